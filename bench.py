"""Benchmark of the Gated DeltaNet layer on GB300 (one JSON line on rank 0).

Step (the timed unit): one decode step of the Qwen3.5-4B-like layer stack --
24 GDN layers (the hybrid's 24 linear-attention layers of "Hybrid transformers
under load: where Gated DeltaNet loses to full attention", braintools.ru), each
with its own fp32 state pool of 256 slots (2 MiB per slot and layer, section
4.1 of that page), B = 64 slots decoding one token each.  The 24 layer calls
are captured in one CUDA graph and replayed (the pure-GPU floor of "Chapter 6:
engine start-up and memory plan", section 6.11); timing uses CUDA events on
the launching stream, outside the capture.

Metric: decode state GB/s = algorithmic bytes per step / time, where a slot
and layer moves 4,325,504 B (state read + write 4,194,304; conv state read +
write 98,304; x 16,384; z 8,192; a, b 128; y 8,192) and each layer call reads
65,920 B of parameters.  The chunked prefill (1 sequence, T = 8192, chunk 64)
is timed too and reported under "prefill" in tokens/s per layer and as a
fraction of the bf16 tensor peak (5.29 MFLOP per token and layer, counted on
the chunk form at C = 64), with its end-to-end figure (inputs copied in from
pinned host memory, y and the final states copied back).  Two more workloads
follow: the wide-GVA one (16/48 heads, 10240 conv channels: a 4 x 32768-token
varlen prefill and verify of r = 4 rows at 4 and 64 slots) under "wide_gva",
and the serving mix (20 sequences of log-uniform length in [500, 30000] packed
into one varlen prefill, then decode of 256 random slots of a 1024-slot pool)
under "serving", the decode step at B = 1, 4, 16 under "decode_small_batch",
and the hybrid's attention layer (decode over paged K/V at 16/4 and 24/2 heads
of 256, prefill at T = 8192, each with its fraction of the measured peak)
under "attention".

--impl reference times the CPU fp64 oracle (test infrastructure) on a bounded
sample of the same workload; it is a deliberately slow reported baseline.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

N_LAYERS = 24
B = 64
POOL = 4 * B
PREFILL_T = 8192
GEOM_ARGS = (16, 32, 128, 128, 4)

# algorithmic bytes of one decode slot-layer and one layer call's parameters
SLOT_BYTES = (2 * 32 * 128 * 128 * 4) + (2 * 3 * 8192 * 2) + 8192 * 2 + 32 * 128 * 2 + 2 * 32 * 2 + 32 * 128 * 2
PARAM_BYTES = 8192 * 4 * 2 + 32 * 4 + 128 * 2
# algorithmic bytes of one prefill token (x, z, y, a, b) and of one sequence's final state and conv state
TOKEN_BYTES = 8192 * 2 + 4096 * 2 + 4096 * 2 + 2 * 32 * 2
STATE_BYTES = 32 * 128 * 128 * 4 + 3 * 8192 * 2
# algorithmic flops per token and layer of the chunk form at C = 64 (16 k-heads, 32 v-heads, d = 128)
C_REF = 64
FLOP_KHEAD = 4 * C_REF * 128                                  # K K^T and Q K^T per k-head
FLOP_VHEAD = C_REF * C_REF / 3 + 2 * C_REF * 256 + 6 * 128 * 128 + 2 * C_REF * 128
FLOP_PER_TOKEN = 16 * FLOP_KHEAD + 32 * FLOP_VHEAD


METRIC = "GDN decode state GB/s (% of HBM peak); chunked-prefill tokens/s/layer (% TC peak)"


def decode_config(world: int) -> dict:
    return {"workload": "Qwen3.5-4B-like GDN decode step: 24 layers x 64 slots, 1 token per slot, "
                        "16 k-heads / 32 v-heads, d_k = d_v = 128, bf16 q/k/v/z, fp32 state (2 MiB per "
                        "slot and layer), pool of 256 slots per layer",
            "layers": N_LAYERS, "slots": B, "pool_slots_per_layer": POOL,
            "working_set_bytes_per_step": N_LAYERS * (B * SLOT_BYTES + PARAM_BYTES),
            "l2": "inputs larger than L2 (6.6 GB touched per step vs 129 MB L2); no flush",
            "parallelism": f"replicas x{world}"}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while it runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "reasons": reasons, "samples": len(rows)}


# -----------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas, no collective on the path)
# -----------------------------------------------------------------------------
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# -----------------------------------------------------------------------------
# the GPU arm
# -----------------------------------------------------------------------------
def _side_stream(torch):
    """A new stream for timed work, after the device has finished everything the
    default stream was given (input initialisation runs there; a side stream
    does not wait for it)."""
    torch.cuda.synchronize()
    return torch.cuda.Stream()


def _dev(stored, torch, device):
    from hybrid_gated_deltanet_gb300 import synth
    if stored.dtype == synth.BF16:
        return torch.from_numpy(np.ascontiguousarray(stored.raw).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(stored.raw)).to(device)


def _rel(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def setup_decode(torch, device, seed: int, n_layers=None, batch=None, pool=None):
    from hybrid_gated_deltanet_gb300 import binding as gb
    from hybrid_gated_deltanet_gb300 import synth
    n_layers, batch, pool = n_layers or N_LAYERS, batch or B, pool or POOL
    geom = synth.QWEN35_4B
    r = synth.rng_for(1, seed)
    cfg = gb.Config(*GEOM_ARGS, chunk=64, act_dtype=gb.BF16)
    p = synth.make_params(geom, r, synth.BF16)
    tok = synth.make_tokens(geom, batch, r, synth.BF16)
    S = synth.make_state(geom, pool, r, std=0.1)
    CS = synth.make_conv_state(geom, pool, r, synth.BF16, std=0.1)
    slots = r.permutation(pool)[:batch].astype(np.int32)
    host = dict(geom=geom, p=p, tok=tok, S=S, CS=CS, slots=slots)
    # layer 0 from the generator; layers 1..23 are device copies (distinct buffers)
    prm0 = gb.Params(conv_w=_dev(p["conv_w"], torch, device), A_log=_dev(p["A_log"], torch, device),
                     norm_w=_dev(p["norm_w"], torch, device))
    s0, c0 = _dev(S, torch, device), _dev(CS, torch, device)
    x0, z0, a0, b0 = (_dev(tok[k], torch, device) for k in ("x", "z", "a", "b"))
    sl = torch.from_numpy(slots).to(device)
    layers = []
    for l in range(n_layers):
        clone = (lambda t: t) if l == 0 else (lambda t: t.clone())
        layers.append(dict(prm=gb.Params(conv_w=clone(prm0.conv_w), A_log=clone(prm0.A_log),
                                         norm_w=clone(prm0.norm_w)),
                           S=clone(s0), C=clone(c0), x=clone(x0), z=clone(z0), a=clone(a0), b=clone(b0),
                           slots=clone(sl), y=torch.empty((batch, geom.value_dim), dtype=torch.bfloat16, device=device)))
    return cfg, host, layers


L2_BYTES = 129 * 1024 * 1024


def small_batch_decode(torch, device, steps, warmup, batches=(1, 4, 16)):
    """The decode step at small batches: per batch, enough layers (each with its own
    pool of 4 B slots) that one step touches at least 4 x L2 of state, replayed from
    a CUDA graph; GB/s of the same algorithmic bytes per slot and layer."""
    out = []
    for bt in batches:
        layer_bytes = bt * SLOT_BYTES + PARAM_BYTES
        n_layers = max(24, -(-4 * L2_BYTES // layer_bytes))
        cfg, _, layers = setup_decode(torch, device, seed=100 + bt, n_layers=n_layers, batch=bt, pool=4 * bt)
        t = time_decode(torch, cfg, layers, steps, warmup)
        us = 1e6 * t / (steps * n_layers)
        out.append({"batch": bt, "layers": n_layers, "working_set_bytes": n_layers * layer_bytes,
                    "us_per_layer": round(us, 3), "gbs": round(layer_bytes / us / 1e3, 1)})
        del layers
        torch.cuda.empty_cache()
    return out


def decode_parity(torch, cfg, host, layers, n_check=8):
    """One decode step on layer 0 checked against the oracle on n_check slots."""
    import oracle
    from hybrid_gated_deltanet_gb300 import binding as gb
    L0 = layers[0]
    S_before = L0["S"].clone()
    C_before = L0["C"].clone()
    gb.gdn_decode_step(cfg, L0["prm"], L0["x"], L0["z"], L0["a"], L0["b"], L0["C"], L0["S"], L0["slots"], L0["y"])
    torch.cuda.synchronize()
    geom, p, tok, S, CS, slots = (host[k] for k in ("geom", "p", "tok", "S", "CS", "slots"))
    yg = L0["y"].float().cpu().numpy()
    ys, yr, ss, sr = [], [], [], []
    for b in range(n_check):
        ref = oracle.run_sequence(geom, tok["x"].f64[b:b + 1], tok["z"].f64[b:b + 1], tok["a"].f64[b:b + 1],
                                  tok["b"].f64[b:b + 1], s0=S.f64[slots[b]], conv0=CS.f64[slots[b]],
                                  conv_w=p["conv_w"].f64, A_log=p["A_log"].f64, norm_w=p["norm_w"].f64)
        ys.append(yg[b]); yr.append(ref["y"][0])
        ss.append(L0["S"][int(slots[b])].cpu().numpy()); sr.append(ref["S"])
    L0["S"].copy_(S_before)
    L0["C"].copy_(C_before)
    return {"y": _rel(ys, yr), "S": _rel(ss, sr), "slots_checked": n_check}


def time_decode(torch, cfg, layers, steps, warmup, use_graph=True, per_step=None):
    """Seconds for `steps` replays of the decode step, timed with CUDA events on the
    launching stream.  If `per_step` is a list, each replay's own duration (an event
    after every replay) is appended to it."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    stream = _side_stream(torch)

    def step():
        for L in layers:
            gb.gdn_decode_step(cfg, L["prm"], L["x"], L["z"], L["a"], L["b"], L["C"], L["S"], L["slots"], L["y"],
                               stream=stream)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step()  # first call outside capture
    torch.cuda.synchronize()
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else step
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(steps):
            run()
            evs[i + 1].record(stream)
    evs[-1].synchronize()
    if per_step is not None:
        per_step.extend(evs[i].elapsed_time(evs[i + 1]) / 1e3 for i in range(steps))
    return evs[0].elapsed_time(evs[-1]) / 1e3  # seconds


def time_decode_e2e(torch, cfg, layers, steps, warmup, graph=False):
    """Same step through the public API, with each step's inputs copied in from
    pinned host memory and its outputs copied back, inside the timed region.
    Three streams pipeline it: layer l's inputs are copied in on a copy stream
    once the previous step's kernel for layer l has read its buffers, layer l
    runs on the compute stream once its inputs have landed and its previous y
    has been read out, and y goes back on a third stream.  The timed region
    ends after the last read-back.  With graph=True one step (its 24 copies in,
    24 API calls and 24 read-backs, on the same three streams) is captured as a
    CUDA graph, as the device-timed step is, and replayed once per step: the
    host-side cost of the eager calls leaves the timed region, the copies stay."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    stream = _side_stream(torch)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    # each layer's x, z, a, b packed into one pinned host buffer and one device
    # buffer (16-byte aligned views): one copy in per layer
    keys = ("x", "z", "a", "b")
    packs = []
    for L in layers:
        sizes = [L[k].numel() for k in keys]
        dbuf = torch.empty(sum(sizes), dtype=L["x"].dtype, device=L["x"].device)
        views, o = {}, 0
        for k, n_el in zip(keys, sizes):
            views[k] = dbuf[o:o + n_el].view(L[k].shape)
            views[k].copy_(L[k])
            o += n_el
        packs.append((dbuf, views, dbuf.cpu().pin_memory()))
    hout = [torch.empty(L["y"].shape, dtype=L["y"].dtype, pin_memory=True) for L in layers]
    h2d = sum(hb.numel() * hb.element_size() for _, _, hb in packs)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    n = len(layers)
    e_in = [torch.cuda.Event() for _ in range(n)]    # inputs of layer l landed
    e_k = [torch.cuda.Event() for _ in range(n)]     # kernel of layer l done
    e_out = [torch.cuda.Event() for _ in range(n)]   # y of layer l copied out
    for l in range(n):  # start state: nothing outstanding
        e_k[l].record(stream)
        e_out[l].record(s_out)

    def step():
        for l, (L, (dbuf, v, hbuf), ho) in enumerate(zip(layers, packs, hout)):
            s_in.wait_event(e_k[l])
            with torch.cuda.stream(s_in):
                dbuf.copy_(hbuf, non_blocking=True)
            e_in[l].record(s_in)
            stream.wait_event(e_in[l])
            stream.wait_event(e_out[l])
            gb.gdn_decode_step(cfg, L["prm"], v["x"], v["z"], v["a"], v["b"], L["C"], L["S"], L["slots"], L["y"],
                               stream=stream)
            e_k[l].record(stream)
            s_out.wait_event(e_k[l])
            with torch.cuda.stream(s_out):
                ho.copy_(L["y"], non_blocking=True)
            e_out[l].record(s_out)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if graph:
        # Replays are serialized, so inside one step no buffer is reused: the kernels
        # wait only for their inputs.  The copies in run ahead on their own stream, in
        # layer order (about 10 us per layer's 1.6 MB here, against about 48 us per
        # layer's kernel), so a wait for copy i covers every layer up to i: layer 0
        # waits for its own, layer 1 for the copies up to layer 4, layer 5 for the
        # last one.  Every other kernel follows its predecessor without a wait, which
        # keeps the programmatic launch (a wait in front of a kernel costs about 4 us).
        ev_fork = torch.cuda.Event()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            ev_fork.record(stream)  # the side streams join the capture here
            s_in.wait_event(ev_fork)
            s_out.wait_event(ev_fork)
            with torch.cuda.stream(s_in):
                for l, (dbuf, v, hbuf) in enumerate(packs):
                    dbuf.copy_(hbuf, non_blocking=True)
                    e_in[l].record(s_in)
            waits = {0: 0, 1: min(4, n - 1), 5: n - 1}  # kernel of layer l: wait for copies up to layer i
            for l, (L, (dbuf, v, hbuf), ho) in enumerate(zip(layers, packs, hout)):
                if l in waits:
                    stream.wait_event(e_in[waits[l]])
                gb.gdn_decode_step(cfg, L["prm"], v["x"], v["z"], v["a"], v["b"], L["C"], L["S"], L["slots"],
                                   L["y"], stream=stream)
                e_k[l].record(stream)
                s_out.wait_event(e_k[l])
                with torch.cuda.stream(s_out):
                    ho.copy_(L["y"], non_blocking=True)
            e_out[n - 1].record(s_out)
            stream.wait_event(e_in[n - 1])  # rejoin: every copy of the step is in the graph
            stream.wait_event(e_out[n - 1])
        with torch.cuda.stream(stream):  # a graph replays on the current stream
            for _ in range(warmup):
                g.replay()
        torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    s_in.wait_event(ev0)
    for _ in range(steps):
        if graph:
            with torch.cuda.stream(stream):  # a graph replays on the current stream
                g.replay()
        else:
            step()
    if not graph:  # (a replayed graph ends with its streams joined: the read-backs are in it)
        for l in range(n):  # every read-back of the last step precedes the end mark
            stream.wait_event(e_out[l])
    ev1.record(stream)
    ev1.synchronize()
    return ev0.elapsed_time(ev1) / 1e3, h2d, d2h


def prefill_measure(torch, device, steps, warmup, seed, check=True, e2e=True):
    """Chunked prefill of one 8192-token sequence: parity on sampled heads, then timing."""
    import oracle
    from hybrid_gated_deltanet_gb300 import binding as gb
    from hybrid_gated_deltanet_gb300 import synth
    geom = synth.QWEN35_4B
    r = synth.rng_for(2, seed)
    cfg = gb.Config(*GEOM_ARGS, chunk=64, act_dtype=gb.BF16)
    p = synth.make_params(geom, r, synth.BF16)
    tok = synth.make_tokens(geom, PREFILL_T, r, synth.BF16)
    prm = gb.Params(conv_w=_dev(p["conv_w"], torch, device), A_log=_dev(p["A_log"], torch, device),
                    norm_w=_dev(p["norm_w"], torch, device))
    x, z, a, b = (_dev(tok[k], torch, device) for k in ("x", "z", "a", "b"))
    s_fin = torch.empty((32, 128, 128), device=device)
    c_fin = torch.empty((3, 8192), dtype=torch.bfloat16, device=device)
    y = torch.empty((PREFILL_T, 4096), dtype=torch.bfloat16, device=device)
    ws = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_CHUNK_PREFILL, PREFILL_T), dtype=torch.uint8, device=device)
    stream = _side_stream(torch)

    def call():
        gb.gdn_chunk_prefill(cfg, prm, x, z, a, b, None, None, s_fin, c_fin, y, ws, stream=stream)

    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    errs = None
    if check:
        heads = [0, 13, 31]
        ref = oracle.run_sequence(geom, tok["x"].f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, heads=heads,
                                  conv_w=p["conv_w"].f64, A_log=p["A_log"].f64, norm_w=p["norm_w"].f64)
        cols = np.concatenate([np.arange(j * 128, (j + 1) * 128) for j in heads])
        yg = y.float().cpu().numpy()
        sg = s_fin.cpu().numpy()
        errs = {"y": _rel(yg[:, cols], ref["y"][:, cols]), "S": _rel(sg[heads], ref["S"][heads]),
                "heads_checked": heads}
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps):
            call()
        ev1.record(stream)
    ev1.synchronize()
    t = ev0.elapsed_time(ev1) / 1e3 / steps
    e2e_line = prefill_e2e(torch, cfg, prm, (x, z, a, b), s_fin, c_fin, y, ws, steps, warmup) if e2e else None
    return t, errs, e2e_line


def prefill_e2e(torch, cfg, prm, inputs, s_fin, c_fin, y, ws, steps, warmup):
    """The same prefill through the public API with its inputs copied in from
    pinned host memory (x, z, a, b packed in one buffer: one copy) and y, the
    final state and the final conv state copied back, all inside the timed
    region.  Calls are pipelined as a serving loop would run them: two sets of
    device buffers, the copy in of call i on a copy stream while call i - 1
    computes, its read-back on a third stream (the host link carries each
    direction at about 0.2 TB/s, so call i's 202 MB in take longer than its
    kernels)."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    stream = _side_stream(torch)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    sizes = [t.numel() for t in inputs]
    sets = []
    for _ in range(2):  # device inputs, outputs and workspace per set
        dbuf = torch.empty(sum(sizes), dtype=inputs[0].dtype, device=inputs[0].device)
        views, o = [], 0
        for t, n_el in zip(inputs, sizes):
            views.append(dbuf[o:o + n_el].view(t.shape))
            views[-1].copy_(t)
            o += n_el
        outs = (torch.empty_like(y), torch.empty_like(s_fin), torch.empty_like(c_fin))
        sets.append((dbuf, views, outs, torch.empty_like(ws)))
    hin = sets[0][0].cpu().pin_memory()
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in sets[0][2]]
    h2d = hin.numel() * hin.element_size()
    d2h = sum(t.numel() * t.element_size() for t in hout)
    e_in = [torch.cuda.Event() for _ in range(2)]   # inputs of set k landed
    e_k = [torch.cuda.Event() for _ in range(2)]    # call on set k done (its inputs free)
    e_out = [torch.cuda.Event() for _ in range(2)]  # outputs of set k read back (free)
    for k in range(2):
        e_k[k].record(stream)
        e_out[k].record(s_out)

    def step(i):
        k = i & 1
        dbuf, (x, z, a, b), (yo, so, co), wsk = sets[k]
        s_in.wait_event(e_k[k])
        with torch.cuda.stream(s_in):
            dbuf.copy_(hin, non_blocking=True)
        e_in[k].record(s_in)
        stream.wait_event(e_in[k])
        stream.wait_event(e_out[k])
        gb.gdn_chunk_prefill(cfg, prm, x, z, a, b, None, None, so, co, yo, wsk, stream=stream)
        e_k[k].record(stream)
        s_out.wait_event(e_k[k])
        with torch.cuda.stream(s_out):
            for ho, t in zip(hout, (yo, so, co)):
                ho.copy_(t, non_blocking=True)
        e_out[k].record(s_out)

    torch.cuda.synchronize()
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    s_in.wait_event(ev0)
    for i in range(steps):
        step(i)
    for k in range(2):  # every read-back precedes the end mark
        stream.wait_event(e_out[k])
    ev1.record(stream)
    ev1.synchronize()
    t = ev0.elapsed_time(ev1) / 1e3 / steps
    return {"value": round(PREFILL_T / t, 1), "unit": "tokens/s/layer", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(1e3 * t, 4), "pipelined": True}


# -----------------------------------------------------------------------------
# the CPU oracle, timed (reported baseline and the reference arm)
# -----------------------------------------------------------------------------
def _oracle_decode_inputs(n_slots: int, seed: int):
    from hybrid_gated_deltanet_gb300 import synth
    geom = synth.QWEN35_4B
    r = synth.rng_for(1, 10_000 + seed)
    p = synth.make_params(geom, r, synth.BF16)
    tok = synth.make_tokens(geom, n_slots, r, synth.BF16)
    S = synth.make_state(geom, n_slots, r, std=0.1)
    CS = synth.make_conv_state(geom, n_slots, r, synth.BF16, std=0.1)
    return geom, p, tok, S, CS


def oracle_decode_rate(n_slots: int, min_seconds: float = 0.0, seed: int = 7, inputs=None, threads=None):
    """Oracle decode of n_slots slots of one layer (repeated from the same initial
    states until min_seconds have passed): GB/s of the same algorithmic bytes."""
    import oracle
    geom, p, tok, S, CS = inputs or _oracle_decode_inputs(n_slots, seed)
    threads = threads or oracle.default_threads()
    kw = dict(conv_w=p["conv_w"].f64, A_log=p["A_log"].f64, norm_w=p["norm_w"].f64, threads=threads)
    done, t0 = 0, time.perf_counter()
    while True:
        for b in range(n_slots):
            oracle.run_sequence(geom, tok["x"].f64[b:b + 1], tok["z"].f64[b:b + 1], tok["a"].f64[b:b + 1],
                                tok["b"].f64[b:b + 1], s0=S.f64[b], conv0=CS.f64[b], **kw)
        done += n_slots
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return done * SLOT_BYTES / dt / 1e9, dt, threads, done


def oracle_prefill_rate(T: int, n_heads: int, min_seconds: float = 0.0, seed: int = 8):
    """Oracle prefill of T tokens on n_heads of the 32 v-heads (repeated until
    min_seconds have passed), scaled to tokens/s for a whole layer."""
    import oracle
    from hybrid_gated_deltanet_gb300 import synth
    geom = synth.QWEN35_4B
    r = synth.rng_for(2, 10_000 + seed)
    p = synth.make_params(geom, r, synth.BF16)
    tok = synth.make_tokens(geom, T, r, synth.BF16)
    threads = oracle.default_threads()
    heads = list(range(n_heads))
    x, z, a, b = (np.asarray(tok[k].f64) for k in ("x", "z", "a", "b"))
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.run_sequence(geom, x, z, a, b, heads=heads, conv_w=p["conv_w"].f64, A_log=p["A_log"].f64,
                            norm_w=p["norm_w"].f64, threads=threads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    # tokens/s per layer: all 32 v-heads take 32/n_heads times as long
    return reps * T / (dt * 32 / n_heads), dt, threads


def _src_hash(names: str) -> str:
    """First 16 hex digits of the sha256 of the named csrc files, concatenated
    in the order given (names separated by '+')."""
    import hashlib
    h = hashlib.sha256()
    for name in names.split("+"):
        with open(os.path.join(ROOT, "hybrid_gated_deltanet_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, source: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed since the counters were taken (hash recorded there)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.strip().split("=", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_sha256_16") != _src_hash(source):
        return None
    try:
        return int(float(vals["dram_bytes_per_full_launch"]))
    except (KeyError, ValueError):
        return None


def profile_case(args):
    """Small cases for ncu captures (a few GB on the device, few launches)."""
    import torch
    from hybrid_gated_deltanet_gb300 import build as gbuild
    from hybrid_gated_deltanet_gb300 import binding as gb
    gbuild.build()
    device = torch.device("cuda", 0)
    if args.case == "decode-small":
        global N_LAYERS, B, POOL
        N_LAYERS = 2  # 2 x 64 slots x 2 MiB of state: 256 MiB, larger than L2
        B = args.batch
        POOL = max(4 * B, 2)
        cfg, host, layers = setup_decode(torch, device, seed=0)
        t = time_decode(torch, cfg, layers, args.steps, args.warmup, use_graph=not args.no_graph)
        us = 1e6 * t / (args.steps * N_LAYERS)
        print(json.dumps({"case": args.case, "batch": B, "launches": (args.steps + args.warmup + 1) * N_LAYERS,
                          "us_per_launch": round(us, 3),
                          "gbs": round((B * SLOT_BYTES + PARAM_BYTES) / us / 1e3, 1),
                          "slices": os.environ.get("GDN_DECODE_SLICES", "auto")}))
    elif args.case == "decode-batches":
        batches = tuple(int(v) for v in args.batches.split(","))
        for rec in small_batch_decode(torch, device, args.steps, args.warmup, batches=batches):
            print(json.dumps(dict(rec, slices=os.environ.get("GDN_DECODE_SLICES", "auto"),
                                  clustered=os.environ.get("GDN_DECODE_CLUSTERED", "auto"))))
    elif args.case == "serving":
        print(json.dumps(serving_measure(torch, device, args.steps, args.warmup)))
    elif args.case == "prefill-varlen":
        print(json.dumps(varlen_prefill_case(torch, device, args.steps, args.warmup)))
    elif args.case == "ckpt":
        print(json.dumps(ckpt_measure(torch, device, args.steps, args.warmup)))
    elif args.case == "proj-prefill":
        print(json.dumps(proj_prefill_case(torch, device, args.steps, args.warmup)))
    elif args.case == "attn-small":
        print(json.dumps(attn_small_case(torch, device, args.steps, args.warmup)))
    elif args.case == "attn-wide":
        print(json.dumps(attn_wide_case(torch, device, args.steps, args.warmup)))
    elif args.case == "attn":
        for rec in attn_measure(torch, device, args.steps, args.warmup):
            print(json.dumps(rec))
    elif args.case == "proj-decode":
        print(json.dumps(proj_decode_case(torch, device, args.steps, args.warmup, args.batch)))
    elif args.case == "layer":
        for rec in layer_measure(torch, device, args.steps, args.warmup):
            print(json.dumps(rec))
    elif args.case == "verify":
        print(json.dumps(wide_prefill_measure(torch, device, args.steps, args.warmup)))
        for nb in (4, 64):
            print(json.dumps(verify_measure(torch, device, args.steps, args.warmup, batch=nb)))
    else:
        t, _, _ = prefill_measure(torch, device, args.steps, args.warmup, seed=0, check=False, e2e=False)
        print(json.dumps({"case": args.case, "ms_per_call": round(1e3 * t, 4)}))
    return 0


def varlen_prefill_case(torch, device, steps, warmup, n_seq=4, T=2048):
    """One varlen prefill of n_seq x T tokens (16/32 heads, d = 128): the prep kernel
    runs as one launch over all chunks (no segments), for ncu captures."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    from hybrid_gated_deltanet_gb300 import synth
    r = synth.rng_for(5, 0)
    cfg = gb.Config(*GEOM_ARGS, chunk=64, act_dtype=gb.BF16)
    p = synth.make_params(synth.QWEN35_4B, r, synth.BF16)
    prm = gb.Params(conv_w=_dev(p["conv_w"], torch, device), A_log=_dev(p["A_log"], torch, device),
                    norm_w=_dev(p["norm_w"], torch, device))
    g = torch.Generator(device=device)
    g.manual_seed(5)
    bf = torch.bfloat16
    N = n_seq * T
    x = torch.randn((N, 8192), generator=g, device=device).to(bf)
    z = torch.randn((N, 4096), generator=g, device=device).to(bf)
    a = torch.randn((N, 32), generator=g, device=device).to(bf)
    b = torch.randn((N, 32), generator=g, device=device).to(bf)
    y = torch.empty((N, 4096), dtype=bf, device=device)
    S = torch.zeros((n_seq, 32, 128, 128), device=device)
    Cp = torch.zeros((n_seq, 3, 8192), dtype=bf, device=device)
    cu = torch.arange(0, N + 1, T, dtype=torch.int32, device=device)
    sl = torch.arange(n_seq, dtype=torch.int32, device=device)
    ws = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_VARLEN_PREFILL, N, n_seq), dtype=torch.uint8, device=device)
    stream = _side_stream(torch)
    with torch.cuda.stream(stream):
        for _ in range(warmup + steps):
            gb.gdn_varlen_prefill(cfg, prm, x, z, a, b, cu, sl, None, Cp, S, y, ws, stream=stream)
    torch.cuda.synchronize()
    return {"case": "prefill-varlen", "n_seq": n_seq, "tokens_each": T, "launches": warmup + steps}


def proj_prefill_case(torch, device, steps, warmup, T=8192):
    """The in-projection GEMM of a T-token prefill alone (12352 x 2560 bf16 weights),
    warmup + steps launches, for ncu captures."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    g = torch.Generator(device=device)
    g.manual_seed(12)
    bf = torch.bfloat16
    w = (torch.randn((12352, 2560), generator=g, device=device) / 50).to(bf)
    h = torch.randn((T, 2560), generator=g, device=device).to(bf)
    u = torch.empty((T, 12352), dtype=bf, device=device)
    for _ in range(warmup + steps):
        gb.gdn_proj_gemm(h, w, u)
    torch.cuda.synchronize()
    return {"case": "proj-prefill", "tokens": T, "launches": warmup + steps}


def attn_wide_case(torch, device, steps, warmup):
    """Wide-GQA decode attention alone (24 query / 2 kv-heads of 256, pages of 528,
    4 sequences x 32768 cached tokens: 268 MB of K and V); warmup + steps calls, for
    ncu captures."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    g = torch.Generator(device=device)
    g.manual_seed(14)
    bf = torch.bfloat16
    cfg = gb.AttnConfig(24, 2, 256, 528)
    B, L = 4, 32768
    per = (L + 1 + 527) // 528
    kp = torch.randn((B * per, 2, 528, 256), generator=g, device=device).to(bf)
    vp = torch.randn((B * per, 2, 528, 256), generator=g, device=device).to(bf)
    table = torch.randperm(B * per, generator=g, device=device).to(torch.int32).view(B, per)
    lens = torch.full((B,), L, dtype=torch.int32, device=device)
    q = torch.randn((B, 24, 256), generator=g, device=device).to(bf)
    kn = torch.randn((B, 2, 256), generator=g, device=device).to(bf)
    o = torch.empty((B, 24, 256), dtype=bf, device=device)
    ws = torch.empty(max(16, gb.gdn_attn_workspace_size(cfg, B, L + 1)), dtype=torch.uint8, device=device)
    torch.cuda.synchronize()
    for _ in range(warmup + steps):
        gb.gdn_attn_decode(cfg, q, kn, kn, kp, vp, table, lens, L + 1, o, ws)
    torch.cuda.synchronize()
    return {"case": "attn-wide", "launches": warmup + steps}


def attn_small_case(torch, device, steps, warmup):
    """Decode attention (16 sequences x 8192 cached tokens) and prefill attention (one
    2048-token prompt), 16 query / 4 kv-heads of 256, pages of 16; warmup + steps of
    each, for ncu captures (about 1.2 GB on the device)."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    g = torch.Generator(device=device)
    g.manual_seed(13)
    bf = torch.bfloat16
    cfg = gb.AttnConfig(16, 4, 256, 16)
    B, L = 16, 8192
    per = (L + 1 + 15) // 16
    kp = torch.randn((B * per, 4, 16, 256), generator=g, device=device).to(bf)
    vp = torch.randn((B * per, 4, 16, 256), generator=g, device=device).to(bf)
    table = torch.randperm(B * per, generator=g, device=device).to(torch.int32).view(B, per)
    lens = torch.full((B,), L, dtype=torch.int32, device=device)
    q = torch.randn((B, 16, 256), generator=g, device=device).to(bf)
    kn = torch.randn((B, 4, 256), generator=g, device=device).to(bf)
    o = torch.empty((B, 16, 256), dtype=bf, device=device)
    ws = torch.empty(max(16, gb.gdn_attn_workspace_size(cfg, B, L + 1)), dtype=torch.uint8, device=device)
    T = 2048
    tab2 = torch.arange(T // 16, dtype=torch.int32, device=device).view(1, -1)
    cu = torch.tensor([0, T], dtype=torch.int32, device=device)
    ctx = torch.zeros(1, dtype=torch.int32, device=device)
    q2 = torch.randn((T, 16, 256), generator=g, device=device).to(bf)
    k2 = torch.randn((T, 4, 256), generator=g, device=device).to(bf)
    o2 = torch.empty((T, 16, 256), dtype=bf, device=device)
    torch.cuda.synchronize()
    for _ in range(warmup + steps):
        gb.gdn_attn_decode(cfg, q, kn, kn, kp, vp, table, lens, L + 1, o, ws)
        gb.gdn_attn_prefill(cfg, q2, k2, k2, kp, vp, tab2, cu, ctx, o2)
    torch.cuda.synchronize()
    return {"case": "attn-small", "launches": 4 * (warmup + steps)}


ATTN_DECODE_CASES = ((16, 4, 256, 16, 1, 8192), (16, 4, 256, 16, 16, 8192), (16, 4, 256, 16, 64, 8192),
                     (24, 2, 256, 528, 4, 32768))
ATTN_PREFILL_CASES = ((16, 4, 256, 16, [(0, 8192)]), (16, 4, 256, 128, [(0, 8192)]),
                      (16, 4, 256, 16, [(8192, 512)] * 4), (24, 2, 256, 528, [(0, 32768)]))


def attn_measure(torch, device, steps, warmup, decode_cases=ATTN_DECODE_CASES, prefill_cases=ATTN_PREFILL_CASES):
    """Decode attention over a paged KV cache (timing only, N(0, 1) bf16 q, K, V
    drawn on the device): 16 query / 4 kv-heads of 256 with pages of 16 tokens at
    B = 1, 16, 64 sequences of 8192 cached tokens, and 24 / 2 heads with pages of
    528 tokens at B = 4 sequences of 32768.  Bytes: K and V of every cached
    token read once, the new token's K and V written, q and o.  Then prefill
    attention (flops: 4 d Hq per (query, visible key) pair)."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    out = []
    g = torch.Generator(device=device)
    g.manual_seed(11)
    bf = torch.bfloat16
    for Hq, Hkv, D, page, B, L in decode_cases:
        cfg = gb.AttnConfig(Hq, Hkv, D, page)
        per = (L + 1 + page - 1) // page
        n_pages = B * per
        kp = torch.randn((n_pages, Hkv, page, D), generator=g, device=device).to(bf)
        vp = torch.randn((n_pages, Hkv, page, D), generator=g, device=device).to(bf)
        table = torch.randperm(n_pages, generator=g, device=device).to(torch.int32).view(B, per)
        lens = torch.full((B,), L, dtype=torch.int32, device=device)
        q = torch.randn((B, Hq, D), generator=g, device=device).to(bf)
        kn = torch.randn((B, Hkv, D), generator=g, device=device).to(bf)
        vn = torch.randn((B, Hkv, D), generator=g, device=device).to(bf)
        o = torch.empty((B, Hq, D), dtype=bf, device=device)
        nws = gb.gdn_attn_workspace_size(cfg, B, L + 1)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=device)
        stream = _side_stream(torch)

        def step():
            gb.gdn_attn_decode(cfg, q, kn, vn, kp, vp, table, lens, L + 1, o, ws, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(warmup):
                step()
        torch.cuda.synchronize()
        n = max(20, steps)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                step()
            e1.record(stream)
        e1.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / n
        nbytes = B * (L * Hkv * D * 2 * 2 + Hkv * D * 2 * 2 * 2 + 2 * Hq * D * 2)
        out.append({"case": "attn", "heads": f"{Hq}/{Hkv}x{D}", "page": page, "batch": B, "context": L,
                    "splits": None if nws == 0 else nws // (B * Hq * (D + 2) * 4),
                    "us": round(1e6 * t, 2), "gbs": round(nbytes / t / 1e9, 1)})
        del kp, vp
    # prefill: (cached, new) tokens per sequence; flops 4 d Hq per (query, visible key) pair
    for Hq, Hkv, D, page, seqs in prefill_cases:
        cfg = gb.AttnConfig(Hq, Hkv, D, page)
        per = [(c + n + page - 1) // page for c, n in seqs]
        n_pages, max_pages = sum(per), max(per)
        N = sum(n for _, n in seqs)
        kp = torch.randn((n_pages, Hkv, page, D), generator=g, device=device).to(bf)
        vp = torch.randn((n_pages, Hkv, page, D), generator=g, device=device).to(bf)
        perm = torch.randperm(n_pages, generator=g, device=device).to(torch.int32)
        table = torch.full((len(seqs), max_pages), -1, dtype=torch.int32, device=device)
        o0 = 0
        for i, pcount in enumerate(per):
            table[i, :pcount] = perm[o0:o0 + pcount]
            o0 += pcount
        cu = torch.tensor([0] + list(np.cumsum([n for _, n in seqs])), dtype=torch.int32, device=device)
        ctx = torch.tensor([c for c, _ in seqs], dtype=torch.int32, device=device)
        q = torch.randn((N, Hq, D), generator=g, device=device).to(bf)
        kn = torch.randn((N, Hkv, D), generator=g, device=device).to(bf)
        vn = torch.randn((N, Hkv, D), generator=g, device=device).to(bf)
        o = torch.empty((N, Hq, D), dtype=bf, device=device)
        stream = _side_stream(torch)

        def pstep():
            gb.gdn_attn_prefill(cfg, q, kn, vn, kp, vp, table, cu, ctx, o, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(warmup):
                pstep()
        torch.cuda.synchronize()
        n = max(5, steps // 4)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                pstep()
            e1.record(stream)
        e1.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / n
        pairs = sum(nn * c + nn * (nn + 1) // 2 for c, nn in seqs)
        fl = 4.0 * D * Hq * pairs
        out.append({"case": "attn-prefill", "heads": f"{Hq}/{Hkv}x{D}", "page": page, "seqs": seqs[:1],
                    "n_seq": len(seqs), "ms": round(1e3 * t, 3), "tflops": round(fl / t / 1e12, 1),
                    "tokens_per_s": round(N / t, 1)})
        del kp, vp
    return out


def proj_decode_case(torch, device, steps, warmup, batch):
    """The two projections of a decode step alone (`batch` tokens, model width
    2560, one layer's weights: 84 MB), for ncu captures: in-projection then
    out-projection, warmup + steps times."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    from hybrid_gated_deltanet_gb300 import synth
    geom = synth.QWEN35_4B
    hid, vd = synth.HIDDEN, geom.value_dim
    n_in = geom.conv_channels + vd + 2 * geom.n_v_heads
    g = torch.Generator(device=device)
    g.manual_seed(9)
    bf = torch.bfloat16
    w_in = (torch.randn((n_in, hid), generator=g, device=device) / hid ** 0.5).to(bf)
    w_out = (torch.randn((hid, vd), generator=g, device=device) / vd ** 0.5).to(bf)
    h = torch.randn((batch, hid), generator=g, device=device).to(bf)
    u = torch.empty((batch, n_in), dtype=bf, device=device)
    y = torch.randn((batch, vd), generator=g, device=device).to(bf)
    o = torch.empty((batch, hid), dtype=bf, device=device)
    nb = max(gb.gdn_proj_workspace_size(batch, n_in, hid), gb.gdn_proj_workspace_size(batch, hid, vd))
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=device)
    for _ in range(warmup + steps):
        gb.gdn_proj_gemm(h, w_in, u, ws)
        gb.gdn_proj_gemm(y, w_out, o, ws)
    torch.cuda.synchronize()
    return {"case": "proj-decode", "batch": batch, "launches": 2 * (warmup + steps)}


def layer_measure(torch, device, steps, warmup, n_layers=4, batch=64):
    """The layer between its projections (model width 2560, Qwen3.5-4B-like
    geometry; timing only, N(0, 1) inputs and N(0, 1/k) weights drawn on the
    device from a fixed seed):
    * the two projection GEMMs of a T = 8192 prefill (tensor-core TFLOP/s);
    * gdn_layer_varlen_prefill of one T = 8192 sequence (tokens/s);
    * gdn_layer_decode of `batch` slots, round-robin over `n_layers` layers
      with their own weights and pools (more than L2 in total), and its
      in-projection alone (weight GB/s).
    Every case is replayed from a CUDA graph (device time)."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    from hybrid_gated_deltanet_gb300 import synth
    geom = synth.QWEN35_4B
    hid = synth.HIDDEN
    cfg = gb.Config(*GEOM_ARGS, chunk=64, act_dtype=gb.BF16)
    r = synth.rng_for(6, 0)
    p = synth.make_params(geom, r, synth.BF16)
    prm = gb.Params(conv_w=_dev(p["conv_w"], torch, device), A_log=_dev(p["A_log"], torch, device),
                    norm_w=_dev(p["norm_w"], torch, device))
    g = torch.Generator(device=device)
    g.manual_seed(6)
    bf = torch.bfloat16
    n_in = geom.conv_channels + geom.value_dim + 2 * geom.n_v_heads
    vd = geom.value_dim
    projs = [gb.Proj((torch.randn((n_in, hid), generator=g, device=device) / hid ** 0.5).to(bf),
                     (torch.randn((hid, vd), generator=g, device=device) / vd ** 0.5).to(bf)) for _ in range(n_layers)]
    stream = _side_stream(torch)

    def timed(fn, n):
        """Device time per fn() call: fn is captured once in a CUDA graph and replayed,
        so host launch costs (tensor-map encoding, ctypes) do not count."""
        torch.cuda.synchronize()  # inputs made on the default stream are complete
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            fn()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                graph.replay()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    out = []
    T = PREFILL_T
    h = torch.randn((T, hid), generator=g, device=device).to(bf)
    u = torch.empty((T, n_in), dtype=bf, device=device)
    yv = torch.randn((T, vd), generator=g, device=device).to(bf)
    o = torch.empty((T, hid), dtype=bf, device=device)
    n = max(10, steps)
    t_in = timed(lambda: gb.gdn_proj_gemm(h, projs[0].w_in, u, stream=stream), n)
    t_out = timed(lambda: gb.gdn_proj_gemm(yv, projs[0].w_out, o, stream=stream), n)  # T tokens: no split, no workspace
    for name, t, nn_, kk in (("in", t_in, n_in, hid), ("out", t_out, hid, vd)):
        fl = 2.0 * T * nn_ * kk
        out.append({"case": "layer", "what": f"{name}-projection GEMM", "tokens": T, "n_out": nn_, "k": kk,
                    "us": round(1e6 * t, 2), "tflops": round(fl / t / 1e12, 1)})
    # whole layer, one T = 8192 sequence
    S = torch.zeros((1, 32, 128, 128), device=device)
    Cp = torch.zeros((1, 3, 8192), dtype=bf, device=device)
    cu = torch.tensor([0, T], dtype=torch.int32, device=device)
    sl = torch.zeros(1, dtype=torch.int32, device=device)
    ws = torch.empty(gb.gdn_layer_workspace_size(cfg, gb.OP_LAYER_VARLEN_PREFILL, T, 1, hid), dtype=torch.uint8,
                     device=device)
    t_pf = timed(lambda: gb.gdn_layer_varlen_prefill(cfg, prm, projs[0], h, cu, sl, None, Cp, S, o, ws,
                                                      stream=stream), n)
    fl_layer = FLOP_PER_TOKEN * T + 2.0 * T * (n_in * hid + hid * vd)
    out.append({"case": "layer", "what": "gdn_layer_varlen_prefill", "tokens": T, "ms": round(1e3 * t_pf, 4),
                "tokens_per_s": round(T / t_pf, 1), "tflops": round(fl_layer / t_pf / 1e12, 1)})
    del h, u, yv, o, ws
    # decode: batch slots per layer, n_layers layers round-robin
    pools = []
    for _ in range(n_layers):
        pools.append((torch.randn((batch, 32, 128, 128), generator=g, device=device) * 0.1,
                      (torch.randn((batch, 3, 8192), generator=g, device=device) * 0.1).to(bf)))
    hd = torch.randn((batch, hid), generator=g, device=device).to(bf)
    od = torch.empty((batch, hid), dtype=bf, device=device)
    si = torch.arange(batch, dtype=torch.int32, device=device)
    wsd = torch.empty(gb.gdn_layer_workspace_size(cfg, gb.OP_LAYER_DECODE, batch, 1, hid), dtype=torch.uint8,
                      device=device)
    wsp = torch.empty(max(16, gb.gdn_proj_workspace_size(batch, n_in, hid), gb.gdn_proj_workspace_size(batch, hid, vd)),
                      dtype=torch.uint8, device=device)
    ud = torch.empty((batch, n_in), dtype=bf, device=device)

    def dec_all():
        for li in range(n_layers):
            gb.gdn_layer_decode(cfg, prm, projs[li], hd, pools[li][1], pools[li][0], si, od, wsd, stream=stream)

    def inproj_all():
        for li in range(n_layers):
            gb.gdn_proj_gemm(hd, projs[li].w_in, ud, wsp, stream=stream)

    yd = torch.randn((batch, vd), generator=g, device=device).to(bf)

    def outproj_all():
        for li in range(n_layers):
            gb.gdn_proj_gemm(yd, projs[li].w_out, od, wsp, stream=stream)

    nd = max(20, steps)
    t_dec = timed(dec_all, nd) / n_layers
    t_ip = timed(inproj_all, nd) / n_layers
    t_op = timed(outproj_all, nd) / n_layers
    wbytes = 2 * (n_in * hid + hid * vd)
    dec_bytes = batch * SLOT_BYTES + PARAM_BYTES + wbytes + 2 * batch * hid * 2 - batch * (8192 + 4096 + 64) * 2 \
        - batch * 4096 * 2
    out.append({"case": "layer", "what": "gdn_layer_decode", "batch": batch, "layers": n_layers,
                "us_per_layer": round(1e6 * t_dec, 2), "algorithmic_bytes": dec_bytes,
                "gbs": round(dec_bytes / t_dec / 1e9, 1)})
    out.append({"case": "layer", "what": "decode in-projection GEMM", "batch": batch,
                "us": round(1e6 * t_ip, 2), "weight_gbs": round(2 * n_in * hid / t_ip / 1e9, 1)})
    out.append({"case": "layer", "what": "decode out-projection GEMM", "batch": batch,
                "us": round(1e6 * t_op, 2), "weight_gbs": round(2 * hid * vd / t_op / 1e9, 1)})
    return out


def ckpt_measure(torch, device, steps, warmup, every=1024):
    """The T = 8192 prefill with a prefix snapshot every `every` tokens (into pool
    slots) against the same prefill without snapshots (timing only)."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    from hybrid_gated_deltanet_gb300 import synth
    r = synth.rng_for(2, 5)
    cfg = gb.Config(*GEOM_ARGS, chunk=64, act_dtype=gb.BF16)
    p = synth.make_params(synth.QWEN35_4B, r, synth.BF16)
    prm = gb.Params(conv_w=_dev(p["conv_w"], torch, device), A_log=_dev(p["A_log"], torch, device),
                    norm_w=_dev(p["norm_w"], torch, device))
    g = torch.Generator(device=device)
    g.manual_seed(5)
    bf, T = torch.bfloat16, PREFILL_T
    x = torch.randn((T, 8192), generator=g, device=device).to(bf)
    z = torch.randn((T, 4096), generator=g, device=device).to(bf)
    a = torch.randn((T, 32), generator=g, device=device).to(bf)
    b = torch.randn((T, 32), generator=g, device=device).to(bf)
    y = torch.empty((T, 4096), dtype=bf, device=device)
    n_ck = T // every
    S = torch.zeros((1 + n_ck, 32, 128, 128), device=device)
    Cp = torch.zeros((1 + n_ck, 3, 8192), dtype=bf, device=device)
    cu = torch.tensor([0, T], dtype=torch.int32, device=device)
    sl = torch.zeros(1, dtype=torch.int32, device=device)
    off = torch.tensor([0, n_ck], dtype=torch.int32, device=device)
    ck = torch.arange(1, 1 + n_ck, dtype=torch.int32, device=device)
    ws = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_VARLEN_PREFILL, T, 1), dtype=torch.uint8, device=device)
    stream = _side_stream(torch)

    def plain():
        gb.gdn_varlen_prefill(cfg, prm, x, z, a, b, cu, sl, None, Cp, S, y, ws, stream=stream)

    def snap():
        gb.gdn_varlen_prefill_ckpt(cfg, prm, x, z, a, b, cu, sl, None, Cp, S, y, every, off, ck, ws, stream=stream)

    def timed(fn, n):
        torch.cuda.synchronize()  # inputs made on the default stream are complete
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    n = max(10, steps)
    t0, t1 = timed(plain, n), timed(snap, n)
    return {"case": "ckpt", "tokens": T, "every": every, "snapshots": n_ck,
            "snapshot_bytes": n_ck * (32 * 128 * 128 * 4 + 3 * 8192 * 2),
            "ms_plain": round(1e3 * t0, 4), "ms_with_snapshots": round(1e3 * t1, 4),
            "overhead_pct": round(100 * (t1 / t0 - 1), 2)}


def wide_prefill_measure(torch, device, steps, warmup, n_seq=4, T=32768):
    """The wide-GVA prefill (16/48 heads, d = 128, 10240 conv channels): n_seq
    sequences of T tokens packed into one gdn_varlen_prefill call, each into its
    own pool slot (the prefill that precedes the verify steps of that workload).
    Timing only: N(0, 1) inputs drawn on the device from a fixed seed."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    from hybrid_gated_deltanet_gb300 import synth
    geom = synth.WIDE_GVA
    hv, dd, cch = geom.n_v_heads, geom.d_k, geom.conv_channels
    cfg = gb.Config(geom.n_k_heads, hv, dd, dd, geom.d_conv, chunk=64, act_dtype=gb.BF16)
    r_ = synth.rng_for(3, 8)
    p = synth.make_params(geom, r_, synth.BF16)
    prm = gb.Params(conv_w=_dev(p["conv_w"], torch, device), A_log=_dev(p["A_log"], torch, device),
                    norm_w=_dev(p["norm_w"], torch, device))
    g = torch.Generator(device=device)
    g.manual_seed(8)
    bf = torch.bfloat16
    N = n_seq * T
    x = torch.randn((N, cch), generator=g, device=device).to(bf)
    z = torch.randn((N, hv * dd), generator=g, device=device).to(bf)
    a = torch.randn((N, hv), generator=g, device=device).to(bf)
    b = torch.randn((N, hv), generator=g, device=device).to(bf)
    y = torch.empty((N, hv * dd), dtype=bf, device=device)
    S = torch.zeros((n_seq, hv, dd, dd), device=device)
    Cp = torch.zeros((n_seq, geom.d_conv - 1, cch), dtype=bf, device=device)
    cu = torch.arange(0, N + 1, T, dtype=torch.int32, device=device)
    sl = torch.arange(n_seq, dtype=torch.int32, device=device)
    ws = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_VARLEN_PREFILL, N, n_seq), dtype=torch.uint8, device=device)
    stream = _side_stream(torch)

    def call():
        gb.gdn_varlen_prefill(cfg, prm, x, z, a, b, cu, sl, None, Cp, S, y, ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
    torch.cuda.synchronize()
    n = max(3, steps // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n):
            call()
        e1.record(stream)
    e1.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / n
    flop_tok = 16 * FLOP_KHEAD + hv * FLOP_VHEAD
    return {"case": "wide-prefill", "n_seq": n_seq, "tokens_each": T, "ms": round(1e3 * t, 3),
            "tokens_per_s_per_layer": round(N / t, 1), "tflops": round(flop_tok * N / t / 1e12, 2),
            "workspace_gb": round(ws.numel() / 1e9, 2)}


def verify_measure(torch, device, steps, warmup, batch=4, r=4):
    """Speculative verify on the wide-GVA geometry (16/48 heads, d = 128, 10240
    conv channels): `batch` slots, r rows each, the state after every row
    written to a snapshot slot, then a commit of a random accepted count.
    Timing only: N(0, 1) inputs drawn on the device from a fixed seed."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    from hybrid_gated_deltanet_gb300 import synth
    geom = synth.WIDE_GVA
    hv, dd, cch = geom.n_v_heads, geom.d_k, geom.conv_channels
    cfg = gb.Config(geom.n_k_heads, hv, dd, dd, geom.d_conv, chunk=64, act_dtype=gb.BF16)
    r_ = synth.rng_for(3, 7)
    p = synth.make_params(geom, r_, synth.BF16)
    prm = gb.Params(conv_w=_dev(p["conv_w"], torch, device), A_log=_dev(p["A_log"], torch, device),
                    norm_w=_dev(p["norm_w"], torch, device))
    n_slots = 2 * batch * (1 + r)
    perm = r_.permutation(n_slots).astype(np.int32)
    slots = torch.from_numpy(perm[:batch].copy()).to(device)
    snaps = torch.from_numpy(perm[batch:batch * (1 + r)].reshape(batch, r).copy()).to(device)
    accept = torch.from_numpy(r_.integers(0, r + 1, size=batch).astype(np.int32)).to(device)
    g = torch.Generator(device=device)
    g.manual_seed(3)
    bf = torch.bfloat16
    S = 0.1 * torch.randn((n_slots, hv, dd, dd), generator=g, device=device)
    Cp = (0.1 * torch.randn((n_slots, geom.d_conv - 1, cch), generator=g, device=device)).to(bf)
    x = torch.randn((batch, r, cch), generator=g, device=device).to(bf)
    z = torch.randn((batch, r, hv * dd), generator=g, device=device).to(bf)
    a = torch.randn((batch, r, hv), generator=g, device=device).to(bf)
    b = torch.randn((batch, r, hv), generator=g, device=device).to(bf)
    y = torch.empty((batch, r, hv * dd), dtype=bf, device=device)
    stream = _side_stream(torch)

    def verify():
        gb.gdn_verify_rows(cfg, prm, x, z, a, b, Cp, S, slots, snaps, y, stream=stream)

    def commit():
        gb.gdn_commit_rows(cfg, Cp, S, slots, snaps, accept, stream=stream)

    def timed(fn, n):
        torch.cuda.synchronize()  # inputs made on the default stream are complete
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    def verify_nosnap():
        gb.gdn_verify_rows_nosnap(cfg, prm, x, z, a, b, Cp, S, slots, y, stream=stream)

    def commit_recompute():
        gb.gdn_commit_rows_recompute(cfg, prm, x, a, b, Cp, S, slots, accept, stream=stream)

    n = max(20, steps)
    t_v = timed(verify, n)
    t_c = timed(commit, n)
    t_vn = timed(verify_nosnap, n)
    t_cr = timed(commit_recompute, n)
    state, conv = hv * dd * dd * 4, (geom.d_conv - 1) * cch * 2
    row_io = cch * 2 + 2 * hv * dd * 2 + 2 * hv * 2  # x, z, y, a, b of one row
    v_bytes = batch * ((1 + r) * (state + conv) + r * row_io)
    return {"case": "verify", "geometry": "16/48 heads, d = 128, 10240 conv channels, bf16, fp32 state",
            "batch": batch, "rows": r, "verify_us": round(1e6 * t_v, 2),
            "verify_gbs": round(v_bytes / t_v / 1e9, 1), "verify_bytes": v_bytes,
            "commit_us": round(1e6 * t_c, 2),
            "recompute_variant": {"verify_us": round(1e6 * t_vn, 2), "commit_us": round(1e6 * t_cr, 2),
                                  "verify_plus_commit_us": round(1e6 * (t_vn + t_cr), 2),
                                  "snapshot_verify_plus_commit_us": round(1e6 * (t_v + t_c), 2)}}


def serving_measure(torch, device, steps, warmup, n_seq=20, pool=1024, batch=256):
    """The serving mix: one varlen prefill of n_seq sequences with lengths
    log-uniform in [500, 30000] into a pool of fp32 states, then decode steps of
    `batch` slots drawn at random from the same pool.  Timing only: inputs are
    N(0, 1) drawn on the device from a fixed seed (the parity of both paths is
    covered by the tests)."""
    from hybrid_gated_deltanet_gb300 import binding as gb
    from hybrid_gated_deltanet_gb300 import synth
    r = synth.rng_for(4, 0)
    lengths = synth.log_uniform_lengths(r, n_seq, 500, 30000)
    n_tok = int(sum(lengths))
    cfg = gb.Config(*GEOM_ARGS, chunk=64, act_dtype=gb.BF16)
    p = synth.make_params(synth.QWEN35_4B, r, synth.BF16)
    prm = gb.Params(conv_w=_dev(p["conv_w"], torch, device), A_log=_dev(p["A_log"], torch, device),
                    norm_w=_dev(p["norm_w"], torch, device))
    g = torch.Generator(device=device)
    g.manual_seed(4)
    bf = torch.bfloat16
    x = torch.randn((n_tok, 8192), generator=g, device=device).to(bf)
    z = torch.randn((n_tok, 4096), generator=g, device=device).to(bf)
    a = torch.randn((n_tok, 32), generator=g, device=device).to(bf)
    b = torch.randn((n_tok, 32), generator=g, device=device).to(bf)
    y = torch.empty((n_tok, 4096), dtype=bf, device=device)
    S = torch.zeros((pool, 32, 128, 128), device=device)
    Cp = torch.zeros((pool, 3, 8192), dtype=bf, device=device)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=device)
    pf_slots = torch.from_numpy(r.permutation(pool)[:n_seq].astype(np.int32)).to(device)
    ws = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_VARLEN_PREFILL, n_tok, n_seq), dtype=torch.uint8, device=device)
    dec_slots = torch.from_numpy(r.permutation(pool)[:batch].astype(np.int32)).to(device)
    dx = torch.randn((batch, 8192), generator=g, device=device).to(bf)
    dz = torch.randn((batch, 4096), generator=g, device=device).to(bf)
    da = torch.randn((batch, 32), generator=g, device=device).to(bf)
    db = torch.randn((batch, 32), generator=g, device=device).to(bf)
    dy = torch.empty((batch, 4096), dtype=bf, device=device)
    stream = _side_stream(torch)

    def prefill():
        gb.gdn_varlen_prefill(cfg, prm, x, z, a, b, cu, pf_slots, None, Cp, S, y, ws, stream=stream)

    def decode():
        gb.gdn_decode_step(cfg, prm, dx, dz, da, db, Cp, S, dec_slots, dy, stream=stream)

    def timed(fn, n):
        torch.cuda.synchronize()  # inputs made on the default stream are complete
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    t_pf = timed(prefill, max(1, steps))
    t_dec = timed(decode, max(1, steps) * 20)
    dec_bytes = batch * SLOT_BYTES + PARAM_BYTES
    return {"case": "serving", "n_seq": n_seq, "lengths": lengths, "tokens": n_tok,
            "prefill_ms": round(1e3 * t_pf, 3), "prefill_tokens_per_s_per_layer": round(n_tok / t_pf, 1),
            "prefill_tflops": round(FLOP_PER_TOKEN * n_tok / t_pf / 1e12, 2),
            "longest_seq_chunks": int(max(lengths) + 63) // 64,
            "decode_batch": batch, "decode_us": round(1e6 * t_dec, 2),
            "decode_gbs": round(dec_bytes / t_dec / 1e9, 1)}


def reference_arm(args):
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    n_slots = 16
    inputs = _oracle_decode_inputs(n_slots, 7)
    for _ in range(args.warmup):
        oracle_decode_rate(2, inputs=inputs)
    t0 = time.perf_counter()
    busy = 0.0
    threads = 1
    for _ in range(args.steps):
        _, dt, threads, _ = oracle_decode_rate(n_slots, inputs=inputs)
        busy += dt
    total = time.perf_counter() - t0
    value = args.steps * n_slots * SLOT_BYTES / busy / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total / max(args.steps, 1), 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": decode_config(1),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step: {n_slots} slots x 1 layer of the decode step (a bounded sample "
                                       f"of its 24 x 64 slot-layers), fp64 token loop, {threads} threads"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def gpu_arm(args):
    import torch
    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from hybrid_gated_deltanet_gb300 import build as gbuild
    if rank == 0:
        gbuild.build()
    barrier(world)
    peaks = _peaks()

    cfg, host, layers = setup_decode(torch, device, seed=rank)
    parity = decode_parity(torch, cfg, host, layers) if rank == 0 else None
    pf_steps = max(3, min(args.steps, 20))
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        step_s = []
        t_dec = time_decode(torch, cfg, layers, args.steps, args.warmup, use_graph=not args.no_graph,
                            per_step=step_s)
        torch.cuda.synchronize()
        barrier(world)
        t_pf, pf_err, pf_e2e = prefill_measure(torch, device, pf_steps, max(3, args.warmup // 4), seed=rank,
                                               check=(rank == 0))
        extra = {}
        if not args.no_workloads:
            # the wide-GVA workload (4 x 32768-token prefill, then verify at 4 and 64
            # slots) and the serving mix (20-sequence prefill, 256-of-1024 decode)
            wide_pf = wide_prefill_measure(torch, device, pf_steps, 3)
            wide_v = [verify_measure(torch, device, max(20, args.steps // 8), 3, batch=nb) for nb in (4, 64)]
            extra["wide_gva"] = {"prefill": wide_pf, "verify": wide_v}
            extra["serving"] = serving_measure(torch, device, max(3, pf_steps // 2), 3)
            sb = small_batch_decode(torch, device, max(10, args.steps // 20), 3)
            for rec in sb:
                rec["frac"] = round(rec["gbs"] / peaks["hbm_gbs"], 4)
            extra["decode_small_batch"] = sb
            # the hybrid's attention layer: decode at 16/4 heads (B = 64) and the wide
            # 24/2 heads (B = 4 x 32768, the tensor-core kernel), prefill at T = 8192
            att = attn_measure(torch, device, args.steps, 3,
                               decode_cases=(ATTN_DECODE_CASES[2], ATTN_DECODE_CASES[3]),
                               prefill_cases=(ATTN_PREFILL_CASES[0],))
            for rec in att:
                if rec["case"] == "attn":
                    rec["frac_hbm"] = round(rec["gbs"] / peaks["hbm_gbs"], 4)
                else:
                    rec["frac_bf16"] = round(rec["tflops"] / peaks["bf16_tflops"], 4)
            extra["attention"] = att
    t_dec = max_over_ranks(t_dec, world)
    e2e_steps = max(3, args.steps // 4)
    e2e_t, h2d, d2h = time_decode_e2e(torch, cfg, layers, e2e_steps, 3, graph=not args.no_graph)
    e2e_t = max_over_ranks(e2e_t, world)
    e2e_eager_t, _, _ = time_decode_e2e(torch, cfg, layers, e2e_steps, 3, graph=False)
    e2e_eager_t = max_over_ranks(e2e_eager_t, world)

    step_bytes = N_LAYERS * (B * SLOT_BYTES + PARAM_BYTES)
    value = world * step_bytes * args.steps / t_dec / 1e9
    launch_s = t_dec / (args.steps * N_LAYERS)
    achieved = (B * SLOT_BYTES + PARAM_BYTES) / launch_s / 1e9
    pf_tflops = FLOP_PER_TOKEN * PREFILL_T / t_pf / 1e12
    if rank != 0:
        return 0
    cpu_base = pf_cpu = None
    if world == 1:  # the oracle baseline is timed on rank 0 at N = 1 only
        cpu_rate, cpu_dt, cpu_thr, cpu_done = oracle_decode_rate(16, min_seconds=args.cpu_seconds)
        pf_heads = min(32, cpu_thr)
        pf_cpu_rate, pf_cpu_dt, _ = oracle_prefill_rate(args.cpu_prefill_tokens, pf_heads,
                                                        min_seconds=args.cpu_seconds)
        cpu_base = {"value": round(cpu_rate, 4), "unit": "GB/s", "cores": cpu_thr, "kind": "oracle",
                    "sample": f"{cpu_done} slot-steps of one layer (16 slots repeated, {cpu_dt:.1f} s)"}
        pf_cpu = {"value": round(pf_cpu_rate, 3), "unit": "tokens/s/layer", "cores": cpu_thr, "kind": "oracle",
                  "sample": f"{args.cpu_prefill_tokens} tokens x {pf_heads} of 32 v-heads ({pf_cpu_dt:.1f} s), "
                            "scaled to 32 heads"}
        one_rate, one_dt, _, one_done = oracle_decode_rate(16, min_seconds=args.cpu_seconds / 2, threads=1)
        cpu_base["single_core"] = {"value": round(one_rate, 4), "unit": "GB/s", "cores": 1,
                                   "sample": f"{one_done} slot-steps of one layer, one thread ({one_dt:.1f} s)"}
    traffic = measured_traffic("k_decode_persist", "gdn_decode.cu")
    pf_traffic = measured_traffic("gdn_chunk_prefill", "gdn_chunk16.cu+gdn_prefill.cu")
    pf_bytes = PREFILL_T * TOKEN_BYTES + STATE_BYTES
    clocks = clk.summary()
    line = {
        "metric": METRIC,
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t_dec / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "step_ms": {"min": round(1e3 * min(step_s), 4), "median": round(1e3 * float(np.median(step_s)), 4),
                    "max": round(1e3 * max(step_s), 4)},
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(decode_config(world), graph=not args.no_graph),
        "parity": {"decode_rel_fro": parity, "prefill_rel_fro": pf_err,
                   "tolerance": {"y": 2e-2, "S": 1e-3}},
        "roofline": {"bound": "hbm",
                     "kernel": "gdn_decode_step = k_decode_persist (state, conv-state roll, y: one launch per layer)",
                     "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "peak_src": peaks["src"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": traffic, "call_us": round(launch_s * 1e6, 3),
                     "algorithmic_bytes_per_launch": B * SLOT_BYTES + PARAM_BYTES},
        "prefill": {"workload": "chunked prefill, 1 sequence, T = 8192, 16/32 heads, d = 128, bf16 in, fp32 state, "
                                "chunk 64 (3 launches: k_prep16, k_chain16, k_conv_final)",
                    "tokens_per_s_per_layer": round(PREFILL_T / t_pf, 1), "ms_per_call": round(t_pf * 1e3, 4),
                    "tflops": round(pf_tflops, 3), "flop_per_token": FLOP_PER_TOKEN,
                    "peak_tflops": peaks["bf16_tflops"], "frac_tc": round(pf_tflops / peaks["bf16_tflops"], 4),
                    "roofline": {"bound": "tensor", "kernel": "one gdn_chunk_prefill call (its 3 launches)",
                                 "achieved": round(pf_tflops, 3), "peak": peaks["bf16_tflops"],
                                 "peak_src": peaks["src"], "unit": "TFLOP/s",
                                 "frac": round(pf_tflops / peaks["bf16_tflops"], 4), "traffic": pf_traffic,
                                 "algorithmic_flops_per_call": FLOP_PER_TOKEN * PREFILL_T,
                                 "algorithmic_bytes_per_call": pf_bytes,
                                 "hbm_view": {"achieved": round(pf_bytes / t_pf / 1e9, 1), "unit": "GB/s",
                                              "frac": round(pf_bytes / t_pf / 1e9 / peaks["hbm_gbs"], 4)}},
                    "e2e": pf_e2e, "cpu_baseline": pf_cpu},
        **extra,
        "cpu_baseline": cpu_base,
        "e2e": {"value": round(world * step_bytes * e2e_steps / e2e_t / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(1e3 * e2e_t / e2e_steps, 4), "graph": not args.no_graph,
                "eager": {"value": round(world * step_bytes * e2e_steps / e2e_eager_t / 1e9, 2),
                          "ms_per_step": round(1e3 * e2e_eager_t / e2e_steps, 4)}},
        "gpu_launches": args.steps * N_LAYERS,  # per layer: the persistent decode kernel
        "clocks": clocks,
    }
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--batch", type=int, default=64, help="slots of the decode-small case")
    ap.add_argument("--batches", default="1,4,16", help="slot counts of the decode-batches case")
    ap.add_argument("--case", default="full", choices=["full", "decode-small", "decode-batches", "prefill-small",
                             "prefill-varlen", "serving",
                             "verify", "ckpt", "layer",
                             "proj-decode", "attn", "proj-prefill", "attn-small", "attn-wide"],
                    help="small cases for ncu captures")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-prefill-tokens", type=int, default=8192)
    ap.add_argument("--no-workloads", action="store_true",
                    help="leave out the wide-GVA and serving-mix figures of the full run")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return reference_arm(args)
    if args.case != "full":
        return profile_case(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
