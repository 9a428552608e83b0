"""The C ABI without a GPU: libgdn loads, exports every entry point that
include/gdn.h declares, and rejects bad arguments on the host with the status
and a message naming the argument, the value found and the value required
(Strata chapter 6, sections 6.2 and 6.5).  No call here reaches a launch."""
import ctypes
import os
import re
import subprocess

import pytest

from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")
FAKE = 0x100000  # an aligned address that is never dereferenced on the host


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gb.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(gdn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for fn in ("gdn_conv_state_update", "gdn_decode_step", "gdn_verify_rows", "gdn_chunk_prefill",
               "gdn_varlen_prefill", "gdn_workspace_size", "gdn_last_error", "gdn_proj_gemm", "gdn_layer_decode",
               "gdn_layer_varlen_prefill"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", gb.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (gdn_\w+)", out))
    assert set(declared_functions()) <= exported
    assert lib.gdn_version().decode().startswith("libgdn")


def _cfg(**kw):
    c = gb.Config(16, 32, 128, 128, 4, 64, gb.BF16)
    for k, v in kw.items():
        setattr(c, k, v)
    return c.c()


def _prm():
    return gb.CParams(FAKE, None, FAKE, None, FAKE)


def _decode(lib, cfg, x=FAKE, B=4, n_slots=8, prm=None):
    prm = prm or _prm()
    return lib.gdn_decode_step(ctypes.byref(cfg), ctypes.byref(prm), x, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B,
                               n_slots, FAKE, None)


def _err(lib):
    return lib.gdn_last_error().decode()


@pytest.mark.parametrize("kw,status,needle", [
    (dict(act_dtype=7), -3, "cfg.act_dtype: found 7"),
    (dict(n_v_heads=30), -2, "cfg.n_v_heads: found 30, required a multiple of n_k_heads = 16"),
    (dict(n_k_heads=2, n_v_heads=32), -7, "required <= 8"),
    (dict(n_k_heads=4096, n_v_heads=8192), -7, "cfg.n_v_heads: found 8192, required <= 4096"),
    (dict(d_k=48, d_v=48), -2, "cfg.d_k: found 48"),
    (dict(d_v=64), -7, "required d_v == d_k = 128"),
    (dict(d_conv=5), -2, "cfg.d_conv: found 5"),
    (dict(flags=16), -2, "cfg.flags"),
])
def test_config_validation(lib, kw, status, needle):
    assert _decode(lib, _cfg(**kw)) == status
    assert needle in _err(lib)


def test_null_and_alignment(lib):
    assert lib.gdn_decode_step(None, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, FAKE, None) == -1
    assert "cfg: found NULL" in _err(lib)
    assert _decode(lib, _cfg(), x=0) == -1
    assert "x: found NULL, required a device pointer" in _err(lib)
    assert _decode(lib, _cfg(), x=FAKE + 1) == -4
    assert "x: found address" in _err(lib) and "16-byte alignment" in _err(lib)
    prm = gb.CParams(FAKE, None, None, None, FAKE)
    assert _decode(lib, _cfg(), prm=prm) == -1 and "prm.A_log" in _err(lib)


def test_counts(lib):
    assert _decode(lib, _cfg(), B=-1) == -5 and "B: found -1" in _err(lib)
    assert _decode(lib, _cfg(), n_slots=0) == -5 and "n_slots: found 0" in _err(lib)
    assert _decode(lib, _cfg(), B=0) == 0 and _err(lib) == ""   # nothing to launch
    cfg = _cfg()
    prm = _prm()
    st = lib.gdn_verify_rows(ctypes.byref(cfg), ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2,
                             17, 8, FAKE, None)
    assert st == -5 and "r: found 17, required 1..16" in _err(lib)
    st = lib.gdn_verify_rows(ctypes.byref(cfg), ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 2,
                             4, 8, FAKE, None)
    assert st == -1 and "snap_idx" in _err(lib)


def test_workspace_size_and_refusal(lib):
    cfg = _cfg()
    need = lib.gdn_workspace_size(ctypes.byref(cfg), gb.OP_CHUNK_PREFILL, 8192, 1)
    # d = 128, chunk 64, bf16: per 64-token chunk slot (8192/64 + 1 sequence + 1 slots), per k-head the
    # fp16 K^ tile (16 KB), per v-head the fp16 [-W; Q'] (32 KB), [T'; PT'] (16 KB) and V (16 KB)
    # tiles and 512 B of gates; the two sections start on 1024-byte boundaries
    slots = 8192 // 64 + 2
    kk = slots * 16 * 16384
    rec = slots * 32 * (32768 + 16384 + 16384 + 512)
    assert need == kk + (rec + 1023) // 1024 * 1024
    # every other geometry: fp32 per token (q^ and k^ 2 x 16 x 128, v 32 x 128, g and beta 2 x 32)
    f32 = _cfg(act_dtype=gb.F32)
    assert lib.gdn_workspace_size(ctypes.byref(f32), gb.OP_CHUNK_PREFILL, 8192, 1) == \
        8192 * (2 * 16 * 128 + 32 * 128 + 2 * 32) * 4
    assert lib.gdn_workspace_size(ctypes.byref(cfg), gb.OP_DECODE_STEP, 64, 1) == 0
    bad = _cfg(chunk=48)
    assert lib.gdn_workspace_size(ctypes.byref(bad), gb.OP_CHUNK_PREFILL, 10, 1) == 0
    assert "cfg.chunk: found 48" in _err(lib)
    prm = _prm()
    st = lib.gdn_chunk_prefill(ctypes.byref(cfg), ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, 8192, None, None, FAKE,
                               FAKE, FAKE, FAKE, need - 1, None)
    assert st == -6
    assert f"workspace: found {need - 1} bytes, required {need} bytes" in _err(lib)
    st = lib.gdn_chunk_prefill(ctypes.byref(cfg), ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, 8192, None, None, FAKE,
                               FAKE, FAKE, None, 0, None)
    assert st == -1 and "workspace" in _err(lib)


def test_varlen_validation(lib):
    cfg = _cfg()
    prm = _prm()
    st = lib.gdn_varlen_prefill(ctypes.byref(cfg), ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, None, 3, 100, FAKE,
                                None, FAKE, FAKE, 8, FAKE, FAKE, 1 << 30, None)
    assert st == -1 and "cu_seqlens" in _err(lib)
    st = lib.gdn_varlen_prefill(ctypes.byref(cfg), ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, FAKE, 0, 5, FAKE,
                                None, FAKE, FAKE, 8, FAKE, FAKE, 0, None)
    assert st == -5 and "n_tokens: found 5 with n_seq = 0" in _err(lib)
    st = lib.gdn_varlen_prefill(ctypes.byref(cfg), ctypes.byref(prm), None, None, None, None, None, 0, 0, None, None,
                                None, None, 8, None, None, 0, None)
    assert st == 0


def test_varlen_ckpt_validation(lib):
    """gdn_varlen_prefill_ckpt: snapshot spacing must be a positive multiple of the
    chunk; the offset and slot arrays are required."""
    cfg = _cfg()
    prm = _prm()

    def call(every, off=FAKE, slots=FAKE):
        return lib.gdn_varlen_prefill_ckpt(ctypes.byref(cfg), ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, FAKE, 2, 100,
                                           FAKE, None, FAKE, FAKE, 8, FAKE, every, off, slots, FAKE, 1 << 30, None)

    assert call(0) == -5 and "ckpt_every: found 0, required a positive multiple of chunk = 64" in _err(lib)
    assert call(96) == -5 and "found 96" in _err(lib)
    assert call(128, off=None) == -1 and "ckpt_offset" in _err(lib)
    assert call(128, slots=None) == -1 and "ckpt_slots" in _err(lib)
    assert call(128, off=FAKE + 2) == -4 and "ckpt_offset" in _err(lib)


def test_recompute_commit_validation(lib):
    cfg = _cfg()
    prm = _prm()
    st = lib.gdn_commit_rows_recompute(ctypes.byref(cfg), ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                       4, 4, 16, None)
    assert st == -1 and "accepted" in _err(lib)
    st = lib.gdn_commit_rows_recompute(ctypes.byref(cfg), ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                       4, 17, 16, None)
    assert st == -5 and "r: found 17" in _err(lib)
    st = lib.gdn_verify_rows_nosnap(ctypes.byref(cfg), ctypes.byref(prm), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                    4, 4, 16, None, None)
    assert st == -1 and "y" in _err(lib)


def test_projection_and_layer_validation(lib):
    cfg = _cfg()
    prm = _prm()
    st = lib.gdn_proj_gemm(FAKE, FAKE, FAKE, 4, 16, 60, 16, None, 0, None)
    assert st == -2 and "k: found 60, required a positive multiple of 8" in _err(lib)
    st = lib.gdn_proj_gemm(FAKE, FAKE, FAKE, 4, 16, 64, 8, None, 0, None)
    assert st == -2 and "ld_out: found 8, required >= n_out = 16" in _err(lib)
    assert lib.gdn_proj_gemm(None, None, None, 0, 16, 64, 16, None, 0, None) == 0
    need = lib.gdn_proj_workspace_size(4, 2560, 4096)
    st = lib.gdn_proj_gemm(FAKE, FAKE, FAKE, 4, 2560, 4096, 2560, FAKE, need - 16, None)
    assert st == -6 and f"required {need} bytes" in _err(lib)

    def dec(cfg_=cfg, proj=gb.CProj(FAKE, FAKE, 2560), ws_bytes=1 << 30):
        return lib.gdn_layer_decode(ctypes.byref(cfg_), ctypes.byref(prm), ctypes.byref(proj) if proj else None,
                                    FAKE, FAKE, FAKE, FAKE, 4, 8, FAKE, FAKE, ws_bytes, None)

    assert dec(proj=None) == -1 and "proj: found NULL" in _err(lib)
    assert dec(proj=gb.CProj(FAKE, FAKE, 2561)) == -2 and "proj.hidden: found 2561" in _err(lib)
    assert dec(proj=gb.CProj(FAKE, None, 2560)) == -1 and "proj.w_out" in _err(lib)
    assert dec(cfg_=_cfg(act_dtype=1)) == -7 and "GDN_DTYPE_BF16" in _err(lib)
    need = lib.gdn_layer_workspace_size(ctypes.byref(cfg), gb.OP_LAYER_DECODE, 4, 1, 2560)
    assert dec(ws_bytes=need - 1) == -6 and f"required {need} bytes" in _err(lib)
    st = lib.gdn_layer_varlen_prefill(ctypes.byref(cfg), ctypes.byref(prm), ctypes.byref(gb.CProj(FAKE, FAKE, 2560)),
                                      FAKE, None, 2, 100, FAKE, None, FAKE, FAKE, 8, FAKE, FAKE, 1 << 30, None)
    assert st == -1 and "cu_seqlens" in _err(lib)


def test_projection_workspace_sizes(lib):
    """Split-K partials: up to 64 tokens in 64-token tiles, more in 256-token tiles;
    when the 128-row tiles number at most 74, K (in 64-wide blocks) is split over
    ks = min(16, 148 // tiles) CTAs, fewer if a CTA would get under 2 blocks; each
    split tile needs ks x tile-width x 128 fp32."""
    def want(n_tok, n_out, k):
        bt = 64 if n_tok <= 64 else 256
        tiles = -(-n_out // 128) * -(-n_tok // bt)
        if tiles * 2 > 148:
            return 0
        ks, kb = min(16, 148 // tiles), -(-k // 64)
        while ks > 1 and kb // ks < 2:
            ks -= 1
        return tiles * ks * bt * 128 * 4 if ks > 1 else 0

    for n_tok, n_out, k in [(1, 12352, 2560), (64, 12352, 2560), (64, 2560, 4096), (4, 100, 64), (300, 2560, 4096),
                            (200, 1, 8), (256, 4096, 2560), (8192, 12352, 2560), (100, 256, 1024)]:
        assert lib.gdn_proj_workspace_size(n_tok, n_out, k) == want(n_tok, n_out, k), (n_tok, n_out, k)
    assert lib.gdn_proj_workspace_size(64, 12352, 2560) == 0
    assert lib.gdn_proj_workspace_size(64, 2560, 4096) == 20 * 7 * 64 * 128 * 4
    assert lib.gdn_proj_workspace_size(256, 2560, 4096) == 20 * 7 * 256 * 128 * 4


def test_varlen_prefill_workspace_holds_the_sequence_order(lib):
    """A varlen prefill of 2 to 1024 sequences adds one int32 per sequence (the chain's
    longest-first order) after the chunk records, in its own 1024-byte-aligned region;
    one sequence, or more than 1024, adds nothing."""
    cfg = _cfg()
    up = lambda v: (v + 1023) // 1024 * 1024

    def records(n, n_seq):
        slots = n // 64 + n_seq + 1
        return up(up(slots * 16 * 16384) + slots * 32 * (32768 + 16384 + 16384 + 512))

    for n, n_seq in [(8192, 1), (8192, 2), (5000, 20), (70000, 1024), (70000, 1025), (300, 3)]:
        want = records(n, n_seq)
        if 1 < n_seq <= 1024:
            want = up(want + 4 * n_seq)
        assert lib.gdn_workspace_size(ctypes.byref(cfg), gb.OP_VARLEN_PREFILL, n, n_seq) == want, (n, n_seq)


def test_layer_workspace_sizes(lib):
    """x [n][8192], z [n][4096], a, b [n][32], y [n][4096] in bf16, then the larger of
    the two projections' partial sums, each region rounded up to 256 bytes; a layer
    prefill adds the prefill's own workspace."""
    cfg = _cfg()
    up = lambda v: (v + 255) // 256 * 256
    for n in (1, 4, 64, 300):
        part = max(lib.gdn_proj_workspace_size(n, 8192 + 4096 + 64, 2560), lib.gdn_proj_workspace_size(n, 2560, 4096))
        want = up(n * 8192 * 2) + up(n * 4096 * 2) + 2 * up(n * 32 * 2) + up(n * 4096 * 2) + up(part)
        assert lib.gdn_layer_workspace_size(ctypes.byref(cfg), gb.OP_LAYER_DECODE, n, 1, 2560) == want
        pf = lib.gdn_workspace_size(ctypes.byref(cfg), gb.OP_VARLEN_PREFILL, n, 3)
        assert lib.gdn_layer_workspace_size(ctypes.byref(cfg), gb.OP_LAYER_VARLEN_PREFILL, n, 3, 2560) == want + pf
    assert lib.gdn_layer_workspace_size(ctypes.byref(cfg), gb.OP_LAYER_DECODE, 4, 1, 2561) == 0
    assert "hidden" in _err(lib)


def test_binding_raises_with_message(lib):
    cfg = gb.Config(16, 30, 128, 128)
    with pytest.raises(gb.GdnError, match="GDN_ERR_SHAPE: cfg.n_v_heads: found 30"):
        gb.gdn_workspace_size(cfg, gb.OP_CHUNK_PREFILL, 10)


def test_attention_validation(lib):
    def cfg(**kw):
        c = gb.AttnConfig(16, 4, 256, 16)
        for k, v in kw.items():
            setattr(c, k, v)
        return c.c()

    def call(c, B=2, ws=None, ws_bytes=0, max_seq=100):
        return lib.gdn_attn_decode(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, 8, 64, max_seq, FAKE,
                                   ws, ws_bytes, None)

    assert call(cfg(n_q_heads=12, n_kv_heads=8)) == -2 and "n_q_heads/n_kv_heads: found 12/8" in _err(lib)
    assert call(cfg(n_q_heads=24, n_kv_heads=4)) == -7 and "G = n_q_heads / n_kv_heads = 6" in _err(lib)
    assert call(cfg(head_dim=64)) == -2 and "head_dim: found 64" in _err(lib)
    assert call(cfg(page_size=12)) == -2 and "page_size: found 12" in _err(lib)
    assert call(cfg(), B=0) == 0
    need = lib.gdn_attn_workspace_size(ctypes.byref(cfg()), 2, 5000)
    assert need > 0
    assert call(cfg(), max_seq=5000) == -1 and "workspace" in _err(lib)
    assert call(cfg(), max_seq=5000, ws=FAKE, ws_bytes=need - 1) == -6 and f"required {need} bytes" in _err(lib)
    assert call(cfg(), max_seq=5000, ws=FAKE + 8, ws_bytes=need) == -4


def test_attention_workspace_sizes(lib):
    """Context splits of gdn_attn_decode: about 1216 CTAs over (sequence, kv-head, head
    group), each split at least 128 tokens, a multiple of 16; a head group is all G query
    heads of the kv-head up to G = 16, groups of 4 beyond; G = 8, 12, 16 (the tensor-core
    kernel, one CTA per SM) aim at 152 CTAs.  The workspace holds B x Hq x splits x
    (d + 2) fp32 (unnormalised o, maximum, sum) when splitting."""
    def want(Hq, Hkv, D, B, max_seq):
        G = Hq // Hkv
        pairs = B * Hkv * (G // 4 if G > 16 else 1)
        target = 152 if G in (8, 12, 16) else 1216
        ns = min(-(-target // pairs), -(-max_seq // 128))
        ns = max(ns, 1)
        span = -(-max_seq // ns)
        span = -(-span // 16) * 16
        ns = -(-max_seq // span)
        return B * Hq * ns * (D + 2) * 4 if ns > 1 else 0

    for Hq, Hkv, D, B, L in [(16, 4, 256, 1, 8193), (16, 4, 256, 64, 8193), (24, 2, 256, 4, 32769),
                             (8, 8, 128, 200, 60), (4, 2, 128, 3, 129), (32, 4, 128, 16, 4000),
                             (32, 2, 128, 1, 5000), (64, 8, 256, 3, 70000)]:
        c = gb.AttnConfig(Hq, Hkv, D, 16).c()
        assert lib.gdn_attn_workspace_size(ctypes.byref(c), B, L) == want(Hq, Hkv, D, B, L), (Hq, Hkv, D, B, L)


def _oracle_check(path):
    import oracle
    return oracle._native(path)


@pytest.mark.parametrize("check, built", [(gbuild._built_here, gbuild.LIB), (_oracle_check, None)],
                         ids=["libgdn", "oracle"])
def test_build_rejects_a_library_of_another_architecture(tmp_path, check, built):
    """A shared library carried over from a machine of another architecture is rebuilt, not
    loaded: each up-to-date check reads the ELF machine field as well as the times."""
    import platform
    here = {"x86_64": 62, "amd64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine().lower())
    if here is None:
        pytest.skip("host architecture without a known ELF machine number")
    other = 183 if here == 62 else 62

    def elf(machine):
        head = bytearray(64)
        head[:4] = b"\x7fELF"
        head[4], head[5] = 2, 1  # 64-bit, little-endian
        head[18:20] = machine.to_bytes(2, "little")
        return bytes(head)

    for name, data, want in (("native.so", elf(here), True), ("foreign.so", elf(other), False),
                             ("text.so", b"not an ELF file at all....", False), ("short.so", b"\x7fELF", False)):
        path = tmp_path / name
        path.write_bytes(data)
        assert check(str(path)) is want, name
    assert check(str(tmp_path / "missing.so")) is False
    if built is not None:
        assert check(built)
