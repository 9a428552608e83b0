"""Thin Python binding of libgdn (ctypes): argument marshalling only.

Every function here has the name of the C entry point it calls (include/gdn.h)
and takes torch tensors for the device buffers.  Sizes come from the tensor
shapes, the stream is torch's current CUDA stream unless one is given.  All
arithmetic happens in libgdn's kernels; nothing here computes any part of the
layer, and there is no fallback: if libgdn.so is missing or its call fails,
the call raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

BF16, F32 = 0, 1
RAW_QKV, NO_L2NORM, GATES_DIRECT, NO_OUTNORM = 1, 2, 4, 8
(OP_CONV_STATE_UPDATE, OP_DECODE_STEP, OP_VERIFY_ROWS, OP_CHUNK_PREFILL, OP_VARLEN_PREFILL, OP_LAYER_DECODE,
 OP_LAYER_VARLEN_PREFILL) = range(7)

STATUS = {0: "GDN_OK", -1: "GDN_ERR_NULL", -2: "GDN_ERR_SHAPE", -3: "GDN_ERR_DTYPE", -4: "GDN_ERR_ALIGN",
          -5: "GDN_ERR_RANGE", -6: "GDN_ERR_WORKSPACE", -7: "GDN_ERR_UNSUPPORTED", -8: "GDN_ERR_CUDA"}


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class CConfig(ctypes.Structure):
    _fields_ = [("n_k_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("d_conv", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("q_scale", ctypes.c_float), ("l2_eps", ctypes.c_float),
                ("norm_eps", ctypes.c_float), ("flags", ctypes.c_uint32)]


class CParams(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("conv_b", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p), ("norm_w", ctypes.c_void_p)]


@dataclasses.dataclass
class Config:
    n_k_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    d_conv: int = 4
    chunk: int = 64
    act_dtype: int = BF16
    q_scale: float = 1.0
    l2_eps: float = 1e-6
    norm_eps: float = 1e-6
    flags: int = 0

    @property
    def conv_channels(self) -> int:
        return 2 * self.n_k_heads * self.d_k + self.n_v_heads * self.d_v

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.act_dtype == BF16 else torch.float32

    def c(self) -> CConfig:
        return CConfig(self.n_k_heads, self.n_v_heads, self.d_k, self.d_v, self.d_conv, self.chunk, self.act_dtype,
                       self.q_scale, self.l2_eps, self.norm_eps, self.flags)


@dataclasses.dataclass
class Params:
    conv_w: Optional[torch.Tensor]
    A_log: Optional[torch.Tensor]
    norm_w: Optional[torch.Tensor]
    conv_b: Optional[torch.Tensor] = None
    dt_bias: Optional[torch.Tensor] = None

    def c(self) -> CParams:
        return CParams(_p(self.conv_w), _p(self.conv_b), _p(self.A_log), _p(self.dt_bias), _p(self.norm_w))


class CProj(ctypes.Structure):
    _fields_ = [("w_in", ctypes.c_void_p), ("w_out", ctypes.c_void_p), ("hidden", ctypes.c_int32)]


@dataclasses.dataclass
class Proj:
    """Projection weights of a layer: w_in bf16 [C_ch + H_v*d_v + 2*H_v, hidden] (rows of
    x, z, a, b), w_out bf16 [hidden, H_v*d_v]."""
    w_in: torch.Tensor
    w_out: torch.Tensor

    def c(self) -> CProj:
        return CProj(_p(self.w_in), _p(self.w_out), self.w_in.shape[1])


class CAttnConfig(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("scale", ctypes.c_float)]


@dataclasses.dataclass
class AttnConfig:
    n_q_heads: int
    n_kv_heads: int
    head_dim: int = 256
    page_size: int = 16
    scale: float = 0.0

    def c(self) -> CAttnConfig:
        return CAttnConfig(self.n_q_heads, self.n_kv_heads, self.head_dim, self.page_size, self.scale)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("libgdn takes dense row-major tensors")
    return t.data_ptr()


_lib = None


def load() -> ctypes.CDLL:
    """Load libgdn.so (built by hybrid_gated_deltanet_gb300.build); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libgdn.so is not built ({LIB_PATH}); run "
                               "`python -m hybrid_gated_deltanet_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        cfgp, prmp = ctypes.POINTER(CConfig), ctypes.POINTER(CParams)
        sigs = {
            "gdn_conv_state_update": [cfgp, prmp, vp, vp, vp, i32, i32, i32, vp, vp],
            "gdn_decode_step": [cfgp, prmp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp],
            "gdn_verify_rows": [cfgp, prmp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, vp],
            "gdn_commit_rows": [cfgp, vp, vp, vp, vp, vp, i32, i32, i32, vp],
            "gdn_chunk_prefill": [cfgp, prmp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp, sz, vp],
            "gdn_chunk_prefill_noalloc": [cfgp, prmp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp],
            "gdn_varlen_prefill": [cfgp, prmp, vp, vp, vp, vp, vp, i32, i64, vp, vp, vp, vp, i32, vp, vp, sz, vp],
            "gdn_verify_rows_nosnap": [cfgp, prmp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, vp],
            "gdn_commit_rows_recompute": [cfgp, prmp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp],
            "gdn_varlen_prefill_ckpt": [cfgp, prmp, vp, vp, vp, vp, vp, i32, i64, vp, vp, vp, vp, i32, vp, i32, vp,
                                        vp, vp, sz, vp],
        }
        projp = ctypes.POINTER(CProj)
        sigs["gdn_proj_gemm"] = [vp, vp, vp, i64, i32, i32, i64, vp, sz, vp]
        sigs["gdn_layer_decode"] = [cfgp, prmp, projp, vp, vp, vp, vp, i32, i32, vp, vp, sz, vp]
        sigs["gdn_layer_varlen_prefill"] = [cfgp, prmp, projp, vp, vp, i32, i64, vp, vp, vp, vp, i32, vp, vp, sz, vp]
        acfgp = ctypes.POINTER(CAttnConfig)
        sigs["gdn_attn_decode"] = [acfgp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, sz, vp]
        sigs["gdn_attn_prefill"] = [acfgp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, vp, vp]
        for name, args in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.gdn_workspace_size.argtypes = [cfgp, i32, i64, i32]
        lib.gdn_workspace_size.restype = sz
        lib.gdn_proj_workspace_size.argtypes = [i64, i32, i32]
        lib.gdn_proj_workspace_size.restype = sz
        lib.gdn_layer_workspace_size.argtypes = [cfgp, i32, i64, i32, i32]
        lib.gdn_layer_workspace_size.restype = sz
        lib.gdn_attn_workspace_size.argtypes = [acfgp, i32, i32]
        lib.gdn_attn_workspace_size.restype = sz
        lib.gdn_last_error.argtypes = []
        lib.gdn_last_error.restype = ctypes.c_char_p
        lib.gdn_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        lib.gdn_device_status.restype = ctypes.c_int
        lib.gdn_version.argtypes = []
        lib.gdn_version.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _check(status: int):
    if status != 0:
        raise GdnError(status, load().gdn_last_error().decode())


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def gdn_device_status() -> int:
    """Reads and clears the device status word (0: no kernel reported a timed-out
    wait).  Synchronises the current device."""
    v = ctypes.c_uint32(0)
    _check(load().gdn_device_status(ctypes.byref(v)))
    return int(v.value)


def gdn_workspace_size(cfg: Config, op: int, n_tokens: int, n_seq: int = 1) -> int:
    c = cfg.c()
    n = load().gdn_workspace_size(ctypes.byref(c), op, n_tokens, n_seq)
    msg = load().gdn_last_error().decode()
    if msg:
        raise GdnError(-2, msg)
    return n


def gdn_conv_state_update(cfg: Config, prm: Params, x: torch.Tensor, conv_pool: torch.Tensor,
                          slot_idx: torch.Tensor, n_tok: int, u_out: Optional[torch.Tensor] = None, stream=None):
    """x [n_seq*n_tok, C_ch]; updates conv_pool[slot_idx] in place; u_out = silu(conv(x))."""
    c, p = cfg.c(), prm.c()
    n_seq = slot_idx.numel()
    _check(load().gdn_conv_state_update(ctypes.byref(c), ctypes.byref(p), _p(x), _p(conv_pool), _p(slot_idx), n_seq,
                                        n_tok, conv_pool.shape[0], _p(u_out), _stream(stream)))


def gdn_decode_step(cfg: Config, prm: Params, x, z, a, b, conv_pool, state_pool, slot_idx, y, stream=None):
    """One token for each of B = x.shape[0] slots; pools updated in place; writes y."""
    c, p = cfg.c(), prm.c()
    _check(load().gdn_decode_step(ctypes.byref(c), ctypes.byref(p), _p(x), _p(z), _p(a), _p(b), _p(conv_pool),
                                  _p(state_pool), _p(slot_idx), x.shape[0], state_pool.shape[0], _p(y),
                                  _stream(stream)))


def gdn_verify_rows(cfg: Config, prm: Params, x, z, a, b, conv_pool, state_pool, slot_idx, snap_idx, y,
                    stream=None):
    """x [B, r, C_ch] ...; state after row i of entry b goes to slot snap_idx[b, i]."""
    c, p = cfg.c(), prm.c()
    B, r = snap_idx.shape
    _check(load().gdn_verify_rows(ctypes.byref(c), ctypes.byref(p), _p(x), _p(z), _p(a), _p(b), _p(conv_pool),
                                  _p(state_pool), _p(slot_idx), _p(snap_idx), B, r, state_pool.shape[0], _p(y),
                                  _stream(stream)))


def gdn_commit_rows(cfg: Config, conv_pool, state_pool, slot_idx, snap_idx, accepted, stream=None):
    """Copies snapshot accepted[b]-1 of entry b into slot_idx[b] (accepted[b] = 0: no copy)."""
    c = cfg.c()
    B, r = snap_idx.shape
    _check(load().gdn_commit_rows(ctypes.byref(c), _p(conv_pool), _p(state_pool), _p(slot_idx), _p(snap_idx),
                                  _p(accepted), B, r, state_pool.shape[0], _stream(stream)))


def gdn_chunk_prefill(cfg: Config, prm: Params, x, z, a, b, s0, conv0, s_final, conv_final, y, workspace,
                      stream=None):
    """One sequence of T = x.shape[0] tokens; s0/conv0 may be None (zeros)."""
    c, p = cfg.c(), prm.c()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_chunk_prefill(ctypes.byref(c), ctypes.byref(p), _p(x), _p(z), _p(a), _p(b), x.shape[0], _p(s0),
                                    _p(conv0), _p(s_final), _p(conv_final), _p(y), _p(workspace), ws_bytes,
                                    _stream(stream)))


def gdn_chunk_prefill_noalloc(cfg: Config, prm: Params, x, z, a, b, s0, conv0, s_final, conv_final, y, stream=None):
    """gdn_chunk_prefill without a workspace argument, for callers that cannot
    allocate: the library's static 64 MiB device scratch is used instead."""
    c, p = cfg.c(), prm.c()
    _check(load().gdn_chunk_prefill_noalloc(ctypes.byref(c), ctypes.byref(p), _p(x), _p(z), _p(a), _p(b),
                                            x.shape[0], _p(s0), _p(conv0), _p(s_final), _p(conv_final), _p(y),
                                            _stream(stream)))


def gdn_varlen_prefill(cfg: Config, prm: Params, x, z, a, b, cu_seqlens, slot_idx, has_init, conv_pool, state_pool, y,
                       workspace, stream=None):
    """Packed sequences [cu_seqlens[s], cu_seqlens[s+1]); pool slots slot_idx[s]."""
    c, p = cfg.c(), prm.c()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_varlen_prefill(ctypes.byref(c), ctypes.byref(p), _p(x), _p(z), _p(a), _p(b), _p(cu_seqlens),
                                     slot_idx.numel(), x.shape[0], _p(slot_idx), _p(has_init), _p(conv_pool),
                                     _p(state_pool), state_pool.shape[0], _p(y), _p(workspace), ws_bytes,
                                     _stream(stream)))


def gdn_varlen_prefill_ckpt(cfg: Config, prm: Params, x, z, a, b, cu_seqlens, slot_idx, has_init, conv_pool,
                            state_pool, y, ckpt_every: int, ckpt_offset, ckpt_slots, workspace, stream=None):
    """gdn_varlen_prefill plus prefix snapshots: the state after (k+1)*ckpt_every
    tokens of sequence s goes to pool slot ckpt_slots[ckpt_offset[s] + k]."""
    c, p = cfg.c(), prm.c()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_varlen_prefill_ckpt(ctypes.byref(c), ctypes.byref(p), _p(x), _p(z), _p(a), _p(b),
                                          _p(cu_seqlens), slot_idx.numel(), x.shape[0], _p(slot_idx), _p(has_init),
                                          _p(conv_pool), _p(state_pool), state_pool.shape[0], _p(y), int(ckpt_every),
                                          _p(ckpt_offset), _p(ckpt_slots), _p(workspace), ws_bytes,
                                          _stream(stream)))


def gdn_verify_rows_nosnap(cfg: Config, prm: Params, x, z, a, b, conv_pool, state_pool, slot_idx, y, stream=None):
    """x [B, r, C_ch] ...: y of every row; the pools are not written."""
    c, p = cfg.c(), prm.c()
    B, r = x.shape[0], x.shape[1]
    _check(load().gdn_verify_rows_nosnap(ctypes.byref(c), ctypes.byref(p), _p(x), _p(z), _p(a), _p(b),
                                         _p(conv_pool), _p(state_pool), _p(slot_idx), B, r, state_pool.shape[0],
                                         _p(y), _stream(stream)))


def gdn_commit_rows_recompute(cfg: Config, prm: Params, x, a, b, conv_pool, state_pool, slot_idx, accepted,
                              stream=None):
    """Applies the first accepted[b] rows of x/a/b [B, r, ...] to slot_idx[b] in place."""
    c, p = cfg.c(), prm.c()
    B, r = x.shape[0], x.shape[1]
    _check(load().gdn_commit_rows_recompute(ctypes.byref(c), ctypes.byref(p), _p(x), _p(a), _p(b), _p(conv_pool),
                                            _p(state_pool), _p(slot_idx), _p(accepted), B, r, state_pool.shape[0],
                                            _stream(stream)))


def gdn_proj_workspace_size(n_tok: int, n_out: int, k: int) -> int:
    return load().gdn_proj_workspace_size(n_tok, n_out, k)


def gdn_layer_workspace_size(cfg: Config, op: int, n_tokens: int, n_seq: int, hidden: int) -> int:
    c = cfg.c()
    n = load().gdn_layer_workspace_size(ctypes.byref(c), op, n_tokens, n_seq, hidden)
    msg = load().gdn_last_error().decode()
    if msg:
        raise GdnError(-2, msg)
    return n


def gdn_proj_gemm(act, w, out, workspace=None, stream=None):
    """out[t, n] = sum_k act[t, k] w[n, k]: act bf16 [n_tok, k], w bf16 [n_out, k],
    out bf16 [n_tok, >= n_out] (row stride out.shape[1]); workspace of
    gdn_proj_workspace_size bytes (or None when that is 0)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_proj_gemm(_p(act), _p(w), _p(out), act.shape[0], w.shape[0], act.shape[1], out.shape[1],
                                _p(workspace), ws_bytes, _stream(stream)))


def gdn_layer_decode(cfg: Config, prm: Params, proj: Proj, h, conv_pool, state_pool, slot_idx, out, workspace,
                     stream=None):
    """One token for each of B = h.shape[0] slots through in-projection, decode step and
    out-projection; h, out bf16 [B, hidden]."""
    c, p, j = cfg.c(), prm.c(), proj.c()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_layer_decode(ctypes.byref(c), ctypes.byref(p), ctypes.byref(j), _p(h), _p(conv_pool),
                                   _p(state_pool), _p(slot_idx), h.shape[0], state_pool.shape[0], _p(out),
                                   _p(workspace), ws_bytes, _stream(stream)))


def gdn_layer_varlen_prefill(cfg: Config, prm: Params, proj: Proj, h, cu_seqlens, slot_idx, has_init, conv_pool,
                             state_pool, out, workspace, stream=None):
    """Packed sequences of h bf16 [n_tokens, hidden] through in-projection, varlen prefill
    and out-projection into out bf16 [n_tokens, hidden]."""
    c, p, j = cfg.c(), prm.c(), proj.c()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_layer_varlen_prefill(ctypes.byref(c), ctypes.byref(p), ctypes.byref(j), _p(h),
                                           _p(cu_seqlens), slot_idx.numel(), h.shape[0], _p(slot_idx),
                                           _p(has_init), _p(conv_pool), _p(state_pool), state_pool.shape[0], _p(out),
                                           _p(workspace), ws_bytes, _stream(stream)))


def gdn_attn_workspace_size(cfg: AttnConfig, B: int, max_seq_len: int) -> int:
    c = cfg.c()
    n = load().gdn_attn_workspace_size(ctypes.byref(c), B, max_seq_len)
    msg = load().gdn_last_error().decode()
    if msg:
        raise GdnError(-2, msg)
    return n


def gdn_attn_decode(cfg: AttnConfig, q, k_new, v_new, k_pool, v_pool, block_table, seq_lens, max_seq_len: int, o,
                    workspace=None, stream=None):
    """q, o [B, Hq, D]; k_new, v_new [B, Hkv, D]; pools [n_pages, Hkv, page, D];
    block_table int32 [B, max_pages]; seq_lens int32 [B] (tokens before the new one)."""
    c = cfg.c()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_attn_decode(ctypes.byref(c), _p(q), _p(k_new), _p(v_new), _p(k_pool), _p(v_pool),
                                  _p(block_table), _p(seq_lens), q.shape[0], block_table.shape[1], k_pool.shape[0],
                                  int(max_seq_len), _p(o), _p(workspace), ws_bytes, _stream(stream)))


def gdn_attn_prefill(cfg: AttnConfig, q, k_new, v_new, k_pool, v_pool, block_table, cu_seqlens, ctx_lens, o,
                     stream=None):
    """q, o [N, Hq, D]; k_new, v_new [N, Hkv, D]; new tokens of sequence s are rows
    cu_seqlens[s] .. cu_seqlens[s+1] at positions ctx_lens[s] + i."""
    c = cfg.c()
    _check(load().gdn_attn_prefill(ctypes.byref(c), _p(q), _p(k_new), _p(v_new), _p(k_pool), _p(v_pool),
                                   _p(block_table), _p(cu_seqlens), _p(ctx_lens), ctx_lens.numel(), q.shape[0],
                                   block_table.shape[1], k_pool.shape[0], _p(o), _stream(stream)))
