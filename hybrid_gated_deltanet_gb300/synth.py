"""Seeded synthetic inputs for the Gated DeltaNet layer.

This module only draws random numbers and stores them in the storage dtypes
the layer reads (bf16 or fp32).  It holds none of the layer's arithmetic: no
convolution, normalisation, gate or recurrence is computed here.  Both the CUDA
path (through the Python binding) and the CPU oracle (tests only) receive the
arrays produced here, so the two sides see bit-identical inputs.

Shapes follow the statement of the layer on the pages:

* "Hybrid transformers under load: where Gated DeltaNet loses to full
  attention" (braintools.ru), section 4.1: the Qwen3.5-4B state is
  32 x 128 x 128 fp32 (2,097,152 B) plus a 49,152 B conv part per layer, i.e.
  16 k-heads, 32 v-heads, d = 128, 8192 conv channels and 3 stored conv rows in
  bf16.
* "Chapter 6: engine start-up and memory plan" (Strata), section 6.2,
  ModelGeometry: 16 k-heads, 48 v-heads, d_state 128, d_conv 4, 10240 conv
  channels = 2*128*16 + 128*48.

Rounding: values are drawn in fp64 with numpy's PCG64, rounded to fp32 (RNE)
and, for bf16 storage, rounded again fp32 -> bf16 (RNE on the bit pattern).
The decoded values (exact in fp64) are what the oracle consumes.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List

import numpy as np

BF16 = "bf16"
F32 = "f32"


# ----------------------------------------------------------------------------
# storage-dtype helpers (pure bit manipulation, no layer arithmetic)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even); returns uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    bias = 0x7FFF + ((u >> 16) & 1)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact decode of bf16 bit patterns to fp64."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


class LazyF64:
    """fp64 view of a stored array, decoded on indexing (only the slice asked for)."""

    def __init__(self, raw: np.ndarray, dtype: str):
        self._raw = raw
        self._dtype = dtype

    @property
    def shape(self):
        return self._raw.shape

    def _decode(self, part):
        if self._dtype == BF16:
            return bf16_bits_to_f64(part)
        return np.asarray(part, dtype=np.float64)

    def __getitem__(self, idx):
        return self._decode(self._raw[idx])

    def __array__(self, dtype=None, copy=None):
        out = self._decode(self._raw)
        return out if dtype is None else out.astype(dtype)

    def __len__(self):
        return self._raw.shape[0]


class Stored:
    """An array in its storage dtype plus its exact fp64 value.

    ``raw`` is what the GPU receives: uint16 bit patterns for bf16, float32
    otherwise.  ``f64`` decodes the same numbers exactly (lazily, per slice).
    """

    def __init__(self, raw: np.ndarray, dtype: str):
        self.raw = raw
        self.dtype = dtype

    @property
    def f64(self) -> LazyF64:
        return LazyF64(self.raw, self.dtype)

    @property
    def shape(self):
        return self.raw.shape


def store(values: np.ndarray, dtype: str) -> Stored:
    f32 = np.asarray(values, dtype=np.float64).astype(np.float32)
    if dtype == BF16:
        return Stored(f32_to_bf16_bits(f32), BF16)
    if dtype == F32:
        return Stored(np.ascontiguousarray(f32), F32)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def _store_rows(draw, n_rows: int, dtype: str, block: int = 4096) -> Stored:
    """Draw n_rows rows block by block (bounded host memory) and store them."""
    parts = [store(draw(min(block, n_rows - r0)), dtype).raw for r0 in range(0, n_rows, block)]
    if not parts:
        parts = [store(draw(0), dtype).raw]
    return Stored(np.ascontiguousarray(np.concatenate(parts, axis=0)), dtype)


# ----------------------------------------------------------------------------
# geometry
# ----------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Geometry:
    n_k_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    d_conv: int = 4

    @property
    def group(self) -> int:
        return self.n_v_heads // self.n_k_heads

    @property
    def conv_channels(self) -> int:
        # [q | k | v] channel order, head-major
        return 2 * self.n_k_heads * self.d_k + self.n_v_heads * self.d_v

    @property
    def value_dim(self) -> int:
        return self.n_v_heads * self.d_v

    def state_bytes_per_slot(self) -> int:
        return self.n_v_heads * self.d_v * self.d_k * 4

    def conv_state_bytes_per_slot(self, act_dtype: str) -> int:
        return (self.d_conv - 1) * self.conv_channels * (2 if act_dtype == BF16 else 4)


QWEN35_4B = Geometry(16, 32, 128, 128, 4)   # braintools.ru, section 4.1
WIDE_GVA = Geometry(16, 48, 128, 128, 4)    # Strata chapter 6, section 6.2
TINY = Geometry(2, 2, 32, 32, 4)


# ----------------------------------------------------------------------------
# generators
# ----------------------------------------------------------------------------
def make_params(geom: Geometry, rng: np.random.Generator, act_dtype: str) -> Dict[str, Stored]:
    """Per-layer parameters.

    conv_w ~ U(-1/2, 1/2) (= +-1/sqrt(d_conv) for d_conv = 4), A_log ~ U(0, ln 16)
    per v-head, norm_w = 1 + 0.1 N(0,1).  No conv bias, no dt_bias.
    """
    C = geom.conv_channels
    conv_w = rng.uniform(-0.5, 0.5, size=(C, geom.d_conv))
    A_log = rng.uniform(0.0, math.log(16.0), size=(geom.n_v_heads,))
    norm_w = 1.0 + 0.1 * rng.standard_normal(geom.d_v)
    return {
        "conv_w": store(conv_w, act_dtype),
        "A_log": store(A_log, F32),
        "norm_w": store(norm_w, act_dtype),
    }


def make_tokens(geom: Geometry, n_tok: int, rng: np.random.Generator, act_dtype: str,
                x_std: float = 1.0, block: int = 4096) -> Dict[str, Stored]:
    """Per-token layer inputs: x (pre-conv [q|k|v]), z, a, b, all ~ N(0,1).

    Drawn in blocks of ``block`` tokens; within a block the order is x, z, a, b.
    """
    C = geom.conv_channels
    raws = {"x": [], "z": [], "a": [], "b": []}
    for t0 in range(0, max(n_tok, 1), block):
        n = min(block, n_tok - t0) if n_tok > 0 else 0
        raws["x"].append(store(x_std * rng.standard_normal((n, C)), act_dtype).raw)
        raws["z"].append(store(rng.standard_normal((n, geom.value_dim)), act_dtype).raw)
        raws["a"].append(store(rng.standard_normal((n, geom.n_v_heads)), act_dtype).raw)
        raws["b"].append(store(rng.standard_normal((n, geom.n_v_heads)), act_dtype).raw)
    return {k: Stored(np.ascontiguousarray(np.concatenate(v, axis=0)), act_dtype) for k, v in raws.items()}


def make_state(geom: Geometry, n_slots: int, rng: np.random.Generator, std: float = 0.1) -> Stored:
    """fp32 recurrent states [n_slots, H_v, d_v, d_k] ~ N(0, std^2)."""
    shape = (geom.n_v_heads, geom.d_v, geom.d_k)
    return _store_rows(lambda n: std * rng.standard_normal((n,) + shape), n_slots, F32, block=64)


def make_conv_state(geom: Geometry, n_slots: int, rng: np.random.Generator, act_dtype: str,
                    std: float = 0.1) -> Stored:
    """Conv states [n_slots, d_conv-1, C_ch] ~ N(0, std^2) in the act dtype."""
    shape = (geom.d_conv - 1, geom.conv_channels)
    return _store_rows(lambda n: std * rng.standard_normal((n,) + shape), n_slots, act_dtype, block=256)


# model width around the layer: n_embd = 2560 in Strata chapter 6, section 6.2
# (ModelGeometry); the Qwen3.5-4B-like geometry uses the same width
HIDDEN = 2560


def make_proj(geom: Geometry, hidden: int, rng: np.random.Generator) -> Dict[str, Stored]:
    """Projection weights, bf16: w_in [C_ch + H_v*d_v + 2*H_v, hidden] ~ N(0, 1/hidden)
    (rows of x, z, a, b; with h ~ N(0, 1) their outputs are ~ N(0, 1) like the layer
    inputs of the other workloads) and w_out [hidden, H_v*d_v] ~ N(0, 1/(H_v*d_v))."""
    n_in = geom.conv_channels + geom.value_dim + 2 * geom.n_v_heads
    w_in = _store_rows(lambda n: rng.standard_normal((n, hidden)) / math.sqrt(hidden), n_in, BF16, block=2048)
    w_out = _store_rows(lambda n: rng.standard_normal((n, geom.value_dim)) / math.sqrt(geom.value_dim), hidden, BF16,
                        block=2048)
    return {"w_in": w_in, "w_out": w_out}


def make_hidden(n_tok: int, hidden: int, rng: np.random.Generator) -> Stored:
    """Hidden states h [n_tok, hidden] ~ N(0, 1), bf16."""
    return _store_rows(lambda n: rng.standard_normal((n, hidden)), n_tok, BF16, block=2048)


def log_uniform_lengths(rng: np.random.Generator, n: int, lo: int, hi: int) -> List[int]:
    """floor(exp(U(ln lo, ln hi))) sequence lengths."""
    return [int(math.floor(math.exp(v))) for v in rng.uniform(math.log(lo), math.log(hi), size=n)]


def orthonormal_rows(rng: np.random.Generator, n: int, d: int) -> np.ndarray:
    """n <= d orthonormal rows (from the QR factor of a Gaussian matrix)."""
    qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    return np.ascontiguousarray(qm[:, :n].T)


# ----------------------------------------------------------------------------
# named workloads (shapes and distributions of the pages' models)
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    name: str
    geom: Geometry
    act_dtype: str
    chunk: int
    seed: int


WORKLOADS = {
    "tiny": Workload("tiny: 1 seq, T=64, 2/2 heads, d=32, fp32, chunk 16", TINY, F32, 16, 0),
    "decode4b": Workload("Qwen3.5-4B-like decode: 16/32 heads, d=128, bf16, fp32 state",
                         QWEN35_4B, BF16, 64, 1),
    "prefill4b": Workload("chunked prefill: 1 seq, T=8192, 16/32 heads, d=128, bf16, chunk 64",
                          QWEN35_4B, BF16, 64, 2),
    "wide": Workload("wide GVA: 16/48 heads, d=128, 10240 conv channels, bf16", WIDE_GVA, BF16, 64, 3),
    "serving": Workload("serving mix: varlen 20 seqs log-U[500,30000] + decode 256 slots",
                        QWEN35_4B, BF16, 64, 4),
}


def rng_for(seed: int, stream: int = 0) -> np.random.Generator:
    """Independent seeded streams: (seed, stream) -> PCG64."""
    return np.random.Generator(np.random.PCG64([seed, stream]))
