"""The byte and flop counts behind the benchmark's roofline figures, checked on CPU
against what fixes them independently: the per-layer state sizes printed by
"Hybrid transformers under load: where Gated DeltaNet loses to full attention"
(braintools.ru, section 4.1; tests/golden/state_geometry.txt), the layer geometry,
and the products the oracle's chunk form actually evaluates."""
import os

import numpy as np
import pytest

import bench
from hybrid_gated_deltanet_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "state_geometry.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def test_decode_bytes_per_slot_follow_the_printed_state_sizes():
    gold = _golden()
    geom = synth.QWEN35_4B
    assert bench.GEOM_ARGS == (geom.n_k_heads, geom.n_v_heads, geom.d_k, geom.d_v, geom.d_conv)
    bf16 = 2
    # the state and the conv state are read and written back once per step
    state_rw = 2 * (gold["qwen35_4b.ssm_state_bytes"] + gold["qwen35_4b.conv_state_bytes"])
    # one token's x (all conv channels), z, a, b in and y out
    token_io = (geom.conv_channels + geom.value_dim + 2 * geom.n_v_heads + geom.value_dim) * bf16
    assert bench.SLOT_BYTES == state_rw + token_io
    # conv weights [C_ch][d_conv], A_log (fp32 per v-head), norm_w [d_v], read once per call
    assert bench.PARAM_BYTES == geom.conv_channels * geom.d_conv * bf16 + geom.n_v_heads * 4 + geom.d_v * bf16


def test_prefill_bytes_follow_the_printed_state_sizes():
    gold = _golden()
    geom = synth.QWEN35_4B
    assert bench.STATE_BYTES == gold["qwen35_4b.layer_state_bytes"]
    assert bench.TOKEN_BYTES == (geom.conv_channels + 2 * geom.value_dim + 2 * geom.n_v_heads) * 2


class _Counting(np.ndarray):
    """An array that records the (m, n, k) shape of every matrix product it takes part in."""
    log = []

    def __array_ufunc__(self, ufunc, method, *inputs, **kwargs):
        args = [np.asarray(x) if isinstance(x, _Counting) else x for x in inputs]
        if ufunc is np.matmul and method == "__call__":
            a, b = args[0], args[1]
            _Counting.log.append((a.shape[-2], b.shape[-1], a.shape[-1]))
        out = getattr(ufunc, method)(*args, **kwargs)
        return out.view(_Counting) if isinstance(out, np.ndarray) else out


class _NumpyWithCountingArrays:
    """numpy, except that the array constructors the chunk form uses return counting arrays."""

    def __getattr__(self, name):
        return getattr(np, name)

    @staticmethod
    def zeros(*a, **k):
        return np.zeros(*a, **k).view(_Counting)

    @staticmethod
    def empty(*a, **k):
        return np.empty(*a, **k).view(_Counting)

    @staticmethod
    def asarray(*a, **k):
        return np.asarray(*a, **k).view(_Counting)

    @staticmethod
    def array(*a, **k):
        return np.array(*a, **k).view(_Counting)


def test_prefill_flops_per_token_match_the_chunk_forms_products(monkeypatch):
    """FLOP_PER_TOKEN against the products oracle.chunk_form evaluates for one v-head.
    Products with a C x C result (K K^T and Q K^T) depend only on the k-head, so the
    layer computes them once per k-head; every other product is per v-head.  The
    oracle inverts I + A with a general solve; the layer's inverse is that of a unit
    lower-triangular C x C matrix, C^3/3 flops per chunk, counted apart."""
    from oracle import chunk_form
    monkeypatch.setattr(chunk_form, "np", _NumpyWithCountingArrays())
    geom = synth.QWEN35_4B
    C, d = bench.C_REF, geom.d_k
    n_chunks = 2
    T = n_chunks * C
    r = np.random.default_rng(0)
    q = r.standard_normal((T, d)) / np.sqrt(d)
    k = r.standard_normal((T, d)) / np.sqrt(d)
    v = r.standard_normal((T, d))
    g = -r.uniform(0.0, 0.5, T)
    beta = r.uniform(0.0, 1.0, T)
    _Counting.log = []
    chunk_form.run_head(q, k, v, g, beta, np.zeros((d, d)), C)
    log = list(_Counting.log)
    assert log, "no matrix product was seen"
    per_khead = sum(2 * m * n * kk for m, n, kk in log if (m, n) == (C, C)) / T
    per_vhead = sum(2 * m * n * kk for m, n, kk in log if (m, n) != (C, C)) / T + C * C / 3
    # K K^T and Q K^T, each 2 C^2 d per chunk
    assert per_khead == pytest.approx(4 * C * d)
    assert per_khead == pytest.approx(bench.FLOP_KHEAD)
    assert per_vhead == pytest.approx(bench.FLOP_VHEAD)
    want = geom.n_k_heads * per_khead + geom.n_v_heads * per_vhead
    assert bench.FLOP_PER_TOKEN == pytest.approx(want, rel=1e-12)
    # 5.29 MFLOP per token and 43.3 GFLOP per 8192-token call, as the prefill roofline states
    assert bench.FLOP_PER_TOKEN * bench.PREFILL_T == pytest.approx(43.3e9, rel=2e-3)
