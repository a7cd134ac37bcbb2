"""Property tests of the float64 oracle over drawn sizes and seeds (hypothesis).

They widen fixed-case pins: the streamed Hessian equals its batch definition under any
chunking; every packed code sits at the bit position the format defines; the column
loop without clipping equals Babai's nearest plane for any shape and block size; the
dequantised weights are linear in the scales and shift with the zero point."""

import numpy as np
import pytest

from oracle import gptq_oracle as O

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

SETTINGS = settings(max_examples=25, deadline=None, derandomize=True)


@SETTINGS
@given(seed=st.integers(0, 2 ** 31 - 1), d=st.integers(1, 24),
       cuts=st.lists(st.integers(0, 40), min_size=1, max_size=6))
def test_streamed_hessian_any_chunking(seed, d, cuts):
    """"GPTQ Architecture, in depth", HessianHook: the running update over any chunking
    (empty chunks included) equals 2/n X^T X of all tokens."""
    rng = np.random.default_rng(seed)
    chunks = [rng.standard_normal((t, d)) for t in cuts]
    n = sum(cuts)
    H, got_n = O.hessian_streaming(chunks)
    assert got_n == n
    if n:
        X = np.concatenate(chunks)
        assert np.allclose(H, 2.0 / n * X.T @ X, rtol=1e-12, atol=1e-12)


@SETTINGS
@given(seed=st.integers(0, 2 ** 31 - 1), bits=st.sampled_from([2, 3, 4, 8]),
       words=st.integers(1, 6), rows=st.integers(1, 3))
def test_pack_bit_positions(seed, bits, words, rows):
    """"04 - GPTQ", section 8 (little-endian streams): bit i of value k is stream bit
    bits*k + i, i.e. bit (bits*k + i) mod 32 of word (bits*k + i) // 32."""
    L = words * 32 // int(np.gcd(bits, 32))      # the shortest whole-word lengths
    rng = np.random.default_rng(seed)
    v = rng.integers(0, 1 << bits, size=(rows, L))
    w = np.asarray(O.pack_bitstream(v, bits)).view(np.uint32)
    for r in range(rows):
        for k in range(L):
            for i in range(bits):
                b = bits * k + i
                assert (int(w[r, b // 32]) >> (b % 32)) & 1 == (int(v[r, k]) >> i) & 1


def _unclipped(s):
    def q(col, w):
        c = np.rint(w / s)
        return c.astype(np.int64), c * s
    return q


@SETTINGS
@given(seed=st.integers(0, 2 ** 31 - 1), d=st.integers(2, 40), m=st.integers(1, 4),
       block=st.sampled_from([1, 3, 8, 128]))
def test_column_loop_is_babai(seed, d, m, block):
    """"04 - GPTQ", section 4: without clipping, GPTQ's codes are Babai's nearest plane
    on the Hessian's lattice, for any shape and block size."""
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((3 * d + 5, d)) * np.exp(rng.standard_normal(d))
    Hd, _ = O.damping(O.hessian(X), 0.01)
    W = rng.standard_normal((m, d)) * 0.02
    s = np.abs(W).max(axis=1) / 7.0 + 1e-6
    r = O.gptq_sweep(W, O.inverse_cholesky_upper(Hd), blocksize=block,
                     column_quantizer=_unclipped(s))
    assert np.array_equal(O.gptq_babai(W, Hd, s), r["codes"])


@SETTINGS
@given(seed=st.integers(0, 2 ** 31 - 1), bits=st.sampled_from([2, 3, 4, 8]),
       c=st.floats(0.25, 4.0))
def test_dequantize_linear_in_scales(seed, bits, c):
    """W_hat = s (code - z): scaling every scale by c scales W_hat by c, and adding 1 to
    every code and zero point (where both stay in range) leaves it unchanged."""
    rng = np.random.default_rng(seed)
    m, d, G = 32, 64, 2
    maxq = (1 << bits) - 1
    codes = rng.integers(0, maxq, size=(m, d))                     # below maxq: room for +1
    zeros = rng.integers(0, maxq, size=(G, m))
    g_idx = (rng.permutation(d) % G).astype(np.int32)
    scales = (rng.random((G, m)) + 0.5).astype(np.float32)
    qw = O.pack_bitstream(codes, bits).T                           # [bits*d/32, m] layout
    qz = O.pack_bitstream(zeros, bits)
    base = O.dequantize(qw, scales, qz, g_idx, bits)
    assert np.allclose(O.dequantize(qw, (scales * np.float32(c)).astype(np.float32), qz,
                                    g_idx, bits),
                       base * np.float64(np.float32(c)), rtol=1e-6)
    shifted = O.dequantize(O.pack_bitstream(codes + 1, bits).T, scales,
                           O.pack_bitstream(zeros + 1, bits), g_idx, bits)
    assert np.array_equal(shifted, base)
