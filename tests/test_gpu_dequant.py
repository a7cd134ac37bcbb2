"""Parity of gptq_dequant_matmul (through the C ABI) with the float64 oracle: y = x W_hat^T
from the packed checkpoint, for checkpoints the oracle and the GPU quantizer wrote."""

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from tests.parity import gpu_quantize, rel_fro, to_np
from workloads import CONFIGS, make_permutation, make_upper_factor, make_weight

pytestmark = pytest.mark.gpu

# float32 products and sums over d_in terms against float64: the relative Frobenius error
# is about sqrt(d_in) float32 epsilons on random data
Y_REL_FRO = 1e-5


def _oracle_checkpoint(rng, m, d, bits, group, sym, static):
    X = rng.standard_normal((4 * d, d)) * np.exp(rng.standard_normal(d))
    W = rng.standard_normal((m, d)) * 0.02
    return O.gptq_layer(W, O.hessian(X), bits, group, sym, actorder=True, static_groups=static)


def _dev(a, dev, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return t if dtype is None else t.to(dtype)


@pytest.mark.parametrize("m,d,bits,group,sym,static,n,xdt", [
    (96, 256, 4, 32, False, False, 1, torch.bfloat16),
    (96, 256, 4, 32, False, False, 5, torch.bfloat16),
    (64, 384, 3, 64, True, True, 16, torch.bfloat16),
    (160, 512, 2, -1, False, False, 11, torch.float32),
    (32, 1024, 8, 128, False, True, 8, torch.float32),
])
def test_dequant_matmul_small(lib, cuda_device, m, d, bits, group, sym, static, n, xdt):
    rng = np.random.default_rng(m + d + bits + n)
    ck = _oracle_checkpoint(rng, m, d, bits, group, sym, static)
    x = _dev(rng.standard_normal((n, d)).astype(np.float32), cuda_device, xdt)
    y = lib.gptq_dequant_matmul(x, _dev(ck["qweight"], cuda_device),
                                _dev(ck["scales"], cuda_device), _dev(ck["qzeros"], cuda_device),
                                _dev(ck["g_idx"], cuda_device), bits)
    torch.cuda.synchronize()
    ref = O.dequant_matmul(to_np(x).astype(np.float64), ck["qweight"], ck["scales"],
                           ck["qzeros"], ck["g_idx"], bits)
    assert y.shape == (n, m)
    assert rel_fro(to_np(y), ref) <= Y_REL_FRO


def test_dequant_matmul_bad_group_index(lib, cuda_device):
    """A g_idx value outside the scales is reported (the kernel reads group 0 for it)."""
    rng = np.random.default_rng(3)
    ck = _oracle_checkpoint(rng, 64, 256, 4, 128, False, False)
    gi = ck["g_idx"].copy()
    gi[17] = 5                                            # G = 2
    x = _dev(rng.standard_normal((2, 256)).astype(np.float32), cuda_device, torch.bfloat16)
    with pytest.raises(lib.GptqError) as e:
        lib.gptq_dequant_matmul(x, _dev(ck["qweight"], cuda_device),
                                _dev(ck["scales"], cuda_device),
                                _dev(ck["qzeros"], cuda_device), _dev(gi, cuda_device), 4)
    assert e.value.status == lib.GPTQ_ERR_INVALID_ARG


@pytest.mark.slow
@pytest.mark.parametrize("static", [False, True])
def test_dequant_matmul_q_proj(lib, cuda_device, static):
    """The q_proj checkpoint as the GPU quantizer writes it, 8 tokens, against the oracle."""
    cfg = CONFIGS["q_proj_4096x4096"]
    dev, m, d = cuda_device, cfg.d_out, cfg.d_in
    W = make_weight(cfg, dev)
    U = make_upper_factor(d, cfg.seed, dev)
    perm = make_permutation(d, cfg.seed, dev)
    ck = gpu_quantize(lib, W, U, perm, None, cfg.bits, cfg.group, cfg.sym, static_groups=static)
    del W, U
    rng = np.random.default_rng(7)
    x = _dev(rng.standard_normal((8, d)).astype(np.float32), dev, torch.bfloat16)
    y = lib.gptq_dequant_matmul(x, _dev(ck["qweight"], dev), _dev(ck["scales"], dev),
                                _dev(ck["qzeros"], dev), _dev(ck["g_idx"], dev), cfg.bits)
    torch.cuda.synchronize()
    ref = O.dequant_matmul(to_np(x).astype(np.float64), ck["qweight"], ck["scales"],
                           ck["qzeros"], ck["g_idx"], cfg.bits)
    assert rel_fro(to_np(y), ref) <= Y_REL_FRO


@pytest.mark.parametrize("m,d,bits,group,n", [
    (64, 32768, 8, 128, 16),   # eight tokens' x does not fit beside the ring: one per pass
    (96, 28672, 4, 128, 3),    # the table (224 groups) does not fit: global lookups
])
def test_dequant_matmul_wide_random(lib, cuda_device, m, d, bits, group, n):
    """Wide layers on a random valid checkpoint (any codes, positive scales, act-order
    style g_idx), against the oracle's dequantise-then-multiply."""
    rng = np.random.default_rng(d + bits)
    G = d // group
    qweight = rng.integers(-2**31, 2**31, size=(bits * d // 32, m), dtype=np.int64).astype(np.int32)
    qzeros = rng.integers(-2**31, 2**31, size=(G, bits * m // 32), dtype=np.int64).astype(np.int32)
    scales = (rng.random((G, m)) * 0.01 + 1e-3).astype(np.float32)
    g_idx = (rng.permutation(d) // group).astype(np.int32)
    x = _dev(rng.standard_normal((n, d)).astype(np.float32), cuda_device, torch.bfloat16)
    y = lib.gptq_dequant_matmul(x, _dev(qweight, cuda_device), _dev(scales, cuda_device),
                                _dev(qzeros, cuda_device), _dev(g_idx, cuda_device), bits)
    torch.cuda.synchronize()
    ref = O.dequant_matmul(to_np(x).astype(np.float64), qweight, scales, qzeros, g_idx, bits)
    assert rel_fro(to_np(y), ref) <= Y_REL_FRO


@pytest.mark.parametrize("bits,group,static", [(4, 32, False), (3, 64, True), (8, -1, False)])
def test_dequantize_dense(lib, cuda_device, bits, group, static):
    """gptq_dequantize: W_hat = s (code - z) per original column's group.  One float32
    multiply of a float32 scale by a small integer rounds like the oracle's float64 value
    rounded to float32, so float32 output matches exactly; bf16 is that value rounded."""
    rng = np.random.default_rng(bits + group)
    m, d = 96, 256
    ck = _oracle_checkpoint(rng, m, d, bits, group, False, static)
    ref = O.dequantize(ck["qweight"], ck["scales"], ck["qzeros"], ck["g_idx"], bits)
    args = [_dev(ck[k], cuda_device) for k in ("qweight", "scales", "qzeros", "g_idx")]
    W32 = lib.gptq_dequantize(*args, bits, dtype=torch.float32)
    Wbf = lib.gptq_dequantize(*args, bits, dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(W32), ref.astype(np.float32))
    assert torch.equal(Wbf, torch.from_numpy(ref.astype(np.float32)).to(cuda_device).bfloat16())


@pytest.mark.parametrize("n,offset", [(4096, 0), (1001, 0), (1001, 1), (3, 2)])
def test_scales_fp16_matches_round_to_nearest_even(lib, cuda_device, n, offset):
    """The checkpoint's fp16 copy of the scales, bit for bit against numpy's float32 ->
    float16 conversion (round to nearest, ties to even): drawn scales across the fp16
    range, exact ties, the all-zero group's 1e-8 (to zero), subnormals, overflow to inf;
    ragged lengths and unaligned starts take the element-wise path."""
    rng = np.random.default_rng(n + offset)
    s = (10.0 ** rng.uniform(-9, 5.5, n)).astype(np.float32)
    special = np.array([1e-8, 6.0e-8, 3.0e-5, 1.0009765625, 1.00048828125, 65504.0, 65520.0,
                        1e6, 2.0 ** -24, 2.0 ** -25], dtype=np.float32)
    k = min(n, special.size)
    s[:k] = special[:k]
    buf = torch.zeros(n + offset, dtype=torch.float32, device=cuda_device)
    buf[offset:] = torch.from_numpy(s).to(cuda_device)
    out = torch.zeros(n + offset, dtype=torch.float16, device=cuda_device)
    lib.gptq_scales_fp16(buf[offset:], out[offset:])
    torch.cuda.synchronize()
    got = out[offset:].cpu().numpy().view(np.uint16)
    with np.errstate(over="ignore"):  # the overflow to infinity is part of the check
        ref = s.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)
