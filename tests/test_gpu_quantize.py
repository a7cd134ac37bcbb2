"""Parity of gptq_quantize_layer (through the C ABI) with the float64 oracle, given the
same W, U and perm on both sides."""

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from tests.parity import check_quantize, gpu_quantize, to_np
from workloads import CONFIGS, make_tokens, make_tokens_chunk, make_weight

pytestmark = pytest.mark.gpu


def _inputs(rng, m, d, n=None, dead=(), actorder=True, wscale=0.02):
    n = 4 * d if n is None else n
    X = rng.standard_normal((n, d)) * np.exp(rng.standard_normal(d))
    for j in dead:
        X[:, j] = 0.0
    H = O.hessian(X)
    prep = O.gptq_prepare(H, 0.01, actorder)
    U32 = prep["U"].astype(np.float32)
    W = (rng.standard_normal((m, d)) * wscale).astype(np.float32)
    return W, U32, prep["perm"], prep["dead"]


def _run(lib, dev, W, U32, perm, dead, bits, group, sym, wdtype=torch.float32, rows=None):
    Wt = torch.from_numpy(W).to(dev).to(wdtype)
    Wn = to_np(Wt).astype(np.float64)        # the values the GPU sees
    Ut = torch.from_numpy(U32).to(dev)
    pt = torch.from_numpy(perm.astype(np.int32)).to(dev)
    dt = torch.from_numpy(dead.astype(np.uint8)).to(dev)
    gpu = gpu_quantize(lib, Wt, Ut, pt, dt, bits, group, sym)
    return check_quantize(Wn, U32.astype(np.float64), perm, dead, bits, group, sym, gpu, rows=rows)


CASES = [
    # (m, d, bits, group, sym, actorder)
    (64, 256, 4, -1, False, False),
    (96, 288, 3, 32, True, True),       # ragged last block of 32 columns
    (64, 384, 2, 64, False, True),
    (32, 256, 8, 128, False, True),
    (64, 640, 4, 256, False, True),     # groups wider than a block, ragged
    (128, 512, 4, 16, True, True),
    (160, 1024, 4, 128, False, True),   # several blocks and row tiles
    (64, 2080, 4, 128, False, True),    # three 1024-column superblocks, the last one a
                                        # ragged block of 32 columns (superblock-end updates)
    (64, 2304, 4, 384, True, True),     # 384-column groups do not nest in a superblock:
                                        # every block is its own, fits outside the loop
]


@pytest.mark.parametrize("m,d,bits,group,sym,actorder", CASES)
def test_quantize_cases(lib, cuda_device, m, d, bits, group, sym, actorder):
    rng = np.random.default_rng(m * 7 + d + bits)
    # wider layers: a full-rank token sample of d + 256 rows keeps the float64 Hessian cheap
    n = None if d <= 1024 else d + 256
    W, U32, perm, dead = _inputs(rng, m, d, n=n, actorder=actorder, dead=(5,))
    rep = _run(lib, cuda_device, W, U32, perm, dead, bits, group, sym)
    assert rep["n_codes"] == m * d


STATIC_CASES = [
    # (m, d, bits, group, sym): act-order on, static groups
    (64, 384, 4, 128, False),
    (96, 288, 3, 32, True),         # ragged last block
    (64, 640, 4, 256, False),       # groups wider than a block, ragged
    (128, 512, 2, 16, False),
    (64, 256, 4, -1, False),        # one group per row: the dynamic mode
    (64, 2080, 4, 128, False),      # three superblocks, the last a ragged block
]


@pytest.mark.parametrize("m,d,bits,group,sym", STATIC_CASES)
def test_quantize_static_groups(lib, cuda_device, m, d, bits, group, sym):
    """Static groups (fixed in the original order before the loop) against the oracle."""
    rng = np.random.default_rng(m * 5 + d + bits + 3)
    n = None if d <= 1024 else d + 256
    W, U32, perm, dead = _inputs(rng, m, d, n=n, actorder=True, dead=(5,))
    Wt = torch.from_numpy(W).to(cuda_device)
    gpu = gpu_quantize(lib, Wt, torch.from_numpy(U32).to(cuda_device),
                       torch.from_numpy(perm.astype(np.int32)).to(cuda_device),
                       torch.from_numpy(dead.astype(np.uint8)).to(cuda_device),
                       bits, group, sym, static_groups=True)
    rep = check_quantize(W.astype(np.float64), U32.astype(np.float64), perm, dead, bits, group,
                         sym, gpu, static_groups=True)
    assert rep["n_codes"] == m * d
    if group != -1:
        assert np.array_equal(gpu["g_idx"], np.arange(d) // group)


def test_quantize_bf16_weights(lib, cuda_device):
    rng = np.random.default_rng(11)
    W, U32, perm, dead = _inputs(rng, 64, 512)
    _run(lib, cuda_device, W, U32, perm, dead, 4, 128, False, wdtype=torch.bfloat16)


def test_quantize_zero_rows_and_constant_groups(lib, cuda_device):
    """All-zero rows (scale 1e-8, zero 0) and rows constant within groups."""
    rng = np.random.default_rng(12)
    W, U32, perm, dead = _inputs(rng, 64, 256)
    W[:8] = 0.0
    W[8:16] = 0.05
    _run(lib, cuda_device, W, U32, perm, dead, 4, 128, False)
    _run(lib, cuda_device, W, U32, perm, dead, 4, 128, True)


def test_quantize_empty_rows(lib, cuda_device):
    d = 128
    dev = cuda_device
    U = torch.eye(d, device=dev)
    loss = torch.full((), 7.0, dtype=torch.float64, device=dev)
    g_idx = torch.empty(d, dtype=torch.int32, device=dev)
    empty = torch.empty(0, device=dev, dtype=torch.int32)
    lib.gptq_quantize_layer(torch.empty(0, d, device=dev), U, None, None, 4, 128, False, 128,
                            empty, empty.float(), empty, g_idx, loss)
    assert float(loss) == 0.0 and bool(torch.all(g_idx == 0))


def test_quantize_nonfinite_weights(lib, cuda_device):
    rng = np.random.default_rng(13)
    W, U32, perm, dead = _inputs(rng, 32, 128)
    W[3, 17] = np.inf
    with pytest.raises(lib.GptqError) as e:
        gpu_quantize(lib, torch.from_numpy(W).to(cuda_device), torch.from_numpy(U32).to(cuda_device),
                     None, None, 4, 128, False)
    assert e.value.status == lib.GPTQ_ERR_NONFINITE


def test_quantize_layer_256(lib, cuda_device):
    """The 256x256 layer: fp32 weights, per-row groups, natural order."""
    cfg = CONFIGS["layer_256x256"]
    X = make_tokens(cfg).numpy()
    prep = O.gptq_prepare(O.hessian(X), cfg.damp, cfg.actorder)
    W = make_weight(cfg).numpy()
    _run(lib, cuda_device, W, prep["U"].astype(np.float32), prep["perm"], prep["dead"],
         cfg.bits, cfg.group, cfg.sym)


@pytest.mark.slow
def test_quantize_q_proj_full(lib, cuda_device):
    """q_proj 4096x4096 bf16 weights, 4-bit asymmetric g128 with act-order, every row."""
    cfg = CONFIGS["q_proj_4096x4096"]
    X = make_tokens_chunk(cfg, 0, "cpu").float().numpy()
    prep = O.gptq_prepare(O.hessian(X), cfg.damp, True)
    W = make_weight(cfg, cuda_device)
    _run(lib, cuda_device, to_np(W), prep["U"].astype(np.float32), prep["perm"], prep["dead"],
         cfg.bits, cfg.group, cfg.sym, wdtype=torch.bfloat16)
