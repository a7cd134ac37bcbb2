"""Parity of gptq_hessian_accumulate (through the C ABI) with the float64 oracle."""

import os

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from tests.parity import H_REL_FRO, rel_fro, to_np, upper_tile_mask
from workloads import CONFIGS, make_tokens, make_tokens_chunk, channel_multipliers

pytestmark = pytest.mark.gpu


def _accumulate(lib, chunks, d, dev):
    H = torch.full((d, d), float("nan"), dtype=torch.float32, device=dev)
    n = 0
    for X in chunks:
        n = lib.gptq_hessian_accumulate(H, n, X.to(dev))
    torch.cuda.synchronize()
    return to_np(H), n


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d,ntok", [(256, 3), (256, 128), (296, 1000), (1024, 4160),
                                   (2056, 6000)])
def test_hessian_small(lib, cuda_device, dtype, d, ntok):
    """Ragged column tiles (296, 2056 = 16 * 128 + 8) and token tails (3, 1000, 4160, 6000)
    against the f64 oracle: bf16 tokens on the tensor-core SYRK (128-token stages below
    d_in = 8192; 4160 and 6000 tokens take several token splits, the last one short of a
    whole stage), float32 tokens on the float32 FMA kernel."""
    g = torch.Generator().manual_seed(d + ntok)
    X = (torch.randn(ntok, d, generator=g) * torch.exp(torch.randn(d, generator=g))).to(dtype)
    H, n = _accumulate(lib, [X], d, cuda_device)
    ref = O.hessian(X.float().numpy())
    mask = upper_tile_mask(d)
    assert n == ntok
    assert rel_fro(H[mask], ref[mask]) <= H_REL_FRO
    assert np.all(np.isfinite(H[mask]))


@pytest.mark.parametrize("d,ntok", [(8264, 6000), (8192, 5000), (8192, 7)])
def test_hessian_wide_clusters(lib, cuda_device, d, ntok):
    """Wide layers (d_in >= 8192) run the SYRK in clusters of two SM pairs that share the
    column strip by multicast: a ragged last row and column tile (8264 = 64 * 128 + 72),
    the padded units of column tiles with an odd number of row-tile pairs, two token
    splits added by the reduction (8192, 5000 tokens) and one stage holding 7 tokens.  Sampled 128-blocks (the first, the last on the
    diagonal, blocks of the last column tile and of padded units) against the float64
    Hessian of their columns; the whole diagonal and two quadratic forms against the
    float64 sums."""
    g = torch.Generator().manual_seed(d + ntok)
    X = (torch.randn(ntok, d, generator=g) * torch.exp(0.5 * torch.randn(d, generator=g)))
    X = X.bfloat16()
    H, n = _accumulate(lib, [X], d, cuda_device)
    assert n == ntok
    Xd = X.double().numpy()
    nb = -(-d // 128)
    picks = [(0, 0), (1, 1), (nb - 1, nb - 1), (0, nb - 1), (nb - 2, nb - 1), (2, 2), (3, 4),
             (4, 5), (5, 5), (1, 60), (62, 63), (30, 31)]
    mask = upper_tile_mask(d)
    num = den = 0.0
    for bi, bj in picks:
        r, c = slice(128 * bi, min(d, 128 * bi + 128)), slice(128 * bj, min(d, 128 * bj + 128))
        ref = (2.0 / ntok) * (Xd[:, r].T @ Xd[:, c])
        got = H[r, c].astype(np.float64)
        assert np.all(mask[r, c]) and np.all(np.isfinite(got))
        num += float(np.sum((got - ref) ** 2))
        den += float(np.sum(ref ** 2))
    assert np.sqrt(num / den) <= H_REL_FRO
    diag_ref = (2.0 / ntok) * np.sum(Xd * Xd, axis=0)
    assert np.max(np.abs(np.diag(H) - diag_ref) / diag_ref) <= 1e-5
    Hs = np.where(mask, H, H.T).astype(np.float64)  # the symmetric H from its upper tiles
    for seed in range(2):
        v = np.random.default_rng(seed).standard_normal(d)
        ref = (2.0 / ntok) * float(np.sum((Xd @ v) ** 2))
        assert abs(float(v @ Hs @ v) - ref) <= 1e-5 * abs(ref)


def test_hessian_streaming_chunks(lib, cuda_device):
    """Three uneven calls follow the hook's recurrence (H <- H n/(n+t) + 2/(n+t) X^T X)."""
    d = 384
    g = torch.Generator().manual_seed(5)
    X = (torch.randn(3000, d, generator=g) * 3.0).bfloat16()
    parts = [X[:700], X[700:701], X[701:]]
    H, n = _accumulate(lib, parts, d, cuda_device)
    ref, nref = O.hessian_streaming([p.float().numpy() for p in parts])
    mask = upper_tile_mask(d)
    assert n == nref == 3000
    assert rel_fro(H[mask], ref[mask]) <= H_REL_FRO


def test_hessian_async_matches_sync(lib, cuda_device):
    """The enqueue-only form runs the same kernels in the same order: H is bit-identical
    to the synchronous calls' (and to the oracle within tolerance), the status is OK."""
    d = 384
    g = torch.Generator().manual_seed(11)
    X = (torch.randn(5000, d, generator=g) * 2.0).bfloat16().to(cuda_device)
    parts = [X[:1800], X[1800:1801], X[1801:4000], X[4000:]]
    ws = lib.workspace(lib.gptq_workspace_size(lib.GPTQ_OP_HESSIAN, 4000, 0, d), cuda_device)
    H_sync = torch.full((d, d), float("nan"), dtype=torch.float32, device=cuda_device)
    H_async = torch.full((d, d), float("nan"), dtype=torch.float32, device=cuda_device)
    n = 0
    for p in parts:
        n = lib.gptq_hessian_accumulate(H_sync, n, p, ws)
    na = 0
    for p in parts:
        na = lib.gptq_hessian_accumulate_async(H_async, na, p, ws)
    lib.gptq_hessian_status(ws)
    assert n == na == 5000
    mask = upper_tile_mask(d)
    Hs, Ha = to_np(H_sync), to_np(H_async)
    assert np.array_equal(Hs[mask], Ha[mask])
    ref, _ = O.hessian_streaming([p.float().cpu().numpy() for p in parts])
    assert rel_fro(Ha[mask], ref[mask]) <= H_REL_FRO


def test_hessian_fp32_layer_256(lib, cuda_device):
    """The 256x256 layer's float32 calibration stream (2048 tokens)."""
    cfg = CONFIGS["layer_256x256"]
    X = make_tokens(cfg)
    H, n = _accumulate(lib, [X], cfg.d_in, cuda_device)
    ref = O.hessian(X.numpy())
    mask = upper_tile_mask(cfg.d_in)
    assert n == cfg.n_tokens
    assert rel_fro(H[mask], ref[mask]) <= H_REL_FRO


def test_hessian_zero_tokens_is_noop(lib, cuda_device):
    d = 64
    H = torch.ones(d, d, device=cuda_device)
    n = lib.gptq_hessian_accumulate(H, 5, torch.empty(0, d, dtype=torch.bfloat16, device=cuda_device))
    assert n == 5 and bool(torch.all(H == 1))


@pytest.mark.slow
def test_hessian_q_proj_full(lib, cuda_device):
    """q_proj 4096x4096, 262,144 bf16 tokens with outlier channels, in one call: sampled
    128x128 blocks against the f64 oracle (the ratio estimate of the whole-matrix relative
    Frobenius error, and every sampled entry relative to sqrt(H_ii H_jj)), the diagonal
    closed form, and v^T H v = 2/n ||X v||^2 for random v."""
    cfg = CONFIGS["q_proj_4096x4096"]
    dev = cuda_device
    mult = channel_multipliers(cfg, dev)
    nch = cfg.n_tokens // cfg.chunk
    X = torch.cat([make_tokens_chunk(cfg, i, dev, mult) for i in range(nch)])
    d, n = cfg.d_in, cfg.n_tokens
    H = torch.empty(d, d, dtype=torch.float32, device=dev)
    assert lib.gptq_hessian_accumulate(H, 0, X) == n
    torch.cuda.synchronize()
    Hn = to_np(H)
    # float64 diagonal on the device: the normalising scale of every entry
    diag_ref = (2.0 / n) * (X.double() ** 2).sum(0).cpu().numpy()
    rng = np.random.default_rng(0)
    blocks = [(i, j) for i in range(32) for j in range(i, 32)]
    picks = [blocks[k] for k in rng.choice(len(blocks), 24, replace=False)] + [(0, 0), (31, 31)]
    num = den = 0.0
    worst = 0.0
    for bi, bj in picks:
        a = X[:, bi * 128:(bi + 1) * 128].float().cpu().numpy()
        b = X[:, bj * 128:(bj + 1) * 128].float().cpu().numpy()
        ref = O.hessian_block(np.concatenate([a, b], 1), slice(0, 128), slice(128, 256))
        got = Hn[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
        num += float(np.sum((got - ref) ** 2))
        den += float(np.sum(ref ** 2))
        # each entry against the Cauchy-Schwarz scale sqrt(H_ii H_jj) of its summands
        scale = np.sqrt(np.outer(diag_ref[bi * 128:(bi + 1) * 128],
                                 diag_ref[bj * 128:(bj + 1) * 128]))
        worst = max(worst, float(np.max(np.abs(got - ref) / scale)))
    # ratio estimate of the whole-matrix relative Frobenius error from the sampled tiles
    assert np.sqrt(num / den) <= H_REL_FRO, np.sqrt(num / den)
    assert worst <= H_REL_FRO, worst
    # diagonal: 2/n sum x^2 in float64 on the device
    assert np.max(np.abs(np.diag(Hn) - diag_ref) / diag_ref) <= 1e-5
    # quadratic forms with the symmetric H built from the upper triangle
    Hs = np.triu(Hn) + np.triu(Hn, 1).T
    for s in range(3):
        v = torch.randn(d, generator=torch.Generator().manual_seed(s), dtype=torch.float64)
        xv = X.double() @ v.to(dev)
        ref = float(2.0 / n * (xv * xv).sum())
        got = float(v.numpy() @ Hs @ v.numpy())
        assert abs(got - ref) <= 1e-5 * abs(ref)
    del X
