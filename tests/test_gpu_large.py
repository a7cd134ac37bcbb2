"""Parity at the full sizes of the larger workloads (down_proj 4096x14336, the Llama-3-8B
block's 3-bit gate/up, the 70B-width 8192x28672 down_proj), through the C ABI.

At these sizes the float64 oracle checks sampled outputs exactly (sampled Hessian blocks,
sampled output rows of the column loop, the trailing block of the inverse Cholesky
factor) and properties that hold at any size (the Hessian's diagonal and quadratic forms,
the ordering of the act-order permutation)."""

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from tests.parity import H_REL_FRO, U_REL_FRO, check_quantize, gpu_quantize, rel_fro, to_np
from workloads import (CONFIGS, channel_multipliers, make_permutation, make_tokens_chunk,
                       make_upper_factor, make_weight)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _tile_checks(Hn, cols, diag_ref, n, picks):
    """Ratio estimate of the whole-matrix relative Frobenius error over sampled 128-blocks
    and the worst entry relative to sqrt(H_ii H_jj)."""
    num = den = worst = 0.0
    for bi, bj in picks:
        a, b = cols[bi].astype(np.float64), cols[bj].astype(np.float64)
        ref = (2.0 / n) * (a.T @ b)
        got = Hn[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
        num += float(np.sum((got - ref) ** 2))
        den += float(np.sum(ref ** 2))
        scale = np.sqrt(np.outer(diag_ref[bi * 128:(bi + 1) * 128], diag_ref[bj * 128:(bj + 1) * 128]))
        worst = max(worst, float(np.max(np.abs(got - ref) / scale)))
    return np.sqrt(num / den), worst


@pytest.mark.parametrize("name,streamed", [("down_proj_4096x14336", False),
                                           ("down_proj_8192x28672", True)])
def test_hessian_large(lib, cuda_device, name, streamed):
    """The Hessian of the down_proj streams: 262,144 tokens at d_in = 14336 in one call,
    and 524,288 tokens at d_in = 28672 in 32 calls of 16,384 tokens (the hook's running
    recurrence across calls)."""
    cfg = CONFIGS[name]
    dev, d, n = cuda_device, cfg.d_in, cfg.n_tokens
    nb = d // 128
    picks = [(0, 0), (nb - 1, nb - 1), (3, 200 % nb), (nb // 2, nb // 2 + 1), (7, nb - 2)]
    blocks = sorted({b for p in picks for b in p})
    mult = channel_multipliers(cfg, dev)
    H = torch.empty(d, d, dtype=torch.float32, device=dev)
    cols = {b: [] for b in blocks}
    diag = torch.zeros(d, dtype=torch.float64, device=dev)
    vs = [torch.randn(d, generator=torch.Generator().manual_seed(s), dtype=torch.float64)
          for s in range(2)]
    xv2 = [0.0, 0.0]
    nchunks = n // cfg.chunk
    seen = 0
    chunk_list = []
    for i in range(nchunks):
        X = make_tokens_chunk(cfg, i, dev, mult)
        for b in blocks:
            cols[b].append(X[:, b * 128:(b + 1) * 128].float().cpu().numpy())
        Xd = X.double()
        diag += (Xd * Xd).sum(0)
        for s, v in enumerate(vs):
            xv2[s] += float(((Xd @ v.to(dev)) ** 2).sum())
        del Xd
        if streamed:
            seen = lib.gptq_hessian_accumulate(H, seen, X)
        else:
            chunk_list.append(X)
    if not streamed:
        Xall = torch.cat(chunk_list)
        del chunk_list
        seen = lib.gptq_hessian_accumulate(H, 0, Xall)
        del Xall
    torch.cuda.synchronize()
    assert seen == n
    Hn = to_np(H)
    cols = {b: np.concatenate(v) for b, v in cols.items()}
    diag_ref = (2.0 / n) * diag.cpu().numpy()
    ratio, worst = _tile_checks(Hn, cols, diag_ref, n, picks)
    assert ratio <= H_REL_FRO, ratio
    assert worst <= H_REL_FRO, worst
    assert np.max(np.abs(np.diag(Hn) - diag_ref) / diag_ref) <= 1e-5
    Hs = np.triu(Hn) + np.triu(Hn, 1).T
    for s, v in enumerate(vs):
        ref = 2.0 / n * xv2[s]
        got = float(v.numpy() @ Hs @ v.numpy())
        assert abs(got - ref) <= 1e-5 * abs(ref)


def test_prepare_down_proj_14336(lib, cuda_device):
    """d_in = 14336 from 2,048 tokens of the down_proj stream (rank-deficient: only the
    damping makes H_damp positive definite).  perm equals the oracle's act-order of the same
    H; the trailing 1024 x 1024 block of U, which depends only on the trailing block of
    H_damp in processing order, matches the oracle's factor of that block."""
    cfg = CONFIGS["down_proj_4096x14336"]
    d = cfg.d_in
    X = make_tokens_chunk(cfg, 0, "cpu")[:2048].float().numpy().astype(np.float64)
    H32 = O.hessian(X).astype(np.float32)
    dev = cuda_device
    Ht = torch.from_numpy(H32).to(dev)
    perm = torch.empty(d, dtype=torch.int32, device=dev)
    dead = torch.empty(d, dtype=torch.uint8, device=dev)
    U = torch.empty(d, d, dtype=torch.float32, device=dev)
    assert lib.gptq_prepare(Ht, cfg.damp, True, perm, dead, U) == 0
    torch.cuda.synchronize()
    perm_np, U_np = to_np(perm).astype(np.int64), to_np(U)
    Hf, dead_ref = O.fix_dead(H32.astype(np.float64))
    assert np.array_equal(perm_np, O.act_order(Hf))
    assert np.array_equal(to_np(dead).astype(bool), dead_ref)
    _, lam = O.damping(Hf, cfg.damp)
    r = 1024
    tail = perm_np[d - r:]
    Hd_tail = Hf[np.ix_(tail, tail)] + lam * np.eye(r)
    U_tail = O.inverse_cholesky_upper(Hd_tail)
    assert rel_fro(U_np[d - r:, d - r:], U_tail) <= U_REL_FRO
    assert np.allclose(np.tril(U_np, -1), 0.0)


@pytest.mark.parametrize("name,rows,static", [
    ("down_proj_4096x14336", 64, False),     # symmetric, 4-bit, group 128
    ("block_gateup_w3", 48, False),          # 3-bit, d_out = 28672
    ("down_proj_8192x28672", 32, False),
    ("q_proj_4096x4096", 64, True),          # static groups
    ("down_proj_4096x14336", 32, True),
    ("block_qkv_w4", 48, False),             # the Llama-3-8B block's stacked q/k/v, 6144 rows
    ("block_o_w3", 48, False),               # 3-bit o_proj
    ("block_down_w3", 32, False),            # 3-bit down_proj, d_in = 14336
])
def test_quantize_large(lib, cuda_device, name, rows, static):
    """The column loop and packing at full size with a drawn inverse Cholesky factor and
    permutation (any positive-diagonal upper-triangular U is the factor of some positive
    definite Hessian); sampled output rows are checked exactly against the oracle."""
    cfg = CONFIGS[name]
    dev, m, d = cuda_device, cfg.d_out, cfg.d_in
    W = make_weight(cfg, dev)
    U = make_upper_factor(d, cfg.seed, dev)
    perm = make_permutation(d, cfg.seed, dev)
    gpu = gpu_quantize(lib, W, U, perm, None, cfg.bits, cfg.group, cfg.sym,
                       static_groups=static)
    sel = np.sort(np.random.default_rng(cfg.seed).choice(m, rows, replace=False))
    Wsel = to_np(W[torch.from_numpy(sel).to(dev)])
    del W
    Un = to_np(U)
    del U
    rep = check_quantize(Wsel, Un, to_np(perm), None, cfg.bits, cfg.group, cfg.sym, gpu,
                         rows=sel, check_loss=False, w_rows_only=True, static_groups=static)
    assert rep["n_codes"] == rows * d
