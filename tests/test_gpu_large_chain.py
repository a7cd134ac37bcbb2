"""The prepare at the wide layers' full widths, the whole GPU chain at q_proj size, and
the column loop as Babai's nearest plane, through the C ABI against the float64 oracle.

* Prepare at d_in = 14336 and 28672 (and at 8264, whose last superpanel and panel are
  ragged) on the Hessian of a token sample (the GPU's own
  Hessian, checked against the oracle): perm bit-exact against the oracle's act-order of
  that Hessian, and rows of U taken across the whole factor (the first, middle and last
  row panels) against the oracle's rows of the factor of the same damped, permuted
  Hessian.
* The whole chain on q_proj (every calibration token): GPU Hessian -> GPU prepare -> GPU
  quantize, with the oracle run on the GPU's Hessian: perm, U, and sampled output rows
  replayed exactly.
* Babai ("04 - GPTQ", section 4): with grids fixed before the loop (static groups) and
  wide enough that no code is clamped, the GPU's codes are Babai's nearest-plane
  coefficients on the lattice the damped Hessian defines.
"""

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from tests.parity import (H_REL_FRO, U_REL_FRO, check_quantize, gpu_quantize, rel_fro, to_np,
                          unpack_codes, upper_tile_mask)
from workloads import CONFIGS, channel_multipliers, make_tokens_chunk, make_weight

pytestmark = pytest.mark.gpu


def _gpu_hessian(lib, cfg, dev, ntok):
    """H of the first ntok tokens of the workload's stream (one call) and those tokens."""
    mult = channel_multipliers(cfg, dev)
    X = make_tokens_chunk(cfg, 0, dev, mult)[:ntok].contiguous()
    H = torch.empty(cfg.d_in, cfg.d_in, dtype=torch.float32, device=dev)
    assert lib.gptq_hessian_accumulate(H, 0, X) == ntok
    return H, X


def _gpu_prepare(lib, H, damp, dev):
    d = H.shape[0]
    perm = torch.empty(d, dtype=torch.int32, device=dev)
    dead = torch.empty(d, dtype=torch.uint8, device=dev)
    U = torch.empty(d, d, dtype=torch.float32, device=dev)
    assert lib.gptq_prepare(H, damp, True, perm, dead, U) == 0
    torch.cuda.synchronize()
    return perm, dead, U


def _sym(Hn):
    """The symmetric float64 matrix of the GPU's H (its upper triangle is authoritative)."""
    H = np.triu(Hn.astype(np.float64))
    return H + np.triu(H, 1).T


@pytest.mark.slow
@pytest.mark.parametrize("name,ntok", [("down_proj_4096x14336", 8192),
                                       ("down_proj_8192x28672", 16384)])
def test_prepare_rows_across_the_factor(lib, cuda_device, name, ntok):
    cfg = CONFIGS[name]
    d = cfg.d_in
    H, X = _gpu_hessian(lib, cfg, cuda_device, ntok)
    # the GPU's Hessian on a sampled diagonal block and the diagonal
    Xb = X[:, :256].double()
    Hn = to_np(H)
    m256 = upper_tile_mask(256)                  # the lower 128-tile is not written
    assert rel_fro(Hn[:256, :256][m256], ((2.0 / ntok) * to_np(Xb.T @ Xb))[m256]) <= H_REL_FRO
    del Xb, X
    perm, dead, U = _gpu_prepare(lib, H, cfg.damp, cuda_device)
    perm_np = to_np(perm).astype(np.int64)
    Hs = _sym(Hn)
    del Hn
    Hf, dead_ref = O.fix_dead(Hs)
    assert np.array_equal(perm_np, O.act_order(Hf))
    assert np.array_equal(to_np(dead).astype(bool), dead_ref)
    Hp = Hf[np.ix_(perm_np, perm_np)]
    del Hf, Hs
    Hd, lam = O.damping(Hp, cfg.damp)
    del Hp
    panels = [np.arange(0, 64), np.arange(d // 2, d // 2 + 64), np.arange(d - 64, d)]
    rows = np.concatenate(panels)
    ref = O.inverse_cholesky_upper_rows(Hd, rows)
    del Hd
    got = to_np(U[torch.from_numpy(rows).to(cuda_device)])
    for k, p in enumerate(panels):
        err = rel_fro(got[k * 64:(k + 1) * 64], ref[k * 64:(k + 1) * 64])
        assert err <= U_REL_FRO, (k, err)
    assert np.all(np.tril(got[:64, :64], -1) == 0.0)


@pytest.mark.slow
def test_prepare_ragged_wide(lib, cuda_device):
    """A wide layer whose width is a whole number of neither superpanels (1024 columns)
    nor panels (128): d_in = 8264 = 8 * 1024 + 72, so the last superpanel and the last
    panel are 72 columns wide.  Perm bit-exact against the oracle's act-order of the
    GPU's Hessian; rows of U across the factor (the first, a middle one, those around the
    ragged superpanel's start, the last) against the oracle's rows of the factor of the
    same damped, permuted Hessian.  16,384 tokens give a full-rank Hessian: with 4096 the
    first rows of U, which condition on the whole matrix, carry 1.3e-4 of rounding at
    d_in = 8192 and 8264 alike (the tail rows 1e-7)."""
    d, ntok, damp = 8264, 16384, 0.01
    g = torch.Generator().manual_seed(d)
    X = (torch.randn(ntok, d, generator=g) * torch.exp(0.5 * torch.randn(d, generator=g)))
    X = X.bfloat16().to(cuda_device)
    H = torch.empty(d, d, dtype=torch.float32, device=cuda_device)
    assert lib.gptq_hessian_accumulate(H, 0, X) == ntok
    del X
    perm, dead, U = _gpu_prepare(lib, H, damp, cuda_device)
    Hs = _sym(to_np(H))
    Hf, dead_ref = O.fix_dead(Hs)
    perm_np = to_np(perm).astype(np.int64)
    assert np.array_equal(perm_np, O.act_order(Hf))
    assert np.array_equal(to_np(dead).astype(bool), dead_ref)
    Hd, _ = O.damping(Hf[np.ix_(perm_np, perm_np)], damp)
    del Hf, Hs
    panels = [np.arange(0, 64), np.arange(4100, 4164), np.arange(8160, 8224),
              np.arange(d - 64, d)]
    rows = np.concatenate(panels)
    assert rows.min() >= 0 and rows.max() < d
    ref = O.inverse_cholesky_upper_rows(Hd, rows)
    got = to_np(U[torch.from_numpy(rows).to(cuda_device)])
    for k, p in enumerate(panels):
        err = rel_fro(got[k * 64:(k + 1) * 64], ref[k * 64:(k + 1) * 64])
        assert err <= U_REL_FRO, (k, err)
    assert np.all(np.tril(got[:64, :64], -1) == 0.0)
    assert np.all(np.tril(got[-64:, d - 64:], -1) == 0.0)


@pytest.mark.slow
def test_whole_chain_q_proj(lib, cuda_device):
    """GPU Hessian over all 262,144 tokens -> GPU prepare -> GPU quantize; the oracle
    prepares the GPU's Hessian and replays 64 sampled output rows."""
    from post_weight_quantization_02_gb300 import LayerEngine
    cfg = CONFIGS["q_proj_4096x4096"]
    dev, m, d = cuda_device, cfg.d_out, cfg.d_in
    eng = LayerEngine(m, d, cfg.bits, cfg.group, cfg.sym, cfg.actorder, cfg.damp,
                      cfg.blocksize, max_chunk_tokens=cfg.chunk, device=dev)
    mult = channel_multipliers(cfg, dev)
    for i in range(cfg.n_tokens // cfg.chunk):
        eng.add_batch(make_tokens_chunk(cfg, i, dev, mult))
    W = make_weight(cfg, dev)
    res = eng.quantize(W)
    torch.cuda.synchronize()
    ref = O.gptq_prepare(_sym(to_np(eng.H)), cfg.damp, cfg.actorder)
    assert np.array_equal(to_np(res.perm).astype(np.int64), ref["perm"])
    assert rel_fro(to_np(eng.Hinv_chol), ref["U"]) <= U_REL_FRO
    sel = np.sort(np.random.default_rng(2).choice(m, 64, replace=False))
    gpu = dict(qweight=to_np(res.qweight), scales=to_np(res.scales), qzeros=to_np(res.qzeros),
               g_idx=to_np(res.g_idx), loss=float(res.loss))
    Wsel = to_np(W[torch.from_numpy(sel).to(dev)]).astype(np.float64)
    rep = check_quantize(Wsel, ref["U"], ref["perm"], ref["dead"], cfg.bits, cfg.group, cfg.sym,
                         gpu, rows=sel, check_loss=False, w_rows_only=True)
    assert rep["n_codes"] == 64 * d


@pytest.mark.parametrize("bits,group", [(8, 64), (8, 128)])
def test_column_loop_is_babai_nearest_plane(lib, cuda_device, bits, group):
    rng = np.random.default_rng(31 + group)
    m, d, n = 512, 256, 1024
    X = rng.standard_normal((n, d)) * np.exp(rng.standard_normal(d))
    W = (rng.standard_normal((m, d)) * 0.02).astype(np.float32).astype(np.float64)
    prep = O.gptq_prepare(O.hessian(X), 0.01, True)
    perm = prep["perm"]
    sc, ze = O.static_group_fit(W, group, bits, False)       # grids fixed before the loop
    gcol = perm // group                                     # group of each processed column
    s_proc = sc[gcol].T.astype(np.float64)                   # [m, d], processing order
    z_proc = ze[gcol].T
    coeff = O.gptq_babai(W[:, perm], prep["Hd"], s_proc)     # Babai's lattice coefficients
    babai = coeff + z_proc                                   # as unsigned codes
    gpu = gpu_quantize(lib, torch.from_numpy(W.astype(np.float32)).to(cuda_device),
                       torch.from_numpy(prep["U"].astype(np.float32)).to(cuda_device),
                       torch.from_numpy(perm.astype(np.int32)).to(cuda_device), None, bits,
                       group, False, static_groups=True)
    codes = unpack_codes(gpu["qweight"], bits, d)[:, perm]   # processing order
    # rows where Babai's coefficients all land on the code grid: there the loop never
    # clamps, so GPTQ and Babai take the same steps.  (Each group's extreme weights sit on
    # the grid's ends, so compensation pushes some of them out in most rows.)
    inside = np.all((babai >= 0) & (babai <= (1 << bits) - 1), axis=1)
    assert inside.sum() >= 32, inside.sum()
    diff = codes[inside] - babai[inside]
    # float32 (GPU) against float64 (Babai): only a pre-rounding value at a tie can go the
    # other way, by one level
    assert np.all(np.abs(diff) <= 1)
    assert np.count_nonzero(diff) <= 1e-3 * diff.size, np.count_nonzero(diff)
