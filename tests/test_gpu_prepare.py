"""Parity of gptq_prepare (through the C ABI) with the float64 oracle."""

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from tests.parity import U_REL_FRO, rel_fro, to_np
from workloads import CONFIGS, make_tokens, make_tokens_chunk

pytestmark = pytest.mark.gpu


def _prepare(lib, H32: np.ndarray, damp, actorder, dev):
    d = H32.shape[0]
    H = torch.from_numpy(np.ascontiguousarray(H32)).to(dev)
    perm = torch.empty(d, dtype=torch.int32, device=dev)
    dead = torch.empty(d, dtype=torch.uint8, device=dev)
    U = torch.empty(d, d, dtype=torch.float32, device=dev)
    info = lib.gptq_prepare(H, damp, actorder, perm, dead, U)
    torch.cuda.synchronize()
    return to_np(perm), to_np(dead), to_np(U), info


def _check(lib, H32, damp, actorder, dev):
    perm, dead, U, info = _prepare(lib, H32, damp, actorder, dev)
    ref = O.gptq_prepare(H32.astype(np.float64), damp, actorder)
    assert info == 0
    assert np.array_equal(perm, ref["perm"])
    assert np.array_equal(dead.astype(bool), ref["dead"])
    assert np.allclose(np.tril(U, -1), 0.0)
    err = rel_fro(U, ref["U"])
    assert err <= U_REL_FRO, err
    return perm, U, ref


def _sym_from(X, dead=()):
    H = O.hessian(X)
    for j in dead:
        H[j, :] = 0.0
        H[:, j] = 0.0
    return H.astype(np.float32)


@pytest.mark.parametrize("actorder", [False, True])
def test_prepare_layer_256(lib, cuda_device, actorder):
    cfg = CONFIGS["layer_256x256"]
    H32 = _sym_from(make_tokens(cfg).numpy())
    _check(lib, H32, 0.01, actorder, cuda_device)


def test_prepare_ragged_dead_and_ties(lib, cuda_device):
    """d = 296 (not a multiple of 64 or 128), three dead channels, exact diagonal ties."""
    rng = np.random.default_rng(2)
    d = 296
    X = rng.standard_normal((600, d)) * np.exp(rng.standard_normal(d))
    X[:, 40] = X[:, 7]            # identical channels: equal diagonals, tie by index
    X[:, 250] = X[:, 7]
    H32 = _sym_from(X, dead=(3, 100, 295))
    perm, U, ref = _check(lib, H32, 0.01, True, cuda_device)
    pos = {int(c): k for k, c in enumerate(perm)}
    assert pos[7] < pos[40] < pos[250]


def test_prepare_rank_deficient_needs_damping(lib, cuda_device):
    """n < d makes H singular; 1% damping makes it positive definite ("Same Ruler",
    section 1.6), and without damping the factorisation reports NOT_PD."""
    rng = np.random.default_rng(4)
    d = 128
    X = rng.standard_normal((40, d))
    H32 = _sym_from(X)
    _check(lib, H32, 0.01, True, cuda_device)
    Hbad = H32.copy()
    Hbad[5, 5] = -1.0
    with pytest.raises(lib.GptqError) as e:
        _prepare(lib, Hbad, 0.0, False, cuda_device)
    assert e.value.status == lib.GPTQ_ERR_NOT_PD
    assert e.value.info > 0


def test_prepare_nonfinite(lib, cuda_device):
    d = 64
    H32 = np.eye(d, dtype=np.float32)
    H32[3, 9] = np.nan
    with pytest.raises(lib.GptqError) as e:
        _prepare(lib, H32, 0.01, True, cuda_device)
    assert e.value.status == lib.GPTQ_ERR_NONFINITE


@pytest.mark.slow
def test_prepare_q_proj(lib, cuda_device):
    """d = 4096 with act-order on a Hessian of the q_proj calibration distribution
    (16,384 tokens of it, so that the f64 oracle H takes seconds)."""
    cfg = CONFIGS["q_proj_4096x4096"]
    X = make_tokens_chunk(cfg, 0, "cpu").float().numpy()
    H32 = _sym_from(X)
    perm, U, ref = _check(lib, H32, 0.01, True, cuda_device)
    # the processed diagonal is non-increasing
    assert np.all(np.diff(np.diag(H32)[perm]) <= 0)
