"""Failure handling on the GPU without a fault: a bounded device wait that can never end
gives up, the call reports GPTQ_ERR_TIMEOUT through the status word, and the context stays
usable (the next calls succeed and match the oracle).  The failing pivot of a matrix that
is not positive definite is covered in the prepare tests."""

import time

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from tests.parity import H_REL_FRO, gpu_quantize, rel_fro, to_np, upper_tile_mask
from workloads import make_permutation, make_upper_factor

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ns", [1, 1_000_000, 50_000_000])
def test_bounded_wait_times_out_and_context_survives(lib, cuda_device, limit_ns):
    ws = lib.workspace(256, cuda_device)
    t0 = time.perf_counter()
    with pytest.raises(lib.GptqError) as e:
        lib.gptq_check_wait_timeout(limit_ns, ws)
    elapsed = time.perf_counter() - t0
    assert e.value.status == lib.GPTQ_ERR_TIMEOUT
    assert "1 device-side wait(s) ran out" in str(e.value)
    assert elapsed < 5.0
    # the status word is per call: a normal call on the same workspace's device succeeds
    d = 256
    g = torch.Generator().manual_seed(limit_ns % 997)
    X = (torch.randn(512, d, generator=g) * 2.0).bfloat16()
    H = torch.empty(d, d, dtype=torch.float32, device=cuda_device)
    assert lib.gptq_hessian_accumulate(H, 0, X.to(cuda_device)) == 512
    torch.cuda.synchronize()
    mask = upper_tile_mask(d)
    assert rel_fro(to_np(H)[mask], O.hessian(X.float().numpy())[mask]) <= H_REL_FRO


def test_wait_limit_is_checked(lib, cuda_device):
    ws = lib.workspace(256, cuda_device)
    with pytest.raises(lib.GptqError) as e:
        lib.gptq_check_wait_timeout(0, ws)
    assert e.value.status == lib.GPTQ_ERR_INVALID_ARG
    with pytest.raises(lib.GptqError) as e:
        lib.gptq_check_wait_timeout(2_000_000_000, ws)
    assert e.value.status == lib.GPTQ_ERR_INVALID_ARG


@pytest.mark.parametrize("d,ntok", [(256, 4096), (1024, 20000), (8192, 1024)])
def test_hessian_timeout_drains_and_context_survives(lib, cuda_device, d, ntok):
    """The SYRK itself: with a wait limit of 1 ns its pipeline waits run out while copies
    and matrix operations are in flight; the kernel drains them before it returns (one SM
    pair per cluster at 256 and 1024, two at 8192 with multicast copies) and the call reports
    GPTQ_ERR_TIMEOUT.  Then, with the default limit, the same call succeeds and matches
    the float64 Hessian."""
    g = torch.Generator().manual_seed(d + ntok)
    X = (torch.randn(ntok, d, generator=g) * 2.0).bfloat16()
    Xd = X.to(cuda_device)
    H = torch.empty(d, d, dtype=torch.float32, device=cuda_device)
    lib.gptq_set_wait_limit(1)
    try:
        t0 = time.perf_counter()
        with pytest.raises(lib.GptqError) as e:
            lib.gptq_hessian_accumulate(H, 0, Xd)
        assert time.perf_counter() - t0 < 5.0
    finally:
        lib.gptq_set_wait_limit(0)
    assert e.value.status == lib.GPTQ_ERR_TIMEOUT
    assert lib.gptq_hessian_accumulate(H, 0, Xd) == ntok
    torch.cuda.synchronize()
    Hn = to_np(H)
    Xn = X.double().numpy()
    for bi, bj in [(0, 0), (0, d // 128 - 1), (d // 128 - 1, d // 128 - 1)]:
        r, c = slice(128 * bi, 128 * bi + 128), slice(128 * bj, 128 * bj + 128)
        ref = (2.0 / ntok) * (Xn[:, r].T @ Xn[:, c])
        assert rel_fro(Hn[r, c], ref) <= H_REL_FRO


def _prepare(lib, H, dev):
    d = H.shape[0]
    perm = torch.empty(d, dtype=torch.int32, device=dev)
    dead = torch.empty(d, dtype=torch.uint8, device=dev)
    U = torch.empty(d, d, dtype=torch.float32, device=dev)
    lib.gptq_prepare(H, 0.01, True, perm, dead, U)
    torch.cuda.synchronize()
    return to_np(perm), to_np(U)


@pytest.mark.parametrize("d", [1024, 8192])
def test_prepare_timeout_drains_and_context_survives(lib, cuda_device, d):
    """The prepare's tf32x3 GEMMs (the K = 128 panel steps on one SM; from 8192 also the
    paired-SM superpanel updates) with a wait limit of 1 ns: the call reports
    GPTQ_ERR_TIMEOUT, and with the default limit the same prepare then gives the same
    permutation and factor, bit for bit, as before the failure."""
    g = torch.Generator(device=cuda_device).manual_seed(d)
    X = torch.randn(2 * d, d, generator=g, device=cuda_device) * (
        1.0 + torch.rand(d, generator=g, device=cuda_device))
    H = (2.0 / X.shape[0]) * (X.T @ X)
    perm0, U0 = _prepare(lib, H, cuda_device)
    lib.gptq_set_wait_limit(1)
    try:
        with pytest.raises(lib.GptqError) as e:
            _prepare(lib, H, cuda_device)
    finally:
        lib.gptq_set_wait_limit(0)
    assert e.value.status == lib.GPTQ_ERR_TIMEOUT
    perm1, U1 = _prepare(lib, H, cuda_device)
    assert np.array_equal(perm0, perm1)
    assert np.array_equal(U0, U1)


def test_quantize_timeout_drains_and_context_survives(lib, cuda_device):
    """The lazy update (paired-SM bf16x3 MMAs) with a wait limit of 1 ns: the quantize
    reports GPTQ_ERR_TIMEOUT, and with the default limit it then gives the same outputs,
    bit for bit, as before the failure."""
    m, d = 512, 2304
    g = torch.Generator(device=cuda_device).manual_seed(7)
    W = torch.randn(m, d, generator=g, device=cuda_device) * 0.02
    U = make_upper_factor(d, 7, cuda_device)
    perm = make_permutation(d, 7, cuda_device)
    ref = gpu_quantize(lib, W, U, perm, None, 4, 128, False)
    lib.gptq_set_wait_limit(1)
    try:
        with pytest.raises(lib.GptqError) as e:
            gpu_quantize(lib, W, U, perm, None, 4, 128, False)
    finally:
        lib.gptq_set_wait_limit(0)
    assert e.value.status == lib.GPTQ_ERR_TIMEOUT
    again = gpu_quantize(lib, W, U, perm, None, 4, 128, False)
    for k in ref:
        assert np.array_equal(ref[k], again[k]), k


def test_wait_limit_is_checked_host_side(lib, cuda_device):
    with pytest.raises(lib.GptqError) as e:
        lib.gptq_set_wait_limit(20_000_000_000)
    assert e.value.status == lib.GPTQ_ERR_INVALID_ARG
    lib.gptq_set_wait_limit(0)
