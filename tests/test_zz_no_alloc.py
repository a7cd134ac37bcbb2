"""gptq_hessian_accumulate_noalloc, the entry point for callers that cannot allocate
device memory (it uses the library's own fixed scratch array instead of a caller
workspace), checked through the C ABI against gptq_hessian_accumulate on two calls in a
row.  This file is collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from tests.parity import H_REL_FRO, rel_fro, to_np, upper_tile_mask

pytestmark = pytest.mark.gpu


def _noalloc(lib, H, n, X):
    c = ctypes.c_int64(n)
    st = lib.lib().gptq_hessian_accumulate_noalloc(
        H.data_ptr(), ctypes.byref(c), X.data_ptr(), lib.GPTQ_BF16 if X.dtype == torch.bfloat16
        else lib.GPTQ_F32, X.shape[0], X.shape[1], torch.cuda.current_stream().cuda_stream)
    assert st == lib.GPTQ_OK, lib.gptq_last_error()
    return int(c.value)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 1024), (torch.float32, 256),
                                     (torch.bfloat16, 2048)])    # 2048: one split fills the array
def test_noalloc_matches_workspace_entry_point(lib, cuda_device, dtype, d):
    g = torch.Generator().manual_seed(d)
    X = (torch.randn(3000, d, generator=g) * torch.exp(torch.randn(d, generator=g))).to(dtype)
    X = X.to(cuda_device)
    parts = [X[:1700].contiguous(), X[1700:].contiguous()]
    H_ref = torch.empty(d, d, dtype=torch.float32, device=cuda_device)
    H_new = torch.full((d, d), float("nan"), dtype=torch.float32, device=cuda_device)
    n_ref = n_new = 0
    mask = upper_tile_mask(d)
    for Xp in parts:                        # two calls in a row: the second continues n
        n_ref = lib.gptq_hessian_accumulate(H_ref, n_ref, Xp)
        n_new = _noalloc(lib, H_new, n_new, Xp)
        torch.cuda.synchronize()
        assert n_new == n_ref
        a, b = to_np(H_new), to_np(H_ref)
        assert np.all(np.isfinite(a[mask]))
        assert rel_fro(a[mask], b[mask]) <= H_REL_FRO
    # and directly against the float64 oracle's Hessian of every token so far
    ref = O.hessian(X.float().cpu().numpy().astype(np.float64))
    assert rel_fro(to_np(H_new)[mask], ref[mask]) <= H_REL_FRO


def test_noalloc_rejects_large_d(lib, cuda_device):
    d = 2056
    H = torch.zeros(8, dtype=torch.float32, device=cuda_device)
    X = torch.zeros(4, d, dtype=torch.bfloat16, device=cuda_device)
    c = ctypes.c_int64(0)
    st = lib.lib().gptq_hessian_accumulate_noalloc(H.data_ptr(), ctypes.byref(c), X.data_ptr(),
                                                   lib.GPTQ_BF16, 4, d, None)
    assert st == lib.GPTQ_ERR_UNSUPPORTED
    assert "2048" in lib.gptq_last_error()
    assert c.value == 0
