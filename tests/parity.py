"""Comparison helpers between the CUDA path (through the C ABI) and the float64 oracle."""

from __future__ import annotations

import numpy as np
import torch

from oracle import gptq_oracle as O

# Tolerances of the parity contract.
H_REL_FRO = 1e-5       # Hessian, relative Frobenius error
U_REL_FRO = 1e-4       # inverse Cholesky factor
SCALE_REL = 1e-5       # scales (and zeros, which are integers: exact after replay)
LOSS_REL = 1e-3        # layer loss
CODE_MATCH = 0.999     # fraction of identical codes
TIE_EPS = 1e-3         # |frac - 0.5| below which a pre-rounding value is a near-tie


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def upper_tile_mask(d: int, tile: int = 128) -> np.ndarray:
    i = np.arange(d)
    return (i[:, None] // tile) <= (i[None, :] // tile)


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.cpu().numpy()


def unpack_codes(qweight: np.ndarray, bits: int, d: int) -> np.ndarray:
    """[bits*d/32, m] int32 -> codes [m, d] in original column order."""
    return O.unpack_bitstream(np.ascontiguousarray(qweight.T), bits, d)


def unpack_zeros(qzeros: np.ndarray, bits: int, m: int) -> np.ndarray:
    return O.unpack_bitstream(qzeros, bits, m)


def check_quantize(W, U, perm, dead, bits, group, sym, gpu, rows=None, check_loss=True,
                   w_rows_only=False, static_groups=False):
    """Replay the oracle on (W, U, perm) with the GPU's codes as near-tie hints and check
    every element.  ``gpu`` holds numpy copies of qweight, scales, qzeros, g_idx, loss.
    With ``w_rows_only`` W holds just the sampled ``rows`` (large layers).
    Returns a report dict."""
    m = gpu["scales"].shape[1]
    sel = np.arange(m) if rows is None else np.asarray(rows)
    if rows is not None and not w_rows_only:
        W = np.asarray(W)[sel]
    W = np.asarray(W, dtype=np.float64)
    d = W.shape[1]
    codes_sel = unpack_codes(gpu["qweight"][:, sel], bits, d)   # only the checked rows
    zeros_gpu = unpack_zeros(gpu["qzeros"], bits, m)
    scales_gpu = gpu["scales"]
    perm_np = np.arange(d) if perm is None else np.asarray(perm, dtype=np.int64)
    hint = dict(codes=codes_sel[:, perm_np], zeros=zeros_gpu[:, sel])
    ref = O.gptq_quantize_layer(W, U, perm_np, dead, bits, group, sym, blocksize=128,
                                hint=hint, tie_eps=TIE_EPS, pack=False,
                                static_groups=static_groups)
    n_codes = codes_sel.size
    mismatch = int(np.count_nonzero(ref["codes"] != codes_sel))
    zero_mismatch = int(np.count_nonzero(ref["zeros"] != zeros_gpu[:, sel]))
    ties = ref["stats"].get("codes", 0) + ref["stats"].get("zeros", 0)
    srel = float(np.max(np.abs(ref["scales"].astype(np.float64) - scales_gpu[:, sel])
                        / np.maximum(np.abs(ref["scales"].astype(np.float64)), 1e-30)))
    gidx_ok = np.array_equal(O.group_index(perm_np, group, static_groups), gpu["g_idx"])
    rep = dict(mismatch=mismatch, zero_mismatch=zero_mismatch, near_ties=ties, n_codes=n_codes,
               scale_rel=srel, g_idx_ok=gidx_ok, loss_ref=ref["loss"], loss_gpu=float(gpu["loss"]))
    assert gidx_ok, "g_idx differs"
    assert mismatch == 0, rep
    assert zero_mismatch == 0, rep
    assert 1.0 - ties / n_codes >= CODE_MATCH, rep
    assert srel <= SCALE_REL, rep
    if check_loss and rows is None:
        assert abs(rep["loss_gpu"] - rep["loss_ref"]) <= LOSS_REL * abs(rep["loss_ref"]), rep
    return rep


def gpu_quantize(lib_mod, Wt, U32, perm_t, dead_t, bits, group, sym, blocksize=128,
                 static_groups=False):
    """Run gptq_quantize_layer on device tensors; returns numpy copies of the outputs."""
    m, d = Wt.shape
    dev = Wt.device
    G = 1 if group == -1 else -(-d // group)
    out = dict(
        qweight=torch.empty(bits * d // 32, m, dtype=torch.int32, device=dev),
        scales=torch.empty(G, m, dtype=torch.float32, device=dev),
        qzeros=torch.empty(G, bits * m // 32, dtype=torch.int32, device=dev),
        g_idx=torch.empty(d, dtype=torch.int32, device=dev),
        loss=torch.empty((), dtype=torch.float64, device=dev),
    )
    lib_mod.gptq_quantize_layer(Wt, U32, perm_t, dead_t, bits, group, sym, blocksize,
                                out["qweight"], out["scales"], out["qzeros"], out["g_idx"],
                                out["loss"], static_groups=static_groups)
    torch.cuda.synchronize()
    return {k: to_np(v) for k, v in out.items()}
