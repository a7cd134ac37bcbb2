"""The block-sequential pipeline on the GPU against the float64 oracle, block by block.

Each block is checked on the inputs the GPU pipeline itself fed it: every group's H
against the oracle's H of the same inputs, its perm exactly, every linear through the
quantize parity check (given the GPU's U), and the quantised block's output against the
oracle's block forward with the GPU's dequantised weights."""

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from oracle import pipeline_oracle as P
from post_weight_quantization_02_gb300.pipeline import (GROUPS, BlockQuantizer, block_forward,
                                                        make_block_weights)
from tests.parity import H_REL_FRO, check_quantize, rel_fro, to_np, upper_tile_mask

pytestmark = pytest.mark.gpu

Y_REL_FRO = 1e-5   # float32 block forward against float64 (hidden 128, MLP 256)
# At the Llama-3-8B widths the float32 forward sums products over up to 14,336 terms in
# each of its seven matrix products; with rounding errors of about sqrt(K) * 2^-24 ~ 7e-6
# per product the block output's relative error reaches a few 1e-5
Y_REL_FRO_WIDE = 1e-4


def _check_block(lib, x, W, layers, y, ex, inputs, heads, kv_heads, bits, group, static,
                 rows=None, y_tol=Y_REL_FRO):
    """Every group's H against the oracle's H of the block's own inputs, perm exactly, every
    linear through the replay check (all rows, or ``rows`` per linear), and the quantised
    block's output against the oracle's block forward with the GPU's dequantised weights."""
    for gname, names in GROUPS:
        Xg = to_np(inputs[gname]).astype(np.float64)
        H_gpu = to_np(ex[gname]["H"]).astype(np.float64)
        H_ref = O.hessian(Xg)
        mask = upper_tile_mask(Xg.shape[1])
        assert rel_fro(H_gpu[mask], H_ref[mask]) <= H_REL_FRO, gname
        del H_ref
        perm = to_np(ex[gname]["perm"]).astype(np.int64)
        H_sym = np.triu(H_gpu) + np.triu(H_gpu, 1).T
        assert np.array_equal(perm, O.act_order(O.fix_dead(H_sym)[0])), gname
        U = to_np(ex[gname]["U"]).astype(np.float64)
        dead = to_np(ex[gname]["dead"]).astype(bool)
        for name in names:
            lay = layers[name]
            gpu = {k: to_np(getattr(lay, k)) for k in
                   ("qweight", "scales", "qzeros", "g_idx", "loss")}
            Wn = to_np(W[name]).astype(np.float64)
            sel = None
            if rows is not None:
                sel = np.sort(np.random.default_rng(len(name)).choice(Wn.shape[0], rows,
                                                                     replace=False))
                Wn = Wn[sel]
            check_quantize(Wn, U, perm, dead, bits, group, False, gpu, rows=sel,
                           check_loss=rows is None, w_rows_only=rows is not None,
                           static_groups=static)
    W_hat = {n: O.dequantize(to_np(l.qweight), to_np(l.scales), to_np(l.qzeros),
                             to_np(l.g_idx), bits) for n, l in layers.items()}
    y_ref, _ = P.block_forward(to_np(x).astype(np.float64), W_hat, heads, kv_heads)
    assert rel_fro(to_np(y).astype(np.float64), y_ref) <= y_tol


@pytest.mark.parametrize("static,kv_heads", [(False, 4), (True, 4), (False, 2)])
def test_block_pipeline_small(lib, cuda_device, static, kv_heads):
    torch.backends.cuda.matmul.allow_tf32 = False
    hidden, inter, heads, B, S = 128, 256, 4, 8, 32
    bits, group = 4, 32
    dev = cuda_device
    g = torch.Generator(device="cpu").manual_seed(21)
    x = torch.randn(B, S, hidden, generator=g).to(dev)
    kv_dim = hidden * kv_heads // heads
    blocks = [make_block_weights(hidden, inter, seed, dev, dtype=torch.float32, std=0.05,
                                 kv_dim=kv_dim) for seed in (1, 2)]
    bq = BlockQuantizer(hidden, inter, heads, bits=bits, group=group, static_groups=static,
                        seqs_per_chunk=3, max_chunk_tokens=3 * S, device=dev, kv_heads=kv_heads)
    for W in blocks:
        _, inputs = block_forward(x, W, heads, kv_heads)
        layers, y, ex = bq.quantize_block(x, W, keep=True)
        torch.cuda.synchronize()
        assert layers["wk"].qweight.shape == (bits * hidden // 32, kv_dim)
        _check_block(lib, x, W, layers, y, ex, inputs, heads, kv_heads, bits, group, static)
        x = y


@pytest.mark.slow
def test_block_pipeline_llama3_8b_width(lib, cuda_device):
    """One block at the Llama-3-8B widths (hidden 4096, 32 query heads, 8 key/value heads,
    MLP 14336), 2 x 256 calibration tokens; 48 sampled rows of every linear replayed."""
    torch.backends.cuda.matmul.allow_tf32 = False
    hidden, inter, heads, kv_heads, B, S = 4096, 14336, 32, 8, 2, 256
    bits, group = 4, 128
    dev = cuda_device
    g = torch.Generator(device="cpu").manual_seed(23)
    x = torch.randn(B, S, hidden, generator=g).to(dev)
    W = make_block_weights(hidden, inter, 5, dev, dtype=torch.float32, std=0.02,
                           kv_dim=hidden * kv_heads // heads)
    bq = BlockQuantizer(hidden, inter, heads, bits=bits, group=group, seqs_per_chunk=1,
                        max_chunk_tokens=S, device=dev, kv_heads=kv_heads)
    _, inputs = block_forward(x, W, heads, kv_heads)
    layers, y, ex = bq.quantize_block(x, W, keep=True)
    torch.cuda.synchronize()
    assert layers["wv"].scales.shape == (hidden // group, 1024)
    _check_block(lib, x, W, layers, y, ex, inputs, heads, kv_heads, bits, group, False, rows=48,
                 y_tol=Y_REL_FRO_WIDE)
