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

Y_REL_FRO = 1e-5   # float32 block forward against float64


@pytest.mark.parametrize("static", [False, True])
def test_block_pipeline_small(lib, cuda_device, static):
    torch.backends.cuda.matmul.allow_tf32 = False
    hidden, inter, heads, B, S = 128, 256, 4, 8, 32
    bits, group = 4, 32
    dev = cuda_device
    g = torch.Generator(device="cpu").manual_seed(21)
    x = torch.randn(B, S, hidden, generator=g).to(dev)
    blocks = [make_block_weights(hidden, inter, seed, dev, dtype=torch.float32, std=0.05)
              for seed in (1, 2)]
    bq = BlockQuantizer(hidden, inter, heads, bits=bits, group=group, static_groups=static,
                        seqs_per_chunk=3, max_chunk_tokens=3 * S, device=dev)
    for W in blocks:
        _, inputs = block_forward(x, W, heads)
        layers, y, ex = bq.quantize_block(x, W, keep=True)
        torch.cuda.synchronize()
        for gname, names in GROUPS:
            Xg = to_np(inputs[gname]).astype(np.float64)
            H_gpu = to_np(ex[gname]["H"]).astype(np.float64)
            H_ref = O.hessian(Xg)
            mask = upper_tile_mask(Xg.shape[1])
            assert rel_fro(H_gpu[mask], H_ref[mask]) <= H_REL_FRO, gname
            perm = to_np(ex[gname]["perm"]).astype(np.int64)
            H_sym = np.triu(H_gpu) + np.triu(H_gpu, 1).T
            assert np.array_equal(perm, O.gptq_prepare(H_sym, 0.01, True)["perm"]), gname
            U = to_np(ex[gname]["U"]).astype(np.float64)
            dead = to_np(ex[gname]["dead"]).astype(bool)
            for name in names:
                lay = layers[name]
                gpu = {k: to_np(getattr(lay, k)) for k in
                       ("qweight", "scales", "qzeros", "g_idx", "loss")}
                check_quantize(to_np(W[name]).astype(np.float64), U, perm, dead, bits, group,
                               False, gpu, static_groups=static)
        W_hat = {n: O.dequantize(to_np(l.qweight), to_np(l.scales), to_np(l.qzeros),
                                 to_np(l.g_idx), bits) for n, l in layers.items()}
        y_ref, _ = P.block_forward(to_np(x).astype(np.float64), W_hat, heads)
        assert rel_fro(to_np(y).astype(np.float64), y_ref) <= Y_REL_FRO
        x = y
