"""The pieces of the multi-GPU split on one GPU, through the C ABI: partial Hessians of
two token slices, each rescaled to the total token count, add up to the one-shot Hessian;
quantising two row slices with the same U and permutation gives the one-call outputs bit
for bit once concatenated.  (The all-reduce and all-gather themselves are exercised by
the gloo test; no test here runs kernels of several ranks on one GPU.)"""

import pytest
import torch

from oracle import gptq_oracle as O
from post_weight_quantization_02_gb300 import LayerEngine, ShardedLayer, shard
from tests.parity import H_REL_FRO, rel_fro, to_np, upper_tile_mask

pytestmark = pytest.mark.gpu


def _inputs(d, m, n, seed):
    g = torch.Generator().manual_seed(seed)
    X = (torch.randn(n, d, generator=g) * torch.exp(torch.randn(d, generator=g))).bfloat16()
    W = (torch.randn(m, d, generator=g) * 0.02).bfloat16()
    return X, W


def _engine(m, d, dev, n, bits=4):
    return LayerEngine(m, d, bits, 128, False, True, 0.01, 128, max_chunk_tokens=n, device=dev)


@pytest.mark.parametrize("bits", [4, 3])
def test_token_split_hessian_and_row_split_quantize(lib, cuda_device, bits):
    d, m, n, cut = 512, 224, 8192, 3000        # 7 row groups of 32: a ragged 128 / 96 split
    X, W = _inputs(d, m, n, 3 + bits)
    Xd, Wd = X.to(cuda_device), W.to(cuda_device)
    full = _engine(m, d, cuda_device, n, bits)
    full.add_batch(Xd)
    full.prepare()
    ref = full.quantize_weights(Wd).to("cpu")
    torch.cuda.synchronize()

    # token split: each slice's partial, rescaled from its own count to the total
    a, b = _engine(m, d, cuda_device, n, bits), _engine(m, d, cuda_device, n, bits)
    a.add_batch(Xd[:cut])
    b.add_batch(Xd[cut:])
    a.rescale_hessian(cut, n)
    b.rescale_hessian(n - cut, n)
    H = to_np(a.H + b.H)                        # the sum an all-reduce forms
    mask = upper_tile_mask(d)
    assert rel_fro(H[mask], to_np(full.H)[mask]) <= H_REL_FRO
    assert rel_fro(H[mask], O.hessian(X.float().numpy())[mask]) <= H_REL_FRO

    # row split with the full engine's U and permutation: bit-exact after concatenation
    parts = []
    for r0, r1 in shard.row_ranges(2, m):
        e = _engine(r1 - r0, d, cuda_device, n, bits)
        e.Hinv_chol.copy_(full.Hinv_chol)
        e.perm.copy_(full.perm)
        e.dead.copy_(full.dead)
        parts.append(e.quantize_weights(Wd[r0:r1].contiguous()).to("cpu"))
    assert [p.qweight.shape[1] for p in parts] == [128, 96]
    for f in ("qweight", "scales", "qzeros"):
        cat = torch.cat([getattr(p, f) for p in parts], dim=1)
        assert torch.equal(cat, getattr(ref, f)), f
    for p in parts:
        assert torch.equal(p.g_idx, ref.g_idx)
    loss = sum(float(p.loss) for p in parts)
    assert abs(loss - float(ref.loss)) <= 1e-12 * abs(float(ref.loss))


def test_sharded_layer_single_process_equals_engine(lib, cuda_device):
    """Without torch.distributed the split is one rank (rescale by n/n = 1): the outputs
    equal the engine's bit for bit."""
    d, m, n = 256, 128, 4096
    X, W = _inputs(d, m, n, 21)
    Xd, Wd = X.to(cuda_device), W.to(cuda_device)
    eng = _engine(m, d, cuda_device, n)
    eng.add_batch(Xd)
    ref = eng.quantize(Wd).to("cpu")
    sl = ShardedLayer(_engine(m, d, cuda_device, n), m)
    sl.add_batch(Xd)
    got = sl.quantize(Wd).to("cpu")
    assert sl.n_total == n
    for f in ("qweight", "scales", "qzeros", "g_idx", "perm", "loss"):
        assert torch.equal(getattr(got, f), getattr(ref, f)), f


def test_rescale_of_an_empty_partial_is_zero(lib, cuda_device):
    d = 256
    H = torch.full((d, d), float("nan"), dtype=torch.float32, device=cuda_device)
    lib.gptq_hessian_rescale(H, 0, 100)
    mask = torch.from_numpy(upper_tile_mask(d)).to(cuda_device)
    assert torch.all(H[mask] == 0)
    assert torch.all(torch.isnan(H[~mask]))      # the rest is left as it was
    H2 = torch.full((d, d), 3.0, dtype=torch.float32, device=cuda_device)
    lib.gptq_hessian_rescale(H2, 1, 4)
    assert torch.all(H2[mask] == 0.75) and torch.all(H2[~mask] == 3.0)
