"""The layer split across ranks (token-sharded Hessian, replicated prepare, row-sharded
quantize) on CPU: two gloo ranks drive ``ShardedLayer`` over an engine stand-in whose
steps are the float64 oracle's, and the assembled outputs must equal the oracle's
single-process layer exactly.  This checks the host logic of the split -- the token and
row ranges, the rescale-and-sum combine of the partial Hessians, the all-gather assembly
of qweight / scales / qzeros and the loss sum -- without a GPU."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from oracle import gptq_oracle as O
from post_weight_quantization_02_gb300 import shard
from post_weight_quantization_02_gb300.api import QuantizedLayer

M, D, N, BITS, GROUP = 96, 64, 700, 3, 32   # 3 row groups of 32 over 2 ranks: ragged split


def _data():
    g = torch.Generator().manual_seed(7)
    X = torch.randn(N, D, generator=g, dtype=torch.float64) * torch.exp(
        torch.randn(D, generator=g, dtype=torch.float64))
    W = torch.randn(M, D, generator=g, dtype=torch.float64) * 0.02
    return X, W


class OracleEngine:
    """The engine's interface with the oracle's float64 steps (test stand-in)."""

    def __init__(self, d_out, d_in):
        self.d_out, self.d_in, self.bits = d_out, d_in, BITS
        self.H = torch.zeros(d_in, d_in, dtype=torch.float64)
        self.nseen = 0

    def reset(self):
        self.nseen = 0

    def add_batch(self, X, stream=None):
        H, n = O.hessian_streaming([X.numpy()])
        t = X.shape[0]
        if t == 0:
            return
        tot = self.nseen + t
        self.H = self.H * (self.nseen / tot) + torch.from_numpy(H) * (t / tot)
        self.nseen = tot

    def rescale_hessian(self, n_from, n_to, stream=None):
        self.H = self.H * (n_from / n_to) if n_from else torch.zeros_like(self.H)

    def prepare(self, stream=None):
        self.prep = O.gptq_prepare(self.H.numpy(), 0.01, True)
        return 0

    def quantize_weights(self, W, stream=None):
        p = self.prep
        out = O.gptq_quantize_layer(W.numpy(), p["U"], p["perm"], p["dead"], BITS, GROUP,
                                    False, 128)
        return QuantizedLayer(torch.from_numpy(out["qweight"]),
                              torch.from_numpy(out["scales"].astype(np.float32)),
                              torch.from_numpy(out["qzeros"]),
                              torch.from_numpy(out["g_idx"].astype(np.int32)),
                              torch.from_numpy(p["perm"].astype(np.int32)),
                              torch.tensor(out["loss"], dtype=torch.float64))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    X, W = _data()
    r0, r1 = shard.row_range(rank, world, M)
    t0, t1 = shard.token_range(rank, world, N)
    sl = shard.ShardedLayer(OracleEngine(r1 - r0, D), M)
    # two uneven batches of the rank's own tokens
    mid = t0 + (t1 - t0) // 3
    sl.add_batch(X[t0:mid])
    sl.add_batch(X[mid:t1])
    res = sl.quantize(W[r0:r1])
    q.put((rank, (r0, r1), (t0, t1), sl.n_total, sl.eng.H.numpy(),
           {f: getattr(res, f).numpy() for f in ("qweight", "scales", "qzeros", "g_idx",
                                                 "perm", "loss")}))
    dist.destroy_process_group()


def test_ranges():
    assert shard.token_range(0, 2, 7) == (0, 4) and shard.token_range(1, 2, 7) == (4, 7)
    assert shard.row_ranges(2, 96) == [(0, 64), (64, 96)]
    assert shard.row_ranges(4, 64) == [(0, 32), (32, 64), (64, 64), (64, 64)]
    for world in (1, 2, 3, 5, 8):
        for m in (0, 32, 96, 4096, 6144):
            rr = shard.row_ranges(world, m)
            assert rr[0][0] == 0 and rr[-1][1] == m
            assert all(a[1] == b[0] for a, b in zip(rr, rr[1:]))
            assert all((r1 - r0) % 32 == 0 for r0, r1 in rr)
            assert max(r1 - r0 for r0, r1 in rr) - min(r1 - r0 for r0, r1 in rr) <= 32
        for n in (0, 1, 700, 524288):
            tr = [shard.token_range(r, world, n) for r in range(world)]
            assert tr[0][0] == 0 and tr[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(tr, tr[1:]))
    with pytest.raises(ValueError):
        shard.row_ranges(2, 100)


def test_two_gloo_ranks_equal_single_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    X, W = _data()
    H = O.hessian(X.numpy())
    ref = O.gptq_layer(W.numpy(), H, BITS, GROUP, False, True, 0.01, 128)
    for rank, rows, toks, n_total, Hr, out in res:
        assert n_total == N
        # the rescaled partials summed over ranks are the whole stream's Hessian
        assert np.allclose(Hr, H, rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(out["perm"], ref["perm"])
        np.testing.assert_array_equal(out["g_idx"], ref["g_idx"])
        np.testing.assert_array_equal(out["qweight"], ref["qweight"])
        np.testing.assert_array_equal(out["qzeros"], ref["qzeros"])
        np.testing.assert_array_equal(out["scales"], ref["scales"].astype(np.float32))
        assert abs(float(out["loss"]) - ref["loss"]) <= 1e-12 * abs(ref["loss"])
    assert [r[1] for r in res] == [(0, 64), (64, 96)]
    assert [r[2] for r in res] == [(0, 350), (350, 700)]
