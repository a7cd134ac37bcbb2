"""One layer split across GPUs: token-sharded Hessian, replicated prepare, row-sharded
quantize.

The split follows two facts the pages state.  The Hessian is a sum over calibration
tokens ("GPTQ Architecture, in depth", "The algorithm in code", HessianHook: every batch
adds 2 x x^T), so token slices on different GPUs give partial Hessians that add up.
The output rows of W are quantised independently once U is known ("GPTQ Architecture,
in depth", "The algorithm on one page": each row's column loop touches only that row),
so rows can be split with no exchange until the packed outputs are assembled.  Per
rank:

1. the hook runs over the rank's own token slice (``token_range``);
2. the partial is rescaled from the rank's token count to the total
   (``gptq_hessian_rescale``, a kernel) and one all-reduce (sum) forms H on every rank;
3. every rank runs the prepare on that identical H (replicated: the kernels are
   deterministic, so perm and U agree bit for bit across ranks);
4. rank r quantises rows ``row_range(r)`` (multiples of 32 rows, so that a rank's packed
   zero points are whole 32-bit words);
5. one all-gather per output assembles qweight, scales and qzeros, and the loss is an
   all-reduce (sum).

Only torch.distributed moves data between GPUs (NCCL on GPUs, gloo on CPU); every
arithmetic step runs in the library's kernels through the engine.  The padding and
concatenation around the all-gathers are data movement only.
"""

from __future__ import annotations

from typing import List, Optional, Tuple

import torch

from .api import QuantizedLayer

__all__ = ["token_range", "row_range", "row_ranges", "ShardedLayer"]

ROW_ALIGN = 32  # rows per packed zero-point word group at any bit width


def token_range(rank: int, world: int, ntok: int) -> Tuple[int, int]:
    """Contiguous token slice [t0, t1) of ``rank``: sizes differ by at most one token."""
    if not (0 <= rank < world) or ntok < 0:
        raise ValueError("need 0 <= rank < world and ntok >= 0")
    per, extra = divmod(ntok, world)
    t0 = rank * per + min(rank, extra)
    return t0, t0 + per + (1 if rank < extra else 0)


def row_ranges(world: int, d_out: int, align: int = ROW_ALIGN) -> List[Tuple[int, int]]:
    """Row slices of every rank: whole multiples of ``align`` rows, sizes differing by at
    most ``align`` (a rank may get none when there are fewer row groups than ranks)."""
    if world < 1 or d_out < 0 or d_out % align:
        raise ValueError(f"need world >= 1 and d_out a multiple of {align}")
    units = d_out // align
    per, extra = divmod(units, world)
    out, r = [], 0
    for k in range(world):
        n = (per + (1 if k < extra else 0)) * align
        out.append((r, r + n))
        r += n
    return out


def row_range(rank: int, world: int, d_out: int, align: int = ROW_ALIGN) -> Tuple[int, int]:
    """Row slice [r0, r1) of ``rank`` (see ``row_ranges``)."""
    return row_ranges(world, d_out, align)[rank]


class ShardedLayer:
    """Drives one rank's share of a layer split across ranks.

    ``engine`` is this rank's ``LayerEngine`` built for the rank's rows
    (``d_out = r1 - r0``) and the full ``d_in``; ``group`` is a torch.distributed process
    group (None: the default group, or a single process when torch.distributed is not
    initialised).  ``d_out`` is the layer's full output size.
    """

    def __init__(self, engine, d_out: int, group=None):
        import torch.distributed as dist
        self.eng = engine
        self.pg = group
        self.dist = dist if dist.is_available() and dist.is_initialized() else None
        self.world = self.dist.get_world_size(group) if self.dist else 1
        self.rank = self.dist.get_rank(group) if self.dist else 0
        self.d_out = int(d_out)
        self.rows = row_ranges(self.world, self.d_out)
        r0, r1 = self.rows[self.rank]
        if engine.d_out != r1 - r0:
            raise ValueError(f"rank {self.rank} owns rows [{r0}, {r1}); the engine has "
                             f"d_out = {engine.d_out}")
        self.n_total = 0

    @property
    def row_slice(self) -> Tuple[int, int]:
        return self.rows[self.rank]

    def reset(self) -> None:
        self.eng.reset()
        self.n_total = 0

    def add_batch(self, X_local: torch.Tensor, stream=None) -> None:
        """The hook over a batch of this rank's own tokens."""
        self.eng.add_batch(X_local, stream)

    def combine_hessian(self, stream=None) -> int:
        """Rescale this rank's partial to the total token count and sum the partials over
        ranks; returns the total token count."""
        n_local = int(self.eng.nseen)
        if self.dist is not None:
            n = torch.tensor([n_local], dtype=torch.int64, device=self.eng.H.device)
            self.dist.all_reduce(n, group=self.pg)
            n_total = int(n.item())
        else:
            n_total = n_local
        if n_total == 0:
            raise RuntimeError("no calibration tokens on any rank")
        self.eng.rescale_hessian(n_local, n_total, stream)
        if self.dist is not None:
            self.dist.all_reduce(self.eng.H, group=self.pg)
        self.eng.nseen = n_total
        self.n_total = n_total
        return n_total

    def quantize(self, W_rows: torch.Tensor, stream=None) -> QuantizedLayer:
        """Combine the Hessian, prepare (replicated), quantise this rank's rows and
        assemble the whole layer's packed outputs on every rank."""
        self.combine_hessian(stream)
        self.eng.prepare(stream)
        res = self.eng.quantize_weights(W_rows, stream)
        return self.gather(res)

    def gather(self, res: QuantizedLayer) -> QuantizedLayer:
        """The whole layer's outputs from every rank's row slice."""
        if self.dist is None:
            return res
        bits = self.eng.bits
        widths = [r1 - r0 for r0, r1 in self.rows]
        qweight = self._gather_cols(res.qweight, widths)
        scales = self._gather_cols(res.scales, widths)
        qzeros = self._gather_cols(res.qzeros, [w * bits // 32 for w in widths])
        loss = res.loss.clone()
        self.dist.all_reduce(loss, group=self.pg)
        return QuantizedLayer(qweight, scales, qzeros, res.g_idx, res.perm, loss)

    def _gather_cols(self, t: torch.Tensor, widths: List[int]) -> torch.Tensor:
        """All-gather a [rows, width_r] tensor along its columns (padded to the widest)."""
        wmax = max(widths)
        pad = t.new_zeros(t.shape[0], wmax)
        pad[:, :t.shape[1]] = t
        bufs = [torch.empty_like(pad) for _ in range(self.world)]
        self.dist.all_gather(bufs, pad, group=self.pg)
        return torch.cat([b[:, :w] for b, w in zip(bufs, widths)], dim=1).contiguous()
