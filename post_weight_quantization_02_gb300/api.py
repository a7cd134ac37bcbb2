"""Public Python API: one GPTQ layer on one GB300, device-resident or from host buffers.

``LayerEngine`` owns the device buffers of one layer shape (torch allocates them; the
library never does) and drives the three C-ABI calls: ``add_batch`` is the Hessian hook,
``quantize`` runs prepare and the column loop.  ``quantize_layer_from_host`` is the
end-to-end path: pinned host activations and weights in, packed checkpoint tensors out,
with the host-to-device copies of token chunks overlapped with the Hessian kernels.
"""

from __future__ import annotations

import dataclasses
from typing import Iterable, Optional

import torch

from . import gptq as G

__all__ = ["LayerEngine", "QuantizedLayer", "quantize_layer_from_host"]


@dataclasses.dataclass
class QuantizedLayer:
    """Packed GPTQ checkpoint tensors of one layer (see include/gptq.h for layouts)."""

    qweight: torch.Tensor   # int32 [bits*d_in/32, d_out]
    scales: torch.Tensor    # float32 [G, d_out]
    qzeros: torch.Tensor    # int32 [G, bits*d_out/32]
    g_idx: torch.Tensor     # int32 [d_in]
    perm: torch.Tensor      # int32 [d_in]
    loss: torch.Tensor      # float64 scalar

    def to(self, device, non_blocking=False) -> "QuantizedLayer":
        return QuantizedLayer(*(getattr(self, f.name).to(device, non_blocking=non_blocking)
                                for f in dataclasses.fields(self)))


class LayerEngine:
    def __init__(self, d_out: int, d_in: int, bits: int = 4, group: int = 128,
                 sym: bool = False, actorder: bool = True, damp: float = 0.01,
                 blocksize: int = 128, max_chunk_tokens: int = 16384,
                 device: Optional[torch.device] = None, static_groups: bool = False):
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        self.d_out, self.d_in = int(d_out), int(d_in)
        self.bits, self.group, self.sym = int(bits), int(group), bool(sym)
        self.actorder, self.damp, self.blocksize = bool(actorder), float(damp), int(blocksize)
        self.static_groups = bool(static_groups)
        dev, d, m = self.device, self.d_in, self.d_out
        ngroups = 1 if group == -1 else -(-d // group)
        self.H = torch.empty(d, d, dtype=torch.float32, device=dev)
        self.nseen = 0
        self.Hinv_chol = torch.empty(d, d, dtype=torch.float32, device=dev)
        self.perm = torch.empty(d, dtype=torch.int32, device=dev)
        self.dead = torch.empty(d, dtype=torch.uint8, device=dev)
        self.qweight = torch.empty(bits * d // 32, m, dtype=torch.int32, device=dev)
        self.scales = torch.empty(ngroups, m, dtype=torch.float32, device=dev)
        self.qzeros = torch.empty(ngroups, bits * m // 32, dtype=torch.int32, device=dev)
        self.g_idx = torch.empty(d, dtype=torch.int32, device=dev)
        self.loss = torch.empty((), dtype=torch.float64, device=dev)
        self.ws_h = G.workspace(G.gptq_workspace_size(G.GPTQ_OP_HESSIAN, max_chunk_tokens, m, d),
                                dev)
        self.ws_p = G.workspace(G.gptq_workspace_size(G.GPTQ_OP_PREPARE, 0, m, d), dev)
        self.ws_q = G.workspace(G.gptq_workspace_size(G.GPTQ_OP_QUANTIZE, 0, m, d, bits, group),
                                dev)

    def reset(self) -> None:
        self.nseen = 0

    def add_batch(self, X: torch.Tensor, stream=None) -> None:
        """The Hessian hook for one batch of activations ``[tokens, d_in]``."""
        X = X.reshape(-1, self.d_in)
        self.nseen = G.gptq_hessian_accumulate(self.H, self.nseen, X, self.ws_h, stream)

    def add_batch_async(self, X: torch.Tensor, stream=None) -> None:
        """The Hessian hook for one batch, enqueued without waiting (X must stay valid
        until the stream reaches the work); hessian_status() reports device failures."""
        X = X.reshape(-1, self.d_in)
        self.nseen = G.gptq_hessian_accumulate_async(self.H, self.nseen, X, self.ws_h, stream)

    def hessian_status(self, stream=None) -> None:
        """Wait for the enqueued Hessian steps and raise the first device-side failure."""
        G.gptq_hessian_status(self.ws_h, stream)

    def prepare(self, stream=None) -> int:
        return G.gptq_prepare(self.H, self.damp, self.actorder, self.perm, self.dead,
                              self.Hinv_chol, self.ws_p, stream)

    def quantize_weights(self, W: torch.Tensor, stream=None) -> QuantizedLayer:
        G.gptq_quantize_layer(W, self.Hinv_chol, self.perm, self.dead, self.bits, self.group,
                              self.sym, self.blocksize, self.qweight, self.scales, self.qzeros,
                              self.g_idx, self.loss, self.ws_q, stream,
                              static_groups=self.static_groups)
        return QuantizedLayer(self.qweight, self.scales, self.qzeros, self.g_idx, self.perm,
                              self.loss)

    def quantize(self, W: torch.Tensor, stream=None) -> QuantizedLayer:
        """Prepare (damping, act-order, inverse Cholesky factor) then the column loop."""
        if self.nseen == 0:
            raise RuntimeError("no calibration tokens: call add_batch first")
        self.prepare(stream)
        return self.quantize_weights(W, stream)


def quantize_layer_from_host(engine: LayerEngine, W_host: torch.Tensor,
                             X_chunks_host: Iterable[torch.Tensor],
                             out: Optional[QuantizedLayer] = None) -> QuantizedLayer:
    """End to end from (pinned) host memory.

    Token chunks are copied host-to-device on a side stream, double buffered, while the
    Hessian kernels of the previous chunk run (enqueued without waiting, so the host
    issues the next copy at once); the weights follow; the packed outputs are copied back
    into ``out`` (pinned host tensors) when given.
    """
    dev = engine.device
    compute = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    bufs = [None, None]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    engine.reset()
    for i, xh in enumerate(X_chunks_host):
        b = i % 2
        if bufs[b] is None or bufs[b].shape != xh.shape or bufs[b].dtype != xh.dtype:
            bufs[b] = torch.empty(xh.shape, dtype=xh.dtype, device=dev)
        with torch.cuda.stream(copy):
            copy.wait_event(done[b])
            bufs[b].copy_(xh, non_blocking=True)
            ready[b].record(copy)
        compute.wait_event(ready[b])
        engine.add_batch_async(bufs[b], compute)
        done[b].record(compute)
    if engine.nseen == 0:
        raise RuntimeError("no calibration tokens: X_chunks_host was empty")
    with torch.cuda.stream(copy):
        Wd = W_host.to(dev, non_blocking=True)
        wready = torch.cuda.Event()
        wready.record(copy)
    engine.hessian_status(compute)
    engine.prepare(compute)
    compute.wait_event(wready)
    res = engine.quantize_weights(Wd, compute)
    if out is None:
        return res.to("cpu")
    for f in dataclasses.fields(out):
        getattr(out, f.name).copy_(getattr(res, f.name), non_blocking=True)
    compute.synchronize()
    return out
