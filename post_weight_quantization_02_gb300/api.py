"""Public Python API: one GPTQ layer on one GB300, device-resident or from host buffers.

``LayerEngine`` owns the device buffers of one layer shape (torch allocates them; the
library never does) and drives the three C-ABI calls: ``add_batch`` is the Hessian hook,
``quantize`` runs prepare and the column loop.  ``quantize_layer_from_host`` is the
end-to-end path: host activations and weights in, packed checkpoint tensors out, in one
call of the C ABI that copies token chunks to the device while the Hessian kernels of the
previous chunk run.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

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

    def rescale_hessian(self, n_from: int, n_to: int, stream=None) -> None:
        """H <- H * n_from / n_to: this engine's partial as its share of an n_to-token
        stream (the token-split combine; see ``shard``)."""
        G.gptq_hessian_rescale(self.H, n_from, n_to, stream)

    def prepare(self, stream=None) -> int:
        return G.gptq_prepare(self.H, self.damp, self.actorder, self.perm, self.dead,
                              self.Hinv_chol, self.ws_p, stream)

    def quantize_weights(self, W: torch.Tensor, stream=None) -> QuantizedLayer:
        """The column loop and packing of W with this engine's U and perm.  W may have
        fewer rows than the engine's d_out (layers that share the Hessian but not the
        output size, such as grouped-query k and v beside q); its outputs are then
        allocated for its own rows."""
        m = W.shape[0]
        if m == self.d_out:
            out = (self.qweight, self.scales, self.qzeros, self.g_idx, self.loss)
        elif 0 < m < self.d_out:
            ngroups = self.scales.shape[0]
            dev = self.device
            out = (torch.empty(self.bits * self.d_in // 32, m, dtype=torch.int32, device=dev),
                   torch.empty(ngroups, m, dtype=torch.float32, device=dev),
                   torch.empty(ngroups, self.bits * m // 32, dtype=torch.int32, device=dev),
                   torch.empty(self.d_in, dtype=torch.int32, device=dev),
                   torch.empty((), dtype=torch.float64, device=dev))
        else:
            raise ValueError(f"W has {m} rows; this engine quantises at most {self.d_out}")
        G.gptq_quantize_layer(W, self.Hinv_chol, self.perm, self.dead, self.bits, self.group,
                              self.sym, self.blocksize, *out, self.ws_q, stream,
                              static_groups=self.static_groups)
        return QuantizedLayer(out[0], out[1], out[2], out[3], self.perm, out[4])

    def quantize(self, W: torch.Tensor, stream=None) -> QuantizedLayer:
        """Prepare (damping, act-order, inverse Cholesky factor) then the column loop."""
        if self.nseen == 0:
            raise RuntimeError("no calibration tokens: call add_batch first")
        self.prepare(stream)
        return self.quantize_weights(W, stream)


def quantize_layer_from_host(engine: LayerEngine, W_host: torch.Tensor, X_host: torch.Tensor,
                             out: Optional[QuantizedLayer] = None,
                             chunk_tokens: int = 16384, stream=None) -> QuantizedLayer:
    """End to end from host memory in one C-ABI call (gptq_quantize_layer_host).

    ``X_host`` ``[ntok, d_in]`` and ``W_host`` ``[d_out, d_in]`` are host tensors (page-
    locked, e.g. ``.pin_memory()``, so that the library's chunked copies overlap the
    Hessian kernels).  The engine supplies the quantiser settings and the device; the
    library's device buffer is allocated here by torch, once per chunk size, and kept on
    the engine.  The packed outputs land in ``out`` (host tensors, allocated pinned when
    not given); ``out.loss`` is a float64 host scalar.
    """
    if X_host.dim() != 2 or X_host.shape[1] != engine.d_in:
        raise ValueError("X_host must be [ntok, d_in]")
    m, d, bits = engine.d_out, engine.d_in, engine.bits
    if out is None:
        ngroups = 1 if engine.group == -1 else -(-d // engine.group)
        out = QuantizedLayer(
            torch.empty(bits * d // 32, m, dtype=torch.int32).pin_memory(),
            torch.empty(ngroups, m, dtype=torch.float32).pin_memory(),
            torch.empty(ngroups, bits * m // 32, dtype=torch.int32).pin_memory(),
            torch.empty(d, dtype=torch.int32).pin_memory(),
            torch.empty(d, dtype=torch.int32).pin_memory(),
            torch.empty((), dtype=torch.float64))
    key = (int(chunk_tokens), _dtype_code(X_host), _dtype_code(W_host))
    buf = getattr(engine, "_host_buf", None)
    if buf is None or buf[0] != key:
        nbytes = G.gptq_layer_host_size(chunk_tokens, m, d, bits, engine.group, key[1], key[2])
        if nbytes == 0:
            raise ValueError("unsupported sizes or element types for the host path")
        engine._host_buf = (key, G.workspace(nbytes, engine.device))
    dev = engine._host_buf[1]
    with torch.cuda.device(engine.device):
        loss, _ = G.gptq_quantize_layer_host(
            X_host, W_host, chunk_tokens, engine.damp, engine.actorder, bits, engine.group,
            engine.sym, engine.blocksize, out.qweight, out.scales, out.qzeros, out.g_idx,
            out.perm, dev, stream, static_groups=engine.static_groups)
    out.loss.fill_(loss)
    return out


def _dtype_code(t: torch.Tensor) -> int:
    """The library's element-type code of a tensor."""
    return G.GPTQ_BF16 if t.dtype == torch.bfloat16 else G.GPTQ_F32
