"""Block-sequential GPTQ over a Llama-shaped decoder block.

"GPTQ Architecture, in depth", "The pipeline, block by block": the calibration batch goes
through the model one block at a time; hooks on every linear layer of the block record
its inputs and accumulate H, each layer is quantised, and the block is run again with
the quantised weights to produce the inputs of the next block, so that later layers
partly compensate errors made upstream.

The block (random init here; the pages name its layers in "Worked example: a 7B model"):

    h1 = rmsnorm(x);  o = causal softmax attention of (h1 Wq^T, h1 Wk^T, h1 Wv^T)
    y1 = x + o Wo^T;  h2 = rmsnorm(y1);  a = silu(h2 Wg^T) * (h2 Wu^T);  y = y1 + a Wd^T

q, k and v share one Hessian (their common input h1), as do gate and up (h2); o and down
have their own.  With grouped-query attention (``kv_heads`` < ``heads``: the Llama-3-8B
block has 32 query heads and 8 key/value heads, so k and v have 1024 rows) key/value head
j serves the query heads j*r .. j*r + r - 1, r = heads / kv_heads.  All four are accumulated in one forward with the block's own weights,
through ``LayerEngine.add_batch_async``; every linear is then quantised by the engine and
the block re-run with the dense dequantised weights (``gptq_dequantize``).  The block's
forward is plain PyTorch (the model the method is applied to, not the method); every
step of GPTQ runs in the library's kernels.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import torch
import torch.nn.functional as F

from . import gptq as G
from .api import LayerEngine, QuantizedLayer

GROUPS = (("qkv", ("wq", "wk", "wv")), ("o", ("wo",)), ("gateup", ("wg", "wu")),
          ("down", ("wd",)))
LINEARS = tuple(n for _, names in GROUPS for n in names)


def rmsnorm(x: torch.Tensor, eps: float = 1e-6) -> torch.Tensor:
    xf = x.float()
    return (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + eps)).to(x.dtype)


def block_forward(x: torch.Tensor, W: Dict[str, torch.Tensor], heads: int,
                  kv_heads: Optional[int] = None
                  ) -> Tuple[torch.Tensor, Dict[str, torch.Tensor]]:
    """The block's output ``[B, S, h]`` and the inputs of its four Hessian groups
    (``[B*S, dim]``)."""
    B, S, h = x.shape
    hd = h // heads
    kv = heads if kv_heads is None else int(kv_heads)
    h1 = rmsnorm(x)
    split = lambda t, n: t.view(B, S, n, hd).transpose(1, 2)
    q = split(h1 @ W["wq"].T, heads)
    k, v = (split(h1 @ W[n].T, kv).repeat_interleave(heads // kv, dim=1) for n in ("wk", "wv"))
    o = F.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(1, 2).reshape(B, S, h)
    y1 = x + o @ W["wo"].T
    h2 = rmsnorm(y1)
    a = F.silu(h2 @ W["wg"].T) * (h2 @ W["wu"].T)
    y = y1 + a @ W["wd"].T
    return y, {"qkv": h1.reshape(B * S, h), "o": o.reshape(B * S, h),
               "gateup": h2.reshape(B * S, h), "down": a.reshape(B * S, -1)}


def make_block_weights(hidden: int, inter: int, seed: int, device, dtype=torch.bfloat16,
                       std: float = 0.02, kv_dim: Optional[int] = None
                       ) -> Dict[str, torch.Tensor]:
    """Random-init block weights ([out, in] per linear), seeded; k and v have ``kv_dim``
    rows (grouped-query attention), ``hidden`` by default."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    kvd = hidden if kv_dim is None else int(kv_dim)
    shapes = {"wq": (hidden, hidden), "wk": (kvd, hidden), "wv": (kvd, hidden),
              "wo": (hidden, hidden), "wg": (inter, hidden), "wu": (inter, hidden),
              "wd": (hidden, inter)}
    return {n: (torch.randn(*s, generator=g) * std).to(device=device, dtype=dtype)
            for n, s in shapes.items()}


class BlockQuantizer:
    """GPTQ for one block at a time: four LayerEngines (one per Hessian group)."""

    def __init__(self, hidden: int, inter: int, heads: int, bits: int = 4, group: int = 128,
                 sym: bool = False, actorder: bool = True, damp: float = 0.01,
                 static_groups: bool = False, seqs_per_chunk: int = 8,
                 max_chunk_tokens: int = 16384, device: Optional[torch.device] = None,
                 kv_heads: Optional[int] = None):
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        self.hidden, self.inter, self.heads = int(hidden), int(inter), int(heads)
        self.kv_heads = self.heads if kv_heads is None else int(kv_heads)
        self.bits, self.seqs_per_chunk = int(bits), int(seqs_per_chunk)
        kw = dict(bits=bits, group=group, sym=sym, actorder=actorder, damp=damp,
                  max_chunk_tokens=max_chunk_tokens, device=self.device,
                  static_groups=static_groups)
        self.engines = {"qkv": LayerEngine(hidden, hidden, **kw),
                        "o": LayerEngine(hidden, hidden, **kw),
                        "gateup": LayerEngine(inter, hidden, **kw),
                        "down": LayerEngine(hidden, inter, **kw)}

    def quantize_block(self, x: torch.Tensor, W: Dict[str, torch.Tensor], keep: bool = False
                       ) -> Tuple[Dict[str, QuantizedLayer], torch.Tensor, Dict]:
        """Quantise every linear of the block on the calibration batch ``x`` [B, S, h] and
        return (the packed layers, the quantised block's output, extras).  With ``keep``
        the extras hold each group's H, U, perm and dead (for checking)."""
        B = x.shape[0]
        stream = torch.cuda.current_stream(self.device)
        for eng in self.engines.values():
            eng.reset()
        for b0 in range(0, B, self.seqs_per_chunk):
            _, inp = block_forward(x[b0:b0 + self.seqs_per_chunk], W, self.heads,
                                   self.kv_heads)
            for gname, eng in self.engines.items():
                eng.add_batch_async(inp[gname], stream)
        extras: Dict = {}
        layers: Dict[str, QuantizedLayer] = {}
        for gname, names in GROUPS:
            eng = self.engines[gname]
            eng.hessian_status(stream)
            eng.prepare(stream)
            if keep:
                extras[gname] = dict(H=eng.H.clone(), U=eng.Hinv_chol.clone(),
                                     perm=eng.perm.clone(), dead=eng.dead.clone())
            for name in names:
                q = eng.quantize_weights(W[name], stream)
                layers[name] = QuantizedLayer(*(getattr(q, f.name).clone()
                                                for f in dataclasses.fields(q)))
        W_hat = {n: G.gptq_dequantize(l.qweight, l.scales, l.qzeros, l.g_idx, self.bits,
                                      dtype=x.dtype, stream=stream)
                 for n, l in layers.items()}
        y = torch.cat([block_forward(x[b0:b0 + self.seqs_per_chunk], W_hat, self.heads,
                                     self.kv_heads)[0]
                       for b0 in range(0, B, self.seqs_per_chunk)])
        return layers, y, extras


def quantize_blocks(x: torch.Tensor, blocks, heads: int, **kw):
    """The whole pipeline: each block quantised on the previous quantised block's output.
    Returns the packed layers of every block and the last output."""
    hidden = x.shape[-1]
    inter = blocks[0]["wg"].shape[0]
    kv_heads = heads * blocks[0]["wk"].shape[0] // hidden
    bq = BlockQuantizer(hidden, inter, heads, device=x.device, kv_heads=kv_heads, **kw)
    out = []
    for W in blocks:
        layers, x, _ = bq.quantize_block(x, W)
        out.append(layers)
    return out, x
