"""Float64 CPU oracle for the block-sequential pipeline.

TEST INFRASTRUCTURE ONLY.  Only ``tests/`` may import it; the product path never does.
It shares no code with the CUDA library.

"GPTQ Architecture, in depth", "The pipeline, block by block": the calibration batch goes
through the model block by block; hooks on every linear layer of a block record its
inputs and accumulate H, each layer is quantised, then the block is run again with the
quantised weights to produce the inputs of the next block.  The block is a random-init
Llama-shaped decoder block (the pages name the layers: q, k, v and o projections, MLP
gate, up and down projections; "Worked example: a 7B model"):

    h1 = rmsnorm(x);  o = attention(h1 Wq^T, h1 Wk^T, h1 Wv^T)   (causal, per head)
    y1 = x + o Wo^T
    h2 = rmsnorm(y1); a = silu(h2 Wg^T) * (h2 Wu^T)
    y  = y1 + a Wd^T

Readings (the pages give no block formula; these are the plainest Llama-style ones):
rmsnorm without a learned gain (random init: gain 1), eps 1e-6; softmax attention scaled
by 1/sqrt(head_dim) with a causal mask; no rotary position encoding; the linears have no
bias.  With grouped-query attention (``kv_heads`` < ``heads``, as in the Llama-3-8B block:
32 query heads, 8 key/value heads, k and v projections of 1024 rows) key/value head j
serves the query heads j*r .. j*r + r - 1, r = heads / kv_heads.  Inputs of the four Hessians: q, k and v share h1 (one H, as the pages' 7B example
shares one Hessian for q, k and v); o sees the attention output; gate and up share h2;
down sees a.  All four come from one forward with the block's own weights, and the block
is re-run once with every linear quantised.
"""

from __future__ import annotations

from typing import Dict, List, Tuple

import numpy as np

from oracle import gptq_oracle as O

F64 = np.float64

GROUPS = (("qkv", ("wq", "wk", "wv")), ("o", ("wo",)), ("gateup", ("wg", "wu")),
          ("down", ("wd",)))


def rmsnorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = np.asarray(x, dtype=F64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, heads: int,
              kv_heads: int = None) -> np.ndarray:
    """Causal multi-head softmax attention; q ``[B, S, h]``, k and v ``[B, S, kv_heads *
    h / heads]`` -> ``[B, S, h]``."""
    B, S, h = q.shape
    hd = h // heads
    kv = heads if kv_heads is None else kv_heads
    def split(t, n):
        return t.reshape(B, S, n, hd).transpose(0, 2, 1, 3)         # [B, n, S, hd]
    qh = split(q, heads)
    # key/value head j serves query heads j*r .. j*r + r - 1
    kh = np.repeat(split(k, kv), heads // kv, axis=1)
    vh = np.repeat(split(v, kv), heads // kv, axis=1)
    scores = qh @ kh.transpose(0, 1, 3, 2) / np.sqrt(hd)            # [B, heads, S, S]
    mask = np.triu(np.ones((S, S), dtype=bool), 1)
    scores = np.where(mask, -np.inf, scores)
    scores = scores - scores.max(axis=-1, keepdims=True)
    p = np.exp(scores)
    p = p / p.sum(axis=-1, keepdims=True)
    return (p @ vh).transpose(0, 2, 1, 3).reshape(B, S, h)


def block_forward(x: np.ndarray, W: Dict[str, np.ndarray], heads: int, kv_heads: int = None
                  ) -> Tuple[np.ndarray, Dict[str, np.ndarray]]:
    """The block's output and the inputs of its four Hessian groups (``[B*S, dim]``)."""
    x = np.asarray(x, dtype=F64)
    B, S, h = x.shape
    h1 = rmsnorm(x)
    o = attention(h1 @ W["wq"].T, h1 @ W["wk"].T, h1 @ W["wv"].T, heads, kv_heads)
    y1 = x + o @ W["wo"].T
    h2 = rmsnorm(y1)
    a = silu(h2 @ W["wg"].T) * (h2 @ W["wu"].T)
    y = y1 + a @ W["wd"].T
    flat = lambda t: t.reshape(B * S, -1)
    return y, {"qkv": flat(h1), "o": flat(o), "gateup": flat(h2), "down": flat(a)}


def quantize_block(x: np.ndarray, W: Dict[str, np.ndarray], heads: int, bits: int = 4,
                   group: int = 128, sym: bool = False, actorder: bool = True,
                   damp: float = 0.01, kv_heads: int = None) -> Dict:
    """One pipeline step: Hessians from the block's own forward, every linear quantised
    (gptq_layer), then the re-forward with the dequantised weights."""
    _, inputs = block_forward(x, W, heads, kv_heads)
    out: Dict = {"inputs": inputs, "H": {}, "layers": {}, "W_hat": {}}
    for gname, names in GROUPS:
        H = O.hessian(inputs[gname])
        out["H"][gname] = H
        for name in names:
            res = O.gptq_layer(W[name], H, bits, group, sym, actorder, damp)
            out["layers"][name] = res
            Q = np.empty_like(res["Q"])
            Q[:, res["perm"]] = res["Q"]                 # original column order
            out["W_hat"][name] = Q
    out["y"], _ = block_forward(x, out["W_hat"], heads, kv_heads)
    return out


def pipeline(x: np.ndarray, blocks: List[Dict[str, np.ndarray]], heads: int, **kw) -> List[Dict]:
    """Blocks in order, each fed the previous quantised block's output."""
    steps = []
    for W in blocks:
        st = quantize_block(x, W, heads, **kw)
        steps.append(st)
        x = st["y"]
    return steps
