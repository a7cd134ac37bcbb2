"""Seeded synthetic layers shaped like the GPTQ pages' workloads.

The pages calibrate on 128 segments of 2048 tokens (GPTQ Architecture, in depth,
"Groups, act-order and other knobs"; 04 - GPTQ, section 5) and quantise Llama-shaped
linears.  No dataset or trained weight is available, so every tensor here is drawn from
a seeded torch generator with the shape, dtype and value distribution of those
workloads:

* weights ``W`` are ``[d_out, d_in]`` Gaussian with a per-layer standard deviation;
* calibration activations ``X`` are token-major ``[n_tokens, d_in]`` (a Linear's input
  flattened to ``[tokens, cols]``), either Gaussian with a log-normal magnitude per input
  channel or a gated-MLP product ``SiLU(N(0,1)) * N(0,1)``, optionally with a fraction of
  outlier channels multiplied by a constant.

``X`` is produced in chunks of ``chunk`` tokens, each from its own seed, so that a long
calibration stream can be regenerated chunk by chunk without ever materialising it.

The generators are device-agnostic: the same seed on the same device type gives the same
tensor; a CPU draw and a CUDA draw differ.  A test that compares the CUDA path with the
oracle hands both sides the very same tensor.
"""

from __future__ import annotations

import dataclasses
from typing import Iterator, Optional, Tuple

import torch

__all__ = [
    "LayerConfig",
    "CONFIGS",
    "channel_multipliers",
    "make_weight",
    "make_tokens_chunk",
    "make_tokens",
    "token_chunks",
]


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """One synthetic linear layer plus its calibration stream and quantiser knobs."""

    name: str
    d_out: int
    d_in: int
    n_tokens: int
    w_std: float
    w_dtype: torch.dtype
    x_dtype: torch.dtype
    x_kind: str  # "lognormal_gauss" or "silu_gated"
    x_sigma: float = 1.0  # log-normal sigma of the per-channel magnitudes
    outlier_frac: float = 0.0
    outlier_mult: float = 1.0
    bits: int = 4
    group: int = 128  # -1: one group per row
    sym: bool = False
    actorder: bool = True
    blocksize: int = 128
    damp: float = 0.01
    seed: int = 0
    chunk: int = 16384

    def replace(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)


# The five workloads.  Seeds follow "seed = index"; the weight, channel and token streams
# of one config draw from disjoint seed ranges.
CONFIGS = {
    "layer_256x256": LayerConfig(
        name="layer_256x256", d_out=256, d_in=256, n_tokens=2048, w_std=0.02,
        w_dtype=torch.float32, x_dtype=torch.float32, x_kind="lognormal_gauss", x_sigma=0.5,
        bits=4, group=-1, sym=False, actorder=False, seed=0, chunk=2048),
    "q_proj_4096x4096": LayerConfig(
        name="q_proj_4096x4096", d_out=4096, d_in=4096, n_tokens=128 * 2048, w_std=0.02,
        w_dtype=torch.bfloat16, x_dtype=torch.bfloat16, x_kind="lognormal_gauss", x_sigma=1.0,
        outlier_frac=0.01, outlier_mult=20.0, bits=4, group=128, sym=False, actorder=True,
        seed=1),
    "down_proj_4096x14336": LayerConfig(
        name="down_proj_4096x14336", d_out=4096, d_in=14336, n_tokens=128 * 2048,
        w_std=0.015, w_dtype=torch.bfloat16, x_dtype=torch.bfloat16, x_kind="silu_gated",
        bits=4, group=128, sym=True, actorder=True, seed=2),
    "down_proj_8192x28672": LayerConfig(
        name="down_proj_8192x28672", d_out=8192, d_in=28672, n_tokens=256 * 2048,
        w_std=0.01, w_dtype=torch.bfloat16, x_dtype=torch.bfloat16, x_kind="silu_gated",
        outlier_frac=0.005, outlier_mult=30.0, bits=4, group=128, sym=False, actorder=True,
        seed=4),
}


def _llama3_8b_block(bits: int) -> dict:
    """The seven linears of one Llama-3-8B-shaped block, grouped by shared input.

    q/k/v read the same hidden state and gate/up read the same normalised state, so each
    group shares one Hessian; their weights are stacked along d_out.
    """
    base = dict(w_std=0.02, w_dtype=torch.bfloat16, x_dtype=torch.bfloat16,
                x_kind="lognormal_gauss", x_sigma=1.0, n_tokens=128 * 2048, bits=bits,
                group=128, sym=False, actorder=True)
    return {
        f"block_qkv_w{bits}": LayerConfig(name=f"block_qkv_w{bits}", d_out=4096 + 1024 + 1024,
                                          d_in=4096, seed=3, **base),
        f"block_o_w{bits}": LayerConfig(name=f"block_o_w{bits}", d_out=4096, d_in=4096,
                                        seed=3 + 10, **base),
        f"block_gateup_w{bits}": LayerConfig(name=f"block_gateup_w{bits}", d_out=2 * 14336,
                                             d_in=4096, seed=3 + 20, **base),
        f"block_down_w{bits}": LayerConfig(name=f"block_down_w{bits}", d_out=4096,
                                           d_in=14336, seed=3 + 30, **base),
    }


BLOCK_CONFIGS = {**_llama3_8b_block(4), **_llama3_8b_block(3)}
CONFIGS.update(BLOCK_CONFIGS)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device).type)
    g.manual_seed(int(seed))
    return g


def channel_multipliers(cfg: LayerConfig, device="cpu") -> torch.Tensor:
    """Per-input-channel magnitudes, float32 ``[d_in]``.

    ``lognormal_gauss``: exp(sigma * N(0,1)) per channel; ``silu_gated``: 1.  Then a random
    ``outlier_frac`` of the channels is multiplied by ``outlier_mult``.
    """
    g = _gen(cfg.seed * 1000 + 3, device)
    d = cfg.d_in
    if cfg.x_kind == "lognormal_gauss":
        mult = torch.exp(cfg.x_sigma * torch.randn(d, generator=g, device=device))
    elif cfg.x_kind == "silu_gated":
        mult = torch.ones(d, device=device)
    else:
        raise ValueError(f"unknown x_kind {cfg.x_kind!r}")
    n_out = int(round(cfg.outlier_frac * d))
    if n_out > 0:
        idx = torch.randperm(d, generator=g, device=device)[:n_out]
        mult[idx] *= cfg.outlier_mult
    return mult.float()


def make_weight(cfg: LayerConfig, device="cpu", rows: Optional[Tuple[int, int]] = None
                ) -> torch.Tensor:
    """``W`` ``[d_out, d_in]`` ~ N(0, w_std^2) in ``cfg.w_dtype``."""
    g = _gen(cfg.seed * 1000 + 2, device)
    w = torch.randn(cfg.d_out, cfg.d_in, generator=g, device=device) * cfg.w_std
    if rows is not None:
        w = w[rows[0]:rows[1]]
    return w.to(cfg.w_dtype).contiguous()


def make_tokens_chunk(cfg: LayerConfig, index: int, device="cpu",
                      mult: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Token chunk ``index`` of the calibration stream, ``[t, d_in]`` in ``cfg.x_dtype``.

    Chunk ``index`` covers tokens ``[index*chunk, min((index+1)*chunk, n_tokens))``.
    """
    t0 = index * cfg.chunk
    t = min(cfg.chunk, cfg.n_tokens - t0)
    if t <= 0:
        raise IndexError(index)
    if mult is None:
        mult = channel_multipliers(cfg, device)
    g = _gen((cfg.seed * 1000 + 1) * 100003 + index, device)
    if cfg.x_kind == "lognormal_gauss":
        x = torch.randn(t, cfg.d_in, generator=g, device=device)
    else:
        a = torch.randn(t, cfg.d_in, generator=g, device=device)
        b = torch.randn(t, cfg.d_in, generator=g, device=device)
        x = torch.nn.functional.silu(a) * b
        del a, b
    x.mul_(mult.to(device)[None, :])
    return x.to(cfg.x_dtype)


def token_chunks(cfg: LayerConfig, device="cpu") -> Iterator[torch.Tensor]:
    """All chunks of the calibration stream in order."""
    mult = channel_multipliers(cfg, device)
    nchunks = (cfg.n_tokens + cfg.chunk - 1) // cfg.chunk
    for i in range(nchunks):
        yield make_tokens_chunk(cfg, i, device, mult)


def make_tokens(cfg: LayerConfig, device="cpu") -> torch.Tensor:
    """The whole calibration stream ``[n_tokens, d_in]`` (only for streams that fit)."""
    return torch.cat(list(token_chunks(cfg, device)), dim=0).contiguous()


def make_upper_factor(d: int, seed: int, device="cpu", offdiag: float = 0.5) -> torch.Tensor:
    """A random upper-triangular float32 ``[d, d]`` with a positive diagonal.

    Any such matrix is the inverse Cholesky factor of some positive-definite Hessian, so
    it is a valid, cheap-to-draw input for the column loop at sizes where the factor of
    a real Hessian is out of the CPU oracle's reach.  Diagonal: exp(0.3 N(0,1)); above
    it: row's diagonal x N(0,1) x offdiag / sqrt(d).
    """
    g = _gen(seed * 1000 + 7, device)
    diag = torch.exp(0.3 * torch.randn(d, generator=g, device=device))
    U = torch.randn(d, d, generator=g, device=device) * (offdiag / d ** 0.5)
    U = torch.triu(U, diagonal=1) * diag[:, None]
    U.diagonal().copy_(diag)
    return U.float().contiguous()


def make_permutation(d: int, seed: int, device="cpu") -> torch.Tensor:
    """A random permutation of ``range(d)`` (int32)."""
    g = _gen(seed * 1000 + 8, device)
    return torch.randperm(d, generator=g, device=device).to(torch.int32)
