"""Float64 CPU oracle for GPTQ layer quantization.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow reference that the CUDA path
is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import or call it; the product path never does.  It shares no code
with the CUDA library and imports nothing from it.

Everything is written in float64 with numpy, step by step in the order the pages give
the method.  Library routines serve only as steps (a matmul, a Cholesky factorisation, a
triangular solve).  Sources, by page:

* "Same Ruler, Smarter Placement: GPTQ" (techscribr), sections 1.4-1.11 and 2:
  H = 2XX^T, the OBS compensating update, damping, the Cholesky trick, lazy batches,
  act-order and the 4x4 worked example.
* "GPTQ Architecture, in depth" (aicassindra), "The algorithm in code" and "Groups,
  act-order and other knobs": the streaming Hessian hook, the dead-column fix, the
  asymmetric min-max group fit, the blocked column loop and the group index.
* "04 - GPTQ: Hessian-Weighted Rounding" (project-fortress), sections 2 and 8: the OBS
  loss w^2 / (2 [H^-1]_qq) and the packed checkpoint format.
* "GPTQ > ActOrder: Activation-Based Column Ordering" (mbrenndoerfer): the act-order
  permutation by descending Hessian diagonal.

Readings where the pages are silent or disagree:

* H is normalised as 2/n * sum(x x^T) (the streaming hook), not 2XX^T; every output but the
  loss is invariant to a positive scale of H because the damping is relative.
* Columns go front to back (after the optional permutation).
* Rounding is half-to-even (``np.rint``), as torch.round in the page's code.
* The symmetric grid has step max|w| / (2^(b-1) - 1) and signed codes in
  [-(2^(b-1)-1), 2^(b-1)-1], stored with the offset 2^(b-1) (the 4x4 example's
  max|w|/7 at 4 bits).
* ``group = -1`` is one group spanning the whole row, fitted before the first column.
* Static groups ("GPTQ Architecture, in depth", "Groups, act-order and other knobs": groups
  fixed in the original order before permuting): group G is original columns
  [G*g, (G+1)*g); its scale and zero are fitted once, before the loop, on W after the dead
  fix (no permutation, no compensation yet); processed column q uses the group of
  original column perm[q]; g_idx[c] = c // g.
* Act-order ties are broken by ascending original index (a stable sort).
* Wherever a float decides an integer (a code, a zero point), the decision is taken in
  float32, the precision of the page's code (``.float()``); the weights themselves evolve
  in float64.
* loss = sum over rows and columns of e^2 / 2 with e = (w - what) / u_qq, the OBS loss
  (w - what)^2 / (2 [H_cond^-1]_qq) with u_qq^2 = [H_cond^-1]_qq.
* Codes are packed as a little-endian bit stream along the packed axis: code k sits at
  bits [b*k, b*k + b) of the stream, word j holds stream bits [32j, 32j + 32).
"""

from __future__ import annotations

import math
from typing import Callable, Dict, Iterable, Optional, Tuple

import numpy as np

F32 = np.float32
F64 = np.float64

__all__ = [
    "hessian", "hessian_streaming", "hessian_block",
    "dead_columns", "fix_dead", "act_order", "damping", "inverse_cholesky_upper",
    "inverse_cholesky_upper_rows",
    "grid", "fit_group", "round_to_grid",
    "gptq_sweep", "gptq_sweep_obs",
    "gptq_prepare", "gptq_quantize_layer", "gptq_layer",
    "group_index", "static_group_fit", "pack_bitstream", "unpack_bitstream",
    "checkpoint_bytes", "dequantize", "dequant_matmul",
    "quadratic_loss", "rtn_quantize",
]


# --------------------------------------------------------------------------------------
# Hessian
# --------------------------------------------------------------------------------------

def hessian(X) -> np.ndarray:
    """H = (2/n) * sum_t x_t x_t^T for token-major X ``[n, d]``.

    "Same Ruler, Smarter Placement: GPTQ", section 1.4 (H = 2XX^T with X as
    ``[d, n]``), normalised by the token count as the streaming hook of "GPTQ
    Architecture, in depth", "The algorithm in code", does.
    """
    X = np.asarray(X, dtype=F64)
    n = X.shape[0]
    if n == 0:
        raise ValueError("no tokens")
    return (2.0 / n) * (X.T @ X)


def hessian_streaming(chunks: Iterable, H: Optional[np.ndarray] = None, n: int = 0
                      ) -> Tuple[np.ndarray, int]:
    """The Hessian hook's running update, one token chunk at a time.

    "GPTQ Architecture, in depth", "The algorithm in code" (HessianHook): for a chunk of
    t tokens, H <- H * n/(n+t); n <- n+t; x <- sqrt(2/n) x; H <- H + x^T x.
    """
    for Xc in chunks:
        Xc = np.asarray(Xc, dtype=F64)
        t = Xc.shape[0]
        if H is None:
            H = np.zeros((Xc.shape[1], Xc.shape[1]), dtype=F64)
        if t == 0:
            continue
        H = H * (n / (n + t))
        n = n + t
        xs = math.sqrt(2.0 / n) * Xc
        H = H + xs.T @ xs
    return H, n


def hessian_block(X, rows: slice, cols: slice, n: Optional[int] = None) -> np.ndarray:
    """One block H[rows, cols] = (2/n) X[:, rows]^T X[:, cols]; for sampling large H."""
    X = np.asarray(X)
    n = X.shape[0] if n is None else n
    a = np.asarray(X[:, rows], dtype=F64)
    b = np.asarray(X[:, cols], dtype=F64)
    return (2.0 / n) * (a.T @ b)


# --------------------------------------------------------------------------------------
# Preparation: dead columns, act-order, damping, inverse Cholesky factor
# --------------------------------------------------------------------------------------

def dead_columns(H) -> np.ndarray:
    """Input channels that never fired: diag(H) == 0 ("GPTQ Architecture, in depth",
    "The algorithm in code"; "Failure modes": channels that are always zero)."""
    return np.diag(np.asarray(H)) == 0


def fix_dead(H, W=None):
    """Set H_jj = 1 and W[:, j] = 0 for every dead channel j (same passage)."""
    H = np.array(H, dtype=F64, copy=True)
    dead = dead_columns(H)
    idx = np.nonzero(dead)[0]
    H[idx, idx] = 1.0
    if W is None:
        return H, dead
    W = np.array(W, dtype=F64, copy=True)
    W[:, dead] = 0.0
    return H, W, dead


def act_order(H) -> np.ndarray:
    """perm = argsort(diag(H), descending), ties by ascending index.

    "GPTQ > ActOrder: Activation-Based Column Ordering" (get_actorder_permutation);
    "Same Ruler, Smarter Placement: GPTQ", section 1.9.  ``perm[k]`` is the original
    column processed k-th.  A stable ascending sort of -diag keeps equal diagonals in
    index order.
    """
    diag = np.diag(np.asarray(H, dtype=F64))
    return np.argsort(-diag, kind="stable").astype(np.int64)


def damping(H, percdamp: float) -> Tuple[np.ndarray, float]:
    """H_damp = H + lambda I with lambda = percdamp * mean(diag H).

    "Same Ruler, Smarter Placement: GPTQ", section 1.6 (percdamp = 0.01).
    """
    H = np.asarray(H, dtype=F64)
    lam = float(percdamp) * float(np.mean(np.diag(H)))
    return H + lam * np.eye(H.shape[0]), lam


def inverse_cholesky_upper(Hd) -> np.ndarray:
    """Upper-triangular U with H_damp^-1 = U^T U, by the pages' four steps.

    "Same Ruler, Smarter Placement: GPTQ", section 1.7 ("In code, this is exactly four
    steps"): L = chol(H_damp); H^-1 = cholesky_inverse(L) = L^-T L^-1; U = chol(H^-1)
    taken as the upper factor.  Raises ``np.linalg.LinAlgError`` if H_damp is not
    positive definite.
    """
    Hd = np.asarray(Hd, dtype=F64)
    L = np.linalg.cholesky(Hd)                      # H_damp = L L^T, L lower
    Linv = _lower_inverse(L)                        # L^-1
    Hinv = Linv.T @ Linv                            # (L L^T)^-1
    Hinv = 0.5 * (Hinv + Hinv.T)                    # exact symmetry for the next factor
    Lh = np.linalg.cholesky(Hinv)                   # Hinv = Lh Lh^T
    return np.ascontiguousarray(Lh.T)               # U = Lh^T, Hinv = U^T U


def inverse_cholesky_upper_rows(Hd, rows) -> np.ndarray:
    """Rows ``rows`` of the same U, for matrices too large for the four steps on a CPU.

    Section 1.7 of "Same Ruler" shows that row q of U holds the conditional inverse at
    step q, i.e. it only depends on H_damp's trailing block from q on.  Ordering the
    columns backwards (J the index reversal) turns those trailing blocks into leading
    ones, so with Lr = chol(J H_damp J) (lower), U = J Lr^-1 J: row q of U is row
    d-1-q of Lr^-1 read backwards, the solution y of Lr^T y = e_(d-1-q).  One Cholesky
    factorisation and one triangular solve with the selected unit vectors; float64.
    """
    import scipy.linalg
    Hd = np.asarray(Hd, dtype=F64)
    d = Hd.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    Lr = np.linalg.cholesky(Hd[::-1, ::-1])          # J H_damp J = Lr Lr^T
    E = np.zeros((d, rows.size), dtype=F64)
    E[d - 1 - rows, np.arange(rows.size)] = 1.0
    Y = scipy.linalg.solve_triangular(Lr, E, trans="T", lower=True)   # Lr^T Y = E
    return np.ascontiguousarray(Y.T[:, ::-1])


def _lower_inverse(L: np.ndarray) -> np.ndarray:
    import scipy.linalg
    return scipy.linalg.solve_triangular(L, np.eye(L.shape[0]), lower=True)


# --------------------------------------------------------------------------------------
# Quantisation grid (decisions in float32)
# --------------------------------------------------------------------------------------

def grid(bits: int, sym: bool) -> Tuple[int, int, Optional[int]]:
    """(maxq, lowest code, fixed zero or None) of the b-bit unsigned code grid."""
    maxq = (1 << bits) - 1
    if sym:
        return maxq, 1, 1 << (bits - 1)
    return maxq, 0, None


def fit_group(wg: np.ndarray, bits: int, sym: bool,
              hint_zero: Optional[np.ndarray] = None, tie_eps: float = 1e-3,
              stats: Optional[dict] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Scale and zero point per row of the group ``wg`` ``[rows, g]`` (float64 values).

    Asymmetric ("GPTQ Architecture, in depth", fit_group): lo = min(min w, 0),
    hi = max(max w, 0), s = max((hi - lo)/maxq, 1e-8), z = round(-lo / s).
    Symmetric (reading of the 4x4 example, "Same Ruler", section 1.11):
    s = max(max|w| / (2^(b-1) - 1), 1e-8), z = 2^(b-1).
    The arithmetic is float32, the precision of the page's code.  Returns float32 scales
    and int64 zeros.  ``hint_zero`` may only move a zero whose pre-rounding value is within
    ``tie_eps`` of a rounding tie to the other neighbour.
    """
    maxq, _, zfix = grid(bits, sym)
    if sym:
        amax = np.max(np.abs(wg), axis=1).astype(F32)
        s = np.maximum(amax / F32((1 << (bits - 1)) - 1), F32(1e-8)).astype(F32)
        return s, np.full(s.shape, zfix, dtype=np.int64)
    lo = np.minimum(np.min(wg, axis=1), 0.0).astype(F32)
    hi = np.maximum(np.max(wg, axis=1), 0.0).astype(F32)
    s = np.maximum((hi - lo) / F32(maxq), F32(1e-8)).astype(F32)
    u = (-lo) / s                                   # float32 division
    z = _round_with_hint(u.astype(F64), hint_zero, tie_eps, stats, "zeros")
    return s, z


def _round_with_hint(u: np.ndarray, hint, tie_eps, stats, key) -> np.ndarray:
    """Half-to-even rounding; at a near-tie, the hinted neighbour wins."""
    r = np.rint(u)
    if hint is None:
        return r.astype(np.int64)
    hint = np.asarray(hint, dtype=F64)
    fl = np.floor(u)
    near = np.abs(u - (fl + 0.5)) < tie_eps
    take = near & (hint != r) & ((hint == fl) | (hint == fl + 1))
    if stats is not None:
        stats[key] = stats.get(key, 0) + int(np.count_nonzero(take))
    return np.where(take, hint, r).astype(np.int64)


def round_to_grid(w: np.ndarray, s: np.ndarray, z: np.ndarray, bits: int, sym: bool,
                  hint_code: Optional[np.ndarray] = None, tie_eps: float = 1e-3,
                  stats: Optional[dict] = None) -> Tuple[np.ndarray, np.ndarray]:
    """code = clamp(round(w / s) + z, lowest, maxq); what = s * (code - z).

    "GPTQ Architecture, in depth", "The algorithm in code".  w / s is a float32 division.
    Returns (codes int64, dequantised float64).
    """
    maxq, lowest, _ = grid(bits, sym)
    v = (w.astype(F32) / s).astype(F64)             # float32 division
    own = np.clip(np.rint(v) + z, lowest, maxq)
    if hint_code is not None:
        fl = np.floor(v)
        lo_c = np.clip(fl + z, lowest, maxq)
        hi_c = np.clip(fl + 1 + z, lowest, maxq)
        near = np.abs(v - (fl + 0.5)) < tie_eps
        hint = np.asarray(hint_code, dtype=F64)
        take = near & (hint != own) & ((hint == lo_c) | (hint == hi_c))
        if stats is not None:
            stats["codes"] = stats.get("codes", 0) + int(np.count_nonzero(take))
        own = np.where(take, hint, own)
    codes = own.astype(np.int64)
    what = s.astype(F64) * (codes - z).astype(F64)
    return codes, what


# --------------------------------------------------------------------------------------
# The column sweep
# --------------------------------------------------------------------------------------

def _group_span(q: int, group: int, d: int) -> Optional[Tuple[int, int]]:
    """Columns [q, q + g) to fit when column q starts a group, else None."""
    if group == -1:
        return (0, d) if q == 0 else None
    if q % group == 0:
        return (q, min(q + group, d))
    return None


def gptq_sweep(Wp, U, bits: int = 4, group: int = 128, sym: bool = False,
               blocksize: int = 128, hint: Optional[dict] = None,
               tie_eps: float = 1e-3, column_quantizer: Optional[Callable] = None,
               static: Optional[dict] = None) -> Dict[str, np.ndarray]:
    """The blocked fixed-order column loop with lazy batch updates.

    "GPTQ Architecture, in depth", "The algorithm in code" (the gptq loop) and
    "Same Ruler, Smarter Placement: GPTQ", sections 1.5 and 1.8.  ``Wp`` ``[m, d]`` are
    the weights already in processing order (dead columns zeroed, columns permuted);
    ``U`` is the upper factor with H_damp^-1 = U^T U in the same order.

    For each block [i1, i2): for each column q, fit (s, z) at a group start on the
    current W[:, q:q+g], quantise column q, e = (w_q - what_q) / u_qq, update the rest
    of the block W[:, q+1:i2] -= e u_q,q+1:i2, store e; after the block,
    W[:, i2:] -= Err U[i1:i2, i2:].

    ``blocksize >= d`` is the unblocked loop (every update applied at once to all later
    columns).  ``hint`` (``codes`` ``[m, d]`` in processing order and ``zeros``
    ``[G, m]``) resolves near-ties only; see ``round_to_grid``.
    ``column_quantizer(q, w_col) -> (codes, what)``, if given, replaces the per-row group
    grid (the 4x4 worked example of "Same Ruler", section 1.11, uses one symmetric scale
    per column); scales and zeros are then not recorded.
    ``static`` (``scales`` ``[G, m]``, ``zeros`` ``[G, m]``, ``gcol`` ``[d]``), if given,
    fixes the grids before the loop: column q uses group ``gcol[q]`` and nothing is fitted
    inside the loop (static groups).

    Returns codes ``[m, d]`` (processing order), scales ``[G, m]`` float32, zeros
    ``[G, m]``, loss_rows ``[m]`` (sum of e^2/2), Q ``[m, d]`` (dequantised, processing
    order) and ``stats`` (number of near-tie adoptions).
    """
    W = np.array(Wp, dtype=F64, copy=True)
    U = np.asarray(U, dtype=F64)
    m, d = W.shape
    G = 1 if group == -1 else -(-d // group)
    codes = np.zeros((m, d), dtype=np.int64)
    Q = np.zeros((m, d), dtype=F64)
    scales = np.zeros((G, m), dtype=F32)
    zeros = np.zeros((G, m), dtype=np.int64)
    loss = np.zeros(m, dtype=F64)
    stats: dict = {}
    s = z = None
    B = max(1, int(blocksize))
    for i1 in range(0, d, B):
        i2 = min(i1 + B, d)
        Err = np.zeros((m, i2 - i1), dtype=F64)
        for q in range(i1, i2):
            if column_quantizer is not None:
                c, what = column_quantizer(q, W[:, q].copy())
            elif static is not None:
                gi = int(static["gcol"][q])
                s, z = static["scales"][gi], static["zeros"][gi]
                hc = None if hint is None else hint["codes"][:, q]
                c, what = round_to_grid(W[:, q], s, z, bits, sym, hc, tie_eps, stats)
            else:
                span = _group_span(q, group, d)
                if span is not None:
                    gi = 0 if group == -1 else q // group
                    hz = None if hint is None else hint["zeros"][gi]
                    s, z = fit_group(W[:, span[0]:span[1]], bits, sym, hz, tie_eps, stats)
                    scales[gi], zeros[gi] = s, z
                hc = None if hint is None else hint["codes"][:, q]
                c, what = round_to_grid(W[:, q], s, z, bits, sym, hc, tie_eps, stats)
            codes[:, q] = c
            Q[:, q] = what
            e = (W[:, q] - what) / U[q, q]
            W[:, q + 1:i2] -= np.outer(e, U[q, q + 1:i2])
            Err[:, q - i1] = e
            loss += 0.5 * e * e
        if i2 < d:
            W[:, i2:] -= Err @ U[i1:i2, i2:]
    if static is not None:
        scales = np.asarray(static["scales"], dtype=F32).copy()
        zeros = np.asarray(static["zeros"], dtype=np.int64).copy()
    return dict(codes=codes, scales=scales, zeros=zeros, loss_rows=loss, Q=Q, stats=stats)


def gptq_sweep_obs(Wp, Hd, bits: int = 4, group: int = 128, sym: bool = False,
                   column_quantizer: Optional[Callable] = None) -> Dict[str, np.ndarray]:
    """The same fixed-order loop with explicit inverse-Hessian rows (OBQ style).

    "Same Ruler, Smarter Placement: GPTQ", sections 1.5 and 1.7: quantise column q,
    w_j -= (w_q - what_q) [H^-1]_qj / [H^-1]_qq for j > q, loss += (w_q - what_q)^2 /
    (2 [H^-1]_qq) ("04 - GPTQ", section 2, OBS loss), then replace H^-1 by its
    conditional inverse for the remaining columns, the Schur complement
    H^-1[q+1:, q+1:] - H^-1[q+1:, q] H^-1[q, q+1:] / H^-1_qq.  Unblocked; O(d^3).
    ``column_quantizer`` as in ``gptq_sweep``.
    """
    W = np.array(Wp, dtype=F64, copy=True)
    Hinv = np.linalg.inv(np.asarray(Hd, dtype=F64))
    m, d = W.shape
    G = 1 if group == -1 else -(-d // group)
    codes = np.zeros((m, d), dtype=np.int64)
    Q = np.zeros((m, d), dtype=F64)
    scales = np.zeros((G, m), dtype=F32)
    zeros = np.zeros((G, m), dtype=np.int64)
    loss = np.zeros(m, dtype=F64)
    s = z = None
    for q in range(d):
        if column_quantizer is not None:
            c, what = column_quantizer(q, W[:, q].copy())
        else:
            span = _group_span(q, group, d)
            if span is not None:
                gi = 0 if group == -1 else q // group
                s, z = fit_group(W[:, span[0]:span[1]], bits, sym)
                scales[gi], zeros[gi] = s, z
            c, what = round_to_grid(W[:, q], s, z, bits, sym)
        codes[:, q] = c
        Q[:, q] = what
        delta = W[:, q] - what
        hqq = Hinv[q, q]
        W[:, q + 1:] -= np.outer(delta / hqq, Hinv[q, q + 1:])
        loss += delta * delta / (2.0 * hqq)
        Hinv[q + 1:, q + 1:] -= np.outer(Hinv[q + 1:, q], Hinv[q, q + 1:]) / hqq
    return dict(codes=codes, scales=scales, zeros=zeros, loss_rows=loss, Q=Q)


# --------------------------------------------------------------------------------------
# Output format
# --------------------------------------------------------------------------------------

def group_index(perm: np.ndarray, group: int, static: bool = False) -> np.ndarray:
    """g_idx[c] = (position of original column c in the processing order) // g.

    "GPTQ Architecture, in depth", "Groups, act-order and other knobs": with act-order
    the groups follow the permuted order, so each original column records its group.
    With static groups the groups stay in the original order: g_idx[c] = c // g.
    ``group = -1`` puts every column in group 0.
    """
    perm = np.asarray(perm, dtype=np.int64)
    if static and group != -1:
        return (np.arange(perm.size) // group).astype(np.int32)
    pos = np.empty_like(perm)
    pos[perm] = np.arange(perm.size)
    if group == -1:
        return np.zeros(perm.size, dtype=np.int32)
    return (pos // group).astype(np.int32)


def static_group_fit(W0, group: int, bits: int, sym: bool, hint_zeros=None,
                     tie_eps: float = 1e-3, stats: Optional[dict] = None
                     ) -> Tuple[np.ndarray, np.ndarray]:
    """Scales and zeros ``[G, m]`` of the static groups: group G is the original columns
    [G*g, (G+1)*g) of ``W0`` (weights after the dead fix, original order, before any
    compensation), fitted once ("GPTQ Architecture, in depth", "Groups, act-order and
    other knobs": groups fixed in the original order before permuting)."""
    W0 = np.asarray(W0, dtype=F64)
    m, d = W0.shape
    if group == -1:
        spans = [(0, d)]
    else:
        spans = [(c, min(c + group, d)) for c in range(0, d, group)]
    scales = np.zeros((len(spans), m), dtype=F32)
    zeros = np.zeros((len(spans), m), dtype=np.int64)
    for gi, (a, b) in enumerate(spans):
        hz = None if hint_zeros is None else hint_zeros[gi]
        scales[gi], zeros[gi] = fit_group(W0[:, a:b], bits, sym, hz, tie_eps, stats)
    return scales, zeros


def pack_bitstream(values: np.ndarray, bits: int) -> np.ndarray:
    """Pack the last axis of non-negative ``values`` into int32 words.

    Value k of a row occupies bits [bits*k, bits*k + bits) of that row's little-endian
    bit stream; word j holds stream bits [32j, 32j + 32).  At 4 bits this is eight codes
    per int32 with code k in bits 4(k mod 8) ("04 - GPTQ", section 8: qweight holds
    eight INT4 values per int32).
    """
    values = np.asarray(values, dtype=np.int64)
    *lead, L = values.shape
    if (L * bits) % 32:
        raise ValueError("row length * bits must be a multiple of 32")
    if values.size and (values.min() < 0 or values.max() >= (1 << bits)):
        raise ValueError("value out of range")
    stream = ((values[..., :, None] >> np.arange(bits)) & 1).reshape(*lead, L * bits)
    stream = stream.reshape(*lead, (L * bits) // 32, 32).astype(np.uint64)
    words = (stream << np.arange(32, dtype=np.uint64)).sum(axis=-1)
    return words.astype(np.uint32).view(np.int32)


def unpack_bitstream(words: np.ndarray, bits: int, L: int) -> np.ndarray:
    """Inverse of ``pack_bitstream``: ``L`` values per row."""
    words = np.asarray(words).view(np.uint32).astype(np.int64)
    *lead, nw = words.shape
    stream = ((words[..., :, None] >> np.arange(32)) & 1).reshape(*lead, nw * 32)
    stream = stream[..., :L * bits].reshape(*lead, L, bits)
    return (stream << np.arange(bits)).sum(axis=-1)


def dequantize(qweight, scales, qzeros, g_idx, bits: int) -> np.ndarray:
    """The weights a packed checkpoint stands for, ``[d_out, d_in]`` float64.

    "GPTQ Architecture, in depth", "Packing, tooling and serving": a serving kernel
    unpacks each code and dequantises it with its group's scale and zero point; the group
    of original column c is g_idx[c]: w_hat[r, c] = s[g, r] * (code[r, c] - z[g, r]),
    g = g_idx[c] (the page's Q = scale * (q - zero)).  ``qweight`` ``[bits*d/32, m]`` and
    ``qzeros`` ``[G, bits*m/32]`` are little-endian bit streams as ``pack_bitstream``
    writes them.
    """
    qweight = np.asarray(qweight)
    m = qweight.shape[1]
    d = qweight.shape[0] * 32 // bits
    codes = unpack_bitstream(qweight.T, bits, d)                    # [m, d]
    zeros = unpack_bitstream(np.asarray(qzeros), bits, m)           # [G, m]
    g = np.asarray(g_idx, dtype=np.int64)
    s = np.asarray(scales, dtype=F64)[g].T                          # [m, d]
    z = zeros[g].T.astype(F64)
    return s * (codes.astype(F64) - z)


def dequant_matmul(x, qweight, scales, qzeros, g_idx, bits: int) -> np.ndarray:
    """y = x W_hat^T, ``x`` ``[n, d_in]``: the product a W4A16-style serving kernel computes
    from the packed checkpoint ("GPTQ Architecture, in depth", "Packing, tooling and
    serving"; "Same Ruler, Smarter Placement: GPTQ", section 1.5: the layer output the
    method preserves is W X)."""
    W = dequantize(qweight, scales, qzeros, g_idx, bits)
    return np.asarray(x, dtype=F64) @ W.T


def checkpoint_bytes(d_out: int, d_in: int, group: int) -> int:
    """Bytes of one W4 layer: qweight + fp16 scales + 4-bit zeros + int32 g_idx.

    "04 - GPTQ", section 8: out*in/2 + out*in/g*2 + out*in/(2g) + 4*in.
    """
    return (d_out * d_in // 2 + d_out * d_in // group * 2 + d_out * d_in // (2 * group)
            + 4 * d_in)


# --------------------------------------------------------------------------------------
# Stages mirroring the library's calls, and the whole layer
# --------------------------------------------------------------------------------------

def gptq_prepare(H, damp: float = 0.01, actorder: bool = True) -> Dict[str, np.ndarray]:
    """Dead fix, act-order, damping and the inverse Cholesky factor.

    "GPTQ Architecture, in depth", "The algorithm in code": dead = diag(H) == 0 with
    H_jj = 1; perm by descending diagonal (after the dead fix); H permuted on both axes;
    H += damp * mean(diag H) * I; U = upper Cholesky factor of H^-1.  Returns perm,
    dead, lam, the damped permuted H ``Hd`` and ``U``.
    """
    H = np.asarray(H, dtype=F64)
    H, dead = fix_dead(H)
    d = H.shape[0]
    perm = act_order(H) if actorder else np.arange(d, dtype=np.int64)
    Hp = H[np.ix_(perm, perm)]
    Hd, lam = damping(Hp, damp)
    U = inverse_cholesky_upper(Hd)
    return dict(perm=perm, dead=dead, lam=lam, Hd=Hd, U=U)


def gptq_quantize_layer(W, U, perm=None, dead=None, bits: int = 4, group: int = 128,
                        sym: bool = False, blocksize: int = 128,
                        rows: Optional[np.ndarray] = None, hint: Optional[dict] = None,
                        tie_eps: float = 1e-3, pack: bool = True,
                        static_groups: bool = False) -> Dict[str, np.ndarray]:
    """Quantise W given U and perm, and produce the packed checkpoint tensors.

    W ``[m, d]`` in original column order.  ``rows`` restricts the work to a subset of
    output rows (rows are independent given U: "GPTQ Architecture, in depth", "The
    algorithm on one page").  Codes come back in original column order (the un-permute,
    ``Q[:, argsort(perm)]``).  With ``pack`` (needs all rows): qweight
    ``[bits*d/32, m]`` packed along d, qzeros ``[G, bits*m/32]`` packed along m (only
    when both lengths fill whole words).  g_idx is always produced.  ``static_groups``
    fits the groups in the original column order before the loop (``static_group_fit``);
    scales and zeros then come in original group order.
    """
    W = np.array(W, dtype=F64, copy=True)
    m, d = W.shape
    if rows is not None:
        W = W[np.asarray(rows)]
    if dead is not None:
        W[:, np.asarray(dead, dtype=bool)] = 0.0
    perm = np.arange(d, dtype=np.int64) if perm is None else np.asarray(perm, np.int64)
    static = None
    if static_groups:
        st_stats: dict = {}
        sc, ze = static_group_fit(W, group, bits, sym,
                                  None if hint is None else hint["zeros"], tie_eps, st_stats)
        gcol = np.zeros(d, dtype=np.int64) if group == -1 else perm // group
        static = dict(scales=sc, zeros=ze, gcol=gcol)
    res = gptq_sweep(W[:, perm], U, bits, group, sym, blocksize, hint, tie_eps,
                     static=static)
    if static_groups and st_stats:
        for k, v in st_stats.items():
            res["stats"][k] = res["stats"].get(k, 0) + v
    codes = np.empty_like(res["codes"])
    codes[:, perm] = res["codes"]
    out = dict(res)
    out["codes_proc"] = res["codes"]
    out["codes"] = codes
    out["loss"] = float(np.sum(res["loss_rows"]))
    out["g_idx"] = group_index(perm, group, static_groups)
    if pack and rows is None and (d * bits) % 32 == 0 and (m * bits) % 32 == 0:
        out["qweight"] = pack_bitstream(codes, bits).T.copy()
        out["qzeros"] = pack_bitstream(res["zeros"], bits)
    return out


def gptq_layer(W, H, bits: int = 4, group: int = 128, sym: bool = False,
               actorder: bool = True, damp: float = 0.01, blocksize: int = 128,
               rows=None, static_groups: bool = False) -> Dict[str, np.ndarray]:
    """The whole per-layer method: prepare, then the column loop and packing."""
    prep = gptq_prepare(H, damp, actorder)
    out = gptq_quantize_layer(W, prep["U"], prep["perm"], prep["dead"], bits, group, sym,
                              blocksize, rows, static_groups=static_groups)
    out.update(perm=prep["perm"], dead=prep["dead"], lam=prep["lam"], U=prep["U"],
               Hd=prep["Hd"])
    return out


# --------------------------------------------------------------------------------------
# Loss measures and the round-to-nearest baseline
# --------------------------------------------------------------------------------------

def quadratic_loss(delta: np.ndarray, H: np.ndarray) -> np.ndarray:
    """Per row 1/2 delta^T H delta ("Same Ruler", section 1.5: the layer error is, up to
    constants, this quadratic in the row perturbation).  With the undamped H = 2/n XX^T
    it equals ||delta X||^2 / n."""
    delta = np.asarray(delta, dtype=F64)
    return 0.5 * np.einsum("ri,ij,rj->r", delta, np.asarray(H, dtype=F64), delta)


def babai_nearest_plane(C, t) -> np.ndarray:
    """Babai's nearest-plane algorithm for the closest vector problem: the integer
    coefficients z of the lattice point sum_j z_j c_j that it returns for the basis
    columns ``C`` ``[n, d]`` and the target ``t`` ``[n]``.

    "04 - GPTQ", section 4 (GPTQ as Babai's nearest-plane algorithm on the lattice the
    calibration Hessian defines).  With C = Q R (R upper triangular) and y = Q^T t, the
    coefficients are fixed from the last to the first: z_j is the integer nearest to
    (y_j - sum_{k>j} R_jk z_k) / R_jj, the hyperplane of the remaining sublattice that
    lies nearest the target.
    """
    C = np.asarray(C, dtype=F64)
    Qm, R = np.linalg.qr(C)
    y = Qm.T @ np.asarray(t, dtype=F64)
    d = C.shape[1]
    z = np.zeros(d, dtype=F64)
    for j in range(d - 1, -1, -1):
        z[j] = np.rint((y[j] - R[j, j + 1:] @ z[j + 1:]) / R[j, j])
    return z.astype(np.int64)


def gptq_babai(Wp, Hd, scales) -> np.ndarray:
    """GPTQ's codes on fixed, unclipped grids, computed as Babai's nearest plane
    ("04 - GPTQ", section 4: GPTQ run back to front is that algorithm).

    ``scales`` is ``[m]`` (one step per row) or ``[m, d]`` (a step per row and column,
    e.g. group-wise grids fixed before the loop).  Row r minimises
    (what - w_r)^T Hd (what - w_r) over what_j in s_rj Z.  With any B such that
    B^T B = Hd (here from the eigendecomposition, so nothing is shared with the Cholesky
    factor the column loop uses), the lattice has the basis vectors s_rj B[:, j] and the
    target is B w_r.  Babai's pass fixes the last basis vector first, so the
    columns are handed over in reverse order and the pass visits column 0 first, as the
    column loop does.  ``Wp`` ``[m, d]`` and ``Hd`` are in processing order; returns the
    codes ``[m, d]`` in that order.
    """
    W = np.asarray(Wp, dtype=F64)
    lam, V = np.linalg.eigh(np.asarray(Hd, dtype=F64))
    B = np.sqrt(lam)[:, None] * V.T
    s = np.asarray(scales, dtype=F64)
    if s.ndim == 1:
        s = np.repeat(s[:, None], W.shape[1], axis=1)
    codes = np.zeros(W.shape, dtype=np.int64)
    for r in range(W.shape[0]):
        codes[r] = babai_nearest_plane((B * s[r][None, :])[:, ::-1], B @ W[r])[::-1]
    return codes


def rtn_quantize(Wp, bits: int = 4, group: int = 128, sym: bool = False
                 ) -> Dict[str, np.ndarray]:
    """Round-to-nearest on the same groups, fitted on the uncompensated weights ("Same
    Ruler", section 2, the per-column RTN control; "GPTQ Architecture, in depth", "Why
    rounding to nearest breaks at 4 bits")."""
    W = np.asarray(Wp, dtype=F64)
    m, d = W.shape
    G = 1 if group == -1 else -(-d // group)
    Q = np.zeros_like(W)
    codes = np.zeros((m, d), dtype=np.int64)
    scales = np.zeros((G, m), dtype=F32)
    zeros = np.zeros((G, m), dtype=np.int64)
    for q in range(d):
        span = _group_span(q, group, d)
        if span is not None:
            s, z = fit_group(W[:, span[0]:span[1]], bits, sym)
            gi = 0 if group == -1 else q // group
            scales[gi], zeros[gi] = s, z
        codes[:, q], Q[:, q] = round_to_grid(W[:, q], s, z, bits, sym)
    return dict(codes=codes, Q=Q, scales=scales, zeros=zeros)
