"""Pins for the float64 oracle: page-printed values, closed forms, invariants, brute force.

Every pin is a function of the oracle module ``O`` so that ``test_oracle_mutations``
can run the same checks against copies of the oracle with a planted mistake and show
that each mistake is caught.
"""

import json
import os

import numpy as np
import pytest

from oracle import gptq_oracle as ORACLE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example_4x4.json")


def golden():
    with open(GOLDEN) as f:
        g = json.load(f)
    return {k: (np.array(v["value"], dtype=float) if isinstance(v, dict) else v)
            for k, v in g.items()}


def page_column_quantizer(seen=None):
    """The 4x4 example's grid: one symmetric scale per column, max|col| / 7, codes in
    [-7, 7] ("Same Ruler", section 1.11), in the page's (float64) hand arithmetic."""
    def q(col_idx, w):
        if seen is not None:
            seen[col_idx] = w.copy()
        delta = np.max(np.abs(w)) / 7.0
        c = np.rint(w / delta)
        return c.astype(np.int64), c * delta
    return q


def spd(rng, d, n=None):
    n = 4 * d if n is None else n
    X = rng.standard_normal((n, d)) * np.exp(rng.standard_normal(d))
    return 2.0 / n * X.T @ X, X


# ----------------------------------------------------------------------------- pins

def pin_worked_example(O):
    g = golden()
    W = g["W_columns"].T.copy()
    sX = g["s_X"]
    assert np.allclose(W @ sX, g["y_true"], atol=6e-4)
    for B in (1, 2, 4):
        seen = {}
        res = O.gptq_sweep(W, g["Hinv_2dp"], blocksize=B,
                           column_quantizer=page_column_quantizer(seen))
        assert np.array_equal(res["codes"].T, g["codes_per_column"]), B
        # the column each step sees, against W^(1), W^(2) and the adjusted column 3
        assert np.allclose(seen[1], g["W1"][:, 1], atol=1.5e-4)
        assert np.allclose(seen[2], g["W2"][:, 2], atol=1.5e-4)
        assert np.allclose(seen[3], [0.1084, -0.0696, 0.1023, 0.0066], atol=1.5e-4)
        assert np.allclose(res["Q"], g["W_hat_gptq"], atol=1.5e-4)
        yhat = res["Q"] @ sX
        assert np.allclose(yhat, g["y_hat_gptq"], atol=1.5e-3)
        loss = float(np.sum((yhat - W @ sX) ** 2))
        assert abs(loss - g["loss_gptq_text"]) < 1e-3


def pin_rtn_per_column():
    g = golden()
    W = g["W_columns"].T.copy()
    q = page_column_quantizer()
    Q = np.stack([q(j, W[:, j])[1] for j in range(4)], axis=1)
    yhat = Q @ g["s_X"]
    assert np.allclose(yhat, g["y_hat_rtn_col"], atol=1e-3)
    assert abs(np.sum((yhat - W @ g["s_X"]) ** 2) - g["loss_rtn_col"]) < 1e-3


def pin_conditioned_example(O):
    """True GPTQ on the printed H (conditioned inverse) differs from the page's
    illustration at one code only: column 3, row 2 becomes 6."""
    g = golden()
    W = g["W_columns"].T.copy()
    for Hd in (g["H"], O.damping(g["H"], 0.01)[0]):
        U = O.inverse_cholesky_upper(Hd)
        a = O.gptq_sweep(W, U, blocksize=4, column_quantizer=page_column_quantizer())
        b = O.gptq_sweep_obs(W, Hd, column_quantizer=page_column_quantizer())
        assert np.array_equal(a["codes"], b["codes"])
        assert np.allclose(a["loss_rows"], b["loss_rows"], rtol=1e-10, atol=1e-14)
        expect = g["codes_per_column"].T.copy()
        expect[2, 3] = 6
        assert np.array_equal(a["codes"], expect)


def pin_two_weight_closed_form(O):
    """d_in = 2: after quantising column 0, w1 moves by (w0 - what0) H01 / H11 and the
    column-0 loss is (w0 - what0)^2 / (2 [H^-1]_00) ("Same Ruler", section 1.5;
    "04 - GPTQ", section 2); column 1 then has conditional inverse 1 / H11."""
    rng = np.random.default_rng(7)
    for _ in range(20):
        H, _ = spd(rng, 2)
        W = rng.standard_normal((5, 2)) * 0.3
        delta = 0.05

        def quant(q, w):
            c = np.rint(w / delta)
            return c.astype(np.int64), c * delta

        seen = {}

        def rec(q, w):
            seen[q] = w.copy()
            return quant(q, w)

        for res in (O.gptq_sweep(W, O.inverse_cholesky_upper(H), blocksize=1,
                                 column_quantizer=rec),
                    O.gptq_sweep_obs(W, H, column_quantizer=rec)):
            e0 = W[:, 0] - np.rint(W[:, 0] / delta) * delta
            w1 = W[:, 1] + e0 * H[0, 1] / H[1, 1]
            assert np.allclose(seen[1], w1, rtol=1e-12, atol=1e-14)
            hinv00 = H[1, 1] / (H[0, 0] * H[1, 1] - H[0, 1] ** 2)
            e1 = w1 - np.rint(w1 / delta) * delta
            loss = e0 ** 2 / (2 * hinv00) + e1 ** 2 * H[1, 1] / 2
            assert np.allclose(res["loss_rows"], loss, rtol=1e-10, atol=1e-16)


def pin_cholesky_2x2(O):
    """U for a 2x2 H^-1 = [[a, b], [b, c]]: u00 = sqrt(a), u01 = b / sqrt(a),
    u11 = sqrt(c - b^2 / a) ("Same Ruler", section 1.7)."""
    rng = np.random.default_rng(3)
    for _ in range(10):
        H, _ = spd(rng, 2)
        Hinv = np.linalg.inv(H)
        a, b, c = Hinv[0, 0], Hinv[0, 1], Hinv[1, 1]
        U = O.inverse_cholesky_upper(H)
        assert np.allclose(U, [[np.sqrt(a), b / np.sqrt(a)], [0.0, np.sqrt(c - b * b / a)]],
                           rtol=1e-12)


def pin_cholesky_general(O):
    """Row q of U carries the conditional inverse at step q: u_qq^2 = [H_c^-1]_qq and
    u_qj / u_qq = [H_c^-1]_qj / [H_c^-1]_qq ("Same Ruler", section 1.7, 'The general
    pattern'); U agrees with the reversed-order Cholesky route U = J chol(J H J)^-1 J."""
    rng = np.random.default_rng(11)
    d = 24
    H, _ = spd(rng, d)
    Hd, _ = O.damping(H, 0.01)
    U = O.inverse_cholesky_upper(Hd)
    assert np.allclose(np.tril(U, -1), 0)
    assert np.all(np.diag(U) > 0)
    assert np.allclose(U.T @ U @ Hd, np.eye(d), atol=1e-10)
    Hc = np.linalg.inv(Hd)
    for q in range(d):
        assert np.isclose(U[q, q] ** 2, Hc[0, 0], rtol=1e-10)
        assert np.allclose(U[q, q + 1:] / U[q, q], Hc[0, 1:] / Hc[0, 0], rtol=1e-9, atol=1e-12)
        Hc = Hc[1:, 1:] - np.outer(Hc[1:, 0], Hc[0, 1:]) / Hc[0, 0]
    J = np.eye(d)[::-1]
    Lr = np.linalg.cholesky(J @ Hd @ J)
    assert np.allclose(J @ np.linalg.inv(Lr) @ J, U, rtol=1e-9, atol=1e-12)
    # selected rows through the reversed factor and one triangular solve: the same rows
    for rows in ([0], [d - 1], [0, 5, 11, d - 1], list(range(d))):
        assert np.allclose(O.inverse_cholesky_upper_rows(Hd, rows), U[rows], rtol=1e-9,
                           atol=1e-12), rows


def _small_layer(rng, m, d, n=None):
    H, X = spd(rng, d, n)
    W = rng.standard_normal((m, d)) * 0.02
    return W, H, X


def pin_obs_equals_cholesky(O):
    """The OBQ-style explicit-inverse loop and the Cholesky-row loop agree."""
    rng = np.random.default_rng(5)
    for bits, group, sym in [(4, -1, False), (3, 4, False), (4, 8, True), (2, 4, True)]:
        W, H, _ = _small_layer(rng, 6, 16)
        Hd, _ = O.damping(H, 0.01)
        U = O.inverse_cholesky_upper(Hd)
        a = O.gptq_sweep(W, U, bits, group, sym, blocksize=10 ** 9)
        b = O.gptq_sweep_obs(W, Hd, bits, group, sym)
        assert np.array_equal(a["codes"], b["codes"])
        assert np.allclose(a["loss_rows"], b["loss_rows"], rtol=1e-10)
        assert np.allclose(a["scales"], b["scales"], rtol=1e-6)


def pin_blocked_equals_unblocked(O):
    """Lazy batching changes only when updates are applied ("Same Ruler", section 1.8)."""
    rng = np.random.default_rng(9)
    for bits, group, sym in [(4, -1, False), (4, 8, False), (3, 4, True), (4, 16, False)]:
        W, H, _ = _small_layer(rng, 7, 48)
        U = O.inverse_cholesky_upper(O.damping(H, 0.01)[0])
        ref = O.gptq_sweep(W, U, bits, group, sym, blocksize=10 ** 9)
        for B in (1, 4, 8, 16, 128):
            if group != -1 and group % B and B % group:
                continue
            r = O.gptq_sweep(W, U, bits, group, sym, blocksize=B)
            assert np.array_equal(r["codes"], ref["codes"]), (B, group)
            assert np.allclose(r["loss_rows"], ref["loss_rows"], rtol=1e-10)
            assert np.array_equal(r["zeros"], ref["zeros"])


def pin_loss_identity(O):
    """sum e^2/2 over a row equals 1/2 delta^T H_damp delta with delta = what - w."""
    rng = np.random.default_rng(13)
    for bits, group, sym in [(4, 8, False), (3, -1, True)]:
        W, H, _ = _small_layer(rng, 5, 32)
        Hd, _ = O.damping(H, 0.01)
        r = O.gptq_sweep(W, O.inverse_cholesky_upper(Hd), bits, group, sym, blocksize=8)
        assert np.allclose(r["loss_rows"], O.quadratic_loss(r["Q"] - W, Hd), rtol=1e-9)


def pin_brute_force_optimum(O):
    """d_in <= 6: the exhaustive minimum of the layer loss ||W X - What X||^2 over every
    assignment on GPTQ's own grid is never above GPTQ's loss."""
    rng = np.random.default_rng(17)
    d, bits = 5, 3
    maxq = (1 << bits) - 1
    grid_codes = np.stack(np.meshgrid(*[np.arange(maxq + 1)] * d, indexing="ij"), -1)
    grid_codes = grid_codes.reshape(-1, d)
    for trial in range(6):
        W, H, X = _small_layer(rng, 3, d, n=12)
        r = O.gptq_layer(W, H, bits=bits, group=-1, sym=False, actorder=bool(trial % 2),
                         damp=0.01, blocksize=128)
        for row in range(W.shape[0]):
            s = float(r["scales"][0, row])
            z = int(r["zeros"][0, row])
            cand = s * (grid_codes - z)                       # all grid points, [N, d]
            err = cand - W[row][None, :]
            layer = np.sum((err @ X.T) ** 2, axis=1)          # ||(what - w) X^T||^2
            mine = float(np.sum(((((r["codes"][row] - z) * s) - W[row]) @ X.T) ** 2))
            assert layer.min() <= mine * (1 + 1e-12) + 1e-18


def pin_gptq_beats_rtn_on_average(O):
    """Over 200 seeds, GPTQ's mean layer loss is below round-to-nearest on the same
    groups ("Same Ruler", section 2; spec: RTN never better on average)."""
    g_loss, r_loss = [], []
    for seed in range(200):
        rng = np.random.default_rng(1000 + seed)
        W, H, X = _small_layer(rng, 4, 16, n=40)
        r = O.gptq_layer(W, H, bits=3, group=8, sym=False, actorder=True, damp=0.01)
        perm = r["perm"]
        rt = O.rtn_quantize(W[:, perm], bits=3, group=8)
        Qr = np.empty_like(W)
        Qr[:, perm] = rt["Q"]
        Qg = np.empty_like(W)
        Qg[:, perm] = r["Q"]
        g_loss.append(np.sum(O.quadratic_loss(Qg - W, H)))
        r_loss.append(np.sum(O.quadratic_loss(Qr - W, H)))
    assert np.mean(g_loss) < np.mean(r_loss)


def pin_act_order(O):
    """perm sorts diag(H) descending ("GPTQ > ActOrder"); ties keep index order."""
    rng = np.random.default_rng(19)
    H, _ = spd(rng, 30)
    perm = O.act_order(H)
    dg = np.diag(H)[perm]
    assert np.all(np.diff(dg) <= 0)
    assert sorted(perm.tolist()) == list(range(30))
    Ht = np.diag([1.0, 3.0, 1.0, 3.0, 2.0, 1.0])
    assert O.act_order(Ht).tolist() == [1, 3, 4, 0, 2, 5]
    prep = O.gptq_prepare(Ht, 0.01, actorder=True)
    assert np.all(np.diff(np.diag(prep["Hd"])) <= 0)


def pin_damping(O):
    """Every eigenvalue moves up by lambda = 0.01 mean(diag H) and each diagonal entry
    of H_damp^-1 is at most 1 / lambda ("Same Ruler", section 1.6)."""
    rng = np.random.default_rng(23)
    H, _ = spd(rng, 20, n=8)           # rank-deficient: n < d
    Hd, lam = O.damping(H, 0.01)
    assert np.isclose(lam, 0.01 * np.trace(H) / 20)
    assert np.allclose(np.linalg.eigvalsh(Hd), np.linalg.eigvalsh(H) + lam, atol=1e-10)
    assert np.all(np.diag(np.linalg.inv(Hd)) <= 1.0 / lam * (1 + 1e-12))


def pin_dead_columns(O):
    rng = np.random.default_rng(29)
    X = rng.standard_normal((50, 6))
    X[:, 2] = 0.0
    H = O.hessian(X)
    W = rng.standard_normal((3, 6))
    Hf, Wf, dead = O.fix_dead(H, W)
    assert dead.tolist() == [False, False, True, False, False, False]
    assert Hf[2, 2] == 1.0 and np.all(Wf[:, 2] == 0.0)
    assert np.allclose(np.delete(np.delete(Hf, 2, 0), 2, 1), np.delete(np.delete(H, 2, 0), 2, 1))
    r = O.gptq_layer(W, H, bits=4, group=-1, actorder=True)
    assert r["dead"][2] and np.isfinite(r["loss"])


def pin_hessian(O):
    rng = np.random.default_rng(31)
    X = rng.standard_normal((7, 4))
    brute = np.zeros((4, 4))
    for t in range(7):
        for i in range(4):
            for j in range(4):
                brute[i, j] += 2.0 / 7 * X[t, i] * X[t, j]
    assert np.allclose(O.hessian(X), brute, rtol=1e-14)
    X = rng.standard_normal((300, 9))
    Hs, n = O.hessian_streaming([X[:100], X[100:101], X[101:250], X[250:]])
    assert n == 300 and np.allclose(Hs, O.hessian(X), rtol=1e-12)
    assert np.allclose(np.diag(O.hessian(X)), 2.0 / 300 * np.sum(X * X, axis=0), rtol=1e-13)
    assert np.allclose(O.hessian_block(X, slice(2, 5), slice(4, 9)), O.hessian(X)[2:5, 4:9])


def pin_fit_and_round(O):
    # asymmetric, 4 bits: lo=-1, hi=2, s=3/15=0.2, z=round(5)=5
    s, z = O.fit_group(np.array([[-1.0, 0.5, 2.0]]), 4, False)
    assert np.isclose(s[0], np.float32(0.2)) and z[0] == 5
    # -lo/s = 0.9 / (2.9/15) = 4.655 rounds to 5
    s, z = O.fit_group(np.array([[-0.9, 2.0, 0.1]]), 4, False)
    assert np.isclose(s[0], np.float32(2.9 / 15)) and z[0] == 5
    # all positive: lo clamps to 0 so z = 0
    s, z = O.fit_group(np.array([[0.5, 1.5]]), 4, False)
    assert np.isclose(s[0], np.float32(0.1)) and z[0] == 0
    # all-zero group: s = 1e-8, z = 0
    s, z = O.fit_group(np.zeros((1, 4)), 4, False)
    assert s[0] == np.float32(1e-8) and z[0] == 0
    # symmetric, 4 bits: s = max|w| / 7, zero 8
    s, z = O.fit_group(np.array([[-0.7, 0.35]]), 4, True)
    assert np.isclose(s[0], np.float32(0.1)) and z[0] == 8
    # rounding: half to even, clamp to the grid
    c, q = O.round_to_grid(np.array([0.25, 0.35, 10.0, -10.0]), np.float32([0.1] * 4),
                           np.array([0, 0, 0, 0]), 4, False)
    assert c.tolist() == [2, 4, 15, 0]
    c, q = O.round_to_grid(np.array([-10.0, 10.0]), np.float32([0.1] * 2),
                           np.array([8, 8]), 4, True)
    assert c.tolist() == [1, 15]


def pin_replay_hint(O):
    """The replay rule that lets a GPU code or zero differ from the oracle's own choice:
    a hint is adopted only where the float32 pre-rounding value lies within tie_eps of a
    rounding tie, and only for the other of the two neighbouring grid points (inside the
    clamped grid).  Everything else keeps the oracle's own rounding (half to even)."""
    s = np.float32([0.1])
    z = np.array([0])

    def code(w, hint, stats=None):
        c, _ = O.round_to_grid(np.array([w]), s, z, 4, False, np.array([hint]), 1e-3, stats)
        return int(c[0])

    # w / s = 2.5 exactly in float32: half to even gives 2; the hint 3 is the other
    # neighbour of the tie, so it is adopted and counted
    assert abs(float(np.float32(0.25) / s[0]) - 2.5) < 1e-3
    st = {}
    assert code(0.25, 3, st) == 3 and st.get("codes") == 1
    # the same hint just outside the band (|v - 2.5| = 2e-3 >= 1e-3) is refused
    st = {}
    assert code(0.2502, 2, st) == 3 and code(0.2498, 3, st) == 2 and st.get("codes", 0) == 0
    # a hint two levels away (or on the far side) is refused even at an exact tie
    st = {}
    assert code(0.25, 4, st) == 2 and code(0.25, 1, st) == 2 and code(0.25, 0, st) == 2
    assert st.get("codes", 0) == 0
    # a hint equal to the oracle's own code changes nothing and is not counted
    st = {}
    assert code(0.25, 2, st) == 2 and st.get("codes", 0) == 0
    # a hint outside the clamped grid is refused: at v = 15.5 both neighbours clamp to 15,
    # at v = -0.5 both clamp to 0
    st = {}
    assert code(1.55, 16, st) == 15 and code(-0.05, -1, st) == 0 and st.get("codes", 0) == 0
    # a code decided on the hint keeps its dequantised value consistent: what = s (c - z)
    c, what = O.round_to_grid(np.array([0.25]), s, z, 4, False, np.array([3]), 1e-3, {})
    assert c[0] == 3 and what[0] == np.float64(s[0]) * 3

    # zero points: -lo / s = 2.5 for lo = -0.25, hi = 1.25 (s = 1.5 / 15 = 0.1)
    def zero(wg, hint, stats=None):
        _, zz = O.fit_group(np.array([wg]), 4, False, np.array([hint]), 1e-3, stats)
        return int(zz[0])

    st = {}
    assert zero([-0.25, 1.25], 3, st) == 3 and st.get("zeros") == 1
    st = {}
    assert zero([-0.25, 1.25], 2, st) == 2 and st.get("zeros", 0) == 0
    # off the band: -lo / s = 2.6 rounds to 3, the hint 2 is refused
    st = {}
    assert zero([-0.26, 1.24], 2, st) == 3 and st.get("zeros", 0) == 0
    # two levels away at the tie: refused
    st = {}
    assert zero([-0.25, 1.25], 4, st) == 2 and zero([-0.25, 1.25], 0, st) == 2
    assert st.get("zeros", 0) == 0
    # no hint: plain half-to-even rounding
    _, zz = O.fit_group(np.array([[-0.25, 1.25]]), 4, False)
    assert int(zz[0]) == 2


def pin_pack(O):
    codes = np.arange(1, 9)[None, :]
    w = O.pack_bitstream(codes, 4)
    assert w.view(np.uint32)[0, 0] == 0x87654321
    # 3 bits: 32 codes in 3 words, code 10 straddles words 0 and 1
    codes = np.zeros((1, 32), dtype=np.int64)
    codes[0, 10] = 0b111
    w = O.pack_bitstream(codes, 3).view(np.uint32)
    assert w[0, 0] == 0b11 << 30 and w[0, 1] == 0b1 and w[0, 2] == 0
    assert O.pack_bitstream(np.array([[0x12, 0x34, 0x56, 0x78]]), 8).view(np.uint32)[0, 0] \
        == 0x78563412
    rng = np.random.default_rng(37)
    for bits in (2, 3, 4, 8):
        v = rng.integers(0, 1 << bits, size=(5, 64))
        assert np.array_equal(O.unpack_bitstream(O.pack_bitstream(v, bits), bits, 64), v)


def pin_checkpoint_format(O):
    """"04 - GPTQ", section 8: 4096x4096 at g128 is out*in/2 + out*in/g*2 + out*in/(2g)
    + 4*in = 8,732,672 bytes; the tensors the oracle packs have exactly these sizes."""
    assert O.checkpoint_bytes(4096, 4096, 128) == 8732672
    # "GPTQ Architecture, in depth", worked example: 4 + (16 + 4)/128 bits per weight
    assert np.isclose((O.checkpoint_bytes(4096, 4096, 128) - 4 * 4096) * 8 / 4096 ** 2,
                      4 + 20 / 128)
    rng = np.random.default_rng(41)
    m, d, g = 32, 256, 128
    W, H, _ = _small_layer(rng, m, d)
    r = O.gptq_layer(W, H, bits=4, group=g, actorder=True)
    nbytes = (r["qweight"].nbytes + r["scales"].astype(np.float16).nbytes
              + r["qzeros"].nbytes + r["g_idx"].nbytes)
    assert r["qweight"].shape == (d // 8, m) and r["qzeros"].shape == (d // g, m // 8)
    assert nbytes == O.checkpoint_bytes(m, d, g)


def pin_format_roundtrip(O):
    """qweight/qzeros/scales/g_idx dequantise to the loop's Q, un-permuted
    ("GPTQ Architecture, in depth": Q[:, argsort(perm)], g_idx per original column)."""
    rng = np.random.default_rng(43)
    m, d = 32, 64
    for bits, group, sym in [(4, 16, False), (3, 32, True), (4, -1, False)]:
        W, H, _ = _small_layer(rng, m, d)
        r = O.gptq_layer(W, H, bits=bits, group=group, sym=sym, actorder=True, blocksize=16)
        codes = O.unpack_bitstream(r["qweight"].T.copy(), bits, d)
        zeros = O.unpack_bitstream(r["qzeros"], bits, m)
        gi = r["g_idx"]
        deq = r["scales"][gi].T.astype(float) * (codes - zeros[gi].T)
        Q = np.empty_like(W)
        Q[:, r["perm"]] = r["Q"]
        assert np.allclose(deq, Q, rtol=0, atol=1e-15)
        assert np.array_equal(codes, r["codes"])


def pin_static_groups(O):
    """Static groups ("GPTQ Architecture, in depth", "Groups, act-order and other knobs":
    groups fixed in the original order before permuting).

    * With a diagonal H the factor U is diagonal, so no error reaches a later column and
      GPTQ with grids fixed before the loop is round-to-nearest on those grids: the codes
      in original column order equal RTN on the original order (act-order on, so a
      column read through the wrong group would show), and differ from dynamic groups.
    * With one group per row the fit sees every column of the row before any update in
      both modes, so static equals dynamic exactly.
    * With a general H the static scales and zeros are the RTN fit of the original,
      uncompensated weights; g_idx[c] = c // g; blocking does not change the result.
    """
    rng = np.random.default_rng(41)
    m, d, g = 5, 32, 8
    for bits, sym in [(4, False), (3, True)]:
        W = rng.standard_normal((m, d)) * 0.02 * np.exp(rng.standard_normal(d))
        H = np.diag(np.exp(rng.standard_normal(d)))
        st = O.gptq_layer(W, H, bits, g, sym, actorder=True, static_groups=True)
        assert not np.array_equal(st["perm"], np.arange(d))
        rtn = O.rtn_quantize(W, bits, g, sym)
        assert np.array_equal(st["codes"], rtn["codes"])
        assert np.array_equal(st["scales"], rtn["scales"])
        assert np.array_equal(st["zeros"], rtn["zeros"])
        dyn = O.gptq_layer(W, H, bits, g, sym, actorder=True)
        assert not np.array_equal(dyn["codes"], st["codes"])
    for bits, sym in [(4, False), (3, True)]:
        W, H, _ = _small_layer(rng, 6, 24)
        a = O.gptq_layer(W, H, bits, -1, sym, actorder=True, static_groups=True)
        b = O.gptq_layer(W, H, bits, -1, sym, actorder=True)
        assert np.array_equal(a["codes"], b["codes"])
        assert np.array_equal(a["scales"], b["scales"]) and np.array_equal(a["zeros"], b["zeros"])
        assert a["loss"] == b["loss"]
        assert np.array_equal(a["g_idx"], b["g_idx"])
    W, H, _ = _small_layer(rng, 6, 48)
    H[7, :] = 0.0
    H[:, 7] = 0.0                                   # a dead channel
    st = O.gptq_layer(W, H, 4, g, False, actorder=True, static_groups=True)
    W0 = W.copy()
    W0[:, 7] = 0.0
    rtn = O.rtn_quantize(W0, 4, g, False)
    assert np.array_equal(st["scales"], rtn["scales"]) and np.array_equal(st["zeros"], rtn["zeros"])
    assert np.array_equal(st["g_idx"], np.arange(48) // g)
    prep = O.gptq_prepare(H, 0.01, True)
    ref = O.gptq_quantize_layer(W, prep["U"], prep["perm"], prep["dead"], 4, g, False,
                                blocksize=10 ** 9, static_groups=True)
    for B in (1, 8, 16):
        r = O.gptq_quantize_layer(W, prep["U"], prep["perm"], prep["dead"], 4, g, False,
                                  blocksize=B, static_groups=True)
        assert np.array_equal(r["codes"], ref["codes"]), B
        assert np.allclose(r["loss_rows"], ref["loss_rows"], rtol=1e-10)


def pin_dequantize(O):
    """Unpacking the checkpoint reproduces the quantizer's own dequantised weights.

    The column loop keeps what = s (code - z) for every weight (Q, processing order);
    ``dequantize`` rebuilds it from qweight / scales / qzeros / g_idx alone, so the two
    agree exactly (in original column order) for dynamic and static groups, every width
    and act-order on; ``dequant_matmul`` is x times that matrix transposed.
    """
    rng = np.random.default_rng(43)
    m, d = 32, 64
    for bits, group, sym, static in [(4, 16, False, False), (3, 32, True, False),
                                     (2, 16, False, True), (8, -1, False, False),
                                     (4, 32, True, True)]:
        W, H, _ = _small_layer(rng, m, d)
        out = O.gptq_layer(W, H, bits, group, sym, actorder=True, static_groups=static)
        Qo = np.empty_like(out["Q"])
        Qo[:, out["perm"]] = out["Q"]
        Wh = O.dequantize(out["qweight"], out["scales"], out["qzeros"], out["g_idx"], bits)
        assert np.array_equal(Wh, Qo), (bits, group, sym, static)
        x = rng.standard_normal((3, d))
        y = O.dequant_matmul(x, out["qweight"], out["scales"], out["qzeros"], out["g_idx"],
                             bits)
        assert np.allclose(y, x @ Qo.T, rtol=1e-13, atol=0)


def pin_block_pipeline(O):
    """The block oracle ("GPTQ Architecture, in depth", "The pipeline, block by block"):
    zero weights make the block the identity (both residual branches vanish); with one
    token the causal softmax has a single term, so attention returns v itself; rmsnorm
    of a constant row is all ones; at 8 bits the quantised block stays close to the
    original one; and a pipeline step feeds its re-forward output to the next block."""
    from oracle import pipeline_oracle as P
    rng = np.random.default_rng(47)
    B, S, h, f, heads = 2, 8, 32, 64, 4
    x = rng.standard_normal((B, S, h))
    zero = {k: np.zeros((f if k in ("wg", "wu") else h, f if k == "wd" else h))
            for k in ("wq", "wk", "wv", "wo", "wg", "wu", "wd")}
    y, _ = P.block_forward(x, zero, heads)
    assert np.array_equal(y, x)
    q, k, v = (rng.standard_normal((B, 1, h)) for _ in range(3))
    assert np.allclose(P.attention(q, k, v, heads), v, rtol=0, atol=1e-15)
    assert np.allclose(P.rmsnorm(np.full((3, h), 2.5)), 1.0, rtol=1e-6)
    W = {k: rng.standard_normal(zero[k].shape) * 0.05 for k in zero}
    st = P.quantize_block(x, W, heads, bits=8, group=32)
    y_ref, inputs = P.block_forward(x, W, heads)
    assert np.linalg.norm(st["y"] - y_ref) <= 1e-2 * np.linalg.norm(y_ref)
    assert set(st["H"]) == {"qkv", "o", "gateup", "down"}
    assert np.allclose(st["H"]["qkv"], O.hessian(inputs["qkv"]))
    steps = P.pipeline(x, [W, W], heads, bits=4, group=32)
    assert np.array_equal(steps[1]["inputs"]["qkv"], P.rmsnorm(steps[0]["y"]).reshape(B * S, h))
    # grouped-query attention is multi-head attention whose key / value heads are repeated:
    # with k and v weights of 2 heads (16 rows), expanding each head's rows to its query
    # heads gives the same block
    kvh = 2
    hd = h // heads
    Wg = dict(W, wk=W["wk"][:kvh * hd], wv=W["wv"][:kvh * hd])
    expand = lambda w: np.concatenate([np.tile(w[j * hd:(j + 1) * hd], (heads // kvh, 1))
                                       for j in range(kvh)])
    Wm = dict(W, wk=expand(Wg["wk"]), wv=expand(Wg["wv"]))
    yg, ig = P.block_forward(x, Wg, heads, kvh)
    ym, im = P.block_forward(x, Wm, heads)
    assert np.allclose(yg, ym, rtol=1e-12, atol=1e-14)
    assert np.allclose(ig["o"], im["o"], rtol=1e-12, atol=1e-14)


def unclipped_grid(s):
    """Fixed grids without clipping (the lattice of the Babai view): s ``[m]`` per row,
    or ``[m, d]`` per row and column."""
    def q(col_idx, w):
        sc = s if s.ndim == 1 else s[:, col_idx]
        c = np.rint(w / sc)
        return c.astype(np.int64), c * sc
    return q


def pin_babai(O):
    """Babai's nearest plane ("04 - GPTQ", section 4).  On an orthogonal basis it rounds
    each coordinate, which solves the closest vector problem exactly (brute force over a
    box); GPTQ without clipping returns exactly its codes on random Hessians, blocked or
    not; and each row's loss stays within the bound that rounding gives,
    sum_q (s/2)^2 / (2 U_qq^2)."""
    rng = np.random.default_rng(23)
    for _ in range(5):
        d = 4
        Qb, _ = np.linalg.qr(rng.standard_normal((d, d)))
        lens = np.exp(rng.standard_normal(d))
        C = Qb * lens                                    # orthogonal columns
        t = rng.standard_normal(d) * 3.0
        z = O.babai_nearest_plane(C, t)
        assert np.array_equal(z, np.rint(Qb.T @ t / lens).astype(np.int64))
        box = np.stack(np.meshgrid(*[np.arange(-2, 3)] * d, indexing="ij"), -1)
        box = box.reshape(-1, d) + z
        dist = np.sum((box @ C.T - t) ** 2, axis=1)
        assert np.sum((C @ z - t) ** 2) <= dist.min() * (1 + 1e-12) + 1e-15
    for d, B in [(16, 10 ** 9), (24, 8), (40, 16), (32, 1)]:
        H, _ = spd(rng, d)
        Hd, _ = O.damping(H, 0.01)
        U = O.inverse_cholesky_upper(Hd)
        W = rng.standard_normal((4, d)) * 0.02
        s = np.abs(W).max(axis=1) / 7.0
        r = O.gptq_sweep(W, U, blocksize=B, column_quantizer=unclipped_grid(s))
        assert np.array_equal(O.gptq_babai(W, Hd, s), r["codes"]), (d, B)
        bound = 0.5 * (s / 2.0) ** 2 * np.sum(1.0 / np.diag(U) ** 2)
        assert np.all(r["loss_rows"] <= bound * (1 + 1e-12))
        assert np.allclose(r["loss_rows"], O.quadratic_loss(r["Q"] - W, Hd), rtol=1e-9)
    # group-wise steps fixed before the loop (as with static groups), in act-order
    d, g = 32, 8
    H, _ = spd(rng, d)
    W0 = rng.standard_normal((5, d)) * 0.02
    perm = O.act_order(H)
    Hd, _ = O.damping(H[np.ix_(perm, perm)], 0.01)
    W = W0[:, perm]
    sg = np.abs(W0).reshape(5, d // g, g).max(axis=2) / 7.0     # per original group
    s = sg[:, perm // g]                                         # step of processed column
    r = O.gptq_sweep(W, O.inverse_cholesky_upper(Hd), blocksize=8,
                     column_quantizer=unclipped_grid(s))
    assert np.array_equal(O.gptq_babai(W, Hd, s), r["codes"])


PINS = [pin_worked_example, pin_conditioned_example, pin_two_weight_closed_form,
        pin_cholesky_2x2, pin_cholesky_general, pin_obs_equals_cholesky,
        pin_blocked_equals_unblocked, pin_loss_identity, pin_brute_force_optimum,
        pin_gptq_beats_rtn_on_average, pin_act_order, pin_damping, pin_dead_columns,
        pin_hessian, pin_fit_and_round, pin_pack, pin_checkpoint_format,
        pin_format_roundtrip, pin_static_groups, pin_dequantize, pin_block_pipeline,
        pin_babai, pin_replay_hint]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(ORACLE)


def test_rtn_per_column_row_of_table():
    pin_rtn_per_column()
