"""Each plausible mistake planted in a copy of the oracle is caught by some pin.

The mistakes are planted in the oracle's source text on the CPU (a dropped term, a
flipped sign, a transposed operand, a wrong index, a wrong constant) and the copy is run
through every pin of ``test_oracle_pins``.
"""

import inspect
import types

import pytest

from oracle import gptq_oracle as ORACLE
from tests.test_oracle_pins import PINS

SOURCE = inspect.getsource(ORACLE)

MUTATIONS = {
    "update_sign": ("W[:, q + 1:i2] -= np.outer(e, U[q, q + 1:i2])",
                    "W[:, q + 1:i2] += np.outer(e, U[q, q + 1:i2])"),
    "update_transposed_row": ("W[:, q + 1:i2] -= np.outer(e, U[q, q + 1:i2])",
                              "W[:, q + 1:i2] -= np.outer(e, U[q + 1:i2, q])"),
    "lazy_update_dropped": ("W[:, i2:] -= Err @ U[i1:i2, i2:]",
                            "W[:, i2:] -= 0.0 * (Err @ U[i1:i2, i2:])"),
    "lazy_update_transposed": ("W[:, i2:] -= Err @ U[i1:i2, i2:]",
                               "W[:, i2:] -= Err @ U[i2:, i1:i2].T"),
    "err_not_scaled": ("e = (W[:, q] - what) / U[q, q]", "e = (W[:, q] - what)"),
    "hessian_factor": ("return (2.0 / n) * (X.T @ X)", "return (1.0 / n) * (X.T @ X)"),
    "hessian_stream_rescale": ("H = H * (n / (n + t))", "H = H"),
    "damping_absolute": ("lam = float(percdamp) * float(np.mean(np.diag(H)))",
                         "lam = float(percdamp)"),
    "act_order_ascending": ("np.argsort(-diag, kind=\"stable\")",
                            "np.argsort(diag, kind=\"stable\")"),
    "zero_floor": ("r = np.rint(u)", "r = np.floor(u)"),
    "lo_not_clamped": ("lo = np.minimum(np.min(wg, axis=1), 0.0).astype(F32)",
                       "lo = np.min(wg, axis=1).astype(F32)"),
    "factor_lower": ("return np.ascontiguousarray(Lh.T)", "return np.ascontiguousarray(Lh)"),
    "schur_sign": ("Hinv[q + 1:, q + 1:] -= np.outer", "Hinv[q + 1:, q + 1:] += np.outer"),
    "loss_half_dropped": ("loss += 0.5 * e * e", "loss += e * e"),
    "pack_big_endian": ("(stream << np.arange(32, dtype=np.uint64))",
                        "(stream << np.arange(31, -1, -1, dtype=np.uint64))"),
    "g_idx_from_perm": ("return (pos // group).astype(np.int32)",
                        "return (perm // group).astype(np.int32)"),
    "sym_step": ("amax / F32((1 << (bits - 1)) - 1)", "amax / F32((1 << bits) - 1)"),
    "round_floor": ("own = np.clip(np.rint(v) + z, lowest, maxq)",
                    "own = np.clip(np.floor(v) + z, lowest, maxq)"),
    "dead_not_zeroed": ("W[:, dead] = 0.0", "pass"),
    "static_group_of_processing_position": (
        "gcol = np.zeros(d, dtype=np.int64) if group == -1 else perm // group",
        "gcol = np.zeros(d, dtype=np.int64) if group == -1 else np.arange(d) // group"),
    "static_fit_on_permuted": ("sc, ze = static_group_fit(W, group, bits, sym,",
                               "sc, ze = static_group_fit(W[:, perm], group, bits, sym,"),
    "static_g_idx_permuted": ("if static and group != -1:", "if False:"),
    "babai_natural_order": (
        "codes[r] = babai_nearest_plane((B * s[r][None, :])[:, ::-1], B @ W[r])[::-1]",
        "codes[r] = babai_nearest_plane(B * s[r][None, :], B @ W[r])"),
    "babai_steps_reversed": (
        "codes[r] = babai_nearest_plane((B * s[r][None, :])[:, ::-1], B @ W[r])[::-1]",
        "codes[r] = babai_nearest_plane((B * s[r][::-1][None, :])[:, ::-1], B @ W[r])[::-1]"),
    "babai_floor": ("z[j] = np.rint((y[j] - R[j, j + 1:] @ z[j + 1:]) / R[j, j])",
                    "z[j] = np.floor((y[j] - R[j, j + 1:] @ z[j + 1:]) / R[j, j])"),
    # the replay rule of the GPU parity check: the near-tie band and the neighbour test
    "hint_band_always_codes": ("near = np.abs(v - (fl + 0.5)) < tie_eps",
                               "near = np.ones(v.shape, dtype=bool)"),
    "hint_band_always_zeros": ("near = np.abs(u - (fl + 0.5)) < tie_eps",
                               "near = np.ones(u.shape, dtype=bool)"),
    "hint_neighbour_widened_codes": (
        "take = near & (hint != own) & ((hint == lo_c) | (hint == hi_c))",
        "take = near & (hint != own) & (np.abs(hint - own) <= 2)"),
    "hint_neighbour_unclamped_codes": ("hi_c = np.clip(fl + 1 + z, lowest, maxq)",
                                       "hi_c = fl + 1 + z"),
    "hint_neighbour_widened_zeros": (
        "take = near & (hint != r) & ((hint == fl) | (hint == fl + 1))",
        "take = near & (hint != r) & (np.abs(hint - r) <= 2)"),
    "rows_unreversed": ("    return np.ascontiguousarray(Y.T[:, ::-1])",
                        "    return np.ascontiguousarray(Y.T)"),
    "rows_wrong_index": ("E[d - 1 - rows, np.arange(rows.size)] = 1.0",
                         "E[rows, np.arange(rows.size)] = 1.0"),
    "dequant_zero_dropped": ("return s * (codes.astype(F64) - z)", "return s * codes.astype(F64)"),
    "dequant_scale_of_position": ("s = np.asarray(scales, dtype=F64)[g].T",
                                  "s = np.asarray(scales, dtype=F64)[np.arange(g.size) * len(scales) // g.size].T"),
}


def mutated_oracle(name):
    old, new = MUTATIONS[name]
    assert SOURCE.count(old) >= 1, f"mutation {name}: pattern not found"
    src = SOURCE.replace(old, new, 1)
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src, mod.__name__, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    mod = mutated_oracle(name)
    caught = []
    for pin in PINS:
        try:
            pin(mod)
        except Exception:  # an AssertionError or a crash both count as caught
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name!r}"
