"""Plants plausible mistakes in a copy of the attention oracle and checks that
the pins catch every one (CPU only).  The oracle on disk is never modified:
each mutant is the oracle's source with one substitution, executed into a
fresh module object."""

import os
import types

import pytest

import pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "attention.py")

MUTATIONS = {
    "dropped_scale_fwd": ("S = scale * (qb[rows] @ Ks.T)\n                    m = S.max(axis=1)\n                    lse = m + np.log(np.exp(S - m[:, None]).sum(axis=1))\n                    P = np.exp(S - lse[:, None])\n                    O[",
                          "S = (qb[rows] @ Ks.T)\n                    m = S.max(axis=1)\n                    lse = m + np.log(np.exp(S - m[:, None]).sum(axis=1))\n                    P = np.exp(S - lse[:, None])\n                    O["),
    "log2_lse": ("lse = m + np.log(np.exp(S - m[:, None]).sum(axis=1))\n                    P = np.exp(S - lse[:, None])\n                    O[",
                 "lse = m + np.log2(np.exp(S - m[:, None]).sum(axis=1))\n                    P = np.exp(S - lse[:, None])\n                    O["),
    "wrong_delta_sign": ("dS = P * (dP - delta[:, None])", "dS = P * (dP + delta[:, None])"),
    "dropped_scale_dk": ("dKs += scale * (dS.T @ qb[rows])", "dKs += (dS.T @ qb[rows])"),
    "dk_uses_keys": ("dKs += scale * (dS.T @ qb[rows])", "dKs += scale * (dS.T @ kb[rows])"),
    "dv_uses_values": ("dVs += P.T @ dob[rows]", "dVs += P.T @ vb[rows]"),
    "dq_transposed_operand": ("dQ[b, rows, hi] = scale * (dS @ Ks)", "dQ[b, rows, hi] = scale * (dS @ Vs)"),
    "padding_admitted": ("seq_row[seq_row >= 0]", "seq_row[seq_row >= -1]"),
    "ids_merged": ("np.nonzero(seq_row == s)[0]", "np.nonzero(seq_row >= s)[0]"),
    "missing_max_shift": ("P = np.exp(S - lse[:, None])\n                    O[", "P = np.exp(S - m[:, None])\n                    O["),
    "keys_take_query_ids": ("yield rows, np.nonzero(np.asarray(k_row) == s)[0]", "yield rows, np.nonzero(np.asarray(q_row) == s)[0]"),
    "dk_at_query_positions": ("dK[b, kidx, hi] = dKs", "dK[b, idx, hi] = dKs"),
    "padding_keys_admitted": ("yield rows, np.nonzero(np.asarray(k_row) == s)[0]", "yield rows, np.nonzero((np.asarray(k_row) == s) | (np.asarray(k_row) < 0))[0]"),
}


def _mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutant(name):
    mod = _mutant(*MUTATIONS[name])
    failures = []
    for pin in pins.ALL_PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failures.append(pin.__name__)
    assert failures, f"no pin caught the planted mistake {name}"


def test_unmutated_copy_passes():
    src = open(SRC).read()
    mod = types.ModuleType("oracle_copy")
    exec(compile(src, "oracle_copy", "exec"), mod.__dict__)
    for pin in pins.ALL_PINS:
        pin(mod)
