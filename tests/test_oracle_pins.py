"""Pin the fp64 oracle to references other than itself (CPU only).

The second half plants plausible mistakes in copies of the oracle source and
checks that at least one pin catches each, so the pins are known to bite.
"""
import importlib.util
import math
import os
import types

import numpy as np
import pytest

import oracle.sparse_mla_ref as orc
from tests import oracle_pins as pins

TOL_LIB = 1e-10     # fp64 vs fp64 library routine
TOL_FD = 1e-6       # central differences with h = 1e-5 (truncation ~h^2, cancellation ~eps/h)
TOL_CLOSED = 1e-12


def test_pin_sdpa_library_routine():
    assert pins.pin_sdpa(orc) < TOL_LIB


def test_pin_finite_differences():
    assert pins.pin_finite_differences(orc) < TOL_FD


def test_pin_closed_forms():
    assert pins.pin_closed_forms(orc) < TOL_CLOSED


def test_pin_padding_invariants_exact():
    assert pins.pin_padding_invariants(orc) == 0.0


def test_pin_sum_rules_and_lse_bounds():
    assert pins.pin_sum_rules(orc) < 1e-9


def test_pin_delta_identity():
    assert pins.pin_delta_identity(orc) < 1e-10


def test_pin_check_indices_hand_count():
    assert pins.pin_check_indices(orc) == 0.0


def test_lse_empty_constant():
    # sumexp floor 1e-30 with the empty max read as 0
    assert orc.LSE_EMPTY == math.log(1e-30)
    assert abs(orc.LSE_EMPTY + 69.07755278982137) < 1e-12


def test_bf16_upcast_exact():
    bits = np.array([0x0000, 0x3F80, 0xBF80, 0x4049, 0x7F7F, 0x0001], dtype=np.uint16)
    want = np.array([0.0, 1.0, -1.0, 3.140625, 3.3895313892515355e38, 9.183549615799121e-41])
    assert np.array_equal(orc.bf16_bits_to_f64(bits), want)


def test_golden_hand_example():
    """tests/golden/hand_example.txt: a 3-row example worked by hand."""
    path = os.path.join(os.path.dirname(__file__), "golden", "hand_example.txt")
    vals = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split("=", 1)
            vals[k.strip()] = float(v)
    T, H = 3, 1
    q = np.zeros((T, H, 576))
    kv = np.zeros((T, 576))
    q[0, 0, 0] = 1.0
    q[0, 0, 512] = 1.0
    kv[0, 0] = 2.0          # score with row 0: 2 (latent) + 0 (tail)
    kv[0, 1] = 1.0
    kv[1, 512] = math.log(3.0)    # score with row 1: 0 (latent) + ln 3 (tail)
    kv[1, 1] = 5.0
    idx = np.array([[0, -1, 1], [-1, -1, -1], [2, 2, -1]], dtype=np.int32)
    out, lse = orc.sparse_mla_fwd(q, kv, idx, 1.0)
    assert abs(lse[0, 0] - vals["lse0"]) < 1e-12
    assert abs(out[0, 0, 0] - vals["out0_d0"]) < 1e-12
    assert abs(out[0, 0, 1] - vals["out0_d1"]) < 1e-12
    assert abs(lse[1, 0] - vals["lse1"]) < 1e-12
    assert np.all(out[1] == 0.0)
    assert abs(lse[2, 0] - vals["lse2"]) < 1e-12


# ---------------------------------------------------------------- planted mistakes

_SRC = open(orc.__file__).read()


def _mutant(old: str, new: str) -> types.ModuleType:
    assert old in _SRC, old
    src = _SRC.replace(old, new)
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src, "<oracle-mutant>", "exec"), mod.__dict__)
    return mod


MUTANTS = {
    "scores drop the rope tail": ("s = scale * (q_t @ K.T)             # [H, n]",
                                  "s = scale * (q_t[:, :512] @ K[:, :512].T)"),
    "value taken from the wrong columns": ("V = K[:, :D_LATENT]                 # the latent part is also the value",
                                           "V = K[:, D_TAIL:]"),
    "dS sign flipped": ("dS = P * (dP - dlt[:, None])", "dS = P * (dlt[:, None] - dP)"),
    "dkv tail dropped": ("G = scale * (dS.T @ q_t)                    # [n, 576]",
                         "G = scale * (dS.T @ q_t); G[:, 512:] = 0"),
    "dq missing scale": ("dq_t = scale * (dS @ K)                     # [H, 576]",
                         "dq_t = dS @ K"),
    "delta from the wrong operand": ("dlt = (dout_t * out_t).sum(axis=1)          # Delta from the given output",
                                     "dlt = (dout_t * dout_t).sum(axis=1)"),
    "lse in base 2": ("return out, m + np.log(l)\n\n\ndef _row",
                      "return out, (m + np.log(l)) / np.log(2.0)\n\n\ndef _row"),
    "padding read as row 0": ("keep = (idx_row >= 0) & (idx_row < T)\n    return idx_row[keep]",
                              "return np.maximum(idx_row, 0)[idx_row < T]"),
    "no sumexp floor on empty rows": ("m = np.zeros(H)\n        l = np.maximum(np.zeros(H), SUMEXP_FLOOR)",
                                      "m = np.full(H, -np.inf)\n        l = np.zeros(H)"),
    "P transposed in the dkv latent term": ("G[:, :D_LATENT] += P.T @ dout_t",
                                            "G[:, :D_LATENT] += (P.T @ dout_t)[::-1]"),
}


def _caught(mod) -> bool:
    checks = [
        lambda: pins.pin_sdpa(mod) < TOL_LIB,
        lambda: pins.pin_finite_differences(mod, n_coords=3) < TOL_FD,
        lambda: pins.pin_closed_forms(mod) < TOL_CLOSED,
        lambda: pins.pin_padding_invariants(mod) == 0.0,
        lambda: pins.pin_sum_rules(mod) < 1e-9,
        lambda: pins.pin_delta_identity(mod) < 1e-10,
    ]
    for c in checks:
        try:
            with np.errstate(all="ignore"):
                if not c():
                    return True
        except Exception:
            return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    old, new = MUTANTS[name]
    assert _caught(_mutant(old, new)), f"no pin caught: {name}"
