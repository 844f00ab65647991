"""The oracle pins are sensitive: plant plausible mistakes in a copy of the
oracle's C source (on the CPU) and check that the pins reject every one."""
import ctypes
import os
import subprocess

import pytest

import oracle
import oracle.oracle as ormod

from . import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(ormod.__file__), "gdn_oracle.c")

MUTATIONS = {
    # e formed from the undecayed state (the walkthrough snippet's reading)
    "undecayed_residual": ("                row[j] *= a;", "                row[j] *= 1.0 + 0.0 * a;"),
    # output read before the write
    "read_before_write": ("/* S_t = S~ + beta_t k_t e_t^T */", "/* write skipped */ if (0)"),
    # wrong sign of the residual
    "residual_sign": ("e[j] -= row[j] * ki;", "e[j] += row[j] * ki;"),
    # transposed state in the read-out
    "transposed_readout": ("yt[j] += row[j] * qi;", "yt[j] += S[(size_t)j * dv + i] * qt[j];"),
    # interleaved instead of contiguous head grouping
    "head_grouping": ("const int hk = hv / group;", "const int hk = hv % J->Hqk;"),
    # beta dropped from the write
    "dropped_beta": ("const double w = bt * kt[i];", "const double w = kt[i];"),
}

PIN_TESTS = [
    lambda: pins.test_transition_matrix_bruteforce(True),
    pins.test_identity_gates_keep_state,
    pins.test_beta_zero_is_pure_decay,
    pins.test_orthonormal_keys_store_and_retrieve,
    pins.test_repeated_key_overwrites,
    pins.test_single_step_from_zero_state,
    pins.test_decay_applies_before_the_residual,
    pins.test_golden_hand_worked_example,
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutation(name, tmp_path, monkeypatch):
    before, after = MUTATIONS[name]
    src = open(SRC).read()
    assert before in src, f"mutation anchor for {name} not found"
    msrc = tmp_path / "gdn_oracle_mut.c"
    msrc.write_text(src.replace(before, after))
    mlib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-shared", "-fPIC", "-pthread", "-o", str(mlib), str(msrc)], check=True)
    lib = ctypes.CDLL(str(mlib))
    dp = ctypes.POINTER(ctypes.c_double)
    lib.gdn_oracle_recurrence.restype = ctypes.c_int
    lib.gdn_oracle_recurrence.argtypes = [ctypes.c_int64, ctypes.c_int64] + [ctypes.c_int] * 4 + [dp] * 8 + [ctypes.c_int]
    monkeypatch.setattr(ormod, "_lib", lib)
    caught = 0
    for t in PIN_TESTS:
        try:
            t()
        except AssertionError:
            caught += 1
    assert caught >= 1, f"no pin rejects the '{name}' mutation"


def test_unmutated_oracle_passes_all_pins():
    oracle.build()
    for t in PIN_TESTS:
        t()
