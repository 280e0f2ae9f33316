"""CPU tests: the fp64 oracle against its pins, and the pins against planted mistakes."""
import os

import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.default())


@pytest.mark.parametrize("D", [4, 6, 8])
def test_finite_differences_sizes(D):
    oracle_pins.pin_finite_differences(oracle.default(), D=D, T=9 + D)


def test_finite_differences_recon():
    oracle_pins.pin_finite_differences(oracle.default(), D=5, T=12, mode="recon")


# Each planted mistake is a plausible slip in the oracle source (a dropped term, a wrong
# index, swapped operands, a wrong sign, an off-by-one).  The mutant is compiled from a
# patched copy of wkv7_oracle.c, on the CPU; at least one pin must reject it.
MUTANTS = {
    "drop_sa_b_term": ("+ v[i] * k[j] + sa[i] * bb[j];", "+ v[i] * k[j];"),
    "decay_by_row_index": ("S[i * D + j] = S[i * D + j] * w[j]", "S[i * D + j] = S[i * D + j] * w[i]"),
    "swap_a_and_b": ("s += S[i * D + j] * a[j];", "s += S[i * D + j] * bb[j];"),
    "transposed_state_in_sa": ("s += S[i * D + j] * a[j];", "s += S[j * D + i] * a[j];"),
    "y_before_update": ("for (int j = 0; j < D; j++) s += S[i * D + j] * r[o + j];",
                        "for (int j = 0; j < D; j++) s += (S[i * D + j] - v[o + i] * k[o + j]) * r[o + j];"),
    "ckpt_off_by_one": ("(t + 1) % chunk == 0", "t % chunk == 0"),
    "bwd_sign_of_a_term": ("* w[o + j] + dsa[i] * a[o + j];", "* w[o + j] - dsa[i] * a[o + j];"),
    "bwd_dk_wrong_vector": ("s_k += G[i * D + j] * v[o + i];", "s_k += G[i * D + j] * k[o + i];"),
    "bwd_dr_pre_update_state": ("s_r += dy[o + i] * Snew[i * D + j];", "s_r += dy[o + i] * S[i * D + j];"),
    "bwd_da_transposed": ("for (int i = 0; i < D; i++) s += dsa[i] * S[i * D + j];",
                          "for (int i = 0; i < D; i++) s += dsa[i] * S[j * D + i];"),
    "bwd_recon_divides_by_row": ("/ w[o + j];", "/ w[o + i];"),
    "bwd_dy_r_transposed": ("G[i * D + j] += dy[o + i] * r[o + j];", "G[i * D + j] += dy[o + j] * r[o + i];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.source_path()).read()
    assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    mpath = os.path.join(tmp_path, "mutant.c")
    with open(mpath, "w") as f:
        f.write(src.replace(old, new))
    mut = oracle.Oracle(oracle.compile_c(mpath, os.path.join(tmp_path, "mutant.so")))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mut)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin rejects the planted mistake {name}"
