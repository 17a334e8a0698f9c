"""Plants plausible mistakes in a copy of the oracle and checks that the pins catch each one.

Every mutation below is a one-place change to the oracle's C source, built
into a temporary library on the CPU.  The real oracle is never modified.
"""
import os

import pytest

from oracle import oracle
from tests import oracle_pins

_STEPS = (
    "        decay_rows(S, g_t, dk, dv);\n"
    "        read_state(S, k_t, vhat, dk, dv);\n"
    "        prediction_error(v_t, vhat, delta, dv);\n"
    "        write_state(S, k_t, J->beta[th], delta, dk, dv);\n"
    "        read_output(S, q_t, o_t, dk, dv);\n"
)

MUTATIONS = {
    # D applied after the rank-one write instead of before it.
    "decay_after_write": (_STEPS, _STEPS.replace("        decay_rows(S, g_t, dk, dv);\n", "")
                          .replace("        read_output", "        decay_rows(S, g_t, dk, dv);\n        read_output")),
    # output read from the state before token t's write.
    "output_before_write": (_STEPS, _STEPS.replace("        read_output(S, q_t, o_t, dk, dv);\n", "")
                            .replace("        write_state", "        read_output(S, q_t, o_t, dk, dv);\n        write_state")),
    "no_decay": (_STEPS, _STEPS.replace("        decay_rows(S, g_t, dk, dv);\n", "")),
    "decay_linearised": ("const double d = exp(g_t[i]);", "const double d = 1.0 + g_t[i];"),
    "decay_sign": ("const double d = exp(g_t[i]);", "const double d = exp(-g_t[i]);"),
    # D multiplies the value columns instead of the key rows (S D instead of D S).
    "decay_on_columns": ("for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= d;",
                         "for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= exp(g_t[j % dk]); (void)d;"),
    "error_sign": ("delta[j] = v_t[j] - vhat[j];", "delta[j] = vhat[j] - v_t[j];"),
    "no_beta": ("write_state(S, k_t, J->beta[th], delta, dk, dv);", "write_state(S, k_t, 1.0, delta, dk, dv);"),
    "output_with_k": ("read_output(S, q_t, o_t, dk, dv);", "read_output(S, k_t, o_t, dk, dv);"),
    # o = S q instead of S^T q (indices wrapped so that every access stays in bounds).
    "output_transposed": ("for (int j = 0; j < dv; ++j) o_t[j] += S[(size_t)i * dv + j] * q_t[i];",
                          "for (int j = 0; j < dv; ++j) o_t[j] += S[(size_t)(j % dk) * dv + (i % dv)] * q_t[i];"),
    # the boundary is off by one: the first token of the next document leaks into this one.
    "boundary_off_by_one": ("const int32_t t0 = J->cu_seqlens[seq], t1 = J->cu_seqlens[seq + 1];",
                            "const int32_t t0 = J->cu_seqlens[seq], t1 = J->cu_seqlens[seq + 1] + "
                            "(seq + 1 < J->num_seqs && J->cu_seqlens[seq + 2] > J->cu_seqlens[seq + 1]);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    with open(oracle._SRC) as f:
        src = f.read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, "mutation anchor not found; update the mutation table"
    mutated = tmp_path / "kda_oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(force=True, src=str(mutated), out=str(tmp_path / "libmut.so")))
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "no pin caught mutation %s" % name
