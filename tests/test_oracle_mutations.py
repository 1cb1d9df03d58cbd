"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant is a textual edit of ``oracle/kkt_oracle.c`` compiled into a
temporary directory; the real oracle is untouched.  The edits are the slips the
page warns about ("TileLang 实战：单位下三角矩阵求逆" §3.2: beta on rows and a
unit diagonal; §3.5/§4: the sign of the coupling term) and ordinary index
errors.  None of them reads or writes outside the buffers it is given.
"""
import os

import pytest

import oracle
from tests.pins import PINS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "kkt_oracle.c")

MUTATIONS = {
    "beta_on_columns": ("a = bc[i] * dot;", "a = bc[j] * dot;"),
    "diagonal_keeps_beta": ("a = 1.0;", "a = 1.0 + bc[i];"),
    "substitution_sign": ("xr[c] -= arj * xj[c];", "xr[c] += arj * xj[c];"),
    "dropped_first_term": ("for (int j = 0; j < r; ++j) {", "for (int j = 1; j < r; ++j) {"),
    "transposed_T_in_products": ("s += X[(int64_t)i * C + j] * f", "s += X[(int64_t)j * C + i] * f"),
    "beta_dropped_in_products": ("double f = bc[j];", "double f = 1.0;"),
    "gram_wrong_row": ("kc[(int64_t)i * dk + d] * kc[(int64_t)j * dk + d]",
                       "kc[(int64_t)i * dk + d] * kc[(int64_t)i * dk + d]"),
    "beta_wrong_head": ("bc[i] = beta[n * H + h];", "bc[i] = beta[n * H + (H - 1 - h)];"),
    "short_chunk_length": ("clen[q] = (int)((t1 - a) < C ? (t1 - a) : C);",
                           "clen[q] = (int)((t1 - a) < C ? (t1 - a) : C - 1);"),
    # the gated coefficient
    "gate_includes_first_token": ("for (int t = j + 1; t <= i; ++t)", "for (int t = j; t <= i; ++t)"),
    "gate_drops_last_token": ("for (int t = j + 1; t <= i; ++t)", "for (int t = j + 1; t < i; ++t)"),
    "gate_sign": ("return exp(s);", "return exp(-s);"),
    "gate_wrong_head": ("gc[i] = g[n * H + h];", "gc[i] = g[n * H + (H - 1 - h)];"),
    "gate_ignored": ("a *= gate_decay(gc, j, i);", "a *= 1.0;"),
    # the decay the keys of W carry from the chunk's start
    "w_decay_ignored": ("f *= decay_from_start(gc, j);", "f *= 1.0;"),
    "w_decay_excludes_own_token": ("for (int t = 0; t <= j; ++t)", "for (int t = 0; t < j; ++t)"),
    "w_decay_on_values_too": ("apply_scaled(X, bz, NULL, vc, Lc, C, dv, U);", "apply_scaled(X, bz, gc, vc, Lc, C, dv, U);"),
    "w_decay_sign": ("return exp(acc);", "return exp(-acc);"),
}


def _pins_failing(lib):
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mut = tmp_path / "kkt_oracle_mut.c"
    mut.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(src=mut, out=tmp_path / "libmut.so"))
    failed = _pins_failing(lib)
    assert failed, f"mutant {name} passed every pin"
