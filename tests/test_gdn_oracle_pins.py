"""The GDN recurrence oracle against its pins (tests/gdn_pins.py), and planted mistakes in a copy of
it, each of which must fail at least one pin.  No GPU.

The mutants are textual edits of ``oracle/gdn_oracle.c`` compiled into a temporary directory: the
decay in the wrong place, the erase term without beta, the state update skipped, the state
transposed in the output, the initial state ignored or taken from the wrong sequence, the scale
dropped, and in the chunkwise form a strict causal mask, the decay dropped from the carried state or
from the output's state term, the sign of W S, and the decay of the chunk's last token.
"""
import os

import pytest

from oracle import gdn
from tests.gdn_pins import PINS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "gdn_oracle.c")

MUTATIONS = {
    # the token recurrence
    "decay_after_write": ("S[x] = at * (S[x] - bt * kt[d] * tmp[e]) + bt * kt[d] * vt[e];",
                          "S[x] = at * (S[x] - bt * kt[d] * tmp[e] + bt * kt[d] * vt[e]);"),
    "erase_without_beta": ("S[x] = at * (S[x] - bt * kt[d] * tmp[e])", "S[x] = at * (S[x] - kt[d] * tmp[e])"),
    "erase_without_decay_of_read": ("S[x] = at * (S[x] - bt * kt[d] * tmp[e]) + bt * kt[d] * vt[e];",
                                    "S[x] = at * S[x] - bt * kt[d] * tmp[e] + bt * kt[d] * vt[e];"),
    "update_skipped": ("    /* S <- alpha (S - beta k (S^T k)^T) + beta k v^T */",
                             "    for (int e = 0; e < dv; ++e) { double s0 = 0.0; for (int d = 0; d < dk; ++d) "
                             "s0 += S[(int64_t)d * dv + e] * qt[d]; ot[e] = scale * s0; } if (0)"),
    "state_transposed_in_output": ("            s += S[(int64_t)d * dv + e] * qt[d];",
                                   "            s += S[(int64_t)(e % dk) * dv + (d % dv)] * qt[d];"),
    "initial_state_ignored_recurrent": ("            if (h0)\n                memcpy(S, h0 + st, sizeof(double) * (size_t)(dk * dv));\n            else\n                memset(S, 0, sizeof(double) * (size_t)(dk * dv));\n            for (int64_t n = t0;",
                                        "            memset(S, 0, sizeof(double) * (size_t)(dk * dv));\n            for (int64_t n = t0;"),
    "scale_dropped": ("        ot[e] = scale * s;", "        ot[e] = s;"),
    "gate_wrong_head": ("const double at = g ? exp(g[n * H + h]) : 1.0;",
                        "const double at = g ? exp(g[n * H + (H - 1 - h)]) : 1.0;"),
    # the chunkwise form
    "chunk_mask_strict": ("for (int j = 0; j <= i; ++j) {", "for (int j = 0; j < i; ++j) {"),
    "chunk_state_term_undecayed": ("        const double gi = exp(G[i]);", "        const double gi = 1.0;"),
    "chunk_carry_undecayed": ("    const double decay = exp(glast);", "    const double decay = 1.0;"),
    "chunk_keys_undecayed": ("        const double f = exp(glast - G[j]);", "        const double f = 1.0;"),
    "chunk_correction_sign": ("Vp[(int64_t)i * dv + e] = ui[e] - s;", "Vp[(int64_t)i * dv + e] = ui[e] + s;"),
    "chunk_gate_exclusive": ("        if (g)\n            acc += g[(n0 + i) * H + h];\n        G[i] = acc;",
                             "        G[i] = acc;\n        if (g)\n            acc += g[(n0 + i) * H + h];"),
    "chunk_wrong_last_token": ("    const double glast = G[Lc - 1];", "    const double glast = G[Lc > 1 ? Lc - 2 : 0];"),
    "chunk_initial_state_next_sequence": ("            if (h0)\n                memcpy(S, h0 + st, sizeof(double) * (size_t)(dk * dv));\n            else\n                memset(S, 0, sizeof(double) * (size_t)(dk * dv));\n            for (int64_t n0 = t0;",
                                          "            if (h0)\n                memcpy(S, h0 + ((s + 1) % nseq * H + h) * dk * dv, sizeof(double) * (size_t)(dk * dv));\n            else\n                memset(S, 0, sizeof(double) * (size_t)(dk * dv));\n            for (int64_t n0 = t0;"),
}


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(gdn.load())


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
    mut = tmp_path / "gdn_oracle_mut.c"
    mut.write_text(src.replace(old, new))
    lib = gdn.load(gdn.build(src=mut, out=tmp_path / "libmut.so"))
    assert _pins_failing(lib), f"mutant {name} passed every pin"
