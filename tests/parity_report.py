"""Prints the whole-tensor errors of every full-size workload against the oracle (GPU).

    python -m tests.parity_report [--gated-only | --plain-only]

One markdown table row per workload: max-abs of T, max-abs and relative Frobenius error of W and
U~, and n_large (elements with |x_ref| >= 8, whose bound is 2e-2 plus half a bf16 ulp).  The
assertions are those of ``tests/test_full_size_gpu.py``.
"""
from __future__ import annotations

import sys

from tests.fullsize import GATED, PLAIN, run_and_compare


def main(argv):
    runs = []
    if "--gated-only" not in argv:
        runs += [(n, False) for n in PLAIN]
    if "--plain-only" not in argv:
        runs += [(n, True) for n in GATED]
    print("| Workload | Gated | Tokens x heads | T max-abs | W max-abs | W rel-Frob | U max-abs | U rel-Frob "
          "| n_large (W, U) |")
    print("|---|---|---|---|---|---|---|---|---|")
    for name, gated in runs:
        st = run_and_compare(name, gated=gated)
        print(f"| {name} | {'yes' if gated else 'no'} | {st['tokens']} x {st['heads']} | {st['T_max_abs']:.2e} "
              f"| {st['W_max_abs']:.2e} | {st['W_rel_fro']:.2e} | {st['U_max_abs']:.2e} | {st['U_rel_fro']:.2e} "
              f"| {st['W_n_large']}, {st['U_n_large']} |", flush=True)


if __name__ == "__main__":
    main(sys.argv[1:])
