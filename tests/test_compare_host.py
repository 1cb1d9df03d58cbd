"""Host logic of the whole-tensor comparison (no GPU): slabs cover every sequence once, and the
accumulated comparison passes the oracle against itself and fails a planted error."""
import numpy as np
import pytest

import oracle
from gdn_chunkwise_ut_gb300.inputs import cu_seqlens_from_lengths, make_inputs, varlen_lengths
from tests.compare import FullComparison, slabs


def test_slabs_cover_fixed_length_batches():
    for B, T in ((4, 8192), (1, 8192), (2, 16384), (3, 100), (5, 20000)):
        sl = slabs(B, T)
        assert sl[0][0] == 0 and sl[-1][1] == B * T
        for (a0, a1, cu), (b0, _, _) in zip(sl, sl[1:]):
            assert a1 == b0 and cu is None and (a1 - a0) % T == 0


def test_slabs_cover_varlen_batches():
    cu = cu_seqlens_from_lengths(varlen_lengths())
    sl = slabs(len(cu) - 1, 0, cu)
    assert sl[0][0] == 0 and sl[-1][1] == cu[-1]
    seen = []
    for n0, n1, rel in sl:
        assert rel[0] == 0 and rel[-1] == n1 - n0 and np.all(np.diff(rel) >= 0)
        seen += [int(x) + n0 for x in rel[1:]]
    assert seen == [int(x) for x in cu[1:]]
    # empty sequences stay inside a slab
    cu2 = cu_seqlens_from_lengths([0, 5, 0, 0, 7, 0])
    sl2 = slabs(6, 0, cu2, max_tokens=6)
    assert sum(len(r) - 1 for _, _, r in sl2) == 6


def test_full_comparison_accepts_exact_and_rejects_planted_error():
    k, v, beta = (x.double().numpy() for x in make_inputs(2, 150, 3, 128, 128, seed=3))
    T, W, U = oracle.oracle_fwd(k, v, beta, 64)
    acc = FullComparison()
    acc.add(T.astype(np.float32), W.astype(np.float32), U.astype(np.float32), T, W, U)
    st = acc.finish()
    assert st["T_max_abs"] < 1e-6 and st["W_rel_fro"] < 1e-6 and st["U_n_large"] == 0
    bad = U.copy()
    bad[1, 7, 2, 5] += 0.05
    acc2 = FullComparison()
    with pytest.raises(AssertionError):
        acc2.add(T, W, bad, T, W, U)
