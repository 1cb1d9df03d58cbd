"""The end-to-end runner's piece planner (host logic, no GPU): the pieces tile the token axis in
order, every cut inside a sequence falls on a chunk boundary of that sequence, and each piece's
sequence offsets describe exactly the sequence parts it holds."""
import random

import pytest

from gdn_chunkwise_ut_gb300.api import _pieces


def _check(bounds, C, parts):
    plan = _pieces(bounds, C, parts)
    total = sum(b - a for a, b in bounds)
    assert sum(n1 - n0 for n0, n1, _ in plan) == total
    # consecutive, covering [first start, last end)
    assert plan[0][0] == bounds[0][0] and plan[-1][1] == bounds[-1][1]
    for (a0, a1, _), (b0, b1, _) in zip(plan, plan[1:]):
        assert a1 == b0
    starts = {a: (a, b) for a, b in bounds}
    for n0, n1, cu in plan:
        assert cu[0] == 0 and cu[-1] == n1 - n0 and all(x < y for x, y in zip(cu, cu[1:]))
        for x, y in zip(cu, cu[1:]):
            s0, s1 = n0 + x, n0 + y
            # the part [s0, s1) lies in one sequence and starts on a chunk boundary of it
            seq = next((a, b) for a, b in bounds if a <= s0 < b)
            assert s1 <= seq[1]
            assert (s0 - seq[0]) % C == 0
    return plan


@pytest.mark.parametrize("C", [32, 64, 128])
@pytest.mark.parametrize("parts", [1, 3, 8, 16])
def test_fixed_length_batch(C, parts):
    bounds = [(b * 8192, (b + 1) * 8192) for b in range(4)]
    plan = _check(bounds, C, parts)
    assert len(plan) <= parts + 1


@pytest.mark.parametrize("seed", range(5))
def test_varlen_batch(seed):
    rng = random.Random(seed)
    lengths = [rng.randint(1, 3000) for _ in range(rng.randint(1, 20))]
    bounds, pos = [], 0
    for n in lengths:
        bounds.append((pos, pos + n))
        pos += n
    for C in (32, 64, 128):
        for parts in (1, 2, 5, 8):
            _check(bounds, C, parts)


def test_empty_batch():
    assert _pieces([(0, 0)], 64, 8) == []
