"""Every element of T, W and U~ against the fp64 oracle, at full size, on every workload (GPU).

Each workload runs in the bench's launch configuration (one call over the whole workload, kernel
"auto", the cached workspace); ``tests/fullsize.py`` compares the whole output with the oracle under
the tolerances of ``tests/compare.py``.  The ungated runs cover the five workload families (the
fp32 case, the 8192-token sequence, the head sweep H in {64, 48, 32, 24, 16, 8}, the 32-sequence
varlen batch and the chunk sizes 32, 64 and 128); the gated runs cover all but the head sweep's
other head counts.
"""
import pytest

from tests.fullsize import GATED, PLAIN, run_and_compare

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", PLAIN)
def test_full_size_every_element(name):
    st = run_and_compare(name)
    assert st["W_elements"] > 0


@pytest.mark.parametrize("name", GATED)
def test_gated_full_size_every_element(name):
    st = run_and_compare(name, gated=True)
    assert st["U_elements"] > 0
