"""Suite-wide near-tie budget: decisions where the GPU and the float64 oracle
differ are allowed only when the oracle's margin is below 1e-6 (checked in each
parity test), and their number must stay at or below 1e-5 of every decision
compared in this run.  This file is collected after the parity tests."""
import pytest

from tests._parity import EXEMPT_RATIO, SESSION

pytestmark = pytest.mark.gpu


def test_near_tie_mismatches_within_budget():
    if SESSION.decisions == 0:
        pytest.skip("no parity decisions were compared in this run")
    print(f"decisions={SESSION.decisions} near-margin={SESSION.near_margin} "
          f"near-tie mismatches={SESSION.exempt}")
    assert SESSION.exempt <= EXEMPT_RATIO * SESSION.decisions
