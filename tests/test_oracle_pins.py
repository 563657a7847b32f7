"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()


def test_replay_plan_exhaustive():
    oc.check_replay_plan_exhaustive(200000)
