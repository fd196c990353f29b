"""The CPU oracle against what the pages and the mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
from pins import ALL_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check(oracle.fwd, np.random.default_rng(20261202))
