"""The CPU oracle against what the pages and the mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
from pins import ALL_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check(oracle.fwd, np.random.default_rng(20261202))


def test_rel_l2_hand_values():
    from pins import check_rel_l2
    check_rel_l2(oracle.rel_l2)


def test_step_recall_and_reset():
    from pins import check_step_recall
    check_step_recall(oracle.step, np.random.default_rng(20261203))


def test_step_chain_equals_forward():
    from pins import check_step_chain
    check_step_chain(oracle.step, oracle.fwd, np.random.default_rng(20261204))
