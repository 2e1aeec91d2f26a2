"""The block step's host decisions: the confidence prefix of a drafted block
and the hybrid rule (confidence-only decoding commits the first draft and
extends through consecutive drafts whose probability clears tau; hybrid
decoding commits that prefix when it is at least m long, else verifies).
CPU only."""
import pytest

from ternary_w2a8_linear_gb300.blockstep import confidence_length, needs_verification


@pytest.mark.parametrize("p,tau,expect", [
    ([], 0.9, 0),
    ([0.1], 0.9, 1),                          # the first draft is always committed
    ([0.1, 0.95, 0.99], 0.9, 3),              # the first draft's own probability does not count
    ([0.99, 0.5, 0.99, 0.99], 0.9, 1),        # stops at the first draft below tau
    ([0.99, 0.95, 0.91, 0.2, 0.99], 0.9, 3),  # consecutive only: the later 0.99 is not reached
    ([0.5, 0.9, 0.9], 0.9, 3),                # p == tau clears it
    ([0.5, 0.8999999, 0.99], 0.9, 1),
    ([1.0] * 8, 0.9, 8),                      # a whole block of D = 8
])
def test_confidence_length(p, tau, expect):
    assert confidence_length(p, tau) == expect


def test_hybrid_rule():
    assert needs_verification(1, 4)
    assert needs_verification(3, 4)
    assert not needs_verification(4, 4)
    assert not needs_verification(8, 4)
    assert needs_verification(0, 1)
