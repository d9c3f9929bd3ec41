"""The CPU oracle against its pins (closed forms, mpmath, torch, scipy,
finite differences, invariants). CPU only."""
import pytest

import oracle_pins as P  # noqa: E402


@pytest.mark.parametrize("case", P.load_golden(), ids=lambda c: c["name"])
def test_golden_closed_form(case):
    P.pin_golden_case(case)


def test_mpmath_bruteforce():
    pytest.importorskip("mpmath")
    P.pin_mpmath_bruteforce()


def test_torch_cross_entropy_float64():
    P.pin_torch_cross_entropy()


def test_scipy_logsumexp():
    pytest.importorskip("scipy")
    P.pin_scipy_logsumexp()


def test_finite_differences():
    P.pin_finite_differences()


def test_invariants():
    P.pin_invariants()


def test_shift_invariance_large_lse():
    P.pin_shift_invariance()


def test_sampled_forms_match_full():
    P.pin_sampled_forms()
