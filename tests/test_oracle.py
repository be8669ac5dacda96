"""The float64 oracle against hand-worked closed forms, brute force, a library routine and invariants."""

import pytest

import oracle_pins


@pytest.mark.parametrize("case", oracle_pins.load_golden(), ids=lambda c: c["name"])
def test_golden_closed_form(case):
    oracle_pins.check_golden(case)


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def test_golden_file_has_citations():
    for case in oracle_pins.load_golden():
        assert case["cite"], case["name"]
