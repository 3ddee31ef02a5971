"""The CPU oracle against its pins (hand-worked examples, library reductions,
brute force, closed forms).  CPU only."""
import pytest

import oracle
import oracle_pins as pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("name,check", pins.ALL_PINS, ids=[n for n, _ in pins.ALL_PINS])
def test_oracle_pin(lib, name, check):
    check(lib)


def test_traced_plan_brute_force(lib):
    import workloads as wl

    pins.pin_plan_brute_force(lib, wl.traced_batch(), dense_extra=3)


def test_config_ragged_closed_forms(lib):
    import workloads as wl

    pins.pin_ragged_closed_forms(lib, wl.ragged_batch())
    pins.pin_ragged_cp1(lib, wl.ragged_batch())
