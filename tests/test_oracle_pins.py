"""The CPU oracle against its pins (no GPU)."""

import numpy as np
import pytest

import oracle
import oracle_pins
import workloads
from checks import check_workload
from golden import load_cases


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c.name)
def test_golden_case(o, case):
    got = np.sort(oracle_pins.run_case(o, case), axis=1)
    assert (got == np.sort(case.expect, axis=1)).all(), case.cites


def test_order_key_is_float_order(o):
    """The key is strictly monotone in float order, with -0.0 just below +0.0."""
    g = np.random.Generator(np.random.PCG64(3))
    bits = g.integers(0, 2**32, size=4000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[~np.isnan(vals)]
    specials = np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 1.0, -1.0,
                         np.finfo(np.float32).max, -np.finfo(np.float32).max], np.float32)
    vals = np.concatenate([vals, specials])
    keys = np.array([o.order_key(float(v)) for v in vals], dtype=np.uint64)
    for i in range(len(vals) - 1):
        a, b = vals[i], vals[i + 1]
        ka, kb = keys[i], keys[i + 1]
        fa = oracle_pins._value_order(a)
        fb = oracle_pins._value_order(b)
        assert (ka < kb) == (fa < fb) and (ka == kb) == (fa == fb), (a, b)


def test_brute_force_tiny_rows(o):
    oracle_pins.pin_brute_force(o)


def test_closed_form_short_rows(o):
    oracle_pins.pin_closed_form(o)


def test_invariants_all_generators(o):
    oracle_pins.pin_invariants(o)


def test_matches_torch_topk_on_continuous_data(o):
    pytest.importorskip("torch")
    oracle_pins.pin_torch_topk(o)


def test_forms_agree(o):
    oracle_pins.pin_forms(o)


def test_threads_agree(o):
    oracle_pins.pin_threads(o)


def test_config1_invariants(o):
    w = workloads.config1()
    assert not check_workload(w, o.run(w))


def test_invalid_arguments_raise(o):
    with pytest.raises(ValueError):
        o.topk_raw(np.zeros((1, 4), np.float32), np.array([4], np.int32), 0)
