"""The oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from oracle_pins import ALL_PINS, _read_golden
from context_ra_forward_gb300 import inputs


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)


def test_alibi_slopes_golden():
    """The slope vector handed to both sides matches the hand-written H=8 values
    ("超长上下文技术" survey §2.1.2)."""
    want = [float(x) for x in _read_golden("alibi_slopes_H8.txt")[0].split()]
    assert inputs.alibi_slopes(8).tolist() == want


def test_inputs_seeded_and_rounded():
    w = inputs.WORKLOADS["C3"]
    a = inputs.make_inputs(w, H=2, S=256)
    b = inputs.make_inputs(w, H=2, S=256)
    for key in ("q", "k", "v"):
        assert a[key].dtype.is_floating_point and a[key].shape == (1, 2, 256, 128)
        assert (a[key].float() == b[key].float()).all()
    x = inputs.to_f64_numpy(a["q"])
    assert x.dtype == np.float64 and np.array_equal(x, a["q"].float().numpy().astype(np.float64))


def test_split_validation():
    with pytest.raises(ValueError):
        oracle.index_maps(10, 3, "contiguous")
    with pytest.raises(ValueError):
        oracle.index_maps(12, 4, "zigzag")
    with pytest.raises(ValueError):
        oracle.index_maps(12, 0, "zigzag")
