"""The fp64 oracle against its pins (CPU only)."""

import numpy as np
import pytest

from oracle import moe_oracle as O
from synth import LAYERS, make_layer, make_x
from tests import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(O)


def test_layer_invariants_tiny():
    spec = LAYERS["tiny"]
    arrays = make_layer(spec)
    x = make_x(spec, 9, 0)
    P.pin_layer_invariants(O, spec, arrays, x)


def test_tiny_selection_brute_force_and_margins():
    spec = LAYERS["tiny"]
    layer = O.Layer.from_spec(spec, make_layer(spec))
    x = make_x(spec, 64, 3)
    scores, sel = layer.route(layer.widen_x(x))
    b = scores + np.asarray(make_layer(spec)["bias"], np.float64)
    for t in range(x.shape[0]):
        want = P.brute_force_select(b[t], spec.n_group, spec.topk_group, spec.top_k)
        assert sorted(sel.ids[t].tolist()) == want
    assert np.all(sel.margin > 0)
