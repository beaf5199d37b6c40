"""GPU tests of the HBM cache of host-resident experts (moe_layer_create_cached): the routed
experts stay in pinned host memory and are copied into HBM slots on demand (LRU), by
router-driven prefetch, or as a pinned hot set.

Outputs of a cached layer are bit-identical to the resident layer's grouped path (the same
kernels read the same packed bytes, only through a slot table), and match the oracle; the
cache's counters and residency follow the LRU, prefetch and pinning rules."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from oracle.moe_oracle import Layer
from synth import LAYERS, make_layer, make_x
from tests.gpu_util import empty_out, out_to_host, x_to_device
from tests.parity import check_out, check_routing

SPEC = LAYERS["small"]      # H = I = 2048, E = 32, k = 4
TMAX = 4                    # a forward needs at most min(E, TMAX * k) = 16 slots
_cache = {}


def layers():
    import quantized_moe_noaux_b300 as moe
    if "l" not in _cache:
        arrays = make_layer(SPEC)
        resident = moe.MoeLayer.from_spec(SPEC, arrays, max_tokens=TMAX)
        resident.set_path(moe.PATH_GROUPED)
        _cache["l"] = (arrays, resident, Layer.from_spec(SPEC, arrays))
    return _cache["l"]


def run(layer, x):
    out = empty_out(x.shape[0], SPEC.hidden, SPEC.act_dtype)
    layer.forward(x_to_device(x, SPEC.act_dtype), out)
    torch.cuda.synchronize()
    assert layer.status() == 0
    return out_to_host(out)


def per_expert_bytes():
    H, I = SPEC.hidden, SPEC.inter
    return 2 * I * (H // 2 + H // 16) + H * (I // 2 + I // 16)   # packed codes + fp16 scales


def test_cached_matches_resident_and_oracle():
    import quantized_moe_noaux_b300 as moe
    arrays, resident, oracle = layers()
    cached = moe.MoeLayer.from_spec(SPEC, arrays, max_tokens=TMAX, cache_slots=16)
    try:
        rng = np.random.default_rng(3)
        for step in range(14):
            T = int(rng.integers(1, TMAX + 1))
            x = make_x(SPEC, T, 100 + step)
            got = run(cached, x)
            assert np.array_equal(got, run(resident, x)), step
            if step % 5 == 0:
                ref = oracle.forward(x)
                rep = check_routing(ref, cached.routing(T), bias=arrays["bias"], n_group=SPEC.n_group,
                                    topk_group=SPEC.topk_group, top_k=SPEC.top_k, n_experts=SPEC.n_experts)
                if rep["mismatch"]:
                    ref = oracle.forward(x, ids=cached.routing(T)["ids"])
                check_out(ref.out, got)
        st = cached.cache_stats()
        assert st["misses"] > 0 and st["hits"] > 0 and st["evictions"] > 0, st
        assert st["bytes_h2d"] == (st["misses"] + st["prefetched"]) * per_expert_bytes(), st
        slot, pinned = cached.cache_query()
        assert (slot >= 0).sum() == 16 and not pinned.any()
        assert len(set(slot[slot >= 0].tolist())) == 16   # one expert per slot
    finally:
        cached.close()


def test_prefetch_makes_the_next_forward_hit():
    import quantized_moe_noaux_b300 as moe
    arrays, resident, _ = layers()
    cached = moe.MoeLayer.from_spec(SPEC, arrays, max_tokens=TMAX, cache_slots=16)
    try:
        for step in range(6):
            x = make_x(SPEC, TMAX, 200 + step)
            xd = x_to_device(x, SPEC.act_dtype)
            before = cached.cache_stats()
            cached.prefetch(xd)
            got = run(cached, x)
            after = cached.cache_stats()
            routed = int(np.count_nonzero(np.diff(cached.routing(TMAX)["offsets"])))
            # the prediction uses the same router on the same x: every routed expert is resident
            assert after["misses"] == before["misses"], (before, after)
            assert after["hits"] - before["hits"] == routed
            assert after["prefetch_hits"] - before["prefetch_hits"] == after["prefetched"] - before["prefetched"]
            assert np.array_equal(got, run(resident, x))
    finally:
        cached.close()


def test_pin_hot_set_stays_resident():
    import quantized_moe_noaux_b300 as moe
    arrays, resident, _ = layers()
    cached = moe.MoeLayer.from_spec(SPEC, arrays, max_tokens=TMAX, cache_slots=24)
    try:
        usage = np.zeros(SPEC.n_experts, np.int64)
        for step in range(10):
            x = make_x(SPEC, TMAX, 300 + step)
            run(cached, x)
            r = cached.routing(TMAX)
            usage[np.flatnonzero(np.diff(r["offsets"]))] += 1
        with pytest.raises(moe.MoeError):
            cached.cache_pin_hot(9)                 # would leave 15 < 16 unpinned slots
        cached.cache_pin_hot(8)
        _, pinned = cached.cache_query()
        order = sorted(range(SPEC.n_experts), key=lambda e: (-usage[e], e))[:8]
        assert sorted(np.flatnonzero(pinned).tolist()) == sorted(order)
        for step in range(12):
            x = make_x(SPEC, TMAX, 400 + step)
            assert np.array_equal(run(cached, x), run(resident, x))
            slot, pinned = cached.cache_query()
            assert np.all(slot[pinned == 1] >= 0)      # pinned experts never evicted
    finally:
        cached.close()


def test_cached_layer_rejects_other_paths():
    import quantized_moe_noaux_b300 as moe
    arrays, _, _ = layers()
    cached = moe.MoeLayer.from_spec(SPEC, arrays, max_tokens=TMAX, cache_slots=16)
    try:
        x = x_to_device(make_x(SPEC, 1, 0), SPEC.act_dtype)
        out = empty_out(1, SPEC.hidden, SPEC.act_dtype)
        for path in (moe.PATH_GEMV, moe.PATH_GENERIC):
            cached.set_path(path)
            with pytest.raises(moe.MoeError) as ei:
                cached.forward(x, out)
            assert ei.value.code == 2
    finally:
        cached.close()
