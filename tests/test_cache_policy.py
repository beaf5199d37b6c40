"""Host policy of the HBM cache of host-resident experts, on the CPU.

The policy follows "Cara kerja eksekusi MoE berbasis streaming disk" in "Show HN: Menjalankan
GLM 5.2 di komputer lambat" (a per-layer least-recently-used cache of experts over slower
storage, a pinned hot store chosen by usage counts) and "Yönlendirici İleriye Dönük
Ön-Getirme" in "Show HN: GLM 5.2 Modelini Yavaş Bilgisayarımda Çalıştırmak" (router-driven
prefetch). The library's own expert_cache.cu is compiled unchanged with g++ against the CUDA
runtime double in tests/cache_host, whose copies run at once and are logged, so the tests
read the exact sequence of copies, stream waits and event records the cache issues.

Checked: residency after every request; slot contents byte-equal to the expert's host
bytes; free slots first, then least-recently-used eviction among experts that are neither
needed by the request nor pinned (ties: lower slot); the pinned hot set (highest usage,
ties lower id, earlier pins released, pinned experts never evicted); the counters; the
fence that makes a request's first copy wait for the layer's last recorded compute; the
completion event that the compute stream waits on; error returns from failing runtime
calls."""

import ctypes
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest

ROOT = Path(__file__).resolve().parent.parent
COPY, WAIT, RECORD, SYNC = 1, 2, 3, 4
OK, INVALID_ARG, UNSUPPORTED, ERR_CUDA = 0, 1, 2, 4
STATS = ("hits", "misses", "prefetched", "prefetch_hits", "bytes_h2d", "evictions")
UP, DN = 96, 80          # bytes per expert of the gate/up and down stores (any sizes serve)


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    out = tmp_path_factory.mktemp("cache_host") / "libcachehost.so"
    here = ROOT / "tests" / "cache_host"
    cmd = [gxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-shared", "-fPIC", "-I", str(here),
           "-x", "c++", str(ROOT / "quantized_moe_noaux_b300" / "csrc" / "expert_cache.cu"),
           str(here / "harness.cpp"), "-o", str(out)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    L = ctypes.CDLL(str(out))
    L.ch_create.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_long, ctypes.c_long]
    L.ch_ensure.argtypes = [ctypes.c_void_p, ctypes.c_int]
    L.ch_pin_hot.argtypes = [ctypes.c_int, ctypes.c_int]
    L.ch_slot_of.argtypes = [ctypes.c_int]
    L.ch_pinned.argtypes = [ctypes.c_int]
    L.ch_stats.argtypes = [ctypes.c_void_p]
    L.ch_take_log.argtypes = [ctypes.c_void_p, ctypes.c_int]
    L.ch_slot_holds.argtypes = [ctypes.c_int, ctypes.c_int]
    L.ch_fail_call.argtypes = [ctypes.c_int]
    assert L.ch_num_stats() == len(STATS)
    yield L
    L.ch_destroy()


class Cache:
    def __init__(self, lib, E, slots):
        lib.ch_fail_call(0)
        assert lib.ch_create(E, slots, UP, DN) == OK
        self.lib, self.E, self.slots = lib, E, slots
        assert lib.ch_slots() == slots
        self.copy_stream = lib.ch_copy_stream()
        self.compute_stream = lib.ch_compute_stream()
        assert self.copy_stream != self.compute_stream
        assert len(self.take()) == 0

    def take(self):
        buf = np.zeros((4096, 7), np.int32)
        n = self.lib.ch_take_log(buf.ctypes.data, 4096)
        return buf[:n].copy()

    def ensure(self, experts, prefetch=False):
        counts = np.zeros(self.E, np.int32)
        counts[list(experts)] = 1
        return self.lib.ch_ensure(counts.ctypes.data, int(prefetch)), self.take()

    def note_compute(self):
        return self.lib.ch_note_compute(), self.take()

    def wait_copies(self):
        return self.lib.ch_wait_copies(), self.take()

    def pin_hot(self, n, min_free):
        return self.lib.ch_pin_hot(n, min_free), self.take()

    def slot_of(self):
        return np.array([self.lib.ch_slot_of(e) for e in range(self.E)])

    def owners(self):
        owner = np.full(self.slots, -1)
        for e, s in enumerate(self.slot_of()):
            if s >= 0:
                assert owner[s] == -1, "two experts in one slot"
                owner[s] = e
        return owner

    def pinned(self):
        return np.array([self.lib.ch_pinned(e) for e in range(self.E)], bool)

    def stats(self):
        buf = np.zeros(len(STATS), np.int64)
        self.lib.ch_stats(buf.ctypes.data)
        return dict(zip(STATS, buf.tolist()))

    def check_contents(self):
        for s, e in enumerate(self.owners()):
            if e >= 0:
                assert self.lib.ch_slot_holds(s, int(e)), (s, e)


def kinds(ops):
    return [int(k) for k in ops[:, 0]]


def copies_of(cache, ops):
    """(expert, slot) per loaded expert, in issue order; each load is a gate/up copy then a
    down copy of the full per-expert size, from the expert's host bytes into one slot, on the
    cache's copy stream."""
    c = ops[ops[:, 0] == COPY]
    assert len(c) % 2 == 0
    loads = []
    for up, dn in c.reshape(-1, 2, 7):
        assert up[1] == dn[1] == cache.copy_stream
        assert (up[3], dn[3]) == (0, 1)
        assert up[4] == dn[4] >= 0 and up[5] == dn[5] >= 0
        assert (up[6], dn[6]) == (UP, DN)
        loads.append((int(up[5]), int(up[4])))
    return loads


# ---------------------------------------------------------------------------------------
# hand-worked sequences


def test_lru_sequence_by_hand(lib):
    c = Cache(lib, E=6, slots=3)
    st, ops = c.ensure({0, 1})
    assert st == OK and copies_of(c, ops) == [(0, 0), (1, 1)]
    assert kinds(ops) == [COPY, COPY, COPY, COPY, RECORD]      # nothing computed yet: no fence
    copied_ev = int(ops[-1, 2])
    assert ops[-1, 1] == c.copy_stream
    st, ops = c.ensure({2})
    assert st == OK and copies_of(c, ops) == [(2, 2)]
    st, ops = c.note_compute()
    assert st == OK and kinds(ops) == [RECORD] and ops[0, 1] == c.compute_stream
    computed_ev = int(ops[0, 2])
    assert computed_ev != copied_ev
    # 0 hits; 3 evicts the older of 1 (request 1) and 2 (request 2): expert 1 in slot 1
    st, ops = c.ensure({0, 3})
    assert st == OK and copies_of(c, ops) == [(3, 1)]
    assert kinds(ops) == [WAIT, COPY, COPY, RECORD]
    assert list(ops[0, 1:3]) == [c.copy_stream, computed_ev]
    assert list(ops[-1, 1:3]) == [c.copy_stream, copied_ev]
    # a prefetch of 4 evicts expert 2, the least recently used (0 and 3: request 3)
    st, ops = c.ensure({4}, prefetch=True)
    assert st == OK and copies_of(c, ops) == [(4, 2)]
    # 1 must evict 0 or 3, both last used by request 3: the tie goes to the lower slot (0)
    st, ops = c.ensure({1, 4})
    assert st == OK and copies_of(c, ops) == [(1, 0)]
    assert list(c.owners()) == [1, 3, 4]
    assert c.stats() == dict(hits=2, misses=5, prefetched=1, prefetch_hits=1,
                             bytes_h2d=6 * (UP + DN), evictions=3)
    # all hits: no copy, no fence, one completion record
    st, ops = c.ensure({1, 3, 4})
    assert st == OK and kinds(ops) == [RECORD]
    st, ops = c.wait_copies()
    assert st == OK and kinds(ops) == [WAIT] and list(ops[0, 1:3]) == [c.compute_stream, copied_ev]
    c.check_contents()


def test_pin_hot_by_hand(lib):
    c = Cache(lib, E=6, slots=4)
    for _ in range(3):                              # prefetches do not count as usage
        assert c.ensure({4}, prefetch=True)[0] == OK
    for req in ({0, 1}, {1, 2}, {1, 3}, {2, 5}):    # 3 evicts 4, then 5 evicts 0
        assert c.ensure(req)[0] == OK
    assert list(c.owners()) == [3, 5, 1, 2]
    # usage: 1 -> 3, 2 -> 2, 0/3/5 -> 1, 4 -> 0
    st, ops = c.pin_hot(2, 2)                       # {1, 2}: resident already
    assert st == OK and kinds(ops) == [RECORD]
    assert sorted(np.flatnonzero(c.pinned())) == [1, 2]
    st, ops = c.pin_hot(3, 2)                       # 4 - 3 < 2 unpinned slots
    assert st == INVALID_ARG and len(ops) == 0
    assert sorted(np.flatnonzero(c.pinned())) == [1, 2]
    assert c.pin_hot(7, 0)[0] == INVALID_ARG        # more than E
    assert c.pin_hot(-1, 0)[0] == INVALID_ARG
    owners = list(c.owners())
    st, ops = c.pin_hot(3, 1)                       # {1, 2} + 0 (usage tie 0/3/5: lower id)
    assert st == OK
    # the victim is the least recently used slot not holding an expert being pinned: 3
    assert copies_of(c, ops) == [(0, owners.index(3))]
    assert sorted(np.flatnonzero(c.pinned())) == [0, 1, 2]
    # one unpinned slot left: a request for two unpinned, non-resident experts cannot fit
    free = [e for e in range(6) if c.slot_of()[e] < 0]
    assert c.ensure(set(free[:2]))[0] == UNSUPPORTED
    # releasing the pins
    assert c.pin_hot(0, 1)[0] == OK and not c.pinned().any()
    c.check_contents()


def test_runtime_failures_are_reported(lib):
    for k in (1, 2, 3):                             # the stream, then each event, fails
        lib.ch_fail_call(k)
        assert lib.ch_create(4, 2, UP, DN) == ERR_CUDA
    lib.ch_destroy()
    c = Cache(lib, E=8, slots=3)
    assert c.ensure({0})[0] == OK
    assert c.note_compute()[0] == OK
    for k, what in ((1, "fence"), (2, "gate/up copy"), (3, "down copy"), (4, "completion record")):
        lib.ch_fail_call(k)
        st, _ = c.ensure({1 + k})
        assert st == ERR_CUDA, what
    lib.ch_fail_call(1)
    assert c.note_compute()[0] == ERR_CUDA
    lib.ch_fail_call(1)
    assert c.wait_copies()[0] == ERR_CUDA
    lib.ch_fail_call(0)


def test_state_after_a_failed_load(lib):
    """A load whose fence fails changes nothing; one whose copy fails leaves the victim's
    slot free (its expert no longer resident, counted once as evicted), and the next
    request takes that free slot."""
    c = Cache(lib, E=8, slots=2)
    assert c.ensure({0})[0] == OK and c.ensure({1})[0] == OK
    assert c.note_compute()[0] == OK
    lib.ch_fail_call(1)                              # the fence
    st, ops = c.ensure({2})
    assert st == ERR_CUDA and COPY not in kinds(ops)
    assert list(c.owners()) == [0, 1] and c.stats()["evictions"] == 0
    lib.ch_fail_call(2)                              # the gate/up copy into slot 0 (expert 0, LRU)
    assert c.ensure({2})[0] == ERR_CUDA
    assert list(c.owners()) == [-1, 1] and c.stats()["evictions"] == 1
    st, ops = c.ensure({3})                          # the free slot, not the LRU expert 1
    assert st == OK and copies_of(c, ops) == [(3, 0)]
    assert list(c.owners()) == [3, 1] and c.stats()["evictions"] == 1
    lib.ch_fail_call(3)                              # the down copy into slot 1 (expert 1)
    assert c.ensure({4})[0] == ERR_CUDA
    assert list(c.owners()) == [3, -1] and c.stats()["evictions"] == 2
    st, ops = c.ensure({1})
    assert st == OK and copies_of(c, ops) == [(1, 1)]
    assert list(c.owners()) == [3, 1]
    c.check_contents()


# ---------------------------------------------------------------------------------------
# randomised sequences against the definitions


class Model:
    """What the test knows independently of the cache: request order (for recency), usage
    counts, the prefetched-and-unused flags, and which events the cache has shown."""

    def __init__(self, E):
        self.tick = 0
        self.last = np.zeros(E, np.int64)
        self.usage = np.zeros(E, np.int64)
        self.pref = np.zeros(E, bool)
        self.noted = False
        self.copied_ev = None
        self.computed_ev = None


def check_fence_and_record(c, m, ops, loaded):
    k = kinds(ops)
    waits = [i for i, x in enumerate(k) if x == WAIT]
    if loaded and m.noted:
        assert len(waits) == 1 and waits[0] < k.index(COPY)
        assert list(ops[waits[0], 1:3]) == [c.copy_stream, m.computed_ev]
    else:
        assert waits == []
    assert k.count(RECORD) == 1 and k[-1] == RECORD
    assert ops[-1, 1] == c.copy_stream
    if m.copied_ev is None:
        m.copied_ev = int(ops[-1, 2])
    assert ops[-1, 2] == m.copied_ev


def replay_loads(c, m, owner, loads, protected, pinned):
    """Checks each load's slot: the lowest free slot if any, else the least recently used
    slot whose expert is not protected (needed by the request) and not pinned, ties to the
    lower slot. Returns the evicted experts."""
    evicted = []
    for e, s in loads:
        free = [t for t in range(c.slots) if owner[t] < 0]
        if free:
            assert s == free[0], (e, s, free)
        else:
            cand = [t for t in range(c.slots) if not protected[owner[t]] and not pinned[owner[t]]]
            best = min(cand, key=lambda t: (m.last[owner[t]], t))
            assert s == best, (e, s, best, owner)
            evicted.append(int(owner[s]))
            m.pref[owner[s]] = False
        owner[s] = e
        m.last[e] = m.tick
    return evicted


def do_ensure(c, m, needed, prefetch):
    before_slot = c.slot_of()
    owner = c.owners()
    pinned = c.pinned()
    stats0 = c.stats()
    m.tick += 1
    st, ops = c.ensure(needed, prefetch)
    assert st == OK
    loads = copies_of(c, ops)
    missing = sorted(e for e in needed if before_slot[e] < 0)
    hits = sorted(e for e in needed if before_slot[e] >= 0)
    assert [e for e, _ in loads] == missing             # issued in expert order
    protected = np.zeros(c.E, bool)
    protected[list(needed)] = True
    evicted = replay_loads(c, m, owner, loads, protected, pinned)
    for e in hits:
        m.last[e] = m.tick
    pref_hits = 0
    if prefetch:
        m.pref[missing] = True
    else:
        m.usage[list(needed)] += 1
        pref_hits = int(m.pref[hits].sum())
        m.pref[hits] = False
    assert list(c.owners()) == list(owner)
    check_fence_and_record(c, m, ops, loads)
    s1 = c.stats()
    d = {k: s1[k] - stats0[k] for k in STATS}
    assert d == dict(hits=0 if prefetch else len(hits), misses=0 if prefetch else len(missing),
                     prefetched=len(missing) if prefetch else 0, prefetch_hits=pref_hits,
                     bytes_h2d=len(loads) * (UP + DN), evictions=len(evicted)), d


def do_pin(c, m, n, min_free):
    before_slot = c.slot_of()
    owner = c.owners()
    pinned0 = c.pinned()
    stats0 = c.stats()
    st, ops = c.pin_hot(n, min_free)
    if n < 0 or n > c.E or c.slots - n < min_free:
        assert st == INVALID_ARG and len(ops) == 0
        assert list(c.pinned()) == list(pinned0)
        return
    m.tick += 1
    assert st == OK
    want = sorted(range(c.E), key=lambda e: (-m.usage[e], e))[:n]
    loads = copies_of(c, ops)
    assert [e for e, _ in loads] == sorted(e for e in want if before_slot[e] < 0)
    protected = np.zeros(c.E, bool)
    protected[want] = True
    evicted = replay_loads(c, m, owner, loads, protected, np.zeros(c.E, bool))
    assert list(c.owners()) == list(owner)
    assert sorted(np.flatnonzero(c.pinned()).tolist()) == sorted(want)
    check_fence_and_record(c, m, ops, loads)
    s1 = c.stats()
    assert s1["bytes_h2d"] - stats0["bytes_h2d"] == len(loads) * (UP + DN)
    assert s1["evictions"] - stats0["evictions"] == len(evicted)
    for k in ("hits", "misses", "prefetched", "prefetch_hits"):
        assert s1[k] == stats0[k]


@pytest.mark.parametrize("E,slots,seed", [(16, 6, 0), (40, 12, 1), (9, 9, 2), (64, 5, 3)])
def test_random_sequences(lib, E, slots, seed):
    rng = np.random.default_rng(seed)
    c = Cache(lib, E, slots)
    m = Model(E)
    for it in range(500):
        r = rng.random()
        pinned = c.pinned()
        if r < 0.6:
            room = slots - int(pinned.sum())
            unp = np.flatnonzero(~pinned)
            k = int(rng.integers(1, min(room, len(unp)) + 1)) if room > 0 else 0
            needed = set(rng.choice(unp, size=k, replace=False).tolist()) if k else set()
            pin_ids = np.flatnonzero(pinned)
            if len(pin_ids):
                needed |= set(rng.choice(pin_ids, size=int(rng.integers(0, len(pin_ids) + 1)),
                                         replace=False).tolist())
            if not needed:
                continue
            do_ensure(c, m, needed, prefetch=r < 0.15)
        elif r < 0.8:
            st, ops = c.note_compute()
            assert st == OK and kinds(ops) == [RECORD] and ops[0, 1] == c.compute_stream
            if m.computed_ev is None:
                m.computed_ev = int(ops[0, 2])
            assert ops[0, 2] == m.computed_ev and ops[0, 2] != m.copied_ev
            m.noted = True
        elif r < 0.9:
            if m.copied_ev is None:
                continue
            st, ops = c.wait_copies()
            assert st == OK and kinds(ops) == [WAIT]
            assert list(ops[0, 1:3]) == [c.compute_stream, m.copied_ev]
        else:
            do_pin(c, m, int(rng.integers(-1, slots + 2)), int(rng.integers(0, 4)))
        # invariants after every call
        slot = c.slot_of()
        assert np.all(slot[c.pinned()] >= 0)
        c.check_contents()
    # with a slot for every expert nothing is ever evicted; otherwise eviction is exercised
    assert (c.stats()["evictions"] > 0) == (E > slots)
