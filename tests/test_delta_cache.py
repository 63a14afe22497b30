"""Delta cache policy on the CPU (host-arena mode of bd_cache: the arena is host
memory and loads are memcpy, no CUDA call): residency, the request-rate-weighted
LRU eviction rule, pinning, references, first-fit arena reuse with coalescing,
single-flight under concurrent acquires, synthetic Zipf traces, errors.

Source: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU" (Hanzo
blog), "Détails d'infrastructure" (cold start, rate-weighted LRU, pinning,
single-flight routing).  The eviction rule is the reading the library states:
rate += 1 per request, halving every half-life; evict the unpinned, unused
resident variant with the lowest decayed rate, the least recently requested on
ties."""
import ctypes
import threading

import numpy as np
import pytest
import torch

from bit_delta_tenant_gb300 import bitdelta as bd
from bit_delta_tenant_gb300 import synth

BLOCK = 4096  # bits bytes per test variant; alpha 256 bytes -> 4352-byte blocks


def make_cache(n_blocks, max_variants=16, half_life=10.0, block=BLOCK):
    arena = torch.zeros(n_blocks * (block + 256), dtype=torch.uint8)
    # the arena must be 256-byte aligned: over-allocate and slice
    raw = torch.zeros(arena.numel() + 256, dtype=torch.uint8)
    off = (-raw.data_ptr()) % 256
    arena = raw[off:off + n_blocks * (block + 256)]
    cache = bd.DeltaCache(max_variants, arena, half_life_s=half_life, host_arena=True)
    cache._raw = raw
    return cache, arena


def host_delta(v, block=BLOCK):
    g = np.random.default_rng(1000 + v)
    bits = torch.from_numpy(g.integers(0, 256, block, dtype=np.uint8))
    alpha = torch.tensor([1e-3 * (v + 1)], dtype=torch.float32)
    return bits, alpha


def register_all(cache, n, block=BLOCK):
    deltas = [host_delta(v, block) for v in range(n)]
    for v, (b, a) in enumerate(deltas):
        cache.register(v, b, a)
    return deltas


def read(ptr, n, dtype=np.uint8):
    return np.ctypeslib.as_array(ctypes.cast(ptr, ctypes.POINTER(np.ctypeslib.as_ctypes_type(dtype))), (n,)).copy()


def use(cache, v, t):
    rc, b, a = cache.acquire(v, now_s=t)
    assert rc == bd.BD_OK, rc
    assert cache.release(v) == bd.BD_OK
    return b, a


def test_load_contents_and_hit():
    cache, _ = make_cache(4)
    deltas = register_all(cache, 3)
    rc, b, a = cache.acquire(1, now_s=0.0)
    assert rc == bd.BD_OK and b % 256 == 0 and a % 256 == 0
    assert np.array_equal(read(b, BLOCK), deltas[1][0].numpy())
    assert read(a, 1, np.float32)[0] == np.float32(2e-3)
    assert cache.release(1) == bd.BD_OK
    rc, b2, _ = cache.acquire(1, now_s=1.0)
    assert rc == bd.BD_OK and b2 == b
    cache.release(1)
    st = cache.stats()
    assert (st.acquires, st.hits, st.misses, st.loads, st.evictions) == (2, 1, 1, 1, 0)
    assert st.bytes_loaded == BLOCK + 4 and st.resident == 1 and st.in_use == 0


def test_evicts_lowest_decayed_rate_not_just_oldest():
    # room for two deltas; 0 is requested often long ago, 1 once recently
    cache, _ = make_cache(2, half_life=10.0)
    register_all(cache, 3)
    for t in (0.0, 0.1, 0.2, 0.3, 0.4):
        use(cache, 0, t)          # rate 5 at t = 0.4
    use(cache, 1, 5.0)            # rate 1 at t = 5
    # at t = 6: rate(0) = 5 * 2^(-5.6/10) ~ 3.4, rate(1) = 2^(-0.1) ~ 0.93 -> evict 1 (plain LRU would evict 0)
    use(cache, 2, 6.0)
    assert cache.is_resident(0) and not cache.is_resident(1) and cache.is_resident(2)
    # much later the old burst has decayed below a single recent request: 0 goes
    use(cache, 1, 80.0)           # evicts the lower of rate(0)~0.02 and rate(2)~0.008 -> 2
    assert cache.is_resident(0) and cache.is_resident(1) and not cache.is_resident(2)
    use(cache, 2, 81.0)           # rate(0) ~ 0.02 < rate(1) ~ 0.93
    assert not cache.is_resident(0) and cache.is_resident(1) and cache.is_resident(2)


def test_ties_go_to_least_recently_requested():
    cache, _ = make_cache(2, half_life=1e9)  # no decay: equal rates
    register_all(cache, 3)
    use(cache, 0, 1.0)
    use(cache, 1, 2.0)
    use(cache, 2, 3.0)
    assert not cache.is_resident(0) and cache.is_resident(1) and cache.is_resident(2)


def test_pinned_and_in_use_are_never_evicted():
    cache, _ = make_cache(2)
    register_all(cache, 4)
    cache.set_pinned(0, True)
    use(cache, 0, 0.0)
    rc, _, _ = cache.acquire(1, now_s=1.0)      # held
    assert rc == bd.BD_OK
    rc, _, _ = cache.acquire(2, now_s=2.0)      # nothing evictable
    assert rc == bd.BD_ERR_NO_SPACE
    assert cache.release(1) == bd.BD_OK
    rc, _, _ = cache.acquire(2, now_s=3.0)      # now 1 goes
    assert rc == bd.BD_OK
    assert cache.is_resident(0) and not cache.is_resident(1) and cache.is_resident(2)
    cache.release(2)
    cache.set_pinned(0, False)
    use(cache, 3, 100.0)                        # 0's rate has decayed most
    assert not cache.is_resident(0)


def test_arena_reuse_coalesces_free_blocks():
    # a large delta needs the space of two small ones that were evicted
    cache, _ = make_cache(3, block=BLOCK)
    small = [host_delta(v) for v in range(3)]
    for v, (b, a) in enumerate(small):
        cache.register(v, b, a)
    g = np.random.default_rng(7)
    big_bits = torch.from_numpy(g.integers(0, 256, 2 * BLOCK + 256, dtype=np.uint8))
    cache.register(3, big_bits, torch.tensor([0.5], dtype=torch.float32))
    for v in range(3):
        use(cache, v, float(v))
    rc, b, a = cache.acquire(3, now_s=10.0)
    assert rc == bd.BD_OK
    assert np.array_equal(read(b, big_bits.numel()), big_bits.numpy())
    st = cache.stats()
    assert st.evictions == 2 and st.resident == 2      # blocks 0 and 1 merged, delta 2 kept
    assert not cache.is_resident(0) and not cache.is_resident(1) and cache.is_resident(2)
    cache.release(3)


def test_single_flight_under_concurrent_acquires():
    cache, _ = make_cache(4)
    deltas = register_all(cache, 2)
    out = []
    barrier = threading.Barrier(8)

    def worker():
        barrier.wait()
        rc, b, _ = cache.acquire(1)
        out.append((rc, b))
        cache.release(1)

    ts = [threading.Thread(target=worker) for _ in range(8)]
    [t.start() for t in ts]
    [t.join() for t in ts]
    assert all(rc == bd.BD_OK for rc, _ in out) and len({b for _, b in out}) == 1
    st = cache.stats()
    assert st.loads == 1 and st.misses == 1 and st.hits == 7 and st.in_use == 0
    assert np.array_equal(read(out[0][1], BLOCK), deltas[1][0].numpy())


def test_zipf_trace_accounting_and_pinned_hot_variant():
    # 14 variants, room for 6; Zipf(1.1) request stream like the page's traffic
    cache, _ = make_cache(6, max_variants=14, half_life=50.0)
    register_all(cache, 14)
    cache.set_pinned(0, True)
    ids = synth.zipf_ids(4000, 14, 1.1, seed=9)
    for i, v in enumerate(ids):
        use(cache, int(v), float(i) * 0.01)
    st = cache.stats()
    assert st.acquires == 4000 and st.hits + st.misses == 4000
    assert st.loads == st.misses and st.evictions == st.loads - st.resident
    assert st.resident <= 6 and cache.is_resident(0)
    # hot variants stay resident: far fewer loads than requests
    assert st.hits / st.acquires > 0.7


def test_errors():
    cache, _ = make_cache(2)
    b, a = host_delta(0)
    cache.register(0, b, a)
    with pytest.raises(bd.BitDeltaError):
        cache.register(0, b, a)                          # twice
    assert cache.acquire(5)[0] == bd.BD_ERR_BAD_VARIANT_ID   # not registered
    assert cache.acquire(99)[0] == bd.BD_ERR_BAD_VARIANT_ID  # out of range
    assert cache.release(0) == bd.BD_ERR_INVALID_ARG     # not acquired
    huge = torch.zeros(10 * BLOCK, dtype=torch.uint8)
    with pytest.raises(bd.BitDeltaError):
        cache.register(1, huge, a)                       # larger than the arena
    lib = bd.load_library()
    assert lib.bd_cache_state_size(0) == 0
    state = ctypes.create_string_buffer(64)
    h = ctypes.c_void_p()
    arena = torch.zeros(4096, dtype=torch.uint8)
    assert lib.bd_cache_create(ctypes.addressof(state), 64, 4, ctypes.c_void_p(arena.data_ptr()), 4096, 1.0, 1,
                               ctypes.byref(h)) == bd.BD_ERR_WORKSPACE
