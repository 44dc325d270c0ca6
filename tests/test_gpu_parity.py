"""GPU parity: the CUDA path against the CPU oracle, byte for byte, over every
replica's whole cache buffer plus 4 KiB red zones on both sides.

Covers the five workloads, hand-derived rows (NaN, Inf, ties, saturation,
subnormals), every bf16 value through the encoder at scale 1, scales from
2^-40 to 2^40, strided input views, padded and invalid slots, 1..8
replicas (8 also on the capacity workload), ragged batch sizes, batches on
both sides of the launch-shape switch (SMs x 8 rows), byte offsets beyond
2^31, the gather-then-insert path, the fused store+epoch launch, and the
failure statuses.
Sources: "[Kernel][PCP] Publish replicated KV updates through PyTorch
symmetric memory", Correctness and current-head validation (fp8_ds_mla,
padded and invalid slots, guard bytes, byte-exact against gather-then-
insert).
"""

import numpy as np
import pytest
import torch

import hand_rows
import oracle
from gpu_util import Caches, DevInputs, assert_matches_oracle, bf16, oracle_caches, run_store
from replication_token_warp_gb300 import build as kbuild
from replication_token_warp_gb300 import inputs, kvpub

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_device):
    kbuild.build()
    kvpub.lib()
    return cuda_device


def workload(name, lat, rope, idx, slots, R, nb):
    return inputs.Workload(name, np.ascontiguousarray(lat, np.uint16),
                           np.ascontiguousarray(rope, np.uint16),
                           np.ascontiguousarray(idx, np.uint16),
                           np.ascontiguousarray(slots, np.int64), R, nb)


@pytest.mark.parametrize("index", [0, 1, 2, 4])
@pytest.mark.parametrize("path", ["fused", "gather", "publish"])
def test_workloads_match_oracle(dev, index, path):
    w = inputs.make(index)
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    c = run_store(w, dev, path, invalid_count=cnt)
    want_main, want_idx, n, inv = oracle_caches(w)
    assert_matches_oracle(c, want_main, want_idx)
    assert int(cnt.item()) == inv == 0


@pytest.mark.parametrize("layer", [0, 29, 60])
def test_prefill_layers_match_oracle(dev, layer):
    w = inputs.make(3, layer=layer)
    c = run_store(w, dev, "fused")
    assert_matches_oracle(c, *oracle_caches(w)[:2])


def test_hand_rows(dev):
    rows = hand_rows.load()["rows"]
    lat = np.stack([hand_rows.build_bf16(r["latent"], 512) for r in rows])
    rope = np.stack([hand_rows.build_bf16(r["rope"], 64) for r in rows])
    idx = np.stack([hand_rows.build_bf16(r["index_k"], 128) for r in rows])
    slots = np.array([r["slot"] for r in rows], np.int64)
    w = workload("hand", lat, rope, idx, slots, 2, 4)
    for path in ("fused", "gather"):
        c = run_store(w, dev, path)
        assert_matches_oracle(c, *oracle_caches(w)[:2])
    # and against the hand-written expectation directly
    c = run_store(w, dev, "fused")
    main, ixc = c.host()
    for r, row in enumerate(rows):
        s = row["slot"]
        body = main[0][4096:-4096]
        want = hand_rows.build_codes(row["expect"]["latent_codes"], 512)
        assert np.array_equal(body[s * 656:s * 656 + 512], want)


def test_every_bf16_value_at_scale_one(dev):
    """Tiles whose amax is 448 have scale exactly 1, so each code is the
    E4M3 conversion of the value itself: all bf16 values with |x| <= 448."""
    pos = np.arange(0x0000, 0x43E1, dtype=np.uint16)       # 0 .. 448
    vals = np.concatenate([pos, pos | 0x8000])
    per_tile = 127
    n_tiles = -(-vals.size // per_tile)
    vals = np.concatenate([vals, np.zeros(n_tiles * per_tile - vals.size, np.uint16)])
    tiles = np.concatenate([np.full((n_tiles, 1), 0x43E0, np.uint16),     # 448
                            vals.reshape(n_tiles, per_tile)], axis=1)
    n_rows = -(-n_tiles // 5)
    tiles = np.concatenate([tiles, np.tile(tiles[:1], (n_rows * 5 - n_tiles, 1))])
    rows = tiles.reshape(n_rows, 5 * 128)
    lat, idx = rows[:, :512], rows[:, 512:]
    rope = np.arange(n_rows * 64, dtype=np.uint16).reshape(n_rows, 64)
    w = workload("all-bf16", lat, rope, idx, np.arange(n_rows) * 3 + 1, 1, -(-n_rows * 3 // 64) + 1)
    c = run_store(w, dev, "fused")
    assert_matches_oracle(c, *oracle_caches(w)[:2])


def test_scales_across_the_exponent_range(dev):
    """Row magnitudes log-uniform in [2^-40, 2^40] with random signs, some
    single-element outliers and some sub-floor rows."""
    rng = np.random.default_rng(11)
    T, nb = 4099, 80
    def block(cols):
        mag = np.exp2(rng.uniform(-40, 40, size=(T, 1))) * rng.standard_normal((T, cols))
        x = torch.from_numpy(mag.astype(np.float32))
        return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    lat, rope, idx = block(512), block(64), block(128)
    lat[::7, 5] = 0x7F7F                                    # bf16 near its max
    idx[::11, 100] = 0x0001                                 # bf16 subnormal
    slots = rng.permutation(nb * 64)[:T]
    slots[::13] = -1
    w = workload("scales", lat, rope, idx, slots, 3, nb)
    for path in ("fused", "gather"):
        c = run_store(w, dev, path)
        assert_matches_oracle(c, *oracle_caches(w)[:2])


def test_strided_input_views(dev):
    w = inputs.make(1)
    T = w.num_tokens
    kv = torch.zeros(T, 576, dtype=torch.bfloat16, device=dev)
    kv[:, :512] = bf16(w.kv_latent, dev)
    kv[:, 512:] = bf16(w.k_rope, dev)
    ik = torch.zeros(T, 136, dtype=torch.bfloat16, device=dev)
    ik[:, :128] = bf16(w.index_k, dev)
    c = Caches(2, w.num_blocks, w.guard, dev)
    kvpub.store_mla_fp8(kv[:, :512], kv[:, 512:], ik[:, :128],
                        torch.from_numpy(w.slot_mapping).to(dev), c.main, c.idx)
    torch.cuda.synchronize()
    assert_matches_oracle(c, *oracle_caches(w)[:2])


def test_padded_and_invalid_slots(dev):
    w = inputs.make(2)
    slots = w.slot_mapping.copy()
    cap = w.num_blocks * 64
    rng = np.random.default_rng(5)
    pos = rng.choice(np.nonzero(slots >= 0)[0], 300, replace=False)
    slots[pos[:100]] = cap + rng.integers(0, 10 ** 6, 100)
    slots[pos[100:200]] = -rng.integers(2, 10 ** 9, 100)
    slots[pos[200:]] = -1
    w.slot_mapping = slots
    for path in ("fused", "gather", "publish"):
        cnt = torch.zeros(1, dtype=torch.int64, device=dev)
        c = run_store(w, dev, path, invalid_count=cnt)
        want_main, want_idx, n, inv = oracle_caches(w)
        assert inv == 200 and int(cnt.item()) == 200
        assert_matches_oracle(c, want_main, want_idx)


@pytest.mark.parametrize("R", [1, 2, 3, 5, 6, 7, 8])
@pytest.mark.parametrize("T", [1, 31, 777])
def test_replica_counts_and_ragged_batches(dev, R, T):
    w = inputs.random_rows(seed=100 + R * 10 + T, num_tokens=T, num_blocks=16,
                           num_replicas=R, pad_fraction=0.1)
    c = run_store(w, dev, "fused")
    assert_matches_oracle(c, *oracle_caches(w)[:2])


def _switch_rows(dev):
    # launches of fewer rows than this take 2-warp blocks, the rest 8-warp blocks
    return torch.cuda.get_device_properties(dev).multi_processor_count * 8


@pytest.mark.parametrize("path", ["fused", "gather", "publish"])
@pytest.mark.parametrize("delta", [-1, 0, 1])
def test_batches_on_both_sides_of_the_block_size_switch(dev, path, delta):
    T = _switch_rows(dev) + delta
    w = inputs.random_rows(seed=300 + delta, num_tokens=T, num_blocks=32, num_replicas=3,
                           pad_fraction=0.05)
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    c = run_store(w, dev, path, invalid_count=cnt)
    assert_matches_oracle(c, *oracle_caches(w)[:2])
    assert int(cnt.item()) == 0


def test_capacity_workload_into_eight_replicas(dev):
    """The capacity workload (706,624-slot caches, random slots) with the
    maximum replica count instead of 4: 8 x 556 MB of caches, all byte-exact."""
    w = inputs.make(4)
    w.num_replicas = 8
    c = run_store(w, dev, "fused")
    assert_matches_oracle(c, *oracle_caches(w)[:2])


def test_empty_and_all_padded(dev):
    w = inputs.make(1)
    c = Caches(2, w.num_blocks, w.guard, dev)
    e = torch.empty(0, 512, dtype=torch.bfloat16, device=dev)
    kvpub.store_mla_fp8(e, e[:, :64], e[:, :128], torch.empty(0, dtype=torch.int64, device=dev),
                        c.main, c.idx)
    w.slot_mapping = np.full(w.num_tokens, -1, np.int64)
    x = DevInputs(w, dev)
    kvpub.store_mla_fp8(x.lat, x.rope, x.idx, x.slots, c.main, c.idx)
    epoch = torch.zeros(1, dtype=torch.int64, device=dev)
    done = torch.zeros(1, dtype=torch.int32, device=dev)
    kvpub.store_mla_fp8_publish(x.lat, x.rope, x.idx, x.slots, c.main, c.idx, epoch, done)
    kvpub.store_mla_fp8_publish(e, e[:, :64], e[:, :128],
                                torch.empty(0, dtype=torch.int64, device=dev),
                                c.main, c.idx, epoch, done)
    torch.cuda.synchronize()
    assert int(epoch.item()) == 2 and int(done.item()) == 0
    main, idx = c.host()
    assert all(np.all(b == w.guard) for b in main + idx)


def test_byte_offsets_beyond_2_pow_31(dev):
    """Slots whose Main row starts past 2 GiB: rows land where the oracle puts
    them and nothing else in the 2.6 GB buffer changes."""
    nb = 62_000                                   # 62,000 * 64 * 656 B = 2.6 GB
    top = nb * 64
    w = inputs.random_rows(seed=9, num_tokens=64, num_blocks=1)
    w.slot_mapping = np.arange(top - 64, top, dtype=np.int64)[::-1].copy()
    w.slot_mapping[::9] = -1
    x = DevInputs(w, dev)
    main = torch.full((nb * 64 * 656,), 0xA5, dtype=torch.uint8, device=dev)
    ixc = torch.full((nb * 8448,), 0xA5, dtype=torch.uint8, device=dev)
    kvpub.store_mla_fp8(x.lat, x.rope, x.idx, x.slots, [main], [ixc])
    torch.cuda.synchronize()
    # oracle on a one-block cache: slot s -> s - (top - 64)
    small = w.slot_mapping - (top - 64)
    small[w.slot_mapping < 0] = -1
    om, oi = oracle.new_caches(1, 1)
    oracle.store_mla_fp8(w.kv_latent, w.k_rope, w.index_k, small, om, oi, 1)
    tail_main = main[(top - 64) * 656:].cpu().numpy()
    tail_idx = ixc[(nb - 1) * 8448:].cpu().numpy()
    assert np.array_equal(tail_main, om[0]) and np.array_equal(tail_idx, oi[0])
    assert int((main[:(top - 64) * 656] != 0xA5).sum().item()) == 0
    assert int((ixc[:(nb - 1) * 8448] != 0xA5).sum().item()) == 0


def _mixed_batch():
    """One batch of contiguous prefill runs interleaved, in chunks of 256 rows, with scattered
    slots, some of them sharing a Main half-sector or an Indexer-scale sector with the end of a
    run (each request's run ends at block offset 40, so offsets 41 and 43 are free), plus padded
    and invalid entries."""
    nb, R = 2048, 3
    a = inputs.prefill_batch(901, 6, 1001, nb, R)
    ends = a.slot_mapping.reshape(6, 1001)[:, -1]
    # the cache's first and last slot too: their part-written sectors are the
    # first and last ones of the buffers
    edges = np.setdiff1d([0, 1, nb * 64 - 2, nb * 64 - 1], a.slot_mapping)
    shared = np.concatenate([ends + 1, ends + 3, edges])
    free = np.setdiff1d(np.arange(nb * 64), np.concatenate([a.slot_mapping, shared]))
    rng = np.random.default_rng(902)
    b_slots = np.concatenate([shared, rng.choice(free, 6000 - shared.size, replace=False)])
    b = inputs.random_rows(903, b_slots.size, nb, R)
    chunks_a = np.array_split(np.arange(a.num_tokens), a.num_tokens // 256)
    chunks_b = np.array_split(np.arange(b_slots.size), b_slots.size // 256)
    parts = []
    for ca, cb in zip(chunks_a, chunks_b):
        parts.append(("a", ca))
        parts.append(("b", cb))
    def take(name):
        xa = getattr(a, name)
        xb = b_slots if name == "slot_mapping" else getattr(b, name)
        return np.concatenate([(xa if w == "a" else xb)[idx] for w, idx in parts])
    slots = take("slot_mapping")
    pad = rng.choice(slots.size, 70, replace=False)
    slots[pad[:50]] = -1
    slots[pad[50:]] = nb * 64 + np.arange(20) * 977
    return workload("mixed", take("kv_latent"), take("k_rope"), take("index_k"), slots, R, nb)


@pytest.mark.parametrize("path", ["fused", "publish", "gather"])
def test_contiguous_runs_and_scattered_slots_in_one_launch(dev, path):
    """Warps whose first row sits in a contiguous run leave the part-sector prefetch off, the
    others turn it on; some scattered slots share a sector with a run's last row, so two warps
    (one prefetching) write the two parts of one sector in the same launch."""
    w = _mixed_batch()
    assert w.num_tokens >= 8 * torch.cuda.get_device_properties(dev).multi_processor_count
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    c = run_store(w, dev, path, invalid_count=cnt)
    want_main, want_idx, _, inv = oracle_caches(w)
    assert inv == 20
    assert_matches_oracle(c, want_main, want_idx)
    assert int(cnt.item()) == inv


def test_gather_equals_fused_on_prefill(dev):
    w = inputs.make(2)
    a = run_store(w, dev, "fused")
    b = run_store(w, dev, "gather")
    for x, y in zip(a.main_full + a.idx_full, b.main_full + b.idx_full):
        assert torch.equal(x, y)


def test_publish_advances_epoch_once_per_call(dev):
    w = inputs.make(1)
    x = DevInputs(w, dev)
    c = Caches(2, w.num_blocks, w.guard, dev)
    epoch = torch.full((1,), 41, dtype=torch.int64, device=dev)
    done = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(5):
        kvpub.store_mla_fp8_publish(x.lat, x.rope, x.idx, x.slots, c.main, c.idx, epoch, done)
    torch.cuda.synchronize()
    assert int(epoch.item()) == 46 and int(done.item()) == 0
    assert_matches_oracle(c, *oracle_caches(w)[:2])


def test_epoch_wait_reached_and_timeout(dev):
    epoch = torch.zeros(1, dtype=torch.int64, device=dev)
    status = torch.full((1,), 7, dtype=torch.int32, device=dev)
    kvpub.epoch_advance(epoch)
    kvpub.epoch_advance(epoch)
    kvpub.epoch_wait(epoch, 2, 1000, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # nothing will ever advance it to 3: the wait gives up and says so
    kvpub.epoch_wait(epoch, 3, 1000, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1 and int(epoch.item()) == 2


def test_failures_change_nothing(dev):
    w = inputs.make(0)
    x = DevInputs(w, dev)
    c = Caches(1, w.num_blocks, w.guard, dev)
    lib = kvpub.lib()
    import ctypes
    mains = (ctypes.c_void_p * 1)(c.main[0].data_ptr())
    idxs = (ctypes.c_void_p * 1)(c.idx[0].data_ptr())
    base = [x.lat.data_ptr(), 512, x.rope.data_ptr(), 64, x.idx.data_ptr(), 128,
            x.slots.data_ptr(), w.num_tokens, mains, idxs, 1, w.num_blocks, 64, None]
    bad = [(0, x.lat.data_ptr() + 2, 2), (1, 516, 2), (1, 504, 1), (10, 0, 1), (10, 9, 3), (12, 16, 1),
           (7, -5, 1), (13, x.slots.data_ptr() + 4, 2)]
    for i, v, st in bad:
        args = list(base)
        args[i] = v
        if i == 10 and v == 9:
            args[8] = (ctypes.c_void_p * 9)(*([c.main[0].data_ptr()] * 9))
            args[9] = (ctypes.c_void_p * 9)(*([c.idx[0].data_ptr()] * 9))
        assert lib.kvpub_store_mla_fp8(*args, None) == st
    torch.cuda.synchronize()
    main, idx = c.host()
    assert np.all(main[0] == w.guard) and np.all(idx[0] == w.guard)


def test_store_sees_the_producer_kernel_that_precedes_it(dev):
    """Every kernel here may be scheduled early (programmatic dependent
    launch) but waits for the previous kernel on the stream before touching
    memory.  A torch kernel rewrites the input rows right before each store;
    the stores must see the new rows, round after round."""
    ws = [inputs.random_rows(seed=900 + k, num_tokens=2048, num_blocks=40, num_replicas=2)
          for k in range(3)]
    slots = ws[0].slot_mapping
    for w in ws:
        w.slot_mapping = slots
    src = [DevInputs(w, dev) for w in ws]
    x = DevInputs(ws[0], dev)
    c = Caches(2, ws[0].num_blocks, ws[0].guard, dev)
    for rnd in range(6):
        w, y = ws[rnd % 3], src[rnd % 3]
        x.lat.copy_(y.lat)
        x.rope.copy_(y.rope)
        x.idx.copy_(y.idx)
        kvpub.store_mla_fp8(x.lat, x.rope, x.idx, x.slots, c.main, c.idx)
        torch.cuda.synchronize()
        assert_matches_oracle(c, *oracle_caches(w)[:2])


def test_large_batch_matches_oracle(dev):
    """131,072 rows (128 prefill requests x 1,024 tokens) into 4 replicas of
    8,192-block caches: many rows per warp, the whole buffers byte-exact."""
    w = inputs.prefill_batch(1000, 128, 1024, 8192)
    c = run_store(w, dev, "fused")
    assert_matches_oracle(c, *oracle_caches(w)[:2])


def test_concurrent_host_threads_on_separate_streams(dev):
    """Four host threads, each with its own CUDA stream and caches, publish
    different batches at the same time; the library's cached launch geometry
    and thread-local error state must not mix them up."""
    import threading
    ws = [inputs.random_rows(seed=700 + k, num_tokens=3000, num_blocks=60, num_replicas=2,
                             pad_fraction=0.05) for k in range(4)]
    xs = [DevInputs(w, dev) for w in ws]
    cs = [Caches(2, w.num_blocks, w.guard, dev) for w in ws]
    streams = [torch.cuda.Stream(device=dev) for _ in ws]
    torch.cuda.synchronize()
    errors = []

    def worker(k):
        try:
            with torch.cuda.stream(streams[k]):
                for _ in range(20):
                    kvpub.store_mla_fp8(xs[k].lat, xs[k].rope, xs[k].idx, xs[k].slots,
                                        cs[k].main, cs[k].idx)
                    # a failing call on this thread must not disturb the others
                    assert kvpub.lib().kvpub_epoch_advance(None, None) == 1
                    assert "epoch" in kvpub.last_error()
        except Exception as e:      # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for w, c in zip(ws, cs):
        assert_matches_oracle(c, *oracle_caches(w)[:2])


def test_prepared_calls_match_the_plain_calls(dev):
    """Calls prepared once (arguments marshalled up front) leave the same
    bytes and advance the epoch the same way as the plain calls."""
    w = inputs.make(2)
    x = DevInputs(w, dev)
    c = Caches(4, w.num_blocks, w.guard, dev)
    c2 = Caches(4, w.num_blocks, w.guard, dev)
    epoch = torch.zeros(1, dtype=torch.int64, device=dev)
    done = torch.zeros(1, dtype=torch.int32, device=dev)
    store = kvpub.prepare_store_mla_fp8(x.lat, x.rope, x.idx, x.slots, c.main, c.idx)
    advance = kvpub.prepare_epoch_advance(epoch)
    publish = kvpub.prepare_store_mla_fp8_publish(x.lat, x.rope, x.idx, x.slots, c2.main, c2.idx,
                                                  epoch, done)
    for _ in range(3):
        store()
        advance()
        publish()
    torch.cuda.synchronize()
    assert int(epoch.item()) == 6 and int(done.item()) == 0
    want = oracle_caches(w)[:2]
    assert_matches_oracle(c, *want)
    assert_matches_oracle(c2, *want)
