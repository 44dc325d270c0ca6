"""The 61-layer prefill (4 requests x 3,584 tokens per layer, 4 replicas, a
separate 1,024-block cache per layer) captured in one CUDA graph and
replayed 10 times.

The device epoch must advance on every replay ("[Perf][PCP] Fuse direct-KV
publication fence", Motivation: a host-side epoch cannot advance inside a
replayed graph; its summary: the replay test checks the epoch on every
replay).  After the replays, every layer's four replicas must equal the
oracle byte for byte, red zones included.
"""

import os

import numpy as np
import pytest
import torch

from gpu_util import Caches, assert_matches_oracle, bf16, oracle_caches
from replication_token_warp_gb300 import build as kbuild
from replication_token_warp_gb300 import inputs, kvpub

pytestmark = pytest.mark.gpu

LAYERS = 61
REPLAYS = 10


@pytest.fixture(scope="module")
def dev(cuda_device):
    kbuild.build()
    kvpub.lib()
    return cuda_device


@pytest.fixture(scope="module")
def layers():
    slots = inputs.layer_slot_mapping()
    return slots, [inputs.prefill_layer(layer, slots) for layer in range(LAYERS)]


def _device_layers(layers, dev):
    slots, ws = layers
    d_slots = torch.from_numpy(slots).to(dev)
    xs = [(bf16(w.kv_latent, dev), bf16(w.k_rope, dev), bf16(w.index_k, dev)) for w in ws]
    caches = [Caches(4, 1024, inputs.GUARD_BYTE, dev) for _ in range(LAYERS)]
    return d_slots, xs, caches


def _check_epoch_per_replay(g, epoch, per_replay):
    start = int(epoch.item())
    for k in range(1, REPLAYS + 1):
        g.replay()
        torch.cuda.synchronize()
        assert int(epoch.item()) == start + k * per_replay


@pytest.mark.parametrize("variant", ["store_then_advance", "fused_publish"])
def test_graph_replay_advances_epoch_and_matches_oracle(dev, layers, variant):
    d_slots, xs, caches = _device_layers(layers, dev)
    epoch = torch.zeros(1, dtype=torch.int64, device=dev)
    done = torch.zeros(1, dtype=torch.int32, device=dev)
    scratch_epoch = torch.zeros(1, dtype=torch.int64, device=dev)

    def step(ep):
        for layer in range(LAYERS):
            lat, rope, idx = xs[layer]
            c = caches[layer]
            if variant == "store_then_advance":
                kvpub.store_mla_fp8(lat, rope, idx, d_slots, c.main, c.idx)
                kvpub.epoch_advance(ep)
            else:
                kvpub.store_mla_fp8_publish(lat, rope, idx, d_slots, c.main, c.idx, ep, done)

    # one eager pass loads the kernels before capture (the store is idempotent)
    step(scratch_epoch)
    torch.cuda.synchronize()
    assert int(scratch_epoch.item()) == LAYERS

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(epoch)
    torch.cuda.synchronize()
    assert int(epoch.item()) == 0              # capture runs nothing
    _check_epoch_per_replay(g, epoch, LAYERS)
    assert int(epoch.item()) == LAYERS * REPLAYS == 610
    assert int(done.item()) == 0

    check = range(LAYERS) if variant == "store_then_advance" else (0, 30, 60)
    _, ws = layers
    for layer in check:
        want_main, want_idx, _, _ = oracle_caches(ws[layer])
        assert_matches_oracle(caches[layer], want_main, want_idx)
    del caches, xs
    torch.cuda.empty_cache()


def test_separate_epoch_lanes_in_one_graph(dev):
    """Two epoch counters (two lanes) advanced in an interleaved order inside
    one graph keep separate counts on every replay ("[Kernel][PCP] Publish
    replicated KV updates through PyTorch symmetric memory", Design: the
    device-epoch barrier supports separate DBO lanes)."""
    lanes = torch.zeros(2, dtype=torch.int64, device=dev)
    kvpub.epoch_advance(lanes[0:1])            # load the kernel
    torch.cuda.synchronize()
    lanes.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for k in range(7):
            kvpub.epoch_advance(lanes[0:1])
            if k % 2 == 0:
                kvpub.epoch_advance(lanes[1:2])
    for k in range(1, 6):
        g.replay()
        torch.cuda.synchronize()
        assert lanes.tolist() == [7 * k, 4 * k]


def test_two_dbo_lanes_on_two_streams_in_one_graph(dev):
    """Two micro-batch lanes, as in dual-batch overlap: each lane stores its
    own layers' rows into its own caches and advances its own epoch after
    every layer, on its own stream forked from the capture stream.  The
    launches are issued interleaved, and lane B's store of layer k also
    waits for lane A's epoch advance of layer k (an event across streams).
    On every one of 10 replays both counters must be exact, and afterwards
    both lanes' caches must equal the oracle's bytes ("[Kernel][PCP] Publish
    replicated KV updates through PyTorch symmetric memory", Design: the
    device-epoch barrier supports CUDA Graph replay and separate DBO
    lanes)."""
    from gpu_util import DevInputs
    layers = {"A": 4, "B": 3}
    R, nb = 2, 96
    ws = {lane: [inputs.prefill_batch(600 + 10 * i + layer, 2, 1024, nb, R)
                 for layer in range(n)] for i, (lane, n) in enumerate(layers.items())}
    xs = {lane: [DevInputs(w, dev) for w in ws[lane]] for lane in layers}
    caches = {lane: [Caches(R, nb, inputs.GUARD_BYTE, dev) for _ in ws[lane]] for lane in layers}
    epochs = torch.zeros(2, dtype=torch.int64, device=dev)
    epoch = {"A": epochs[0:1], "B": epochs[1:2]}

    def store(lane, layer):
        x, c = xs[lane][layer], caches[lane][layer]
        kvpub.store_mla_fp8(x.lat, x.rope, x.idx, x.slots, c.main, c.idx, nb)
        kvpub.epoch_advance(epoch[lane])

    for lane in layers:                        # load the kernels before capture
        store(lane, 0)
    torch.cuda.synchronize()
    epochs.zero_()

    lane_a, lane_b = torch.cuda.Stream(), torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        main = torch.cuda.current_stream()
        lane_a.wait_stream(main)
        lane_b.wait_stream(main)
        for layer in range(max(layers.values())):
            done_a = torch.cuda.Event()
            if layer < layers["A"]:
                with torch.cuda.stream(lane_a):
                    store("A", layer)
                    done_a.record(lane_a)
            if layer < layers["B"]:
                with torch.cuda.stream(lane_b):
                    if layer < layers["A"]:
                        lane_b.wait_event(done_a)
                    store("B", layer)
        main.wait_stream(lane_a)
        main.wait_stream(lane_b)
    torch.cuda.synchronize()
    assert epochs.tolist() == [0, 0]           # capture runs nothing
    for k in range(1, REPLAYS + 1):
        g.replay()
        torch.cuda.synchronize()
        assert epochs.tolist() == [layers["A"] * k, layers["B"] * k]
    for lane in layers:
        for w, c in zip(ws[lane], caches[lane]):
            assert_matches_oracle(c, *oracle_caches(w)[:2])


def test_scattered_slots_replay_in_a_graph(dev):
    """The capacity batch (slots scattered over 706,624, so every warp takes
    the part-sector prefetch) stored into two layers' caches, each store
    followed by an epoch advance, captured once and replayed three times:
    the epoch counts every replay and both layers equal the oracle."""
    from gpu_util import DevInputs
    w = inputs.make(4)
    x = DevInputs(w, dev)
    caches = [Caches(4, w.num_blocks, w.guard, dev) for _ in range(2)]
    epoch = torch.zeros(1, dtype=torch.int64, device=dev)

    def step():
        for c in caches:
            kvpub.store_mla_fp8(x.lat, x.rope, x.idx, x.slots, c.main, c.idx, w.num_blocks)
            kvpub.epoch_advance(epoch)

    step()
    torch.cuda.synchronize()
    epoch.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for c in caches:                       # replays must rewrite every byte
        for b in c.main + c.idx:
            b.fill_(w.guard)
    for k in range(1, 4):
        g.replay()
        torch.cuda.synchronize()
        assert int(epoch.item()) == 2 * k
    want_main, want_idx, _, _ = oracle_caches(w)
    for c in caches:
        assert_matches_oracle(c, want_main, want_idx)
    del caches, x, g
    torch.cuda.empty_cache()


def test_bench_step_matches_oracle(dev):
    """The benchmark's own launch configuration: packed [T, 704] rows passed
    as strided views, one graph of 61 x (store + epoch advance), and the
    end-to-end graph that copies the inputs from pinned host memory."""
    import bench

    step = bench.Step(dev, bench.SPECS[bench.WORKLOAD]())
    g = step.capture(with_epoch=True)
    g.replay()
    torch.cuda.synchronize()
    assert int(step.epoch.item()) == LAYERS
    slots = inputs.layer_slot_mapping()
    for layer in (0, 31, 60):
        w = inputs.prefill_layer(layer, slots)
        want_main, want_idx, _, _ = oracle_caches(w)
        for r in range(4):
            assert np.array_equal(step.main[layer][r].cpu().numpy(), want_main[r])
            assert np.array_equal(step.idx[layer][r].cpu().numpy(), want_idx[r])
    # end to end: wipe the device rows and caches, then one replay must
    # bring the rows back from host memory and rewrite the same bytes
    step.rows.zero_()
    for layer in (0, 60):
        for c in step.main[layer] + step.idx[layer]:
            c.fill_(inputs.GUARD_BYTE)
    ge = step.capture_end_to_end()
    ge.replay()
    torch.cuda.synchronize()
    assert int(step.host_epoch.item()) == 2 * LAYERS
    for layer in (0, 60):
        w = inputs.prefill_layer(layer, slots)
        want_main, want_idx, _, _ = oracle_caches(w)
        for r in range(4):
            assert np.array_equal(step.main[layer][r].cpu().numpy(), want_main[r])
            assert np.array_equal(step.idx[layer][r].cpu().numpy(), want_idx[r])
    del step, g, ge
    torch.cuda.empty_cache()


def test_bench_publish_path_matches_oracle(dev):
    """The benchmark's fused path: one store + epoch launch per layer in one
    graph; one replay advances the epoch by 61 and layers 0 and 60 equal the
    oracle."""
    import bench

    step = bench.Step(dev, bench.SPECS[bench.WORKLOAD](), "publish")
    assert step.launches_per_layer() == 1
    g = step.capture(with_epoch=True)
    torch.cuda.synchronize()
    before = int(step.epoch.item())
    g.replay()
    torch.cuda.synchronize()
    assert int(step.epoch.item()) == before + LAYERS
    assert int(step.done.item()) == 0
    slots = inputs.layer_slot_mapping()
    for layer in (0, 60):
        want_main, want_idx, _, _ = oracle_caches(inputs.prefill_layer(layer, slots))
        for r in range(4):
            assert np.array_equal(step.main[layer][r].cpu().numpy(), want_main[r])
            assert np.array_equal(step.idx[layer][r].cpu().numpy(), want_idx[r])
    del step, g
    torch.cuda.empty_cache()


def test_every_capturable_call_replays_in_a_graph(dev):
    """gather-then-insert, the bf16 store and the bounded wait, captured with
    the epoch advance and replayed twice: bytes as the oracle's, epoch and
    wait status as expected on every replay."""
    import oracle
    w = inputs.make(1)
    from gpu_util import Caches, DevInputs
    x = DevInputs(w, dev)
    c_gather = Caches(2, w.num_blocks, w.guard, dev)
    ws = torch.empty(kvpub.gather_workspace_bytes(w.num_tokens), dtype=torch.uint8, device=dev)
    nb = w.num_blocks
    main16 = [torch.full((nb * 64 * 1152,), w.guard, dtype=torch.uint8, device=dev) for _ in range(2)]
    idx16 = [torch.full((nb * 64 * 256,), w.guard, dtype=torch.uint8, device=dev) for _ in range(2)]
    epoch = torch.zeros(1, dtype=torch.int64, device=dev)
    status = torch.full((1,), 7, dtype=torch.int32, device=dev)
    scratch = torch.zeros(1, dtype=torch.int64, device=dev)

    def step(ep, target):
        kvpub.gather_insert(x.lat, x.rope, x.idx, x.slots, c_gather.main, c_gather.idx, ws, nb)
        kvpub.store_mla_bf16(x.lat, x.rope, x.idx, x.slots, main16, idx16, nb)
        kvpub.epoch_advance(ep)
        kvpub.epoch_wait(ep, target, 1000, status)

    step(scratch, 1)                              # load the kernels before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(epoch, 1)                            # reached on every replay: epoch >= 1
    for k in (1, 2):
        status.fill_(7)
        g.replay()
        torch.cuda.synchronize()
        assert int(epoch.item()) == k and int(status.item()) == 0
    assert_matches_oracle(c_gather, *oracle_caches(w)[:2])
    want16_main, want16_idx = oracle.new_caches_bf16(2, nb, w.guard)
    oracle.store_mla_bf16(w.kv_latent, w.k_rope, w.index_k, w.slot_mapping, want16_main,
                          want16_idx, nb)
    for got, want in zip(main16 + idx16, want16_main + want16_idx):
        assert np.array_equal(got.cpu().numpy(), want)


def test_first_call_of_a_process_can_be_captured(cuda_device):
    """A fresh process whose first kvpub call is inside graph capture."""
    import json
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    kbuild.build()
    res = subprocess.run([sys.executable, os.path.join(here, "capture_first_call.py")],
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    out = json.loads(res.stdout.strip().splitlines()[-1])
    assert out == {"captured_first_call": True, "bytes_ok": True, "epoch": 1}, out
