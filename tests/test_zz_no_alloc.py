"""The allocation-free gather-then-insert against the allocating one.

Some callers cannot allocate device memory:
  * a serving loop that reserves all of its device memory at start-up;
  * a plugin inside another runtime that owns the device's memory;
  * a latency-critical path where cudaMalloc could synchronise the device.
kvpub_gather_insert_noalloc serves them with a fixed workspace inside the
library.

This file calls that entry point through the C ABI twice in a row, each
time with different rows and a different replica count. Both calls must
leave the same bytes as kvpub_gather_insert with a caller-owned workspace,
and the same bytes as the CPU oracle computes from the same inputs: byte for
byte over whole buffers and red zones, the tolerance of every cache test
here. A batch above the fixed limit must be refused with nothing launched.

The file sits last in collection order, so a run that stops at its first
failure has already run every other test.
"""

import ctypes

import pytest
import torch

from gpu_util import Caches, DevInputs, assert_matches_oracle, oracle_caches
from replication_token_warp_gb300 import build as kbuild
from replication_token_warp_gb300 import inputs, kvpub

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_device):
    kbuild.build()
    kvpub.lib()
    return cuda_device


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _noalloc_call(x, w, c, count):
    lib = kvpub.lib()
    return lib.kvpub_gather_insert_noalloc(
        x.lat.data_ptr(), x.lat.stride(0), x.rope.data_ptr(), x.rope.stride(0),
        x.idx.data_ptr(), x.idx.stride(0), x.slots.data_ptr(), w.num_tokens,
        _ptrs(c.main), _ptrs(c.idx), c.R, w.num_blocks, 64, count.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_gather_insert_twice(dev):
    calls = [inputs.make(1),
             inputs.random_rows(seed=77, num_tokens=kvpub.STATIC_GATHER_MAX_TOKENS,
                                num_blocks=80, num_replicas=3, pad_fraction=0.05)]
    for w in calls:
        x = DevInputs(w, dev)
        want = Caches(w.num_replicas, w.num_blocks, w.guard, dev)
        ws = torch.empty(kvpub.gather_workspace_bytes(w.num_tokens), dtype=torch.uint8,
                         device=dev)
        n_want = torch.zeros(1, dtype=torch.int64, device=dev)
        kvpub.gather_insert(x.lat, x.rope, x.idx, x.slots, want.main, want.idx, ws,
                            w.num_blocks, invalid_count=n_want)

        got = Caches(w.num_replicas, w.num_blocks, w.guard, dev)
        n_got = torch.zeros(1, dtype=torch.int64, device=dev)
        assert _noalloc_call(x, w, got, n_got) == 0, kvpub.last_error()
        torch.cuda.synchronize()

        for a, b in zip(want.main_full + want.idx_full, got.main_full + got.idx_full):
            assert torch.equal(a, b)
        assert int(n_got.item()) == int(n_want.item())
        want_main, want_idx, _, n_invalid = oracle_caches(w)
        assert_matches_oracle(got, want_main, want_idx)
        assert int(n_got.item()) == n_invalid
        written = sum(int((b != w.guard).sum().item()) for b in got.main)
        assert written > 0.9 * 656 * w.num_valid * w.num_replicas


def test_noalloc_refuses_batches_above_its_limit(dev):
    w = inputs.random_rows(seed=78, num_tokens=kvpub.STATIC_GATHER_MAX_TOKENS + 1,
                           num_blocks=80, num_replicas=1)
    x = DevInputs(w, dev)
    c = Caches(1, w.num_blocks, w.guard, dev)
    count = torch.zeros(1, dtype=torch.int64, device=dev)
    assert _noalloc_call(x, w, c, count) == 5
    assert "static workspace limit" in kvpub.last_error()
    torch.cuda.synchronize()
    assert all(bool((b == w.guard).all().item()) for b in c.main_full + c.idx_full)
