"""GPU parity of the unquantised (bf16) cache variant against the oracle,
byte for byte over every replica's whole buffer plus red zones: the five
workloads' shapes, strided input views, padded and invalid slots, 1..8
replicas and ragged batches (the BF16 main/indexer cache cases of "[Feature]
[KV Connector] Support QSA HiSparse in disaggregated serving", Validation).
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import RED, DevInputs, bf16
from replication_token_warp_gb300 import build as kbuild
from replication_token_warp_gb300 import inputs, kvpub

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_device):
    kbuild.build()
    kvpub.lib()
    return cuda_device


def caches(R, nb, guard, dev):
    mb, ib = nb * 64 * 1152, nb * 64 * 256
    main = [torch.full((mb + 2 * RED,), guard, dtype=torch.uint8, device=dev) for _ in range(R)]
    idx = [torch.full((ib + 2 * RED,), guard, dtype=torch.uint8, device=dev) for _ in range(R)]
    return main, idx, [m[RED:RED + mb] for m in main], [x[RED:RED + ib] for x in idx]


def check(w, main_full, idx_full):
    want_main, want_idx = oracle.new_caches_bf16(len(main_full), w.num_blocks, w.guard)
    oracle.store_mla_bf16(w.kv_latent, w.k_rope, w.index_k, w.slot_mapping, want_main, want_idx,
                          w.num_blocks)
    for got, want in zip(main_full + idx_full, want_main + want_idx):
        g = got.cpu().numpy()
        assert np.all(g[:RED] == w.guard) and np.all(g[-RED:] == w.guard)
        assert np.array_equal(g[RED:-RED], want)


def run(w, dev, R=None, cnt=None):
    R = w.num_replicas if R is None else R
    x = DevInputs(w, dev)
    mf, xf, m, xi = caches(R, w.num_blocks, w.guard, dev)
    kvpub.store_mla_bf16(x.lat, x.rope, x.idx, x.slots, m, xi, w.num_blocks, invalid_count=cnt)
    torch.cuda.synchronize()
    return mf, xf


@pytest.mark.parametrize("index", [0, 1, 2, 4])
def test_workloads_match_oracle(dev, index):
    w = inputs.make(index)
    check(w, *run(w, dev))


def test_prefill_layer_matches_oracle(dev):
    w = inputs.make(3, layer=17)
    check(w, *run(w, dev))


def test_strided_views(dev):
    w = inputs.make(1)
    T = w.num_tokens
    kv = torch.zeros(T, 576, dtype=torch.bfloat16, device=dev)
    kv[:, :512] = bf16(w.kv_latent, dev)
    kv[:, 512:] = bf16(w.k_rope, dev)
    ik = torch.zeros(T, 136, dtype=torch.bfloat16, device=dev)
    ik[:, :128] = bf16(w.index_k, dev)
    mf, xf, m, xi = caches(2, w.num_blocks, w.guard, dev)
    kvpub.store_mla_bf16(kv[:, :512], kv[:, 512:], ik[:, :128],
                         torch.from_numpy(w.slot_mapping).to(dev), m, xi)
    torch.cuda.synchronize()
    check(w, mf, xf)


def test_padded_and_invalid_slots(dev):
    w = inputs.make(2)
    cap = w.num_blocks * 64
    slots = w.slot_mapping.copy()
    slots[[5, 50, 500]] = [cap, -9, cap + 12345]
    w.slot_mapping = slots
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    mf, xf = run(w, dev, cnt=cnt)
    assert int(cnt.item()) == 3
    check(w, mf, xf)


@pytest.mark.parametrize("delta", [-1, 0, 1])
def test_batches_on_both_sides_of_the_block_size_switch(dev, delta):
    # launches of fewer rows than SMs x 8 take 2-warp blocks, the rest 8-warp blocks
    T = torch.cuda.get_device_properties(dev).multi_processor_count * 8 + delta
    w = inputs.random_rows(seed=700 + delta, num_tokens=T, num_blocks=32, num_replicas=2,
                           pad_fraction=0.05)
    check(w, *run(w, dev))


@pytest.mark.parametrize("R", [1, 3, 8])
@pytest.mark.parametrize("T", [1, 33, 1000])
def test_replicas_and_ragged_batches(dev, R, T):
    w = inputs.random_rows(seed=500 + R + T, num_tokens=T, num_blocks=20, num_replicas=R,
                           pad_fraction=0.1)
    check(w, *run(w, dev))
