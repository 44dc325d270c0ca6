"""Seeded random parity cases: every case draws its own batch size, replica
count, cache size, row strides, padding, invalid slots and value range, and
runs one of the four store paths (direct, gather-then-insert, fused publish,
bf16 cache) against the CPU oracle, byte for byte over every replica's whole
buffer and its red zones.  A second set draws only launches large enough for
the kernel with the part-sector prefetch, mixing scattered slots with
contiguous runs in caches 1.1x to 30x the batch.

Each case also fills the row padding beyond the 512 / 64 / 128 used values
with NaN bit patterns, so a kernel that read past a row's used columns would
change the scales and codes.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import RED
from replication_token_warp_gb300 import build as kbuild
from replication_token_warp_gb300 import kvpub

pytestmark = pytest.mark.gpu

PATHS = ("fused", "gather", "publish", "bf16")
NAN_BITS = 0x7FC0


@pytest.fixture(scope="module")
def dev(cuda_device):
    kbuild.build()
    kvpub.lib()
    return cuda_device


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _values(rng, T, cols):
    """Rows of N(0,1) x 2^e (e uniform in [-60, 60] per row) with a few
    all-zero rows, rows holding +-Inf, rows holding NaN and signed zeros."""
    x = rng.standard_normal((T, cols)) * np.exp2(rng.uniform(-60, 60, size=(T, 1)))
    kind = rng.random(T)
    x[kind < 0.03] = 0.0
    inf_rows = np.nonzero((kind >= 0.03) & (kind < 0.05))[0]
    x[inf_rows, rng.integers(0, cols, size=inf_rows.size)] = np.inf * rng.choice([-1, 1], inf_rows.size)
    nan_rows = np.nonzero((kind >= 0.05) & (kind < 0.06))[0]
    x[nan_rows, rng.integers(0, cols, size=nan_rows.size)] = np.nan
    zeros = rng.random((T, cols)) < 0.01
    x[zeros] = -0.0
    return _bf16_bits(x)


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    T = int(round(np.exp(rng.uniform(0, np.log(4000)))))
    R = int(rng.integers(1, 9))
    nb = int(-(-T // 64) + rng.integers(1, 40))
    cap = nb * 64
    slots = rng.permutation(cap)[:T].astype(np.int64)
    slots[rng.random(T) < rng.uniform(0, 0.3)] = -1
    for _ in range(int(rng.integers(0, 4))):
        slots[rng.integers(0, T)] = int(rng.choice([cap + int(rng.integers(0, 1000)),
                                                    -2 - int(rng.integers(0, 1000))]))
    strides = (int(rng.choice([512, 520, 576, 640, 704])), int(rng.choice([64, 72, 80, 576])),
               int(rng.choice([128, 136, 200])))
    return dict(T=T, R=R, nb=nb, slots=slots, strides=strides,
                lat=_values(rng, T, 512), rope=_values(rng, T, 64), idx=_values(rng, T, 128),
                path=PATHS[seed % len(PATHS)])


def _strided(bits: np.ndarray, stride: int, dev) -> torch.Tensor:
    T, cols = bits.shape
    buf = np.full((T, stride), NAN_BITS, np.uint16)
    buf[:, :cols] = bits
    t = torch.from_numpy(buf.view(np.int16)).view(torch.bfloat16).to(dev)
    return t[:, :cols]


@pytest.mark.parametrize("seed", range(40))
def test_random_case_matches_oracle(dev, seed):
    _run_case(dev, _case(seed), seed)


def _run_case(dev, c, seed):
    T, R, nb, path = c["T"], c["R"], c["nb"], c["path"]
    bf16_cache = path == "bf16"
    main_bytes = nb * 64 * (1152 if bf16_cache else 656)
    idx_bytes = nb * (64 * 256 if bf16_cache else 8448)
    main_full = [torch.full((main_bytes + 2 * RED,), 0xA5, dtype=torch.uint8, device=dev)
                 for _ in range(R)]
    idx_full = [torch.full((idx_bytes + 2 * RED,), 0xA5, dtype=torch.uint8, device=dev)
                for _ in range(R)]
    main = [b[RED:RED + main_bytes] for b in main_full]
    idx = [b[RED:RED + idx_bytes] for b in idx_full]
    ls, rs, xs = c["strides"]
    lat, rope, ik = _strided(c["lat"], ls, dev), _strided(c["rope"], rs, dev), \
        _strided(c["idx"], xs, dev)
    slots = torch.from_numpy(c["slots"]).to(dev)
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    if path == "fused":
        kvpub.store_mla_fp8(lat, rope, ik, slots, main, idx, nb, invalid_count=cnt)
    elif path == "gather":
        ws = torch.empty(kvpub.gather_workspace_bytes(T), dtype=torch.uint8, device=dev)
        kvpub.gather_insert(lat, rope, ik, slots, main, idx, ws, nb, invalid_count=cnt)
    elif path == "publish":
        epoch = torch.zeros(1, dtype=torch.int64, device=dev)
        done = torch.zeros(1, dtype=torch.int32, device=dev)
        kvpub.store_mla_fp8_publish(lat, rope, ik, slots, main, idx, epoch, done, nb,
                                    invalid_count=cnt)
    else:
        kvpub.store_mla_bf16(lat, rope, ik, slots, main, idx, nb, invalid_count=cnt)
    torch.cuda.synchronize()
    if path == "publish":
        assert int(epoch.item()) == 1 and int(done.item()) == 0

    if bf16_cache:
        want_main, want_idx = oracle.new_caches_bf16(R, nb)
        _, inv = oracle.store_mla_bf16(c["lat"], c["rope"], c["idx"], c["slots"], want_main,
                                       want_idx, nb)
    else:
        want_main, want_idx = oracle.new_caches(R, nb)
        _, inv = oracle.store_mla_fp8(c["lat"], c["rope"], c["idx"], c["slots"], want_main,
                                      want_idx, nb)
    assert int(cnt.item()) == inv
    for got, want in zip(main_full + idx_full, want_main + want_idx):
        g = got.cpu().numpy()
        assert np.all(g[:RED] == 0xA5) and np.all(g[-RED:] == 0xA5), "red zone touched"
        assert np.array_equal(g[RED:-RED], want), f"case {seed}: T={T} R={R} nb={nb} {path}"


def _large_case(seed):
    """A launch of at least SMs x 8 rows (the instantiation with the part-sector
    prefetch): the cache is 1.1x, 4x or 30x the batch, and each case mixes
    scattered slots with contiguous runs of 64 to 1,024 slots, so some warps
    take the prefetch and others do not."""
    rng = np.random.default_rng(5000 + seed)
    T = int(rng.integers(1216, 16385))
    R = int(rng.integers(1, 9))
    nb = int(-(-int(T * float(rng.choice([1.1, 4.0, 30.0]))) // 64))
    cap = nb * 64
    slots = np.empty(T, np.int64)
    perm = rng.permutation(cap)
    blocks = rng.permutation(nb)
    used, t, bi, pi = set(), 0, 0, 0
    while t < T:
        if rng.random() < 0.5 and bi < nb:               # a contiguous run in a fresh block
            run = int(min(T - t, rng.integers(64, 1025)))
            start = int(blocks[bi]) * 64
            bi += 1
            cand = [s for s in range(start, min(start + run, cap)) if s not in used]
        else:                                           # scattered slots
            run = int(min(T - t, rng.integers(1, 257)))
            cand = []
            while len(cand) < run and pi < cap:
                s = int(perm[pi])
                pi += 1
                if s not in used:
                    cand.append(s)
        cand = cand[:T - t]
        if not cand:
            cand = [int(s) for s in np.setdiff1d(np.arange(cap), list(used))[:T - t]]
        used.update(cand)
        slots[t:t + len(cand)] = cand
        t += len(cand)
    slots[rng.random(T) < 0.03] = -1
    return dict(T=T, R=R, nb=nb, slots=slots, strides=(512, 64, 128),
                lat=_values(rng, T, 512), rope=_values(rng, T, 64), idx=_values(rng, T, 128),
                path=PATHS[seed % 3])


@pytest.mark.parametrize("seed", range(12))
def test_large_mixed_case_matches_oracle(dev, seed):
    _run_case(dev, _large_case(seed), seed)
