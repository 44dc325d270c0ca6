"""Seeded synthetic workloads for the replicated KV-cache store.

This module only draws inputs: bf16 token rows, a slot_mapping and the cache
geometry.  It holds none of the store's arithmetic, imports neither the CUDA
library nor the oracle, and is the one module both sides use.

The shapes follow the workloads on the pages:
  * "[Kernel][PCP] Publish replicated KV updates through PyTorch symmetric
    memory" (vLLM #52863), Performance evidence: 1,024-token prompts at
    concurrency 16 and 3,584-token prompts at concurrency 4; KV capacity
    706,624 tokens.
  * "[Feature][KV Connector] Support QSA HiSparse in disaggregated serving",
    Performance configuration: at most 64 sequences, maximum length 40,960.
Values are drawn as fp32 from a CPU ``torch.Generator`` seeded per workload
and rounded to bf16 (round to nearest even).  Every array is returned on the
host; callers copy to the device.

Workloads (one token row = Main-KV latent [512] | rope [64] | Indexer-K [128]):
  0 tiny      16 rows, R=1, 4 blocks; row 3 all zero; row 7 holds 1e4 at
              column 0 of latent and Indexer-K; 2 padded (-1) entries.
  1 decode    64 rows (one per sequence), R=2, 2048 blocks; 1% of channels
              x20; each sequence's next slot at a length U[1, 40960] in its
              own random block; the last 4 entries padded.
  2 prefill   16 requests x 1024 tokens, R=4, 4096 blocks; outlier channels
              as in decode; each request fills a contiguous run in randomly
              permuted blocks; the last 128 entries padded.
  3 layers    4 requests x 3584 tokens per layer, R=4, 1024 blocks per layer,
              61 layers; rows regenerated per layer from seed 3 + layer; one
              slot_mapping shared by every layer; no padding.
  4 capacity  32,768 rows, R=4, 11,041 blocks (706,624 slots); 97% N(0,1)
              rows, 2% all-zero rows, 1% rows U(-6e4, 6e4); distinct random
              slots over the whole cache with 5% padded entries.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

LATENT_DIM = 512
ROPE_DIM = 64
INDEXER_DIM = 128
BLOCK_SIZE = 64
GUARD_BYTE = 0xA5

NAMES = ("tiny", "decode", "prefill_c16x1024", "prefill_c4x3584_61layers",
         "capacity_706624")


@dataclasses.dataclass
class Workload:
    """One layer's store: bf16 rows as uint16 bit patterns plus geometry."""

    name: str
    kv_latent: np.ndarray      # uint16 [T, 512]
    k_rope: np.ndarray         # uint16 [T, 64]
    index_k: np.ndarray        # uint16 [T, 128]
    slot_mapping: np.ndarray   # int64 [T]; -1 = padded
    num_replicas: int
    num_blocks: int
    guard: int = GUARD_BYTE

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def num_valid(self) -> int:
        s = self.slot_mapping
        return int(np.count_nonzero((s >= 0) & (s < self.num_blocks * BLOCK_SIZE)))


@dataclasses.dataclass(frozen=True)
class Spec:
    index: int
    name: str
    num_tokens: int
    num_replicas: int
    num_blocks: int
    num_layers: int = 1


SPECS = (
    Spec(0, NAMES[0], 16, 1, 4),
    Spec(1, NAMES[1], 64, 2, 2048),
    Spec(2, NAMES[2], 16 * 1024, 4, 4096),
    Spec(3, NAMES[3], 4 * 3584, 4, 1024, num_layers=61),
    Spec(4, NAMES[4], 32768, 4, 11041),
)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    """fp32 tensor -> bf16 (RNE) -> uint16 bit patterns."""
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _normal(g, rows, cols):
    return torch.randn(rows, cols, generator=g, dtype=torch.float32)


def _outlier_channels(g, x: torch.Tensor) -> torch.Tensor:
    """Scale max(1, round(1% of the columns)) random columns by 20."""
    cols = x.shape[1]
    k = max(1, int(round(0.01 * cols)))
    pick = torch.randperm(cols, generator=g)[:k]
    x[:, pick] *= 20.0
    return x


def _rows_with_outlier_channels(g, T):
    lat = _outlier_channels(g, _normal(g, T, LATENT_DIM))
    rope = _outlier_channels(g, _normal(g, T, ROPE_DIM))
    idx = _outlier_channels(g, _normal(g, T, INDEXER_DIM))
    return lat, rope, idx


def _tiny() -> Workload:
    g = _gen(0)
    T, nb = 16, 4
    lat, rope, idx = _normal(g, T, LATENT_DIM), _normal(g, T, ROPE_DIM), _normal(g, T, INDEXER_DIM)
    for x in (lat, rope, idx):
        x[3].zero_()
    lat[7, 0] = 1e4
    idx[7, 0] = 1e4
    slots = torch.randperm(nb * BLOCK_SIZE, generator=g)[:T].to(torch.int64)
    pad = torch.randperm(T, generator=g)[:2]
    slots[pad] = -1
    return Workload(NAMES[0], _bf16_bits(lat), _bf16_bits(rope), _bf16_bits(idx),
                    slots.numpy().copy(), 1, nb)


def _decode() -> Workload:
    g = _gen(1)
    T, nb, max_len = 64, 2048, 40960
    lat, rope, idx = _rows_with_outlier_channels(g, T)
    lengths = torch.randint(1, max_len + 1, (T,), generator=g, dtype=torch.int64)
    blocks = torch.randperm(nb, generator=g)[:T].to(torch.int64)
    slots = blocks * BLOCK_SIZE + (lengths - 1) % BLOCK_SIZE
    slots[T - 4:] = -1
    return Workload(NAMES[1], _bf16_bits(lat), _bf16_bits(rope), _bf16_bits(idx),
                    slots.numpy().copy(), 2, nb)


def _prefill_slots(g, num_requests, tokens_per_request, num_blocks):
    """Each request fills a contiguous token run in its own permuted blocks."""
    per = (tokens_per_request + BLOCK_SIZE - 1) // BLOCK_SIZE
    perm = torch.randperm(num_blocks, generator=g).to(torch.int64)
    pos = torch.arange(tokens_per_request, dtype=torch.int64)
    out = []
    for r in range(num_requests):
        blocks = perm[r * per:(r + 1) * per]
        out.append(blocks[pos // BLOCK_SIZE] * BLOCK_SIZE + pos % BLOCK_SIZE)
    return torch.cat(out)


def _prefill_c16() -> Workload:
    g = _gen(2)
    T, nb = 16 * 1024, 4096
    lat, rope, idx = _rows_with_outlier_channels(g, T)
    slots = _prefill_slots(g, 16, 1024, nb)
    slots[T - 128:] = -1
    return Workload(NAMES[2], _bf16_bits(lat), _bf16_bits(rope), _bf16_bits(idx),
                    slots.numpy().copy(), 4, nb)


def layer_slot_mapping() -> np.ndarray:
    """The slot_mapping shared by all 61 layers of the c4 x 3584 prefill."""
    g = _gen(3)
    return _prefill_slots(g, 4, 3584, 1024).numpy().copy()


def prefill_layer(layer: int, slots: np.ndarray | None = None) -> Workload:
    """Layer ``layer`` (0..60) of the c4 x 3584 prefill: rows from seed 3+layer."""
    g = _gen(3 + int(layer))
    T = 4 * 3584
    lat, rope, idx = _rows_with_outlier_channels(g, T)
    if slots is None:
        slots = layer_slot_mapping()
    return Workload(f"{NAMES[3]}[{layer}]", _bf16_bits(lat), _bf16_bits(rope),
                    _bf16_bits(idx), slots, 4, 1024)


def _capacity() -> Workload:
    g = _gen(4)
    T, nb = 32768, 11041
    n_zero, n_big = int(0.02 * T), int(0.01 * T)
    lat, rope, idx = _normal(g, T, LATENT_DIM), _normal(g, T, ROPE_DIM), _normal(g, T, INDEXER_DIM)
    order = torch.randperm(T, generator=g)
    zero_rows, big_rows = order[:n_zero], order[n_zero:n_zero + n_big]
    for x in (lat, rope, idx):
        x[zero_rows] = 0.0
        big = torch.rand(n_big, x.shape[1], generator=g, dtype=torch.float32)
        x[big_rows] = (big * 2.0 - 1.0) * 6e4
    n_pad = int(0.05 * T)
    slots = torch.randperm(nb * BLOCK_SIZE, generator=g)[:T].to(torch.int64)
    pad = torch.randperm(T, generator=g)[:n_pad]
    slots[pad] = -1
    return Workload(NAMES[4], _bf16_bits(lat), _bf16_bits(rope), _bf16_bits(idx),
                    slots.numpy().copy(), 4, nb)


def make(index: int, layer: int = 0) -> Workload:
    """Workload ``index`` (0..4); for the 61-layer prefill, one layer of it."""
    if index == 0:
        return _tiny()
    if index == 1:
        return _decode()
    if index == 2:
        return _prefill_c16()
    if index == 3:
        return prefill_layer(layer)
    if index == 4:
        return _capacity()
    raise ValueError(f"no workload {index}")


def prefill_batch(seed: int, num_requests: int, tokens_per_request: int, num_blocks: int,
                  num_replicas: int = 4) -> Workload:
    """A generic prefill batch: outlier-channel rows, each request filling a
    contiguous token run in its own randomly permuted blocks."""
    g = _gen(seed)
    T = num_requests * tokens_per_request
    lat, rope, idx = _rows_with_outlier_channels(g, T)
    slots = _prefill_slots(g, num_requests, tokens_per_request, num_blocks)
    return Workload(f"prefill(seed={seed},{num_requests}x{tokens_per_request})",
                    _bf16_bits(lat), _bf16_bits(rope), _bf16_bits(idx), slots.numpy().copy(),
                    int(num_replicas), int(num_blocks))


def random_rows(seed: int, num_tokens: int, num_blocks: int, num_replicas: int = 1,
                pad_fraction: float = 0.0, scale: float = 1.0) -> Workload:
    """A generic seeded workload: N(0, scale^2) rows, distinct random slots."""
    g = _gen(seed)
    T = int(num_tokens)
    lat = _normal(g, T, LATENT_DIM) * scale
    rope = _normal(g, T, ROPE_DIM) * scale
    idx = _normal(g, T, INDEXER_DIM) * scale
    cap = num_blocks * BLOCK_SIZE
    if T > cap:
        raise ValueError("more tokens than slots")
    slots = torch.randperm(cap, generator=g)[:T].to(torch.int64)
    n_pad = int(pad_fraction * T)
    if n_pad:
        slots[torch.randperm(T, generator=g)[:n_pad]] = -1
    return Workload(f"random(seed={seed},T={T})", _bf16_bits(lat), _bf16_bits(rope),
                    _bf16_bits(idx), slots.numpy().copy(), int(num_replicas),
                    int(num_blocks))
