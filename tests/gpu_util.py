"""Helpers for the GPU parity tests: device inputs, guarded cache buffers
with red zones, and byte comparison against the CPU oracle."""

import numpy as np
import torch

import oracle
from replication_token_warp_gb300 import kvpub

RED = 4096            # red-zone bytes before and after every cache buffer


def bf16(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


class Caches:
    """R Main + R Indexer caches, each inside a buffer with red zones."""

    def __init__(self, R, num_blocks, guard, dev):
        self.R, self.num_blocks, self.guard = R, num_blocks, guard
        self.main_bytes = num_blocks * 64 * 656
        self.idx_bytes = num_blocks * 8448
        self.main_full = [torch.full((self.main_bytes + 2 * RED,), guard, dtype=torch.uint8,
                                     device=dev) for _ in range(R)]
        self.idx_full = [torch.full((self.idx_bytes + 2 * RED,), guard, dtype=torch.uint8,
                                    device=dev) for _ in range(R)]
        self.main = [b[RED:RED + self.main_bytes] for b in self.main_full]
        self.idx = [b[RED:RED + self.idx_bytes] for b in self.idx_full]

    def host(self):
        return ([b.cpu().numpy() for b in self.main_full],
                [b.cpu().numpy() for b in self.idx_full])


class DevInputs:
    def __init__(self, w, dev):
        self.lat = bf16(w.kv_latent, dev)
        self.rope = bf16(w.k_rope, dev)
        self.idx = bf16(w.index_k, dev)
        self.slots = torch.from_numpy(w.slot_mapping).to(dev)


def oracle_caches(w, R=None, guard=None):
    R = w.num_replicas if R is None else R
    main, ixc = oracle.new_caches(R, w.num_blocks, w.guard if guard is None else guard)
    n, inv = oracle.store_mla_fp8(w.kv_latent, w.k_rope, w.index_k, w.slot_mapping, main, ixc,
                                  w.num_blocks)
    return main, ixc, n, inv


def assert_matches_oracle(caches: Caches, want_main, want_idx):
    """Byte-exact over every replica's whole buffer, red zones included."""
    got_main, got_idx = caches.host()
    for r in range(caches.R):
        for got, want, what in ((got_main[r], want_main[r], "Main"),
                                (got_idx[r], want_idx[r], "Indexer")):
            assert np.all(got[:RED] == caches.guard), f"{what}[{r}] front red zone written"
            assert np.all(got[-RED:] == caches.guard), f"{what}[{r}] back red zone written"
            body = got[RED:-RED]
            if not np.array_equal(body, want):
                bad = np.nonzero(body != want)[0]
                raise AssertionError(
                    f"{what}[{r}]: {bad.size} bytes differ, first at {bad[:8].tolist()}: "
                    f"got {body[bad[:8]].tolist()} want {want[bad[:8]].tolist()}")


def run_store(w, dev, path="fused", R=None, invalid_count=None):
    R = w.num_replicas if R is None else R
    x = DevInputs(w, dev)
    c = Caches(R, w.num_blocks, w.guard, dev)
    if path == "fused":
        kvpub.store_mla_fp8(x.lat, x.rope, x.idx, x.slots, c.main, c.idx, w.num_blocks,
                            invalid_count=invalid_count)
    elif path == "gather":
        ws = torch.empty(max(1, kvpub.gather_workspace_bytes(w.num_tokens)), dtype=torch.uint8,
                         device=dev)
        kvpub.gather_insert(x.lat, x.rope, x.idx, x.slots, c.main, c.idx, ws, w.num_blocks,
                            invalid_count=invalid_count)
    elif path == "publish":
        epoch = torch.zeros(1, dtype=torch.int64, device=dev)
        done = torch.zeros(1, dtype=torch.int32, device=dev)
        kvpub.store_mla_fp8_publish(x.lat, x.rope, x.idx, x.slots, c.main, c.idx, epoch, done,
                                    w.num_blocks, invalid_count=invalid_count)
        torch.cuda.synchronize()
        assert int(epoch.item()) == 1 and int(done.item()) == 0
    else:
        raise ValueError(path)
    torch.cuda.synchronize()
    return c
