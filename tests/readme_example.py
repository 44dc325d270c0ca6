"""The library's Python usage example, as its front-page documentation shows it.

Publishes 1,024 token rows into 4 replicas of a 256-block fp8 cache, then
advances the device epoch.  tests/test_gpu_readme.py runs this file and
checks every written slot against the CPU oracle.
"""
import torch
from replication_token_warp_gb300 import kvpub

T, R, num_blocks = 1024, 4, 256
kv = torch.randn(T, 576, dtype=torch.bfloat16, device="cuda")      # latent | rope, one buffer
index_k = torch.randn(T, 128, dtype=torch.bfloat16, device="cuda")
slot_mapping = torch.randperm(num_blocks * 64, device="cuda")[:T]  # int64; -1 = padded
main = [torch.empty(num_blocks * 64 * 656, dtype=torch.uint8, device="cuda") for _ in range(R)]
indexer = [torch.empty(num_blocks * 64 * 132, dtype=torch.uint8, device="cuda") for _ in range(R)]
epoch = torch.zeros(1, dtype=torch.int64, device="cuda")

kvpub.store_mla_fp8(kv[:, :512], kv[:, 512:], index_k, slot_mapping, main, indexer)
kvpub.epoch_advance(epoch)      # or store_mla_fp8_publish(...) for both in one launch
