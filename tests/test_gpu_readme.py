"""The repository's Python usage example (tests/readme_example.py, shown in
the front-page documentation) runs as written, and every slot it writes holds the bytes the
CPU oracle computes from the example's own inputs.  The example's caches
start uninitialised, so only the written slots are compared; the
whole-buffer checks are in test_gpu_parity.py."""

import os
import runpy

import numpy as np
import pytest
import torch

import oracle
from replication_token_warp_gb300 import build as kbuild
from replication_token_warp_gb300 import kvpub

pytestmark = pytest.mark.gpu

EXAMPLE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "readme_example.py")


def test_readme_example_matches_the_oracle(cuda_device):
    kbuild.build()
    kvpub.lib()
    ns = runpy.run_path(EXAMPLE)
    torch.cuda.synchronize()
    assert int(ns["epoch"].item()) == 1

    def bits(t):
        return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    kv, R, nb = ns["kv"], ns["R"], ns["num_blocks"]
    slots = ns["slot_mapping"].cpu().numpy()
    want_main, want_idx = oracle.new_caches(R, nb)
    oracle.store_mla_fp8(bits(kv[:, :512]), bits(kv[:, 512:]), bits(ns["index_k"]), slots,
                         want_main, want_idx, nb)
    for r in range(R):
        got_main = ns["main"][r].cpu().numpy().reshape(nb * 64, 656)
        got_idx = ns["indexer"][r].cpu().numpy().reshape(nb, 8448)
        wm = want_main[r].reshape(nb * 64, 656)
        wi = want_idx[r].reshape(nb, 8448)
        for s in slots[slots >= 0].tolist():
            blk, off = divmod(s, 64)
            assert np.array_equal(got_main[s], wm[s])
            assert np.array_equal(got_idx[blk, off * 128:(off + 1) * 128],
                                  wi[blk, off * 128:(off + 1) * 128])
            assert np.array_equal(got_idx[blk, 8192 + 4 * off:8196 + 4 * off],
                                  wi[blk, 8192 + 4 * off:8196 + 4 * off])
