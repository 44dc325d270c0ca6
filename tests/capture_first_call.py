"""Run in a fresh process by test_gpu_graph.py: the first kvpub call of the
process happens inside CUDA-graph capture (occupancy queries and module
loading included); one replay must leave the oracle's bytes and epoch 1."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from gpu_util import Caches, DevInputs, oracle_caches  # noqa: E402
from replication_token_warp_gb300 import inputs, kvpub  # noqa: E402

dev = torch.device("cuda:0")
w = inputs.make(1)
x = DevInputs(w, dev)
c = Caches(2, w.num_blocks, w.guard, dev)
epoch = torch.zeros(1, dtype=torch.int64, device=dev)
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
try:
    with torch.cuda.graph(g):
        kvpub.store_mla_fp8(x.lat, x.rope, x.idx, x.slots, c.main, c.idx)
        kvpub.epoch_advance(epoch)
    g.replay()
    torch.cuda.synchronize()
    main, idx = c.host()
    wm, wi, _, _ = oracle_caches(w)
    ok = all(np.array_equal(main[r][4096:-4096], wm[r]) and np.array_equal(idx[r][4096:-4096], wi[r]) for r in range(2))
    print(json.dumps({"captured_first_call": True, "bytes_ok": ok, "epoch": int(epoch.item())}))
except Exception as e:
    print(json.dumps({"captured_first_call": False, "error": str(e)[:300]}))
