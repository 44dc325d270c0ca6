"""Benchmark: the fused replicated fp8 KV-cache store on GB300.

One step is one prefill's publication: 61 sparse-MLA layers, each storing
4 requests x 3,584 tokens (14,336 rows) into 4 replicas of that layer's
1,024-block cache, followed by that layer's device-epoch advance; the 122
launches are captured in one CUDA graph and one step is one replay.  The
workload follows "[Kernel][PCP] Publish replicated KV updates through
PyTorch symmetric memory", Performance evidence (3,584-token prompts at
concurrency 4, GLM-5.2's sparse layers) with seeded synthetic bf16 rows.

Prints one JSON line: rows stored per second x replicas (whole job), the
roofline of the store kernel against the measured HBM copy bandwidth, the
end-to-end figure through the public API with host inputs, the CPU oracle
timed on the host as a baseline, and under "workloads" the store kernel's
roofline fraction on each bandwidth-bound workload: the c16 x 1,024 prefill,
this c4 x 3,584 prefill and the 706,624-slot capacity batch.  Before any
timing, the timed buffers are compared byte for byte with the oracle's.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--path direct|publish|gather] [--workload NAME]

--path publish times the same step with the store and the epoch advance
fused into one launch per layer; --path gather the unfused
gather-then-insert path.  --eager issues the step's calls one by one from
the host (arguments marshalled once) instead of replaying a graph.

With --gpus N > 1 outside torchrun, the script starts itself again under
torch.distributed.run with N local ranks (one per GPU).

The DRAM traffic in the roofline comes from profiles/store_mla_fp8_prefill_
c4x3584.json, which ``--write-traffic`` writes from the CSV of this ncu
capture (a 3-layer run of the same launches; 3 captured store launches):

  python bench.py --layers 3 --steps 1 --warmup 3 --no-cpu-baseline --no-e2e \
      --no-workloads
  ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --print-units base \
      --cache-control none --clock-control none -k regex:store_mla_fp8_kernel \
      -s 14 -c 3 --csv --log-file dram_prefill.csv \
      python bench.py --layers 3 --steps 1 --warmup 3 --no-cpu-baseline --no-e2e \
      --no-workloads
  python bench.py --write-traffic dram_prefill.csv
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from replication_token_warp_gb300 import build as kbuild  # noqa: E402
from replication_token_warp_gb300 import inputs, kvpub  # noqa: E402

METRIC = "KV rows stored/sec ×R replicas and achieved HBM GB/s vs GB300 peak"
UNIT = "rows/s"
WORKLOAD = "prefill_c4x3584_61layers"
LAYERS = 61
ROWS = 4 * 3584
R = 4
NUM_BLOCKS = 1024
ROW_IN = 1408                  # bf16 bytes read per valid row
ROW_OUT = 656 + 132            # bytes written per valid row and replica
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "store_mla_fp8_prefill_c4x3584.json")
TRAFFIC_LAYERS = 3
# store_mla_fp8_kernel launches before the first timed replay of a
# --layers 3 --no-cpu-baseline run: the direct-vs-gather check (1 + 4),
# two eager passes before the captures (3 + 3) and one replay (3).
TRAFFIC_SKIP = 5 + 3 * TRAFFIC_LAYERS
TRAFFIC_RUN = (f"python bench.py --layers {TRAFFIC_LAYERS} --steps 1 --warmup 3 "
               "--no-cpu-baseline --no-e2e --no-workloads")
TRAFFIC_CMD = ("ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --print-units base "
               "--cache-control none --clock-control none -k regex:store_mla_fp8_kernel "
               f"-s {TRAFFIC_SKIP} -c {TRAFFIC_LAYERS} --csv --log-file <csv> {TRAFFIC_RUN}")


def gather_insert_bytes(num_tokens: int, num_valid: int, replicas: int) -> int:
    """Algorithmic HBM bytes of the unfused path for one layer: the gather
    copies every row (read + write 1408 B), then each replica's insert reads
    the slots and the gathered rows and writes 788 B per valid row."""
    return 2 * ROW_IN * num_tokens + replicas * (8 * num_tokens + num_valid * (ROW_IN + ROW_OUT))


def store_bytes(num_tokens: int, num_valid: int, replicas: int, bf16_cache: bool = False) -> int:
    """Algorithmic HBM bytes of one store launch: slots + rows read once +
    the bytes written per valid row and replica (788 for the fp8 cache,
    1408 for the unquantised bf16 cache)."""
    out = ROW_IN if bf16_cache else ROW_OUT
    return 8 * num_tokens + num_valid * (ROW_IN + out * replicas)


# ------------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """Source text without comments and with whitespace runs collapsed, so
    that an edit to a comment does not count as a change of the kernel."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """Hash of the code the kernels are built from: every file under csrc/
    and the public header (its layout constants are compiled in)."""
    h = hashlib.sha256()
    paths = [os.path.join(kbuild.CSRC, n) for n in sorted(os.listdir(kbuild.CSRC))]
    for path in paths + [os.path.join(kbuild.INCLUDE, "kvpub.h")]:
        with open(path, encoding="utf-8") as f:
            h.update(os.path.basename(path).encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes of the headline store kernel from the committed
    ncu summary, if it was captured on the kernel source as it stands (else
    None)."""
    try:
        with open(TRAFFIC_JSON) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    return int(rec["dram_bytes_per_launch"])


_UNIT_SCALE = {"byte": 1, "kbyte": 10**3, "mbyte": 10**6, "gbyte": 10**9,
               "kibyte": 2**10, "mibyte": 2**20, "gibyte": 2**30}


def read_ncu_csv(path: str, kernel: str = "store_mla_fp8_kernel"):
    """{launch id: {metric: bytes}} for the launches of ``kernel`` in an ncu
    --csv --metrics log (the log's own banner lines are skipped)."""
    import csv
    with open(path, newline="") as f:
        lines = f.read().splitlines()
    start = next((i for i, l in enumerate(lines) if l.startswith('"ID"')), None)
    if start is None:
        raise SystemExit(f"{path}: no ncu --csv metrics table in it")
    launches = {}
    for row in csv.DictReader(lines[start:]):
        if kernel not in row["Kernel Name"]:
            continue
        unit = row.get("Metric Unit", "byte").strip().lower() or "byte"
        value = float(row["Metric Value"].replace(",", "")) * _UNIT_SCALE.get(unit, 1)
        launches.setdefault(int(row["ID"]), {})[row["Metric Name"]] = value
    return launches


def write_traffic(csv_path: str) -> dict:
    """Turn the ncu capture named in the module docstring into the traffic
    record that the roofline reads, stamped with the current source hash."""
    launches = read_ncu_csv(csv_path)
    if not launches:
        raise SystemExit(f"no store_mla_fp8_kernel launches in {csv_path}")
    reads = [m["dram__bytes_read.sum"] for m in launches.values()]
    writes = [m["dram__bytes_write.sum"] for m in launches.values()]
    slots = inputs.layer_slot_mapping()
    rec = {
        "kernel": f"store_mla_fp8_kernel<{R}>",
        "workload": f"prefill_c4x3584 ({TRAFFIC_LAYERS} of {LAYERS} layers: the same "
                    f"{ROWS}-row, {R}-replica launches as the timed graph)",
        "kernel_source_sha256_16": kernel_source_hash(),
        "launches": len(launches),
        "dram_bytes_read_per_launch": int(round(statistics.mean(reads))),
        "dram_bytes_write_per_launch": int(round(statistics.mean(writes))),
        "dram_bytes_per_launch": int(round(statistics.mean(reads) + statistics.mean(writes))),
        "algorithmic_bytes_per_launch": store_bytes(ROWS, int(np.count_nonzero(slots >= 0)), R),
        "per_launch": [{"read": int(m["dram__bytes_read.sum"]),
                        "write": int(m["dram__bytes_write.sum"])}
                       for _, m in sorted(launches.items())],
        "command": TRAFFIC_CMD,
    }
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu, self.period = gpu_index, period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self, t0: float, t1: float):
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4)
                          if r[3][5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


# ------------------------------------------------------------------ our arm

class Spec:
    """A benchmark workload: `layers` store launches per step, each on its
    own inputs and caches (distinct buffers, so a step's working set is
    larger than L2), every launch followed by an epoch advance."""

    def __init__(self, name, layers, make, replicas, num_blocks, note, bf16_cache=False):
        self.name, self.layers, self.make = name, layers, make
        self.replicas, self.num_blocks, self.note = replicas, num_blocks, note
        self.bf16_cache = bf16_cache


def _copy_of(index):
    w = inputs.make(index)
    return lambda layer: w


def _stress(layer):
    """128 requests x 1,024 tokens (131,072 rows) into 8,192-block caches:
    one launch moves ~600 MB (~4.6x L2), so ncu's DRAM counters see the
    writes; about 1.9 GB on the device."""
    return inputs.prefill_batch(1000 + layer, 128, 1024, 8192)


def _prefill_layer_fn():
    slots = inputs.layer_slot_mapping()
    return lambda layer: inputs.prefill_layer(layer, slots)


SPECS = {
    "prefill_c4x3584_61layers": lambda: Spec(
        WORKLOAD, LAYERS, _prefill_layer_fn(), 4, 1024,
        "61 layers, seeds 3+layer, one shared slot_mapping"),
    "prefill_c4x3584_61layers_bf16": lambda: Spec(
        "prefill_c4x3584_61layers_bf16", LAYERS, _prefill_layer_fn(), 4, 1024,
        "the 61-layer prefill into unquantised bf16 caches", bf16_cache=True),
    "prefill_c16x1024": lambda: Spec(
        "prefill_c16x1024", 8, _copy_of(2), 4, 4096,
        "8 buffer copies of the c16 x 1024 batch per step"),
    "capacity_706624": lambda: Spec(
        "capacity_706624", 4, _copy_of(4), 4, 11041,
        "4 buffer copies of the 706,624-slot capacity batch per step"),
    "decode_c64_61layers": lambda: Spec(
        "decode_c64_61layers", LAYERS, _copy_of(1), 2, 2048,
        "a 64-sequence decode batch published in each of 61 layers (latency-bound)"),
    "capacity_706624_x1": lambda: Spec(
        "capacity_706624_x1", 1, _copy_of(4), 4, 11041,
        "one copy of the capacity batch (profiling case, ~2.3 GB)"),
    "capacity_706624_bf16": lambda: Spec(
        "capacity_706624_bf16", 4, _copy_of(4), 4, 11041,
        "4 buffer copies of the capacity batch, unquantised bf16 caches", bf16_cache=True),
    "stress_131072": lambda: Spec(
        "stress_131072", 1, _stress, 4, 8192,
        "one 131,072-row launch (profiling case)"),
}


class Step:
    """All layers resident in HBM: packed bf16 rows [T, 704] per layer
    (latent | rope | Indexer-K as strided views), a slot_mapping and R
    replica caches per layer, one epoch counter."""

    def __init__(self, dev, spec: Spec, path: str = "direct"):
        self.dev, self.spec, self.path = dev, spec, path
        L = spec.layers
        ws = [spec.make(layer) for layer in range(L)]
        T = ws[0].num_tokens
        self.num_tokens = T
        self.valid = [w.num_valid for w in ws]
        host = torch.empty(L, T, 704, dtype=torch.bfloat16, pin_memory=True)
        for layer, w in enumerate(ws):
            row = np.concatenate([w.kv_latent, w.k_rope, w.index_k], axis=1)
            host[layer].copy_(torch.from_numpy(row.view(np.int16)).view(torch.bfloat16))
        self.host_rows = host
        self.rows = host.to(dev)
        self.host_slots = torch.from_numpy(np.stack([w.slot_mapping for w in ws])).pin_memory()
        self.slots = self.host_slots.to(dev)
        nb = spec.num_blocks
        main_bytes = nb * 64 * (1152 if spec.bf16_cache else 656)
        idx_bytes = nb * 64 * (256 if spec.bf16_cache else 132)
        self.main = [[torch.full((main_bytes,), inputs.GUARD_BYTE, dtype=torch.uint8,
                                 device=dev) for _ in range(spec.replicas)] for _ in range(L)]
        self.idx = [[torch.full((idx_bytes,), inputs.GUARD_BYTE, dtype=torch.uint8,
                                device=dev) for _ in range(spec.replicas)] for _ in range(L)]
        self.epoch = torch.zeros(1, dtype=torch.int64, device=dev)
        self.invalid = torch.zeros(1, dtype=torch.int64, device=dev)
        self.workspace = None
        if path == "gather":
            self.workspace = torch.empty(kvpub.gather_workspace_bytes(T), dtype=torch.uint8,
                                         device=dev)
        self.done = torch.zeros(1, dtype=torch.int32, device=dev)     # publish path only

    def launches_per_layer(self, with_epoch: bool = True) -> int:
        if self.path == "publish":
            return 1                        # the store advances the epoch itself
        n = 1 + self.spec.replicas if self.path == "gather" else 1
        return n + (1 if with_epoch else 0)

    def views(self, layer):
        x = self.rows[layer]
        return x[:, :512], x[:, 512:576], x[:, 576:704]

    def launch_layers(self, with_epoch: bool = True):
        for layer in range(self.spec.layers):
            self.launch_layer(layer, with_epoch)

    def launch_layer(self, layer: int, with_epoch: bool = True):
        """One layer's publication.  On the publish path the single fused
        launch stores and advances the epoch, whatever with_epoch says."""
        lat, rope, idx = self.views(layer)
        if self.path == "publish":
            kvpub.store_mla_fp8_publish(lat, rope, idx, self.slots[layer], self.main[layer],
                                        self.idx[layer], self.epoch, self.done,
                                        self.spec.num_blocks, invalid_count=self.invalid)
            return
        if self.path == "gather":
            kvpub.gather_insert(lat, rope, idx, self.slots[layer], self.main[layer],
                                self.idx[layer], self.workspace, self.spec.num_blocks,
                                invalid_count=self.invalid)
        else:
            store = kvpub.store_mla_bf16 if self.spec.bf16_cache else kvpub.store_mla_fp8
            store(lat, rope, idx, self.slots[layer], self.main[layer], self.idx[layer],
                  self.spec.num_blocks, invalid_count=self.invalid)
        if with_epoch:
            kvpub.epoch_advance(self.epoch)

    def prepared_calls(self):
        """Every layer's calls with their arguments marshalled once (for an
        eager loop): store + epoch advance, or the fused store + epoch."""
        if self.path == "gather" or self.spec.bf16_cache:
            raise SystemExit("--eager times the direct and publish paths of the fp8 cache")
        calls = []
        for layer in range(self.spec.layers):
            lat, rope, idx = self.views(layer)
            args = (lat, rope, idx, self.slots[layer], self.main[layer], self.idx[layer])
            if self.path == "publish":
                calls.append(kvpub.prepare_store_mla_fp8_publish(
                    *args, self.epoch, self.done, self.spec.num_blocks,
                    invalid_count=self.invalid))
            else:
                calls.append(kvpub.prepare_store_mla_fp8(
                    *args, self.spec.num_blocks, invalid_count=self.invalid))
                calls.append(kvpub.prepare_epoch_advance(self.epoch))
        return calls

    def capture(self, with_epoch: bool = True):
        """One graph of all layers: store (+ epoch advance) per layer."""
        self.launch_layers(with_epoch=False)    # load the kernels before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.launch_layers(with_epoch)
        return g

    def capture_end_to_end(self):
        """One graph of a whole step from host memory: the slot maps and each
        layer's pinned host rows are copied on a side stream, layer by layer,
        while the stores of the layers already copied run; the epoch is read
        back into pinned host memory at the end."""
        L = self.spec.layers
        self.host_epoch = torch.zeros(1, dtype=torch.int64, pin_memory=True)
        copy_stream = torch.cuda.Stream()
        ready = [torch.cuda.Event() for _ in range(L)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            main = torch.cuda.current_stream()
            copy_stream.wait_stream(main)
            with torch.cuda.stream(copy_stream):
                self.slots.copy_(self.host_slots, non_blocking=True)
                for layer in range(L):
                    self.rows[layer].copy_(self.host_rows[layer], non_blocking=True)
                    ready[layer].record(copy_stream)
            for layer in range(L):
                main.wait_event(ready[layer])
                self.launch_layer(layer)
            self.host_epoch.copy_(self.epoch, non_blocking=True)
            main.wait_stream(copy_stream)
        return g


def check_direct_equals_gather(step: Step):
    """Before any timing: layer 0 published directly must leave the same
    bytes as the unfused gather-then-insert path on the same inputs ("byte-
    exact against gather-then-insert oracles before timing", as on
    "[Kernel][PCP] Publish replicated KV updates through PyTorch symmetric
    memory", Correctness and current-head validation)."""
    if step.spec.bf16_cache:
        return None
    lat, rope, idx = step.views(0)
    nb = step.spec.num_blocks
    direct_main = [torch.full_like(c, inputs.GUARD_BYTE) for c in step.main[0]]
    direct_idx = [torch.full_like(c, inputs.GUARD_BYTE) for c in step.idx[0]]
    kvpub.store_mla_fp8(lat, rope, idx, step.slots[0], direct_main, direct_idx, nb)
    gather_main = [torch.full_like(c, inputs.GUARD_BYTE) for c in step.main[0]]
    gather_idx = [torch.full_like(c, inputs.GUARD_BYTE) for c in step.idx[0]]
    ws = torch.empty(kvpub.gather_workspace_bytes(step.num_tokens), dtype=torch.uint8,
                     device=step.dev)
    kvpub.gather_insert(lat, rope, idx, step.slots[0], gather_main, gather_idx, ws, nb)
    torch.cuda.synchronize()
    same = all(torch.equal(a, b) for a, b in zip(direct_main + direct_idx,
                                                 gather_main + gather_idx))
    if not same:
        raise RuntimeError("direct publication and gather-then-insert disagree on layer 0")
    return True


def time_graph(g, steps, warmup):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    start.record()
    for _ in range(steps):
        g.replay()
    end.record()
    torch.cuda.synchronize()
    t1 = time.monotonic()
    barrier()
    return start.elapsed_time(end), t0, t1


def time_eager(calls, steps, warmup):
    """K steps of the calls issued one by one from the host (no graph), with
    CUDA events around them: the host's cost per call shows in the time.
    Each call gets the current stream's raw handle, looked up once."""
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(warmup):
        for c in calls:
            c(stream)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    start.record()
    for _ in range(steps):
        for c in calls:
            c(stream)
    end.record()
    torch.cuda.synchronize()
    t1 = time.monotonic()
    barrier()
    return start.elapsed_time(end), t0, t1


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(x: float) -> float:
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        t = torch.tensor([x], dtype=torch.float64,
                         device="cuda" if torch.distributed.get_backend() == "nccl" else "cpu")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())
    return x


def whole_job_rate(world: int, units_per_rank: float, ms_per_step_max: float) -> float:
    """Weak scaling: every rank processes the same per-rank work in each step,
    so the job's rate is all ranks' units over the slowest rank's time."""
    return world * units_per_rank / (ms_per_step_max / 1e3)


def e2e_measure(step: Step, steps: int, warmup: int):
    """Through the public API with host inputs: every step copies all layers'
    pinned host rows and slot maps to the device, runs every store and epoch
    advance, and reads the epoch back to pinned host memory."""
    h2d = step.host_rows.numel() * 2 + step.host_slots.numel() * 8
    d2h = 8
    g = step.capture_end_to_end()
    # the transfer floor: this machine's host->device rate for the same bytes
    for _ in range(2):
        step.rows.copy_(step.host_rows, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        step.rows.copy_(step.host_rows, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    h2d_gbs = 3 * step.host_rows.numel() * 2 / e0.elapsed_time(e1) / 1e6
    before = int(step.epoch.item())
    ms, _, _ = time_graph(g, steps, warmup)
    after = int(step.host_epoch.item())
    if after != before + step.spec.layers * (warmup + steps):
        raise RuntimeError(f"end-to-end epoch read back {after}, expected "
                           f"{before + step.spec.layers * (warmup + steps)}")
    return ms, h2d, d2h, h2d_gbs


def cpu_model() -> str:
    """The host CPU's model name (/proc/cpuinfo, else lscpu, else platform)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


class OracleLeg:
    """The CPU-baseline leg: the oracle as it stands (one thread) on a
    bounded sample of the benchmark's own inputs.  The bytes it computes are
    also compared with the GPU's timed buffers before any timing ("byte-
    exact against gather-then-insert oracles before timing", as on
    "[Kernel][PCP] Publish replicated KV updates through PyTorch symmetric
    memory", Correctness and current-head validation).  Rank 0 of a
    single-rank run only."""

    def __init__(self):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.elapsed = 0.0          # oracle seconds on the headline workload
        self.row_replicas = 0
        self.layers = []
        self.checked = {}

    def _store(self, w, replicas, num_blocks):
        main, idx = self.oracle.new_caches(replicas, num_blocks, inputs.GUARD_BYTE)
        t = time.perf_counter()
        n, _ = self.oracle.store_mla_fp8(w.kv_latent, w.k_rope, w.index_k, w.slot_mapping,
                                         main, idx, num_blocks)
        return main, idx, n, time.perf_counter() - t

    def check(self, name: str, w, gpu_main, gpu_idx, replicas: int, num_blocks: int,
              headline_layer: int | None = None):
        """Compare one launch's GPU caches (every replica's whole buffer) with
        the oracle's bytes; raise on any difference."""
        main, idx, n, dt = self._store(w, replicas, num_blocks)
        if headline_layer is not None:
            self.elapsed += dt
            self.row_replicas += n * replicas
            self.layers.append(headline_layer)
        for r in range(replicas):
            for got, want, what in ((gpu_main[r], main[r], "Main"), (gpu_idx[r], idx[r], "Indexer")):
                if not np.array_equal(got.cpu().numpy(), want):
                    raise RuntimeError(f"{name}: {what} cache of replica {r} differs from "
                                       "the oracle")
        self.checked[name] = f"{replicas} replicas x (Main + Indexer), whole buffers"

    def fill(self, budget_s: float):
        """More headline layers, timed, until about budget_s oracle seconds."""
        slots = inputs.layer_slot_mapping()
        layer = 1
        while self.elapsed < budget_s and layer < LAYERS:
            if layer not in self.layers:
                _, _, n, dt = self._store(inputs.prefill_layer(layer, slots), R, NUM_BLOCKS)
                self.elapsed += dt
                self.row_replicas += n * R
                self.layers.append(layer)
            layer += 1

    def baseline(self):
        return {"value": self.row_replicas / self.elapsed, "unit": UNIT, "cores": 1,
                "kind": "oracle",
                "sample": f"{len(self.layers)} of {LAYERS} layers of {WORKLOAD} "
                          f"({self.row_replicas // R} rows x {R} replicas), scalar C oracle, "
                          f"1 thread, {self.elapsed:.1f} s",
                "host_cpus": os.cpu_count(), "cpu_model": cpu_model()}


def roofline_entry(spec: Spec, step: Step, store_ms: float, steps: int, peak: float,
                   clocks: dict, checked: bool):
    """One workload's store-kernel figures: mean launch time from a graph of
    all its store launches, algorithmic bytes per launch, GB/s, fraction of
    the measured copy peak."""
    L = spec.layers
    per_launch = sum(store_bytes(step.num_tokens, v, spec.replicas, spec.bf16_cache)
                     for v in step.valid) / L
    kernel_ms = store_ms / (steps * L)
    achieved = per_launch / (kernel_ms / 1e3) / 1e9
    return {"kernel": f"store_mla_{'bf16' if spec.bf16_cache else 'fp8'}_kernel<{spec.replicas}>",
            "rows_per_launch": step.num_tokens, "valid_rows_per_launch": step.valid[0],
            "replicas": spec.replicas, "blocks_per_replica": spec.num_blocks,
            "launches_per_step": L, "kernel_us": round(kernel_ms * 1e3, 3),
            "algorithmic_bytes": int(round(per_launch)), "achieved": round(achieved, 1),
            "unit": "GB/s", "frac": round(achieved / peak, 4), "clocks": clocks,
            "oracle_checked_before_timing": checked, "note": spec.note}


# the bandwidth-bound workloads timed after the headline, each one
# launch per buffer copy, copies distinct so a step exceeds L2
SIDE_WORKLOADS = ("prefill_c16x1024", "capacity_706624")


def run_ours(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kbuild.build()
    kvpub.lib()
    spec = SPECS[args.workload]()
    if args.layers is not None:
        if not 1 <= args.layers <= spec.layers:
            raise SystemExit(f"--layers must be in 1..{spec.layers}")
        spec.layers = args.layers
        spec.note += f" (first {args.layers} layers only)"
    if args.replicas is not None:
        if not 1 <= args.replicas <= kvpub.MAX_REPLICAS:
            raise SystemExit(f"--replicas must be in 1..{kvpub.MAX_REPLICAS}")
        spec.replicas = args.replicas
        spec.note += f" ({args.replicas} replicas)"
    if args.path != "direct" and spec.bf16_cache:
        raise SystemExit(f"the {args.path} path exists for the fp8 cache only")
    leg = OracleLeg() if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    step = Step(dev, spec, args.path)
    L, Rr = spec.layers, spec.replicas
    checked = check_direct_equals_gather(step)
    g = step.capture(with_epoch=True)
    g_store = step.capture(with_epoch=False)
    # one replay fills the timed buffers; the oracle checks them before timing
    g.replay()
    torch.cuda.synchronize()
    oracle_checked = False
    if leg is not None and spec.name == WORKLOAD and args.path in ("direct", "publish"):
        for layer in sorted({0, L - 1}):
            w = spec.make(layer)
            leg.check(f"{WORKLOAD}[{layer}]", w, step.main[layer], step.idx[layer], Rr,
                      spec.num_blocks, headline_layer=layer)
        oracle_checked = True
    peak, peak_kind = measured_peak()
    epoch_before = int(step.epoch.item())
    with ClockSampler(local) as sampler:
        if args.eager:
            total_ms, t0, t1 = time_eager(step.prepared_calls(), args.steps, args.warmup)
        else:
            total_ms, t0, t1 = time_graph(g, args.steps, args.warmup)
        epoch_after = int(step.epoch.item())
        store_ms, s0, s1 = time_graph(g_store, args.steps, args.warmup)
        clocks = sampler.summary(t0, t1)
        store_clocks = sampler.summary(s0, s1)
        total_ms = max_over_ranks(total_ms)
        store_ms = max_over_ranks(store_ms)
        ms_per_step = total_ms / args.steps
        expected = L * (args.warmup + args.steps)
        if epoch_after - epoch_before != expected:
            raise RuntimeError(f"the epoch advanced by {epoch_after - epoch_before} over the "
                               f"timed replays, not {expected}: launches were lost")

        rows_x_r = sum(step.valid) * Rr
        value = whole_job_rate(world, rows_x_r, ms_per_step)
        if args.path == "gather":
            launch_bytes = [gather_insert_bytes(step.num_tokens, v, Rr) for v in step.valid]
            kernel_name = f"gather_rows_kernel + {Rr} x store_mla_fp8_kernel<1> (per layer)"
        elif args.path == "publish":
            launch_bytes = [store_bytes(step.num_tokens, v, Rr) for v in step.valid]
            kernel_name = f"store_mla_fp8_publish_kernel<{Rr}>"
        else:
            launch_bytes = [store_bytes(step.num_tokens, v, Rr, spec.bf16_cache)
                            for v in step.valid]
            kernel_name = f"store_mla_{'bf16' if spec.bf16_cache else 'fp8'}_kernel<{Rr}>"
        per_launch = sum(launch_bytes) / L
        kernel_ms = store_ms / (args.steps * L)
        timing = (f"CUDA events around {args.steps} replays of a graph of the same {L} layers' "
                  f"store launches (no separate epoch kernels) / {args.steps * L} layers, "
                  "gaps included")
        achieved = per_launch / (kernel_ms / 1e3) / 1e9
        traffic = (profiled_traffic()
                   if (spec.name == WORKLOAD and args.path == "direct" and Rr == R) else None)
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                    "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                    "kernel": kernel_name, "algorithmic_bytes": int(round(per_launch)),
                    "kernel_us": round(kernel_ms * 1e3, 2),
                    "peak_source": f"{peak_kind} hbm_gbs", "timing": timing,
                    "traffic_source": (f"{os.path.relpath(TRAFFIC_JSON, ROOT)} (ncu, "
                                       f"{TRAFFIC_LAYERS}-layer run of the same launches)"
                                       if traffic is not None else None)}

        e2e = None
        if not args.no_e2e:
            e2e_steps = max(3, min(args.steps, 50))
            e2e_ms, h2d, d2h, h2d_gbs = e2e_measure(step, e2e_steps,
                                                    max(1, min(args.warmup, 3)))
            e2e_ms = max_over_ranks(e2e_ms)
            floor_ms = h2d / (h2d_gbs * 1e6)
            e2e = {"value": whole_job_rate(world, rows_x_r, e2e_ms / e2e_steps), "unit": UNIT,
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                   "ms_per_step": round(e2e_ms / e2e_steps, 4), "steps": e2e_steps,
                   "h2d_gbs_measured": round(h2d_gbs, 1),
                   "transfer_floor_ms": round(floor_ms, 4),
                   "frac_of_transfer_floor": round(floor_ms / (e2e_ms / e2e_steps), 4)}

        workloads = {}
        if spec.name == WORKLOAD and args.path == "direct" and not spec.bf16_cache:
            workloads[WORKLOAD] = roofline_entry(spec, step, store_ms, args.steps, peak,
                                                 store_clocks, oracle_checked)
        launches_per_step = step.launches_per_layer() * L
        rows_per_layer, valid_per_layer = step.num_tokens, step.valid[0]
        l2_note = ("inputs larger than L2: one step touches "
                   f"{sum(launch_bytes) / 1e9:.2f} GB")
        del g, g_store, step
        torch.cuda.empty_cache()
        if not args.no_workloads and spec.name == WORKLOAD and args.path == "direct":
            for name in SIDE_WORKLOADS:
                workloads[name] = time_side_workload(dev, name, args, peak, sampler, leg)

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": spec.name, "layers": L, "rows_per_layer": rows_per_layer,
                   "valid_rows_per_layer": valid_per_layer, "replicas": Rr, "blocks_per_replica": spec.num_blocks,
                   "launches_per_step": launches_per_step, "path": args.path,
                   "graph": not args.eager,
                   "parallelism": f"replicas only x{world}", "note": spec.note,
                   "direct_equals_gather_before_timing": checked,
                   "oracle_checked_before_timing": oracle_checked,
                   "l2": l2_note,
                   "hbm_gbs_step": round(sum(launch_bytes) / (ms_per_step / 1e3) / 1e9, 1)},
        "roofline": roofline,
        "workloads": workloads or None,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if leg is not None:
        leg.fill(args.cpu_budget)
        out["cpu_baseline"] = leg.baseline()
        out["oracle_check"] = leg.checked
    if rank == 0:
        print(json.dumps(out), flush=True)


def time_side_workload(dev, name: str, args, peak: float, sampler, leg):
    """Time one more bandwidth-bound workload's store launches (a graph of
    all its buffer copies, no epoch kernels) after checking its first copy
    against the oracle; free its buffers afterwards."""
    spec = SPECS[name]()
    step = Step(dev, spec)
    g = step.capture(with_epoch=False)
    g.replay()
    torch.cuda.synchronize()
    checked = False
    if leg is not None:
        leg.check(f"{name}[copy 0]", spec.make(0), step.main[0], step.idx[0], spec.replicas,
                  spec.num_blocks)
        checked = True
    store_ms, t0, t1 = time_graph(g, args.steps, args.warmup)
    store_ms = max_over_ranks(store_ms)
    entry = roofline_entry(spec, step, store_ms, args.steps, peak, sampler.summary(t0, t1),
                           checked)
    del g, step
    torch.cuda.empty_cache()
    return entry


# ------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle as it stands, on the same workload and metric."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    slots = inputs.layer_slot_mapping()
    w = inputs.prefill_layer(0, slots)
    main, idx = oracle.new_caches(R, NUM_BLOCKS)
    # size each step so warmup + steps take about --ref-seconds in total
    t = time.perf_counter()
    oracle.store_mla_fp8(w.kv_latent[:256], w.k_rope[:256], w.index_k[:256],
                         w.slot_mapping[:256], main, idx, NUM_BLOCKS)
    per_row = (time.perf_counter() - t) / 256
    rows = int(min(ROWS, max(64, args.ref_seconds / (args.steps + args.warmup) / per_row)))
    sample = slice(0, rows)
    valid = int(np.count_nonzero(w.slot_mapping[sample] >= 0))
    call = (w.kv_latent[sample], w.k_rope[sample], w.index_k[sample], w.slot_mapping[sample],
            main, idx, NUM_BLOCKS)
    for _ in range(args.warmup):
        oracle.store_mla_fp8(*call)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.store_mla_fp8(*call)
    elapsed = time.perf_counter() - t
    value = valid * R * args.steps / elapsed
    desc = (f"{rows} of {ROWS} rows of layer 0 per step, scalar C oracle, 1 thread")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(elapsed / args.steps * 1e3, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "config": {"workload": WORKLOAD, "layers": LAYERS, "rows_per_layer": ROWS,
                      "replicas": R, "blocks_per_replica": NUM_BLOCKS},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                            "sample": desc, "host_cpus": os.cpu_count(), "cpu_model": cpu_model()},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def free_port() -> int:
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        return sock.getsockname()[1]


def relaunch(n: int) -> int:
    """Run this script again under torch.distributed.run with n local ranks
    (one per GPU) and the same arguments; return its exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1",
           "--master-port", str(free_port()), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline field")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the CPU-baseline leg (and with it the oracle check)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time the headline workload only")
    ap.add_argument("--layers", type=int, default=None,
                    help="publish only the first K layers (a small profiling case)")
    ap.add_argument("--replicas", type=int, default=None,
                    help="store into R replicas instead of the workload's own count")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: about this many seconds of oracle work in all")
    ap.add_argument("--write-traffic", metavar="CSV",
                    help="write the roofline's DRAM traffic record from an ncu CSV and exit")
    ap.add_argument("--path", choices=["direct", "publish", "gather"], default="direct",
                    help="direct publication with a separate epoch launch (the measured "
                         "line), the store + epoch fused in one launch, or the unfused "
                         "gather-then-insert path, for comparison")
    ap.add_argument("--eager", action="store_true",
                    help="time the step as calls issued one by one from the host, "
                         "arguments marshalled once, instead of a CUDA graph replay")
    ap.add_argument("--workload", choices=sorted(SPECS), default=WORKLOAD,
                    help="the default is the measured line; the others are for "
                         "per-workload roofline figures and ncu captures")
    args = ap.parse_args()
    if args.write_traffic:
        print(json.dumps(write_traffic(args.write_traffic)))
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.gpus < 1:
        raise SystemExit("--gpus must be at least 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        raise SystemExit(relaunch(args.gpus))
    world, rank, local = dist_env()
    if world != args.gpus and rank == 0:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE is {world}; using {world} ranks",
              file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        run_ours(args)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
