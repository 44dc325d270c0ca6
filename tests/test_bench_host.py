"""Host-side pieces of bench.py that need no GPU: the ncu CSV reader behind
the roofline's DRAM traffic, the traffic record it writes, and the record's
source-hash gate."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
          '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
          '"Metric Value"')


def _row(launch, kernel, metric, unit, value):
    return (f'"{launch}","1","python3","127.0.0.1","{kernel}","1","7","(256, 1, 1)",'
            f'"(608, 1, 1)","0","10.3","Command line profiler metrics","{metric}","{unit}",'
            f'"{value}"')


def _csv(tmp_path):
    store = "void kvpub::store_mla_fp8_kernel<4>(kvpub::StoreArgs)"
    lines = ["==PROF== Connected to process 1", HEADER,
             _row(14, store, "dram__bytes_read.sum", "byte", "20,000,000"),
             _row(14, store, "dram__bytes_write.sum", "byte", "44000000"),
             _row(15, "void kvpub::epoch_advance_kernel(unsigned long long*)",
                  "dram__bytes_read.sum", "byte", "64"),
             _row(16, store, "dram__bytes_read.sum", "Mbyte", "21"),
             _row(16, store, "dram__bytes_write.sum", "Kbyte", "46000")]
    path = tmp_path / "dram.csv"
    path.write_text("\n".join(lines) + "\n")
    return str(path)


def test_reader_keeps_the_store_launches_and_scales_units(tmp_path):
    got = bench.read_ncu_csv(_csv(tmp_path))
    assert sorted(got) == [14, 16]
    assert got[14] == {"dram__bytes_read.sum": 20e6, "dram__bytes_write.sum": 44e6}
    assert got[16] == {"dram__bytes_read.sum": 21e6, "dram__bytes_write.sum": 46e6}


def test_traffic_record_is_per_launch_and_gated_on_the_source_hash(tmp_path, monkeypatch):
    out = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(out))
    rec = bench.write_traffic(_csv(tmp_path))
    assert rec["launches"] == 2
    assert rec["dram_bytes_read_per_launch"] == 20_500_000
    assert rec["dram_bytes_write_per_launch"] == 45_000_000
    assert rec["dram_bytes_per_launch"] == 65_500_000
    assert rec["algorithmic_bytes_per_launch"] == 8 * 14336 + 14336 * (1408 + 788 * 4)
    assert json.loads(out.read_text()) == rec
    assert bench.profiled_traffic() == 65_500_000
    stale = dict(rec, kernel_source_sha256_16="0" * 16)
    out.write_text(json.dumps(stale))
    assert bench.profiled_traffic() is None


def test_committed_traffic_record_if_present_matches_its_command():
    if not os.path.exists(bench.TRAFFIC_JSON):
        pytest.skip("no traffic record committed")
    rec = json.load(open(bench.TRAFFIC_JSON))
    assert rec["command"] == bench.TRAFFIC_CMD
    assert rec["launches"] == bench.TRAFFIC_LAYERS


def test_kernel_hash_ignores_comments_but_not_code():
    a = "int x = 1; // one\n/* block\n comment */ int y =  2;\n"
    b = "int x = 1;\nint y = 2; // edited comment\n"
    c = "int x = 1;\nint y = 3;\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_reader_refuses_a_file_without_a_metrics_table(tmp_path):
    path = tmp_path / "empty.csv"
    path.write_text("==PROF== Connected to process 1\n==ERROR== nothing profiled\n")
    with pytest.raises(SystemExit, match="no ncu --csv metrics table"):
        bench.read_ncu_csv(str(path))


def test_oracle_leg_checks_every_byte_and_times_headline_layers_only():
    """The bench's pre-timing check: buffers equal to the oracle's bytes pass,
    one flipped byte anywhere raises; only headline layers count toward the
    CPU baseline."""
    import numpy as np
    import torch

    import oracle
    from replication_token_warp_gb300 import inputs

    w = inputs.make(0)
    main, idx = oracle.new_caches(w.num_replicas, w.num_blocks, inputs.GUARD_BYTE)
    oracle.store_mla_fp8(w.kv_latent, w.k_rope, w.index_k, w.slot_mapping, main, idx,
                         w.num_blocks)
    got_main = [torch.from_numpy(m.copy()) for m in main]
    got_idx = [torch.from_numpy(x.copy()) for x in idx]
    leg = bench.OracleLeg()
    leg.check("tiny", w, got_main, got_idx, w.num_replicas, w.num_blocks)
    assert leg.row_replicas == 0 and leg.layers == []
    leg.check("tiny as layer 5", w, got_main, got_idx, w.num_replicas, w.num_blocks,
              headline_layer=5)
    assert leg.layers == [5] and leg.row_replicas == w.num_valid * w.num_replicas
    got_idx[0][int(np.flatnonzero(idx[0] != inputs.GUARD_BYTE)[-1])] ^= 1
    with pytest.raises(RuntimeError, match="Indexer cache of replica 0 differs"):
        leg.check("tiny", w, got_main, got_idx, w.num_replicas, w.num_blocks)
