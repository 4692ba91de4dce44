"""Host-side logic of bench.py on the CPU: the cross-rank aggregation (two gloo
ranks with different timings), the algorithmic work counts, the clock-sample
parsing and the traffic record's staleness check."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_varlen_flash_gb300 import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, nbytes = bench.aggregate_ranks(10.0 + 5.0 * rank, 1000 + rank, torch.device("cpu"))
    with open("%s.%d" % (out_path, rank), "w") as f:
        json.dump([ms, nbytes], f)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    out = str(tmp_path / "agg")
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        with open("%s.%d" % (out, r)) as f:
            ms, nbytes = json.load(f)
        assert ms == 15.0          # the slowest rank sets the job time
        assert nbytes == 2001      # every rank's bytes count


def test_aggregate_single_process_is_identity():
    assert bench.aggregate_ranks(3.5, 77, torch.device("cpu")) == (3.5, 77)


def test_workload_units_count_kv_once_per_kv_head():
    w = W.build("u", 8, 2, 64, 16, [1, 3], [40, 3], 8, 0.125, values=False, poison=False)
    nbytes, flops = bench.workload_units(w)
    kv = (40 + 3) * 2 * 64 * 2 * 2
    qo = 2 * 4 * 8 * 64 * 2
    meta = (3 + 1) * 4 + (2 * 2 + 1) * 4
    assert nbytes == kv + qo + meta
    # visible pairs: seq0 row0 sees 40 keys; seq1 rows see 1, 2, 3 keys
    assert flops == 4.0 * 64 * 8 * (40 + 6)


def test_clock_summary_parses_reasons():
    c = bench.ClockSampler(0)
    c.samples = [(1.0, "1900, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active"),
                 (1.1, "2000, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
                 (9.0, "500, 2070, 100.0, 0x0, Active, Not Active, Not Active, Not Active")]
    s = c.summary(1.0, 1.1)
    assert s["sm_mhz"] == 1950.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_traffic_record_goes_stale_when_the_kernel_changes(tmp_path, monkeypatch):
    rec = {"split_kernel": {"workload": "decode", "dram_bytes_per_launch": 123,
                            "source_sha256": bench.kernel_source_hash("split_kernel")}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.recorded_traffic("split_kernel", "decode") == 123
    assert bench.recorded_traffic("split_kernel", "chunked") is None
    rec["split_kernel"]["source_sha256"] = "0" * 64
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("split_kernel", "decode") is None


def test_dominant_kernel_follows_the_reported_path():
    assert bench.dominant_kernel("decode_tc+combine") == "decode_tc_kernel"
    assert bench.dominant_kernel("topk_tc+combine") == "topk_kernel"
    assert bench.dominant_kernel("tensor_core_cta2") == "prefill_cta2_kernel"
    assert bench.dominant_kernel("tensor_core_pair+combine") == "prefill_pair_kernel"
    assert bench.dominant_kernel("tensor_core_grid") == "prefill_grid_kernel"
    assert bench.dominant_kernel("split_kv+combine") == "split_kernel"


def test_workload_units_of_a_topk_workload_count_listed_keys():
    w = W.make("decode_topk", values=False)
    nbytes, flops = bench.workload_units(w)
    listed = 256 * 2048
    kv = listed * w.hk * w.d * 2 * 2
    qo = 2 * w.total_q * w.hq * w.d * 2
    meta = listed * 4 + w.total_q * 4 + (2 * w.num_seqs + 1) * 4
    assert nbytes == kv + qo + meta
    assert flops == 4.0 * w.d * w.hq * listed
