"""Host-side logic of bench.py on CPU: the max/sum over ranks of the
multi-replica run (gloo, world size 2), clock-log parsing, and the rule that
a recorded DRAM-traffic figure is dropped once the kernel source changes."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out_path):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    step_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    tokens = 73
    mx = bench.reduce_max_over_ranks(step_ms, world)
    sm = bench.reduce_sum_over_ranks(100.0 * (rank + 1), world)
    bench.barrier(world)
    value = tokens * world / (mx / 1e3)
    with open(f"{out_path}.{rank}", "w") as f:
        json.dump({"max": mx, "sum": sm, "value": value}, f)
    dist.destroy_process_group()


def test_two_rank_reduction_gloo(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    out = str(tmp_path / "r")
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    res = [json.load(open(f"{out}.{r}")) for r in range(2)]
    for r in res:
        assert r["max"] == 15.0          # max over ranks, on every rank
        assert r["sum"] == 300.0
        assert abs(r["value"] - 73 * 2 / 0.015) < 1e-6  # all ranks' tokens / slowest rank


def test_single_rank_reduction_is_identity():
    assert bench.reduce_max_over_ranks(3.5, 1) == 3.5
    assert bench.reduce_sum_over_ranks(3.5, 1) == 3.5


def test_clock_log_parsing(tmp_path):
    import datetime
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.path = str(tmp_path / "c.csv")
    base = datetime.datetime(2026, 1, 2, 3, 4, 5)

    def stamp(dt_s):
        return (base + datetime.timedelta(seconds=dt_s)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]

    with open(s.path, "w") as f:
        f.write(f"{stamp(0.0)}, 0, 345, 2070, 100.0, 0x0000000000000001\n")    # before the region
        f.write(f"{stamp(1.00)}, 0, 1965, 2070, 900.1, 0x0000000000000000\n")
        f.write(f"{stamp(1.05)}, 0, 1980, 2070, 950.2, 0x0000000000000004\n")  # sw_power_cap
        f.write(f"{stamp(1.10)}, 0, 1995, 2070, 950.2, 0x0000000000000000\n")
        f.write(f"{stamp(3.0)}, 0, 345, 2070, 100.0, 0x0000000000000020\n")    # after: ignored
        f.write("garbage line\n")
    s.t0 = base.timestamp() + 0.99
    s.t1 = base.timestamp() + 1.11
    c = s.parse()
    assert c["samples"] == 3 and c["sm_max_mhz"] == 2070
    assert c["sm_mhz"] == 1980
    assert c["reasons"] == ["sw_power_cap"]


def test_traffic_record_requires_same_source(tmp_path, monkeypatch):
    csrc = tmp_path / "mxfp4_routed_expert_k3_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"gateup_gemv_kernel": {"source": "k.cu", "source_sha": bench.source_sha(str(csrc / "k.cu")),
                                  "workload": "w", "dram_bytes_per_active_expert": 123.0}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("gateup_gemv_kernel", "w") == 123.0
    assert bench.recorded_traffic("gateup_gemv_kernel", "other") is None
    (csrc / "k.cu").write_text("kernel v2")
    assert bench.recorded_traffic("gateup_gemv_kernel", "w") is None
