"""Host logic of bench.py that needs no GPU: the max-over-ranks timing and the
whole-job aggregate under a 2-rank gloo process group, the clock-sample
parser, and the traffic record's source-hash check."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [12.5, 20.0][rank]
    mx = bench.aggregate_max(local_ms, dist)
    value = bench.whole_job_tflops(1e12, world, 10, mx)
    q.put((rank, mx, value))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, value in out:
        assert mx == 20.0  # every rank sees the slowest rank's time
        # 2 ranks x 10 steps x 1e12 FLOP over 20 ms
        assert value == pytest.approx(2 * 10 * 1e12 / 0.020 / 1e12)


def test_aggregate_without_process_group_is_identity():
    assert bench.aggregate_max(3.5, None) == 3.5
    assert bench.whole_job_tflops(1e12, 1, 1, 1000.0) == pytest.approx(1.0)


def test_clock_summary_parses_samples_and_reasons():
    s = bench.ClockSampler(0)
    s.lines = [
        "0, 2070, 2070, 650.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1300.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2010, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    ]
    r = s.summary(0)
    assert r["sm_mhz"] == 2010.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]
    assert r["samples"] == 3
    assert s.summary(3)["samples"] == 0


def test_traffic_record_requires_current_kernel_source(tmp_path, monkeypatch):
    from fa_inputs import workload

    for key, wname, other in (("sm103", "causal", "mha"), ("d256", "hd256", "causal")):
        name, src, _ = bench.BWD_KERNELS[key]
        rec = tmp_path / f"traffic_{key}.txt"
        rec.write_text(f"# comment\nkernel_sha256 {bench.kernel_sha(src)}\nbytes_per_launch_{wname} 1234\n")
        monkeypatch.setitem(bench.BWD_KERNELS, key, (name, src, str(rec)))
        w = workload(wname)
        assert bench.bwd_kernel(w)[0] == name
        assert bench.recorded_traffic(w) == 1234.0
        assert bench.recorded_traffic(w.with_(name=other)) is None
        rec.write_text(f"kernel_sha256 0000\nbytes_per_launch_{wname} 1234\n")
        assert bench.recorded_traffic(w) is None


def test_committed_traffic_records_match_the_kernel_sources():
    """The committed ncu DRAM figures were taken on the kernels as they are now:
    each record's hash is that of its kernel source, and it has a figure for
    the workloads bench.py reports it on."""
    from fa_inputs import workload

    for wname in ("causal", "long", "hd256"):
        w = workload(wname)
        traffic = bench.recorded_traffic(w)
        assert traffic is not None and traffic > 0, wname
        # at least the compulsory bytes: Q, K, V, dO read and dK, dV written once (bf16)
        assert traffic >= 6 * w.B * w.H * w.N * w.d * 2 * 0.9, wname
