"""Host logic of bench.py, without a GPU: work counts, roofline selection, sharding and the
max-over-ranks time across two gloo ranks."""
import json
import os
import socket

import pytest

import bench


def test_fwd_work_counts_the_bench_workload():
    # 8 x 1536 x 2048 x 16, bf16 in, f32 out, h_last written, no h0
    w = bench.fwd_work(8, 1536, 2048, 16, in_bytes=2, out_bytes=4, h0=False, h_last=True)
    elems = 8 * 1536 * 2048
    assert w["elements"] == elems
    per_elem = 3 * 2 + 4                       # u, δ, z read; out written
    bc = 2 * 8 * 16 * 2048 * 2                 # B and C once per (b, n, t)
    small = 1536 * 16 * 4 + 2 * 1536 * 4       # A, D, Δ_bias
    h_last = 8 * 1536 * 16 * 4
    assert w["bytes"] == elems * per_elem + bc + small + h_last == 253_603_840
    assert w["mufu"] == elems * 20 and w["fp32"] == elems * 72
    assert w["sfu"] == {"ex2": elems * 18, "lg2": elems, "rcp": elems}


def test_bwd_work_counts_the_backward_of_the_bench_workload():
    # 8 x 1536 x 2048 x 16, bf16 inputs and dout; gradients du, dδ, dz in bf16, dB, dC fp32
    w = bench.bwd_work(8, 1536, 2048, 16, in_bytes=2, dout_bytes=2)
    elems = 8 * 1536 * 2048
    per_elem = 3 * 2 + 2 + 3 * 2               # u, δ, z, dout read; du, dδ, dz written
    bc = 8 * 16 * 2048 * (2 * 2 + 2 * 4)       # B, C read (bf16); dB, dC written (fp32)
    small = 2 * 1536 * 16 * 4 + 4 * 1536 * 4  # A, dA; D, Δ_bias, dD, dΔ_bias
    states = 3 * 8 * 1536 * 16 * 4             # h0, dh_last, dh0
    assert w["bytes"] == elems * per_elem + bc + small + states
    assert w["sfu"] == {"ex2": elems * 34, "lg2": elems, "rcp": 2 * elems}
    t = bench.roofline_times(w, sms=148, hbm_gbs=6493.4, sm_mhz=2032.0)
    assert t["mufu"] > t["hbm"]  # the backward is bound by its exponentials, as the forward is


def test_step_work_counts_the_decode_workload():
    w = bench.step_work(256, 5120, 16)
    rows = 256 * 5120
    assert w["bytes"] == rows * (2 * 16 * 4 + 3 * 2 + 4) + 2 * 256 * 16 * 2 + 5120 * 16 * 4 + 2 * 5120 * 4


def test_roofline_picks_the_slowest_resource():
    w = bench.fwd_work(8, 1536, 2048, 16)
    t = bench.roofline_times(w, sms=148, hbm_gbs=6516.4, sm_mhz=2032.0)
    assert t["mufu"] > t["fp32"] > t["hbm"]
    # N + 2 exponentials at 32 per clock per SM, the logarithm and the reciprocal at 16
    elems = 8 * 1536 * 2048
    want = elems * (18 / 32 + 1 / 16 + 1 / 16) / (148 * 2.032e9)
    assert abs(t["mufu"] - want) < 1e-12 and abs(t["mufu"] * 1e6 - 57.53) < 0.05
    e = bench.roofline_entry(w, t_kernel=2 * t["mufu"], sms=148, hbm_gbs=6516.4, sm_mhz=2032.0)
    assert e["bound"] == "alu" and e["resource"] == "mufu" and e["unit"] == "TFLOP/s"
    assert abs(e["frac"] - 0.5) < 1e-12
    assert abs(e["peak"] - 148 * 32 * 2.032e9 / 1e12) < 1e-9
    # the decode step is bound by HBM
    s = bench.step_work(256, 5120, 16)
    s = dict(s, mufu=s["elements"] * 20, fp32=s["elements"] * 72)
    e2 = bench.roofline_entry(s, t_kernel=1e-4, sms=148, hbm_gbs=6516.4, sm_mhz=2032.0)
    assert e2["bound"] == "hbm" and e2["unit"] == "GB/s"


@pytest.mark.parametrize("batch,world", [(8, 1), (8, 2), (7, 2), (3, 4), (16, 8), (5, 8)])
def test_shard_batch_partitions_the_batch(batch, world):
    ranges = [bench.shard_batch(batch, r, world) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == batch
    for (lo, hi), (lo2, _) in zip(ranges, ranges[1:]):
        assert hi == lo2 and hi >= lo
    sizes = [hi - lo for lo, hi in ranges]
    assert max(sizes) - min(sizes) <= 1


def test_aggregate_uses_the_slowest_rank():
    assert bench.aggregate([100, 100], [1.0, 2.0]) == 100.0


def test_measured_peaks_fallback(tmp_path):
    assert bench.measured_peaks(str(tmp_path / "missing.json"))[2] == "fallback"
    p = tmp_path / "peaks.json"
    p.write_text(json.dumps({"hbm_gbs": 6000.0, "sm_max_mhz": 2000.0}))
    assert bench.measured_peaks(str(p)) == (6000.0, 2000.0, "measured")


def test_recorded_traffic_needs_the_current_sources(tmp_path):
    p = tmp_path / "traffic.json"
    rec = {"selscan_fwd": {"w": {"source_hash": bench.kernel_source_hash("selscan_fwd"), "dram_bytes_per_launch": 123.0}},
           "selscan_step": {"w": {"source_hash": "stale", "dram_bytes_per_launch": 5.0}}}
    p.write_text(json.dumps(rec))
    assert bench.recorded_traffic("selscan_fwd", "w", str(p)) == 123.0
    assert bench.recorded_traffic("selscan_step", "w", str(p)) is None
    assert bench.recorded_traffic("selscan_fwd", "other", str(p)) is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lo, hi = bench.shard_batch(8 * world, rank, world)
        secs = 1.0 + rank  # rank 1 is the slow one
        t = bench.max_over_ranks(secs, dist, "cpu")
        value = (hi - lo) * 1536 * 2048 * world / t
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"lo": lo, "hi": hi, "t": t, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_take_the_max_time(tmp_path):
    import torch.multiprocessing as mp

    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.loads((tmp_path / f"r{r}.json").read_text()) for r in range(world)]
    assert [(r["lo"], r["hi"]) for r in res] == [(0, 8), (8, 16)]
    assert all(r["t"] == 2.0 for r in res)  # every rank sees the slowest rank's time
    assert res[0]["value"] == bench.aggregate([8 * 1536 * 2048] * 2, [1.0, 2.0])
