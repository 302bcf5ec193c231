"""Host-side logic of bench.py: the N>1 aggregation over ranks (two gloo ranks on CPU),
clock-log parsing, peaks and the recorded-traffic guard."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r processed 10 units in r + 1 seconds: the job did 20 units in 2 s (the slowest)
    value, slowest = bench.aggregate_throughput(10.0, rank + 1.0, world)
    bench.barrier(world)
    out[rank] = (value, slowest, bench.max_over_ranks(float(rank * 7), world))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        assert out[r] == (10.0, 2.0, 7.0)


def test_single_rank_aggregate_is_identity():
    assert bench.aggregate_throughput(5.0, 2.0, 1) == (2.5, 2.0)


def test_clock_summary_parses_reasons(tmp_path):
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "c.csv")
    cs.proc = object()
    with open(cs.path, "w") as f:
        f.write("0, 1900, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 1950, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 300, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    s = cs.summary()
    assert s["sm_max_mhz"] == 2070 and s["sm_mhz"] == 1925 and s["reasons"] == ["sw_power_cap"]


def test_recorded_traffic_requires_matching_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    monkeypatch.setitem(bench.KERNEL_SOURCES, "prefill", ("k.cu",))
    sha = bench.source_sha("k.cu")
    (prof / "dram_traffic.json").write_text(json.dumps(
        {"w": {"source_sha": sha, "dram_bytes_per_launch": 123}}))
    assert bench.recorded_traffic("prefill", "w") == 123
    src.write_text("kernel v2")
    assert bench.recorded_traffic("prefill", "w") is None


def test_measured_peaks_reads_driver_file():
    p = bench.measured_peaks()
    assert p["hbm_gbs"] > 1000 and p["bf16_tflops"] > 100


def test_packed_prefill_flops_count_the_allowed_pairs():
    """The benchmark's FLOP count of a packed workload equals 4 d hq times the allowed
    (query, key) pairs counted one by one with the oracle's mask predicate."""
    import oracle
    from workloads import configs as C

    pw = C.PackedPrefillWorkload("tiny_packed", 2, 1, 8, 5, 3, 40, 17, seed=5)
    cu_q, cu_k = pw.offsets()
    pairs = 0
    for s in range(pw.nseq):
        nq, nk = cu_q[s + 1] - cu_q[s], cu_k[s + 1] - cu_k[s]
        for i in range(nq):
            qp = oracle.q_pos(i, nq, nk)
            pairs += sum(oracle.allowed(j, nk, qp, True, 0) for j in range(nk))
    assert pw.flops() == 4 * pw.d * pw.hq * pairs


def test_cpu_baselines_run_on_small_host_inputs(monkeypatch):
    """The oracle timing legs of the benchmark on CPU tensors of small workloads: the full
    and the sampled prefill, the packed prefill and every decode variant the benchmark
    times (their sampling, page compaction and byte counts)."""
    import torch

    from workloads import configs as C

    cpu = torch.device("cpu")
    small = C.PrefillWorkload("small", 1, 2, 1, 300, 300, 64, True, 0, seed=3)
    big = C.PrefillWorkload("big", 1, 16, 4, 1024, 1024, 64, True, 200, seed=4)
    monkeypatch.setattr(bench, "FULL_PREFILL_FLOP", 1e8)  # small is below it, big above
    for w, full in ((small, True), (big, False)):
        q, k, v = C.prefill_inputs_torch(w, cpu)
        ent = bench.cpu_prefill(w, q, k, v, 2, C.sink_logits(w.hq))
        assert ent["value"] > 0 and ent["kind"] == "oracle" and ent["cores"] == 2
        assert ("extrapolated_full_s" in ent) == (not full)
    pw = C.PackedPrefillWorkload("small_packed", 4, 2, 64, 5, 20, 200, 50, seed=9)
    q, k, v = C.prefill_inputs_torch(pw.as_prefill(), cpu)
    assert bench.cpu_packed(pw, q, k, v, 2)["value"] > 0
    wd = C.DecodeWorkload("small_decode", 3, 8, 2, 128, 4, len_lo=40, len_hi=300, seed=8)
    t = C.decode_inputs_torch(wd, cpu)
    te = C.decode_inputs_e4m3_torch(wd, cpu)
    inv = bench.rope_inv_freq(wd.d)
    for kw, tt in ((dict(), t), (dict(sink=C.sink_logits(wd.hq)), t), (dict(e4m3=True), te),
                   (dict(window=64, inv_freq=inv), t)):
        ent = bench.cpu_decode(wd, tt, 2, **kw)  # small caches: the whole workload
        assert ent["value"] > 0 and ent["unit"] == "GB/s" and "whole workload" in ent["sample"]
        assert "extrapolated_full_s" not in ent
    monkeypatch.setattr(bench, "DECODE_FULL_MAX_BYTES", 0)  # as for caches too large to copy
    for kw, tt in ((dict(), t), (dict(e4m3=True), te), (dict(window=64, inv_freq=inv), t)):
        ent = bench.cpu_decode(wd, tt, 2, **kw)
        assert ent["value"] > 0 and "2 of 3 sequences" in ent["sample"]
        assert ent["extrapolated_full_s"] > 0


def test_final_line_summary_is_compact():
    ent = {"value": 1454.123, "unit": "TFLOP/s", "ms_per_step": 6.0512, "roofline": {"frac": 0.7461},
           "cpu_baseline": {"value": 0.0351234}}
    assert bench.compact(ent) == {"v": 1454.1, "u": "TFLOP/s", "ms": 6.0512, "frac": 0.746,
                                  "cpu": 0.0351}
    assert "error" in bench.compact({"workload": "x", "error": "device error"})
