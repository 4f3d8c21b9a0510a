"""The benchmark's multi-rank host logic on CPU (gloo, world size 2): the timed region's
time is the max over ranks and the work is the sum over ranks."""
import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        t, u = bench.aggregate(elapsed_s=1.0 + rank, units=10.0 * (rank + 1))
        q.put((rank, t, u))
    finally:
        dist.destroy_process_group()


def test_aggregate_max_time_sum_units_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, t, u in res:
        assert t == 2.0 and u == 30.0


def test_aggregate_single_process_passthrough():
    import bench
    assert bench.aggregate(0.5, 7.0) == (0.5, 7.0)


def test_traffic_lookup_is_tied_to_the_kernel_source(tmp_path, monkeypatch):
    import json
    import bench
    k = "i8_gemm_kernel"
    rec = {"w": {"kernel": k, "source_sha256": bench.kernel_source_hash(k),
                 "dram_bytes_per_launch": 123.0}}
    f = tmp_path / "t.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.measured_traffic("w", k) == 123.0
    assert bench.measured_traffic("other", k) is None
    assert bench.measured_traffic("w", "gemv_i8_kernel") is None
    rec["w"]["source_sha256"] = "0" * 64
    f.write_text(json.dumps(rec))
    assert bench.measured_traffic("w", k) is None


def test_matmul_path_selection_follows_the_library_rule():
    import bench
    import synth
    assert bench.matmul_kernel(synth.WORKLOADS["decode_176b_t1"]) == "gemv_i8_kernel"
    assert bench.matmul_kernel(synth.WORKLOADS["decode_176b_t8"]) == "gemv_i8_kernel"
    assert bench.matmul_kernel(synth.WORKLOADS["tiny"]) == "gemv_mma_kernel"
    assert bench.matmul_kernel(synth.WORKLOADS["decode_176b_t64"]) == "i8_gemm_kernel"
    assert bench.matmul_kernel(synth.WORKLOADS["ffn_6.7b_up"]) == "i8_gemm_kernel"


def test_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    import bench
    src = "// header\nint f(int a) {  /* inline */ return a + 1; }\n\n// tail\n"
    for name in ("a.cu", "b.h"):
        (tmp_path / name).write_text(src)
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    monkeypatch.setitem(bench.KERNEL_SOURCES, "k", ("a.cu", "b.h"))
    h0 = bench.kernel_source_hash("k")
    (tmp_path / "a.cu").write_text("// other words\n" + src + "\n// more\n")
    assert bench.kernel_source_hash("k") == h0
    (tmp_path / "a.cu").write_text(src.replace("a + 1", "a + 2"))
    assert bench.kernel_source_hash("k") != h0


def test_roofline_bound_and_fraction_follow_the_workload():
    import bench
    import synth
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1500.0}
    w = synth.WORKLOADS["decode_176b_t8"]
    r = bench.roofline(w, 0.2, peaks, "test")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - bench.matmul_bytes(w) / 0.2e-3 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / 6000.0) < 1e-12
    w = synth.WORKLOADS["ffn_6.7b_up"]
    r = bench.roofline(w, 0.25, peaks, "test")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - bench.workload_ops(w) / 0.25e-3 / 1e12) < 1e-9
    # the zeropoint variant runs on the tensor-core kernel at every size; no traffic record
    r = bench.roofline(synth.WORKLOADS["decode_176b_t8"], 0.2, peaks, "test", zeropoint=True)
    assert r["kernel"].startswith("i8_gemm_kernel") and r["traffic"] is None


def test_cpu_baselines_run_the_oracle_on_bounded_samples():
    import bench
    import oracle
    import synth
    w = synth.WORKLOADS["tiny"]
    X, W, b = synth.make_x(w), synth.make_w(w), synth.make_bias(w)
    CB, SCB = oracle.quantize_weight(W)
    for zp in (False, True):
        r = bench.cpu_baseline_sample(w, X, CB, SCB, b, 2, seconds=0.2, zeropoint=zp)
        assert r["kind"] == "oracle" and r["cores"] == 2 and r["value"] > 0
        assert ("zeropoint" in r["sample"]) == zp
    f = synth.FFN_WORKLOADS["ffn_small"].with_(T=24)
    r = bench.ffn_cpu_baseline(f, synth.make_ffn(f), 2, seconds=0.2)
    assert r["kind"] == "oracle" and r["value"] > 0 and "of 24 tokens" in r["sample"]
