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
