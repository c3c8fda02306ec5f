"""The benchmark's multi-rank host logic on CPU: two gloo ranks (127.0.0.1)
agree on the slowest rank's time and report the whole-job weak-scaling rate.
No GPU: the data path has no collective; only this timing reduction does."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, _ = bench.dist_env()
    my_ms = 10.0 + 5.0 * rank           # rank 1 is the slow one
    mx = bench.reduce_max(my_ms, ws)
    rate = bench.weak_scaling_rate(1e9, ws, 4, mx)
    dist.barrier()
    q.put((r, ws, mx, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_and_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, mx, rate in res:
        assert ws == 2 and mx == 15.0
        assert rate == pytest.approx(2 * 4 * 1e9 / 15e-3 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.weak_scaling_rate(2e9, 1, 10, 1000.0) == pytest.approx(20.0)


def test_peaks_file_forms(tmp_path, monkeypatch):
    """bench.peaks(): measured figures at the top level or one level down; a
    malformed or partial file falls back to the recipe's figures."""
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = tmp_path / "MEASURED_PEAKS.json"
    assert bench.peaks()["source"] == "fallback"
    f.write_text('{"hbm_gbs": 7000, "bf16_tflops": 2000, "bf16_tflops_sustained": 1750}')
    p = bench.peaks()
    assert p["source"] == "measured" and p["hbm_gbs"] == 7000 and p["bf16_tflops_sustained"] == 1750
    f.write_text('{"gb300": {"hbm_gbs": 7100, "bf16_tflops": 1950}}')
    p = bench.peaks()
    assert p["source"] == "measured" and p["bf16_tflops_sustained"] == 1950
    for bad in ("not json", "[1, 2]", '{"hbm_gbs": 7000}', '{"hbm_gbs": true, "bf16_tflops": 1}'):
        f.write_text(bad)
        assert bench.peaks()["source"] == "fallback", bad


def test_gemm_traffic_record_matches_source():
    """The roofline's DRAM traffic comes from a committed ncu record keyed by
    the GEMM source's hash; it must still match the source in the tree."""
    import bench
    t = bench.traffic_for("k_gemm_e1m2_moe124b")
    assert isinstance(t, int) and t > 0
