"""Multi-rank logic of bench.py on CPU with the gloo backend (world size 2):
each rank renders its own frames (replicas / views dealt round-robin) and only
the timing is reduced; no collective touches the data path."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, lr, w = bench.dist_env()
    frame_ms = 2.0 + 3.0 * rank                  # rank 1 is the slow one
    m = bench.max_over_ranks(frame_ms, w, "cpu")
    out[rank] = (r, lr, w, m, bench.job_value(m, w), bench.rank_view(0, r, 8), bench.rank_view(0, r, 1))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_and_views():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for rank in range(world):
        r, lr, w, m, value, view8, view1 = res[rank]
        assert (r, lr, w) == (rank, rank, world)
        assert m == 5.0                          # the slowest rank's frame time
        assert value == pytest.approx(world * 1e3 / 5.0)
        assert view8 == rank and view1 == 0      # views dealt out; one-view scenes are replicated


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_value(2.0, 1) == 500.0
    assert [bench.rank_view(2, r, 4) for r in range(4)] == [2, 3, 0, 1]


def test_traffic_figure_only_for_its_workload_and_code(tmp_path, monkeypatch):
    """roofline.traffic comes from a committed ncu summary only for the workload the
    counters were taken on and only while the code of the named files is unchanged;
    comments and whitespace do not count as code."""
    csrc = tmp_path / "gaussian_splatting_tile_02_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text("int f() { return 1; }  // one\n")
    (csrc / "h.cuh").write_text("/* helper */ int g();\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.code_hash(["k.cu", "h.cuh"])
    (tmp_path / "profiles" / "k.md").write_text(
        f"# k\n- workload: 1M\n- code_files: k.cu h.cuh\n- code_sha256_16: {h}\n- dram_bytes_per_launch: 1234\n")
    assert bench.traffic_from_profile("k.md", "1M") == 1234.0
    assert bench.traffic_from_profile("k.md", "5M") is None
    (csrc / "k.cu").write_text("int f() {\n    return 1;   // a reworded comment\n}\n")
    assert bench.traffic_from_profile("k.md", "1M") == 1234.0
    (csrc / "h.cuh").write_text("/* helper */ int g(int);\n")
    assert bench.traffic_from_profile("k.md", "1M") is None


def test_clock_summary_median_under_load_and_reasons(tmp_path):
    """The clocks record of the JSON line: median SM clock over the samples taken under load,
    the throttle reasons seen active, and the raw file kept only when asked for."""
    rows = [
        "0, 1200, 2032, 150.0, 0, Not Active, Not Active, Not Active, Not Active, Not Active",
        "0, 2032, 2032, 400.0, 97, Active, Not Active, Not Active, Not Active, Active",
        "0, 2010, 2032, 420.0, 99, Not Active, Not Active, Not Active, Not Active, Not Active",
        "0, 1990, 2032, 430.0, 98, Not Active, Not Active, Not Active, Not Active, Not Active",
    ]
    kept = tmp_path / "clocks.csv"
    kept.write_text("\n".join(rows) + "\n")
    s = bench.ClockSampler(0, str(kept)).summary()
    assert s["sm_mhz"] == 2010 and s["sm_max_mhz"] == 2032
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 4 and s["samples_under_load"] == 3
    assert s["power_w_max"] == 430.0 and kept.exists()
    temp = bench.ClockSampler(0)
    with open(temp.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    assert temp.summary()["sm_mhz"] == 2010
    assert not os.path.exists(temp.path)


def test_clock_sampler_closes_its_file_when_the_sampler_cannot_start(tmp_path, monkeypatch):
    """nvidia-smi missing: Popen raises inside __enter__; the record file is still closed on exit
    and the summary reports no samples."""
    def no_smi(*a, **k):
        raise FileNotFoundError("nvidia-smi")
    monkeypatch.setattr(bench.subprocess, "Popen", no_smi)
    sampler = bench.ClockSampler(0, str(tmp_path / "c.csv"))
    with sampler:
        assert sampler.proc is None and sampler.fh is not None
    assert sampler.fh is None
    assert sampler.summary()["samples"] == 0


def test_frame_launch_count():
    """gpu_launches per frame: 18 at 1920x1080 (8160 tiles, 13-bit tile ids, two passes) and at
    64x64 (16 tiles, one pass and a copy back); 19 at 8192x4320 (138240 tiles, three passes
    and a copy back, and the one-kernel tile order beyond 186 blocks of tiles)."""
    assert bench.frame_launches(120 * 68) == 18
    assert bench.frame_launches(4 * 4) == 18
    assert bench.frame_launches(512 * 270) == 19
    assert bench.frame_launches(240 * 135) == 18   # 3840x2160: 15 bits, two passes, 127 order blocks
    # tile-first frames sort each tile's list instead of all Gaussians by depth: one kernel per
    # list-size class the key capacity allows (up to 512, 2048, 8192 entries, and longer)
    assert bench.frame_launches(120 * 68, tile_first=True, key_capacity=400_000) == 17
    assert bench.frame_launches(120 * 68, tile_first=True, key_capacity=8192) == 16
    assert bench.frame_launches(4 * 4, tile_first=True, key_capacity=2000) == 15
    assert bench.frame_launches(4 * 4, tile_first=True, key_capacity=512) == 14
    assert [bench.tile_depth_launches(c) for c in (0, 1, 2, 512, 513, 2048, 2049, 8192, 8193)] == \
        [0, 0, 1, 1, 2, 2, 3, 3, 4]
    # from 4096 tiles up the tile keys hold the 8x4-tile block and 5 bits of tile within it
    assert bench.tile_key_bits(120, 68) == 13 and bench.tile_key_bits(40, 30) == 11
    assert bench.tile_key_bits(512, 270) == 18 and bench.tile_key_bits(240, 135) == 15
    # the ranges from the tile rectangles on a second stream (two kernels) up to 2^21
    # Gaussians where the grid's difference array fits in shared memory: 1080p yes, 8K no
    assert bench.side_ranges(10**6, 120, 68) and not bench.side_ranges(5 * 10**6, 120, 68)
    assert not bench.side_ranges(10**6, 240, 135)
    assert bench.frame_launches(120 * 68, tiles_xy=(120, 68), n=10**6) == 19
    assert bench.frame_launches(120 * 68, tiles_xy=(120, 68), n=5 * 10**6) == 18
    assert bench.frame_launches(512 * 270, tiles_xy=(512, 270), n=10**6) == 19
    assert bench.frame_launches(240 * 135, tiles_xy=(240, 135), n=10**6) == 18
