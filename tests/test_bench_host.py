"""Host-side pieces of bench.py on CPU: the work counting behind the FLOP figure and the parsing of the
clock samples that decides whether a run was throttled."""
import numpy as np

import bench
import oracle as orc
from dynamic_block_sparse_rank_gb300 import inputs


def test_block_sizes_cover_every_token_of_the_ragged_grid():
    wl = inputs.WORKLOADS["merge_131k"]  # 21 x 60 x 104 in 2 x 8 x 8 tiles: clipped tiles on t and h
    sz = bench.block_sizes(wl)
    assert sz.sum() == wl.N and len(sz) == wl.n_blocks == 1144
    counts = {int(v): int(c) for v, c in zip(*np.unique(sz, return_counts=True))}
    assert counts == {32: 13, 64: 221, 128: 910}
    geom = orc.Geometry(wl.T, wl.H, wl.W, wl.bt, wl.bh, wl.bw)
    assert all(sz[I] == len(geom.tokens(I)) for I in range(0, wl.n_blocks, 37))


def test_kept_pairs_counts_the_attended_token_pairs():
    wl = inputs.Workload("ragged", 2, 3, 5, 12, 20, 64, 2, 8, 8, 16, 0.4, "bf16", 3.0, 16)
    geom = orc.Geometry(wl.T, wl.H, wl.W, wl.bt, wl.bh, wl.bw)
    rng = np.random.default_rng(0)
    idx = np.stack([np.stack([np.stack([np.sort(rng.choice(geom.n_blocks, wl.k, replace=False))
                                        for _ in range(geom.n_blocks)]) for _ in range(wl.heads)])
                    for _ in range(wl.B)]).astype(np.int32)
    brute = 0
    for b in range(wl.B):
        for h in range(wl.heads):
            for I in range(geom.n_blocks):
                brute += len(geom.tokens(I)) * sum(len(geom.tokens(int(J))) for J in idx[b, h, I])
    assert bench.kept_pairs(wl, idx) == brute


def _summary(tmp_path, lines):
    cs = bench.ClockSampler(0)
    cs.tmp = open(tmp_path / "clocks.csv", "w+")
    cs.tmp.write("\n".join(lines) + "\n")
    cs.proc = object()  # a sampler that ran
    return cs.summary()  # reads and removes the file


def test_clock_summary_takes_the_loaded_median_and_reports_throttle_reasons(tmp_path):
    idle = "0, 345, 2070, 120.5, 0x0, Not Active, Not Active, Not Active, Not Active"
    busy = ["0, {}, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, {}".format(mhz, cap)
            for mhz, cap in ((2010, "Active"), (1995, "Active"), (2040, "Not Active"))]
    s = _summary(tmp_path, [idle] + busy)
    assert s["sm_mhz"] == 2010 and s["sm_max_mhz"] == 2070 and s["samples"] == 4
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1350.0
    hot = "0, 1500, 2070, 1390.0, 0x40, Not Active, Active, Not Active, Not Active"
    assert "hw_thermal_slowdown" in _summary(tmp_path, [hot, hot])["reasons"]


def test_clock_summary_without_samples_says_so(tmp_path):
    assert _summary(tmp_path, [])["reasons"] == ["no samples"]
    cs = bench.ClockSampler(0)
    assert cs.summary()["reasons"] == ["nvidia-smi unavailable"]
