"""The knob sweep's candidate list (CPU) and one small sweep on the GPU."""
import pytest

import tensor_core_gemm_multistage_gb300 as gsr
from tensor_core_gemm_multistage_gb300 import sweep


def test_candidates_respect_each_kernels_limits():
    big = sweep.candidates(8192, 8192, 8192)
    kernels = {c["kernel"] for c in big}
    assert kernels == {"tiled_128x256", "tiled_128x128", "tiled_128x64", "pair_256x256",
                       "pair_256x128"}   # no small-M above 256 rows
    assert "small_m" in {c["kernel"] for c in sweep.candidates(256, 4096, 4096)}
    assert {c["b_copy"] for c in big if c["kernel"] == "pair_256x256"} == {"3d", "2d"}
    assert {c["b_copy"] for c in big if c["kernel"] == "pair_256x128"} == {"3d", "2d"}
    assert {c["l2"] for c in big if c["kernel"] == "pair_256x256"} == set(sweep.L2_MODES)
    assert {c["l2"] for c in big if c["kernel"].startswith("tiled")} == {"default"}
    small = sweep.candidates(16, 1000, 4096)                                    # N % 64 != 0
    assert "small_m" in {c["kernel"] for c in small}
    assert {c["b_copy"] for c in small} == {"default"}
    assert all(c["raster"] == 0 for c in small if c["kernel"] == "small_m")
    # split-K only for the small-M kernel, never more slabs than 64-wide k-blocks (4096 / 64)
    assert {c["split"] for c in small if c["kernel"] == "small_m"} == set(sweep.SPLITS)
    assert {c["split"] for c in small if c["kernel"] != "small_m"} == {0}
    assert {c["split"] for c in sweep.candidates(16, 1024, 256) if c["kernel"] == "small_m"} == {0, 1, 2, 4}


@pytest.mark.gpu
def test_sweep_runs_every_candidate():
    gsr.build()
    results, best, auto = sweep.sweep(48, 1024, 512, iters=3, rounds=2)
    assert len(results) == len(sweep.candidates(48, 1024, 512))
    assert all(r["ms"] > 0 and len(r["ms_all"]) == 2 for r in results)
    assert best in results and auto in ("tiled", "small_m", "pair_256x256", "pair_256x128")


def test_choice_shapes_straddle_the_pair_threshold():
    # the boundary list must keep shapes on both sides of 76 pair tiles (half of 152 SMs)
    tiles = [((M + 255) // 256) * ((N + 255) // 256) for M, N, _ in sweep.CHOICE_SHAPES]
    assert min(tiles) < 76 <= max(tiles)
    assert any(70 <= t < 76 for t in tiles) and any(76 <= t <= 81 for t in tiles)


@pytest.mark.gpu
def test_check_choice_runs_on_two_shapes():
    gsr.build()
    rows = sweep.check_choice(shapes=[(1024, 1024, 512), (2048, 2560, 512)], rounds=1)
    assert [r["choice"] for r in rows] == ["tiled", "pair_256x256"]
    for r in rows:
        assert set(r["us"]) == set(sweep.CHOICE_KERNELS) and all(t > 0 for t in r["us"].values())
        assert r["fastest"] in sweep.CHOICE_KERNELS and r["choice_over_fastest"] > 0
