"""The benchmark's host-side arithmetic, on the CPU: the tile-covering
sample the CPU oracle table runs on, the even sub-sampling, the binning of
clock-study chunks and the roofline classification."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("M,N", [(8192, 8192), (32768, 256), (1000, 1000), (16, 8), (129, 257), (1, 1)])
def test_tile_covering_sample_covers_every_tile_once_per_element(M, N):
    rows, cols = bench.tile_covering_entries(M, N)
    assert rows.dtype == np.int64 and cols.dtype == np.int64 and len(rows) == len(cols)
    assert rows.min() >= 0 and rows.max() < M and cols.min() >= 0 and cols.max() < N
    flat = rows * N + cols
    assert len(np.unique(flat)) == len(flat), "an output element is listed twice"
    # every 128 x 256 output tile holds at least one sampled element
    tiles = set(zip((rows // 128).tolist(), (cols // 256).tolist()))
    assert tiles == {(i, j) for i in range((M + 127) // 128) for j in range((N + 255) // 256)}
    # one full row per row block and one full column per column block
    n_rb, n_cb = (M + 127) // 128, (N + 255) // 256
    full_rows = [r for r in np.unique(rows) if np.count_nonzero(rows == r) >= N]
    full_cols = [c for c in np.unique(cols) if np.count_nonzero(cols == c) >= M]
    assert len(full_rows) == n_rb and len(full_cols) == n_cb
    assert len(rows) == n_rb * N + n_cb * (M - n_rb)


def test_tile_covering_sample_size_at_the_headline():
    rows, _ = bench.tile_covering_entries(8192, 8192)
    assert len(rows) == 64 * 8192 + 32 * (8192 - 64)


@pytest.mark.parametrize("total,keep", [(10, 3), (10, 10), (10, 50), (786432, 1000), (5, 1)])
def test_every_nth_is_even_and_bounded(total, keep):
    idx = bench.every_nth(total, keep)
    assert len(idx) == min(total, keep)
    assert idx.min() >= 0 and idx.max() <= total - 1
    assert np.all(np.diff(idx) > 0)
    if keep >= 2 and keep < total:
        gaps = np.diff(idx)
        assert gaps.max() - gaps.min() <= 1


def test_clock_bins_group_and_average():
    chunks = [{"mhz": 1410.0, "launches": 16, "ms": 16 * 0.7}, {"mhz": 1440.0, "launches": 16, "ms": 16 * 0.68},
              {"mhz": 2060.0, "launches": 16, "ms": 16 * 0.62}]
    bins = bench.clock_bins(chunks, width_mhz=50.0)
    assert [(b["mhz_lo"], b["chunks"], b["launches"]) for b in bins] == [(1400.0, 2, 32), (2050.0, 1, 16)]
    assert bins[0]["ms_per_launch"] == pytest.approx(0.69)
    assert bins[0]["mhz_mean"] == pytest.approx(1425.0)
    assert bins[1]["ms_per_launch"] == pytest.approx(0.62)


def test_roofline_classification():
    # 8192^3 f16: tensor-bound, 2048 flop per byte
    r = bench.roofline_of(2 * 8192 ** 3, 536870912, 0.62e-3, 1882.7, 6772.2)
    assert r["bound"] == "tensor" and r["frac"] == pytest.approx(2 * 8192 ** 3 / 1882.7e12 / 0.62e-3)
    # 8192^2 x 256: HBM-bound
    r = bench.roofline_of(2 * 8192 * 8192 * 256, 2 * (8192 * 256 * 2) + 4 * 8192 * 8192, 55e-6, 1882.7, 6772.2)
    assert r["bound"] == "hbm" and "limited_by" not in r
    # the single atom: latency
    r = bench.roofline_of(2 * 16 * 8 * 16, 2 * (16 * 16 + 16 * 8) + 4 * 16 * 8, 8e-6, 1882.7, 6772.2)
    assert r["limited_by"] == "latency"


def test_clock_series_from_probe_samples():
    """Consecutive (globaltimer ns, clock64, smid) samples give the clock in
    MHz between them; pairs across a change of SM (the counters are per SM)
    or with a non-advancing timer are skipped."""
    samples = [(1000, 5000, 7), (21000, 5000 + 40000, 7), (41000, 45000 + 33800, 7),
               (61000, 10, 9), (81000, 10 + 20700 * 2, 9), (81000, 99999, 9)]
    series = bench.clock_series(samples)
    assert [round(m) for _, m in series] == [2000, 1690, 2070]
    assert [t for t, _ in series] == [11000.0, 31000.0, 71000.0]
    assert bench.clock_between(series, 10000, 40000) == [series[0][1], series[1][1]]
    assert bench.clock_between(series, 72000, 90000) == []
