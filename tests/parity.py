"""Comparison of the CUDA path's results with the oracle's, under one rule for every test:

  * sampled indices are bit-exact, except on rows whose top-two oracle scores differ by less
    than NEAR_TIE; there the CUDA index is accepted if the oracle scores it within NEAR_TIE of
    the top, and the row is counted as a near-tie;
  * per-tile maximum scores agree within TILE_RTOL * (1 + |s|); per-tile indices are equal
    unless the oracle's own tile has a near-tie (checked the same way);
  * statuses are equal.

The kernels compute in fp32 (fp32 accumulation of bf16 products, fp32 noise) and the oracle in
fp64.  The difference per score is bounded by the fp32 GEMM error (~1e-6 relative to the
sum of |products|) plus the noise error (~1e-5 absolute at the far tail), so both tolerances
are orders of magnitude above what a correct kernel produces and far below what a wrong index,
term or sign would give.
"""
import numpy as np

NEAR_TIE = 1e-3
TILE_RTOL = 2e-4

# Per-test counts of what was compared and how many comparisons fell under the near-tie rule
# (and, through record(), other counts a test reports, such as tail misses).  conftest.py sets
# CURRENT to the running test's id, prints the counts at the end of the session and, when
# LMS_PARITY_RECORD names a file, writes them there as JSON.
RECORD = {}
CURRENT = ["(outside a test)"]


def _add(**counts):
    d = RECORD.setdefault(CURRENT[0], {})
    for k, v in counts.items():
        d[k] = d.get(k, 0) + int(v)


def record(**facts):
    """Attach facts (numbers, short lists) to the running test's record."""
    RECORD.setdefault(CURRENT[0], {}).update(facts)


def tile_tol(s):
    return TILE_RTOL * (1.0 + np.abs(s))


def check_rows(gpu_out, gpu_status, orc, score_of=None, rows=None):
    """Compare per-row results.  `score_of(i, v)` returns the oracle's score of index v in
    result row i (needed only when an index differs).  Returns the number of near-ties."""
    gpu_out = np.asarray(gpu_out)
    gpu_status = np.asarray(gpu_status)
    assert gpu_out.shape == orc.out.shape
    bad_status = np.nonzero(gpu_status != orc.status)[0]
    assert bad_status.size == 0, (
        f"status differs on rows {bad_status[:8]}: gpu {gpu_status[bad_status[:8]]} "
        f"oracle {orc.status[bad_status[:8]]}")
    near = 0
    for i in np.nonzero(gpu_out != orc.out)[0]:
        gap = orc.top1[i] - orc.top2[i]
        assert gap < NEAR_TIE, (
            f"row {i if rows is None else rows[i]}: gpu {gpu_out[i]} oracle {orc.out[i]}, "
            f"top-two gap {gap:.3e} is not a near-tie")
        assert score_of is not None, "index differs on a near-tie row; need the oracle's scores"
        s = score_of(i, int(gpu_out[i]))
        assert s >= orc.top1[i] - NEAR_TIE, (i, gpu_out[i], s, orc.top1[i])
        near += 1
    # rows whose top two oracle scores sit within the near-tie distance, whether or not the
    # indices happened to agree
    close = int(np.count_nonzero((orc.top1 - orc.top2 < NEAR_TIE) & (orc.status == 0)))
    _add(rows=gpu_out.shape[0], rows_index_differs_near_tie=near, rows_top2_within_near_tie=close)
    return near


def check_tiles(gpu_score, gpu_index, orc, score_of=None):
    """Compare Stage-1 candidates [rows, n_tiles]."""
    gpu_score = np.asarray(gpu_score, np.float64)
    gpu_index = np.asarray(gpu_index, np.int64)
    assert gpu_score.shape == orc.tile_max.shape
    both_empty = (gpu_index == -1) & (orc.tile_idx == -1)
    finite = ~both_empty
    assert (gpu_index[both_empty] == -1).all()
    assert ((gpu_index == -1) == (orc.tile_idx == -1)).all(), "a tile is empty on one side only"
    d = np.abs(gpu_score[finite] - orc.tile_max[finite])
    inf_same = np.isinf(orc.tile_max[finite]) & (gpu_score[finite] == orc.tile_max[finite])
    ok = inf_same | (d <= tile_tol(np.where(np.isinf(orc.tile_max[finite]), 0, orc.tile_max[finite])))
    if not ok.all():
        k = np.nonzero(~ok)[0][:5]
        raise AssertionError(f"tile scores differ: gpu {gpu_score[finite][k]} oracle {orc.tile_max[finite][k]}")
    near = 0
    for i, t in zip(*np.nonzero(gpu_index != orc.tile_idx)):
        assert score_of is not None, f"tile ({i},{t}) index differs: {gpu_index[i, t]} vs {orc.tile_idx[i, t]}"
        s = score_of(i, int(gpu_index[i, t]))
        assert s >= orc.tile_max[i, t] - NEAR_TIE, (i, t, gpu_index[i, t], s, orc.tile_max[i, t])
        near += 1
    _add(tiles=int(finite.sum()), tiles_index_differs_near_tie=near)
    return near
