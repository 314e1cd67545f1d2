"""The comparison rules themselves (CPU): the lazily evaluated per-row
scale gives the same verdict as the full one, and a planted difference
beyond the bar is caught and located."""
import numpy as np
import pytest

from oracle import tolerance as T


def _case(seed=0, s=64, k=3, rows=200, m=16):
    rng = np.random.default_rng(seed)
    row = rng.integers(-1, rows, size=(s, k)).astype(np.int32)
    gate = rng.random((s, k)).astype(np.float32)
    y = rng.standard_normal((rows, m)).astype(np.float32)
    return row, gate, y


def test_lazy_scale_matches_full_scale():
    row, gate, y = _case()
    ora = np.zeros((row.shape[0], y.shape[1]), np.float32)
    full = T.combine_scale(row, gate, y)
    ora[:] = full.astype(np.float32)  # any values; the check below moves a few by less than the bar
    gpu = ora.copy()
    gpu[5, 3] = np.nextafter(gpu[5, 3], np.float32(np.inf))  # 1 ulp, well inside 1e-6 of the scale
    T.assert_close(gpu, ora, full, "eager")
    T.assert_close(gpu, ora, lambda ts: T.combine_scale(row[ts], gate[ts], y), "lazy")
    # the lazy scale is only asked for the rows that differ
    asked = []
    T.assert_close(gpu, ora, lambda ts: asked.append(ts.copy()) or T.combine_scale(row[ts], gate[ts], y), "lazy")
    assert [a.tolist() for a in asked] == [[5]]


def test_lazy_scale_reports_a_planted_error_at_its_row():
    row, gate, y = _case(1)
    full = T.combine_scale(row, gate, y)
    ora = full.astype(np.float32)
    gpu = ora.copy()
    gpu[41, 7] += 1e-3 * (full[41, 7] + 1.0)
    with pytest.raises(AssertionError, match=r"first at \(41, 7\)"):
        T.assert_close(gpu, ora, lambda ts: T.combine_scale(row[ts], gate[ts], y), "lazy")
    with pytest.raises(AssertionError, match=r"first at \(41, 7\)"):
        T.assert_close(gpu, ora, full, "eager")


def test_bf16_rule_needs_no_scale():
    ora = np.array([[0x3F80, 0x4000]], np.uint16)  # 1.0, 2.0
    T.assert_close(np.array([[0x3F81, 0x4000]], np.uint16), ora, lambda ts: 1 / 0, "one ulp")
    with pytest.raises(AssertionError):
        T.assert_close(np.array([[0x3F83, 0x4000]], np.uint16), ora, lambda ts: 1 / 0, "three ulps")
