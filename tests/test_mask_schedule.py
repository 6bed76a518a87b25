"""The block-sparse forward's static task schedule, through the C ABI (host logic, no GPU).

Every (query tile, batch-head) task must appear exactly once, each CTA runs two streams, each stream
runs its tasks by (batch-head, descending query tile), and longest-first assignment leaves the
streams' loads within one task's cost of each other.
"""
import ctypes

import numpy as np
import pytest

import attention_causal_attn_gb300 as attn
import seeded_inputs as si


@pytest.fixture(scope="module")
def lib():
    attn.build()
    return attn.load_library()


def _check_schedule(rp, bh, num_ctas):
    rp = np.asarray(rp, dtype=np.int64)
    nrows = len(rp) - 1
    n = nrows * bh
    tasks, offsets = attn.attn_mask_schedule(rp, bh, num_ctas)
    ctas = (len(offsets) - 1) // 2
    assert ctas == min(num_ctas, (n + 1) // 2)
    assert offsets[0] == 0 and offsets[-1] == n
    assert np.all(np.diff(offsets) >= 0)
    assert np.array_equal(np.sort(tasks), np.arange(n))  # every task exactly once
    cost = (rp[1:] - rp[:-1]) + 1.0  # listed tiles + the fixed cost, per row of tiles
    tcost = cost[tasks // bh]
    loads = np.array([tcost[offsets[j]:offsets[j + 1]].sum() for j in range(2 * ctas)])
    # longest-first into the least loaded stream: the last task a stream received went to the lightest
    # stream, so no stream ends more than one task's cost above the lightest (run order does not
    # change a stream's load)
    assert loads.max() - loads.min() <= tcost.max() + 1e-9
    for j in range(2 * ctas):
        seg = tasks[offsets[j]:offsets[j + 1]].astype(np.int64)
        key = (seg % bh) * (nrows + 1) + (nrows - seg // bh)  # (batch-head, descending query tile)
        assert np.all(np.diff(key) > 0), "a stream runs its tasks by batch-head, then descending query tile"
    return tasks, offsets, loads


def test_bigbird_mask_schedule_covers_every_task_once():
    rp, _ = si.bigbird_block_mask(4096, window=0, n_global=1, n_random=1, seed=4096, causal=False)
    _, _, loads = _check_schedule(rp, bh=4 * 32, num_ctas=152)
    assert loads.max() <= 1.05 * loads.mean() + 33  # the heaviest task (the global row) is 33


def test_causal_band_schedule_with_empty_rows():
    # rows 0..9: row r lists r + 1 tiles, except rows 3 and 7 list none
    counts = np.array([0 if r in (3, 7) else r + 1 for r in range(10)])
    rp = np.concatenate([[0], np.cumsum(counts)])
    _check_schedule(rp, bh=5, num_ctas=152)  # 50 tasks: 25 CTAs, two streams each
    _check_schedule(rp, bh=48, num_ctas=152)
    _check_schedule(rp, bh=1, num_ctas=3)


def test_tiny_schedules():
    _check_schedule([0, 1], bh=1, num_ctas=152)     # one task: one CTA, its second stream empty
    _check_schedule([0, 0], bh=3, num_ctas=152)     # nothing listed: the tasks still write O = 0
    _check_schedule([0, 2, 4], bh=1, num_ctas=1)    # one CTA, two streams


def test_schedule_argument_errors(lib):
    rp = np.array([0, 1, 2], dtype=np.int32)
    assert lib.attn_mask_schedule(None, 2, 1, 152, None, None, None) == -1          # ATTN_ERR_NULL
    assert lib.attn_mask_schedule(rp.ctypes.data, 2, 0, 152, None, None, None) == -2  # bh < 1
    assert lib.attn_mask_schedule(rp.ctypes.data, 2, 1, 0, None, None, None) == -2   # no CTA
    bad = np.array([0, 2, 1], dtype=np.int32)                                          # decreasing row pointers
    assert lib.attn_mask_schedule(bad.ctypes.data, 2, 1, 152, None, None, None) == -2
    assert lib.attn_mask_schedule(rp.ctypes.data, 2, 2 ** 31, 152, None, None, None) == -2  # too many tasks
    ctas = ctypes.c_int(0)
    assert lib.attn_mask_schedule(rp.ctypes.data, 2, 3, 152, None, None, ctypes.byref(ctas)) == 0
    assert ctas.value == 3
