"""The forward's static tile schedule, through the C ABI (host logic, no GPU).

A unit is two 128-row query tiles that share one KV head; the estimated cost
of query tile bm is 2(bm + 1) + 4 ("Flash Attention: Causal Prefill D=128",
Step 4).  Checked: every query tile of every (batch, head) is covered exactly
once, the per-CTA cost is balanced, and with the K/V windows each CTA walks
the KV heads window by window.
"""
import numpy as np
import pytest

import attention_causal_attn_gb300 as attn

SHAPES = [
    # B, Hq, Hkv, S, D, causal
    (4, 32, 32, 8192, 128, True),     # the metric's workload
    (4, 32, 32, 4096, 128, True),
    (1, 32, 8, 16384, 128, True),     # GQA pairs
    (2, 3, 1, 257, 64, True),         # odd group: one paired and one single-head unit per tile
    (1, 4, 4, 640, 128, False),       # full attention: every tile costs the same
    (300, 1, 1, 129, 64, True),       # many more units than CTAs
    (1, 2, 2, 128, 64, True),         # fewer units than CTAs
]


def _decode(words, S, Hq, Hkv, causal):
    nqt = (S + 127) // 128
    G = Hq // Hkv
    tiles, costs, kv = [], [], []
    for x, y in words:
        qt = [int(x) & 0xFFFF, int(x) >> 16]
        h = [int(y) & 0xFF, (int(y) >> 8) & 0xFF]
        b = int(y) >> 16
        cost = 4.0
        for s in range(2):
            if qt[s] == 0xFFFF:
                continue
            if s == 1 and qt[1] == qt[0] and h[1] == h[0]:
                raise AssertionError("a unit names one tile twice")
            tiles.append((b, h[s], qt[s]))
            cost += 2.0 * ((qt[s] if causal else nqt - 1) + 1)
        assert h[0] // G == h[1] // G, "both stages of a unit share one KV head"
        costs.append(cost)
        kv.append(b * Hkv + h[0] // G)
    return tiles, np.array(costs), np.array(kv)


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal", SHAPES)
@pytest.mark.parametrize("window_mb", [0, 32])
def test_every_query_tile_once_and_balanced(B, Hq, Hkv, S, D, causal, window_mb):
    words, offsets = attn.attn_fwd_schedule(B, Hq, Hkv, S, D, causal, 152, window_mb * 2 ** 20)
    nqt = (S + 127) // 128
    ctas = len(offsets) - 1
    assert offsets[0] == 0 and np.all(np.diff(offsets) >= 1)  # every CTA has work
    tiles, costs, _ = _decode(words, S, Hq, Hkv, causal)
    expect = {(b, h, t) for b in range(B) for h in range(Hq) for t in range(nqt)}
    assert len(tiles) == len(expect) and set(tiles) == expect
    assert ctas == min(152, len(words))
    loads = np.array([costs[offsets[c]:offsets[c + 1]].sum() for c in range(ctas)])
    if len(words) >= 3 * ctas:
        # longest-first into the least loaded CTA: within one unit of the mean
        assert loads.max() - loads.mean() <= costs.max()
    if (B, Hq, Hkv, S) in [(4, 32, 32, 8192), (4, 32, 32, 4096), (1, 32, 8, 16384)]:
        assert loads.max() / loads.mean() < 1.012


def _window_of(B, Hkv, S, D, units, ctas, window):
    """The documented window rule: KV heads (b * Hkv + g) in windows of at most `window` bytes of
    K and V; the last window widened to at least three units per CTA; the heads before it split
    into windows whose sizes differ by at most one."""
    kv_heads = B * Hkv
    cap = max(1, min(kv_heads, int(window // (4 * S * D)))) if window > 0 else kv_heads
    per_kv = -(-units // kv_heads)
    tail = min(kv_heads, max(cap, -(-3 * ctas // per_kv)))
    front = kv_heads - tail
    nfront = -(-front // cap)
    return lambda kv: nfront if kv >= front else kv * nfront // front


@pytest.mark.parametrize("B,Hq,Hkv,S,D", [(4, 32, 32, 8192, 128), (4, 32, 32, 4096, 128), (8, 8, 2, 16384, 128),
                                          (2, 32, 8, 16384, 128)])
def test_ctas_walk_the_kv_heads_window_by_window(B, Hq, Hkv, S, D):
    window = 32 * 2 ** 20
    words, offsets = attn.attn_fwd_schedule(B, Hq, Hkv, S, D, True, 152, window)
    _, costs, kv = _decode(words, S, Hq, Hkv, True)
    ctas = len(offsets) - 1
    win = np.array([_window_of(B, Hkv, S, D, len(words), ctas, window)(int(x)) for x in kv])
    assert win.max() >= 1, "the workload spans several windows"
    sizes = np.bincount(win)
    for c in range(ctas):
        w = win[offsets[c]:offsets[c + 1]]
        assert np.all(np.diff(w) >= 0), f"CTA {c} returns to an earlier window"
        for x in np.unique(w):  # heaviest first inside each window
            assert np.all(np.diff(costs[offsets[c]:offsets[c + 1]][w == x]) <= 0)
    # every window but the last holds at most `window` bytes of K and V
    heads = np.bincount(win[np.unique(kv, return_index=True)[1]])
    assert np.all(heads[:-1] * 4 * S * D <= window)
    assert sizes.sum() == len(words)
    # loads stay balanced at every window boundary: within one unit's cost
    ends = np.zeros((ctas, win.max() + 1))
    for c in range(ctas):
        seg_w = win[offsets[c]:offsets[c + 1]]
        seg_c = costs[offsets[c]:offsets[c + 1]]
        for x in range(win.max() + 1):
            ends[c, x] = seg_c[seg_w <= x].sum()
    assert np.all(ends.max(axis=0) - ends.min(axis=0) <= 2 * costs.max())


def test_one_window_is_plain_longest_first():
    words, offsets = attn.attn_fwd_schedule(4, 32, 32, 8192, 128, True, 152, 0.0)
    _, costs, _ = _decode(words, 8192, 32, 32, True)
    for c in range(len(offsets) - 1):
        seg = costs[offsets[c]:offsets[c + 1]]
        assert np.all(np.diff(seg) <= 0), "each CTA runs its units heaviest first"


def test_schedule_argument_errors():
    lib = attn.load_library()
    assert lib.attn_fwd_schedule(0, 2, 2, 128, 64, 1, 152, 0.0, None, None, None) == -2
    assert lib.attn_fwd_schedule(1, 3, 2, 128, 64, 1, 152, 0.0, None, None, None) == -2   # Hq % Hkv
    assert lib.attn_fwd_schedule(1, 2, 2, 128, 96, 1, 152, 0.0, None, None, None) == -2   # D
    assert lib.attn_fwd_schedule(1, 2, 2, 128, 64, 1, 0, 0.0, None, None, None) == -2     # no CTA
    assert lib.attn_fwd_schedule(1, 2, 2, 128, 64, 2, 152, 0.0, None, None, None) == -4   # causal flag
