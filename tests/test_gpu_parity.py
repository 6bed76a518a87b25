"""GPU parity: the sm_103a kernel through the C ABI against the float64 oracle.

Tolerances (the attention prefill gate): O max-abs <= 2e-2 and mean-abs <=
2e-3; LSE |error| <= 1e-3 * max(1, |LSE|).  Small cases compare every row;
the benchmark-sized workloads compare 256 seeded query rows of 8 seeded heads.
"""
import numpy as np
import pytest
import torch

import attention_causal_attn_gb300 as attn
import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_REL = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    attn.build()
    oracle.build()
    yield
    torch.cuda.synchronize()


def _dev(a):
    return torch.from_numpy(a).view(torch.bfloat16).cuda()


def _check(o, lse, o_ref, lse_ref, tag=""):
    o = np.asarray(o, dtype=np.float64)
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all(), f"{tag}: non-finite output"
    assert err.max() <= O_MAX, f"{tag}: max|dO| {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{tag}: mean|dO| {err.mean():.3e}"
    if lse is not None:
        # the gate: |dLSE| <= 1e-3 * max(1, |LSE|) (a row's LSE can be near 0, e.g. row 0's is one
        # score); the plain relative error is reported beside it
        d = np.abs(np.asarray(lse, np.float64) - lse_ref)
        lerr = d / np.maximum(1.0, np.abs(lse_ref))
        rel = d / np.maximum(1e-6, np.abs(lse_ref))
        assert lerr.max() <= LSE_REL, f"{tag}: max dLSE/max(1,|LSE|) {lerr.max():.3e} (plain relative {rel.max():.3e})"
    return err.max()


SMALL = [
    # B, Hq, Hkv, S, D, causal, rope_base
    (1, 2, 2, 128, 64, True, 10000.0),    # the tiny benchmark configuration
    (2, 4, 4, 384, 128, True, None),      # odd number of query tiles (last unit has one stage)
    (1, 4, 2, 300, 128, True, 10000.0),   # GQA pairs, ragged tail
    (2, 3, 1, 257, 64, True, 500000.0),   # group of 3: one paired unit and one single-head unit
    (1, 2, 2, 1, 128, True, 10000.0),     # S = 1
    (1, 2, 2, 2, 64, True, None),         # S = 2
    (1, 2, 1, 200, 128, False, None),     # full attention, ragged
    (2, 2, 2, 129, 64, False, 10000.0),   # full attention with RoPE, one key past a tile
    (1, 8, 8, 1024, 128, True, 10000.0),  # eight query tiles per head
    (1, 4, 4, 640, 128, False, 500000.0),
]


EDGE = [
    # B, Hq, Hkv, S, D, causal, rope_base
    (1, 255, 5, 130, 64, True, 10000.0),   # query heads at the API limit, GQA groups of 51
    (1, 16, 1, 257, 128, True, 500000.0),  # every query head on one KV head
    (300, 1, 1, 129, 64, True, None),      # many more work units than CTAs
    (65535, 1, 1, 1, 64, True, 10000.0),   # batch at the API limit, one key per row
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base", EDGE)
def test_limits_all_rows(B, Hq, Hkv, S, D, causal, base):
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=303 + S)
    o, lse = attn.attn_fwd(_dev(q), _dev(k), _dev(v), causal=causal, rope_base=base)
    attn.attn_check()
    o_ref, lse_ref = oracle.attn_full(q, k, v, causal=causal, rope_base=base)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"B={B} Hq={Hq} S={S}")


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base", SMALL)
def test_small_all_rows(B, Hq, Hkv, S, D, causal, base):
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=101 + S)
    o, lse = attn.attn_fwd(_dev(q), _dev(k), _dev(v), causal=causal, rope_base=base)
    attn.attn_check()
    o_ref, lse_ref = oracle.attn_full(q, k, v, causal=causal, rope_base=base)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"S={S} D={D}")


def test_no_lse_and_side_stream_and_determinism():
    B, Hq, Hkv, S, D = 1, 4, 2, 513, 128
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=5)
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = attn.attn_fwd(qd, kd, vd, causal=True, rope_base=10000.0, stream=s)
        o2, none = attn.attn_fwd(qd, kd, vd, causal=True, rope_base=10000.0, return_lse=False, stream=s)
    attn.attn_check(stream=s)
    assert none is None
    assert torch.equal(o1, o2)  # same schedule, same arithmetic: bitwise reproducible
    o_ref, lse_ref = oracle.attn_full(q, k, v, causal=True, rope_base=10000.0)
    _check(o1.float().cpu().numpy(), l1.cpu().numpy(), o_ref, lse_ref)


_INPUT_CACHE = {}


def _sampled(B, Hq, Hkv, S, D, causal, base, outliers=0.0, nrows=256, nheads=8, seed=si.MASTER_SEED, window_k=None):
    key = (B, Hq, Hkv, S, D, outliers, seed)
    if key not in _INPUT_CACHE:  # the long-context workload is generated once for its three window settings
        _INPUT_CACHE.clear()
        _INPUT_CACHE[key] = si.make_qkv(B, Hq, Hkv, S, D, outliers=outliers, seed=seed)
    q, k, v = _INPUT_CACHE[key]
    o, lse = attn.attn_fwd(_dev(q), _dev(k), _dev(v), causal=causal, rope_base=base, window_k=window_k)
    attn.attn_check()
    rows = si.sample_rows(seed, S, nrows)
    heads = si.sample_heads(seed, B, Hq, Hkv, nheads)
    rb = np.repeat([b for b, _ in heads], len(rows))
    rh = np.repeat([h for _, h in heads], len(rows))
    ri = np.tile(rows, len(heads))
    o_ref, lse_ref = oracle.attn_rows(q, k, v, rb, rh, ri, causal=causal, rope_base=base, window_k=window_k)
    idx_b = torch.from_numpy(rb).long().cuda()
    idx_h = torch.from_numpy(rh).long().cuda()
    idx_i = torch.from_numpy(ri).long().cuda()
    o_s = o[idx_b, idx_i, idx_h].float().cpu().numpy()
    l_s = lse[idx_b, idx_h, idx_i].cpu().numpy()
    del o, lse
    torch.cuda.empty_cache()
    return _check(o_s, l_s, o_ref, lse_ref, f"S={S}")


def test_plain_causal_s4096_sampled():
    _sampled(4, 32, 32, 4096, 128, True, None)


def test_rope_causal_s8192_sampled():
    _sampled(4, 32, 32, 8192, 128, True, 10000.0)


def test_gqa_outliers_s16384_sampled():
    _sampled(1, 32, 8, 16384, 128, True, 500000.0, outliers=0.01)


@pytest.mark.parametrize("base", [None, 10000.0])
def test_late_large_score_rescales_running_max(base):
    """A key visited last (key 100: chunk 3 of tile 0, reverse traversal) whose
    score exceeds every earlier one by ~24 in log2 units (the rescale threshold
    is 16).  The running max must move mid-tile: O, the P chunks already written
    and the partial sums are rescaled (the softmax's rare path)."""
    B, H, S, D = 1, 2, 640, 128
    q = si.bf16_bits_to_f64(si.bshd_bf16(31, 1, B, S, H, D)) * 0.3 + 1.0
    k = si.bf16_bits_to_f64(si.bshd_bf16(31, 2, B, S, H, D)) * 0.3
    k[:, 100] = 1.5
    v = si.bf16_bits_to_f64(si.bshd_bf16(31, 3, B, S, H, D))
    q, k, v = (si.f64_to_bf16_bits(x.reshape(-1)).reshape(x.shape) for x in (q, k, v))
    o, lse = attn.attn_fwd(_dev(q), _dev(k), _dev(v), causal=True, rope_base=base)
    attn.attn_check()
    o_ref, lse_ref = oracle.attn_full(q, k, v, causal=True, rope_base=base)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "late large score")


@pytest.mark.parametrize("base", [None, 10000.0])
def test_running_max_moves_inside_tiles(base):
    """Planted keys that move a row's running max inside a tile, where the
    softmax decides per 32-key chunk:
    - key 40 (chunk 1 of the diagonal tile 0): rows 40..127 move on their
      first tile, while rows 0..39 must not see it (masked chunk);
    - keys 168 and 228 (chunks 1 and 3 of tile 1), each above the running max
      by more than the threshold: two moves in one tile for rows 256..299;
    - key 300 (chunk 1 of the diagonal tile 2) for rows 300..383.
    (Scores in log2 units without RoPE: about 23, 21, 42 and 29 for the planted
    keys against about 1 for the others; the rescale threshold is 16.)  Large scores on causally
    hidden keys must never reach earlier rows."""
    B, H, S, D = 1, 2, 512, 128
    q = si.bf16_bits_to_f64(si.bshd_bf16(37, 1, B, S, H, D)) * 0.3 + 1.0
    k = si.bf16_bits_to_f64(si.bshd_bf16(37, 2, B, S, H, D)) * 0.3
    k[:, 40] = 1.4
    k[:, 168] = 1.3
    k[:, 228] = 2.6
    k[:, 300] = 1.8
    v = si.bf16_bits_to_f64(si.bshd_bf16(37, 3, B, S, H, D))
    q, k, v = (si.f64_to_bf16_bits(x.reshape(-1)).reshape(x.shape) for x in (q, k, v))
    o, lse = attn.attn_fwd(_dev(q), _dev(k), _dev(v), causal=True, rope_base=base)
    attn.attn_check()
    o_ref, lse_ref = oracle.attn_full(q, k, v, causal=True, rope_base=base)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "running max moves inside tiles")


WINDOW_SMALL = [
    # B, Hq, Hkv, S, D, rope_base, k
    (1, 2, 2, 640, 128, 10000.0, 0.05),   # heavy pruning: whole channel groups skipped, many boundary pairs
    (1, 4, 2, 700, 128, 100.0, 0.3),      # GQA pairs, small base: every tile has boundary pairs
    (1, 2, 1, 300, 64, 500.0, 1.0),       # D = 64, ragged
    (2, 4, 4, 1024, 128, 10000.0, 1.0),   # MHA pairs of query tiles (the two stages drop different pairs)
    (1, 2, 2, 400, 128, 10000.0, 1e-9),   # W_r = 0: only the diagonal keeps its terms (all groups dropped)
    (1, 2, 2, 256, 128, 500000.0, 4.0),   # window barely bites
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,base,k", WINDOW_SMALL)
def test_window_small_all_rows(B, Hq, Hkv, S, D, base, k):
    q, k_, v = si.make_qkv(B, Hq, Hkv, S, D, seed=202 + S)
    o, lse = attn.attn_fwd(_dev(q), _dev(k_), _dev(v), causal=True, rope_base=base, window_k=k)
    attn.attn_check()
    o_ref, lse_ref = oracle.attn_full(q, k_, v, causal=True, rope_base=base, window_k=k)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"window k={k} S={S} D={D}")
    # the window must change the result where it prunes (not silently ignored)
    o_off, _ = oracle.attn_full(q, k_, v, causal=True, rope_base=base)
    if k < 1.0:
        assert np.abs(o_off - o_ref).max() > 5e-2


def _sampled_window(k):
    return _sampled(1, 32, 8, 131072, 128, True, 500000.0, window_k=k)


@pytest.mark.parametrize("k", [1.0, 4.0, None])
def test_window_s131072_sampled(k):
    _sampled_window(k)


HOST = [
    # B, Hq, Hkv, S, D, causal, rope_base, window_k
    (4, 4, 4, 300, 128, True, 10000.0, None),    # one chunk per batch element
    (2, 8, 4, 257, 64, True, None, None),        # two KV-head groups per batch element
    (1, 8, 8, 1030, 128, True, 500000.0, None),  # four head groups, ragged
    (1, 4, 2, 700, 128, True, 10000.0, 1.0),     # window
    (3, 2, 1, 129, 64, False, None, None),       # full attention, one KV head
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base,wk", HOST)
def test_host_entry_matches_device_entry_bitwise(B, Hq, Hkv, S, D, causal, base, wk):
    """attn_fwd_host cuts the work into (batch, KV-head group) chunks; each head's
    arithmetic is unchanged, so O and LSE equal attn_fwd's bit for bit."""
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=404 + S)
    qp, kp, vp = (torch.from_numpy(x).view(torch.bfloat16).pin_memory() for x in (q, k, v))
    o_h, l_h = attn.attn_fwd_host(qp, kp, vp, causal=causal, rope_base=base, window_k=wk)
    o_d, l_d = attn.attn_fwd(qp.cuda(), kp.cuda(), vp.cuda(), causal=causal, rope_base=base, window_k=wk)
    attn.attn_check()
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(l_h, l_d.cpu())
    if S <= 300:
        o_ref, lse_ref = oracle.attn_full(q, k, v, causal=causal, rope_base=base, window_k=wk)
        _check(o_h.float().numpy(), l_h.numpy(), o_ref, lse_ref, "host entry")


def test_host_entry_pageable_memory_and_no_lse():
    B, Hq, Hkv, S, D = 2, 4, 2, 333, 128
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=505)
    qt, kt, vt = (torch.from_numpy(x).view(torch.bfloat16) for x in (q, k, v))  # not pinned
    o_h, none = attn.attn_fwd_host(qt, kt, vt, causal=True, rope_base=10000.0, return_lse=False)
    assert none is None
    o_d, _ = attn.attn_fwd(qt.cuda(), kt.cuda(), vt.cuda(), causal=True, rope_base=10000.0)
    attn.attn_check()
    assert torch.equal(o_h, o_d.cpu())


@pytest.mark.parametrize("B,S,H,D,base", [(2, 1000, 3, 128, 10000.0), (1, 257, 4, 64, 500000.0),
                                          (1, 131072, 1, 128, 500000.0)])
def test_pre_rotation_matches_oracle_rotation(B, S, H, D, base):
    """attn_rope_rotate (fp16 out) against the float64 rotation, within fp16 rounding
    plus a few fp32 ulps of angle error; long rows check the angles at large positions."""
    x = si.bshd_bf16(606, 1, B, S, H, D)
    y = attn.attn_rope_rotate(_dev(x), base)
    torch.cuda.synchronize()
    ref = oracle.rope_rotate(x, base)
    got = y.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert np.all(err <= 1e-3 * np.abs(ref) + 2e-4), f"max err {err.max():.3e}"


PRE = [
    # B, Hq, Hkv, S, D, causal, rope_base
    (2, 4, 4, 384, 128, True, 10000.0),
    (1, 4, 2, 300, 128, True, 500000.0),
    (2, 3, 1, 257, 64, False, 10000.0),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base", PRE)
def test_pre_rotated_forward_matches_oracle_and_fused(B, Hq, Hkv, S, D, causal, base):
    """attn_rope_rotate on Q and K, then attn_fwd_rotated: the same attention as
    the fused path ("AttnFuse", sec. 5.3: pre-rotation against fusion)."""
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=707 + S)
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    o, lse = attn.attn_fwd_rotated(attn.attn_rope_rotate(qd, base), attn.attn_rope_rotate(kd, base), vd,
                                   causal=causal)
    o_f, lse_f = attn.attn_fwd(qd, kd, vd, causal=causal, rope_base=base)
    attn.attn_check()
    o_ref, lse_ref = oracle.attn_full(q, k, v, causal=causal, rope_base=base)
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "pre-rotated")
    # both paths round the rotated operands to fp16; only the angles' last fp32 bits differ
    assert (o.float() - o_f.float()).abs().max().item() <= 1e-2


DECODE = [
    # B, Hq, Hkv, S, D, rope_base, window_k
    (2, 8, 2, 1000, 128, 10000.0, None),     # GQA groups of 4, several splits
    (3, 4, 4, 257, 64, None, None),          # MHA, RoPE off, ragged split tail
    (1, 32, 1, 700, 128, 10000.0, None),     # all 32 query heads on one KV head
    (1, 16, 2, 1, 128, 10000.0, None),       # a cache of one key
    (1, 32, 8, 5000, 128, 500000.0, 1.0),    # windowed decode
    (1, 8, 8, 3000, 128, 100.0, 0.3),        # small base: the window drops most pairs of far keys
    (2, 6, 2, 2500, 64, 10000.0, None),      # groups of 3, D = 64
    (1, 40, 2, 1500, 128, 10000.0, 2.0),     # groups of 20: two 16-head tiles, the second partly empty
    (2, 8, 4, 1800, 64, 500.0, 0.5),         # windowed, D = 64
]


def _decode_check(B, Hq, Hkv, S, D, base, wk, seed):
    q_full, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=seed)
    q_dec = np.ascontiguousarray(q_full[:, S - 1])  # the newest token of each sequence
    o, lse = attn.attn_decode(_dev(q_dec), _dev(k), _dev(v), rope_base=base, window_k=wk)
    attn.attn_check()
    rb = np.repeat(np.arange(B), Hq)
    rh = np.tile(np.arange(Hq), B)
    ri = np.full(B * Hq, S - 1)
    o_ref, lse_ref = oracle.attn_rows(q_full, k, v, rb, rh, ri, causal=True, rope_base=base, window_k=wk)
    _check(o.float().cpu().numpy().reshape(B * Hq, D), lse.cpu().numpy().reshape(-1), o_ref, lse_ref,
           f"decode S={S}")


@pytest.mark.parametrize("B,Hq,Hkv,S,D,base,wk", DECODE)
def test_decode_matches_oracle_last_row(B, Hq, Hkv, S, D, base, wk):
    """attn_decode: the query at position S-1 against the whole cache, i.e. the
    last row of the causal prefill, split across CTAs and merged by LSE."""
    _decode_check(B, Hq, Hkv, S, D, base, wk, seed=808 + S)


@pytest.mark.parametrize("wk", [4.0, None])
def test_decode_long_cache_s131072(wk):
    _decode_check(1, 32, 8, 131072, 128, 500000.0, wk, seed=909)


# ---------------------------------------------------------------- backward
# Gradients are compared per tensor, relative to the reference's scale: the
# bf16 outputs alone carry up to 2^-9 = 1.95e-3 of it, and P enters dV in bf16
# and dS enters dQ/dK in fp16 (bf16 without RoPE).  Measured on GB300: at most
# 4.1e-3 (max) and 2.4e-3 (mean) over the cases below; the gate keeps about a
# factor 2.5.  A reference that is exactly zero (a cache of one key gives
# dS = 0) is held to 1e-3 of an absolute unit scale.
BWD_MAX, BWD_MEAN = 1e-2, 5e-3

BWD = [
    # B, Hq, Hkv, S, D, causal, rope_base
    (1, 2, 2, 128, 64, True, 10000.0),
    (2, 4, 2, 300, 128, True, 10000.0),    # GQA, ragged tail
    (1, 2, 2, 256, 128, True, None),       # RoPE off: bf16 operands throughout
    (1, 2, 1, 200, 64, False, 500000.0),   # full attention, group of 2
    (2, 3, 1, 129, 128, True, 10000.0),    # group of 3, one key past a tile
    (1, 2, 2, 1, 128, True, 10000.0),      # S = 1
    (1, 4, 4, 1024, 128, True, 10000.0),   # eight tiles per head
]


def _check_grad(got, ref, tag):
    got = np.asarray(got, dtype=np.float64)
    assert np.isfinite(got).all(), f"{tag}: non-finite gradient"
    err = np.abs(got - ref)
    scale_max, scale_mean = max(np.abs(ref).max(), 1e-3), max(np.abs(ref).mean(), 1e-3)
    assert err.max() <= BWD_MAX * scale_max, f"{tag}: max err {err.max():.3e} vs scale {scale_max:.3e}"
    assert err.mean() <= BWD_MEAN * scale_mean, f"{tag}: mean err {err.mean():.3e} vs scale {scale_mean:.3e}"


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base", BWD)
def test_backward_matches_oracle(B, Hq, Hkv, S, D, causal, base):
    """attn_bwd on the GPU forward's own O and LSE against the float64 chain rule."""
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=600 + S)
    dO = si.bshd_bf16(601 + S, 9, B, S, Hq, D)
    qd, kd, vd, dOd = _dev(q), _dev(k), _dev(v), _dev(dO)
    o, lse = attn.attn_fwd(qd, kd, vd, causal=causal, rope_base=base)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dOd, causal=causal, rope_base=base)
    attn.attn_check()
    rq, rk, rv = oracle.attn_bwd(q, k, v, dO, causal=causal, rope_base=base)
    tag = f"B{B} Hq{Hq} Hkv{Hkv} S{S} D{D} causal{causal} base{base}"
    _check_grad(dv.float().cpu().numpy(), rv, tag + " dV")
    _check_grad(dk.float().cpu().numpy(), rk, tag + " dK")
    _check_grad(dq.float().cpu().numpy(), rq, tag + " dQ")


def test_backward_rope_causal_s8192_two_heads():
    """The timed backward's own shape (B=4, H=32, S=8192, D=128, RoPE, causal): every gradient row of
    two heads of the last batch against the chain rule on those heads alone (heads are independent
    when Hq = Hkv, and the rotation does not depend on the head)."""
    B, Hq, Hkv, S, D, base = 4, 32, 32, 8192, 128, 10000.0
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=2024)
    dO = si.bshd_bf16(2025, 9, B, S, Hq, D)
    qd, kd, vd, dOd = _dev(q), _dev(k), _dev(v), _dev(dO)
    o, lse = attn.attn_fwd(qd, kd, vd, causal=True, rope_base=base)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dOd, causal=True, rope_base=base)
    attn.attn_check()
    b, heads = B - 1, [5, 30]
    sl = lambda a: np.ascontiguousarray(a[b:b + 1][:, :, heads])
    rq, rk, rv = oracle.attn_bwd(sl(q), sl(k), sl(v), sl(dO), causal=True, rope_base=base)
    got = lambda t: t[b:b + 1][:, :, heads].float().cpu().numpy()
    tag = "rope_causal_s8192 backward, batch 3, heads 5 and 30"
    _check_grad(got(dv), rv, tag + " dV")
    _check_grad(got(dk), rk, tag + " dK")
    _check_grad(got(dq), rq, tag + " dQ")


# ---------------------------------------------------------------- block-sparse forward
BS = [
    # B, Hq, Hkv, S, D, causal, rope_base, mask
    (2, 4, 2, 1000, 128, False, 10000.0, "bigbird"),
    (1, 4, 4, 1024, 128, True, 10000.0, "bigbird"),
    (1, 2, 1, 300, 64, True, None, "full"),
    (2, 3, 3, 640, 128, False, 500000.0, "empty_row"),
    (1, 2, 2, 4096, 128, False, 10000.0, "bigbird"),
]


def _bs_mask(kind, S, causal):
    nb = (S + 127) // 128
    if kind == "bigbird":
        return si.bigbird_block_mask(S, window=0, n_global=1, n_random=1, seed=S, causal=causal)
    if kind == "full":
        return attn.create_block_mask(lambda qb, kb: (kb <= qb) or not causal, S)
    return attn.create_block_mask(lambda qb, kb: qb != 2 and (kb == qb or kb == 0), S)  # block row 2 empty


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base,kind", BS)
def test_blocksparse_forward_matches_oracle(B, Hq, Hkv, S, D, causal, base, kind):
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=700 + S)
    rp, ci = _bs_mask(kind, S, causal)
    o, lse = attn.attn_fwd_blocksparse(_dev(q), _dev(k), _dev(v), rp, ci, causal=causal, rope_base=base)
    attn.attn_check()
    if S <= 1024:
        o_ref, lse_ref = oracle.attn_full_bs(q, k, v, rp, ci, causal=causal, rope_base=base)
        og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
        empty = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lg), empty)
        assert np.all(og.transpose(0, 2, 1, 3)[empty] == 0.0)
        keep = ~empty
        _check(og.transpose(0, 2, 1, 3)[keep], lg[keep], o_ref.transpose(0, 2, 1, 3)[keep], lse_ref[keep],
               f"block-sparse {kind} S={S}")
    else:  # sampled rows
        rows = si.sample_rows(S, S, n=128)
        rb = np.zeros(len(rows), int)
        rh = np.arange(len(rows)) % Hq
        o_ref, lse_ref = oracle.attn_rows_bs(q, k, v, rp, ci, rb, rh, rows, causal=causal, rope_base=base)
        og = o.float().cpu().numpy()[rb, rows, rh]
        lg = lse.cpu().numpy()[rb, rh, rows]
        _check(og, lg, o_ref, lse_ref, f"block-sparse {kind} S={S} (sampled)")


# Shapes with several tasks (query tile, batch, head) per CTA of the persistent block-sparse
# kernel (B * Hq * ceil(S/128) well above the 152 CTAs), so ring slots, barrier phases and the
# overlap of one task's epilogue with the next task's loads and products run across tasks.
# Rows are sampled over every batch, head and query tile.
BS_MANY = [
    # B, Hq, Hkv, S, D, causal, rope_base, mask
    (4, 16, 8, 2048, 128, True, 10000.0, "bigbird"),     # 1024 tasks, RoPE, GQA
    (8, 8, 8, 1024, 64, False, None, "empty_row"),       # 512 tasks: rows of 0, 1 and 2 listed tiles
    (2, 16, 16, 4000, 128, False, 500000.0, "bigbird"),  # 1024 tasks, ragged last tile
]


def _sample_bhi(seed, B, Hq, S, n):
    w = si.uniform_words(seed, 4242, 0, 3 * n)
    rb = (w[:n] % np.uint64(B)).astype(np.int64)
    rh = (w[n:2 * n] % np.uint64(Hq)).astype(np.int64)
    ri = (w[2 * n:] % np.uint64(S)).astype(np.int64)
    # every batch-head's last row and a row of every query tile of batch-head (0, 0)
    bb, hh = np.meshgrid(np.arange(B), np.arange(Hq), indexing="ij")
    tiles = np.arange(0, S, 128) + 127
    rb = np.concatenate([rb, bb.ravel(), np.zeros(len(tiles), np.int64)])
    rh = np.concatenate([rh, hh.ravel(), np.zeros(len(tiles), np.int64)])
    ri = np.concatenate([ri, np.full(B * Hq, S - 1), np.minimum(tiles, S - 1)])
    return rb, rh, ri


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base,kind", BS_MANY)
def test_blocksparse_forward_many_tasks_per_cta(B, Hq, Hkv, S, D, causal, base, kind):
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=750 + S)
    rp, ci = _bs_mask(kind, S, causal)
    o, lse = attn.attn_fwd_blocksparse(_dev(q), _dev(k), _dev(v), rp, ci, causal=causal, rope_base=base)
    attn.attn_check()
    rb, rh, ri = _sample_bhi(S + B, B, Hq, S, 768)
    o_ref, lse_ref = oracle.attn_rows_bs(q, k, v, rp, ci, rb, rh, ri, causal=causal, rope_base=base)
    og = o.float().cpu().numpy()[rb, ri, rh]
    lg = lse.cpu().numpy()[rb, rh, ri]
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), empty)
    assert np.all(og[empty] == 0.0)
    _check(og[~empty], lg[~empty], o_ref[~empty], lse_ref[~empty], f"block-sparse {kind} S={S} B={B} Hq={Hq}")
    # the same call again gives the same bits (static schedule, no atomics)
    o2, lse2 = attn.attn_fwd_blocksparse(_dev(q), _dev(k), _dev(v), rp, ci, causal=causal, rope_base=base)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


LOCAL_MANY = [
    # B, Hq, Hkv, S, D, causal, rope_base, window, alibi
    (4, 12, 12, 4096, 64, True, None, 512, False),   # the sliding-window workload's shape
    (4, 12, 12, 2048, 64, True, None, 0, True),      # ALiBi, 768 tasks
    (2, 8, 4, 3000, 128, False, 10000.0, 300, True),  # both, non-causal, RoPE, ragged
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base,window,alibi", LOCAL_MANY)
def test_local_forward_many_tasks_per_cta(B, Hq, Hkv, S, D, causal, base, window, alibi):
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=950 + S)
    o, lse = attn.attn_fwd_local(_dev(q), _dev(k), _dev(v), causal=causal, rope_base=base, window=window,
                                 alibi=alibi)
    attn.attn_check()
    rb, rh, ri = _sample_bhi(S + 7, B, Hq, S, 768)
    o_ref, lse_ref = oracle.attn_rows_local(q, k, v, rb, rh, ri, causal=causal, rope_base=base, window=window,
                                            alibi=alibi)
    _check(o.float().cpu().numpy()[rb, ri, rh], lse.cpu().numpy()[rb, rh, ri], o_ref, lse_ref,
           f"local w={window} alibi={alibi} S={S} B={B} Hq={Hq}")


def test_blocksparse_full_mask_matches_dense_forward():
    """Every block listed: the same attention as the dense kernel (both round operands alike)."""
    B, Hq, Hkv, S, D, base = 1, 4, 2, 700, 128, 10000.0
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=777)
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    rp, ci = attn.create_block_mask(lambda qb, kb: kb <= qb, S)
    o, lse = attn.attn_fwd_blocksparse(qd, kd, vd, rp, ci, causal=True, rope_base=base)
    o_d, lse_d = attn.attn_fwd(qd, kd, vd, causal=True, rope_base=base)
    attn.attn_check()
    assert (o.float() - o_d.float()).abs().max().item() <= 1e-2
    assert (lse - lse_d).abs().max().item() <= 1e-3


BS_BWD = [
    # B, Hq, Hkv, S, D, causal, rope_base, mask
    (1, 4, 2, 1000, 128, False, 10000.0, "bigbird"),
    (1, 2, 2, 640, 128, True, 10000.0, "bigbird"),
    (2, 2, 1, 384, 64, False, None, "empty_row"),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base,kind", BS_BWD)
def test_blocksparse_backward_matches_oracle(B, Hq, Hkv, S, D, causal, base, kind):
    """attn_bwd under a block mask, on attn_fwd_blocksparse's own O and LSE, against the masked chain rule."""
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=800 + S)
    dO = si.bshd_bf16(801 + S, 9, B, S, Hq, D)
    rp, ci = _bs_mask(kind, S, causal)
    qd, kd, vd, dOd = _dev(q), _dev(k), _dev(v), _dev(dO)
    o, lse = attn.attn_fwd_blocksparse(qd, kd, vd, rp, ci, causal=causal, rope_base=base)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dOd, causal=causal, rope_base=base, block_mask=(rp, ci))
    attn.attn_check()
    rq, rk, rv = oracle.attn_bwd(q, k, v, dO, causal=causal, rope_base=base, block_mask=(rp, ci))
    tag = f"block-sparse backward {kind} S={S}"
    _check_grad(dv.float().cpu().numpy(), rv, tag + " dV")
    _check_grad(dk.float().cpu().numpy(), rk, tag + " dK")
    _check_grad(dq.float().cpu().numpy(), rq, tag + " dQ")


# ---------------------------------------------------------------- sliding window and ALiBi
LOCAL = [
    # B, Hq, Hkv, S, D, causal, rope_base, window, alibi
    (1, 4, 4, 1000, 64, True, None, 256, False),     # GPT-2-small head size, causal sliding window
    (2, 4, 2, 700, 128, True, 10000.0, 0, True),     # ALiBi over the whole causal range, RoPE, GQA
    (1, 2, 2, 640, 64, False, None, 100, True),      # both, non-causal window
    (1, 3, 3, 300, 128, True, 10000.0, 1, True),     # a window of one key: O_i = V_i
    (1, 2, 2, 520, 128, True, None, 45, False),      # both window edges inside one tile and one 32-key chunk
    (1, 4, 2, 900, 64, True, 10000.0, 200, True),    # causal window and ALiBi: masked biased tiles, ragged
    (1, 8, 2, 777, 128, True, 10000.0, 128, False),  # a window of exactly one tile, GQA group of 4, RoPE
    (1, 2, 2, 513, 64, False, None, 512, False),     # non-causal window of S - 1 keys, ragged
    (2, 2, 1, 384, 64, False, 500000.0, 0, True),    # non-causal ALiBi over the whole range, GQA, RoPE
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base,window,alibi", LOCAL)
def test_local_forward_matches_oracle(B, Hq, Hkv, S, D, causal, base, window, alibi):
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=900 + S)
    o, lse = attn.attn_fwd_local(_dev(q), _dev(k), _dev(v), causal=causal, rope_base=base, window=window,
                                 alibi=alibi)
    attn.attn_check()
    o_ref, lse_ref = oracle.attn_full_local(q, k, v, causal=causal, rope_base=base, window=window, alibi=alibi)
    tag = f"local w={window} alibi={alibi} S={S}"
    if window != 1:
        _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, tag)
        return
    # one key per row: O_i = V_i, and LSE_i is the single score, whose error is not averaged over
    # keys.  Rounding the rotated q', k' to fp16 (relative 2^-11 each) bounds it by
    # 2 * 2^-11 * sum_d |q'_d k'_d| / sqrt(D) (+ fp32 slack).
    _check(o.float().cpu().numpy(), None, o_ref, None, tag)
    qr = oracle.rope_rotate(q, base) if base else si.bf16_bits_to_f64(q)
    kr = oracle.rope_rotate(k, base) if base else si.bf16_bits_to_f64(k)
    kr = np.repeat(kr, Hq // Hkv, axis=2)
    bound = 2 * 2.0 ** -11 * np.abs(qr * kr).sum(-1).transpose(0, 2, 1) / np.sqrt(D) + 1e-5
    assert np.all(np.abs(lse.cpu().numpy() - lse_ref) <= bound), f"{tag}: LSE beyond the fp16 rounding bound"


def test_local_window_of_s_or_more_is_no_window():
    """|i - j| < window holds for every pair once window >= S: the host treats it as no window."""
    q, k, v = si.make_qkv(1, 2, 2, 600, 64, seed=977)
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    for alibi in (False, True):
        o0, l0 = attn.attn_fwd_local(qd, kd, vd, causal=True, window=0, alibi=alibi)
        o1, l1 = attn.attn_fwd_local(qd, kd, vd, causal=True, window=2 ** 31 - 1, alibi=alibi)
        o2, l2 = attn.attn_fwd_local(qd, kd, vd, causal=True, window=600, alibi=alibi)
        attn.attn_check()
        assert torch.equal(o0, o1) and torch.equal(l0, l1) and torch.equal(o0, o2) and torch.equal(l0, l2)


LOCAL_BWD = [
    # B, Hq, Hkv, S, D, causal, rope_base, window, alibi
    (1, 4, 4, 1000, 64, True, None, 256, False),     # causal sliding window, ragged tail
    (2, 4, 2, 700, 128, True, 10000.0, 0, True),     # ALiBi over the whole causal range, RoPE, GQA
    (1, 2, 2, 640, 64, False, None, 100, True),      # both, non-causal window (bias changes sign in a tile)
    (1, 4, 2, 900, 64, True, 10000.0, 200, True),    # causal window and ALiBi, ragged
    (1, 2, 2, 520, 128, True, None, 45, False),      # both window edges inside one tile
    (1, 3, 3, 300, 128, True, 10000.0, 1, True),     # a window of one key: dV = dO, dQ = dK = 0
    (1, 8, 2, 777, 128, True, 10000.0, 128, False),  # a window of exactly one tile, GQA group of 4, RoPE
    (1, 2, 2, 513, 64, False, None, 512, False),     # non-causal window of S - 1 keys, ragged
    (2, 2, 1, 384, 64, False, 500000.0, 0, True),    # non-causal ALiBi over the whole range, GQA, RoPE
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base,window,alibi", LOCAL_BWD)
def test_local_backward_matches_oracle(B, Hq, Hkv, S, D, causal, base, window, alibi):
    """attn_bwd_local on attn_fwd_local's own O and LSE against the float64 chain rule with the band and bias."""
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=1900 + S)
    dO = si.bshd_bf16(1901 + S, 9, B, S, Hq, D)
    qd, kd, vd, dOd = _dev(q), _dev(k), _dev(v), _dev(dO)
    o, lse = attn.attn_fwd_local(qd, kd, vd, causal=causal, rope_base=base, window=window, alibi=alibi)
    dq, dk, dv = attn.attn_bwd_local(qd, kd, vd, o, lse, dOd, causal=causal, rope_base=base, window=window,
                                     alibi=alibi)
    attn.attn_check()
    rq, rk, rv = oracle.attn_bwd(q, k, v, dO, causal=causal, rope_base=base, window=window, alibi=alibi)
    tag = f"local backward w={window} alibi={alibi} S={S}"
    _check_grad(dv.float().cpu().numpy(), rv, tag + " dV")
    if window == 1:
        # P = 1 up to its bf16 rounding, so dS = P dO.(V - O) is a rounding residue, not 0
        bound = 2e-2 * np.abs(rv).max()
        assert np.abs(dq.float().cpu().numpy()).max() <= bound and np.abs(dk.float().cpu().numpy()).max() <= bound
        return
    _check_grad(dk.float().cpu().numpy(), rk, tag + " dK")
    _check_grad(dq.float().cpu().numpy(), rq, tag + " dQ")


@pytest.mark.parametrize("window,alibi", [(512, False), (0, True)])
def test_local_backward_full_shape_one_batch(window, alibi):
    """The timed local backward's own shape (B=4, H=12, S=4096, D=64, causal; the sliding window of 512
    keys, or ALiBi): every gradient row of one batch element, all heads, against the chain rule on that
    batch element alone (batch elements are independent; the ALiBi slopes depend only on h and Hq)."""
    B, Hq, Hkv, S, D = 4, 12, 12, 4096, 64
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=2030)
    dO = si.bshd_bf16(2031, 9, B, S, Hq, D)
    qd, kd, vd, dOd = _dev(q), _dev(k), _dev(v), _dev(dO)
    o, lse = attn.attn_fwd_local(qd, kd, vd, causal=True, window=window, alibi=alibi)
    dq, dk, dv = attn.attn_bwd_local(qd, kd, vd, o, lse, dOd, causal=True, window=window, alibi=alibi)
    attn.attn_check()
    b = 2
    sl = lambda a: np.ascontiguousarray(a[b:b + 1])
    rq, rk, rv = oracle.attn_bwd(sl(q), sl(k), sl(v), sl(dO), causal=True, window=window, alibi=alibi)
    got = lambda t: t[b:b + 1].float().cpu().numpy()
    tag = f"local backward S=4096 window={window} alibi={alibi}, batch 2"
    _check_grad(got(dv), rv, tag + " dV")
    _check_grad(got(dk), rk, tag + " dK")
    _check_grad(got(dq), rq, tag + " dQ")


def test_blocksparse_backward_bigbird_full_shape_two_heads():
    """The timed block-sparse backward's own shape (bigbird_s4096: B=4, H=32, S=4096, D=128, full
    attention over the BigBird-style mask): every gradient row of two heads of one batch element against
    the masked chain rule on those heads alone (the mask is shared by every head)."""
    w = si.WORKLOADS["bigbird_s4096"]
    B, Hq, Hkv, S, D = w["B"], w["Hq"], w["Hkv"], w["S"], w["D"]
    rp, ci = si.bigbird_block_mask(S, causal=w["causal"], **w["block_mask"])
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=2040)
    dO = si.bshd_bf16(2041, 9, B, S, Hq, D)
    qd, kd, vd, dOd = _dev(q), _dev(k), _dev(v), _dev(dO)
    o, lse = attn.attn_fwd_blocksparse(qd, kd, vd, rp, ci, causal=w["causal"])
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dOd, causal=w["causal"], block_mask=(rp, ci))
    attn.attn_check()
    b, heads = 1, [0, 19]
    sl = lambda a: np.ascontiguousarray(a[b:b + 1][:, :, heads])
    rq, rk, rv = oracle.attn_bwd(sl(q), sl(k), sl(v), sl(dO), causal=w["causal"], block_mask=(rp, ci))
    got = lambda t: t[b:b + 1][:, :, heads].float().cpu().numpy()
    tag = "bigbird_s4096 backward, batch 1, heads 0 and 19"
    _check_grad(got(dv), rv, tag + " dV")
    _check_grad(got(dk), rk, tag + " dK")
    _check_grad(got(dq), rq, tag + " dQ")

