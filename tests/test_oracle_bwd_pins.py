"""Pins for the oracle's backward pass (gradients of sum(O * dO)).

Each test ties it to something other than itself:
- torch autograd through scaled_dot_product_attention in float64, with RoPE
  written as complex multiplication (a library routine and a different
  formulation of the rotation);
- central finite differences of a forward written with explicit 2x2 rotation
  matrices, on a tiny case (brute force);
- invariants: the value gradients sum to the output gradients, a constant
  added to every value row leaves dQ and dK unchanged, the gradients of a
  fully masked-out key are zero, and GQA equals MHA with repeated K/V.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si


def _inputs(B, Hq, Hkv, S, D, seed):
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=seed)
    dO = si.bshd_bf16(seed + 1000, 9, B, S, Hq, D)
    return q, k, v, dO


def _rope_torch(x, base):
    """RoPE as complex multiplication on a float64 BSHD tensor: z_r * exp(i p theta_r)."""
    B, S, H, D = x.shape
    h = D // 2
    theta = base ** (-2.0 * torch.arange(h, dtype=torch.float64) / D)
    ang = torch.arange(S, dtype=torch.float64)[:, None] * theta[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)[None, :, None, :]
    z = torch.complex(x[..., :h], x[..., h:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def _autograd_ref(q, k, v, dO, causal, base):
    G = q.shape[2] // k.shape[2]
    qt, kt, vt = (torch.from_numpy(oracle.bf16_to_f64(a)).requires_grad_(True) for a in (q, k, v))
    qr = _rope_torch(qt, base) if base else qt
    kr = _rope_torch(kt, base) if base else kt
    qh = qr.permute(0, 2, 1, 3)
    kh = kr.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    vh = vt.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, is_causal=causal)
    loss = (o.permute(0, 2, 1, 3) * torch.from_numpy(oracle.bf16_to_f64(dO))).sum()
    loss.backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Hq,Hkv,base", [(2, 2, None), (4, 2, 10000.0), (3, 1, 500000.0), (2, 1, 37.0)])
def test_backward_equals_torch_autograd(causal, Hq, Hkv, base):
    q, k, v, dO = _inputs(2, Hq, Hkv, 23, 16, seed=5)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, causal=causal, rope_base=base)
    rq, rk, rv = _autograd_ref(q, k, v, dO, causal, base)
    np.testing.assert_allclose(dq, rq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, rk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, rv, rtol=0, atol=1e-11)


def _loss_explicit(q, k, v, dO, causal, base):
    """sum(O * dO) with RoPE as an explicit 2x2 rotation matrix per (position, pair)."""
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    h = D // 2

    def rot(x):
        out = np.empty_like(x)
        for s in range(S):
            for r in range(h):
                a = s * base ** (-2.0 * r / D) if base else 0.0
                m = np.array([[math.cos(a), -math.sin(a)], [math.sin(a), math.cos(a)]])
                pair = np.stack([x[:, s, :, r], x[:, s, :, r + h]], axis=-1)  # [B, H, 2]
                res = pair @ m.T
                out[:, s, :, r], out[:, s, :, r + h] = res[..., 0], res[..., 1]
        return out

    qr, kr = rot(q), rot(k)
    total = 0.0
    for b in range(B):
        for hh in range(Hq):
            g = hh // G
            s = qr[b, :, hh, :] @ kr[b, :, g, :].T / math.sqrt(D)
            if causal:
                s = np.where(np.tril(np.ones((S, S), bool)), s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            total += float(np.sum((p @ v[b, :, g, :]) * dO[b, :, hh, :]))
    return total


@pytest.mark.parametrize("causal,base", [(True, 10000.0), (False, 10.0), (True, None)])
def test_backward_matches_finite_differences(causal, base):
    rng = np.random.default_rng(3)
    B, Hq, Hkv, S, D = 1, 2, 1, 5, 4
    q = rng.standard_normal((B, S, Hq, D))
    k = rng.standard_normal((B, S, Hkv, D))
    v = rng.standard_normal((B, S, Hkv, D))
    dO = rng.standard_normal((B, S, Hq, D))
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, causal=causal, rope_base=base)
    eps = 1e-6
    for x, grad in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            up = _loss_explicit(q, k, v, dO, causal, base)
            x[idx] = old - eps
            dn = _loss_explicit(q, k, v, dO, causal, base)
            x[idx] = old
            num[idx] = (up - dn) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8)


def test_value_gradients_sum_to_output_gradients():
    """Each probability row sums to one, so sum_j dV_j = sum_i dO_i over a KV group's heads."""
    q, k, v, dO = _inputs(2, 4, 2, 31, 32, seed=8)
    _, _, dv = oracle.attn_bwd(q, k, v, dO, causal=True, rope_base=10000.0)
    dOf = oracle.bf16_to_f64(dO)
    for g in range(2):
        np.testing.assert_allclose(dv[:, :, g, :].sum(axis=1), dOf[:, :, 2 * g:2 * g + 2, :].sum(axis=(1, 2)),
                                   rtol=0, atol=1e-11)


def test_constant_value_shift_leaves_query_and_key_gradients():
    """V_j + c for every j shifts O_i by c; dP and Dlt shift alike, so dS, dQ and dK do not change."""
    q, k, v, dO = _inputs(1, 2, 2, 19, 16, seed=9)
    vf = oracle.bf16_to_f64(v)
    dq0, dk0, _ = oracle.attn_bwd(q, k, vf, dO, causal=True, rope_base=500000.0)
    dq1, dk1, _ = oracle.attn_bwd(q, k, vf + np.linspace(-3, 3, 16), dO, causal=True, rope_base=500000.0)
    np.testing.assert_allclose(dq1, dq0, rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk1, dk0, rtol=0, atol=1e-10)


def test_last_key_gets_gradient_only_from_the_last_query():
    """Under the causal mask key S-1 is seen by query S-1 alone; with that row's dO zero its dK, dV are zero."""
    q, k, v, dO = _inputs(1, 2, 1, 13, 16, seed=10)
    dOf = oracle.bf16_to_f64(dO)
    dOf[:, -1] = 0.0
    _, dk, dv = oracle.attn_bwd(q, k, v, dOf, causal=True, rope_base=10000.0)
    assert np.all(dk[:, -1] == 0.0) and np.all(dv[:, -1] == 0.0)
    assert np.abs(dk[:, :-1]).max() > 0 and np.abs(dv[:, :-1]).max() > 0


def test_gqa_backward_equals_mha_with_repeated_kv():
    """A KV head shared by G query heads gets the sum of the G heads' gradients."""
    q, k, v, dO = _inputs(1, 4, 2, 17, 16, seed=12)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, causal=True, rope_base=10000.0)
    k2, v2 = np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2)
    dq2, dk2, dv2 = oracle.attn_bwd(q, k2, v2, dO, causal=True, rope_base=10000.0)
    np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, dk2.reshape(1, 17, 2, 2, 16).sum(axis=3), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, dv2.reshape(1, 17, 2, 2, 16).sum(axis=3), rtol=0, atol=1e-12)


def _mask_autograd_ref(q, k, v, dO, causal, base, cell):
    """torch autograd through float64 SDPA with a cell mask; rows that see nothing are left out."""
    G = q.shape[2] // k.shape[2]
    qt, kt, vt = (torch.from_numpy(oracle.bf16_to_f64(a)).requires_grad_(True) for a in (q, k, v))
    qr = _rope_torch(qt, base) if base else qt
    kr = _rope_torch(kt, base) if base else kt
    qh = qr.permute(0, 2, 1, 3)
    kh = kr.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    vh = vt.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    seen = torch.from_numpy(cell.any(axis=1))
    s = torch.matmul(qh, kh.transpose(-1, -2)) / math.sqrt(q.shape[-1])
    s = s.masked_fill(~torch.from_numpy(cell), float("-inf"))
    pr = torch.softmax(s[..., seen, :], dim=-1)
    o = torch.matmul(pr, vh)
    dOt = torch.from_numpy(oracle.bf16_to_f64(dO)).permute(0, 2, 1, 3)[..., seen, :]
    (o * dOt).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("causal,base", [(False, 10000.0), (True, None)])
def test_block_sparse_backward_equals_masked_autograd(causal, base):
    """Under a CSR block mask (with one empty block row): torch autograd with the expanded cell mask."""
    S, blk = 37, 8
    q, k, v, dO = _inputs(1, 4, 2, S, 16, seed=31)
    nb = (S + blk - 1) // blk
    rows = [[0, 2], [1], [], [0, 3], [1, 2, 4]]
    if causal:
        rows = [[c for c in r if c <= i] for i, r in enumerate(rows)]
    rp = np.zeros(nb + 1, np.int32)
    rp[1:] = np.cumsum([len(r) for r in rows])
    ci = np.array([c for r in rows for c in r], np.int32)
    act = np.zeros((nb, nb), bool)
    for i, r in enumerate(rows):
        act[i, r] = True
    cell = act[np.arange(S)[:, None] // blk, np.arange(S)[None, :] // blk]
    if causal:
        cell &= np.tril(np.ones((S, S), bool))
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, causal=causal, rope_base=base, block_mask=(rp, ci), block=blk)
    rq, rk, rv = _mask_autograd_ref(q, k, v, dO, causal, base, cell)
    np.testing.assert_allclose(dq, rq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, rk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, rv, rtol=0, atol=1e-11)
    assert np.all(dq[:, 16:24] == 0.0)  # block row 2 sees nothing


def test_block_sparse_backward_with_every_block_is_dense():
    S, blk = 40, 16
    q, k, v, dO = _inputs(1, 2, 1, S, 16, seed=32)
    nb = (S + blk - 1) // blk
    rp = np.arange(nb + 1, dtype=np.int32) * nb
    ci = np.tile(np.arange(nb, dtype=np.int32), nb)
    a = oracle.attn_bwd(q, k, v, dO, causal=True, rope_base=10000.0, block_mask=(rp, ci), block=blk)
    b = oracle.attn_bwd(q, k, v, dO, causal=True, rope_base=10000.0)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def _local_autograd_ref(q, k, v, dO, causal, base, window, alibi):
    """torch autograd through float64 SDPA whose float mask carries the band (-inf outside
    |i - j| < window, and j > i when causal) and the ALiBi bias -m_h |i - j|, m_h = 2^(-8 (h+1) / Hq)."""
    B, S, Hq, D = q.shape
    G = Hq // k.shape[2]
    qt, kt, vt = (torch.from_numpy(oracle.bf16_to_f64(a)).requires_grad_(True) for a in (q, k, v))
    qr = _rope_torch(qt, base) if base else qt
    kr = _rope_torch(kt, base) if base else kt
    qh = qr.permute(0, 2, 1, 3)
    kh = kr.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    vh = vt.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    i = torch.arange(S)[:, None]
    j = torch.arange(S)[None, :]
    dist = (i - j).abs().to(torch.float64)
    ok = torch.ones(S, S, dtype=torch.bool)
    if causal:
        ok &= j <= i
    if window:
        ok &= dist < window
    slopes = (2.0 ** (-8.0 * (torch.arange(Hq, dtype=torch.float64) + 1) / Hq)) if alibi else torch.zeros(Hq,
                                                                                                          dtype=torch.float64)
    bias = torch.where(ok[None], -slopes[:, None, None] * dist[None], torch.tensor(float("-inf"), dtype=torch.float64))
    o = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=bias[None])
    loss = (o.permute(0, 2, 1, 3) * torch.from_numpy(oracle.bf16_to_f64(dO))).sum()
    loss.backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("causal,window,alibi,base", [(True, 7, False, 10000.0), (False, 5, False, None),
                                                      (True, 0, True, 500000.0), (False, 0, True, 10000.0),
                                                      (True, 9, True, None), (False, 6, True, 37.0)])
def test_local_backward_equals_banded_biased_autograd(causal, window, alibi, base):
    """Sliding window and/or ALiBi ("AttnFuse", sec. 3 combinators): torch autograd with the band and bias."""
    q, k, v, dO = _inputs(2, 4, 2, 29, 16, seed=41)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, causal=causal, rope_base=base, window=window, alibi=alibi)
    rq, rk, rv = _local_autograd_ref(q, k, v, dO, causal, base, window, alibi)
    np.testing.assert_allclose(dq, rq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, rk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, rv, rtol=0, atol=1e-11)


def test_local_backward_matches_finite_differences():
    """Window 3 and ALiBi on a tiny causal case: central differences of sum(O * dO), forward written out."""
    rng = np.random.default_rng(4)
    B, Hq, Hkv, S, D, W = 1, 2, 1, 6, 4, 3
    q = rng.standard_normal((B, S, Hq, D))
    k = rng.standard_normal((B, S, Hkv, D))
    v = rng.standard_normal((B, S, Hkv, D))
    dO = rng.standard_normal((B, S, Hq, D))

    def loss(q, k, v):
        total = 0.0
        for hh in range(Hq):
            m = 2.0 ** (-8.0 * (hh + 1) / Hq)
            for a in range(S):
                keys = [b for b in range(S) if b <= a and a - b < W]
                s = np.array([q[0, a, hh] @ k[0, b, 0] / math.sqrt(D) - m * (a - b) for b in keys])
                p = np.exp(s - s.max())
                p /= p.sum()
                total += float((p @ v[0, keys, 0]) @ dO[0, a, hh])
        return total

    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, causal=True, window=W, alibi=True)
    eps = 1e-6
    for x, grad in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            up = loss(q, k, v)
            x[idx] = old - eps
            dn = loss(q, k, v)
            x[idx] = old
            num[idx] = (up - dn) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8)


def test_local_backward_window_of_one_key_passes_dO_to_V():
    """A window of one key: O_i = V_i, so dV_j = dO_j (summed over the group's heads) and dQ = dK = 0."""
    q, k, v, dO = _inputs(1, 4, 2, 21, 16, seed=42)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, causal=True, rope_base=10000.0, window=1, alibi=True)
    dOf = oracle.bf16_to_f64(dO)
    np.testing.assert_array_equal(dq, 0.0)
    np.testing.assert_array_equal(dk, 0.0)
    np.testing.assert_allclose(dv, dOf.reshape(1, 21, 2, 2, 16).sum(axis=3), rtol=0, atol=1e-12)
