"""Pins for the oracle's sliding-window and ALiBi attention.

- no window and no ALiBi: the dense oracle (special case);
- a window: float64 SDPA with the boolean band mask, RoPE as complex multiplication;
- ALiBi: float64 SDPA with the additive bias -m_h |i - j|, m_h = 2^(-8 (h+1) / H)
  (slopes of the linear-bias paper), causal and full;
- both together; and the window of one key, O_i = V_i (closed form).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si


def _rope_torch(x, base):
    B, S, H, D = x.shape
    h = D // 2
    theta = base ** (-2.0 * torch.arange(h, dtype=torch.float64) / D)
    ang = torch.arange(S, dtype=torch.float64)[:, None] * theta[None, :]
    z = torch.complex(x[..., :h], x[..., h:]) * torch.polar(torch.ones_like(ang), ang)[None, :, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def _sdpa(q, k, v, base, bias):
    G = q.shape[2] // k.shape[2]
    qt = torch.from_numpy(si.bf16_bits_to_f64(q))
    kt = torch.from_numpy(si.bf16_bits_to_f64(k))
    if base:
        qt, kt = _rope_torch(qt, base), _rope_torch(kt, base)
    qh = qt.permute(0, 2, 1, 3)
    kh = kt.permute(0, 2, 1, 3).repeat_interleave(G, 1)
    vh = torch.from_numpy(si.bf16_bits_to_f64(v)).permute(0, 2, 1, 3).repeat_interleave(G, 1)
    o = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=bias)
    s = torch.matmul(qh, kh.transpose(-1, -2)) / math.sqrt(q.shape[-1]) + bias
    return o.permute(0, 2, 1, 3).numpy(), torch.logsumexp(s, dim=-1).numpy()


def _bias(S, H, causal, window, alibi):
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    dist = np.abs(i - j)
    ok = np.ones((S, S), bool)
    if causal:
        ok &= j <= i
    if window:
        ok &= dist < window
    slopes = 2.0 ** (-8.0 * (np.arange(H) + 1) / H) if alibi else np.zeros(H)
    b = -slopes[:, None, None] * dist[None]
    b = np.where(ok[None], b, -np.inf)
    return torch.from_numpy(b[None])


@pytest.mark.parametrize("causal,window,alibi,base", [(True, 40, False, 10000.0), (False, 17, False, None),
                                                      (True, 0, True, 10000.0), (False, 0, True, None),
                                                      (True, 25, True, 500000.0)])
def test_local_attention_equals_biased_library_sdpa(causal, window, alibi, base):
    B, Hq, Hkv, S, D = 1, 4, 2, 90, 16
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=41)
    o, lse = oracle.attn_full_local(q, k, v, causal=causal, rope_base=base, window=window, alibi=alibi)
    o_ref, lse_ref = _sdpa(q, k, v, base, _bias(S, Hq, causal, window, alibi))
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_no_window_no_bias_is_the_dense_oracle():
    q, k, v = si.make_qkv(1, 2, 2, 77, 32, seed=42)
    o, lse = oracle.attn_full_local(q, k, v, causal=True, rope_base=10000.0)
    o2, lse2 = oracle.attn_full(q, k, v, causal=True, rope_base=10000.0)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)


def test_window_of_one_key_returns_the_value_row():
    q, k, v = si.make_qkv(1, 2, 1, 33, 16, seed=43)
    o, _ = oracle.attn_full_local(q, k, v, causal=True, rope_base=10000.0, window=1, alibi=True)
    np.testing.assert_allclose(o, np.repeat(si.bf16_bits_to_f64(v), 2, axis=2), rtol=0, atol=1e-15)
