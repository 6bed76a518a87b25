"""Pins for the CPU oracle: each test ties it to something other than itself.

- a library routine (torch scaled_dot_product_attention / logsumexp in float64),
- RoPE written as complex multiplication instead of the oracle's cos/sin formulas,
- a per-cell brute force that uses only the relative angle (i-j)*theta_r,
- closed forms (S=1, constant V, a window narrower than one position),
- invariants (softmax rows sum to one, causal zeros, shift invariance, GQA = MHA),
- the window rule's closed-form pruned count, and the pruned share the
  ATFlash page prints.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-12


def _qkv(B, Hq, Hkv, S, D, seed=7):
    return si.make_qkv(B, Hq, Hkv, S, D, seed=seed)


def _f64(bits):
    return si.bf16_bits_to_f64(bits)


def _sdpa_ref(q, k, v, causal, G):
    """torch SDPA (float64, CPU) + torch logsumexp of the masked scaled scores."""
    qt = torch.from_numpy(_f64(q)).permute(0, 2, 1, 3)  # B H S D
    kt = torch.from_numpy(_f64(k)).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    vt = torch.from_numpy(_f64(v)).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal)
    s = torch.matmul(qt, kt.transpose(-1, -2)) / math.sqrt(qt.shape[-1])
    if causal:
        S = s.shape[-1]
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy()


def _rope_complex(x_bits, base, offset=0):
    """RoPE as complex multiplication: z_r = x_r + i x_{r+D/2}, z'_r = z_r * exp(i p theta_r)."""
    x = _f64(x_bits)
    B, S, H, D = x.shape
    h = D // 2
    theta = base ** (-2.0 * np.arange(h) / D)
    pos = (np.arange(S) + offset)[None, :, None, None]
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * pos * theta[None, None, None, :])
    return np.concatenate([z.real, z.imag], axis=-1)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2), (3, 1)])
def test_rope_off_equals_library_sdpa(causal, Hq, Hkv):
    B, S, D = 2, 37, 16
    q, k, v = _qkv(B, Hq, Hkv, S, D)
    o, lse = oracle.attn_full(q, k, v, causal=causal)
    o_ref, lse_ref = _sdpa_ref(q, k, v, causal, Hq // Hkv)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=TOL)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=TOL)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("base", [10000.0, 500000.0, 37.0])
def test_rope_equals_complex_rotation_then_sdpa(causal, base):
    B, Hq, Hkv, S, D = 1, 4, 2, 29, 32
    q, k, v = _qkv(B, Hq, Hkv, S, D, seed=11)
    o, lse = oracle.attn_full(q, k, v, causal=causal, rope_base=base)
    qr = _rope_complex(q, base)
    kr = _rope_complex(k, base)
    G = Hq // Hkv
    qt = torch.from_numpy(qr).permute(0, 2, 1, 3)
    kt = torch.from_numpy(kr).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    vt = torch.from_numpy(_f64(v)).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    o_ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal)
    s = torch.matmul(qt, kt.transpose(-1, -2)) / math.sqrt(D)
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(o, o_ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("base", [10000.0, 500000.0, 37.0])
def test_standalone_rotation_equals_complex_rotation(base):
    """The oracle's standalone rotation (used to check the pre-rotation kernel)
    against multiplication by e^{i p theta_r}: a different formulation."""
    x = si.bshd_bf16(7, 1, 2, 33, 3, 64)
    got = oracle.rope_rotate(x, base)
    np.testing.assert_allclose(got, _rope_complex(x, base), rtol=0, atol=1e-12)
    # a rotation keeps each pair's length, and position 0 is the identity
    xf = _f64(x)
    h = 32
    np.testing.assert_allclose(got[..., :h] ** 2 + got[..., h:] ** 2, xf[..., :h] ** 2 + xf[..., h:] ** 2,
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(got[:, 0], xf[:, 0])


def _brute_relative(q, k, v, base, window_k):
    """Per-cell brute force from unrotated q, k and the relative angle only.

    q'_i . k'_j = sum_r cos(d theta_r) (q_r k_r + q_{r+h} k_{r+h}) + sin(d theta_r) (q_r k_{r+h} - q_{r+h} k_r),
    d = i - j: the pair's contribution depends only on the distance.  The
    window drops pair r when d > floor(k * 2 pi / theta_r).  Two-pass softmax
    with math.fsum.  Causal, one batch, one head.
    """
    S, D = q.shape
    h = D // 2
    theta = [base ** (-2.0 * r / D) for r in range(h)]
    W = [math.floor(window_k * 2 * math.pi / t) if window_k else math.inf for t in theta]
    O = np.zeros((S, D))
    L = np.zeros(S)
    for i in range(S):
        s = []
        for j in range(i + 1):
            d = i - j
            terms = []
            for r in range(h):
                if d > W[r]:
                    continue
                c, sn = math.cos(d * theta[r]), math.sin(d * theta[r])
                terms.append(c * (q[i, r] * k[j, r] + q[i, r + h] * k[j, r + h]))
                terms.append(sn * (q[i, r] * k[j, r + h] - q[i, r + h] * k[j, r]))
            s.append(math.fsum(terms) / math.sqrt(D))
        m = max(s)
        e = [math.exp(x - m) for x in s]
        l = math.fsum(e)
        for dd in range(D):
            O[i, dd] = math.fsum(e[j] * v[j, dd] for j in range(i + 1)) / l
        L[i] = m + math.log(l)
    return O, L


@pytest.mark.parametrize("window_k", [None, 0.5, 1.0])
def test_relative_angle_brute_force(window_k):
    B, H, S, D = 1, 1, 16, 8
    base = 100.0
    q, k, v = _qkv(B, H, H, S, D, seed=3)
    o, lse = oracle.attn_full(q, k, v, causal=True, rope_base=base, window_k=window_k)
    O, L = _brute_relative(_f64(q)[0, :, 0], _f64(k)[0, :, 0], _f64(v)[0, :, 0], base, window_k)
    np.testing.assert_allclose(o[0, :, 0], O, rtol=0, atol=TOL)
    np.testing.assert_allclose(lse[0, 0], L, rtol=0, atol=TOL)
    if window_k:
        # the window really prunes something at these sizes, so this case is not the unwindowed one
        o_off, _ = oracle.attn_full(q, k, v, causal=True, rope_base=base)
        assert np.abs(o_off - o).max() > 1e-3


@pytest.mark.parametrize("rope_base", [None, 10000.0])
def test_single_position_closed_form(rope_base):
    q, k, v = _qkv(2, 4, 2, 1, 64, seed=5)
    o, lse = oracle.attn_full(q, k, v, causal=True, rope_base=rope_base)
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    for b in range(2):
        for h in range(4):
            g = h // 2
            assert np.array_equal(o[b, 0, h], vf[b, 0, g])  # softmax of one key is exactly 1
            assert abs(lse[b, h, 0] - qf[b, 0, h] @ kf[b, 0, g] / 8.0) < TOL  # position 0: no rotation


def test_constant_values_give_constant_output():
    B, H, S, D = 1, 2, 50, 16
    q, k, _ = _qkv(B, H, H, S, D, seed=9)
    c = si.f64_to_bf16_bits(np.linspace(-3, 3, D))
    v = np.broadcast_to(c, (B, S, H, D)).copy()
    for causal in (True, False):
        o, _ = oracle.attn_full(q, k, v, causal=causal, rope_base=10000.0)
        np.testing.assert_allclose(o, np.broadcast_to(_f64(c), o.shape), rtol=0, atol=TOL)


@pytest.mark.parametrize("window_k", [None, 0.25])
def test_one_hot_values_expose_probabilities(window_k):
    """V_j = e_j makes O_i the probability row i: non-negative, sums to 1, zero above the diagonal."""
    S = D = 32
    q, k, _ = _qkv(1, 1, 1, S, D, seed=13)
    v = si.f64_to_bf16_bits(np.eye(S)).reshape(1, S, 1, D)
    o, _ = oracle.attn_full(q, k, v, causal=True, rope_base=50.0, window_k=window_k)
    P = o[0, :, 0, :]
    assert (P >= 0).all()
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=TOL)
    assert np.all(P[np.triu_indices(S, 1)] == 0.0)
    assert np.all(np.diag(P) > 0)


@pytest.mark.parametrize("window_k", [None, 1.0])
def test_rope_shift_invariance(window_k):
    """RoPE scores depend only on relative position: shifting every position changes nothing."""
    q, k, v = _qkv(1, 2, 1, 40, 32, seed=17)
    o0, l0 = oracle.attn_full(q, k, v, causal=True, rope_base=100.0, window_k=window_k)
    o1, l1 = oracle.attn_full(q, k, v, causal=True, rope_base=100.0, window_k=window_k, pos_offset=12345)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-9)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-9)


def test_window_infinite_k_is_window_off():
    q, k, v = _qkv(1, 2, 2, 64, 32, seed=19)
    o0, l0 = oracle.attn_full(q, k, v, causal=True, rope_base=10000.0)
    o1, l1 = oracle.attn_full(q, k, v, causal=True, rope_base=10000.0, window_k=1e30)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_window_below_one_position_closed_form():
    """k so small that W_r = 0 for every pair: only the diagonal keeps its terms.

    Then s_ij = 0 for j < i and s_ii = q_i . k_i / sqrt(D) (same position, the
    rotations cancel), so O_i = (sum_{j<i} V_j + e^{s_ii} V_i) / (i + e^{s_ii})
    and LSE_i = ln(i + e^{s_ii}).
    """
    S, D = 24, 16
    q, k, v = _qkv(1, 1, 1, S, D, seed=23)
    o, lse = oracle.attn_full(q, k, v, causal=True, rope_base=10000.0, window_k=1e-9)
    qf, kf, vf = _f64(q)[0, :, 0], _f64(k)[0, :, 0], _f64(v)[0, :, 0]
    for i in range(S):
        sii = qf[i] @ kf[i] / math.sqrt(D)
        e = math.exp(sii)
        O = (vf[:i].sum(axis=0) + e * vf[i]) / (i + e)
        np.testing.assert_allclose(o[0, i, 0], O, rtol=0, atol=1e-11)
        assert abs(lse[0, 0, i] - math.log(i + e)) < 1e-11


def test_gqa_equals_mha_with_repeated_kv():
    B, Hq, Hkv, S, D = 2, 6, 2, 33, 32
    q, k, v = _qkv(B, Hq, Hkv, S, D, seed=29)
    G = Hq // Hkv
    o, l = oracle.attn_full(q, k, v, causal=True, rope_base=10000.0, window_k=2.0)
    k2 = np.repeat(k, G, axis=2)
    v2 = np.repeat(v, G, axis=2)
    o2, l2 = oracle.attn_full(q, k2, v2, causal=True, rope_base=10000.0, window_k=2.0)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


def _closed_form_pruned(S, D, base, k):
    """sum_r T(max(0, S-1-W_r)), T(n) = n(n+1)/2: cells at distance d > W_r number S-d."""
    total = 0
    for r in range(D // 2):
        W = math.floor(k * 2 * math.pi / base ** (-2.0 * r / D))
        n = max(0, S - 1 - W)
        total += n * (n + 1) // 2
    return total


@pytest.mark.parametrize("S", [16, 128, 2048])
@pytest.mark.parametrize("base,k", [(10000.0, 1.0), (10000.0, 4.0), (500000.0, 1.0), (500000.0, 0.05)])
def test_pruned_count_matches_closed_form(S, base, k):
    assert oracle.pruned_terms(S, 128, base, k) == _closed_form_pruned(S, 128, base, k)


def test_pruned_share_matches_page():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "atflash_pruned_share.txt")) if l.strip() and not l.startswith("#")]
    for base, D, S, k, lo, hi in rows:
        base, D, S, k, lo, hi = float(base), int(D), int(S), float(k), float(lo), float(hi)
        frac = _closed_form_pruned(S, D, base, k) / ((D // 2) * S * (S + 1) / 2)
        assert lo <= frac <= hi, (k, frac)


def test_window_widths_are_floor_k_wavelength():
    w = oracle.window_widths(128, 500000.0, 4.0)
    lam = 2 * math.pi / (500000.0 ** (-2.0 * np.arange(64) / 128))
    assert np.array_equal(w, np.floor(4.0 * lam))
    assert np.all(np.diff(w) >= 0)  # low frequencies keep longer distances
    assert np.all(np.isinf(oracle.window_widths(128, 500000.0, 0.0)))


def test_oracle_rejects_window_without_rope_or_causal():
    q, k, v = _qkv(1, 1, 1, 8, 16)
    with pytest.raises(ValueError):
        oracle.attn_full(q, k, v, causal=True, rope_base=None, window_k=1.0)
    with pytest.raises(ValueError):
        oracle.attn_full(q, k, v, causal=False, rope_base=10000.0, window_k=1.0)


def test_exp2_scale_constant_matches_page():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "exp2_scale.txt")) if l.strip() and not l.startswith("#")]
    for D, printed, digits in rows:
        assert round(math.log2(math.e) / math.sqrt(int(D)), int(digits)) == float(printed)
