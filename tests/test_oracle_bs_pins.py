"""Pins for the oracle's block-sparse attention (a CSR BlockMask over 128 x 128 blocks).

- every block listed: the dense oracle (a special case that reduces to it);
- a random mask: torch scaled_dot_product_attention in float64 with the boolean
  mask expanded cell by cell, RoPE written as complex multiplication (a library
  routine and a different formulation);
- only the diagonal blocks: each block attends to itself alone, i.e. the dense
  oracle run on the block with its positions shifted (brute force by pieces);
- a row of blocks with nothing listed: O = 0 and LSE = -inf (the stated convention).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

BLK = 128


def _full_mask(S):
    nb = (S + BLK - 1) // BLK
    return np.arange(nb + 1, dtype=np.int32) * nb, np.tile(np.arange(nb, dtype=np.int32), nb)


@pytest.mark.parametrize("causal,Hq,Hkv,base", [(True, 2, 2, 10000.0), (False, 4, 2, None), (True, 3, 1, 500000.0)])
def test_all_blocks_listed_is_the_dense_oracle(causal, Hq, Hkv, base):
    S = 300
    q, k, v = si.make_qkv(1, Hq, Hkv, S, 32, seed=21)
    rp, ci = _full_mask(S)
    o, lse = oracle.attn_full_bs(q, k, v, rp, ci, causal=causal, rope_base=base)
    o2, lse2 = oracle.attn_full(q, k, v, causal=causal, rope_base=base)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)


def _rope_torch(x, base):
    B, S, H, D = x.shape
    h = D // 2
    theta = base ** (-2.0 * torch.arange(h, dtype=torch.float64) / D)
    ang = torch.arange(S, dtype=torch.float64)[:, None] * theta[None, :]
    z = torch.complex(x[..., :h], x[..., h:]) * torch.polar(torch.ones_like(ang), ang)[None, :, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


@pytest.mark.parametrize("causal", [False, True])
def test_random_mask_equals_masked_library_sdpa(causal):
    B, Hq, Hkv, S, D, base = 1, 4, 2, 520, 32, 10000.0
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=22)
    rp, ci = si.bigbird_block_mask(S, block=BLK, window=0, n_global=1, n_random=1, seed=5, causal=causal)
    o, lse = oracle.attn_full_bs(q, k, v, rp, ci, causal=causal, rope_base=base)
    nb = len(rp) - 1
    act = np.zeros((nb, nb), bool)
    for r in range(nb):
        act[r, ci[rp[r]:rp[r + 1]]] = True
    cell = act[np.arange(S)[:, None] // BLK, np.arange(S)[None, :] // BLK]
    if causal:
        cell &= np.tril(np.ones((S, S), bool))
    G = Hq // Hkv
    qt = _rope_torch(torch.from_numpy(si.bf16_bits_to_f64(q)), base).permute(0, 2, 1, 3)
    kt = _rope_torch(torch.from_numpy(si.bf16_bits_to_f64(k)), base).permute(0, 2, 1, 3).repeat_interleave(G, 1)
    vt = torch.from_numpy(si.bf16_bits_to_f64(v)).permute(0, 2, 1, 3).repeat_interleave(G, 1)
    mask = torch.from_numpy(cell)
    o_ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    s = torch.matmul(qt, kt.transpose(-1, -2)) / math.sqrt(D)
    lse_ref = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
    np.testing.assert_allclose(o, o_ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref.numpy(), rtol=0, atol=1e-12)


def test_diagonal_blocks_are_independent_attentions():
    """Block r alone: the dense oracle on rows/keys [128r, 128r+128) with positions shifted by 128r."""
    B, Hq, Hkv, S, D, base = 1, 2, 2, 300, 32, 10000.0
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=23)
    nb = (S + BLK - 1) // BLK
    rp = np.arange(nb + 1, dtype=np.int32)
    ci = np.arange(nb, dtype=np.int32)
    o, lse = oracle.attn_full_bs(q, k, v, rp, ci, causal=True, rope_base=base)
    for r in range(nb):
        sl = slice(BLK * r, min(S, BLK * r + BLK))
        qb, kb, vb = (np.ascontiguousarray(a[:, sl]) for a in (q, k, v))
        n = qb.shape[1]
        bb, hh, ii = np.meshgrid(np.arange(B), np.arange(Hq), np.arange(n), indexing="ij")
        ob, lb = oracle.attn_rows(qb, kb, vb, bb.ravel(), hh.ravel(), ii.ravel(), causal=True, rope_base=base,
                                  pos_offset=BLK * r)
        np.testing.assert_allclose(o[:, sl].transpose(0, 2, 1, 3).reshape(-1, D), ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, :, sl].reshape(-1), lb, rtol=0, atol=1e-12)


def test_row_without_blocks_is_zero_with_minus_infinite_lse():
    q, k, v = si.make_qkv(1, 2, 2, 256, 32, seed=24)
    rp = np.array([0, 1, 1], dtype=np.int32)  # block row 1 lists nothing
    ci = np.array([0], dtype=np.int32)
    o, lse = oracle.attn_full_bs(q, k, v, rp, ci, causal=False)
    assert np.all(o[:, 128:] == 0.0) and np.all(np.isneginf(lse[:, :, 128:]))
    assert np.all(np.isfinite(lse[:, :, :128]))


def test_oracle_rejects_out_of_range_blocks():
    q, k, v = si.make_qkv(1, 2, 2, 256, 32, seed=25)
    with pytest.raises(ValueError):
        oracle.attn_full_bs(q, k, v, np.array([0, 1, 2], np.int32), np.array([0, 2], np.int32))
