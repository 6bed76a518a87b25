"""The device status word through the C ABI: bounded waits that run out, and non-finite rows.

Failure detection without a fault: attn_selftest_wait_timeout launches the
forward with a producer that issues no load, so every in-kernel wait runs out
after a short limit; the CTAs leave with nothing in flight and attn_check
reports ATTN_ERR_TIMEOUT.  The same process then runs a normal forward that
must match the float64 oracle.  The fp16 range guard is driven by plain input
data past the documented bound.
"""
import ctypes

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


def _status(stream=None):
    return attn.load_library().attn_check(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base", [
    (1, 2, 2, 256, 128, True, 10000.0),
    (4, 8, 2, 2048, 128, True, 500000.0),  # more work units than SMs: every CTA runs out
    (2, 4, 4, 300, 64, False, None),
])
def test_wait_timeout_is_reported_then_a_normal_forward_matches(B, Hq, Hkv, S, D, causal, base):
    lib = attn.load_library()
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=404 + S)
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.attn_selftest_wait_timeout(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        B, Hq, Hkv, S, D, int(causal), float(base or 0.0), 1_000_000, stream)
    assert rc == 0
    assert _status() == attn.ATTN_STATUS["ATTN_ERR_TIMEOUT"]
    assert _status() == 0  # read and cleared
    assert torch.isnan(o).all() and torch.isnan(lse).all()  # nothing was written
    # the context is intact: a normal forward in the same process matches the oracle
    o2, lse2 = attn.attn_fwd(qd, kd, vd, causal=causal, rope_base=base)
    attn.attn_check()
    o_ref, lse_ref = oracle.attn_full(q, k, v, causal=causal, rope_base=base)
    err = np.abs(o2.float().cpu().numpy().astype(np.float64) - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN
    lerr = np.abs(lse2.cpu().numpy().astype(np.float64) - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    assert lerr.max() <= LSE_REL


def test_selftest_rejects_wait_limits_out_of_range():
    lib = attn.load_library()
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    for limit in (0, 99_999, 2_000_000_001):
        assert lib.attn_selftest_wait_timeout(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), None,
                                              1, 1, 1, 1, 64, 1, 0.0, limit, None) == \
            attn.ATTN_STATUS["ATTN_ERR_UNSUPPORTED"]


def _pair_inputs(value):
    """RoPE inputs with one pair (channels 0 and D/2) of query row 5 set to `value`: at angle
    5 rad the rotated first member is value * (cos 5 - sin 5) = 1.2426 * value."""
    B, Hq, Hkv, S, D = 1, 2, 2, 256, 128
    q, k, v = si.make_qkv(B, Hq, Hkv, S, D, seed=505)
    big = np.array([value], dtype=np.float32).view(np.uint32) >> 16  # bf16 bits (both values are exact in bf16)
    q = q.copy()
    q[0, 5, 0, 0] = big[0]
    q[0, 5, 0, D // 2] = big[0]
    return q, k, v


def test_rotated_operand_past_fp16_range_is_reported():
    q, k, v = _pair_inputs(59904.0)  # 1.2426 * 59904 > 65504: the rotated value overflows fp16
    o, lse = attn.attn_fwd(_dev(q), _dev(k), _dev(v), causal=True, rope_base=10000.0)
    with pytest.raises(attn.AttnError) as e:
        attn.attn_check()
    assert e.value.code == attn.ATTN_STATUS["ATTN_ERR_NONFINITE"]
    assert not np.isfinite(lse[0, 0, 5].item())
    assert _status() == 0  # cleared
    # inside the bound every rotated value stays finite (a rotation keeps the pair's norm)
    q, k, v = _pair_inputs(45056.0)
    o, lse = attn.attn_fwd(_dev(q), _dev(k), _dev(v), causal=True, rope_base=10000.0)
    attn.attn_check()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
