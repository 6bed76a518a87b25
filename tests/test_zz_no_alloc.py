"""attn_fwd_noalloc, the entry point for callers that must not allocate device memory.

Some callers cannot call cudaMalloc (a fixed device-memory budget, an allocator
that owns every byte, a hot loop that must not touch the allocator).  For them
attn_fwd_noalloc keeps its RoPE table and tile schedule in a static 16 MiB
device array inside the library.  This test calls it through the C ABI twice
in a row and checks each result against attn_fwd, the entry point that keeps
its tables in cached cudaMalloc'd buffers.  It lives in its own file, named to
be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import attention_causal_attn_gb300 as attn
import seeded_inputs as si

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_REL = 2e-2, 2e-3, 1e-3


def _dev(a):
    return torch.from_numpy(a).view(torch.bfloat16).cuda()


def _noalloc(lib, q, k, v, o, lse, causal, base, stream):
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    return lib.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                B, Hq, Hkv, S, D, int(causal), float(base or 0.0), 0.0,
                                ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,base", [
    (2, 4, 2, 700, 128, True, 10000.0),
    (1, 4, 4, 300, 64, False, None),
])
def test_noalloc_matches_attn_fwd_on_two_calls(B, Hq, Hkv, S, D, causal, base):
    attn.build()
    lib = attn.load_library()
    q, k, v = (_dev(x) for x in si.make_qkv(B, Hq, Hkv, S, D, seed=77))
    stream = torch.cuda.current_stream()
    o_ref, lse_ref = attn.attn_fwd(q, k, v, causal=causal, rope_base=base)
    attn.attn_check()
    o_ref = o_ref.float().cpu().numpy()
    lse_ref = lse_ref.cpu().numpy()
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device=q.device)
        assert _noalloc(lib, q, k, v, o, lse, causal, base, stream) == 0
        attn.attn_check()
        err = np.abs(o.float().cpu().numpy() - o_ref)
        assert np.isfinite(err).all()
        assert err.max() <= O_MAX and err.mean() <= O_MEAN
        lerr = np.abs(lse.cpu().numpy() - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
        assert lerr.max() <= LSE_REL


def test_noalloc_rejects_requests_beyond_its_scratch():
    lib = attn.load_library()
    q = torch.empty(16, dtype=torch.bfloat16, device="cuda")  # never read: the size check comes first
    # 64 x 128 heads x 2^22 rows is 134M work units, 1 GiB of schedule > 16 MiB
    rc = lib.attn_fwd_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), None,
                              64, 128, 128, 1 << 22, 128, 1, 10000.0, 0.0, None)
    assert rc == attn.ATTN_STATUS["ATTN_ERR_SCRATCH"]
    assert "static scratch" in attn.attn_error_string(rc)
