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


def test_noalloc_waits_for_an_upload_enqueued_on_another_stream():
    """A call whose tables were uploaded on stream A, repeated with the same shape on stream B
    before A has run, must wait for the upload rather than read the array's previous contents.

    Stream A is held back by a sleep kernel, so B would otherwise launch first.  The previous
    contents come from a smaller RoPE shape whose upload covers only the start of the array
    (below the larger shape's schedule), so a launch that did not wait would read wrong RoPE
    factors but nothing outside its tensors."""
    lib = attn.load_library()
    big = (2, 4, 2, 700, 128)     # its RoPE table ends below its schedule's offset in the array
    small = (1, 2, 2, 128, 128)   # its whole upload lies below the larger shape's schedule
    base = 10000.0

    def inputs(shape, seed):
        B, Hq, Hkv, S, D = shape
        return [_dev(x) for x in si.make_qkv(B, Hq, Hkv, S, D, seed=seed)]

    qb, kb, vb = inputs(big, 91)
    qs, ks, vs = inputs(small, 92)
    o_ref, lse_ref = attn.attn_fwd(qb, kb, vb, causal=True, rope_base=base)
    attn.attn_check()
    o_ref, lse_ref = o_ref.float().cpu().numpy(), lse_ref.cpu().numpy()

    def outputs(q):
        B, S, Hq, D = q.shape
        return (torch.full_like(q, float("nan")),
                torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device=q.device))

    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    o1, l1 = outputs(qb)
    assert _noalloc(lib, qb, kb, vb, o1, l1, True, base, sa) == 0   # the larger shape's tables
    o2, l2 = outputs(qs)
    assert _noalloc(lib, qs, ks, vs, o2, l2, True, base, sa) == 0   # overwritten at the start
    torch.cuda.synchronize()
    o3, l3 = outputs(qb)
    with torch.cuda.stream(sa):
        torch.cuda._sleep(200_000_000)  # holds stream A back by tens of milliseconds
    assert _noalloc(lib, qb, kb, vb, o3, l3, True, base, sa) == 0   # re-upload, enqueued behind the sleep
    assert _noalloc(lib, qb, kb, vb, o3, l3, True, base, sb) == 0   # same shape on stream B: must wait
    torch.cuda.synchronize()
    attn.attn_check()
    err = np.abs(o3.float().cpu().numpy() - o_ref)
    assert np.isfinite(err).all()
    assert err.max() <= O_MAX and err.mean() <= O_MEAN
    lerr = np.abs(l3.cpu().numpy() - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    assert lerr.max() <= LSE_REL


def test_noalloc_rejects_requests_beyond_its_scratch():
    lib = attn.load_library()
    q = torch.empty(16, dtype=torch.bfloat16, device="cuda")  # never read: the size check comes first
    # 64 x 128 heads x 2^22 rows is 134M work units, 1 GiB of schedule > 16 MiB
    rc = lib.attn_fwd_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), None,
                              64, 128, 128, 1 << 22, 128, 1, 10000.0, 0.0, None)
    assert rc == attn.ATTN_STATUS["ATTN_ERR_SCRATCH"]
    assert "static scratch" in attn.attn_error_string(rc)
