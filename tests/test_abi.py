"""The C ABI without a GPU: symbols, host-side argument checks, host tables."""
import ctypes
import math
import subprocess

import numpy as np
import pytest

import attention_causal_attn_gb300 as attn
import oracle


@pytest.fixture(scope="module")
def lib():
    attn.build()
    return attn.load_library()


def test_exports_every_declared_symbol(lib):
    names = attn.header_functions()
    assert set(names) == {"attn_fwd", "attn_fwd_noalloc", "attn_fwd_host", "attn_rope_rotate", "attn_fwd_rotated",
                          "attn_decode", "attn_bwd", "attn_fwd_blocksparse", "attn_bwd_blocksparse", "attn_fwd_local", "attn_bwd_local", "attn_mask_schedule", "attn_fwd_schedule", "attn_selftest_wait_timeout",
                          "attn_build_tables", "attn_check", "attn_error_string", "attn_release_cache"}
    out = subprocess.run(["nm", "-D", "--defined-only", attn._build.LIB], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_error_strings(lib):
    for name, code in attn.ATTN_STATUS.items():
        assert attn.attn_error_string(code).startswith(name)
    assert "unknown" in attn.attn_error_string(12345)


def _call(lib, q=16, k=16, v=16, o=16, lse=0, B=1, Hq=2, Hkv=2, S=128, D=64, causal=1, base=10000.0, win=0.0):
    return lib.attn_fwd(q, k, v, o, lse or None, B, Hq, Hkv, S, D, causal, base, win, None)


def test_argument_errors_are_caught_on_the_host(lib):
    E = attn.ATTN_STATUS
    assert _call(lib, q=0) == E["ATTN_ERR_NULL"]
    assert _call(lib, o=0) == E["ATTN_ERR_NULL"]
    assert _call(lib, B=0) == E["ATTN_ERR_SHAPE"]
    assert _call(lib, S=0) == E["ATTN_ERR_SHAPE"]
    assert _call(lib, D=96) == E["ATTN_ERR_SHAPE"]
    assert _call(lib, Hq=6, Hkv=4) == E["ATTN_ERR_SHAPE"]
    assert _call(lib, Hq=2, Hkv=4) == E["ATTN_ERR_SHAPE"]
    assert _call(lib, Hq=256, Hkv=1) == E["ATTN_ERR_SHAPE"]
    assert _call(lib, B=65536) == E["ATTN_ERR_SHAPE"]  # the batch index is 16 bits of a work unit
    assert _call(lib, S=(1 << 22) + 1) == E["ATTN_ERR_SHAPE"]
    assert _call(lib, q=24) == E["ATTN_ERR_ALIGN"]
    assert _call(lib, lse=18) == E["ATTN_ERR_ALIGN"]
    assert _call(lib, causal=2) == E["ATTN_ERR_UNSUPPORTED"]
    assert _call(lib, base=0.0, win=1.0) == E["ATTN_ERR_UNSUPPORTED"]  # window needs RoPE
    assert _call(lib, causal=0, win=1.0) == E["ATTN_ERR_UNSUPPORTED"]  # window needs causal
    assert _call(lib, base=math.inf) == E["ATTN_ERR_UNSUPPORTED"]


def test_host_entry_checks_arguments_before_any_device_call(lib):
    E = attn.ATTN_STATUS
    call = lambda **kw: lib.attn_fwd_host(*(kw.get(n, 16) for n in ("q", "k", "v", "o")), None,
                                           kw.get("B", 1), kw.get("Hq", 2), kw.get("Hkv", 2), kw.get("S", 128),
                                           kw.get("D", 64), kw.get("causal", 1), kw.get("base", 1e4), kw.get("win", 0.0))
    assert call(q=0) == E["ATTN_ERR_NULL"]
    assert call(B=0) == E["ATTN_ERR_SHAPE"]
    assert call(Hq=6, Hkv=4) == E["ATTN_ERR_SHAPE"]
    assert call(D=80) == E["ATTN_ERR_SHAPE"]
    assert call(causal=3) == E["ATTN_ERR_UNSUPPORTED"]
    assert call(causal=0, win=2.0) == E["ATTN_ERR_UNSUPPORTED"]


def test_rotation_entries_check_arguments_on_the_host(lib):
    E = attn.ATTN_STATUS
    assert lib.attn_rope_rotate(None, 16, 1, 128, 2, 128, 1e4, None) == E["ATTN_ERR_NULL"]
    assert lib.attn_rope_rotate(16, 16, 1, 128, 2, 96, 1e4, None) == E["ATTN_ERR_SHAPE"]
    assert lib.attn_rope_rotate(16, 16, 1, 128, 2, 128, 0.0, None) == E["ATTN_ERR_UNSUPPORTED"]
    assert lib.attn_rope_rotate(24, 16, 1, 128, 2, 128, 1e4, None) == E["ATTN_ERR_ALIGN"]
    assert lib.attn_fwd_rotated(16, 16, 16, 16, None, 1, 6, 4, 128, 128, 1, None) == E["ATTN_ERR_SHAPE"]
    assert lib.attn_fwd_rotated(16, 16, 16, 16, None, 1, 2, 2, 128, 128, 2, None) == E["ATTN_ERR_UNSUPPORTED"]


def test_decode_checks_arguments_on_the_host(lib):
    E = attn.ATTN_STATUS
    call = lambda **kw: lib.attn_decode(*(kw.get(n, 16) for n in ("q", "k", "v", "o")), None, kw.get("B", 1),
                                         kw.get("Hq", 2), kw.get("Hkv", 2), kw.get("S", 128), kw.get("D", 128),
                                         kw.get("base", 1e4), kw.get("win", 0.0), None)
    assert call(q=0) == E["ATTN_ERR_NULL"]
    assert call(S=0) == E["ATTN_ERR_SHAPE"]
    assert call(Hq=66, Hkv=2) == E["ATTN_ERR_UNSUPPORTED"]  # more than 32 query heads per KV head
    assert call(base=0.0, win=1.0) == E["ATTN_ERR_UNSUPPORTED"]  # window needs RoPE
    assert call(k=24) == E["ATTN_ERR_ALIGN"]


def test_backward_checks_arguments_on_the_host(lib):
    E = attn.ATTN_STATUS
    call = lambda **kw: lib.attn_bwd(*(kw.get(n, 16) for n in ("q", "k", "v", "o", "dO", "lse", "dq", "dk", "dv")),
                                      kw.get("B", 1), kw.get("Hq", 2), kw.get("Hkv", 2), kw.get("S", 128),
                                      kw.get("D", 128), kw.get("causal", 1), kw.get("base", 1e4), None)
    assert call(dO=0) == E["ATTN_ERR_NULL"]
    assert call(lse=0) == E["ATTN_ERR_NULL"]
    assert call(dv=0) == E["ATTN_ERR_NULL"]
    assert call(D=96) == E["ATTN_ERR_SHAPE"]
    assert call(Hq=6, Hkv=4) == E["ATTN_ERR_SHAPE"]
    assert call(causal=2) == E["ATTN_ERR_UNSUPPORTED"]
    assert call(dq=24) == E["ATTN_ERR_ALIGN"]
    assert call(lse=18) == E["ATTN_ERR_ALIGN"]


def test_blocksparse_mask_is_checked_on_the_host(lib):
    E = attn.ATTN_STATUS
    import numpy as np

    def call(rp, ci, causal=0, S=256):
        rp = np.asarray(rp, np.int32)
        ci = np.asarray(ci, np.int32)
        return lib.attn_fwd_blocksparse(16, 16, 16, 16, None, 1, 2, 2, S, 128, causal, 1e4, rp.ctypes.data,
                                        ci.ctypes.data if ci.size else None, None)
    assert call([1, 1, 2], [0, 1]) == E["ATTN_ERR_SHAPE"]         # row_ptr[0] != 0
    assert call([0, 2, 1], [0, 1]) == E["ATTN_ERR_SHAPE"]         # decreasing
    assert call([0, 1, 2], [0, 2]) == E["ATTN_ERR_SHAPE"]         # column out of range
    assert call([0, 2, 2], [1, 0]) == E["ATTN_ERR_SHAPE"]         # not ascending
    assert call([0, 2, 2], [0, 0]) == E["ATTN_ERR_SHAPE"]         # repeated
    assert call([0, 2, 2], [0, 1], causal=1) == E["ATTN_ERR_SHAPE"]  # above the diagonal
    assert lib.attn_fwd_blocksparse(16, 16, 16, 16, None, 1, 2, 2, 256, 128, 0, 1e4, None, None,
                                    None) == E["ATTN_ERR_NULL"]
    bad = np.asarray([0, 2, 1], np.int32)
    ci = np.asarray([0, 1], np.int32)
    assert lib.attn_bwd_blocksparse(*([16] * 9), 1, 2, 2, 256, 128, 0, 1e4, bad.ctypes.data, ci.ctypes.data,
                                    None) == E["ATTN_ERR_SHAPE"]
    assert lib.attn_bwd_blocksparse(*([16] * 9), 1, 2, 2, 256, 128, 0, 1e4, None, None, None) == E["ATTN_ERR_NULL"]


def test_local_entry_checks_arguments_on_the_host(lib):
    E = attn.ATTN_STATUS
    call = lambda **kw: lib.attn_fwd_local(16, 16, 16, 16, None, 1, 2, 2, kw.get("S", 256), kw.get("D", 128),
                                            kw.get("causal", 1), 1e4, kw.get("window", 64), kw.get("alibi", 0), None)
    assert call(window=-1) == E["ATTN_ERR_UNSUPPORTED"]
    assert call(alibi=2) == E["ATTN_ERR_UNSUPPORTED"]
    assert call(D=80) == E["ATTN_ERR_SHAPE"]
    assert call(S=0) == E["ATTN_ERR_SHAPE"]
    bwd = lambda **kw: lib.attn_bwd_local(*([16] * 9), 1, 2, 2, kw.get("S", 256), kw.get("D", 128),
                                          kw.get("causal", 1), 1e4, kw.get("window", 64), kw.get("alibi", 0), None)
    assert bwd(window=-1) == E["ATTN_ERR_UNSUPPORTED"]
    assert bwd(alibi=2) == E["ATTN_ERR_UNSUPPORTED"]
    assert bwd(D=80) == E["ATTN_ERR_SHAPE"]
    assert bwd(S=0) == E["ATTN_ERR_SHAPE"]


def test_create_block_mask_lists_the_predicate():
    rp, ci = attn.create_block_mask(lambda qb, kb: kb <= qb and (qb - kb) % 2 == 0, 640)
    assert rp.tolist() == [0, 1, 2, 4, 6, 9]
    assert ci.tolist() == [0, 1, 0, 2, 1, 3, 0, 2, 4]


def test_rope_tables_are_float64_cos_sin_rounded(lib):
    S, D, base = 300, 128, 10000.0
    c, s, _ = attn.attn_build_tables(S, D, base, None, pos_offset=7)
    theta = [base ** (-2.0 * r / D) for r in range(D // 2)]
    for p in (0, 1, 17, 299):
        for r in range(D // 2):
            a = (p + 7) * theta[r]
            assert c[p, r] == np.float32(math.cos(a)) and s[p, r] == np.float32(math.sin(a))


@pytest.mark.parametrize("base,k", [(10000.0, 1.0), (500000.0, 4.0), (500000.0, 1.0)])
def test_window_widths_match_oracle_and_closed_form(lib, base, k):
    _, _, w = attn.attn_build_tables(16, 128, base, k)
    np.testing.assert_array_equal(w.astype(np.float64), oracle.window_widths(128, base, k))
    # the library's widths give the page's closed-form pruned count
    S = 2048
    closed = sum(max(0, S - 1 - int(x)) * (max(0, S - 1 - int(x)) + 1) // 2 for x in w)
    assert closed == oracle.pruned_terms(S, 128, base, k)


def test_window_off_widths_are_int_max(lib):
    _, _, w = attn.attn_build_tables(16, 64, 10000.0, None)
    assert np.all(w == np.iinfo(np.int32).max)
    _, _, w = attn.attn_build_tables(16, 64, 10000.0, math.inf)
    assert np.all(w == np.iinfo(np.int32).max)


def test_build_tables_rejects_bad_arguments(lib):
    with pytest.raises(attn.AttnError):
        attn.attn_build_tables(16, 128, 0.0)
    with pytest.raises(attn.AttnError):
        attn.attn_build_tables(16, 80, 10000.0)


def test_tmem_io_matches_its_generator(tmp_path):
    """tmem_io.inc (the tcgen05.ld / ld.red / st wrappers with long operand lists) is what
    gen_tmem_io.py writes: an edit of either alone fails here."""
    import sys
    from pathlib import Path
    csrc = Path(__file__).resolve().parents[1] / "attention_causal_attn_gb300" / "csrc"
    out = tmp_path / "tmem_io.inc"
    subprocess.run([sys.executable, str(csrc / "gen_tmem_io.py"), str(out)], check=True)
    assert out.read_text() == (csrc / "tmem_io.inc").read_text()
