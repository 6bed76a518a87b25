"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds no attention arithmetic.  It only draws numbers: a
counter-based generator (splitmix64, Steele/Lea/Flood 2014) gives every
element its own pair of 64-bit words, Box-Muller turns the pair into one
standard normal in float64, and the value is rounded to bfloat16 with
round-to-nearest-even.  Because each element depends only on
(seed, tensor id, element index), any slice of a tensor can be regenerated
without generating the rest, and the host-side bits handed to the CUDA path
and to the CPU oracle are identical.

Workload recipes follow the configurations of the fused RoPE + causal
attention prefill benchmark: iid N(0, 1) Q/K/V in BSHD layout, optionally
with 1% "outlier" (head, dim) channels of Q and K scaled by 8.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

MASTER_SEED = 42

# tensor ids: each tensor of a workload draws from its own counter stream
TENSOR_Q, TENSOR_K, TENSOR_V = 1, 2, 3
TENSOR_BLOCK_MASK = 20  # stream id of the random blocks of a block mask
_OUTLIER_STREAM = 1000

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function (the finaliser applied to a counter)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, tensor_id: int) -> np.uint64:
    start = (int(seed) * 0x9E3779B97F4A7C15 + int(tensor_id)) & 0xFFFFFFFFFFFFFFFF
    one = np.array([start], dtype=np.uint64)
    return _mix(_mix(one))[0]


def uniform_words(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """64-bit words number start..start+count-1 of the (seed, tensor_id) stream."""
    key = _stream_key(seed, tensor_id)
    with np.errstate(over="ignore"):
        idx = np.arange(start, start + count, dtype=np.uint64)
        return _mix(key + (idx + np.uint64(1)) * _GOLDEN)


def _normals_chunk(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    w = uniform_words(seed, tensor_id, 2 * start, 2 * count)
    a = w[0::2]
    b = w[1::2]
    inv53 = 1.0 / 9007199254740992.0  # 2**-53
    u1 = ((a >> np.uint64(11)).astype(np.float64) + 1.0) * inv53  # (0, 1]
    u2 = (b >> np.uint64(11)).astype(np.float64) * inv53  # [0, 1)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def normals_f64(seed: int, tensor_id: int, start: int, count: int, threads: int | None = None) -> np.ndarray:
    """Standard normals (float64) for elements start..start+count-1 of a stream."""
    out = np.empty(count, dtype=np.float64)
    chunks = [(s, min(_CHUNK, count - s)) for s in range(0, count, _CHUNK)]
    if threads is None:
        threads = min(16, os.cpu_count() or 1)

    def work(c):
        s, n = c
        out[s:s + n] = _normals_chunk(seed, tensor_id, start + s, n)

    if len(chunks) <= 1 or threads <= 1:
        for c in chunks:
            work(c)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, chunks))
    return out


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 to bfloat16 bits (uint16): float64 -> float32 (RNE) -> bf16 (RNE).

    The inputs drawn here are finite and far from the float32 range limits,
    so the two roundings never meet a NaN or an overflow.
    """
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (f >> np.uint32(16)) & np.uint32(1)
    r = (f + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def outlier_channels(seed: int, tensor_id: int, heads: int, dim: int, fraction: float = 0.01) -> np.ndarray:
    """Seeded choice of round(fraction*heads*dim) distinct (head, dim) channels, as flat indices h*dim+d."""
    n = heads * dim
    count = int(round(fraction * n))
    keys = uniform_words(seed, _OUTLIER_STREAM + tensor_id, 0, n)
    return np.sort(np.argsort(keys, kind="stable")[:count])


def bshd_bf16(seed: int, tensor_id: int, B: int, S: int, H: int, D: int,
              outlier_fraction: float = 0.0, outlier_scale: float = 8.0,
              threads: int | None = None) -> np.ndarray:
    """A [B, S, H, D] tensor of bf16 bits (uint16), iid N(0,1), optional outlier channels.

    Outlier channels are (head, dim) pairs scaled at every (batch, position)
    before the rounding to bf16.
    """
    count = B * S * H * D
    x = normals_f64(seed, tensor_id, 0, count, threads).reshape(B, S, H, D)
    if outlier_fraction > 0.0:
        ch = outlier_channels(seed, tensor_id, H, D, outlier_fraction)
        flat = x.reshape(B, S, H * D)
        flat[:, :, ch] *= outlier_scale
    return f64_to_bf16_bits(x.reshape(-1)).reshape(B, S, H, D)


# ---------------------------------------------------------------------------
# Workload recipes (shapes of the attention prefill benchmark configurations).
# ---------------------------------------------------------------------------

WORKLOADS = {
    # name: dict of shape + attention options
    "tiny_rope_causal": dict(B=1, Hq=2, Hkv=2, S=128, D=64, causal=True, rope_base=10000.0,
                             window_k=None, outliers=0.0),
    "plain_causal_s4096": dict(B=4, Hq=32, Hkv=32, S=4096, D=128, causal=True, rope_base=None,
                               window_k=None, outliers=0.0),
    "rope_causal_s8192": dict(B=4, Hq=32, Hkv=32, S=8192, D=128, causal=True, rope_base=10000.0,
                              window_k=None, outliers=0.0),
    "gqa_llama3_s16384": dict(B=1, Hq=32, Hkv=8, S=16384, D=128, causal=True, rope_base=500000.0,
                              window_k=None, outliers=0.01),
    "window_s131072": dict(B=1, Hq=32, Hkv=8, S=131072, D=128, causal=True, rope_base=500000.0,
                           window_k=1.0, outliers=0.0),
    # block-sparse forward ("AttnFuse", sec. 4.3: BigBird at N = 4096): a BigBird-style mask over
    # 128 x 128 blocks, the diagonal, one global block row/column and one seeded random block per row
    "bigbird_s4096": dict(B=4, Hq=32, Hkv=32, S=4096, D=128, causal=False, rope_base=None,
                          window_k=None, outliers=0.0, block_mask=dict(window=0, n_global=1, n_random=1)),
    # sliding window and ALiBi ("AttnFuse", sec. 6.1: GPT-2-small geometry B=4, H=12, D=64)
    "sliding_window_s4096": dict(B=4, Hq=12, Hkv=12, S=4096, D=64, causal=True, rope_base=None,
                                 window_k=None, outliers=0.0, local=dict(window=512, alibi=False)),
    "alibi_s4096": dict(B=4, Hq=12, Hkv=12, S=4096, D=64, causal=True, rope_base=None,
                        window_k=None, outliers=0.0, local=dict(window=0, alibi=True)),
}


def make_qkv(B: int, Hq: int, Hkv: int, S: int, D: int, outliers: float = 0.0,
             seed: int = MASTER_SEED, threads: int | None = None):
    """Q [B,S,Hq,D], K and V [B,S,Hkv,D] as bf16 bits (uint16 numpy arrays)."""
    q = bshd_bf16(seed, TENSOR_Q, B, S, Hq, D, outliers, threads=threads)
    k = bshd_bf16(seed, TENSOR_K, B, S, Hkv, D, outliers, threads=threads)
    v = bshd_bf16(seed, TENSOR_V, B, S, Hkv, D, 0.0, threads=threads)
    return q, k, v


def sample_rows(seed: int, S: int, n: int = 256, block: int = 128) -> np.ndarray:
    """Seeded sorted set of query rows: always 0, 1, block-1, block, S-1 and tile edges, then random rows."""
    fixed = {0, 1, block - 1, block, S - 1, S // 2}
    for t in range(block, S, block * max(1, (S // block) // 8)):
        fixed.add(t - 1)
        fixed.add(t)
    fixed = {r for r in fixed if 0 <= r < S}
    rows = set(fixed)
    if n > len(rows):
        w = uniform_words(seed, 7777, 0, 4 * n)
        for x in (w % np.uint64(S)).astype(np.int64):
            if len(rows) >= min(n, S):
                break
            rows.add(int(x))
    return np.array(sorted(rows), dtype=np.int32)


def sample_heads(seed: int, B: int, Hq: int, Hkv: int, n: int = 8):
    """Seeded (b, h) pairs: (0,0) and (B-1,Hq-1) always, covering every KV group when n allows."""
    G = Hq // Hkv
    pairs = [(0, 0)]
    if (B - 1, Hq - 1) != (0, 0):
        pairs.append((B - 1, Hq - 1))
    covered = {h // G for _, h in pairs}
    w = uniform_words(seed, 8888, 0, 64 * n + 64)
    i = 0
    for g in range(Hkv):
        if len(pairs) >= n:
            break
        if g in covered:
            continue
        h = g * G + int(w[i] % np.uint64(G))
        b = int(w[i + 1] % np.uint64(B))
        i += 2
        pairs.append((b, h))
        covered.add(g)
    while len(pairs) < min(n, B * Hq) and i + 1 < len(w):
        b = int(w[i] % np.uint64(B))
        h = int(w[i + 1] % np.uint64(Hq))
        i += 2
        if (b, h) not in pairs:
            pairs.append((b, h))
    return pairs[:n]


def bigbird_block_mask(S: int, block: int = 128, window: int = 1, n_global: int = 1, n_random: int = 1,
                       seed: int = MASTER_SEED, causal: bool = False):
    """A BigBird-style block mask as CSR (row_ptr, col_idx) over ceil(S/block) blocks per side.

    Row r lists: the blocks within `window` of the diagonal, the first `n_global` blocks (global
    columns), `n_random` further blocks drawn from the splitmix64 stream of (seed, block-mask
    id) at counters 256 r ..; the first
    `n_global` rows list every block (global rows).  With causal=True blocks above the diagonal
    are dropped.  Columns are sorted and unique.  Structure only: no attention arithmetic.
    """
    nb = (S + block - 1) // block
    rows = []
    for r in range(nb):
        cols = set(range(max(0, r - window), min(nb, r + window + 1)))
        cols.update(range(min(n_global, nb)))
        if r < n_global:
            cols.update(range(nb))
        words = uniform_words(seed, TENSOR_BLOCK_MASK, r * 256, 256)
        drawn = 0
        for word in words:
            if drawn >= n_random or len(cols) >= nb:
                break
            c = int(word % np.uint64(nb))
            if c not in cols:
                cols.add(c)
                drawn += 1
        if causal:
            cols = {c for c in cols if c <= r}
        rows.append(sorted(cols))
    row_ptr = np.zeros(nb + 1, dtype=np.int32)
    row_ptr[1:] = np.cumsum([len(c) for c in rows])
    col_idx = np.array([c for cs in rows for c in cs], dtype=np.int32)
    return row_ptr, col_idx
