// Block-sparse attention forward ("AttnFuse", sec. 4.3 Block-Sparse Attention:
// a CSR BlockMask lists the active key blocks of each row of blocks, and the
// kernel visits only those, so its work is proportional to the active share).
//
// Blocks are the kernel's 128 x 128 tiles.  CTA i * (B * Hq) + b * Hq + h
// computes query tile i of head h (tile by tile across heads, so a mask's
// heavy rows start first): Q is loaded and rotated once, then the listed key tiles
// are streamed (two slots) in descending order, each through
//   S = Q K^T (tcgen05, TMEM)  ->  online softmax, P in bf16 over S  ->  O += P V.
// Roles as in the backward kernels: two softmax warpgroups (one thread per
// query row and half of the 128 key columns), four RoPE warps, a TMA warp and
// an MMA warp.  Each half keeps its own running maximum and sum (log2 units)
// and its own O accumulator in TMEM, fed by its half of P; the halves merge
// by their maxima once, in the epilogue.  A row of blocks with nothing listed
// writes O = 0 and LSE = -inf.  Every wait is bounded.
//
// The EXT variant adds the sliding_window and alibi combinators ("AttnFuse",
// sec. 3): key j is visible to query i only when |i - j| < window, and the
// score gains -m_h |i - j| with m_h = 2^(-8 (h+1) / Hq); its softmax keeps
// the running maximum in log2 units of the biased score.
#pragma once

#include "bwd_kernel.cuh"

namespace attn {

struct BsParams {
    FwdParams f;           // tm_q, tm_k, tm_v, o, lse, RoPE factor table, shape, scale, status, wait limit
    const int* row_ptr;    // [ceil(S/128) + 1]
    const int* col_idx;    // listed key tiles of each row of tiles, ascending
    int window;            // EXT: visible iff |i - j| < window (0: no window)
    int alibi;             // EXT: ALiBi bias on
};

// EXT: the score of column col of a tile for this row in log2 units (biased), or -inf when the
// key lies outside [lo, hi).  rel0 = first key of the tile - row; m2 = m_h * log2(e).
__device__ __forceinline__ float ext_score(uint32_t raw, int col, int lo, int hi, float c, float m2, int rel0) {
    const float dist = fabsf(static_cast<float>(rel0 + col));
    return (col >= lo && col < hi) ? __uint_as_float(raw) * c - m2 * dist : -INFINITY;
}

constexpr int kBsThreads = 448;  // warps 0-7 softmax (two halves), 8-11 RoPE, 12 TMA, 13 MMA
constexpr int kBsWarpRope = 8, kBsWarpTma = 12, kBsWarpMma = 13;

template <int D>
struct BsLayout {
    static constexpr uint32_t kTile = 128u * D * 2u;
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kStr0 = kTile;  // slot s: K at kStr0 + 2 s kTile, V after it
    static constexpr uint32_t kBars = 5 * kTile;
    static constexpr uint32_t kMisc = kBars + 256;
    static constexpr uint32_t kMerge = kMisc + 64;  // [2 halves][128 rows] float2 (m, l)
    static constexpr uint32_t kBytes = kMerge + 2 * 128 * 8;
    static constexpr uint32_t kAlloc = kBytes + 1024;
};

// Without the EXT terms: the raw-score maximum of one half (columns [c0, c0 + 64), keys at or past
// limit hidden), and P = exp2(S c - m c) packed into the half's first 32 columns with its sum, by
// the prefill's own chunk routines (raw scores, paired fp32 arithmetic).
template <bool MASKED>
__device__ __forceinline__ float half_row_max_raw(uint32_t tS, int c0, int limit) {
    uint32_t a[32], b[32];
    tmem_load_32_async(tS + c0, a);
    tmem_load_32_async(tS + c0 + 32, b);
    tmem_wait_ld_32(a);
    tmem_wait_ld_32(b);
    return row_max32<MASKED>(b, c0 + 32, limit, row_max32<MASKED>(a, c0, limit, -INFINITY));
}

template <bool MASKED>
__device__ __forceinline__ float half_exp_to_p_raw(uint32_t tS, int c0, int limit, float c, float mc) {
    const uint64_t c2 = f2_pack(c, c), nmc2 = f2_pack(-mc, -mc);
    uint64_t sum2 = f2_pack(0.f, 0.f);
#pragma unroll
    for (int cc = 0; cc < 64; cc += 32) {
        uint32_t r[32], pk[16];
        tmem_load_32(tS + c0 + cc, r);
        exp_pack32<MASKED>(r, c0 + cc, limit, c2, nmc2, sum2, pk);
        tmem_store_16(tS + c0 + cc / 2, pk);
    }
    float s0, s1;
    f2_unpack(sum2, s0, s1);
    return s0 + s1;
}

// Row maximum of one half (columns [c0, c0 + 64)) of a tile, of score(raw, column).
template <typename F>
__device__ __forceinline__ float half_row_max(uint32_t tS, int c0, F score) {
    uint32_t a[32], b[32];
    tmem_load_32_async(tS + c0, a);
    tmem_load_32_async(tS + c0 + 32, b);
    tmem_wait_ld_32(a);
    tmem_wait_ld_32(b);
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        m0 = fmaxf(m0, score(a[j], c0 + j));
        m1 = fmaxf(m1, score(b[j], c0 + 32 + j));
    }
    return fmaxf(m0, m1);
}

// P = exp2(score - m) (0 for hidden keys) of one half in bf16, packed into the half's own first 32
// columns (never a column still to be read); returns the half's sum of P.
template <typename F>
__device__ __forceinline__ float half_exp_to_p(uint32_t tS, int c0, F score, float m) {
    float sum = 0.f;
#pragma unroll
    for (int cc = 0; cc < 64; cc += 32) {
        uint32_t r[32];
        tmem_load_32(tS + c0 + cc, r);
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const float v0 = score(r[j], c0 + cc + j), v1 = score(r[j + 1], c0 + cc + j + 1);
            const float p0 = v0 == -INFINITY ? 0.f : ex2_approx(v0 - m);
            const float p1 = v1 == -INFINITY ? 0.f : ex2_approx(v1 - m);
            sum += p0 + p1;
            pk[j / 2] = pack_bf16x2(p0, p1);
        }
        tmem_store_16(tS + c0 + cc / 2, pk);
    }
    return sum;
}

template <int D, bool CAUSAL, bool ROPE, bool EXT = false>
__global__ void __launch_bounds__(kBsThreads, 1) bs_fwd_kernel(const __grid_constant__ BsParams p) {
    using L = BsLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smg = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sm = smem_addr(smg);
    const uint32_t bar0 = sm + L::kBars;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smg + L::kMisc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smg + L::kMisc + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const FwdParams& f = p.f;
    const int bhs = f.B * f.Hq;
    const int i = static_cast<int>(blockIdx.x / bhs);
    const int b = static_cast<int>(blockIdx.x % bhs) / f.Hq, h = static_cast<int>(blockIdx.x % bhs) % f.Hq;
    const int g = h / (f.Hq / f.Hkv);
    const int q0 = i * 128;
    const int e0 = p.row_ptr[i];
    const int nblk = p.row_ptr[i + 1] - e0;  // listed tiles, visited from the last listed down

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        bwd_init_bars(bar0, 256);  // P is handed over by the 256 softmax threads
    }
    if (warp == kBsWarpTma && lane == 0) {
        tma_prefetch_desc(&f.tm_q);
        tma_prefetch_desc(&f.tm_k);
        tma_prefetch_desc(&f.tm_v);
    }
    if (warp == kBsWarpMma) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, f.status, f.wait_limit_ns};

    if (warp < 8) {
        // ---- softmax warpgroups: thread t owns query row q0 + t (TMEM lane t) and key columns
        // [64 x, 64 x + 64) of every tile, x = half; scores, maxima and sums in log2 units
        const int t = threadIdx.x % 128, x = threadIdx.x / 128;
        const int row = q0 + t;
        const uint32_t trow = tmem + (static_cast<uint32_t>(t & ~31) << 16);
        const uint32_t tS = trow, tO = trow + 128u + static_cast<uint32_t>(x * D);  // this half's O
        const float c = f.scale_log2;
        const float m2 = (EXT && p.alibi) ? exp2f(-8.f * static_cast<float>(h + 1) / static_cast<float>(f.Hq)) *
                                                1.4426950408889634f
                                          : 0.f;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int it = 0; it < nblk && ok; ++it) {
            const int kv0 = p.col_idx[e0 + nblk - 1 - it] * 128;
            ok = bwd_wait(bar_at(bar0, BB_S_FULL), it & 1, ctl, kStatusSoftmax);
            if (!ok) break;
            tc_fence_after();
            // keys kv0 + [lo, limit) are visible to this row
            int limit = min(128, f.S - kv0);
            if (CAUSAL) limit = min(limit, row - kv0 + 1);
            int lo = 0;
            if (EXT && p.window > 0) {
                lo = max(0, row - p.window + 1 - kv0);
                if (!CAUSAL) limit = min(limit, row + p.window - kv0);
            }
            const int rel0 = kv0 - row;
            auto score = [&](uint32_t raw, int col) {
                if (EXT) return ext_score(raw, col, lo, limit, c, m2, rel0);
                return col < limit ? __uint_as_float(raw) * c : -INFINITY;
            };
            // EXT: m in log2 units of the biased score; otherwise raw score units (as the prefill)
            const bool masked = __any_sync(0xffffffffu, limit < 128);
            float mx;
            if constexpr (EXT) mx = half_row_max(tS, 64 * x, score);
            else mx = masked ? half_row_max_raw<true>(tS, 64 * x, limit) : half_row_max_raw<false>(tS, 64 * x, limit);
            const float m_new = fmaxf(m_used, mx);
            const float unit = EXT ? 1.f : c;
            if (it == 0) {
                m_used = m_new;
            } else {
                const bool need = (m_new - m_used) * unit > kRescaleThreshold;
                if (__any_sync(0xffffffffu, need)) {
                    float alpha = 1.f;
                    if (need) {
                        alpha = m_used == -INFINITY ? 0.f : ex2_approx((m_used - m_new) * unit);
                        m_used = m_new;
                        l *= alpha;
                    }
                    const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                    for (int cc = 0; cc < D; cc += 32) {
                        uint32_t r[32];
                        tmem_load_32(tO + cc, r);
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            float x0, x1;
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), a2), x0, x1);
                            r[j] = __float_as_uint(x0);
                            r[j + 1] = __float_as_uint(x1);
                        }
                        tmem_store_32(tO + cc, r);
                    }
                }
            }
            if constexpr (EXT) l += half_exp_to_p(tS, 64 * x, score, m_used);
            else {
                // a half that has seen no key yet (m = -inf: every key it held was masked) gets P = 0
                const float mc = m_used == -INFINITY ? 0.f : m_used * c;
                l += masked ? half_exp_to_p_raw<true>(tS, 64 * x, limit, c, mc)
                            : half_exp_to_p_raw<false>(tS, 64 * x, limit, c, mc);
            }
            tmem_store_wait();
            tc_fence_before();
            mbar_arrive(bar_at(bar0, BB_P_FULL));
        }
        // epilogue: merge the halves by their maxima; each half writes D/2 output channels
        const bool have = nblk > 0;
        if (ok && have) ok = bwd_wait(bar_at(bar0, BB_ACC_FULL), 0, ctl, kStatusSoftmax);
        float2* ml = reinterpret_cast<float2*>(smg + L::kMerge);
        ml[x * 128 + t] = make_float2(EXT ? m_used : m_used * c, l);  // log2 units
        mbar_arrive(bar_at(bar0, BB_MERGE));
        if (ok) ok = bwd_wait(bar_at(bar0, BB_MERGE), 0, ctl, kStatusSoftmax);
        if (ok) {
            tc_fence_after();
            const float2 mine = ml[x * 128 + t], other = ml[(1 - x) * 128 + t];
            const float ma = x == 0 ? mine.x : other.x, mb = x == 0 ? other.x : mine.x;
            const float la = x == 0 ? mine.y : other.y, lb = x == 0 ? other.y : mine.y;
            const float M = fmaxf(ma, mb);
            const float sa = ma == -INFINITY ? 0.f : ex2_approx(ma - M), sb = mb == -INFINITY ? 0.f : ex2_approx(mb - M);
            const float Lsum = la * sa + lb * sb;
            const float inv = (have && Lsum > 0.f) ? 1.0f / Lsum : 0.f;
            const bool store = row < f.S;
            __nv_bfloat16* dst = f.o + ((static_cast<size_t>(b) * f.S + (store ? row : 0)) * f.Hq + h) * D;
            const uint32_t tOa = trow + 128u, tOb = trow + 128u + D;
#pragma unroll
            for (int cc = 0; cc < D / 2; cc += 32) {
                const int d0 = x * (D / 2) + cc;  // this half's output channels
                uint32_t ra[32], rb[32];
                if (have) {
                    tmem_load_32_async(tOa + d0, ra);
                    tmem_load_32_async(tOb + d0, rb);
                    tmem_wait_ld_32(ra);
                    tmem_wait_ld_32(rb);
                }
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float o0 = have ? (__uint_as_float(ra[j]) * sa + __uint_as_float(rb[j]) * sb) * inv : 0.f;
                    const float o1 = have ? (__uint_as_float(ra[j + 1]) * sa + __uint_as_float(rb[j + 1]) * sb) * inv : 0.f;
                    pk[j / 2] = pack_bf16x2(o0, o1);
                }
                if (store) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + d0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            if (x == 0 && store && f.lse != nullptr)
                f.lse[(static_cast<size_t>(b) * f.Hq + h) * f.S + row] =
                    (have && Lsum > 0.f) ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
        }
    } else if (warp < kBsWarpTma) {
        // ---- RoPE warps: Q once, then each streamed K tile
        if (ROPE && nblk > 0) {
            const int t = threadIdx.x - kBsWarpRope * 32;
            RopeConsts k;
            rope_load_consts<D>(f, t, k);
            uint64_t cb[4], sb[4];
            rope_load_base<D>(f, i, t, cb, sb);
            bool ok = bwd_wait(bar_at(bar0, BB_RES_FULL), 0, ctl, kStatusRope);
            if (ok) {
                rope_rotate_tile<D, false>(smg + L::kQ, k, cb, sb, t);
                fence_proxy_async_smem();
                mbar_arrive(bar_at(bar0, BB_RES_ROT));
            }
            for (int it = 0; it < nblk && ok; ++it) {
                const int s = it & 1;
                rope_load_base<D>(f, p.col_idx[e0 + nblk - 1 - it], t, cb, sb);
                ok = bwd_wait(bar_at(bar0, BB_STR_FULL + s), (it >> 1) & 1, ctl, kStatusRope);
                if (!ok) break;
                rope_rotate_tile<D, false>(smg + L::kStr0 + s * 2 * L::kTile, k, cb, sb, t);
                fence_proxy_async_smem();
                mbar_arrive(bar_at(bar0, BB_STR_ROT + s));
            }
        }
    } else if (warp == kBsWarpTma) {
        // ---- producer: Q once, then K and V of each listed tile
        if (lane == 0 && nblk > 0) {
            const uint32_t rb = bar_at(bar0, BB_RES_FULL);
            mbar_arrive_expect_tx(rb, L::kTile);
#pragma unroll
            for (int sub = 0; sub < D / 64; ++sub)
                tma_load_4d(sm + L::kQ + sub * kSubTileBytes, &f.tm_q, rb, sub * 64, h, q0, b);
            for (int it = 0; it < nblk; ++it) {
                const int s = it & 1, n = it >> 1;
                const int kv0 = p.col_idx[e0 + nblk - 1 - it] * 128;
                if (n >= 1 && !mbar_wait(bar_at(bar0, BB_STR_EMPTY + s), (n - 1) & 1, ctl, kStatusProducer)) break;
                const uint32_t fb = bar_at(bar0, BB_STR_FULL + s);
                mbar_arrive_expect_tx(fb, 2 * L::kTile);
                const uint32_t ka = sm + L::kStr0 + s * 2 * L::kTile;
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub) {
                    tma_load_4d(ka + sub * kSubTileBytes, &f.tm_k, fb, sub * 64, g, kv0, b);
                    tma_load_4d(ka + L::kTile + sub * kSubTileBytes, &f.tm_v, fb, sub * 64, g, kv0, b);
                }
            }
        }
        __syncwarp();
    } else if (warp == kBsWarpMma && lane == 0 && nblk > 0) {
        // ---- MMA issuer: S = Q K^T (K-major, fp16 after RoPE), then O += P V (P from TMEM, V MN-major)
        const uint32_t kIdescS = umma_idesc_f16(ROPE ? 0u : 1u, 0u, 128, 128);
        constexpr uint32_t kIdescPV = umma_idesc_f16(1u, 1u, 128, D);
        const uint32_t tS = tmem, tO = tmem + 128u;
        const uint64_t qdesc = sw128_desc(sm + L::kQ, 16u, 1024u);
        bool ok = mbar_wait(bar_at(bar0, BB_RES_FULL), 0, ctl, kStatusMma);
        if (ok && ROPE) ok = mbar_wait(bar_at(bar0, BB_RES_ROT), 0, ctl, kStatusMma);
        for (int it = 0; it < nblk && ok; ++it) {
            const int s = it & 1, n = it >> 1;
            ok = mbar_wait(bar_at(bar0, BB_STR_FULL + s), n & 1, ctl, kStatusMma);
            if (ok && ROPE) ok = mbar_wait(bar_at(bar0, BB_STR_ROT + s), n & 1, ctl, kStatusMma);
            if (!ok) break;
            tc_fence_after();
            const uint32_t ka = sm + L::kStr0 + s * 2 * L::kTile, va = ka + L::kTile;
            const uint64_t kdesc = sw128_desc(ka, 16u, 1024u);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_ss(tS, desc_advance(qdesc, kmajor_units(kk)), desc_advance(kdesc, kmajor_units(kk)), kIdescS,
                        kk > 0 ? 1u : 0u);
            tc_commit(bar_at(bar0, BB_S_FULL));
            ok = mbar_wait(bar_at(bar0, BB_P_FULL), it & 1, ctl, kStatusMma);
            if (!ok) break;
            tc_fence_after();
            const uint64_t vdesc = sw128_desc(va, kSubTileBytes, 1024u);
            // each half of P (keys 0-63, 64-127, packed in its half's first 32 columns) into its own O;
            // 16 keys per step: 2048 bytes of V, 8 TMEM columns of P
#pragma unroll
            for (int hx = 0; hx < 2; ++hx)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_ts(tO + static_cast<uint32_t>(hx * D), tS + 64u * hx + kk * 8u,
                            desc_advance(vdesc, (4 * hx + kk) * 128u), kIdescPV, (it > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bar_at(bar0, BB_STR_EMPTY + s));
        }
        if (ok) tc_commit(bar_at(bar0, BB_ACC_FULL));
        bwd_drain(bar0, ctl);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kBsWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace attn
