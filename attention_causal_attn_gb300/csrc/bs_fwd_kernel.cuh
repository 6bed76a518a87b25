// Block-sparse attention forward ("AttnFuse", sec. 4.3 Block-Sparse Attention:
// a CSR BlockMask lists the active key blocks of each row of blocks, and the
// kernel visits only those, so its work is proportional to the active share).
//
// Blocks are the kernel's 128 x 128 tiles.  CTA i * (B * Hq) + b * Hq + h
// computes query tile i of head h (tile by tile across heads, so a mask's
// heavy rows start first).  Q is loaded and rotated once; the listed key tiles
// are visited in descending order and dealt alternately to two softmax
// streams, as the prefill deals two query tiles to its two stages:
//   S_s = Q K^T (tcgen05, TMEM)  ->  online softmax of stream s, P in bf16 over S_s  ->  O_s += P V.
// Each stream keeps its own running maximum, sum and O accumulator; the two
// merge by their maxima once, in the epilogue.  While one stream's softmax
// works, the tensor cores form the other stream's S and accumulate its last
// P V.  K and V tiles sit in separate three-slot rings, so a K slot refills as
// soon as its S is formed.  Roles: two softmax warpgroups (one thread per query
// row), four RoPE warps, a TMA warp and an MMA warp.  A row of blocks with
// nothing listed writes O = 0 and LSE = -inf.  Every wait is bounded.
//
// The EXT variant adds the sliding_window and alibi combinators ("AttnFuse",
// sec. 3): key j is visible to query i only when |i - j| < window, and the
// score gains -m_h |i - j| with m_h = 2^(-8 (h+1) / Hq).
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

constexpr int kBsThreads = 448;  // warps 0-7 softmax (two streams), 8-11 RoPE, 12 TMA, 13 MMA
constexpr int kBsWarpRope = 8, kBsWarpTma = 12, kBsWarpMma = 13;
constexpr int kBsSlots = 3;      // K slots and V slots

template <int D>
struct BsLayout {
    static constexpr uint32_t kTile = 128u * D * 2u;
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK0 = kTile;                   // K slot r at kK0 + r kTile
    static constexpr uint32_t kV0 = kK0 + kBsSlots * kTile;  // V slot r at kV0 + r kTile
    static constexpr uint32_t kBars = kV0 + kBsSlots * kTile;
    static constexpr uint32_t kMisc = kBars + 256;
    static constexpr uint32_t kBytes = kMisc + 64;
    static constexpr uint32_t kAlloc = kBytes + 1024;
    static constexpr uint32_t kMerge = kK0;  // epilogue: [2 streams][128 rows] float2 (m, l) over K slot 0
};

enum : int {
    BS_Q_FULL = 0,
    BS_Q_ROT,
    BS_K_FULL,                          // [3]
    BS_K_ROT = BS_K_FULL + kBsSlots,    // [3]
    BS_K_EMPTY = BS_K_ROT + kBsSlots,   // [3] S of the slot's tile formed
    BS_V_FULL = BS_K_EMPTY + kBsSlots,  // [3]
    BS_V_EMPTY = BS_V_FULL + kBsSlots,  // [3] P V of the slot's tile done
    BS_S_FULL = BS_V_EMPTY + kBsSlots,  // [2] per stream
    BS_P_FULL = BS_S_FULL + 2,          // [2] per stream
    BS_O_FULL = BS_P_FULL + 2,
    BS_DRAIN,
    BS_MERGE,
    BS_NUM
};
static_assert(BS_NUM * 8 <= 256, "barrier block");

__device__ __forceinline__ void bs_init_bars(uint32_t bar0) {
    mbar_init(bar_at(bar0, BS_Q_FULL), 1);
    mbar_init(bar_at(bar0, BS_Q_ROT), 128);
    for (int r = 0; r < kBsSlots; ++r) {
        mbar_init(bar_at(bar0, BS_K_FULL + r), 1);
        mbar_init(bar_at(bar0, BS_K_ROT + r), 128);
        mbar_init(bar_at(bar0, BS_K_EMPTY + r), 1);
        mbar_init(bar_at(bar0, BS_V_FULL + r), 1);
        mbar_init(bar_at(bar0, BS_V_EMPTY + r), 1);
    }
    for (int s = 0; s < 2; ++s) {
        mbar_init(bar_at(bar0, BS_S_FULL + s), 1);
        mbar_init(bar_at(bar0, BS_P_FULL + s), 128);
    }
    mbar_init(bar_at(bar0, BS_O_FULL), 1);
    mbar_init(bar_at(bar0, BS_DRAIN), 1);
    mbar_init(bar_at(bar0, BS_MERGE), 256);
    fence_barrier_init();
    fence_proxy_async_smem();
}

// EXT: the score of column col of a tile for this row in log2 units (biased), or -inf when the
// key lies outside [lo, hi).  rel0 = first key of the tile - row; m2 = m_h * log2(e).
__device__ __forceinline__ float ext_score(uint32_t raw, int col, int lo, int hi, float c, float m2, int rel0) {
    const float dist = fabsf(static_cast<float>(rel0 + col));
    return (col >= lo && col < hi) ? __uint_as_float(raw) * c - m2 * dist : -INFINITY;
}

__device__ __forceinline__ float ext_row_max(uint32_t tS, int lo, int hi, float c, float m2, int rel0) {
    float mx = -INFINITY;
    tmem_stream_128(tS, [&](const uint32_t (&r)[32], int cc) {
#pragma unroll
        for (int j = 0; j < 32; ++j) mx = fmaxf(mx, ext_score(r[j], cc + j, lo, hi, c, m2, rel0));
    });
    return mx;
}

// P = exp2(score - m) in bf16 over the S columns (hidden keys 0; none computed while m = -inf),
// and the row sum of P.
__device__ __forceinline__ float ext_exp_to_p(uint32_t tS, int lo, int hi, float c, float m2, int rel0, float m) {
    float sum = 0.f;
    tmem_stream_128(tS, [&](const uint32_t (&r)[32], int cc) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const float v0 = ext_score(r[j], cc + j, lo, hi, c, m2, rel0);
            const float v1 = ext_score(r[j + 1], cc + j + 1, lo, hi, c, m2, rel0);
            const float p0 = v0 == -INFINITY ? 0.f : ex2_approx(v0 - m);
            const float p1 = v1 == -INFINITY ? 0.f : ex2_approx(v1 - m);
            sum += p0 + p1;
            pk[j / 2] = pack_bf16x2(p0, p1);
        }
        tmem_store_16(tS + cc / 2, pk);
    });
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
    const int nblk = p.row_ptr[i + 1] - e0;
    auto ktile = [&](int it) { return p.col_idx[e0 + nblk - 1 - it]; };  // listed tiles, last first

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        bs_init_bars(bar0);
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
        // ---- softmax stream st (tiles st, st + 2, ...): thread t owns query row q0 + t (TMEM lane t)
        const int t = threadIdx.x % 128, st = threadIdx.x / 128;
        const int row = q0 + t;
        const uint32_t trow = tmem + (static_cast<uint32_t>(t & ~31) << 16);
        const uint32_t tS = trow + 128u * st, tO = trow + 256u + static_cast<uint32_t>(st * D);
        const float c = f.scale_log2;
        const float m2 = (EXT && p.alibi) ? exp2f(-8.f * static_cast<float>(h + 1) / static_cast<float>(f.Hq)) *
                                                1.4426950408889634f
                                          : 0.f;
        // m: raw score units (as the prefill), or log2 units of the biased score with EXT
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int it = st; it < nblk && ok; it += 2) {
            const int kv0 = ktile(it) * 128;
            ok = bwd_wait(bar_at(bar0, BS_S_FULL + st), (it >> 1) & 1, ctl, kStatusSoftmax);
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
            const bool masked = __any_sync(0xffffffffu, limit < 128);
            float mx;
            if constexpr (EXT) mx = ext_row_max(tS, lo, limit, c, m2, rel0);
            else mx = masked ? tile_row_max<true>(tS, limit) : tile_row_max<false>(tS, limit);
            const float m_new = fmaxf(m_used, mx);
            const float unit = EXT ? 1.f : c;
            if (it == st) {
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
            if constexpr (EXT) {
                l += ext_exp_to_p(tS, lo, limit, c, m2, rel0, m_used);
            } else {
                // a row that has seen only masked keys so far (m = -inf) gets P = 0
                const float mc = m_used == -INFINITY ? 0.f : m_used * c;
                l += masked ? tile_exp_to_p<true>(tS, limit, c, mc) : tile_exp_to_p<false>(tS, limit, c, mc);
            }
            tmem_store_wait();
            tc_fence_before();
            mbar_arrive(bar_at(bar0, BS_P_FULL + st));
        }
        // epilogue: merge the two streams by their maxima (log2 units); each writes D/2 channels.
        // The (m, l) exchange uses K slot 0, free once the last P V is done.
        if (ok && nblk > 0) ok = bwd_wait(bar_at(bar0, BS_O_FULL), 0, ctl, kStatusSoftmax);
        float2* ml = reinterpret_cast<float2*>(smg + L::kMerge);
        ml[st * 128 + t] = make_float2(EXT ? m_used : m_used * c, l);
        mbar_arrive(bar_at(bar0, BS_MERGE));
        if (ok) ok = bwd_wait(bar_at(bar0, BS_MERGE), 0, ctl, kStatusSoftmax);
        if (ok) {
            tc_fence_after();
            const float2 a = ml[t], bb = ml[128 + t];
            const float M = fmaxf(a.x, bb.x);
            const float sa = a.x == -INFINITY ? 0.f : ex2_approx(a.x - M);
            const float sb = bb.x == -INFINITY ? 0.f : ex2_approx(bb.x - M);
            const float Lsum = a.y * sa + bb.y * sb;
            const bool have0 = nblk >= 1, have1 = nblk >= 2;  // stream 1 sees tiles only from the second on
            const float inv = Lsum > 0.f ? 1.0f / Lsum : 0.f;
            const bool store = row < f.S;
            __nv_bfloat16* dst = f.o + ((static_cast<size_t>(b) * f.S + (store ? row : 0)) * f.Hq + h) * D;
            const uint32_t tO0 = trow + 256u, tO1 = trow + 256u + D;
#pragma unroll
            for (int cc = 0; cc < D / 2; cc += 32) {
                const int d0 = st * (D / 2) + cc;  // this stream's output channels
                uint32_t ra[32], rb[32];
                if (have0) tmem_load_32_async(tO0 + d0, ra);
                if (have1) tmem_load_32_async(tO1 + d0, rb);
                if (have0) tmem_wait_ld_32(ra);
                if (have1) tmem_wait_ld_32(rb);
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    float o0 = 0.f, o1 = 0.f;
                    if (have0) {
                        o0 += __uint_as_float(ra[j]) * sa;
                        o1 += __uint_as_float(ra[j + 1]) * sa;
                    }
                    if (have1) {
                        o0 += __uint_as_float(rb[j]) * sb;
                        o1 += __uint_as_float(rb[j + 1]) * sb;
                    }
                    pk[j / 2] = pack_bf16x2(o0 * inv, o1 * inv);
                }
                if (store) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + d0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            if (st == 0 && store && f.lse != nullptr)
                f.lse[(static_cast<size_t>(b) * f.Hq + h) * f.S + row] =
                    Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
        }
    } else if (warp < kBsWarpTma) {
        // ---- RoPE warps: Q once, then each K tile in its slot
        if (ROPE && nblk > 0) {
            const int t = threadIdx.x - kBsWarpRope * 32;
            RopeConsts k;
            rope_load_consts<D>(f, t, k);
            uint64_t cb[4], sb[4];
            rope_load_base<D>(f, i, t, cb, sb);
            bool ok = bwd_wait(bar_at(bar0, BS_Q_FULL), 0, ctl, kStatusRope);
            if (ok) {
                rope_rotate_tile<D, false>(smg + L::kQ, k, cb, sb, t);
                fence_proxy_async_smem();
                mbar_arrive(bar_at(bar0, BS_Q_ROT));
            }
            for (int it = 0; it < nblk && ok; ++it) {
                const int r = it % kBsSlots;
                rope_load_base<D>(f, ktile(it), t, cb, sb);
                ok = bwd_wait(bar_at(bar0, BS_K_FULL + r), (it / kBsSlots) & 1, ctl, kStatusRope);
                if (!ok) break;
                rope_rotate_tile<D, false>(smg + L::kK0 + r * L::kTile, k, cb, sb, t);
                fence_proxy_async_smem();
                mbar_arrive(bar_at(bar0, BS_K_ROT + r));
            }
        }
    } else if (warp == kBsWarpTma) {
        // ---- producer: Q once, then each listed tile's K and V into their rings
        if (lane == 0 && nblk > 0) {
            const uint32_t qb = bar_at(bar0, BS_Q_FULL);
            mbar_arrive_expect_tx(qb, L::kTile);
#pragma unroll
            for (int sub = 0; sub < D / 64; ++sub)
                tma_load_4d(sm + L::kQ + sub * kSubTileBytes, &f.tm_q, qb, sub * 64, h, q0, b);
            for (int it = 0; it < nblk; ++it) {
                const int r = it % kBsSlots, n = it / kBsSlots;
                const int kv0 = ktile(it) * 128;
                if (n >= 1 && !mbar_wait(bar_at(bar0, BS_K_EMPTY + r), (n - 1) & 1, ctl, kStatusProducer)) break;
                const uint32_t kb = bar_at(bar0, BS_K_FULL + r);
                mbar_arrive_expect_tx(kb, L::kTile);
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_4d(sm + L::kK0 + r * L::kTile + sub * kSubTileBytes, &f.tm_k, kb, sub * 64, g, kv0, b);
                if (n >= 1 && !mbar_wait(bar_at(bar0, BS_V_EMPTY + r), (n - 1) & 1, ctl, kStatusProducer)) break;
                const uint32_t vb = bar_at(bar0, BS_V_FULL + r);
                mbar_arrive_expect_tx(vb, L::kTile);
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_4d(sm + L::kV0 + r * L::kTile + sub * kSubTileBytes, &f.tm_v, vb, sub * 64, g, kv0, b);
            }
        }
        __syncwarp();
    } else if (warp == kBsWarpMma && lane == 0 && nblk > 0) {
        // ---- MMA issuer.  Tile it goes to stream it % 2: S_s = Q K^T (K-major, fp16 after RoPE),
        // then, once that stream's softmax has handed P back, O_s += P V (P from TMEM, V MN-major).
        // Issue order S(it), then P V(it - 1): the tensor cores form one stream's S while the other
        // stream's softmax works.
        const uint32_t kIdescS = umma_idesc_f16(ROPE ? 0u : 1u, 0u, 128, 128);
        constexpr uint32_t kIdescPV = umma_idesc_f16(1u, 1u, 128, D);
        const uint64_t qdesc = sw128_desc(sm + L::kQ, 16u, 1024u);
        bool ok = mbar_wait(bar_at(bar0, BS_Q_FULL), 0, ctl, kStatusMma);
        if (ok && ROPE) ok = mbar_wait(bar_at(bar0, BS_Q_ROT), 0, ctl, kStatusMma);
        for (int it = 0; it <= nblk && ok; ++it) {
            if (it < nblk) {
                const int r = it % kBsSlots, n = it / kBsSlots, s = it & 1;
                ok = mbar_wait(bar_at(bar0, BS_K_FULL + r), n & 1, ctl, kStatusMma);
                if (ok && ROPE) ok = mbar_wait(bar_at(bar0, BS_K_ROT + r), n & 1, ctl, kStatusMma);
                if (!ok) break;
                tc_fence_after();
                const uint64_t kdesc = sw128_desc(sm + L::kK0 + r * L::kTile, 16u, 1024u);
                const uint32_t tS = tmem + 128u * s;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_ss(tS, desc_advance(qdesc, kmajor_units(kk)), desc_advance(kdesc, kmajor_units(kk)), kIdescS,
                            kk > 0 ? 1u : 0u);
                tc_commit(bar_at(bar0, BS_K_EMPTY + r));  // the K slot refills once this S is formed
                tc_commit(bar_at(bar0, BS_S_FULL + s));
            }
            if (it >= 1) {
                const int pt = it - 1, ps = pt & 1, pr = pt % kBsSlots;
                ok = mbar_wait(bar_at(bar0, BS_P_FULL + ps), (pt >> 1) & 1, ctl, kStatusMma);
                if (ok) ok = mbar_wait(bar_at(bar0, BS_V_FULL + pr), (pt / kBsSlots) & 1, ctl, kStatusMma);
                if (!ok) break;
                tc_fence_after();
                const uint64_t vdesc = sw128_desc(sm + L::kV0 + pr * L::kTile, kSubTileBytes, 1024u);
                const uint32_t tS = tmem + 128u * ps, tO = tmem + 256u + static_cast<uint32_t>(ps * D);
                // 16 keys per step: 2048 bytes of V, 8 TMEM columns of P
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts(tO, tS + kk * 8u, desc_advance(vdesc, kk * 128u), kIdescPV, (pt >= 2 || kk > 0) ? 1u : 0u);
                tc_commit(bar_at(bar0, BS_V_EMPTY + pr));
            }
        }
        if (ok) tc_commit(bar_at(bar0, BS_O_FULL));
        tc_commit(bar_at(bar0, BS_DRAIN));
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar_at(bar0, BS_DRAIN), 0)) {
            if (global_timer_ns() - t0 > ctl.limit_ns) {
                atomicOr(ctl.status, kStatusDrain);
                break;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kBsWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace attn
