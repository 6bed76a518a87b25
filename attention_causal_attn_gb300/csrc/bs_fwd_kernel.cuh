// Block-sparse attention forward ("AttnFuse", sec. 4.3 Block-Sparse Attention:
// a CSR BlockMask lists the active key blocks of each row of blocks, and the
// kernel visits only those, so its work is proportional to the active share).
//
// Blocks are the kernel's 128 x 128 tiles.  A task is one query tile of one
// (batch, head).  One persistent CTA per SM runs a host-built list of tasks
// (heaviest rows first, balanced by listed tiles), so that the fixed costs of
// a task overlap the neighbouring tasks: the next task's K/V tiles and its Q
// load and rotation start while the current task's softmax runs its merge and
// output stores, and its first Q K^T products form before those stores end.
// Per task, Q is loaded and rotated once; the listed key tiles are visited in
// descending order and dealt alternately to two softmax streams, as the
// prefill deals two query tiles to its two stages:
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
    const int* tasks;      // task t = query tile * (B * Hq) + b * Hq + h, per-CTA lists
    const int* task_off;   // [gridDim.x + 1]: CTA c runs tasks[task_off[c] .. task_off[c+1])
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
    // epilogue: [2 streams][128 rows] float2 (m, l) over the Q tile, which every product of the
    // task has read by then; the next task's Q is loaded once both streams have read it
    static constexpr uint32_t kMerge = kQ;
};

enum : int {
    BS_Q_FULL = 0,
    BS_Q_ROT,
    BS_Q_EMPTY,                         // both streams read the merge values: Q may be reloaded
    BS_K_FULL,                          // [3]
    BS_K_ROT = BS_K_FULL + kBsSlots,    // [3]
    BS_K_EMPTY = BS_K_ROT + kBsSlots,   // [3] S of the slot's tile formed
    BS_V_FULL = BS_K_EMPTY + kBsSlots,  // [3]
    BS_V_EMPTY = BS_V_FULL + kBsSlots,  // [3] P V of the slot's tile done
    BS_S_FULL = BS_V_EMPTY + kBsSlots,  // [2] per stream
    BS_P_FULL = BS_S_FULL + 2,          // [2] per stream
    BS_O_FULL = BS_P_FULL + 2,
    BS_O_FREE,                          // both streams read O_0 and O_1: the next task may accumulate
    BS_DRAIN,
    BS_MERGE,
    BS_NUM
};
static_assert(BS_NUM * 8 <= 256, "barrier block");

__device__ __forceinline__ void bs_init_bars(uint32_t bar0) {
    mbar_init(bar_at(bar0, BS_Q_FULL), 1);
    mbar_init(bar_at(bar0, BS_Q_ROT), 128);
    mbar_init(bar_at(bar0, BS_Q_EMPTY), 256);
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
    mbar_init(bar_at(bar0, BS_O_FREE), 256);
    mbar_init(bar_at(bar0, BS_DRAIN), 1);
    mbar_init(bar_at(bar0, BS_MERGE), 256);
    fence_barrier_init();
    fence_proxy_async_smem();
}

// EXT: the score of column col of a tile for this row in log2 units (biased), or -inf when the
// key lies outside [lo, hi).  rel0 = first key of the tile - row; m2 = m_h * log2(e).  col is a
// compile-time constant once the TMEM stream is unrolled, so the distance costs one add.
__device__ __forceinline__ float ext_score(uint32_t raw, int col, int lo, int hi, float c, float m2, float rel0f) {
    const float s = fmaf(-m2, fabsf(rel0f + static_cast<float>(col)), __uint_as_float(raw) * c);
    return (col >= lo && col < hi) ? s : -INFINITY;
}

__device__ __forceinline__ float ext_row_max(uint32_t tS, int lo, int hi, float c, float m2, float rel0f) {
    float mx = -INFINITY;
    tmem_stream_128(tS, [&](const uint32_t (&r)[32], int cc) {
#pragma unroll
        for (int j = 0; j < 32; ++j) mx = fmaxf(mx, ext_score(r[j], cc + j, lo, hi, c, m2, rel0f));
    });
    return mx;
}

// P = exp2(score - m) in bf16 over the S columns (hidden keys 0), and the row sum of P.
// m is finite or, while the row has seen no key, -inf; then every score is -inf and P = 0.
__device__ __forceinline__ float ext_exp_to_p(uint32_t tS, int lo, int hi, float c, float m2, float rel0f, float m) {
    const float mm = m == -INFINITY ? 0.f : m;
    float sum = 0.f;
    tmem_stream_128(tS, [&](const uint32_t (&r)[32], int cc) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const float p0 = ex2_approx(ext_score(r[j], cc + j, lo, hi, c, m2, rel0f) - mm);
            const float p1 = ex2_approx(ext_score(r[j + 1], cc + j + 1, lo, hi, c, m2, rel0f) - mm);
            sum += p0 + p1;
            pk[j / 2] = pack_bf16x2(p0, p1);
        }
        tmem_store_16(tS + cc / 2, pk);
    });
    return sum;
}

// ALiBi on a tile whose 128 keys this row all sees and which lies on one side of the row:
// |rel0 + j| = sgn (rel0 + j), so the biased score is raw c + a j + b0 with a = -m2 sgn and
// b0 = a rel0, linear in the column.
__device__ __forceinline__ float alibi_row_max(uint32_t tS, float c, float a, float b0) {
    float mx = -INFINITY;
    tmem_stream_128(tS, [&](const uint32_t (&r)[32], int cc) {
        float m0 = mx, m1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            float v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                v[q] = fmaf(__uint_as_float(r[j + q]), c, fmaf(a, static_cast<float>(cc + j + q), b0));
            m0 = fmax3(m0, v[0], v[1]);
            m1 = fmax3(m1, v[2], v[3]);
        }
        mx = fmaxf(m0, m1);
    });
    return mx;
}

__device__ __forceinline__ float alibi_exp_to_p(uint32_t tS, float c, float a, float b0, float m) {
    const float bm = b0 - m;
    float sum = 0.f;
    tmem_stream_128(tS, [&](const uint32_t (&r)[32], int cc) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(r[j]), c, fmaf(a, static_cast<float>(cc + j), bm)));
            const float p1 = ex2_approx(fmaf(__uint_as_float(r[j + 1]), c, fmaf(a, static_cast<float>(cc + j + 1), bm)));
            sum += p0 + p1;
            pk[j / 2] = pack_bf16x2(p0, p1);
        }
        tmem_store_16(tS + cc / 2, pk);
    });
    return sum;
}

// One task: query tile i of batch b, head h (KV head g); its listed key tiles are
// col_idx[e0 .. e0 + nblk), visited last first.
struct BsTask {
    int i, b, h, g, e0, nblk;
};

__device__ __forceinline__ BsTask bs_task(const BsParams& p, int ti) {
    const FwdParams& f = p.f;
    const int bhs = f.B * f.Hq;
    const int t = p.tasks[ti];
    BsTask k;
    k.i = t / bhs;
    k.b = (t % bhs) / f.Hq;
    k.h = (t % bhs) % f.Hq;
    k.g = k.h / (f.Hq / f.Hkv);
    k.e0 = p.row_ptr[k.i];
    k.nblk = p.row_ptr[k.i + 1] - k.e0;
    return k;
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
    const int t_begin = p.task_off[blockIdx.x], t_end = p.task_off[blockIdx.x + 1];
    // Every role walks the same task list and skips the empty rows the same way; ring slots and
    // barrier phases count K/V tiles (kit) and non-empty tasks (qn) over the whole list.

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
        // ---- softmax stream st (tiles st, st + 2, ... of each task): thread t owns query row 128 i + t
        const int t = threadIdx.x % 128, st = threadIdx.x / 128;
        const uint32_t trow = tmem + (static_cast<uint32_t>(t & ~31) << 16);
        const uint32_t tS = trow + 128u * st, tO = trow + 256u + static_cast<uint32_t>(st * D);
        const float c = f.scale_log2;
        float2* ml = reinterpret_cast<float2*>(smg + L::kMerge);
        int sit = 0, qn = 0;  // S tiles of this stream, non-empty tasks
        bool ok = true;
        for (int ti = t_begin; ti < t_end && ok; ++ti) {
            const BsTask k = bs_task(p, ti);
            const int row = k.i * 128 + t;
            const bool store = row < f.S;
            __nv_bfloat16* dst = f.o + ((static_cast<size_t>(k.b) * f.S + (store ? row : 0)) * f.Hq + k.h) * D;
            const size_t lse_at = (static_cast<size_t>(k.b) * f.Hq + k.h) * f.S + row;
            if (k.nblk == 0) {
                // nothing listed: O = 0 (this stream's half of the channels), LSE = -inf
                if (store) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + st * (D / 2));
#pragma unroll
                    for (int q = 0; q < D / 16; ++q) d4[q] = make_uint4(0u, 0u, 0u, 0u);
                    if (st == 0 && f.lse != nullptr) f.lse[lse_at] = -INFINITY;
                }
                continue;
            }
            const float m2 = (EXT && p.alibi) ? exp2f(-8.f * static_cast<float>(k.h + 1) / static_cast<float>(f.Hq)) *
                                                    1.4426950408889634f
                                              : 0.f;
            // m: raw score units (as the prefill), or log2 units of the biased score with EXT
            float m_used = -INFINITY, l = 0.f;
            for (int it = st; it < k.nblk && ok; it += 2) {
                const int kv0 = p.col_idx[k.e0 + k.nblk - 1 - it] * 128;
                ok = bwd_wait(bar_at(bar0, BS_S_FULL + st), sit & 1, ctl, kStatusSoftmax);
                ++sit;
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
                // EXT tile kinds (uniform across the warp): 1 = no bias and no lower edge (the plain
                // path, in log2 units), 2 = ALiBi on fully visible keys on one side of every row,
                // 0 = the general form
                int kind = 0;
                float a_lin = 0.f, b_lin = 0.f;
                if constexpr (EXT) {
                    if (m2 == 0.f && __all_sync(0xffffffffu, lo <= 0)) {
                        kind = 1;
                    } else if (__all_sync(0xffffffffu, lo <= 0 && limit >= 128 && (kv0 >= row || kv0 + 127 <= row))) {
                        kind = 2;
                        a_lin = kv0 >= row ? -m2 : m2;
                        b_lin = a_lin * static_cast<float>(rel0);
                    }
                }
                float mx;
                if (EXT && kind == 0) mx = ext_row_max(tS, lo, limit, c, m2, static_cast<float>(rel0));
                else if (EXT && kind == 2) mx = alibi_row_max(tS, c, a_lin, b_lin);
                else mx = (masked ? tile_row_max<true>(tS, limit) : tile_row_max<false>(tS, limit)) * (EXT ? c : 1.f);
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
                if (EXT && kind == 0) {
                    l += ext_exp_to_p(tS, lo, limit, c, m2, static_cast<float>(rel0), m_used);
                } else if (EXT && kind == 2) {
                    l += alibi_exp_to_p(tS, c, a_lin, b_lin, m_used);  // m is finite: every key is seen
                } else if (EXT) {
                    const float mc = m_used == -INFINITY ? 0.f : m_used;  // log2 units
                    l += masked ? tile_exp_to_p<true>(tS, limit, c, mc) : tile_exp_to_p<false>(tS, limit, c, mc);
                } else {
                    // a row that has seen only masked keys so far (m = -inf) gets P = 0
                    const float mc = m_used == -INFINITY ? 0.f : m_used * c;
                    l += masked ? tile_exp_to_p<true>(tS, limit, c, mc) : tile_exp_to_p<false>(tS, limit, c, mc);
                }
                tmem_store_wait();
                tc_fence_before();
                mbar_arrive(bar_at(bar0, BS_P_FULL + st));
            }
            // epilogue: merge the two streams by their maxima (log2 units); each writes D/2 channels
            if (ok) ok = bwd_wait(bar_at(bar0, BS_O_FULL), qn & 1, ctl, kStatusSoftmax);
            if (!ok) break;
            tc_fence_after();
            ml[st * 128 + t] = make_float2(EXT ? m_used : m_used * c, l);
            mbar_arrive(bar_at(bar0, BS_MERGE));
            ok = bwd_wait(bar_at(bar0, BS_MERGE), qn & 1, ctl, kStatusSoftmax);
            if (!ok) break;
            const float2 a = ml[t], bb = ml[128 + t];
            fence_proxy_async_smem();  // the next task's Q copy overwrites the merge values
            mbar_arrive(bar_at(bar0, BS_Q_EMPTY));
            const float M = fmaxf(a.x, bb.x);
            const float sa = a.x == -INFINITY ? 0.f : ex2_approx(a.x - M);
            const float sb = bb.x == -INFINITY ? 0.f : ex2_approx(bb.x - M);
            const float Lsum = a.y * sa + bb.y * sb;
            const bool have1 = k.nblk >= 2;  // stream 1 sees tiles only from the second on
            const float inv = Lsum > 0.f ? 1.0f / Lsum : 0.f;
            const uint32_t tO0 = trow + 256u, tO1 = trow + 256u + D;
#pragma unroll
            for (int cc = 0; cc < D / 2; cc += 32) {
                const int d0 = st * (D / 2) + cc;  // this stream's output channels
                uint32_t ra[32], rb[32];
                tmem_load_32_async(tO0 + d0, ra);
                if (have1) tmem_load_32_async(tO1 + d0, rb);
                tmem_wait_ld_32(ra);
                if (have1) tmem_wait_ld_32(rb);
                if (cc + 32 >= D / 2) {  // last read of O_0 and O_1 by this thread
                    tc_fence_before();
                    mbar_arrive(bar_at(bar0, BS_O_FREE));
                }
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    float o0 = __uint_as_float(ra[j]) * sa, o1 = __uint_as_float(ra[j + 1]) * sa;
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
                f.lse[lse_at] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
            ++qn;
        }
    } else if (warp < kBsWarpTma) {
        // ---- RoPE warps: each task's Q once, then each of its K tiles in its slot
        if (ROPE) {
            const int t = threadIdx.x - kBsWarpRope * 32;
            RopeConsts rc;
            rope_load_consts<D>(f, t, rc);
            uint64_t cb[4], sb[4];
            int kit = 0, qn = 0;
            bool ok = true;
            for (int ti = t_begin; ti < t_end && ok; ++ti) {
                const BsTask k = bs_task(p, ti);
                if (k.nblk == 0) continue;
                rope_load_base<D>(f, k.i, t, cb, sb);
                ok = bwd_wait(bar_at(bar0, BS_Q_FULL), qn & 1, ctl, kStatusRope);
                if (!ok) break;
                rope_rotate_tile<D, false>(smg + L::kQ, rc, cb, sb, t);
                fence_proxy_async_smem();
                mbar_arrive(bar_at(bar0, BS_Q_ROT));
                for (int it = 0; it < k.nblk && ok; ++it) {
                    const int gi = kit + it, r = gi % kBsSlots;
                    rope_load_base<D>(f, p.col_idx[k.e0 + k.nblk - 1 - it], t, cb, sb);
                    ok = bwd_wait(bar_at(bar0, BS_K_FULL + r), (gi / kBsSlots) & 1, ctl, kStatusRope);
                    if (!ok) break;
                    rope_rotate_tile<D, false>(smg + L::kK0 + r * L::kTile, rc, cb, sb, t);
                    fence_proxy_async_smem();
                    mbar_arrive(bar_at(bar0, BS_K_ROT + r));
                }
                kit += k.nblk;
                ++qn;
            }
        }
    } else if (warp == kBsWarpTma) {
        // ---- producer: per task, the first K/V tile, then Q (once the previous task's merge has
        // read its copy of Q), then the other K/V tiles, into their rings
        if (lane == 0) {
            int kit = 0, qn = 0;
            bool ok = true;
            for (int ti = t_begin; ti < t_end && ok; ++ti) {
                const BsTask k = bs_task(p, ti);
                if (k.nblk == 0) continue;
                for (int it = 0; it < k.nblk && ok; ++it) {
                    const int gi = kit + it, r = gi % kBsSlots, n = gi / kBsSlots;
                    const int kv0 = p.col_idx[k.e0 + k.nblk - 1 - it] * 128;
                    if (n >= 1 && !mbar_wait(bar_at(bar0, BS_K_EMPTY + r), (n - 1) & 1, ctl, kStatusProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t kb = bar_at(bar0, BS_K_FULL + r);
                    mbar_arrive_expect_tx(kb, L::kTile);
#pragma unroll
                    for (int sub = 0; sub < D / 64; ++sub)
                        tma_load_4d(sm + L::kK0 + r * L::kTile + sub * kSubTileBytes, &f.tm_k, kb, sub * 64, k.g, kv0, k.b);
                    if (n >= 1 && !mbar_wait(bar_at(bar0, BS_V_EMPTY + r), (n - 1) & 1, ctl, kStatusProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t vb = bar_at(bar0, BS_V_FULL + r);
                    mbar_arrive_expect_tx(vb, L::kTile);
#pragma unroll
                    for (int sub = 0; sub < D / 64; ++sub)
                        tma_load_4d(sm + L::kV0 + r * L::kTile + sub * kSubTileBytes, &f.tm_v, vb, sub * 64, k.g, kv0, k.b);
                    if (it == 0) {
                        if (qn >= 1 && !mbar_wait(bar_at(bar0, BS_Q_EMPTY), (qn - 1) & 1, ctl, kStatusProducer)) {
                            ok = false;
                            break;
                        }
                        const uint32_t qb = bar_at(bar0, BS_Q_FULL);
                        mbar_arrive_expect_tx(qb, L::kTile);
#pragma unroll
                        for (int sub = 0; sub < D / 64; ++sub)
                            tma_load_4d(sm + L::kQ + sub * kSubTileBytes, &f.tm_q, qb, sub * 64, k.h, k.i * 128, k.b);
                    }
                }
                kit += k.nblk;
                ++qn;
            }
        }
        __syncwarp();
    } else if (warp == kBsWarpMma && lane == 0) {
        // ---- MMA issuer.  Tile it of a task goes to stream it % 2: S_s = Q K^T (K-major, fp16 after
        // RoPE), then, once that stream's softmax has handed P back, O_s += P V (P from TMEM, V
        // MN-major).  Issue order S(it), then P V(it - 1): the tensor cores form one stream's S while
        // the other stream's softmax works.  A task's first P V waits until the previous task's
        // epilogue has read O_0 and O_1; its S products need not.
        const uint32_t kIdescS = umma_idesc_f16(ROPE ? 0u : 1u, 0u, 128, 128);
        constexpr uint32_t kIdescPV = umma_idesc_f16(1u, 1u, 128, D);
        const uint64_t qdesc = sw128_desc(sm + L::kQ, 16u, 1024u);
        int kit = 0, qn = 0, pc0 = 0, pc1 = 0;
        bool ok = true;
        for (int ti = t_begin; ti < t_end && ok; ++ti) {
            const BsTask k = bs_task(p, ti);
            if (k.nblk == 0) continue;
            ok = mbar_wait(bar_at(bar0, BS_Q_FULL), qn & 1, ctl, kStatusMma);
            if (ok && ROPE) ok = mbar_wait(bar_at(bar0, BS_Q_ROT), qn & 1, ctl, kStatusMma);
            for (int it = 0; it <= k.nblk && ok; ++it) {
                if (it < k.nblk) {
                    const int gi = kit + it, r = gi % kBsSlots, n = gi / kBsSlots, s = it & 1;
                    ok = mbar_wait(bar_at(bar0, BS_K_FULL + r), n & 1, ctl, kStatusMma);
                    if (ok && ROPE) ok = mbar_wait(bar_at(bar0, BS_K_ROT + r), n & 1, ctl, kStatusMma);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t kdesc = sw128_desc(sm + L::kK0 + r * L::kTile, 16u, 1024u);
                    const uint32_t tS = tmem + 128u * s;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma_ss(tS, desc_advance(qdesc, kmajor_units(kk)), desc_advance(kdesc, kmajor_units(kk)),
                                kIdescS, kk > 0 ? 1u : 0u);
                    tc_commit(bar_at(bar0, BS_K_EMPTY + r));  // the K slot refills once this S is formed
                    tc_commit(bar_at(bar0, BS_S_FULL + s));
                }
                if (it >= 1) {
                    const int pt = it - 1, ps = pt & 1, gp = kit + pt, pr = gp % kBsSlots;
                    const int pc = ps ? pc1++ : pc0++;
                    ok = mbar_wait(bar_at(bar0, BS_P_FULL + ps), pc & 1, ctl, kStatusMma);
                    if (ok) ok = mbar_wait(bar_at(bar0, BS_V_FULL + pr), (gp / kBsSlots) & 1, ctl, kStatusMma);
                    if (ok && pt == 0 && qn >= 1) ok = mbar_wait(bar_at(bar0, BS_O_FREE), (qn - 1) & 1, ctl, kStatusMma);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t vdesc = sw128_desc(sm + L::kV0 + pr * L::kTile, kSubTileBytes, 1024u);
                    const uint32_t tS = tmem + 128u * ps, tO = tmem + 256u + static_cast<uint32_t>(ps * D);
                    // 16 keys per step: 2048 bytes of V, 8 TMEM columns of P
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_ts(tO, tS + kk * 8u, desc_advance(vdesc, kk * 128u), kIdescPV,
                                (pt >= 2 || kk > 0) ? 1u : 0u);
                    tc_commit(bar_at(bar0, BS_V_EMPTY + pr));
                }
            }
            if (ok) tc_commit(bar_at(bar0, BS_O_FULL));
            kit += k.nblk;
            ++qn;
        }
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
