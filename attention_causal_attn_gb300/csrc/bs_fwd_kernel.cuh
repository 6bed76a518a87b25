// Block-sparse attention forward ("AttnFuse", sec. 4.3 Block-Sparse Attention:
// a CSR BlockMask lists the active key blocks of each row of blocks, and the
// kernel visits only those, so its work is proportional to the active share).
//
// Blocks are the kernel's 128 x 128 tiles.  A task is one query tile of one
// (batch, head): Q is loaded and rotated once, and the listed key tiles are
// visited in descending order,
//   S = Q K^T (tcgen05, TMEM)  ->  online softmax, P in bf16 over S  ->  O += P V.
// One persistent CTA per SM runs two task streams side by side, as the prefill
// runs its two query-tile stages: each stream has its own Q slot, S and O in
// TMEM, and softmax warpgroup (one thread per query row), and walks its own
// host-built task list (heaviest tasks first, the streams balanced by listed
// tiles).  The tensor cores alternate between the streams: while one stream's
// softmax works on its S, they accumulate the other stream's P V and form its
// next S.  One stream's task boundary (the epilogue, the next Q load and
// rotation) thus overlaps the other stream's tiles.  K and V tiles of both
// streams pass through one K ring (three slots) and one V ring (two slots) in
// the order the tensor cores consume them.  Roles: two softmax warpgroups,
// four RoPE warps, a TMA warp and an MMA warp.  A row of blocks with nothing
// listed writes O = 0 and LSE = -inf.  Every wait is bounded.
//
// The EXT variants add the sliding_window and alibi combinators ("AttnFuse",
// sec. 3): key j is visible to query i only when |i - j| < window, and the
// score gains -m_h |i - j| with m_h = 2^(-8 (h+1) / Hq).  EXT = 1 is the window
// alone, EXT = 2 ALiBi with or without the window; each instance carries only
// the softmax forms it can take, which keeps the code within the instruction
// cache.
#pragma once

#include "bwd_kernel.cuh"

namespace attn {

struct BsParams {
    FwdParams f;           // tm_q, tm_k, tm_v, o, lse, RoPE factor table, shape, scale, status, wait limit
    const int* row_ptr;    // [ceil(S/128) + 1]
    const int* col_idx;    // listed key tiles of each row of tiles, ascending
    int window;            // EXT: visible iff |i - j| < window (0: no window)
    int alibi;             // EXT: ALiBi bias on
    const int* tasks;      // task t = query tile * (B * Hq) + b * Hq + h
    const int* task_off;   // [2 gridDim.x + 1]: stream s of CTA c runs tasks[task_off[2c+s] .. task_off[2c+s+1])
};

constexpr int kBsThreads = 448;  // warps 0-7 softmax (two streams), 8-11 RoPE, 12 TMA, 13 MMA
constexpr int kBsWarpRope = 8, kBsWarpTma = 12, kBsWarpMma = 13;
constexpr int kBsMaxSlots = 5;  // barrier room per ring

template <int D>
struct BsLayout {
    // Paired ring (D = 64): a tile's K and V share a slot index, land on one barrier (K_FULL) and
    // are released together after its P V (K_EMPTY), so the issuer waits once and commits once
    // less per tile.  D = 128 has room only for K and V rings of 3 and 2 slots (with the two Q
    // slots in 227 KB): separate barriers.
    static constexpr bool kPairKV = D == 64;
    static constexpr int KS = kPairKV ? 4 : 3, VS = kPairKV ? 4 : 2;
    static_assert(KS <= kBsMaxSlots && VS <= kBsMaxSlots, "ring depth");
    static constexpr uint32_t kTile = 128u * D * 2u;
    static constexpr uint32_t kQ0 = 0;                 // Q slot of stream s at kQ0 + s kTile
    static constexpr uint32_t kK0 = 2 * kTile;         // K slot r at kK0 + r kTile
    static constexpr uint32_t kV0 = kK0 + KS * kTile;  // V slot r at kV0 + r kTile
    static constexpr uint32_t kBars = kV0 + VS * kTile;
    static constexpr uint32_t kMisc = kBars + 512;
    static constexpr uint32_t kBytes = kMisc + 64;
    static constexpr uint32_t kAlloc = kBytes + 1024;
};

enum : int {
    BS_Q_FULL = 0,                         // [2] per stream
    BS_Q_ROT = BS_Q_FULL + 2,              // [2]
    BS_Q_EMPTY = BS_Q_ROT + 2,             // [2] the task's last S formed: the slot may be reloaded
    BS_K_FULL = BS_Q_EMPTY + 2,              // [K slots]
    BS_K_ROT = BS_K_FULL + kBsMaxSlots,      // [K slots]
    BS_K_EMPTY = BS_K_ROT + kBsMaxSlots,     // [K slots] S of the slot's tile formed
    BS_V_FULL = BS_K_EMPTY + kBsMaxSlots,    // [V slots]
    BS_V_EMPTY = BS_V_FULL + kBsMaxSlots,    // [V slots] P V of the slot's tile done
    BS_S_FULL = BS_V_EMPTY + kBsMaxSlots,    // [2] per stream
    BS_P_FULL = BS_S_FULL + 2,             // [2]
    BS_O_FULL = BS_P_FULL + 2,             // [2] the task's last P V done
    BS_O_FREE = BS_O_FULL + 2,             // [2] the epilogue read O: the next task may accumulate
    BS_DRAIN = BS_O_FREE + 2,
    BS_NUM
};
static_assert(BS_NUM * 8 <= 512, "barrier block");

__device__ __forceinline__ void bs_init_bars(uint32_t bar0) {
    for (int s = 0; s < 2; ++s) {
        mbar_init(bar_at(bar0, BS_Q_FULL + s), 1);
        mbar_init(bar_at(bar0, BS_Q_ROT + s), 128);
        mbar_init(bar_at(bar0, BS_Q_EMPTY + s), 1);
        mbar_init(bar_at(bar0, BS_S_FULL + s), 1);
        mbar_init(bar_at(bar0, BS_P_FULL + s), 128);
        mbar_init(bar_at(bar0, BS_O_FULL + s), 1);
        mbar_init(bar_at(bar0, BS_O_FREE + s), 128);
    }
    for (int r = 0; r < kBsMaxSlots; ++r) {
        mbar_init(bar_at(bar0, BS_K_FULL + r), 1);
        mbar_init(bar_at(bar0, BS_K_ROT + r), 128);
        mbar_init(bar_at(bar0, BS_K_EMPTY + r), 1);
    }
    for (int r = 0; r < kBsMaxSlots; ++r) {
        mbar_init(bar_at(bar0, BS_V_FULL + r), 1);
        mbar_init(bar_at(bar0, BS_V_EMPTY + r), 1);
    }
    mbar_init(bar_at(bar0, BS_DRAIN), 1);
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

// One-pass softmax of a local tile, m in log2 units of the biased score: the
// window tiles with no bias (BIAS false) and the ALiBi tiles whose visible keys
// all lie on one side of the row (BIAS: score = raw c + a j + b0, linear in the
// column j).  MASKED: the row sees only the keys [lo, limit) of the tile (a
// lower window edge, the diagonal, a ragged end); the hidden scores become
// -inf before the exponential, so their P is exactly 0.  Each 32-key chunk's
// reference is a bound on its largest score: the chunk maximum that
// tcgen05.ld.red returns times c (recomputed from the visible keys on chunks
// with hidden ones), plus the chunk's largest bias.  A bound at or above the
// true maximum is as good a reference as the maximum itself (P is formed
// against it and stays below 2^threshold); the moves and the deferred rescale
// of O and earlier P chunks are those of tile_exp_online.
template <int D, bool MASKED, bool BIAS>
__device__ __forceinline__ void local_exp_online(uint32_t tS, uint32_t tO, float c, int lo, int limit, float a,
                                                 float b0, bool first, float& m_used, float& l) {
    const uint64_t c2 = f2_pack(c, c);
    float nm = m_used == -INFINITY ? 0.f : -m_used;  // a row that has seen no key forms P against 0
    uint64_t sum2 = f2_pack(0.f, 0.f);
    float alpha_all = 1.f, fac0 = 1.f, fac1 = 1.f, fac2 = 1.f;
    bool moved = false;
    auto step = [&](uint32_t (&r)[32], float cm, int k) {
        if (MASKED && (32 * k < lo || 32 * k + 31 >= limit)) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (32 * k + j < lo || 32 * k + j >= limit) r[j] = __float_as_uint(-INFINITY);
            cm = row_max32<false>(r, 0, 0, -INFINITY);
        }
        float ub = cm * c;
        if (BIAS) ub += fmaf(a, static_cast<float>(a > 0.f ? 32 * k + 31 : 32 * k), b0);
        if (ub - m_used > kRescaleThreshold) {
            if (m_used != -INFINITY) {
                const float alpha = ex2_approx(m_used - ub);
                l *= alpha;
                sum2 = f2_mul(sum2, f2_pack(alpha, alpha));
                alpha_all *= alpha;
                if (k > 0) fac0 *= alpha;
                if (k > 1) fac1 *= alpha;
                if (k > 2) fac2 *= alpha;
                moved = true;
            }
            m_used = ub;
            nm = -m_used;
        }
        uint32_t pk[16];
        if constexpr (BIAS) {
            // x_j = raw_j c + (a j + b0 - m), the bias term advanced two columns at a time
            const float bm = b0 + nm;
            uint64_t bias2 = f2_pack(fmaf(a, static_cast<float>(32 * k), bm), fmaf(a, static_cast<float>(32 * k + 1), bm));
            const uint64_t step2 = f2_pack(2.f * a, 2.f * a);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), c2, bias2), x0, x1);
                bias2 = f2_add(bias2, step2);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                sum2 = f2_add(sum2, f2_pack(p0, p1));
                pk[j / 2] = pack_bf16x2(p0, p1);
            }
        } else {
            exp_pack32<false>(r, 32 * k, limit, c2, f2_pack(nm, nm), sum2, pk);
        }
        tmem_store_16(tS + 16 * k, pk);
    };
    uint32_t ra[32], rb[32];
    float ma, mb;
    tmem_load_32_max(tS, ra, ma);
    tmem_load_32_max_async(tS + 32, rb, mb);
    step(ra, ma, 0);
    tmem_wait_ld_32_max(rb, mb);
    tmem_load_32_max_async(tS + 64, ra, ma);
    step(rb, mb, 1);
    tmem_wait_ld_32_max(ra, ma);
    tmem_load_32_max_async(tS + 96, rb, mb);
    step(ra, ma, 2);
    tmem_wait_ld_32_max(rb, mb);
    step(rb, mb, 3);
    float s0, s1;
    f2_unpack(sum2, s0, s1);
    l += s0 + s1;
    if (__any_sync(0xffffffffu, moved)) rescale_o_and_p<D>(tO, tS, alpha_all, fac0, fac1, fac2, !first);
}

// The general local tile (an ALiBi bias whose sign changes across a row's
// visible keys: the diagonal tile of a two-sided window): two passes over S
// (the biased maximum, then P), m in log2 units.  Rare per task, so it is kept
// out of line: the one-pass paths then keep their registers.  Called by the
// whole warp.
template <int D>
__device__ __noinline__ void local_tile_general(uint32_t tS, uint32_t tO, int lo, int limit, float c, float m2,
                                                float rel0f, bool first, float& m_used, float& l) {
    const float mx = ext_row_max(tS, lo, limit, c, m2, rel0f);
    const float m_new = fmaxf(m_used, mx);
    if (first) {
        m_used = m_new;
    } else {
        const bool need = m_new - m_used > kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
            float alpha = 1.f;
            if (need) {
                alpha = m_used == -INFINITY ? 0.f : ex2_approx(m_used - m_new);
                m_used = m_new;
                l *= alpha;
            }
            rescale_o_and_p<D>(tO, tS, alpha, 1.f, 1.f, 1.f, true);  // no P formed yet: its factors are 1
        }
    }
    l += ext_exp_to_p(tS, lo, limit, c, m2, rel0f, m_used);
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

// A stream's position in its flattened tile sequence (the listed tiles of its
// non-empty tasks, task by task).  The TMA, RoPE and MMA roles each walk both
// streams' sequences in the same interleaved order.
struct BsCursor {
    int ti, te;  // current task index, end of the stream's list
    int it;      // tile of the current task
    BsTask k;
    __device__ __forceinline__ void skip_empty(const BsParams& p) {
        for (; ti < te; ++ti) {
            k = bs_task(p, ti);
            if (k.nblk > 0) return;
        }
    }
    __device__ __forceinline__ void init(const BsParams& p, int begin, int end) {
        ti = begin;
        te = end;
        it = 0;
        skip_empty(p);
    }
    __device__ __forceinline__ bool valid() const { return ti < te; }
    __device__ __forceinline__ bool first() const { return it == 0; }
    __device__ __forceinline__ bool last() const { return it == k.nblk - 1; }
    __device__ __forceinline__ int ktile(const BsParams& p) const { return p.col_idx[k.e0 + k.nblk - 1 - it]; }
    __device__ __forceinline__ void next(const BsParams& p) {
        if (++it < k.nblk) return;
        it = 0;
        ++ti;
        skip_empty(p);
    }
};

template <typename T>
__device__ __forceinline__ void bs_swap(T& a, T& b) {
    const T t = a;
    a = b;
    b = t;
}

template <int D, bool CAUSAL, bool ROPE, int EXT = 0>
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
    // stream 0 runs tasks [tb0, tb1), stream 1 runs [tb1, te1)
    const int tb0 = p.task_off[2 * blockIdx.x], tb1 = p.task_off[2 * blockIdx.x + 1];
    const int te1 = p.task_off[2 * blockIdx.x + 2];

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
        // ---- softmax of stream st: thread t owns query row 128 i + t (TMEM lane t) of each task
        const int t = threadIdx.x % 128, st = threadIdx.x / 128;
        const uint32_t trow = tmem + (static_cast<uint32_t>(t & ~31) << 16);
        const uint32_t tS = trow + 128u * st, tO = trow + 256u + static_cast<uint32_t>(st * D);
        const float c = f.scale_log2;
        const int tb = st ? tb1 : tb0, te = st ? te1 : tb1;
        int sit = 0, oit = 0;  // S tiles and finished tasks of this stream (barrier phases)
        bool ok = true;
        for (int ti = tb; ti < te && ok; ++ti) {
            const BsTask k = bs_task(p, ti);
            const int row = k.i * 128 + t;
            const bool store = row < f.S;
            __nv_bfloat16* dst = f.o + ((static_cast<size_t>(k.b) * f.S + (store ? row : 0)) * f.Hq + k.h) * D;
            const size_t lse_at = (static_cast<size_t>(k.b) * f.Hq + k.h) * f.S + row;
            if (k.nblk == 0) {  // nothing listed: O = 0, LSE = -inf
                if (store) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                    for (int q = 0; q < D / 8; ++q) d4[q] = make_uint4(0u, 0u, 0u, 0u);
                    if (f.lse != nullptr) f.lse[lse_at] = -INFINITY;
                }
                continue;
            }
            const float m2 = (EXT == 2 && p.alibi) ? exp2f(-8.f * static_cast<float>(k.h + 1) / static_cast<float>(f.Hq)) *
                                                    1.4426950408889634f
                                              : 0.f;
            // m: raw score units (as the prefill), or log2 units of the biased score with EXT
            float m_used = -INFINITY, l = 0.f;
            for (int it = 0; it < k.nblk && ok; ++it) {
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
                const bool edged = EXT != 0 && __any_sync(0xffffffffu, lo > 0 || limit < 128);
                // EXT tile kinds (uniform across the warp): 1 = no bias (window edges as masks, in
                // log2 units), 2 = ALiBi whose visible keys lie on one side of every row, 0 = the
                // general form (an ALiBi tile that a row's visible keys straddle)
                int kind = 0;
                float a_lin = 0.f, b_lin = 0.f;
                if constexpr (EXT == 1) {
                    kind = 1;
                } else if constexpr (EXT == 2) {
                    if (__all_sync(0xffffffffu, kv0 + lo >= row || kv0 + limit - 1 <= row)) {
                        kind = 2;
                        a_lin = kv0 + lo >= row ? -m2 : m2;
                        b_lin = a_lin * static_cast<float>(rel0);
                    }
                }
                if constexpr (EXT == 0) {
                    // the prefill's one-pass softmax (raw score units, chunk maxima from tcgen05.ld.red)
                    if (masked) tile_exp_online<D, true>(tS, tO, c, limit, it == 0, m_used, l);
                    else tile_exp_online<D, false>(tS, tO, c, limit, it == 0, m_used, l);
                } else if (EXT == 1 && kind == 1) {
                    if (edged) local_exp_online<D, true, false>(tS, tO, c, lo, limit, 0.f, 0.f, it == 0, m_used, l);
                    else local_exp_online<D, false, false>(tS, tO, c, 0, 128, 0.f, 0.f, it == 0, m_used, l);
                } else if (EXT == 2 && kind == 2) {
                    if (edged) local_exp_online<D, true, true>(tS, tO, c, lo, limit, a_lin, b_lin, it == 0, m_used, l);
                    else local_exp_online<D, false, true>(tS, tO, c, 0, 128, a_lin, b_lin, it == 0, m_used, l);
                } else {  // the general local tile: a lower edge or a bias across the row
                    local_tile_general<D>(tS, tO, lo, limit, c, m2, static_cast<float>(rel0), it == 0, m_used, l);
                }
                tmem_store_wait();
                tc_fence_before();
                mbar_arrive(bar_at(bar0, BS_P_FULL + st));
            }
            // epilogue: O / l in bf16, LSE in natural log
            if (ok) ok = bwd_wait(bar_at(bar0, BS_O_FULL + st), oit & 1, ctl, kStatusSoftmax);
            ++oit;
            if (!ok) break;
            tc_fence_after();
            const float inv = l > 0.f ? 1.0f / l : 0.f;
            const uint64_t il2 = f2_pack(inv, inv);
#pragma unroll
            for (int cc = 0; cc < D; cc += 32) {
                uint32_t r[32];
                tmem_load_32(tO + cc, r);
                if (cc + 32 == D) {  // the last read of O_st by this thread
                    tc_fence_before();
                    mbar_arrive(bar_at(bar0, BS_O_FREE + st));
                }
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float x0, x1;
                    f2_unpack(f2_mul(f2_pack(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), il2), x0, x1);
                    pk[j] = pack_bf16x2(x0, x1);
                }
                if (store) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
                    for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            if (store && f.lse != nullptr)
                f.lse[lse_at] = l > 0.f ? ((EXT ? m_used : m_used * c) + log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    } else if (warp < kBsWarpTma) {
        // ---- RoPE warps: Q of each task once, then each K tile in its slot, in the order the
        // tensor cores consume them
        if (ROPE) {
            const int t = threadIdx.x - kBsWarpRope * 32;
            RopeConsts rc;
            rope_load_consts<D>(f, t, rc);
            uint64_t cb[4], sb[4];
            BsCursor c0, c1;
            c0.init(p, tb0, tb1);
            c1.init(p, tb1, te1);
            int kq = 0, qn0 = 0, qn1 = 0;
            auto rope_for_s = [&](const BsCursor& cu, int s, int& qn) -> bool {
                if (cu.first()) {
                    rope_load_base<D>(f, cu.k.i, t, cb, sb);
                    if (!bwd_wait(bar_at(bar0, BS_Q_FULL + s), qn & 1, ctl, kStatusRope)) return false;
                    ++qn;
                    rope_rotate_tile<D, false>(smg + L::kQ0 + s * L::kTile, rc, cb, sb, t);
                    fence_proxy_async_smem();
                    mbar_arrive(bar_at(bar0, BS_Q_ROT + s));
                }
                const int r = kq % L::KS;
                rope_load_base<D>(f, cu.ktile(p), t, cb, sb);
                if (!bwd_wait(bar_at(bar0, BS_K_FULL + r), (kq / L::KS) & 1, ctl, kStatusRope)) return false;
                ++kq;
                rope_rotate_tile<D, false>(smg + L::kK0 + r * L::kTile, rc, cb, sb, t);
                fence_proxy_async_smem();
                mbar_arrive(bar_at(bar0, BS_K_ROT + r));
                return true;
            };
            // c0 is the stream whose turn it is (s); it swaps with c1 after each turn, so every
            // step has one copy in the code
            bool ok = true, go0 = false, go1 = false;
            int s = 0;
            while (ok && (c0.valid() || c1.valid())) {
                if (c0.valid()) {
                    if (go0) c0.next(p);
                    go0 = true;
                    if (c0.valid()) ok = rope_for_s(c0, s, qn0);
                }
                bs_swap(c0, c1);
                bs_swap(qn0, qn1);
                bs_swap(go0, go1);
                s ^= 1;
            }
        }
    } else if (warp == kBsWarpTma) {
        // ---- producer: Q, K and V tiles of both streams in the order the tensor cores consume
        // them (S_0, S_1 first, then per round P V_0, the next S_0, P V_1, the next S_1)
        if (lane == 0) {
            BsCursor c0, c1;
            c0.init(p, tb0, tb1);
            c1.init(p, tb1, te1);
            int kq = 0, vq = 0, ql0 = 0, ql1 = 0;
            auto load_for_s = [&](const BsCursor& cu, int s, int& ql) -> bool {
                if (cu.first()) {  // the task's Q, once the stream's previous task formed its last S
                    if (ql >= 1 && !mbar_wait(bar_at(bar0, BS_Q_EMPTY + s), (ql - 1) & 1, ctl, kStatusProducer))
                        return false;
                    ++ql;
                    const uint32_t qb = bar_at(bar0, BS_Q_FULL + s);
                    mbar_arrive_expect_tx(qb, L::kTile);
#pragma unroll
                    for (int sub = 0; sub < D / 64; ++sub)
                        tma_load_4d(sm + L::kQ0 + s * L::kTile + sub * kSubTileBytes, &f.tm_q, qb, sub * 64, cu.k.h,
                                    cu.k.i * 128, cu.k.b);
                }
                const int r = kq % L::KS, n = kq / L::KS;
                if (n >= 1 && !mbar_wait(bar_at(bar0, BS_K_EMPTY + r), (n - 1) & 1, ctl, kStatusProducer)) return false;
                ++kq;
                const uint32_t kb = bar_at(bar0, BS_K_FULL + r);
                mbar_arrive_expect_tx(kb, L::kPairKV ? 2 * L::kTile : L::kTile);
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_4d(sm + L::kK0 + r * L::kTile + sub * kSubTileBytes, &f.tm_k, kb, sub * 64, cu.k.g,
                                cu.ktile(p) * 128, cu.k.b);
                if constexpr (L::kPairKV) {  // the tile's V into the same slot index, on the same barrier
#pragma unroll
                    for (int sub = 0; sub < D / 64; ++sub)
                        tma_load_4d(sm + L::kV0 + r * L::kTile + sub * kSubTileBytes, &f.tm_v, kb, sub * 64, cu.k.g,
                                    cu.ktile(p) * 128, cu.k.b);
                }
                return true;
            };
            auto load_v = [&](const BsCursor& cu) -> bool {
                const int r = vq % L::VS, n = vq / L::VS;
                if (n >= 1 && !mbar_wait(bar_at(bar0, BS_V_EMPTY + r), (n - 1) & 1, ctl, kStatusProducer)) return false;
                ++vq;
                const uint32_t vb = bar_at(bar0, BS_V_FULL + r);
                mbar_arrive_expect_tx(vb, L::kTile);
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_4d(sm + L::kV0 + r * L::kTile + sub * kSubTileBytes, &f.tm_v, vb, sub * 64, cu.k.g,
                                cu.ktile(p) * 128, cu.k.b);
                return true;
            };
            // c0 is the stream whose turn it is (s), as in the RoPE loop: its first turn loads
            // for S only, each later turn the V tile of its last S and then its next S
            bool ok = true, go0 = false, go1 = false;
            int s = 0;
            while (ok && (c0.valid() || c1.valid())) {
                if (c0.valid()) {
                    if (go0) {
                        if (!L::kPairKV) ok = load_v(c0);
                        c0.next(p);
                    }
                    go0 = true;
                    if (ok && c0.valid()) ok = load_for_s(c0, s, ql0);
                }
                bs_swap(c0, c1);
                bs_swap(ql0, ql1);
                bs_swap(go0, go1);
                s ^= 1;
            }
            // On the way out, whether the lists ended or a wait gave up: the last load of every
            // slot has landed before the CTA may exit (ql0 belongs to stream s, ql1 to the other).
            drain_ring(bar_at(bar0, BS_Q_FULL + s), 1, ql0, ctl, kStatusDrain);
            drain_ring(bar_at(bar0, BS_Q_FULL + (s ^ 1)), 1, ql1, ctl, kStatusDrain);
            drain_ring(bar_at(bar0, BS_K_FULL), L::KS, kq, ctl, kStatusDrain);
            if (!L::kPairKV) drain_ring(bar_at(bar0, BS_V_FULL), L::VS, vq, ctl, kStatusDrain);
        }
        __syncwarp();
    } else if (warp == kBsWarpMma) {  // the whole warp: one elected thread issues
        // ---- MMA issuer.  Per stream s: S_s = Q_s K^T (K-major, fp16 after RoPE), then, once the
        // stream's softmax has handed P back, O_s += P V (P from TMEM, V MN-major) followed at once
        // by the stream's next S, as the prefill issues its stages.  The streams alternate, so the
        // tensor cores work on one stream while the other's softmax runs.  A task's first P V
        // waits until the stream's previous epilogue has read O_s.
        const uint32_t kIdescS = umma_idesc_f16(ROPE ? 0u : 1u, 0u, 128, 128);
        constexpr uint32_t kIdescPV = umma_idesc_f16(1u, 1u, 128, D);
        BsCursor c0, c1;
        c0.init(p, tb0, tb1);
        c1.init(p, tb1, te1);
        int kq = 0, vq = 0, qn0 = 0, qn1 = 0, pq0 = 0, pq1 = 0, dn0 = 0, dn1 = 0;
        auto issue_s = [&](const BsCursor& cu, int s, int& qn, int& kt) -> bool {
            if (cu.first()) {
                if (!mbar_wait_warp(bar_at(bar0, BS_Q_FULL + s), qn & 1, ctl, kStatusMma)) return false;
                if (ROPE && !mbar_wait_warp(bar_at(bar0, BS_Q_ROT + s), qn & 1, ctl, kStatusMma)) return false;
                ++qn;
            }
            const int r = kq % L::KS, n = kq / L::KS;
            if (!mbar_wait_warp(bar_at(bar0, BS_K_FULL + r), n & 1, ctl, kStatusMma)) return false;
            if (ROPE && !mbar_wait_warp(bar_at(bar0, BS_K_ROT + r), n & 1, ctl, kStatusMma)) return false;
            kt = kq++;  // the tile's ticket: with the paired ring its P V reads V slot kt % VS
            tc_fence_after();
            const uint64_t qdesc = sw128_desc(sm + L::kQ0 + s * L::kTile, 16u, 1024u);
            const uint64_t kdesc = sw128_desc(sm + L::kK0 + r * L::kTile, 16u, 1024u);
            const uint32_t tS = tmem + 128u * s;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_ss(tS, desc_advance(qdesc, kmajor_units(kk)), desc_advance(kdesc, kmajor_units(kk)), kIdescS,
                        kk > 0 ? 1u : 0u);
            if (!L::kPairKV) tc_commit(bar_at(bar0, BS_K_EMPTY + r));  // the K slot refills once this S is formed
            if (cu.last()) tc_commit(bar_at(bar0, BS_Q_EMPTY + s));  // and Q_s after the task's last S
            tc_commit(bar_at(bar0, BS_S_FULL + s));
            return true;
        };
        auto issue_pv = [&](const BsCursor& cu, int s, int& pq, int& dn, int kt) -> bool {
            if (!mbar_wait_warp(bar_at(bar0, BS_P_FULL + s), pq & 1, ctl, kStatusMma)) return false;
            ++pq;
            // paired ring: V landed with the tile's K (waited before its S)
            const int r = L::kPairKV ? kt % L::VS : vq % L::VS, n = vq / L::VS;
            if (!L::kPairKV && !mbar_wait_warp(bar_at(bar0, BS_V_FULL + r), n & 1, ctl, kStatusMma)) return false;
            if (cu.first() && dn >= 1 && !mbar_wait_warp(bar_at(bar0, BS_O_FREE + s), (dn - 1) & 1, ctl, kStatusMma))
                return false;
            ++vq;
            tc_fence_after();
            const uint64_t vdesc = sw128_desc(sm + L::kV0 + r * L::kTile, kSubTileBytes, 1024u);
            const uint32_t tS = tmem + 128u * s, tO = tmem + 256u + static_cast<uint32_t>(s * D);
            // 16 keys per step: 2048 bytes of V, 8 TMEM columns of P
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                umma_ts(tO, tS + kk * 8u, desc_advance(vdesc, kk * 128u), kIdescPV, (!cu.first() || kk > 0) ? 1u : 0u);
            tc_commit(bar_at(bar0, L::kPairKV ? BS_K_EMPTY + r : BS_V_EMPTY + r));  // K and V, or V, refill
            if (cu.last()) {
                tc_commit(bar_at(bar0, BS_O_FULL + s));
                ++dn;
            }
            return true;
        };
        // c0 is the stream whose turn it is (s): its first turn forms S only, each later turn
        // accumulates P V of its last S and forms its next S
        bool ok = true, go0 = false, go1 = false;
        int s = 0, kt0 = 0, kt1 = 0;  // ticket of each stream's last S
        while (ok && (c0.valid() || c1.valid())) {
            if (c0.valid()) {
                if (go0) {
                    ok = issue_pv(c0, s, pq0, dn0, kt0);
                    c0.next(p);
                }
                go0 = true;
                if (ok && c0.valid()) ok = issue_s(c0, s, qn0, kt0);
            }
            bs_swap(c0, c1);
            bs_swap(qn0, qn1);
            bs_swap(pq0, pq1);
            bs_swap(dn0, dn1);
            bs_swap(go0, go1);
            bs_swap(kt0, kt1);
            s ^= 1;
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
