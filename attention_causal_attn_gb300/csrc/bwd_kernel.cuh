// Backward pass of the fused RoPE + causal attention forward ("AttnFuse",
// sec. 4.4 Backward Pass: FlashAttention-2's split into a row-reduction
// kernel, a dK/dV kernel and a dQ kernel, each writing its own output tiles,
// with the softmax probabilities re-derived from the forward's per-row LSE).
//
// For a loss with gradient dO with respect to O:
//   P_ij  = exp2(S_ij * log2(e)/sqrt(D) - LSE_i * log2(e)),  S = Q' K'^T on the
//           rotated operands (rounded to fp16 as in the forward)
//   Dlt_i = dO_i . O_i                            (bwd_dot_kernel)
//   dS_ij = P_ij (dO_i . V_j - Dlt_i)
//   dV_j  = sum_i P_ij dO_i,  dK'_j = sum_i dS_ij Q'_i / sqrt(D)   (bwd_dkdv_kernel)
//   dQ'_i = sum_j dS_ij K'_j / sqrt(D)                              (bwd_dq_kernel)
//   dQ_i  = R(i)^T dQ'_i,  dK_j = R(j)^T dK'_j  (the rotation run backwards)
//
// Both tile kernels follow the forward's GB300 structure: TMA loads into
// 128-byte-swizzled shared memory, one converged warp issues tcgen05 MMAs
// into TMEM, and the elementwise warps (one thread per TMEM lane) turn S and
// dP into P and dS in TMEM, which the next MMAs read as their A operand.  Two
// warpgroups share that work, one per half of the 128 columns, each writing
// its packed P / dS inside its own half.  The elementwise work runs in two
// phases (P from S, then dS from dP and P), so each phase overlaps the tensor
// cores' next products (see the MMA issuers).  With RoPE, Q and K arrive
// rotated once by the rotation pass (prerot); the RoPE warps rotate tiles in
// place only when they do not.  Every wait is bounded.
#pragma once

#include "attn_fwd_kernel.cuh"

namespace attn {

struct BwdParams {
    FwdParams f;            // tm_q, tm_k, tm_v, the RoPE factor table, shape, scale, status, wait limit
    CUtensorMap tm_do;      // dO [B][S][Hq][D] bf16, box {64, 1, 128, 1}, 128-byte swizzle
    const float* lse;       // [B][Hq][S] natural log, from the forward
    const float* dlt;       // [B][Hq][S] dO_i . O_i
    __nv_bfloat16* dq;      // [B][S][Hq][D]
    __nv_bfloat16* dk;      // [B][S][Hkv][D]
    __nv_bfloat16* dv;      // [B][S][Hkv][D]
    const float2* rot_base; // (cos, sin)(32*m*theta_r), [m][r] (RoPE only)
    const float2* rot_row;  // (cos, sin)(rr*theta_r), [rr][r], rr < 32
    float inv_sqrt_d;
    // block mask (null: dense).  The dQ kernel walks row i's listed key tiles (CSR), the dK/dV
    // kernel key tile j's listed query tiles (the same mask by columns).
    const int* q_ptr;       // [ntiles + 1]
    const int* q_idx;
    const int* k_ptr;       // [ntiles + 1]
    const int* k_idx;
    // CTA order: 1 = a head's tiles together (they share the streamed tiles in L2; dense masks),
    // 0 = tile by tile across heads (a mask's heavy rows or columns first)
    int head_major;
    // RoPE: 1 = tm_q and tm_k hold Q and K already rotated (fp16, one rotation pass before the
    // kernels), so no tile is rotated inside the loops; 0 = the RoPE warps rotate each tile
    int prerot;
    // the local kernels (EXT): key j is visible to query i only if |i - j| < window (window > 0),
    // and alibi = 1 adds -m_h |i - j| to the score, as the local forward did
    int window;
    int alibi;
};

// A local tile's elementwise terms for one thread's 64 columns x: visible iff lo <= x < hi, and
// the score in log2 units gains -m2 |rel0 + sgn x| (the query - key distance of column x;
// m2 = m_h log2(e), 0 without ALiBi).
struct BwdLocal {
    int lo, hi;
    float m2, rel0, sgn;
};

// The ALiBi slope of query head h in log2 units, the local forward's expression.
__device__ __forceinline__ float bwd_alibi_m2(const BwdParams& p, int h) {
    return p.alibi ? exp2f(-8.f * static_cast<float>(h + 1) / static_cast<float>(p.f.Hq)) * 1.4426950408889634f
                   : 0.f;
}

// (tile, batch-head) of CTA x among bh batch-heads x ntiles tiles, in the order p.head_major picks.
__device__ __forceinline__ void bwd_cta_coords(const BwdParams& p, int bh, int ntiles, int& tile, int& bhi) {
    const long long x = blockIdx.x;
    if (p.head_major) {
        tile = static_cast<int>(x % ntiles);
        bhi = static_cast<int>(x / ntiles);
    } else {
        tile = static_cast<int>(x / bh);
        bhi = static_cast<int>(x % bh);
    }
}

// Dlt for every row i = (b, s, h): dO_i . O_i, dlt [B][H][S].  Each thread reads 16-byte pieces
// (8 values) of a row and the D/8 threads of a row add up through shuffles; a thread takes
// kDotPasses rows, one block row-count apart, and issues all their loads first, so that enough
// bytes are in flight per SM to stream O and dO at HBM rate.
constexpr int kDotPasses = 4;
template <int D>
__host__ __device__ constexpr int dot_rows_per_block() { return 256 / (D / 8) * kDotPasses; }

template <int D>
__global__ void __launch_bounds__(256) bwd_dot_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dO, float* __restrict__ dlt,
                                                      int B, int S, int H) {
    constexpr int kLanes = D / 8;              // threads per row
    constexpr int kRowsPerPass = 256 / kLanes;
    const long long nrows = static_cast<long long>(B) * S * H;
    const long long base = static_cast<long long>(blockIdx.x) * dot_rows_per_block<D>();
    const int sub = threadIdx.x % kLanes, rloc = threadIdx.x / kLanes;
    uint4 a[kDotPasses], b[kDotPasses];
#pragma unroll
    for (int k = 0; k < kDotPasses; ++k) {
        const long long row = base + k * kRowsPerPass + rloc;
        a[k] = b[k] = make_uint4(0u, 0u, 0u, 0u);
        if (row < nrows) {
            a[k] = __ldg(reinterpret_cast<const uint4*>(o + row * D) + sub);
            b[k] = __ldg(reinterpret_cast<const uint4*>(dO + row * D) + sub);
        }
    }
#pragma unroll
    for (int k = 0; k < kDotPasses; ++k) {
        const uint32_t av[4] = {a[k].x, a[k].y, a[k].z, a[k].w}, bv[4] = {b[k].x, b[k].y, b[k].z, b[k].w};
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = fmaf(bf16_lo(av[e]), bf16_lo(bv[e]), acc);
            acc = fmaf(bf16_hi(av[e]), bf16_hi(bv[e]), acc);
        }
#pragma unroll
        for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const long long row = base + k * kRowsPerPass + rloc;
        if (sub == 0 && row < nrows) {
            const long long h = row % H, s = (row / H) % S, bb = row / (static_cast<long long>(H) * S);
            dlt[(bb * H + h) * S + s] = acc;
        }
    }
}

// Warp roles of the two tile kernels (448 threads): warps 0-7 elementwise (two warpgroups, one per
// half of the columns), 8-11 RoPE, 12 TMA, 13 MMA.
constexpr int kBwdThreads = 448;
constexpr int kBwdEw = 256;
constexpr int kBwdWarpRope = 8;
constexpr int kBwdWarpTma = 12;
constexpr int kBwdWarpMma = 13;

// Shared memory of a tile kernel: two resident tiles, two stages of two streamed tiles, two
// stages of 2 x 128 per-row floats, then barriers and the abort flag / TMEM slot.
template <int D>
struct BwdLayout {
    static constexpr uint32_t kTile = 128u * D * 2u;
    static constexpr uint32_t kRes0 = 0, kRes1 = kTile;
    static constexpr uint32_t kStr0 = 2 * kTile;              // stage s: tiles at kStr0 + s * 2 * kTile (+ kTile)
    static constexpr uint32_t kRows = 6 * kTile;              // stage s: 256 floats at kRows + s * 1024
    static constexpr uint32_t kBars = kRows + 2048;
    static constexpr uint32_t kMisc = kBars + 256;
    static constexpr uint32_t kBytes = kMisc + 64;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // room to align the base to 1024 bytes
};

enum : int {
    BB_RES_FULL = 0,  // resident tiles landed
    BB_RES_ROT,       // resident RoPE tile rotated
    BB_STR_FULL,      // [2] streamed tiles landed
    BB_STR_ROT = BB_STR_FULL + 2,    // [2] streamed RoPE tile rotated
    BB_STR_EMPTY = BB_STR_ROT + 2,   // [2] the MMAs reading the stage are done
    BB_S_FULL = BB_STR_EMPTY + 2,    // S of the iteration in TMEM
    BB_P_FULL,        // P formed (dK/dV kernel: written to TMEM; dQ kernel: S read)
    BB_DP_FULL,       // dP of the iteration in TMEM
    BB_DS_FULL,       // dS written to TMEM
    BB_ACC_FULL,      // last accumulation done
    BB_DRAIN,
    BB_NUM
};
static_assert(BB_NUM * 8 <= 256, "barrier block");

// (cos, sin) of position pos for pairs r and r + 1 (r even), from the per-32-key factor tables.
__device__ __forceinline__ void bwd_factor2(const BwdParams& p, int pos, int r, int half, float4& f) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p.rot_base + static_cast<size_t>(pos >> 5) * half + r));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p.rot_row + static_cast<size_t>(pos & 31) * half + r));
    f = make_float4(a.x * b.x - a.y * b.y, a.y * b.x + a.x * b.y, a.z * b.z - a.w * b.w, a.w * b.z + a.z * b.w);
}

// Epilogue of one row held in TMEM columns [taddr, taddr + D): scale, rotate back by the row's
// position (RoPE), round to bf16 and store D contiguous elements at dst.
// zero: the tile saw no listed block; the row is 0 and TMEM is not read.
template <int D, bool ROPE>
__device__ __forceinline__ void bwd_store_row(const BwdParams& p, uint32_t taddr, float scale, int pos, bool store,
                                              __nv_bfloat16* dst, int c_begin = 0, int c_end = D / 2,
                                              bool zero = false) {
    constexpr int kHalf = D / 2;
#pragma unroll
    for (int c0 = 0; c0 < kHalf; c0 += 32) {
        if (c0 < c_begin || c0 >= c_end) continue;  // pairs [c_begin, c_end) of this thread's share
        uint32_t x[32], y[32];
        if (zero) {
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = y[e] = 0u;
        } else {
            tmem_load_32(taddr + c0, x);
            tmem_load_32(taddr + kHalf + c0, y);
        }
        uint32_t px[16], py[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            float x0 = __uint_as_float(x[e]) * scale, x1 = __uint_as_float(x[e + 1]) * scale;
            float y0 = __uint_as_float(y[e]) * scale, y1 = __uint_as_float(y[e + 1]) * scale;
            if (ROPE && store) {  // rows past S have no table entry and are not stored
                float4 f;
                bwd_factor2(p, pos, c0 + e, kHalf, f);  // (cos, sin) of pairs c0+e, c0+e+1
                const float a0 = x0 * f.x + y0 * f.y, b0 = -x0 * f.y + y0 * f.x;
                const float a1 = x1 * f.z + y1 * f.w, b1 = -x1 * f.w + y1 * f.z;
                x0 = a0;
                y0 = b0;
                x1 = a1;
                y1 = b1;
            }
            px[e / 2] = pack_bf16x2(x0, x1);
            py[e / 2] = pack_bf16x2(y0, y1);
        }
        if (store) {
            uint4* dx = reinterpret_cast<uint4*>(dst + c0);
            uint4* dy = reinterpret_cast<uint4*>(dst + kHalf + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                dx[q] = make_uint4(px[4 * q], px[4 * q + 1], px[4 * q + 2], px[4 * q + 3]);
                dy[q] = make_uint4(py[4 * q], py[4 * q + 1], py[4 * q + 2], py[4 * q + 3]);
            }
        }
    }
}

// The dK/dV kernel's elementwise work in two phases, so that each overlaps tensor-core work:
// the P phase needs only S^T, the dS phase only dP^T and P.  P phase: P^T = exp2(S^T c -
// LSE2_col) (0 where the query is before the key), packed to bf16 over the half's S^T columns
// (for dV) and kept in pp (for dS: the next S^T overwrites those columns meanwhile).
template <bool MASKED, bool LOCAL = false>
__device__ __forceinline__ void bwd_ew_p(uint32_t tS, const float* nls, float c, int lim, uint32_t (&pp)[32],
                                         const BwdLocal& lc = BwdLocal{0, 64, 0.f, 0.f, 1.f}) {
    // nls: -LSE2 of the half's 64 query columns (-inf for padded queries: P = 0)
    const uint64_t c2 = f2_pack(c, c);
    auto chunk = [&](const uint32_t (&rs)[32], int cc) {
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(nls + cc + e);
            float x0, x1, x2, x3;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(rs[e]), __uint_as_float(rs[e + 1])), c2, f2_pack(l4.x, l4.y)), x0, x1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(rs[e + 2]), __uint_as_float(rs[e + 3])), c2, f2_pack(l4.z, l4.w)),
                      x2, x3);
            if (LOCAL) {
                x0 = fmaf(-lc.m2, fabsf(fmaf(lc.sgn, static_cast<float>(cc + e), lc.rel0)), x0);
                x1 = fmaf(-lc.m2, fabsf(fmaf(lc.sgn, static_cast<float>(cc + e + 1), lc.rel0)), x1);
                x2 = fmaf(-lc.m2, fabsf(fmaf(lc.sgn, static_cast<float>(cc + e + 2), lc.rel0)), x2);
                x3 = fmaf(-lc.m2, fabsf(fmaf(lc.sgn, static_cast<float>(cc + e + 3), lc.rel0)), x3);
            }
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            if (MASKED) {
                if (cc + e < lim) p0 = 0.f;
                if (cc + e + 1 < lim) p1 = 0.f;
                if (cc + e + 2 < lim) p2 = 0.f;
                if (cc + e + 3 < lim) p3 = 0.f;
            }
            if (LOCAL) {
                if (cc + e < lc.lo || cc + e >= lc.hi) p0 = 0.f;
                if (cc + e + 1 < lc.lo || cc + e + 1 >= lc.hi) p1 = 0.f;
                if (cc + e + 2 < lc.lo || cc + e + 2 >= lc.hi) p2 = 0.f;
                if (cc + e + 3 < lc.lo || cc + e + 3 >= lc.hi) p3 = 0.f;
            }
            pp[(cc + e) / 2] = pack_bf16x2(p0, p1);
            pp[(cc + e) / 2 + 1] = pack_bf16x2(p2, p3);
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pp[cc / 2 + e];
        tmem_store_16(tS + cc / 2, pk);  // columns [cc/2, cc/2 + 16): never a column still to be read
    };
    // the second chunk's load is in flight while the first is processed
    uint32_t ra[32], rb[32];
    tmem_load_32(tS, ra);
    tmem_load_32_async(tS + 32, rb);
    chunk(ra, 0);
    tmem_wait_ld_32(rb);
    chunk(rb, 32);
}
// dS phase: dS^T = P^T (dP^T - Dlt_col) from the bf16 P^T of the P phase (the value dV
// accumulates), fp16 after RoPE, else bf16, over the half's dP^T columns.
template <bool ROPE>
__device__ __forceinline__ void bwd_ew_ds(uint32_t tdP, const float* dl, const uint32_t (&pp)[32]) {
    auto chunk = [&](const uint32_t (&rd)[32], int cc) {
        uint32_t pd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(dl + cc + e);
            const uint32_t pa = pp[(cc + e) / 2], pb = pp[(cc + e) / 2 + 1];
            float s0, s1, s2, s3;
            f2_unpack(f2_mul(f2_pack(bf16_lo(pa), bf16_hi(pa)),
                             f2_sub(f2_pack(__uint_as_float(rd[e]), __uint_as_float(rd[e + 1])), f2_pack(d4.x, d4.y))),
                      s0, s1);
            f2_unpack(f2_mul(f2_pack(bf16_lo(pb), bf16_hi(pb)),
                             f2_sub(f2_pack(__uint_as_float(rd[e + 2]), __uint_as_float(rd[e + 3])), f2_pack(d4.z, d4.w))),
                      s2, s3);
            pd[e / 2] = ROPE ? pack_f16x2(s0, s1) : pack_bf16x2(s0, s1);
            pd[e / 2 + 1] = ROPE ? pack_f16x2(s2, s3) : pack_bf16x2(s2, s3);
        }
        tmem_store_16(tdP + cc / 2, pd);
    };
    uint32_t ra[32], rb[32];
    tmem_load_32(tdP, ra);
    tmem_load_32_async(tdP + 32, rb);
    chunk(ra, 0);
    tmem_wait_ld_32(rb);
    chunk(rb, 32);
}

// The dQ kernel's elementwise work in the same two phases, one thread per query row and half of
// the columns (64 keys).  P phase: P = exp2(S c - LSE2_row), 0 for keys after the query (columns
// c > lim), kept in pp as bf16 (the P of the dK/dV kernel's dS, so both kernels form one dS).
template <bool MASKED, bool LOCAL = false>
__device__ __forceinline__ void bwd_ew_p_row(uint32_t tS, float l2, float c, int lim, uint32_t (&pp)[32],
                                             const BwdLocal& lc = BwdLocal{0, 64, 0.f, 0.f, 1.f}) {
    const uint64_t c2 = f2_pack(c, c), nl2 = f2_pack(-l2, -l2);  // -inf for a padded row: P = 0
    auto chunk = [&](const uint32_t (&rs)[32], int cc) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(rs[e]), __uint_as_float(rs[e + 1])), c2, nl2), x0, x1);
            if (LOCAL) {
                x0 = fmaf(-lc.m2, fabsf(fmaf(lc.sgn, static_cast<float>(cc + e), lc.rel0)), x0);
                x1 = fmaf(-lc.m2, fabsf(fmaf(lc.sgn, static_cast<float>(cc + e + 1), lc.rel0)), x1);
            }
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if (MASKED) {
                if (cc + e > lim) p0 = 0.f;
                if (cc + e + 1 > lim) p1 = 0.f;
            }
            if (LOCAL) {
                if (cc + e < lc.lo || cc + e >= lc.hi) p0 = 0.f;
                if (cc + e + 1 < lc.lo || cc + e + 1 >= lc.hi) p1 = 0.f;
            }
            pp[(cc + e) / 2] = pack_bf16x2(p0, p1);
        }
    };
    uint32_t ra[32], rb[32];
    tmem_load_32(tS, ra);
    tmem_load_32_async(tS + 32, rb);
    chunk(ra, 0);
    tmem_wait_ld_32(rb);
    chunk(rb, 32);
}
// dS phase: dS = P (dP - Dlt_row) over the half's dP columns (fp16 after RoPE, else bf16).
template <bool ROPE>
__device__ __forceinline__ void bwd_ew_ds_row(uint32_t tdP, float dl, const uint32_t (&pp)[32]) {
    const uint64_t dl2 = f2_pack(dl, dl);
    auto chunk = [&](const uint32_t (&rd)[32], int cc) {
        uint32_t pd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            const uint32_t pa = pp[(cc + e) / 2];
            float s0, s1;
            f2_unpack(f2_mul(f2_pack(bf16_lo(pa), bf16_hi(pa)),
                             f2_sub(f2_pack(__uint_as_float(rd[e]), __uint_as_float(rd[e + 1])), dl2)),
                      s0, s1);
            pd[e / 2] = ROPE ? pack_f16x2(s0, s1) : pack_bf16x2(s0, s1);
        }
        tmem_store_16(tdP + cc / 2, pd);
    };
    uint32_t ra[32], rb[32];
    tmem_load_32(tdP, ra);
    tmem_load_32_async(tdP + 32, rb);
    chunk(ra, 0);
    tmem_wait_ld_32(rb);
    chunk(rb, 32);
}

// TMEM column of k-step kk (16 rows of the streamed tile) of packed P / dS: each half of 64
// columns keeps its packed values in its own first 32 columns.
__device__ __forceinline__ uint32_t packed_col(int kk) { return static_cast<uint32_t>((kk / 4) * 64 + (kk % 4) * 8); }

// One K-major 128 x D tile (D/64 column blocks of [128 rows][128 B]): the descriptor units of k-step kk.
__device__ __forceinline__ uint32_t kmajor_units(int kk) {
    return static_cast<uint32_t>((kk / 4) * (kSubTileBytes >> 4) + (kk % 4) * 2);
}

__device__ __forceinline__ bool bwd_wait(uint32_t bar, uint32_t parity, const WaitCtl& ctl, int code) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, code));
}

// Every issued MMA completes before TMEM is released (bounded).
__device__ __forceinline__ void bwd_drain(uint32_t bar0, const WaitCtl& ctl) {
    tc_commit(bar_at(bar0, BB_DRAIN));
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar_at(bar0, BB_DRAIN), 0)) {
        if (global_timer_ns() - t0 > ctl.limit_ns) {
            atomicOr(ctl.status, kStatusDrain);
            break;
        }
    }
}

__device__ __forceinline__ void bwd_init_bars(uint32_t bar0) {
    mbar_init(bar_at(bar0, BB_RES_FULL), 1);
    mbar_init(bar_at(bar0, BB_RES_ROT), 128);
    for (int s = 0; s < 2; ++s) {
        mbar_init(bar_at(bar0, BB_STR_FULL + s), 1);
        mbar_init(bar_at(bar0, BB_STR_ROT + s), 128);
        mbar_init(bar_at(bar0, BB_STR_EMPTY + s), 1);
    }
    mbar_init(bar_at(bar0, BB_S_FULL), 1);
    mbar_init(bar_at(bar0, BB_P_FULL), kBwdEw);
    mbar_init(bar_at(bar0, BB_DP_FULL), 1);
    mbar_init(bar_at(bar0, BB_DS_FULL), kBwdEw);
    mbar_init(bar_at(bar0, BB_ACC_FULL), 1);
    mbar_init(bar_at(bar0, BB_DRAIN), 1);
    fence_barrier_init();
    fence_proxy_async_smem();
}

// dK and dV of one 128-key tile j of KV head g (CTA order: bwd_cta_coords) walk the query tiles
// i >= j (all of them without the causal mask) of each of the group's query heads.  With the
// head-major order the CTAs of one KV head run together and read the Q and dO tiles they all
// stream from L2 rather than HBM.
// TMEM: S^T [0,128), dP^T [128,256), dV [256, 256+D), dK [256+D, 256+2D).
template <int D, bool CAUSAL, bool ROPE, bool EXT = false>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using L = BwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smg = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sm = smem_addr(smg);
    const uint32_t bar0 = sm + L::kBars;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smg + L::kMisc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smg + L::kMisc + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const FwdParams& f = p.f;
    const int ntiles = (f.S + 127) / 128;
    int j, bg;
    bwd_cta_coords(p, f.B * f.Hkv, ntiles, j, bg);
    const int b = bg / f.Hkv, g = bg % f.Hkv;
    const int G = f.Hq / f.Hkv;
    const int kv0 = j * 128;
    const int i_lo = CAUSAL ? j : 0;
    const int lbase = p.k_ptr != nullptr ? p.k_ptr[j] : 0;
    const int per_head = p.k_ptr != nullptr ? p.k_ptr[j + 1] - lbase : ntiles - i_lo;
    const int iters = G * per_head;  // iteration it: head g*G + it / per_head, query tile qtile(it % per_head)
    auto qtile = [&](int x) { return p.k_ptr != nullptr ? p.k_idx[lbase + x] : i_lo + x; };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        bwd_init_bars(bar0);
    }
    if (warp == kBwdWarpTma && lane == 0) {
        tma_prefetch_desc(&f.tm_q);
        tma_prefetch_desc(&f.tm_k);
        tma_prefetch_desc(&f.tm_v);
        tma_prefetch_desc(&p.tm_do);
    }
    if (warp == kBwdWarpMma) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, f.status, f.wait_limit_ns};

    if (warp < 8) {
        // ---- elementwise warpgroups: thread t owns key row kv0 + t (TMEM lane t), columns 64 half ..
        const int t = threadIdx.x % 128, half = threadIdx.x / 128;
        const uint32_t trow = tmem + (static_cast<uint32_t>(t & ~31) << 16);
        const uint32_t tS = trow, tdP = trow + 128u, tdV = trow + 256u, tdK = trow + 256u + D;
        const float c = f.scale_log2;
        bool ok = true;
        for (int it = 0; it < iters && ok; ++it) {
            const int s = it & 1;
            const int q0 = qtile(it % per_head) * 128;
            ok = bwd_wait(bar_at(bar0, BB_STR_FULL + s), (it >> 1) & 1, ctl, kStatusSoftmax);  // per-column values
            if (!ok) break;
            ok = bwd_wait(bar_at(bar0, BB_S_FULL), it & 1, ctl, kStatusSoftmax);
            if (!ok) break;
            tc_fence_after();
            const float* ls = reinterpret_cast<const float*>(smg + L::kRows + s * 1024) + 64 * half;
            const int lim = kv0 + t - (q0 + 64 * half);  // query columns c < lim precede the key
            const uint32_t hS = tS + 64u * half, hdP = tdP + 64u * half;
            uint32_t pp[32];
            if constexpr (EXT) {
                // query column x is q0 + 64 half + x: its distance to the key is x - lim
                int lo = CAUSAL ? lim : -(1 << 30), hi = 1 << 30;
                if (p.window > 0) {
                    hi = lim + p.window;
                    if (!CAUSAL) lo = lim - p.window + 1;
                }
                const BwdLocal lc{lo, hi, bwd_alibi_m2(p, g * G + it / per_head), static_cast<float>(-lim), 1.f};
                if (p.alibi || __any_sync(0xffffffffu, lo > 0 || hi < 64))
                    bwd_ew_p<false, true>(hS, ls, c, 0, pp, lc);
                else
                    bwd_ew_p<false>(hS, ls, c, 0, pp);
            } else if (CAUSAL && __any_sync(0xffffffffu, lim > 0)) {
                bwd_ew_p<true>(hS, ls, c, lim, pp);
            } else {
                bwd_ew_p<false>(hS, ls, c, lim, pp);
            }
            tmem_store_wait();
            tc_fence_before();
            mbar_arrive(bar_at(bar0, BB_P_FULL));
            ok = bwd_wait(bar_at(bar0, BB_DP_FULL), it & 1, ctl, kStatusSoftmax);
            if (!ok) break;
            tc_fence_after();
            bwd_ew_ds<ROPE>(hdP, ls + 128, pp);
            tmem_store_wait();
            tc_fence_before();
            mbar_arrive(bar_at(bar0, BB_DS_FULL));
        }
        const bool none = iters == 0;  // no listed query tile: dK = dV = 0
        if (ok && (none || bwd_wait(bar_at(bar0, BB_ACC_FULL), 0, ctl, kStatusSoftmax))) {
            tc_fence_after();
            const int key = kv0 + t;
            const bool store = key < f.S;
            const size_t off = ((static_cast<size_t>(b) * f.S + (store ? key : 0)) * f.Hkv + g) * D;
            if (half == 0)
                bwd_store_row<D, false>(p, tdV, 1.0f, key, store, p.dv + off, 0, D / 2, none);
            else
                bwd_store_row<D, ROPE>(p, tdK, p.inv_sqrt_d, key, store, p.dk + off, 0, D / 2, none);
        }
    } else if (warp < kBwdWarpTma) {
        // ---- RoPE warps: the resident K tile once, then each streamed Q tile
        if (ROPE && !p.prerot) {
            const int t = threadIdx.x - kBwdWarpRope * 32;
            RopeConsts k;
            rope_load_consts<D>(f, t, k);
            uint64_t cb[4], sb[4];
            rope_load_base<D>(f, j, t, cb, sb);
            bool ok = bwd_wait(bar_at(bar0, BB_RES_FULL), 0, ctl, kStatusRope);
            if (ok) {
                rope_rotate_tile<D, false>(smg + L::kRes0, k, cb, sb, t);
                fence_proxy_async_smem();
                mbar_arrive(bar_at(bar0, BB_RES_ROT));
            }
            for (int it = 0; it < iters && ok; ++it) {
                const int s = it & 1;
                rope_load_base<D>(f, qtile(it % per_head), t, cb, sb);
                ok = bwd_wait(bar_at(bar0, BB_STR_FULL + s), (it >> 1) & 1, ctl, kStatusRope);
                if (!ok) break;
                rope_rotate_tile<D, false>(smg + L::kStr0 + s * 2 * L::kTile, k, cb, sb, t);
                fence_proxy_async_smem();
                mbar_arrive(bar_at(bar0, BB_STR_ROT + s));
            }
        }
    } else if (warp == kBwdWarpTma) {
        // ---- producer: K and V once; per iteration Q and dO by TMA, LSE2 and Dlt by the lanes
        if (lane == 0) {
            const uint32_t rb = bar_at(bar0, BB_RES_FULL);
            mbar_arrive_expect_tx(rb, 2 * L::kTile);
#pragma unroll
            for (int sub = 0; sub < D / 64; ++sub) {
                tma_load_4d(sm + L::kRes0 + sub * kSubTileBytes, &f.tm_k, rb, sub * 64, g, kv0, b);
                tma_load_4d(sm + L::kRes1 + sub * kSubTileBytes, &f.tm_v, rb, sub * 64, g, kv0, b);
            }
        }
        int armed = 0;  // streamed loads armed so far
        for (int it = 0; it < iters; ++it) {
            const int s = it & 1, n = it >> 1;
            const int h = g * G + it / per_head;
            const int q0 = qtile(it % per_head) * 128;
            // the tile's per-row values are read before the slot frees up, off the refill's path
            const float* lse_row = p.lse + (static_cast<size_t>(b) * f.Hq + h) * f.S;
            const float* dlt_row = p.dlt + (static_cast<size_t>(b) * f.Hq + h) * f.S;
            float lv[4], dv4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = q0 + lane + 32 * q;
                const bool in = r < f.S;
                lv[q] = in ? -(__ldg(lse_row + r) * 1.4426950408889634f) : -INFINITY;  // -LSE2; padded queries: P = 0
                dv4[q] = in ? __ldg(dlt_row + r) : 0.f;
            }
            if (n >= 1 && !bwd_wait(bar_at(bar0, BB_STR_EMPTY + s), (n - 1) & 1, ctl, kStatusProducer)) break;
            float* ls = reinterpret_cast<float*>(smg + L::kRows + s * 1024);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                ls[lane + 32 * q] = lv[q];
                ls[128 + lane + 32 * q] = dv4[q];
            }
            __syncwarp();
            if (lane == 0) {
                const uint32_t fb = bar_at(bar0, BB_STR_FULL + s);
                mbar_arrive_expect_tx(fb, 2 * L::kTile);
                const uint32_t dq = sm + L::kStr0 + s * 2 * L::kTile;
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub) {
                    tma_load_4d(dq + sub * kSubTileBytes, &f.tm_q, fb, sub * 64, h, q0, b);
                    tma_load_4d(dq + L::kTile + sub * kSubTileBytes, &p.tm_do, fb, sub * 64, h, q0, b);
                }
            }
            ++armed;
            __syncwarp();
        }
        // on the way out (loop ended or a wait gave up): every load has landed before the CTA may exit
        if (lane == 0) {
            mbar_drain(bar_at(bar0, BB_RES_FULL), 0, ctl, kStatusDrain);
            drain_ring(bar_at(bar0, BB_STR_FULL), 2, armed, ctl, kStatusDrain);
        }
        __syncwarp();
    } else if (warp == kBwdWarpMma) {  // the whole warp: one elected thread issues
        // ---- MMA issuer
        // S^T = K Q^T (A = K tile, B = Q tile, both K-major; fp16 after RoPE) and dP^T = V dO^T (bf16)
        const uint32_t kIdescS = umma_idesc_f16(ROPE ? 0u : 1u, 0u, 128, 128);
        constexpr uint32_t kIdescDP = umma_idesc_f16(1u, 0u, 128, 128);
        // dV += P^T dO and dK += dS^T Q: A from TMEM, B = the [queries][D] tile, MN-major
        constexpr uint32_t kIdescDV = umma_idesc_f16(1u, 1u, 128, D);
        const uint32_t kIdescDK = umma_idesc_f16(ROPE ? 0u : 1u, 1u, 128, D);
        const uint32_t tS = tmem, tdP = tmem + 128u, tdV = tmem + 256u, tdK = tmem + 256u + D;
        const uint64_t kdesc = sw128_desc(sm + L::kRes0, 16u, 1024u);
        const uint64_t vdesc = sw128_desc(sm + L::kRes1, 16u, 1024u);
        // Issue order dV(i), S^T(i+1), dK(i), dP^T(i+1): the elementwise warps turn dP^T(i) into
        // dS^T(i) while dV(i) and S^T(i+1) run, and S^T(i+1) into P^T(i+1) while dK(i) and
        // dP^T(i+1) run.  S^T(i+1) overwrites the columns of P^T(i) after dV(i) has read them,
        // dP^T(i+1) those of dS^T(i) after dK(i).
        auto stage_a = [&](int it) { return sm + L::kStr0 + (it & 1) * 2 * L::kTile; };  // Q; dO follows
        auto issue_s = [&](int it) -> bool {  // the stage's tiles, its rotated Q, then S^T = K Q^T
            const int s = it & 1, n = it >> 1;
            if (!mbar_wait_warp(bar_at(bar0, BB_STR_FULL + s), n & 1, ctl, kStatusMma)) return false;
            if (ROPE && !p.prerot) {
                if (it == 0 && !mbar_wait_warp(bar_at(bar0, BB_RES_ROT), 0, ctl, kStatusMma)) return false;
                if (!mbar_wait_warp(bar_at(bar0, BB_STR_ROT + s), n & 1, ctl, kStatusMma)) return false;
            }
            tc_fence_after();
            const uint64_t qdesc = sw128_desc(stage_a(it), 16u, 1024u);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_ss(tS, desc_advance(kdesc, kmajor_units(kk)), desc_advance(qdesc, kmajor_units(kk)), kIdescS,
                        kk > 0 ? 1u : 0u);
            tc_commit(bar_at(bar0, BB_S_FULL));
            return true;
        };
        auto issue_dp = [&](int it) {  // dP^T = V dO^T (the stage's tiles were waited for by issue_s)
            const uint64_t ddesc = sw128_desc(stage_a(it) + L::kTile, 16u, 1024u);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_ss(tdP, desc_advance(vdesc, kmajor_units(kk)), desc_advance(ddesc, kmajor_units(kk)), kIdescDP,
                        kk > 0 ? 1u : 0u);
            tc_commit(bar_at(bar0, BB_DP_FULL));
        };
        bool ok = mbar_wait_warp(bar_at(bar0, BB_RES_FULL), 0, ctl, kStatusMma);
        if (ok && iters > 0) {
            ok = issue_s(0);
            if (ok) issue_dp(0);
        }
        for (int it = 0; it < iters && ok; ++it) {
            const int s = it & 1;
            const uint32_t qa = stage_a(it), da = qa + L::kTile;
            const uint64_t dmn = sw128_desc(da, kSubTileBytes, 1024u), qmn = sw128_desc(qa, kSubTileBytes, 1024u);
            ok = mbar_wait_warp(bar_at(bar0, BB_P_FULL), it & 1, ctl, kStatusMma);
            if (!ok) break;
            tc_fence_after();
            // 16 queries per k-step: 2048 bytes of the tile, 8 TMEM columns of P^T / dS^T
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                umma_ts(tdV, tS + packed_col(kk), desc_advance(dmn, kk * 128u), kIdescDV, (it > 0 || kk > 0) ? 1u : 0u);
            if (it + 1 < iters && !(ok = issue_s(it + 1))) break;
            ok = mbar_wait_warp(bar_at(bar0, BB_DS_FULL), it & 1, ctl, kStatusMma);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                umma_ts(tdK, tdP + packed_col(kk), desc_advance(qmn, kk * 128u), kIdescDK, (it > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bar_at(bar0, BB_STR_EMPTY + s));
            if (it + 1 < iters) issue_dp(it + 1);
        }
        if (ok) tc_commit(bar_at(bar0, BB_ACC_FULL));
        bwd_drain(bar0, ctl);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kBwdWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// dQ of one 128-row query tile i of head h (CTA order: bwd_cta_coords) walks the key tiles j <= i
// (all of them without the causal mask); the heaviest tiles go first under the causal mask
// (i = ntiles-1-y).
// TMEM: S [0,128), dP [128,256), dQ [256, 256+D).
template <int D, bool CAUSAL, bool ROPE, bool EXT = false>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using L = BwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smg = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sm = smem_addr(smg);
    const uint32_t bar0 = sm + L::kBars;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smg + L::kMisc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smg + L::kMisc + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const FwdParams& f = p.f;
    const int ntiles = (f.S + 127) / 128;
    int y, bh;
    bwd_cta_coords(p, f.B * f.Hq, ntiles, y, bh);
    const int i = (CAUSAL && p.q_ptr == nullptr) ? ntiles - 1 - y : y;
    const int b = bh / f.Hq, h = bh % f.Hq;
    const int g = h / (f.Hq / f.Hkv);
    const int q0 = i * 128;
    const int lbase = p.q_ptr != nullptr ? p.q_ptr[i] : 0;
    const int iters = p.q_ptr != nullptr ? p.q_ptr[i + 1] - lbase : (CAUSAL ? i + 1 : ntiles);
    auto ktile = [&](int x) { return p.q_ptr != nullptr ? p.q_idx[lbase + x] : x; };  // key tile of iteration x

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        bwd_init_bars(bar0);
    }
    if (warp == kBwdWarpTma && lane == 0) {
        tma_prefetch_desc(&f.tm_q);
        tma_prefetch_desc(&f.tm_k);
        tma_prefetch_desc(&f.tm_v);
        tma_prefetch_desc(&p.tm_do);
    }
    if (warp == kBwdWarpMma) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, f.status, f.wait_limit_ns};

    if (warp < 8) {
        // ---- elementwise warpgroups: thread t owns query row q0 + t (TMEM lane t), columns 64 half ..
        const int t = threadIdx.x % 128, half = threadIdx.x / 128;
        const int row = q0 + t;
        const uint32_t trow = tmem + (static_cast<uint32_t>(t & ~31) << 16);
        const uint32_t tS = trow, tdP = trow + 128u, tdQ = trow + 256u;
        const float c = f.scale_log2;
        const size_t rix = (static_cast<size_t>(b) * f.Hq + h) * f.S + (row < f.S ? row : 0);
        const float l2 = row < f.S ? p.lse[rix] * 1.4426950408889634f : INFINITY;  // padded rows get P = 0
        const float dl = row < f.S ? p.dlt[rix] : 0.f;
        const float m2 = EXT ? bwd_alibi_m2(p, h) : 0.f;
        bool ok = true;
        for (int it = 0; it < iters && ok; ++it) {
            ok = bwd_wait(bar_at(bar0, BB_S_FULL), it & 1, ctl, kStatusSoftmax);
            if (!ok) break;
            tc_fence_after();
            const int lim = q0 + t - (ktile(it) * 128 + 64 * half);  // key columns c > lim follow the query
            const uint32_t hS = tS + 64u * half, hdP = tdP + 64u * half;
            uint32_t pp[32];
            if constexpr (EXT) {
                // key column x is ktile * 128 + 64 half + x: the query's distance to it is lim - x
                int lo = -(1 << 30), hi = CAUSAL ? lim + 1 : 1 << 30;
                if (p.window > 0) {
                    lo = lim - p.window + 1;
                    if (!CAUSAL) hi = lim + p.window;
                }
                const BwdLocal lc{lo, hi, m2, static_cast<float>(lim), -1.f};
                if (p.alibi || __any_sync(0xffffffffu, lo > 0 || hi < 64))
                    bwd_ew_p_row<false, true>(hS, l2, c, 0, pp, lc);
                else
                    bwd_ew_p_row<false>(hS, l2, c, 0, pp);
            } else if (CAUSAL && __any_sync(0xffffffffu, lim < 63)) {
                bwd_ew_p_row<true>(hS, l2, c, lim, pp);
            } else {
                bwd_ew_p_row<false>(hS, l2, c, lim, pp);
            }
            tc_fence_before();
            mbar_arrive(bar_at(bar0, BB_P_FULL));  // S is read: the next S may overwrite it
            ok = bwd_wait(bar_at(bar0, BB_DP_FULL), it & 1, ctl, kStatusSoftmax);
            if (!ok) break;
            tc_fence_after();
            bwd_ew_ds_row<ROPE>(hdP, dl, pp);
            tmem_store_wait();
            tc_fence_before();
            mbar_arrive(bar_at(bar0, BB_DS_FULL));
        }
        const bool none = iters == 0;  // no listed key tile: dQ = 0
        if (ok && (none || bwd_wait(bar_at(bar0, BB_ACC_FULL), 0, ctl, kStatusSoftmax))) {
            tc_fence_after();
            const bool store = row < f.S;
            const size_t off = ((static_cast<size_t>(b) * f.S + (store ? row : 0)) * f.Hq + h) * D;
            // each warpgroup stores its share of the row's pairs (all of them at D = 64: one share)
            if (D == 128 || half == 0)
                bwd_store_row<D, ROPE>(p, tdQ, p.inv_sqrt_d, row, store, p.dq + off, D == 128 ? 32 * half : 0,
                                       D == 128 ? 32 * half + 32 : D / 2, none);
        }
    } else if (warp < kBwdWarpTma) {
        // ---- RoPE warps: the resident Q tile once, then each streamed K tile
        if (ROPE && !p.prerot) {
            const int t = threadIdx.x - kBwdWarpRope * 32;
            RopeConsts k;
            rope_load_consts<D>(f, t, k);
            uint64_t cb[4], sb[4];
            rope_load_base<D>(f, i, t, cb, sb);
            bool ok = bwd_wait(bar_at(bar0, BB_RES_FULL), 0, ctl, kStatusRope);
            if (ok) {
                rope_rotate_tile<D, false>(smg + L::kRes0, k, cb, sb, t);
                fence_proxy_async_smem();
                mbar_arrive(bar_at(bar0, BB_RES_ROT));
            }
            for (int it = 0; it < iters && ok; ++it) {
                const int s = it & 1;
                rope_load_base<D>(f, ktile(it), t, cb, sb);
                ok = bwd_wait(bar_at(bar0, BB_STR_FULL + s), (it >> 1) & 1, ctl, kStatusRope);
                if (!ok) break;
                rope_rotate_tile<D, false>(smg + L::kStr0 + s * 2 * L::kTile, k, cb, sb, t);
                fence_proxy_async_smem();
                mbar_arrive(bar_at(bar0, BB_STR_ROT + s));
            }
        }
    } else if (warp == kBwdWarpTma) {
        // ---- producer: Q and dO once; per iteration K and V
        if (lane == 0) {
            const uint32_t rb = bar_at(bar0, BB_RES_FULL);
            mbar_arrive_expect_tx(rb, 2 * L::kTile);
#pragma unroll
            for (int sub = 0; sub < D / 64; ++sub) {
                tma_load_4d(sm + L::kRes0 + sub * kSubTileBytes, &f.tm_q, rb, sub * 64, h, q0, b);
                tma_load_4d(sm + L::kRes1 + sub * kSubTileBytes, &p.tm_do, rb, sub * 64, h, q0, b);
            }
            int armed = 0;  // streamed loads armed so far
            for (int it = 0; it < iters; ++it) {
                const int s = it & 1, n = it >> 1;
                if (n >= 1 && !mbar_wait(bar_at(bar0, BB_STR_EMPTY + s), (n - 1) & 1, ctl, kStatusProducer)) break;
                const uint32_t fb = bar_at(bar0, BB_STR_FULL + s);
                mbar_arrive_expect_tx(fb, 2 * L::kTile);
                const uint32_t ka = sm + L::kStr0 + s * 2 * L::kTile;
#pragma unroll
                for (int sub = 0; sub < D / 64; ++sub) {
                    tma_load_4d(ka + sub * kSubTileBytes, &f.tm_k, fb, sub * 64, g, ktile(it) * 128, b);
                    tma_load_4d(ka + L::kTile + sub * kSubTileBytes, &f.tm_v, fb, sub * 64, g, ktile(it) * 128, b);
                }
                ++armed;
            }
            // on the way out (loop ended or a wait gave up): every load has landed before the CTA may exit
            mbar_drain(bar_at(bar0, BB_RES_FULL), 0, ctl, kStatusDrain);
            drain_ring(bar_at(bar0, BB_STR_FULL), 2, armed, ctl, kStatusDrain);
        }
        __syncwarp();
    } else if (warp == kBwdWarpMma) {  // the whole warp: one elected thread issues
        // ---- MMA issuer: S = Q K^T, dP = dO V^T (K-major operands), then dQ += dS K (K tile MN-major)
        const uint32_t kIdescS = umma_idesc_f16(ROPE ? 0u : 1u, 0u, 128, 128);
        constexpr uint32_t kIdescDP = umma_idesc_f16(1u, 0u, 128, 128);
        const uint32_t kIdescDQ = umma_idesc_f16(ROPE ? 0u : 1u, 1u, 128, D);
        const uint32_t tS = tmem, tdP = tmem + 128u, tdQ = tmem + 256u;
        const uint64_t qdesc = sw128_desc(sm + L::kRes0, 16u, 1024u);
        const uint64_t ddesc = sw128_desc(sm + L::kRes1, 16u, 1024u);
        // Issue order S(j+1), dQ(j), dP(j+1): the elementwise warps form dS(j) while S(j+1) runs and
        // P(j+1) while dQ(j) and dP(j+1) run.  S(j+1) overwrites S(j) once P(j) is in registers,
        // dP(j+1) overwrites dS(j) after dQ(j) has read it.
        auto stage_a = [&](int it) { return sm + L::kStr0 + (it & 1) * 2 * L::kTile; };  // K; V follows
        auto issue_s = [&](int it) -> bool {  // the stage's tiles, its rotated K, then S = Q K^T
            const int s = it & 1, n = it >> 1;
            if (!mbar_wait_warp(bar_at(bar0, BB_STR_FULL + s), n & 1, ctl, kStatusMma)) return false;
            if (ROPE && !p.prerot) {
                if (it == 0 && !mbar_wait_warp(bar_at(bar0, BB_RES_ROT), 0, ctl, kStatusMma)) return false;
                if (!mbar_wait_warp(bar_at(bar0, BB_STR_ROT + s), n & 1, ctl, kStatusMma)) return false;
            }
            tc_fence_after();
            const uint64_t kdesc = sw128_desc(stage_a(it), 16u, 1024u);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_ss(tS, desc_advance(qdesc, kmajor_units(kk)), desc_advance(kdesc, kmajor_units(kk)), kIdescS,
                        kk > 0 ? 1u : 0u);
            tc_commit(bar_at(bar0, BB_S_FULL));
            return true;
        };
        auto issue_dp = [&](int it) {  // dP = dO V^T (the stage's tiles were waited for by issue_s)
            const uint64_t vdesc = sw128_desc(stage_a(it) + L::kTile, 16u, 1024u);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_ss(tdP, desc_advance(ddesc, kmajor_units(kk)), desc_advance(vdesc, kmajor_units(kk)), kIdescDP,
                        kk > 0 ? 1u : 0u);
            tc_commit(bar_at(bar0, BB_DP_FULL));
        };
        bool ok = mbar_wait_warp(bar_at(bar0, BB_RES_FULL), 0, ctl, kStatusMma);
        if (ok && iters > 0) {
            ok = issue_s(0);
            if (ok) issue_dp(0);
        }
        for (int it = 0; it < iters && ok; ++it) {
            const int s = it & 1;
            ok = mbar_wait_warp(bar_at(bar0, BB_P_FULL), it & 1, ctl, kStatusMma);
            if (!ok) break;
            if (it + 1 < iters && !(ok = issue_s(it + 1))) break;
            ok = mbar_wait_warp(bar_at(bar0, BB_DS_FULL), it & 1, ctl, kStatusMma);
            if (!ok) break;
            tc_fence_after();
            const uint64_t kmn = sw128_desc(stage_a(it), kSubTileBytes, 1024u);
            // 16 keys per k-step: 2048 bytes of K, 8 TMEM columns of dS
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                umma_ts(tdQ, tdP + packed_col(kk), desc_advance(kmn, kk * 128u), kIdescDQ, (it > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bar_at(bar0, BB_STR_EMPTY + s));
            if (it + 1 < iters) issue_dp(it + 1);
        }
        if (ok) tc_commit(bar_at(bar0, BB_ACC_FULL));
        bwd_drain(bar0, ctl);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kBwdWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace attn
