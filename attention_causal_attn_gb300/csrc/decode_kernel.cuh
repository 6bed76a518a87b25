// Split-KV decode: one query token per sequence (at position S-1) against a
// KV cache of S rows, with RoPE applied to K as it is loaded and an optional
// per-RoPE-pair distance window whose dropped pairs are never loaded.
// ("AttnFuse", sec. 4.2 Decode: the key range is split across blocks whose
// partial results merge through their log-sum-exp; "ATFlash", decode: the
// window becomes a predicate on the K loads.)
//
// Decode reads every K/V byte once and does a few FLOPs per byte, so it is
// bound by HBM; what the SM must keep low is the instruction count per byte.
// Kernel 1 (split): CTA (split * mtiles + mt, b * Hkv + g) covers keys
// [j0, j1) for query heads 16 mt .. 16 mt + 15 of KV head g (the warp-level
// MMA's 16 rows; heads past the group are zero rows).  Each warp walks 32-key
// tiles: cp.async stages the K and V tiles in XOR-swizzled shared memory (K of
// the next tile is fetched while this tile's P V runs), ldmatrix hands each
// lane its K fragment, the lane rotates its pairs in fp32 and rounds them to
// fp16 (the prefill's rounding of rotated operands), and mma.sync forms
// S = Q K^T; the online softmax runs on the accumulator fragment in log2
// units, whose bf16 P feeds the P V mma.sync directly (V through transposed
// ldmatrix).  The angle of key j and pair r is the product of a per-32-key
// factor (staged with each K tile) and a per-offset factor j % 32 (held in
// shared memory for the whole CTA).  The four warps' partials merge in
// shared memory, and the CTA writes one partial (m, log2 l, O / l) per head.
// Kernel 2 (combine): per (b, h), the splits' partials merge by their
// log-sum-exp.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace attn {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = 32 * kDecWarps;
constexpr int kDecMaxGroup = 32;  // query heads per KV head
constexpr int kDecTile = 32;      // keys per warp tile
constexpr int kDecHeads = 16;     // query heads per CTA (the MMA's M)
constexpr int kDecMaxParts = 1024;  // splits per row the combine kernel takes

struct DecodeParams {
    const __nv_bfloat16* q;   // [B][Hq][D]
    const __nv_bfloat16* k;   // [B][S][Hkv][D]
    const __nv_bfloat16* v;
    float* part_o;            // [B][Hq][nsplit][D]   O_i / l_i of each split
    float* part_ml;           // [B][Hq][nsplit][2]   (m_i, log2 l_i), scores in log2 units
    const float2* rot_base;   // (cos, sin)(32*m*theta_r), [m][r], or null (RoPE off)
    const float2* rot_row;    // (cos, sin)(rr*theta_r), [rr][r], rr < 32
    int B, Hq, Hkv, S, nsplit, split_len, mtiles;
    float scale_log2;         // log2(e) / sqrt(D)
    int win[64];              // W_r ascending (windowed decode)
};

// Dynamic shared memory of the split kernel: per warp a K and a V tile and the K tile's
// per-32-key angle factors, then the CTA's per-offset factors (rows padded by 64 bytes so that
// the 8 rows one load touches spread over both halves of the banks), then the window widths.
template <int D>
struct DecSmem {
    static constexpr int kTile = kDecTile * D * 2;
    static constexpr int kFac = D / 2 * 8;            // one row of (cos, sin) pairs
    static constexpr int kRowPitch = kFac + 64;
    static constexpr int kWarp = 2 * kTile + kFac;    // K tile, V tile, base factors
    static constexpr int kRows = kDecWarps * kWarp;   // offset of the per-offset factors
    static constexpr int kWin = kRows + kDecTile * kRowPitch;
    static constexpr int kBytes = kWin + 64 * 4;
};
template <int D>
constexpr int decode_smem_bytes() { return DecSmem<D>::kBytes; }

// Byte offset of 16-byte chunk c of row `row` in a tile of D bf16 per row; the chunk index is
// XORed with row % 8 so that the 8 rows an ldmatrix phase reads fall in distinct banks.
template <int D>
__device__ __forceinline__ uint32_t dec_tile_off(int row, int c) {
    return static_cast<uint32_t>(row * (D * 2) + ((c ^ (row & 7)) << 4));
}

// (cos, sin) of position pos for pair r from the two factor tables.
template <int HALF>
__device__ __forceinline__ float2 dec_factor(const DecodeParams& p, int pos, int r) {
    const float2 a = __ldg(p.rot_base + static_cast<size_t>(pos / kDecTile) * HALF + r);
    const float2 b = __ldg(p.rot_row + static_cast<size_t>(pos % kDecTile) * HALF + r);
    return make_float2(a.x * b.x - a.y * b.y, a.y * b.x + a.x * b.y);
}

// Number of pairs r with W_r < dist (W ascending): the pairs a key at that distance drops.
template <int HALF>
__device__ __forceinline__ int window_cut(const int* win, int dist) {
    int lo = 0, hi = HALF;  // first r with W_r >= dist lies in [lo, hi]
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (win[mid] < dist) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Stage rows [t0, t0 + 32) of one K or V tile (zero-filled past j1; with the window, K chunks
// whose 8 pairs all lie below the row's cut are zero-filled without being read).
template <int D, bool WIN>
__device__ __forceinline__ void dec_stage(uint32_t dst, const __nv_bfloat16* base, size_t row_stride, int t0, int j1,
                                          int lane, int rcut) {
    constexpr int kChunks = D / 8;
    static_assert(D == 64 || D == 128, "one or two rows per lane and copy");
    constexpr int kRowsPerCopy = 32 / kChunks;
#pragma unroll
    for (int i = 0; i < kDecTile / kRowsPerCopy; ++i) {
        const int row = i * kRowsPerCopy + lane / kChunks;
        const int ch = lane % kChunks;
        const bool ok = t0 + row < j1;
        uint32_t bytes = ok ? 16u : 0u;
        if (WIN) {
            const int rc = __shfl_sync(0xffffffffu, rcut, row);
            if ((ch % (kChunks / 2)) * 8 + 8 <= rc) bytes = 0u;
        }
        const __nv_bfloat16* src = base + static_cast<size_t>(ok ? t0 + row : t0) * row_stride + 8 * ch;
        cp_async_16(dst + dec_tile_off<D>(row, ch), src, bytes);
    }
}

template <int D, bool ROPE, bool WIN>
__global__ void __launch_bounds__(kDecThreads, 2) decode_split_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int kHalf = D / 2;
    constexpr int kSteps = D / 16;        // MMA k-steps over D
    constexpr int kPairSteps = kSteps / 2;  // k-step s pairs with s + kPairSteps (RoPE pairs r, r + D/2)
    constexpr int kChunks = D / 8;
    constexpr int kNT = kDecTile / 8;     // key n-tiles of S
    constexpr int kDT = D / 8;            // dimension n-tiles of O
    using L = DecSmem<D>;
    static_assert(!WIN || ROPE, "the window is defined on RoPE pairs");

    extern __shared__ __align__(128) uint8_t dsm[];
    int* win_s = reinterpret_cast<int*>(dsm + L::kWin);

    const int mt = blockIdx.x % p.mtiles, split = blockIdx.x / p.mtiles;
    const int b = blockIdx.y / p.Hkv, g = blockIdx.y % p.Hkv;
    const int G = p.Hq / p.Hkv;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int gr = lane >> 2, tq = lane & 3;  // fragment row and column pair
    const int j0 = split * p.split_len;
    const int j1 = min(p.S, j0 + p.split_len);
    const int qpos = p.S - 1;
    const uint32_t sbase = smem_addr(dsm);
    if (WIN)
        for (int i = threadIdx.x; i < 64; i += kDecThreads) win_s[i] = p.win[i];
    if (ROPE) {  // per-offset factors of the 32 keys of a tile, once per CTA
        constexpr int kRowChunks = L::kFac / 16;
        for (int i = threadIdx.x; i < kDecTile * kRowChunks; i += kDecThreads) {
            const int rr = i / kRowChunks, c = i % kRowChunks;
            cp_async_16(sbase + L::kRows + rr * L::kRowPitch + 16 * c,
                        reinterpret_cast<const uint8_t*>(p.rot_row) + rr * L::kFac + 16 * c, 16u);
        }
        cp_async_commit();
    }

    // Q as MMA A fragments: rows gr, gr + 8 of the head tile; columns 2tq, 2tq+1 (+8) of each k-step.
    // Rotated at position S-1 in fp32 and rounded to fp16 (bf16 as loaded when RoPE is off).
    uint32_t qa[kSteps][4];
#pragma unroll
    for (int s = 0; s < kPairSteps; ++s) {
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
            const int h = mt * kDecHeads + gr + 8 * hi;
            const __nv_bfloat16* qrow = p.q + (static_cast<size_t>(b) * p.Hq + g * G + min(h, G - 1)) * D;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float x[2], y[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = 16 * s + 8 * c + 2 * tq + e;
                    x[e] = h < G ? __bfloat162float(qrow[r]) : 0.f;
                    y[e] = h < G ? __bfloat162float(qrow[r + kHalf]) : 0.f;
                    if (ROPE) {
                        const float2 f = dec_factor<kHalf>(p, qpos, r);
                        const float xr = x[e] * f.x - y[e] * f.y;
                        y[e] = y[e] * f.x + x[e] * f.y;
                        x[e] = xr;
                    }
                }
                qa[s][hi + 2 * c] = ROPE ? pack_f16x2(x[0], x[1]) : pack_bf16x2(x[0], x[1]);
                qa[s + kPairSteps][hi + 2 * c] = ROPE ? pack_f16x2(y[0], y[1]) : pack_bf16x2(y[0], y[1]);
            }
        }
    }

    cp_async_wait<0>();
    __syncthreads();  // factors and window widths visible to every warp

    float o[kDT][4];
#pragma unroll
    for (int d = 0; d < kDT; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows gr and gr + 8

    const size_t row_stride = static_cast<size_t>(p.Hkv) * D;  // elements from one key to the next
    const __nv_bfloat16* kbase = p.k + (static_cast<size_t>(b) * p.S * p.Hkv + g) * D;
    const __nv_bfloat16* vbase = p.v + (static_cast<size_t>(b) * p.S * p.Hkv + g) * D;
    const uint32_t kt = sbase + static_cast<uint32_t>(warp * L::kWarp);
    const uint32_t vt = kt + L::kTile;
    const uint32_t fbase = vt + L::kTile;  // this warp's per-32-key factors of its current K tile
    const uint8_t* fbase_p = dsm + warp * L::kWarp + 2 * L::kTile;
    const uint8_t* frow_p = dsm + L::kRows;
    constexpr int kStride = kDecWarps * kDecTile;  // 128: a warp's next tile
    // the K tile's per-32-key factors ride in the K tile's copy group
    auto stage_factors = [&](int t) {
        if (ROPE && lane < L::kFac / 16)
            cp_async_16(fbase + 16 * lane,
                        reinterpret_cast<const uint8_t*>(p.rot_base + static_cast<size_t>(t / kDecTile) * kHalf) + 16 * lane,
                        16u);
    };

    int t0 = j0 + warp * kDecTile;
    int rcut = (WIN && t0 + lane < j1) ? window_cut<kHalf>(win_s, qpos - (t0 + lane)) : 0;  // key t0 + lane
    if (t0 < j1) {
        dec_stage<D, WIN>(kt, kbase, row_stride, t0, j1, lane, rcut);
        stage_factors(t0);
        cp_async_commit();
        dec_stage<D, false>(vt, vbase, row_stride, t0, j1, lane, 0);
        cp_async_commit();
    }
    for (; t0 < j1; t0 += kStride) {
        const bool more = t0 + kStride < j1;
        cp_async_wait<1>();  // this tile's K
        __syncwarp();

        // ---- S = Q K^T over the tile: n-tile nt holds keys 8nt .. 8nt+7, this lane's key 8nt + gr
        float sacc[kNT][4];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
        const int lrow = (lane & 7);  // ldmatrix row this lane addresses
        // with the window, k-step pairs (s, s + kPairSteps) whose 16 pairs every key of the tile
        // drops are skipped: their loads, rotations and MMAs would only add zeros
        // the next tile's cuts, ahead of the S arithmetic so that their lookups do not delay its K copy
        const int rcut_next =
            (WIN && t0 + kStride + lane < j1) ? window_cut<kHalf>(win_s, qpos - (t0 + kStride + lane)) : 0;
        const int s_lo = WIN ? __reduce_min_sync(0xffffffffu, static_cast<unsigned>(t0 + lane < j1 ? rcut : kHalf)) / 16
                             : 0;
#pragma unroll
        for (int s = 0; s < kPairSteps; ++s) {
            if (WIN && s < s_lo) continue;
            float4 fb[2];
            if (ROPE) {
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    fb[c] = *reinterpret_cast<const float4*>(fbase_p + 8 * (16 * s + 8 * c + 2 * tq));
            }
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                // matrices: x chunks 2s, 2s+1 and y chunks kChunks/2 + 2s, +1 of keys 8nt .. 8nt+7
                const int mi = lane >> 3;
                const int chunk = (mi >> 1) * (kChunks / 2) + 2 * s + (mi & 1);
                uint32_t w[4];
                ldmatrix_x4(kt + dec_tile_off<D>(8 * nt + lrow, chunk), w[0], w[1], w[2], w[3]);
                if (ROPE) {
                    const int n = 8 * nt + gr;  // this lane's key in the tile
                    const int rc = WIN ? __shfl_sync(0xffffffffu, rcut, n) : 0;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const float4 fr = *reinterpret_cast<const float4*>(frow_p + n * L::kRowPitch +
                                                                           8 * (16 * s + 8 * c + 2 * tq));
                        float xr[2], yr[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float ax = e ? fb[c].z : fb[c].x, ay = e ? fb[c].w : fb[c].y;
                            const float bx = e ? fr.z : fr.x, by = e ? fr.w : fr.y;
                            const float cs = ax * bx - ay * by, sn = ay * bx + ax * by;
                            const float x = e ? bf16_hi(w[c]) : bf16_lo(w[c]);
                            const float y = e ? bf16_hi(w[2 + c]) : bf16_lo(w[2 + c]);
                            xr[e] = x * cs - y * sn;
                            yr[e] = y * cs + x * sn;
                            if (WIN && 16 * s + 8 * c + 2 * tq + e < rc) xr[e] = yr[e] = 0.f;  // pair dropped
                        }
                        w[c] = pack_f16x2(xr[0], xr[1]);
                        w[2 + c] = pack_f16x2(yr[0], yr[1]);
                    }
                    mma_f16_16816(sacc[nt], qa[s], w[0], w[1]);
                    mma_f16_16816(sacc[nt], qa[s + kPairSteps], w[2], w[3]);
                } else {
                    mma_bf16_16816(sacc[nt], qa[s], w[0], w[1]);
                    mma_bf16_16816(sacc[nt], qa[s + kPairSteps], w[2], w[3]);
                }
            }
        }
        __syncwarp();  // every lane has read this tile's K
        // fetch the next tile's K behind the softmax and P V of this one
        if (more) {
            rcut = rcut_next;
            dec_stage<D, WIN>(kt, kbase, row_stride, t0 + kStride, j1, lane, rcut);
            stage_factors(t0 + kStride);
        }
        cp_async_commit();

        // ---- online softmax on the fragment: elements 0,1 are row gr, 2,3 row gr + 8; key 8nt + 2tq + (e & 1)
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool live = t0 + 8 * nt + 2 * tq + (e & 1) < j1;
                sacc[nt][e] = live ? sacc[nt][e] * p.scale_log2 : -INFINITY;
                if (e < 2) mx0 = fmaxf(mx0, sacc[nt][e]);
                else mx1 = fmaxf(mx1, sacc[nt][e]);
            }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: key t0 is live
        const float al0 = ex2_approx(m0 - mn0), al1 = ex2_approx(m1 - mn1);  // 0 on the first tile
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            sacc[nt][0] = ex2_approx(sacc[nt][0] - mn0);
            sacc[nt][1] = ex2_approx(sacc[nt][1] - mn0);
            sacc[nt][2] = ex2_approx(sacc[nt][2] - mn1);
            sacc[nt][3] = ex2_approx(sacc[nt][3] - mn1);
            ps0 += sacc[nt][0] + sacc[nt][1];
            ps1 += sacc[nt][2] + sacc[nt][3];
        }
        l0 = l0 * al0 + ps0;  // this lane's share of the row sums
        l1 = l1 * al1 + ps1;
#pragma unroll
        for (int d = 0; d < kDT; ++d) {
            o[d][0] *= al0;
            o[d][1] *= al0;
            o[d][2] *= al1;
            o[d][3] *= al1;
        }
        // P as A fragments: k-step ks covers keys 16ks .. 16ks+15 = S n-tiles 2ks, 2ks+1
        uint32_t pa[kNT / 2][4];
#pragma unroll
        for (int ks = 0; ks < kNT / 2; ++ks) {
            pa[ks][0] = pack_bf16x2(sacc[2 * ks][0], sacc[2 * ks][1]);
            pa[ks][1] = pack_bf16x2(sacc[2 * ks][2], sacc[2 * ks][3]);
            pa[ks][2] = pack_bf16x2(sacc[2 * ks + 1][0], sacc[2 * ks + 1][1]);
            pa[ks][3] = pack_bf16x2(sacc[2 * ks + 1][2], sacc[2 * ks + 1][3]);
        }

        // ---- O += P V (rows past j1 were zero-filled, and their P is 0)
        cp_async_wait<1>();  // this tile's V
        __syncwarp();
#pragma unroll
        for (int ks = 0; ks < kNT / 2; ++ks) {
#pragma unroll
            for (int dp = 0; dp < kDT / 2; ++dp) {
                // matrices: keys 16ks + {0..7, 8..15} of dimension chunks 2dp, 2dp+1
                const int key = 16 * ks + ((lane >> 3) & 1) * 8 + (lane & 7);
                const int chunk = 2 * dp + (lane >> 4);
                uint32_t r0, r1, r2, r3;
                ldmatrix_x4_trans(vt + dec_tile_off<D>(key, chunk), r0, r1, r2, r3);
                mma_bf16_16816(o[2 * dp], pa[ks], r0, r1);
                mma_bf16_16816(o[2 * dp + 1], pa[ks], r2, r3);
            }
        }
        __syncwarp();  // every lane has read this tile's V
        if (more) dec_stage<D, false>(vt, vbase, row_stride, t0 + kStride, j1, lane, 0);
        cp_async_commit();
    }
    cp_async_wait<0>();

    // ---- merge the four warps' partials in shared memory (the tiles are no longer needed)
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    constexpr int kOPitch = D + 8;  // floats per row of a warp's O
    float* o_s = reinterpret_cast<float*>(dsm);                                 // [warp][16][kOPitch]
    float* ml_s = reinterpret_cast<float*>(dsm + kDecWarps * kDecHeads * kOPitch * 4);  // [warp][16][2]
    static_assert(kDecWarps * kDecHeads * (kOPitch + 2) * 4 <= L::kRows, "merge fits in the tile space");
    __syncthreads();  // every warp is done with its tiles
    if (tq == 0) {
        ml_s[(warp * kDecHeads + gr) * 2] = m0;
        ml_s[(warp * kDecHeads + gr) * 2 + 1] = l0;
        ml_s[(warp * kDecHeads + gr + 8) * 2] = m1;
        ml_s[(warp * kDecHeads + gr + 8) * 2 + 1] = l1;
    }
    __syncthreads();
    // row maximum over the warps and each warp's weight 2^(m_w - M)
    auto row_max = [&](int row) {
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, ml_s[(w * kDecHeads + row) * 2]);
        return mm;
    };
    const float sc0 = ex2_approx(m0 - row_max(gr)), sc1 = ex2_approx(m1 - row_max(gr + 8));  // 0 for a warp without keys
#pragma unroll
    for (int d = 0; d < kDT; ++d) {
        *reinterpret_cast<float2*>(o_s + (warp * kDecHeads + gr) * kOPitch + 8 * d + 2 * tq) =
            make_float2(o[d][0] * sc0, o[d][1] * sc0);
        *reinterpret_cast<float2*>(o_s + (warp * kDecHeads + gr + 8) * kOPitch + 8 * d + 2 * tq) =
            make_float2(o[d][2] * sc1, o[d][3] * sc1);
    }
    __syncthreads();
    const int nsplit = p.nsplit;
    for (int idx = threadIdx.x; idx < kDecHeads * D; idx += kDecThreads) {
        const int row = idx / D, d = idx % D;
        const int h = mt * kDecHeads + row;
        if (h >= G) break;  // rows are visited in order
        const float mm = row_max(row);
        float lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
            lsum += ml_s[(w * kDecHeads + row) * 2 + 1] * ex2_approx(ml_s[(w * kDecHeads + row) * 2] - mm);
            acc += o_s[(w * kDecHeads + row) * kOPitch + d];
        }
        const size_t slot = (static_cast<size_t>(b) * p.Hq + g * G + h) * nsplit + split;
        p.part_o[slot * D + d] = acc / lsum;  // lsum > 0: the split holds at least its first key
        if (d == 0) {
            p.part_ml[2 * slot] = mm;
            p.part_ml[2 * slot + 1] = log2f(lsum);
        }
    }
}

// One CTA per (b, h): merge the splits' partials by their log-sum-exp (base 2).  The weights
// 2^(m_i + log2 l_i - max) go to shared memory; then thread t sums dimension t % D over every
// (128 / D)-th partial, eight partials in flight at a time.
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const float* __restrict__ part_o,
                                                             const float* __restrict__ part_ml,
                                                             __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                             int nparts) {
    constexpr int kGroups = 128 / D;  // threads per dimension
    __shared__ float w_s[kDecMaxParts];
    __shared__ float red[4];
    __shared__ float acc_s[kGroups][D];
    const int row = blockIdx.x;
    const int t = threadIdx.x, lane = t % 32, warp = t / 32;
    const float* ml = part_ml + static_cast<size_t>(row) * nparts * 2;
    float mx = -INFINITY;
    for (int i = t; i < nparts; i += 128) mx = fmaxf(mx, ml[2 * i] + ml[2 * i + 1]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    float ws = 0.f;
    for (int i = t; i < nparts; i += 128) {
        const float w = ex2_approx(ml[2 * i] + ml[2 * i + 1] - mx);
        w_s[i] = w;
        ws += w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, off);
    __syncthreads();  // red[] reads above are done before it is reused
    if (lane == 0) red[warp] = ws;
    __syncthreads();
    ws = red[0] + red[1] + red[2] + red[3];
    // O = sum_i w_i (O_i / l_i) / sum_i w_i
    const int d = t % D, grp = t / D;
    const float* po = part_o + static_cast<size_t>(row) * nparts * D + d;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int i = grp;
    for (; i + 7 * kGroups < nparts; i += 8 * kGroups) {
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = fmaf(w_s[i + u * kGroups], po[static_cast<size_t>(i + u * kGroups) * D], acc[u]);
    }
    for (; i < nparts; i += kGroups) acc[0] = fmaf(w_s[i], po[static_cast<size_t>(i) * D], acc[0]);
    acc_s[grp][d] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    __syncthreads();
    if (grp == 0) {
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < kGroups; ++q) sum += acc_s[q][d];
        o[static_cast<size_t>(row) * D + d] = __float2bfloat16(sum / ws);
        if (lse != nullptr && d == 0) lse[row] = (mx + log2f(ws)) * 0.69314718055994531f;
    }
}

}  // namespace attn
