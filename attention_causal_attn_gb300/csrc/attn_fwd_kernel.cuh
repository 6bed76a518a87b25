// Fused RoPE + causal attention forward for sm_103a (tcgen05 / TMEM / TMA).
//
// One persistent CTA per SM walks a host-built list of work units.  A unit is
// two 128-row query tiles ("stages") that share one KV head, so every K/V tile
// loaded into shared memory (and, with RoPE, every rotation of it) serves 256
// query rows:
//   - MHA: the two stages are consecutive query tiles of one head;
//   - GQA: the two stages are two query heads of one KV group at the same tile.
//
// Warp roles (16 warps = 4 warpgroups, registers rebalanced with setmaxnreg):
//   warps 0-3   softmax stage 0: online softmax on S0 in TMEM, P0 back to TMEM,
//               O0 rescale, epilogue (O/l -> bf16 -> global, LSE)
//   warps 4-7   softmax stage 1 (same, on S1/P1/O1)
//   warps 8-11  RoPE: rotate each loaded Q tile once and each loaded K tile in
//               place ("AttnFuse", sec. 4.1: Q rotated once before the loop, K
//               rotated tile by tile inside it), writing fp16 operands
//   warp 12     TMA producer: Q tiles, then K/V tiles from the diagonal down to
//               tile 0 ("Flash Attention: Causal Prefill D=128", reverse
//               traversal isolates the causal mask to the first tile)
//   warp 13     tcgen05 issuer (the converged warp, one elected thread issues;
//               one thread in the windowed variant) and TMEM owner
//   warps 14-15 idle (they complete the fourth warpgroup)
//
// TMEM (512 columns x 128 lanes x 32 bit): S0 [0,128), S1 [128,256), O0 [256,
// 256+D), O1 [384, 384+D).  P_s (bf16, two per column) overwrites the first 64
// columns of S_s once the softmax has read them; the PV product takes P from
// TMEM as its A operand.
//
// Per stage, the issue order is PV_s(n+1) then S_s(n): the next QK^T of a stage
// is queued behind the PV that reads its P, and the commit that reports S_s(n)
// also covers PV_s(n+1), so the softmax may rescale O_s as soon as S_s(n) is
// reported.  Softmax of one stage overlaps the tensor-core work of the other
// (FlashAttention-3 style ping-pong, "AttnFuse" sec. 7 / "Fused Kernels on
// Tensor Cores", FlashAttention-3 paragraph).
//
// Online softmax ("Flash Attention: Causal Prefill D=128", Online softmax):
// scores stay raw in TMEM; with c = log2(e)/sqrt(D), P = exp2(S*c - m*c),
// l = alpha*l + rowsum(P), O = alpha*O + P V, alpha = exp2((m_old - m_new)*c).
// The running max used for P is only moved (and O, l rescaled) when the true
// row max exceeds it by more than 16 in log2 units; P then stays below 2^16 and
// the final O/l and LSE = ln2*(m*c + log2 l) are unchanged up to rounding (P is
// bf16 and l, O accumulate in fp32, all with fp32's exponent range, so the
// bound only has to keep l * max|V| * S far below 2^128).
// That test is made per 32-key chunk with the maximum that tcgen05.ld.red
// (sm_103a) returns along with the chunk's scores, so each S tile is read from
// TMEM once: no separate max pass.
// One thread owns one query row (TMEM lane), so the row sums need no
// cross-lane reduction at all.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "host_tables.h"
#include "ptx.cuh"

namespace attn {

constexpr int kBlockM = 128;  // query rows per stage
constexpr int kBlockN = 128;  // keys per KV tile
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kNumThreads = 512;  // four warpgroups; launched at 128 registers per thread
constexpr int kWarpRope = 8;
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;
// Register split per warpgroup (softmax x2, RoPE, producer/MMA): the sum of
// 128 x budget over the four warpgroups must not exceed 512 x 128.
constexpr uint32_t kRegsSoftmax = 152, kRegsRope = 120, kRegsOther = 88;
static_assert(128 * (2 * kRegsSoftmax + kRegsRope + kRegsOther) <= kNumThreads * 128, "register split");
constexpr uint32_t kSubTileBytes = 128u * 128u;  // 128 rows x 128 B: one 64-wide bf16 column block
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 16.0f;  // log2 units

// status word bits (OR-ed by the CTA whose wait ran out)
constexpr int kStatusProducer = 1, kStatusRope = 2, kStatusMma = 4, kStatusSoftmax = 8, kStatusDrain = 16;
constexpr int kStatusTimeoutMask = 255;
// OR-ed by a row whose LSE came out non-finite: a score overflowed (with RoPE,
// a rotated Q or K value past the fp16 range) or an input was not finite
constexpr int kStatusNonFinite = 256;

struct FwdParams {
    CUtensorMap tm_q;  // [B][S][Hq][D] bf16, box {64, 1, 128, 1}, 128B swizzle
    CUtensorMap tm_k;  // [B][S][Hkv][D]
    CUtensorMap tm_v;
    CUtensorMap tm_k16; // K again, box {16, 1, 128, 1}, 32-byte swizzle (windowed variant: one 16-channel group per load)
    CUtensorMap tm_o;   // O [B][S][Hq][D] bf16, box {64, 1, 32, 1}, 128B swizzle: one warp's rows of one 64-channel block
    __nv_bfloat16* o;   // [B][S][Hq][D]
    float* lse;         // [B][Hq][S] or null
    const float2* rope; // RoPE factor tables (see RopeGeom), null when RoPE is off
    const uint2* tasks; // unit words, see decode_unit
    const int* task_off;// [gridDim.x + 1]: CTA c runs tasks[task_off[c] .. task_off[c+1])
    int* status;
    int B, Hq, Hkv, S;
    float scale_log2;   // log2(e) / sqrt(D)
    unsigned long long wait_limit_ns;
    int win[64];        // W_r = floor(k * 2*pi / theta_r), ascending in r (windowed variant)
    int qk_f16;         // without in-kernel RoPE: Q and K hold fp16 (already rotated) rather than bf16
    const short2* wtab; // windowed variant, per tile distance: (first pair kept at the tile's smallest distance,
                        // first pair kept at its largest), see window_tile
    int test_no_loads;  // test mode for the bounded waits: the producer issues nothing, so every
                        // consumer's first wait runs out after wait_limit_ns (0 in every real launch)
};

// barrier slots
enum : int {
    BAR_Q_FULL = 0,   // [2] TMA landed Q_s
    BAR_Q_ROT = 2,    // [2] Q_s rotated (RoPE)
    BAR_Q_EMPTY = 4,  // [2] last QK^T of the unit read Q_s
    BAR_K_FULL = 6,   // [kKStages]
    BAR_K_ROT = BAR_K_FULL + kKStages,
    BAR_K_EMPTY = BAR_K_ROT + kKStages,
    BAR_V_FULL = BAR_K_EMPTY + kKStages,  // [kVStages]
    BAR_V_EMPTY = BAR_V_FULL + kVStages,
    BAR_S_FULL = BAR_V_EMPTY + kVStages,  // [2] S_s(n) in TMEM (and PV_s(n+1) done)
    BAR_P_FULL = BAR_S_FULL + 2,          // [2] P_s(n) in TMEM, O_s rescaled
    BAR_O_FULL = BAR_P_FULL + 2,          // [2] last PV of the unit done
    BAR_O_FREE = BAR_O_FULL + 2,          // [2] epilogue finished reading O_s
    BAR_DRAIN = BAR_O_FREE + 2,
    NUM_BARS = BAR_DRAIN + 1
};

// Output staging for the TMA-store epilogue: per stage, one [32 rows][128 B]
// block (64 channels, 128-byte swizzle) per warp of the softmax warpgroup.
constexpr uint32_t kEpiWarpBytes = 32u * 128u;
constexpr uint32_t kEpiStageBytes = 4u * kEpiWarpBytes;

template <int D>
struct SmemLayout {
    static constexpr uint32_t kTileBytes = 128u * D * 2u;
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + 2 * kTileBytes;
    static constexpr uint32_t kV = kK + kKStages * kTileBytes;
    static constexpr uint32_t kO = kV + kVStages * kTileBytes;  // 1024-byte aligned (tiles are multiples of 16 KB)
    static constexpr uint32_t kBars = kO + 2 * kEpiStageBytes;
    static constexpr uint32_t kMisc = kBars + 8 * NUM_BARS;
    static constexpr uint32_t kBytes = kMisc + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

struct Unit {
    int b, kvh;
    int h[2], row0[2], nhi[2];
    bool valid[2];
    int nmax;
};

// Unit word: x = qtile0 | qtile1 << 16 (0xFFFF = no stage), y = h0 | h1 << 8 | b << 16.
__device__ __forceinline__ Unit decode_unit(uint2 w, const FwdParams& p, bool causal) {
    Unit u;
    const int qt[2] = {static_cast<int>(w.x & 0xFFFFu), static_cast<int>(w.x >> 16)};
    u.h[0] = static_cast<int>(w.y & 0xFFu);
    u.h[1] = static_cast<int>((w.y >> 8) & 0xFFu);
    u.b = static_cast<int>(w.y >> 16);
    u.kvh = u.h[0] / (p.Hq / p.Hkv);
    const int last_tile = (p.S - 1) / kBlockN;
    u.nmax = -1;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        u.valid[s] = qt[s] != 0xFFFF && qt[s] * kBlockM < p.S;
        u.row0[s] = qt[s] * kBlockM;
        u.nhi[s] = causal ? qt[s] : last_tile;
        if (u.valid[s] && u.nhi[s] > u.nmax) u.nmax = u.nhi[s];
    }
    return u;
}

__device__ __forceinline__ uint32_t bar_at(uint32_t bar0, int i) { return bar0 + 8u * static_cast<uint32_t>(i); }

// ------------------------------------------------------------------ window geometry
// Per-RoPE-pair window ("ATFlash", The idea): pair r of cell (i, j) is kept
// iff the distance i - j <= W_r.  W_r grows with r, so the pairs a cell drops
// are a prefix.  Query tile qt against key tile n covers distances
// 128*(qt-n) - 127 .. 128*(qt-n) + 127, so the bounds depend on the tile
// distance qt - n only; the host tabulates, per tile distance,
//   .x = first pair kept at the tile's smallest distance (pairs below are
//        dropped for every cell),
//   .y = first pair kept at its largest distance (pairs from here on are kept
//        for every cell); pairs in [.x, .y) are the tile's boundary pairs.
//
// Pairs below z are dropped for every cell of the KV tile against every query
// tile of the unit.  The windowed variant holds K as D/16 groups of 16
// channels (one K=16 MMA step each, 32-byte swizzle); the 16-pair blocks below
// m0 = z / 16 are never loaded, rotated nor multiplied (block m is channel
// groups m and m + D/32: the pairs' first and second members), and the pairs
// of block m0 below z are zeroed in shared memory by the rotation.
struct WinTile {
    int z, m0;
};
template <int D>
__device__ __forceinline__ WinTile window_tile(const FwdParams& p, const Unit& u, int n) {
    // only the stages that visit key tile n count (n <= nhi, so the tile distance is >= 0)
    int z = D / 2;
#pragma unroll
    for (int s = 0; s < 2; ++s)
        if (u.valid[s] && n <= u.nhi[s]) z = min(z, static_cast<int>(p.wtab[u.row0[s] / kBlockM - n].x));
    WinTile w;
    w.z = z;
    w.m0 = min(z / 16, D / 32 - 1);
    return w;
}

// ------------------------------------------------------------------ producer
// Issues the CTA's Q, K and V loads; kit, vit, qit count the loads armed so far.
template <int D, bool WINDOW>
__device__ void producer_issue(const FwdParams& p, bool causal, uint32_t sm, uint32_t bar0, int t_begin, int t_end,
                               const WaitCtl& ctl, int& kit, int& vit, int (&qit)[2]) {
    using L = SmemLayout<D>;
    for (int ti = t_begin; ti < t_end; ++ti) {
        const Unit u = decode_unit(p.tasks[ti], p, causal);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (!u.valid[s]) continue;
            if (!mbar_wait(bar_at(bar0, BAR_Q_EMPTY + s), (qit[s] & 1) ^ 1, ctl, kStatusProducer)) return;
            const uint32_t fb = bar_at(bar0, BAR_Q_FULL + s);
            mbar_arrive_expect_tx(fb, L::kTileBytes);
            for (int sub = 0; sub < D / 64; ++sub)
                tma_load_4d(sm + L::kQ + s * L::kTileBytes + sub * kSubTileBytes, &p.tm_q, fb, sub * 64, u.h[s],
                            u.row0[s], u.b);
            ++qit[s];
        }
        for (int n = u.nmax; n >= 0; --n) {
            const int ks = kit % kKStages;
            const WinTile w = WINDOW ? window_tile<D>(p, u, n) : WinTile{0, 0};  // before the wait: load in flight
            if (!mbar_wait(bar_at(bar0, BAR_K_EMPTY + ks), ((kit / kKStages) & 1) ^ 1, ctl, kStatusProducer)) return;
            const uint32_t kb = bar_at(bar0, BAR_K_FULL + ks);
            if (WINDOW) {
                // only the 16-pair blocks with a kept pair: 16 channels x 128 rows = 4 KB per group, two per block
                constexpr int kBlocks = D / 32;
                mbar_arrive_expect_tx(kb, static_cast<uint32_t>(2 * (kBlocks - w.m0)) * 4096u);
                for (int m = w.m0; m < kBlocks; ++m) {
                    tma_load_4d(sm + L::kK + ks * L::kTileBytes + m * 4096u, &p.tm_k16, kb, 16 * m, u.kvh,
                                n * kBlockN, u.b);
                    tma_load_4d(sm + L::kK + ks * L::kTileBytes + (m + kBlocks) * 4096u, &p.tm_k16, kb,
                                D / 2 + 16 * m, u.kvh, n * kBlockN, u.b);
                }
            } else {
                mbar_arrive_expect_tx(kb, L::kTileBytes);
                for (int sub = 0; sub < D / 64; ++sub)
                    tma_load_4d(sm + L::kK + ks * L::kTileBytes + sub * kSubTileBytes, &p.tm_k, kb, sub * 64, u.kvh,
                                n * kBlockN, u.b);
            }
            ++kit;
            const int vs = vit % kVStages;
            if (!mbar_wait(bar_at(bar0, BAR_V_EMPTY + vs), ((vit / kVStages) & 1) ^ 1, ctl, kStatusProducer)) return;
            const uint32_t vb = bar_at(bar0, BAR_V_FULL + vs);
            mbar_arrive_expect_tx(vb, L::kTileBytes);
            for (int sub = 0; sub < D / 64; ++sub)
                tma_load_4d(sm + L::kV + vs * L::kTileBytes + sub * kSubTileBytes, &p.tm_v, vb, sub * 64, u.kvh,
                            n * kBlockN, u.b);
            ++vit;
        }
    }
}

template <int D, bool WINDOW>
__device__ void producer_role(const FwdParams& p, bool causal, uint32_t sm, uint32_t bar0, int t_begin, int t_end,
                              const WaitCtl& ctl) {
    int kit = 0, vit = 0;
    int qit[2] = {0, 0};
    if (!p.test_no_loads) producer_issue<D, WINDOW>(p, causal, sm, bar0, t_begin, t_end, ctl, kit, vit, qit);
    // On the way out, whether the loop ended or a wait gave up: the last load of
    // every slot has landed before the CTA may exit (the earlier ones were consumed).
#pragma unroll
    for (int s = 0; s < 2; ++s) drain_ring(bar_at(bar0, BAR_Q_FULL + s), 1, qit[s], ctl, kStatusDrain);
    drain_ring(bar_at(bar0, BAR_K_FULL), kKStages, kit, ctl, kStatusDrain);
    drain_ring(bar_at(bar0, BAR_V_FULL), kVStages, vit, ctl, kStatusDrain);
}

// ------------------------------------------------------------------ RoPE
// Rotation of one 128-row tile in place.  Q and K tiles are stored as D/64
// column blocks of [128 rows][128 B] with the 128-byte swizzle (16-byte chunk
// c of row r sits at chunk c ^ (r & 7)).  Pair (r, r + D/2) has both members
// at the same swizzled offset in column blocks 0 and 1 for D = 128, and in
// chunks c and c + 4 of the single block for D = 64, so each thread rotates
// whole pairs from two 16-byte loads.  The windowed variant stores K as D/16
// channel groups of [128 rows][32 B] with the 32-byte swizzle (group g at
// g * 4 KB; the 16-byte half h of row r sits at half h ^ ((r >> 2) & 1)), so
// that dropped groups are never loaded.  Input bf16, math fp32, output fp16.
//
// Thread t owns chunk c = t / kRows (pairs 8c..8c+7) of rows rr + kRows*i,
// rr = t % kRows: eight consecutive threads touch eight rows of one chunk,
// which is free of bank conflicts in both layouts.  Angles come from the angle-addition rule, as complex
// numbers: the angle of row pos0 + rr is base(pos0) * rowfac(rr), with
// base(pos0) = (cos, sin)(pos0 theta) read once per tile, and each pass
// advances it by step = (cos, sin)(kRows theta).  The host computes every
// factor in float64; the recurrence adds a few float32 ulps.  Pairs are
// processed two at a time in packed fp32x2 arithmetic.
template <int D>
struct RopeGeom {
    static constexpr int kHalf = D / 2;
    static constexpr int kChunks = kHalf / 8;     // 16-byte chunks per half row
    static constexpr int kRows = 128 / kChunks;   // rows covered by one pass of the 128 threads
    static constexpr int kIters = kChunks;        // passes per 128-row tile
    static_assert(kRows == attn_host::rope_rows_per_pass(D), "host factor table must match the rotating threads");
    static_assert(kRows * kIters == 128, "passes must cover the tile");
};

// Table layout (float2 = (cos, sin)): base[ntiles][D/2] | rowfac[kRows][D/2] | step[D/2].
// Packed pairs of pairs: element q holds pairs (8c + 2q, 8c + 2q + 1).
struct RopeConsts {
    uint64_t cr[4], sr[4];  // rowfac of this thread's rr
    uint64_t cs[4], ss[4];  // step
};

__device__ __forceinline__ void load8_packed(const float2* src, uint64_t (&c)[4], uint64_t (&s)[4]) {
    const float4* p4 = reinterpret_cast<const float4*>(src);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float4 v = __ldg(p4 + k);  // (cos, sin) of pairs 2k and 2k+1
        c[k] = f2_pack(v.x, v.z);
        s[k] = f2_pack(v.y, v.w);
    }
}

template <int D>
__device__ __forceinline__ void rope_load_consts(const FwdParams& p, int t, RopeConsts& k) {
    using G = RopeGeom<D>;
    const int ntiles = (p.S + kBlockM - 1) / kBlockM;
    const int c = t / G::kRows, rr = t % G::kRows;
    load8_packed(p.rope + (static_cast<size_t>(ntiles) + rr) * G::kHalf + 8 * c, k.cr, k.sr);
    load8_packed(p.rope + (static_cast<size_t>(ntiles) + G::kRows) * G::kHalf + 8 * c, k.cs, k.ss);
}

template <int D>
__device__ __forceinline__ void rope_load_base(const FwdParams& p, int tile, int t, uint64_t (&cb)[4],
                                               uint64_t (&sb)[4]) {
    using G = RopeGeom<D>;
    load8_packed(p.rope + static_cast<size_t>(tile) * G::kHalf + 8 * (t / G::kRows), cb, sb);
}

// (c, s) <- (c, s) * (fc, fs) as complex numbers, two pairs per operand.
__device__ __forceinline__ void cmul2(uint64_t& c, uint64_t& s, uint64_t fc, uint64_t fs) {
    const uint64_t nc = f2_sub(f2_mul(c, fc), f2_mul(s, fs));
    s = f2_fma(s, fc, f2_mul(c, fs));
    c = nc;
}

// LAYOUT_GROUPS: the windowed K layout; pairs below `zero_below` come out as 0.
template <int D, bool LAYOUT_GROUPS>
__device__ __forceinline__ void rope_rotate_tile(uint8_t* tile, const RopeConsts& k, uint64_t (&cb)[4],
                                                 uint64_t (&sb)[4], int t, int zero_below = 0) {
    using G = RopeGeom<D>;
    const int c = t / G::kRows, rr = t % G::kRows;
    // angle of this thread's first row
#pragma unroll
    for (int q = 0; q < 4; ++q) cmul2(cb[q], sb[q], k.cr[q], k.sr[q]);
#pragma unroll 2
    for (int i = 0; i < G::kIters; ++i) {
        const int row = rr + G::kRows * i;
        uint32_t lo_off, hi_off;
        if (LAYOUT_GROUPS) {
            const uint32_t half = static_cast<uint32_t>(((c & 1) ^ ((row >> 2) & 1)) << 4);
            lo_off = static_cast<uint32_t>((c >> 1) * 4096 + row * 32) + half;
            hi_off = lo_off + static_cast<uint32_t>(G::kChunks / 2 * 4096);
        } else if (D == 128) {
            lo_off = static_cast<uint32_t>(row * 128 + ((c ^ (row & 7)) << 4));
            hi_off = lo_off + kSubTileBytes;
        } else {
            lo_off = static_cast<uint32_t>(row * 128 + ((c ^ (row & 7)) << 4));
            hi_off = static_cast<uint32_t>(row * 128 + (((c + 4) ^ (row & 7)) << 4));
        }
        const uint4 lo = *reinterpret_cast<const uint4*>(tile + lo_off);
        const uint4 hi = *reinterpret_cast<const uint4*>(tile + hi_off);
        const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w};
        const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w};
        uint32_t lo_out[4], hi_out[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint64_t x = f2_pack(bf16_lo(lw[q]), bf16_hi(lw[q]));
            const uint64_t y = f2_pack(bf16_lo(hw[q]), bf16_hi(hw[q]));
            float a0, a1, b0, b1;
            f2_unpack(f2_sub(f2_mul(x, cb[q]), f2_mul(y, sb[q])), a0, a1);  // x cos - y sin
            f2_unpack(f2_fma(y, cb[q], f2_mul(x, sb[q])), b0, b1);           // y cos + x sin
            lo_out[q] = pack_f16x2(a0, a1);
            hi_out[q] = pack_f16x2(b0, b1);
            if (LAYOUT_GROUPS) {  // pairs 8c+2q, 8c+2q+1 below zero_below are dropped
                const int pr = 8 * c + 2 * q;
                const uint32_t keep = (pr >= zero_below ? 0x0000FFFFu : 0u) | (pr + 1 >= zero_below ? 0xFFFF0000u : 0u);
                lo_out[q] &= keep;
                hi_out[q] &= keep;
            }
        }
        *reinterpret_cast<uint4*>(tile + lo_off) = make_uint4(lo_out[0], lo_out[1], lo_out[2], lo_out[3]);
        *reinterpret_cast<uint4*>(tile + hi_off) = make_uint4(hi_out[0], hi_out[1], hi_out[2], hi_out[3]);
#pragma unroll
        for (int q = 0; q < 4; ++q) cmul2(cb[q], sb[q], k.cs[q], k.ss[q]);
    }
}

template <int D, bool WINDOW>
__device__ void rope_role(const FwdParams& p, bool causal, uint8_t* smg, uint32_t bar0, int t_begin, int t_end,
                          const WaitCtl& ctl, int t) {
    using L = SmemLayout<D>;
    RopeConsts k;
    rope_load_consts<D>(p, t, k);
    int kit = 0;
    int qit[2] = {0, 0};
    uint64_t cb[4], sb[4];
    for (int ti = t_begin; ti < t_end; ++ti) {
        const Unit u = decode_unit(p.tasks[ti], p, causal);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (!u.valid[s]) continue;
            rope_load_base<D>(p, u.row0[s] / kBlockM, t, cb, sb);
            if (!__all_sync(0xffffffffu, mbar_wait(bar_at(bar0, BAR_Q_FULL + s), qit[s] & 1, ctl, kStatusRope)))
                return;
            rope_rotate_tile<D, false>(smg + L::kQ + s * L::kTileBytes, k, cb, sb, t);
            fence_proxy_async_smem();
            mbar_arrive(bar_at(bar0, BAR_Q_ROT + s));
            ++qit[s];
        }
        for (int n = u.nmax; n >= 0; --n) {
            const int ks = kit % kKStages;
            rope_load_base<D>(p, n, t, cb, sb);
            const WinTile w = WINDOW ? window_tile<D>(p, u, n) : WinTile{0, 0};  // before the wait: load in flight
            if (!__all_sync(0xffffffffu,
                            mbar_wait(bar_at(bar0, BAR_K_FULL + ks), (kit / kKStages) & 1, ctl, kStatusRope)))
                return;
            if (WINDOW) {
                using G = RopeGeom<D>;
                const int c = t / G::kRows;
                // chunk c (pairs 8c..8c+7) is in 16-pair block c / 2; the blocks below m0 were not
                // loaded and are not multiplied, and the pairs of block m0 below z are zeroed
                if (c / 2 >= w.m0) rope_rotate_tile<D, true>(smg + L::kK + ks * L::kTileBytes, k, cb, sb, t, w.z);
            } else {
                rope_rotate_tile<D, false>(smg + L::kK + ks * L::kTileBytes, k, cb, sb, t);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar_at(bar0, BAR_K_ROT + ks));
            ++kit;
        }
    }
}

// ------------------------------------------------------------------ MMA issuer
// Issuer form: the whole warp runs the loop and one elected thread issues,
// so the warp stays converged; the alternative runs the loop on one thread.
// Each is the faster one measured for its variant: converged without the
// window (1215 against 1130 TFLOP/s on the RoPE + causal S=8192 prefill), one
// thread with it (141 against 153 ms on the windowed S=131072 prefill, k=1).
template <bool WINDOW>
__host__ __device__ constexpr bool issue_one_thread() { return WINDOW; }

template <int D, bool ROPE, bool WINDOW>
__device__ void mma_role(const FwdParams& p, bool causal, uint32_t sm, uint32_t bar0, uint32_t tmem, int t_begin,
                         int t_end, const WaitCtl& ctl) {
    constexpr bool kWarp = !issue_one_thread<WINDOW>();
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if constexpr (kWarp) return mbar_wait_warp(bar, parity, ctl, kStatusMma);
        else return mbar_wait(bar, parity, ctl, kStatusMma);
    };
    auto commit = [&](uint32_t bar) {
        if constexpr (kWarp) tc_commit(bar);
        else tc_commit_one(bar);
    };
    auto mma_ss = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
        if constexpr (kWarp) umma_ss(d, a, b, idesc, acc);
        else umma_ss_one(d, a, b, idesc, acc);
    };
    auto mma_ts = [&](uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
        if constexpr (kWarp) umma_ts(d, a, b, idesc, acc);
        else umma_ts_one(d, a, b, idesc, acc);
    };
    using L = SmemLayout<D>;
    // QK^T: A = Q tile, B = K tile, both K-major; fp16 after rotation, bf16 otherwise.
    const uint32_t kIdescQK = umma_idesc_f16((ROPE || p.qk_f16) ? 0u : 1u, 0u, kBlockM, kBlockN);
    // PV: A = P (bf16, TMEM), B = V tile [keys][D] with D contiguous: MN-major.
    constexpr uint32_t kIdescPV = umma_idesc_f16(1u, 1u, kBlockM, D);
    const int kbar_ready = ROPE ? BAR_K_ROT : BAR_K_FULL;
    const int qbar_ready = ROPE ? BAR_Q_ROT : BAR_Q_FULL;

    static_assert(kVStages == 2, "descriptor selects below assume two V stages");
    // operand descriptors, built once; each MMA step only advances the start address
    const uint64_t qdesc0 = sw128_desc(sm + L::kQ, 16u, 1024u);
    const uint64_t qdesc1 = sw128_desc(sm + L::kQ + L::kTileBytes, 16u, 1024u);
    // windowed K: one 16-channel group of [128 rows][32 B] per K=16 step, 32-byte swizzle, 8-row atoms 256 B apart
    const uint64_t kdesc0 = WINDOW ? sw32_desc(sm + L::kK, 256u) : sw128_desc(sm + L::kK, 16u, 1024u);
    const uint64_t vdesc0 = sw128_desc(sm + L::kV, kSubTileBytes, 1024u);
    const uint64_t vdesc1 = sw128_desc(sm + L::kV + L::kTileBytes, kSubTileBytes, 1024u);
    int kit = 0, vit = 0;
    int qit[2] = {0, 0}, pit[2] = {0, 0}, oit[2] = {0, 0};
    bool ok = true;
    for (int ti = t_begin; ti < t_end && ok; ++ti) {
        const Unit u = decode_unit(p.tasks[ti], p, causal);
        bool first_pv[2] = {true, true};
        for (int n = u.nmax; n >= -1 && ok; --n) {
            const int ks = kit % kKStages;
            const int vs = vit % kVStages;
            const bool do_s = n >= 0;
            const bool do_pv = n + 1 <= u.nmax;
            // each wait sits right before the first MMA that needs it, so a PV
            // never waits for the next K tile (or its rotation)
            bool k_ready = false, v_ready = false;
#pragma unroll
            for (int s = 0; s < 2 && ok; ++s) {
                if (!u.valid[s]) continue;
                const uint32_t tS = tmem + static_cast<uint32_t>(s * 128);
                const uint32_t tO = tmem + 256u + static_cast<uint32_t>(s * 128);
                if (do_pv && n + 1 <= u.nhi[s]) {
                    if (!v_ready) {
                        ok = wait(bar_at(bar0, BAR_V_FULL + vs), (vit / kVStages) & 1);
                        if (!ok) break;
                        v_ready = true;
                    }
                    ok = wait(bar_at(bar0, BAR_P_FULL + s), pit[s] & 1);
                    if (!ok) break;
                    ++pit[s];
                    if (first_pv[s]) {
                        ok = wait(bar_at(bar0, BAR_O_FREE + s), (oit[s] & 1) ^ 1);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const uint64_t vdesc = vs ? vdesc1 : vdesc0;
                    // 16 keys per step: 2048 bytes of V, 8 TMEM columns of P
                    mma_ts(tO, tS, vdesc, kIdescPV, first_pv[s] ? 0u : 1u);
#pragma unroll
                    for (int kk = 1; kk < kBlockN / 16; ++kk)
                        mma_ts(tO, tS + kk * 8u, desc_advance(vdesc, kk * 128u), kIdescPV, 1u);
                    first_pv[s] = false;
                }
                if (do_s && n <= u.nhi[s]) {
                    if (!k_ready) {
                        ok = wait(bar_at(bar0, kbar_ready + ks), (kit / kKStages) & 1);
                        if (!ok) break;
                        k_ready = true;
                        tc_fence_after();
                    }
                    if (n == u.nhi[s]) {
                        ok = wait(bar_at(bar0, qbar_ready + s), qit[s] & 1);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    const uint64_t qdesc = s ? qdesc1 : qdesc0;
                    const uint64_t kdesc = desc_advance(kdesc0, static_cast<uint32_t>(ks) * (L::kTileBytes >> 4));
                    if (WINDOW) {
                        // k-step kk covers pairs of block kk % (D/32); blocks below m0 hold only dropped pairs
                        const int m0 = window_tile<D>(p, u, n).m0;
                        uint32_t acc = 0u;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            if (kk % (D / 32) < m0) continue;
                            const uint32_t qunits = (kk / 4) * (kSubTileBytes >> 4) + (kk % 4) * 2u;
                            mma_ss(tS, desc_advance(qdesc, qunits), desc_advance(kdesc, kk * 256u), kIdescQK, acc);
                            acc = 1u;
                        }
                    } else {
                        // 16 channels per step: 32 bytes inside a 128-byte row, next column block every 4 steps
                        mma_ss(tS, qdesc, kdesc, kIdescQK, 0u);
#pragma unroll
                        for (int kk = 1; kk < D / 16; ++kk) {
                            const uint32_t units = (kk / 4) * (kSubTileBytes >> 4) + (kk % 4) * 2u;
                            mma_ss(tS, desc_advance(qdesc, units), desc_advance(kdesc, units), kIdescQK, 1u);
                        }
                    }
                    commit(bar_at(bar0, BAR_S_FULL + s));
                    if (n == 0) ++qit[s];  // Q_s is released by its softmax (see softmax_loop)
                }
            }
            if (!ok) break;
            // The K/V slots are released by the softmax (see softmax_loop): each
            // commit here would take a slot of the tensor core's short
            // instruction queue between two groups of MMAs.
            if (do_s) ++kit;
            if (do_pv) ++vit;
        }
        if (!ok) break;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (!u.valid[s]) continue;
            commit(bar_at(bar0, BAR_O_FULL + s));
            ++oit[s];
        }
    }
    // Drain: every issued MMA must finish before TMEM is released.  This wait
    // ignores the abort flag but keeps its own time limit.
    commit(bar_at(bar0, BAR_DRAIN));
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar_at(bar0, BAR_DRAIN), 0)) {
        if (global_timer_ns() - t0 > ctl.limit_ns) {
            atomicOr(ctl.status, kStatusDrain);
            break;
        }
    }
}

// ------------------------------------------------------------------ softmax + epilogue
// Streams the 128 columns of this thread's row of a tile from TMEM in
// 32-column chunks: the load of chunk k + 1 is in flight while f(chunk k, its
// first column) runs.
template <typename F>
__device__ __forceinline__ void tmem_stream_128(uint32_t taddr, F&& f) {
    uint32_t a[32], b[32];
    tmem_load_32(taddr, a);
    tmem_load_32_async(taddr + 32, b);
    f(a, 0);
    tmem_wait_ld_32(b);
    tmem_load_32_async(taddr + 64, a);
    f(b, 32);
    tmem_wait_ld_32(a);
    tmem_load_32_async(taddr + 96, b);
    f(a, 64);
    tmem_wait_ld_32(b);
    f(b, 96);
}

// Masked row maximum of 32 raw scores: keys at or past `limit` are ignored.
template <bool MASKED>
__device__ __forceinline__ float row_max32(const uint32_t (&r)[32], int col0, int limit, float mx) {
    float m0 = mx, m1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[q] = __uint_as_float(r[j + q]);
            if (MASKED && col0 + j + q >= limit) v[q] = -INFINITY;
        }
        m0 = fmax3(m0, v[0], v[1]);
        m1 = fmax3(m1, v[2], v[3]);
    }
    return fmaxf(m0, m1);
}

// P = exp2(S*c - m*c) for 32 scores (masked keys give exactly 0), the running
// pair sum of P in fp32, and P packed to bf16 pairs (even key in the low half).
template <bool MASKED>
__device__ __forceinline__ void exp_pack32(const uint32_t (&r)[32], int col0, int limit, uint64_t c2, uint64_t nmc2,
                                           uint64_t& sum2, uint32_t (&pk)[16]) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        float a = __uint_as_float(r[j]), b = __uint_as_float(r[j + 1]);
        if (MASKED) {
            if (col0 + j >= limit) a = -INFINITY;
            if (col0 + j + 1 >= limit) b = -INFINITY;
        }
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(a, b), c2, nmc2), x0, x1);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        sum2 = f2_add(sum2, f2_pack(p0, p1));
        pk[j / 2] = pack_bf16x2(p0, p1);
    }
}

template <bool MASKED>
__device__ __forceinline__ float tile_row_max(uint32_t taddr, int limit) {
    static_assert(kBlockN == 128, "the TMEM stream covers 128 columns");
    float mx = -INFINITY;
    tmem_stream_128(taddr, [&](const uint32_t (&r)[32], int cc) { mx = row_max32<MASKED>(r, cc, limit, mx); });
    return mx;
}

template <bool MASKED>
__device__ __forceinline__ float tile_exp_to_p(uint32_t taddr, int limit, float c, float mc) {
    const uint64_t c2 = f2_pack(c, c), nmc2 = f2_pack(-mc, -mc);
    uint64_t sum2 = f2_pack(0.f, 0.f);
    // P of keys cc.. goes to columns cc/2..: never a column whose S is still to be read
    tmem_stream_128(taddr, [&](const uint32_t (&r)[32], int cc) {
        uint32_t pk[16];
        exp_pack32<MASKED>(r, cc, limit, c2, nmc2, sum2, pk);
        tmem_store_16(taddr + cc / 2, pk);
    });
    float s0, s1;
    f2_unpack(sum2, s0, s1);
    return s0 + s1;
}

// Rare path of tile_exp_online, after the tile's P is formed: O_s's row is
// multiplied by alpha (unless with_o is false: on the unit's first tile O_s
// holds nothing yet) and the P of the tile's first three 32-key chunks (bf16
// pairs in columns [16k, 16k+16)) by fac[k] (all 1 for rows whose maximum
// stayed).  Called by the whole warp.
template <int D>
__device__ __forceinline__ void rescale_o_and_p(uint32_t tO, uint32_t tS, float alpha, float fac0, float fac1,
                                                float fac2, bool with_o) {
    const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
    for (int oc = 0; oc < (with_o ? D : 0); oc += 32) {
        uint32_t r[32];
        tmem_load_32(tO + oc, r);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            float x0, x1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), a2), x0, x1);
            r[j] = __float_as_uint(x0);
            r[j + 1] = __float_as_uint(x1);
        }
        tmem_store_32(tO + oc, r);
    }
    tmem_store_wait();  // the P stores have landed before they are read back
#pragma unroll 1
    for (int k = 0; k < 3; ++k) {
        const float f = k == 0 ? fac0 : (k == 1 ? fac1 : fac2);
        const uint64_t f2 = f2_pack(f, f);
        uint32_t r[16];
        tmem_load_16(tS + 16 * k, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r[j]));
            float x0, x1;
            f2_unpack(f2_mul(f2_pack(x.x, x.y), f2), x0, x1);
            r[j] = pack_bf16x2(x0, x1);
        }
        tmem_store_16(tS + 16 * k, r);
    }
}

// One pass over a tile: P is formed against the running maximum m_used, and
// each 32-key chunk's maximum comes with its load (tcgen05.ld.red; on the
// masked tiles, the diagonal and the ragged last one, recomputed from the
// visible keys), so no separate max pass is needed.  A chunk whose maximum
// exceeds m_used by more than the rescale threshold moves m_used there before
// its own P is formed (l and the tile's partial sum rescaled at once); O_s and
// the P of the tile's earlier chunks are rescaled after the tile, by the
// product of the factors that apply to each.  While m_used is -inf (no key
// seen yet) a chunk only sets it: nothing has been accumulated.  Keys
// [0, limit) are visible to this row; `first` marks the unit's first tile.
template <int D, bool MASKED>
__device__ __forceinline__ void tile_exp_online(uint32_t tS, uint32_t tO, float c, int limit, bool first,
                                                float& m_used, float& l) {
    static_assert(kBlockN == 128, "four 32-key chunks");
    const uint64_t c2 = f2_pack(c, c);
    // a row that has seen no key yet forms P against 0: its masked keys give exp2(-inf) = 0
    const float nmc0 = m_used == -INFINITY ? 0.f : -m_used * c;
    uint64_t nmc2 = f2_pack(nmc0, nmc0);
    uint64_t sum2 = f2_pack(0.f, 0.f);
    float alpha_all = 1.f, fac0 = 1.f, fac1 = 1.f, fac2 = 1.f;
    bool moved = false;
    auto step = [&](const uint32_t (&r)[32], float cm, int k) {
        if (MASKED && 32 * k + 31 >= limit) cm = row_max32<true>(r, 32 * k, limit, -INFINITY);
        if ((cm - m_used) * c > kRescaleThreshold) {
            if (m_used != -INFINITY) {
                const float alpha = ex2_approx((m_used - cm) * c);
                l *= alpha;
                sum2 = f2_mul(sum2, f2_pack(alpha, alpha));
                alpha_all *= alpha;
                if (k > 0) fac0 *= alpha;
                if (k > 1) fac1 *= alpha;
                if (k > 2) fac2 *= alpha;
                moved = true;
            }
            m_used = cm;
            nmc2 = f2_pack(-m_used * c, -m_used * c);
        }
        uint32_t pk[16];
        exp_pack32<MASKED>(r, 32 * k, limit, c2, nmc2, sum2, pk);
        tmem_store_16(tS + 16 * k, pk);  // keys 32k.. to columns 16k..: never a column still to be read
    };
    uint32_t a[32], b[32];
    float ma, mb;
    tmem_load_32_max(tS, a, ma);
    tmem_load_32_max_async(tS + 32, b, mb);
    step(a, ma, 0);
    tmem_wait_ld_32_max(b, mb);
    tmem_load_32_max_async(tS + 64, a, ma);
    step(b, mb, 1);
    tmem_wait_ld_32_max(a, ma);
    tmem_load_32_max_async(tS + 96, b, mb);
    step(a, ma, 2);
    tmem_wait_ld_32_max(b, mb);
    step(b, mb, 3);
    float s0, s1;
    f2_unpack(sum2, s0, s1);
    l += s0 + s1;
    if (__any_sync(0xffffffffu, moved)) rescale_o_and_p<D>(tO, tS, alpha_all, fac0, fac1, fac2, !first);
}

// Windowed variant, boundary pairs: pairs in [r_begin, r_end) are kept by the
// QK^T product for this tile but dropped for some of its cells (distance
// i - j > W_r).  Their exact terms q'_r k'_r + q'_{r+D/2} k'_{r+D/2} are
// subtracted from those cells of this thread's row, from the same fp16
// operands the tensor cores multiplied (the products are exact in fp32, so
// only the summation order differs).  rel = row - first key of the tile.
// Per 32-key chunk and pair, the K values of the chunk's keys are read first
// (broadcast loads: every row needs the same ones), then applied with selects.
// W_r ascends in r and the dropped keys of a row are those with j < rel - W_r,
// so once no row of the warp drops a key, later pairs and later chunks drop
// none either.  Called by the whole warp; most tiles have no boundary pair.
template <int D>
__device__ __noinline__ void window_correct(uint32_t tS, const uint8_t* qtile, const uint8_t* ktile,
                                            const FwdParams& p, int r_begin, int r_end, int rel, int t) {
    constexpr int kHalf = D / 2;
#pragma unroll 1
    for (int cc = 0; cc < kBlockN; cc += 32) {
        if (!__any_sync(0xffffffffu, rel - p.win[r_begin] - cc > 0)) break;
        uint32_t r[32];
        tmem_load_32(tS + cc, r);
#pragma unroll 1
        for (int pr = r_begin; pr < r_end; ++pr) {
            const int lim = rel - p.win[pr] - cc;  // this row drops the pair for keys cc + j, j < lim
            if (!__any_sync(0xffffffffu, lim > 0)) break;
            const int dx = pr, dy = pr + kHalf;  // channels of the pair
            const float qx = f16_at(qtile + (dx / 64) * kSubTileBytes + t * 128 + ((((dx % 64) / 8) ^ (t & 7)) << 4) +
                                    (dx % 8) * 2);
            const float qy = f16_at(qtile + (dy / 64) * kSubTileBytes + t * 128 + ((((dy % 64) / 8) ^ (t & 7)) << 4) +
                                    (dy % 8) * 2);
            // K in 16-channel groups with the 32-byte swizzle: channel d of key row j at
            // (d/16)*4096 + j*32 + ((((d%16)/8) ^ ((j>>2)&1)) << 4) + (d%8)*2; cc is a multiple of 8,
            // so the swizzle bit of key cc + j is (j >> 2) & 1
            const uint8_t* kx = ktile + (dx / 16) * 4096 + (dx % 8) * 2 + cc * 32;
            const uint8_t* ky = ktile + (dy / 16) * 4096 + (dy % 8) * 2 + cc * 32;
            const int hx = ((dx % 16) / 8) << 4, hy = ((dy % 16) / 8) << 4;
            float kxv[32], kyv[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int sw = ((j >> 2) & 1) << 4;
                kxv[j] = f16_at(kx + j * 32 + (hx ^ sw));
                kyv[j] = f16_at(ky + j * 32 + (hy ^ sw));
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float v = __uint_as_float(r[j]);
                const float term = fmaf(qx, kxv[j], qy * kyv[j]);
                r[j] = __float_as_uint(j < lim ? v - term : v);
            }
        }
        tmem_store_32(tS + cc, r);
    }
    tmem_store_wait();
}

// One body serves both stages (stage is a runtime value: a second copy of this
// code measurably costs instruction-cache capacity).  Per-stage fields of the
// unit are picked with selects so nothing is indexed at run time.
template <int D, bool CAUSAL, bool WINDOW>
__device__ void softmax_loop(const FwdParams& p, int stage, uint8_t* smg, uint32_t bar0, uint32_t tmem, int t_begin,
                             int t_end, const WaitCtl& ctl, int t) {
    using L = SmemLayout<D>;
    int kit = 0;  // K tiles seen by the unit loop (which K stage holds tile n)
    const uint32_t lane_base = static_cast<uint32_t>(t & ~31);  // this warp's TMEM lane quarter
    const uint32_t trow = tmem + (lane_base << 16);
    const uint32_t tS = trow + static_cast<uint32_t>(stage * 128);
    const uint32_t tO = trow + 256u + static_cast<uint32_t>(stage * 128);
    const float c = p.scale_log2;
    const int last_tile = (p.S - 1) / kBlockN;
    const bool ragged = (p.S % kBlockN) != 0;
    int sit = 0, oit = 0;
    for (int ti = t_begin; ti < t_end; ++ti) {
        const Unit u = decode_unit(p.tasks[ti], p, CAUSAL);
        const int kit_unit = kit;  // K tiles of earlier units (tile n of this unit is the (nmax-n)-th after them)
        kit += u.nmax + 1;
        const bool valid = stage ? u.valid[1] : u.valid[0];
        if (!valid) continue;
        // The stage that visits every K/V tile of the unit releases the K/V
        // slots: stage 1 when present (its first tile is the unit's first, and
        // its products are issued after stage 0's), else stage 0.
        const bool releaser = stage == 1 || !u.valid[1];
        const int nhi = stage ? u.nhi[1] : u.nhi[0];
        const int head = stage ? u.h[1] : u.h[0];
        const int row = (stage ? u.row0[1] : u.row0[0]) + t;
        float m_used = -INFINITY;
        float l = 0.f;
        for (int n = nhi; n >= 0; --n) {
            if (!__all_sync(0xffffffffu,
                            mbar_wait(bar_at(bar0, BAR_S_FULL + stage), sit & 1, ctl, kStatusSoftmax << stage)))
                return;
            ++sit;
            tc_fence_after();
            const int it = kit_unit + u.nmax - n;  // load index of K(n) and V(n)
            if (releaser && t == 0) {
                // S_s(n) landed, and the issue order puts it after every other
                // product that reads V(n+1) (and K(n)): the slots are free again
                if (n + 1 <= u.nmax) mbar_arrive(bar_at(bar0, BAR_V_EMPTY + (it - 1) % kVStages));
                if (!WINDOW) mbar_arrive(bar_at(bar0, BAR_K_EMPTY + it % kKStages));
            }
            if (!WINDOW && n == 0 && t == 0)  // the unit's last product reading Q_s has landed
                mbar_arrive(bar_at(bar0, BAR_Q_EMPTY + stage));
            if (WINDOW) {
                // boundary pairs: kept for the tile by the MMA, dropped beyond W_r for some of its cells
                const int z = window_tile<D>(p, u, n).z;
                const int rel0 = (stage ? u.row0[1] : u.row0[0]) - n * kBlockN;  // first row - first key
                const int r_end = p.wtab[rel0 / kBlockM].y;                       // kept everywhere from here on
                if (z < r_end)
                    window_correct<D>(tS, smg + L::kQ + stage * L::kTileBytes,
                                      smg + L::kK + (it % kKStages) * L::kTileBytes, p, z, r_end, rel0 + t, t);
                // K(n), and Q_s after tile 0, are free once both stages' corrections have read them:
                // one arrival per warp and stage, doubled when the other stage does not visit tile n
                __syncwarp();
                if ((t & 31) == 0) {
                    const bool other = stage ? (u.valid[0] && n <= u.nhi[0]) : (u.valid[1] && n <= u.nhi[1]);
                    mbar_arrive_cnt(bar_at(bar0, BAR_K_EMPTY + it % kKStages), other ? 1u : 2u);
                    if (n == 0) mbar_arrive(bar_at(bar0, BAR_Q_EMPTY + stage));
                }
            }
            // keys [0, limit) of this tile are visible to this row; only the
            // diagonal tile (causal) and the ragged last tile have a limit < 128
            const bool diag = CAUSAL && n == nhi;
            const bool tail = ragged && n == last_tile;
            int limit = kBlockN;
            if (diag) limit = t + 1;
            if (tail) limit = min(limit, p.S - n * kBlockN);
            if (diag || tail)  // uniform across the warp
                tile_exp_online<D, true>(tS, tO, c, limit, n == nhi, m_used, l);
            else
                tile_exp_online<D, false>(tS, tO, c, limit, n == nhi, m_used, l);
            tmem_store_wait();
            tc_fence_before();
            mbar_arrive(bar_at(bar0, BAR_P_FULL + stage));
        }
        // epilogue: O / l in bf16, LSE in natural log
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar_at(bar0, BAR_O_FULL + stage), oit & 1, ctl, kStatusSoftmax << stage)))
            return;
        ++oit;
        tc_fence_after();
        if (releaser && t == 0)  // the unit's last products (PV of tile 0) are done: V(0) is free
            mbar_arrive(bar_at(bar0, BAR_V_EMPTY + (kit_unit + u.nmax) % kVStages));
        const float inv_l = 1.0f / l;
        const uint64_t il2 = f2_pack(inv_l, inv_l);
        const bool row_ok = row < p.S;
        const float lse2 = m_used * c + log2f(l);  // every row sees at least one key: finite for finite scores
        if (row_ok && !isfinite(lse2)) atomicOr(p.status, kStatusNonFinite);
        if (row_ok && p.lse != nullptr)
            p.lse[(static_cast<size_t>(u.b) * p.Hq + head) * p.S + row] = lse2 * 0.69314718055994531f;
        // Each warp stages its 32 rows one 64-channel block at a time (128-byte
        // swizzle: chunk c of row r at chunk c ^ (r & 7)) and stores the block
        // with one TMA copy; rows past S are clipped by the copy.  O_s is
        // handed back as soon as its last columns are in registers.
        const int lane = t & 31, wq = t >> 5;
        uint8_t* blk = smg + L::kO + static_cast<uint32_t>(stage) * kEpiStageBytes + static_cast<uint32_t>(wq) * kEpiWarpBytes;
        const int row0 = (stage ? u.row0[1] : u.row0[0]) + 32 * wq;
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub) {
            if (lane == 0) bulk_wait_group_read<0>();  // the previous copy has read the block
            __syncwarp();
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // 32 channels (four 16-byte chunks) at a time
                uint32_t r[32];
                tmem_load_32(tO + 64 * sub + 32 * h, r);
                if (sub == D / 64 - 1 && h == 1) {
                    tc_fence_before();
                    mbar_arrive(bar_at(bar0, BAR_O_FREE + stage));
                }
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float x0, x1;
                    f2_unpack(f2_mul(f2_pack(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), il2), x0, x1);
                    pk[j] = pack_bf16x2(x0, x1);
                }
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int c8 = 4 * h + c4;
                    *reinterpret_cast<uint4*>(blk + lane * 128 + ((c8 ^ (lane & 7)) << 4)) =
                        make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_4d(&p.tm_o, smem_addr(blk), 64 * sub, head, row0, u.b);
                bulk_commit_group();
            }
        }
    }
}

// The softmax warpgroup's role; before the warps leave, each warp's output
// copies must have finished (their source is this CTA's shared memory).
template <int D, bool CAUSAL, bool WINDOW>
__device__ void softmax_role(const FwdParams& p, int stage, uint8_t* smg, uint32_t bar0, uint32_t tmem, int t_begin,
                             int t_end, const WaitCtl& ctl, int t) {
    softmax_loop<D, CAUSAL, WINDOW>(p, stage, smg, bar0, tmem, t_begin, t_end, ctl, t);
    if ((t & 31) == 0) bulk_wait_group<0>();
}

// ------------------------------------------------------------------ kernel
template <int D, bool CAUSAL, bool ROPE, bool WINDOW>
__global__ void __launch_bounds__(kNumThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
    static_assert(!WINDOW || (CAUSAL && ROPE), "the window is defined with RoPE and causal masking");
    using L = SmemLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smg = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sm = smem_addr(smg);
    const uint32_t bar0 = sm + L::kBars;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smg + L::kMisc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smg + L::kMisc + 4);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        *abort_flag = 0;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_at(bar0, BAR_Q_FULL + s), 1);
            mbar_init(bar_at(bar0, BAR_Q_ROT + s), 128);
            mbar_init(bar_at(bar0, BAR_Q_EMPTY + s), WINDOW ? 4 : 1);  // windowed: one arrival per warp
            mbar_init(bar_at(bar0, BAR_S_FULL + s), 1);
            mbar_init(bar_at(bar0, BAR_P_FULL + s), 128);
            mbar_init(bar_at(bar0, BAR_O_FULL + s), 1);
            mbar_init(bar_at(bar0, BAR_O_FREE + s), 128);
        }
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(bar_at(bar0, BAR_K_FULL + i), 1);
            mbar_init(bar_at(bar0, BAR_K_ROT + i), 128);
            mbar_init(bar_at(bar0, BAR_K_EMPTY + i), WINDOW ? 8 : 1);  // windowed: per warp of both stages
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(bar_at(bar0, BAR_V_FULL + i), 1);
            mbar_init(bar_at(bar0, BAR_V_EMPTY + i), 1);
        }
        mbar_init(bar_at(bar0, BAR_DRAIN), 1);
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kWarpTma && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns};
    const int t_begin = p.task_off[blockIdx.x];
    const int t_end = p.task_off[blockIdx.x + 1];

    if (warp < 8) {
        regs_increase<kRegsSoftmax>();
        softmax_role<D, CAUSAL, WINDOW>(p, warp / 4, smg, bar0, tmem, t_begin, t_end, ctl, threadIdx.x % 128);
    } else if (warp < kWarpTma) {
        regs_decrease<kRegsRope>();
        if (ROPE) rope_role<D, WINDOW>(p, CAUSAL, smg, bar0, t_begin, t_end, ctl, threadIdx.x - kWarpRope * 32);
    } else {
        regs_decrease<kRegsOther>();
        if (warp == kWarpTma) {
            if (lane == 0) producer_role<D, WINDOW>(p, CAUSAL, sm, bar0, t_begin, t_end, ctl);
            __syncwarp();
        } else if (warp == kWarpMma) {
            if constexpr (issue_one_thread<WINDOW>()) {
                if (lane == 0) mma_role<D, ROPE, WINDOW>(p, CAUSAL, sm, bar0, tmem, t_begin, t_end, ctl);
                __syncwarp();
            } else {
                mma_role<D, ROPE, WINDOW>(p, CAUSAL, sm, bar0, tmem, t_begin, t_end, ctl);  // the whole warp
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace attn
