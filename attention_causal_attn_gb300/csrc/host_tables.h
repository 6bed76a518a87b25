// Host-side tables and the static tile schedule of the attention forward.
// Plain C++ (no CUDA): compiled by the host compiler and unit-tested through
// the C ABI without a GPU.
#pragma once

#include <cstdint>
#include <vector>

namespace attn_host {

// theta_r = base^(-2r/D), r = 0..D/2-1 (RoFormer's frequencies, NeoX pairing r <-> r + D/2).
std::vector<double> rope_thetas(int D, double base);

// (cos, sin) of (p + pos_offset) * theta_r for p = 0..S-1, interleaved as
// [S][D/2][2] float32, computed in float64.
std::vector<float> rope_table(int S, int D, double base, long long pos_offset);

// Rows of a 128-row tile that one pass of 128 rotating threads covers: each
// thread takes one 16-byte chunk (8 pairs) of the D/2 pairs of a row, so a
// pass covers 128 / (D/16) = 2048/D rows (16 for D = 128, 32 for D = 64).
// Shared with the kernel.
constexpr int rope_rows_per_pass(int D) { return 2048 / D; }

// The factor tables the kernel rotates with (float2 = (cos, sin), float32 from
// float64), for positions p = 128*m + rows*i + rr, rows = rope_rows_per_pass(D):
//   base[m][r]    = angle 128*m*theta_r,  m = 0..ceil(S/128)-1
//   rowfac[rr][r] = angle rr*theta_r,     rr = 0..rows-1
//   step[r]       = angle rows*theta_r
// The kernel forms the angle of position p by complex multiplication of these factors.
std::vector<float> rope_factor_table(int S, int D, double base);
size_t rope_factor_table_floats(int S, int D);

// Factor tables of the pre-rotation pass (block = 128) and of decode
// (block = 32), float2 = (cos, sin), float32 from float64:
// base[m][r] = angle block*m*theta_r for m = 0..ceil(S/block)-1, then
// row[rr][r] = angle rr*theta_r for rr = 0..block-1.
std::vector<float> rope_split_tables(int S, int D, double base, int block);

// W_r = floor(k * 2*pi / theta_r) clamped to [0, INT32_MAX]; INT32_MAX when
// the window is off (k <= 0 or infinite).  ("ATFlash", The idea.)
std::vector<int32_t> window_widths(int D, double base, double k);

// Window bounds per tile distance t = 0..ceil(S/128)-1 (query tile minus key
// tile), as int16 pairs: [2t] = first pair r with W_r >= max(0, 128t - 127)
// (the tile's smallest distance), [2t+1] = first pair with W_r >= 128t + 127
// (its largest).  D/2 when no pair qualifies.
std::vector<int16_t> window_tile_table(int S, int D, double base, double k);

// One work unit = two 128-row query tiles sharing a KV head, encoded as the
// kernel reads it: x = qtile0 | qtile1 << 16 (0xFFFF: no second tile),
// y = h0 | h1 << 8 | b << 16.
struct Schedule {
    std::vector<uint32_t> words;  // 2 per unit, in per-CTA order
    std::vector<int32_t> offsets; // ctas + 1 prefix offsets into units
    int ctas = 0;
    double max_cost = 0, mean_cost = 0;  // per-CTA estimated cost
};

// Cost-guided static schedule ("Flash Attention: Causal Prefill D=128", Step 4:
// estimated cost 2(bm+1) + 4 per query tile, heaviest units first into the
// lightest CTA).
//
// K/V locality in L2: the KV heads, in (batch, KV head) order, are cut into
// windows whose K and V together take at most kv_window_bytes (at least one
// KV head per window).  Windows are scheduled one after another: the units of
// a window go heaviest first into the CTA with the least load accumulated over
// all earlier windows, and each CTA runs its units in that order.  The loads
// stay balanced at every window boundary (to within one unit), so the CTAs
// move through the windows together and the K/V tiles that the units running
// at one time read from L2 belong to one or two windows.  The last window,
// which has to even out what the earlier ones leave, is widened to at least
// three units per CTA.  kv_window_bytes <= 0 puts every KV head into one
// window (plain longest-first).
constexpr double kScheduleWindowBytes = 64.0 * 1024.0 * 1024.0;
Schedule build_schedule(int B, int Hq, int Hkv, int S, int D, bool causal, int num_ctas,
                        double kv_window_bytes = kScheduleWindowBytes);

// Number of work units build_schedule makes for a shape, without building it.
long long schedule_units(int B, int Hq, int Hkv, int S);

// Static schedule of the persistent block-sparse forward.  A task is one query
// tile i of one batch-head x, encoded i * bh + x.  Its cost is the number of
// key tiles the mask lists for row i plus a fixed cost per task (the Q load
// and rotation and the output stores).  Each CTA runs two task streams; the
// heaviest tasks go first into the least loaded stream.  Each stream then runs
// its tasks by (batch-head, descending query tile), so that all streams sweep
// the batch-heads in the same order and share K/V tiles in L2.
constexpr double kMaskTileFixedCost = 1.0;
struct MaskSchedule {
    std::vector<int32_t> tasks;    // per-stream lists, concatenated: stream s of CTA c is list 2c + s
    std::vector<int32_t> offsets;  // 2 ctas + 1 prefix offsets into tasks
    int ctas = 0;
};
MaskSchedule build_mask_schedule(const int* row_ptr, int nrows, long long bh, int num_ctas);

}  // namespace attn_host
