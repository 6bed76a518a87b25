// Pre-rotation pass: RoPE applied to a whole BSHD bf16 tensor in one memory-
// bound sweep, written as fp16 (the precision the fused path gives its
// rotated operands).  It is the other side of "AttnFuse" sec. 5.3, The
// Rotation Calculus: rotate Q and K once and run the attention kernel without
// in-loop rotation, against rotating K tiles inside the loop every time a
// query tile visits them.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace attn {

// Thread i rotates chunk c = i % (D/16) (pairs 8c..8c+7) of row i / (D/16):
// eight consecutive threads cover one row's two 128-byte halves.  The angle of
// position s = 128*m + rr is the product of two float64-built factors:
// base[m][r] = (cos, sin)(128*m*theta_r) and row[rr][r] = (cos, sin)(rr*theta_r).
template <int D>
__global__ void __launch_bounds__(256) rope_rotate_kernel(const uint4* __restrict__ x, uint4* __restrict__ y,
                                                           const float2* __restrict__ base_tab,
                                                           const float2* __restrict__ row_tab, long long rows, int S,
                                                           int H) {
    constexpr int kHalf = D / 2;
    constexpr int kChunks = kHalf / 8;  // 16-byte chunks per half row
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= rows * kChunks) return;
    const long long row = i / kChunks;
    const int c = static_cast<int>(i % kChunks);
    const int s = static_cast<int>((row / H) % S);
    // (cos, sin) factors of pairs 8c..8c+7, two pairs per 16-byte load
    const float4* bf = reinterpret_cast<const float4*>(base_tab + static_cast<size_t>(s / 128) * kHalf + 8 * c);
    const float4* rf = reinterpret_cast<const float4*>(row_tab + static_cast<size_t>(s % 128) * kHalf + 8 * c);
    const uint4 lo = __ldg(x + row * (D / 8) + c);
    const uint4 hi = __ldg(x + row * (D / 8) + kChunks + c);
    const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w};
    const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w};
    uint32_t lo_out[4], hi_out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 f1v = __ldg(bf + q), f2v = __ldg(rf + q);
        float a[2], b[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float2 f1 = e ? make_float2(f1v.z, f1v.w) : make_float2(f1v.x, f1v.y);
            const float2 f2 = e ? make_float2(f2v.z, f2v.w) : make_float2(f2v.x, f2v.y);
            const float cs = f1.x * f2.x - f1.y * f2.y;  // cos(A + B)
            const float sn = f1.y * f2.x + f1.x * f2.y;  // sin(A + B)
            const float xv = e ? bf16_hi(lw[q]) : bf16_lo(lw[q]);
            const float yv = e ? bf16_hi(hw[q]) : bf16_lo(hw[q]);
            a[e] = xv * cs - yv * sn;
            b[e] = yv * cs + xv * sn;
        }
        lo_out[q] = pack_f16x2(a[0], a[1]);
        hi_out[q] = pack_f16x2(b[0], b[1]);
    }
    y[row * (D / 8) + c] = make_uint4(lo_out[0], lo_out[1], lo_out[2], lo_out[3]);
    y[row * (D / 8) + kChunks + c] = make_uint4(hi_out[0], hi_out[1], hi_out[2], hi_out[3]);
}

}  // namespace attn
