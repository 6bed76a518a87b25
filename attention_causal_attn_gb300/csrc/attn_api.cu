// C ABI of the fused RoPE + causal attention forward (declared in attn.h):
// argument checks, the per-device cache of RoPE tables and tile schedules,
// TMA descriptor encoding, and the launch of the sm_103a kernel.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "attn.h"
#include "attn_fwd_kernel.cuh"
#include "host_tables.h"

// Raised (bitwise OR) by a CTA whose bounded wait ran out; read and cleared by attn_check().
__device__ int g_attn_status;

namespace {

using attn::FwdParams;

constexpr int kMaxDevices = 64;
constexpr int kMaxS = 1 << 22;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait

struct RopeEntry {
    int dev, S, D;
    double base;
    float2* table;
};
struct WinEntry {
    int dev, S, D;
    double base, k;
    short2* table;
};
struct SchedEntry {
    int dev, B, Hq, Hkv, S, causal, ctas;
    uint2* tasks;
    int* offsets;
};
struct DevInfo {
    bool probed = false, ok = false;
    int sms = 0;
    int* status = nullptr;
    unsigned configured = 0;  // kernel variants whose smem attribute was set (bit per variant)
};

std::mutex g_mu;

// With ATTN_VERBOSE=1 in the environment, failures name the CUDA call and its error.
bool verbose() {
    static const bool v = [] {
        const char* e = std::getenv("ATTN_VERBOSE");
        return e != nullptr && e[0] == '1';
    }();
    return v;
}
int cuda_fail(const char* what, cudaError_t e, int code = ATTN_ERR_CUDA) {
    if (verbose()) std::fprintf(stderr, "attn: %s failed: %s (%d)\n", what, cudaGetErrorString(e), static_cast<int>(e));
    return code;
}
std::vector<RopeEntry> g_rope;
std::vector<SchedEntry> g_sched;
std::vector<WinEntry> g_win;
DevInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// [B][S][H][D] bf16 as a 4-D tensor (innermost first: D, H, S, B); box
// {64, 1, 128, 1} = 128 rows of one head and 64 channels, 128-byte swizzle.
// Rows past S read as zero.
bool encode_bshd(CUtensorMap* m, const void* base, int B, int S, int H, int D, int box_inner = 64,
                 CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B, int box_rows = 128) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                                   static_cast<cuuint64_t>(S) * H * D * 2};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_inner), 1, static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t elem[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q, K, V loads (128-row boxes) and the O store (32-row boxes: one warp's rows).
bool encode_operands(FwdParams* prm, const void* q, const void* k, const void* v, void* o, int B, int S, int Hq,
                     int Hkv, int D) {
    return encode_bshd(&prm->tm_q, q, B, S, Hq, D) && encode_bshd(&prm->tm_k, k, B, S, Hkv, D) &&
           encode_bshd(&prm->tm_v, v, B, S, Hkv, D) &&
           encode_bshd(&prm->tm_o, o, B, S, Hq, D, 64, CU_TENSOR_MAP_SWIZZLE_128B, 32);
}

int probe_device(int dev) {
    DevInfo& di = g_dev[dev];
    if (!di.probed) {
        di.probed = true;
        int major = 0, minor = 0;
        cudaError_t e;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail("cudaDeviceGetAttribute", e);
        if (major != 10 || minor != 3) return cuda_fail("compute capability 10.3 check", cudaSuccess, ATTN_ERR_NO_DEVICE);
        if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&di.status), g_attn_status)) != cudaSuccess)
            return cuda_fail("cudaGetSymbolAddress(status word)", e);
        di.ok = true;
    }
    return di.ok ? ATTN_OK : ATTN_ERR_NO_DEVICE;
}

int get_rope(int dev, int S, int D, double base, float2** out) {
    for (auto& e : g_rope)
        if (e.dev == dev && e.S == S && e.D == D && e.base == base) {
            *out = e.table;
            return ATTN_OK;
        }
    const std::vector<float> host = attn_host::rope_factor_table(S, D, base);
    float2* d = nullptr;
    cudaError_t e;
    if ((e = cudaMalloc(&d, host.size() * sizeof(float))) != cudaSuccess) return cuda_fail("cudaMalloc(rope)", e, ATTN_ERR_OOM);
    if ((e = cudaMemcpy(d, host.data(), host.size() * sizeof(float), cudaMemcpyHostToDevice)) != cudaSuccess) {
        cudaFree(d);
        return cuda_fail("cudaMemcpy(rope)", e);
    }
    g_rope.push_back({dev, S, D, base, d});
    *out = d;
    return ATTN_OK;
}

int get_wtab(int dev, int S, int D, double base, double k, short2** out) {
    for (auto& e : g_win)
        if (e.dev == dev && e.S == S && e.D == D && e.base == base && e.k == k) {
            *out = e.table;
            return ATTN_OK;
        }
    const std::vector<int16_t> host = attn_host::window_tile_table(S, D, base, k);
    short2* d = nullptr;
    cudaError_t e;
    if ((e = cudaMalloc(&d, host.size() * sizeof(int16_t))) != cudaSuccess)
        return cuda_fail("cudaMalloc(window table)", e, ATTN_ERR_OOM);
    if ((e = cudaMemcpy(d, host.data(), host.size() * sizeof(int16_t), cudaMemcpyHostToDevice)) != cudaSuccess) {
        cudaFree(d);
        return cuda_fail("cudaMemcpy(window table)", e);
    }
    g_win.push_back({dev, S, D, base, k, d});
    *out = d;
    return ATTN_OK;
}

int get_schedule(int dev, int B, int Hq, int Hkv, int S, int causal, int sms, const SchedEntry** out) {
    for (auto& e : g_sched)
        if (e.dev == dev && e.B == B && e.Hq == Hq && e.Hkv == Hkv && e.S == S && e.causal == causal) {
            *out = &e;
            return ATTN_OK;
        }
    const attn_host::Schedule sc = attn_host::build_schedule(B, Hq, Hkv, S, causal != 0, sms);
    uint2* tasks = nullptr;
    int* offs = nullptr;
    cudaError_t e;
    if ((e = cudaMalloc(&tasks, sc.words.size() * sizeof(uint32_t))) != cudaSuccess)
        return cuda_fail("cudaMalloc(tasks)", e, ATTN_ERR_OOM);
    if ((e = cudaMalloc(&offs, sc.offsets.size() * sizeof(int32_t))) != cudaSuccess) {
        cudaFree(tasks);
        return cuda_fail("cudaMalloc(offsets)", e, ATTN_ERR_OOM);
    }
    if ((e = cudaMemcpy(tasks, sc.words.data(), sc.words.size() * sizeof(uint32_t), cudaMemcpyHostToDevice)) !=
            cudaSuccess ||
        (e = cudaMemcpy(offs, sc.offsets.data(), sc.offsets.size() * sizeof(int32_t), cudaMemcpyHostToDevice)) !=
            cudaSuccess) {
        cudaFree(tasks);
        cudaFree(offs);
        return cuda_fail("cudaMemcpy(schedule)", e);
    }
    g_sched.push_back({dev, B, Hq, Hkv, S, causal, sc.ctas, tasks, offs});
    *out = &g_sched.back();
    return ATTN_OK;
}

template <int D, bool CAUSAL, bool ROPE, bool WINDOW = false>
int launch(const FwdParams& prm, int grid, cudaStream_t stream, DevInfo& di) {
    constexpr unsigned bit = 1u << ((WINDOW ? 8 : 0) | (D == 128 ? 4 : 0) | (CAUSAL ? 2 : 0) | (ROPE ? 1 : 0));
    auto kern = attn::attn_fwd_kernel<D, CAUSAL, ROPE, WINDOW>;
    // At least 120 KB so that only one CTA fits on an SM: each CTA takes all 512 TMEM columns.
    using Layout = attn::SmemLayout<D, WINDOW>;
    constexpr int smem = static_cast<int>(Layout::kAlloc) > 120 * 1024 ? static_cast<int>(Layout::kAlloc) : 120 * 1024;
    cudaError_t e;
    if (!(di.configured & bit)) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
            return cuda_fail("cudaFuncSetAttribute(max dynamic smem)", e);
        di.configured |= bit;
    }
    kern<<<grid, attn::kNumThreads, smem, stream>>>(prm);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail("kernel launch", e);
    return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int S, int D, int causal, double rope_base, double window_k, void* stream) {
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return ATTN_ERR_NULL;
    if (B < 1 || B > 65535 || S < 1 || S > kMaxS || Hq < 1 || Hq > 255 || Hkv < 1 || Hkv > Hq || Hq % Hkv != 0)
        return ATTN_ERR_SHAPE;
    if (D != 64 && D != 128) return ATTN_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
        return ATTN_ERR_ALIGN;
    if (causal != 0 && causal != 1) return ATTN_ERR_UNSUPPORTED;
    const bool rope = rope_base > 0.0 && std::isfinite(rope_base);
    if (rope_base > 0.0 && !std::isfinite(rope_base)) return ATTN_ERR_UNSUPPORTED;
    const bool window = window_k > 0.0 && !std::isinf(window_k);
    if (window && !(rope && causal)) return ATTN_ERR_UNSUPPORTED;
    if (std::isnan(window_k) || std::isnan(rope_base)) return ATTN_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_NO_DEVICE;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;

    FwdParams prm;
    SchedEntry sched;  // copied under the lock: the cache vector may grow later
    float2* rope_tab = nullptr;
    short2* wtab = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int rc = probe_device(dev);
        if (rc != ATTN_OK) return rc;
        if (rope && (rc = get_rope(dev, S, D, rope_base, &rope_tab)) != ATTN_OK) return rc;
        if (window && (rc = get_wtab(dev, S, D, rope_base, window_k, &wtab)) != ATTN_OK) return rc;
        const SchedEntry* se = nullptr;
        if ((rc = get_schedule(dev, B, Hq, Hkv, S, causal, g_dev[dev].sms, &se)) != ATTN_OK) return rc;
        sched = *se;
        prm.status = g_dev[dev].status;
    }
    if (!encode_operands(&prm, q, k, v, o, B, S, Hq, Hkv, D) ||
        (window && !encode_bshd(&prm.tm_k16, k, B, S, Hkv, D, 16, CU_TENSOR_MAP_SWIZZLE_32B)))
        return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
    {
        const std::vector<int32_t> w = attn_host::window_widths(D, rope ? rope_base : 10000.0, window ? window_k : 0.0);
        for (int r = 0; r < 64; ++r) prm.win[r] = r < D / 2 ? w[r] : INT32_MAX;
    }
    prm.wtab = wtab;
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.lse = lse;
    prm.rope = rope_tab;
    prm.tasks = sched.tasks;
    prm.task_off = sched.offsets;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.S = S;
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    prm.wait_limit_ns = kWaitLimitNs;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DevInfo& di = g_dev[dev];
    const int grid = sched.ctas;
    if (window)  // RoPE and causal masking are implied (checked above)
        return D == 128 ? launch<128, true, true, true>(prm, grid, st, di) : launch<64, true, true, true>(prm, grid, st, di);
    if (D == 128) {
        if (causal) return rope ? launch<128, true, true>(prm, grid, st, di) : launch<128, true, false>(prm, grid, st, di);
        return rope ? launch<128, false, true>(prm, grid, st, di) : launch<128, false, false>(prm, grid, st, di);
    }
    if (causal) return rope ? launch<64, true, true>(prm, grid, st, di) : launch<64, true, false>(prm, grid, st, di);
    return rope ? launch<64, false, true>(prm, grid, st, di) : launch<64, false, false>(prm, grid, st, di);
}

// ---------------------------------------------------------------------------
// attn_fwd_noalloc: the same forward for callers that may not allocate device
// memory.  Its RoPE table and tile schedule live in one file-scope device
// array instead of cudaMalloc'd buffers.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB, held by every device that loads the library

// Host code may not use this name as a device address (it is a host-side
// stand-in); the device address comes from cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDev {
    bool ready = false;
    unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    // what the scratch currently holds (re-uploaded only when the request differs)
    bool have = false;
    int S = 0, D = 0, B = 0, Hq = 0, Hkv = 0, causal = 0, rope = 0, ctas = 0;
    double base = 0.0;
    size_t off_tasks = 0, off_offsets = 0;
};
NoAllocDev g_noalloc[kMaxDevices];

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                int Hkv, int S, int D, int causal, double rope_base, double window_k, void* stream) {
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return ATTN_ERR_NULL;
    if (B < 1 || B > 65535 || S < 1 || S > kMaxS || Hq < 1 || Hq > 255 || Hkv < 1 || Hkv > Hq || Hq % Hkv != 0)
        return ATTN_ERR_SHAPE;
    if (D != 64 && D != 128) return ATTN_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
        return ATTN_ERR_ALIGN;
    if (causal != 0 && causal != 1) return ATTN_ERR_UNSUPPORTED;
    if (std::isnan(window_k) || std::isnan(rope_base)) return ATTN_ERR_UNSUPPORTED;
    if (rope_base > 0.0 && !std::isfinite(rope_base)) return ATTN_ERR_UNSUPPORTED;
    const bool rope = rope_base > 0.0;
    const bool window = window_k > 0.0 && !std::isinf(window_k);
    if (window) return ATTN_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(g_mu);
    int rc = probe_device(dev);
    if (rc != ATTN_OK) return rc;
    NoAllocDev& na = g_noalloc[dev];
    cudaError_t e;
    if (!na.ready) {
        // once per device, with that device current
        if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&na.scratch), g_noalloc_scratch)) != cudaSuccess)
            return cuda_fail("cudaGetSymbolAddress(no-alloc scratch)", e);
        na.ready = true;
    }
    const bool same = na.have && na.S == S && na.D == D && na.B == B && na.Hq == Hq && na.Hkv == Hkv &&
                      na.causal == causal && na.rope == static_cast<int>(rope) && (!rope || na.base == rope_base);
    if (!same) {
        // size check first, from the shape alone
        const size_t rope_bytes = rope ? attn_host::rope_factor_table_floats(S, D) * sizeof(float) : 0;
        const long long units = attn_host::schedule_units(B, Hq, Hkv, S);
        const long long ctas = std::min<long long>(units, g_dev[dev].sms);
        const size_t off_tasks = align256(rope_bytes);
        const size_t need_tasks = static_cast<size_t>(units) * 2 * sizeof(uint32_t);
        const size_t off_offsets = align256(off_tasks + need_tasks);
        if (units > static_cast<long long>(kNoAllocScratchBytes) ||
            off_offsets + static_cast<size_t>(ctas + 1) * sizeof(int32_t) > kNoAllocScratchBytes)
            return ATTN_ERR_SCRATCH;
        const attn_host::Schedule sc = attn_host::build_schedule(B, Hq, Hkv, S, causal != 0, g_dev[dev].sms);
        na.have = false;  // contents are in flux until the copies below are enqueued
        // Pageable host sources: each copy returns once its source has been staged,
        // so the host vectors may go out of scope; the copies are ordered on `st`.
        if (rope) {
            const std::vector<float> host = attn_host::rope_factor_table(S, D, rope_base);
            if ((e = cudaMemcpyAsync(na.scratch, host.data(), rope_bytes, cudaMemcpyHostToDevice, st)) != cudaSuccess)
                return cuda_fail("cudaMemcpyAsync(no-alloc rope table)", e);
        }
        if ((e = cudaMemcpyAsync(na.scratch + off_tasks, sc.words.data(), sc.words.size() * sizeof(uint32_t),
                                 cudaMemcpyHostToDevice, st)) != cudaSuccess ||
            (e = cudaMemcpyAsync(na.scratch + off_offsets, sc.offsets.data(), sc.offsets.size() * sizeof(int32_t),
                                 cudaMemcpyHostToDevice, st)) != cudaSuccess)
            return cuda_fail("cudaMemcpyAsync(no-alloc schedule)", e);
        na.have = true;
        na.S = S, na.D = D, na.B = B, na.Hq = Hq, na.Hkv = Hkv, na.causal = causal;
        na.rope = static_cast<int>(rope), na.base = rope_base, na.ctas = sc.ctas;
        na.off_tasks = off_tasks, na.off_offsets = off_offsets;
    }

    FwdParams prm;
    if (!encode_operands(&prm, q, k, v, o, B, S, Hq, Hkv, D))
        return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.lse = lse;
    prm.rope = rope ? reinterpret_cast<const float2*>(na.scratch) : nullptr;
    prm.wtab = nullptr;
    prm.tasks = reinterpret_cast<const uint2*>(na.scratch + na.off_tasks);
    prm.task_off = reinterpret_cast<const int*>(na.scratch + na.off_offsets);
    prm.status = g_dev[dev].status;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.S = S;
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    prm.wait_limit_ns = kWaitLimitNs;
    DevInfo& di = g_dev[dev];
    const int grid = na.ctas;
    if (D == 128) {
        if (causal) return rope ? launch<128, true, true>(prm, grid, st, di) : launch<128, true, false>(prm, grid, st, di);
        return rope ? launch<128, false, true>(prm, grid, st, di) : launch<128, false, false>(prm, grid, st, di);
    }
    if (causal) return rope ? launch<64, true, true>(prm, grid, st, di) : launch<64, true, false>(prm, grid, st, di);
    return rope ? launch<64, false, true>(prm, grid, st, di) : launch<64, false, false>(prm, grid, st, di);
}

extern "C" int attn_build_tables(int S, int D, double rope_base, double window_k, long long pos_offset,
                                 float* cos_out, float* sin_out, int* win_out) {
    if (S < 1 || S > kMaxS || (D != 64 && D != 128)) return ATTN_ERR_SHAPE;
    if (!(rope_base > 0.0) || !std::isfinite(rope_base)) return ATTN_ERR_UNSUPPORTED;
    if (cos_out != nullptr || sin_out != nullptr) {
        const std::vector<float> t = attn_host::rope_table(S, D, rope_base, pos_offset);
        const size_t n = static_cast<size_t>(S) * (D / 2);
        for (size_t i = 0; i < n; ++i) {
            if (cos_out != nullptr) cos_out[i] = t[2 * i];
            if (sin_out != nullptr) sin_out[i] = t[2 * i + 1];
        }
    }
    if (win_out != nullptr) {
        const std::vector<int32_t> w = attn_host::window_widths(D, rope_base, window_k);
        for (int r = 0; r < D / 2; ++r) win_out[r] = w[r];
    }
    return ATTN_OK;
}

extern "C" int attn_check(void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    int v = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_attn_status, sizeof(int))) != cudaSuccess)
        return cuda_fail("cudaMemcpyFromSymbol(status word)", e);
    if (v != 0 && verbose()) std::fprintf(stderr, "attn: device status word 0x%x\n", v);
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int));
        return ATTN_ERR_TIMEOUT;
    }
    return ATTN_OK;
}

extern "C" const char* attn_error_string(int status) {
    switch (status) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_NULL: return "ATTN_ERR_NULL: a required pointer is NULL";
        case ATTN_ERR_SHAPE: return "ATTN_ERR_SHAPE: B, S, H or D out of range";
        case ATTN_ERR_ALIGN: return "ATTN_ERR_ALIGN: tensor pointer not 16-byte aligned";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: option combination not implemented";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: a CUDA call failed";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a bounded in-kernel wait ran out";
        case ATTN_ERR_OOM: return "ATTN_ERR_OOM: table allocation failed";
        case ATTN_ERR_NO_DEVICE: return "ATTN_ERR_NO_DEVICE: no sm_103 device is current";
        case ATTN_ERR_SCRATCH:
            return "ATTN_ERR_SCRATCH: the request needs more than the 16 MiB static scratch of attn_fwd_noalloc";
        default: return "unknown attn status";
    }
}

extern "C" void attn_release_cache(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = 0;
    const bool have = cudaGetDevice(&cur) == cudaSuccess;
    for (auto& e : g_rope) {
        cudaSetDevice(e.dev);
        cudaFree(e.table);
    }
    for (auto& e : g_sched) {
        cudaSetDevice(e.dev);
        cudaFree(e.tasks);
        cudaFree(e.offsets);
    }
    for (auto& e : g_win) {
        cudaSetDevice(e.dev);
        cudaFree(e.table);
    }
    g_rope.clear();
    g_sched.clear();
    g_win.clear();
    if (have) cudaSetDevice(cur);
}
