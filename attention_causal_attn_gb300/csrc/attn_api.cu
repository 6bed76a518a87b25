// C ABI of the fused RoPE + causal attention forward (declared in attn.h):
// argument checks, the per-device cache of RoPE tables and tile schedules,
// TMA descriptor encoding, and the launch of the sm_103a kernel.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "attn.h"
#include "attn_fwd_kernel.cuh"
#include "rope_rotate_kernel.cuh"
#include "decode_kernel.cuh"
#include "bwd_kernel.cuh"
#include "bs_fwd_kernel.cuh"
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
    int dev, B, Hq, Hkv, S, D, causal, ctas;
    uint2* tasks;
    int* offsets;
};
struct DevInfo {
    bool probed = false, ok = false;
    int sms = 0;
    int* status = nullptr;
    std::atomic<unsigned> configured{0};  // kernel variants whose smem attribute was set (bit per variant);
                                          // set by launches, which run outside the mutex
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
// K/V bytes per scheduling window of the forward's tile schedule: the built-in
// default, or ATTN_SCHEDULE_WINDOW_MB from the environment (read once; 0 turns
// the windows off).
double schedule_window_bytes() {
    static const double b = [] {
        const char* e = std::getenv("ATTN_SCHEDULE_WINDOW_MB");
        if (e == nullptr || e[0] == '\0') return attn_host::kScheduleWindowBytes;
        return std::max(0.0, std::atof(e)) * 1024.0 * 1024.0;
    }();
    return b;
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

int get_schedule(int dev, int B, int Hq, int Hkv, int S, int D, int causal, int sms, const SchedEntry** out) {
    for (auto& e : g_sched)
        if (e.dev == dev && e.B == B && e.Hq == Hq && e.Hkv == Hkv && e.S == S && e.D == D && e.causal == causal) {
            *out = &e;
            return ATTN_OK;
        }
    const attn_host::Schedule sc =
        attn_host::build_schedule(B, Hq, Hkv, S, D, causal != 0, sms, schedule_window_bytes());
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
    g_sched.push_back({dev, B, Hq, Hkv, S, D, causal, sc.ctas, tasks, offs});
    *out = &g_sched.back();
    return ATTN_OK;
}

template <int D, bool CAUSAL, bool ROPE, bool WINDOW = false>
int launch(const FwdParams& prm, int grid, cudaStream_t stream, DevInfo& di) {
    constexpr unsigned bit = 1u << ((WINDOW ? 8 : 0) | (D == 128 ? 4 : 0) | (CAUSAL ? 2 : 0) | (ROPE ? 1 : 0));
    auto kern = attn::attn_fwd_kernel<D, CAUSAL, ROPE, WINDOW>;
    // At least 120 KB so that only one CTA fits on an SM: each CTA takes all 512 TMEM columns.
    using Layout = attn::SmemLayout<D>;
    constexpr int smem = static_cast<int>(Layout::kAlloc) > 120 * 1024 ? static_cast<int>(Layout::kAlloc) : 120 * 1024;
    cudaError_t e;
    if (!(di.configured.load(std::memory_order_acquire) & bit)) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
            return cuda_fail("cudaFuncSetAttribute(max dynamic smem)", e);
        di.configured.fetch_or(bit, std::memory_order_release);
    }
    kern<<<grid, attn::kNumThreads, smem, stream>>>(prm);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail("kernel launch", e);
    return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace {
// Argument checks shared by the entry points (pointer alignment aside).
int check_args(const void* q, const void* k, const void* v, const void* o, int B, int Hq, int Hkv, int S, int D,
               int causal, double rope_base, double window_k) {
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return ATTN_ERR_NULL;
    if (B < 1 || B > 65535 || S < 1 || S > kMaxS || Hq < 1 || Hq > 255 || Hkv < 1 || Hkv > Hq || Hq % Hkv != 0)
        return ATTN_ERR_SHAPE;
    if (D != 64 && D != 128) return ATTN_ERR_SHAPE;
    if (causal != 0 && causal != 1) return ATTN_ERR_UNSUPPORTED;
    const bool rope = rope_base > 0.0 && std::isfinite(rope_base);
    if (rope_base > 0.0 && !std::isfinite(rope_base)) return ATTN_ERR_UNSUPPORTED;
    const bool window = window_k > 0.0 && !std::isinf(window_k);
    if (window && !(rope && causal)) return ATTN_ERR_UNSUPPORTED;
    if (std::isnan(window_k) || std::isnan(rope_base)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}
}  // namespace

namespace {
// The forward; qk_f16: Q and K hold fp16 values (already rotated) rather than bf16.
// test_no_loads: the bounded-wait test mode (the producer issues nothing), with
// wait_limit_ns per wait.
int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int S, int D,
             int causal, double rope_base, double window_k, void* stream, bool qk_f16, bool test_no_loads = false,
             unsigned long long wait_limit_ns = kWaitLimitNs) {
    int arc = check_args(q, k, v, o, B, Hq, Hkv, S, D, causal, rope_base, window_k);
    if (arc == ATTN_OK && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
                           (reinterpret_cast<uintptr_t>(lse) & 3u) != 0))
        arc = ATTN_ERR_ALIGN;
    if (arc != ATTN_OK) return arc;
    const bool rope = rope_base > 0.0 && std::isfinite(rope_base);
    const bool window = window_k > 0.0 && !std::isinf(window_k);

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
        if ((rc = get_schedule(dev, B, Hq, Hkv, S, D, causal, g_dev[dev].sms, &se)) != ATTN_OK) return rc;
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
    prm.wait_limit_ns = wait_limit_ns;
    prm.qk_f16 = qk_f16 ? 1 : 0;
    prm.test_no_loads = test_no_loads ? 1 : 0;

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
}  // namespace

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int S, int D, int causal, double rope_base, double window_k, void* stream) {
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, S, D, causal, rope_base, window_k, stream, false);
}

extern "C" int attn_selftest_wait_timeout(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                          int Hq, int Hkv, int S, int D, int causal, double rope_base,
                                          unsigned long long wait_limit_ns, void* stream) {
    if (wait_limit_ns < 100000ull || wait_limit_ns > kWaitLimitNs) return ATTN_ERR_UNSUPPORTED;
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, S, D, causal, rope_base, 0.0, stream, false, true, wait_limit_ns);
}

extern "C" int attn_fwd_rotated(const void* q_rot, const void* k_rot, const void* v, void* o, float* lse, int B,
                                int Hq, int Hkv, int S, int D, int causal, void* stream) {
    return fwd_impl(q_rot, k_rot, v, o, lse, B, Hq, Hkv, S, D, causal, 0.0, 0.0, stream, true);
}

// ---------------------------------------------------------------------------
// Pre-rotation pass ("AttnFuse", sec. 5.3, The Rotation Calculus).
namespace {
struct SplitEntry {
    int dev, S, D, block;
    double base;
    float2* table;
};
std::vector<SplitEntry> g_split;

int get_split(int dev, int S, int D, double base, int block, float2** out) {
    for (auto& e : g_split)
        if (e.dev == dev && e.S == S && e.D == D && e.block == block && e.base == base) {
            *out = e.table;
            return ATTN_OK;
        }
    const std::vector<float> host = attn_host::rope_split_tables(S, D, base, block);
    float2* d = nullptr;
    cudaError_t e;
    if ((e = cudaMalloc(&d, host.size() * sizeof(float))) != cudaSuccess)
        return cuda_fail("cudaMalloc(rotation tables)", e, ATTN_ERR_OOM);
    if ((e = cudaMemcpy(d, host.data(), host.size() * sizeof(float), cudaMemcpyHostToDevice)) != cudaSuccess) {
        cudaFree(d);
        return cuda_fail("cudaMemcpy(rotation tables)", e);
    }
    g_split.push_back({dev, S, D, block, base, d});
    *out = d;
    return ATTN_OK;
}
}  // namespace

extern "C" int attn_rope_rotate(const void* x, void* y, int B, int S, int H, int D, double rope_base, void* stream) {
    if (x == nullptr || y == nullptr) return ATTN_ERR_NULL;
    if (B < 1 || B > 65535 || S < 1 || S > kMaxS || H < 1 || H > 255 || (D != 64 && D != 128)) return ATTN_ERR_SHAPE;
    if (!(rope_base > 0.0) || !std::isfinite(rope_base)) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(y)) return ATTN_ERR_ALIGN;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;
    float2* tab = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int rc = probe_device(dev);
        if (rc != ATTN_OK) return rc;
        if ((rc = get_split(dev, S, D, rope_base, 128, &tab)) != ATTN_OK) return rc;
    }
    const long long rows = static_cast<long long>(B) * S * H;
    const long long threads = rows * (D / 16);
    const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
    const float2* base_tab = tab;
    const float2* row_tab = tab + static_cast<size_t>((S + 127) / 128) * (D / 2);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (D == 128)
        attn::rope_rotate_kernel<128><<<blocks, 256, 0, st>>>(static_cast<const uint4*>(x), static_cast<uint4*>(y),
                                                              base_tab, row_tab, rows, S, H);
    else
        attn::rope_rotate_kernel<64><<<blocks, 256, 0, st>>>(static_cast<const uint4*>(x), static_cast<uint4*>(y),
                                                             base_tab, row_tab, rows, S, H);
    cudaError_t e;
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail("rotation kernel launch", e);
    return ATTN_OK;
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
    // Recorded on the upload stream after the last upload; a launch on another
    // stream waits for it until the upload has been seen complete.
    cudaEvent_t uploaded = nullptr;
    cudaStream_t upload_stream = nullptr;
    bool upload_done = true;
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
    int arc = check_args(q, k, v, o, B, Hq, Hkv, S, D, causal, rope_base, window_k);
    if (arc == ATTN_OK && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
                           (reinterpret_cast<uintptr_t>(lse) & 3u) != 0))
        arc = ATTN_ERR_ALIGN;
    if (arc != ATTN_OK) return arc;
    const bool rope = rope_base > 0.0 && std::isfinite(rope_base);
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
        // once per device, with that device current (an event allocates no device memory)
        if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&na.scratch), g_noalloc_scratch)) != cudaSuccess)
            return cuda_fail("cudaGetSymbolAddress(no-alloc scratch)", e);
        if ((e = cudaEventCreateWithFlags(&na.uploaded, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail("cudaEventCreateWithFlags(no-alloc upload)", e);
        na.ready = true;
    }
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(st, &capture)) != cudaSuccess) return cuda_fail("cudaStreamIsCapturing", e);
    const bool capturing = capture != cudaStreamCaptureStatusNone;
    const bool same = na.have && na.S == S && na.D == D && na.B == B && na.Hq == Hq && na.Hkv == Hkv &&
                      na.causal == causal && na.rope == static_cast<int>(rope) && (!rope || na.base == rope_base);
    // An upload enqueues copies from host vectors that end with this call: not
    // while the stream is being captured.
    if (!same && capturing) return ATTN_ERR_UNSUPPORTED;
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
        const attn_host::Schedule sc =
            attn_host::build_schedule(B, Hq, Hkv, S, D, causal != 0, g_dev[dev].sms, schedule_window_bytes());
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
        if ((e = cudaEventRecord(na.uploaded, st)) != cudaSuccess) return cuda_fail("cudaEventRecord(no-alloc upload)", e);
        na.upload_stream = st;
        na.upload_done = false;
        na.have = true;
        na.S = S, na.D = D, na.B = B, na.Hq = Hq, na.Hkv = Hkv, na.causal = causal;
        na.rope = static_cast<int>(rope), na.base = rope_base, na.ctas = sc.ctas;
        na.off_tasks = off_tasks, na.off_offsets = off_offsets;
    }

    if (!na.upload_done && st != na.upload_stream) {
        // The tables were enqueued on another stream: this launch must not start before they land.
        if (capturing) return ATTN_ERR_UNSUPPORTED;
        e = cudaEventQuery(na.uploaded);
        if (e == cudaSuccess) {
            na.upload_done = true;
        } else if (e == cudaErrorNotReady) {
            if ((e = cudaStreamWaitEvent(st, na.uploaded, 0)) != cudaSuccess)
                return cuda_fail("cudaStreamWaitEvent(no-alloc upload)", e);
        } else {
            return cuda_fail("cudaEventQuery(no-alloc upload)", e);
        }
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
    prm.qk_f16 = 0;
    prm.test_no_loads = 0;
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

// ---------------------------------------------------------------------------
// Host-buffer forward: chunks of (batch, KV heads) go host -> device, through
// attn_fwd and back while the neighbouring chunks move, on three streams.
namespace {
struct HostPipe {
    size_t slot_bytes = 0;   // one staging slot: q, k, v, o, lse of the largest chunk
    uint8_t* buf = nullptr;  // two slots
    cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
    cudaEvent_t ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {};
    bool ready = false;
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;

// `rows` rows of `width` bytes, `pitch` bytes apart in host memory, to or from a
// packed device buffer (one plain copy when the rows are contiguous).
cudaError_t copy_rows(void* dst_packed, const void* src, size_t width, size_t pitch, int rows, cudaMemcpyKind kind,
                      cudaStream_t st) {
    if (width == pitch) return cudaMemcpyAsync(dst_packed, src, width * rows, kind, st);
    return cudaMemcpy2DAsync(dst_packed, width, src, pitch, width, rows, kind, st);
}
cudaError_t copy_rows_out(void* dst, size_t pitch, const void* src_packed, size_t width, int rows, cudaStream_t st) {
    if (width == pitch) return cudaMemcpyAsync(dst, src_packed, width * rows, cudaMemcpyDeviceToHost, st);
    return cudaMemcpy2DAsync(dst, pitch, src_packed, width, width, rows, cudaMemcpyDeviceToHost, st);
}

int pipe_setup(HostPipe& hp, size_t slot_bytes) {
    cudaError_t e;
    if (!hp.ready) {
        if ((e = cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&hp.s_comp, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail("cudaStreamCreate(host pipeline)", e);
        for (int i = 0; i < 2; ++i)
            if ((e = cudaEventCreateWithFlags(&hp.ev_in[i], cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&hp.ev_comp[i], cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&hp.ev_out[i], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail("cudaEventCreate(host pipeline)", e);
        hp.ready = true;
    }
    if (hp.slot_bytes < slot_bytes) {
        if (hp.buf != nullptr) {
            cudaFree(hp.buf);
            hp.buf = nullptr;
            hp.slot_bytes = 0;
        }
        if ((e = cudaMalloc(&hp.buf, 2 * slot_bytes)) != cudaSuccess)
            return cuda_fail("cudaMalloc(host pipeline staging)", e, ATTN_ERR_OOM);
        hp.slot_bytes = slot_bytes;
    }
    return ATTN_OK;
}
}  // namespace

extern "C" int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                             int Hkv, int S, int D, int causal, double rope_base, double window_k) {
    const int arc = check_args(q, k, v, o, B, Hq, Hkv, S, D, causal, rope_base, window_k);
    if (arc != ATTN_OK) return arc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_NO_DEVICE;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;

    int sms = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);  // released before the pipeline's lock (lock order)
        if (int rc0 = probe_device(dev); rc0 != ATTN_OK) return rc0;
        sms = g_dev[dev].sms;
    }
    // Chunks: one batch element and a group of KV heads (with their query heads).
    // Up to eight per call, so that the copies of the first chunk in and the last
    // one out (which nothing overlaps) stay short, but each chunk keeps at least
    // two work units per SM for the kernel's load balance.
    const int G = Hq / Hkv;
    const long long nqt = (S + 127) / 128;
    auto units_for = [&](int hkv) {
        return G >= 2 ? static_cast<long long>(hkv) * nqt * ((G + 1) / 2) : static_cast<long long>(hkv) * ((nqt + 1) / 2);
    };
    int groups = std::max(1, std::min(Hkv, (8 + B - 1) / B));
    while (groups > 1 && units_for(Hkv / groups) < 2LL * sms) --groups;
    const int gmax = (Hkv + groups - 1) / groups;
    const size_t e2 = 2;  // bytes per bf16 element
    const size_t q_bytes = align256(static_cast<size_t>(S) * gmax * G * D * e2);
    const size_t kv_bytes = align256(static_cast<size_t>(S) * gmax * D * e2);
    const size_t lse_bytes = align256(static_cast<size_t>(gmax) * G * S * sizeof(float));
    const size_t slot_bytes = 2 * q_bytes + 2 * kv_bytes + lse_bytes;  // q, o, k, v, lse

    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe& hp = g_pipe[dev];
    int rc = pipe_setup(hp, slot_bytes);
    if (rc != ATTN_OK) return rc;
    const char* hq = static_cast<const char*>(q);
    const char* hk = static_cast<const char*>(k);
    const char* hv = static_cast<const char*>(v);
    char* ho = static_cast<char*>(o);
    // The chunk list: equal chunks, except that the last is cut into up to four
    // pieces.  The input copies run back to back on one copy engine and the kernels
    // hide behind them, so what shows is the last chunk's compute and copy out.
    struct Chunk {
        int b, g0, g1;
    };
    std::vector<Chunk> chunks;
    for (int b = 0; b < B; ++b)
        for (int gi = 0; gi < groups; ++gi) {
            const int g0 = Hkv * gi / groups, g1 = Hkv * (gi + 1) / groups;
            if (g1 > g0) chunks.push_back({b, g0, g1});
        }
    if (!chunks.empty()) {
        const Chunk last = chunks.back();
        const int pieces = std::min(4, last.g1 - last.g0);
        chunks.pop_back();
        for (int i = 0; i < pieces; ++i)
            chunks.push_back({last.b, last.g0 + (last.g1 - last.g0) * i / pieces,
                              last.g0 + (last.g1 - last.g0) * (i + 1) / pieces});
    }
    cudaError_t e = cudaSuccess;
    for (int c = 0; c < static_cast<int>(chunks.size()) && rc == ATTN_OK; ++c) {
        const int b = chunks[c].b, g0 = chunks[c].g0, g1 = chunks[c].g1;
        const int hkv = g1 - g0, hq_n = hkv * G, h0 = g0 * G;
        const int slot = c & 1;
        uint8_t* base = hp.buf + slot * hp.slot_bytes;
        uint8_t* dq = base;
        uint8_t* dout = base + q_bytes;
        uint8_t* dk = base + 2 * q_bytes;
        uint8_t* dv = dk + kv_bytes;
        float* dl = reinterpret_cast<float*>(dv + kv_bytes);
        const size_t row_q = static_cast<size_t>(Hq) * D * e2, row_kv = static_cast<size_t>(Hkv) * D * e2;
        const size_t w_q = static_cast<size_t>(hq_n) * D * e2, w_kv = static_cast<size_t>(hkv) * D * e2;
        const size_t off_q = (static_cast<size_t>(b) * S * Hq + h0) * D * e2;
        const size_t off_kv = (static_cast<size_t>(b) * S * Hkv + g0) * D * e2;
        // in: the slot's previous chunk must have been read by its kernel
        if (c >= 2 && (e = cudaStreamWaitEvent(hp.s_in, hp.ev_comp[slot], 0)) != cudaSuccess) break;
        if ((e = copy_rows(dq, hq + off_q, w_q, row_q, S, cudaMemcpyHostToDevice, hp.s_in)) != cudaSuccess ||
            (e = copy_rows(dk, hk + off_kv, w_kv, row_kv, S, cudaMemcpyHostToDevice, hp.s_in)) != cudaSuccess ||
            (e = copy_rows(dv, hv + off_kv, w_kv, row_kv, S, cudaMemcpyHostToDevice, hp.s_in)) != cudaSuccess ||
            (e = cudaEventRecord(hp.ev_in[slot], hp.s_in)) != cudaSuccess)
            break;
        // compute: after the inputs landed and the slot's previous outputs left
        if ((e = cudaStreamWaitEvent(hp.s_comp, hp.ev_in[slot], 0)) != cudaSuccess) break;
        if (c >= 2 && (e = cudaStreamWaitEvent(hp.s_comp, hp.ev_out[slot], 0)) != cudaSuccess) break;
        rc = attn_fwd(dq, dk, dv, dout, lse != nullptr ? dl : nullptr, 1, hq_n, hkv, S, D, causal, rope_base,
                      window_k, hp.s_comp);
        if (rc != ATTN_OK) break;
        if ((e = cudaEventRecord(hp.ev_comp[slot], hp.s_comp)) != cudaSuccess) break;
        // out
        if ((e = cudaStreamWaitEvent(hp.s_out, hp.ev_comp[slot], 0)) != cudaSuccess ||
            (e = copy_rows_out(ho + off_q, row_q, dout, w_q, S, hp.s_out)) != cudaSuccess)
            break;
        if (lse != nullptr &&
            (e = cudaMemcpyAsync(lse + (static_cast<size_t>(b) * Hq + h0) * S, dl,
                                 static_cast<size_t>(hq_n) * S * sizeof(float), cudaMemcpyDeviceToHost,
                                 hp.s_out)) != cudaSuccess)
            break;
        if ((e = cudaEventRecord(hp.ev_out[slot], hp.s_out)) != cudaSuccess) break;
    }
    // the call returns once every chunk is back in host memory
    const cudaError_t e_sync = cudaStreamSynchronize(hp.s_out);
    cudaStreamSynchronize(hp.s_comp);
    cudaStreamSynchronize(hp.s_in);
    if (rc != ATTN_OK) return rc;
    if (e != cudaSuccess) return cuda_fail("host pipeline", e);
    if (e_sync != cudaSuccess) return cuda_fail("cudaStreamSynchronize(host pipeline)", e_sync);
    return attn_check(hp.s_comp);
}

// ---------------------------------------------------------------------------
// Split-KV decode ("AttnFuse", sec. 4.2 Decode; "ATFlash", decode window).
namespace {
struct DecodeScratch {
    size_t floats = 0;
    float* buf = nullptr;
};
DecodeScratch g_dec[kMaxDevices];
int g_dec_occ[kMaxDevices][2][3];  // resident split CTAs per SM, by [D == 128][variant], 0 = not yet queried

using DecodeKernel = void (*)(attn::DecodeParams);

template <int D>
DecodeKernel decode_kernel(int variant) {  // 0: RoPE off, 1: RoPE, 2: RoPE + window
    if (variant == 0) return attn::decode_split_kernel<D, false, false>;
    if (variant == 1) return attn::decode_split_kernel<D, true, false>;
    return attn::decode_split_kernel<D, true, true>;
}

// Opt the split kernel into its shared memory and read its residency (caller holds g_mu).
int decode_occupancy(int dev, int D, int variant, int* occ) {
    int& cached = g_dec_occ[dev][D == 128][variant];
    if (cached == 0) {
        const DecodeKernel kern = D == 128 ? decode_kernel<128>(variant) : decode_kernel<64>(variant);
        const int smem = D == 128 ? attn::decode_smem_bytes<128>() : attn::decode_smem_bytes<64>();
        cudaError_t e;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
            return cuda_fail("cudaFuncSetAttribute(decode)", e);
        int n = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, attn::kDecThreads, smem)) != cudaSuccess)
            return cuda_fail("cudaOccupancyMaxActiveBlocksPerMultiprocessor(decode)", e);
        cached = std::max(1, n);
    }
    *occ = cached;
    return ATTN_OK;
}
}  // namespace

extern "C" int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                           int S, int D, double rope_base, double window_k, void* stream) {
    int arc = check_args(q, k, v, o, B, Hq, Hkv, S, D, 1, rope_base, window_k);
    if (arc == ATTN_OK && Hq / Hkv > attn::kDecMaxGroup) arc = ATTN_ERR_UNSUPPORTED;
    if (arc == ATTN_OK && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
                           (reinterpret_cast<uintptr_t>(lse) & 3u) != 0))
        arc = ATTN_ERR_ALIGN;
    if (arc != ATTN_OK) return arc;
    const bool rope = rope_base > 0.0 && std::isfinite(rope_base);
    const bool window = window_k > 0.0 && !std::isinf(window_k);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;

    // Splits are whole multiples of 128 keys (one 32-key tile per warp).  Among split counts up to
    // about two waves of resident CTAs, take the one with the least estimated time, counted as
    // waves x tiles per split.
    const int tile = attn::kDecWarps * attn::kDecTile;
    const int variant = !rope ? 0 : (window ? 2 : 1);
    const int mtiles = (Hq / Hkv + attn::kDecHeads - 1) / attn::kDecHeads;
    float2* tab = nullptr;
    float* scratch = nullptr;
    int nsplit = 1, split_len = S;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int rc = probe_device(dev);
        if (rc != ATTN_OK) return rc;
        if (rope && (rc = get_split(dev, S, D, rope_base, attn::kDecTile, &tab)) != ATTN_OK) return rc;
        int occ = 1;
        if ((rc = decode_occupancy(dev, D, variant, &occ)) != ATTN_OK) return rc;
        const long long slots = static_cast<long long>(occ) * g_dev[dev].sms;
        const long long units = static_cast<long long>(B) * Hkv * mtiles;
        const int tiles = (S + tile - 1) / tile;
        const long long cap = std::max(
            1LL, std::min<long long>({static_cast<long long>(tiles), (2 * slots + units - 1) / units,
                                      static_cast<long long>(attn::kDecMaxParts)}));
        long long best = -1;
        for (long long n = 1; n <= cap; ++n) {
            const int per = static_cast<int>((tiles + n - 1) / n);  // tiles per split
            const long long used = (tiles + per - 1) / per;         // splits actually made
            const long long waves = (used * units + slots - 1) / slots;
            const long long cost = waves * per;
            if (best < 0 || cost < best) {
                best = cost;
                nsplit = static_cast<int>(used);
                split_len = per * tile;
            }
        }
        const size_t need = static_cast<size_t>(B) * Hq * nsplit * (D + 2);
        DecodeScratch& ds = g_dec[dev];
        if (ds.floats < need) {
            if (ds.buf != nullptr) cudaFree(ds.buf);
            ds.buf = nullptr;
            ds.floats = 0;
            cudaError_t e;
            if ((e = cudaMalloc(&ds.buf, need * sizeof(float))) != cudaSuccess)
                return cuda_fail("cudaMalloc(decode partials)", e, ATTN_ERR_OOM);
            ds.floats = need;
        }
        scratch = ds.buf;
    }
    attn::DecodeParams dp;
    dp.q = static_cast<const __nv_bfloat16*>(q);
    dp.k = static_cast<const __nv_bfloat16*>(k);
    dp.v = static_cast<const __nv_bfloat16*>(v);
    dp.part_o = scratch;
    dp.part_ml = scratch + static_cast<size_t>(B) * Hq * nsplit * D;
    dp.rot_base = rope ? tab : nullptr;
    dp.rot_row = rope ? tab + static_cast<size_t>((S + attn::kDecTile - 1) / attn::kDecTile) * (D / 2) : nullptr;
    dp.B = B;
    dp.Hq = Hq;
    dp.Hkv = Hkv;
    dp.S = S;
    dp.nsplit = nsplit;
    dp.split_len = split_len;
    dp.mtiles = mtiles;
    dp.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    {
        const std::vector<int32_t> w = attn_host::window_widths(D, rope ? rope_base : 10000.0, window ? window_k : 0.0);
        for (int r = 0; r < 64; ++r) dp.win[r] = r < D / 2 ? w[r] : INT32_MAX;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid(static_cast<unsigned>(nsplit * mtiles), static_cast<unsigned>(B * Hkv));
    if (D == 128)
        decode_kernel<128>(variant)<<<grid, attn::kDecThreads, attn::decode_smem_bytes<128>(), st>>>(dp);
    else
        decode_kernel<64>(variant)<<<grid, attn::kDecThreads, attn::decode_smem_bytes<64>(), st>>>(dp);
    cudaError_t e;
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail("decode split kernel launch", e);
    const unsigned rows = static_cast<unsigned>(B * Hq);
    if (D == 128)
        attn::decode_combine_kernel<128><<<rows, 128, 0, st>>>(dp.part_o, dp.part_ml, static_cast<__nv_bfloat16*>(o), lse,
                                                             nsplit);
    else
        attn::decode_combine_kernel<64><<<rows, 128, 0, st>>>(dp.part_o, dp.part_ml, static_cast<__nv_bfloat16*>(o), lse,
                                                            nsplit);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail("decode combine kernel launch", e);
    return ATTN_OK;
}

// ---------------------------------------------------------------------------
// Backward ("AttnFuse", sec. 4.4 Backward Pass: row reduction, dK/dV, dQ).
namespace {
DecodeScratch g_bwd[kMaxDevices];  // Dlt rows, [B][Hq][S] floats
// RoPE: Q and K rotated once before the backward's tile kernels (fp16, the layouts of Q and K)
struct RotScratch {
    void* buf = nullptr;
    size_t bytes = 0;
};
RotScratch g_bwd_rot[kMaxDevices];
// as DevInfo::configured, for the backward (bits 0-7, local 32-39) and block-sparse (8-31) kernels
std::atomic<unsigned long long> g_bwd_configured[kMaxDevices];

template <int D, bool CAUSAL, bool ROPE, bool EXT = false>
int launch_bwd(const attn::BwdParams& bp, int dev, int ntiles, cudaStream_t st) {
    using L = attn::BwdLayout<D>;
    // at least 120 KB so that one CTA fits on an SM: each CTA takes all 512 TMEM columns
    constexpr int smem = static_cast<int>(L::kAlloc) > 120 * 1024 ? static_cast<int>(L::kAlloc) : 120 * 1024;
    constexpr unsigned long long bit = 1ull << ((EXT ? 32 : 0) + ((D == 128 ? 2 : 0) | (CAUSAL ? 1 : 0) | (ROPE ? 4 : 0)));
    auto kv = attn::bwd_dkdv_kernel<D, CAUSAL, ROPE, EXT>;
    auto kq = attn::bwd_dq_kernel<D, CAUSAL, ROPE, EXT>;
    cudaError_t e;
    if (!(g_bwd_configured[dev].load(std::memory_order_acquire) & bit)) {
        if ((e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
            return cuda_fail("cudaFuncSetAttribute(backward)", e);
        g_bwd_configured[dev].fetch_or(bit, std::memory_order_release);
    }
    const int B = bp.f.B, Hq = bp.f.Hq, Hkv = bp.f.Hkv;
    kv<<<static_cast<unsigned>(static_cast<long long>(B) * Hkv * ntiles), attn::kBwdThreads, smem, st>>>(bp);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail("dK/dV kernel launch", e);
    kq<<<static_cast<unsigned>(static_cast<long long>(B) * Hq * ntiles), attn::kBwdThreads, smem, st>>>(bp);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail("dQ kernel launch", e);
    return ATTN_OK;
}
}  // namespace

int check_mask(const int* row_ptr, const int* col_idx, int nrows, bool causal);
namespace {
struct MaskEntry;
}
int get_mask(int dev, const int* row_ptr, const int* col_idx, int nrows, int** out, MaskEntry** entry = nullptr);

// The backward; row_ptr / col_idx: an optional host CSR block mask (null: dense); ext: the local
// kernels, with the sliding window (window > 0) and ALiBi (alibi = 1) of the local forward.
int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dq,
             void* dk, void* dv, int B, int Hq, int Hkv, int S, int D, int causal, double rope_base,
             const int* row_ptr, const int* col_idx, void* stream, bool ext = false, int window = 0, int alibi = 0) {
    int arc = check_args(q, k, v, o, B, Hq, Hkv, S, D, causal, rope_base, 0.0);
    const int ntiles = (S + 127) / 128;
    if (arc == ATTN_OK && row_ptr != nullptr) arc = check_mask(row_ptr, col_idx, ntiles, causal != 0);
    if (arc == ATTN_OK && (dO == nullptr || lse == nullptr || dq == nullptr || dk == nullptr || dv == nullptr))
        arc = ATTN_ERR_NULL;
    if (arc == ATTN_OK && static_cast<long long>(B) * Hq * ((S + 127) / 128) > INT_MAX) arc = ATTN_ERR_SHAPE;  // CTAs
    if (arc == ATTN_OK && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
                           !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
                           (reinterpret_cast<uintptr_t>(lse) & 3u) != 0))
        arc = ATTN_ERR_ALIGN;
    if (arc != ATTN_OK) return arc;
    const bool rope = rope_base > 0.0 && std::isfinite(rope_base);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;

    attn::BwdParams bp;
    float2* rope_tab = nullptr;
    float2* split_tab = nullptr;
    float2* rot_tab = nullptr;  // the rotation pass's tables (128-row blocks)
    uint8_t* qk_rot = nullptr;  // rotated Q, then rotated K
    float* dlt = nullptr;
    int* mask = nullptr;
    const int nnz = row_ptr != nullptr ? row_ptr[ntiles] : 0;
    const size_t rows = static_cast<size_t>(B) * Hq * S;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int rc = probe_device(dev);
        if (rc != ATTN_OK) return rc;
        if (rope && ((rc = get_rope(dev, S, D, rope_base, &rope_tab)) != ATTN_OK ||
                     (rc = get_split(dev, S, D, rope_base, 32, &split_tab)) != ATTN_OK ||
                     (rc = get_split(dev, S, D, rope_base, 128, &rot_tab)) != ATTN_OK))
            return rc;
        if (rope) {
            RotScratch& rs = g_bwd_rot[dev];
            const size_t need = static_cast<size_t>(B) * S * (Hq + Hkv) * D * 2;
            if (rs.bytes < need) {
                if (rs.buf != nullptr) cudaFree(rs.buf);
                rs.buf = nullptr;
                rs.bytes = 0;
                cudaError_t e;
                if ((e = cudaMalloc(&rs.buf, need)) != cudaSuccess)
                    return cuda_fail("cudaMalloc(backward rotated Q, K)", e, ATTN_ERR_OOM);
                rs.bytes = need;
            }
            qk_rot = static_cast<uint8_t*>(rs.buf);
        }
        DecodeScratch& ds = g_bwd[dev];
        if (ds.floats < rows) {
            if (ds.buf != nullptr) cudaFree(ds.buf);
            ds.buf = nullptr;
            ds.floats = 0;
            cudaError_t e;
            if ((e = cudaMalloc(&ds.buf, rows * sizeof(float))) != cudaSuccess)
                return cuda_fail("cudaMalloc(backward rows)", e, ATTN_ERR_OOM);
            ds.floats = rows;
        }
        dlt = ds.buf;
        if (row_ptr != nullptr && (rc = get_mask(dev, row_ptr, col_idx, ntiles, &mask)) != ATTN_OK) return rc;
        bp.f.status = g_dev[dev].status;
    }
    // With RoPE the tile kernels read Q and K rotated once by the rotation pass (fp16): each Q tile
    // is used by every key tile of its head and each K tile by every query tile, so rotating
    // inside the loops would repeat each rotation about S/256 times ("AttnFuse", sec. 5.3).
    const void* q_in = rope ? static_cast<const void*>(qk_rot) : q;
    const void* k_in = rope ? static_cast<const void*>(qk_rot + static_cast<size_t>(B) * S * Hq * D * 2) : k;
    if (!encode_bshd(&bp.f.tm_q, q_in, B, S, Hq, D) || !encode_bshd(&bp.f.tm_k, k_in, B, S, Hkv, D) ||
        !encode_bshd(&bp.f.tm_v, v, B, S, Hkv, D) || !encode_bshd(&bp.tm_do, dO, B, S, Hq, D))
        return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
    bp.prerot = rope ? 1 : 0;
    bp.f.rope = rope_tab;
    bp.f.B = B;
    bp.f.Hq = Hq;
    bp.f.Hkv = Hkv;
    bp.f.S = S;
    bp.f.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    bp.f.wait_limit_ns = kWaitLimitNs;
    bp.lse = lse;
    bp.dlt = dlt;
    bp.dq = static_cast<__nv_bfloat16*>(dq);
    bp.dk = static_cast<__nv_bfloat16*>(dk);
    bp.dv = static_cast<__nv_bfloat16*>(dv);
    bp.rot_base = rope ? split_tab : nullptr;
    bp.rot_row = rope ? split_tab + static_cast<size_t>((S + 31) / 32) * (D / 2) : nullptr;
    bp.inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
    bp.head_major = mask == nullptr ? 1 : 0;
    bp.q_ptr = mask;
    bp.q_idx = mask != nullptr ? mask + ntiles + 1 : nullptr;
    bp.k_ptr = mask != nullptr ? mask + ntiles + 1 + nnz : nullptr;
    bp.k_idx = mask != nullptr ? mask + 2 * (ntiles + 1) + nnz : nullptr;
    bp.window = window;
    bp.alibi = alibi;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long dot_rows = D == 128 ? attn::dot_rows_per_block<128>() : attn::dot_rows_per_block<64>();
    const unsigned dot_blocks = static_cast<unsigned>((static_cast<long long>(rows) + dot_rows - 1) / dot_rows);
    if (D == 128)
        attn::bwd_dot_kernel<128><<<dot_blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(o),
                                                                static_cast<const __nv_bfloat16*>(dO), dlt, B, S, Hq);
    else
        attn::bwd_dot_kernel<64><<<dot_blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(o),
                                                               static_cast<const __nv_bfloat16*>(dO), dlt, B, S, Hq);
    cudaError_t e;
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail("backward row-reduction launch", e);
    if (rope) {
        const float2* row_tab = rot_tab + static_cast<size_t>(ntiles) * (D / 2);
        for (int which = 0; which < 2; ++which) {
            const int H = which ? Hkv : Hq;
            const long long nrows = static_cast<long long>(B) * S * H;
            const unsigned blocks = static_cast<unsigned>((nrows * (D / 16) + 255) / 256);
            const uint4* src = static_cast<const uint4*>(which ? k : q);
            uint4* dst = reinterpret_cast<uint4*>(const_cast<void*>(which ? k_in : q_in));
            if (D == 128)
                attn::rope_rotate_kernel<128><<<blocks, 256, 0, st>>>(src, dst, rot_tab, row_tab, nrows, S, H);
            else
                attn::rope_rotate_kernel<64><<<blocks, 256, 0, st>>>(src, dst, rot_tab, row_tab, nrows, S, H);
            if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail("backward rotation launch", e);
        }
    }
    if (ext) {
        if (D == 128) {
            if (causal) return rope ? launch_bwd<128, true, true, true>(bp, dev, ntiles, st) : launch_bwd<128, true, false, true>(bp, dev, ntiles, st);
            return rope ? launch_bwd<128, false, true, true>(bp, dev, ntiles, st) : launch_bwd<128, false, false, true>(bp, dev, ntiles, st);
        }
        if (causal) return rope ? launch_bwd<64, true, true, true>(bp, dev, ntiles, st) : launch_bwd<64, true, false, true>(bp, dev, ntiles, st);
        return rope ? launch_bwd<64, false, true, true>(bp, dev, ntiles, st) : launch_bwd<64, false, false, true>(bp, dev, ntiles, st);
    }
    if (D == 128) {
        if (causal) return rope ? launch_bwd<128, true, true>(bp, dev, ntiles, st) : launch_bwd<128, true, false>(bp, dev, ntiles, st);
        return rope ? launch_bwd<128, false, true>(bp, dev, ntiles, st) : launch_bwd<128, false, false>(bp, dev, ntiles, st);
    }
    if (causal) return rope ? launch_bwd<64, true, true>(bp, dev, ntiles, st) : launch_bwd<64, true, false>(bp, dev, ntiles, st);
    return rope ? launch_bwd<64, false, true>(bp, dev, ntiles, st) : launch_bwd<64, false, false>(bp, dev, ntiles, st);
}

// ---------------------------------------------------------------------------
// Block-sparse forward ("AttnFuse", sec. 4.3 Block-Sparse Attention).
namespace {
struct MaskSched {
    long long bh;
    int ctas;
    int* d;  // tasks | offsets (2 ctas + 1)
};
struct MaskEntry {
    int dev;
    std::vector<int> csr;  // row_ptr then col_idx, as given
    int* d = nullptr;      // row_ptr | col_idx | col_ptr | row_idx (the same mask by columns)
    std::vector<MaskSched> sched;  // persistent forward schedules, by batch-heads
};
std::vector<MaskEntry> g_masks;  // device copies of the block masks seen, by content
}  // namespace

// A CSR block mask over nrows x nrows tiles: row_ptr[0] = 0, non-decreasing; each row's columns
// ascending, distinct, in range, and at most the row with the causal mask (tiles above the
// diagonal hold no visible key).
int check_mask(const int* row_ptr, const int* col_idx, int nrows, bool causal) {
    if (row_ptr[0] != 0) return ATTN_ERR_SHAPE;
    for (int r = 0; r < nrows; ++r) {
        if (row_ptr[r + 1] < row_ptr[r]) return ATTN_ERR_SHAPE;
        for (int e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
            if (col_idx == nullptr) return ATTN_ERR_NULL;
            const int cidx = col_idx[e];
            if (cidx < 0 || cidx >= nrows || (causal && cidx > r) || (e > row_ptr[r] && cidx <= col_idx[e - 1]))
                return ATTN_ERR_SHAPE;
        }
    }
    return ATTN_OK;
}

// The device copy of a (checked) mask, with its column-major form; caller holds g_mu.
int get_mask(int dev, const int* row_ptr, const int* col_idx, int nrows, int** out, MaskEntry** entry) {
    const int nnz = row_ptr[nrows];
    for (auto& e : g_masks) {
        if (e.dev != dev || e.csr.size() != static_cast<size_t>(nrows + 1 + nnz)) continue;
        if (std::equal(row_ptr, row_ptr + nrows + 1, e.csr.begin()) &&
            std::equal(col_idx, col_idx + nnz, e.csr.begin() + nrows + 1)) {
            *out = e.d;
            if (entry != nullptr) *entry = &e;
            return ATTN_OK;
        }
    }
    MaskEntry me;
    me.dev = dev;
    me.csr.assign(row_ptr, row_ptr + nrows + 1);
    me.csr.insert(me.csr.end(), col_idx, col_idx + nnz);
    // by columns: col_ptr[c] .. col_ptr[c+1] list the rows that list c, ascending
    std::vector<int> all(me.csr);
    std::vector<int> col_ptr(nrows + 1, 0), row_idx(nnz);
    for (int e = 0; e < nnz; ++e) ++col_ptr[col_idx[e] + 1];
    for (int c = 0; c < nrows; ++c) col_ptr[c + 1] += col_ptr[c];
    std::vector<int> fill(col_ptr.begin(), col_ptr.end() - 1);
    for (int r = 0; r < nrows; ++r)
        for (int e = row_ptr[r]; e < row_ptr[r + 1]; ++e) row_idx[fill[col_idx[e]]++] = r;
    all.insert(all.end(), col_ptr.begin(), col_ptr.end());
    all.insert(all.end(), row_idx.begin(), row_idx.end());
    cudaError_t e;
    if ((e = cudaMalloc(&me.d, all.size() * sizeof(int))) != cudaSuccess)
        return cuda_fail("cudaMalloc(block mask)", e, ATTN_ERR_OOM);
    if ((e = cudaMemcpy(me.d, all.data(), all.size() * sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess) {
        cudaFree(me.d);
        return cuda_fail("cudaMemcpy(block mask)", e);
    }
    *out = me.d;
    g_masks.push_back(std::move(me));
    if (entry != nullptr) *entry = &g_masks.back();
    return ATTN_OK;
}

// The persistent block-sparse forward's task lists for a mask and B * Hq, built once
// (attn_host::build_mask_schedule) and kept on the device; caller holds g_mu.
int get_mask_sched(int dev, MaskEntry& me, int nrows, long long bh, const MaskSched** out) {
    for (auto& s : me.sched)
        if (s.bh == bh) {
            *out = &s;
            return ATTN_OK;
        }
    const attn_host::MaskSchedule sc = attn_host::build_mask_schedule(me.csr.data(), nrows, bh, g_dev[dev].sms);
    std::vector<int> all(sc.tasks.begin(), sc.tasks.end());
    all.insert(all.end(), sc.offsets.begin(), sc.offsets.end());
    MaskSched ms{bh, sc.ctas, nullptr};
    cudaError_t e;
    if ((e = cudaMalloc(&ms.d, all.size() * sizeof(int))) != cudaSuccess)
        return cuda_fail("cudaMalloc(block-sparse schedule)", e, ATTN_ERR_OOM);
    if ((e = cudaMemcpy(ms.d, all.data(), all.size() * sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess) {
        cudaFree(ms.d);
        return cuda_fail("cudaMemcpy(block-sparse schedule)", e);
    }
    me.sched.push_back(ms);
    *out = &me.sched.back();
    return ATTN_OK;
}

namespace {

template <int D, bool CAUSAL, bool ROPE, int EXT = 0>
int launch_bs(const attn::BsParams& bp, int dev, int ctas, cudaStream_t st) {
    constexpr int kMin = 120 * 1024;  // one CTA per SM: each takes all 512 TMEM columns
    constexpr int smem = static_cast<int>(attn::BsLayout<D>::kAlloc) > kMin ? static_cast<int>(attn::BsLayout<D>::kAlloc) : kMin;
    constexpr unsigned long long bit = 1ull << (8 + 8 * EXT + (D == 128 ? 2 : 0) + (CAUSAL ? 1 : 0) + (ROPE ? 4 : 0));
    auto kern = attn::bs_fwd_kernel<D, CAUSAL, ROPE, EXT>;
    cudaError_t e;
    if (!(g_bwd_configured[dev].load(std::memory_order_acquire) & bit)) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
            return cuda_fail("cudaFuncSetAttribute(block-sparse)", e);
        g_bwd_configured[dev].fetch_or(bit, std::memory_order_release);
    }
    kern<<<static_cast<unsigned>(ctas), attn::kBsThreads, smem, st>>>(bp);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail("block-sparse kernel launch", e);
    return ATTN_OK;
}
}  // namespace

// The block-sparse forward, with the sliding window and ALiBi of the EXT variant when `ext`.
int bs_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int S, int D,
            int causal, double rope_base, const int* row_ptr, const int* col_idx, bool ext, int window, int alibi,
            void* stream) {
    int arc = check_args(q, k, v, o, B, Hq, Hkv, S, D, causal, rope_base, 0.0);
    if (arc == ATTN_OK && row_ptr == nullptr) arc = ATTN_ERR_NULL;
    if (arc == ATTN_OK && static_cast<long long>(B) * Hq * ((S + 127) / 128) > INT_MAX) arc = ATTN_ERR_SHAPE;  // CTAs
    if (arc == ATTN_OK && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
                           (reinterpret_cast<uintptr_t>(lse) & 3u) != 0))
        arc = ATTN_ERR_ALIGN;
    if (arc != ATTN_OK) return arc;
    const int nrows = (S + 127) / 128;
    if ((arc = check_mask(row_ptr, col_idx, nrows, causal != 0)) != ATTN_OK) return arc;
    const bool rope = rope_base > 0.0 && std::isfinite(rope_base);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;
    attn::BsParams bp;
    float2* rope_tab = nullptr;
    int* dmask = nullptr;
    int ctas = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int rc = probe_device(dev);
        if (rc != ATTN_OK) return rc;
        if (rope && (rc = get_rope(dev, S, D, rope_base, &rope_tab)) != ATTN_OK) return rc;
        MaskEntry* me = nullptr;
        if ((rc = get_mask(dev, row_ptr, col_idx, nrows, &dmask, &me)) != ATTN_OK) return rc;
        const MaskSched* ms = nullptr;
        if ((rc = get_mask_sched(dev, *me, nrows, static_cast<long long>(B) * Hq, &ms)) != ATTN_OK) return rc;
        const long long ntasks = static_cast<long long>(B) * Hq * nrows;
        bp.tasks = ms->d;
        bp.task_off = ms->d + ntasks;
        ctas = ms->ctas;
        bp.f.status = g_dev[dev].status;
    }
    if (!encode_bshd(&bp.f.tm_q, q, B, S, Hq, D) || !encode_bshd(&bp.f.tm_k, k, B, S, Hkv, D) ||
        !encode_bshd(&bp.f.tm_v, v, B, S, Hkv, D))
        return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
    bp.f.o = static_cast<__nv_bfloat16*>(o);
    bp.f.lse = lse;
    bp.f.rope = rope_tab;
    bp.f.B = B;
    bp.f.Hq = Hq;
    bp.f.Hkv = Hkv;
    bp.f.S = S;
    bp.f.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    bp.f.wait_limit_ns = kWaitLimitNs;
    bp.row_ptr = dmask;
    bp.col_idx = dmask + nrows + 1;
    bp.window = window;
    bp.alibi = alibi;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (ext) {
        if (alibi) {
            if (D == 128) {
                if (causal) return rope ? launch_bs<128, true, true, 2>(bp, dev, ctas, st) : launch_bs<128, true, false, 2>(bp, dev, ctas, st);
                return rope ? launch_bs<128, false, true, 2>(bp, dev, ctas, st) : launch_bs<128, false, false, 2>(bp, dev, ctas, st);
            }
            if (causal) return rope ? launch_bs<64, true, true, 2>(bp, dev, ctas, st) : launch_bs<64, true, false, 2>(bp, dev, ctas, st);
            return rope ? launch_bs<64, false, true, 2>(bp, dev, ctas, st) : launch_bs<64, false, false, 2>(bp, dev, ctas, st);
        }
        if (D == 128) {
            if (causal) return rope ? launch_bs<128, true, true, 1>(bp, dev, ctas, st) : launch_bs<128, true, false, 1>(bp, dev, ctas, st);
            return rope ? launch_bs<128, false, true, 1>(bp, dev, ctas, st) : launch_bs<128, false, false, 1>(bp, dev, ctas, st);
        }
        if (causal) return rope ? launch_bs<64, true, true, 1>(bp, dev, ctas, st) : launch_bs<64, true, false, 1>(bp, dev, ctas, st);
        return rope ? launch_bs<64, false, true, 1>(bp, dev, ctas, st) : launch_bs<64, false, false, 1>(bp, dev, ctas, st);
    }
    if (D == 128) {
        if (causal) return rope ? launch_bs<128, true, true>(bp, dev, ctas, st) : launch_bs<128, true, false>(bp, dev, ctas, st);
        return rope ? launch_bs<128, false, true>(bp, dev, ctas, st) : launch_bs<128, false, false>(bp, dev, ctas, st);
    }
    if (causal) return rope ? launch_bs<64, true, true>(bp, dev, ctas, st) : launch_bs<64, true, false>(bp, dev, ctas, st);
    return rope ? launch_bs<64, false, true>(bp, dev, ctas, st) : launch_bs<64, false, false>(bp, dev, ctas, st);
}

extern "C" int attn_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                    int Hkv, int S, int D, int causal, double rope_base, const int* row_ptr,
                                    const int* col_idx, void* stream) {
    return bs_impl(q, k, v, o, lse, B, Hq, Hkv, S, D, causal, rope_base, row_ptr, col_idx, false, 0, 0, stream);
}

namespace {
// The key tiles that any row of query tile i can see under the window (keys in
// [128 i - window + 1, 128 i + 127 (+ window - 1 without the causal mask)]), as a CSR block mask.
void local_tiles(int S, int causal, int window, std::vector<int>& row_ptr, std::vector<int>& col_idx) {
    const int nrows = (S + 127) / 128;
    row_ptr.assign(1, 0);
    col_idx.clear();
    for (int i = 0; i < nrows; ++i) {
        long long lo = 0, hi = causal ? 128LL * i + 127 : S - 1LL;
        if (window > 0) {
            lo = std::max(0LL, 128LL * i - window + 1);
            if (!causal) hi = 128LL * i + 127 + window - 1;
        }
        hi = std::min(hi, S - 1LL);
        for (long long t = lo / 128; t <= hi / 128; ++t) col_idx.push_back(static_cast<int>(t));
        row_ptr.push_back(static_cast<int>(col_idx.size()));
    }
}
}  // namespace

extern "C" int attn_fwd_local(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                              int Hkv, int S, int D, int causal, double rope_base, int window, int alibi,
                              void* stream) {
    if (window < 0 || (alibi != 0 && alibi != 1)) return ATTN_ERR_UNSUPPORTED;
    if (S < 1 || S > kMaxS) return ATTN_ERR_SHAPE;
    if (window >= S) window = 0;  // every distance is below S: the same as no window (and no overflow)
    std::vector<int> row_ptr, col_idx;
    local_tiles(S, causal, window, row_ptr, col_idx);
    return bs_impl(q, k, v, o, lse, B, Hq, Hkv, S, D, causal, rope_base, row_ptr.data(),
                   col_idx.empty() ? nullptr : col_idx.data(), true, window, alibi, stream);
}

extern "C" int attn_bwd_local(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int D,
                              int causal, double rope_base, int window, int alibi, void* stream) {
    if (window < 0 || (alibi != 0 && alibi != 1)) return ATTN_ERR_UNSUPPORTED;
    if (S < 1 || S > kMaxS) return ATTN_ERR_SHAPE;
    if (window >= S) window = 0;
    std::vector<int> row_ptr, col_idx;
    local_tiles(S, causal, window, row_ptr, col_idx);
    return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, S, D, causal, rope_base, row_ptr.data(),
                    col_idx.empty() ? nullptr : col_idx.data(), stream, true, window, alibi);
}

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                        void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int D, int causal,
                        double rope_base, void* stream) {
    return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, S, D, causal, rope_base, nullptr, nullptr, stream);
}

extern "C" int attn_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S,
                                    int D, int causal, double rope_base, const int* row_ptr, const int* col_idx,
                                    void* stream) {
    if (row_ptr == nullptr) return ATTN_ERR_NULL;
    return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, S, D, causal, rope_base, row_ptr, col_idx, stream);
}

extern "C" int attn_mask_schedule(const int* row_ptr, int nrows, long long bh, int num_ctas, int* tasks_out,
                                  int* offsets_out, int* ctas_out) {
    if (row_ptr == nullptr) return ATTN_ERR_NULL;
    if (nrows < 1 || bh < 1 || num_ctas < 1 || static_cast<long long>(nrows) * bh > INT_MAX) return ATTN_ERR_SHAPE;
    if (row_ptr[0] != 0) return ATTN_ERR_SHAPE;
    for (int r = 0; r < nrows; ++r)
        if (row_ptr[r + 1] < row_ptr[r]) return ATTN_ERR_SHAPE;
    const attn_host::MaskSchedule sc = attn_host::build_mask_schedule(row_ptr, nrows, bh, num_ctas);
    if (tasks_out != nullptr) std::copy(sc.tasks.begin(), sc.tasks.end(), tasks_out);
    if (offsets_out != nullptr) std::copy(sc.offsets.begin(), sc.offsets.end(), offsets_out);
    if (ctas_out != nullptr) *ctas_out = sc.ctas;
    return ATTN_OK;
}

extern "C" int attn_fwd_schedule(int B, int Hq, int Hkv, int S, int D, int causal, int num_ctas,
                                 double kv_window_bytes, unsigned* words_out, int* offsets_out, int* ctas_out) {
    if (B < 1 || B > 65535 || S < 1 || S > kMaxS || Hq < 1 || Hq > 255 || Hkv < 1 || Hkv > Hq || Hq % Hkv != 0 ||
        (D != 64 && D != 128) || num_ctas < 1)
        return ATTN_ERR_SHAPE;
    if (causal != 0 && causal != 1) return ATTN_ERR_UNSUPPORTED;
    if (attn_host::schedule_units(B, Hq, Hkv, S) > INT_MAX / 2) return ATTN_ERR_SHAPE;
    if (std::isnan(kv_window_bytes)) return ATTN_ERR_UNSUPPORTED;
    const attn_host::Schedule sc = attn_host::build_schedule(B, Hq, Hkv, S, D, causal != 0, num_ctas, kv_window_bytes);
    if (words_out != nullptr) std::copy(sc.words.begin(), sc.words.end(), words_out);
    if (offsets_out != nullptr) std::copy(sc.offsets.begin(), sc.offsets.end(), offsets_out);
    if (ctas_out != nullptr) *ctas_out = sc.ctas;
    return ATTN_OK;
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
        return (v & attn::kStatusTimeoutMask) != 0 ? ATTN_ERR_TIMEOUT : ATTN_ERR_NONFINITE;
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
        case ATTN_ERR_NONFINITE:
            return "ATTN_ERR_NONFINITE: a result row came out non-finite (an input, or a rotated fp16 operand, out of range)";
        case ATTN_ERR_SCRATCH:
            return "ATTN_ERR_SCRATCH: the request needs more than the 16 MiB static scratch of attn_fwd_noalloc";
        default: return "unknown attn status";
    }
}

extern "C" void attn_release_cache(void) {
    int cur = 0;
    const bool have = cudaGetDevice(&cur) == cudaSuccess;
    // lock order: the host pipeline's lock before the table caches' (attn_fwd_host calls attn_fwd)
    std::lock_guard<std::mutex> plock(g_pipe_mu);
    {
        for (int d = 0; d < kMaxDevices; ++d) {
            HostPipe& hp = g_pipe[d];
            if (!hp.ready) continue;
            cudaSetDevice(d);
            cudaFree(hp.buf);
            for (int i = 0; i < 2; ++i) {
                cudaEventDestroy(hp.ev_in[i]);
                cudaEventDestroy(hp.ev_comp[i]);
                cudaEventDestroy(hp.ev_out[i]);
            }
            cudaStreamDestroy(hp.s_in);
            cudaStreamDestroy(hp.s_comp);
            cudaStreamDestroy(hp.s_out);
            hp = HostPipe();
        }
    }
    std::lock_guard<std::mutex> lock(g_mu);
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
    for (auto& e : g_split) {
        cudaSetDevice(e.dev);
        cudaFree(e.table);
    }
    for (int d = 0; d < kMaxDevices; ++d) {
        if (g_dec[d].buf == nullptr) continue;
        cudaSetDevice(d);
        cudaFree(g_dec[d].buf);
        g_dec[d] = DecodeScratch();
    }
    for (auto& e : g_masks) {
        cudaSetDevice(e.dev);
        cudaFree(e.d);
        for (auto& ms : e.sched) cudaFree(ms.d);
    }
    g_masks.clear();
    for (int d = 0; d < kMaxDevices; ++d) {
        if (g_bwd_rot[d].buf != nullptr) {
            cudaSetDevice(d);
            cudaFree(g_bwd_rot[d].buf);
            g_bwd_rot[d] = RotScratch();
        }
        if (g_bwd[d].buf == nullptr) continue;
        cudaSetDevice(d);
        cudaFree(g_bwd[d].buf);
        g_bwd[d] = DecodeScratch();
    }
    g_split.clear();
    g_rope.clear();
    g_sched.clear();
    g_win.clear();
    if (have) cudaSetDevice(cur);
}
