// noalloc.cu - the streamed-weight GEMM for callers that cannot allocate device memory.
//
// eagle_linear_bf16 needs a caller-provided, zero-initialised scratch buffer for its split-K
// partial sums and tile tickets.  Some callers cannot provide one: code that runs where
// cudaMalloc is not allowed or not wanted (it synchronises the device and can fail under memory
// pressure), plug-ins living inside a framework whose own allocator owns all device memory, and
// latency-critical loops that must not allocate per call.  This file gives them a variant whose
// scratch is a fixed array in this library's device memory, so the caller passes only its
// inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds it
// (kNoAllocScratchBytes, about 5 MiB) until the process exits.  Host code cannot use the
// variable's name as a device address, so the first call on each device looks the address up
// with cudaGetSymbolAddress while that device is current, and later calls reuse it.
#include <mutex>

#include "../../include/eagle_tree.h"
#include "kernels.cuh"

namespace {

constexpr int32_t kNoAllocMaxRows = 32;            // MMA N of at most 32
constexpr int32_t kNoAllocMaxGrid = 160;           // CTAs (one per SM, capped)
constexpr int32_t kNoAllocMaxOut = 131072;         // output features (1024 weight tiles)
constexpr size_t kCountersBytes = 4096;            // 1024 tile tickets
constexpr size_t kPartialsBytes =
    static_cast<size_t>(kNoAllocMaxGrid) * 2 * kNoAllocMaxRows * eagle::kLinearTileM * sizeof(float);
constexpr size_t kNoAllocScratchBytes = kCountersBytes + kPartialsBytes;  // 5 MiB + 4 KiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's scratch array (looked up once per device).
eagle_status scratch_for_current_device(void **out, int *num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return EAGLE_ERR_CUDA;
    if (cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return EAGLE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return EAGLE_ERR_CUDA;
        if (eagle::prepare_kernels() != cudaSuccess) return EAGLE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return EAGLE_OK;
}

}  // namespace

extern "C" {

size_t eagle_linear_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

eagle_status eagle_linear_bf16_noalloc(const void *d_w, int64_t ldw, const void *d_x, int64_t ldx,
                                       const void *d_bias, int32_t out_features, int32_t in_features,
                                       int32_t rows, void *d_y, int64_t ldy, int32_t out_bf16,
                                       eagle_stream_t stream) {
    if (out_features < 1 || in_features < 1 || rows < 1) return EAGLE_ERR_INVALID_ARG;
    if (rows > kNoAllocMaxRows || out_features > kNoAllocMaxOut) return EAGLE_ERR_INVALID_ARG;
    if (!d_w || !d_x || !d_y) return EAGLE_ERR_INVALID_ARG;
    if (ldw < in_features || ldx < in_features || ldy < out_features) return EAGLE_ERR_INVALID_ARG;
    if (ldw % 8 != 0 || ldx % 8 != 0) return EAGLE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_w) & 15u) || (reinterpret_cast<uintptr_t>(d_x) & 15u))
        return EAGLE_ERR_INVALID_ARG;
    void *scratch = nullptr;
    int num_sms = 0;
    const eagle_status s = scratch_for_current_device(&scratch, &num_sms);
    if (s != EAGLE_OK) return s;
    const int32_t grid = num_sms < kNoAllocMaxGrid ? num_sms : kNoAllocMaxGrid;
    int32_t *counters = reinterpret_cast<int32_t *>(scratch);
    float *partials = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(scratch) + kCountersBytes);
    eagle::LinearPlan p;
    if (!eagle::plan_linear_bf16(&p, d_w, ldw, out_features, in_features, d_x, ldx, rows, d_bias, d_y, ldy,
                                 out_bf16, partials, counters, nullptr, grid))
        return EAGLE_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // The tickets must start at zero; a completed launch leaves them zero, an aborted one may not.
    if (cudaMemsetAsync(counters, 0, eagle::linear_counters_bytes(out_features), st) != cudaSuccess)
        return EAGLE_ERR_CUDA;
    if (eagle::launch_linear_bf16(p, st) != cudaSuccess) return EAGLE_ERR_CUDA;
    return EAGLE_OK;
}

}  // extern "C"
