// W8A8 GEMM for callers that cannot allocate device memory.
//
// Some callers must not allocate GPU memory while they run: code replayed
// from a CUDA graph whose memory was fixed at capture, real-time serving
// loops that forbid allocator calls (and their possible synchronisation or
// failure) on the hot path, and hosts that hand the library only the tensors
// they already own.  w8a8_gemm needs a workspace for large M (the fp16 codes
// of the tokens) and takes it from the stream-ordered allocator; this
// entry point instead uses one fixed array compiled into the library.
//
// The array lives in device global memory: every GPU that loads the library
// holds its kNoAllocBytes until the process exits.  Every call shares it and
// it keeps the last call's contents; the kernels overwrite every byte they
// read, so nothing needs clearing between calls.  Calls whose kernels may
// overlap on the GPU (different streams, no ordering between them) race on
// the array and must not be issued.

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace i8ql {
namespace {

constexpr int64_t kNoAllocElements = I8QL_NOALLOC_MAX_ELEMENTS;  // fp16 workspace elements

static __device__ __align__(256) uint16_t g_noalloc_scratch[kNoAllocElements];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
std::atomic<uint16_t*> g_scratch_ptr[kMaxDevices];

// The device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress, once per device, with that device current.
i8ql_status scratch_address(int dev, uint16_t** out) {
    uint16_t* ptr = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (ptr == nullptr) {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        ptr = g_scratch_ptr[dev].load(std::memory_order_relaxed);
        if (ptr == nullptr) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
                cudaGetLastError();
                return I8QL_ERR_CUDA;
            }
            ptr = static_cast<uint16_t*>(addr);
            g_scratch_ptr[dev].store(ptr, std::memory_order_release);
        }
    }
    *out = ptr;
    return I8QL_OK;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace i8ql

using namespace i8ql;

extern "C" i8ql_status w8a8_gemm_noalloc(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw,
                                         const i8ql_bf16* bias, i8ql_bf16* y, int32_t* acc_debug, int64_t M,
                                         int64_t N, int64_t K, void* stream) {
    // Host-side argument checks: the same rules as w8a8_gemm.
    if (M < 0 || N <= 0 || K <= 0) return I8QL_ERR_INVALID_ARG;
    if (K % 16 != 0 || K > I8QL_MAX_K || M >= kMaxRows || N >= kMaxRows) return I8QL_ERR_UNSUPPORTED;
    if (qw == nullptr || !aligned_to(qw, 16) || sw == nullptr || !aligned_to(sw, 4)) return I8QL_ERR_INVALID_ARG;
    if (M > 0) {
        if (qx == nullptr || !aligned_to(qx, 16) || sx == nullptr || !aligned_to(sx, 4)) return I8QL_ERR_INVALID_ARG;
        if (y == nullptr || !aligned_to(y, 16)) return I8QL_ERR_INVALID_ARG;
    }
    if (bias != nullptr && !aligned_to(bias, 2)) return I8QL_ERR_INVALID_ARG;
    if (acc_debug != nullptr && !aligned_to(acc_debug, 16)) return I8QL_ERR_INVALID_ARG;
    if (M == 0) return I8QL_OK;
    // The fixed array bounds the problem size on the large-M path.
    if (w8a8_workspace_bytes(M, N, K) > (size_t)kNoAllocElements * sizeof(uint16_t)) return I8QL_ERR_WORKSPACE_LIMIT;

    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return I8QL_ERR_NO_DEVICE;
    }
    uint16_t* scratch = nullptr;
    if ((s = scratch_address(dev, &scratch)) != I8QL_OK) return s;
    // no stream-K: its workspace would not fit a fixed array
    const cudaError_t e = launch_w8a8_ws(qx, sx, qw, sw, bias, y, acc_debug, M, N, K, scratch, nullptr, 0, env);
    return e == cudaSuccess ? I8QL_OK : I8QL_ERR_CUDA;
}
