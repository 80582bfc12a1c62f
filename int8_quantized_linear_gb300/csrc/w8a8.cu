// W8A8 GEMM entry: routes a problem to the decode kernel (M <= 64, int8
// mma.sync weight streaming, decode_gemm.cu) or, for larger M, to the
// tcgen05 tensor-core kernel (w8a8_fused.cu) after one small pass that turns
// the token codes into fp16 codes.
//
// Sources: "feat(quantization): support compressed-tensors W8A8 and mixed
// modules", Design and Supported Execution Scheme, and "Day 6 -- Quantize It
// Yourself", The mechanism, block 5.
//
// The token pass exists because the tensor-core kernel reads the token tile
// of every k-block once per output tile it meets (N / BN times): reading
// ready fp16 codes through TMA costs nothing there, while converting them in
// the kernel would compete with the weight conversion for issue slots.  The
// pass touches 3*M*K bytes, small next to the weights and the GEMM.

#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "tc_common.cuh"

namespace i8ql {
namespace {

// int8 codes -> fp16 codes (exact), grid-stride over 16-byte vectors.
__global__ void __launch_bounds__(256) i8_to_f16_kernel(const int8_t* __restrict__ src, int64_t vecs,
                                                        uint16_t* __restrict__ dst) {
    pdl_wait();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vecs; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
        uint32_t h[8];
        tc::i8x4_to_f16(v.x, h[0], h[1]);
        tc::i8x4_to_f16(v.y, h[2], h[3]);
        tc::i8x4_to_f16(v.z, h[4], h[5]);
        tc::i8x4_to_f16(v.w, h[6], h[7]);
        uint4* o = reinterpret_cast<uint4*>(dst) + 2 * i;
        o[0] = make_uint4(h[0], h[1], h[2], h[3]);
        o[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
}

}  // namespace

size_t w8a8_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    (void)N;
    if (M <= kW8A8DecodeMaxM) return 0;
    return (size_t)M * (size_t)K * 2;
}

cudaError_t launch_w8a8_ws(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw,
                           const uint16_t* bias, uint16_t* y, int32_t* acc, int64_t M, int64_t N, int64_t K,
                           uint16_t* ws, const LaunchEnv& env) {
    if (M <= kW8A8DecodeMaxM) return launch_w8a8_decode(qx, sx, qw, sw, bias, y, acc, M, N, K, env);
    const int64_t vecs = M * K / 16;  // K is a multiple of 16
    const int64_t blocks = std::min<int64_t>((vecs + 255) / 256, (int64_t)env.sm_count * 8);
    cudaError_t e = launch_kernel(i8_to_f16_kernel, dim3((unsigned)blocks), dim3(256), 0, env.stream, kNoCluster, qx,
                                  vecs, ws);
    if (e != cudaSuccess) return e;
    return launch_w8a8_fused(ws, sx, qw, sw, bias, y, acc, M, N, K, env);
}

cudaError_t launch_w8a8(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw, const uint16_t* bias,
                        uint16_t* y, int32_t* acc, int64_t M, int64_t N, int64_t K, const LaunchEnv& env) {
    if (M <= kW8A8DecodeMaxM) return launch_w8a8_decode(qx, sx, qw, sw, bias, y, acc, M, N, K, env);
    // Stream-ordered workspace for the fp16 token codes (from the device's
    // default memory pool, returned when the stream reaches the free).
    void* ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, w8a8_workspace_bytes(M, N, K), env.stream);
    if (e != cudaSuccess) return e;
    e = launch_w8a8_ws(qx, sx, qw, sw, bias, y, acc, M, N, K, static_cast<uint16_t*>(ws), env);
    const cudaError_t f = cudaFreeAsync(ws, env.stream);
    return e != cudaSuccess ? e : f;
}

}  // namespace i8ql
