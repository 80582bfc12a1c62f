// W8A8 GEMM entry: routes a problem to the decode kernel (M <= 32, int8
// mma.sync weight streaming, decode_gemm.cu) or, for larger M, to the
// tcgen05 tensor-core kernel (w8a8_fused.cu) after one small pass that turns
// the token codes into fp16 codes.  The fused linear layer (w8a8_linear)
// lets the activation quantization pass write those fp16 codes itself.
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

// int8 codes -> fp16 codes (exact), grid-stride over 16-byte vectors.  CTA
// 0 also sets the `nzero` words at `zero` to 0 (the stream-K flags of the
// GEMM launched next; nullable).
__global__ void __launch_bounds__(256) i8_to_f16_kernel(const int8_t* __restrict__ src, int64_t vecs,
                                                        uint16_t* __restrict__ dst, unsigned* __restrict__ zero,
                                                        int nzero) {
    pdl_wait();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0u;
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

size_t pad256(size_t n) { return (n + 255) / 256 * 256; }

}  // namespace

size_t w8a8_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    (void)N;
    if (M <= kW8A8DecodeMaxM) return 0;
    return (size_t)M * (size_t)K * 2;
}

cudaError_t launch_w8a8_ws(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw,
                           const uint16_t* bias, uint16_t* y, int32_t* acc, int64_t M, int64_t N, int64_t K,
                           uint16_t* ws, void* sk_ws, size_t sk_bytes, const LaunchEnv& env) {
    if (M <= kW8A8DecodeMaxM) return launch_w8a8_decode(qx, sx, qw, sw, bias, y, acc, M, N, K, env);
    size_t need = 0;
    int flags = 0;
    cudaError_t e = sk_ws ? w8a8_sk_workspace(M, N, K, env.sm_count, &need, &flags) : cudaSuccess;
    if (e != cudaSuccess) return e;
    if (need == 0 || sk_bytes < need) {
        sk_ws = nullptr;
        flags = 0;
    }
    const int64_t vecs = M * K / 16;  // K is a multiple of 16
    const int64_t blocks = std::min<int64_t>((vecs + 255) / 256, (int64_t)env.sm_count * 8);
    e = launch_kernel(i8_to_f16_kernel, dim3((unsigned)blocks), dim3(256), 0, env.stream, kNoCluster, qx, vecs, ws,
                      static_cast<unsigned*>(sk_ws), flags);
    if (e != cudaSuccess) return e;
    return launch_w8a8_fused(ws, sx, qw, sw, bias, y, acc, M, N, K, sk_ws, sk_ws ? sk_bytes : 0, env);
}

cudaError_t launch_w8a8(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw, const uint16_t* bias,
                        uint16_t* y, int32_t* acc, int64_t M, int64_t N, int64_t K, const LaunchEnv& env) {
    if (M <= kW8A8DecodeMaxM) return launch_w8a8_decode(qx, sx, qw, sw, bias, y, acc, M, N, K, env);
    // One stream-ordered allocation (from the device's default memory pool,
    // returned when the stream reaches the free): the fp16 token codes, then
    // the stream-K workspace.
    size_t sk = 0;
    int flags = 0;
    cudaError_t e = w8a8_sk_workspace(M, N, K, env.sm_count, &sk, &flags);
    if (e != cudaSuccess) return e;
    const size_t tok = pad256(w8a8_workspace_bytes(M, N, K));
    void* ws = nullptr;
    if ((e = cudaMallocAsync(&ws, tok + sk, env.stream)) != cudaSuccess) return e;
    uint8_t* w = static_cast<uint8_t*>(ws);
    e = launch_w8a8_ws(qx, sx, qw, sw, bias, y, acc, M, N, K, reinterpret_cast<uint16_t*>(w), sk ? w + tok : nullptr,
                       sk, env);
    const cudaError_t f = cudaFreeAsync(ws, env.stream);
    return e != cudaSuccess ? e : f;
}

namespace {

// Workspace of the fused linear layer: the token codes (int8 for the decode
// kernel unless the caller keeps them, fp16 for the tensor-core kernel), the
// scales unless the caller keeps them, then the stream-K workspace.
struct LinearLayout {
    size_t codes, scales, sk;
    int flags;
    size_t total() const { return codes + scales + sk; }
};

cudaError_t linear_layout(int64_t M, int64_t N, int64_t K, bool have_qx, bool have_sx, int sms, LinearLayout* l) {
    const size_t codes = M > kW8A8DecodeMaxM ? (size_t)M * (size_t)K * 2 : (have_qx ? 0 : (size_t)M * (size_t)K);
    l->codes = pad256(codes);
    l->scales = have_sx ? 0 : pad256((size_t)M * 4);
    l->sk = 0;
    l->flags = 0;
    if (M <= kW8A8DecodeMaxM) return cudaSuccess;
    return w8a8_sk_workspace(M, N, K, sms, &l->sk, &l->flags);
}

}  // namespace

cudaError_t launch_w8a8_linear(const uint16_t* x, const int8_t* qw, const float* sw, const uint16_t* bias, uint16_t* y,
                               int8_t* qx, float* sx, int32_t* acc, int64_t M, int64_t N, int64_t K,
                               const LaunchEnv& env) {
    // Few tokens and a weight whose decode GEMM is one unsplit wave: the
    // one-launch form, which quantizes the tokens inside the GEMM, measured
    // faster there (Qwen3-4B gate_up: 14.7 against 16.0 us) and slower on
    // split-K shapes (qkv 9.1 against 8.3 us) and beyond one wave (Qwen3-8B
    // gate_up); its results are the same bit for bit, and it needs no
    // workspace.
    if (w8a8_linear_one_launch(M, N, K, env.sm_count))
        return launch_w8a8_decode_fused(x, qw, sw, bias, y, qx, sx, acc, M, N, K, env);
    LinearLayout l;
    cudaError_t e = linear_layout(M, N, K, qx != nullptr, sx != nullptr, env.sm_count, &l);
    if (e != cudaSuccess) return e;
    void* ws = nullptr;
    if (l.total() > 0 && (e = cudaMallocAsync(&ws, l.total(), env.stream)) != cudaSuccess) return e;
    uint8_t* w = static_cast<uint8_t*>(ws);
    float* s = sx ? sx : reinterpret_cast<float*>(w + l.codes);
    if (M <= kW8A8DecodeMaxM) {
        // int8 codes for the decode kernel
        int8_t* q8 = qx ? qx : reinterpret_cast<int8_t*>(w);
        e = launch_quant_rows(x, M, K, q8, nullptr, s, env);
        if (e == cudaSuccess) e = launch_w8a8_decode(q8, s, qw, sw, bias, y, acc, M, N, K, env);
    } else {
        // fp16 codes for the tensor-core kernel, written by the quantization
        // pass itself (and the int8 codes only if the caller asked for
        // them); the same pass zeroes the stream-K flags
        uint16_t* x16 = reinterpret_cast<uint16_t*>(w);
        void* sk = l.sk ? w + l.codes + l.scales : nullptr;
        e = launch_quant_rows(x, M, K, qx, x16, s, env, static_cast<unsigned*>(sk), l.flags);
        if (e == cudaSuccess) e = launch_w8a8_fused(x16, s, qw, sw, bias, y, acc, M, N, K, sk, l.sk, env);
    }
    if (ws != nullptr) {
        const cudaError_t f = cudaFreeAsync(ws, env.stream);
        if (e == cudaSuccess) e = f;
    }
    return e;
}

}  // namespace i8ql
