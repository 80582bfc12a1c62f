// Internal helpers shared by the i8ql CUDA sources (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/i8ql.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "i8ql kernels are written for sm_103a (GB300) only"
#endif

namespace i8ql {

// Sticky per-device kernel fault word.  Kernels OR a status bit into it:
constexpr unsigned kErrBitTimeout = 1u;
constexpr unsigned kErrBitBadOffsets = 2u;

// Largest supported sizes (indices stay well inside 64-bit arithmetic and
// grid limits).
constexpr int64_t kMaxRows = (int64_t)1 << 31;

// Wall-clock limit of every bounded wait inside a kernel (nanoseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_fault(unsigned* err, unsigned bit) {
    if (err) atomicOr(err, bit);
}

// Programmatic dependent launch: every kernel is launched with programmatic
// stream serialization and waits here, before touching global memory, for the
// grids it depends on to complete (a no-op when launched without it).  Its
// launch and prologue can then overlap the tail of the previous kernel.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream begin launching (its CTAs still wait in
// pdl_wait() for this grid to finish).  Called only by grids that fit in one
// wave, so early dependents never take SM slots this grid still needs.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Warms L2 with `bytes` bytes at p (multiple of 16, 16-byte aligned).  Safe
// before pdl_wait() even if the previous grid writes those bytes: L2 is the
// point of coherence, so a line written later is updated there, and the
// loads after pdl_wait() read through it.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// cudaLaunchKernelEx with programmatic stream serialization and, when
// cluster.x > 0, thread-block clusters of the given shape.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          dim3 cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    unsigned n = 0;
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster.x > 0) {
        attrs[n].id = cudaLaunchAttributeClusterDimension;
        attrs[n].val.clusterDim.x = cluster.x;
        attrs[n].val.clusterDim.y = cluster.y;
        attrs[n].val.clusterDim.z = cluster.z;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// No thread-block clusters.
constexpr dim3 kNoCluster(0, 0, 0);

// Launch parameters every entry point passes down.
struct LaunchEnv {
    cudaStream_t stream;
    unsigned* err;   // device address of the sticky word of the current device
    int sm_count;
};

// Returns the environment of the current device, creating per-device state
// on first use.  Returns false (and sets *status) on failure.
bool launch_env(void* stream, LaunchEnv* env, i8ql_status* status);

// Test hook (i8ql_debug_stream_k_timeout): stream-K finishers wait for a
// flag value that is never written, with a 1 ms limit.
bool debug_sk_timeout();
// i8ql_set_early_weight_loads: decode GEMMs may load weights before waiting
// for the previous kernel on the stream.
bool early_weight_loads();

// Kernel launchers.  They assume validated arguments.
// W8A8 up to this many tokens runs on the decode kernel (int8 mma.sync,
// weight streaming); larger M runs on the tcgen05 kernel.
constexpr int64_t kW8A8DecodeMaxM = I8QL_W8A8_DECODE_MAX_M;
// Per-row quantization; the codes go to q (int8) and/or qh (fp16), either
// nullable.  The kernel also sets the `nzero` words at `zero` to 0 (the
// stream-K flags of the GEMM launched after it; nullable).
cudaError_t launch_quant_rows(const uint16_t* src, int64_t rows, int64_t K, int8_t* q, uint16_t* qh, float* s,
                              const LaunchEnv& env, unsigned* zero = nullptr, int nzero = 0);
// W8A16 (offsets null) or grouped W8A16; grouped calls may gather their token
// rows (gather[r] = row of x feeding grouped row r) and may fuse the
// SiLU-gated product of a gate/up projection with N = 2 * glu rows.
cudaError_t launch_w8a16(const uint16_t* x, const int32_t* offsets, int64_t E, const int8_t* qw,
                         const float* sw, uint16_t* y, int64_t M, int64_t N, int64_t K,
                         const LaunchEnv& env, const int32_t* gather = nullptr, int64_t glu = 0);
// MoE routing over device logits, and the weighted combine of expert rows.
cudaError_t launch_moe_route(const float* logits, int64_t T, int64_t E, int64_t topk, int64_t shared,
                             int32_t* offsets, int32_t* row_token, int32_t* token_row, float* slot_weight,
                             const LaunchEnv& env);
cudaError_t launch_moe_combine(const uint16_t* yd, const int32_t* token_row, const float* slot_weight, uint16_t* out,
                               int64_t T, int64_t S, int64_t H, const LaunchEnv& env);
// Shared memory of the routing kernel for T tokens over E routed experts
// (kRouteTooLarge when one CTA cannot hold it).
constexpr size_t kRouteTooLarge = ~(size_t)0;
size_t moe_route_smem(int64_t T, int64_t E);
// The MoE expert MLP: routing, grouped gate/up with the SiLU-gated product,
// grouped down, combine; intermediates in a stream-ordered workspace.
cudaError_t launch_moe_mlp(const uint16_t* x, const float* logits, int64_t E_routed, int64_t topk, int64_t shared,
                           const int8_t* qw_gu, const float* sw_gu, const int8_t* qw_d, const float* sw_d,
                           uint16_t* out, int64_t T, int64_t H, int64_t I, const LaunchEnv& env);
cudaError_t launch_w8a8_decode(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw,
                               const uint16_t* bias, uint16_t* y, int32_t* acc, int64_t M, int64_t N,
                               int64_t K, const LaunchEnv& env);
// W8A8 from bf16 tokens in one launch (M <= kW8A8FusedMaxM): the decode
// kernel quantizes its token rows itself; qx / sx receive the codes and
// scales when not null.
constexpr int64_t kW8A8FusedMaxM = 8;
// Whether the one-launch kernel runs an N x K weight as one unsplit wave
// (where it measured faster than a quantization launch plus the GEMM).
bool w8a8_decode_fused_preferred(int64_t N, int64_t K, int sms);
// Whether w8a8_linear takes the one-launch form for this problem.
inline bool w8a8_linear_one_launch(int64_t M, int64_t N, int64_t K, int sms) {
    return M > 0 && M <= kW8A8FusedMaxM && w8a8_decode_fused_preferred(N, K, sms);
}
cudaError_t launch_w8a8_decode_fused(const uint16_t* x, const int8_t* qw, const float* sw, const uint16_t* bias,
                                     uint16_t* y, int8_t* qx, float* sx, int32_t* acc, int64_t M, int64_t N, int64_t K,
                                     const LaunchEnv& env);
// Tile width (N side of the output tile), split-K factor and CTA-pair mode
// (0 single CTAs, 1 pairs, 2 pairs with stream-K) the tcgen05 kernel uses
// for a W8A8 problem, with or without a stream-K workspace; all 0 when M is
// in the decode range.
cudaError_t w8a8_plan(int64_t M, int64_t N, int64_t K, int sms, bool allow_sk, int* tile_n, int* split_k, int* pair);
// Bytes of the token workspace launch_w8a8_ws needs (the fp16 token codes,
// M * K * 2, when M exceeds the decode range; 0 otherwise).
size_t w8a8_workspace_bytes(int64_t M, int64_t N, int64_t K);
// Stream-K workspace of the tensor-core kernel: its bytes (0 when the plan
// does not use stream-K) and the number of 32-bit flags at its start that
// must read zero when the kernel starts.
cudaError_t w8a8_sk_workspace(int64_t M, int64_t N, int64_t K, int sms, size_t* bytes, int* flags);
// W8A8 with a given token workspace `ws` and an optional stream-K workspace
// (sk_ws, sk_bytes; null or too small: no stream-K).
cudaError_t launch_w8a8_ws(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw,
                           const uint16_t* bias, uint16_t* y, int32_t* acc, int64_t M, int64_t N, int64_t K,
                           uint16_t* ws, void* sk_ws, size_t sk_bytes, const LaunchEnv& env);
// tcgen05 W8A8 for M > kW8A8DecodeMaxM: the token codes as fp16 (x16, [M, K]), the weight
// codes as int8 (converted inside the kernel).  Stream-K runs when the plan
// wants it and sk_ws holds sk_bytes >= what w8a8_sk_workspace reports, its
// flags zeroed by an earlier kernel of the stream.
cudaError_t launch_w8a8_fused(const uint16_t* x16, const float* sx, const int8_t* qw, const float* sw,
                              const uint16_t* bias, uint16_t* y, int32_t* acc, int64_t M, int64_t N, int64_t K,
                              void* sk_ws, size_t sk_bytes, const LaunchEnv& env);
cudaError_t launch_w8a8_linear(const uint16_t* x, const int8_t* qw, const float* sw, const uint16_t* bias, uint16_t* y,
                               int8_t* qx, float* sx, int32_t* acc, int64_t M, int64_t N, int64_t K,
                               const LaunchEnv& env);
cudaError_t launch_w8a8(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw,
                        const uint16_t* bias, uint16_t* y, int32_t* acc, int64_t M, int64_t N,
                        int64_t K, const LaunchEnv& env);
// FP8 E4M3: per-row codes (s = absmax / 448), the tcgen05 kind::f8f6f4 GEMM,
// and the linear layer from bf16 activations (quantization, then the GEMM).
cudaError_t launch_quant_rows_fp8(const uint16_t* src, int64_t rows, int64_t K, uint8_t* q, float* s,
                                  const LaunchEnv& env);
// The plan launch_fp8_gemm would run (tile width, split-K, CTA pairs).
cudaError_t fp8_plan(int64_t M, int64_t N, int64_t K, int sms, int* tile_n, int* split_k, int* pair);
cudaError_t launch_fp8_gemm(const uint8_t* qx, const float* sx, const uint8_t* qw, const float* sw,
                            const uint16_t* bias, uint16_t* y, int64_t M, int64_t N, int64_t K, const LaunchEnv& env);
// W4A16 with bf16 group-128 scales: the quantization of bf16 weights to
// packed int4 codes and the decode GEMM.
cudaError_t launch_quant_w4(const uint16_t* w, int64_t N, int64_t K, uint8_t* packed, uint16_t* scale,
                            const LaunchEnv& env);
cudaError_t launch_w4a16(const uint16_t* x, const uint8_t* q, const uint16_t* s, uint16_t* y, int64_t M, int64_t N,
                         int64_t K, const LaunchEnv& env);
cudaError_t launch_fp8_linear(const uint16_t* x, const uint8_t* qw, const float* sw, const uint16_t* bias,
                              uint16_t* y, uint8_t* qx, float* sx, int64_t M, int64_t N, int64_t K,
                              const LaunchEnv& env);

}  // namespace i8ql
