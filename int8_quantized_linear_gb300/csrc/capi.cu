// C ABI of libi8ql.so: argument validation, per-device state and dispatch.
//
// Every entry point validates its arguments on the host before touching the
// CUDA runtime, so argument errors never launch anything and can be tested
// without a GPU.

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace i8ql {

// The sticky kernel-fault word; one instance per device context.
__device__ unsigned g_kernel_faults;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    std::atomic<bool> ready{false};
    unsigned* err = nullptr;
    int sm_count = 0;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
std::atomic<int> g_debug_sk_timeout{0};
std::atomic<int> g_early_weights{0};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

i8ql_status check_k(int64_t K) {
    if (K <= 0) return I8QL_ERR_INVALID_ARG;
    if (K % 16 != 0 || K > I8QL_MAX_K) return I8QL_ERR_UNSUPPORTED;
    return I8QL_OK;
}

i8ql_status check_rows(int64_t R) {
    if (R < 0) return I8QL_ERR_INVALID_ARG;
    if (R >= kMaxRows) return I8QL_ERR_UNSUPPORTED;
    return I8QL_OK;
}

i8ql_status check_matrix(const void* p, int64_t rows) {
    if (rows == 0) return I8QL_OK;
    if (p == nullptr || !aligned(p, 16)) return I8QL_ERR_INVALID_ARG;
    return I8QL_OK;
}

i8ql_status check_vec(const void* p, int64_t n, uintptr_t align) {
    if (n == 0) return I8QL_OK;
    if (p == nullptr || !aligned(p, align)) return I8QL_ERR_INVALID_ARG;
    return I8QL_OK;
}

#define I8QL_TRY(expr)                       \
    do {                                     \
        i8ql_status _s = (expr);             \
        if (_s != I8QL_OK) return _s;        \
    } while (0)

i8ql_status from_cuda(cudaError_t e) { return e == cudaSuccess ? I8QL_OK : I8QL_ERR_CUDA; }

}  // namespace

bool debug_sk_timeout() { return g_debug_sk_timeout.load(std::memory_order_relaxed) != 0; }
bool early_weight_loads() { return g_early_weights.load(std::memory_order_relaxed) != 0; }

bool launch_env(void* stream, LaunchEnv* env, i8ql_status* status) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        *status = I8QL_ERR_NO_DEVICE;
        return false;
    }
    DeviceState& st = g_devices[dev];
    if (!st.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!st.ready.load(std::memory_order_relaxed)) {
            int major = 0, minor = 0, sms = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
                cudaGetLastError();
                *status = I8QL_ERR_CUDA;
                return false;
            }
            if (major != 10 || minor != 3) {
                *status = I8QL_ERR_NO_DEVICE;
                return false;
            }
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_kernel_faults) != cudaSuccess) {
                cudaGetLastError();
                *status = I8QL_ERR_CUDA;
                return false;
            }
            st.err = static_cast<unsigned*>(addr);
            st.sm_count = sms;
            st.ready.store(true, std::memory_order_release);
        }
    }
    env->stream = static_cast<cudaStream_t>(stream);
    env->err = st.err;
    env->sm_count = st.sm_count;
    return true;
}

}  // namespace i8ql

using namespace i8ql;

extern "C" {

i8ql_status quantize_weight_per_channel_int8(const i8ql_bf16* w, int64_t N, int64_t K, int8_t* q,
                                             float* scale, void* stream) {
    I8QL_TRY(check_rows(N));
    I8QL_TRY(check_k(K));
    I8QL_TRY(check_matrix(w, N));
    I8QL_TRY(check_matrix(q, N));
    I8QL_TRY(check_vec(scale, N, 4));
    if (N == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_quant_rows(w, N, K, q, nullptr, scale, env));
}

i8ql_status quantize_act_per_token_int8(const i8ql_bf16* x, int64_t M, int64_t K, int8_t* q,
                                        float* scale, void* stream) {
    I8QL_TRY(check_rows(M));
    I8QL_TRY(check_k(K));
    I8QL_TRY(check_matrix(x, M));
    I8QL_TRY(check_matrix(q, M));
    I8QL_TRY(check_vec(scale, M, 4));
    if (M == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_quant_rows(x, M, K, q, nullptr, scale, env));
}

i8ql_status w8a8_gemm(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw,
                      const i8ql_bf16* bias, i8ql_bf16* y, int32_t* acc_debug, int64_t M, int64_t N,
                      int64_t K, void* stream) {
    I8QL_TRY(check_rows(M));
    I8QL_TRY(check_k(K));
    if (N <= 0) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_rows(N));
    I8QL_TRY(check_matrix(qx, M));
    I8QL_TRY(check_vec(sx, M, 4));
    I8QL_TRY(check_matrix(qw, N));
    I8QL_TRY(check_vec(sw, N, 4));
    if (bias != nullptr && !aligned(bias, 2)) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_matrix(y, M));
    if (acc_debug != nullptr && !aligned(acc_debug, 16)) return I8QL_ERR_INVALID_ARG;
    if (M == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_w8a8(qx, sx, qw, sw, bias, y, acc_debug, M, N, K, env));
}

i8ql_status w8a8_linear(const i8ql_bf16* x, const int8_t* qw, const float* sw, const i8ql_bf16* bias,
                        i8ql_bf16* y, int8_t* qx, float* sx, int32_t* acc_debug, int64_t M, int64_t N, int64_t K,
                        void* stream) {
    I8QL_TRY(check_rows(M));
    I8QL_TRY(check_k(K));
    if (N <= 0) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_rows(N));
    I8QL_TRY(check_matrix(x, M));
    I8QL_TRY(check_matrix(qw, N));
    I8QL_TRY(check_vec(sw, N, 4));
    if (bias != nullptr && !aligned(bias, 2)) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_matrix(y, M));
    if (qx != nullptr) I8QL_TRY(check_matrix(qx, M));
    if (sx != nullptr && !aligned(sx, 4)) return I8QL_ERR_INVALID_ARG;
    if (acc_debug != nullptr && !aligned(acc_debug, 16)) return I8QL_ERR_INVALID_ARG;
    if (M == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_w8a8_linear(x, qw, sw, bias, y, qx, sx, acc_debug, M, N, K, env));
}

i8ql_status w8a8_linear_fused(const i8ql_bf16* x, const int8_t* qw, const float* sw, const i8ql_bf16* bias,
                              i8ql_bf16* y, int8_t* qx, float* sx, int32_t* acc_debug, int64_t M, int64_t N, int64_t K,
                              void* stream) {
    I8QL_TRY(check_rows(M));
    I8QL_TRY(check_k(K));
    if (N <= 0) return I8QL_ERR_INVALID_ARG;
    if (M > kW8A8FusedMaxM) return I8QL_ERR_UNSUPPORTED;
    I8QL_TRY(check_rows(N));
    I8QL_TRY(check_matrix(x, M));
    I8QL_TRY(check_matrix(qw, N));
    I8QL_TRY(check_vec(sw, N, 4));
    if (bias != nullptr && !aligned(bias, 2)) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_matrix(y, M));
    if (qx != nullptr) I8QL_TRY(check_matrix(qx, M));
    if (sx != nullptr && !aligned(sx, 4)) return I8QL_ERR_INVALID_ARG;
    if (acc_debug != nullptr && !aligned(acc_debug, 16)) return I8QL_ERR_INVALID_ARG;
    if (M == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_w8a8_decode_fused(x, qw, sw, bias, y, qx, sx, acc_debug, M, N, K, env));
}

i8ql_status w8a16_gemm(const i8ql_bf16* x, const int8_t* qw, const float* sw, i8ql_bf16* y,
                       int64_t M, int64_t N, int64_t K, void* stream) {
    I8QL_TRY(check_rows(M));
    I8QL_TRY(check_k(K));
    if (N <= 0) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_rows(N));
    I8QL_TRY(check_matrix(x, M));
    I8QL_TRY(check_matrix(qw, N));
    I8QL_TRY(check_vec(sw, N, 4));
    I8QL_TRY(check_matrix(y, M));
    if (M == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_w8a16(x, nullptr, 1, qw, sw, y, M, N, K, env));
}

i8ql_status grouped_w8a16_gemm(const i8ql_bf16* x, const int32_t* offsets, int64_t E,
                               const int8_t* qw, const float* sw, i8ql_bf16* y, int64_t T_total,
                               int64_t N, int64_t K, void* stream) {
    I8QL_TRY(check_rows(T_total));
    I8QL_TRY(check_k(K));
    if (N <= 0 || E <= 0) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_rows(N));
    if (E > 65535) return I8QL_ERR_UNSUPPORTED;
    if ((double)E * (double)N * (double)K > 9.0e18) return I8QL_ERR_UNSUPPORTED;
    if (offsets == nullptr || !aligned(offsets, 4)) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_matrix(x, T_total));
    if (qw == nullptr || !aligned(qw, 16)) return I8QL_ERR_INVALID_ARG;
    if (sw == nullptr || !aligned(sw, 4)) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_matrix(y, T_total));
    if (T_total == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_w8a16(x, offsets, E, qw, sw, y, T_total, N, K, env));
}

i8ql_status quantize_weight_per_channel_fp8(const i8ql_bf16* w, int64_t N, int64_t K, uint8_t* q, float* scale,
                                            void* stream) {
    I8QL_TRY(check_rows(N));
    I8QL_TRY(check_k(K));
    I8QL_TRY(check_matrix(w, N));
    I8QL_TRY(check_matrix(q, N));
    I8QL_TRY(check_vec(scale, N, 4));
    if (N == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_quant_rows_fp8(w, N, K, q, scale, env));
}

i8ql_status quantize_act_per_token_fp8(const i8ql_bf16* x, int64_t M, int64_t K, uint8_t* q, float* scale,
                                       void* stream) {
    return quantize_weight_per_channel_fp8(x, M, K, q, scale, stream);
}

i8ql_status w8a8_fp8_gemm(const uint8_t* qx, const float* sx, const uint8_t* qw, const float* sw,
                          const i8ql_bf16* bias, i8ql_bf16* y, int64_t M, int64_t N, int64_t K, void* stream) {
    I8QL_TRY(check_rows(M));
    I8QL_TRY(check_k(K));
    if (N <= 0) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_rows(N));
    I8QL_TRY(check_matrix(qx, M));
    I8QL_TRY(check_vec(sx, M, 4));
    I8QL_TRY(check_matrix(qw, N));
    I8QL_TRY(check_vec(sw, N, 4));
    if (bias != nullptr && !aligned(bias, 2)) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_matrix(y, M));
    if (M == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_fp8_gemm(qx, sx, qw, sw, bias, y, M, N, K, env));
}

i8ql_status w8a8_fp8_linear(const i8ql_bf16* x, const uint8_t* qw, const float* sw, const i8ql_bf16* bias,
                            i8ql_bf16* y, uint8_t* qx, float* sx, int64_t M, int64_t N, int64_t K, void* stream) {
    I8QL_TRY(check_rows(M));
    I8QL_TRY(check_k(K));
    if (N <= 0) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_rows(N));
    I8QL_TRY(check_matrix(x, M));
    I8QL_TRY(check_matrix(qw, N));
    I8QL_TRY(check_vec(sw, N, 4));
    if (bias != nullptr && !aligned(bias, 2)) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_matrix(y, M));
    if (qx != nullptr) I8QL_TRY(check_matrix(qx, M));
    if (sx != nullptr && !aligned(sx, 4)) return I8QL_ERR_INVALID_ARG;
    if (M == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_fp8_linear(x, qw, sw, bias, y, qx, sx, M, N, K, env));
}

i8ql_status quantize_weight_w4_g128(const i8ql_bf16* w, int64_t N, int64_t K, uint8_t* q, i8ql_bf16* scale,
                                    void* stream) {
    I8QL_TRY(check_rows(N));
    I8QL_TRY(check_k(K));
    if (K % 128 != 0) return I8QL_ERR_UNSUPPORTED;
    I8QL_TRY(check_matrix(w, N));
    I8QL_TRY(check_matrix(q, N));
    I8QL_TRY(check_vec(scale, N, 2));
    if (N == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_quant_w4(w, N, K, q, scale, env));
}

i8ql_status w4a16_gemm(const i8ql_bf16* x, const uint8_t* q, const i8ql_bf16* scale, i8ql_bf16* y, int64_t M,
                       int64_t N, int64_t K, void* stream) {
    I8QL_TRY(check_rows(M));
    I8QL_TRY(check_k(K));
    if (K % 128 != 0) return I8QL_ERR_UNSUPPORTED;
    if (N <= 0) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_rows(N));
    I8QL_TRY(check_matrix(x, M));
    I8QL_TRY(check_matrix(q, N));
    I8QL_TRY(check_vec(scale, N, 2));
    I8QL_TRY(check_matrix(y, M));
    if (M == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_w4a16(x, q, scale, y, M, N, K, env));
}

i8ql_status moe_route_topk(const float* logits, int64_t T, int64_t E, int64_t top_k, int64_t n_shared,
                           int32_t* offsets, int32_t* row_token, int32_t* token_row, float* slot_weight,
                           void* stream) {
    if (T < 0 || E <= 0 || top_k <= 0 || top_k > E || n_shared < 0) return I8QL_ERR_INVALID_ARG;
    if (E > 256 || n_shared > 64 || T > 65535 || moe_route_smem(T, E) == kRouteTooLarge)
        return I8QL_ERR_UNSUPPORTED;
    if (offsets == nullptr || !aligned(offsets, 4)) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_vec(logits, T, 4));
    I8QL_TRY(check_vec(row_token, T, 4));
    I8QL_TRY(check_vec(token_row, T, 4));
    I8QL_TRY(check_vec(slot_weight, T, 4));
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_moe_route(logits, T, E, top_k, n_shared, offsets, row_token, token_row, slot_weight, env));
}

i8ql_status grouped_w8a16_silu_mul(const i8ql_bf16* x, const int32_t* row_token, const int32_t* offsets, int64_t E,
                                   const int8_t* qw, const float* sw, i8ql_bf16* h, int64_t T_total, int64_t I,
                                   int64_t K, void* stream) {
    I8QL_TRY(check_rows(T_total));
    I8QL_TRY(check_k(K));
    if (I <= 0 || E <= 0) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_rows(2 * I));
    if (E > 65535) return I8QL_ERR_UNSUPPORTED;
    if ((double)E * (double)(2 * I) * (double)K > 9.0e18) return I8QL_ERR_UNSUPPORTED;
    if (offsets == nullptr || !aligned(offsets, 4)) return I8QL_ERR_INVALID_ARG;
    if (row_token != nullptr && !aligned(row_token, 4)) return I8QL_ERR_INVALID_ARG;
    if (x == nullptr && T_total > 0) return I8QL_ERR_INVALID_ARG;
    if (x != nullptr && !aligned(x, 16)) return I8QL_ERR_INVALID_ARG;
    if (qw == nullptr || !aligned(qw, 16)) return I8QL_ERR_INVALID_ARG;
    if (sw == nullptr || !aligned(sw, 4)) return I8QL_ERR_INVALID_ARG;
    if (T_total > 0 && (h == nullptr || !aligned(h, 2))) return I8QL_ERR_INVALID_ARG;
    if (T_total == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_w8a16(x, offsets, E, qw, sw, h, T_total, 2 * I, K, env, row_token, I));
}

i8ql_status moe_combine(const i8ql_bf16* yd, const int32_t* token_row, const float* slot_weight, i8ql_bf16* out,
                        int64_t T, int64_t S, int64_t H, void* stream) {
    if (T < 0 || S <= 0 || H <= 0) return I8QL_ERR_INVALID_ARG;
    if (H % 8 != 0 || T > 65535) return I8QL_ERR_UNSUPPORTED;
    I8QL_TRY(check_vec(token_row, T, 4));
    I8QL_TRY(check_vec(slot_weight, T, 4));
    I8QL_TRY(check_matrix(yd, T));
    I8QL_TRY(check_matrix(out, T));
    if (T == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_moe_combine(yd, token_row, slot_weight, out, T, S, H, env));
}

i8ql_status moe_expert_mlp_w8a16(const i8ql_bf16* x, const float* logits, int64_t E_routed, int64_t top_k,
                                 int64_t n_shared, const int8_t* qw_gate_up, const float* sw_gate_up,
                                 const int8_t* qw_down, const float* sw_down, i8ql_bf16* out, int64_t T, int64_t H,
                                 int64_t I, void* stream) {
    if (T < 0 || E_routed <= 0 || top_k <= 0 || top_k > E_routed || n_shared < 0 || H <= 0 || I <= 0)
        return I8QL_ERR_INVALID_ARG;
    if (E_routed > 256 || n_shared > 64 || T > 65535 || moe_route_smem(T, E_routed) == kRouteTooLarge)
        return I8QL_ERR_UNSUPPORTED;
    I8QL_TRY(check_k(H));
    I8QL_TRY(check_k(I));
    I8QL_TRY(check_matrix(x, T));
    I8QL_TRY(check_vec(logits, T, 4));
    I8QL_TRY(check_matrix(out, T));
    if (qw_gate_up == nullptr || !aligned(qw_gate_up, 16) || qw_down == nullptr || !aligned(qw_down, 16))
        return I8QL_ERR_INVALID_ARG;
    if (sw_gate_up == nullptr || !aligned(sw_gate_up, 4) || sw_down == nullptr || !aligned(sw_down, 4))
        return I8QL_ERR_INVALID_ARG;
    if (T == 0) return I8QL_OK;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    return from_cuda(launch_moe_mlp(x, logits, E_routed, top_k, n_shared, qw_gate_up, sw_gate_up, qw_down, sw_down,
                                    out, T, H, I, env));
}

i8ql_status i8ql_get_device_error(void* stream) {
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(stream, &env, &s)) return s;
    if (cudaStreamSynchronize(env.stream) != cudaSuccess) return I8QL_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, env.err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return I8QL_ERR_CUDA;
    if (word != 0) {
        const unsigned zero = 0;
        if (cudaMemcpy(env.err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return I8QL_ERR_CUDA;
    }
    if (word & kErrBitTimeout) return I8QL_ERR_TIMEOUT;
    if (word & kErrBitBadOffsets) return I8QL_ERR_BAD_OFFSETS;
    return I8QL_OK;
}

namespace {

i8ql_status plan_query(int64_t M, int64_t N, int64_t K, bool allow_sk, int32_t* tile_n, int32_t* split_k,
                       int32_t* cta_pair) {
    I8QL_TRY(check_rows(M));
    I8QL_TRY(check_k(K));
    if (N <= 0) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_rows(N));
    if (tile_n == nullptr || split_k == nullptr || cta_pair == nullptr) return I8QL_ERR_INVALID_ARG;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(nullptr, &env, &s)) return s;
    int bn = 0, split = 0, pair = 0;
    I8QL_TRY(from_cuda(w8a8_plan(M, N, K, env.sm_count, allow_sk, &bn, &split, &pair)));
    *tile_n = bn;
    *split_k = split;
    *cta_pair = pair;
    return I8QL_OK;
}

}  // namespace

i8ql_status i8ql_w8a8_plan(int64_t M, int64_t N, int64_t K, int32_t* tile_n, int32_t* split_k, int32_t* cta_pair) {
    return plan_query(M, N, K, true, tile_n, split_k, cta_pair);
}

i8ql_status i8ql_w8a8_noalloc_plan(int64_t M, int64_t N, int64_t K, int32_t* tile_n, int32_t* split_k,
                                   int32_t* cta_pair) {
    return plan_query(M, N, K, false, tile_n, split_k, cta_pair);
}

i8ql_status i8ql_w8a8_linear_launches(int64_t M, int64_t N, int64_t K, int32_t* launches) {
    I8QL_TRY(check_rows(M));
    I8QL_TRY(check_k(K));
    if (N <= 0) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_rows(N));
    if (launches == nullptr) return I8QL_ERR_INVALID_ARG;
    if (M == 0) {
        *launches = 0;
        return I8QL_OK;
    }
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(nullptr, &env, &s)) return s;
    *launches = w8a8_linear_one_launch(M, N, K, env.sm_count) ? 1 : 2;
    return I8QL_OK;
}

i8ql_status i8ql_fp8_plan(int64_t M, int64_t N, int64_t K, int32_t* tile_n, int32_t* split_k, int32_t* cta_pair) {
    I8QL_TRY(check_rows(M));
    I8QL_TRY(check_k(K));
    if (N <= 0) return I8QL_ERR_INVALID_ARG;
    I8QL_TRY(check_rows(N));
    if (tile_n == nullptr || split_k == nullptr || cta_pair == nullptr) return I8QL_ERR_INVALID_ARG;
    LaunchEnv env;
    i8ql_status s;
    if (!launch_env(nullptr, &env, &s)) return s;
    int bn = 0, split = 0, pair = 0;
    I8QL_TRY(from_cuda(fp8_plan(M, N, K, env.sm_count, &bn, &split, &pair)));
    *tile_n = bn;
    *split_k = split;
    *cta_pair = pair;
    return I8QL_OK;
}

const char* i8ql_status_string(i8ql_status status) {
    switch (status) {
        case I8QL_OK: return "ok";
        case I8QL_ERR_INVALID_ARG: return "invalid argument (null, negative size or misaligned pointer)";
        case I8QL_ERR_UNSUPPORTED: return "unsupported size (K must be a positive multiple of 16, at most 133144)";
        case I8QL_ERR_CUDA: return "CUDA runtime or launch failure";
        case I8QL_ERR_TIMEOUT: return "a kernel's bounded wait timed out";
        case I8QL_ERR_BAD_OFFSETS: return "grouped offsets are not 0..T_total and non-decreasing";
        case I8QL_ERR_NO_DEVICE: return "no usable sm_103 CUDA device";
        case I8QL_ERR_WORKSPACE_LIMIT:
            return "problem too large for the fixed workspace of w8a8_gemm_noalloc (M * K > 16 Mi for M > 32)";
        default: return "unknown status";
    }
}

int32_t i8ql_version(void) { return 1 * 10000 + 1 * 100 + 0; }

void i8ql_debug_stream_k_timeout(int32_t on) { g_debug_sk_timeout.store(on != 0 ? 1 : 0, std::memory_order_relaxed); }

void i8ql_set_early_weight_loads(int32_t on) { g_early_weights.store(on != 0 ? 1 : 0, std::memory_order_relaxed); }

int32_t i8ql_early_weight_loads(void) { return g_early_weights.load(std::memory_order_relaxed); }

}  // extern "C"
