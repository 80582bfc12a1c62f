// Per-row symmetric quantization: per-output-channel weights and per-token
// activations share this kernel, to int8 codes or to FP8 E4M3 codes.
//
// Sources: "Phase 5a: int8 weight-only quantization", Summary (per-output-
// channel int8, float32 scale arithmetic, zero-channel guard only for
// all-zero channels); "Day 6 -- Quantize It Yourself", The mechanism,
// blocks 1, 4 and 5 (q = clamp(round(w / s)), s = absmax / 127, round to
// nearest, per-token dynamic activation scales) and block 2 (the E4M3 grid,
// largest value 448: s = absmax / 448 for FP8 codes).
//
// One fused pass: each row is read once from HBM into registers (16-byte
// vector loads), its absmax is reduced across the threads that own it, and
// the codes are written from the same registers.  Rows longer than the
// register budget are read a second time (an L2 hit).  The arithmetic is
// IEEE fp32: __fdiv_rn for a / 127; the code of each element is the
// round-half-even of the IEEE quotient v / s, obtained from a multiply by the
// correctly rounded reciprocal except near ties, where the division itself
// is taken (see codes8()); no flush of subnormals (built without fast math).
// HBM traffic: 2 bytes read + 1 byte written per element, plus 4 bytes per row.

#include <cuda_runtime.h>

#include "common.cuh"
#include "quant_math.cuh"

namespace i8ql {
namespace {

constexpr int kQuantThreads = 256;


// Eight int8 codes (two words) -> eight fp16 codes (four words), exact: the
// biased byte u = q + 128 becomes the low mantissa byte of fp16 1024, and
// 1152 is subtracted.
__device__ __forceinline__ uint4 codes_to_f16(const uint2& c) {
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t u = (i == 0 ? c.x : c.y) ^ 0x80808080u;
        uint32_t lo = __byte_perm(u, 0x64646464u, 0x5150);
        uint32_t hi = __byte_perm(u, 0x64646464u, 0x5352);
        asm("sub.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
        asm("sub.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
        h[2 * i] = lo;
        h[2 * i + 1] = hi;
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

__device__ __forceinline__ uint4 load_nc(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// E4M3 codes of 8 values (two words of bf16 pairs): v / s by IEEE division,
// then the conversion instruction rounds to nearest even onto the E4M3 grid
// and saturates at +-448 (satfinite), keeping the sign of zero.
__device__ __forceinline__ uint2 codes8_fp8(const uint4& v, float s) {
    const float x[8] = {lo_bf16(v.x), hi_bf16(v.x), lo_bf16(v.y), hi_bf16(v.y),
                        lo_bf16(v.z), hi_bf16(v.z), lo_bf16(v.w), hi_bf16(v.w)};
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float t0 = __fdiv_rn(x[2 * i], s), t1 = __fdiv_rn(x[2 * i + 1], s);
        uint16_t pair;
        // the first source lands in the upper byte
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(t1), "f"(t0));
        h[i] = pair;
    }
    return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

// TPR threads own one row; VPT > 0 keeps up to VPT 8-element vectors per
// thread in registers, VPT == 0 streams the row twice.  INT8: the codes go to
// q (int8) and/or qh (the same codes as fp16, for the tensor-core GEMM);
// either may be null.  FP8 (E4M3, s = absmax / 448): the codes go to q.
template <int TPR, int VPT, bool FP8>
__global__ void __launch_bounds__(kQuantThreads)
quant_rows_kernel(const uint16_t* __restrict__ src, int64_t rows, int64_t K,
                  int8_t* __restrict__ q, uint16_t* __restrict__ qh, float* __restrict__ scale, int one_wave,
                  unsigned* __restrict__ zero, int nzero) {
    constexpr int kRowsPerCta = kQuantThreads / TPR;
    constexpr int kWarpsPerRow = TPR / 32;
    __shared__ float warp_max[kQuantThreads / 32];

    const int tid = threadIdx.x;
    const int rloc = tid / TPR;
    const int lt = tid % TPR;
    const int64_t row = (int64_t)blockIdx.x * kRowsPerCta + rloc;
    const bool valid = row < rows;
    // A one-wave grid may start while the previous kernel still runs: pull
    // the row into L2 meanwhile (the entry points bound K, so 2 * K fits the
    // 32-bit size).
    if (one_wave && valid && lt == 0) prefetch_l2(src + row * K, (uint32_t)(K * 2));
    pdl_wait();
    if (one_wave) pdl_launch_dependents();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < nzero; i += kQuantThreads) zero[i] = 0u;
    const int64_t nvec = K / 8;
    const uint4* rp = reinterpret_cast<const uint4*>(src) + (valid ? row : 0) * nvec;

    constexpr int kRegs = VPT > 0 ? VPT : 1;
    uint4 v[kRegs];
    float a = 0.0f;
    if constexpr (VPT > 0) {
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t idx = lt + (int64_t)i * TPR;
            if (valid && idx < nvec) {
                v[i] = load_nc(rp + idx);
            } else {
                v[i] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) a = absmax8(v[i], a);
    } else {
        if (valid)
            for (int64_t idx = lt; idx < nvec; idx += TPR) a = absmax8(rp[idx], a);
    }

#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if constexpr (kWarpsPerRow > 1) {
        if ((tid & 31) == 0) warp_max[tid >> 5] = a;
        __syncthreads();
        const int w0 = rloc * kWarpsPerRow;
#pragma unroll
        for (int w = 0; w < kWarpsPerRow; ++w) a = fmaxf(a, warp_max[w0 + w]);
    }

    // Zero-channel guard: only an all-zero row is special.
    const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, FP8 ? 448.0f : 127.0f);
    if (!valid) return;
    if (lt == 0) scale[row] = s;
    if constexpr (FP8) {
        uint2* fp = reinterpret_cast<uint2*>(q + row * K);
        if constexpr (VPT > 0) {
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int64_t idx = lt + (int64_t)i * TPR;
                if (idx < nvec) fp[idx] = codes8_fp8(v[i], s);
            }
        } else {
            for (int64_t idx = lt; idx < nvec; idx += TPR) fp[idx] = codes8_fp8(rp[idx], s);
        }
        return;
    }
    const RowScale rs = make_row_scale(s);

    uint2* qp = q ? reinterpret_cast<uint2*>(q + row * K) : nullptr;
    uint4* hp = qh ? reinterpret_cast<uint4*>(qh + row * K) : nullptr;
    auto put = [&](int64_t idx, const uint2& c) {
        if (qp) qp[idx] = c;
        if (hp) hp[idx] = codes_to_f16(c);
    };
    if constexpr (VPT > 0) {
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t idx = lt + (int64_t)i * TPR;
            if (idx < nvec) put(idx, codes8(v[i], rs));
        }
    } else {
        for (int64_t idx = lt; idx < nvec; idx += TPR) {
            const uint4 u = rp[idx];
            put(idx, codes8(u, rs));
        }
    }
}

template <int TPR, int VPT, bool FP8>
cudaError_t launch_cfg(const uint16_t* src, int64_t rows, int64_t K, int8_t* q, uint16_t* qh, float* s,
                       const LaunchEnv& env, unsigned* zero, int nzero) {
    constexpr int kRowsPerCta = kQuantThreads / TPR;
    const int64_t blocks = (rows + kRowsPerCta - 1) / kRowsPerCta;
    // one wave: every CTA resident at once (at least 2 per SM fit, 256 threads each)
    const int one_wave = blocks <= 2LL * env.sm_count ? 1 : 0;
    return launch_kernel(quant_rows_kernel<TPR, VPT, FP8>, dim3((unsigned)blocks), dim3(kQuantThreads), 0, env.stream,
                         kNoCluster, src, rows, K, q, qh, s, one_wave, zero, nzero);
}

template <bool FP8>
cudaError_t launch_rows(const uint16_t* src, int64_t rows, int64_t K, int8_t* q, uint16_t* qh, float* s,
                        const LaunchEnv& env, unsigned* zero, int nzero) {
    // Threads per row and vectors per thread (measured on weight and
    // activation shapes): many rows of moderate length go two warps to a
    // row (more CTAs resident, no CTA barrier per row pair); long rows keep
    // at most five vectors per thread, so that more CTAs fit on an SM.
    const int64_t nvec = K / 8;
    if (nvec <= 32 * 4) return launch_cfg<32, 4, FP8>(src, rows, K, q, qh, s, env, zero, nzero);
    if (nvec <= 64 * 6 && rows >= 4096) return launch_cfg<64, 6, FP8>(src, rows, K, q, qh, s, env, zero, nzero);
    if (nvec <= 128 * 4) return launch_cfg<128, 4, FP8>(src, rows, K, q, qh, s, env, zero, nzero);
    if (nvec <= 256 * 5) return launch_cfg<256, 5, FP8>(src, rows, K, q, qh, s, env, zero, nzero);
    if (nvec <= 256 * 8) return launch_cfg<256, 8, FP8>(src, rows, K, q, qh, s, env, zero, nzero);
    return launch_cfg<256, 0, FP8>(src, rows, K, q, qh, s, env, zero, nzero);
}

}  // namespace

cudaError_t launch_quant_rows(const uint16_t* src, int64_t rows, int64_t K, int8_t* q, uint16_t* qh, float* s,
                              const LaunchEnv& env, unsigned* zero, int nzero) {
    return launch_rows<false>(src, rows, K, q, qh, s, env, zero, nzero);
}

cudaError_t launch_quant_rows_fp8(const uint16_t* src, int64_t rows, int64_t K, uint8_t* q, float* s,
                                  const LaunchEnv& env) {
    return launch_rows<true>(src, rows, K, reinterpret_cast<int8_t*>(q), nullptr, s, env, nullptr, 0);
}

}  // namespace i8ql
