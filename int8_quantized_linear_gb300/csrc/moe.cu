// The MoE layer around the grouped W8A16 GEMM: routing of tokens to experts
// on the device, and the weighted combine of the experts' output rows.
//
// Source: "Phase 5a: int8 weight-only quantization", Summary (the grouped
// int8 GEMM serves the MoE layer of deepseek-moe-16b: stacked expert
// weights, per-expert token groups), with that model's layer as the
// benchmark configuration states it: softmax over the gate logits, top-6 of
// 64 routed experts per token, plus 2 shared experts that see every token.
//
//   routing: p[t,e] = softmax_e(logits[t,:]); the top_k experts of largest
//     logit (equal logits: the lower expert index first; the softmax is
//     increasing in the logit); rows grouped by expert (routed 0 .. E-1,
//     then shared E .. E+shared-1), tokens increasing within an expert;
//     slot weights p[t,e] for routed slots, 1 for shared ones;
//   combine: out[t,:] = bf16(sum_s w[t,s] * yd[token_row[t,s], :]), slots in
//     order, fp32.
//
// Routing is two kernels.  The selection spreads the tokens over the GPU,
// one warp per token (softmax denominator and top-k by warp reductions, ties
// to the lower index).  The grouping runs in one CTA: it marks each chosen
// (expert, token) in a per-expert token bitmap in shared memory, and then
// every (token, slot) finds its row as the expert's offset plus the number
// of earlier tokens in the expert's bitmap.  The grouping is therefore
// deterministic and identical to the definition, with no atomics on global
// memory.  Up to 32 tokens the grouping CTA's warps select them first (one
// launch); beyond, one CTA doing both measured 19.7 us at T = 64, issue-bound
// on its one SM, so the selection is its own launch.

#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"

namespace i8ql {
namespace {

constexpr int kRouteThreads = 1024;
constexpr int kSelectThreads = 256;
constexpr int kInlineSelectTokens = kRouteThreads / 32;  // tokens the grouping CTA selects itself
constexpr int kMaxLogitsPerLane = 8;  // E <= 256

struct RouteParams {
    const float* logits;
    int64_t T, E, topk, shared;
    int32_t* offsets;
    int32_t* row_token;
    int32_t* token_row;  // [T, topk + shared]; holds expert ids until the rows are known
    float* slot_weight;  // [T, topk + shared]
};

// Selection of token t by one warp: the softmax denominator and the top_k
// largest logits by repeated warp argmax (equal logits: the lower index).
// Writes each routed slot's expert id into token_row (the grouping turns it
// into a row) and its weight, and weight 1 for the shared slots.
__device__ __forceinline__ void select_token(const RouteParams& p, int t, int lane) {
    const int E = (int)p.E, topk = (int)p.topk, S = (int)(p.topk + p.shared);
    const float* lt = p.logits + (int64_t)t * E;
    float l[kMaxLogitsPerLane];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxLogitsPerLane; ++i) {
        const int e = lane + 32 * i;
        l[i] = e < E ? __ldg(lt + e) : -INFINITY;
        mx = fmaxf(mx, l[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxLogitsPerLane; ++i)
        if (lane + 32 * i < E) sum += expf(l[i] - mx);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    unsigned taken = 0u;  // this lane's chosen logits
    for (int s = 0; s < topk; ++s) {
        // the lane's best untaken logit, lowest index first among equals
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kMaxLogitsPerLane; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !(taken >> i & 1u) && (l[i] > bv || bi == 0x7fffffff)) {
                bv = l[i];
                bi = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == (bi & 31)) taken |= 1u << (bi >> 5);
        if (lane == (s & 31)) {  // slot s is written by one lane (top_k may exceed 32)
            p.token_row[(int64_t)t * S + s] = bi;
            p.slot_weight[(int64_t)t * S + s] = expf(bv - mx) / sum;
        }
    }
    for (int s = topk + lane; s < S; s += 32) p.slot_weight[(int64_t)t * S + s] = 1.0f;
}

// Selection, one warp per token, the tokens spread over the whole GPU.
__global__ void __launch_bounds__(kSelectThreads) moe_select_kernel(const RouteParams p) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    pdl_wait();
    for (int t = blockIdx.x * (kSelectThreads / 32) + warp; t < (int)p.T; t += gridDim.x * (kSelectThreads / 32))
        select_token(p, t, lane);
}

// Grouping, one CTA: each (token, routed slot) marks its expert's token
// bitmap in shared memory; per-expert counts give the offsets (a warp scan),
// and every (token, slot) finds its row as the expert's offset plus the
// number of earlier tokens in the expert's bitmap -- deterministic, with no
// atomics on global memory.
__global__ void __launch_bounds__(kRouteThreads) moe_group_kernel(const RouteParams p) {
    extern __shared__ uint32_t route_smem[];
    const int T = (int)p.T, E = (int)p.E, topk = (int)p.topk, shared = (int)p.shared;
    const int S = topk + shared;
    const int W = (T + 31) / 32;               // bitmap words per expert
    uint32_t* bits = route_smem;               // [E][W]
    uint32_t* before = route_smem + E * W;     // [E][W] set bits in earlier words
    __shared__ int32_t offs[257 + 64];
    pdl_wait();
    if (T <= kInlineSelectTokens) {
        // few tokens: this CTA's warps select them too (no separate launch)
        if ((int)(threadIdx.x >> 5) < T) select_token(p, (int)(threadIdx.x >> 5), (int)(threadIdx.x & 31));
    }
    for (int i = threadIdx.x; i < E * W; i += kRouteThreads) bits[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < T * topk; i += kRouteThreads) {
        const int t = i / topk, s = i - t * topk;
        const int e = p.token_row[(int64_t)t * S + s];
        atomicOr(&bits[e * W + (t >> 5)], 1u << (t & 31));
    }
    __syncthreads();

    // ---- per-expert counts and running counts of earlier words
    for (int e = threadIdx.x; e < E; e += kRouteThreads) {
        uint32_t run = 0;
        for (int w = 0; w < W; ++w) {
            before[e * W + w] = run;
            run += __popc(bits[e * W + w]);
        }
        offs[e] = (int32_t)run;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        // offsets: exclusive scan of the counts (routed, then shared: T each),
        // each lane summing a run of consecutive experts
        const int lane = threadIdx.x;
        const int n = E + shared;
        const int per = (n + 31) / 32;
        const int lo = min(n, lane * per), hi = min(n, lo + per);
        int32_t local = 0;
        for (int e = lo; e < hi; ++e) local += e < E ? offs[e] : T;
        int32_t incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        int32_t acc = incl - local;
        __syncwarp();
        for (int e = lo; e < hi; ++e) {
            const int32_t c = e < E ? offs[e] : T;
            offs[e] = acc;
            p.offsets[e] = acc;
            acc += c;
        }
        if (lane == 31) {
            offs[n] = incl;
            p.offsets[n] = incl;
        }
    }
    __syncthreads();

    // ---- rows of every (token, slot)
    for (int i = threadIdx.x; i < T * S; i += kRouteThreads) {
        const int t = i / S, s = i - t * S;
        int row;
        if (s < topk) {
            const int e = p.token_row[i];
            const uint32_t mask = (1u << (t & 31)) - 1u;
            row = offs[e] + (int)before[e * W + (t >> 5)] + __popc(bits[e * W + (t >> 5)] & mask);
        } else {
            row = offs[E + (s - topk)] + t;
        }
        p.token_row[i] = row;
        p.row_token[row] = t;
    }
}

// out[t, :] for 8 columns per thread: the slots' rows weighted in order.
// The slot rows and weights, then the slots' output vectors, are loaded in
// batches of 8 ahead of the arithmetic, so the gathers overlap.
__global__ void __launch_bounds__(256) moe_combine_kernel(const uint16_t* __restrict__ yd,
                                                          const int32_t* __restrict__ token_row,
                                                          const float* __restrict__ slot_weight,
                                                          uint16_t* __restrict__ out, int64_t S, int64_t H) {
    pdl_wait();
    const int64_t t = blockIdx.y;
    const int64_t c = ((int64_t)blockIdx.x * 256 + threadIdx.x) * 8;
    if (c >= H) return;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int64_t s0 = 0; s0 < S; s0 += 8) {
        int32_t row[8];
        float w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const bool ok = s0 + j < S;
            row[j] = ok ? __ldg(token_row + t * S + s0 + j) : 0;
            w[j] = ok ? __ldg(slot_weight + t * S + s0 + j) : 0.0f;
        }
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = s0 + j < S ? __ldg(reinterpret_cast<const uint4*>(yd + (int64_t)row[j] * H + c)) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (s0 + j >= S) break;
            const uint32_t words[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[2 * q] = fmaf(w[j], __uint_as_float(words[q] << 16), acc[2 * q]);
                acc[2 * q + 1] = fmaf(w[j], __uint_as_float(words[q] & 0xffff0000u), acc[2 * q + 1]);
            }
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        o[j] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * j])) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * j + 1])) << 16);
    *reinterpret_cast<uint4*>(out + t * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

// Shared memory the routing kernel needs (kRouteTooLarge: beyond what one
// CTA holds).
size_t moe_route_smem(int64_t T, int64_t E) {
    const int64_t W = (T + 31) / 32;
    const size_t bytes = (size_t)(2 * E * W) * sizeof(uint32_t);
    return bytes <= 200 * 1024 ? bytes : kRouteTooLarge;
}

cudaError_t launch_moe_route(const float* logits, int64_t T, int64_t E, int64_t topk, int64_t shared,
                             int32_t* offsets, int32_t* row_token, int32_t* token_row, float* slot_weight,
                             const LaunchEnv& env) {
    const size_t smem = moe_route_smem(T, E);
    if (smem == kRouteTooLarge) return cudaErrorInvalidValue;
    static bool opted[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !opted[dev]) {
        if ((e = cudaFuncSetAttribute(moe_group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024)) !=
            cudaSuccess)
            return e;
        opted[dev] = true;
    }
    RouteParams p{logits, T, E, topk, shared, offsets, row_token, token_row, slot_weight};
    if (T > kInlineSelectTokens) {
        const int64_t blocks = std::min<int64_t>((T + kSelectThreads / 32 - 1) / (kSelectThreads / 32), 4 * env.sm_count);
        e = launch_kernel(moe_select_kernel, dim3((unsigned)blocks), dim3(kSelectThreads), 0, env.stream, kNoCluster, p);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(moe_group_kernel, dim3(1), dim3(kRouteThreads), smem, env.stream, kNoCluster, p);
}

cudaError_t launch_moe_combine(const uint16_t* yd, const int32_t* token_row, const float* slot_weight, uint16_t* out,
                               int64_t T, int64_t S, int64_t H, const LaunchEnv& env) {
    const dim3 grid((unsigned)((H / 8 + 255) / 256), (unsigned)T);
    return launch_kernel(moe_combine_kernel, grid, dim3(256), 0, env.stream, kNoCluster, yd, token_row, slot_weight,
                         out, S, H);
}

cudaError_t launch_moe_mlp(const uint16_t* x, const float* logits, int64_t E_routed, int64_t topk, int64_t shared,
                           const int8_t* qw_gu, const float* sw_gu, const int8_t* qw_d, const float* sw_d,
                           uint16_t* out, int64_t T, int64_t H, int64_t I, const LaunchEnv& env) {
    const int64_t E = E_routed + shared;
    const int64_t S = topk + shared;
    const int64_t rows = T * S;  // every token in top_k routed and all shared experts
    auto pad = [](size_t n) { return (n + 255) / 256 * 256; };
    const size_t off_b = pad((size_t)(E + 1) * 4), idx_b = pad((size_t)rows * 4);
    const size_t h_b = pad((size_t)rows * (size_t)I * 2), yd_b = pad((size_t)rows * (size_t)H * 2);
    void* ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, off_b + 3 * idx_b + h_b + yd_b, env.stream);
    if (e != cudaSuccess) return e;
    uint8_t* w = static_cast<uint8_t*>(ws);
    int32_t* offsets = reinterpret_cast<int32_t*>(w);
    int32_t* row_token = reinterpret_cast<int32_t*>(w + off_b);
    int32_t* token_row = reinterpret_cast<int32_t*>(w + off_b + idx_b);
    float* slot_weight = reinterpret_cast<float*>(w + off_b + 2 * idx_b);
    uint16_t* h = reinterpret_cast<uint16_t*>(w + off_b + 3 * idx_b);
    uint16_t* yd = reinterpret_cast<uint16_t*>(w + off_b + 3 * idx_b + h_b);
    e = launch_moe_route(logits, T, E_routed, topk, shared, offsets, row_token, token_row, slot_weight, env);
    if (e == cudaSuccess) e = launch_w8a16(x, offsets, E, qw_gu, sw_gu, h, rows, 2 * I, H, env, row_token, I);
    if (e == cudaSuccess) e = launch_w8a16(h, offsets, E, qw_d, sw_d, yd, rows, H, I, env);
    if (e == cudaSuccess) e = launch_moe_combine(yd, token_row, slot_weight, out, T, S, H, env);
    const cudaError_t f = cudaFreeAsync(ws, env.stream);
    return e != cudaSuccess ? e : f;
}

}  // namespace i8ql
