// Weight-only W8A16 GEMM/GEMV for decode, plain and grouped over MoE experts.
//
// Sources: "Day 6 -- Quantize It Yourself", The mechanism, block 5 (int8
// weights dequantized inside the kernel, the product on bf16 tensor math, a
// pure memory-bandwidth win for decode) and "Phase 5a: int8 weight-only
// quantization", Summary (grouped GEMM over MoE experts with stacked
// [E, N, K] int8 weights and per-output-channel scales).
//
//   y[m,n] = bf16_rne(sw[n] * sum_k q[n,k] * x[m,k])
//
// Design (bandwidth kernel, one HBM pass over the int8 weights):
//  * Each lane streams 16-byte vectors of int8 weights (ld.global.nc, two
//    k-steps in flight per lane), so a warp reads 64 contiguous bytes of each
//    of its rows per k-step.
//  * The int8 codes become bf16 in registers (exact: |q| <= 127) and feed
//    legacy mma.sync m16n8k16 bf16 with weights as the 16-row A operand and
//    the tokens as the 8-wide B operand ("swap AB"), fp32 accumulation.  The
//    fp32 scale is applied once per output in the epilogue, so s * q is
//    never rounded to bf16.
//  * The k order inside each 64-wide k-step is permuted identically for A
//    and B (lane t owns k = 16t .. 16t+15), which lets every lane load its
//    weights and tokens with plain 16-byte vectors and no shuffles.
//  * Split-K without global scratch: the S CTAs of a thread-block cluster
//    own disjoint k-ranges of the same rows; the four warps of a CTA are
//    reduced in shared memory, then the cluster is reduced through
//    distributed shared memory in a fixed rank order (deterministic).
//  * Grouped: blockIdx.z is the expert; an expert with no rows exits before
//    reading any weight.  Offsets are validated on the device; a bad expert
//    is skipped and reported through the sticky fault word.
// HBM traffic per launch: N*K weight bytes (+4N scale bytes) per active
// expert, + 2*M*K token bytes + 2*M*N output bytes.

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace i8ql {
namespace {

constexpr int kW8A16Threads = 128;
constexpr int kW8A16Warps = kW8A16Threads / 32;
constexpr int kMaxClusterSplit = 8;

struct W8A16Params {
    const uint16_t* x;
    const int32_t* offsets;  // null for the plain GEMM
    const int8_t* qw;
    const float* sw;
    uint16_t* y;
    int64_t rows;  // M (plain) or T_total (grouped)
    int64_t N;
    int64_t K;
    int64_t E;
    unsigned* err;
};

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_cached(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// Four int8 codes -> two bf16x2 words (exact).  Each byte b is biased to
// u = b + 128, placed in the low mantissa bits of 2^23 (float 2^23 + u),
// and 2^23 + 128 is subtracted (packed f32x2); the upper halves of the exact
// fp32 results are the bf16 values.
__device__ __forceinline__ void i8x4_to_bf16(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t f0 = __byte_perm(u, 0x4b000000u, 0x7440);
    const uint32_t f1 = __byte_perm(u, 0x4b000000u, 0x7441);
    const uint32_t f2 = __byte_perm(u, 0x4b000000u, 0x7442);
    const uint32_t f3 = __byte_perm(u, 0x4b000000u, 0x7443);
    const uint64_t bias = 0xcb000080cb000080ull;  // (-(2^23 + 128), -(2^23 + 128))
    uint64_t p01 = ((uint64_t)f1 << 32) | f0;
    uint64_t p23 = ((uint64_t)f3 << 32) | f2;
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(p01) : "l"(bias));
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(p23) : "l"(bias));
    lo = __byte_perm((uint32_t)p01, (uint32_t)(p01 >> 32), 0x7632);
    hi = __byte_perm((uint32_t)p23, (uint32_t)(p23 >> 32), 0x7632);
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <int MT>
struct WeightRegs {
    uint4 r[MT][2];  // rows g and g+8 of each 16-row m-tile
};

// MT 16-row m-tiles per warp, NT 8-token n-tiles per pass.
template <int MT, int NT, bool GROUPED>
__global__ void __launch_bounds__(kW8A16Threads)
w8a16_kernel(const W8A16Params p) {
    constexpr int kRows = 16 * MT;
    constexpr int kToks = 8 * NT;
    __shared__ float part[kW8A16Warps][kToks * kRows];

    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int64_t N = p.N, K = p.K;
    const int64_t n0 = (int64_t)blockIdx.x * kRows;

    // Row range of this expert (grouped) or of the whole batch.
    int64_t lo = 0, hi = p.rows;
    const int8_t* qw = p.qw;
    const float* sw = p.sw;
    if constexpr (GROUPED) {
        const int64_t e = blockIdx.z;
        const int64_t a = p.offsets[e], b = p.offsets[e + 1];
        const bool bad = a < 0 || b < a || b > p.rows || (e == 0 && a != 0) ||
                         (e == p.E - 1 && b != p.rows);
        if (bad) {
            if (blockIdx.x == 0 && rank == 0 && threadIdx.x == 0) record_fault(p.err, kErrBitBadOffsets);
            return;  // the whole cluster shares e, so all of it leaves here
        }
        lo = a;
        hi = b;
        qw += e * N * K;
        sw += e * N;
    }
    if (hi <= lo) return;  // an empty expert reads no weights

    // This warp's k-steps (64 k each) within the cluster's split of K.
    const int64_t ksteps = (K + 63) / 64;
    const int units = S * kW8A16Warps;
    const int unit = rank * kW8A16Warps + warp;
    const int64_t ks_begin = ksteps * unit / units;
    const int64_t ks_end = ksteps * (unit + 1) / units;

    // Weight row pointers of this lane (clamped rows are never loaded).
    const int8_t* wrow[MT][2];
    bool wok[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = n0 + mt * 16 + g + 8 * h;
            wok[mt][h] = n < N;
            wrow[mt][h] = qw + (wok[mt][h] ? n : 0) * K + 16 * t;
        }

    auto load_w = [&](WeightRegs<MT>& w, int64_t ks) {
        const int64_t k0 = ks * 64;
        const bool kok = k0 + 16 * t < K;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                w.r[mt][h] = (kok && wok[mt][h]) ? ldg_stream(wrow[mt][h] + k0) : make_uint4(0, 0, 0, 0);
    };

    for (int64_t c0 = lo; c0 < hi; c0 += kToks) {
        const int64_t chunk = min((int64_t)kToks, hi - c0);
        const int nt_active = (int)((chunk + 7) / 8);

        float acc[MT][NT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.0f;

        auto compute = [&](const WeightRegs<MT>& w, int64_t ks) {
            const int64_t k0 = ks * 64 + 16 * t;
            const bool kok = k0 < K;
            uint32_t xb[NT][8];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int64_t m = c0 + nt * 8 + g;
                if (nt < nt_active && kok && m < hi) {
                    const uint16_t* xp = p.x + m * K + k0;
                    const uint4 v0 = ldg_cached(xp);
                    const uint4 v1 = ldg_cached(xp + 8);
                    xb[nt][0] = v0.x; xb[nt][1] = v0.y; xb[nt][2] = v0.z; xb[nt][3] = v0.w;
                    xb[nt][4] = v1.x; xb[nt][5] = v1.y; xb[nt][6] = v1.z; xb[nt][7] = v1.w;
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) xb[nt][i] = 0u;
                }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const uint32_t wg[4] = {w.r[mt][0].x, w.r[mt][0].y, w.r[mt][0].z, w.r[mt][0].w};
                const uint32_t wh[4] = {w.r[mt][1].x, w.r[mt][1].y, w.r[mt][1].z, w.r[mt][1].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t a0, a2, a1, a3;
                    i8x4_to_bf16(wg[j], a0, a2);  // row g:   k 16t+4j+{0,1} | {2,3}
                    i8x4_to_bf16(wh[j], a1, a3);  // row g+8: same k
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        if (nt < nt_active) mma_bf16(acc[mt][nt], a0, a1, a2, a3, xb[nt][2 * j], xb[nt][2 * j + 1]);
                }
            }
        };

        if (ks_begin < ks_end) {
            WeightRegs<MT> wa, wb;
            load_w(wa, ks_begin);
            for (int64_t ks = ks_begin; ks < ks_end; ks += 2) {
                const bool two = ks + 1 < ks_end;
                if (two) load_w(wb, ks + 1);
                compute(wa, ks);
                if (two) {
                    if (ks + 2 < ks_end) load_w(wa, ks + 2);
                    compute(wb, ks + 1);
                }
            }
        }

        // Warp partials -> shared memory, laid out [token][row].
        float* mine = part[warp];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int r = mt * 16 + g;
                const int c = nt * 8 + 2 * t;
                mine[c * kRows + r] = acc[mt][nt][0];
                mine[(c + 1) * kRows + r] = acc[mt][nt][1];
                mine[c * kRows + r + 8] = acc[mt][nt][2];
                mine[(c + 1) * kRows + r + 8] = acc[mt][nt][3];
            }
        __syncthreads();
        // Sum the four warps in order into part[0].
        for (int i = threadIdx.x; i < kToks * kRows; i += kW8A16Threads) {
            float s = part[0][i];
#pragma unroll
            for (int w = 1; w < kW8A16Warps; ++w) s += part[w][i];
            part[0][i] = s;
        }
        // Publish to the cluster, then each rank finishes a slice of the tile.
        cluster.sync();
        const int total = nt_active * 8 * kRows;
        const int per = (total + S - 1) / S;
        const int i_begin = rank * per;
        const int i_end = min(total, i_begin + per);
        for (int i = i_begin + (int)threadIdx.x; i < i_end; i += kW8A16Threads) {
            float s = 0.0f;
            for (int r = 0; r < S; ++r) s += cluster.map_shared_rank(&part[0][0], r)[i];
            const int row = i % kRows;
            const int tok = i / kRows;
            const int64_t n = n0 + row;
            const int64_t m = c0 + tok;
            if (n < N && m < hi) p.y[m * N + n] = f32_to_bf16_rn(s * sw[n]);
        }
        cluster.sync();  // peers are done reading this CTA's shared memory
    }
}

template <int MT, int NT, bool GROUPED>
cudaError_t launch_cfg(const W8A16Params& p, int split, int64_t experts, cudaStream_t stream) {
    constexpr int kRows = 16 * MT;
    const int64_t row_blocks = (p.N + kRows - 1) / kRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)row_blocks, (unsigned)split, (unsigned)experts);
    cfg.blockDim = dim3(kW8A16Threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)split;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, w8a16_kernel<MT, NT, GROUPED>, p);
}

template <bool GROUPED>
cudaError_t dispatch(const W8A16Params& p, int64_t tokens_hint, int64_t active_hint, int sms,
                     cudaStream_t stream) {
    const int64_t ksteps = (p.K + 63) / 64;
    const int mt = tokens_hint <= 16 ? 4 : 2;
    const int64_t row_blocks = (p.N + 16 * mt - 1) / (16 * mt);
    const int64_t want = 3LL * sms;
    int64_t split = (want + row_blocks * active_hint - 1) / (row_blocks * active_hint);
    split = std::min<int64_t>(split, std::max<int64_t>(1, ksteps / (2 * kW8A16Warps)));
    split = std::max<int64_t>(1, std::min<int64_t>(split, kMaxClusterSplit));
    const int s = (int)split;
    if (tokens_hint <= 8) return launch_cfg<4, 1, GROUPED>(p, s, p.E, stream);
    if (tokens_hint <= 16) return launch_cfg<4, 2, GROUPED>(p, s, p.E, stream);
    if (tokens_hint <= 32) return launch_cfg<2, 4, GROUPED>(p, s, p.E, stream);
    return launch_cfg<2, 8, GROUPED>(p, s, p.E, stream);
}

}  // namespace

cudaError_t launch_w8a16(const uint16_t* x, const int32_t* offsets, int64_t E, const int8_t* qw,
                         const float* sw, uint16_t* y, int64_t M, int64_t N, int64_t K,
                         const LaunchEnv& env) {
    W8A16Params p{x, offsets, qw, sw, y, M, N, K, E, env.err};
    if (offsets == nullptr) return dispatch<false>(p, M, 1, env.sm_count, env.stream);
    // Grouped: at most min(E, T_total) experts have rows; an expert sees at
    // most T_total rows, and on average T_total / active.
    const int64_t active = std::min<int64_t>(E, M);
    const int64_t per_expert = (M + active - 1) / active;
    return dispatch<true>(p, std::max<int64_t>(per_expert, 1), active, env.sm_count, env.stream);
}

}  // namespace i8ql
