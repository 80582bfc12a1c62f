// W4A16 with one bf16 scale per 128 weights along K (group-128 int4).
//
// Source: "Day 6 -- Quantize It Yourself", The mechanism, block 1 (a
// W4A16-g128 tensor is int4 codes plus one bf16 scale per 128 weights along
// the input dimension; q = clamp(round(w / s)), s = absmax(group) / 7) and
// block 5 (W4A16: the weights are dequantized inside the kernel and the
// product runs on bf16 math, a pure memory-bandwidth win).
//
// Storage: codes [N, K / 2] bytes, two per byte (even k in the low nibble,
// 4-bit two's complement), scales [N, K / 128] bf16.  K % 128 == 0.
//
//   quantization: per group g of row n, a = max |w|, s = bf16_rne(a / 7)
//     (fp32 IEEE division; s = 1 if a == 0), q = clamp(rint(w / s), -7, 7)
//     with one IEEE fp32 division by the stored scale;
//   GEMM: y[m,n] = bf16_rne(sum_g s[n,g] * sum_{k in g} q[n,k] * x[m,k]),
//     each group's sum in fp32 on the tensor cores, scaled in fp32.
//
// GEMM design (decode sizes; the weight stream is the cost, half the bytes
// of W8A16): one 128-wide k-step is one scale group.  Each lane streams one
// 16-byte vector (32 codes) of each of its rows per k-step through a
// register ring; warps are the 16-row A operand of mma.sync m16n8k16 bf16
// and the tokens the 8-wide B operand ("swap AB").  Nibbles become bf16 with
// two logic ops and one packed subtraction per pair (the biased nibble in
// the mantissa of 128, minus 136: exact), which pairs code i with code i + 4
// of an 8-code word; the token operand is permuted the same way with byte
// permutes, so the k order the MMA sees is consistent.  Per k-step the
// group's partial sums start at zero and are added, times the row's scale,
// into the fp32 totals.  Split-K over a thread-block cluster reduces through
// distributed shared memory in rank order, as in the W8A16 kernel.

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "quant_math.cuh"

namespace cg = cooperative_groups;

namespace i8ql {
namespace {

constexpr int kW4Threads = 128;
constexpr int kW4Warps = kW4Threads / 32;
constexpr int kW4MaxSplit = 8;
constexpr int kGroup = 128;

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t bf16r(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// ------------------------------------------------------------------ quantization

__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}


// Four threads own one group of 128 weights (32 per thread: four 16-byte
// vectors, all loaded before any arithmetic so that 64 bytes per thread are
// in flight).  The codes are the int8 quantization's arithmetic with the
// stored bf16 scale as divisor (codes8: rint of the quotient through the
// correctly rounded reciprocal, with the IEEE division near half-integers).
// Its fast-path argument holds here a fortiori: s = bf16(fl32(a / 7)) is at
// least (a / 7)(1 - 2^-24)(1 - 2^-9), so |w / s| <= 7.014 and rint never
// leaves [-7, 7].  A scale that is subnormal in bf16 (a group whose absmax is
// below 7 * 2^-126) loses that bound, so such a group takes the IEEE division
// with the clamp, element by element.
__device__ __forceinline__ uint32_t nibbles8(uint2 b) {
    // bytes c0..c7 (two's complement) -> c0 | c1 << 4 | ... | c7 << 28
    uint32_t lo = b.x & 0x0f0f0f0fu, hi = b.y & 0x0f0f0f0fu;
    lo |= lo >> 4;
    hi |= hi >> 4;
    return __byte_perm(lo, hi, 0x6420);
}

__global__ void __launch_bounds__(256) quant_w4_kernel(const uint16_t* __restrict__ w, int64_t groups,
                                                        uint8_t* __restrict__ packed, uint16_t* __restrict__ scale) {
    pdl_wait();
    const int64_t gidx = ((int64_t)blockIdx.x * 256 + threadIdx.x) / 4;
    const int sub = threadIdx.x & 3;
    const bool valid = gidx < groups;
    // the matrix is contiguous and K % 128 == 0: group g covers elements
    // [128 g, 128 g + 128), its codes bytes [64 g, 64 g + 64)
    const uint4* src = reinterpret_cast<const uint4*>(w + gidx * kGroup + sub * 32);
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = valid ? ldg_stream16(src + i) : make_uint4(0, 0, 0, 0);
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) a = absmax8(v[i], a);
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    if (!valid) return;
    // the stored scale is bf16; the codes divide by it (zero group: 1)
    const uint16_t sb = a == 0.0f ? bf16r(1.0f) : bf16r(__fdiv_rn(a, 7.0f));
    const float s = bf16f(sb);
    if (sub == 0) scale[gidx] = sb;
    const RowScale rs = make_row_scale(s);
    uint32_t word[4];
    if ((sb & 0x7f80u) != 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) word[i] = nibbles8(codes8(v[i], rs));
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t vw[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            uint32_t acc = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float x = (j & 1) ? hi_bf16(vw[j / 2]) : lo_bf16(vw[j / 2]);
                const int c = max(-7, min(7, __float2int_rn(__fdiv_rn(x, s))));
                acc |= (uint32_t)(c & 15) << (4 * j);
            }
            word[i] = acc;
        }
    }
    *reinterpret_cast<uint4*>(packed + gidx * (kGroup / 2) + sub * 16) = make_uint4(word[0], word[1], word[2], word[3]);
}

// ------------------------------------------------------------------ GEMM

struct W4Params {
    const uint16_t* x;
    const uint8_t* q;
    const uint16_t* s;
    uint16_t* y;
    int64_t M, N, K;
    int one_wave;
};

// Eight codes of one 32-bit word (code i in bits 4i..4i+3) -> four bf16x2
// words holding the code pairs (0, 4), (1, 5), (2, 6), (3, 7), exactly: the
// biased nibble u = q + 8 goes into the mantissa of bf16 128 (0x4300 | u =
// 128 + u) and 136 is subtracted.
__device__ __forceinline__ void i4x8_to_bf16(uint32_t w, uint32_t (&out)[4]) {
    const uint32_t u = w ^ 0x88888888u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h = ((u >> (4 * i)) & 0x000f000fu) | 0x43004300u;
        asm("sub.rn.bf16x2 %0, %0, %1;" : "+r"(h) : "r"(0x43084308u));
        out[i] = h;
    }
}

// Eight token values (bf16 words (x0,x1), (x2,x3), (x4,x5), (x6,x7)) in the
// same pairing: (x0,x4), (x1,x5), (x2,x6), (x3,x7).
__device__ __forceinline__ void pair_tokens(const uint4& v, uint32_t (&out)[4]) {
    out[0] = __byte_perm(v.x, v.z, 0x5410);
    out[1] = __byte_perm(v.x, v.z, 0x7632);
    out[2] = __byte_perm(v.y, v.w, 0x5410);
    out[3] = __byte_perm(v.y, v.w, 0x7632);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int MT>
struct W4Regs {
    uint4 q[MT][2];      // rows g and g+8 of each 16-row m-tile: 32 codes each
    uint32_t s[MT];      // the two rows' group scales (bf16 bits, g low, g+8 high)
    uint4 x[4];          // one token tile (NT == 1): the step's 32 token values
};

// MT 16-row m-tiles per warp, NT 8-token n-tiles per pass.
template <int MT, int NT, int STAGES>
__global__ void __launch_bounds__(kW4Threads, NT >= 4 ? 2 : (NT == 1 ? 3 : 4)) w4a16_kernel(const W4Params p) {
    constexpr int kRows = 16 * MT;
    constexpr int kToks = 8 * NT;
    __shared__ float part[kW4Warps][kToks * kRows];
    {
        // stream this CTA's codes into L2 while the previous kernel drains
        const int64_t r0 = (int64_t)blockIdx.x * kRows;
        const int64_t ksteps = p.K / kGroup;
        const int S0 = (int)gridDim.y;
        const int64_t kb0 = ksteps * (int64_t)blockIdx.y / S0, kb1 = ksteps * ((int64_t)blockIdx.y + 1) / S0;
        const int r = (int)threadIdx.x;
        if (r < kRows && r0 + r < p.N && kb1 > kb0)
            prefetch_l2(p.q + (r0 + r) * (p.K / 2) + kb0 * (kGroup / 2), (uint32_t)((kb1 - kb0) * (kGroup / 2)));
    }
    pdl_wait();
    if (p.one_wave) pdl_launch_dependents();
    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int64_t N = p.N, K = p.K;
    const int64_t n0 = (int64_t)blockIdx.x * kRows;
    const int64_t G = K / kGroup;

    // this warp's k-steps (one scale group each) within the cluster's split
    const int units = S * kW4Warps;
    const int unit = rank * kW4Warps + warp;
    const int64_t ks_begin = G * unit / units;
    const int count = (int)(G * (unit + 1) / units - ks_begin);

    // Lane base pointers: lane t owns codes k = 32t .. 32t+31 of a k-step
    // (16 bytes).  Rows past N read row N-1, tokens past M the last token:
    // their products land only in outputs that are never stored.
    const uint8_t* qbase[MT][2];
    const uint16_t* sbase[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = min(n0 + mt * 16 + g + 8 * h, N - 1);
            qbase[mt][h] = p.q + n * (K / 2) + 16 * t + ks_begin * (kGroup / 2);
            sbase[mt][h] = p.s + n * G + ks_begin;
        }

    for (int64_t c0 = 0; c0 < p.M; c0 += kToks) {
        const int64_t chunk_hi = min(p.M, c0 + (int64_t)kToks);
        const int nt_active = (int)((chunk_hi - c0 + 7) / 8);
        const uint16_t* xbase[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            xbase[nt] = p.x + min(c0 + nt * 8 + g, chunk_hi - 1) * K + 32 * t + ks_begin * kGroup;

        float acc[MT][NT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.0f;

        auto load_w = [&](W4Regs<MT>& w, int i) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int h = 0; h < 2; ++h) w.q[mt][h] = ldg_stream16(qbase[mt][h] + (int64_t)i * (kGroup / 2));
                w.s[mt] = (uint32_t)__ldg(sbase[mt][0] + i) | ((uint32_t)__ldg(sbase[mt][1] + i) << 16);
            }
            if constexpr (NT == 1) {
                // the token values travel in the ring too: their L1 latency
                // then stays off the step's critical path
#pragma unroll
                for (int v = 0; v < 4; ++v) w.x[v] = __ldg(reinterpret_cast<const uint4*>(xbase[0] + (int64_t)i * kGroup) + v);
            }
        };
        auto step = [&](const W4Regs<MT>& w, int i) {
            float part_acc[MT][NT][4];  // this k-step's group sums
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) part_acc[mt][nt][r] = 0.0f;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                // word v: codes k = 32t + 8v .. +7, and the same 8 token
                // values, paired alike -> two MMAs of 4 pairs per tile
                uint32_t xb[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if constexpr (NT == 1) {
                        pair_tokens(w.x[v], xb[nt]);
                    } else if (nt < nt_active) {
                        pair_tokens(__ldg(reinterpret_cast<const uint4*>(xbase[nt] + (int64_t)i * kGroup) + v), xb[nt]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) xb[nt][j] = 0u;
                    }
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const uint32_t wgv = v == 0 ? w.q[mt][0].x : v == 1 ? w.q[mt][0].y : v == 2 ? w.q[mt][0].z : w.q[mt][0].w;
                    const uint32_t whv = v == 0 ? w.q[mt][1].x : v == 1 ? w.q[mt][1].y : v == 2 ? w.q[mt][1].z : w.q[mt][1].w;
                    uint32_t ag[4], ah[4];
                    i4x8_to_bf16(wgv, ag);
                    i4x8_to_bf16(whv, ah);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        if (nt < nt_active) {
                            mma16816(part_acc[mt][nt], ag[0], ah[0], ag[1], ah[1], xb[nt][0], xb[nt][1]);
                            mma16816(part_acc[mt][nt], ag[2], ah[2], ag[3], ah[3], xb[nt][2], xb[nt][3]);
                        }
                }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const float sg = bf16f((uint16_t)(w.s[mt] & 0xffffu)), sh = bf16f((uint16_t)(w.s[mt] >> 16));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    acc[mt][nt][0] = fmaf(sg, part_acc[mt][nt][0], acc[mt][nt][0]);
                    acc[mt][nt][1] = fmaf(sg, part_acc[mt][nt][1], acc[mt][nt][1]);
                    acc[mt][nt][2] = fmaf(sh, part_acc[mt][nt][2], acc[mt][nt][2]);
                    acc[mt][nt][3] = fmaf(sh, part_acc[mt][nt][3], acc[mt][nt][3]);
                }
            }
        };
        {
            W4Regs<MT> ring[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s)
                if (s < count) load_w(ring[s], s);
            for (int i0 = 0; i0 < count; i0 += STAGES) {
#pragma unroll
                for (int s = 0; s < STAGES; ++s) {
                    const int i = i0 + s;
                    if (i < count) {
                        step(ring[s], i);
                        if (i + STAGES < count) load_w(ring[s], i + STAGES);
                    }
                }
            }
        }

        // warp partials -> shared memory [token][row], then the cluster
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
        for (int i = threadIdx.x; i < kToks * kRows; i += kW4Threads) {
            float s = part[0][i];
#pragma unroll
            for (int w = 1; w < kW4Warps; ++w) s += part[w][i];
            part[0][i] = s;
        }
        if (S == 1)
            __syncthreads();
        else
            cluster.sync();
        const int total = nt_active * 8 * kRows;
        const int per = (total + S - 1) / S;
        const int i_begin = rank * per;
        const int i_end = min(total, i_begin + per);
        for (int i = i_begin + (int)threadIdx.x; i < i_end; i += kW4Threads) {
            float s;
            if (S == 1) {
                s = part[0][i];
            } else {
                float v[kW4MaxSplit];
#pragma unroll
                for (int r = 0; r < kW4MaxSplit; ++r) v[r] = r < S ? cluster.map_shared_rank(&part[0][0], r)[i] : 0.0f;
                s = v[0];
#pragma unroll
                for (int r = 1; r < kW4MaxSplit; ++r)
                    if (r < S) s += v[r];
            }
            const int row = i % kRows;
            const int tok = i / kRows;
            const int64_t n = n0 + row;
            const int64_t m = c0 + tok;
            if (n < N && m < p.M) p.y[m * N + n] = bf16r(s);
        }
        if (S == 1)
            __syncthreads();
        else
            asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
    }
}

template <int MT, int NT, int STAGES>
int w4_resident() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 1;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, w4a16_kernel<MT, NT, STAGES>, kW4Threads, 0) !=
                cudaSuccess || n < 1)
            n = 1;
        cached[dev] = n;
    }
    return cached[dev];
}

template <int MT, int NT, int STAGES>
cudaError_t w4_launch(W4Params p, const LaunchEnv& env) {
    constexpr int kRows = 16 * MT;
    const int64_t row_blocks = (p.N + kRows - 1) / kRows;
    const int64_t capacity = (int64_t)env.sm_count * w4_resident<MT, NT, STAGES>();
    const int64_t groups = p.K / kGroup;
    // split-K: fill one wave, keep at least two k-steps per warp, one portable cluster
    int64_t split = std::max<int64_t>(1, capacity / std::max<int64_t>(1, row_blocks));
    split = std::min<int64_t>(split, std::max<int64_t>(1, groups / (2 * kW4Warps)));
    split = std::min<int64_t>(split, kW4MaxSplit);
    p.one_wave = row_blocks * split <= capacity ? 1 : 0;
    return launch_kernel(w4a16_kernel<MT, NT, STAGES>, dim3((unsigned)row_blocks, (unsigned)split, 1),
                         dim3(kW4Threads), 0, env.stream, dim3(1, (unsigned)split, 1), p);
}

}  // namespace

cudaError_t launch_quant_w4(const uint16_t* w, int64_t N, int64_t K, uint8_t* packed, uint16_t* scale,
                            const LaunchEnv& env) {
    const int64_t groups = N * (K / kGroup);
    const int64_t blocks = (groups * 4 + 255) / 256;
    return launch_kernel(quant_w4_kernel, dim3((unsigned)blocks), dim3(256), 0, env.stream, kNoCluster, w, groups,
                         packed, scale);
}

cudaError_t launch_w4a16(const uint16_t* x, const uint8_t* q, const uint16_t* s, uint16_t* y, int64_t M, int64_t N,
                         int64_t K, const LaunchEnv& env) {
    W4Params p{x, q, s, y, M, N, K, 0};
    if (M <= 8) return w4_launch<2, 1, 2>(p, env);
    if (M <= 16) return w4_launch<1, 2, 3>(p, env);
    if (M <= 32) return w4_launch<1, 4, 2>(p, env);
    return w4_launch<1, 8, 2>(p, env);
}

}  // namespace i8ql
