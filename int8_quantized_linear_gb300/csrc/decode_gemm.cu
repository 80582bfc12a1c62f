// Decode-size GEMMs (few tokens, weight streaming): W8A16, grouped W8A16 over
// MoE experts, and W8A8 for small M.
//
// Sources: "Day 6 -- Quantize It Yourself", The mechanism, block 5 (weight-
// only int8 is dequantized inside the kernel and multiplied on bf16 math, a
// pure memory-bandwidth win for decode; W8A8 multiplies 8-bit operands on the
// tensor cores); "Phase 5a: int8 weight-only quantization", Summary (grouped
// GEMM over MoE experts with stacked [E, N, K] int8 weights and per-output-
// channel scales); "feat(quantization): support compressed-tensors W8A8 and
// mixed modules", Design and Supported Execution Scheme (per-channel int8
// weights, per-token int8 activations, no output quantization).
//
//   W8A16: y[m,n] = bf16_rne(sw[n] * sum_k q[n,k] * x[m,k])          (fp32 acc)
//   W8A8:  y[m,n] = bf16_rne(((float)acc * sx[m]) * sw[n] (+ bias[n])),
//          acc = sum_k qx[m,k] * qw[n,k]                              (exact int32)
//
// Design (bandwidth kernel, one HBM pass over the int8 weights):
//  * Each lane streams 16-byte vectors of int8 weights (ld.global.nc) through
//    a 4-deep register ring (three k-steps in flight per lane while one is
//    computed): a warp reads 64 contiguous bytes of each of its 32 rows per
//    64-wide k-step.  The grid is one wave of resident CTAs.
//  * Weights are the 16-row A operand of legacy warp-level mma.sync and the
//    tokens the 8-wide B operand ("swap AB"), so the MMA does no work on
//    absent tokens beyond the 8-token granule.
//      W8A16: int8 codes become bf16 in registers (exact, |q| <= 127) and run
//      m16n8k16 bf16 with fp32 accumulation; the fp32 scale is applied once
//      per output, so s * q is never rounded to bf16.
//      W8A8: codes and token codes go straight into m16n8k32 s8 x s8 -> s32,
//      with no conversion at all and an exact int32 accumulator.
//  * The k order inside a 64-wide k-step is permuted identically for A and B
//    (lane t owns k = 16t .. 16t+15), so every lane loads weights and tokens
//    with plain 16-byte vectors and no shuffles.
//  * Split-K without global scratch: the S CTAs of a thread-block cluster own
//    disjoint k-ranges of the same rows; the four warps of a CTA are reduced
//    in shared memory, then the cluster through distributed shared memory, in
//    a fixed rank order (deterministic; exact for the int32 W8A8 sums).
//  * Grouped: blockIdx.z walks the experts from the last one down (the
//    hardware dispatches z in increasing order), so the experts at the end
//    of the list -- the shared experts of an MoE layer, which see every
//    token and loop over the most token chunks -- start first instead of
//    forming the grid's tail (DeepSeek-MoE T = 64: gate_up 114.6 -> 89.8 us,
//    down 73.0 -> 52.0 us).  An expert without rows exits before reading any
//    weight.  Offsets are validated on the device; a bad expert is skipped
//    and reported through the sticky fault word.
// HBM traffic per launch: N*K weight bytes + 4N scale bytes (per active
// expert) + token and output bytes.

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "quant_math.cuh"

namespace cg = cooperative_groups;

namespace i8ql {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxClusterSplit = 8;

// kW8A8Q: W8A8 whose token rows arrive in bf16 and are quantized per token
// inside the kernel (the activation quantization fused into the GEMM).
enum class Op { kW8A16, kW8A8, kW8A8Q };

struct DecodeParams {
    const void* x;           // bf16 [rows, K] (W8A16) or int8 [rows, K] (W8A8)
    const float* sx;         // W8A8 per-token scales [rows]
    const int32_t* offsets;  // grouped: [E + 1]; null otherwise
    const int8_t* qw;
    const float* sw;
    const uint16_t* bias;    // W8A8 only, nullable
    uint16_t* y;
    int32_t* acc;            // W8A8 only, nullable
    int64_t rows;            // M (plain) or T_total (grouped)
    int64_t N;
    int64_t K;
    int64_t E;
    unsigned* err;
    int one_wave;            // every CTA of the grid is resident at once
    const int32_t* gather;   // grouped: token row of x for each grouped row (null: row r is x's row r)
    int8_t* qx_out;          // kW8A8Q: receives the token codes and scales when not null
    float* sx_out;
    int64_t glu;             // grouped W8A16: intermediate size I of a fused gate/up
                             // projection (N = 2I) whose SiLU-gated product is the
                             // output [rows, I]; 0: plain outputs
    int early_weights;       // (not grouped) the first ring stages of weights are
                             // loaded before the wait for the previous kernel: the
                             // caller promised that it does not write them
};

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_cached(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// Four int8 codes -> two bf16x2 words (exact).  Each byte b is biased to
// u = b + 128, placed in the low mantissa bits of 2^23 (float 2^23 + u),
// and 2^23 + 128 is subtracted with packed f32x2 adds; the upper halves of
// the exact fp32 results are the bf16 values.
__device__ __forceinline__ void i8x4_to_bf16(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t"
        ".reg .b32 u, f0, f1, f2, f3;\n\t"
        ".reg .b64 pa, pb;\n\t"
        "xor.b32 u, %2, 0x80808080;\n\t"
        "prmt.b32 f0, u, 0x4b000000, 0x7440;\n\t"
        "prmt.b32 f1, u, 0x4b000000, 0x7441;\n\t"
        "prmt.b32 f2, u, 0x4b000000, 0x7442;\n\t"
        "prmt.b32 f3, u, 0x4b000000, 0x7443;\n\t"
        "mov.b64 pa, {f0, f1};\n\t"
        "mov.b64 pb, {f2, f3};\n\t"
        "add.rn.f32x2 pa, pa, %3;\n\t"
        "add.rn.f32x2 pb, pb, %3;\n\t"
        "mov.b64 {f0, f1}, pa;\n\t"
        "mov.b64 {f2, f3}, pb;\n\t"
        "prmt.b32 %0, f0, f1, 0x7632;\n\t"
        "prmt.b32 %1, f2, f3, 0x7632;\n\t"
        "}"
        : "=r"(lo), "=r"(hi)
        : "r"(w), "l"(0xcb000080cb000080ull));  // (-(2^23 + 128), -(2^23 + 128))
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_s8(int32_t (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                       uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

template <int MT>
struct WeightRegs {
    uint4 r[MT][2];  // rows g and g+8 of each 16-row m-tile
};

// Per-configuration tuning (each choice measured on the decode shapes):
//  kStages  depth of the per-lane register ring of weight loads (while one
//           k-step is converted and multiplied, the next kStages - 1 are in
//           flight);
//  kMinCtas CTAs per SM the register budget is sized for;
//  kXAhead  the token operand (an L1/L2 hit that still queues behind the
//           weight stream) is loaded one k-step ahead.
// W8A8 streams without conversion and keeps a deep ring.  W8A16 with one
// token tile trades ring depth for the token prefetch; its grouped form
// (many short expert GEMMs) does better with more CTAs per SM instead, and
// with 16-row warps (MT = 1, small launches only) with more still.
// Wider token tiles have no registers to spare for the prefetch.
template <Op OP, int MT, int NT, bool GROUPED>
struct Tuning {
    static constexpr bool kW8A16One = OP == Op::kW8A16 && NT == 1;
    static constexpr bool kInt = OP != Op::kW8A16;  // int8 x int8 -> int32
    // (the token quantization of kW8A8Q needs the registers of one stage)
    static constexpr int kStages = OP == Op::kW8A8 ? 4 : (OP == Op::kW8A8Q ? 3 : (NT == 1 ? 2 : 3));
    static constexpr int kMinCtas =
        (kW8A16One && GROUPED) ? (MT == 1 ? 8 : 6) : (NT <= 2 ? 4 : (NT <= 4 ? 3 : 2));
    static constexpr bool kXAhead = kInt ? NT <= 2 : (kW8A16One && !GROUPED);
};

// MT 16-row m-tiles per warp, NT 8-token n-tiles per pass.
constexpr int kCompactExperts = 256;  // grouped: largest E for per-row expert slots

template <Op OP, int MT, int NT, bool GROUPED>
__global__ void __launch_bounds__(kThreads, (Tuning<OP, MT, NT, GROUPED>::kMinCtas))
    decode_gemm_kernel(const DecodeParams p) {
    using Acc = std::conditional_t<OP != Op::kW8A16, int32_t, float>;
    constexpr int kRows = 16 * MT;
    constexpr int kToks = 8 * NT;
    constexpr int kStages = Tuning<OP, MT, NT, GROUPED>::kStages;
    __shared__ Acc part[kWarps][kToks * kRows];

    // Before waiting for the previous kernel, start streaming this CTA's
    // weight rows into L2, so the DRAM ramp overlaps that kernel's tail.  This
    // is safe even if the previous kernel writes these weights: L2 is the
    // point of coherence (a line it writes later is updated in L2), and the
    // loads after pdl_wait() read through it.
    {
        const int64_t rows_n = p.N;
        const int64_t r0 = (int64_t)blockIdx.x * kRows;
        const int8_t* qw0 = p.qw + (GROUPED ? (int64_t)blockIdx.z * rows_n * p.K : 0);
        const int64_t ksteps = (p.K + 63) / 64;
        const int S0 = (int)gridDim.y;
        const int64_t kb0 = ksteps * (int64_t)blockIdx.y / S0, kb1 = ksteps * ((int64_t)blockIdx.y + 1) / S0;
        const int64_t k_lo = kb0 * 64, k_hi = min(kb1 * 64, p.K);
        const int r = (int)threadIdx.x;
        // (not for the grouped kernel: its multi-wave grid measured slower with it)
        if (!GROUPED && r < kRows && r0 + r < rows_n && k_hi > k_lo)
            prefetch_l2(qw0 + (r0 + r) * p.K + k_lo, (uint32_t)(k_hi - k_lo));
    }
    // With early weight loads the wait comes after the first ring fill (the
    // weights are not the previous kernel's output); tokens, scales and
    // offsets are read only after it.
    const bool early = !GROUPED && p.early_weights;
    if (!early) {
        pdl_wait();
        if (p.one_wave) pdl_launch_dependents();
    }
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
        int64_t e = p.E - 1 - (int64_t)blockIdx.z;  // last expert first
        if (gridDim.z < p.E) {
            // Few rows (the launch gives fewer expert slots than experts, and
            // E <= kCompactExperts): slot z takes the z-th expert with rows,
            // counted from the last.  Every warp loads all offsets at once,
            // scans them 32 experts per ballot and reaches the same answer;
            // the scan also checks every expert's offsets.
            const unsigned need = blockIdx.z;
            unsigned seen = 0;
            bool any_bad = false;
            e = -1;
            int32_t oa[kCompactExperts / 32], ob[kCompactExperts / 32];
#pragma unroll
            for (int j = 0; j < kCompactExperts / 32; ++j) {
                const int64_t ee = p.E - 1 - 32 * j - lane;
                oa[j] = ee >= 0 ? p.offsets[ee] : 0;
                ob[j] = ee >= 0 ? p.offsets[ee + 1] : 0;
            }
#pragma unroll
            for (int j = 0; j < kCompactExperts / 32; ++j) {
                const int64_t ee = p.E - 1 - 32 * j - lane;
                const int64_t a = oa[j], b = ob[j];
                const bool bad_e = ee >= 0 && (a < 0 || b < a || b > p.rows || (ee == 0 && a != 0) ||
                                                (ee == p.E - 1 && b != p.rows));
                const unsigned has = __ballot_sync(0xffffffffu, ee >= 0 && b > a);
                any_bad |= __any_sync(0xffffffffu, bad_e);
                if (e < 0 && need < seen + __popc(has))
                    e = p.E - 1 - 32 * j - (int64_t)__fns(has, 0, (int)(need - seen) + 1);
                seen += __popc(has);
            }
            if (any_bad && blockIdx.x == 0 && blockIdx.z == 0 && rank == 0 && threadIdx.x == 0)
                record_fault(p.err, kErrBitBadOffsets);
            if (e < 0) return;  // fewer experts with rows than slots (the cluster agrees)
        }
        const int64_t a = p.offsets[e], b = p.offsets[e + 1];
        const bool bad = a < 0 || b < a || b > p.rows || (e == 0 && a != 0) || (e == p.E - 1 && b != p.rows);
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

    // This warp's k-steps (64 k each) within the cluster's split of K.  All
    // k-steps are full except possibly the last of the matrix (K % 64 != 0),
    // which is handled once, with predicates, after the main loop.
    const int64_t ksteps = (K + 63) / 64;
    const int64_t full_steps = K / 64;
    const int units = S * kWarps;
    const int unit = rank * kWarps + warp;
    const int64_t ks_begin = ksteps * unit / units;
    const int64_t ks_end = ksteps * (unit + 1) / units;
    const int64_t main_end = min(ks_end, full_steps);
    const int main_count = (int)max((int64_t)0, main_end - ks_begin);
    const bool has_tail = ks_end > full_steps;  // this warp owns the partial k-step

    // Lane base pointers.  Rows past N read row N-1 and tokens past the
    // chunk read its last token: their products land only in outputs that
    // are never stored, so the main loop needs no predicates.
    // With a fused gate/up projection (p.glu = I) a CTA owns 16 output
    // columns j0 .. j0+15: m-tile 0 holds their gate rows, m-tile 1 the up
    // rows I + j0 .. (MT == 2 there).
    const int8_t* wbase[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            int64_t n;
            if (p.glu) {
                const int64_t j = min((int64_t)blockIdx.x * 16 + g + 8 * h, p.glu - 1);
                n = mt == 0 ? j : p.glu + j;
            } else {
                n = min(n0 + mt * 16 + g + 8 * h, N - 1);
            }
            wbase[mt][h] = qw + n * K + 16 * t + ks_begin * 64;
        }

    // kW8A8Q: the per-token scales s = absmax / 127 over all of K, from
    // the cluster's CTAs (each takes the absmax over its own k range; 16
    // threads per token, at most 8 tokens), before any code is formed.
    __shared__ float tok_amax[8];
    __shared__ float tok_scale[8];
    // kW8A8Q: called once the first weight loads are in flight, so that
    // this pass over the tokens overlaps their latency.
    auto quant_prologue = [&]() {
        const int64_t k_lo = ksteps * rank / S * 64, k_hi = min(ksteps * (rank + 1) / S * 64, K);
        const int tok = threadIdx.x >> 4, sub = threadIdx.x & 15;
        const uint16_t* xr = static_cast<const uint16_t*>(p.x) + min((int64_t)tok, p.rows - 1) * K;
        float a = 0.0f;
        if (tok < p.rows)
            for (int64_t k = k_lo + sub * 8; k < k_hi; k += 128) a = absmax8(ldg_cached(xr + k), a);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        if (sub == 0) tok_amax[tok] = a;
        if (S == 1)
            __syncthreads();
        else
            cluster.sync();
        if (threadIdx.x < 8) {
            float full = tok_amax[threadIdx.x];
            for (int r = 0; r < S; ++r) full = fmaxf(full, cluster.map_shared_rank(&tok_amax[0], r)[threadIdx.x]);
            const float sc = full == 0.0f ? 1.0f : __fdiv_rn(full, 127.0f);  // zero-row guard
            tok_scale[threadIdx.x] = sc;
            if (p.sx_out && blockIdx.x == 0 && rank == 0 && threadIdx.x < p.rows) p.sx_out[threadIdx.x] = sc;
        }
        __syncthreads();
        if (p.qx_out && blockIdx.x == 0 && tok < p.rows) {
            // the codes themselves, for a caller that keeps them: row block 0
            // writes each CTA's k range
            const RowScale rs = make_row_scale(tok_scale[tok]);
            for (int64_t k = k_lo + sub * 8; k < k_hi; k += 128)
                *reinterpret_cast<uint2*>(p.qx_out + tok * K + k) = codes8(ldg_cached(xr + k), rs);
        }
    };

    using XT = std::conditional_t<OP != Op::kW8A8, uint16_t, int8_t>;
    constexpr int kXW = OP == Op::kW8A16 ? 8 : 4;  // 32-bit words of x per lane per k-step

    for (int64_t c0 = lo; c0 < hi; c0 += kToks) {
        const int64_t chunk_hi = min(hi, c0 + (int64_t)kToks);
        const int nt_active = (int)((chunk_hi - c0 + 7) / 8);
        const XT* xbase[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int64_t r = min(c0 + nt * 8 + g, chunk_hi - 1);
            const int64_t src = p.gather ? (int64_t)p.gather[r] : r;  // the token feeding grouped row r
            xbase[nt] = static_cast<const XT*>(p.x) + src * K + 16 * t + ks_begin * 64;
        }

        Acc acc[MT][NT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[mt][nt][i] = Acc(0);

        // kW8A8Q: each lane's token scale (for the reciprocal-based codes),
        // set once the scales are known, before the first token load
        RowScale rsx[NT];
        auto load_x = [&](uint32_t (&xb)[NT][kXW], int i, bool ok) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if constexpr (OP == Op::kW8A8Q) {
                    if (nt < nt_active && ok) {
                        // 16 bf16 values -> 16 int8 codes, exactly as the
                        // quantization kernel forms them
                        const XT* xp = xbase[nt] + (int64_t)i * 64;
                        const uint2 c0w = codes8(ldg_cached(xp), rsx[nt]);
                        const uint2 c1w = codes8(ldg_cached(xp + 8), rsx[nt]);
                        xb[nt][0] = c0w.x; xb[nt][1] = c0w.y; xb[nt][2] = c1w.x; xb[nt][3] = c1w.y;
                    } else {
#pragma unroll
                        for (int q = 0; q < kXW; ++q) xb[nt][q] = 0u;
                    }
                } else if (nt < nt_active && ok) {
                    const XT* xp = xbase[nt] + (int64_t)i * 64;
                    const uint4 v0 = ldg_cached(xp);
                    xb[nt][0] = v0.x; xb[nt][1] = v0.y; xb[nt][2] = v0.z; xb[nt][3] = v0.w;
                    if constexpr (OP == Op::kW8A16) {
                        const uint4 v1 = ldg_cached(xp + 8);
                        xb[nt][4] = v1.x; xb[nt][5] = v1.y; xb[nt][6] = v1.z; xb[nt][7] = v1.w;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < kXW; ++q) xb[nt][q] = 0u;
                }
            }
        };
        auto mma_step = [&](const WeightRegs<MT>& w, const uint32_t (&xb)[NT][kXW]) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const uint32_t wg[4] = {w.r[mt][0].x, w.r[mt][0].y, w.r[mt][0].z, w.r[mt][0].w};
                const uint32_t wh[4] = {w.r[mt][1].x, w.r[mt][1].y, w.r[mt][1].z, w.r[mt][1].w};
                if constexpr (OP == Op::kW8A16) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t a0, a2, a1, a3;
                        i8x4_to_bf16(wg[j], a0, a2);  // row g:   k 16t+4j+{0,1} | {2,3}
                        i8x4_to_bf16(wh[j], a1, a3);  // row g+8: same k
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            if (nt < nt_active)
                                mma_bf16(acc[mt][nt], a0, a1, a2, a3, xb[nt][2 * j], xb[nt][2 * j + 1]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        // k 16t+8j+{0..3} -> fragment slot 4t.., k 16t+8j+{4..7} -> slot 16+4t..
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            if (nt < nt_active)
                                mma_s8(acc[mt][nt], wg[2 * j], wh[2 * j], wg[2 * j + 1], wh[2 * j + 1],
                                       xb[nt][2 * j], xb[nt][2 * j + 1]);
                    }
                }
            }
        };
        auto load_w = [&](WeightRegs<MT>& w, int i) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) w.r[mt][h] = ldg_stream(wbase[mt][h] + (int64_t)i * 64);
        };

        {
            // main loop: full k-steps through a kStages-deep register ring
            // of weights (the token operand one k-step ahead if kXAhead)
            constexpr bool kXAhead = Tuning<OP, MT, NT, GROUPED>::kXAhead;
            WeightRegs<MT> ring[kStages];
#pragma unroll
            for (int s = 0; s < kStages; ++s)
                if (s < main_count) load_w(ring[s], s);
            if (early && c0 == lo) {
                pdl_wait();
                if (p.one_wave) pdl_launch_dependents();
            }
            if constexpr (OP == Op::kW8A8Q) {
                // (a single token chunk: M <= 8)
                quant_prologue();
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    rsx[nt] = make_row_scale(tok_scale[min(c0 + nt * 8 + g, chunk_hi - 1) - c0]);
            }
            uint32_t xb[NT][kXW];
            if constexpr (kXAhead) load_x(xb, 0, main_count > 0);
            for (int i0 = 0; i0 < main_count; i0 += kStages) {
#pragma unroll
                for (int s = 0; s < kStages; ++s) {
                    const int i = i0 + s;
                    if (i < main_count) {
                        if constexpr (kXAhead) {
                            uint32_t xn[NT][kXW];
                            load_x(xn, i + 1, i + 1 < main_count);
                            mma_step(ring[s], xb);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int q = 0; q < kXW; ++q) xb[nt][q] = xn[nt][q];
                        } else {
                            load_x(xb, i, true);
                            mma_step(ring[s], xb);
                        }
                        if (i + kStages < main_count) load_w(ring[s], i + kStages);
                    }
                }
            }
        }
        if (has_tail) {
            // the partial last k-step of the matrix: lanes past K load zeros
            const int i = main_count;
            const bool kok = full_steps * 64 + 16 * t < K;
            WeightRegs<MT> w;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    w.r[mt][h] = kok ? ldg_stream(wbase[mt][h] + (int64_t)i * 64) : make_uint4(0, 0, 0, 0);
            uint32_t xb[NT][kXW];
            load_x(xb, i, kok);
            mma_step(w, xb);
        }

        // Warp partials -> shared memory, laid out [token][row].
        Acc* mine = part[warp];
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
        for (int i = threadIdx.x; i < kToks * kRows; i += kThreads) {
            Acc s = part[0][i];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) s += part[w][i];
            part[0][i] = s;
        }
        // Publish to the cluster, then each rank finishes a slice of the tile.
        // (A one-CTA cluster needs only a CTA barrier: the release semantics
        // of a cluster barrier would also wait for earlier global stores.)
        if (S == 1)
            __syncthreads();
        else
            cluster.sync();
        // the sum over the cluster of tile entry i, in rank order
        auto reduced = [&](int i) -> Acc {
            if (S == 1) return part[0][i];
            Acc v[kMaxClusterSplit];
#pragma unroll
            for (int r = 0; r < kMaxClusterSplit; ++r)
                v[r] = r < S ? cluster.map_shared_rank(&part[0][0], r)[i] : Acc(0);
            Acc s = v[0];
#pragma unroll
            for (int r = 1; r < kMaxClusterSplit; ++r)
                if (r < S) s += v[r];
            return s;
        };
        if (OP == Op::kW8A16 && p.glu) {
            // SiLU-gated product of the fused gate/up rows: tile rows r and
            // 16 + r hold gate and up of output column j0 + r
            const int64_t j0 = (int64_t)blockIdx.x * 16;
            const int total = nt_active * 8 * 16;
            const int per = (total + S - 1) / S;
            const int i_begin = rank * per;
            const int i_end = min(total, i_begin + per);
            for (int i = i_begin + (int)threadIdx.x; i < i_end; i += kThreads) {
                const int r = i % 16;
                const int tok = i / 16;
                const Acc gs = reduced(tok * kRows + r), us = reduced(tok * kRows + 16 + r);
                const int64_t j = j0 + r;
                const int64_t m = c0 + tok;
                if (j < p.glu && m < hi) {
                    const float gv = (float)gs * sw[j];
                    const float uv = (float)us * sw[p.glu + j];
                    p.y[m * p.glu + j] = f32_to_bf16_rn(gv / (1.0f + expf(-gv)) * uv);
                }
            }
        }
        const int total = (OP == Op::kW8A16 && p.glu) ? 0 : nt_active * 8 * kRows;
        const int per = (total + S - 1) / S;
        const int i_begin = rank * per;
        const int i_end = min(total, i_begin + per);
        for (int i = i_begin + (int)threadIdx.x; i < i_end; i += kThreads) {
            const Acc s = reduced(i);  // all peers' loads in flight before the rank-ordered sum
            const int row = i % kRows;
            const int tok = i / kRows;
            const int64_t n = n0 + row;
            const int64_t m = c0 + tok;
            if (n < N && m < hi) {
                if constexpr (OP == Op::kW8A16) {
                    p.y[m * N + n] = f32_to_bf16_rn(s * sw[n]);
                } else {
                    const float sxm = OP == Op::kW8A8Q ? tok_scale[m - c0] : p.sx[m];
                    float f = __fmul_rn(__fmul_rn(__int2float_rn(s), sxm), sw[n]);
                    if (p.bias) f = __fadd_rn(f, bf16_to_f32(p.bias[n]));
                    p.y[m * N + n] = f32_to_bf16_rn(f);
                    if (p.acc) p.acc[m * N + n] = s;
                }
            }
        }
        // Peers are done reading this CTA's shared memory (their loads have
        // returned: the values are summed).  A relaxed arrive does not wait
        // for this thread's output stores to drain.
        if (S == 1)
            __syncthreads();
        else
            asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
    }
}

// Row blocks of the grid: 16 * MT weight rows each, or 16 gated output
// columns each with a fused gate/up projection.
template <int MT>
int64_t row_blocks_of(const DecodeParams& p) {
    return p.glu ? (p.glu + 15) / 16 : (p.N + 16 * MT - 1) / (16 * MT);
}

// Expert slots of a grouped launch: one per expert, or, when at most half
// of the experts can have rows (rows <= E / 2, E <= kCompactExperts), one
// per row -- the CTAs of experts without rows then never launch (DeepSeek-
// MoE at one token: 8 slots instead of 66, gate_up 17.6 -> 15.9 us).
template <bool GROUPED>
int64_t expert_slots(const DecodeParams& p) {
    if (!GROUPED) return 1;
    if (p.E <= kCompactExperts && 2 * p.rows <= p.E) return std::max<int64_t>(1, p.rows);
    return p.E;
}

template <Op OP, int MT, int NT, bool GROUPED>
cudaError_t launch_cfg(const DecodeParams& p, int split, cudaStream_t stream) {
    const int64_t row_blocks = row_blocks_of<MT>(p);
    return launch_kernel(decode_gemm_kernel<OP, MT, NT, GROUPED>,
                         dim3((unsigned)row_blocks, (unsigned)split, (unsigned)expert_slots<GROUPED>(p)), dim3(kThreads),
                         0, stream, dim3(1, (unsigned)split, 1), p);
}

// CTAs of this configuration that fit on one SM at once (cached per device).
template <Op OP, int MT, int NT, bool GROUPED>
int resident_ctas() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 1;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_gemm_kernel<OP, MT, NT, GROUPED>, kThreads, 0) !=
                cudaSuccess || n < 1)
            n = 1;
        cached[dev] = n;
    }
    return cached[dev];
}

// Split-K factor: fill one wave of resident CTAs (no tail wave), keep at
// least two k-steps per warp, and stay within one portable cluster.
int choose_split(int64_t row_blocks, int64_t groups, int64_t K, int64_t capacity) {
    const int64_t ksteps = (K + 63) / 64;
    int64_t split = capacity / std::max<int64_t>(1, row_blocks * groups);
    split = std::min<int64_t>(split, std::max<int64_t>(1, ksteps / (2 * kWarps)));
    return (int)std::max<int64_t>(1, std::min<int64_t>(split, kMaxClusterSplit));
}

template <Op OP, int MT, int NT, bool GROUPED>
cudaError_t launch_auto(DecodeParams p, int64_t groups_hint, int sms, cudaStream_t stream) {
    const int64_t row_blocks = row_blocks_of<MT>(p);
    const int64_t capacity = (int64_t)sms * resident_ctas<OP, MT, NT, GROUPED>();
    const int split = choose_split(row_blocks, groups_hint, p.K, capacity);
    p.one_wave = row_blocks * split * expert_slots<GROUPED>(p) <= capacity ? 1 : 0;
    // Early weight loads pay off for split-K launches (short CTAs whose
    // first-load latency is a large part of their time: Qwen3-4B o 4.53 ->
    // 4.17 us, W8A8 qkv 6.11 -> 5.51 us) and not for unsplit full waves
    // (gate_up 12.48 -> 13.00 us), so they are kept to the former.
    if (split == 1) p.early_weights = 0;
    return launch_cfg<OP, MT, NT, GROUPED>(p, split, stream);
}

template <Op OP, bool GROUPED>
cudaError_t dispatch(const DecodeParams& p, int64_t tokens_hint, int64_t groups_hint, int sms, cudaStream_t stream) {
    if constexpr (GROUPED && OP == Op::kW8A16) {
        // A grouped launch small enough that its 16-row CTAs still fit in
        // one wave spreads over more SMs with them (DeepSeek-MoE down at one
        // token: 12.3 -> 10.5 us; gate_up, past one wave, stays at 32 rows).
        // The fused gate/up form pairs 16 gate and 16 up rows: 32 rows.
        if (tokens_hint <= 8 && !p.glu &&
            row_blocks_of<1>(p) * expert_slots<GROUPED>(p) <= (int64_t)sms * resident_ctas<OP, 1, 1, GROUPED>())
            return launch_auto<OP, 1, 1, GROUPED>(p, groups_hint, sms, stream);
    }
    if (tokens_hint <= 8) return launch_auto<OP, 2, 1, GROUPED>(p, groups_hint, sms, stream);
    if (tokens_hint <= 16) return launch_auto<OP, 2, 2, GROUPED>(p, groups_hint, sms, stream);
    if (tokens_hint <= 32) return launch_auto<OP, 2, 4, GROUPED>(p, groups_hint, sms, stream);
    return launch_auto<OP, 2, 8, GROUPED>(p, groups_hint, sms, stream);
}

}  // namespace

cudaError_t launch_w8a16(const uint16_t* x, const int32_t* offsets, int64_t E, const int8_t* qw, const float* sw,
                         uint16_t* y, int64_t M, int64_t N, int64_t K, const LaunchEnv& env, const int32_t* gather,
                         int64_t glu) {
    DecodeParams p{x, nullptr, offsets, qw, sw, nullptr, y, nullptr, M, N, K, E, env.err, 0, gather, nullptr, nullptr, glu};
    if (offsets == nullptr) {
        p.early_weights = early_weight_loads() ? 1 : 0;
        return dispatch<Op::kW8A16, false>(p, M, 1, env.sm_count, env.stream);
    }
    // Grouped: at most min(E, T_total) experts have rows, on average
    // T_total / active rows each.
    const int64_t active = std::min<int64_t>(E, M);
    const int64_t per_expert = (M + active - 1) / active;
    return dispatch<Op::kW8A16, true>(p, std::max<int64_t>(per_expert, 1), active, env.sm_count, env.stream);
}

bool w8a8_decode_fused_preferred(int64_t N, int64_t K, int sms) {
    DecodeParams p{};
    p.N = N;
    p.K = K;
    const int64_t capacity = (int64_t)sms * resident_ctas<Op::kW8A8Q, 2, 1, false>();
    const int64_t row_blocks = row_blocks_of<2>(p);
    return choose_split(row_blocks, 1, K, capacity) == 1 && row_blocks <= capacity;
}

cudaError_t launch_w8a8_decode_fused(const uint16_t* x, const int8_t* qw, const float* sw, const uint16_t* bias,
                                     uint16_t* y, int8_t* qx, float* sx, int32_t* acc, int64_t M, int64_t N, int64_t K,
                                     const LaunchEnv& env) {
    DecodeParams p{x, nullptr, nullptr, qw, sw, bias, y, acc, M, N, K, 1, env.err, 0, nullptr, qx, sx, 0};
    p.early_weights = early_weight_loads() ? 1 : 0;
    return launch_auto<Op::kW8A8Q, 2, 1, false>(p, 1, env.sm_count, env.stream);
}

cudaError_t launch_w8a8_decode(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw,
                               const uint16_t* bias, uint16_t* y, int32_t* acc, int64_t M, int64_t N, int64_t K,
                               const LaunchEnv& env) {
    DecodeParams p{qx, sx, nullptr, qw, sw, bias, y, acc, M, N, K, 1, env.err, 0, nullptr, nullptr, nullptr, 0};
    p.early_weights = early_weight_loads() ? 1 : 0;
    return dispatch<Op::kW8A8, false>(p, M, 1, env.sm_count, env.stream);
}

}  // namespace i8ql
