// W8A8 GEMM for M > 64: int8 x int8 -> exact int32 -> scale/bias epilogue -> bf16.
//
// Sources: "feat(quantization): support compressed-tensors W8A8 and mixed
// modules", Design and Supported Execution Scheme (static symmetric int8
// per-channel weights, dynamic symmetric int8 per-token activations, no
// output quantization) and "Day 6 -- Quantize It Yourself", The mechanism,
// block 5 (W8A8: both operands 8-bit, the GEMM on the tensor cores).
//
//   acc[m,n] = sum_k qx[m,k] * qw[n,k]          (exact int32)
//   y[m,n]   = bf16_rne(((float)acc * sx[m]) * sw[n] (+ bias[n]))
//
// sm_103a has no integer kind of tcgen05.mma, so the product runs on the
// fifth-generation tensor cores as kind::f16 with exact arithmetic:
//  * every int8 code is exactly representable in fp16, and every product of
//    two codes (|p| <= 16129) is exact in the fp32 accumulator;
//  * the fp32 accumulator in tensor memory (TMEM) stays exact while its
//    magnitude is below 2^24, which holds for any 1024-deep chunk of k
//    (1024 * 127^2 = 16,516,096 < 16,777,216);
//  * after each chunk the epilogue warps drain the fp32 chunk sum from TMEM,
//    convert it to int32 (exact) and add it to int32 running sums held in
//    their registers; chunks alternate between two TMEM buffers, so the next
//    chunk accumulates while the previous one drains.
//
// Two launches per call:
//  1. i8_to_f16_kernel turns both code matrices into fp16 codes (exact) in a
//     workspace, one HBM pass.  Converting once per call instead of once per
//     output tile cuts the conversion work from M*N*K*3/256 to (M+N)*K
//     elements, and lets the GEMM stream operands with TMA.
//  2. w8a8_tc_kernel: persistent, one CTA per SM, 320 threads.  Warp 9
//     issues TMA tile loads (cp.async.bulk.tensor, 128-byte swizzle, ragged
//     edges zero-filled by the tensor map) into a 4-stage ring, running ahead
//     across tiles; warp 8 allocates TMEM and issues
//     tcgen05.mma.cta_group::1.kind::f16 (M = 128, N = 256; for M <= 128,
//     "swap AB": weights fill the 128-row operand and tokens the N side,
//     padded to 128); warps 0-7 drain the chunk buffers into register
//     running sums and write the epilogue of a tile while the MMA works on
//     the next.  Tiles are rasterized in groups of 8 A row-blocks for L2
//     reuse.
//
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the CTA
// records I8QL_ERR_TIMEOUT in the sticky fault word, all roles leave their
// loops, the MMA issuer waits (bounded) for its outstanding MMAs, and the
// TMEM is freed before the CTA exits.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace i8ql {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;  // fp16 per stage row: one 128-byte swizzle atom
constexpr int kStages = 4;
constexpr int kMaxBN = 256;
constexpr int kChunkKB = 16;  // k-blocks per exact fp32 chunk (1024 k)
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each owning half of the columns
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kThreads = 10 * 32;  // 320 threads; SMSPs 0 and 1 host three warps: <= 168 registers
constexpr int kGroupA = 8;  // tile rows of A swept together (L2 reuse of B tiles)
constexpr int kAStageBytes = kBM * kBK * 2;
constexpr int kBStageBytes = kMaxBN * kBK * 2;
constexpr int kSmemBytes = kStages * (kAStageBytes + kBStageBytes) + 1024 /*align*/ + 256 /*barriers*/;

struct W8A8Params {
    int64_t rows_a, rows_b, K;
    const float* sx;
    const float* sw;
    const uint16_t* bias;
    uint16_t* y;
    int32_t* acc;
    int64_t M, N;
    int64_t tiles_a;
    int64_t tiles_b;
    int bn;
    int swap;
    uint32_t tmem_cols;
    unsigned* err;
};

struct SmemCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[2];   // fp32 chunk accumulator buffers in TMEM
    uint64_t acc_empty[2];
    uint64_t drained;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `bar` with the given parity.  Returns false
// if the CTA is aborting or the wall-clock limit expired (which starts the
// abort and records the fault).
__device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, SmemCtl* ctl, unsigned* err) {
    const uint32_t addr = smem_u32(bar);
    uint64_t t0 = 0;
    bool started = false;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try(addr, parity)) return true;
        if ((it & 63u) == 63u) {
            if (*reinterpret_cast<volatile int*>(&ctl->abort_flag)) return false;
            const uint64_t now = global_ns();
            if (!started) {
                t0 = now;
                started = true;
            } else if (now - t0 > kWaitLimitNs) {
                record_fault(err, kErrBitTimeout);
                *reinterpret_cast<volatile int*>(&ctl->abort_flag) = 1;
                return false;
            }
        }
    }
}

// Every lane of a warp waits (each gets the barrier's acquire), then the
// warp agrees: if any lane gave up, all of them take the abort path, so the
// warp stays converged for the .sync.aligned tcgen05 instructions.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, SmemCtl* ctl, unsigned* err) {
    const bool ok = mbar_wait(bar, parity, ctl, err);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3ffffu) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset
    d |= (uint64_t)1 << 46;            // version
    d |= (uint64_t)2 << 61;            // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: fp16 A and B, fp32 D, both K-major.
__device__ __forceinline__ uint32_t f16_idesc(int bn) {
    return (1u << 4) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Four int8 codes -> two fp16x2 words (exact): the biased byte u = q + 128
// becomes the low mantissa byte of fp16 1024 (value 1024 + u); subtracting
// 1152 leaves q.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    lo = __byte_perm(u, 0x64646464u, 0x5150);
    hi = __byte_perm(u, 0x64646464u, 0x5352);
    asm("sub.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
    asm("sub.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }


__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// int8 codes -> fp16 codes, both matrices in one grid-stride pass (exact).
__global__ void __launch_bounds__(256) i8_to_f16_kernel(const int8_t* __restrict__ a, int64_t a_vec,
                                                        const int8_t* __restrict__ b, int64_t b_vec,
                                                        uint16_t* __restrict__ out_a, uint16_t* __restrict__ out_b) {
    pdl_wait();
    const int64_t total = a_vec + b_vec;  // 16-byte vectors of int8
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const bool in_a = i < a_vec;
        const int64_t j = in_a ? i : i - a_vec;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(in_a ? a : b) + j);
        uint32_t h[8];
        i8x4_to_f16(v.x, h[0], h[1]);
        i8x4_to_f16(v.y, h[2], h[3]);
        i8x4_to_f16(v.z, h[4], h[5]);
        i8x4_to_f16(v.w, h[6], h[7]);
        uint4* o = reinterpret_cast<uint4*>(in_a ? out_a : out_b) + 2 * j;
        o[0] = make_uint4(h[0], h[1], h[2], h[3]);
        o[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
}

// Persistent: CTA b handles tiles b, b + grid, ...  The fp32 chunk sums
// alternate between two TMEM buffers, and the exact int32 running sums live
// in the registers of the 8 epilogue warps (warp w owns TMEM lane quarter
// w % 4 and column half w / 4), so the MMA never waits for a drain and the
// epilogue of one tile overlaps the main loop of the next.
template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    w8a8_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const W8A8Params p) {
    constexpr int kHalf = BN / 2;     // columns per epilogue warp
    constexpr int kGroups = kHalf / 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* a_stages = smem;
    uint8_t* b_stages = smem + kStages * kAStageBytes;
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(b_stages + kStages * kBStageBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t K = p.K;
    const int nkb = (int)((K + kBK - 1) / kBK);
    const int nchunks = (nkb + kChunkKB - 1) / kChunkKB;
    const int64_t tiles = p.tiles_a * p.tiles_b;
    const uint32_t stage_tx = (uint32_t)(kAStageBytes + BN * kBK * 2);

    // Grouped raster: consecutive tiles sweep kGroupA tile rows of A for each
    // tile column of B, so CTAs running together share A row blocks and B
    // tiles in L2.
    auto coords = [&](int64_t tile, int64_t& ta, int64_t& tb) {
        const int64_t group_tiles = (int64_t)kGroupA * p.tiles_b;
        const int64_t first_a = (tile / group_tiles) * kGroupA;
        const int64_t rows_in_group = min((int64_t)kGroupA, p.tiles_a - first_a);
        const int64_t local = tile % group_tiles;
        ta = first_a + local % rows_in_group;
        tb = local / rows_in_group;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->acc_full[b], 1);
            mbar_init(&ctl->acc_empty[b], kEpiWarps);
        }
        mbar_init(&ctl->drained, 1);
        ctl->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTmaWarp && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&ctl->tmem_base)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();  // the fp16 codes come from the conversion launch
    const uint32_t tmem = ctl->tmem_base;

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t a_base = smem_u32(a_stages);
            const uint32_t b_base = smem_u32(b_stages);
            int64_t kg = 0;  // k-blocks issued by this CTA
            bool alive = true;
            for (int64_t tile = blockIdx.x; tile < tiles && alive; tile += gridDim.x) {
                int64_t ta, tb;
                coords(tile, ta, tb);
                for (int kb = 0; kb < nkb; ++kb, ++kg) {
                    const int st = (int)(kg % kStages);
                    if (!mbar_wait(&ctl->empty[st], (uint32_t)(((kg / kStages) & 1) ^ 1), ctl, p.err)) {
                        alive = false;
                        break;
                    }
                    mbar_expect_tx(&ctl->full[st], stage_tx);
                    tma_load_2d(a_base + st * kAStageBytes, &map_a, kb * kBK, (int32_t)(ta * kBM), &ctl->full[st]);
                    tma_load_2d(b_base + st * kBStageBytes, &map_b, kb * kBK, (int32_t)(tb * BN), &ctl->full[st]);
                }
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = f16_idesc(BN);
            const uint32_t a_base = smem_u32(a_stages);
            const uint32_t b_base = smem_u32(b_stages);
            int64_t kg = 0;  // k-blocks consumed
            int64_t cg = 0;  // chunks accumulated
            bool alive = true;
            for (int64_t tile = blockIdx.x; tile < tiles && alive; tile += gridDim.x) {
                for (int c = 0; c < nchunks && alive; ++c, ++cg) {
                    const int b = (int)(cg & 1);
                    // the epilogue must have drained this buffer's previous chunk
                    if (!mbar_wait(&ctl->acc_empty[b], (uint32_t)(((cg >> 1) & 1) ^ 1), ctl, p.err)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(b * BN);
                    const int kb_end = min(nkb, (c + 1) * kChunkKB);
                    for (int kb = c * kChunkKB; kb < kb_end; ++kb, ++kg) {
                        const int st = (int)(kg % kStages);
                        if (!mbar_wait(&ctl->full[st], (uint32_t)((kg / kStages) & 1), ctl, p.err)) {
                            alive = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            const uint64_t ad = sw128_desc(a_base + st * kAStageBytes + kk * 32);
                            const uint64_t bd = sw128_desc(b_base + st * kBStageBytes + kk * 32);
                            mma_f16(d, ad, bd, idesc, (kb != c * kChunkKB || kk != 0) ? 1u : 0u);
                        }
                        mma_commit(&ctl->empty[st]);
                    }
                    if (alive) mma_commit(&ctl->acc_full[b]);
                }
            }
            // Wait (bounded) until every MMA issued above has completed.
            mma_commit(&ctl->drained);
            const uint64_t t0 = global_ns();
            while (!mbar_try(smem_u32(&ctl->drained), 0)) {
                if (global_ns() - t0 > kWaitLimitNs) {
                    record_fault(p.err, kErrBitTimeout);
                    ctl->abort_flag = 1;
                    break;
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int half = warp >> 2;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        int32_t run[kHalf];
        int64_t cg = 0;
        bool alive = true;
        for (int64_t tile = blockIdx.x; tile < tiles && alive; tile += gridDim.x) {
            int64_t ta, tb;
            coords(tile, ta, tb);
            for (int c = 0; c < nchunks; ++c, ++cg) {
                const int b = (int)(cg & 1);
                if (!warp_wait(&ctl->acc_full[b], (uint32_t)((cg >> 1) & 1), ctl, p.err)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col0 = (uint32_t)(b * BN + half * kHalf);
#pragma unroll
                for (int grp = 0; grp < 2 * kGroups; ++grp) {
                    uint32_t r[8];
                    tmem_ld8(lane_base + col0 + grp * 8, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int32_t v = __float2int_rn(__uint_as_float(r[j]));  // exact: |v| < 2^24
                        run[grp * 8 + j] = (c == 0) ? v : run[grp * 8 + j] + v;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->acc_empty[b]);  // the MMA may refill this buffer
            }
            if (!alive) break;
            // Scale/bias epilogue and stores from the registers, while the MMA
            // already runs the next tile.
            const int64_t arow = ta * kBM + quarter * 32 + lane;
            const int64_t bcol = tb * BN + half * kHalf;
            if (!p.swap) {
                const int64_t m = arow;
                if (m < p.M) {
                    const float sxm = p.sx[m];
#pragma unroll
                    for (int grp = 0; grp < kGroups; ++grp) {
                        const int64_t n0 = bcol + grp * 16;
                        if (n0 + 16 <= p.N && (p.N & 7) == 0) {
#pragma unroll
                            for (int h8 = 0; h8 < 2; ++h8) {
                                uint32_t packed[4];
#pragma unroll
                                for (int j = 0; j < 8; j += 2) {
                                    const int64_t n = n0 + h8 * 8 + j;
                                    const int i = grp * 16 + h8 * 8 + j;
                                    float f0 = __fmul_rn(__fmul_rn(__int2float_rn(run[i]), sxm), __ldg(p.sw + n));
                                    float f1 = __fmul_rn(__fmul_rn(__int2float_rn(run[i + 1]), sxm), __ldg(p.sw + n + 1));
                                    if (p.bias) {
                                        f0 = __fadd_rn(f0, bf16_to_f32(__ldg(p.bias + n)));
                                        f1 = __fadd_rn(f1, bf16_to_f32(__ldg(p.bias + n + 1)));
                                    }
                                    packed[j / 2] = (uint32_t)f32_to_bf16_rn(f0) | ((uint32_t)f32_to_bf16_rn(f1) << 16);
                                }
                                *reinterpret_cast<uint4*>(p.y + m * p.N + n0 + h8 * 8) =
                                    make_uint4(packed[0], packed[1], packed[2], packed[3]);
                            }
                            if (p.acc) {
                                int4* ap = reinterpret_cast<int4*>(p.acc + m * p.N + n0);
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    ap[q] = make_int4(run[grp * 16 + 4 * q], run[grp * 16 + 4 * q + 1],
                                                      run[grp * 16 + 4 * q + 2], run[grp * 16 + 4 * q + 3]);
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int64_t n = n0 + j;
                                if (n < p.N) {
                                    float f = __fmul_rn(__fmul_rn(__int2float_rn(run[grp * 16 + j]), sxm), __ldg(p.sw + n));
                                    if (p.bias) f = __fadd_rn(f, bf16_to_f32(__ldg(p.bias + n)));
                                    p.y[m * p.N + n] = f32_to_bf16_rn(f);
                                    if (p.acc) p.acc[m * p.N + n] = run[grp * 16 + j];
                                }
                            }
                        }
                    }
                }
            } else {
                const int64_t n = arow;
                if (n < p.N) {
                    const float swn = p.sw[n];
                    const float bias_n = p.bias ? bf16_to_f32(p.bias[n]) : 0.0f;
#pragma unroll
                    for (int grp = 0; grp < kGroups; ++grp) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int64_t m = bcol + grp * 16 + j;
                            if (m < p.M) {
                                float f = __fmul_rn(__fmul_rn(__int2float_rn(run[grp * 16 + j]), __ldg(p.sx + m)), swn);
                                if (p.bias) f = __fadd_rn(f, bias_n);
                                p.y[m * p.N + n] = f32_to_bf16_rn(f);
                                if (p.acc) p.acc[m * p.N + n] = run[grp * 16 + j];
                            }
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols)
                     : "memory");
    }
}

uint32_t pow2_cols(int need) {
    uint32_t c = 32;
    while ((int)c < need) c <<= 1;
    return c;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        cudaGetLastError();
    });
    return fn;
}

// 2-D fp16 tensor map over a row-major [rows, K] matrix, box = 64 k x box_rows
// rows, 128-byte swizzle (the K-major canonical layout the MMA reads),
// out-of-range elements read as zero.
bool make_map(CUtensorMap* map, const uint16_t* base, int64_t rows, int64_t K, int box_rows) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t w8a8_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= kW8A8DecodeMaxM) return 0;
    return (size_t)(M + N) * (size_t)K * 2;
}

cudaError_t launch_w8a8_ws(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw,
                           const uint16_t* bias, uint16_t* y, int32_t* acc, int64_t M, int64_t N, int64_t K,
                           uint16_t* ws, const LaunchEnv& env) {
    if (M <= kW8A8DecodeMaxM) return launch_w8a8_decode(qx, sx, qw, sw, bias, y, acc, M, N, K, env);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(w8a8_tc_kernel<kMaxBN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(w8a8_tc_kernel<kBM>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    uint16_t* x16 = ws;
    uint16_t* w16 = ws + M * K;
    // 1. fp16 codes of both operands
    {
        const int64_t vec = (M + N) * K / 16;
        const int64_t blocks = std::min<int64_t>((vec + 255) / 256, (int64_t)env.sm_count * 8);
        e = launch_kernel(i8_to_f16_kernel, dim3((unsigned)blocks), dim3(256), 0, env.stream, 0, qx, M * K / 16, qw,
                          N * K / 16, x16, w16);
        if (e != cudaSuccess) return e;
    }
    // 2. the tensor-core GEMM
    W8A8Params p{};
    p.K = K;
    p.sx = sx;
    p.sw = sw;
    p.bias = bias;
    p.y = y;
    p.acc = acc;
    p.M = M;
    p.N = N;
    p.err = env.err;
    const uint16_t* a16;
    const uint16_t* b16;
    if (M <= kBM) {
        // swap AB: weights fill the 128-row MMA operand, tokens the N side
        // (padded to 128 columns; the tensor map reads zeros past M)
        p.swap = 1;
        a16 = w16;
        p.rows_a = N;
        b16 = x16;
        p.rows_b = M;
        p.bn = kBM;
        p.tiles_b = 1;
        p.tiles_a = (N + kBM - 1) / kBM;
    } else {
        p.swap = 0;
        a16 = x16;
        p.rows_a = M;
        b16 = w16;
        p.rows_b = N;
        p.bn = kMaxBN;
        p.tiles_b = (N + kMaxBN - 1) / kMaxBN;
        p.tiles_a = (M + kBM - 1) / kBM;
    }
    p.tmem_cols = pow2_cols(2 * p.bn);  // two fp32 chunk buffers
    CUtensorMap map_a, map_b;
    if (!make_map(&map_a, a16, p.rows_a, K, kBM) || !make_map(&map_b, b16, p.rows_b, K, p.bn))
        return cudaErrorInvalidValue;
    const int64_t tiles = p.tiles_a * p.tiles_b;
    const int64_t grid = std::min<int64_t>(tiles, env.sm_count);  // persistent: one CTA per SM
    if (p.swap)
        return launch_kernel(w8a8_tc_kernel<kBM>, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, env.stream, 0,
                             map_a, map_b, p);
    return launch_kernel(w8a8_tc_kernel<kMaxBN>, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, env.stream, 0,
                         map_a, map_b, p);
}

cudaError_t launch_w8a8(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw, const uint16_t* bias,
                        uint16_t* y, int32_t* acc, int64_t M, int64_t N, int64_t K, const LaunchEnv& env) {
    if (M <= kW8A8DecodeMaxM) return launch_w8a8_decode(qx, sx, qw, sw, bias, y, acc, M, N, K, env);
    // Stream-ordered workspace for the fp16 codes (from the device's default
    // memory pool, returned when the stream reaches the free).
    void* ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, w8a8_workspace_bytes(M, N, K), env.stream);
    if (e != cudaSuccess) return e;
    e = launch_w8a8_ws(qx, sx, qw, sw, bias, y, acc, M, N, K, static_cast<uint16_t*>(ws), env);
    const cudaError_t f = cudaFreeAsync(ws, env.stream);
    return e != cudaSuccess ? e : f;
}

}  // namespace i8ql
