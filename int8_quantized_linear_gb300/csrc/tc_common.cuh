// Device helpers of the tcgen05 W8A8 kernels (sm_103a): mbarriers with
// bounded waits, TMA tile loads, tcgen05 MMA / commit / TMEM loads, shared-
// memory matrix descriptors, exact int8 -> fp16 code conversion, the W8A8
// scale/bias epilogue, and cluster (DSMEM) helpers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace i8ql {
namespace tc {

constexpr int kBM = 128;      // rows of the MMA A operand per CTA (TMEM lanes)
constexpr int kBK = 64;       // k per pipeline stage: one 128-byte fp16 swizzle atom row
constexpr int kChunkKB = 16;  // k-blocks per exact fp32 chunk (1024 k)
constexpr int kGroupA = 8;    // tile rows of A swept together (L2 reuse of B tiles)
constexpr int kMaxSplit = 8;  // split-K CTAs per cluster (portable cluster size)

// Problem and tile description shared by both W8A8 tensor-core kernels.
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
    int swap;   // A holds the weights and B the tokens (M <= 128)
    int split;  // CTAs of a cluster sharing one tile's k range (1: persistent, no split)
    uint32_t tmem_cols;
    unsigned* err;
    // Stream-K (CTA pairs only): sk_units pairs share the tiles * nkb
    // k-block iterations evenly; a pair whose range ends inside a tile parks
    // that partial tile (int32, this CTA's 128 rows) in its slot of sk_part
    // and counts it done in sk_flags (zeroed before the launch); the pair
    // holding the tile's last k-block adds the parked partials of the
    // earlier pairs.
    int sk;
    int64_t sk_units;
    int32_t* sk_part;   // [sk_units][2][128 * bn] int32
    unsigned* sk_flags; // [sk_units][2]
    unsigned sk_flag_target;  // flag value of a parked part (one count per epilogue thread)
    uint64_t sk_wait_ns;      // limit of a finisher's wait for one parked part
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

// Non-blocking test of the phase with the given parity (cheap when it has
// already completed, the common case of a well-fed pipeline).
__device__ __forceinline__ bool mbar_test(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
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
// if the CTA is aborting (*abort set) or the wall-clock limit expired (which
// sets *abort and records the fault).  Inlined into kernels that rebalance
// registers with setmaxnreg (a call inside such a region defeats the
// register allocator); the out-of-line copy keeps other kernels small.
__device__ __forceinline__ bool mbar_wait_inline(uint64_t* bar, uint32_t parity, int* abort, unsigned* err) {
    const uint32_t addr = smem_u32(bar);
    if (mbar_test(addr, parity)) return true;
    uint64_t t0 = 0;
    bool started = false;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try(addr, parity)) return true;
        if ((it & 63u) == 63u) {
            if (*reinterpret_cast<volatile int*>(abort)) return false;
            const uint64_t now = global_ns();
            if (!started) {
                t0 = now;
                started = true;
            } else if (now - t0 > kWaitLimitNs) {
                record_fault(err, kErrBitTimeout);
                *reinterpret_cast<volatile int*>(abort) = 1;
                return false;
            }
        }
    }
}

static __device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* abort, unsigned* err) {
    return mbar_wait_inline(bar, parity, abort, err);
}

// Every lane of a warp waits (each gets the barrier's acquire), then the
// warp agrees: if any lane gave up, all of them take the abort path, so the
// warp stays converged for .sync.aligned instructions.
template <bool kInline = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* abort, unsigned* err) {
    const bool ok = kInline ? mbar_wait_inline(bar, parity, abort, err) : mbar_wait(bar, parity, abort, err);
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

// Instruction descriptor of kind::f16: fp16 A and B, fp32 D, both K-major,
// M = 128, N = bn.
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

// Arrives on `bar` once every MMA this thread issued before has completed.
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

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t tmem, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols) : "memory");
}

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

// 2-D TMA tile load into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (the tensor core reading them as MMA operands).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// cuTensorMapEncodeTiled from the driver (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ int4 ld_dsmem_v4(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    int4 v;
    asm volatile("ld.shared::cluster.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}

// ---------------------------------------------------------------- CTA pairs
// A pair is a cluster of two CTAs (rank 0 leads) sharing one MMA of M = 256:
// each CTA holds 128 rows of A and half of the N rows of B in its shared
// memory, and receives its 128 rows of D in its own TMEM.

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    return remote;
}

// Arrive on an mbarrier given by its cluster address (either CTA of the
// pair).  Default semantics (release at CTA scope), as for a local arrive:
// the data a remote arrive announces reaches the tensor core through the
// async proxy (TMA, or generic stores followed by a proxy fence), whose
// visibility the MMA's barrier wait covers.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx_cluster(uint32_t cluster_addr, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_addr), "r"(bytes)
                 : "memory");
}

// 2-D TMA tile load into this CTA's shared memory that completes on an
// mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t bar_cluster_addr) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster_addr)
        : "memory");
}

// Instruction descriptor of kind::f16 for the pair MMA: M = 256, N = bn.
__device__ __forceinline__ uint32_t f16_idesc_pair(int bn) {
    return (1u << 4) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)((2 * kBM) >> 4) << 24);
}

__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on the mbarrier at the same offset in both CTAs of the pair once
// every pair MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)0x3)
        : "memory");
}

// TMEM allocation and release for a pair: one warp of each CTA executes them.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t tmem, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols) : "memory");
}

// ---------------------------------------------------------------- epilogue

// Scale/bias epilogue of W consecutive tile columns (c .. c+W-1, W = 4 or 8,
// c a multiple of W) of tile row `row`, from exact int32 sums:
//   y = bf16_rne(((float)acc * sx[m]) * sw[n] (+ bias[n]))
// Non-swapped tiles have tokens on the rows and output channels on the
// columns; swapped tiles the reverse.
template <int W>
__device__ __forceinline__ void epilogue_cols(const W8A8Params& p, int64_t ta, int64_t tb, int bn, int row, int c,
                                              const int32_t* v) {
    if (!p.swap) {
        const int64_t m = ta * kBM + row;
        const int64_t n0 = tb * bn + c;
        if (m >= p.M) return;
        const float sxm = p.sx[m];
        if (n0 + W <= p.N && (p.N % W) == 0) {
            uint32_t packed[W / 2];
#pragma unroll
            for (int j = 0; j < W; j += 2) {
                float f0 = __fmul_rn(__fmul_rn(__int2float_rn(v[j]), sxm), __ldg(p.sw + n0 + j));
                float f1 = __fmul_rn(__fmul_rn(__int2float_rn(v[j + 1]), sxm), __ldg(p.sw + n0 + j + 1));
                if (p.bias) {
                    f0 = __fadd_rn(f0, bf16_to_f32(__ldg(p.bias + n0 + j)));
                    f1 = __fadd_rn(f1, bf16_to_f32(__ldg(p.bias + n0 + j + 1)));
                }
                packed[j / 2] = (uint32_t)f32_to_bf16_rn(f0) | ((uint32_t)f32_to_bf16_rn(f1) << 16);
            }
            if constexpr (W == 8)
                *reinterpret_cast<uint4*>(p.y + m * p.N + n0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            else
                *reinterpret_cast<uint2*>(p.y + m * p.N + n0) = make_uint2(packed[0], packed[1]);
            if (p.acc) {
#pragma unroll
                for (int q = 0; q < W; q += 4)
                    *reinterpret_cast<int4*>(p.acc + m * p.N + n0 + q) = make_int4(v[q], v[q + 1], v[q + 2], v[q + 3]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) {
                const int64_t n = n0 + j;
                if (n < p.N) {
                    float f = __fmul_rn(__fmul_rn(__int2float_rn(v[j]), sxm), __ldg(p.sw + n));
                    if (p.bias) f = __fadd_rn(f, bf16_to_f32(__ldg(p.bias + n)));
                    p.y[m * p.N + n] = f32_to_bf16_rn(f);
                    if (p.acc) p.acc[m * p.N + n] = v[j];
                }
            }
        }
    } else {
        const int64_t n = ta * kBM + row;
        if (n >= p.N) return;
        const float swn = p.sw[n];
        const float bias_n = p.bias ? bf16_to_f32(p.bias[n]) : 0.0f;
#pragma unroll
        for (int j = 0; j < W; ++j) {
            const int64_t m = tb * bn + c + j;
            if (m < p.M) {
                float f = __fmul_rn(__fmul_rn(__int2float_rn(v[j]), __ldg(p.sx + m)), swn);
                if (p.bias) f = __fadd_rn(f, bias_n);
                p.y[m * p.N + n] = f32_to_bf16_rn(f);
                if (p.acc) p.acc[m * p.N + n] = v[j];
            }
        }
    }
}

// Grouped raster: consecutive tiles sweep kGroupA tile rows of A for each
// tile column of B, so CTAs running together share A row blocks and B tiles
// in L2.
__device__ __forceinline__ void tile_coords(const W8A8Params& p, int64_t tile, int64_t& ta, int64_t& tb) {
    const int64_t group_tiles = (int64_t)kGroupA * p.tiles_b;
    const int64_t first_a = (tile / group_tiles) * kGroupA;
    const int64_t rows_in_group = min((int64_t)kGroupA, p.tiles_a - first_a);
    const int64_t local = tile % group_tiles;
    ta = first_a + local % rows_in_group;
    tb = local / rows_in_group;
}

}  // namespace tc
}  // namespace i8ql
