// FP8 E4M3 W8A8 GEMM on the tensor cores (tcgen05.mma kind::f8f6f4).
//
// Sources: "Day 6 -- Quantize It Yourself", The mechanism, block 2 (the E4M3
// grid: sign, 4 exponent and 3 mantissa bits, largest value 448) and block 5
// (W8A8 with fp8 operands: activations quantized per token on the fly, the
// GEMM on 8-bit tensor cores, which also makes the compute ~2x faster), with
// the page's FP8_DYNAMIC recipe (per-channel weights, dynamic per-token
// activations).
//
//   acc[m,n] = sum_k dec(qx[m,k]) * dec(qw[n,k])          (fp32, in TMEM)
//   y[m,n]   = bf16_rne((acc[m,n] * sx[m]) * sw[n] (+ bias[n]))
//
// sm_103a multiplies E4M3 operands natively, so unlike the int8 path there is
// no conversion stage and no chunked exact accumulation: TMA lands 128-row
// token tiles and BN-row weight tiles (128 k per stage, one 128-byte swizzle
// row per tile row) straight in the K-major layout the MMA reads, and the
// fp32 accumulator stays in tensor memory for the whole k range.
//
// Warp roles (320 threads, one CTA per SM, persistent over output tiles in a
// grouped raster for L2 reuse):
//   warp 8: TMA producer (both operands of a stage complete on one barrier);
//   warp 9: TMEM allocation and the MMA issuer (one thread): four
//     tcgen05.mma.kind::f8f6f4 of K = 32 per stage, M = 128, N = BN, then
//     one commit that frees the stage;
//   warps 0-7: epilogue, two per TMEM lane quarter (one per column half):
//     TMEM -> fp32 -> scales and bias -> bf16, staged per warp in 32 x 32
//     boxes of shared memory and written by TMA tensor stores, from one of
//     two accumulator buffers while the MMA fills the other with the next
//     tile.  (Direct per-thread stores, each warp instruction touching 32
//     output rows, held the whole kernel at half its main-loop rate.)
// For M > 128 two CTAs on two SMs form a pair (cluster of 2) and share one
// cta_group::2 MMA of M = 256: each loads its 128 token rows and half of the
// BN weight rows, so each SM pulls a quarter less from L2 per k-block; the
// copies of both complete on the leader's barrier, the leader issues the
// MMAs and its commits reach both CTAs.
// With few tiles (small M or N) single CTAs split K instead: a cluster of S
// CTAs shares one tile, CTA r running k-blocks [nkb*r/S, nkb*(r+1)/S); each
// parks its fp32 partial tile in its idle stage memory, and after a cluster
// barrier CTA r reduces rows [128r/S, 128(r+1)/S) over all partials through
// distributed shared memory, in rank order, and writes them.
// Every mbarrier wait is bounded (1 s); on expiry the CTA records
// I8QL_ERR_TIMEOUT, all roles leave, the MMA issuer waits (bounded) for its
// MMAs, a 50 us pause lets bulk copies in flight land, and TMEM is freed.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tc_common.cuh"

namespace i8ql {
namespace {

using namespace tc;

constexpr int kF8BK = 128;  // k per stage: one 128-byte swizzle row of E4M3 codes
constexpr int kF8EpiWarps = 8;
constexpr int kF8LoadWarp = 8;
constexpr int kF8MmaWarp = 9;
constexpr int kF8Threads = 10 * 32;
constexpr int kF8SmemOptin = 232448;  // largest dynamic shared memory of one CTA (227 KiB)
constexpr int kF8MaxStages = 8;
constexpr int kF8CtlBytes = 1024;
constexpr uint64_t kF8AbortDrainNs = 50000;

struct Fp8Params {
    const float* sx;
    const float* sw;
    const uint16_t* bias;
    uint16_t* y;
    int64_t M, N, K;
    int64_t tiles_a, tiles_b;  // token tiles (128 or 256 rows) x BN-wide weight tiles
    uint32_t tmem_cols;
    int tma_store;             // outputs leave through TMA tensor stores (N % 8 == 0)
    int split;                 // split-K CTAs per tile (a cluster; single CTAs only)
    unsigned* err;
};

// Output staging: per epilogue warp two buffers of 32 rows x 32 bf16 (64
// bytes a row, 64-byte swizzle: the 16-byte chunk c of row r sits at chunk
// c ^ ((r >> 1) & 3), so a warp's 16-byte stores to 32 rows hit every bank
// once per 8 rows), each written out by one TMA tensor store.
constexpr int kF8OutBuf = 32 * 64;
constexpr int kF8OutBytes = kF8EpiWarps * 2 * kF8OutBuf;

struct F8Ctl {
    uint64_t full[kF8MaxStages];   // both operands of a stage landed
    uint64_t empty[kF8MaxStages];  // the MMA is done with a stage
    uint64_t acc_full[2];          // an accumulator buffer holds a finished tile
    uint64_t acc_empty[2];         // the epilogue drained an accumulator buffer
    uint64_t drained;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(F8Ctl) <= kF8CtlBytes, "control block");

// A pair (PAIR) is a cluster of two CTAs on two SMs sharing one MMA of
// M = 256: each holds 128 token rows and half of the BN weight rows of a
// stage, and receives its 128 rows of D in its own TMEM.
template <int BN, bool PAIR>
struct F8Cfg {
    static constexpr int kWRows = PAIR ? BN / 2 : BN;
    static constexpr int kTileM = PAIR ? 2 * kBM : kBM;  // token rows of a tile
    static constexpr int kAStage = kBM * kF8BK;      // tokens: 128 rows x 128 bytes
    static constexpr int kBStage = kWRows * kF8BK;   // weights: this CTA's rows x 128 bytes
    static constexpr int kStage = kAStage + kBStage;
    static constexpr int kFit = (kF8SmemOptin - 1024 - kF8CtlBytes - kF8OutBytes) / kStage;
    static constexpr int kStages = kFit < kF8MaxStages ? kFit : kF8MaxStages;
    static constexpr int kOutOff = kStages * kStage;          // output staging, 1024-byte aligned
    static constexpr int kCtlOff = kOutOff + kF8OutBytes;      // barriers and flags after it
    static constexpr int kSmemBytes = kCtlOff + kF8CtlBytes + 1024;
    static_assert(kStages >= 3, "ring depth");
    // split-K: the fp32 partial tile parks in the idle stage memory
    static constexpr int kPartStride = BN + 4;  // floats per partial row (padding against bank conflicts)
    static_assert(PAIR || kBM * kPartStride * 4 <= kStages * kStage, "split-K partial tile must fit the stages");
    static_assert(kAStage % 1024 == 0 && kBStage % 1024 == 0, "stages keep 1024-byte alignment");
};

// Instruction descriptor of kind::f8f6f4: fp32 D (bits 4-5 = 1), E4M3 A and
// B (format 0 in bits 7-9 and 10-12), both K-major, N >> 3 in bits 17-22,
// M >> 4 in bits 24-28 (M = 128, or 256 for a pair).
__device__ __forceinline__ uint32_t f8_idesc(int bn, int m) {
    return (1u << 4) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The pair form: issued by the leader, it reads the same shared-memory
// offsets in both CTAs and writes each CTA's 128 rows of D to its own TMEM.
__device__ __forceinline__ void mma_f8_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Grouped raster: consecutive tiles sweep 8 token tiles for each weight
// tile column, so CTAs running together share weight tiles in L2.
__device__ __forceinline__ void f8_tile_coords(const Fp8Params& p, int64_t tile, int64_t& ta, int64_t& tb) {
    const int64_t group_tiles = (int64_t)kGroupA * p.tiles_b;
    const int64_t first_a = (tile / group_tiles) * kGroupA;
    const int64_t rows_in_group = min((int64_t)kGroupA, p.tiles_a - first_a);
    const int64_t local = tile % group_tiles;
    ta = first_a + local % rows_in_group;
    tb = local / rows_in_group;
}

// Epilogue of 8 consecutive columns n0 .. n0+7 of token row m, as packed
// bf16 pairs:  y = bf16_rne((acc * sx[m]) * sw[n] (+ bias[n])).  Columns
// past N get 0.
__device__ __forceinline__ void f8_epi8(const Fp8Params& p, int64_t n0, float sxm, const uint32_t (&r)[8],
                                        uint32_t (&w)[4]) {
    float f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t n = n0 + j;
        const float sw = n < p.N ? __ldg(p.sw + n) : 0.0f;
        f[j] = __fmul_rn(__fmul_rn(__uint_as_float(r[j]), sxm), sw);
        if (p.bias && n < p.N) f[j] = __fadd_rn(f[j], bf16_to_f32(__ldg(p.bias + n)));
    }
#pragma unroll
    for (int j = 0; j < 8; j += 2) w[j / 2] = (uint32_t)f32_to_bf16_rn(f[j]) | ((uint32_t)f32_to_bf16_rn(f[j + 1]) << 16);
}

// Direct stores of 8 columns (outputs whose rows are not 16-byte aligned).
__device__ __forceinline__ void f8_store8(const Fp8Params& p, int64_t m, int64_t n0, float sxm, const uint32_t (&r)[8]) {
    uint32_t w[4];
    f8_epi8(p, n0, sxm, r, w);
    uint16_t* out = p.y + m * p.N + n0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (n0 + j < p.N) out[j] = (uint16_t)(w[j / 2] >> (16 * (j & 1)));
}

__device__ __forceinline__ void f8_sts128(uint32_t addr, const uint32_t (&w)[4]) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                 : "memory");
}

// TMA tensor store of a staged box; rows and columns outside the tensor are
// not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int BN, bool PAIR>
__global__ void __launch_bounds__(kF8Threads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                    const __grid_constant__ CUtensorMap map_y, const Fp8Params p) {
    using Cfg = F8Cfg<BN, PAIR>;
    constexpr int S = Cfg::kStages;
    constexpr int kHalf = BN / 2;  // columns per epilogue warp
    // Barriers the MMA issuer waits on live in the leader; a pair's CTAs
    // arrive on them through cluster addresses.
    constexpr uint32_t kArrivers = PAIR ? 2 : 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    F8Ctl* ctl = reinterpret_cast<F8Ctl*>(smem + Cfg::kCtlOff);
    const uint32_t base = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nkb = (int)((p.K + kF8BK - 1) / kF8BK);
    const int64_t tiles = p.tiles_a * p.tiles_b;
    const int prank = PAIR ? (int)cluster_rank() : 0;  // half of the pair this CTA holds
    const bool leader = prank == 0;
    // split-K (single CTAs): this CTA's k-blocks of its cluster's tile
    const int ksplit = PAIR ? 1 : p.split;
    const int krank = ksplit > 1 ? (int)cluster_rank() : 0;
    const int kb_lo = (int)((int64_t)nkb * krank / ksplit), kb_hi = (int)((int64_t)nkb * (krank + 1) / ksplit);
    const int csize = PAIR ? 2 : ksplit;
    const int64_t unit0 = blockIdx.x / csize;
    const int64_t unit_step = gridDim.x / csize;
    int* abort = &ctl->abort_flag;
    auto leader_addr = [&](uint64_t* bar) -> uint32_t { return PAIR ? mapa(smem_u32(bar), 0) : smem_u32(bar); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&ctl->full[s], kArrivers);  // one arrive-with-bytes per CTA
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->acc_full[b], 1);
            mbar_init(&ctl->acc_empty[b], kArrivers * kF8EpiWarps);
        }
        mbar_init(&ctl->drained, 1);
        ctl->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kF8LoadWarp && lane == 0) {
        prefetch_map(&map_x);
        prefetch_map(&map_w);
        if (p.tma_store) prefetch_map(&map_y);
    }
    if (warp == kF8MmaWarp) {
        if constexpr (PAIR)
            tmem_alloc_pair(&ctl->tmem_base, p.tmem_cols);
        else
            tmem_alloc(&ctl->tmem_base, p.tmem_cols);
    }
    tc_fence_before();
    if constexpr (PAIR)
        cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrive
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    pdl_wait();  // the codes and scales come from earlier launches

    if (warp < kF8EpiWarps) {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int half = warp >> 2;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const int row = quarter * 32 + lane;
        const uint32_t out0 = base + (uint32_t)(Cfg::kOutOff + warp * 2 * kF8OutBuf);
        uint32_t nbox = 0;  // boxes this warp has stored
        int64_t lt = 0;
        for (int64_t tile = unit0; tile < tiles; tile += unit_step, ++lt) {
            const int b = (int)(lt & 1);
            if (!warp_wait(&ctl->acc_full[b], (uint32_t)((lt >> 1) & 1), abort, p.err)) break;
            tc_fence_after();
            int64_t ta, tb;
            f8_tile_coords(p, tile, ta, tb);
            const int64_t m0 = ta * Cfg::kTileM + prank * kBM + quarter * 32;  // this warp's first row
            const int64_t m = m0 + lane;
            const float sxm = m < p.M ? __ldg(p.sx + m) : 0.0f;
            const int64_t n_half = tb * BN + half * kHalf;
            if (ksplit > 1) {
                // park this warp's 32 rows x kHalf columns of the fp32
                // partial in the stage memory (every MMA of the tile, and so
                // every read of the stages, has completed)
                float* prow = reinterpret_cast<float*>(smem) + row * Cfg::kPartStride + half * kHalf;
#pragma unroll 4
                for (int c = 0; c < kHalf; c += 8) {
                    uint32_t r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                    if (kb_hi > kb_lo) {
                        tmem_ld8(lane_base + (uint32_t)(b * BN + half * kHalf + c), r);
                        tmem_wait_ld();
                    }
                    *reinterpret_cast<uint4*>(prow + c) = make_uint4(r[0], r[1], r[2], r[3]);
                    *reinterpret_cast<uint4*>(prow + c + 4) = make_uint4(r[4], r[5], r[6], r[7]);
                }
            } else if (p.tma_store) {
                // 32 columns at a time: stage the warp's 32 x 32 box, then
                // one thread stores it; the buffer used two boxes earlier is
                // free once that store has read it
#pragma unroll 1
                for (int j = 0; j < kHalf / 32; ++j, ++nbox) {
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    const uint32_t buf = out0 + (nbox & 1) * kF8OutBuf;
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint32_t r[8], w[4];
                        tmem_ld8(lane_base + (uint32_t)(b * BN + half * kHalf + j * 32 + c), r);
                        tmem_wait_ld();
                        f8_epi8(p, n_half + j * 32 + c, sxm, r, w);
                        f8_sts128(buf + (uint32_t)(lane * 64 + ((((c >> 3) ^ (lane >> 1)) & 3) << 4)), w);
                    }
                    fence_proxy_async_smem();  // the bulk copy reads these stores
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&map_y, buf, (int32_t)(n_half + j * 32), (int32_t)m0);
                        bulk_commit();
                    }
                }
            } else {
#pragma unroll 4
                for (int c = 0; c < kHalf; c += 8) {
                    uint32_t r[8];
                    tmem_ld8(lane_base + (uint32_t)(b * BN + half * kHalf + c), r);
                    tmem_wait_ld();
                    if (m < p.M && n_half + c < p.N) f8_store8(p, m, n_half + c, sxm, r);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {  // the MMA may refill this buffer
                if constexpr (PAIR)
                    mbar_arrive_cluster(leader_addr(&ctl->acc_empty[b]));
                else
                    mbar_arrive(&ctl->acc_empty[b]);
            }
        }
        if (lane == 0) bulk_wait_all();  // the outputs are written before the CTA ends
        __syncwarp();
    } else if (warp == kF8LoadWarp) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            int64_t kg = 0;
            bool alive = true;
            for (int64_t tile = unit0; alive && tile < tiles; tile += unit_step) {
                int64_t ta, tb;
                f8_tile_coords(p, tile, ta, tb);
                const int32_t xrow = (int32_t)(ta * Cfg::kTileM + prank * kBM);
                const int32_t wrow = (int32_t)(tb * BN + prank * Cfg::kWRows);
                for (int kb = kb_lo; kb < kb_hi; ++kb, ++kg) {
                    const int s = (int)(kg % S);
                    if (!mbar_wait(&ctl->empty[s], (uint32_t)(((kg / S) & 1) ^ 1), abort, p.err)) {
                        alive = false;
                        break;
                    }
                    const uint32_t st = base + (uint32_t)(s * Cfg::kStage);
                    if constexpr (PAIR) {
                        // both CTAs' halves complete on the leader's barrier
                        const uint32_t bar = leader_addr(&ctl->full[s]);
                        mbar_expect_tx_cluster(bar, (uint32_t)Cfg::kStage);
                        tma_load_2d_pair(st, &map_x, kb * kF8BK, xrow, bar);
                        tma_load_2d_pair(st + Cfg::kAStage, &map_w, kb * kF8BK, wrow, bar);
                    } else {
                        mbar_expect_tx(&ctl->full[s], (uint32_t)Cfg::kStage);
                        tma_load_2d(st, &map_x, kb * kF8BK, xrow, &ctl->full[s]);
                        tma_load_2d(st + Cfg::kAStage, &map_w, kb * kF8BK, wrow, &ctl->full[s]);
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && leader) {
            const uint32_t idesc = f8_idesc(BN, Cfg::kTileM);
            auto commit = [&](uint64_t* bar) {
                if constexpr (PAIR)
                    mma_commit_pair(bar);
                else
                    mma_commit(bar);
            };
            int64_t kg = 0, lt = 0;
            bool alive = true;
            for (int64_t tile = unit0; alive && tile < tiles; tile += unit_step, ++lt) {
                const int b = (int)(lt & 1);
                // the epilogue must have drained this buffer's previous tile
                if (!mbar_wait(&ctl->acc_empty[b], (uint32_t)(((lt >> 1) & 1) ^ 1), abort, p.err)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * BN);
                for (int kb = kb_lo; kb < kb_hi; ++kb, ++kg) {
                    const int s = (int)(kg % S);
                    if (!mbar_wait(&ctl->full[s], (uint32_t)((kg / S) & 1), abort, p.err)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_st = base + (uint32_t)(s * Cfg::kStage);
                    const uint32_t b_st = a_st + Cfg::kAStage;
#pragma unroll
                    for (int kk = 0; kk < kF8BK / 32; ++kk) {
                        const uint64_t ad = sw128_desc(a_st + kk * 32);
                        const uint64_t bd = sw128_desc(b_st + kk * 32);
                        const uint32_t acc = (kb != kb_lo || kk != 0) ? 1u : 0u;
                        if constexpr (PAIR)
                            mma_f8_pair(d, ad, bd, idesc, acc);
                        else
                            mma_f8(d, ad, bd, idesc, acc);
                    }
                    commit(&ctl->empty[s]);
                }
                if (alive) commit(&ctl->acc_full[b]);
            }
            // Wait (bounded) until every MMA issued above has completed.
            commit(&ctl->drained);
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
    }

    tc_fence_before();
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(&ctl->abort_flag)) {
        // bulk copies of a CTA that gave up land before its shared memory
        // and TMEM are released (at most one per stage, microseconds); the
        // fault is on record however the flag was set
        if (threadIdx.x == 0) {
            record_fault(p.err, kErrBitTimeout);
            const uint64_t t0 = global_ns();
            while (global_ns() - t0 < kF8AbortDrainNs) __nanosleep(1000);
        }
        __syncthreads();
    }
    tc_fence_after();
    if constexpr (PAIR) {
        // Neither CTA leaves (or frees TMEM) while the pair's MMAs, copies or
        // remote arrives may still touch it.
        cluster_sync_all();
        tc_fence_after();
        if (warp == kF8MmaWarp) tmem_dealloc_pair(tmem, p.tmem_cols);
        return;
    }
    if (ksplit > 1) {
        // Split-K: reduce this CTA's rows of the tile over the cluster's
        // partials (rank order: deterministic), apply the epilogue, store.
        cluster_sync_all();  // every partial is parked
        if (unit0 < tiles) {
            int64_t ta, tb;
            f8_tile_coords(p, unit0, ta, tb);
            const int r_lo = kBM * krank / ksplit, r_hi = kBM * (krank + 1) / ksplit;
            constexpr int kC8 = BN / 8;
            for (int i = threadIdx.x; i < (r_hi - r_lo) * kC8; i += kF8Threads) {
                const int row = r_lo + i / kC8, c = (i % kC8) * 8;
                const int64_t m = ta * kBM + row, n0 = tb * BN + c;
                if (m >= p.M || n0 >= p.N) continue;
                const uint32_t off = base + (uint32_t)((row * Cfg::kPartStride + c) * 4);
                float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int q = 0; q < ksplit; ++q) {
                    const int4 v0 = ld_dsmem_v4(off, (uint32_t)q), v1 = ld_dsmem_v4(off + 16, (uint32_t)q);
                    a[0] += __int_as_float(v0.x);
                    a[1] += __int_as_float(v0.y);
                    a[2] += __int_as_float(v0.z);
                    a[3] += __int_as_float(v0.w);
                    a[4] += __int_as_float(v1.x);
                    a[5] += __int_as_float(v1.y);
                    a[6] += __int_as_float(v1.z);
                    a[7] += __int_as_float(v1.w);
                }
                uint32_t r[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) r[j] = __float_as_uint(a[j]);
                const float sxm = __ldg(p.sx + m);
                if (p.tma_store) {  // rows start on 16-byte boundaries
                    uint32_t w[4];
                    f8_epi8(p, n0, sxm, r, w);
                    *reinterpret_cast<uint4*>(p.y + m * p.N + n0) = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
                    f8_store8(p, m, n0, sxm, r);
                }
            }
        }
        cluster_sync_all();  // no partial is released while another CTA reads it
    }
    if (warp == kF8MmaWarp) tmem_dealloc(tmem, p.tmem_cols);
}

// 2-D bf16 tensor map over the row-major [M, N] output: box = 32 columns x
// 32 rows, 64-byte swizzle (the staging layout of the epilogue warps).
bool make_map_out(CUtensorMap* map, const uint16_t* base, int64_t rows, int64_t N) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)N * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D E4M3 tensor map over a row-major [rows, K] code matrix: box = 128 k x
// box_rows rows, 128-byte swizzle (the K-major layout the MMA reads),
// out-of-range elements read as zero (code 0x00 = +0).
bool make_map_fp8(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t K, int box_rows) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K};
    cuuint32_t box[2] = {(cuuint32_t)kF8BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool PAIR>
cudaError_t prepare_fp8(int dev) {
    static std::mutex mu;
    static bool done[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(fp8_gemm_kernel<BN, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               F8Cfg<BN, PAIR>::kSmemBytes);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

template <int BN, bool PAIR>
cudaError_t launch_bn(const uint8_t* qx, const float* sx, const uint8_t* qw, const float* sw, const uint16_t* bias,
                      uint16_t* y, int64_t M, int64_t N, int64_t K, int split, const LaunchEnv& env) {
    using Cfg = F8Cfg<BN, PAIR>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = prepare_fp8<BN, PAIR>(dev)) != cudaSuccess) return e;
    Fp8Params p = {};
    p.sx = sx;
    p.sw = sw;
    p.bias = bias;
    p.y = y;
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_a = (M + Cfg::kTileM - 1) / Cfg::kTileM;
    p.tiles_b = (N + BN - 1) / BN;
    // two fp32 accumulator buffers of BN columns (the allocation is a power of two)
    p.tmem_cols = BN <= 128 ? 256u : 512u;
    p.split = PAIR ? 1 : split;
    p.err = env.err;
    CUtensorMap map_x, map_w, map_y = {};
    if (!make_map_fp8(&map_x, qx, M, K, kBM) || !make_map_fp8(&map_w, qw, N, K, Cfg::kWRows))
        return cudaErrorInvalidValue;
    // rows of y start on 16-byte boundaries only when N % 8 == 0
    p.tma_store = (N % 8) == 0 ? 1 : 0;
    if (p.tma_store && !make_map_out(&map_y, y, M, N)) return cudaErrorInvalidValue;
    const int64_t tiles = p.tiles_a * p.tiles_b;
    if (p.split > 1) {
        // one tile per cluster of `split` CTAs (the planner keeps them to one wave)
        return launch_kernel(fp8_gemm_kernel<BN, PAIR>, dim3((unsigned)(tiles * p.split)), dim3(kF8Threads),
                             Cfg::kSmemBytes, env.stream, dim3((unsigned)p.split, 1, 1), map_x, map_w, map_y, p);
    }
    const int64_t units = std::min<int64_t>(tiles, PAIR ? env.sm_count / 2 : env.sm_count);
    const int64_t grid = PAIR ? 2 * units : units;
    return launch_kernel(fp8_gemm_kernel<BN, PAIR>, dim3((unsigned)grid), dim3(kF8Threads), Cfg::kSmemBytes,
                         env.stream, PAIR ? dim3(2, 1, 1) : kNoCluster, map_x, map_w, map_y, p);
}

// Clusters of `csize` CTAs of the single-CTA kernel that fit on the GPU at
// once (one CTA per SM; clusters do not span GPCs).
template <int BN>
int f8_active_clusters(int dev, int csize) {
    static std::mutex mu;
    static int cache[64][kMaxSplit + 1] = {};
    if (dev < 0 || dev >= 64 || csize < 1 || csize > kMaxSplit) return 0;
    std::lock_guard<std::mutex> lock(mu);
    int& slot = cache[dev][csize];
    if (slot == 0) {
        if (prepare_fp8<BN, false>(dev) != cudaSuccess) return 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)csize);
        cfg.blockDim = dim3(kF8Threads);
        cfg.dynamicSmemBytes = F8Cfg<BN, false>::kSmemBytes;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)csize;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_kernel<BN, false>, &cfg) != cudaSuccess) n = 0;
        slot = n > 0 ? n : -1;
    }
    return slot > 0 ? slot : 0;
}

struct F8Plan {
    int bn;
    bool pair;
    int split;
};

// Tile width, CTA pairs, and split-K.  Pair tiles are 256 x 256 or 256 x
// 192 (the narrower one when its tiles fill the last wave of pairs better:
// N = 2560 at M = 4096 is 160 wide tiles, 2.1 waves of 76 pairs, or 224
// narrower ones, 2.9 waves).  A k-block of a 128 x BN tile costs
// BN + 64 (MMA and weight bytes, plus the token tile); a persistent launch
// costs its waves of tiles times the k-blocks of a tile, a split launch the
// k-blocks of one CTA plus a fixed allowance for the cluster reduction (one
// wave of clusters, each within the GPU's cluster occupancy).  Pairs (M >
// 128) measured no faster per SM than single CTAs, and win ties.
F8Plan plan_fp8(int dev, int64_t M, int64_t N, int64_t K, int sms) {
    const int64_t nkb = (K + kF8BK - 1) / kF8BK;
    F8Plan best{N > 128 ? 256 : 128, false, 1};
    double best_cost = 1e300;
    auto waves = [](int64_t units, int64_t slots) { return (double)((units + slots - 1) / slots); };
    if (M > kBM && N > 128) {
        // 192-wide pair tiles when they fill the last wave of pairs better
        for (int bn : {256, 192}) {
            const int64_t tiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + bn - 1) / bn);
            const double cost = waves(tiles, sms / 2) * (double)nkb * (bn + 64);
            if (cost < best_cost) {
                best_cost = cost;
                best = F8Plan{bn, true, 1};
            }
        }
    }
    for (int bn : {256, 128}) {
        if (bn == 256 && N <= 128) continue;
        const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + bn - 1) / bn);
        const double per_kb = bn + 64.0;
        double cost = waves(tiles, sms) * (double)nkb * per_kb;
        int split = 1;
        if (tiles < sms) {
            for (int s = 2; s <= kMaxSplit && 2 * s <= nkb; ++s) {
                if (tiles * s > sms) break;
                const int fit = bn == 256 ? f8_active_clusters<256>(dev, s) : f8_active_clusters<128>(dev, s);
                if (tiles > fit) continue;
                const double c = ((double)((nkb + s - 1) / s) + 6.0) * per_kb;
                if (c < cost) {
                    cost = c;
                    split = s;
                }
            }
        }
        if (cost < best_cost) {
            best_cost = cost;
            best = F8Plan{bn, false, split};
        }
    }
    return best;
}

}  // namespace

cudaError_t launch_fp8_gemm(const uint8_t* qx, const float* sx, const uint8_t* qw, const float* sw,
                            const uint16_t* bias, uint16_t* y, int64_t M, int64_t N, int64_t K, const LaunchEnv& env) {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const F8Plan plan = plan_fp8(dev, M, N, K, env.sm_count);
    if (plan.pair && plan.bn == 192) return launch_bn<192, true>(qx, sx, qw, sw, bias, y, M, N, K, 1, env);
    if (plan.pair) return launch_bn<256, true>(qx, sx, qw, sw, bias, y, M, N, K, 1, env);
    if (plan.bn == 256) return launch_bn<256, false>(qx, sx, qw, sw, bias, y, M, N, K, plan.split, env);
    return launch_bn<128, false>(qx, sx, qw, sw, bias, y, M, N, K, plan.split, env);
}

cudaError_t fp8_plan(int64_t M, int64_t N, int64_t K, int sms, int* tile_n, int* split_k, int* pair) {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const F8Plan plan = plan_fp8(dev, M, N, K, sms);
    *tile_n = plan.bn;
    *split_k = plan.split;
    *pair = plan.pair ? 1 : 0;
    return cudaSuccess;
}

cudaError_t launch_fp8_linear(const uint16_t* x, const uint8_t* qw, const float* sw, const uint16_t* bias,
                              uint16_t* y, uint8_t* qx, float* sx, int64_t M, int64_t N, int64_t K,
                              const LaunchEnv& env) {
    // Workspace for the token codes and scales the caller does not keep,
    // from the stream-ordered allocator.
    const size_t codes = qx ? 0 : ((size_t)M * (size_t)K + 255) / 256 * 256;
    const size_t scales = sx ? 0 : (size_t)M * 4;
    void* ws = nullptr;
    cudaError_t e = cudaSuccess;
    if (codes + scales > 0 && (e = cudaMallocAsync(&ws, codes + scales, env.stream)) != cudaSuccess) return e;
    uint8_t* q = qx ? qx : static_cast<uint8_t*>(ws);
    float* s = sx ? sx : reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + codes);
    e = launch_quant_rows_fp8(x, M, K, q, s, env);
    if (e == cudaSuccess) e = launch_fp8_gemm(q, s, qw, sw, bias, y, M, N, K, env);
    if (ws != nullptr) {
        const cudaError_t f = cudaFreeAsync(ws, env.stream);
        if (e == cudaSuccess) e = f;
    }
    return e;
}

}  // namespace i8ql
