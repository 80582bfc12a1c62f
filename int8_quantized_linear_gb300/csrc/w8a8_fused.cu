// W8A8 GEMM for M > 32: int8 weight tiles are converted to fp16 codes inside
// the GEMM, between their TMA loads and the tensor core.
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
// sm_103a has no integer kind of tcgen05.mma, so the product runs as
// kind::f16 with exact arithmetic: int8 codes are exact in fp16, every
// product of two codes is exact in fp32, and the fp32 accumulator in tensor
// memory (TMEM) stays exact over any 1024-deep chunk of k (1024 * 127^2 <
// 2^24).  After each chunk the epilogue warps drain the chunk sum, convert it
// to int32 (exact) and add it to int32 running sums in their registers; the
// chunks alternate between two TMEM buffers.
//
// The token codes arrive already as fp16 (one small pass over M x K before
// this launch).  The weight codes, the large operand, stay int8 in HBM and
// L2 and are converted per k-block here, so the weights cross HBM once, at
// one byte per code, with no conversion pass over them.
//
// Warp roles (512 threads, one CTA per SM):
//   warp 13: token TMA (fp16, 128-byte swizzle, straight into the operand
//     stage the MMA reads);
//   warp 14: weight TMA (int8 rows of 64 bytes) into an int8 ring of up to 8
//     stages; ragged edges of both operands are zero-filled by the maps;
//   warps 8-12: converters, int8 -> fp16 codes (exact), written in the
//     128-byte-swizzled K-major layout into the operand stage;
//   warp 15: TMEM allocation and the MMA issuer (one thread),
//     tcgen05.mma.cta_group::1.kind::f16, M = 128, N = BN;
//   warps 0-7: epilogue: TMEM -> exact int32 running sums -> scales, bias,
//     bf16 stores, overlapping the next tile's main loop.  The scales and
//     bias of a tile are staged in shared memory before its first chunk
//     completes.
// Tiles: tokens on the 128-row MMA side and weights on the BN side, or for
// M <= 128 the reverse ("swap AB": weights fill the 128 rows, the tokens a
// 128-wide N side).  Registers are rebalanced with setmaxnreg: the epilogue
// warpgroups hold the running sums (up to 128 per thread), the others need
// few.
//
// Persistent without split-K (CTA b walks tiles b, b + grid, ... in a grouped
// raster for L2 reuse).  With split-K (few tiles, deep K) a cluster of S CTAs
// shares one tile: CTA r runs k-blocks [nkb*r/S, nkb*(r+1)/S), parks its
// exact int32 partial tile in its idle stage memory, and after a cluster
// barrier reduces rows [128r/S, 128(r+1)/S) over all partials through
// distributed shared memory, in rank order (integer sums: identical to the
// unsplit result).
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
#include <type_traits>

#include "common.cuh"
#include "tc_common.cuh"

namespace i8ql {
namespace {

using namespace tc;

constexpr int kEpiWarps = 8;     // warps 0-7: two per TMEM lane quarter, one per column half
constexpr int kConvWarp0 = 8;    // warps 8-13 convert, in two teams of three
constexpr int kConvWarps = 6;
constexpr int kTeamWarps = 3;    // team t converts the k-blocks kg with kg % 2 == t
constexpr int kLoadWarp = 14;    // token and weight TMA
constexpr int kMmaWarp = 15;
constexpr int kThreads = 16 * 32;
// setmaxnreg split: the launch gives 128 registers to each of the 512
// threads (65,536); the two epilogue warpgroups take 176 and the two others
// keep 80.
constexpr int kLaunchRegs = 128;
constexpr int kEpiRegs = 176;
constexpr int kAuxRegs = 80;
static_assert(256 * kEpiRegs + 256 * kAuxRegs <= kThreads * kLaunchRegs, "register split exceeds the launch allocation");
constexpr int kSmemOptin = 232448;  // largest dynamic shared memory of one CTA (227 KiB)
constexpr int kMaxStages8 = 8;
constexpr int kMaxStagesOp = 4;
constexpr int kCtlBytes = 5120;  // barriers + two sets of staged epilogue parameters
constexpr uint64_t kAbortDrainNs = 50000;  // pause of a CTA that gave up, before it releases its resources

// Shared-memory rings of one CTA for tile width BN (all stages 1024-byte
// aligned), with W = BN weight rows per CTA, or BN / 2 for a CTA pair:
//   operand stages, each the two MMA operands of one k-block:
//     tokens: fp16, 128 rows x 64 k, 128-byte swizzle (TMA writes the
//       layout the MMA reads);
//     weights fp16: W rows x 64 k, same layout (written by the converters);
//   weight stages: int8, W rows x 64 k, 64 bytes per row (TMA).
// One full and one empty barrier per operand stage: the MMA issuer waits
// once and commits once per k-block.
// The weights are the BN side, or with swapped operands the 128-row side
// (swap only uses BN = 128, never pairs).
template <int BN, bool PAIR>
struct FusedCfg {
    static constexpr int kWRows = PAIR ? BN / 2 : BN;
    static constexpr int kTileM = PAIR ? 2 * kBM : kBM;  // token rows of a (non-swapped) tile
    static constexpr int kTokStage = kBM * kBK * 2;
    static constexpr int kStage16 = kWRows * kBK * 2;
    static constexpr int kStage8 = kWRows * kBK;
    static constexpr int kOpStage = kTokStage + kStage16;
    // deeper operand rings measured no faster: the main loop is bound by
    // throughput, not by load latency
    static constexpr int kStagesOp = kWRows <= 128 ? 4 : 3;
    static constexpr int kFixed = kStagesOp * kOpStage;
    static constexpr int kFree = kSmemOptin - 1024 /*alignment slack*/ - kCtlBytes - kFixed;
    static constexpr int kStages8 = kFree / kStage8 < kMaxStages8 ? kFree / kStage8 : kMaxStages8;
    static constexpr int kW8Off = kFixed;
    // Output staging (2 KB per epilogue warp: 32 rows x 32 bf16 columns),
    // only where it fits beside full rings.
    static constexpr int kOutBytes = kEpiWarps * 32 * 64;
    static constexpr bool kStageOut = kFree - kStages8 * kStage8 >= kOutBytes;
    static constexpr int kOutOff = kFixed + kStages8 * kStage8;
    static constexpr int kStageBytes = kFixed + kStages8 * kStage8 + (kStageOut ? kOutBytes : 0);
    static constexpr int kSmemBytes = kStageBytes + 1024 + kCtlBytes;
    static constexpr int kGroups = kWRows / 8;  // 8-row groups of weights per stage
    static constexpr int kGroupsPerWarp = (kGroups + kTeamWarps - 1) / kTeamWarps;
    static constexpr int kPartStride = BN + 4;  // split-K partial tile row (int32), padded against bank conflicts
    static_assert(BN % 32 == 0 && BN >= 128 && BN <= 256, "tile width");
    static_assert(kStages8 >= 3 && kStagesOp <= kMaxStagesOp, "ring depths");
    static_assert(kStage16 % 1024 == 0 && kStage8 % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert(kBM * kPartStride * 4 <= kStageBytes, "split-K partial tile must fit the stages");
    static_assert(kWRows % 8 == 0, "weight rows fill whole swizzle atoms");
};

// Epilogue parameters of one tile, staged in shared memory before its first
// chunk completes: per tile column the column-side scale (sw[n], or sx[m]
// when swapped) and bias bits, per tile row the row-side scale and bias
// bits.  Missing entries (past M or N, or no bias) are zero and never used.
struct EpiParams {
    float col_scale[256];
    float row_scale[kBM];
    uint16_t col_bias[256];
    uint16_t row_bias[kBM];
};

struct Ctl {
    uint64_t op_full[kMaxStagesOp];   // token TMA landed and the converters filled an operand stage
    uint64_t op_empty[kMaxStagesOp];  // the MMA is done with an operand stage
    uint64_t w8_full[kMaxStages8];    // the weight TMA landed an int8 stage
    uint64_t w8_empty[kMaxStages8];   // a converter team is done with an int8 stage
    uint64_t acc_full[2];             // fp32 chunk accumulator buffers in TMEM
    uint64_t acc_empty[2];
    uint64_t drained;
    uint64_t epi_ready[2];  // all epilogue warps staged the parameters of a set
    uint64_t epi_free[2];   // all epilogue warps finished the tile of a set
    uint32_t tmem_base;
    int abort_flag;
    EpiParams epi[2];       // double-buffered by local tile parity
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");

// Epilogue threads t = 0..255 stage the parameters of tile (ta, tb).
__device__ __forceinline__ void stage_epi_params(const W8A8Params& p, int64_t row_base, int64_t col_base, int bn,
                                                 EpiParams& e, int t) {
    if (t < bn) {
        const int64_t j = col_base + t;
        float scale = 0.0f;
        uint16_t bias = 0;
        if (!p.swap) {
            if (j < p.N) {
                scale = __ldg(p.sw + j);
                if (p.bias) bias = __ldg(p.bias + j);
            }
        } else if (j < p.M) {
            scale = __ldg(p.sx + j);
        }
        e.col_scale[t] = scale;
        e.col_bias[t] = bias;
    }
    if (t < kBM) {
        const int64_t i = row_base + t;
        float scale = 0.0f;
        uint16_t bias = 0;
        if (!p.swap) {
            if (i < p.M) scale = __ldg(p.sx + i);
        } else if (i < p.N) {
            scale = __ldg(p.sw + i);
            if (p.bias) bias = __ldg(p.bias + i);
        }
        e.row_scale[t] = scale;
        e.row_bias[t] = bias;
    }
}

// Scale/bias epilogue and stores of W consecutive tile columns c .. c+W-1
// (W = 4 or 8, c a multiple of W) of tile row `row`, from exact int32 sums,
// in the order the method defines:
//   y = bf16_rne(((float)acc * sx[m]) * sw[n] (+ bias[n]))
// Non-swapped tiles hold tokens on the rows, swapped tiles output channels.
template <int W>
__device__ __forceinline__ void store_out(const W8A8Params& p, const EpiParams& e, int64_t row_base,
                                          int64_t col_base, int row, int c, const int32_t* v) {
    if (!p.swap) {
        const int64_t m = row_base + row;
        if (m >= p.M) return;
        const int64_t n0 = col_base + c;
        const float rs = e.row_scale[row];
        float f[W];
#pragma unroll
        for (int j = 0; j < W; ++j) {
            f[j] = __fmul_rn(__fmul_rn(__int2float_rn(v[j]), rs), e.col_scale[c + j]);
            if (p.bias) f[j] = __fadd_rn(f[j], bf16_to_f32(e.col_bias[c + j]));
        }
        if (n0 + W <= p.N && (p.N % W) == 0) {
            uint32_t packed[W / 2];
#pragma unroll
            for (int j = 0; j < W; j += 2)
                packed[j / 2] = (uint32_t)f32_to_bf16_rn(f[j]) | ((uint32_t)f32_to_bf16_rn(f[j + 1]) << 16);
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
                if (n0 + j < p.N) {
                    p.y[m * p.N + n0 + j] = f32_to_bf16_rn(f[j]);
                    if (p.acc) p.acc[m * p.N + n0 + j] = v[j];
                }
            }
        }
    } else {
        const int64_t n = row_base + row;
        if (n >= p.N) return;
        const float rs = e.row_scale[row];
        const float rb = bf16_to_f32(e.row_bias[row]);
#pragma unroll
        for (int j = 0; j < W; ++j) {
            const int64_t m = col_base + c + j;
            if (m < p.M) {
                float f = __fmul_rn(__fmul_rn(__int2float_rn(v[j]), e.col_scale[c + j]), rs);
                if (p.bias) f = __fadd_rn(f, rb);
                p.y[m * p.N + n] = f32_to_bf16_rn(f);
                if (p.acc) p.acc[m * p.N + n] = v[j];
            }
        }
    }
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d);
__device__ __forceinline__ uint4 lds128(uint32_t addr);

// The same epilogue as store_out for a non-swapped tile, KH columns of one
// warp's 32 rows, written through the warp's staging buffer: each whole
// block of 32 columns goes to shared memory row by row (16-byte units
// XOR-swizzled by row pair, no bank conflicts), then out as 8 rows x 64
// contiguous bytes per store instruction instead of 32 rows x 16 bytes; the
// KH % 32 columns left over go out directly.  Needs N % 8 == 0.
template <int KH>
__device__ __forceinline__ void store_staged(const W8A8Params& p, const EpiParams& e, int64_t row_base,
                                             int64_t col_base, int quarter, int half, int lane, uint32_t stage,
                                             const int32_t* run) {
    const int row = quarter * 32 + lane;
    const float rs = e.row_scale[row];
    const int swz = (lane >> 1) & 3;
#pragma unroll
    for (int blk = 0; blk < KH / 32; ++blk) {
        const int c0 = half * KH + blk * 32;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                const int c = c0 + 8 * u + j;
                float f0 = __fmul_rn(__fmul_rn(__int2float_rn(run[blk * 32 + 8 * u + j]), rs), e.col_scale[c]);
                float f1 = __fmul_rn(__fmul_rn(__int2float_rn(run[blk * 32 + 8 * u + j + 1]), rs), e.col_scale[c + 1]);
                if (p.bias) {
                    f0 = __fadd_rn(f0, bf16_to_f32(e.col_bias[c]));
                    f1 = __fadd_rn(f1, bf16_to_f32(e.col_bias[c + 1]));
                }
                w[j / 2] = (uint32_t)f32_to_bf16_rn(f0) | ((uint32_t)f32_to_bf16_rn(f1) << 16);
            }
            sts128(stage + (uint32_t)(lane * 64 + ((u ^ swz) << 4)), w[0], w[1], w[2], w[3]);
        }
        __syncwarp();
#pragma unroll 1  // (unrolled, it pushed the epilogue past its registers)
        for (int r = 0; r < 4; ++r) {
            const int lr = 8 * r + (lane >> 2);
            const int u = lane & 3;
            const uint4 v = lds128(stage + (uint32_t)(lr * 64 + ((u ^ ((lr >> 1) & 3)) << 4)));
            const int64_t m = row_base + quarter * 32 + lr;
            const int64_t n = col_base + c0 + 8 * u;
            if (m < p.M && n < p.N) *reinterpret_cast<uint4*>(p.y + m * p.N + n) = v;
        }
        __syncwarp();
    }
#pragma unroll
    for (int q = (KH / 32) * 4; q < KH / 8; ++q) store_out<8>(p, e, row_base, col_base, row, half * KH + 8 * q, run + 8 * q);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// The work of one unit (a CTA, a split-K cluster or a CTA pair) as a
// sequence of segments, each a tile and a range of its k-blocks.
// Persistent: tiles unit, unit + step, ... each over the unit's split-K
// range [kb_lo, kb_hi).  Stream-K: the iterations [total * u / U,
// total * (u + 1) / U) of the tile-major order (total = tiles * nkb), cut
// at tile boundaries and walked from the END of the range backwards: the
// first segment a unit processes is the head of a tile that later units
// finish (it is parked at once), the last one is the tail of a tile whose
// head earlier units parked long before.  Every role walks the same
// sequence.
struct Work {
    int64_t cur, end, step;  // stream-K: cur is the range start, end moves down
    int kb_lo, kb_hi, nkb;
    bool sk;

    __device__ __forceinline__ bool next(int64_t& tile, int& lo, int& hi) {
        if (cur >= end) return false;
        if (!sk) {
            tile = cur;
            lo = kb_lo;
            hi = kb_hi;
            cur += step;
            return true;
        }
        tile = (end - 1) / nkb;
        const int64_t t0 = tile * nkb;
        lo = (int)(max(cur, t0) - t0);
        hi = (int)(end - t0);
        end = t0 + lo;
        return true;
    }
    // k-blocks of the whole sequence
    __device__ __forceinline__ int64_t kblocks() const {
        if (sk) return end > cur ? end - cur : 0;
        return (end > cur ? (end - cur + step - 1) / step : 0) * (kb_hi - kb_lo);
    }
};

// First stream-K iteration of unit u.
__device__ __forceinline__ int64_t sk_first(int64_t total, int64_t u, int64_t units) { return total * u / units; }

// (Stream-K runs on CTA pairs only; SK = false compiles it out.)
template <bool SK>
__device__ __forceinline__ Work make_work(const W8A8Params& p, int64_t unit0, int64_t unit_step, int kb_lo, int kb_hi,
                                          int nkb) {
    Work w;
    w.nkb = nkb;
    w.kb_lo = kb_lo;
    w.kb_hi = kb_hi;
    w.sk = SK && p.sk != 0;
    w.step = unit_step;
    const int64_t tiles = p.tiles_a * p.tiles_b;
    if (w.sk) {
        const int64_t total = tiles * nkb;
        w.cur = sk_first(total, unit0, p.sk_units);
        w.end = sk_first(total, unit0 + 1, p.sk_units);
    } else {
        w.cur = unit0;
        w.end = tiles;
    }
    return w;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int BN, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    w8a8_fused_kernel(const __grid_constant__ CUtensorMap map_tok, const __grid_constant__ CUtensorMap map_wgt,
                      const W8A8Params p) {
    using Cfg = FusedCfg<BN, PAIR>;
    constexpr int S8 = Cfg::kStages8;
    constexpr int SO = Cfg::kStagesOp;
    constexpr int kHalf = BN / 2;  // columns per epilogue warp
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + Cfg::kStageBytes);
    int32_t* part = reinterpret_cast<int32_t*>(smem);  // split-K partial tile (after the main loop)
    // operand stage s: tokens at op_base + s * kOpStage, fp16 weights
    // kTokStage bytes after them
    const uint32_t op_base = smem_u32(smem);
    const uint32_t w8_base = op_base + Cfg::kW8Off;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t K = p.K;
    const int nkb = (int)((K + kBK - 1) / kBK);
    // A pair (cluster of 2) shares every tile; split-K clusters (p.split
    // CTAs, never pairs) share one tile's k range.
    const int S = PAIR ? 1 : p.split;
    const int csize = PAIR ? 2 : S;
    const int rank = csize > 1 ? (int)cluster_rank() : 0;
    const int krank = PAIR ? 0 : rank;
    const int prank = PAIR ? rank : 0;  // half of the pair this CTA holds
    const bool leader = prank == 0;
    const int kb_lo = (int)((int64_t)nkb * krank / S);
    const int kb_hi = (int)((int64_t)nkb * (krank + 1) / S);
    const int64_t tiles = p.tiles_a * p.tiles_b;
    const int64_t unit0 = blockIdx.x / csize;
    const int64_t unit_step = gridDim.x / csize;
    int* abort = &ctl->abort_flag;
    // Barriers the MMA issuer waits on live in the leader; a pair's CTAs
    // arrive on them through cluster addresses.
    constexpr uint32_t kArrivers = PAIR ? 2 : 1;
    auto leader_addr = [&](uint64_t* bar) -> uint32_t { return PAIR ? mapa(smem_u32(bar), 0) : smem_u32(bar); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < SO; ++s) {
            // per CTA of the pair: the token producer's arrive-with-bytes and
            // one arrive per converter warp of the team
            mbar_init(&ctl->op_full[s], kArrivers * (1 + kTeamWarps));
            mbar_init(&ctl->op_empty[s], 1);
        }
        for (int s = 0; s < S8; ++s) {
            mbar_init(&ctl->w8_full[s], 1);
            mbar_init(&ctl->w8_empty[s], kTeamWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->acc_full[b], 1);
            mbar_init(&ctl->acc_empty[b], kArrivers * kEpiWarps);
            mbar_init(&ctl->epi_ready[b], kEpiWarps);
            mbar_init(&ctl->epi_free[b], kEpiWarps);
        }
        mbar_init(&ctl->drained, 1);
        ctl->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kLoadWarp && lane == 0) {
        prefetch_map(&map_tok);
        prefetch_map(&map_wgt);
    }
    if (warp == kMmaWarp) {
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

    if (warp < kEpiWarps) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int half = warp >> 2;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const int row = quarter * 32 + lane;  // tile row of this thread
        int32_t run[kHalf];
        int64_t cg = 0;
        int64_t lt = 0;  // tiles of this CTA so far
        bool alive = true;
        Work work = make_work<PAIR>(p, unit0, unit_step, kb_lo, kb_hi, nkb);
        int64_t tile;
        int seg_lo, seg_hi;
        for (; alive && work.next(tile, seg_lo, seg_hi); ++lt) {
            const int nch = (seg_hi - seg_lo + kChunkKB - 1) / kChunkKB;
            int64_t ta, tb;
            tile_coords(p, tile, ta, tb);
            // Stage this tile's scales and bias in parameter set lt % 2 once
            // every epilogue warp is done with the tile that used it before;
            // the loads overlap the MMA of the first chunk.
            const int eb = (int)(lt & 1);
            const uint32_t eu = (uint32_t)((lt >> 1) & 1);
            if (!warp_wait<true>(&ctl->epi_free[eb], eu ^ 1u, abort, p.err)) break;
            EpiParams& ep = ctl->epi[eb];
            const int64_t row_base = ta * Cfg::kTileM + prank * kBM;
            const int64_t col_base = tb * BN;
            stage_epi_params(p, row_base, col_base, BN, ep, (int)threadIdx.x);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->epi_ready[eb]);
            if (!warp_wait<true>(&ctl->epi_ready[eb], eu, abort, p.err)) break;
            for (int c = 0; c < nch; ++c, ++cg) {
                const int b = (int)(cg & 1);
                if (!warp_wait<true>(&ctl->acc_full[b], (uint32_t)((cg >> 1) & 1), abort, p.err)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col0 = (uint32_t)(b * BN + half * kHalf);
#pragma unroll
                for (int grp = 0; grp < kHalf / 8; ++grp) {
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
                if (lane == 0) {  // the MMA may refill this buffer
                    if constexpr (PAIR)
                        mbar_arrive_cluster(leader_addr(&ctl->acc_empty[b]));
                    else
                        mbar_arrive(&ctl->acc_empty[b]);
                }
            }
            if (!alive) break;
            if (S > 1) {
                // Split-K: park the partial tile in the idle stage memory (the
                // last chunk's completion covers every MMA, hence every load
                // and conversion of this CTA).
                int4* dst = reinterpret_cast<int4*>(part + row * Cfg::kPartStride + half * kHalf);
#pragma unroll
                for (int q = 0; q < kHalf / 4; ++q)
                    dst[q] = make_int4(run[4 * q], run[4 * q + 1], run[4 * q + 2], run[4 * q + 3]);
                continue;
            }
            if (PAIR && p.sk && seg_hi < nkb) {
                // Stream-K, a part of a tile finished by a later unit (the
                // first segment this unit processes): park it for the
                // finisher (coalesced: consecutive lanes, consecutive rows)
                // and count this thread's stores done with a release.
                int4* slot = reinterpret_cast<int4*>(p.sk_part + (unit0 * 2 + prank) * (int64_t)(kBM * BN));
#pragma unroll
                for (int q = 0; q < kHalf / 4; ++q)
                    __stcg(slot + (q * 2 + half) * kBM + row,
                           make_int4(run[4 * q], run[4 * q + 1], run[4 * q + 2], run[4 * q + 3]));
                red_release_gpu_add(p.sk_flags + unit0 * 2 + prank, 1u);
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->epi_free[eb]);
                continue;
            }
            if (PAIR && p.sk && seg_lo > 0) {
                // Stream-K, the tile's finisher (it holds the last k-block;
                // this is the last segment it processes): add the parts
                // parked by the earlier units whose ranges reach into the
                // tile.  Each parked its part as the first segment it
                // processed, before waiting for anything itself, and was
                // dispatched no later than this unit, so the wait is short
                // and never depends on a unit that is not resident yet.
                const int64_t total = tiles * nkb;
                const int64_t tile_start = tile * nkb;
                for (int64_t q = unit0 - 1; q >= 0 && sk_first(total, q + 1, p.sk_units) > tile_start; --q) {
                    if (sk_first(total, q, p.sk_units) == sk_first(total, q + 1, p.sk_units)) continue;  // no work
                    const unsigned* f = p.sk_flags + q * 2 + prank;
                    const uint64_t t0 = global_ns();
                    while (true) {
                        const bool seen = ld_acquire_gpu(f) >= p.sk_flag_target;
                        if (__all_sync(0xffffffffu, seen)) break;
                        const bool give_up =
                            *reinterpret_cast<volatile int*>(abort) != 0 || global_ns() - t0 > p.sk_wait_ns;
                        if (__any_sync(0xffffffffu, give_up)) {
                            alive = false;
                            break;
                        }
                        __nanosleep(128);
                    }
                    if (!alive) {
                        if (lane == 0) {
                            record_fault(p.err, kErrBitTimeout);
                            *reinterpret_cast<volatile int*>(abort) = 1;
                        }
                        break;
                    }
                    const int4* slot = reinterpret_cast<const int4*>(p.sk_part + (q * 2 + prank) * (int64_t)(kBM * BN));
#pragma unroll
                    for (int v = 0; v < kHalf / 4; ++v) {
                        const int4 t = __ldcg(slot + (v * 2 + half) * kBM + row);
                        run[4 * v] += t.x;
                        run[4 * v + 1] += t.y;
                        run[4 * v + 2] += t.z;
                        run[4 * v + 3] += t.w;
                    }
                }
                if (!alive) break;
            }
            if (Cfg::kStageOut && !p.swap && p.acc == nullptr && (p.N % 8) == 0) {
                store_staged<kHalf>(p, ep, row_base, col_base, quarter, half, lane,
                                    op_base + (uint32_t)(Cfg::kOutOff + warp * 2048), run);
            } else {
#pragma unroll
                for (int q = 0; q < kHalf / 8; ++q)
                    store_out<8>(p, ep, row_base, col_base, row, half * kHalf + 8 * q, run + 8 * q);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->epi_free[eb]);
        }
        // back to the launch share for the common tail
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLaunchRegs));
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kAuxRegs));
        if (warp == kLoadWarp) {
            // ---------------------------------------------------------- TMA producer
            // Token and weight loads of a k-block are issued together; each
            // waits for its own ring.
            if (lane == 0) {
                int64_t kg = 0;  // k-blocks issued by this CTA
                bool alive = true;
                Work work = make_work<PAIR>(p, unit0, unit_step, kb_lo, kb_hi, nkb);
                int64_t tile;
                int seg_lo, seg_hi;
                while (alive && work.next(tile, seg_lo, seg_hi)) {
                    int64_t ta, tb;
                    tile_coords(p, tile, ta, tb);
                    const int32_t tok_row = (int32_t)(p.swap ? tb * kBM : ta * Cfg::kTileM + prank * kBM);
                    const int32_t wgt_row = (int32_t)(p.swap ? ta * kBM : tb * BN + prank * Cfg::kWRows);
                    for (int kb = seg_lo; kb < seg_hi; ++kb, ++kg) {
                        const int s8 = (int)(kg % S8);
                        const int so = (int)(kg % SO);
                        if (!mbar_wait_inline(&ctl->w8_empty[s8], (uint32_t)(((kg / S8) & 1) ^ 1), abort, p.err)) {
                            alive = false;
                            break;
                        }
                        mbar_expect_tx(&ctl->w8_full[s8], (uint32_t)Cfg::kStage8);
                        tma_load_2d(w8_base + (uint32_t)(s8 * Cfg::kStage8), &map_wgt, kb * kBK, wgt_row,
                                    &ctl->w8_full[s8]);
                        if (!mbar_wait_inline(&ctl->op_empty[so], (uint32_t)(((kg / SO) & 1) ^ 1), abort, p.err)) {
                            alive = false;
                            break;
                        }
                        if constexpr (PAIR) {
                            // both halves of the token tile complete on the leader's barrier
                            const uint32_t bar = leader_addr(&ctl->op_full[so]);
                            mbar_expect_tx_cluster(bar, (uint32_t)Cfg::kTokStage);
                            tma_load_2d_pair(op_base + (uint32_t)(so * Cfg::kOpStage), &map_tok, kb * kBK, tok_row,
                                             bar);
                        } else {
                            mbar_expect_tx(&ctl->op_full[so], (uint32_t)Cfg::kTokStage);
                            tma_load_2d(op_base + (uint32_t)(so * Cfg::kOpStage), &map_tok, kb * kBK, tok_row,
                                        &ctl->op_full[so]);
                        }
                    }
                }
            }
            __syncwarp();
        } else if (warp == kMmaWarp) {
            // ---------------------------------------------------------- MMA issuer
            if (lane == 0 && leader) {
                const uint32_t idesc = PAIR ? f16_idesc_pair(BN) : f16_idesc(BN);
                auto wait = [&](uint64_t* bar, uint32_t parity) { return mbar_wait_inline(bar, parity, abort, p.err); };
                auto commit = [&](uint64_t* bar) {
                    if constexpr (PAIR)
                        mma_commit_pair(bar);
                    else
                        mma_commit(bar);
                };
                int64_t kg = 0;  // k-blocks consumed
                int64_t cg = 0;  // chunks accumulated
                bool alive = true;
                Work work = make_work<PAIR>(p, unit0, unit_step, kb_lo, kb_hi, nkb);
                int64_t tile;
                int seg_lo, seg_hi;
                while (alive && work.next(tile, seg_lo, seg_hi)) {
                    const int nch = (seg_hi - seg_lo + kChunkKB - 1) / kChunkKB;
                    for (int c = 0; c < nch && alive; ++c, ++cg) {
                        const int b = (int)(cg & 1);
                        // the epilogue must have drained this buffer's previous chunk
                        if (!wait(&ctl->acc_empty[b], (uint32_t)(((cg >> 1) & 1) ^ 1))) {
                            alive = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem + (uint32_t)(b * BN);
                        const int kb_first = seg_lo + c * kChunkKB;
                        const int kb_end = min(seg_hi, kb_first + kChunkKB);
                        for (int kb = kb_first; kb < kb_end; ++kb, ++kg) {
                            const int so = (int)(kg % SO);
                            if (!wait(&ctl->op_full[so], (uint32_t)((kg / SO) & 1))) {
                                alive = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t tok_st = op_base + (uint32_t)(so * Cfg::kOpStage);
                            const uint32_t wgt_st = tok_st + Cfg::kTokStage;
                            const uint32_t a_st = p.swap ? wgt_st : tok_st;
                            const uint32_t b_st = p.swap ? tok_st : wgt_st;
#pragma unroll
                            for (int kk = 0; kk < kBK / 16; ++kk) {
                                const uint64_t ad = sw128_desc(a_st + kk * 32);
                                const uint64_t bd = sw128_desc(b_st + kk * 32);
                                const uint32_t acc = (kb != kb_first || kk != 0) ? 1u : 0u;
                                if constexpr (PAIR)
                                    mma_f16_pair(d, ad, bd, idesc, acc);
                                else
                                    mma_f16(d, ad, bd, idesc, acc);
                            }
                            commit(&ctl->op_empty[so]);
                        }
                        if (alive) commit(&ctl->acc_full[b]);
                    }
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
        } else {
            // ---------------------------------------------------------- converters
            // Two teams of three warps take alternate k-blocks, so one team's
            // waits and fences overlap the other team's conversions; a warp
            // issues all its loads before its conversions.
            constexpr int G = Cfg::kGroups;
            const int cw = warp - kConvWarp0;
            const int team = cw / kTeamWarps;
            const int tw = cw % kTeamWarps;
            // A unit is 4 weight rows x 64 k: lane l converts the 8 codes
            // k = 8c .. 8c+7 (c = l % 8) of row 4u + l / 8.  Each 8-lane group
            // then stores one whole 128-byte row of the 128-byte swizzle (the
            // 8 chunks land at c ^ (row % 8)) and reads 64 contiguous bytes,
            // so neither access has bank conflicts.
            constexpr int U = 2 * G;                                  // units per stage
            constexpr int UPW = (U + kTeamWarps - 1) / kTeamWarps;  // per warp
            const int r_in = lane >> 3;
            const int c = lane & 7;
            const uint32_t src0 = w8_base + (uint32_t)(r_in * kBK + c * 8);
            const uint32_t dst0 = op_base + Cfg::kTokStage + (uint32_t)(r_in * (kBK * 2));
            const int64_t total = make_work<PAIR>(p, unit0, unit_step, kb_lo, kb_hi, nkb).kblocks();
            for (int64_t kg = team; kg < total; kg += 2) {
                const int s8 = (int)(kg % S8);
                const int so = (int)(kg % SO);
                if (!warp_wait<true>(&ctl->w8_full[s8], (uint32_t)((kg / S8) & 1), abort, p.err) ||
                    !warp_wait<true>(&ctl->op_empty[so], (uint32_t)(((kg / SO) & 1) ^ 1), abort, p.err))
                    break;
                const uint32_t src = src0 + (uint32_t)(s8 * Cfg::kStage8);
                const uint32_t dst = dst0 + (uint32_t)(so * Cfg::kOpStage);
                uint2 v[UPW];
#pragma unroll
                for (int i = 0; i < UPW; ++i) {
                    const int u = tw + i * kTeamWarps;
                    if (u < U) v[i] = lds64(src + (uint32_t)(u * 4 * kBK));
                }
#pragma unroll
                for (int i = 0; i < UPW; ++i) {
                    const int u = tw + i * kTeamWarps;
                    if (u < U) {
                        uint32_t h[4];
                        i8x4_to_f16(v[i].x, h[0], h[1]);
                        i8x4_to_f16(v[i].y, h[2], h[3]);
                        const int row7 = (4 * u + r_in) & 7;
                        sts128(dst + (uint32_t)(u * 4 * (kBK * 2)) + (uint32_t)((c ^ row7) << 4), h[0], h[1], h[2],
                               h[3]);
                    }
                }
                fence_proxy_async_smem();  // the tensor core reads these stores
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        mbar_arrive_cluster(leader_addr(&ctl->op_full[so]));
                    else
                        mbar_arrive(&ctl->op_full[so]);
                    mbar_arrive(&ctl->w8_empty[s8]);
                }
            }
        }
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kLaunchRegs));
    }

    tc_fence_before();
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(&ctl->abort_flag)) {
        // A CTA that gave up may still have bulk copies in flight into its
        // shared memory (at most one k-block per ring stage, tens of KB);
        // they land within microseconds, so a fixed pause lets them complete
        // before the CTA's shared memory and TMEM are released.
        if (threadIdx.x == 0) {
            record_fault(p.err, kErrBitTimeout);  // on record however the flag was set
            const uint64_t t0 = global_ns();
            while (global_ns() - t0 < kAbortDrainNs) __nanosleep(1000);
        }
        __syncthreads();
    }
    tc_fence_after();
    if constexpr (PAIR) {
        // Neither CTA leaves (or frees TMEM) while the pair's MMAs, TMA
        // completions or remote arrives may still touch it.
        cluster_sync_all();
        tc_fence_after();
        if (warp == kMmaWarp) tmem_dealloc_pair(tmem, p.tmem_cols);
        return;
    }
    if (warp == kMmaWarp) tmem_dealloc(tmem, p.tmem_cols);
    if (S > 1) {
        // Every CTA of the cluster reaches both barriers, on the abort path too.
        cluster_sync_all();  // all partial tiles are in place
        if (unit0 < tiles && !*reinterpret_cast<volatile int*>(&ctl->abort_flag)) {
            int64_t ta, tb;
            tile_coords(p, unit0, ta, tb);
            const int64_t row_base = ta * kBM, col_base = tb * BN;
            const int r0 = kBM * rank / S, r1 = kBM * (rank + 1) / S;
            const int nrows = r1 - r0;
            constexpr int kVecs = BN / 4;
            const uint32_t part_addr = smem_u32(part);
            const EpiParams& ep = ctl->epi[0];  // the CTA's only tile staged set 0
            for (int i = threadIdx.x; i < nrows * kVecs; i += kThreads) {
                // consecutive threads take consecutive output channels, so
                // the stores coalesce in both orientations
                const int row = p.swap ? r0 + i % nrows : r0 + i / kVecs;
                const int c = (p.swap ? i / nrows : i % kVecs) * 4;
                const uint32_t off = part_addr + (uint32_t)(row * Cfg::kPartStride + c) * 4u;
                // every rank's partial in flight before the rank-ordered sum
                // (a load after each add would wait out each load in turn)
                int4 t[kMaxSplit];
#pragma unroll
                for (int q = 0; q < kMaxSplit; ++q)
                    if (q < S) t[q] = ld_dsmem_v4(off, (uint32_t)q);
                int32_t v[4] = {0, 0, 0, 0};
#pragma unroll
                for (int q = 0; q < kMaxSplit; ++q) {
                    if (q < S) {
                        v[0] += t[q].x;
                        v[1] += t[q].y;
                        v[2] += t[q].z;
                        v[3] += t[q].w;
                    }
                }
                store_out<4>(p, ep, row_base, col_base, row, c, v);
            }
        }
        cluster_sync_all();  // peers are done reading this CTA's partial tile
    }
}

// 2-D int8 tensor map over a row-major [rows, K] code matrix: box = 64 k x
// box_rows rows, no swizzle (rows of 64 bytes in shared memory),
// out-of-range elements read as zero.
bool make_map_i8(CUtensorMap* map, const int8_t* base, int64_t rows, int64_t K, int box_rows) {
    auto enc = tc::tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp16 tensor map over the row-major [rows, K] token codes: box = 64 k x
// 128 rows, 128-byte swizzle (the K-major canonical layout the MMA reads),
// out-of-range elements read as zero.
bool make_map_f16(CUtensorMap* map, const uint16_t* base, int64_t rows, int64_t K) {
    auto enc = tc::tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tile widths the kernel is built for (single CTAs), and those of CTA
// pairs.
constexpr int kTileWidths[] = {256, 224, 192, 160, 128};
constexpr int kPairWidths[] = {256, 224, 192, 160, 128};
// A pair moves a 256 x BN tile through two SMs with half the shared-memory
// operand traffic and conversion work per SM of a single-CTA 128 x BN tile;
// its k-blocks are costed at this fraction of the single-CTA ones.
constexpr double kPairCost = 0.75;

// Calls f with (integral_constant BN, integral_constant PAIR) for a built
// configuration.
template <typename F>
auto with_cfg(int bn, bool pair, F&& f) {
    using std::integral_constant;
    if (pair) {
        switch (bn) {
            case 256: return f(integral_constant<int, 256>{}, integral_constant<bool, true>{});
            case 224: return f(integral_constant<int, 224>{}, integral_constant<bool, true>{});
            case 192: return f(integral_constant<int, 192>{}, integral_constant<bool, true>{});
            case 160: return f(integral_constant<int, 160>{}, integral_constant<bool, true>{});
            default: return f(integral_constant<int, 128>{}, integral_constant<bool, true>{});
        }
    }
    switch (bn) {
        case 256: return f(integral_constant<int, 256>{}, integral_constant<bool, false>{});
        case 224: return f(integral_constant<int, 224>{}, integral_constant<bool, false>{});
        case 192: return f(integral_constant<int, 192>{}, integral_constant<bool, false>{});
        case 160: return f(integral_constant<int, 160>{}, integral_constant<bool, false>{});
        default: return f(integral_constant<int, 128>{}, integral_constant<bool, false>{});
    }
}

// Opt every configuration into its dynamic shared memory, once per device.
// Occupancy queries and launches both need it.
cudaError_t prepare_device(int dev) {
    static std::mutex mu;
    static bool done[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    auto set = [](auto w, auto pr) {
        constexpr int BN = decltype(w)::value;
        constexpr bool PAIR = decltype(pr)::value;
        return cudaFuncSetAttribute(w8a8_fused_kernel<BN, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    FusedCfg<BN, PAIR>::kSmemBytes);
    };
    for (int bn : kTileWidths) {
        const cudaError_t e = with_cfg(bn, false, set);
        if (e != cudaSuccess) return e;
    }
    for (int bn : kPairWidths) {
        const cudaError_t e = with_cfg(bn, true, set);
        if (e != cudaSuccess) return e;
    }
    done[dev] = true;
    return cudaSuccess;
}

// Clusters of `csize` CTAs of a configuration that can run at once on
// device `dev` (cached; 0 if none or on error).  Needs prepare_device(dev).
int active_clusters(int dev, int bn, bool pair, int csize) {
    static std::mutex mu;
    static int cache[64][2][5][kMaxSplit + 1] = {};
    int bi = 0;
    while (kTileWidths[bi] != bn) ++bi;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64 || csize < 1 || csize > kMaxSplit) return 0;
    int& slot = cache[dev][pair ? 1 : 0][bi][csize];
    if (slot == 0) {
        int n = 0;
        cudaError_t e = with_cfg(bn, pair, [&](auto w, auto pr) {
            constexpr int BN = decltype(w)::value;
            constexpr bool PAIR = decltype(pr)::value;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)csize);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = FusedCfg<BN, PAIR>::kSmemBytes;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = (unsigned)csize;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            return cudaOccupancyMaxActiveClusters(&n, w8a8_fused_kernel<BN, PAIR>, &cfg);
        });
        if (e != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        slot = n > 0 ? n : -1;
    }
    return slot > 0 ? slot : 0;
}

struct Plan {
    int bn;
    int split;
    bool pair;
    int64_t units;  // CTAs (or clusters) the persistent grid runs
    int64_t tiles_a, tiles_b;
    bool sk = false;  // stream-K over `units` pairs
};

// Stream-K fix-up (parking partial tiles, owners adding them, the extra
// segment ends), as measured: about this many pair k-blocks per launch.
constexpr int64_t kSkFixupKb = 40;

// Bytes of the stream-K workspace of a plan: the flags (2 per pair, padded
// to 256 bytes), then one int32 partial tile half (128 x BN) per CTA.
size_t sk_flag_count(const Plan& plan) { return plan.sk ? (size_t)plan.units * 2 : 0; }
size_t sk_bytes(const Plan& plan) {
    if (!plan.sk) return 0;
    return (sk_flag_count(plan) * 4 + 255) / 256 * 256 + (size_t)plan.units * 2 * kBM * plan.bn * 4;
}

// Tile width, CTA pairs or single CTAs, split-K factor, and stream-K.  A
// k-block of a 128 x BN tile is costed BN + 96 (MMA work plus the fixed
// A-side work); a persistent launch costs its number of waves of tiles, a
// split launch one wave of clusters plus a fixed allowance for the cross-CTA
// reduction, a stream-K launch its even share of k-blocks plus the fix-up.
Plan choose_plan(int dev, int64_t M, int64_t N, int64_t K, int sms, bool swap, bool allow_sk) {
    const int64_t nkb = (K + kBK - 1) / kBK;
    Plan best{128, 1, false, 1, 1, 1};
    double best_cost = 1e300;
    for (int bn : kTileWidths) {
        if (swap && bn != kBM) continue;  // tokens fill a 128-wide N side
        const int64_t ta = swap ? (N + kBM - 1) / kBM : (M + kBM - 1) / kBM;
        const int64_t tb = swap ? 1 : (N + bn - 1) / bn;
        const int64_t tiles = ta * tb;
        const double per_kb = bn + 96.0;
        const double waves = (double)((tiles + sms - 1) / sms);
        double cost = waves * (double)nkb * per_kb + 4.0 * per_kb;
        int split = 1;
        if (tiles < sms) {
            for (int s = 2; s <= kMaxSplit && s * 4 <= nkb; ++s) {
                if (tiles * s > sms || tiles > active_clusters(dev, bn, false, s)) continue;
                const double c = ((double)((nkb + s - 1) / s) + 8.0) * per_kb;
                if (c < cost) {
                    cost = c;
                    split = s;
                }
            }
        }
        if (cost < best_cost) {
            best_cost = cost;
            best = Plan{bn, split, false, split > 1 ? tiles : std::min<int64_t>(tiles, sms), ta, tb};
        }
    }
    if (!swap) {
        for (int bn : kPairWidths) {
            const int64_t pairs = active_clusters(dev, bn, true, 2);
            if (pairs == 0) continue;
            const int64_t ta = (M + 2 * kBM - 1) / (2 * kBM);
            const int64_t tb = (N + bn - 1) / bn;
            const int64_t tiles = ta * tb;
            const double per_kb = bn + 96.0;
            const double waves = (double)((tiles + pairs - 1) / pairs);
            const double cost = (waves * (double)nkb * kPairCost + 4.0) * per_kb;
            if (cost < best_cost) {
                best_cost = cost;
                best = Plan{bn, 1, true, std::min<int64_t>(tiles, pairs), ta, tb};
            }
        }
    }
    if (!swap && allow_sk) {
        // Stream-K on 256-wide pair tiles, for tiles that outnumber the
        // pairs.  Measured with every SM busy, a pair k-block costs about
        // the same at any tile width, so the alternative costs its fewest
        // waves of whole tiles times nkb; stream-K costs an even share of
        // all k-blocks plus the fix-up.
        // Its per-pair ranges spread the tiles running at one time over the
        // whole problem, so the operand panels they share stop hitting in
        // L2: with deep K over many waves that costs more DRAM traffic than
        // the tail it removes (Qwen3-8B down at M = 8,192, K = 12,288, 6.7
        // waves: 680 against 570 us, DRAM traffic 7x the algorithmic bytes),
        // while at K = 4,096 and 10 waves stream-K still wins (qkv at
        // M = 8,192: 300 against 322 us).
        constexpr int bn = 256;
        const int64_t pairs = active_clusters(dev, bn, true, 2);
        const int64_t ta = (M + 2 * kBM - 1) / (2 * kBM);
        const int64_t tiles = ta * ((N + bn - 1) / bn);
        const bool deep_many_waves = K >= 8192 && tiles > 3 * pairs;
        if (pairs >= 2 && tiles > pairs && !deep_many_waves) {
            int64_t whole = INT64_MAX;
            for (int w : kPairWidths) {
                const int64_t pw = active_clusters(dev, w, true, 2);
                if (pw == 0) continue;
                const int64_t tw = ta * ((N + w - 1) / w);
                whole = std::min(whole, (tw + pw - 1) / pw * nkb);
            }
            const int64_t total = tiles * nkb;
            if ((total + pairs - 1) / pairs + kSkFixupKb < whole) best = Plan{bn, 1, true, pairs, ta, tiles / ta, true};
        }
    }
    return best;
}

uint32_t pow2_cols(int need) {
    uint32_t c = 32;
    while ((int)c < need) c <<= 1;
    return c;
}

}  // namespace

namespace tc {

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

}  // namespace tc

cudaError_t w8a8_plan(int64_t M, int64_t N, int64_t K, int sms, bool allow_sk, int* tile_n, int* split_k, int* pair) {
    if (M <= kW8A8DecodeMaxM) {
        *tile_n = 0;
        *split_k = 0;
        *pair = 0;
        return cudaSuccess;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = prepare_device(dev)) != cudaSuccess) return e;
    const Plan plan = choose_plan(dev, M, N, K, sms, M <= kBM, allow_sk);
    *tile_n = plan.bn;
    *split_k = plan.split;
    *pair = plan.sk ? 2 : (plan.pair ? 1 : 0);
    return cudaSuccess;
}

cudaError_t w8a8_sk_workspace(int64_t M, int64_t N, int64_t K, int sms, size_t* bytes, int* flags) {
    *bytes = 0;
    *flags = 0;
    if (M <= kBM) return cudaSuccess;  // swapped operands: no pairs, no stream-K
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = prepare_device(dev)) != cudaSuccess) return e;
    const Plan plan = choose_plan(dev, M, N, K, sms, false, true);
    *bytes = sk_bytes(plan);
    *flags = (int)sk_flag_count(plan);
    return cudaSuccess;
}

cudaError_t launch_w8a8_fused(const uint16_t* x16, const float* sx, const int8_t* qw, const float* sw,
                              const uint16_t* bias, uint16_t* y, int32_t* acc, int64_t M, int64_t N, int64_t K,
                              void* sk_ws, size_t sk_ws_bytes, const LaunchEnv& env) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = prepare_device(dev)) != cudaSuccess) return e;
    W8A8Params p = {};
    p.K = K;
    p.sx = sx;
    p.sw = sw;
    p.bias = bias;
    p.y = y;
    p.acc = acc;
    p.M = M;
    p.N = N;
    p.err = env.err;
    // For M <= 128, "swap AB": weights fill the 128-row MMA operand and the
    // tokens the N side (a 128-row box; the tensor map reads zeros past M).
    p.swap = M <= kBM ? 1 : 0;
    Plan plan = choose_plan(dev, M, N, K, env.sm_count, p.swap != 0, sk_ws != nullptr);
    if (plan.sk && sk_ws_bytes < sk_bytes(plan)) plan = choose_plan(dev, M, N, K, env.sm_count, p.swap != 0, false);
    p.bn = plan.bn;
    p.split = plan.split;
    p.tiles_a = plan.tiles_a;
    p.tiles_b = plan.tiles_b;
    p.rows_a = p.swap ? N : M;
    p.rows_b = p.swap ? M : N;
    p.tmem_cols = pow2_cols(2 * p.bn);  // two fp32 chunk buffers
    p.sk_flag_target = kEpiWarps * 32;
    p.sk_wait_ns = kWaitLimitNs;
    if (debug_sk_timeout()) {
        // test hook: finishers wait for a flag value no unit ever writes,
        // with a short limit, so that the bounded wait runs out
        p.sk_flag_target = 0xffffffffu;
        p.sk_wait_ns = 1000000ull;
    }
    if (plan.sk) {
        // flags first (zeroed by the launch before this one), then the
        // partial tiles
        p.sk = 1;
        p.sk_units = plan.units;
        p.sk_flags = static_cast<unsigned*>(sk_ws);
        p.sk_part = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(sk_ws) + (sk_flag_count(plan) * 4 + 255) / 256 * 256);
    }
    const int wgt_box = p.swap ? kBM : (plan.pair ? p.bn / 2 : p.bn);
    CUtensorMap map_tok, map_wgt;
    if (!make_map_f16(&map_tok, x16, M, K) || !make_map_i8(&map_wgt, qw, N, K, wgt_box)) return cudaErrorInvalidValue;
    // pairs and split-K run clusters; otherwise one CTA per SM, persistent
    const int csize = plan.pair ? 2 : plan.split;
    const int64_t grid = plan.units * csize;
    const dim3 cluster = csize > 1 ? dim3((unsigned)csize, 1, 1) : kNoCluster;
    return with_cfg(p.bn, plan.pair, [&](auto w, auto pr) {
        constexpr int BN = decltype(w)::value;
        constexpr bool PAIR = decltype(pr)::value;
        return launch_kernel(w8a8_fused_kernel<BN, PAIR>, dim3((unsigned)grid), dim3(kThreads),
                             FusedCfg<BN, PAIR>::kSmemBytes, env.stream, cluster, map_tok, map_wgt, p);
    });
}

}  // namespace i8ql
