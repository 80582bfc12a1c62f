/*
 * i8ql -- int8 quantized linear layers on GB300 (sm_103a).
 *
 * C ABI of libi8ql.so.  Five operations make up the quantized linear layer
 * of LLM serving: per-output-channel weight quantization, per-token
 * activation quantization, the W8A8 GEMM with its scale/bias epilogue, the
 * weight-only W8A16 GEMM/GEMV, and the grouped W8A16 GEMM over MoE experts.
 * Beside them: the fused W8A8 linear layer, FP8 E4M3 W8A8, and the calls
 * declared after those.
 *
 * Conventions shared by every call:
 *  - Every pointer is a DEVICE pointer to a buffer the caller owns, allocates
 *    and frees.  The library keeps no copy of any weight or activation.
 *  - Matrices are dense row-major with no padding: an [R, K] matrix stores
 *    element (r, k) at r * K + k.  bf16 values are passed as their raw
 *    16-bit patterns (i8ql_bf16).  Matrix base pointers must be 16-byte
 *    aligned; scale and offset arrays 4-byte aligned; bias 2-byte aligned.
 *  - K must be a positive multiple of 16 and at most I8QL_MAX_K.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Calls only enqueue work: they return before the GPU finishes
 *    and never synchronise the host.
 *  - Errors are returned, never thrown or trapped.  Argument errors are
 *    found on the host before anything is launched.  Faults seen by a
 *    running kernel (a bounded wait that gave up, bad group offsets) are
 *    recorded in a per-device sticky word, read by i8ql_get_device_error.
 *  - A call with an empty problem (M = 0 or T_total = 0) returns I8QL_OK and
 *    launches nothing.
 *  - Inputs must be finite; NaN or Inf inputs give unspecified codes.
 */
#ifndef I8QL_H
#define I8QL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t i8ql_bf16; /* raw bfloat16 bits */
typedef int32_t i8ql_status;

enum {
    I8QL_OK = 0,
    I8QL_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misaligned pointer  */
    I8QL_ERR_UNSUPPORTED = 2,  /* K not a multiple of 16, K > I8QL_MAX_K, size too large */
    I8QL_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed          */
    I8QL_ERR_TIMEOUT = 4,      /* a kernel's bounded wait gave up (sticky word)        */
    I8QL_ERR_BAD_OFFSETS = 5,  /* grouped offsets not 0 .. T_total, non-decreasing     */
    I8QL_ERR_NO_DEVICE = 6,    /* no CUDA device, or not an sm_103 device              */
    I8QL_ERR_WORKSPACE_LIMIT = 7 /* w8a8_gemm_noalloc: problem exceeds its fixed array  */
};

/* Largest K whose worst-case int8 dot product fits int32:
 * floor((2^31 - 1) / 127^2) = 133,144. */
#define I8QL_MAX_K 133144

/* W8A8 with at most this many tokens runs on the decode kernel (int8
 * mma.sync, weight streaming); larger M runs on the tcgen05 tensor-core
 * kernel.  Measured crossover on GB300: at M = 48 and 64 the tensor-core
 * kernel takes half the time (Qwen3-8B gate_up at M = 64: 60 against
 * 123 us); at M <= 32 the decode kernel is as fast or faster on most
 * shapes. */
#define I8QL_W8A8_DECODE_MAX_M 32

/*
 * Per-output-channel symmetric int8 weight quantization.
 *
 * Source: "Phase 5a: int8 weight-only quantization", Summary (self-computed
 * per-output-channel int8 weights; float32 scale arithmetic; a zero-channel
 * guard that touches only all-zero channels) and "Day 6 -- Quantize It
 * Yourself", The mechanism, blocks 1 and 4 (q = clamp(round(w / s)),
 * s = absmax / qmax, round-to-nearest).
 *
 * For every row n of w (bf16 [N, K], one row per output channel):
 *   a = max_k |w[n,k]|;  scale[n] = a / 127 (fp32 IEEE division), or 1 if a == 0;
 *   q[n,k] = clamp(rint(w[n,k] / scale[n]), -127, 127), ties to even,
 *            one IEEE fp32 division per element, no flush of subnormals.
 * Outputs: q int8 [N, K], scale fp32 [N].  N >= 0.
 */
i8ql_status quantize_weight_per_channel_int8(const i8ql_bf16* w, int64_t N, int64_t K,
                                             int8_t* q, float* scale, void* stream);

/*
 * Dynamic symmetric per-token int8 activation quantization.
 *
 * Source: "feat(quantization): support compressed-tensors W8A8 and mixed
 * modules", Design and Supported Execution Scheme (dynamic symmetric INT8
 * per-token input activations) and "Day 6 -- Quantize It Yourself", The
 * mechanism, block 5 (per-token dynamic scales computed on the fly).
 *
 * The same arithmetic as quantize_weight_per_channel_int8, applied to each
 * token row m of x (bf16 [M, K]).  Outputs: q int8 [M, K], scale fp32 [M].
 */
i8ql_status quantize_act_per_token_int8(const i8ql_bf16* x, int64_t M, int64_t K,
                                        int8_t* q, float* scale, void* stream);

/*
 * W8A8 GEMM: int8 x int8 -> exact int32, then the scale/bias epilogue.
 *
 * Source: "feat(quantization): support compressed-tensors W8A8 and mixed
 * modules", Design and Supported Execution Scheme (static per-channel int8
 * weights, dynamic per-token int8 activations, no output quantization) and
 * "Day 6 -- Quantize It Yourself", The mechanism, block 5 (W8A8 runs the GEMM
 * on 8-bit operands).
 *
 *   acc[m,n] = sum_k qx[m,k] * qw[n,k]                      (exact int32)
 *   y[m,n]   = bf16_rne(((float)acc[m,n] * sx[m]) * sw[n] (+ (float)bias[n]))
 * Inputs: qx int8 [M, K], sx fp32 [M], qw int8 [N, K] (both K-contiguous),
 * sw fp32 [N], bias bf16 [N] or NULL.  Outputs: y bf16 [M, N]; acc_debug
 * int32 [M, N] or NULL (when given, receives the exact accumulator).
 * The epilogue may fuse multiply-adds: y is within one bf16 ulp of the
 * value above.  For M > I8QL_W8A8_DECODE_MAX_M (32) the call takes a temporary stream-ordered
 * workspace (cudaMallocAsync / cudaFreeAsync on `stream`): the fp16 codes of
 * the tokens, 2*M*K bytes, plus, when the plan runs stream-K (see
 * i8ql_w8a8_plan), one int32 partial tile of 128 x 256 per CTA pair half
 * (128 KiB per CTA, about 19 MiB on 152 SMs) and a flag per CTA.
 * Stream-K hands partial tiles from lower-numbered CTA pairs to higher ones:
 * a pair waits only for pairs dispatched before it, which park their part
 * before they wait for anything.  Its grid is sized to the pairs that fit on
 * the device at once; it relies on the hardware dispatching a grid's CTAs in
 * order (a later pair is never resident while an earlier one waits to be
 * scheduled).  A wait that still runs out (1 s) records I8QL_ERR_TIMEOUT and
 * leaves the tile unstored.
 */
i8ql_status w8a8_gemm(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw,
                      const i8ql_bf16* bias, i8ql_bf16* y, int32_t* acc_debug,
                      int64_t M, int64_t N, int64_t K, void* stream);

/*
 * W8A8 linear layer from bf16 activations: per-token activation
 * quantization fused into the W8A8 GEMM.
 *
 * Source: "feat(quantization): support compressed-tensors W8A8 and mixed
 * modules", Design and Supported Execution Scheme (activations quantized per
 * token, dynamically, at run time, feeding the int8 GEMM with the static
 * per-channel weights) and "Day 6 -- Quantize It Yourself", The mechanism,
 * block 5 (the per-forward activation quantization of W8A8).
 *
 * Computes exactly what quantize_act_per_token_int8(x) followed by w8a8_gemm
 * computes (same codes, scales, accumulators and outputs), in fewer passes
 * over memory: for M > 32 the quantization pass writes the codes in the form
 * the tensor-core GEMM reads, so the GEMM needs no separate conversion pass;
 * for M <= 8 with a weight whose decode GEMM is one wave without split-K
 * (large N, up to about 600 row blocks of 32) it is w8a8_linear_fused (one
 * launch); otherwise a quantization launch and the GEMM
 * (i8ql_w8a8_linear_launches reports which).
 * Inputs: x bf16 [M, K], qw int8 [N, K], sw fp32 [N], bias bf16 [N] or NULL.
 * Outputs: y bf16 [M, N]; qx int8 [M, K] and sx fp32 [M] receive the token
 * codes and scales when given (each may be NULL); acc_debug int32 [M, N] or
 * NULL.  Takes a temporary stream-ordered workspace (at most 2*M*K + 4*M
 * bytes, plus the stream-K workspace of w8a8_gemm when the plan runs
 * stream-K; none in the one-launch case).  Errors and argument rules as
 * w8a8_gemm, with x checked like y.
 */
i8ql_status w8a8_linear(const i8ql_bf16* x, const int8_t* qw, const float* sw, const i8ql_bf16* bias,
                        i8ql_bf16* y, int8_t* qx, float* sx, int32_t* acc_debug,
                        int64_t M, int64_t N, int64_t K, void* stream);

/*
 * The W8A8 linear layer from bf16 activations in ONE launch, for up to 8
 * tokens: the per-token activation quantization runs inside the decode
 * GEMM itself (its prologue and its token loads), not as a separate pass.
 *
 * Source: "Day 6 -- Quantize It Yourself", "Some interesting facts I
 * recently learned", item 2 (per-token activation quantization is extra work
 * in every forward pass) and The mechanism, block 5.
 *
 * Computes exactly what w8a8_linear computes (the same codes, scales,
 * accumulators and outputs, bit for bit; same arguments).  The CTAs that
 * split one row block's k range share each token's absmax through
 * distributed shared memory, then form the int8 codes from the bf16 tokens
 * in their main loop.  No workspace.  M > 8 returns I8QL_ERR_UNSUPPORTED.
 * Measured on GB300 it is faster than a quantization launch plus the GEMM
 * when the GEMM runs unsplit (Qwen3-4B gate_up at M <= 8: 14.7 against
 * 16.0 us), and slower on split-K shapes, where the cluster's absmax
 * exchange sits in front of the token loads (qkv: 9.1 against 8.3 us), and
 * beyond one wave of CTAs; w8a8_linear takes it in the first case.
 */
i8ql_status w8a8_linear_fused(const i8ql_bf16* x, const int8_t* qw, const float* sw, const i8ql_bf16* bias,
                              i8ql_bf16* y, int8_t* qx, float* sx, int32_t* acc_debug, int64_t M, int64_t N, int64_t K,
                              void* stream);

/*
 * Weight-only W8A16 GEMM / GEMV (decode).
 *
 * Source: "Day 6 -- Quantize It Yourself", The mechanism, block 5 (int8
 * weights dequantized inside the kernel, the product on bf16 math: a
 * memory-bandwidth win) and "Phase 5a: int8 weight-only quantization",
 * Summary (weight-only quantization saves memory bandwidth, not FLOPs).
 *
 *   y[m,n] = bf16_rne(sw[n] * sum_k q[n,k] * x[m,k])
 * with bf16 x [M, K], int8 qw [N, K], fp32 sw [N]; y bf16 [M, N].  The codes
 * enter the bf16 product exactly and the fp32 scale is applied once per
 * output, so s * q is never rounded to bf16.  Accumulation is fp32.  Any M
 * is accepted; the kernels are built for M <= 64.
 */
i8ql_status w8a16_gemm(const i8ql_bf16* x, const int8_t* qw, const float* sw, i8ql_bf16* y,
                       int64_t M, int64_t N, int64_t K, void* stream);

/*
 * Grouped W8A16 over MoE experts.
 *
 * Source: "Phase 5a: int8 weight-only quantization", Summary (a grouped
 * GEMM over MoE experts on stacked [E, N, K] expert weights with
 * per-output-channel int8 scales).
 *
 * Rows offsets[e] .. offsets[e+1]-1 of x (bf16 [T_total, K], grouped by
 * expert) go through expert e:
 *   y[r,n] = bf16_rne(sw[e,n] * sum_k qw[e,n,k] * x[r,k]).
 * offsets: int32 [E + 1] in DEVICE memory, offsets[0] = 0, non-decreasing,
 * offsets[E] = T_total; the host never reads it.  An expert with no rows
 * reads none of its weights (with T_total <= E / 2 and E <= 256 its CTAs are
 * not even launched: one expert slot per row, each finding its expert in
 * the offsets).  If the offsets break these rules the kernel skips the bad
 * experts (and, in the per-row slot form, any expert with rows beyond the
 * first T_total found from the last) and records I8QL_ERR_BAD_OFFSETS in the
 * sticky word.
 * qw int8 [E, N, K], sw fp32 [E, N], y bf16 [T_total, N].  E >= 1.
 */
i8ql_status grouped_w8a16_gemm(const i8ql_bf16* x, const int32_t* offsets, int64_t E,
                               const int8_t* qw, const float* sw, i8ql_bf16* y,
                               int64_t T_total, int64_t N, int64_t K, void* stream);

/*
 * FP8 E4M3 per-row quantization (weights per output channel, activations per
 * token; the two entry points run the same arithmetic on different rows).
 *
 * Source: "Day 6 -- Quantize It Yourself", The mechanism, block 2 (E4M3: sign,
 * 4 exponent and 3 mantissa bits, largest value 448), block 1 (q =
 * clamp(round(w / s)), s = absmax / largest representable value) and block 5
 * with its FP8_DYNAMIC recipe (per-channel weights, dynamic per-token
 * activations).
 *
 * For every row r of src (bf16 [R, K]):
 *   a = max_k |src[r,k]|;  scale[r] = a / 448 (fp32 IEEE division), or 1 if a == 0;
 *   q[r,k] = E4M3 code of (src[r,k] / scale[r]) (one IEEE fp32 division),
 *            rounded to nearest with ties to the even code, saturated at
 *            +-448, the sign of a value that rounds to zero kept.
 * Code layout: bits s eeee mmm, exponent bias 7, no infinities (0x7f and
 * 0xff are NaN and never produced).  Outputs: q uint8 [R, K], scale fp32 [R].
 */
i8ql_status quantize_weight_per_channel_fp8(const i8ql_bf16* w, int64_t N, int64_t K,
                                            uint8_t* q, float* scale, void* stream);
i8ql_status quantize_act_per_token_fp8(const i8ql_bf16* x, int64_t M, int64_t K,
                                       uint8_t* q, float* scale, void* stream);

/*
 * FP8 E4M3 W8A8 GEMM on the tensor cores.
 *
 * Source: "Day 6 -- Quantize It Yourself", The mechanism, block 5 (W8A8 with
 * fp8 operands runs the GEMM on 8-bit tensor cores) and block 2 (E4M3).
 *
 *   acc[m,n] = sum_k e4m3(qx[m,k]) * e4m3(qw[n,k])      (fp32 accumulation)
 *   y[m,n]   = bf16_rne((acc[m,n] * sx[m]) * sw[n] (+ (float)bias[n]))
 * Inputs: qx uint8 [M, K] and qw uint8 [N, K] E4M3 codes (K-contiguous),
 * sx fp32 [M], sw fp32 [N], bias bf16 [N] or NULL.  Output y bf16 [M, N].
 * Every product of two E4M3 values is exact in fp32; the sum is accumulated
 * in fp32 by the tensor core (with split-K, see i8ql_fp8_plan, as the sum of
 * the CTAs' fp32 partial sums in a fixed order), so y differs from the exact
 * value by fp32 accumulation rounding and one bf16 rounding.  No workspace.
 * Argument rules and errors as w8a8_gemm.
 */
i8ql_status w8a8_fp8_gemm(const uint8_t* qx, const float* sx, const uint8_t* qw, const float* sw,
                          const i8ql_bf16* bias, i8ql_bf16* y, int64_t M, int64_t N, int64_t K, void* stream);

/*
 * FP8 W8A8 linear layer from bf16 activations: quantize_act_per_token_fp8
 * then w8a8_fp8_gemm in one call (bit-identical to the two calls).
 *
 * Source: "Day 6 -- Quantize It Yourself", The mechanism, block 5 (the
 * per-token activation quantization of W8A8 at run time).
 *
 * Inputs: x bf16 [M, K], qw uint8 [N, K], sw fp32 [N], bias bf16 [N] or NULL.
 * Outputs: y bf16 [M, N]; qx uint8 [M, K] and sx fp32 [M] receive the token
 * codes and scales when given (each may be NULL).  Takes a temporary
 * stream-ordered workspace (cudaMallocAsync / cudaFreeAsync on `stream`) for
 * the codes and scales the caller does not keep: at most M*K + 4*M bytes.
 */
i8ql_status w8a8_fp8_linear(const i8ql_bf16* x, const uint8_t* qw, const float* sw, const i8ql_bf16* bias,
                            i8ql_bf16* y, uint8_t* qx, float* sx, int64_t M, int64_t N, int64_t K,
                            void* stream);

/*
 * Group-128 int4 weight quantization (W4A16-g128).
 *
 * Source: "Day 6 -- Quantize It Yourself", The mechanism, block 1 (a
 * W4A16-g128 tensor is int4 codes plus one bf16 scale per 128 weights along
 * the input dimension; q = clamp(round(w / s)), s = absmax(group) / largest
 * code).
 *
 * For every row n of w (bf16 [N, K]) and group g (k = 128g .. 128g+127):
 *   a = max |w[n,k]|;  scale[n,g] = bf16_rne(a / 7) (fp32 IEEE division),
 *                      or 1 if a == 0;
 *   q[n,k] = clamp(rint(w[n,k] / scale[n,g]), -7, 7) with one IEEE fp32
 *            division by the stored (bf16) scale, ties to even.
 * Outputs: q uint8 [N, K/2], two codes per byte (even k in the low nibble,
 * 4-bit two's complement); scale bf16 [N, K/128].  K must be a multiple of
 * 128 (else I8QL_ERR_UNSUPPORTED).  q 16-byte and scale 2-byte aligned.  A
 * nonzero group whose absmax is below about 2^-131 (its scale rounds to zero
 * in bf16) is outside the contract.
 */
i8ql_status quantize_weight_w4_g128(const i8ql_bf16* w, int64_t N, int64_t K, uint8_t* q, i8ql_bf16* scale,
                                    void* stream);

/*
 * Weight-only W4A16 GEMM / GEMV with group-128 scales (decode).
 *
 * Source: "Day 6 -- Quantize It Yourself", The mechanism, block 5 (W4A16:
 * int4 weights dequantized inside the kernel, the product on bf16 math; a
 * pure memory-bandwidth win) and block 1 (group-128 scales).
 *
 *   y[m,n] = bf16_rne(sum_g scale[n,g] * sum_{k in g} q[n,k] * x[m,k])
 * with bf16 x [M, K], q and scale as quantize_weight_w4_g128 writes them,
 * y bf16 [M, N].  The codes enter the bf16 product exactly; each group's
 * sum is accumulated in fp32 and scaled in fp32, so s * q is never rounded.
 * K % 128 == 0.  Any M is accepted; the kernels are built for M <= 64.
 */
i8ql_status w4a16_gemm(const i8ql_bf16* x, const uint8_t* q, const i8ql_bf16* scale, i8ql_bf16* y,
                       int64_t M, int64_t N, int64_t K, void* stream);

/*
 * MoE routing of T tokens on the device (the layer around the grouped GEMM).
 *
 * Source: "Phase 5a: int8 weight-only quantization", Summary (the grouped
 * int8 GEMM serves the MoE layer of deepseek-moe-16b), with that layer's
 * routing as its benchmark configuration states it: softmax over the gate
 * logits, top-k routed experts per token, plus shared experts that see every
 * token.
 *
 * Inputs: logits fp32 [T, E] (finite).  For every token t the top_k experts
 * of largest logit are chosen (equal logits: the lower expert index first;
 * the softmax is increasing in the logit), in decreasing order.  Outputs
 * (S = top_k + n_shared slots per token, T * S grouped rows):
 *   offsets int32 [E + n_shared + 1]: rows of expert e are offsets[e] ..
 *     offsets[e+1]-1 (routed experts 0 .. E-1, then the shared experts),
 *     tokens in increasing order within an expert;
 *   row_token int32 [T * S]: the token of each grouped row;
 *   token_row int32 [T, S]: the grouped row of each (token, slot), routed
 *     slots first in decreasing logit order, then the shared experts;
 *   slot_weight fp32 [T, S]: softmax probability (over all E experts, not
 *     renormalised over the chosen ones) of each routed slot, 1 for shared.
 * Limits: E <= 256, n_shared <= 64, T <= 65535 and 8 * E * ceil(T / 32) <=
 * 200 KiB (one CTA), else I8QL_ERR_UNSUPPORTED.  T = 0 writes zero offsets.
 */
i8ql_status moe_route_topk(const float* logits, int64_t T, int64_t E, int64_t top_k, int64_t n_shared,
                           int32_t* offsets, int32_t* row_token, int32_t* token_row, float* slot_weight,
                           void* stream);

/*
 * Grouped W8A16 of a fused gate/up projection with the SiLU-gated product in
 * its epilogue: the expert MLP's first half.
 *
 * Source: "Phase 5a: int8 weight-only quantization", Summary (grouped GEMM
 * over stacked [E, N, K] expert weights with per-output-channel scales) and
 * "feat(quantization): support compressed-tensors W8A8 and mixed modules",
 * Summary (fused gate/up projections).
 *
 * Expert e's weights qw[e] (int8 [2I, K], gate rows 0 .. I-1, up rows
 * I .. 2I-1) and scales sw[e] (fp32 [2I]) act on grouped rows offsets[e] ..
 * offsets[e+1]-1, row r reading token row_token[r] of x (bf16 [*, K]; or row
 * r itself when row_token is NULL):
 *   g = sw[e,j] * sum_k qw[e,j,k] x[k],  u = sw[e,I+j] * sum_k qw[e,I+j,k] x[k]
 *   h[r,j] = bf16_rne(g / (1 + exp(-g)) * u)                     (fp32)
 * Output h bf16 [T_total, I].  Offsets rules and errors as
 * grouped_w8a16_gemm.
 */
i8ql_status grouped_w8a16_silu_mul(const i8ql_bf16* x, const int32_t* row_token, const int32_t* offsets, int64_t E,
                                   const int8_t* qw, const float* sw, i8ql_bf16* h, int64_t T_total, int64_t I,
                                   int64_t K, void* stream);

/*
 * Weighted combine of the experts' output rows into each token's output.
 *
 * Source: as moe_route_topk.
 *
 *   out[t,:] = bf16_rne(sum_s slot_weight[t,s] * yd[token_row[t,s], :])
 * slots in order, fp32 accumulation.  yd bf16 [rows, H], token_row int32 and
 * slot_weight fp32 [T, S], out bf16 [T, H].  H % 8 == 0, T <= 65535.
 */
i8ql_status moe_combine(const i8ql_bf16* yd, const int32_t* token_row, const float* slot_weight, i8ql_bf16* out,
                        int64_t T, int64_t S, int64_t H, void* stream);

/*
 * The MoE expert MLP with int8 weight-only experts, end to end: routing,
 * grouped gate/up with the SiLU-gated product (token rows gathered),
 * grouped down, combine.
 *
 * Source: "Phase 5a: int8 weight-only quantization", Summary (the grouped
 * int8 kernel inside MoE decode of deepseek-moe-16b).
 *
 * Inputs: x bf16 [T, H], logits fp32 [T, E_routed]; experts E = E_routed +
 * n_shared (routed first): qw_gate_up int8 [E, 2I, H] with sw_gate_up fp32
 * [E, 2I], qw_down int8 [E, H, I] with sw_down fp32 [E, H].  Output out bf16
 * [T, H].  Four kernels (five beyond 32 tokens, where the routing's token
 * selection is its own launch); the intermediates (routing arrays, h [T*S, I] and
 * the down outputs [T*S, H], bf16) live in a temporary stream-ordered
 * workspace (cudaMallocAsync / cudaFreeAsync on `stream`).  Limits as
 * moe_route_topk; H and I multiples of 16.
 */
i8ql_status moe_expert_mlp_w8a16(const i8ql_bf16* x, const float* logits, int64_t E_routed, int64_t top_k,
                                 int64_t n_shared, const int8_t* qw_gate_up, const float* sw_gate_up,
                                 const int8_t* qw_down, const float* sw_down, i8ql_bf16* out, int64_t T, int64_t H,
                                 int64_t I, void* stream);

/*
 * W8A8 GEMM that allocates nothing.
 *
 * No counterpart on the pages: this entry point exists for callers that
 * cannot allocate device memory while they run (code replayed from a CUDA
 * graph whose memory was fixed at capture, serving loops that forbid
 * allocator calls on the hot path, hosts that own every buffer).  It computes
 * exactly what w8a8_gemm computes, with the same arguments, layouts and
 * errors, but where w8a8_gemm takes a temporary workspace from the
 * stream-ordered allocator (for M > 32: the fp16 codes of the tokens,
 * 2 * M * K bytes, and a stream-K workspace when its plan uses one), this
 * one never runs stream-K (i8ql_w8a8_noalloc_plan) and uses a fixed array
 * compiled into the
 * library: I8QL_NOALLOC_MAX_ELEMENTS 16-bit elements (32 MiB), held by every
 * GPU that loads the library until the process exits.
 *
 *  - For M > 32, M * K must not exceed I8QL_NOALLOC_MAX_ELEMENTS, else
 *    the call returns I8QL_ERR_WORKSPACE_LIMIT and launches nothing.  For
 *    M <= 32 the computation needs no workspace and any size is accepted.
 *  - The first call on a device looks up the array's device address (once
 *    per device, with that device current); make that first call before any
 *    stream capture.
 *  - All calls share the array and it keeps the last call's contents (every
 *    byte a call reads is written by the same call first).  Calls whose work
 *    may overlap on the GPU, e.g. on two streams without ordering, race on
 *    the array: order them on one stream or serialise them.
 */
#define I8QL_NOALLOC_MAX_ELEMENTS (16 * 1024 * 1024)
i8ql_status w8a8_gemm_noalloc(const int8_t* qx, const float* sx, const int8_t* qw, const float* sw,
                              const i8ql_bf16* bias, i8ql_bf16* y, int32_t* acc_debug,
                              int64_t M, int64_t N, int64_t K, void* stream);

/*
 * Reports how w8a8_fp8_gemm would run a problem of this size on the current
 * device, without launching anything.
 *
 * No counterpart on the pages: a query for tests and profiling.  *tile_n is
 * the width (N side) of the output tiles (128 or 256), *split_k the number
 * of CTAs of a thread-block cluster that share one tile's k range (1: no
 * split; each CTA then walks tiles persistently), *cta_pair 1 when pairs of
 * CTAs on two SMs share 256-row tiles through one two-SM MMA.  Same argument
 * rules as w8a8_fp8_gemm; the outputs are HOST pointers.
 */
i8ql_status i8ql_fp8_plan(int64_t M, int64_t N, int64_t K, int32_t* tile_n, int32_t* split_k, int32_t* cta_pair);

/*
 * Reports how w8a8_gemm would run a problem of this size on the current
 * device, without launching anything.
 *
 * No counterpart on the pages: a query for tests and profiling.  For
 * M <= I8QL_W8A8_DECODE_MAX_M (the decode kernel) all outputs are 0.  Otherwise *tile_n is the
 * width (N side) of the output tiles of the tensor-core kernel (128, 160,
 * 192, 224 or 256; for M <= 128 the operands are swapped and the tokens fill
 * a 128-wide side), *split_k the number of CTAs of a thread-block cluster
 * that share one tile's k range (1: no split), and *cta_pair 1 when pairs of
 * CTAs on two SMs share 256-row tiles through one two-SM MMA (0: one CTA per
 * 128-row tile), 2 when such pairs also run stream-K: every pair takes an
 * equal share of all (tile, k-block) steps, and a tile cut between pairs is
 * finished by the pair holding its last k-block, which adds the earlier
 * pairs' exact int32 partial sums (w8a8_gemm and w8a8_linear only: the
 * stream-K workspace is part of their temporary allocation).  Same argument
 * rules as w8a8_gemm; the outputs are HOST pointers.
 */
i8ql_status i8ql_w8a8_plan(int64_t M, int64_t N, int64_t K, int32_t* tile_n, int32_t* split_k,
                           int32_t* cta_pair);

/*
 * The same report for w8a8_gemm_noalloc, which never runs stream-K (its
 * fixed array holds only the token codes): *cta_pair is 0 or 1.  No
 * counterpart on the pages: a query for tests and profiling.
 */
i8ql_status i8ql_w8a8_noalloc_plan(int64_t M, int64_t N, int64_t K, int32_t* tile_n, int32_t* split_k,
                                   int32_t* cta_pair);

/*
 * Reports how many kernels one w8a8_linear call of this size launches on
 * the current device, without launching anything: 0 for M == 0; 1 when the
 * per-token quantization runs inside the decode GEMM (M <= 8 and a weight
 * whose decode GEMM is one wave without split-K); 2 otherwise (the
 * quantization launch, then the GEMM).
 *
 * No counterpart on the pages: a query for tests and profiling.  Same
 * argument rules as w8a8_linear for M, N and K; *launches is a HOST pointer
 * (null: I8QL_ERR_INVALID_ARG).
 */
i8ql_status i8ql_w8a8_linear_launches(int64_t M, int64_t N, int64_t K, int32_t* launches);

/*
 * Waits for `stream`, then reads and clears the current device's sticky
 * kernel-error word.  Returns I8QL_OK, I8QL_ERR_TIMEOUT or
 * I8QL_ERR_BAD_OFFSETS (the first fault recorded since the last read), or
 * I8QL_ERR_CUDA if the wait itself failed.  No counterpart on the pages:
 * the failure signal of the kernels' bounded waits and offset checks.
 */
i8ql_status i8ql_get_device_error(void* stream);

/* Static, NUL-terminated description of a status code (no counterpart on
 * the pages; never NULL, "unknown status" for codes outside the enum). */
const char* i8ql_status_string(i8ql_status status);

/* Library version as major * 10000 + minor * 100 + patch (no counterpart
 * on the pages). */
int32_t i8ql_version(void);

/*
 * Test hook, no counterpart on the pages: exercises the timeout path of the
 * stream-K hand-over without faulting or hanging anything.  While `on` is
 * nonzero (process-wide), every stream-K finisher launched by w8a8_gemm or
 * w8a8_linear waits for a flag value that no CTA ever writes, with a 1 ms
 * limit instead of 1 s: the wait runs out, the CTA records I8QL_ERR_TIMEOUT
 * in the sticky word, leaves the tiles it finishes unstored and exits
 * cleanly (its other work, and every other CTA's, is unaffected).  Only
 * tests should call it; calls with it off behave exactly as before.
 */
void i8ql_debug_stream_k_timeout(int32_t on);

/*
 * Early weight loads for the decode GEMMs (serving option, no counterpart on
 * the pages).  Every kernel of this library waits for the kernel launched
 * before it on the same stream (programmatic dependent launch) before it
 * reads anything.  With `on` nonzero (process-wide; default off) the
 * decode-size GEMMs -- w8a16_gemm, w8a8_gemm and w8a8_linear with M <= 32,
 * w8a8_linear_fused; not the grouped ones, whose weight addresses depend on
 * device offsets -- instead load the first few k-steps of their weights
 * before that wait, so the weight stream starts while the previous kernel
 * drains; tokens, scales, bias and outputs still wait.  The caller promises
 * that the kernel launched immediately before such a call on its stream does
 * not write that call's weights (a weight quantization followed directly by
 * a GEMM on its output needs the option off, or any other kernel between
 * them).  Results are identical either way.
 */
void i8ql_set_early_weight_loads(int32_t on);
int32_t i8ql_early_weight_loads(void);

#ifdef __cplusplus
}
#endif

#endif /* I8QL_H */
