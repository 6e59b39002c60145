/*
 * moe.h -- C ABI of the GB300 (sm_103a) sparse MoE expert-layer forward.
 *
 * The forward pass of a sparse Mixture-of-Experts expert layer as served for
 * Qwen3-MoE and Hy3 models, split into the steps the serving pages name:
 *
 *   moe_gating_topk          top-k expert choice and routing weights
 *   moe_init_routing         stable sort of token-expert pairs by expert,
 *                            per-expert counts/offsets, permutation, row gather
 *   moe_grouped_gemm_swiglu  all experts' gate/up projections in one launch,
 *                            SwiGLU fused into the epilogue
 *   moe_grouped_gemm         all experts' down projections in one launch,
 *                            the routing weight fused into the epilogue
 *   moe_finalize_routing     unpermute + weighted sum (+ shared expert)
 *   moe_layer_forward        the whole path on one stream
 *
 * and around it: moe_add_rms_norm_cast / moe_add_rms_norm_mxfp8 and
 * moe_router_logits (the step before gating), moe_init_routing_range (routing
 * restricted to a local expert range), moe_prepack_w13 (one-time weight layout),
 * the 4-bit-weight decode GEMMs on f16 operands (moe_mxfp4_quantize,
 * moe_mxfp4_prepack, moe_gather_rows_f16, moe_grouped_gemm_swiglu_mxfp4,
 * moe_grouped_gemm_mxfp4) and the W4A8 path on the block-scaled MMA
 * (moe_w4a8_prepack, moe_gather_rows_mx, moe_grouped_gemm_swiglu_w4a8,
 * moe_grouped_gemm_w4a8, moe_layer_forward_w4a8).
 *
 * Sources (page titles and sections):
 *  [Q3]  "Qwen3-MoE low-latency inference practice on Atlas A3/950 clusters"
 *        (cann-recipes-infer), sections "MoE TP optimisation: computation
 *        decomposition" and "GMM enablement and routing optimisation".
 *        Also its W4A8 / EP sections (MXFP8 activation quantisation, MXFP4
 *        expert weights, expert-range routing) and "fused RMSNorm + Cast".
 *  [HY3] "Hy3 295B MoE end-to-end inference optimisation practice on Atlas A3"
 *        (cann-recipes-infer), sections 1.1-1.3, 5.1, 6.2, 8.1.
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or keeps device memory.  `stream` is a cudaStream_t
 *    (NULL = legacy default stream).  Every call only enqueues work on `stream`
 *    and returns without synchronising (except moe_get_device_status).
 *  - bf16 tensors are passed as uint16_t bit patterns; all matrices are dense
 *    row-major; every pointer must be 16-byte aligned.
 *  - Notation: T tokens, H hidden size, E routed experts, k experts per token,
 *    I expert intermediate size, P = T*k token-expert pairs, pair p = t*k + j
 *    (j = slot in the top-k order), pos = index in expert-sorted order.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns a negative moe_status and launches nothing.  A failed
 *    launch returns MOE_ERR_CUDA.  Problems seen on the device (a bounded
 *    pipeline wait that ran out, an index outside its buffer) never trap: the
 *    kernel skips the access, sets a bit in the sticky status word at the
 *    start of the workspace and finishes; read it with moe_get_device_status.
 *  - Limits: 1 <= k <= min(E, 32); 1 <= E <= 1024; H % 64 == 0; I % 64 == 0;
 *    T*k < 2^31; T*k*max(H, I) < 2^40.
 */
#ifndef MOE_GB300_MOE_H_
#define MOE_GB300_MOE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,   /* null pointer, bad size, misaligned pointer */
  MOE_ERR_UNSUPPORTED = -2,   /* valid but outside the limits above */
  MOE_ERR_WORKSPACE = -3,     /* workspace missing or smaller than *_workspace_size() */
  MOE_ERR_CUDA = -4,          /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = -5,       /* device status: a bounded wait ran out */
  MOE_ERR_DEVICE_CHECK = -6   /* device status: an index check failed, access skipped */
} moe_status;

/* Gate function.  Values follow norm_type of the Hy3 router call ([HY3] 1.3):
 * 0 = softmax, 1 = sigmoid. */
/* MOE_GATE_SIGMOID_INNER_BIAS: the fused routing op's placement of the correction bias, inside
 * the sigmoid ([HY3] 5.1, P1 precision note), where the model adds it after the sigmoid. */
typedef enum { MOE_GATE_SOFTMAX = 0, MOE_GATE_SIGMOID = 1, MOE_GATE_SIGMOID_INNER_BIAS = 2 } moe_gate;

/* Shape and gating parameters of one MoE layer. */
typedef struct moe_layer_desc {
  int32_t T;                    /* tokens */
  int32_t H;                    /* hidden size */
  int32_t E;                    /* routed experts */
  int32_t k;                    /* experts per token */
  int32_t I;                    /* routed expert intermediate size */
  int32_t gate;                 /* moe_gate */
  float routed_scaling_factor;  /* sigmoid only: weights are multiplied by it (Hy3: 2.826) */
  float eps;                    /* sigmoid only: added to the weight normaliser (Hy3: 1e-20) */
  int32_t n_shared;             /* 0 or 1 shared experts ([HY3] 1.1) */
  int32_t I_s;                  /* shared expert intermediate size (ignored if n_shared == 0) */
} moe_layer_desc;

/* Human-readable name of a moe_status value (static string). */
MOE_API const char* moe_status_string(int status);

/* ABI version (major * 100 + minor). */
MOE_API int moe_abi_version(void);

/* Bytes of workspace header holding the sticky device status word; every
 * workspace starts with it. */
MOE_API size_t moe_status_bytes(void);

/* Clears the sticky device status word of a workspace (async on `stream`).
 * Call once after allocating a workspace, and after handling an error. */
MOE_API int moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Failure injection, for testing the bounded waits (process-wide, not thread-safe; set it back to
 * 0 afterwards).  what = 1: the limit, in ns, of every wait inside the grouped GEMMs (0: the
 * default, 2 s).  what = 2: value != 0 makes the gate/up GEMM's in-kernel row gather (taken by
 * compute-bound problems inside moe_layer_forward) write nothing and set none of its flags, so its
 * producers wait for flags that nothing sets: after the limit the kernel records MOE_ERR_TIMEOUT in
 * the workspace status, every CTA leaves its loops, waits for nothing in flight, frees its tensor
 * memory and returns; the rest of the layer runs on whatever act then holds.  Unknown `what` ->
 * MOE_ERR_INVALID_ARG.  The pages have no counterpart.
 */
MOE_API int moe_debug_set(int what, unsigned long long value);

/* Synchronises `stream`, then reads the sticky status word of `ws`.
 * Returns MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_CHECK (or MOE_ERR_CUDA). */
MOE_API int moe_get_device_status(const void* ws, void* stream);

/*
 * Front end (the step before a1).  [Q3] "fused RMSNorm + Cast": the norm before the MoE gives
 * the hidden state in FP32 for the gate and in BF16 for the experts, and one op does the
 * residual add, the RMSNorm and the casts; without a residual (first layer) it is RMSNorm +
 * cast.  The FP32 output feeds moe_router_logits, the BF16 one the experts (x of
 * moe_layer_forward).
 *
 *  hidden        [T,H] bf16 in.
 *  residual      [T,H] bf16 in, or NULL (no add: the residual stream is `hidden`).
 *  norm_weight   [H] bf16.
 *  eps           variance epsilon (>= 0).
 *  y_fp32        [T,H] fp32 out: r * rsqrt(mean_h(r^2) + eps) * norm_weight, with
 *                r = bf16(hidden + residual) (rounded once) or hidden; fp32 arithmetic.
 *  y_bf16        [T,H] bf16 out (NULL: not written): y_fp32 rounded to nearest even.
 *  residual_out  [T,H] bf16 out: r, the residual stream for the next layer; required when
 *                residual is given, optional (NULL) otherwise.  May alias `residual`.
 *  Constraints: H % 64 == 0, H <= 8192 (one token row is held in registers), 16-byte aligned
 *  pointers.  Errors as everywhere: negative status, nothing launched.
 */
MOE_API int moe_add_rms_norm_cast(const uint16_t* hidden, const uint16_t* residual, const uint16_t* norm_weight,
                                  int T, int H, float eps, float* y_fp32, uint16_t* y_bf16, uint16_t* residual_out,
                                  void* stream);

/*
 * Front end of the W4A8 path: fused residual add + RMSNorm + MXFP8 dynamic quantisation ([Q3]
 * W4A8 section: add_rms_norm_dynamic_mx_quant, round_mode 'rint', dst_type float8_e4m3fn; without
 * a residual, rms_norm_dynamic_mx_quant).  The normalised row y (fp32, as moe_add_rms_norm_cast
 * computes it) is cut into blocks of 32 consecutive elements; a block's scale is
 * X = 2^(floor(log2 max|y|) - 8) (8: the largest E4M3 exponent), stored as an E8M0 byte
 * (exponent + 127, clamped to [-127, 127]; an all-zero block gets 0); each element y / X is
 * rounded to E4M3 (the "fn" variant: no infinities), nearest even, saturating at +-448.
 *
 *  y_fp8         [T,H] uint8 out: E4M3 codes.
 *  y_scale       [T,H/32] uint8 out: E8M0 scale bytes (no alignment requirement).
 *  y_fp32        [T,H] fp32 out, or NULL: the unquantised y (e.g. for the gate GEMM).
 *  others        as moe_add_rms_norm_cast; same constraints (H % 64 == 0, H <= 8192).
 */
MOE_API int moe_add_rms_norm_mxfp8(const uint16_t* hidden, const uint16_t* residual, const uint16_t* norm_weight,
                                   int T, int H, float eps, uint8_t* y_fp8, uint8_t* y_scale, float* y_fp32,
                                   uint16_t* residual_out, void* stream);

/*
 * Router gate GEMM (the step before a1): router_logits = y_fp32 . w_gate^T in fp32 ([Q3] "fused
 * RMSNorm + Cast": the gate is computed from the FP32 hidden state).  Runs on the FP32 pipes:
 * the tensor-core bf16/tf32 paths would round the fp32 input.
 *
 *  y_fp32  [T,H] fp32 (moe_add_rms_norm_cast's FP32 output).
 *  w_gate  [E,H] bf16 gate weight ([out_features, in_features]), widened exactly.
 *  logits  [T,E] fp32 out.  H is cut into S slices (S chosen from T, H, E and the SM count);
 *          each slice is summed in ascending h with fp32 FMA and the slices are added in order,
 *          so the result is the same on every run.
 *  ws      at least moe_router_logits_workspace_size(T, H, E) bytes (the slices' partial sums).
 *  Constraints: H % 64 == 0, E <= 1024, 16-byte aligned pointers.
 */
MOE_API size_t moe_router_logits_workspace_size(int T, int H, int E);
MOE_API int moe_router_logits(const float* y_fp32, const uint16_t* w_gate, int T, int H, int E, float* logits,
                              void* ws, size_t ws_bytes, void* stream);

/*
 * a1. Gating top-k.  [Q3] "GMM enablement and routing optimisation" (one fused
 * op replaces top-k followed by softmax); [HY3] 1.3 (sigmoid router with
 * correction bias, norm_type=1, routed_scaling_factor, eps) and 5.1 (the bias
 * is added after the sigmoid and only changes which experts are chosen).
 *
 *  logits   [T,E] fp32 router logits.
 *  bias     [E] fp32 correction bias, sigmoid gates only; NULL = none.  Must be
 *           NULL for softmax.
 *  gate     moe_gate.  Selection key: softmax -> the logit; sigmoid ->
 *           sigmoid(logit) + bias[e] (the model's placement, [HY3] 5.1);
 *           sigmoid_inner_bias -> sigmoid(logit + bias[e]) (the fused op's
 *           placement, [HY3] 5.1 P1 note; the fp32 sum rounded once).  The
 *           sigmoid is a fixed sequence of IEEE fp32 operations so the choice
 *           is reproducible bit for bit.  Ties go to the lower expert index.
 *  topk_idx [T,k] int32 out: chosen experts, best first.
 *  topk_w   [T,k] fp32 out: softmax -> softmax of the k chosen logits;
 *           sigmoid -> s_j / (sum_j s_j + eps) * routed_scaling_factor with
 *           s_j = sigmoid(logit_j) (sigmoid) or sigmoid(logit_j + bias_j)
 *           (sigmoid_inner_bias).
 */
MOE_API int moe_gating_topk(const float* logits, const float* bias, int T, int E, int k, int gate,
                    float routed_scaling_factor, float eps, float* topk_w, int32_t* topk_idx, void* stream);

/*
 * a2. Init-routing.  [Q3] "GMM enablement and routing optimisation"
 * (init-routing gives the expert sort order; compute-expert-tokens gives the
 * number of tokens per expert); [HY3] 6.2 (group_list = per-expert counts).
 *
 *  topk_idx    [T,k] int32 in, values in [0,E).
 *  counts      [E] int32 out: pairs routed to each expert.
 *  offsets     [E+1] int32 out: exclusive prefix sum of counts, offsets[E] = P.
 *  sorted_pair [P] int32 out: pos -> p; expert-major, ascending p inside an expert.
 *  pair_pos    [P] int32 out: p -> pos (inverse permutation).
 *  x, x_exp    optional (both NULL or both set): x [T,H] bf16 in,
 *              x_exp [P,H] bf16 out, x_exp[pos] = x[sorted_pair[pos] / k].
 *  ws          workspace of at least moe_init_routing_workspace_size(T,E,k) bytes.
 * Indices outside [0,E) are counted nowhere, flagged as MOE_ERR_DEVICE_CHECK
 * in the status word, and leave the outputs unspecified.
 */
MOE_API size_t moe_init_routing_workspace_size(int T, int E, int k);
MOE_API int moe_init_routing(const int32_t* topk_idx, int T, int E, int k, const uint16_t* x, int H, uint16_t* x_exp,
                     int32_t* counts, int32_t* offsets, int32_t* sorted_pair, int32_t* pair_pos, void* ws,
                     size_t ws_bytes, void* stream);

/*
 * Init-routing restricted to a local expert range [e0, e1), the expert-parallel
 * form of a2: [Q3] MoE EP with AllGather + ReduceScatter (W4A8 section) routes the
 * gathered tokens with init_routing_v2 keeping only the tokens of the experts in
 * this rank's range, runs the GMMs on those experts and finalises a partial sum
 * that a reduce-scatter adds up across ranks.  On one device: the partial outputs
 * of a partition of [0, E) into ranges sum to the whole layer's output.
 *
 *  e0, e1      0 <= e0 < e1 <= E; the local experts are l = e - e0, EL = e1 - e0.
 *  counts      [EL] int32 out: pairs routed to each local expert.
 *  offsets     [EL+1] int32 out: exclusive prefix of counts; offsets[EL] = the
 *              number of local pairs P_loc.
 *  sorted_pair [P] int32 out: positions 0..P_loc-1 hold the local pairs sorted by
 *              local expert, ascending pair index inside an expert; the rest is
 *              left alone.
 *  pair_pos    [P] int32 out: pair_pos[p] = its position, or -1 when the pair's
 *              expert is outside [e0, e1) (moe_finalize_routing skips those, which
 *              gives the range's partial output).
 *  x, x_exp    optional as for moe_init_routing; rows 0..P_loc-1 of x_exp are written.
 *  ws          moe_init_routing_workspace_size(T, E, k) bytes suffice.
 *  Expert indices outside [0, E) raise MOE_ERR_DEVICE_CHECK as in moe_init_routing.
 *  Feed the GEMMs the local slice: weights w + e0 * (rows per expert) * K, E = EL,
 *  these offsets, and M = P (rows past P_loc are never read).
 */
MOE_API int moe_init_routing_range(const int32_t* topk_idx, int T, int E, int k, int e0, int e1, const uint16_t* x,
                                   int H, uint16_t* x_exp, int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                                   int32_t* pair_pos, void* ws, size_t ws_bytes, void* stream);

/*
 * Init-routing without a workspace, for callers that cannot allocate device
 * memory (code running inside an allocator or memory-pool callback, runtimes
 * whose device memory is entirely pre-reserved by someone else, or host
 * threads that must not take the allocator's locks).  The pages have no
 * counterpart of this entry point: it is a deployment convenience.
 *
 * Same arguments, outputs and results as moe_init_routing, minus the
 * workspace.  Its scratch is a fixed 1 MiB device array inside the library
 * (held by every GPU that loads the library until the process exits), so the
 * problem must satisfy 2 * n_chunks * E * 4 <= 1 MiB, where n_chunks is the
 * number of pair chunks init-routing uses: ceil(T*k / 32) when T*k <= 4096,
 * else ceil(T*k / max(512, ceil(T*k/256) rounded up to 32)); never above 256,
 * and at most 128 when T*k <= 65536 -- so any E <= 512 fits at any T*k, and
 * E = 1024 fits for T*k <= 65536; larger problems return MOE_ERR_UNSUPPORTED
 * and launch nothing.  Out-of-range expert indices are
 * skipped without a status report.  The call allocates nothing.
 *  - Every call on a device shares the array.  Each call overwrites all the
 *    scratch it reads, so nothing has to be cleared between calls, but calls
 *    whose kernels may overlap on the GPU (different streams or threads) race.
 *  - The first call on a device resolves the array's device address with that
 *    device current; make it before any stream capture starts.
 */
MOE_API int moe_init_routing_static_scratch(const int32_t* topk_idx, int T, int E, int k, const uint16_t* x, int H,
                                            uint16_t* x_exp, int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                                            int32_t* pair_pos, void* stream);

/*
 * One-time weight layout for the gate/up GEMMs (the analogue of the pages'
 * process-weights-after-loading step, [HY3] 6.2): w13 [E,2I,H] with rows
 * [gate_proj; up_proj] per expert ([Q3] "MoE TP optimisation") is rewritten so
 * that every group of 32 rows holds 16 gate rows followed by the up rows of the
 * same 16 features: packed[e][32g + r] = w13[e][16g + r] (r < 16) and
 * w13[e][I + 16g + r - 16] (r >= 16).  Same size; not in place (w13 != packed).
 * The grouped gate/up GEMM and moe_layer_forward read this layout.
 */
MOE_API int moe_prepack_w13(const uint16_t* w13, int E, int I, int H, uint16_t* w13_packed, void* stream);

/*
 * a3. Grouped gate/up GEMM with fused SwiGLU.  [Q3] "MoE TP optimisation:
 * computation decomposition" (w13 = [gate_proj; up_proj]; SwiGLU splits the
 * last axis in two halves and returns SiLU(x[0]) * x[1]) and "GMM enablement"
 * (all experts in one grouped matmul, in the order init-routing gives).
 *
 *  x        row_src == NULL: [M,H] bf16 rows already in expert-sorted order (x_exp of
 *           moe_init_routing).  row_src != NULL: [T,H] bf16 token rows; row pos of the
 *           GEMM is x[row_src[pos] / k], gathered by the call itself (pass sorted_pair of
 *           moe_init_routing / moe_init_routing_range as row_src).
 *  row_src  [M] int32 device or NULL; only entries pos < offsets[E] are read, each must
 *           lie in [0, T*k): one outside is skipped (its row of act is unspecified) and
 *           raises MOE_ERR_DEVICE_CHECK in the workspace status word.
 *  k, T     experts per token and token rows of x; used only with row_src.
 *  w13      [E,2I,H] bf16 in the packed layout of moe_prepack_w13 (made from the
 *           checkpoint [out_features, in_features] rows [gate; up], [HY3] 6.2).
 *  offsets  [E+1] int32 device: expert e owns rows [offsets[e], offsets[e+1]);
 *           offsets[E] <= M.
 *  act      [M,I] bf16 out: act[pos] = SiLU(g) * u, (g, u) = row(pos) . w13[e]^T,
 *           accumulated in fp32, rounded once to bf16.  Rows >= offsets[E] untouched.
 *  ws       at least moe_grouped_gemm_swiglu_workspace_size(M, H, row_src != NULL)
 *           bytes: the status header, and with row_src the gathered rows (M*H*2 bytes)
 *           and one flag per 16 of them.
 *  The gather runs as moe_layer_forward runs it: inside the GEMM (two extra warps per
 *  CTA, overlapping the matmuls) when the problem takes the CTA-pair instances (more than
 *  32 rows per expert on average), else as a separate kernel before it.
 */
MOE_API size_t moe_grouped_gemm_workspace_size(void);
MOE_API size_t moe_grouped_gemm_swiglu_workspace_size(int M, int H, int gather);
MOE_API int moe_grouped_gemm_swiglu(const uint16_t* x, const int32_t* row_src, int k, int T, const uint16_t* w13,
                                    const int32_t* offsets, int E, int M, int H, int I, uint16_t* act, void* ws,
                                    size_t ws_bytes, void* stream);

/*
 * a4. Grouped GEMM (down projection) with the routing weight fused.  [Q3]
 * "MoE TP optimisation" (x = down(...)) and "GMM enablement"; [HY3] 6.2.
 *
 *  a           [M,K] bf16 rows in expert-sorted order (act of a3).
 *  w           [E,N,K] bf16 (down_proj, [out_features, in_features]).
 *  offsets     [E+1] int32 device, as in a3.
 *  topk_w, sorted_pair  optional (both NULL or both set): row pos is scaled by
 *              topk_w[sorted_pair[pos]] ([T,k] fp32 and [M] int32 from a1/a2).
 *  out         [M,N] bf16 out = scale * (a[pos] . w[e]^T), fp32 accumulation,
 *              rounded once.  Rows >= offsets[E] untouched.
 */
MOE_API int moe_grouped_gemm(const uint16_t* a, const uint16_t* w, const int32_t* offsets, const float* topk_w,
                     const int32_t* sorted_pair, int E, int M, int N, int K, uint16_t* out, void* ws,
                     size_t ws_bytes, void* stream);

/*
 * MXFP4 expert weights (decode): a3/a4 on 4-bit weights.  [Q3] MoE EP / W4A8
 * section (MXFP4 expert weights read by the grouped matmuls).  Format (OCP
 * microscaling): blocks of 32 consecutive elements along K share an E8M0 scale
 * byte s (2^(s - 127)); each element is an E2M1 code (sign bit 3, magnitude
 * index 0-7 of {0, 0.5, 1, 1.5, 2, 3, 4, 6} in bits 0-2), two per byte, element
 * 2j in the low nibble of byte j.  The 4-bit GEMMs compute on f16 operands:
 * token rows and act are f16 (saturated to +-65504), products accumulate in fp32.
 *
 * moe_mxfp4_quantize: w [rows,K] bf16 (K % 32 == 0) -> codes [rows,K/2] and
 *   scales [rows,K/32]: scale 2^(floor(log2 amax) - 2) (exponent clamped to
 *   [-127,127]; an all-zero block gets byte 0), element v / scale rounded to the
 *   E2M1 grid nearest-even, saturating at +-6.  w finite.
 *
 * moe_mxfp4_prepack: one-time layout for the GEMMs.  codes/scales of [E,n_out,K]
 *   weights (n_out % 128 == 0, K % 64 == 0) -> codes_p [E*n_out,K/2] (rows in the
 *   packed gate/up order of moe_prepack_w13 when gate_up, else unchanged),
 *   scales_p (E*n_out*K/32 bytes: per 128-row tile, K/32 lines of the tile's 128
 *   rows) holding each block's exponent relative to its row, and omega
 *   [E*n_out] fp32, the power of two the epilogue applies to the row: with
 *   W = (largest scale exponent of the row) - 13, omega = 2^W and a block of
 *   exponent X enters the f16 operand scaled by 2^(X - W) (exact for
 *   X - W >= -23, i.e. blocks within 36 binades of the row's largest; blocks
 *   below 2^-24 relative are dropped).  Scale byte 255 (NaN) unsupported.
 *   Not in place.
 *
 * moe_gather_rows_f16: x_rows16[pos] = f16(x[sorted_pair[pos] / k]) for pos < M
 *   (x [T,H] bf16, H % 64 == 0); an index outside [0,T*k) skips the row and
 *   raises MOE_ERR_DEVICE_CHECK in ws's status word.
 *
 * moe_grouped_gemm_swiglu_mxfp4: as moe_grouped_gemm_swiglu with x_rows16 [M,H]
 *   f16, the w13 weights prepacked with gate_up = 1 (n_out = 2I), and act16 [M,I]
 *   f16 out: act = SiLU(g) * u of (g, u) = x_rows16[pos] . dequant(w13[e])^T.
 * moe_grouped_gemm_mxfp4: as moe_grouped_gemm with a16 [M,K] f16 and the down
 *   weights [E,N,K] prepacked with gate_up = 0 (N % 128 == 0); out [M,N] bf16.
 * Both walk 32 token columns per tile: meant for decode (a few rows per expert);
 * correct for any M.  ws: at least moe_grouped_gemm_workspace_size() bytes.
 * Local expert range [e0, e1) (with moe_init_routing_range's offsets): pass
 * codes_p + e0*n_out*K/2, scales_p + e0*n_out*K/32, omega + e0*n_out and E = e1 - e0
 * (every expert owns whole 128-row tiles of the prepacked layout).
 */
MOE_API int moe_mxfp4_quantize(const uint16_t* w, long long rows, int K, uint8_t* codes, uint8_t* scales,
                               void* stream);
MOE_API int moe_mxfp4_prepack(const uint8_t* codes, const uint8_t* scales, int E, int n_out, int K, int gate_up,
                              uint8_t* codes_p, uint8_t* scales_p, float* omega, void* stream);
MOE_API int moe_gather_rows_f16(const uint16_t* x, const int32_t* sorted_pair, int T, int k, int H, int M,
                                uint16_t* x_rows16, void* ws, size_t ws_bytes, void* stream);
MOE_API int moe_grouped_gemm_swiglu_mxfp4(const uint16_t* x_rows16, const uint8_t* w13_codes,
                                          const uint8_t* w13_scales, const float* w13_omega, const int32_t* offsets,
                                          int E, int M, int H, int I, uint16_t* act16, void* ws, size_t ws_bytes,
                                          void* stream);
MOE_API int moe_grouped_gemm_mxfp4(const uint16_t* a16, const uint8_t* w_codes, const uint8_t* w_scales,
                                   const float* w_omega, const int32_t* offsets, const float* topk_w,
                                   const int32_t* sorted_pair, int E, int M, int N, int K, uint16_t* out, void* ws,
                                   size_t ws_bytes, void* stream);

/*
 * W4A8: MXFP8 activations x MXFP4 expert weights on the block-scaled tensor-core MMA
 * (tcgen05.mma kind::mxf8f6f4 with the E8M0 scale factors of both operands applied by the
 * hardware).  [Q3] MoE EP section, "computation decomposition (AllGather scheme, W4A8)": the hidden
 * state is quantised to MXFP8 (data + scale), routed, and the grouped matmuls run on it with MXFP4
 * expert weights; [HY3] 5.2: on the quantised path the SwiGLU is fused with a group quantisation, so
 * act enters the down projection as MXFP8 too.  Formats as above (MXFP8: E4M3 codes, E8M0 scale per
 * 32 along K, the rule of moe_add_rms_norm_mxfp8; MXFP4: the codes and scales moe_mxfp4_quantize
 * writes).  Products are exact; accumulation in fp32.
 *
 * Token-row scales inside this path are "padded scale rows": [rows, K/128, 16] bytes, per row and
 * 128-K chunk the chunk's four E8M0 scales followed by twelve zero bytes.
 *
 * moe_w4a8_prepack: one-time layout.  codes [E,n_out,K/2] and scales [E,n_out,K/32] of MXFP4
 *   weights -> codes_p [E*n_out/256][K/128][256][64] (per 256-row tile and 128-K chunk the 64 code
 *   bytes of the chunk for each of the tile's rows, so every block the GEMM loads is one contiguous
 *   16 KB; E*n_out*K/2 bytes) and sf_p [E*n_out/256][K/128][2][512] (E*n_out*K/32 bytes).
 *   gate_up = 1 (w13, n_out = 2I, I % 128 == 0): packed row R of an expert is the gate (R % 32 < 16)
 *   or up row of feature 128*(R/256) + 32*((R/32)%4) + 16*((R/128)%2) + R%16, so every 256-row tile
 *   holds 128 whole features.  gate_up = 0: rows unchanged.  n_out % 256 == 0.  sf_p: per 256-row
 *   tile, 128-K chunk and 128-row half a 512-byte atom, byte (r%32)*16 + (r/32)*4 + b = the scale of
 *   half row r, block b of the chunk.  K % 128 == 0.  Not in place.  Local expert range [e0, e1):
 *   codes_p + e0*n_out*K/2 and sf_p + e0*n_out*K/32.
 *
 * moe_gather_rows_mx: out_codes[pos] = x_codes[t], out_sf[pos] = the padded scale row of
 *   x_scales[t], t = sorted_pair[pos] / k, for pos < M (x_codes [T,H], x_scales [T,H/32]; H % 128
 *   == 0).  sorted_pair NULL: t = pos (M <= T), only out_sf written (out_codes may be NULL).  A
 *   pair index outside [0, T*k) skips its row and raises MOE_ERR_DEVICE_CHECK in ws's status word.
 *
 * moe_grouped_gemm_swiglu_w4a8: act = SiLU(g) * u of (g, u) = row(pos) . w13[e]^T in fp32, then
 *   MXFP8 along I: act [M,I] E4M3 codes and act_sf [M,I/128,16] padded scale rows (block scale
 *   2^(floor(log2 amax) - 8), E4M3 nearest-even, saturating at 448).  x [M,H] E4M3 codes in
 *   expert-sorted order with x_sf [M,H/128,16]; w13 prepacked with gate_up = 1.  H % 128 == 0,
 *   I % 128 == 0.  Rows >= offsets[E] untouched.
 * moe_grouped_gemm_w4a8: out [M,N] bf16 = topk_w[sorted_pair[pos]] (optional) *
 *   (a[pos] . w[e]^T), a [M,K] E4M3 with a_sf [M,K/128,16], w prepacked with gate_up = 0;
 *   N % 256 == 0, K % 128 == 0.
 * Both walk 32 token columns per tile when M <= 32*E (decode: a few rows per expert), else 112 (prefill:
 * each weight tile read once per 112 rows); the same results either way, within the stated rounding.
 * ws: at least moe_grouped_gemm_workspace_size() bytes.
 *
 * moe_layer_forward_w4a8: the whole layer a1 -> a6 on MXFP8 x (x_codes [T,H], x_scales [T,H/32],
 *   e.g. from moe_add_rms_norm_mxfp8): gating, routing, the MXFP8 row gather, the W4A8 gate/up GEMM
 *   (+ the shared expert as one more segment, act_s in MXFP8 as well), the W4A8 down GEMM
 *   (+ shared), finalize; y [T,H] bf16.  Weights prepacked by moe_w4a8_prepack (w13 with gate_up = 1,
 *   w2 with 0; the shared expert's likewise with E = 1, or all four NULL when d->n_shared == 0).
 *   H % 256 == 0; I, I_s multiples of 128.  ws: moe_w4a8_layer_workspace_size(d) bytes.
 *   moe_layer_forward_w4a8_events records six caller events as moe_layer_forward_events does (before
 *   gating, routing, the gate/up GEMM (after the row gather), the down GEMM, finalize; after it).
 *   moe_w4a8_layer_kernel_launches: kernels per call.
 */
MOE_API int moe_w4a8_prepack(const uint8_t* codes, const uint8_t* scales, int E, int n_out, int K, int gate_up,
                             uint8_t* codes_p, uint8_t* sf_p, void* stream);
MOE_API int moe_gather_rows_mx(const uint8_t* x_codes, const uint8_t* x_scales, const int32_t* sorted_pair, int T,
                               int k, int H, int M, uint8_t* out_codes, uint8_t* out_sf, void* ws, size_t ws_bytes,
                               void* stream);
MOE_API int moe_grouped_gemm_swiglu_w4a8(const uint8_t* x, const uint8_t* x_sf, const uint8_t* w13_codes,
                                         const uint8_t* w13_sf, const int32_t* offsets, int E, int M, int H, int I,
                                         uint8_t* act, uint8_t* act_sf, void* ws, size_t ws_bytes, void* stream);
MOE_API int moe_grouped_gemm_w4a8(const uint8_t* a, const uint8_t* a_sf, const uint8_t* w_codes, const uint8_t* w_sf,
                                  const int32_t* offsets, const float* topk_w, const int32_t* sorted_pair, int E,
                                  int M, int N, int K, uint16_t* out, void* ws, size_t ws_bytes, void* stream);
MOE_API size_t moe_w4a8_layer_workspace_size(const moe_layer_desc* d);
MOE_API int moe_layer_forward_w4a8(const moe_layer_desc* d, const uint8_t* x_codes, const uint8_t* x_scales,
                                   const float* logits, const float* bias, const uint8_t* w13_codes,
                                   const uint8_t* w13_sf, const uint8_t* w2_codes, const uint8_t* w2_sf,
                                   const uint8_t* w13s_codes, const uint8_t* w13s_sf, const uint8_t* w2s_codes,
                                   const uint8_t* w2s_sf, uint16_t* y, float* topk_w, int32_t* topk_idx,
                                   int32_t* counts, void* ws, size_t ws_bytes, void* stream);
MOE_API int moe_layer_forward_w4a8_events(const moe_layer_desc* d, const uint8_t* x_codes, const uint8_t* x_scales,
                                          const float* logits, const float* bias, const uint8_t* w13_codes,
                                          const uint8_t* w13_sf, const uint8_t* w2_codes, const uint8_t* w2_sf,
                                          const uint8_t* w13s_codes, const uint8_t* w13s_sf,
                                          const uint8_t* w2s_codes, const uint8_t* w2s_sf, uint16_t* y,
                                          float* topk_w, int32_t* topk_idx, int32_t* counts, void* ws,
                                          size_t ws_bytes, void* stream, void* const* events, int n_events);
MOE_API int moe_w4a8_layer_kernel_launches(const moe_layer_desc* d);

/*
 * a6. Finalize-routing.  [Q3] "GMM enablement and routing optimisation"
 * (expert outputs back to token order and weighted sum); [HY3] 8.1 (the
 * shared-expert term belongs to this combine step).
 *
 *  y_perm   [P,H] bf16: per-pair outputs, already scaled by the routing weight.
 *  pair_pos [P] int32: p -> pos.
 *  shared   [T,H] bf16 shared-expert output or NULL.
 *  y        [T,H] bf16 out: y[t] = sum_{j<k} y_perm[pair_pos[t*k+j]] (+ shared[t]),
 *           summed in fp32 in slot order, rounded once.
 */
MOE_API int moe_finalize_routing(const uint16_t* y_perm, const int32_t* pair_pos, const uint16_t* shared, int T, int k,
                         int H, uint16_t* y, void* stream);

/*
 * The whole layer: a1 -> a2 -> a3 (+ shared gate/up) -> a4 (+ shared down) -> a6,
 * enqueued on one stream.  The shared expert ([HY3] 1.1) runs inside the same
 * grouped-GEMM launches as one more segment covering all T rows, weight 1.
 *
 *  d        layer shape (host pointer).
 *  x        [T,H] bf16; logits [T,E] fp32; bias [E] fp32 or NULL (sigmoid only).
 *  w13      [E,2I,H] bf16 packed by moe_prepack_w13; w2 [E,H,I] bf16.
 *  w13_s    [2I_s,H] bf16 packed by moe_prepack_w13 (E = 1); w2_s [H,I_s] bf16
 *           (both NULL when d->n_shared == 0).
 *  y        [T,H] bf16 out.
 *  topk_w   [T,k] fp32 out; topk_idx [T,k] int32 out; counts [E] int32 out.
 *  ws       at least moe_layer_workspace_size(d) bytes; holds offsets, the
 *           permutation, x_exp, act, y_perm and the shared-expert buffers.
 *           moe_layer_workspace_offsets() gives where each one lives.
 */
MOE_API size_t moe_layer_workspace_size(const moe_layer_desc* d);
MOE_API int moe_layer_forward(const moe_layer_desc* d, const uint16_t* x, const float* logits, const float* bias,
                      const uint16_t* w13, const uint16_t* w2, const uint16_t* w13_s, const uint16_t* w2_s,
                      uint16_t* y, float* topk_w, int32_t* topk_idx, int32_t* counts, void* ws, size_t ws_bytes,
                      void* stream);

/* Same as moe_layer_forward, and additionally records caller-created CUDA
 * events (cudaEvent_t, passed as void*) on `stream` around the steps, for
 * per-step device timing: events[0] before gating, [1] before init-routing,
 * [2] before the gate/up grouped GEMM, [3] before the down grouped GEMM(s),
 * [4] before finalize, [5] after finalize.  n_events must be 6; the events
 * stay owned by the caller.  A small batch (T*k <= 4096, rows gathered by a separate kernel)
 * is gated and sorted by one kernel, between events[0] and [1]; between [1] and [2] there is
 * then only the row gather. */
MOE_API int moe_layer_forward_events(const moe_layer_desc* d, const uint16_t* x, const float* logits,
                                     const float* bias, const uint16_t* w13, const uint16_t* w2,
                                     const uint16_t* w13_s, const uint16_t* w2_s, uint16_t* y, float* topk_w,
                                     int32_t* topk_idx, int32_t* counts, void* ws, size_t ws_bytes, void* stream,
                                     void* const* events, int n_events);

/* Number of kernel launches one moe_layer_forward call makes for this shape
 * (0 if the shape is invalid or T == 0): gating 1 + routing 3 (the four in 1 for T*k <= 4096
 * when the rows are gathered by a separate kernel) + row gather 1 (unless the compute-bound
 * gate/up GEMM gathers its rows itself) + gate/up 1 + down 1 (+1 for a shared expert with
 * I_s != I) + finalize 1. */
MOE_API int moe_layer_kernel_launches(const moe_layer_desc* d);

/* Byte offsets, inside the moe_layer_forward workspace, of its intermediates
 * (valid after a call on the same desc): index 0 offsets[E+1], 1 sorted_pair[P],
 * 2 pair_pos[P], 3 x_exp[P,H], 4 act[P,I], 5 y_perm[P,H], 6 act_s[T,I_s],
 * 7 shared[T,H].  Writes min(n, 8) values into out; returns 8. */
MOE_API int moe_layer_workspace_offsets(const moe_layer_desc* d, size_t* out, int n);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_MOE_H_ */
