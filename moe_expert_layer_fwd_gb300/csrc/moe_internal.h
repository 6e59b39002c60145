// Host-side launchers shared between the kernel files and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// `pdl`: launch so the kernel may overlap its predecessor on the stream (only
// between the library's own kernels inside moe_layer_forward).
cudaError_t launch_gating_topk(const float* logits, const float* bias, int T, int E, int k, int gate, float rsf,
                               float eps, float* topk_w, int32_t* topk_idx, cudaStream_t stream, bool pdl = false);
// Gating and init-routing of a small batch in one CTA (one launch instead of four), with the
// results of launch_gating_topk followed by launch_init_routing (no row gather): T*k <= 4096,
// E <= 1024, k <= 32 (gate_route_small_fits).
bool gate_route_small_fits(int T, int E, int k);
cudaError_t launch_gate_route_small(const float* logits, const float* bias, int T, int E, int k, int gate, float rsf,
                                    float eps, float* topk_w, int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                                    int32_t* sorted_pair, int32_t* pair_pos, cudaStream_t stream, bool pdl = false);

// Init-routing scratch: per-chunk expert histograms and bases.
int routing_chunk_pairs(int P);
size_t routing_scratch_bytes(int P, int E);
// `zero`, `n_zero`: optional words zeroed by the routing kernels (the gather flags of the
// following gate/up GEMM).  [e0, e1): the local expert range (e1 < 0: all E experts); counts
// and offsets then have e1-e0 (+1) entries and pair_pos is -1 for pairs routed elsewhere.
cudaError_t launch_init_routing(const int32_t* topk_idx, int P, int E, int k, const uint16_t* x, int H,
                                uint16_t* x_exp, int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                                int32_t* pair_pos, int32_t* scratch, unsigned* status, cudaStream_t stream,
                                bool pdl = false, unsigned* zero = nullptr, int n_zero = 0, int e0 = 0,
                                int e1 = -1);
// n_rows: optional device count of the rows to gather (the rest of x_exp is left alone).
// T: token rows of x (< 0: P / k).  status: optional; a source index outside [0, T*k) skips its
// row and sets DEV_ERR_BOUNDS there.
cudaError_t launch_expand_rows(const uint16_t* x, const int32_t* sorted_pair, int P, int k, int H,
                               uint16_t* x_exp, cudaStream_t stream, bool pdl = false,
                               const int32_t* n_rows = nullptr, int T = -1, unsigned* status = nullptr);

// One grouped GEMM launch: routed experts (+ optionally one dense "shared" segment).
struct GroupedGemmProblem {
  int mode;                    // 0: SwiGLU epilogue (w13), 1: scaled epilogue (down)
  // routed experts
  const uint16_t* a_rows;      // [M,K] token rows in expert-sorted order
  const uint16_t* w;           // [E, n_out, K] (mode 0: packed gate/up layout of moe_prepack_w13)
  const int32_t* offsets;      // [E+1] device
  int E, M, K, n_out;          // n_out = 2I (mode 0) or N (mode 1)
  uint16_t* out;               // [M, ld_out]
  int ld_out;                  // I (mode 0) or N (mode 1)
  const float* topk_w;         // mode 1: row scale topk_w[sorted_pair[pos]] (NULL: 1)
  const int32_t* sorted_pair;
  // optional shared segment (weight 1, rows 0..T_s-1 of s_rows)
  const uint16_t* s_rows;      // [T_s, K] or NULL
  const uint16_t* s_w;         // [n_out_s, K]
  int T_s, n_out_s;
  uint16_t* s_out;             // [T_s, ld_out_s]
  int ld_out_s;
  unsigned* status;
  // Mode 0 only, optional: gather the routed rows while the GEMM runs, a_rows[pos] =
  // g_x[g_sorted_pair[pos] / g_k] (a_rows is then written, not only read).  g_flags: one word
  // per 16 rows of a_rows, zeroed before the launch.
  const uint16_t* g_x;
  const int32_t* g_sorted_pair;
  int g_k, g_T;
  unsigned* g_flags;
};

// Failure injection (tests only): what 1 = wait limit of the grouped GEMMs' waits in ns (0: the
// default 2 s), what 2 = nonzero: the gate/up GEMM's in-kernel gather writes nothing and sets no
// flag.  Returns 0, or -1 for an unknown `what`.
int grouped_gemm_debug_set(int what, unsigned long long value);

// Whether the problem takes the 32-column (decode) instances; whether its CTA-pair instance
// streams weights (under 256 rows per expert); whether a gate/up GEMM asked to gather its rows
// does so inside the GEMM (the CTA-pair instances; else a separate gather kernel runs first).
bool grouped_gemm_narrow(int M, int E, bool has_shared, int T_s);
bool grouped_gemm_streaming(int M, int E);
bool grouped_gemm_gathers_inline(int M, int E, bool has_shared, int T_s);

cudaError_t launch_grouped_gemm(const GroupedGemmProblem& p, cudaStream_t stream, bool pdl = false);

// w13 [E,2I,H] -> packed gate/up layout read by the mode-0 grouped GEMM.
cudaError_t launch_prepack_w13(const uint16_t* w13, int E, int I, int H, uint16_t* w13p, cudaStream_t stream);

// Front end: fused residual add + RMSNorm + cast (H <= 8192), router gate GEMM in fp32.
// mx_codes / mx_scales (optional): the MXFP8 output, E4M3 codes [T,H] and E8M0 scales [T,H/32].
cudaError_t launch_add_rms_norm_cast(const uint16_t* h, const uint16_t* res, const uint16_t* w, int T, int H,
                                     float eps, float* y32, uint16_t* y16, uint16_t* res_out, cudaStream_t stream,
                                     uint8_t* mx_codes = nullptr, uint8_t* mx_scales = nullptr);
// S K-slices (router_splits); with S > 1, part holds S*T*E fp32 partial sums.
int router_splits(int T, int H, int E, int n_sms);
cudaError_t launch_router_logits(const float* y32, const uint16_t* w_gate, int T, int H, int E, float* logits,
                                 float* part, int S, cudaStream_t stream);

cudaError_t launch_finalize(const uint16_t* y_perm, const int32_t* pair_pos, const uint16_t* shared, int T, int k,
                            int H, uint16_t* y, cudaStream_t stream, bool pdl = false);

// MXFP4 expert weights (decode).  Grouped GEMMs on f16 token rows and prepacked MXFP4 weights:
// mode 0 writes act [M, ld_out] in f16 (SwiGLU), mode 1 writes bf16 [M, ld_out] times the routing
// weight.  n_out a multiple of 128, K of 64.
struct Mxfp4GemmProblem {
  int mode;
  const uint16_t* a_rows;    // [M,K] f16 token rows in expert-sorted order
  const uint8_t* codes;      // [E*n_out, K/2] prepacked E2M1 codes
  const uint8_t* scales;     // prepacked scale lines (E*n_out/128 tiles x K/32 lines x 128 bytes)
  const float* omega;        // [E*n_out] per-row 2^W_r
  const int32_t* offsets;    // [E+1] device
  int E, M, K, n_out;
  uint16_t* out;
  int ld_out;
  const float* topk_w;       // mode 1, optional (with sorted_pair)
  const int32_t* sorted_pair;
  unsigned* status;
};
cudaError_t launch_grouped_gemm_mxfp4(const Mxfp4GemmProblem& p, cudaStream_t stream, bool pdl = false);
cudaError_t launch_mxfp4_quantize(const uint16_t* w, long long rows, int K, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t stream);
cudaError_t launch_mxfp4_prepack(const uint8_t* codes, const uint8_t* scales, int E, int n_out, int K, int gate_up,
                                 uint8_t* codes_p, uint8_t* scales_p, float* omega, cudaStream_t stream);
cudaError_t launch_gather_rows_f16(const uint16_t* x, const int32_t* sorted_pair, int M, int k, int T, int H,
                                   uint16_t* out, unsigned* status, cudaStream_t stream, bool pdl = false);

// W4A8: MXFP8 token rows x MXFP4 expert weights on the block-scaled MMA.  Token rows: E4M3 codes
// [rows, K] with padded scale rows [rows, K/128, 16] (four E8M0 scales, twelve zero bytes).  Weights
// prepacked by launch_w4a8_prepack.  Mode 0: act codes [M, n_out/2] + padded scale rows; mode 1: bf16
// out [M, n_out] times the routing weight.  K % 128 == 0; n_out % 256 (mode 0) or % 128 (mode 1).
struct W4a8GemmProblem {
  int mode;
  const uint8_t* a_rows;     // [M, K] E4M3 codes in expert-sorted order
  const uint8_t* a_sf;       // [M, K/128, 16] padded scale rows
  const uint8_t* codes;      // [E*n_out, K/2] prepacked E2M1 codes
  const uint8_t* sf;         // scale atoms [E*n_out/128][K/128][512]
  const int32_t* offsets;    // [E+1] device
  int E, M, K, n_out;
  uint8_t* act;              // mode 0 out: [M, n_out/2] E4M3
  uint8_t* act_sf;           // mode 0 out: [M, n_out/256, 16]
  uint16_t* out;             // mode 1 out: [M, n_out] bf16
  const float* topk_w;       // mode 1, optional (with sorted_pair)
  const int32_t* sorted_pair;
  // optional shared segment (weight 1, token rows 0..T_s-1 of s_rows)
  const uint8_t* s_rows;
  const uint8_t* s_rows_sf;
  const uint8_t* s_codes;
  const uint8_t* s_sf;
  int T_s, n_out_s;
  uint8_t* s_act;
  uint8_t* s_act_sf;
  uint16_t* s_out;
  unsigned* status;
};
cudaError_t launch_grouped_gemm_w4a8(const W4a8GemmProblem& p, cudaStream_t stream, bool pdl = false);
// True when the W4A8 GEMMs take the 32-column (decode) instance, else the 112-column one.
bool w4a8_narrow(int M, int E, bool has_shared, int T_s);
cudaError_t launch_w4a8_prepack(const uint8_t* codes, const uint8_t* scales, int E, int n_out, int K, int gate_up,
                                uint8_t* codes_p, uint8_t* sf_p, cudaStream_t stream);
// sorted_pair NULL: identity rows and no codes written (the padded scale rows of x itself).
cudaError_t launch_gather_rows_mx(const uint8_t* x_codes, const uint8_t* x_scales, const int32_t* sorted_pair, int M,
                                  int k, int T, int H, uint8_t* out_codes, uint8_t* out_sf, const int32_t* n_rows,
                                  unsigned* status, cudaStream_t stream, bool pdl = false);

}  // namespace moe
