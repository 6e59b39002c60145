// C-ABI entry points: host-side validation, workspace carving and launches.
// Declarations and full argument documentation are in include/moe.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "../../include/moe.h"
#include "moe_common.cuh"
#include "moe_internal.h"

namespace {

constexpr size_t kHeader = 256;  // status word + padding
constexpr size_t kAlign = 256;
constexpr int kAbiVersion = 200;

inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SMs of the current device (152 on a GB300; also the answer without a device, so that a
// workspace size computed on the host matches the one the launch uses there).
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

inline unsigned* status_word(void* ws) { return reinterpret_cast<unsigned*>(ws); }

int check_common(int T, int E, int k) {
  if (T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || k > 32 || k > E) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int check_dims(long long P, int H, int I) {
  if (H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 64 != 0 || I % 64 != 0) return MOE_ERR_UNSUPPORTED;
  const long long mx = H > I ? H : I;
  if (P * mx >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Layout of the moe_layer_forward workspace.
struct LayerWs {
  size_t offsets, scratch, sorted_pair, pair_pos, gflags, x_exp, act, y_perm, act_s, shared, total;
};

LayerWs layer_ws(const moe_layer_desc* d) {
  LayerWs w{};
  const size_t P = (size_t)d->T * d->k;
  size_t o = kHeader;
  w.offsets = o;     o = align_up(o + (size_t)(d->E + 1) * 4);
  w.scratch = o;     o = align_up(o + moe::routing_scratch_bytes((int)P, d->E));
  w.sorted_pair = o; o = align_up(o + P * 4);
  w.pair_pos = o;    o = align_up(o + P * 4);
  w.gflags = o;      o = align_up(o + (P + 15) / 16 * 4);  // one flag per 16 gathered rows
  w.x_exp = o;       o = align_up(o + P * d->H * 2);
  w.act = o;         o = align_up(o + P * d->I * 2);
  w.y_perm = o;      o = align_up(o + P * d->H * 2);
  const bool sh = d->n_shared > 0;
  w.act_s = o;       o = align_up(o + (sh ? (size_t)d->T * d->I_s * 2 : 0));
  w.shared = o;      o = align_up(o + (sh ? (size_t)d->T * d->H * 2 : 0));
  w.total = o;
  return w;
}

int check_desc(const moe_layer_desc* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  int s = check_common(d->T, d->E, d->k);
  if (s) return s;
  if ((s = check_dims((long long)d->T * d->k, d->H, d->I))) return s;
  if (d->gate != MOE_GATE_SOFTMAX && d->gate != MOE_GATE_SIGMOID && d->gate != MOE_GATE_SIGMOID_INNER_BIAS)
    return MOE_ERR_INVALID_ARG;
  if (d->n_shared < 0) return MOE_ERR_INVALID_ARG;
  if (d->n_shared > 1) return MOE_ERR_UNSUPPORTED;
  if (d->n_shared == 1) {
    if (d->I_s <= 0) return MOE_ERR_INVALID_ARG;
    if (d->I_s % 64 != 0) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_abi_version(void) { return kAbiVersion; }

size_t moe_status_bytes(void) { return kHeader; }

int moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < kHeader) return MOE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, kHeader, as_stream(stream)));
}

int moe_get_device_status(const void* ws, void* stream) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  unsigned word = 0;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (word & moe::DEV_ERR_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (word & (moe::DEV_ERR_BOUNDS | moe::DEV_ERR_CONFIG)) return MOE_ERR_DEVICE_CHECK;
  return MOE_OK;
}

int moe_gating_topk(const float* logits, const float* bias, int T, int E, int k, int gate,
                    float routed_scaling_factor, float eps, float* topk_w, int32_t* topk_idx, void* stream) {
  int s = check_common(T, E, k);
  if (s) return s;
  if (gate != MOE_GATE_SOFTMAX && gate != MOE_GATE_SIGMOID && gate != MOE_GATE_SIGMOID_INNER_BIAS)
    return MOE_ERR_INVALID_ARG;
  if (gate == MOE_GATE_SOFTMAX && bias) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_w || !topk_idx) return MOE_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(topk_w) || !aligned16(topk_idx) || (bias && !aligned16(bias)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_gating_topk(logits, bias, T, E, k, gate, routed_scaling_factor, eps, topk_w,
                                             topk_idx, as_stream(stream)));
}

size_t moe_init_routing_workspace_size(int T, int E, int k) {
  if (check_common(T, E, k)) return 0;
  return align_up(kHeader + moe::routing_scratch_bytes(T * k, E));
}

}  // extern "C"

namespace {

int init_routing_impl(const int32_t* topk_idx, int T, int E, int k, int e0, int e1, const uint16_t* x, int H,
                      uint16_t* x_exp, int32_t* counts, int32_t* offsets, int32_t* sorted_pair, int32_t* pair_pos,
                      void* ws, size_t ws_bytes, void* stream) {
  int s = check_common(T, E, k);
  if (s) return s;
  if (e0 < 0 || e1 <= e0 || e1 > E) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || !ws) return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_exp == nullptr)) return MOE_ERR_INVALID_ARG;
  if (x) {
    if ((s = check_dims((long long)T * k, H, 64))) return s;
    if (!aligned16(x) || !aligned16(x_exp)) return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16(counts) || !aligned16(offsets) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_init_routing_workspace_size(T, E, k)) return MOE_ERR_WORKSPACE;
  if (T > 0 && (!topk_idx || !sorted_pair || !pair_pos || !aligned16(topk_idx) || !aligned16(sorted_pair) ||
                !aligned16(pair_pos)))
    return MOE_ERR_INVALID_ARG;
  int32_t* scratch = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kHeader);
  return cuda_status(moe::launch_init_routing(topk_idx, T * k, E, k, x, H, x_exp, counts, offsets, sorted_pair,
                                              pair_pos, scratch, status_word(ws), as_stream(stream), false, nullptr,
                                              0, e0, e1));
}

}  // namespace

extern "C" {

int moe_init_routing(const int32_t* topk_idx, int T, int E, int k, const uint16_t* x, int H, uint16_t* x_exp,
                     int32_t* counts, int32_t* offsets, int32_t* sorted_pair, int32_t* pair_pos, void* ws,
                     size_t ws_bytes, void* stream) {
  return init_routing_impl(topk_idx, T, E, k, 0, E, x, H, x_exp, counts, offsets, sorted_pair, pair_pos, ws,
                           ws_bytes, stream);
}

int moe_init_routing_range(const int32_t* topk_idx, int T, int E, int k, int e0, int e1, const uint16_t* x, int H,
                           uint16_t* x_exp, int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                           int32_t* pair_pos, void* ws, size_t ws_bytes, void* stream) {
  return init_routing_impl(topk_idx, T, E, k, e0, e1, x, H, x_exp, counts, offsets, sorted_pair, pair_pos, ws,
                           ws_bytes, stream);
}

int moe_debug_set(int what, unsigned long long value) {
  return moe::grouped_gemm_debug_set(what, value) == 0 ? MOE_OK : MOE_ERR_INVALID_ARG;
}

int moe_add_rms_norm_cast(const uint16_t* hidden, const uint16_t* residual, const uint16_t* norm_weight, int T,
                          int H, float eps, float* y_fp32, uint16_t* y_bf16, uint16_t* residual_out, void* stream) {
  if (T < 0 || H <= 0 || !(eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
  if (H % 64 != 0 || H > 8192) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!hidden || !norm_weight || !y_fp32) return MOE_ERR_INVALID_ARG;
  if (residual && !residual_out) return MOE_ERR_INVALID_ARG;  // the new residual stream must go somewhere
  const void* ptrs[] = {hidden, residual, norm_weight, y_fp32, y_bf16, residual_out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_add_rms_norm_cast(hidden, residual, norm_weight, T, H, eps, y_fp32, y_bf16,
                                                   residual_out, as_stream(stream)));
}

int moe_add_rms_norm_mxfp8(const uint16_t* hidden, const uint16_t* residual, const uint16_t* norm_weight, int T,
                           int H, float eps, uint8_t* y_fp8, uint8_t* y_scale, float* y_fp32, uint16_t* residual_out,
                           void* stream) {
  if (T < 0 || H <= 0 || !(eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
  if (H % 64 != 0 || H > 8192) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!hidden || !norm_weight || !y_fp8 || !y_scale) return MOE_ERR_INVALID_ARG;
  if (residual && !residual_out) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {hidden, residual, norm_weight, y_fp8, y_fp32, residual_out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_add_rms_norm_cast(hidden, residual, norm_weight, T, H, eps, y_fp32, nullptr,
                                                   residual_out, as_stream(stream), y_fp8, y_scale));
}

size_t moe_router_logits_workspace_size(int T, int H, int E) {
  if (T <= 0 || H <= 0 || E <= 0) return kHeader;
  const int S = moe::router_splits(T, H, E, sm_count());
  return align_up(kHeader + (S > 1 ? (size_t)S * T * E * sizeof(float) : 0));
}

int moe_router_logits(const float* y_fp32, const uint16_t* w_gate, int T, int H, int E, float* logits, void* ws,
                      size_t ws_bytes, void* stream) {
  if (T < 0 || H <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 64 != 0 || E > 1024) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y_fp32 || !w_gate || !logits || !ws || !aligned16(y_fp32) || !aligned16(w_gate) || !aligned16(logits) ||
      !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_router_logits_workspace_size(T, H, E)) return MOE_ERR_WORKSPACE;
  const int S = moe::router_splits(T, H, E, sm_count());
  float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + kHeader);
  return cuda_status(moe::launch_router_logits(y_fp32, w_gate, T, H, E, logits, part, S, as_stream(stream)));
}

int moe_prepack_w13(const uint16_t* w13, int E, int I, int H, uint16_t* w13_packed, void* stream) {
  if (E < 1) return MOE_ERR_INVALID_ARG;
  int s = check_dims(1, H, I);
  if (s) return s;
  if (!w13 || !w13_packed || w13 == w13_packed) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w13) || !aligned16(w13_packed)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_prepack_w13(w13, E, I, H, w13_packed, as_stream(stream)));
}

size_t moe_grouped_gemm_workspace_size(void) { return kHeader; }

size_t moe_grouped_gemm_swiglu_workspace_size(int M, int H, int gather) {
  if (M < 0 || H <= 0) return 0;
  if (!gather) return kHeader;
  return kHeader + align_up((size_t)(M + 15) / 16 * 4) + align_up((size_t)M * H * 2);
}

int moe_grouped_gemm_swiglu(const uint16_t* x, const int32_t* row_src, int k, int T, const uint16_t* w13,
                            const int32_t* offsets, int E, int M, int H, int I, uint16_t* act, void* ws,
                            size_t ws_bytes, void* stream) {
  if (E < 1 || M < 0) return MOE_ERR_INVALID_ARG;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  int s = check_dims(M, H, I);
  if (s) return s;
  const bool gather = row_src != nullptr;
  if (gather) {
    if (k < 1 || T < 0) return MOE_ERR_INVALID_ARG;
    if (k > 32 || (long long)T * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  }
  if (!w13 || !offsets || !ws) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_grouped_gemm_swiglu_workspace_size(M, H, gather ? 1 : 0)) return MOE_ERR_WORKSPACE;
  if (M == 0) return MOE_OK;
  if (!x || !act) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w13) || !aligned16(offsets) || !aligned16(act) || !aligned16(ws) ||
      (gather && !aligned16(row_src)))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  moe::GroupedGemmProblem p{};
  p.mode = 0;
  p.a_rows = x;
  p.w = w13;
  p.offsets = offsets;
  p.E = E;
  p.M = M;
  p.K = H;
  p.n_out = 2 * I;
  p.out = act;
  p.ld_out = I;
  p.status = status_word(ws);
  if (gather) {
    // The gathered rows live in the workspace after the status header and the gather flags.
    char* base = static_cast<char*>(ws);
    const size_t flags_off = kHeader;
    const size_t rows_off = kHeader + align_up((size_t)(M + 15) / 16 * 4);
    unsigned* flags = reinterpret_cast<unsigned*>(base + flags_off);
    p.a_rows = reinterpret_cast<const uint16_t*>(base + rows_off);
    p.g_x = x;
    p.g_sorted_pair = row_src;
    p.g_k = k;
    p.g_T = T;
    p.g_flags = flags;
    // the in-kernel gather publishes one flag per 16 rows: they start at zero
    if (moe::grouped_gemm_gathers_inline(M, E, false, 0) &&
        cudaMemsetAsync(flags, 0, (size_t)(M + 15) / 16 * 4, st) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return cuda_status(moe::launch_grouped_gemm(p, st));
}

int moe_grouped_gemm(const uint16_t* a, const uint16_t* w, const int32_t* offsets, const float* topk_w,
                     const int32_t* sorted_pair, int E, int M, int N, int K, uint16_t* out, void* ws,
                     size_t ws_bytes, void* stream) {
  if (E < 1 || M < 0) return MOE_ERR_INVALID_ARG;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  int s = check_dims(M, N, K);
  if (s) return s;
  if ((topk_w == nullptr) != (sorted_pair == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!w || !offsets || !ws) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < kHeader) return MOE_ERR_WORKSPACE;
  if (M == 0) return MOE_OK;
  if (!a || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(w) || !aligned16(offsets) || !aligned16(out) || !aligned16(ws) ||
      (topk_w && (!aligned16(topk_w) || !aligned16(sorted_pair))))
    return MOE_ERR_INVALID_ARG;
  moe::GroupedGemmProblem p{};
  p.mode = 1;
  p.a_rows = a;
  p.w = w;
  p.offsets = offsets;
  p.E = E;
  p.M = M;
  p.K = K;
  p.n_out = N;
  p.out = out;
  p.ld_out = N;
  p.topk_w = topk_w;
  p.sorted_pair = sorted_pair;
  p.status = status_word(ws);
  return cuda_status(moe::launch_grouped_gemm(p, as_stream(stream)));
}

int moe_mxfp4_quantize(const uint16_t* w, long long rows, int K, uint8_t* codes, uint8_t* scales, void* stream) {
  if (rows < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 32 != 0 || rows * (long long)K >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  if (!w || !codes || !scales || !aligned16(w) || !aligned16(codes)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_mxfp4_quantize(w, rows, K, codes, scales, as_stream(stream)));
}

int moe_mxfp4_prepack(const uint8_t* codes, const uint8_t* scales, int E, int n_out, int K, int gate_up,
                      uint8_t* codes_p, uint8_t* scales_p, float* omega, void* stream) {
  if (E < 1 || n_out <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (n_out % 128 != 0 || K % 64 != 0 || (long long)E * n_out * K >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
  if (!codes || !scales || !codes_p || !scales_p || !omega) return MOE_ERR_INVALID_ARG;
  if (codes == codes_p || scales == scales_p) return MOE_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(codes_p) || !aligned16(scales_p) || !aligned16(omega)) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      moe::launch_mxfp4_prepack(codes, scales, E, n_out, K, gate_up ? 1 : 0, codes_p, scales_p, omega, as_stream(stream)));
}

int moe_gather_rows_f16(const uint16_t* x, const int32_t* sorted_pair, int T, int k, int H, int M, uint16_t* x_rows16,
                        void* ws, size_t ws_bytes, void* stream) {
  if (T < 0 || k < 1 || M < 0 || H <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 64 != 0 || (long long)T * k >= (1LL << 31) || (long long)M * H >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < kHeader || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  if (M == 0) return MOE_OK;
  if (!x || !sorted_pair || !x_rows16 || !aligned16(x) || !aligned16(x_rows16)) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      moe::launch_gather_rows_f16(x, sorted_pair, M, k, T, H, x_rows16, status_word(ws), as_stream(stream)));
}

namespace {
int mxfp4_gemm(int mode, const uint16_t* a, const uint8_t* codes, const uint8_t* scales, const float* omega,
               const int32_t* offsets, const float* topk_w, const int32_t* sorted_pair, int E, int M, int n_out,
               int K, uint16_t* out, int ld_out, void* ws, size_t ws_bytes, void* stream) {
  if (E < 1 || M < 0) return MOE_ERR_INVALID_ARG;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  int s = check_dims(M, n_out, K);
  if (s) return s;
  if (n_out % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if ((topk_w == nullptr) != (sorted_pair == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!codes || !scales || !omega || !offsets || !ws) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < kHeader) return MOE_ERR_WORKSPACE;
  if (M == 0) return MOE_OK;
  if (!a || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(codes) || !aligned16(scales) || !aligned16(omega) || !aligned16(offsets) ||
      !aligned16(out) || !aligned16(ws) || (topk_w && (!aligned16(topk_w) || !aligned16(sorted_pair))))
    return MOE_ERR_INVALID_ARG;
  moe::Mxfp4GemmProblem p{};
  p.mode = mode;
  p.a_rows = a;
  p.codes = codes;
  p.scales = scales;
  p.omega = omega;
  p.offsets = offsets;
  p.E = E;
  p.M = M;
  p.K = K;
  p.n_out = n_out;
  p.out = out;
  p.ld_out = ld_out;
  p.topk_w = topk_w;
  p.sorted_pair = sorted_pair;
  p.status = status_word(ws);
  return cuda_status(moe::launch_grouped_gemm_mxfp4(p, as_stream(stream)));
}
}  // namespace

int moe_grouped_gemm_swiglu_mxfp4(const uint16_t* x_rows16, const uint8_t* w13_codes, const uint8_t* w13_scales,
                                  const float* w13_omega, const int32_t* offsets, int E, int M, int H, int I,
                                  uint16_t* act16, void* ws, size_t ws_bytes, void* stream) {
  if (I <= 0) return MOE_ERR_INVALID_ARG;
  return mxfp4_gemm(0, x_rows16, w13_codes, w13_scales, w13_omega, offsets, nullptr, nullptr, E, M, 2 * I, H, act16,
                    I, ws, ws_bytes, stream);
}

int moe_grouped_gemm_mxfp4(const uint16_t* a16, const uint8_t* w_codes, const uint8_t* w_scales, const float* w_omega,
                           const int32_t* offsets, const float* topk_w, const int32_t* sorted_pair, int E, int M,
                           int N, int K, uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  return mxfp4_gemm(1, a16, w_codes, w_scales, w_omega, offsets, topk_w, sorted_pair, E, M, N, K, out, N, ws, ws_bytes,
                    stream);
}

// ---------------------------------------------------------------- W4A8 (MXFP8 x MXFP4, block-scaled MMA)
int moe_w4a8_prepack(const uint8_t* codes, const uint8_t* scales, int E, int n_out, int K, int gate_up,
                     uint8_t* codes_p, uint8_t* sf_p, void* stream) {
  if (E < 1 || n_out <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (n_out % 256 != 0 || K % 128 != 0 || (long long)E * n_out * K >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
  if (!codes || !scales || !codes_p || !sf_p || codes == codes_p) return MOE_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(codes_p) || !aligned16(sf_p)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_w4a8_prepack(codes, scales, E, n_out, K, gate_up ? 1 : 0, codes_p, sf_p,
                                              as_stream(stream)));
}

int moe_gather_rows_mx(const uint8_t* x_codes, const uint8_t* x_scales, const int32_t* sorted_pair, int T, int k,
                       int H, int M, uint8_t* out_codes, uint8_t* out_sf, void* ws, size_t ws_bytes, void* stream) {
  if (T < 0 || k < 1 || M < 0 || H <= 0) return MOE_ERR_INVALID_ARG;
  if (H % 128 != 0 || (long long)T * k >= (1LL << 31) || (long long)M * H >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < kHeader || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  if (!sorted_pair && M > T) return MOE_ERR_INVALID_ARG;  // identity rows: at most the T token rows
  if (M == 0) return MOE_OK;
  if (!x_codes || !x_scales || !out_sf || (sorted_pair && !out_codes)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_codes) || !aligned16(out_sf) || (out_codes && !aligned16(out_codes)) ||
      (reinterpret_cast<uintptr_t>(x_scales) & 3u))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_gather_rows_mx(x_codes, x_scales, sorted_pair, M, k, T, H,
                                                sorted_pair ? out_codes : nullptr, out_sf, nullptr, status_word(ws),
                                                as_stream(stream)));
}

namespace {
int w4a8_gemm(int mode, const uint8_t* a, const uint8_t* a_sf, const uint8_t* codes, const uint8_t* sf,
              const int32_t* offsets, const float* topk_w, const int32_t* sorted_pair, int E, int M, int n_out, int K,
              uint8_t* act, uint8_t* act_sf, uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  if (E < 1 || M < 0 || n_out <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  if (K % 128 != 0 || n_out % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if ((long long)M * (n_out > K ? n_out : K) >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
  if ((topk_w == nullptr) != (sorted_pair == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!codes || !sf || !offsets || !ws) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < kHeader) return MOE_ERR_WORKSPACE;
  if (M == 0) return MOE_OK;
  if (!a || !a_sf || (mode == 0 && (!act || !act_sf)) || (mode == 1 && !out)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {a, a_sf, codes, sf, offsets, ws, act, act_sf, out, topk_w, sorted_pair};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  moe::W4a8GemmProblem p{};
  p.mode = mode;
  p.a_rows = a;
  p.a_sf = a_sf;
  p.codes = codes;
  p.sf = sf;
  p.offsets = offsets;
  p.E = E;
  p.M = M;
  p.K = K;
  p.n_out = n_out;
  p.act = act;
  p.act_sf = act_sf;
  p.out = out;
  p.topk_w = topk_w;
  p.sorted_pair = sorted_pair;
  p.status = status_word(ws);
  return cuda_status(moe::launch_grouped_gemm_w4a8(p, as_stream(stream)));
}
}  // namespace

int moe_grouped_gemm_swiglu_w4a8(const uint8_t* x, const uint8_t* x_sf, const uint8_t* w13_codes,
                                 const uint8_t* w13_sf, const int32_t* offsets, int E, int M, int H, int I,
                                 uint8_t* act, uint8_t* act_sf, void* ws, size_t ws_bytes, void* stream) {
  if (I <= 0) return MOE_ERR_INVALID_ARG;
  return w4a8_gemm(0, x, x_sf, w13_codes, w13_sf, offsets, nullptr, nullptr, E, M, 2 * I, H, act, act_sf, nullptr, ws,
                   ws_bytes, stream);
}

int moe_grouped_gemm_w4a8(const uint8_t* a, const uint8_t* a_sf, const uint8_t* w_codes, const uint8_t* w_sf,
                          const int32_t* offsets, const float* topk_w, const int32_t* sorted_pair, int E, int M, int N,
                          int K, uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  return w4a8_gemm(1, a, a_sf, w_codes, w_sf, offsets, topk_w, sorted_pair, E, M, N, K, nullptr, nullptr, out, ws,
                   ws_bytes, stream);
}

int moe_finalize_routing(const uint16_t* y_perm, const int32_t* pair_pos, const uint16_t* shared, int T, int k,
                         int H, uint16_t* y, void* stream) {
  if (T < 0 || k < 1 || H <= 0) return MOE_ERR_INVALID_ARG;
  if (k > 32 || H % 64 != 0 || (long long)T * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y_perm || !pair_pos || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(pair_pos) || !aligned16(y) || (shared && !aligned16(shared)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_finalize(y_perm, pair_pos, shared, T, k, H, y, as_stream(stream)));
}

size_t moe_layer_workspace_size(const moe_layer_desc* d) {
  if (check_desc(d)) return 0;
  return layer_ws(d).total;
}

int moe_layer_workspace_offsets(const moe_layer_desc* d, size_t* out, int n) {
  if (check_desc(d) || !out || n < 0) return MOE_ERR_INVALID_ARG;
  const LayerWs w = layer_ws(d);
  const size_t v[8] = {w.offsets, w.sorted_pair, w.pair_pos, w.x_exp, w.act, w.y_perm, w.act_s, w.shared};
  for (int i = 0; i < n && i < 8; ++i) out[i] = v[i];
  return 8;
}

}  // extern "C"

namespace {

int layer_forward_impl(const moe_layer_desc* d, const uint16_t* x, const float* logits, const float* bias,
                       const uint16_t* w13, const uint16_t* w2, const uint16_t* w13_s, const uint16_t* w2_s,
                       uint16_t* y, float* topk_w, int32_t* topk_idx, int32_t* counts, void* ws, size_t ws_bytes,
                       void* stream, void* const* events) {
  int s = check_desc(d);
  if (s) return s;
  if (d->gate == MOE_GATE_SOFTMAX && bias) return MOE_ERR_INVALID_ARG;
  if (!ws || !counts) return MOE_ERR_INVALID_ARG;
  const LayerWs L = layer_ws(d);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (d->T == 0) return MOE_OK;
  if (!x || !logits || !w13 || !w2 || !y || !topk_w || !topk_idx) return MOE_ERR_INVALID_ARG;
  if (d->n_shared && (!w13_s || !w2_s)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, logits, w13, w2, y, topk_w, topk_idx, counts, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if ((bias && !aligned16(bias)) || (w13_s && !aligned16(w13_s)) || (w2_s && !aligned16(w2_s)))
    return MOE_ERR_INVALID_ARG;

  cudaStream_t st = as_stream(stream);
  char* base = static_cast<char*>(ws);
  unsigned* status = status_word(ws);
  int32_t* offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  int32_t* scratch = reinterpret_cast<int32_t*>(base + L.scratch);
  int32_t* sorted_pair = reinterpret_cast<int32_t*>(base + L.sorted_pair);
  int32_t* pair_pos = reinterpret_cast<int32_t*>(base + L.pair_pos);
  uint16_t* x_exp = reinterpret_cast<uint16_t*>(base + L.x_exp);
  unsigned* gflags = reinterpret_cast<unsigned*>(base + L.gflags);
  uint16_t* act = reinterpret_cast<uint16_t*>(base + L.act);
  uint16_t* y_perm = reinterpret_cast<uint16_t*>(base + L.y_perm);
  uint16_t* act_s = reinterpret_cast<uint16_t*>(base + L.act_s);
  uint16_t* shared = reinterpret_cast<uint16_t*>(base + L.shared);
  const int T = d->T, E = d->E, k = d->k, H = d->H, I = d->I, P = T * k;
  const bool sh = d->n_shared > 0;

  auto mark = [&](int i) {
    return events ? cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), st) : cudaSuccess;
  };
  // Every kernel may start while its predecessor on the stream finishes (programmatic dependent
  // launch; for gating that is whatever the caller ran before, e.g. the previous layer's
  // finalize); each waits for its predecessor's completion before touching memory.
  constexpr bool kPdl = true;
  // A gate/up GEMM on CTA pairs (prefill sizes) gathers the token rows into x_exp itself
  // (overlapping the gather with its matmuls): routing then only sorts, and clears the GEMM's
  // gather flags.  Otherwise (decode) a row gather kernel follows routing, and a small batch is
  // gated and sorted by one kernel instead of four.
  const bool inline_gather = moe::grouped_gemm_gathers_inline(P, E, sh, T);
  const bool small = !inline_gather && moe::gate_route_small_fits(T, E, k);
  if (mark(0) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t e;
  if (small) {
    e = moe::launch_gate_route_small(logits, bias, T, E, k, d->gate, d->routed_scaling_factor, d->eps, topk_w,
                                     topk_idx, counts, offsets, sorted_pair, pair_pos, st, kPdl);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(1) != cudaSuccess) return MOE_ERR_CUDA;
    e = moe::launch_expand_rows(x, sorted_pair, P, k, H, x_exp, st, kPdl);
  } else {
    e = moe::launch_gating_topk(logits, bias, T, E, k, d->gate, d->routed_scaling_factor, d->eps, topk_w, topk_idx,
                                st, kPdl);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (mark(1) != cudaSuccess) return MOE_ERR_CUDA;
    e = moe::launch_init_routing(topk_idx, P, E, k, inline_gather ? nullptr : x, H, inline_gather ? nullptr : x_exp,
                                 counts, offsets, sorted_pair, pair_pos, scratch, status, st, kPdl,
                                 inline_gather ? gflags : nullptr, inline_gather ? (P + 15) / 16 : 0);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  moe::GroupedGemmProblem g1{};
  g1.mode = 0;
  g1.a_rows = x_exp;
  g1.w = w13;
  g1.offsets = offsets;
  g1.E = E;
  g1.M = P;
  g1.K = H;
  g1.n_out = 2 * I;
  g1.out = act;
  g1.ld_out = I;
  if (inline_gather) {
    g1.g_x = x;
    g1.g_sorted_pair = sorted_pair;
    g1.g_k = k;
    g1.g_T = T;
    g1.g_flags = gflags;
  }
  if (sh) {
    g1.s_rows = x;
    g1.s_w = w13_s;
    g1.T_s = T;
    g1.n_out_s = 2 * d->I_s;
    g1.s_out = act_s;
    g1.ld_out_s = d->I_s;
  }
  g1.status = status;
  if (mark(2) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_grouped_gemm(g1, st, kPdl) != cudaSuccess) return MOE_ERR_CUDA;
  if (mark(3) != cudaSuccess) return MOE_ERR_CUDA;

  // The down projection's K is I for routed experts and I_s for the shared
  // one; one launch covers both only when they agree.
  moe::GroupedGemmProblem g2{};
  g2.mode = 1;
  g2.a_rows = act;
  g2.w = w2;
  g2.offsets = offsets;
  g2.E = E;
  g2.M = P;
  g2.K = I;
  g2.n_out = H;
  g2.out = y_perm;
  g2.ld_out = H;
  g2.topk_w = topk_w;
  g2.sorted_pair = sorted_pair;
  g2.status = status;
  moe::GroupedGemmProblem g2s{};
  const bool fused_shared = sh && d->I_s == I;
  if (sh) {
    moe::GroupedGemmProblem& gs = fused_shared ? g2 : g2s;
    gs.s_rows = act_s;
    gs.s_w = w2_s;
    gs.T_s = T;
    gs.n_out_s = H;
    gs.s_out = shared;
    gs.ld_out_s = H;
  }
  if (moe::launch_grouped_gemm(g2, st, kPdl) != cudaSuccess) return MOE_ERR_CUDA;
  if (sh && !fused_shared) {
    // separate launch for the shared expert's down projection (K = I_s)
    g2s.mode = 1;
    g2s.a_rows = nullptr;
    g2s.w = w2_s;
    g2s.offsets = nullptr;
    g2s.E = 1;
    g2s.M = 0;
    g2s.K = d->I_s;
    g2s.n_out = H;
    g2s.status = status;
    if (moe::launch_grouped_gemm(g2s, st, kPdl) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (mark(4) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_finalize(y_perm, pair_pos, sh ? shared : nullptr, T, k, H, y, st, kPdl) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cuda_status(mark(5));
}

}  // namespace

extern "C" {

int moe_layer_forward(const moe_layer_desc* d, const uint16_t* x, const float* logits, const float* bias,
                      const uint16_t* w13, const uint16_t* w2, const uint16_t* w13_s, const uint16_t* w2_s,
                      uint16_t* y, float* topk_w, int32_t* topk_idx, int32_t* counts, void* ws, size_t ws_bytes,
                      void* stream) {
  return layer_forward_impl(d, x, logits, bias, w13, w2, w13_s, w2_s, y, topk_w, topk_idx, counts, ws, ws_bytes,
                            stream, nullptr);
}

int moe_layer_forward_events(const moe_layer_desc* d, const uint16_t* x, const float* logits, const float* bias,
                             const uint16_t* w13, const uint16_t* w2, const uint16_t* w13_s, const uint16_t* w2_s,
                             uint16_t* y, float* topk_w, int32_t* topk_idx, int32_t* counts, void* ws,
                             size_t ws_bytes, void* stream, void* const* events, int n_events) {
  if (!events || n_events != 6) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 6; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return layer_forward_impl(d, x, logits, bias, w13, w2, w13_s, w2_s, y, topk_w, topk_idx, counts, ws, ws_bytes,
                            stream, events);
}

int moe_layer_kernel_launches(const moe_layer_desc* d) {
  if (check_desc(d)) return 0;
  if (d->T == 0) return 0;
  // gating 1 + routing (hist, scan, scatter) 3, or both in 1 for a small batch + row gather 1
  // (unless the gate/up GEMM gathers its rows itself) + gate/up GEMM 1 + down GEMM 1 (+1 when the
  // shared expert's intermediate size differs) + finalize 1
  const bool sh = d->n_shared > 0;
  const bool gather_kernel = !moe::grouped_gemm_gathers_inline(d->T * d->k, d->E, sh, d->T);
  const bool small = gather_kernel && moe::gate_route_small_fits(d->T, d->E, d->k);
  return (small ? 1 : 4) + 3 + (gather_kernel ? 1 : 0) + ((sh && d->I_s != d->I) ? 1 : 0);
}

}  // extern "C"

namespace {

// Layout of the moe_layer_forward_w4a8 workspace.
struct W8Ws {
  size_t offsets, scratch, sorted_pair, pair_pos, x8, x8_sf, act, act_sf, y_perm, x_sf_tok, act_s, act_sf_s, shared,
      total;
};

W8Ws w8_ws(const moe_layer_desc* d) {
  W8Ws w{};
  const size_t P = (size_t)d->T * d->k, T = (size_t)d->T, H = (size_t)d->H, I = (size_t)d->I;
  const bool sh = d->n_shared > 0;
  const size_t Is = sh ? (size_t)d->I_s : 0;
  size_t o = kHeader;
  w.offsets = o;     o = align_up(o + (size_t)(d->E + 1) * 4);
  w.scratch = o;     o = align_up(o + moe::routing_scratch_bytes((int)P, d->E));
  w.sorted_pair = o; o = align_up(o + P * 4);
  w.pair_pos = o;    o = align_up(o + P * 4);
  w.x8 = o;          o = align_up(o + P * H);
  w.x8_sf = o;       o = align_up(o + P * (H / 128) * 16);
  w.act = o;         o = align_up(o + P * I);
  w.act_sf = o;      o = align_up(o + P * (I / 128) * 16);
  w.y_perm = o;      o = align_up(o + P * H * 2);
  w.x_sf_tok = o;    o = align_up(o + (sh ? T * (H / 128) * 16 : 0));
  w.act_s = o;       o = align_up(o + T * Is);
  w.act_sf_s = o;    o = align_up(o + T * (Is / 128) * 16);
  w.shared = o;      o = align_up(o + (sh ? T * H * 2 : 0));
  w.total = o;
  return w;
}

int check_desc_w4a8(const moe_layer_desc* d) {
  int s = check_desc(d);
  if (s) return s;
  if (d->H % 256 != 0 || d->I % 128 != 0 || (d->n_shared && d->I_s % 128 != 0)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int layer_forward_w4a8_impl(const moe_layer_desc* d, const uint8_t* x_codes, const uint8_t* x_scales,
                            const float* logits, const float* bias, const uint8_t* w13_codes, const uint8_t* w13_sf,
                            const uint8_t* w2_codes, const uint8_t* w2_sf, const uint8_t* w13s_codes,
                            const uint8_t* w13s_sf, const uint8_t* w2s_codes, const uint8_t* w2s_sf, uint16_t* y,
                            float* topk_w, int32_t* topk_idx, int32_t* counts, void* ws, size_t ws_bytes,
                            void* stream, void* const* events) {
  int s = check_desc_w4a8(d);
  if (s) return s;
  if (d->gate == MOE_GATE_SOFTMAX && bias) return MOE_ERR_INVALID_ARG;
  if (!ws || !counts) return MOE_ERR_INVALID_ARG;
  const W8Ws L = w8_ws(d);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (d->T == 0) return MOE_OK;
  if (!x_codes || !x_scales || !logits || !w13_codes || !w13_sf || !w2_codes || !w2_sf || !y || !topk_w || !topk_idx)
    return MOE_ERR_INVALID_ARG;
  const bool sh = d->n_shared > 0;
  if (sh && (!w13s_codes || !w13s_sf || !w2s_codes || !w2s_sf)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x_codes, logits, w13_codes, w13_sf, w2_codes, w2_sf, y, topk_w, topk_idx, counts, ws,
                        bias, w13s_codes, w13s_sf, w2s_codes, w2s_sf};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(x_scales) & 3u) return MOE_ERR_INVALID_ARG;

  cudaStream_t st = as_stream(stream);
  char* base = static_cast<char*>(ws);
  unsigned* status = status_word(ws);
  int32_t* offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  int32_t* scratch = reinterpret_cast<int32_t*>(base + L.scratch);
  int32_t* sorted_pair = reinterpret_cast<int32_t*>(base + L.sorted_pair);
  int32_t* pair_pos = reinterpret_cast<int32_t*>(base + L.pair_pos);
  uint8_t* x8 = reinterpret_cast<uint8_t*>(base + L.x8);
  uint8_t* x8_sf = reinterpret_cast<uint8_t*>(base + L.x8_sf);
  uint8_t* act = reinterpret_cast<uint8_t*>(base + L.act);
  uint8_t* act_sf = reinterpret_cast<uint8_t*>(base + L.act_sf);
  uint16_t* y_perm = reinterpret_cast<uint16_t*>(base + L.y_perm);
  uint8_t* x_sf_tok = reinterpret_cast<uint8_t*>(base + L.x_sf_tok);
  uint8_t* act_s = reinterpret_cast<uint8_t*>(base + L.act_s);
  uint8_t* act_sf_s = reinterpret_cast<uint8_t*>(base + L.act_sf_s);
  uint16_t* shared = reinterpret_cast<uint16_t*>(base + L.shared);
  const int T = d->T, E = d->E, k = d->k, H = d->H, I = d->I, P = T * k;

  auto mark = [&](int i) {
    return events ? cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), st) : cudaSuccess;
  };
  constexpr bool kPdl = true;
  if (mark(0) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::gate_route_small_fits(T, E, k)) {  // a small batch (decode): gated and sorted by one kernel
    if (moe::launch_gate_route_small(logits, bias, T, E, k, d->gate, d->routed_scaling_factor, d->eps, topk_w,
                                     topk_idx, counts, offsets, sorted_pair, pair_pos, st, kPdl) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (mark(1) != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    if (moe::launch_gating_topk(logits, bias, T, E, k, d->gate, d->routed_scaling_factor, d->eps, topk_w, topk_idx,
                                st, kPdl) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (mark(1) != cudaSuccess) return MOE_ERR_CUDA;
    if (moe::launch_init_routing(topk_idx, P, E, k, nullptr, H, nullptr, counts, offsets, sorted_pair, pair_pos,
                                 scratch, status, st, kPdl) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  // the routed MXFP8 rows in expert order, and (shared expert) the padded scale rows of x itself
  if (moe::launch_gather_rows_mx(x_codes, x_scales, sorted_pair, P, k, T, H, x8, x8_sf, nullptr, status, st,
                                 kPdl) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (sh && moe::launch_gather_rows_mx(x_codes, x_scales, nullptr, T, 1, T, H, nullptr, x_sf_tok, nullptr, status,
                                       st, kPdl) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (mark(2) != cudaSuccess) return MOE_ERR_CUDA;
  moe::W4a8GemmProblem g1{};
  g1.mode = 0;
  g1.a_rows = x8;
  g1.a_sf = x8_sf;
  g1.codes = w13_codes;
  g1.sf = w13_sf;
  g1.offsets = offsets;
  g1.E = E;
  g1.M = P;
  g1.K = H;
  g1.n_out = 2 * I;
  g1.act = act;
  g1.act_sf = act_sf;
  if (sh) {
    g1.s_rows = x_codes;
    g1.s_rows_sf = x_sf_tok;
    g1.s_codes = w13s_codes;
    g1.s_sf = w13s_sf;
    g1.T_s = T;
    g1.n_out_s = 2 * d->I_s;
    g1.s_act = act_s;
    g1.s_act_sf = act_sf_s;
  }
  g1.status = status;
  if (moe::launch_grouped_gemm_w4a8(g1, st, kPdl) != cudaSuccess) return MOE_ERR_CUDA;
  if (mark(3) != cudaSuccess) return MOE_ERR_CUDA;
  // the down projection's K is I for routed experts and I_s for the shared one: one launch covers
  // both only when they agree
  moe::W4a8GemmProblem g2{};
  g2.mode = 1;
  g2.a_rows = act;
  g2.a_sf = act_sf;
  g2.codes = w2_codes;
  g2.sf = w2_sf;
  g2.offsets = offsets;
  g2.E = E;
  g2.M = P;
  g2.K = I;
  g2.n_out = H;
  g2.out = y_perm;
  g2.topk_w = topk_w;
  g2.sorted_pair = sorted_pair;
  g2.status = status;
  moe::W4a8GemmProblem g2s{};
  const bool fused_shared = sh && d->I_s == I;
  if (sh) {
    moe::W4a8GemmProblem& gs = fused_shared ? g2 : g2s;
    gs.s_rows = act_s;
    gs.s_rows_sf = act_sf_s;
    gs.s_codes = w2s_codes;
    gs.s_sf = w2s_sf;
    gs.T_s = T;
    gs.n_out_s = H;
    gs.s_out = shared;
  }
  if (moe::launch_grouped_gemm_w4a8(g2, st, kPdl) != cudaSuccess) return MOE_ERR_CUDA;
  if (sh && !fused_shared) {
    g2s.mode = 1;
    g2s.codes = w2s_codes;
    g2s.sf = w2s_sf;
    g2s.E = 1;
    g2s.M = 0;
    g2s.K = d->I_s;
    g2s.n_out = H;
    g2s.status = status;
    if (moe::launch_grouped_gemm_w4a8(g2s, st, kPdl) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (mark(4) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_finalize(y_perm, pair_pos, sh ? shared : nullptr, T, k, H, y, st, kPdl) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cuda_status(mark(5));
}

}  // namespace

extern "C" {

size_t moe_w4a8_layer_workspace_size(const moe_layer_desc* d) {
  if (check_desc_w4a8(d)) return 0;
  return w8_ws(d).total;
}

int moe_layer_forward_w4a8(const moe_layer_desc* d, const uint8_t* x_codes, const uint8_t* x_scales,
                           const float* logits, const float* bias, const uint8_t* w13_codes, const uint8_t* w13_sf,
                           const uint8_t* w2_codes, const uint8_t* w2_sf, const uint8_t* w13s_codes,
                           const uint8_t* w13s_sf, const uint8_t* w2s_codes, const uint8_t* w2s_sf, uint16_t* y,
                           float* topk_w, int32_t* topk_idx, int32_t* counts, void* ws, size_t ws_bytes,
                           void* stream) {
  return layer_forward_w4a8_impl(d, x_codes, x_scales, logits, bias, w13_codes, w13_sf, w2_codes, w2_sf, w13s_codes,
                                 w13s_sf, w2s_codes, w2s_sf, y, topk_w, topk_idx, counts, ws, ws_bytes, stream,
                                 nullptr);
}

int moe_layer_forward_w4a8_events(const moe_layer_desc* d, const uint8_t* x_codes, const uint8_t* x_scales,
                                  const float* logits, const float* bias, const uint8_t* w13_codes,
                                  const uint8_t* w13_sf, const uint8_t* w2_codes, const uint8_t* w2_sf,
                                  const uint8_t* w13s_codes, const uint8_t* w13s_sf, const uint8_t* w2s_codes,
                                  const uint8_t* w2s_sf, uint16_t* y, float* topk_w, int32_t* topk_idx,
                                  int32_t* counts, void* ws, size_t ws_bytes, void* stream, void* const* events,
                                  int n_events) {
  if (!events || n_events != 6) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 6; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return layer_forward_w4a8_impl(d, x_codes, x_scales, logits, bias, w13_codes, w13_sf, w2_codes, w2_sf, w13s_codes,
                                 w13s_sf, w2s_codes, w2s_sf, y, topk_w, topk_idx, counts, ws, ws_bytes, stream,
                                 events);
}

int moe_w4a8_layer_kernel_launches(const moe_layer_desc* d) {
  if (check_desc_w4a8(d) || d->T == 0) return 0;
  // gating 1 + routing 3 (both in 1 for a small batch) + MXFP8 row gather 1 (+1 for the shared
  // expert's scale rows) + gate/up GEMM 1 + down GEMM 1 (+1 when I_s != I) + finalize 1
  const bool sh = d->n_shared > 0;
  const bool small = moe::gate_route_small_fits(d->T, d->E, d->k);
  return (small ? 1 : 4) + 4 + (sh ? 1 : 0) + ((sh && d->I_s != d->I) ? 1 : 0);
}

}  // extern "C"
