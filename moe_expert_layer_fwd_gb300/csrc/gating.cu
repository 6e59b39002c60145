// a1. Gating top-k on GB300: one warp per token.
//
// Source: Qwen3-MoE low-latency inference practice, "GMM enablement and
// routing optimisation" (one fused op computes routing scores and the top-k
// experts, replacing top-k then softmax); Hy3 295B MoE practice, section 1.3
// (sigmoid router: sigmoid, top-k, gather, normalise with eps = 1e-20, scale by
// routed_scaling_factor = 2.826) and section 5.1 (the correction bias is added
// after the sigmoid and only decides which experts are chosen; the fused op adds
// it inside the sigmoid instead, MOE_GATE_SIGMOID_INNER_BIAS here).
//
// Each lane holds experts e = lane + 32*i.  The selection key is turned into
// an order-preserving 32-bit integer (0 marks a removed or absent expert).
// Each of k rounds takes the warp-wide maximum key (redux.sync), then the
// lowest expert index holding it (each lane's lowest slot with that key, then
// a warp-wide minimum): "largest key, then lowest index", k experts in order.  The sigmoid key is
// computed with a fixed sequence of IEEE fp32 operations (Cody-Waite reduced
// exp with a degree-7 Taylor polynomial, each multiply and add rounded
// separately), so the choice is reproducible bit for bit on any IEEE machine.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

// e^x by the fixed operation sequence: n = rint(x*log2e); r = (x - n*C1) - n*C2
// with ln2 = C1 + C2 (C1 = 355/512); p = Horner of sum r^m/m!, m <= 7, each
// step one rounded multiply and one rounded add; result p * 2^n.  x is clamped
// to [-87, 88] so 2^n is a normal float.
__device__ __forceinline__ float exp_fixed_f32(float x) {
  x = fminf(fmaxf(x, -87.0f), 88.0f);
  const float n = rintf(__fmul_rn(x, 1.4426950408889634f));
  const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(n, 0.693359375f)), __fmul_rn(n, -2.12194440e-4f));
  float p = 1.0f / 5040.0f;
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 720.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 120.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 24.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 6.0f);
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  const float scale = __int_as_float(((int)n + 127) << 23);
  return __fmul_rn(p, scale);
}

__device__ __forceinline__ float sigmoid_fixed_f32(float l) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, exp_fixed_f32(-l)));
}

// Order-preserving map float -> uint32 (larger float -> larger integer), with
// -0 and +0 mapped to the same value.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  if (f == 0.0f) f = 0.0f;
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// This lane's logits of token t (experts lane + 32 i), 0 past E.
template <int VPL>
__device__ __forceinline__ void load_logits(const float* __restrict__ logits, int t, int E, int lane, float (&raw)[VPL]) {
  const float* row = logits + (size_t)t * E;
#pragma unroll
  for (int i = 0; i < VPL; ++i) raw[i] = lane + 32 * i < E ? __ldg(row + lane + 32 * i) : 0.0f;
}

// Top-k of token t by one warp from its logits already in registers (raw, as load_logits gives them).
// VPL = keys held per lane (E <= 32 * VPL); a compile-time bound keeps them in registers.  Lane j < k
// writes the j-th choice; returns it (-1 on lanes >= k).
template <int VPL>
__device__ __forceinline__ int gate_token_from(const float (&raw)[VPL], const float* __restrict__ logits,
                                               const float* __restrict__ bias, int t, int E, int k, int gate,
                                               float rsf, float eps, float* __restrict__ topk_w,
                                               int32_t* __restrict__ topk_idx, int lane) {
  const float* row = logits + (size_t)t * E;
  uint32_t keys[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    keys[i] = 0u;  // below every real key: never chosen
    const int e = lane + 32 * i;
    if (e < E) {
      const float l = raw[i];
      float key = l;
      if (gate == MOE_GATE_SIGMOID) {
        key = sigmoid_fixed_f32(l);
        if (bias) key = __fadd_rn(key, __ldg(bias + e));
      } else if (gate == MOE_GATE_SIGMOID_INNER_BIAS) {
        key = sigmoid_fixed_f32(bias ? __fadd_rn(l, __ldg(bias + e)) : l);
      }
      keys[i] = ordered_key(key);
    }
  }

  int my_e = -1;  // lane j keeps the j-th chosen expert
  for (int j = 0; j < k; ++j) {
    uint32_t lm = 0u;
#pragma unroll
    for (int i = 0; i < VPL; ++i) lm = keys[i] > lm ? keys[i] : lm;
    const uint32_t m = __reduce_max_sync(0xffffffffu, lm);
    uint32_t cand = 0xFFFFFFFFu;  // this lane's lowest expert holding the maximum key
#pragma unroll
    for (int i = VPL - 1; i >= 0; --i) cand = keys[i] == m ? (uint32_t)(lane + 32 * i) : cand;
    const int e = (int)__reduce_min_sync(0xffffffffu, cand);
    const bool mine = lane == (e & 31);
    const int slot = e >> 5;
#pragma unroll
    for (int i = 0; i < VPL; ++i) keys[i] = (mine && i == slot) ? 0u : keys[i];
    if (lane == j) my_e = e;
  }

  const float l = (lane < k) ? __ldg(row + my_e) : 0.0f;
  const float l0 = __shfl_sync(0xffffffffu, l, 0);  // softmax: slot 0 holds the largest logit
  float w = 0.0f;
  if (lane < k) {
    if (gate == MOE_GATE_SOFTMAX) w = expf(l - l0);
    else if (gate == MOE_GATE_SIGMOID_INNER_BIAS && bias) w = sigmoid_fixed_f32(__fadd_rn(l, __ldg(bias + my_e)));
    else w = sigmoid_fixed_f32(l);
  }
  const float s = warp_sum(w);
  if (lane < k) {
    w = (gate == MOE_GATE_SOFTMAX) ? w / s : w / (s + eps) * rsf;
    topk_w[(size_t)t * k + lane] = w;
    topk_idx[(size_t)t * k + lane] = my_e;
  }
  return lane < k ? my_e : -1;
}

template <int VPL>
__device__ __forceinline__ int gate_token(const float* __restrict__ logits, const float* __restrict__ bias, int t,
                                          int E, int k, int gate, float rsf, float eps, float* __restrict__ topk_w,
                                          int32_t* __restrict__ topk_idx, int lane) {
  float raw[VPL];
  load_logits<VPL>(logits, t, E, lane, raw);
  return gate_token_from<VPL>(raw, logits, bias, t, E, k, gate, rsf, eps, topk_w, topk_idx, lane);
}

// kTPW tokens per warp: all their logits are loaded before the first is gated, so a large batch
// takes one wave of warps with one load latency instead of two.
constexpr int kTPW = 2;

template <int VPL>
__global__ void __launch_bounds__(256) gating_topk_kernel(const float* __restrict__ logits,
                                                          const float* __restrict__ bias, int T, int E, int k,
                                                          int gate, float rsf, float eps,
                                                          float* __restrict__ topk_w,
                                                          int32_t* __restrict__ topk_idx) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int t0 = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kTPW;
  if (t0 >= T) return;
  float raw[kTPW][VPL];
#pragma unroll
  for (int u = 0; u < kTPW; ++u)
    if (t0 + u < T) load_logits<VPL>(logits, t0 + u, E, lane, raw[u]);
#pragma unroll
  for (int u = 0; u < kTPW; ++u)
    if (t0 + u < T) gate_token_from<VPL>(raw[u], logits, bias, t0 + u, E, k, gate, rsf, eps, topk_w, topk_idx, lane);
}

// Gating and init-routing of a small batch (P = T*k <= kSmallPairs) in one CTA of 32 warps: the
// four launches of gating, histogram, scan and scatter become one (decode: their launch and
// hand-over latencies are most of their time).  Same results, bit for bit:
//   1. warp w gates tokens w, w + 32, ...; the choices also go to shared memory (pair order);
//   2. warp w takes pairs [w*CH, (w+1)*CH) and counts them per expert (shared-memory atomics:
//      counts do not depend on order);
//   3. thread e sums expert e over the warps (counts), a block scan gives offsets, and thread e
//      turns the per-warp counts into each warp's first position for expert e;
//   4. warp w walks its pairs in ascending order, 32 at a time: lanes with the same expert are
//      grouped by __match_any_sync and ranked by the lower lanes of their group, so positions
//      follow pair order (the stable sort) with no atomics deciding the order.
constexpr int kSmallPairs = 4096;
constexpr int kSmallWarps = 32;

template <int VPL>
__global__ void __launch_bounds__(kSmallWarps * 32) gate_route_small_kernel(
    const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k, int gate, float rsf,
    float eps, float* __restrict__ topk_w, int32_t* __restrict__ topk_idx, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_pair, int32_t* __restrict__ pair_pos) {
  extern __shared__ int sh[];
  const int P = T * k;
  int* idx_s = sh;                               // [P] the chosen expert of every pair
  int* hist = sh + kSmallPairs;                  // [kSmallWarps][E] counts, then first positions
  __shared__ int wsum[kSmallWarps];
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  for (int i = tid; i < kSmallWarps * E; i += blockDim.x) hist[i] = 0;
  for (int t = warp; t < T; t += kSmallWarps) {
    const int e = gate_token<VPL>(logits, bias, t, E, k, gate, rsf, eps, topk_w, topk_idx, lane);
    if (lane < k) idx_s[t * k + lane] = e;
  }
  __syncthreads();
  const int CH = ((P + kSmallWarps - 1) / kSmallWarps + 31) & ~31;  // pairs per warp, whole steps
  const int p0 = min(P, warp * CH), p1 = min(P, p0 + CH);
  int* h = hist + warp * E;
  for (int p = p0 + lane; p < p1; p += 32) atomicAdd(&h[idx_s[p]], 1);
  __syncthreads();
  // per expert: total, then (after the scan) each warp's first position
  int v = 0;
  for (int e = tid; e < E; e += blockDim.x)  // E <= 1024 = blockDim.x: at most one expert per thread
    for (int w = 0; w < kSmallWarps; ++w) v += hist[w * E + e];
  if (tid < E) counts[tid] = v;
  int x = v;  // block-wide exclusive scan of v over tid
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int ws = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ws, o);
      if (lane >= o) ws += y;
    }
    wsum[lane] = ws;
  }
  __syncthreads();
  const int excl = x + (warp > 0 ? wsum[warp - 1] : 0) - v;
  if (tid < E) {
    offsets[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + v;
    int run = excl;
    for (int w = 0; w < kSmallWarps; ++w) {
      const int c = hist[w * E + tid];
      hist[w * E + tid] = run;
      run += c;
    }
  }
  __syncthreads();
  const unsigned lower = (1u << lane) - 1u;
  for (int pg = p0; pg < p1; pg += 32) {  // warp-uniform
    const int p = pg + lane;
    const bool ok = p < p1;
    const int e = ok ? idx_s[p] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1 - lane);
    const int rank = __popc(peers & lower);
    const int bs = ok ? h[e] : 0;
    __syncwarp();
    if (ok) {
      const int pos = bs + rank;
      sorted_pair[pos] = p;
      pair_pos[p] = pos;
      if ((peers >> lane) == 1u) h[e] = bs + __popc(peers);  // highest lane of the group
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_gating_topk(const float* logits, const float* bias, int T, int E, int k, int gate, float rsf,
                               float eps, float* topk_w, int32_t* topk_idx, cudaStream_t stream, bool pdl) {
  if (T == 0) return cudaSuccess;
  const int warps = 8;
  dim3 grid((T + warps * kTPW - 1) / (warps * kTPW));
  const int vpl = (E + 31) / 32;
#define MOE_GATING_LAUNCH(V)                                                                                 \
  launch_kernel(gating_topk_kernel<V>, grid, dim3(warps * 32), 0, stream, pdl, logits, bias, T, E, k, gate, rsf, \
                eps, topk_w, topk_idx)
  if (vpl <= 1) return MOE_GATING_LAUNCH(1);
  if (vpl <= 2) return MOE_GATING_LAUNCH(2);
  if (vpl <= 4) return MOE_GATING_LAUNCH(4);
  if (vpl <= 8) return MOE_GATING_LAUNCH(8);
  if (vpl <= 16) return MOE_GATING_LAUNCH(16);
  return MOE_GATING_LAUNCH(32);
#undef MOE_GATING_LAUNCH
}

bool gate_route_small_fits(int T, int E, int k) {
  return (long long)T * k <= kSmallPairs && E <= 1024 && k <= 32;
}

cudaError_t launch_gate_route_small(const float* logits, const float* bias, int T, int E, int k, int gate, float rsf,
                                    float eps, float* topk_w, int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                                    int32_t* sorted_pair, int32_t* pair_pos, cudaStream_t stream, bool pdl) {
  if (T == 0) return cudaSuccess;
  if (!gate_route_small_fits(T, E, k)) return cudaErrorInvalidValue;
  const size_t smem = (size_t)(kSmallPairs + kSmallWarps * E) * sizeof(int);
  const int vpl = (E + 31) / 32;
#define MOE_SMALL_LAUNCH(V)                                                                                        \
  do {                                                                                                             \
    cudaError_t err = cudaFuncSetAttribute(gate_route_small_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                           (int)smem);                                                             \
    if (err != cudaSuccess) return err;                                                                            \
    return launch_kernel(gate_route_small_kernel<V>, dim3(1), dim3(kSmallWarps * 32), smem, stream, pdl, logits,    \
                         bias, T, E, k, gate, rsf, eps, topk_w, topk_idx, counts, offsets, sorted_pair, pair_pos);  \
  } while (0)
  if (vpl <= 1) MOE_SMALL_LAUNCH(1);
  if (vpl <= 2) MOE_SMALL_LAUNCH(2);
  if (vpl <= 4) MOE_SMALL_LAUNCH(4);
  if (vpl <= 8) MOE_SMALL_LAUNCH(8);
  if (vpl <= 16) MOE_SMALL_LAUNCH(16);
  MOE_SMALL_LAUNCH(32);
#undef MOE_SMALL_LAUNCH
}

}  // namespace moe
