// a2. Init-routing on GB300: per-expert counts, offsets, a stable sort of the
// token-expert pairs by expert (and its inverse), and the row gather x_exp.
//
// Source: Qwen3-MoE low-latency inference practice, "GMM enablement and
// routing optimisation" (init-routing gives the expert sort order;
// compute-expert-tokens gives each expert's token count); Hy3 295B MoE
// practice, section 6.2 (group_list = per-expert token counts).
//
// Design: the P = T*k pairs are cut into chunks of CH consecutive pairs, one
// warp per chunk.
//   1. hist:    each warp counts its chunk per expert (shared-memory atomics;
//               counts do not depend on order).
//   2. scan:    one CTA turns the chunk histograms into counts, offsets and,
//               for every (chunk, expert), the first output position.
//   3. scatter: each warp walks its chunk in ascending pair order, 32 pairs at
//               a time; __match_any_sync groups lanes with the same expert and
//               the rank inside the group is the number of lower lanes in it,
//               so positions follow pair order exactly (a stable sort) with no
//               atomics deciding the order.
//   4. expand:  x_exp[pos] = x[sorted_pair[pos] / k], 16-byte vector copies,
//               several independent ones per thread.
//
// Expert range: with a local slice [e0, e0 + EL) of the E experts (routing that
// keeps only the pairs whose expert this device owns, the expert-parallel form of
// init-routing: Qwen3-MoE practice, W4A8 EP section, "init_routing_v2 ... only the
// tokens in this rank's expert range"), the histograms, counts and offsets cover the
// EL local experts, sorted_pair lists only local pairs (local expert order, then
// pair order), and pair_pos is -1 for every other pair.  The whole range (e0 = 0,
// EL = E) is ordinary init-routing.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) route_hist_kernel(const int32_t* __restrict__ idx, int P, int E,
                                                                 int e0, int EL, int CH, int n_chunks,
                                                                 int32_t* __restrict__ hist, unsigned* status) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kWarps + warp;
  if (c >= n_chunks) return;
  int* h = sh + warp * EL;
  for (int e = lane; e < EL; e += 32) h[e] = 0;
  __syncwarp();
  const int p0 = c * CH, p1 = min(P, p0 + CH);
  bool bad = false;
#pragma unroll 8
  for (int p = p0 + lane; p < p1; p += 32) {
    const int e = __ldg(idx + p);
    if ((unsigned)e >= (unsigned)E)
      bad = true;
    else if ((unsigned)(e - e0) < (unsigned)EL)
      atomicAdd(&h[e - e0], 1);
  }
  if (bad) set_status(status, DEV_ERR_BOUNDS);
  __syncwarp();
  for (int e = lane; e < EL; e += 32) hist[(size_t)c * EL + e] = h[e];
}

// One CTA of 1024 threads: thread (seg, e) owns expert e over the seg-th slice of chunks.
__global__ void __launch_bounds__(1024) route_scan_kernel(const int32_t* __restrict__ hist,
                                                          int32_t* __restrict__ base, int n_chunks, int E,
                                                          int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offsets,
                                                          unsigned* __restrict__ zero, int n_zero) {
  __shared__ int part[1024];
  __shared__ int excl_s[1024];
  __shared__ int wsum[32];
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < n_zero; i += 1024) zero[i] = 0u;
  const int S = max(1, 1024 / E);
  const int e = tid % E, seg = tid / E;
  const bool active = seg < S;
  const int cps = (n_chunks + S - 1) / S;
  const int c0 = min(n_chunks, seg * cps), c1 = min(n_chunks, c0 + cps);
  // A thread's chunk histograms are all loaded at once and kept in registers for the second pass when
  // there are at most kReg of them (one load latency instead of four); otherwise they are read kU at a
  // time, twice.
  constexpr int kReg = 32, kU = 16;
  const bool in_regs = c1 - c0 <= kReg;
  int hv[kReg];
  if (active) {
    int s = 0;
    if (in_regs) {
#pragma unroll
      for (int u = 0; u < kReg; ++u) hv[u] = c0 + u < c1 ? __ldg(hist + (size_t)(c0 + u) * E + e) : 0;
#pragma unroll
      for (int u = 0; u < kReg; ++u) s += hv[u];
    } else {
      int c = c0;
      for (; c + kU <= c1; c += kU) {
        int v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) v[u] = __ldg(hist + (size_t)(c + u) * E + e);
#pragma unroll
        for (int u = 0; u < kU; ++u) s += v[u];
      }
      for (; c < c1; ++c) s += __ldg(hist + (size_t)c * E + e);
    }
    part[seg * E + e] = s;
  }
  __syncthreads();
  int v = 0;
  if (tid < E) {
    for (int g = 0; g < S; ++g) v += part[g * E + tid];
    counts[tid] = v;
  }
  // block-wide exclusive scan of v over tid (E <= 1024)
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  const int incl = x + (warp > 0 ? wsum[warp - 1] : 0);
  if (tid < E) {
    excl_s[tid] = incl - v;
    offsets[tid] = incl - v;
    if (tid == E - 1) offsets[E] = incl;
  }
  __syncthreads();
  if (active && in_regs) {
    int run = excl_s[e];
    for (int g = 0; g < seg; ++g) run += part[g * E + e];
#pragma unroll
    for (int u = 0; u < kReg; ++u)
      if (c0 + u < c1) {
        base[(size_t)(c0 + u) * E + e] = run;
        run += hv[u];
      }
  } else if (active) {
    int run = excl_s[e];
    for (int g = 0; g < seg; ++g) run += part[g * E + e];
    int c = c0;
    for (; c + kU <= c1; c += kU) {
      int v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) v[u] = __ldg(hist + (size_t)(c + u) * E + e);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        base[(size_t)(c + u) * E + e] = run;
        run += v[u];
      }
    }
    for (; c < c1; ++c) {
      base[(size_t)c * E + e] = run;
      run += __ldg(hist + (size_t)c * E + e);
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32) route_scatter_kernel(const int32_t* __restrict__ idx, int P,
                                                                    int e0, int E, int CH, int n_chunks,
                                                                    const int32_t* __restrict__ base,
                                                                    int32_t* __restrict__ sorted_pair,
                                                                    int32_t* __restrict__ pair_pos) {
  // E here is the number of local experts (the histogram width); e0 the first one.
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int sh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kWarps + warp;
  if (c >= n_chunks) return;
  int* cnt = sh + warp * E;
  for (int e = lane; e < E; e += 32) cnt[e] = base[(size_t)c * E + e];
  __syncwarp();
  const int p0 = c * CH, p1 = min(P, p0 + CH);
  const unsigned lower = (1u << lane) - 1u;
  constexpr int kBatch = 8;  // steps whose expert indices are loaded together
  for (int pg = p0; pg < p1; pg += 32 * kBatch) {
    int ev[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int p = pg + b * 32 + lane;
      ev[b] = (p < p1) ? __ldg(idx + p) - e0 : -1;  // local expert index
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (pg + b * 32 >= p1) break;  // warp-uniform
      const int p = pg + b * 32 + lane;
      const int e = ev[b];
      const bool ok = (unsigned)e < (unsigned)E;
      const int key = ok ? e : -1 - lane;  // lanes without a valid expert form singleton groups
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      const int rank = __popc(peers & lower);
      const int bs = ok ? cnt[e] : 0;
      __syncwarp();
      if (ok) {
        const int pos = bs + rank;
        if ((unsigned)pos < (unsigned)P) {
          sorted_pair[pos] = p;
          pair_pos[p] = pos;
        }
        if ((peers >> lane) == 1u) cnt[e] = bs + __popc(peers);  // highest lane of the group
      } else if (p < p1) {
        pair_pos[p] = -1;  // not routed here (outside the local expert range, or an invalid index)
      }
      __syncwarp();
    }
  }
}

// x_exp[pos] = x[sorted_pair[pos] / k].  A block moves kExpandRows consecutive rows of x_exp;
// its threads stride over the 16-byte words of a row, and each thread loads its word of every
// one of the block's rows before storing any, so kExpandRows independent loads per thread are
// in flight.  Indices are 32-bit: row * H8 + column stays below 2^31 words per row block.
constexpr int kExpandRows = 4;

__global__ void __launch_bounds__(512) expand_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ sorted_pair, int P, int k,
                                                          int T, int H8, uint4* __restrict__ x_exp,
                                                          const int32_t* __restrict__ n_rows,
                                                          unsigned* __restrict__ status) {
  pdl_wait();
  pdl_launch_dependents();
  if (n_rows) P = min(P, __ldg(n_rows));  // rows routed here (an expert range routes fewer than P)
  const int r0 = blockIdx.x * kExpandRows;
  const uint4* src[kExpandRows];
  bool bad = false;
#pragma unroll
  for (int u = 0; u < kExpandRows; ++u) {
    src[u] = nullptr;
    if (r0 + u < P) {
      const int sp = __ldg(sorted_pair + r0 + u);
      const int t = sp / k;
      if (sp >= 0 && (unsigned)t < (unsigned)T) src[u] = x + (size_t)t * H8;
      else bad = true;
    }
  }
  if (bad && threadIdx.x == 0) set_status(status, DEV_ERR_BOUNDS);
  uint4* dst = x_exp + (size_t)r0 * H8;
  for (int c = threadIdx.x; c < H8; c += blockDim.x) {
    uint4 v[kExpandRows];
#pragma unroll
    for (int u = 0; u < kExpandRows; ++u)
      if (src[u]) v[u] = __ldg(src[u] + c);
#pragma unroll
    for (int u = 0; u < kExpandRows; ++u)
      if (src[u]) dst[u * H8 + c] = v[u];
  }
}

}  // namespace

int routing_chunk_pairs(int P) {
  if (P <= 4096) return 32;  // decode-sized: one 32-pair step per warp, up to 128 warps
  int ch = (P + 255) / 256;
  ch = (ch + 31) / 32 * 32;
  return ch < 512 ? 512 : ch;
}

size_t routing_scratch_bytes(int P, int E) {
  const int CH = routing_chunk_pairs(P);
  const size_t n_chunks = (size_t)((P + CH - 1) / CH);
  return 2 * n_chunks * (size_t)E * sizeof(int32_t);
}

cudaError_t launch_expand_rows(const uint16_t* x, const int32_t* sorted_pair, int P, int k, int H,
                               uint16_t* x_exp, cudaStream_t stream, bool pdl, const int32_t* n_rows, int T,
                               unsigned* status) {
  if (P == 0) return cudaSuccess;
  if (T < 0) T = P / k;
  const int H8 = H / 8;
  const int threads = H8 >= 512 ? 512 : (H8 + 31) / 32 * 32;
  return launch_kernel(expand_rows_kernel, dim3((unsigned)((P + kExpandRows - 1) / kExpandRows)), dim3(threads), 0,
                       stream, pdl, reinterpret_cast<const uint4*>(x), sorted_pair, P, k, T, H8,
                       reinterpret_cast<uint4*>(x_exp), n_rows, status);
}

cudaError_t launch_init_routing(const int32_t* topk_idx, int P, int E, int k, const uint16_t* x, int H,
                                uint16_t* x_exp, int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                                int32_t* pair_pos, int32_t* scratch, unsigned* status, cudaStream_t stream,
                                bool pdl, unsigned* zero, int n_zero, int e0, int e1) {
  if (e1 < 0) e1 = E;
  const int EL = e1 - e0;  // local experts: [e0, e1)
  const int CH = routing_chunk_pairs(P);
  const int n_chunks = (P + CH - 1) / CH;
  int32_t* hist = scratch;
  int32_t* base = scratch + (size_t)n_chunks * EL;
  const size_t smem = (size_t)kWarps * EL * sizeof(int);
  const int blocks = (n_chunks + kWarps - 1) / kWarps;
  cudaError_t err;
  if (smem > 48 * 1024) {
    err = cudaFuncSetAttribute(route_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(route_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  if (n_chunks > 0) {
    err = launch_kernel(route_hist_kernel, dim3(blocks), dim3(kWarps * 32), smem, stream, pdl, topk_idx, P, E, e0,
                        EL, CH, n_chunks, hist, status);
    if (err != cudaSuccess) return err;
  }
  err = launch_kernel(route_scan_kernel, dim3(1), dim3(1024), 0, stream, pdl, (const int32_t*)hist, base, n_chunks,
                      EL, counts, offsets, zero, n_zero);
  if (err != cudaSuccess) return err;
  if (n_chunks > 0) {
    err = launch_kernel(route_scatter_kernel, dim3(blocks), dim3(kWarps * 32), smem, stream, pdl, topk_idx, P, e0,
                        EL, CH, n_chunks, (const int32_t*)base, sorted_pair, pair_pos);
    if (err != cudaSuccess) return err;
  }
  if (x != nullptr && x_exp != nullptr)
    return launch_expand_rows(x, sorted_pair, P, k, H, x_exp, stream, pdl, EL < E ? offsets + EL : nullptr);
  return cudaSuccess;
}

}  // namespace moe
