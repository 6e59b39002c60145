// a3/a4. Grouped expert GEMMs on GB300: tcgen05 (5th-gen tensor cores) with
// the accumulator in TMEM, operands staged by TMA, one persistent CTA per SM.
//
// Source: Qwen3-MoE low-latency inference practice, "GMM enablement and
// routing optimisation" (all experts' matmuls in one grouped op instead of a
// per-expert loop) and "MoE TP optimisation: computation decomposition"
// (x = down(SiLU(gate(x)) * up(x)), gate/up concatenated as w13, SwiGLU =
// SiLU(first half) * second half); Hy3 295B MoE practice, section 6.2 (the
// grouped matmul walks per-expert token counts; expert weights keep the
// checkpoint [out_features, in_features] layout) and 1.1 (one shared expert).
//
// Layout of the product: the WEIGHT rows are the UMMA M operand (128 output
// features per tile) and the expert's TOKEN rows are the N operand (16..256
// columns, chosen per tile as the rows actually present, rounded up to 16).
// Decode has 1-8 rows per expert, so this keeps the tensor core work
// proportional to the real rows while every weight byte is streamed once.
// Both operands are K-major in global memory and land in shared memory as
// 128-byte swizzled rows (64 bf16 of K per stage).
//
//   tile = (segment, feature tile f, token tile m); segments are the routed
//   experts in order, then optionally one dense "shared" segment over all T
//   rows.  Tiles of one expert are numbered f-major so that the token tiles
//   that reuse a weight tile run next to each other (L2 reuse).
//
// Warp roles (192 threads, 1 CTA/SM, static round-robin tile schedule):
//   warp 0      TMA producer: per stage 8 boxes of 16 weight rows + up to 16
//               boxes of 16 token rows, one lane per box.
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//               (M=128, N=rows, K=16 x 4 per stage), double-buffered accumulator.
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 16 columns, then
//               mode 0 (w13): SwiGLU.  The w13 tile is loaded so that in each
//                 32-row quarter, rows 0-15 are gate features and rows 16-31 the
//                 matching up features; a shfl_xor(16) pairs them in registers.
//               mode 1 (down): multiply by the routing weight of the row.
// Every wait is bounded (default 2 s); on expiry the CTA raises an abort flag,
// records DEV_ERR_TIMEOUT, drains its in-flight copies and MMAs and frees TMEM.
#include "moe_common.cuh"
#include "moe_internal.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kBM = 128;                     // weight rows per tile (UMMA M)
constexpr int kBK = 64;                      // K per stage: one 128-byte swizzle row of bf16
constexpr int kBoxRows = 16;                 // rows per TMA box
constexpr int kBoxBytes = kBoxRows * kBK * 2;  // 2 KB
constexpr int kABytes = kBM * kBK * 2;       // 16 KB
constexpr int kThreads = 192;
constexpr unsigned long long kTimeoutNs = 2000000000ull;

struct GemmParams {
  const int32_t* offsets;
  int E, M, K;
  int n_out, n_ftiles, half;        // routed: rows per expert, feature tiles, up-half row offset (mode 0)
  uint16_t* out;
  int ld_out;
  int has_shared, T_s, n_out_s, n_ftiles_s, half_s;
  uint16_t* s_out;
  int ld_out_s;
  int NT;                           // token rows per tile (multiple of 16)
  const float* topk_w;
  const int32_t* sorted_pair;
  unsigned* status;
  unsigned long long timeout_ns;
};

template <int NTMAX, int STAGES>
struct Layout {
  static constexpr int kBBytes = NTMAX * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;  // multiple of 1024
  static constexpr int kBarOff = STAGES * kStageBytes;
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kTabOff = kMiscOff + 16;
  static constexpr uint32_t kTmemCols = (2 * NTMAX <= 32) ? 32 : (2 * NTMAX <= 64 ? 64 : (2 * NTMAX <= 128 ? 128 : (2 * NTMAX <= 256 ? 256 : 512)));
  static size_t bytes(int E) { return 1024 + kTabOff + 2 * (size_t)(E + 1) * 4; }
};

struct Tile {
  int shared, e, f, row_base, rows;
};

__device__ __forceinline__ Tile decode_tile(int tile, int routed_total, const int* s_off, const int* s_tt,
                                            const GemmParams& p) {
  Tile t;
  if (tile < routed_total) {
    const int q = tile / p.n_ftiles;
    int lo = 0, hi = p.E;  // s_tt[lo] <= q < s_tt[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tt[mid] <= q) lo = mid; else hi = mid;
    }
    const int nt = s_tt[lo + 1] - s_tt[lo];
    const int local = tile - s_tt[lo] * p.n_ftiles;
    const int m = local % nt;
    t.shared = 0;
    t.e = lo;
    t.f = local / nt;
    t.row_base = s_off[lo] + m * p.NT;
    t.rows = min(p.NT, s_off[lo + 1] - t.row_base);
  } else {
    const int local = tile - routed_total;
    const int nt = (p.T_s + p.NT - 1) / p.NT;
    const int m = local % nt;
    t.shared = 1;
    t.e = -1;
    t.f = local / nt;
    t.row_base = m * p.NT;
    t.rows = min(p.NT, p.T_s - t.row_base);
  }
  return t;
}

template <int NTMAX, int STAGES, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmAs, const __grid_constant__ CUtensorMap tmBs,
                        const GemmParams p) {
  using L = Layout<NTMAX, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  volatile int* cfg_bad = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 8);
  int* s_off = reinterpret_cast<int*>(smem + L::kTabOff);
  int* s_tt = s_off + (p.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    *cfg_bad = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (p.has_shared) {
      tma_prefetch_desc(&tmAs);
      tma_prefetch_desc(&tmBs);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, L::kTmemCols);
  for (int i = threadIdx.x; i <= E; i += kThreads) s_off[i] = p.offsets ? __ldg(p.offsets + i) : 0;
  __syncthreads();
  if (warp == 2) {
    // Validate offsets and build the prefix of token tiles per expert.
    const int per = (E + 31) >> 5;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int sum = 0;
    bool bad = (lane == 0) && (s_off[0] < 0 || s_off[E] > p.M);
    for (int e = e0; e < e1; ++e) {
      const int n = s_off[e + 1] - s_off[e];
      if (n < 0) bad = true;
      else sum += (n + p.NT - 1) / p.NT;
    }
    int x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    int run = x - sum;
    for (int e = e0; e < e1; ++e) {
      s_tt[e] = run;
      const int n = s_off[e + 1] - s_off[e];
      run += n > 0 ? (n + p.NT - 1) / p.NT : 0;
    }
    if (lane == 31) s_tt[E] = x;
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
      *cfg_bad = 1;
      set_status(p.status, DEV_ERR_CONFIG);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int routed_total = *cfg_bad ? 0 : s_tt[E] * p.n_ftiles;
  const int shared_total = (*cfg_bad || !p.has_shared) ? 0 : ((p.T_s + p.NT - 1) / p.NT) * p.n_ftiles_s;
  const int total = routed_total + shared_total;
  const int KB = p.K / kBK;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      const Tile t = decode_tile(tile, routed_total, s_off, s_tt, p);
      const CUtensorMap* mA = t.shared ? &tmAs : &tmA;
      const CUtensorMap* mB = t.shared ? &tmBs : &tmB;
      const int nbox = (t.rows + kBoxRows - 1) / kBoxRows;
      const int a_row0 = t.shared ? 0 : t.e * p.n_out;
      const int half = t.shared ? p.half_s : p.half;
      int a_row;
      if (MODE == 0)  // box i: quarter i/2, gate (i even) or up (i odd) half, 16 features
        a_row = a_row0 + (lane & 1) * half + t.f * 64 + (lane >> 1) * kBoxRows;
      else
        a_row = a_row0 + t.f * kBM + lane * kBoxRows;
      for (int kb = 0; kb < KB; ++kb) {
        bool w = (lane == 0) ? mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.timeout_ns, p.status)
                             : false;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[stage], kABytes + nbox * kBoxBytes);
        __syncwarp();
        uint8_t* sA = smem + stage * L::kStageBytes;
        uint8_t* sB = sA + kABytes;
        if (lane < 8) {
          tma_load_2d(sA + lane * kBoxBytes, mA, kb * kBK, a_row, &full[stage], pol_w);
        } else if (lane < 8 + nbox) {
          const int j = lane - 8;
          tma_load_2d(sB + j * kBoxBytes, mB, kb * kBK, t.row_base + j * kBoxRows, &full[stage], pol_x);
        }
        __syncwarp();
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Drain: the last fill of every stage must have landed before the CTA exits.
    if (lane == 0) {
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t n = issued / STAGES + ((uint32_t)s < issued % STAGES ? 1u : 0u);
        if (n) mbar_wait_bounded(&full[s], (n - 1u) & 1u, abort_flag, p.timeout_ns, p.status, false);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++it) {
        const Tile t = decode_tile(tile, routed_total, s_off, s_tt, p);
        const int buf = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_bounded(&tempty[buf], aph ^ 1u, abort_flag, p.timeout_ns, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * NTMAX);
        const int nmma = (t.rows + 15) & ~15;
        const uint32_t idesc = umma_idesc_bf16(kBM, nmma);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(smem + stage * L::kStageBytes);
          const uint32_t b = a + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16(d, umma_desc_sw128(a + kk * 32), umma_desc_sw128(b + kk * 32), idesc, (kb | kk) != 0);
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[buf]);
      }
      // Drain: every MMA issued by this thread must be complete before TMEM is freed.
      umma_commit(done);
      mbar_wait_bounded(done, 0, abort_flag, p.timeout_ns, p.status, false);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int qw = warp & 3;  // TMEM lane quarter this warp may access
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const Tile t = decode_tile(tile, routed_total, s_off, s_tt, p);
      const int buf = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      bool w = (lane == 0) ? mbar_wait_bounded(&tfull[buf], aph, abort_flag, p.timeout_ns, p.status) : false;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(qw * 32) << 16) + (uint32_t)(buf * NTMAX);
      const int nch = (t.rows + 15) >> 4;
      uint16_t* out = t.shared ? p.s_out : p.out;
      const size_t ld = (size_t)(t.shared ? p.ld_out_s : p.ld_out);
      if (MODE == 0) {
        const bool is_gate = lane < 16;
        const int feat = t.f * 64 + qw * 16 + (lane & 15);
        for (int c = 0; c < nch; ++c) {
          float v[16];
          tmem_ld16(tb + (uint32_t)(c * 16), v);
          const int col0 = c * 16 + (is_gate ? 0 : 8);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float send = is_gate ? v[8 + i] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
            const float g = is_gate ? v[i] : recv;
            const float u = is_gate ? recv : v[8 + i];
            const float a = g / (1.0f + expf(-g)) * u;
            const int col = col0 + i;
            if (col < t.rows) out[(size_t)(t.row_base + col) * ld + feat] = f32_to_bf16_rne(a);
          }
        }
      } else {
        const int feat = t.f * kBM + qw * 32 + lane;
        const int n_out = t.shared ? p.n_out_s : p.n_out;
        const bool scale = !t.shared && p.topk_w != nullptr;
        for (int c = 0; c < nch; ++c) {
          float v[16];
          tmem_ld16(tb + (uint32_t)(c * 16), v);
          float sc = 1.0f;
          if (scale) {
            const int col = c * 16 + (lane & 15);
            if (col < t.rows) sc = __ldg(p.topk_w + __ldg(p.sorted_pair + t.row_base + col));
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float s = scale ? __shfl_sync(0xffffffffu, sc, i) : 1.0f;
            const int col = c * 16 + i;
            if (col < t.rows && feat < n_out) out[(size_t)(t.row_base + col) * ld + feat] = f32_to_bf16_rne(v[i] * s);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Row-major bf16 matrix [rows, K] as a 2-D tensor map with 64 x 16 boxes and
// the 128-byte swizzle; rows past the end read as zeros.
bool make_map(CUtensorMap* m, const void* base, int K, long long rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBoxRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int NTMAX, int STAGES, int MODE>
cudaError_t launch_instance(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& as,
                            const CUtensorMap& bs, const GemmParams& gp, cudaStream_t stream) {
  using L = Layout<NTMAX, STAGES>;
  auto kern = grouped_gemm_kernel<NTMAX, STAGES, MODE>;
  const size_t smem = L::bytes(gp.E);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  kern<<<num_sms(), kThreads, smem, stream>>>(a, b, as, bs, gp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm(const GroupedGemmProblem& pr, cudaStream_t stream) {
  const bool has_shared = pr.s_rows != nullptr && pr.T_s > 0;
  if (pr.M <= 0 && !has_shared) return cudaSuccess;
  GemmParams gp{};
  gp.offsets = pr.offsets;
  gp.E = pr.E;
  gp.M = pr.M;
  gp.K = pr.K;
  gp.n_out = pr.n_out;
  gp.n_ftiles = pr.mode == 0 ? pr.n_out / 128 : (pr.n_out + kBM - 1) / kBM;
  gp.half = pr.n_out / 2;
  gp.out = pr.out;
  gp.ld_out = pr.ld_out;
  gp.has_shared = has_shared ? 1 : 0;
  gp.T_s = has_shared ? pr.T_s : 0;
  gp.n_out_s = has_shared ? pr.n_out_s : 0;
  gp.n_ftiles_s = has_shared ? (pr.mode == 0 ? pr.n_out_s / 128 : (pr.n_out_s + kBM - 1) / kBM) : 0;
  gp.half_s = has_shared ? pr.n_out_s / 2 : 0;
  gp.s_out = pr.s_out;
  gp.ld_out_s = pr.ld_out_s;
  gp.topk_w = pr.topk_w;
  gp.sorted_pair = pr.sorted_pair;
  gp.status = pr.status;
  gp.timeout_ns = kTimeoutNs;

  // With no routed rows the routed maps are never read: alias the shared ones.
  if (pr.M <= 0) gp.offsets = nullptr;
  CUtensorMap ta, tb, tas, tbs;
  if (pr.M > 0) {
    if (!make_map(&ta, pr.w, pr.K, (long long)pr.E * pr.n_out)) return cudaErrorInvalidValue;
    if (!make_map(&tb, pr.a_rows, pr.K, pr.M)) return cudaErrorInvalidValue;
  }
  if (has_shared) {
    if (!make_map(&tas, pr.s_w, pr.K, pr.n_out_s)) return cudaErrorInvalidValue;
    if (!make_map(&tbs, pr.s_rows, pr.K, pr.T_s)) return cudaErrorInvalidValue;
  }
  if (pr.M <= 0) {
    ta = tas;
    tb = tbs;
  } else if (!has_shared) {
    tas = ta;
    tbs = tb;
  }
  // Token tile: decode-like problems (few rows per expert) use the narrow
  // instance with deep pipelining; prefill-like ones the 256-column instance.
  const bool narrow = (long long)pr.M <= 32LL * pr.E && (!has_shared || pr.T_s <= 32);
  if (narrow) {
    gp.NT = 32;
    return pr.mode == 0 ? launch_instance<32, 10, 0>(ta, tb, tas, tbs, gp, stream)
                        : launch_instance<32, 10, 1>(ta, tb, tas, tbs, gp, stream);
  }
  gp.NT = 256;
  return pr.mode == 0 ? launch_instance<256, 4, 0>(ta, tb, tas, tbs, gp, stream)
                      : launch_instance<256, 4, 1>(ta, tb, tas, tbs, gp, stream);
}

}  // namespace moe
