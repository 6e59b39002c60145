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
// Layout of the product: the WEIGHT rows are the UMMA M operand and the
// expert's TOKEN rows are the N operand (16..256 columns, chosen per tile as
// the rows actually present, rounded up to 16).  Decode has 1-8 rows per
// expert, so this keeps the tensor core work proportional to the real rows
// while every weight byte is streamed once.  Both operands are K-major in
// global memory and land in shared memory as 128-byte swizzled rows (64 bf16
// of K per stage).
//
// The gate/up weight (mode 0) is read in the packed layout of
// moe_prepack_w13: in every 32-row group the first 16 rows are gate rows and
// the next 16 the up rows of the same 16 features, so a 128-row box holds 64
// whole features and, in TMEM, lane l and lane l^16 of each warp hold the
// gate and the up value of one feature: shfl_xor(16) pairs them for SwiGLU.
//
//   tile = (segment, feature tile f, token tile m); segments are the routed
//   experts in order, then optionally one dense "shared" segment over all T
//   rows.  Inside a segment tiles run f-major (the token tiles that reuse a
//   weight tile run next to each other) unless the segment has more token rows
//   than weight rows, then m-major (the feature tiles that reuse a token tile
//   run together and the segment's weights stay in L2).
//
// Few, large TMA boxes: the per-SM rate of TMA box operations, not their
// bytes, limits a stream of small boxes, so each stage moves the weight rows
// in 128-row boxes (16 KB) and the token rows in BBOX-row boxes.
//
// Two instance families:
//   PAIR = 1 (decode-like, 32 token columns): one CTA per tile, cta_group::1
//     UMMA M=128; APARTS weight boxes per stage, each into its own accumulator.
//   PAIR = 2 (prefill-like, 256 token columns): a cluster of two CTAs computes
//     one tile with the 2-SM UMMA (cta_group::2, M=256): each CTA stages its
//     own 128 weight rows and HALF of the token rows, so shared-memory traffic
//     per FLOP is half that of a 1-SM 128x256 tile; the 1-SM kernel is bound by
//     shared-memory bandwidth (operand reads plus TMA writes) at prefill sizes.
//     The leader CTA (rank 0) issues the MMAs; both CTAs' TMA loads complete on
//     the leader's barriers; MMA commits are multicast to both CTAs.
//
// Warp roles (64 + 32*(EPI + GW) threads per CTA, 1 CTA/SM, static round-robin tiles):
//   warp 0      TMA producer (one lane per box).
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer (the leader's
//               only, when PAIR = 2), double-buffered accumulator.
//   warps 2..   epilogue, EPI/4 warps per TMEM lane quarter taking interleaved
//               32-column chunks: tcgen05.ld 32 lanes x 32 columns, then
//               mode 0 (w13): SwiGLU = SiLU(gate) * up in fp32;
//               mode 1 (down): multiply by the routing weight of the row.
//   warps 2+EPI.. GW row-gather warps (the CTA-pair gate/up instances): copy the
//               routed token rows x[sorted_pair / k] into x_exp while the GEMM
//               runs, publishing one flag per 16 rows that the producer waits on.
// Every wait is bounded (default 2 s); on expiry the CTA raises an abort flag,
// records DEV_ERR_TIMEOUT, drains its in-flight copies and MMAs and frees TMEM.
#include "moe_common.cuh"
#include "moe_internal.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kBM = 128;                     // weight rows per box (UMMA M per CTA)
constexpr int kBK = 64;                      // K per chunk: one 128-byte swizzle row of bf16
constexpr int kRowBytes = kBK * 2;           // 128 B per operand row per chunk
constexpr int kABox = kBM * kRowBytes;       // one 128-row weight box: 16 KB
constexpr int kMaxDynSmem = 232448;          // 227 KB per CTA
constexpr unsigned long long kTimeoutNs = 2000000000ull;

struct GemmParams {
  const int32_t* offsets;
  int E, M, K;
  int n_out, n_ftiles;              // routed: weight rows per expert, feature tiles per expert
  int n_feat;                       // output features per row (I in mode 0, N in mode 1)
  uint16_t* out;
  int ld_out;
  int has_shared, T_s, n_out_s, n_ftiles_s, n_feat_s;
  uint16_t* s_out;
  int ld_out_s;
  int NT;                           // token rows per tile (multiple of 16)
  const float* topk_w;
  const int32_t* sorted_pair;
  unsigned* status;
  unsigned long long timeout_ns;
  // In-kernel row gather (mode 0 with gather warps; g_flags == nullptr: off).  The routed token
  // rows are then copied x -> a_rows (= g_xexp) by the gather warps while the GEMM runs:
  // a_rows[pos] = x[sorted_pair[pos] / k], in chunks of kGatherRows rows whose flags
  // (zeroed before the launch) are set once the chunk is written.
  const uint4* g_x;
  const int32_t* g_sp;
  uint4* g_xexp;
  int g_k, g_T, g_H8;
  unsigned* g_flags;
  int g_skip;  // failure injection (tests only): nobody gathers, so no flag is ever set
};

constexpr int kGatherRows = 16;  // rows per gather chunk (one flag each)

// Acquire load of a flag written with release semantics by another CTA.
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders this thread's generic-proxy global accesses with its async-proxy (TMA) ones.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

template <int NTMAX, int STAGES, int MODE, int BBOX, int EPI, int APARTS, int PAIR, int KC, int GW>
struct Layout {
  static constexpr int kThreads = 64 + 32 * (EPI + GW);          // producer, MMA, EPI epilogue, GW gather warps
  static constexpr int kBRows = NTMAX / PAIR;                    // token rows staged by one CTA
  // A stage holds KC chunks of K = 64 (one 128-byte swizzle row each): KC x [APARTS weight
  // boxes], then KC x [kBRows token rows].  The tensor pipe only runs at full rate when the
  // MMA thread issues about 8 MMAs between two waits, so CTA pairs (4 MMAs per chunk) use KC = 2.
  static constexpr int kAChunk = APARTS * kABox;
  static constexpr int kBChunk = kBRows * kRowBytes;
  static constexpr int kABytes = KC * kAChunk;
  static constexpr int kBBytes = KC * kBChunk;
  static constexpr int kStageK = KC * kBK;
  static constexpr int kStageBytes = kABytes + kBBytes;          // multiple of 1024
  static constexpr int kBarOff = STAGES * kStageBytes;
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kScaleOff = kMiscOff + 16;                // mode 1: per-epilogue-warp row scales
  static constexpr int kTabOff = kScaleOff + (MODE == 1 ? EPI * NTMAX * 4 : 0);  // then offsets, tile starts
  static constexpr int kAccCols = APARTS * NTMAX;                // TMEM columns of one accumulator buffer
  static constexpr uint32_t kTmemCols = (2 * kAccCols <= 32) ? 32 : (2 * kAccCols <= 64 ? 64 : (2 * kAccCols <= 128 ? 128 : (2 * kAccCols <= 256 ? 256 : 512)));
  static constexpr int kFeatPerBox = MODE == 0 ? 64 : 128;       // output features of one weight box
  static constexpr int kFeatPerTile = kFeatPerBox * APARTS * PAIR;
  static_assert(2 * kAccCols <= 512, "accumulators exceed TMEM");
  static_assert(kBRows % BBOX == 0 && KC * (kBRows / BBOX) <= 24 && KC * APARTS <= 8, "boxes per stage");
  static_assert(kAChunk % 1024 == 0 && kBChunk % 1024 == 0, "chunk alignment");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static constexpr int kMaxE = (kMaxDynSmem - 1024 - kTabOff) / 8 - 1;  // experts whose tables fit
  static_assert(kMaxE >= 64, "shared memory");
  static size_t bytes(int E) { return 1024 + kTabOff + 2 * (size_t)(E + 1) * 4; }
};

struct Tile {
  int shared, e, f, row_base, rows;
  int nt;  // token tiles of this segment: how many tiles reuse this tile's weight rows
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
    const int cnt = s_off[lo + 1] - s_off[lo];
    // An expert with more token rows than weight rows walks token-tile-major so its
    // weights stay in L2 while its token tiles stream; otherwise feature-tile-major.
    const bool m_major = cnt > p.n_out;
    const int m = m_major ? local / p.n_ftiles : local % nt;
    t.shared = 0;
    t.e = lo;
    t.nt = nt;
    t.f = m_major ? local - m * p.n_ftiles : local / nt;
    t.row_base = s_off[lo] + m * p.NT;
    t.rows = min(p.NT, s_off[lo + 1] - t.row_base);
  } else {
    const int local = tile - routed_total;
    const int nt = (p.T_s + p.NT - 1) / p.NT;
    const bool m_major = p.T_s > p.n_out_s;
    const int m = m_major ? local / p.n_ftiles_s : local % nt;
    t.shared = 1;
    t.e = -1;
    t.nt = nt;
    t.f = m_major ? local - m * p.n_ftiles_s : local / nt;
    t.row_base = m * p.NT;
    t.rows = min(p.NT, p.T_s - t.row_base);
  }
  return t;
}

// Stores 16 token columns [col0, col0+16) of this lane's output feature, two features per
// 32-bit store.  Lanes l and l^1 hold adjacent features (the even lane the even feature),
// so after one shfl_xor(1) per column pair the even lane holds both features of the even
// column and the odd lane both features of the odd one.  `orow` points at this lane's
// feature in token row 0 of the tile; `ok` says the feature exists (output widths are
// multiples of 64, so both lanes of a pair agree on it).
__device__ __forceinline__ void store_pairs16(const float* v, int lane, uint16_t* orow, size_t ld, int col0,
                                              int rows, bool ok) {
  const bool odd = lane & 1;
  uint16_t* base = odd ? orow - 1 : orow;  // the pair's even feature
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float send = odd ? v[2 * m] : v[2 * m + 1];
    const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
    const float lo = odd ? recv : v[2 * m];
    const float hi = odd ? v[2 * m + 1] : recv;
    const int col = col0 + 2 * m + (odd ? 1 : 0);
    if (ok && col < rows) *reinterpret_cast<uint32_t*>(base + (size_t)col * ld) = pack_bf16x2(lo, hi);
  }
}

template <int NTMAX, int STAGES, int MODE, int BBOX, int EPI, int APARTS, int PAIR, int KC, int GW>
__global__ void __launch_bounds__(64 + 32 * (EPI + GW), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmAs, const __grid_constant__ CUtensorMap tmBs,
                        const GemmParams p) {
  using L = Layout<NTMAX, STAGES, MODE, BBOX, EPI, APARTS, PAIR, KC, GW>;
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
  volatile uint32_t* peer_issued = reinterpret_cast<volatile uint32_t*>(smem + L::kMiscOff + 12);
  float* s_scale = reinterpret_cast<float*>(smem + L::kScaleOff);
  int* s_off = reinterpret_cast<int*>(smem + L::kTabOff);
  int* s_tt = s_off + (p.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const uint32_t rank = PAIR == 2 ? cluster_ctarank() : 0u;  // 0 = leader of the CTA pair
  const int group = PAIR == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ngroups = PAIR == 2 ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], PAIR * EPI);  // every epilogue warp of the pair releases the buffer
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    *cfg_bad = 0;
    *peer_issued = 0;
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
  if (warp == 1) {
    if (PAIR == 2) tmem_alloc_pair(tmem_slot, L::kTmemCols);
    else tmem_alloc(tmem_slot, L::kTmemCols);
  }
  // The routing offsets are read before griddepcontrol.wait: every launch sequence that chains
  // this kernel (moe_layer_forward) writes them two or more launches earlier (routing's scan or the
  // fused small-batch kernel, then at least the scatter or the row gather), and a kernel starts only
  // after its predecessor has waited for the one before.  Waiting here instead measured ~3 us more
  // per decode layer.
  for (int i = threadIdx.x; i <= E; i += L::kThreads) s_off[i] = p.offsets ? __ldg(p.offsets + i) : 0;
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
  if (PAIR == 2) cluster_sync();  // the pair's barriers are initialised before any cross-CTA signal
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int routed_total = *cfg_bad ? 0 : s_tt[E] * p.n_ftiles;
  const int shared_total = (*cfg_bad || !p.has_shared) ? 0 : ((p.T_s + p.NT - 1) / p.NT) * p.n_ftiles_s;
  const int total = routed_total + shared_total;
  const int KB = (p.K + L::kStageK - 1) / L::kStageK;  // stages per tile; K is a multiple of kBK
  uint32_t issued = 0;  // producer: stages filled by this CTA

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    // Inside moe_layer_forward this kernel may start while the previous one finishes
    // (programmatic dependent launch): the token rows it loads may still be being
    // written, so wait for that kernel first, then let the next kernel launch.
    pdl_wait();
    pdl_launch_dependents();
    for (int tile = group; ok && tile < total; tile += ngroups) {
      const Tile t = decode_tile(tile, routed_total, s_off, s_tt, p);
      const CUtensorMap* mA = t.shared ? &tmAs : &tmA;
      const CUtensorMap* mB = t.shared ? &tmBs : &tmB;
      const int nmma = (t.rows + 15) & ~15;
      const int brows = nmma / PAIR;  // token rows this CTA stages (its half when PAIR = 2)
      const int nbox = (brows + BBOX - 1) / BBOX;
      const int b_row = t.row_base + (int)rank * brows;
      // weight box `apart` (< APARTS) of this CTA
      const int a_row = (t.shared ? 0 : t.e * p.n_out) + t.f * (kBM * APARTS * PAIR) +
                        ((int)rank * APARTS + (lane % APARTS)) * kBM;
      // Weight rows read by one tile only are streamed past L2 (evict first); weight rows that
      // the segment's other token tiles read again are kept (evict last), like the token rows.
      const uint64_t pol_a = t.nt > 1 ? pol_x : pol_w;
      // lanes 0..KC*APARTS-1 load weight boxes, lanes 8..8+KC*nbox-1 token boxes
      const int ac = lane / APARTS, apart = lane % APARTS;
      const int bc = (lane - 8) / max(nbox, 1), bj = (lane - 8) % max(nbox, 1);
      if (GW > 0 && p.g_flags != nullptr && !t.shared) {
        // The token rows this CTA stages must have been gathered: wait for the flags of the
        // chunks holding rows [b_row, b_end), one lane per chunk, then order the TMA reads
        // after the gathering CTAs' writes.
        const int b_end = min(b_row + brows, t.row_base + t.rows);
        const int q0 = b_row / kGatherRows;
        const int nq = b_end > b_row ? (b_end - 1) / kGatherRows - q0 + 1 : 0;
        bool fine = true;
        if (lane < nq) {
          const unsigned* f = p.g_flags + q0 + lane;
          if (ld_acquire_gpu(f) == 0u) {
            const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
            while (ld_acquire_gpu(f) == 0u) {
              if (*abort_flag || globaltimer_ns() > deadline) {
                fine = false;
                break;
              }
              __nanosleep(64);
            }
          }
        }
        if (!__all_sync(0xffffffffu, fine)) {
          if (lane == 0) {
            *abort_flag = 1;
            set_status(p.status, DEV_ERR_TIMEOUT);
          }
          ok = false;
          break;
        }
        fence_proxy_async_global();
      }
      for (int kb = 0; kb < KB; ++kb) {
        const int nch = min(KC, (p.K - kb * L::kStageK) / kBK);  // chunks in this stage
        const uint32_t tx = (uint32_t)(PAIR * nch) * (uint32_t)(L::kAChunk + nbox * BBOX * kRowBytes);
        bool w = (lane == 0) ? mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.timeout_ns, p.status)
                             : false;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        if (lane == 0 && rank == 0) mbar_arrive_expect_tx(&full[stage], tx);  // both CTAs' bytes
        __syncwarp();
        uint8_t* sA = smem + stage * L::kStageBytes;
        uint8_t* sB = sA + L::kABytes;
        const bool a_op = lane < KC * APARTS && ac < nch;
        const bool b_op = lane >= 8 && lane < 8 + KC * nbox && bc < nch;
        uint8_t* dst = a_op ? sA + ac * L::kAChunk + apart * kABox : sB + bc * L::kBChunk + bj * BBOX * kRowBytes;
        const CUtensorMap* map = a_op ? mA : mB;
        const int x = kb * L::kStageK + (a_op ? ac : bc) * kBK;
        const int y = a_op ? a_row : b_row + bj * BBOX;
        const uint64_t pol = a_op ? pol_a : pol_x;
        if (a_op || b_op) {
          if (PAIR == 1 || rank == 0) tma_load_2d(dst, map, x, y, &full[stage], pol);
          else tma_load_2d_pair(dst, map, x, y, mapa_shared(smem_u32(&full[stage]), 0), pol);  // leader's barrier
        }
        __syncwarp();
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (PAIR == 1) {
      // Drain: the last fill of every stage must have landed before the CTA exits.  One deadline
      // covers all stages, so a stalled pipeline costs one wait limit, not one per stage.
      if (lane == 0) {
        const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
        for (int s = 0; s < STAGES; ++s) {
          const uint32_t n = issued / STAGES + ((uint32_t)s < issued % STAGES ? 1u : 0u);
          const uint64_t now = globaltimer_ns();
          if (n) mbar_wait_bounded(&full[s], (n - 1u) & 1u, abort_flag, deadline > now ? deadline - now : 0,
                                   p.status, false);
        }
      }
    } else if (lane == 0) {
      // A CTA that gave up tells its peer, whose waits would otherwise run to their own limit.
      if (*abort_flag) st_shared_cluster_u32(mapa_shared(smem_u32((const void*)abort_flag), rank ^ 1u), 1u);
      // the follower's loads complete on the leader's barriers: tell the leader how many it issued
      if (rank == 1) st_shared_cluster_u32(mapa_shared(smem_u32((const void*)peer_issued), 0), issued);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      const uint64_t desc0 = umma_desc_sw128(smem_u32(smem));
      for (int tile = group; ok && tile < total; tile += ngroups, ++it) {
        const Tile t = decode_tile(tile, routed_total, s_off, s_tt, p);
        const int buf = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_bounded(&tempty[buf], aph ^ 1u, abort_flag, p.timeout_ns, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * L::kAccCols);
        const int nmma = (t.rows + 15) & ~15;
        const uint32_t idesc = umma_idesc_bf16(kBM * PAIR, nmma);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // descriptors of the stage's first chunk; the address field (bits 0-13, in 16-byte
          // units) of a later chunk or K step is reached by adding its offset / 16
          const uint64_t ad0 = desc0 + (uint64_t)((stage * L::kStageBytes) >> 4);
          const uint64_t bd0 = ad0 + (uint64_t)(L::kABytes >> 4);
          const bool two = KC == 1 || kb * L::kStageK + kBK < p.K;  // false: last stage holds one chunk
#pragma unroll
          for (int c = 0; c < KC; ++c) {
            if (c > 0 && !two) break;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint64_t bd = bd0 + (uint64_t)((c * L::kBChunk + kk * 32) >> 4);
#pragma unroll
              for (int part = 0; part < APARTS; ++part) {
                const uint64_t ad = ad0 + (uint64_t)((c * L::kAChunk + part * kABox + kk * 32) >> 4);
                const uint32_t acc = (kb | c | kk) != 0;
                if (PAIR == 2) umma_bf16_pair(d + part * NTMAX, ad, bd, idesc, acc);
                else umma_bf16(d + part * NTMAX, ad, bd, idesc, acc);
              }
            }
          }
          if (PAIR == 2) umma_commit_pair(&empty[stage], 0x3);
          else umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR == 2) umma_commit_pair(&tfull[buf], 0x3);
        else umma_commit(&tfull[buf]);
      }
      // Drain: every MMA issued by this thread must be complete before TMEM is freed.
      if (PAIR == 2) umma_commit_pair(done, 0x1);
      else umma_commit(done);
      mbar_wait_bounded(done, 0, abort_flag, p.timeout_ns, p.status, false);
    }
    __syncwarp();
  } else if (warp < 2 + EPI) {
    // ------------------------------------------------------------ epilogue
    const int qw = warp & 3;                 // TMEM lane quarter this warp may access
    constexpr int kPerQ = EPI / 4;           // epilogue warps sharing one TMEM lane quarter
    const int half_c = (warp - 2) >> 2;      // this warp takes 32-column chunks half_c, half_c + kPerQ, ...
    const uint32_t tempty_leader = PAIR == 2 ? mapa_shared(smem_u32(&tempty[0]), 0) : 0u;
    if (GW > 0 && p.g_flags != nullptr && !p.g_skip) {
      // Until the first accumulator is ready the epilogue warps are idle: they gather this CTA's
      // first GW row chunks (one row per warp at a time), which the first tiles of the GPU wait for;
      // the gather warps take the CTA's later chunks.
      pdl_wait();  // sorted_pair comes from the previous kernel
      const int ew = warp - 2;
      const int g_rows = min(p.M, s_off[E]);  // rows past offsets[E] are never read
      const int n_chunks = (g_rows + kGatherRows - 1) / kGatherRows;
      bool bad = false;  // an out-of-range row source, reported once after the loop
      for (int g = 0; g < GW; ++g) {
        const int q = GW * (int)blockIdx.x + g;
        if (q >= n_chunks) break;  // uniform over the epilogue warps
        const int r0 = q * kGatherRows, nrow = min(kGatherRows, g_rows - r0);
        for (int i = ew; i < nrow; i += EPI) {
          const int sp = __ldg(p.g_sp + r0 + i);
          const int t = sp / p.g_k;
          if (sp < 0 || (unsigned)t >= (unsigned)p.g_T) {
            bad = true;
            continue;
          }
          const uint4* src = p.g_x + (size_t)t * p.g_H8;
          uint4* dst = p.g_xexp + (size_t)(r0 + i) * p.g_H8;
          for (int c = lane; c < p.g_H8; c += 4 * 32) {
            uint4 v[4];
#pragma unroll
            for (int w = 0; w < 4; ++w)
              if (c + 32 * w < p.g_H8) v[w] = __ldg(src + c + 32 * w);
#pragma unroll
            for (int w = 0; w < 4; ++w)
              if (c + 32 * w < p.g_H8) dst[c + 32 * w] = v[w];
          }
        }
        // every epilogue warp has written its rows of chunk q: publish it
        asm volatile("bar.sync 1, %0;" ::"r"(32 * EPI) : "memory");
        if (warp == 2 && lane == 0) {
          fence_proxy_async_global();
          __threadfence();
          st_release_gpu(p.g_flags + q, 1u);
        }
      }
      if (bad && lane == 0) set_status(p.status, DEV_ERR_BOUNDS);
    }
    int it = 0;
    for (int tile = group; tile < total; tile += ngroups, ++it) {
      const Tile t = decode_tile(tile, routed_total, s_off, s_tt, p);
      const int buf = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      // Mode 1: fetch the routing weights of the tile's rows before waiting for
      // the accumulator, so their latency overlaps the mainloop.  They are kept in shared memory,
      // where the epilogue reads them as broadcast vector loads (in registers, one shuffle per
      // column made the compute-bound down GEMM ~18 % slower).
      float* wsc = s_scale + (warp - 2) * NTMAX;
      constexpr int kMine = (NTMAX / 32 + kPerQ - 1) / kPerQ;  // chunks of 32 columns this warp handles
      const bool scale = MODE == 1 && !t.shared && p.topk_w != nullptr;
      if (scale) {
        int pr[kMine];
#pragma unroll
        for (int r = 0; r < kMine; ++r) {
          const int col = (kPerQ * r + half_c) * 32 + lane;
          pr[r] = (col < t.rows && col < NTMAX) ? __ldg(p.sorted_pair + t.row_base + col) : -1;
        }
#pragma unroll
        for (int r = 0; r < kMine; ++r) {
          const int col = (kPerQ * r + half_c) * 32 + lane;
          if (col < NTMAX) wsc[col] = pr[r] >= 0 ? __ldg(p.topk_w + pr[r]) : 0.0f;
        }
        __syncwarp();
      }
      // The epilogue has slack: it sleeps in the barrier instead of polling.
      bool w = (lane == 0) ? mbar_wait_sleep(&tfull[buf], aph, abort_flag, p.timeout_ns, p.status) : false;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(qw * 32) << 16) + (uint32_t)(buf * L::kAccCols);
      const int nch = (t.rows + 31) >> 5;  // 32-column chunks
      uint16_t* out = t.shared ? p.s_out : p.out;
      const size_t ld = (size_t)(t.shared ? p.ld_out_s : p.ld_out);
      const int n_feat = t.shared ? p.n_feat_s : p.n_feat;
      if (MODE == 0) {
        // packed gate/up: lanes 0-15 hold gate rows, lanes 16-31 the matching up rows
        const bool is_gate = lane < 16;
#pragma unroll
        for (int part = 0; part < APARTS; ++part) {
          const int feat = t.f * L::kFeatPerTile + ((int)rank * APARTS + part) * L::kFeatPerBox + qw * 16 +
                           (lane & 15);
          const bool feat_ok = feat < n_feat;
          uint16_t* orow = out + (size_t)t.row_base * ld + feat;
          for (int c = half_c; c < nch; c += kPerQ) {
            uint32_t v[32];
            tmem_ld32_async(tb + (uint32_t)(part * NTMAX + c * 32), v);
            tmem_wait_ld();
            // gate lanes finish columns 0-15 of the chunk, up lanes columns 16-31
            const int col0 = c * 32 + (is_gate ? 0 : 16);
            float a[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float send = __uint_as_float(is_gate ? v[16 + i] : v[i]);
              const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
              const float g = is_gate ? __uint_as_float(v[i]) : recv;
              const float u = is_gate ? recv : __uint_as_float(v[16 + i]);
              // SiLU(g) * u with the fast exponential and an approximate divide: a few fp32 ulps,
              // far below the bf16 rounding of the result; g -> -inf gives -0, g -> +inf gives g
              a[i] = __fdividef(g, 1.0f + __expf(-g)) * u;
            }
            store_pairs16(a, lane, orow, ld, col0, t.rows, feat_ok);
          }
        }
      } else {
#pragma unroll
        for (int part = 0; part < APARTS; ++part) {
          const int feat = t.f * L::kFeatPerTile + ((int)rank * APARTS + part) * kBM + qw * 32 + lane;
          const bool feat_ok = feat < n_feat;
          uint16_t* orow = out + (size_t)t.row_base * ld + feat;
          for (int c = half_c; c < nch; c += kPerQ) {
            uint32_t v[32];
            tmem_ld32_async(tb + (uint32_t)(part * NTMAX + c * 32), v);
            tmem_wait_ld();
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]) * (scale ? wsc[c * 32 + i] : 1.0f);
            store_pairs16(o, lane, orow, ld, c * 32, t.rows, feat_ok);
            store_pairs16(o + 16, lane, orow, ld, c * 32 + 16, t.rows, feat_ok);
          }
        }
        __syncwarp();  // the next tile rewrites this warp's scales
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR == 2) mbar_arrive_cluster(tempty_leader + (uint32_t)(buf * 8));  // the leader's barrier
        else mbar_arrive(&tempty[buf]);
      }
    }
  } else if (GW > 0 && p.g_flags != nullptr && !p.g_skip) {
    // ------------------------------------------------------------ row gather
    // Chunk q (rows [16q, 16q+16)) belongs to CTA (q / GW) % gridDim.x, warp q % GW; every warp
    // walks its chunks in ascending order, so rows are gathered in the order the tiles need them
    // (tiles are dealt out in expert order).  Nothing here waits on another CTA.
    pdl_wait();  // sorted_pair comes from the previous kernel
    const int gw = warp - 2 - EPI;
    const int g_rows = min(p.M, s_off[E]);  // rows past offsets[E] are never read
    const int n_chunks = (g_rows + kGatherRows - 1) / kGatherRows;
    const int H8 = p.g_H8;
    // the CTA's first GW chunks are gathered by the epilogue warps
    bool bad = false;  // an out-of-range row source, reported once after the loop
    for (int q = GW * ((int)blockIdx.x + (int)gridDim.x) + gw; q < n_chunks; q += GW * (int)gridDim.x) {
      const int r0 = q * kGatherRows, nrow = min(kGatherRows, g_rows - r0);
      int tl = -1;  // lane i < nrow: source token of row r0 + i
      if (lane < nrow) {
        const int sp = __ldg(p.g_sp + r0 + lane);
        tl = sp / p.g_k;
        if (sp < 0 || (unsigned)tl >= (unsigned)p.g_T) {
          tl = -1;
          bad = true;
        }
      }
      for (int i = 0; i < nrow; i += 4) {
        int tr[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          tr[u] = __shfl_sync(0xffffffffu, tl, min(i + u, 31));
          if (i + u >= nrow) tr[u] = -1;
        }
        for (int c = lane; c < H8; c += 2 * 32) {
          uint4 v[4][2];
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int w = 0; w < 2; ++w)
              if (tr[u] >= 0 && c + 32 * w < H8) v[u][w] = __ldg(p.g_x + (size_t)tr[u] * H8 + c + 32 * w);
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int w = 0; w < 2; ++w)
              if (tr[u] >= 0 && c + 32 * w < H8) p.g_xexp[(size_t)(r0 + i + u) * H8 + c + 32 * w] = v[u][w];
        }
      }
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async_global();
        __threadfence();
        st_release_gpu(p.g_flags + q, 1u);
      }
    }
    if (bad) set_status(p.status, DEV_ERR_BOUNDS);
  }

  tc_fence_before();
  if (PAIR == 2) {
    cluster_sync();  // both CTAs have stopped issuing; the follower's load count has arrived
    if (rank == 0 && warp == 0 && lane == 0) {
      // Drain: every stage's last fill, by either CTA, must have landed before either CTA exits
      // (one deadline for all stages).
      const uint32_t pi = *peer_issued;
      const uint32_t n_all = issued > pi ? issued : pi;
      const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t n = n_all / STAGES + ((uint32_t)s < n_all % STAGES ? 1u : 0u);
        const uint64_t now = globaltimer_ns();
        if (n) mbar_wait_bounded(&full[s], (n - 1u) & 1u, abort_flag, deadline > now ? deadline - now : 0, p.status,
                                 false);
      }
    }
    cluster_sync();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem_base, L::kTmemCols);
    }
  } else {
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_base, L::kTmemCols);
    }
  }
}

// Packed gate/up layout: w13p[e][32g + r] = w13[e][16g + r] for r < 16 (gate), and
// w13[e][I + 16g + r - 16] for r >= 16 (up).  One thread per 16 bytes.
__global__ void __launch_bounds__(256) prepack_w13_kernel(const uint4* __restrict__ w13, int E, int I, int H8,
                                                          uint4* __restrict__ w13p) {
  const size_t n = (size_t)E * 2 * I * H8;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const size_t row = i / H8;
  const int col = (int)(i - row * H8);
  const int e = (int)(row / (2 * I));
  const int r = (int)(row - (size_t)e * 2 * I);
  const int g = r >> 5, q = r & 31;
  const int src = q < 16 ? g * 16 + q : I + g * 16 + (q - 16);
  w13p[i] = __ldg(w13 + ((size_t)e * 2 * I + src) * H8 + col);
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

// Row-major bf16 matrix [rows, K] as a 2-D tensor map with 64 x box_rows boxes
// and the 128-byte swizzle; rows past the end read as zeros.
bool make_map(CUtensorMap* m, const void* base, int K, long long rows, int box_rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
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

template <int NTMAX, int STAGES, int MODE, int BBOX, int EPI, int APARTS, int PAIR, int KC, int GW>
cudaError_t launch_instance(const GroupedGemmProblem& pr, GemmParams gp, cudaStream_t stream, bool pdl) {
  using L = Layout<NTMAX, STAGES, MODE, BBOX, EPI, APARTS, PAIR, KC, GW>;
  const bool has_shared = gp.has_shared != 0;
  gp.NT = NTMAX;
  gp.n_ftiles = (gp.n_feat + L::kFeatPerTile - 1) / L::kFeatPerTile;
  gp.n_ftiles_s = has_shared ? (gp.n_feat_s + L::kFeatPerTile - 1) / L::kFeatPerTile : 0;
  CUtensorMap ta, tb, tas, tbs;
  if (pr.M > 0) {
    if (!make_map(&ta, pr.w, pr.K, (long long)pr.E * pr.n_out, kBM)) return cudaErrorInvalidValue;
    if (!make_map(&tb, pr.a_rows, pr.K, pr.M, BBOX)) return cudaErrorInvalidValue;
  }
  if (has_shared) {
    if (!make_map(&tas, pr.s_w, pr.K, pr.n_out_s, kBM)) return cudaErrorInvalidValue;
    if (!make_map(&tbs, pr.s_rows, pr.K, pr.T_s, BBOX)) return cudaErrorInvalidValue;
  }
  // With no routed rows the routed maps are never read (and vice versa): alias them.
  if (pr.M <= 0) {
    ta = tas;
    tb = tbs;
  } else if (!has_shared) {
    tas = ta;
    tbs = tb;
  }
  auto kern = grouped_gemm_kernel<NTMAX, STAGES, MODE, BBOX, EPI, APARTS, PAIR, KC, GW>;
  if (gp.E > L::kMaxE) return cudaErrorInvalidValue;
  const size_t smem = L::bytes(gp.E);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int grid = PAIR == 2 ? (num_sms() & ~1) : num_sms();
  if (PAIR == 2) {
    // Persistent grid: no more CTA pairs than can be resident at once (the gather flags are
    // waited on across CTAs, which needs every CTA of the grid running).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters > 0 && 2 * clusters < grid)
      grid = 2 * clusters;
  }
  return launch_kernel_cluster(kern, dim3(grid), dim3(L::kThreads), smem, stream, pdl, PAIR, ta, tb, tas, tbs, gp);
}

}  // namespace

// Failure injection for the tests of the bounded waits (moe_debug_set): a shorter wait limit, and
// a gate/up GEMM whose gather sets no flag, so that its producers' waits run out.
static unsigned long long g_debug_timeout_ns = 0;
static int g_debug_no_gather = 0;

int grouped_gemm_debug_set(int what, unsigned long long value) {
  if (what == 1) g_debug_timeout_ns = value;
  else if (what == 2) g_debug_no_gather = value != 0;
  else return -1;
  return 0;
}

bool grouped_gemm_narrow(int M, int E, bool has_shared, int T_s) {
  // Decode-like problems (a few rows per expert) take the 32-column single-CTA instances with
  // a deep pipeline; prefill-like ones the 256-column CTA-pair instances.
  return (long long)M <= 32LL * E && (!has_shared || T_s <= 32);
}

bool grouped_gemm_streaming(int M, int E) {
  // Segments averaging fewer than 256 rows do fewer than 256 FLOPs per weight byte, below the
  // GPU's ratio of tensor rate to HBM bandwidth: those GEMMs stream weights.
  return (long long)M < 256LL * E;
}

bool grouped_gemm_gathers_inline(int M, int E, bool has_shared, int T_s) {
  // The CTA-pair gate/up GEMMs gather their rows themselves: the compute-bound one hides the
  // gather's HBM traffic behind its matmuls; the weight-streaming one is bound by the latency of
  // its loads, not by HBM bandwidth, and overlapping the gather saves the separate kernel's time
  // (hy3_prefill: routing 0.080 -> 0.019 ms, the GEMM 0.960 -> 1.010 ms).
  return !grouped_gemm_narrow(M, E, has_shared, T_s);
}

cudaError_t launch_grouped_gemm(const GroupedGemmProblem& pr, cudaStream_t stream, bool pdl) {
  const bool has_shared = pr.s_rows != nullptr && pr.T_s > 0;
  if (pr.M <= 0 && !has_shared) return cudaSuccess;
  GemmParams gp{};
  gp.offsets = pr.M > 0 ? pr.offsets : nullptr;
  gp.E = pr.E;
  gp.M = pr.M;
  gp.K = pr.K;
  gp.n_out = pr.n_out;
  gp.n_feat = pr.mode == 0 ? pr.n_out / 2 : pr.n_out;
  gp.out = pr.out;
  gp.ld_out = pr.ld_out;
  gp.has_shared = has_shared ? 1 : 0;
  if (has_shared) {
    gp.T_s = pr.T_s;
    gp.n_out_s = pr.n_out_s;
    gp.n_feat_s = pr.mode == 0 ? pr.n_out_s / 2 : pr.n_out_s;
  }
  gp.s_out = pr.s_out;
  gp.ld_out_s = pr.ld_out_s;
  gp.topk_w = pr.topk_w;
  gp.sorted_pair = pr.sorted_pair;
  gp.status = pr.status;
  gp.timeout_ns = g_debug_timeout_ns ? g_debug_timeout_ns : kTimeoutNs;
  gp.g_skip = g_debug_no_gather;
  const bool gather = pr.mode == 0 && pr.g_x != nullptr && pr.M > 0;
  // Among the CTA-pair instances, segments averaging fewer than 256 rows do fewer than
  // 256 FLOPs per weight byte, below the GPU's ratio of tensor rate to HBM bandwidth:
  // they stream weights, and six or seven 64-deep stages keep more weight bytes in flight.
  // Longer segments are compute-bound and take three 128-deep stages, which let the
  // MMA thread issue 8 MMAs between two waits (the tensor pipe idles otherwise).
  // The CTA-pair gate/up instances run 2 extra warps that gather the token rows while the GEMM
  // runs (when asked to); the decode instance has the rows gathered by a separate kernel first.
  if (gather && !grouped_gemm_gathers_inline(pr.M, pr.E, has_shared, pr.T_s)) {
    // rows past offsets[E] are never read by the GEMM: gather only the routed ones
    cudaError_t e = launch_expand_rows(pr.g_x, pr.g_sorted_pair, pr.M, pr.g_k, pr.K, const_cast<uint16_t*>(pr.a_rows),
                                       stream, pdl, pr.offsets + pr.E, pr.g_T, pr.status);
    if (e != cudaSuccess) return e;
  }
  if (grouped_gemm_narrow(pr.M, pr.E, has_shared, pr.T_s))
    return pr.mode == 0 ? launch_instance<32, 5, 0, 16, 8, 2, 1, 1, 0>(pr, gp, stream, pdl)
                        : launch_instance<32, 10, 1, 16, 8, 1, 1, 1, 0>(pr, gp, stream, pdl);
  if (gather) {
    gp.g_x = reinterpret_cast<const uint4*>(pr.g_x);
    gp.g_sp = pr.g_sorted_pair;
    gp.g_xexp = reinterpret_cast<uint4*>(const_cast<uint16_t*>(pr.a_rows));
    gp.g_k = pr.g_k;
    gp.g_T = pr.g_T;
    gp.g_H8 = pr.K / 8;
    gp.g_flags = pr.g_flags;
  }
  // Eight epilogue warps except in the compute-bound gate/up instance, whose epilogue warps also
  // gather the first row chunks (with sixteen the others measured 2-5 % slower).
  if (grouped_gemm_streaming(pr.M, pr.E)) {
    // gate/up: seven stages where the expert tables leave room for them, else six; down: six (its
    // routing weights take the room of a seventh)
    if (pr.mode == 1) return launch_instance<256, 6, 1, 64, 8, 1, 2, 1, 0>(pr, gp, stream, pdl);
    if (pr.E <= Layout<256, 7, 0, 64, 8, 1, 2, 1, 2>::kMaxE)
      return launch_instance<256, 7, 0, 64, 8, 1, 2, 1, 2>(pr, gp, stream, pdl);
    return launch_instance<256, 6, 0, 64, 8, 1, 2, 1, 2>(pr, gp, stream, pdl);
  }
  return pr.mode == 0 ? launch_instance<256, 3, 0, 64, 16, 1, 2, 2, 2>(pr, gp, stream, pdl)
                      : launch_instance<256, 3, 1, 64, 8, 1, 2, 2, 0>(pr, gp, stream, pdl);
}

cudaError_t launch_prepack_w13(const uint16_t* w13, int E, int I, int H, uint16_t* w13p, cudaStream_t stream) {
  const size_t n = (size_t)E * 2 * I * (H / 8);
  if (n == 0) return cudaSuccess;
  prepack_w13_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(reinterpret_cast<const uint4*>(w13), E, I,
                                                                      H / 8, reinterpret_cast<uint4*>(w13p));
  return cudaGetLastError();
}

}  // namespace moe
