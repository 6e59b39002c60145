// a3/a4 in W4A8 on GB300: MXFP8 token rows times MXFP4 expert weights on the block-scaled tensor
// core MMA (tcgen05.mma kind::mxf8f6f4 .block_scale), fp32 accumulators in TMEM.
//
// Source: Qwen3-MoE low-latency inference practice (Atlas A3/950), MoE EP section, "computation
// decomposition (AllGather scheme, W4A8 quantisation)": the hidden state is quantised to MXFP8
// (data + scale), routed, and the grouped matmuls run on it with the experts' MXFP4 weights;
// Hy3 295B MoE practice 5.2: on the quantised path the SwiGLU is fused with a group quantisation,
// so the activation entering the down projection is MXFP8 as well.  The matmuls and SwiGLU are
// those of "MoE TP optimisation: computation decomposition", as in the bf16 GEMMs.
//
// Formats (OCP microscaling; blocks of 32 consecutive elements along K share one E8M0 scale):
//   weights  E2M1 codes, two per byte (element 2j in the low nibble of byte j), prepacked by
//            moe_w4a8_prepack: rows of the gate/up weight regrouped so that a 256-row tile holds
//            128 whole features (below), and the scales rearranged into 512-byte atoms, one per
//            (128-row tile, 128-K chunk): byte (r % 32) * 16 + (r / 32) * 4 + b holds the scale of
//            row r, block b -- the layout tcgen05.cp .32x128b.warpx4 turns into the tensor-memory
//            scale-factor layout of an M = 128 block-scaled MMA (row r at lane r % 32 of every lane
//            quarter, column r / 32, byte b = the MMA's scale-factor id).
//   tokens   E4M3 codes [rows, K] and "padded scale rows" [rows, K/128, 16]: per row and 128-K
//            chunk, 16 bytes whose first four are the chunk's four block scales (the rest zero).  A
//            32-row TMA box of them is the 32 x 16-byte source of one tcgen05.cp for the token
//            operand's scale factors (token n at lane n, column 0).
//
// Product (swap-AB, as the bf16 decode instances): weight rows are the MMA's M = 128 operand A,
// read from shared memory in the padded E2M1 layout that TMA writes for
// CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B (each 16 codes = 8 bytes followed by 8 zero bytes, so a
// 128-code row is a 128-byte swizzled row); the expert's token rows are the N = 32 operand B
// (E4M3, 128-byte swizzled rows).  One 128-K stage = 4 MMAs of K = 32, each naming its block with
// the scale-factor ids of the instruction descriptor; both operands' scale factors are copied into
// a per-stage tensor-memory slot by the MMA thread (tcgen05.cp, which the MMAs issued after it by
// the same thread are ordered behind).
//
// Mode 0 (gate/up + SwiGLU + MXFP8 of act): two 128-row weight boxes per stage, each into its own
// accumulator.  The prepacked gate/up tile of 256 rows holds features [128 f, 128 f + 128): box p,
// lane quarter q, lane l holds the gate (l < 16) or up (l >= 16) row of feature
// 128 f + 32 q + 16 p + (l % 16), so one epilogue warp ends up with a whole 32-feature block of act
// for each token column: the block maximum is a 4-step shuffle reduction, and the warp writes the
// E4M3 codes and the E8M0 scale byte of that block for the down GEMM.
// Mode 1 (down + routing weight): one 128-row box, bf16 output times topk_w[sorted_pair[pos]].
//
// Warp roles (64 + 32 * 4 threads, one persistent CTA per SM, static round-robin tiles; an expert's
// token tiles that reuse a weight tile run next to each other): warp 0 TMA producer, warp 1 TMEM
// allocator + MMA issuer, warps 2-5 epilogue (one per TMEM lane quarter).  Every wait is bounded
// (2 s): on expiry the CTA raises its abort flag, records DEV_ERR_TIMEOUT, lets its copies land,
// drains its MMAs and frees TMEM.
#include "moe_common.cuh"
#include "moe_internal.h"

#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kBM = 128;                  // weight rows per box (MMA M)
constexpr int kNT = 32;                   // token columns per tile (MMA N)
constexpr int kKC = 128;                  // K per stage: 4 MMAs of K = 32
constexpr int kABox = kBM * 128;          // shared-memory bytes of one weight box (padded codes): 16 KB
constexpr int kATx = kBM * kKC / 2;       // bytes the weight box moves (and counts on the barrier): 8 KB
constexpr int kBBox = kNT * kKC;          // 32 token rows x 128 E4M3 codes: 4 KB
constexpr int kSF = 512;                  // one scale-factor atom / one 32-row box of padded scale rows
constexpr int kEPI = 4;                   // epilogue warps, one per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kEPI;
constexpr int kMaxDynSmem = 232448;
constexpr unsigned long long kTimeoutNs = 2000000000ull;

template <int MODE, int STAGES>
struct W8Layout {
  static constexpr int kParts = MODE == 0 ? 2 : 1;                 // weight boxes per stage
  static constexpr int kAOff = 0;
  static constexpr int kBOff = kParts * kABox;
  static constexpr int kSFAOff = kBOff + kBBox;
  static constexpr int kSFBOff = kSFAOff + kParts * kSF;
  static constexpr int kStageBytes = (kSFBOff + kSF + 1023) / 1024 * 1024;
  static constexpr int kBarOff = STAGES * kStageBytes;
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kScaleOff = kMiscOff + 16;                  // mode 1: routing weights per epilogue warp
  static constexpr int kTabOff = kScaleOff + kEPI * kNT * 4;
  static constexpr uint32_t kTx = kParts * (kATx + kSF) + kBBox + kSF;
  // tensor memory: two accumulator buffers of kParts x 32 columns, then a scale-factor slot per
  // stage (4 columns per weight box, 4 for the tokens)
  static constexpr int kAccCols = kParts * kNT;
  static constexpr int kSFCol0 = 2 * kAccCols;
  static constexpr int kSFColsPerStage = 4 * (kParts + 1);
  static constexpr int kColsNeeded = kSFCol0 + STAGES * kSFColsPerStage;
  static constexpr uint32_t kTmemCols = kColsNeeded <= 64 ? 64 : (kColsNeeded <= 128 ? 128 : (kColsNeeded <= 256 ? 256 : 512));
  static constexpr int kFeatPerTile = 128;
  static_assert(kColsNeeded <= 512, "TMEM");
  static_assert(kABox % 1024 == 0 && kBOff % 1024 == 0 && kSFAOff % 16 == 0, "alignment");
  static_assert(1024 + kTabOff + 2 * 1025 * 4 <= kMaxDynSmem, "shared memory");
  static size_t bytes(int E) { return 1024 + kTabOff + 2 * (size_t)(E + 1) * 4; }
};

struct W8Params {
  const int32_t* offsets;
  int E, M, K;
  int n_out, n_ftiles, n_feat;      // routed: weight rows per expert, feature tiles per expert, features
  const uint8_t* sfa;               // weight scale atoms
  uint8_t* act;                     // mode 0: [M, n_feat] E4M3 codes
  uint8_t* act_sf;                  // mode 0: [M, n_feat/128, 16] padded scale rows
  uint16_t* out;                    // mode 1: [M, n_feat] bf16
  const float* topk_w;
  const int32_t* sorted_pair;
  int has_shared, T_s, n_out_s, n_ftiles_s, n_feat_s;
  const uint8_t* sfa_s;
  uint8_t* act_s;
  uint8_t* act_sf_s;
  uint16_t* out_s;
  unsigned* status;
  unsigned long long timeout_ns;
};

struct W8Tile {
  int shared, e, f, row_base, rows;
  int nt;  // token tiles of this segment (> 1: the weight tile is read again)
};

__device__ __forceinline__ W8Tile w8_tile(int tile, int routed_total, const int* s_off, const int* s_tt,
                                          const W8Params& p) {
  W8Tile t;
  if (tile < routed_total) {
    const int q = tile / p.n_ftiles;
    int lo = 0, hi = p.E;  // largest lo with s_tt[lo] <= q
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tt[mid] <= q) lo = mid; else hi = mid;
    }
    const int nt = s_tt[lo + 1] - s_tt[lo];
    const int local = tile - s_tt[lo] * p.n_ftiles;
    const int cnt = s_off[lo + 1] - s_off[lo];
    const bool m_major = cnt > p.n_out;  // more token rows than weight rows: token tiles outermost
    const int m = m_major ? local / p.n_ftiles : local % nt;
    t.shared = 0;
    t.e = lo;
    t.nt = nt;
    t.f = m_major ? local - m * p.n_ftiles : local / nt;
    t.row_base = s_off[lo] + m * kNT;
    t.rows = min(kNT, s_off[lo + 1] - t.row_base);
  } else {
    const int local = tile - routed_total;
    const int nt = (p.T_s + kNT - 1) / kNT;
    const bool m_major = p.T_s > p.n_out_s;
    const int m = m_major ? local / p.n_ftiles_s : local % nt;
    t.shared = 1;
    t.e = -1;
    t.nt = nt;
    t.f = m_major ? local - m * p.n_ftiles_s : local / nt;
    t.row_base = m * kNT;
    t.rows = min(kNT, p.T_s - t.row_base);
  }
  return t;
}

// Instruction descriptor of tcgen05.mma kind::mxf8f6f4 .block_scale: A E2M1 (5), B E4M3 (0), both
// K-major, E8M0 scale factors, M = 128, N = 32; the scale-factor ids of A (bits 29-30) and B
// (bits 4-5) select the byte of each 32-bit tensor-memory scale column, i.e. the K block.
__device__ __forceinline__ uint32_t w4a8_idesc(uint32_t sf_id) {
  uint32_t d = 0;
  d |= sf_id << 4;                 // B scale-factor id
  d |= 5u << 7;                    // A format: E2M1
  d |= 0u << 10;                   // B format: E4M3
  d |= (uint32_t)(kNT >> 3) << 17; // N / 8
  d |= 1u << 23;                   // scale-factor type: UE8M0
  d |= (uint32_t)(kBM >> 4) << 24; // M / 16
  d |= sf_id << 29;                // A scale-factor id
  return d;
}

__device__ __forceinline__ void umma_w4a8(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor of a 32-row x 16-byte matrix stored row after row (no swizzle): the source
// of tcgen05.cp .32x128b (8-row core matrices 128 bytes apart; the leading offset is set equal so
// that either reading of the two offsets addresses the same rows).
__device__ __forceinline__ uint64_t sf_src_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)(128u >> 4) << 16;
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  return d;
}

// 32 lanes x 128 bits from shared memory into tensor memory, the same 32 rows into every lane quarter.
__device__ __forceinline__ void tmem_cp_32x128_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// One-dimensional bulk copy global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// floor(log2 m) - 8 clamped to the E8M0 range (m == 0 -> -127): the block's shared exponent.
__device__ __forceinline__ int mx_shared_exponent(float m) {
  const uint32_t b = __float_as_uint(m);
  const int e8 = (int)((b >> 23) & 0xFF);
  if ((b & 0x7FFFFFFFu) == 0) return -127;
  const int fl = e8 != 0 ? e8 - 127 : (31 - __clz((int)(b & 0x7FFFFFu))) - 149;
  return max(-127, min(127, fl - 8));
}

// 2^-s for an E8M0 shared exponent s in [-127, 127] (exact; subnormal at s = 127).
__device__ __forceinline__ float pow2_neg(int s) {
  const int k = -s;
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ void store_pairs16_bf16(const float* v, int lane, uint16_t* orow, size_t ld, int col0,
                                                   int rows, bool ok) {
  const bool odd = lane & 1;
  uint16_t* base = odd ? orow - 1 : orow;
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

template <int MODE, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_w4a8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmSB, const __grid_constant__ CUtensorMap tmAs,
                             const __grid_constant__ CUtensorMap tmBs, const __grid_constant__ CUtensorMap tmSBs,
                             const W8Params p) {
  using L = W8Layout<MODE, STAGES>;
  constexpr int P = L::kParts;
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
  float* s_scale = reinterpret_cast<float*>(smem + L::kScaleOff);
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
      mbar_init(&tempty[b], kEPI);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    *cfg_bad = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmSB);
    if (p.has_shared) {
      tma_prefetch_desc(&tmAs);
      tma_prefetch_desc(&tmBs);
      tma_prefetch_desc(&tmSBs);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, L::kTmemCols);
  for (int i = threadIdx.x; i <= E; i += kThreads) s_off[i] = p.offsets ? __ldg(p.offsets + i) : 0;
  __syncthreads();
  if (warp == 2) {
    // Validate the offsets and build the prefix of token tiles per expert.
    const int per = (E + 31) >> 5;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int sum = 0;
    bool bad = (lane == 0) && (s_off[0] < 0 || s_off[E] > p.M);
    for (int e = e0; e < e1; ++e) {
      const int n = s_off[e + 1] - s_off[e];
      if (n < 0) bad = true;
      else sum += (n + kNT - 1) / kNT;
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
      run += n > 0 ? (n + kNT - 1) / kNT : 0;
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
  const int shared_total = (*cfg_bad || !p.has_shared) ? 0 : ((p.T_s + kNT - 1) / kNT) * p.n_ftiles_s;
  const int total = routed_total + shared_total;
  const int KB = p.K / kKC;  // stages per tile (K is a multiple of 128)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_first = policy_evict_first();
    const uint64_t pol_last = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;
    bool ok = true;
    // Inside a layer forward this kernel may start while its predecessor finishes (programmatic
    // dependent launch): wait for it before reading the rows it writes, then let the next launch.
    pdl_wait();
    pdl_launch_dependents();
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      const W8Tile t = w8_tile(tile, routed_total, s_off, s_tt, p);
      const CUtensorMap* mA = t.shared ? &tmAs : &tmA;
      const CUtensorMap* mB = t.shared ? &tmBs : &tmB;
      const CUtensorMap* mSB = t.shared ? &tmSBs : &tmSB;
      const int n_out = t.shared ? p.n_out_s : p.n_out;
      // first 128-row box of this tile, counted in rows of the prepacked weight
      const int a_row = (t.shared ? 0 : t.e * n_out) + t.f * (kBM * P);
      const uint8_t* sfa = (t.shared ? p.sfa_s : p.sfa) + (size_t)(a_row / kBM) * KB * kSF;
      const uint64_t pol_a = t.nt > 1 ? pol_last : pol_first;  // weight tiles read again stay in L2
      for (int kb = 0; kb < KB; ++kb) {
        bool w = (lane == 0) ? mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.timeout_ns, p.status)
                             : false;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[stage], L::kTx);
        __syncwarp();
        uint8_t* st = smem + stage * L::kStageBytes;
        if (lane < P) {
          tma_load_2d(st + L::kAOff + lane * kABox, mA, kb * kKC, a_row + lane * kBM, &full[stage], pol_a);
        } else if (lane == 8) {
          tma_load_2d(st + L::kBOff, mB, kb * kKC, t.row_base, &full[stage], pol_last);
        } else if (lane >= 16 && lane < 16 + P) {
          const int part = lane - 16;
          bulk_load(st + L::kSFAOff + part * kSF, sfa + ((size_t)part * KB + kb) * kSF, kSF, &full[stage], pol_a);
        } else if (lane == 24) {
          tma_load_2d(st + L::kSFBOff, mSB, kb * 16, t.row_base, &full[stage], pol_last);
        }
        __syncwarp();
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Drain: the last fill of every stage must have landed before the CTA exits (one deadline).
    if (lane == 0) {
      const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
      for (int s = 0; s < STAGES; ++s) {
        const uint32_t n = issued / STAGES + ((uint32_t)s < issued % STAGES ? 1u : 0u);
        const uint64_t now = globaltimer_ns();
        if (n) mbar_wait_bounded(&full[s], (n - 1u) & 1u, abort_flag, deadline > now ? deadline - now : 0,
                                 p.status, false);
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
      const uint64_t desc0 = umma_desc_sw128(smem_u32(smem));
      const uint64_t sfd0 = sf_src_desc(smem_u32(smem));
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_bounded(&tempty[buf], aph ^ 1u, abort_flag, p.timeout_ns, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * L::kAccCols);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t soff = (uint32_t)(stage * L::kStageBytes);
          const uint32_t sf_slot = tmem_base + (uint32_t)(L::kSFCol0 + stage * L::kSFColsPerStage);
          const uint32_t sfb_t = sf_slot + 4u * P;
#pragma unroll
          for (int part = 0; part < P; ++part)
            tmem_cp_32x128_x4(sf_slot + 4u * part, sfd0 + (uint64_t)((soff + L::kSFAOff + part * kSF) >> 4));
          tmem_cp_32x128_x4(sfb_t, sfd0 + (uint64_t)((soff + L::kSFBOff) >> 4));
          const uint64_t ad0 = desc0 + (uint64_t)((soff + L::kAOff) >> 4);
          const uint64_t bd0 = desc0 + (uint64_t)((soff + L::kBOff) >> 4);
#pragma unroll
          for (int kk = 0; kk < kKC / 32; ++kk) {
            const uint32_t idesc = w4a8_idesc((uint32_t)kk);
#pragma unroll
            for (int part = 0; part < P; ++part)
              umma_w4a8(d + part * kNT, ad0 + (uint64_t)((part * kABox + kk * 32) >> 4), bd0 + (uint64_t)((kk * 32) >> 4),
                        idesc, sf_slot + 4u * part, sfb_t, (kb | kk) != 0);
          }
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
      const W8Tile t = w8_tile(tile, routed_total, s_off, s_tt, p);
      const int buf = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      float* wsc = s_scale + (warp - 2) * kNT;
      const bool scale = MODE == 1 && !t.shared && p.topk_w != nullptr;
      if (scale) {
        // routing weights of the tile's rows, fetched before the accumulator wait
        const int pr = lane < t.rows ? __ldg(p.sorted_pair + t.row_base + lane) : -1;
        wsc[lane] = pr >= 0 ? __ldg(p.topk_w + pr) : 0.0f;
        __syncwarp();
      }
      bool w = (lane == 0) ? mbar_wait_sleep(&tfull[buf], aph, abort_flag, p.timeout_ns, p.status) : false;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(qw * 32) << 16) + (uint32_t)(buf * L::kAccCols);
      if (MODE == 0) {
        uint32_t v[2][32];
        tmem_ld32_async(tb, v[0]);
        tmem_ld32_async(tb + kNT, v[1]);
        tmem_wait_ld();
        // release the accumulator early: everything below works on registers
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        // SwiGLU: lanes 0-15 hold gate rows, lanes 16-31 the up rows of the same features; the gate
        // lanes finish token columns 0-15, the up lanes columns 16-31
        const bool is_gate = lane < 16;
        float a[2][16];
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float send = __uint_as_float(is_gate ? v[part][16 + i] : v[part][i]);
            const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
            const float g = is_gate ? __uint_as_float(v[part][i]) : recv;
            const float u = is_gate ? recv : __uint_as_float(v[part][16 + i]);
            a[part][i] = __fdividef(g, 1.0f + __expf(-g)) * u;
          }
        // MXFP8 of act: per token column, the 32 features of this warp's block are 16 lanes x 2 parts
        uint8_t* act = t.shared ? p.act_s : p.act;
        uint8_t* act_sf = t.shared ? p.act_sf_s : p.act_sf;
        const int n_feat = t.shared ? p.n_feat_s : p.n_feat;
        const int col_half = is_gate ? 0 : 16;
        const int feat = t.f * L::kFeatPerTile + qw * 32 + (lane & 15);
        int my_shared = -127;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float m = fmaxf(fabsf(a[0][i]), fabsf(a[1][i]));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
          const int sh = mx_shared_exponent(m);
          if ((lane & 15) == i) my_shared = sh;
          const float inv = pow2_neg(sh);
          const int col = col_half + i;
          if (col < t.rows) {
            const __nv_fp8x2_storage_t c2 =
                __nv_cvt_float2_to_fp8x2(make_float2(a[0][i] * inv, a[1][i] * inv), __NV_SATFINITE, __NV_E4M3);
            uint8_t* orow = act + (size_t)(t.row_base + col) * n_feat + feat;
            orow[0] = (uint8_t)(c2 & 0xFF);
            orow[16] = (uint8_t)(c2 >> 8);
          }
        }
        // lane j of each half writes the scale byte of token column (half + j); the quarter-0 warp
        // also clears the entry's 12 padding bytes
        const int col = col_half + (lane & 15);
        if (col < t.rows) {
          uint8_t* e = act_sf + ((size_t)(t.row_base + col) * (n_feat / 128) + t.f) * 16;
          e[qw] = (uint8_t)(my_shared + 127);
          if (qw == 0) {
            reinterpret_cast<uint32_t*>(e)[1] = 0u;
            reinterpret_cast<uint32_t*>(e)[2] = 0u;
            reinterpret_cast<uint32_t*>(e)[3] = 0u;
          }
        }
      } else {
        uint32_t v[32];
        tmem_ld32_async(tb, v);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        uint16_t* out = t.shared ? p.out_s : p.out;
        const int n_feat = t.shared ? p.n_feat_s : p.n_feat;
        const int feat = t.f * L::kFeatPerTile + qw * 32 + lane;
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]) * (scale ? wsc[i] : 1.0f);
        uint16_t* orow = out + (size_t)t.row_base * n_feat + feat;
        store_pairs16_bf16(o, lane, orow, (size_t)n_feat, 0, t.rows, feat < n_feat);
        store_pairs16_bf16(o + 16, lane, orow, (size_t)n_feat, 16, t.rows, feat < n_feat);
        __syncwarp();  // the next tile rewrites this warp's routing weights
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

// ---------------------------------------------------------------- one-time weight layout
// codes [E, n_out, K/2], scales [E, n_out, K/32] (moe_mxfp4_quantize) -> codes_p [E*n_out, K/2]
// (gate/up rows regrouped when gate_up) and the scale atoms sf_p [E*n_out/128][K/128][512].
// Gate/up (n_out = 2I, I % 128 == 0): packed row R of an expert, with tile = R / 256,
// p = (R / 128) % 2, q = (R / 32) % 4, l = R % 32, is the gate (l < 16) or up (l >= 16) row of
// feature 128 tile + 32 q + 16 p + l % 16.  One warp per packed row.
__global__ void __launch_bounds__(256) w4a8_prepack_kernel(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ scales, int E, int n_out,
                                                           int K, int gate_up, uint8_t* __restrict__ codes_p,
                                                           uint8_t* __restrict__ sf_p) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)E * n_out) return;
  const int e = (int)(row / n_out), R = (int)(row - (long long)e * n_out);
  int src = R;
  if (gate_up) {
    const int I = n_out / 2;
    const int tile = R >> 8, part = (R >> 7) & 1, q = (R >> 5) & 3, l = R & 31;
    const int f = tile * 128 + q * 32 + part * 16 + (l & 15);
    src = l < 16 ? f : I + f;
  }
  const long long srow = (long long)e * n_out + src;
  const uint4* cs = reinterpret_cast<const uint4*>(codes + srow * (K / 2));
  uint4* cd = reinterpret_cast<uint4*>(codes_p + row * (K / 2));
  for (int c = lane; c < K / 32; c += 32) cd[c] = __ldg(cs + c);
  const int nb = K / 32;
  const long long tile128 = row / kBM;
  const int r = (int)(row % kBM);
  for (int b = lane; b < nb; b += 32) {
    const int chunk = b >> 2, kb = b & 3;
    sf_p[(tile128 * (K / kKC) + chunk) * kSF + (r % 32) * 16 + (r / 32) * 4 + kb] = __ldg(scales + srow * nb + b);
  }
}

// MXFP8 token rows for the W4A8 GEMMs: out_codes[pos] = x_codes[t] and the padded scale row
// out_sf[pos] = (x_scales[t][4c .. 4c+3], 0 x 12) per 128-K chunk c, with t = sorted_pair[pos] / k
// (sorted_pair NULL: t = pos, and no codes are written -- the scale rows of the token rows
// themselves, for the shared expert).  One block per row; n_rows: optional device bound on the
// rows (rows past it are left alone).
__global__ void __launch_bounds__(128) gather_rows_mx_kernel(const uint8_t* __restrict__ x_codes,
                                                             const uint8_t* __restrict__ x_scales,
                                                             const int32_t* __restrict__ sorted_pair, int M, int k,
                                                             int T, int H, uint8_t* __restrict__ out_codes,
                                                             uint8_t* __restrict__ out_sf,
                                                             const int32_t* __restrict__ n_rows, unsigned* status) {
  pdl_wait();
  pdl_launch_dependents();
  const int pos = blockIdx.x;
  if (pos >= M) return;
  if (n_rows && pos >= __ldg(n_rows)) return;
  int t = pos;
  if (sorted_pair) {
    const int sp = __ldg(sorted_pair + pos);
    if (sp < 0 || (long long)sp >= (long long)T * k) {
      if (threadIdx.x == 0) set_status(status, DEV_ERR_BOUNDS);
      return;
    }
    t = sp / k;
  }
  if (out_codes) {
    const uint4* src = reinterpret_cast<const uint4*>(x_codes + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(out_codes + (size_t)pos * H);
    for (int c = threadIdx.x; c < H / 16; c += blockDim.x) dst[c] = __ldg(src + c);
  }
  const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(x_scales + (size_t)t * (H / 32));
  uint4* sdst = reinterpret_cast<uint4*>(out_sf + (size_t)pos * (H / kKC) * 16);
  for (int c = threadIdx.x; c < H / kKC; c += blockDim.x) sdst[c] = make_uint4(__ldg(ssrc + c), 0u, 0u, 0u);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_w8() {
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

// E2M1 codes [rows, K] (K/2 bytes per row) in 128-row x 128-code boxes, each 16 codes landing as 8
// bytes followed by 8 zero bytes (the operand layout of the block-scaled MMA for 4-bit A), 128-byte
// swizzle.
bool make_map_e2m1(CUtensorMap* m, const void* base, int K, long long rows) {
  auto fn = encode_fn_w8();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K / 2};
  cuuint32_t box[2] = {(cuuint32_t)kKC, (cuuint32_t)kBM};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bytes [rows, width] in boxes of box_w x box_h (128-byte swizzle or none); rows past the end read as zeros.
bool make_map_bytes(CUtensorMap* m, const void* base, long long width, long long rows, int box_w, int box_h,
                    bool swizzle) {
  auto fn = encode_fn_w8();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)width};
  cuuint32_t box[2] = {(cuuint32_t)box_w, (cuuint32_t)box_h};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int STAGES>
cudaError_t launch_w8(const W4a8GemmProblem& pr, W8Params gp, cudaStream_t stream, bool pdl) {
  using L = W8Layout<MODE, STAGES>;
  const bool has_shared = gp.has_shared != 0;
  CUtensorMap ta, tb, tsb, tas, tbs, tsbs;
  if (pr.M > 0) {
    if (!make_map_e2m1(&ta, pr.codes, pr.K, (long long)pr.E * pr.n_out)) return cudaErrorInvalidValue;
    if (!make_map_bytes(&tb, pr.a_rows, pr.K, pr.M, kKC, kNT, true)) return cudaErrorInvalidValue;
    if (!make_map_bytes(&tsb, pr.a_sf, pr.K / kKC * 16, pr.M, 16, kNT, false)) return cudaErrorInvalidValue;
  }
  if (has_shared) {
    if (!make_map_e2m1(&tas, pr.s_codes, pr.K, pr.n_out_s)) return cudaErrorInvalidValue;
    if (!make_map_bytes(&tbs, pr.s_rows, pr.K, pr.T_s, kKC, kNT, true)) return cudaErrorInvalidValue;
    if (!make_map_bytes(&tsbs, pr.s_rows_sf, pr.K / kKC * 16, pr.T_s, 16, kNT, false)) return cudaErrorInvalidValue;
  }
  // With no routed rows the routed maps are never read (and vice versa): alias them.
  if (pr.M <= 0) {
    ta = tas;
    tb = tbs;
    tsb = tsbs;
  } else if (!has_shared) {
    tas = ta;
    tbs = tb;
    tsbs = tsb;
  }
  auto kern = grouped_gemm_w4a8_kernel<MODE, STAGES>;
  const size_t smem = L::bytes(gp.E);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, n_sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
  return launch_kernel(kern, dim3(n_sms > 0 ? n_sms : 1), dim3(kThreads), smem, stream, pdl, ta, tb, tsb, tas, tbs,
                       tsbs, gp);
}

}  // namespace

cudaError_t launch_grouped_gemm_w4a8(const W4a8GemmProblem& pr, cudaStream_t stream, bool pdl) {
  const bool has_shared = pr.s_rows != nullptr && pr.T_s > 0;
  if (pr.M <= 0 && !has_shared) return cudaSuccess;
  W8Params gp{};
  gp.offsets = pr.M > 0 ? pr.offsets : nullptr;
  gp.E = pr.E;
  gp.M = pr.M;
  gp.K = pr.K;
  gp.n_out = pr.n_out;
  gp.n_feat = pr.mode == 0 ? pr.n_out / 2 : pr.n_out;
  gp.n_ftiles = pr.mode == 0 ? pr.n_out / 256 : pr.n_out / 128;
  gp.sfa = pr.sf;
  gp.act = pr.act;
  gp.act_sf = pr.act_sf;
  gp.out = pr.out;
  gp.topk_w = pr.topk_w;
  gp.sorted_pair = pr.sorted_pair;
  gp.has_shared = has_shared ? 1 : 0;
  if (has_shared) {
    gp.T_s = pr.T_s;
    gp.n_out_s = pr.n_out_s;
    gp.n_feat_s = pr.mode == 0 ? pr.n_out_s / 2 : pr.n_out_s;
    gp.n_ftiles_s = pr.mode == 0 ? pr.n_out_s / 256 : pr.n_out_s / 128;
    gp.sfa_s = pr.s_sf;
    gp.act_s = pr.s_act;
    gp.act_sf_s = pr.s_act_sf;
    gp.out_s = pr.s_out;
  }
  gp.status = pr.status;
  gp.timeout_ns = kTimeoutNs;
  return pr.mode == 0 ? launch_w8<0, 5>(pr, gp, stream, pdl) : launch_w8<1, 10>(pr, gp, stream, pdl);
}

cudaError_t launch_w4a8_prepack(const uint8_t* codes, const uint8_t* scales, int E, int n_out, int K, int gate_up,
                                uint8_t* codes_p, uint8_t* sf_p, cudaStream_t stream) {
  const long long threads = (long long)E * n_out * 32;
  if (threads == 0) return cudaSuccess;
  w4a8_prepack_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(codes, scales, E, n_out, K, gate_up,
                                                                             codes_p, sf_p);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows_mx(const uint8_t* x_codes, const uint8_t* x_scales, const int32_t* sorted_pair, int M,
                                  int k, int T, int H, uint8_t* out_codes, uint8_t* out_sf, const int32_t* n_rows,
                                  unsigned* status, cudaStream_t stream, bool pdl) {
  if (M <= 0) return cudaSuccess;
  return launch_kernel(gather_rows_mx_kernel, dim3(M), dim3(128), 0, stream, pdl, x_codes, x_scales, sorted_pair, M,
                       k, T, H, out_codes, out_sf, n_rows, status);
}

}  // namespace moe
