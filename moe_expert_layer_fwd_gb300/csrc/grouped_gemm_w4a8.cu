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
//            (128-row half of a 256-row tile, 128-K chunk), the two halves' atoms of a chunk side by
//            side: byte (r % 32) * 16 + (r / 32) * 4 + b holds the scale of half-tile row r, block b --
//            the layout tcgen05.cp .32x128b.warpx4 turns into the tensor-memory scale-factor layout of
//            an M = 128 block-scaled MMA (row r at lane r % 32 of every lane quarter, column r / 32,
//            byte b = the MMA's scale-factor id).
//   tokens   E4M3 codes [rows, K] and "padded scale rows" [rows, K/128, 16]: per row and 128-K
//            chunk, 16 bytes whose first four are the chunk's four block scales (the rest zero).  A
//            32-row slice of one chunk is the 32 x 16-byte source of one tcgen05.cp for the token
//            operand's scale factors (token n at lane n, column 0).
//
// Product (swap-AB, as the bf16 decode instances): weight rows are the MMA's operand A, two M = 128
// halves of a 256-row tile into two accumulators, read from shared memory in the padded E2M1 layout
// that TMA writes for CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B (each 16 codes = 8 bytes followed by 8
// zero bytes, so a 128-code row is a 128-byte swizzled row); the expert's token rows are the operand B
// (E4M3, 128-byte swizzled rows; N = 32 in the decode instance, below).  One 128-K chunk = 4 MMAs of K = 32 per half, each
// naming its block with the scale-factor ids of the instruction descriptor; the scale factors are
// copied into a per-stage tensor-memory slot by the MMA thread (tcgen05.cp, which the MMAs issued
// after it by the same thread are ordered behind).
//
// Loads (decode instance).  Each SM's TMA engine works through its copies one after another (about
// 0.33 us per 16 KB), so it carries only the weights: one 16-KB copy per 128-K chunk of the tile's 256 weight rows (A ring,
// 32 KB in shared memory in the padded layout; the prepacked codes of a (tile, chunk) are one contiguous
// block) and one bulk copy of the weight scale atoms per 512-K window (4 chunks).  The window's 32 token
// rows and their scale rows, read from L2 again by every feature tile of an expert, are copied by two
// loader warps with cp.async (T ring).  Two MMA-issuing threads, one per 128-row weight half, keep the
// tensor pipe fed: an N = 32 block-scaled MMA takes about as long to issue as a wide one.
//
// Mode 0 (gate/up + SwiGLU + MXFP8 of act): the prepacked gate/up tile of 256 rows holds features
// [128 f, 128 f + 128): half p, lane quarter q, lane l holds the gate (l < 16) or up (l >= 16) row
// of feature 128 f + 32 q + 16 p + (l % 16), so one epilogue warp ends up with a whole 32-feature
// block of act for each token column: the block maximum is a 4-step shuffle reduction, and the warp
// writes the E4M3 codes and the E8M0 scale byte of that block for the down GEMM.
// Mode 1 (down + routing weight): 256 output features per tile, bf16 times topk_w[sorted_pair[pos]].
//
// Warp roles of the decode instance (288 threads, one persistent CTA per SM, static round-robin tiles;
// an expert's token tiles that reuse a weight tile run next to each other): warp 0 TMA producer, warp 1 TMEM allocator +
// MMA issuer of weight half 0, warps 2-5 epilogue (one per TMEM lane quarter), warp 6 MMA issuer of
// half 1, warps 7-8 token loaders.
//
// Prefill-sized problems (more than 32 rows per expert on average) take a wide instance of the same
// kernel: tiles of 112 token columns (MMA N = the tile's rows rounded up to 16), so a weight tile is
// read once per 112 rows instead of once per 32.  Its token rows come by TMA (one 112-row box per
// 128-K chunk, completing on the window's barrier by byte count); its single loader warp only places
// each token's four block scales at byte (r % 32) * 16 + (r / 32) * 4 of the chunk's 512-byte block,
// the tensor-memory scale-factor layout of an operand of up to 128 rows (token r at lane r % 32,
// column r / 32, as for the weights), then fences and arrives.  Eight epilogue warps, two per lane
// quarter, split a tile's four 32-column chunks (with four, the epilogue bounded the GEMMs).  Windows
// of two chunks, three of them in flight where the expert tables leave room.  Every wait is bounded
// (2 s): on expiry the CTA raises its abort flag, records DEV_ERR_TIMEOUT, lets its copies land,
// drains its MMAs and frees TMEM.
#include "moe_common.cuh"
#include "moe_internal.h"

#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kBM = 128;                  // weight rows per MMA (M), one half of a tile
constexpr int kTR = 256;                  // weight rows per tile and per A copy
constexpr int kKC = 128;                  // K per chunk: 4 MMAs of K = 32 per half
constexpr int kABox = kTR * 128;          // shared-memory bytes of one A copy (padded codes): 32 KB
constexpr int kATx = kTR * kKC / 2;       // bytes the A copy moves (and counts on the barrier): 16 KB
constexpr int kSF = 512;                  // one scale-factor block: 128 rows' atom, or 32 padded token scale rows
// Warp roles of an instance with NT token columns per tile: warp 0 producer, warp 1 MMA issuer of weight
// half 0, kEPI epilogue warps, the MMA issuer of half 1, kLW loader warps.  The decode instance has one
// epilogue warp per TMEM lane quarter and two loader warps (token rows and scales by cp.async); the wide
// one two epilogue warps per quarter (its tiles have up to four 32-column chunks) and one loader warp
// (the token rows come by TMA, the loader only places their scales).
template <int NT>
struct W8Roles {
  static constexpr int kEPI = NT > 32 ? 8 : 4;
  static constexpr int kPerQ = kEPI / 4;      // epilogue warps sharing a TMEM lane quarter
  static constexpr int kMMA2 = 2 + kEPI;
  static constexpr int kLD0 = kMMA2 + 1;
  static constexpr int kLW = NT > 32 ? 1 : 2;
  static constexpr int kLoaders = 32 * kLW;
  static constexpr int kThreads = 32 * (kLD0 + kLW);
};
constexpr int kMaxDynSmem = 232448;
constexpr unsigned long long kTimeoutNs = 2000000000ull;

// NT token columns per tile (MMA N at most), WIN 128-K chunks per token window.
template <int MODE, int STAGES, int TSLOTS, int NT, int WIN>
struct W8Layout {
  static constexpr int kNTPad = (NT + 31) / 32 * 32;               // epilogue: 32-column chunks
  static constexpr int kTB = WIN * NT * kKC;                       // token rows of a window
  static constexpr int kTSB = WIN * kSF;                           // their scales: one 512-byte block per chunk
  static constexpr int kTSA = WIN * 2 * kSF;                       // the window's weight scale atoms
  static constexpr int kTSlot = kTB + kTSB + kTSA;
  static constexpr int kAOff = 0;                                  // STAGES x 32 KB
  static constexpr int kTOff = STAGES * kABox;                     // TSLOTS x kTSlot
  static constexpr int kBarOff = kTOff + TSLOTS * kTSlot;
  static constexpr int kNumBars = 2 * STAGES + 2 * TSLOTS + 6;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // mode 1: the routing weights of each epilogue warp's columns (kMine 32-column chunks per warp)
  static constexpr int kMine = (kNTPad / 32 + W8Roles<NT>::kPerQ - 1) / W8Roles<NT>::kPerQ;
  static constexpr int kScaleOff = kMiscOff + 16;
  static constexpr int kTabOff = kScaleOff + (MODE == 1 ? W8Roles<NT>::kEPI * kMine * 32 * 4 : 0);
  // tensor memory: two accumulator buffers of 2 x NT columns, then a scale-factor slot per A stage:
  // per weight half (one per MMA issuer) 4 columns of weight scales and 4 of token scales
  static constexpr int kAccCols = 2 * NT;
  static constexpr int kSFCol0 = 2 * kAccCols;
  static constexpr int kSFColsPerStage = 16;
  static constexpr int kColsNeeded = kSFCol0 + STAGES * kSFColsPerStage;
  static constexpr uint32_t kTmemCols = kColsNeeded <= 64 ? 64 : (kColsNeeded <= 128 ? 128 : (kColsNeeded <= 256 ? 256 : 512));
  static constexpr int kFeatPerTile = MODE == 0 ? 128 : 256;
  static_assert(kColsNeeded <= 512, "TMEM");
  // the epilogue reads whole 32-column chunks: the last one may run past NT, never past TMEM
  static_assert(kAccCols + NT + kNTPad <= (int)kTmemCols, "TMEM reads");
  static_assert(NT % 16 == 0 && NT >= 32 && NT <= 128, "token tile");
  static_assert(kABox % 1024 == 0 && kTOff % 1024 == 0 && kTSlot % 1024 == 0 && (NT * kKC) % 1024 == 0, "alignment");
  static constexpr int kMaxE = (kMaxDynSmem - 1024 - kTabOff) / 8 - 1;  // experts whose tables fit
  static_assert(kMaxE >= 64, "shared memory");
  static size_t bytes(int E) { return 1024 + kTabOff + 2 * (size_t)(E + 1) * 4; }
};

struct W8Params {
  const int32_t* offsets;
  int E, M, K;
  int n_out, n_ftiles, n_feat;      // routed: weight rows per expert, 256-row tiles per expert, features
  const uint8_t* b_rows;            // token rows [M, K] E4M3 (read by the loader warps)
  const uint8_t* b_sf;              // their padded scale rows [M, K/128, 16]
  const uint8_t* bs_rows;           // shared segment: [T_s, K] and [T_s, K/128, 16]
  const uint8_t* bs_sf;
  const uint8_t* sfa;               // weight scale atoms [E*n_out/256][K/128][2][512]
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

template <int NT>
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
    t.row_base = s_off[lo] + m * NT;
    t.rows = min(NT, s_off[lo + 1] - t.row_base);
  } else {
    const int local = tile - routed_total;
    const int nt = (p.T_s + NT - 1) / NT;
    const bool m_major = p.T_s > p.n_out_s;
    const int m = m_major ? local / p.n_ftiles_s : local % nt;
    t.shared = 1;
    t.e = -1;
    t.nt = nt;
    t.f = m_major ? local - m * p.n_ftiles_s : local / nt;
    t.row_base = m * NT;
    t.rows = min(NT, p.T_s - t.row_base);
  }
  return t;
}

// Instruction descriptor of tcgen05.mma kind::mxf8f6f4 .block_scale: A E2M1 (5), B E4M3 (0), both
// K-major, E8M0 scale factors, M = 128, N = n (a multiple of 16); the scale-factor ids of A (bits 29-30)
// and B (bits 4-5) select the byte of each 32-bit tensor-memory scale column, i.e. the K block.
__device__ __forceinline__ uint32_t w4a8_idesc(uint32_t sf_id, int n) {
  uint32_t d = 0;
  d |= sf_id << 4;                 // B scale-factor id
  d |= 5u << 7;                    // A format: E2M1
  d |= 0u << 10;                   // B format: E4M3
  d |= (uint32_t)(n >> 3) << 17;   // N / 8
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

// cp.async of 16 bytes global -> shared (zero-filled when src_bytes is 0).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
               : "memory");
}

// cp.async of 4 bytes global -> shared (zero-filled when src_bytes is 0).
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
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

template <int MODE, int STAGES, int TSLOTS, int NT, int WIN>
__global__ void __launch_bounds__(W8Roles<NT>::kThreads, 1)
    grouped_gemm_w4a8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAs,
                             const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmBs,
                             const W8Params p) {
  using L = W8Layout<MODE, STAGES, TSLOTS, NT, WIN>;
  using R = W8Roles<NT>;
  constexpr int kEPI = R::kEPI, kMMA2 = R::kMMA2, kLD0 = R::kLD0, kLoaders = R::kLoaders, kThreads = R::kThreads;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* afull = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* aempty = afull + STAGES;
  uint64_t* wfull = aempty + STAGES;     // T ring (512-K windows)
  uint64_t* wempty = wfull + TSLOTS;
  uint64_t* tfull = wempty + TSLOTS;     // accumulators
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;           // one per MMA issuer
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
      mbar_init(&afull[s], 1);
      mbar_init(&aempty[s], 2);                // both MMA issuers release a stage
    }
    for (int s = 0; s < TSLOTS; ++s) {
      mbar_init(&wfull[s], 1 + kLoaders);      // the producer (scale atoms) and every loader thread
      mbar_init(&wempty[s], 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 2);
      mbar_init(&tempty[b], kEPI);
    }
    mbar_init(&done[0], 1);
    mbar_init(&done[1], 1);
    *abort_flag = 0;
    *cfg_bad = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    if (p.has_shared) tma_prefetch_desc(&tmAs);
    if (NT > 32) {
      tma_prefetch_desc(&tmB);
      if (p.has_shared) tma_prefetch_desc(&tmBs);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, L::kTmemCols);
  // The routing offsets are read before griddepcontrol.wait: moe_layer_forward_w4a8 writes them two
  // or more launches earlier (then at least the MXFP8 row gather runs), and a kernel starts only
  // after its predecessor has waited for the one before.  Waiting here instead measured ~3 us more
  // per decode layer.
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
      else sum += (n + NT - 1) / NT;
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
      run += n > 0 ? (n + NT - 1) / NT : 0;
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
  const int shared_total = (*cfg_bad || !p.has_shared) ? 0 : ((p.T_s + NT - 1) / NT) * p.n_ftiles_s;
  const int total = routed_total + shared_total;
  const int KB = p.K / kKC;  // chunks per tile (K is a multiple of 128)

  if (warp == 0) {
    // ------------------------------------------------------------ producer (one lane)
    if (lane == 0) {
      const uint64_t pol_first = policy_evict_first();
      const uint64_t pol_last = policy_evict_last();
      int as = 0, ws = 0;
      uint32_t aph = 0, wph = 0;
      uint32_t a_issued = 0, w_issued = 0;
      bool ok = true;
      // Inside a layer forward this kernel may start while its predecessor finishes (programmatic
      // dependent launch): wait for it before reading the rows it writes, then let the next launch.
      pdl_wait();
      pdl_launch_dependents();
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const W8Tile t = w8_tile<NT>(tile, routed_total, s_off, s_tt, p);
        const CUtensorMap* mA = t.shared ? &tmAs : &tmA;
        const CUtensorMap* mB = t.shared ? &tmBs : &tmB;
        const int n_out = t.shared ? p.n_out_s : p.n_out;
        const int a_tile = ((t.shared ? 0 : t.e * n_out) + t.f * kTR) / kTR;  // 256-row tile of the weights
        const uint8_t* sfa = (t.shared ? p.sfa_s : p.sfa) + (size_t)a_tile * KB * 2 * kSF;
        const uint64_t pol_a = t.nt > 1 ? pol_last : pol_first;  // weight tiles read again stay in L2
        for (int kb = 0; kb < KB && ok; ++kb) {
          if (kb % WIN == 0) {
            // the window's weight scale atoms (the loader warps copy its token rows and their scales)
            if (!mbar_wait_bounded(&wempty[ws], wph ^ 1u, abort_flag, p.timeout_ns, p.status)) {
              ok = false;
              break;
            }
            const int nch = min(WIN, KB - kb);
            uint8_t* slot = smem + L::kTOff + ws * L::kTSlot;
            // the wide instance's token rows come by TMA too: one NT-row box per chunk (rows past the
            // end of the matrix read as zeros)
            const uint32_t tx = (uint32_t)(nch * 2 * kSF) + (NT > 32 ? (uint32_t)(nch * NT * kKC) : 0u);
            mbar_arrive_expect_tx(&wfull[ws], tx);
            bulk_load(slot + L::kTB + L::kTSB, sfa + (size_t)kb * 2 * kSF, (uint32_t)(nch * 2 * kSF), &wfull[ws],
                      pol_a);
            if (NT > 32)
              for (int c = 0; c < nch; ++c)
                tma_load_2d(slot + c * (NT * kKC), mB, (kb + c) * kKC, t.row_base, &wfull[ws], pol_last);
            ++w_issued;
            if (++ws == TSLOTS) {
              ws = 0;
              wph ^= 1u;
            }
          }
          if (!mbar_wait_bounded(&aempty[as], aph ^ 1u, abort_flag, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&afull[as], (uint32_t)kATx);
          tma_load_2d(smem + L::kAOff + as * kABox, mA, 0, ((int)a_tile * KB + kb) * kTR, &afull[as], pol_a);
          ++a_issued;
          if (++as == STAGES) {
            as = 0;
            aph ^= 1u;
          }
        }
      }
      // Drain: the last fill of every stage and window slot must have landed before the CTA exits
      // (one deadline for all).
      const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
      for (int s = 0; s < STAGES + TSLOTS; ++s) {
        const bool is_a = s < STAGES;
        const uint32_t issued = is_a ? a_issued : w_issued;
        const int nst = is_a ? STAGES : TSLOTS;
        const int k = is_a ? s : s - STAGES;
        const uint32_t n = issued / nst + ((uint32_t)k < issued % nst ? 1u : 0u);
        const uint64_t now = globaltimer_ns();
        if (n) mbar_wait_bounded(is_a ? &afull[k] : &wfull[k], (n - 1u) & 1u, abort_flag,
                                 deadline > now ? deadline - now : 0, p.status, false);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == kMMA2) {
    // ------------------------------------------------------------ MMA issuers, one per weight half
    // Each issues its half's MMAs into its own accumulator and copies the scale factors it needs into
    // its own tensor-memory columns (tcgen05 operations of different threads are not ordered).
    if (lane == 0) {
      const int half = warp == 1 ? 0 : 1;
      int as = 0, ws = 0;
      uint32_t aph = 0, wph = 0;
      bool ok = true;
      int it = 0;
      const uint64_t desc0 = umma_desc_sw128(smem_u32(smem));
      const uint64_t sfd0 = sf_src_desc(smem_u32(smem));
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++it) {
        const int buf = it & 1;
        const uint32_t acc_ph = (uint32_t)(it >> 1) & 1u;
        // MMA N: the tile's rows rounded up to 16 (the narrow instance always takes its 32 columns)
        const int nmma = NT == 32 ? 32 : ((w8_tile<NT>(tile, routed_total, s_off, s_tt, p).rows + 15) & ~15);
        if (!mbar_wait_bounded(&tempty[buf], acc_ph ^ 1u, abort_flag, p.timeout_ns, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * L::kAccCols + half * NT);
        for (int kb = 0; kb < KB; ++kb) {
          const int ci = kb % WIN;  // chunk inside the window
          if (ci == 0) {
            if (!mbar_wait_bounded(&wfull[ws], wph, abort_flag, p.timeout_ns, p.status)) {
              ok = false;
              break;
            }
          }
          if (!mbar_wait_bounded(&afull[as], aph, abort_flag, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t woff = (uint32_t)(L::kTOff + ws * L::kTSlot);
          const uint32_t sfa_t = tmem_base + (uint32_t)(L::kSFCol0 + as * L::kSFColsPerStage + 8 * half);
          const uint32_t sfb_t = sfa_t + 4u;
          tmem_cp_32x128_x4(sfa_t, sfd0 + (uint64_t)((woff + L::kTB + L::kTSB + (ci * 2 + half) * kSF) >> 4));
          tmem_cp_32x128_x4(sfb_t, sfd0 + (uint64_t)((woff + L::kTB + ci * kSF) >> 4));
          const uint64_t ad0 = desc0 + (uint64_t)((L::kAOff + as * kABox + half * kBM * 128) >> 4);
          const uint64_t bd0 = desc0 + (uint64_t)((woff + ci * NT * kKC) >> 4);
#pragma unroll
          for (int kk = 0; kk < kKC / 32; ++kk)
            umma_w4a8(d, ad0 + (uint64_t)((kk * 32) >> 4), bd0 + (uint64_t)((kk * 32) >> 4),
                      w4a8_idesc((uint32_t)kk, nmma), sfa_t, sfb_t, (kb | kk) != 0);
          umma_commit(&aempty[as]);
          if (++as == STAGES) {
            as = 0;
            aph ^= 1u;
          }
          if (ci == WIN - 1 || kb == KB - 1) {
            umma_commit(&wempty[ws]);  // the window's token rows and scales are no longer read
            if (++ws == TSLOTS) {
              ws = 0;
              wph ^= 1u;
            }
          }
        }
        if (!ok) break;
        umma_commit(&tfull[buf]);
      }
      // Drain: every MMA issued by this thread must be complete before TMEM is freed.
      umma_commit(&done[half]);
      mbar_wait_bounded(&done[half], 0, abort_flag, p.timeout_ns, p.status, false);
    }
    __syncwarp();
  } else if (warp >= kLD0) {
    // ------------------------------------------------------------ token loaders
    // Decode instance (cp.async): the window's 32 token rows x 4 chunks (128 bytes each, written in the
    // 128-byte swizzle the MMA's operand descriptor expects: 16-byte unit j of row r at j ^ (r % 8)) and
    // their padded scale rows; rows and chunks past the end are zero-filled.  Each thread waits for its
    // own copies and fences them to the async proxy before arriving, one window behind the copies it
    // issues.
    const int lt = (warp - kLD0) * 32 + lane;
    pdl_wait();  // the token rows come from the previous kernel
    if constexpr (NT > 32) {
      // Wide instance: the producer's TMA brings the token rows; the loaders only put each token's four
      // block scales (the first 4 bytes of its padded scale row) at byte (r % 32) * 16 + (r / 32) * 4 of
      // the chunk's 512-byte block -- the scale-factor layout of an operand of up to 128 rows, as for
      // the weights: token r at lane r % 32, column r / 32 -- then fence them to the async proxy and
      // arrive.
      constexpr int kPer = (WIN * NT + kLoaders - 1) / kLoaders;
      int ws = 0;
      uint32_t wph = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const W8Tile t = w8_tile<NT>(tile, routed_total, s_off, s_tt, p);
        const uint8_t* sfr = t.shared ? p.bs_sf : p.b_sf;
        const int nrows = t.shared ? p.T_s : p.M;
        const int nmma = (t.rows + 15) & ~15;  // token rows the tile's MMAs read
        bool ok = true;
        for (int kb0 = 0; kb0 < KB; kb0 += WIN) {
          uint32_t wv[kPer];
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            const int piece = lt + i * kLoaders;  // (chunk, row)
            const int c = piece / NT, r = piece - c * NT;
            const int row = t.row_base + r, kc = kb0 + c;
            const bool valid = piece < WIN * NT && r < nmma && row < nrows && kc < KB;
            wv[i] = valid ? __ldg(reinterpret_cast<const uint32_t*>(sfr + ((size_t)row * KB + kc) * 16)) : 0u;
          }
          bool w = (lane == 0) ? mbar_wait_bounded(&wempty[ws], wph ^ 1u, abort_flag, p.timeout_ns, p.status) : false;
          w = __shfl_sync(0xffffffffu, w, 0);
          if (!w) {
            ok = false;
            break;
          }
          uint8_t* blk = smem + L::kTOff + ws * L::kTSlot + L::kTB;
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            const int piece = lt + i * kLoaders;
            const int c = piece / NT, r = piece - c * NT;
            if (piece < WIN * NT && r < nmma)
              *reinterpret_cast<uint32_t*>(blk + c * kSF + (r & 31) * 16 + (r >> 5) * 4) = wv[i];
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(&wfull[ws]);
          if (++ws == TSLOTS) {
            ws = 0;
            wph ^= 1u;
          }
        }
        if (!ok) break;
      }
    } else {
    int ws = 0, prev = -1;
    uint32_t wph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      const W8Tile t = w8_tile<NT>(tile, routed_total, s_off, s_tt, p);
      const uint8_t* rows = t.shared ? p.bs_rows : p.b_rows;
      const uint8_t* sfr = t.shared ? p.bs_sf : p.b_sf;
      const int nrows = t.shared ? p.T_s : p.M;
      for (int kb0 = 0; kb0 < KB; kb0 += WIN) {
        bool w = (lane == 0) ? mbar_wait_bounded(&wempty[ws], wph ^ 1u, abort_flag, p.timeout_ns, p.status) : false;
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        uint8_t* slot = smem + L::kTOff + ws * L::kTSlot;
#pragma unroll 4
        for (int i = 0; i < L::kTB / 16 / kLoaders; ++i) {
          const int piece = lt + i * kLoaders;  // (chunk, row, 16-byte unit)
          const int c = piece >> 8, r = (piece >> 3) & 31, j = piece & 7;
          const int row = t.row_base + r, kc = kb0 + c;
          const bool valid = row < nrows && kc < KB;
          const uint8_t* src = valid ? rows + (size_t)row * p.K + kc * kKC + j * 16 : rows;
          cp_async16(slot + c * (NT * kKC) + r * kKC + ((j ^ (r & 7)) << 4), src, valid ? 16u : 0u);
        }
        // the 32 padded scale rows of each chunk as they are: token r lands at lane r, column 0
#pragma unroll
        for (int i = 0; i < L::kTSB / 16 / kLoaders; ++i) {
          const int piece = lt + i * kLoaders;  // (chunk, row)
          const int c = piece >> 5, r = piece & 31;
          const int row = t.row_base + r, kc = kb0 + c;
          const bool valid = row < nrows && kc < KB;
          const uint8_t* src = valid ? sfr + ((size_t)row * KB + kc) * 16 : sfr;
          cp_async16(slot + L::kTB + c * kSF + r * 16, src, valid ? 16u : 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (prev >= 0) {
          asm volatile("cp.async.wait_group 1;" ::: "memory");
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(&wfull[prev]);
        }
        prev = ws;
        if (++ws == TSLOTS) {
          ws = 0;
          wph ^= 1u;
        }
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (prev >= 0) mbar_arrive(&wfull[prev]);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-5)
    const int qw = warp & 3;             // TMEM lane quarter this warp may access
    const int half_c = (warp - 2) >> 2;  // which of the quarter's warps this is
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const W8Tile t = w8_tile<NT>(tile, routed_total, s_off, s_tt, p);
      const int buf = it & 1;
      const uint32_t acc_ph = (uint32_t)(it >> 1) & 1u;
      // Mode 1: the routing weights of the tile's rows, fetched before the accumulator wait, in shared
      // memory (read back as broadcast vector loads): wsc[32 r + j] is the weight of column 32 cc + j of
      // this warp's r-th chunk cc = half_c + kPerQ r.
      constexpr int kMine = L::kMine;
      float* wsc = s_scale + (warp - 2) * kMine * 32;
      const bool scale = MODE == 1 && !t.shared && p.topk_w != nullptr;
      if (scale) {
        int pr[kMine];
#pragma unroll
        for (int r = 0; r < kMine; ++r) {
          const int col = (half_c + R::kPerQ * r) * 32 + lane;
          pr[r] = col < t.rows ? __ldg(p.sorted_pair + t.row_base + col) : -1;
        }
#pragma unroll
        for (int r = 0; r < kMine; ++r) wsc[32 * r + lane] = pr[r] >= 0 ? __ldg(p.topk_w + pr[r]) : 0.0f;
        __syncwarp();
      }
      bool w = (lane == 0) ? mbar_wait_sleep(&tfull[buf], acc_ph, abort_flag, p.timeout_ns, p.status) : false;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(qw * 32) << 16) + (uint32_t)(buf * L::kAccCols);
      // 32 token columns at a time (the last chunk may read past the tile's columns: not stored); the
      // kPerQ warps of a lane quarter take chunks half_c, half_c + kPerQ, ...
      const int nch = (t.rows + 31) >> 5;
      const int last = nch > half_c ? half_c + (nch - 1 - half_c) / R::kPerQ * R::kPerQ : -1;  // this warp's last
      if (last < 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
#pragma unroll
      for (int r = 0; r < kMine; ++r) {
      const int cc = half_c + R::kPerQ * r;
      if (cc >= nch) break;
      const int c0 = cc * 32;
      uint32_t v[2][32];
      tmem_ld32_async(tb + (uint32_t)c0, v[0]);
      tmem_ld32_async(tb + (uint32_t)(NT + c0), v[1]);
      tmem_wait_ld();
      if (cc == last) {
        // release the accumulator after this warp's last load: everything below works on registers
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
      if (MODE == 0) {
        // SwiGLU: lanes 0-15 hold gate rows, lanes 16-31 the up rows of the same features; the gate
        // lanes finish token columns 0-15, the up lanes columns 16-31
        const bool is_gate = lane < 16;
        float a[2][16];
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float send = __uint_as_float(is_gate ? v[half][16 + i] : v[half][i]);
            const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
            const float g = is_gate ? __uint_as_float(v[half][i]) : recv;
            const float u = is_gate ? recv : __uint_as_float(v[half][16 + i]);
            a[half][i] = __fdividef(g, 1.0f + __expf(-g)) * u;
          }
        // MXFP8 of act: per token column, the 32 features of this warp's block are 16 lanes x 2 halves
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
          const int col = c0 + col_half + i;
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
        const int col = c0 + col_half + (lane & 15);
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
        uint16_t* out = t.shared ? p.out_s : p.out;
        const int n_feat = t.shared ? p.n_feat_s : p.n_feat;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int feat = t.f * L::kFeatPerTile + half * kBM + qw * 32 + lane;
          float o[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[half][i]) * (scale ? wsc[32 * r + i] : 1.0f);
          uint16_t* orow = out + (size_t)t.row_base * n_feat + feat;
          store_pairs16_bf16(o, lane, orow, (size_t)n_feat, c0, t.rows, feat < n_feat);
          store_pairs16_bf16(o + 16, lane, orow, (size_t)n_feat, c0 + 16, t.rows, feat < n_feat);
        }
      }
      }
      if (MODE == 1) __syncwarp();  // the next tile rewrites this warp's routing weights
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
// codes [E, n_out, K/2], scales [E, n_out, K/32] (moe_mxfp4_quantize) -> codes_p
// [E*n_out/256][K/128][256][64] (per 256-row tile and 128-K chunk, the tile's rows' 64 code bytes of
// the chunk: every block the GEMM loads is one contiguous 16 KB; gate/up rows regrouped when gate_up)
// and the scale atoms sf_p [E*n_out/256][K/128][2][512].
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
  const long long tile256 = row / kTR;
  const int r256 = (int)(row % kTR);
  for (int c = lane; c < K / 32; c += 32) {  // 16-byte piece c of the row: K chunk c / 4
    const long long blk = tile256 * (K / kKC) + c / 4;
    uint4* cd = reinterpret_cast<uint4*>(codes_p + (blk * kTR + r256) * (kKC / 2));
    cd[c % 4] = __ldg(cs + c);
  }
  const int nb = K / 32;
  const int half = (int)((row / kBM) % 2);
  const int r = (int)(row % kBM);
  for (int b = lane; b < nb; b += 32) {
    const int chunk = b >> 2, kb = b & 3;
    sf_p[((tile256 * (K / kKC) + chunk) * 2 + half) * kSF + (r % 32) * 16 + (r / 32) * 4 + kb] =
        __ldg(scales + srow * nb + b);
  }
}

// MXFP8 token rows for the W4A8 GEMMs: out_codes[pos] = x_codes[t] and the padded scale row
// out_sf[pos] = (x_scales[t][4c .. 4c+3], 0 x 12) per 128-K chunk c, with t = sorted_pair[pos] / k
// (sorted_pair NULL: t = pos, and no codes are written -- the scale rows of the token rows
// themselves, for the shared expert).  A block moves kMxRows consecutive rows; each thread loads its
// 16-byte piece of every one of them before storing any, so kMxRows independent loads are in flight.
// n_rows: optional device bound on the rows (rows past it are left alone); a row whose pair index is
// out of range is skipped and reported.
constexpr int kMxRows = 8;

__global__ void __launch_bounds__(256) gather_rows_mx_kernel(const uint8_t* __restrict__ x_codes,
                                                             const uint8_t* __restrict__ x_scales,
                                                             const int32_t* __restrict__ sorted_pair, int M, int k,
                                                             int T, int H, uint8_t* __restrict__ out_codes,
                                                             uint8_t* __restrict__ out_sf,
                                                             const int32_t* __restrict__ n_rows, unsigned* status) {
  __shared__ int s_t[kMxRows];  // source token of each row of the block, -1: left alone
  pdl_wait();
  pdl_launch_dependents();
  const int r0 = blockIdx.x * kMxRows;
  if (threadIdx.x < kMxRows) {
    const int pos = r0 + threadIdx.x;
    int t = -1;
    if (pos < M && (!n_rows || pos < __ldg(n_rows))) {
      t = pos;
      if (sorted_pair) {
        const int sp = __ldg(sorted_pair + pos);
        if (sp < 0 || (long long)sp >= (long long)T * k) {
          set_status(status, DEV_ERR_BOUNDS);
          t = -1;
        } else {
          t = sp / k;
        }
      }
    }
    s_t[threadIdx.x] = t;
  }
  __syncthreads();
  int src[kMxRows];
#pragma unroll
  for (int u = 0; u < kMxRows; ++u) src[u] = s_t[u];
  if (out_codes) {
    const int H16 = H / 16;
    for (int c = threadIdx.x; c < H16; c += blockDim.x) {
      uint4 v[kMxRows];
#pragma unroll
      for (int u = 0; u < kMxRows; ++u)
        if (src[u] >= 0) v[u] = __ldg(reinterpret_cast<const uint4*>(x_codes + (size_t)src[u] * H) + c);
#pragma unroll
      for (int u = 0; u < kMxRows; ++u)
        if (src[u] >= 0) reinterpret_cast<uint4*>(out_codes + (size_t)(r0 + u) * H)[c] = v[u];
    }
  }
  const int nc = H / kKC;  // padded scale entries per row
  for (int i = threadIdx.x; i < kMxRows * nc; i += blockDim.x) {
    const int u = i / nc, c = i - u * nc;
    const int t = s_t[u];
    if (t < 0) continue;
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(x_scales + (size_t)t * (H / 32)) + c);
    reinterpret_cast<uint4*>(out_sf + (size_t)(r0 + u) * nc * 16)[c] = make_uint4(w, 0u, 0u, 0u);
  }
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

// E2M1 codes in 256-row x 128-code boxes, each 16 codes landing as 8 bytes followed by 8 zero bytes
// (the operand layout of the block-scaled MMA for 4-bit A), 128-byte swizzle.
// The prepacked codes are seen as one matrix of (rows * K/128) rows of 128 codes (the chunk-major
// blocks stacked): block (tile, chunk) starts at row (tile * K/128 + chunk) * 256.
// E4M3 token rows [rows, K] in NT-row x 128-byte boxes, 128-byte swizzle (the wide instance's operand B).
bool make_map_rows_e4m3(CUtensorMap* m, const void* base, int K, long long rows, int box_rows) {
  auto fn = encode_fn_w8();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {(cuuint32_t)kKC, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_e2m1(CUtensorMap* m, const void* base, int K, long long rows) {
  auto fn = encode_fn_w8();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kKC, (cuuint64_t)rows * (K / kKC)};
  cuuint64_t strides[1] = {(cuuint64_t)kKC / 2};
  cuuint32_t box[2] = {(cuuint32_t)kKC, (cuuint32_t)kTR};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int STAGES, int TSLOTS, int NT, int WIN>
cudaError_t launch_w8(const W4a8GemmProblem& pr, W8Params gp, cudaStream_t stream, bool pdl) {
  using L = W8Layout<MODE, STAGES, TSLOTS, NT, WIN>;
  const bool has_shared = gp.has_shared != 0;
  CUtensorMap ta, tas, tb, tbs;
  if (pr.M > 0 && !make_map_e2m1(&ta, pr.codes, pr.K, (long long)pr.E * pr.n_out)) return cudaErrorInvalidValue;
  if (has_shared && !make_map_e2m1(&tas, pr.s_codes, pr.K, pr.n_out_s)) return cudaErrorInvalidValue;
  if (NT > 32) {
    if (pr.M > 0 && !make_map_rows_e4m3(&tb, pr.a_rows, pr.K, pr.M, NT)) return cudaErrorInvalidValue;
    if (has_shared && !make_map_rows_e4m3(&tbs, pr.s_rows, pr.K, pr.T_s, NT)) return cudaErrorInvalidValue;
  }
  // with no routed rows the routed maps are never read (and vice versa): alias them
  if (pr.M <= 0) {
    ta = tas;
    tb = tbs;
  } else if (!has_shared) {
    tas = ta;
    tbs = tb;
  }
  if (NT == 32) {  // the token rows come by cp.async: the maps are not read
    tb = ta;
    tbs = ta;
  }
  auto kern = grouped_gemm_w4a8_kernel<MODE, STAGES, TSLOTS, NT, WIN>;
  if (gp.E > L::kMaxE) return cudaErrorInvalidValue;
  const size_t smem = L::bytes(gp.E);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, n_sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
  return launch_kernel(kern, dim3(n_sms > 0 ? n_sms : 1), dim3(W8Roles<NT>::kThreads), smem, stream, pdl, ta, tas, tb, tbs, gp);
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
  gp.n_ftiles = pr.n_out / kTR;
  gp.b_rows = pr.a_rows;
  gp.b_sf = pr.a_sf;
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
    gp.n_ftiles_s = pr.n_out_s / kTR;
    gp.bs_rows = pr.s_rows;
    gp.bs_sf = pr.s_rows_sf;
    gp.sfa_s = pr.s_sf;
    gp.act_s = pr.s_act;
    gp.act_sf_s = pr.s_act_sf;
    gp.out_s = pr.s_out;
  }
  gp.status = pr.status;
  gp.timeout_ns = kTimeoutNs;
  // Decode-like problems (a few rows per expert) walk 32 token columns per tile behind a deep weight
  // ring; prefill-like ones take 112 columns per tile, so each weight tile is read once per 112 rows.
  if (w4a8_narrow(pr.M, pr.E, has_shared, pr.T_s))
    return pr.mode == 0 ? launch_w8<0, 4, 3, 32, 4>(pr, gp, stream, pdl) : launch_w8<1, 4, 3, 32, 4>(pr, gp, stream, pdl);
  // three token windows where the expert tables (and the down GEMM's routing weights) leave room for
  // them, else two
  if (pr.mode == 0)
    return pr.E <= W8Layout<0, 4, 3, 112, 2>::kMaxE ? launch_w8<0, 4, 3, 112, 2>(pr, gp, stream, pdl)
                                                    : launch_w8<0, 4, 2, 112, 2>(pr, gp, stream, pdl);
  return pr.E <= W8Layout<1, 4, 3, 112, 2>::kMaxE ? launch_w8<1, 4, 3, 112, 2>(pr, gp, stream, pdl)
                                                  : launch_w8<1, 4, 2, 112, 2>(pr, gp, stream, pdl);
}

bool w4a8_narrow(int M, int E, bool has_shared, int T_s) {
  return (long long)M <= 32LL * E && (!has_shared || T_s <= 32);
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
  const int threads = H / 16 >= 256 ? 256 : ((H / 16 + 31) / 32 * 32);
  return launch_kernel(gather_rows_mx_kernel, dim3((unsigned)((M + kMxRows - 1) / kMxRows)), dim3(threads), 0, stream,
                       pdl, x_codes, x_scales, sorted_pair, M, k, T, H, out_codes, out_sf, n_rows, status);
}

}  // namespace moe
