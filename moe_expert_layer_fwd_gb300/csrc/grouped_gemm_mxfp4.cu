// a3/a4 with MXFP4 expert weights on GB300: the grouped gate/up GEMM (+ SwiGLU) and the grouped
// down GEMM (+ routing weight) of decode, the expert weights stored as E2M1 codes with one E8M0
// scale per 32 elements of K, and the kernels that make and lay out those weights.
//
// Source: Qwen3-MoE low-latency inference practice (Atlas A3/950), MoE EP / W4A8 section: the
// expert weights are MXFP4 and the grouped matmuls read them; the matmul and SwiGLU themselves
// are those of "MoE TP optimisation: computation decomposition", as in the bf16 GEMMs.
//
// Decode streams every active expert's weights once per step (HBM-bound), so 4-bit weights move
// about a quarter of the bf16 bytes.  The product stays on the f16 tensor-core path
// (tcgen05.mma kind::f16, fp32 accumulators in TMEM) with the weight operand A in TMEM:
// dequantising warps turn each 128-row x 128-K operand stage of codes into f16 and store it straight
// into tensor memory (tcgen05.st, thread = weight row = TMEM lane), while TMA streams the next codes;
// one MMA thread issues 8 MMAs of K = 16 per stage.
// Staging the f16 weights in shared memory instead would move 8 bytes through it (a write and the
// MMA's read) per code byte, more than shared memory delivers at HBM rate; with A in TMEM shared
// memory only carries the codes and the token rows.  The dequantisation is exact: an E2M1 value times a
// power of two is an f16 value while the power stays in f16's range, so every weight row r carries
// an exponent offset W_r = (largest scale exponent of the row) - 13, applied in fp32 by the
// epilogue, and a block with scale 2^X enters the f16 operand as e2m1 * 2^(X - W_r), at most
// 6 * 2^13.  Blocks more than 36 binades below the row's largest block would round in f16's
// subnormal range (their share of the row's sum is below fp32 resolution).  Token rows and act
// are f16 on this path (saturated to +-65504).
//
// Warp roles (480 threads, one CTA per SM, static round-robin tiles of 128 weight rows x 32 token
// columns; f-major inside an expert, like the bf16 decode instances):
//   warp 0      TMA: codes (128 rows x 256 K = 16 KB, 128-byte swizzle) and their scales (1 KB)
//               into a RAW-deep ring;
//   warp 1      TMEM allocation + the single MMA-issuing thread (M = 128, N = 16 or 32, A from
//               TMEM, B from shared memory);
//   warp 2      TMA: the token rows of each raw stage (32 rows x 256 K f16 as four 64-K boxes,
//               128-byte swizzle) into an RB-deep ring, released when the stage's MMAs are done;
//   warps 3-10  dequantisation, two groups of four warps taking alternate operand stages (two
//               stages in flight); in a group, warp w covers TMEM lane quarter w % 4 and thread =
//               weight row: 128 codes (cvt e2m1x2 -> f16x2, times the block's f16 multiplier)
//               -> 64 TMEM columns (two tcgen05.st), then wait::st, fence, one arrival per warp;
//   warps 11-14 epilogue: tcgen05.ld 32 lanes x 32 columns, times 2^W_r, then SwiGLU (mode 0,
//               act in f16) or times the routing weight (mode 1, bf16 out).
// Every wait is bounded (2 s): on expiry the CTA raises its abort flag, records DEV_ERR_TIMEOUT,
// lets its copies land, drains its MMAs and frees TMEM.
#include "moe_common.cuh"
#include "moe_internal.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kBM = 128;                       // weight rows per tile (UMMA M)
constexpr int kNT = 32;                        // token columns per tile (UMMA N <= 32)
constexpr int kAK = 128;                       // K per operand stage (8 MMAs of K = 16 between two waits)
constexpr int kBK = 64;                        // K per token-row TMA box: one 128-byte row of f16
constexpr int kRawK = 256;                     // K per raw stage: one 128-byte row of codes
constexpr int kPerRaw = kRawK / kAK;           // operand stages per raw stage
constexpr int kCodeBytes = kBM * kRawK / 2;    // 16 KB
constexpr int kScaleBytes = (kRawK / 32) * kBM;  // 1 KB: 8 scale lines of 128 rows
constexpr int kBBox = kNT * kBK * 2;           // 4 KB: 32 token rows x 64 K f16 (one swizzled TMA box)
constexpr int kBBytes = (kRawK / kBK) * kBBox; // 16 KB: token rows of one raw stage (256 K)
constexpr int kACols = kAK / 2;                // TMEM columns of one f16 weight operand stage
constexpr int kDQ = 8;                         // dequantising warps: two groups of four
constexpr int kDQG = 4;                        // warps per group (one per TMEM lane quarter)
constexpr int kEPI = 4;                        // epilogue warps
constexpr int kThreads = 32 * (3 + kDQ + kEPI);
constexpr int kMaxDynSmem = 232448;
constexpr unsigned long long kTimeoutNs = 2000000000ull;
static_assert(kDQG * 32 == kBM, "one dequantising thread per weight row in a group");

template <int RAW, int RB, int OPS>
struct W4Layout {
  static constexpr int kCodeOff = 0;
  static constexpr int kBOff = RAW * kCodeBytes;
  static constexpr int kScaleOff = kBOff + RB * kBBytes;
  static constexpr int kBarOff = kScaleOff + RAW * kScaleBytes;
  // full_r, empty_r (RAW each), full_b, empty_b (RB each), full_a, empty_o (OPS each), tfull[2], tempty[2], done
  static constexpr int kNumBars = 2 * RAW + 2 * RB + 2 * OPS + 5;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kRowScaleOff = kMiscOff + 16;  // mode 1: routing weight per token column, per epilogue warp
  static constexpr int kTabOff = kRowScaleOff + kEPI * kNT * 4;
  static constexpr int kACol0 = 2 * kNT;             // TMEM: two 32-column accumulators, then OPS A stages
  static constexpr int kColsNeeded = kACol0 + OPS * kACols;
  static constexpr uint32_t kTmemCols = kColsNeeded <= 128 ? 128 : (kColsNeeded <= 256 ? 256 : 512);
  static_assert(kColsNeeded <= 512, "TMEM");
  static_assert(1024 + kTabOff + 2 * 1025 * 4 <= kMaxDynSmem, "shared memory");
  static size_t bytes(int E) { return 1024 + kTabOff + 2 * (size_t)(E + 1) * 4; }
};

struct W4Params {
  const int32_t* offsets;
  int E, M, K;
  int n_out, n_ftiles, n_feat;  // weight rows per expert, feature tiles per expert, output features per row
  void* out;                    // mode 0: f16 act [M, ld_out]; mode 1: bf16 [M, ld_out]
  int ld_out;
  const float* omega;           // [E * n_out] 2^W_r (row order of the prepacked weights)
  const float* topk_w;
  const int32_t* sorted_pair;
  unsigned* status;
  unsigned long long timeout_ns;
};

struct W4Tile {
  int e, f, row_base, rows;
};

__device__ __forceinline__ W4Tile w4_tile(int tile, const int* s_off, const int* s_tt, const W4Params& p) {
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
  W4Tile t;
  t.e = lo;
  t.f = m_major ? local - m * p.n_ftiles : local / nt;
  t.row_base = s_off[lo] + m * kNT;
  t.rows = min(kNT, s_off[lo + 1] - t.row_base);
  return t;
}

// Instruction descriptor of tcgen05.mma kind::f16 with f16 A and B (both K-major), fp32
// accumulator, shape M x N (A and B formats 0 = f16).
__device__ __forceinline__ uint32_t umma_idesc_f16(int M, int N) {
  uint32_t d = 0;
  d |= 1u << 4;                   // D format: f32
  d |= (uint32_t)(N >> 3) << 17;  // N / 8
  d |= (uint32_t)(M >> 4) << 24;  // M / 16
  return d;
}

// 32 lanes x 32 bits, 32 consecutive columns (thread = lane).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] . B[smem]^T, kind::f16: A is M x 16 in tensor memory (lane = row, column c
// holding the f16 pair of K elements 2c, 2c + 1), B a shared-memory descriptor.
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Two E2M1 codes (bits 0-3 and 4-7 of v) -> f16x2 (the low nibble in the low half).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t v) {
  uint32_t d;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(d) : "r"(v));
  return d;
}

__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The f16 multiplier of a block, from its prepacked scale byte u: 0 -> 0, else 2^(u - 25)
// (u in [1, 38]; u <= 11 is a subnormal or the smallest normal power, bits 1 << (u - 1); above,
// the exponent field is u - 10).  Replicated into both halves.
__device__ __forceinline__ uint32_t block_multiplier_f16x2(uint32_t u) {
  const uint32_t h = u == 0u ? 0u : (u <= 11u ? (1u << (u - 1u)) : ((u - 10u) << 10));
  return h | (h << 16);
}

// f32 pair -> f16x2 rounded to nearest even, saturated to +-65504 (first operand -> high half).
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// All lanes wait (each lane's wait acquires the phase); false on any lane's timeout or abort.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          const W4Params& p) {
  const bool ok = mbar_wait_bounded(bar, parity, abort_flag, p.timeout_ns, p.status);
  return __all_sync(0xffffffffu, ok);
}

// Stores 16 token columns [col0, col0 + 16) of this lane's output feature, two features per
// 32-bit store (lanes l and l^1 hold adjacent features; one shfl_xor(1) per column pair).
template <bool F16>
__device__ __forceinline__ void store_pairs16_w4(const float* v, int lane, uint16_t* orow, size_t ld, int col0,
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
    if (ok && col < rows)
      *reinterpret_cast<uint32_t*>(base + (size_t)col * ld) = F16 ? pack_f16x2_sat(lo, hi) : pack_bf16x2(lo, hi);
  }
}

template <int RAW, int RB, int OPS, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_mxfp4_kernel(const __grid_constant__ CUtensorMap tmCodes, const __grid_constant__ CUtensorMap tmScales,
                              const __grid_constant__ CUtensorMap tmB, const W4Params p) {
  using L = W4Layout<RAW, RB, OPS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_r = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty_r = full_r + RAW;
  uint64_t* full_b = empty_r + RAW;
  uint64_t* empty_b = full_b + RB;
  uint64_t* full_a = empty_b + RB;
  uint64_t* empty_o = full_a + OPS;
  uint64_t* tfull = empty_o + OPS;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  volatile int* cfg_bad = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 8);
  float* s_rowscale = reinterpret_cast<float*>(smem + L::kRowScaleOff);
  int* s_off = reinterpret_cast<int*>(smem + L::kTabOff);
  int* s_tt = s_off + (p.E + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW; ++s) {
      mbar_init(&full_r[s], 1);
      mbar_init(&empty_r[s], kDQ);
    }
    for (int s = 0; s < RB; ++s) {
      mbar_init(&full_b[s], 1);
      mbar_init(&empty_b[s], 1);
    }
    for (int s = 0; s < OPS; ++s) {
      mbar_init(&full_a[s], kDQG);
      mbar_init(&empty_o[s], 1);
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
    tma_prefetch_desc(&tmCodes);
    tma_prefetch_desc(&tmScales);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, L::kTmemCols);
  // Offsets come from init-routing two launches back (see the bf16 GEMMs): complete before this
  // kernel may start.
  for (int i = threadIdx.x; i <= E; i += kThreads) s_off[i] = __ldg(p.offsets + i);
  __syncthreads();
  if (warp == 3) {
    // Validate offsets and build the prefix of token tiles per expert.
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

  const int total = *cfg_bad ? 0 : s_tt[E] * p.n_ftiles;
  const int KA = (p.K + kAK - 1) / kAK;          // operand stages per tile (K is a multiple of 64: the
                                                 // last one may hold 64)
  const int KR = (KA + kPerRaw - 1) / kPerRaw;   // raw stages per tile
  const int lines_per_tile = p.K / 32;           // scale lines of one 128-row weight tile

  if (warp == 0) {
    // ------------------------------------------------------------ codes + scales (TMA)
    // The weights do not depend on the previous kernel: stream them at once.
    pdl_launch_dependents();
    uint32_t issued = 0;
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const W4Tile t = w4_tile(tile, s_off, s_tt, p);
        const int wrow = t.e * p.n_out + t.f * kBM;
        const int line0 = (wrow / kBM) * lines_per_tile;
        for (int kr = 0; kr < KR; ++kr) {
          if (!mbar_wait_bounded(&empty_r[stage], phase ^ 1u, abort_flag, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_r[stage], kCodeBytes + kScaleBytes);
          tma_load_2d(smem + L::kCodeOff + stage * kCodeBytes, &tmCodes, kr * (kRawK / 2), wrow, &full_r[stage], pol);
          tma_load_2d(smem + L::kScaleOff + stage * kScaleBytes, &tmScales, 0, line0 + kr * (kRawK / 32),
                      &full_r[stage], pol);
          ++issued;
          if (++stage == RAW) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the last fill of every stage must have landed before the CTA exits.
      for (int s = 0; s < RAW; ++s) {
        const uint32_t n = issued / RAW + ((uint32_t)s < issued % RAW ? 1u : 0u);
        if (n) mbar_wait_bounded(&full_r[s], (n - 1u) & 1u, abort_flag, p.timeout_ns, p.status, false);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, bst = 0;
      uint32_t phase = 0, bph = 0;
      bool ok = true;
      int it = 0;
      const uint64_t bdesc0 = umma_desc_sw128(smem_u32(smem + L::kBOff));
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++it) {
        const W4Tile t = w4_tile(tile, s_off, s_tt, p);
        const int buf = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_bounded(&tempty[buf], aph ^ 1u, abort_flag, p.timeout_ns, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * kNT);
        const uint32_t idesc = umma_idesc_f16(kBM, (t.rows + 15) & ~15);
        for (int ka = 0; ka < KA; ++ka) {
          const int j = ka % kPerRaw;
          if ((j == 0 && !mbar_wait_bounded(&full_b[bst], bph, abort_flag, p.timeout_ns, p.status)) ||
              !mbar_wait_bounded(&full_a[stage], phase, abort_flag, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tm = tmem_base + (uint32_t)(L::kACol0 + stage * kACols);
          const uint64_t bd = bdesc0 + (uint64_t)((bst * kBBytes + j * (kAK / kBK) * kBBox) >> 4);
          const bool full_k = p.K - ka * kAK >= kAK;  // false: the tile's last stage holds 64 of K
#pragma unroll
          for (int kk = 0; kk < kAK / 16; ++kk) {
            if (kk >= kBK / 16 && !full_k) break;
            // K step kk: TMEM columns 8kk.., token box kk / 4, 32-byte step kk % 4 inside it
            const uint64_t bk = bd + (uint64_t)(((kk / (kBK / 16)) * kBBox + (kk % (kBK / 16)) * 32) >> 4);
            umma_f16_tmem_a(d, a_tm + (uint32_t)(kk * 8), bk, idesc, (ka | kk) != 0);
          }
          umma_commit(&empty_o[stage]);
          if (++stage == OPS) {
            stage = 0;
            phase ^= 1u;
          }
          if (j == kPerRaw - 1 || ka == KA - 1) {
            umma_commit(&empty_b[bst]);  // the token rows of this raw stage are no longer read
            if (++bst == RB) {
              bst = 0;
              bph ^= 1u;
            }
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
  } else if (warp == 2) {
    // ------------------------------------------------------------ token rows (TMA)
    if (lane == 0) {
      pdl_wait();  // the token rows come from the previous kernel
      const uint64_t pol = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const W4Tile t = w4_tile(tile, s_off, s_tt, p);
        for (int kr = 0; kr < KR; ++kr) {
          const int nbox = min(kRawK / kBK, (p.K - kr * kRawK) / kBK);
          if (!mbar_wait_bounded(&empty_b[stage], phase ^ 1u, abort_flag, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_b[stage], (uint32_t)(nbox * kBBox));
          for (int j = 0; j < nbox; ++j)
            tma_load_2d(smem + L::kBOff + stage * kBBytes + j * kBBox, &tmB, kr * kRawK + j * kBK, t.row_base,
                        &full_b[stage], pol);
          ++issued;
          if (++stage == RB) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < RB; ++s) {
        const uint32_t n = issued / RB + ((uint32_t)s < issued % RB ? 1u : 0u);
        if (n) mbar_wait_bounded(&full_b[s], (n - 1u) & 1u, abort_flag, p.timeout_ns, p.status, false);
      }
    }
    __syncwarp();
  } else if (warp < 3 + kDQ) {
    // ------------------------------------------------------------ dequantisation
    const int g = (warp - 3) / kDQG;    // group: operand stages ka with ka % 2 == g
    const int q = warp & 3;             // TMEM lane quarter
    const int r = q * 32 + lane;        // weight row of the tile = TMEM lane
    const uint32_t sw = (uint32_t)(r & 7);
    const uint32_t a_lane = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)L::kACol0;
    int rs = 0, os = 0;
    uint32_t rph = 0, oph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      for (int ka = 0; ka < KA; ++ka) {
        const int j = ka % kPerRaw;
        if (j == 0 && !warp_wait(&full_r[rs], rph, abort_flag, p)) {
          ok = false;
          break;
        }
        if ((ka & 1) == g) {
          if (!warp_wait(&empty_o[os], oph ^ 1u, abort_flag, p)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* codes = smem + L::kCodeOff + rs * kCodeBytes + r * 128;
          const uint8_t* scl = smem + L::kScaleOff + rs * kScaleBytes + r;
#pragma unroll
          for (int hh = 0; hh < kAK / 64; ++hh) {
            uint32_t v[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              // 16-byte chunk of the row's 128 code bytes (32 codes, one scale block)
              const uint32_t chunk = (uint32_t)((kAK / 32) * j + 2 * hh + h);
              const uint4 cw = *reinterpret_cast<const uint4*>(codes + ((chunk ^ sw) << 4));
              const uint32_t mult = block_multiplier_f16x2(scl[chunk * kBM]);
              const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int by = 0; by < 4; ++by)
                  v[16 * h + 4 * i + by] = mul_f16x2(e2m1x2_to_f16x2(words[i] >> (8 * by)), mult);
              }
            }
            tmem_st32(a_lane + (uint32_t)(os * kACols + 32 * hh), v);
          }
          tmem_wait_st();
          tc_fence_before();  // the MMA thread reads these columns after the barrier
          __syncwarp();
          if (lane == 0) mbar_arrive(&full_a[os]);
        }
        if (j == kPerRaw - 1 || ka == KA - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_r[rs]);
          if (++rs == RAW) {
            rs = 0;
            rph ^= 1u;
          }
        }
        if (++os == OPS) {
          os = 0;
          oph ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int qw = warp & 3;  // TMEM lane quarter this warp may access
    const int ew = warp - 3 - kDQ;
    float* wsc = s_rowscale + ew * kNT;
    pdl_wait();  // routing weights and sorted_pair come from earlier kernels
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const W4Tile t = w4_tile(tile, s_off, s_tt, p);
      const int buf = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      const int wrow = t.e * p.n_out + t.f * kBM + qw * 32 + lane;  // this lane's weight row
      const float om = __ldg(p.omega + wrow);
      const bool scale = MODE == 1 && p.topk_w != nullptr;
      if (scale) {
        const int pr = lane < t.rows ? __ldg(p.sorted_pair + t.row_base + lane) : -1;
        wsc[lane] = pr >= 0 ? __ldg(p.topk_w + pr) : 0.0f;
        __syncwarp();
      }
      bool w = (lane == 0) ? mbar_wait_sleep(&tfull[buf], aph, abort_flag, p.timeout_ns, p.status) : false;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) break;
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32_async(tmem_base + ((uint32_t)(qw * 32) << 16) + (uint32_t)(buf * kNT), v);
      tmem_wait_ld();
      if (MODE == 0) {
        // packed gate/up: lanes 0-15 hold gate rows, lanes 16-31 the up rows of the same features
        const bool is_gate = lane < 16;
        const int feat = t.f * (kBM / 2) + qw * 16 + (lane & 15);
        const bool feat_ok = feat < p.n_feat;
        uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + (size_t)t.row_base * p.ld_out + feat;
        float a[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float mine_g = __uint_as_float(v[i]) * om;         // gate lanes: columns 0-15
          const float mine_u = __uint_as_float(v[16 + i]) * om;    // up lanes: columns 16-31
          const float send = is_gate ? __uint_as_float(v[16 + i]) * om : __uint_as_float(v[i]) * om;
          const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
          const float g = is_gate ? mine_g : recv;
          const float u = is_gate ? recv : mine_u;
          a[i] = __fdividef(g, 1.0f + __expf(-g)) * u;
        }
        store_pairs16_w4<true>(a, lane, orow, (size_t)p.ld_out, is_gate ? 0 : 16, t.rows, feat_ok);
      } else {
        const int feat = t.f * kBM + qw * 32 + lane;
        const bool feat_ok = feat < p.n_feat;
        uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + (size_t)t.row_base * p.ld_out + feat;
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]) * om * (scale ? wsc[i] : 1.0f);
        store_pairs16_w4<false>(o, lane, orow, (size_t)p.ld_out, 0, t.rows, feat_ok);
        store_pairs16_w4<false>(o + 16, lane, orow, (size_t)p.ld_out, 16, t.rows, feat_ok);
        __syncwarp();  // the next tile rewrites this warp's routing weights
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

// ---------------------------------------------------------------- weight preparation
// MXFP4 quantisation of bf16 rows [rows, K], one thread per block of 32 elements of K: scale
// exponent X = floor(log2 amax) - 2 (clamped to [-127, 127]; an all-zero block gets -127), the
// element v / 2^X rounded to the E2M1 grid nearest-even and saturated at 6; code = sign << 3 |
// magnitude index, element 2j in the low nibble of byte j.  The rounding is done on the exact
// fp32 quotient: quantum 0.5 below 2, 1 below 4, 2 above.
__global__ void __launch_bounds__(256) mxfp4_quantize_kernel(const uint4* __restrict__ w, long long n_blocks,
                                                             uint4* __restrict__ codes, uint8_t* __restrict__ scales) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_blocks) return;
  uint32_t u[16];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 q = __ldg(w + i * 4 + c);
    u[4 * c + 0] = q.x;
    u[4 * c + 1] = q.y;
    u[4 * c + 2] = q.z;
    u[4 * c + 3] = q.w;
  }
  uint32_t amax_bits = 0;  // |bf16| bit patterns order like their values
#pragma unroll
  for (int c = 0; c < 16; ++c) amax_bits = max(amax_bits, max(u[c] & 0x7FFFu, (u[c] >> 16) & 0x7FFFu));
  int shared;
  if (amax_bits == 0) {
    shared = -127;
  } else {
    const uint32_t f = amax_bits << 16;  // the fp32 bits of amax
    const int e8 = (int)(f >> 23);
    const int fl = e8 != 0 ? e8 - 127 : (31 - __clz((int)(f & 0x7FFFFFu))) - 149;
    shared = max(-127, min(127, fl - 2));
  }
  const float inv = ldexpf(1.0f, -shared);
  uint32_t out[4] = {0, 0, 0, 0};
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const uint32_t bits = (e & 1) ? (u[e >> 1] >> 16) : (u[e >> 1] & 0xFFFFu);
    const float q = __uint_as_float(bits << 16) * inv;
    const float a = fminf(fabsf(q), 6.0f);
    const float quantum = a < 2.0f ? 0.5f : (a < 4.0f ? 1.0f : 2.0f);
    const float rr = fminf(rintf(a / quantum) * quantum, 6.0f);
    const int r2 = (int)(rr * 2.0f);  // 0,1,2,3,4,6,8,12
    const uint32_t idx = r2 <= 4 ? (uint32_t)r2 : (r2 == 6 ? 5u : (r2 == 8 ? 6u : 7u));
    const uint32_t code = ((bits & 0x8000u) && idx ? 8u : 0u) | idx;
    out[e >> 3] |= code << (4 * (e & 7));
  }
  codes[i] = make_uint4(out[0], out[1], out[2], out[3]);
  scales[i] = (uint8_t)(shared + 127);
}

// Kernel layout of MXFP4 weights [E, n_out, K], one warp per row of the output:
//   codes_p   rows in the packed gate/up order when gate_up (as moe_prepack_w13), else unchanged;
//   scales_p  per 128-row tile, K/32 lines of 128 bytes (line kb holds the 128 rows' block kb):
//             u = X - W_r + 25 (0 when below 2^-24, i.e. X - W_r < -24);
//   omega     2^W_r, W_r = (largest X of the row) - 13.
__global__ void __launch_bounds__(256) mxfp4_prepack_kernel(const uint8_t* __restrict__ codes,
                                                            const uint8_t* __restrict__ scales, int E, int n_out,
                                                            int K, int gate_up, uint8_t* __restrict__ codes_p,
                                                            uint8_t* __restrict__ scales_p, float* __restrict__ omega) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)E * n_out) return;
  const int e = (int)(row / n_out), rr = (int)(row - (long long)e * n_out);
  int src = rr;
  if (gate_up) {
    const int g = rr >> 5, q = rr & 31;
    src = q < 16 ? g * 16 + q : n_out / 2 + g * 16 + (q - 16);
  }
  const long long srow = (long long)e * n_out + src;
  const int nb = K / 32;
  int xmax = -1000;
  for (int kb = lane; kb < nb; kb += 32) xmax = max(xmax, (int)__ldg(scales + srow * nb + kb) - 127);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) xmax = max(xmax, __shfl_xor_sync(0xffffffffu, xmax, o));
  const int W = xmax - 13;
  if (lane == 0) omega[row] = ldexpf(1.0f, W);
  uint8_t* sp = scales_p + ((row / kBM) * nb) * kBM + (row % kBM);
  for (int kb = lane; kb < nb; kb += 32) {
    const int j = (int)__ldg(scales + srow * nb + kb) - 127 - W;
    sp[(long long)kb * kBM] = (uint8_t)(j >= -24 ? j + 25 : 0);
  }
  const uint4* cs = reinterpret_cast<const uint4*>(codes + srow * (K / 2));
  uint4* cd = reinterpret_cast<uint4*>(codes_p + row * (K / 2));
  for (int c = lane; c < K / 32; c += 32) cd[c] = __ldg(cs + c);
}

// Routed token rows in f16: out[pos] = f16(x[sorted_pair[pos] / k]) (saturated), one block of
// 128 threads per row, 8 elements per thread and step.
__global__ void __launch_bounds__(128) gather_rows_f16_kernel(const uint4* __restrict__ x,
                                                              const int32_t* __restrict__ sorted_pair, int M, int k,
                                                              int T, int H8, uint4* __restrict__ out,
                                                              unsigned* status) {
  pdl_wait();
  pdl_launch_dependents();
  const int pos = blockIdx.x;
  if (pos >= M) return;
  const int sp = __ldg(sorted_pair + pos);
  if (sp < 0 || (long long)sp >= (long long)T * k) {  // the pair index itself, before the division
    if (threadIdx.x == 0) set_status(status, DEV_ERR_BOUNDS);
    return;
  }
  const int t = sp / k;
  for (int c = threadIdx.x; c < H8; c += blockDim.x) {
    const uint4 v = __ldg(x + (size_t)t * H8 + c);
    uint4 h;
    h.x = pack_f16x2_sat(bf16_lo(v.x), bf16_hi(v.x));
    h.y = pack_f16x2_sat(bf16_lo(v.y), bf16_hi(v.y));
    h.z = pack_f16x2_sat(bf16_lo(v.z), bf16_hi(v.z));
    h.w = pack_f16x2_sat(bf16_lo(v.w), bf16_hi(v.w));
    out[(size_t)pos * H8 + c] = h;
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

bool make_map_u8(CUtensorMap* m, const void* base, long long width, long long rows, int box_w, int box_h,
                 bool swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)width};
  cuuint32_t box[2] = {(cuuint32_t)box_w, (cuuint32_t)box_h};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_f16(CUtensorMap* m, const void* base, int K, long long rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kNT};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int RAW, int RB, int OPS, int MODE>
cudaError_t launch_w4(const Mxfp4GemmProblem& pr, const W4Params& gp, cudaStream_t stream, bool pdl) {
  using L = W4Layout<RAW, RB, OPS>;
  const long long wrows = (long long)pr.E * pr.n_out;
  CUtensorMap tc, ts, tb;
  if (!make_map_u8(&tc, pr.codes, pr.K / 2, wrows, kRawK / 2, kBM, true)) return cudaErrorInvalidValue;
  if (!make_map_u8(&ts, pr.scales, kBM, wrows / kBM * (pr.K / 32), kBM, kRawK / 32, false))
    return cudaErrorInvalidValue;
  if (!make_map_f16(&tb, pr.a_rows, pr.K, pr.M)) return cudaErrorInvalidValue;
  auto kern = grouped_gemm_mxfp4_kernel<RAW, RB, OPS, MODE>;
  const size_t smem = L::bytes(pr.E);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, n_sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
  return launch_kernel(kern, dim3(n_sms > 0 ? n_sms : 1), dim3(kThreads), smem, stream, pdl, tc, ts, tb, gp);
}

}  // namespace

cudaError_t launch_grouped_gemm_mxfp4(const Mxfp4GemmProblem& pr, cudaStream_t stream, bool pdl) {
  if (pr.M <= 0) return cudaSuccess;
  W4Params gp{};
  gp.offsets = pr.offsets;
  gp.E = pr.E;
  gp.M = pr.M;
  gp.K = pr.K;
  gp.n_out = pr.n_out;
  gp.n_feat = pr.mode == 0 ? pr.n_out / 2 : pr.n_out;
  gp.n_ftiles = pr.n_out / kBM;
  gp.out = pr.out;
  gp.ld_out = pr.ld_out;
  gp.omega = pr.omega;
  gp.topk_w = pr.topk_w;
  gp.sorted_pair = pr.sorted_pair;
  gp.status = pr.status;
  gp.timeout_ns = kTimeoutNs;
  return pr.mode == 0 ? launch_w4<7, 4, 7, 0>(pr, gp, stream, pdl) : launch_w4<7, 4, 7, 1>(pr, gp, stream, pdl);
}

cudaError_t launch_mxfp4_quantize(const uint16_t* w, long long rows, int K, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t stream) {
  const long long nb = rows * (K / 32);
  if (nb == 0) return cudaSuccess;
  mxfp4_quantize_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, stream>>>(reinterpret_cast<const uint4*>(w), nb,
                                                                          reinterpret_cast<uint4*>(codes), scales);
  return cudaGetLastError();
}

cudaError_t launch_mxfp4_prepack(const uint8_t* codes, const uint8_t* scales, int E, int n_out, int K, int gate_up,
                                 uint8_t* codes_p, uint8_t* scales_p, float* omega, cudaStream_t stream) {
  const long long threads = (long long)E * n_out * 32;
  if (threads == 0) return cudaSuccess;
  mxfp4_prepack_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(codes, scales, E, n_out, K, gate_up,
                                                                              codes_p, scales_p, omega);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows_f16(const uint16_t* x, const int32_t* sorted_pair, int M, int k, int T, int H,
                                   uint16_t* out, unsigned* status, cudaStream_t stream, bool pdl) {
  if (M <= 0) return cudaSuccess;
  return launch_kernel(gather_rows_f16_kernel, dim3(M), dim3(128), 0, stream, pdl, reinterpret_cast<const uint4*>(x),
                       sorted_pair, M, k, T, H / 8, reinterpret_cast<uint4*>(out), status);
}

}  // namespace moe
