// a6. Finalize-routing on GB300: unpermute + weighted sum (+ shared expert).
//
// Source: Qwen3-MoE low-latency inference practice, "GMM enablement and
// routing optimisation" (expert outputs are re-arranged back to token order
// and summed with their weights); Hy3 295B MoE practice, section 8.1 (the
// shared-expert term is added in this combine step).  The routing weight is
// already applied by the down-projection epilogue, so this step only sums.
//
// One block per token, its threads striding over the token's 16-byte column words:
// y[t, c:c+8] = sum_j y_perm[pair_pos[t*k+j], c:c+8] (+ shared[t]), in fp32 in slot order,
// rounded once to bf16.  The block reads the token's k row positions first, then issues the
// loads of up to kSlotBatch rows back to back, so that many independent loads are in flight.
// HBM-bound: reads P*H*2 + T*H*2 bytes, writes T*H*2.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__device__ __forceinline__ void acc8(float (&a)[8], const uint4& v) {
  a[0] += bf16_lo(v.x); a[1] += bf16_hi(v.x);
  a[2] += bf16_lo(v.y); a[3] += bf16_hi(v.y);
  a[4] += bf16_lo(v.z); a[5] += bf16_hi(v.z);
  a[6] += bf16_lo(v.w); a[7] += bf16_hi(v.w);
}

constexpr int kSlotBatch = 8;

__global__ void __launch_bounds__(512) finalize_kernel(const uint4* __restrict__ y_perm,
                                                       const int32_t* __restrict__ pair_pos,
                                                       const uint4* __restrict__ shared, int T, int k, int H8,
                                                       uint4* __restrict__ y) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int P = T * k;
  const int32_t* pp = pair_pos + (size_t)t * k;
  for (int c = threadIdx.x; c < H8; c += blockDim.x) {
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const size_t o_idx = (size_t)t * H8 + c;
    // the shared expert's word is loaded with the routed rows (it is still added last)
    uint4 sv = make_uint4(0u, 0u, 0u, 0u);
    if (shared) sv = __ldg(shared + o_idx);
    for (int j0 = 0; j0 < k; j0 += kSlotBatch) {
      const uint4* row[kSlotBatch];
#pragma unroll
      for (int j = 0; j < kSlotBatch; ++j) {
        const int pos = j0 + j < k ? __ldg(pp + j0 + j) : -1;
        row[j] = (unsigned)pos < (unsigned)P ? y_perm + (size_t)pos * H8 : nullptr;
      }
      uint4 v[kSlotBatch];
#pragma unroll
      for (int j = 0; j < kSlotBatch; ++j)
        if (row[j]) v[j] = __ldg(row[j] + c);
#pragma unroll
      for (int j = 0; j < kSlotBatch; ++j)
        if (row[j]) acc8(a, v[j]);
    }
    if (shared) acc8(a, sv);
    uint4 o;
    o.x = pack_bf16x2(a[0], a[1]);
    o.y = pack_bf16x2(a[2], a[3]);
    o.z = pack_bf16x2(a[4], a[5]);
    o.w = pack_bf16x2(a[6], a[7]);
    y[o_idx] = o;
  }
}

}  // namespace

cudaError_t launch_finalize(const uint16_t* y_perm, const int32_t* pair_pos, const uint16_t* shared, int T, int k,
                            int H, uint16_t* y, cudaStream_t stream, bool pdl) {
  if (T == 0 || H == 0) return cudaSuccess;
  const int H8 = H / 8;
  // Large batches: 128 threads per token, each taking every 128th column word (long_prefill 0.099 ->
  // 0.095 ms against one word per thread in blocks of up to 512).  Small batches keep the wide blocks:
  // with a few dozen tokens, 128-thread blocks leave most of the GPU idle (qwen3_decode 0.007 -> 0.011 ms).
  const int cap = T >= 1024 ? 128 : 512;
  const int threads = H8 >= cap ? cap : (H8 + 31) / 32 * 32;
  return launch_kernel(finalize_kernel, dim3((unsigned)T), dim3(threads), 0, stream, pdl,
                       reinterpret_cast<const uint4*>(y_perm), pair_pos, reinterpret_cast<const uint4*>(shared), T, k,
                       H8, reinterpret_cast<uint4*>(y));
}

}  // namespace moe
