// The step before gating on GB300: fused residual add + RMSNorm + cast, and the router gate GEMM.
//
// Source: Qwen3-MoE low-latency inference practice, section "fused RMSNorm + Cast": the norm
// before the MoE gives the hidden state in FP32 (for the gate) and in BF16 (for the experts), the
// residual add, the RMSNorm and the casts done by one op; without a residual (first layer) the op
// is RMSNorm + cast.  The router gate GEMM then maps the FP32 hidden state to router_logits.
//
// add_rms_norm_cast_kernel: one block per token, the row held in registers (VPT 16-byte words of 8
// bf16 per thread): r = bf16(h + res) rounded once (the residual stream, stored), sum of r^2 in
// fp32, one block reduction, y = r * rsqrt(mean + eps) * w, stored as fp32 and/or bf16 and/or
// MXFP8 (the same section's fused add + RMSNorm + dynamic MX quantisation, W4A8 path): blocks of
// 32 elements (4 words, held by 4 adjacent lanes) share the scale 2^(floor(log2 amax) - 8) as an
// E8M0 byte; each element y / scale is rounded to E4M3, nearest even, saturating at 448.
// HBM-bound: reads 2*T*H*2 B (+ H*2 weight), writes T*H*(4 + 2 + 2) B (cast outputs).
//
// router_logits_kernel: logits[T,E] = y32[T,H] . w_gate[E,H]^T in fp32 on the FP32 pipes (the
// fp32 input would be rounded by the bf16/tf32 tensor-core paths).  128 x 128 output tiles, 256
// threads with 8 x 8 outputs each, K in steps of 32 staged in shared memory (the bf16 weight
// widened there), split over K into slices added in order by a second kernel when there are
// too few tiles for the GPU; each slice accumulates in ascending k.  ALU-bound: 2*T*H*E FLOPs.
#include <cuda_fp8.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  return red[0];
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
  f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
  f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

template <int VPT>
__global__ void __launch_bounds__(kNormThreads) add_rms_norm_cast_kernel(
    const uint4* __restrict__ h, const uint4* res, const uint4* __restrict__ w, int H8, float eps,
    float4* __restrict__ y32, uint4* __restrict__ y16, uint4* res_out, uint2* __restrict__ mx_codes,
    uint8_t* __restrict__ mx_scales) {
  // res_out may alias res: each word is read and then written by the same thread
  __shared__ float red[32];
  const size_t row = (size_t)blockIdx.x * H8;
  float r[VPT][8];
  float ss = 0.0f;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = threadIdx.x + v * kNormThreads;
    if (c < H8) {
      float a[8];
      unpack8(__ldg(h + row + c), a);
      if (res) {
        float b[8];
        unpack8(res[row + c], b);
        // the residual stream: the sum rounded once to bf16
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = __uint_as_float((uint32_t)f32_to_bf16_rne(a[i] + b[i]) << 16);
      }
      if (res_out) {
        uint4 o;
        o.x = pack_bf16x2(a[0], a[1]);
        o.y = pack_bf16x2(a[2], a[3]);
        o.z = pack_bf16x2(a[4], a[5]);
        o.w = pack_bf16x2(a[6], a[7]);
        res_out[row + c] = o;  // exact: the values are bf16 already
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        r[v][i] = a[i];
        ss = fmaf(a[i], a[i], ss);
      }
    }
  }
  const float total = block_sum(ss, red);
  const float rstd = rsqrtf(total / (float)(H8 * 8) + eps);
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = threadIdx.x + v * kNormThreads;
    float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (c < H8) {
      float g[8];
      unpack8(__ldg(w + c), g);
#pragma unroll
      for (int i = 0; i < 8; ++i) y[i] = r[v][i] * rstd * g[i];
    }
    if (mx_codes) {  // uniform: every lane takes part in the block maximum
      float m = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(y[i]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      // shared exponent floor(log2 m) - 8, clamped to the E8M0 range; m == 0 or subnormal -> -127
      const int eb = (int)((__float_as_uint(m) >> 23) & 0xFF);
      const int shared = eb == 0 ? -127 : max(-127, min(127, eb - 127 - 8));
      const int k = -shared;  // y * 2^k: exact power-of-two scaling
      const float inv = k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
      if (c < H8) {
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 4; i += 2) {
          const __nv_fp8x2_storage_t a = __nv_cvt_float2_to_fp8x2(make_float2(y[i] * inv, y[i + 1] * inv),
                                                                  __NV_SATFINITE, __NV_E4M3);
          const __nv_fp8x2_storage_t b = __nv_cvt_float2_to_fp8x2(make_float2(y[i + 4] * inv, y[i + 5] * inv),
                                                                  __NV_SATFINITE, __NV_E4M3);
          lo |= (uint32_t)a << (8 * i);
          hi |= (uint32_t)b << (8 * i);
        }
        mx_codes[row + c] = make_uint2(lo, hi);
        if ((c & 3) == 0) mx_scales[(row + c) / 4] = (uint8_t)(shared + 127);
      }
    }
    if (c < H8) {
      if (y32) {
        y32[2 * (row + c)] = make_float4(y[0], y[1], y[2], y[3]);
        y32[2 * (row + c) + 1] = make_float4(y[4], y[5], y[6], y[7]);
      }
      if (y16) {
        uint4 o;
        o.x = pack_bf16x2(y[0], y[1]);
        o.y = pack_bf16x2(y[2], y[3]);
        o.z = pack_bf16x2(y[4], y[5]);
        o.w = pack_bf16x2(y[6], y[7]);
        y16[row + c] = o;
      }
    }
  }
}

constexpr int kRBM = 128, kRBN = 128, kRBK = 32;

// Split-K: blockIdx.z takes K slice [z * kslice, (z + 1) * kslice); with S > 1 slices each block
// writes its partial sums to part[z][T][E] and router_reduce_kernel adds them in slice order.
// A 128 x 128 output tile per 256-thread block, 8 x 8 outputs per thread: tokens ty*4..+3 and
// 64+ty*4..+3, experts tx*4..+3 and 64+tx*4..+3, so that the 128-bit shared-memory reads of a
// half-warp cover consecutive words.
__global__ void __launch_bounds__(256) router_logits_kernel(const float* __restrict__ y32,
                                                            const uint16_t* __restrict__ wg, int T, int H, int E,
                                                            int kslice, float* __restrict__ out) {
  __shared__ __align__(16) float As[kRBK][kRBM + 4];  // [k][token]
  __shared__ __align__(16) float Bs[kRBK][kRBN + 4];  // [k][expert]
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.x * kRBM, e0 = blockIdx.y * kRBN;
  const int kbeg = blockIdx.z * kslice, kend = min(H, kbeg + kslice);
  float* logits = out + (size_t)blockIdx.z * T * E;
  float acc[8][8] = {};
  // loaders: A 128 tokens x 32 k (16 floats per thread), B 128 experts x 32 k (16 bf16 per thread)
  const int l_row = tid >> 1, l_col = (tid & 1) * 16;
  for (int k0 = kbeg; k0 < kend; k0 += kRBK) {
    {
      const int t = t0 + l_row;
      float a[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) a[q] = 0.0f;
      if (t < T) {
        const float4* src = reinterpret_cast<const float4*>(y32 + (size_t)t * H + k0 + l_col);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 v = __ldg(src + q);
          a[4 * q] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
        }
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) As[l_col + q][l_row] = a[q];
    }
    {
      const int e = e0 + l_row;
      float f[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) f[q] = 0.0f;
      if (e < E) {
        const uint4* src = reinterpret_cast<const uint4*>(wg + (size_t)e * H + k0 + l_col);
        float g[8];
        unpack8(__ldg(src), g);
#pragma unroll
        for (int q = 0; q < 8; ++q) f[q] = g[q];
        unpack8(__ldg(src + 1), g);
#pragma unroll
        for (int q = 0; q < 8; ++q) f[8 + q] = g[q];
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) Bs[l_col + q][l_row] = f[q];
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < kRBK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[k][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[k][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[k][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[k][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
      if (e < E) logits[(size_t)t * E + e] = acc[i][j];
    }
  }
}

__global__ void __launch_bounds__(256) router_reduce_kernel(const float* __restrict__ part, int S, size_t n,
                                                            float* __restrict__ logits) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float s = part[i];
  for (int z = 1; z < S; ++z) s += part[(size_t)z * n + i];  // slice order: deterministic
  logits[i] = s;
}

}  // namespace

int router_splits(int T, int H, int E, int n_sms) {
  // enough blocks for two waves; slices of at least 64 of K
  const long long tiles = (long long)((T + kRBM - 1) / kRBM) * ((E + kRBN - 1) / kRBN);
  int S = (int)((2LL * n_sms + tiles - 1) / tiles);
  S = S < 1 ? 1 : S;
  const int max_s = H / 64 > 0 ? H / 64 : 1;
  return S > max_s ? max_s : S;
}

cudaError_t launch_add_rms_norm_cast(const uint16_t* h, const uint16_t* res, const uint16_t* w, int T, int H,
                                     float eps, float* y32, uint16_t* y16, uint16_t* res_out, cudaStream_t stream,
                                     uint8_t* mx_codes, uint8_t* mx_scales) {
  if (T == 0) return cudaSuccess;
  const int H8 = H / 8;
  const int vpt = (H8 + kNormThreads - 1) / kNormThreads;
  auto args = [&](auto kern) {
    kern<<<T, kNormThreads, 0, stream>>>(reinterpret_cast<const uint4*>(h), reinterpret_cast<const uint4*>(res),
                                          reinterpret_cast<const uint4*>(w), H8, eps, reinterpret_cast<float4*>(y32),
                                          reinterpret_cast<uint4*>(y16), reinterpret_cast<uint4*>(res_out),
                                          reinterpret_cast<uint2*>(mx_codes), mx_scales);
    return cudaGetLastError();
  };
  if (vpt <= 1) return args(add_rms_norm_cast_kernel<1>);
  if (vpt <= 2) return args(add_rms_norm_cast_kernel<2>);
  return args(add_rms_norm_cast_kernel<4>);
}

cudaError_t launch_router_logits(const float* y32, const uint16_t* w_gate, int T, int H, int E, float* logits,
                                 float* part, int S, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  // K slices: a multiple of the 32-deep step
  const int kslice = ((H + S - 1) / S + kRBK - 1) / kRBK * kRBK;
  S = (H + kslice - 1) / kslice;
  dim3 grid((T + kRBM - 1) / kRBM, (E + kRBN - 1) / kRBN, S);
  router_logits_kernel<<<grid, 256, 0, stream>>>(y32, w_gate, T, H, E, kslice, S > 1 ? part : logits);
  if (S == 1) return cudaGetLastError();
  const size_t n = (size_t)T * E;
  router_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(part, S, n, logits);
  return cudaGetLastError();
}

}  // namespace moe
