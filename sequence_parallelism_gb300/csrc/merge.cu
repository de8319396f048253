// merge.cu -- combine per-block partial attention results by their
// log-sum-exp weights: the cross-device combine of ring attention ("Ring
// Attention", "Cómo funciona la atención en anillo": partial results are
// combined with the same cumulative softmax FlashAttention uses).
//
//   lse = log sum_p exp(lse_p),  out = sum_p exp(lse_p - lse) * out_p
//
// One warp per (b, t, h) row; float32 arithmetic; memory-bound (it reads P
// partial rows and writes one).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"

namespace sp {
namespace {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <typename T>
__global__ void __launch_bounds__(256) merge_kernel(const T* __restrict__ outs,
                                                    const float* __restrict__ lses, int P, int B,
                                                    int S, int H, int d, T* __restrict__ out,
                                                    float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const long long nrows = static_cast<long long>(B) * S * H;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long lse_pstride = static_cast<long long>(B) * H * S;
  const long long out_pstride = nrows * d;
  for (long long row = warp; row < nrows; row += nwarps) {
    const int h = static_cast<int>(row % H);
    const long long bt = row / H;
    const int t = static_cast<int>(bt % S);
    const int b = static_cast<int>(bt / S);
    const long long lse_off = (static_cast<long long>(b) * H + h) * S + t;
    float m = -INFINITY;
    for (int p = lane; p < P; p += 32) m = fmaxf(m, lses[p * lse_pstride + lse_off]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    T* orow = out + row * d;
    if (m == -INFINITY) {  // every partial empty
      for (int c = lane; c < d; c += 32) orow[c] = from_f<T>(0.f);
      if (lse && lane == 0) lse[lse_off] = -INFINITY;
      continue;
    }
    float w = 0.f;
    for (int p = lane; p < P; p += 32) w += expf(lses[p * lse_pstride + lse_off] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    const float inv_w = 1.f / w;
    for (int c0 = 0; c0 < d; c0 += 128) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int p = 0; p < P; ++p) {
        const float lp = lses[p * lse_pstride + lse_off];
        const float coef = (lp == -INFINITY) ? 0.f : expf(lp - m) * inv_w;
        const T* prow = outs + p * out_pstride + row * d;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = c0 + k * 32 + lane;
          if (c < d) acc[k] = fmaf(coef, to_f<T>(prow[c]), acc[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = c0 + k * 32 + lane;
        if (c < d) orow[c] = from_f<T>(acc[k]);
      }
    }
    if (lse && lane == 0) lse[lse_off] = m + logf(w);
  }
}

}  // namespace
}  // namespace sp

extern "C" sp_status sp_attn_merge_partials(const void* outs, const float* lses, int P, int B,
                                            int S, int H, int d, sp_dtype dtype, void* out,
                                            float* lse, sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_attn_merge_partials");
  sp::g_last_launches = 0;
  if (!outs || !lses || !out) return SP_ERR_INVALID_ARG;
  if (P < 1 || B < 1 || S < 1 || H < 1 || d < 1) return SP_ERR_INVALID_ARG;
  if (dtype != SP_BF16 && dtype != SP_F32) return SP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const long long nrows = static_cast<long long>(B) * S * H;
  long long blocks = (nrows + 7) / 8;
  const long long cap = static_cast<long long>(sp::device_sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (dtype == SP_BF16)
    sp::merge_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(outs), lses, P, B, S, H, d,
        static_cast<__nv_bfloat16*>(out), lse);
  else
    sp::merge_kernel<float><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const float*>(outs), lses, P, B, S, H, d, static_cast<float*>(out), lse);
  if (cudaGetLastError() != cudaSuccess) return SP_ERR_CUDA;
  sp::g_last_launches = 1;
  return SP_OK;
}
