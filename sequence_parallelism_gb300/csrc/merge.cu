// merge.cu -- combine per-block partial attention results by their
// log-sum-exp weights: the cross-device combine of ring attention ("Ring
// Attention", "Cómo funciona la atención en anillo": partial results are
// combined with the same cumulative softmax FlashAttention uses).
//
//   lse = log sum_p exp(lse_p),  out = sum_p exp(lse_p - lse) * out_p
//
// Memory-bound (it reads P partial rows and writes one); float32
// arithmetic.  merge_vec_kernel: every lane owns one 16-byte piece of a row
// (8 bf16 or 4 float32 values; a row of d = 128 bf16 is 16 lanes, so a warp
// merges two rows with 16-byte loads), and computes the row's weights from
// the P log-sum-exps itself; merge_kernel (one warp per row, element loads)
// takes the head sizes that do not split into 16-byte pieces.
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

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
  __device__ static void load(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      f[2 * e] = x.x;
      f[2 * e + 1] = x.y;
    }
  }
  __device__ static uint4 store(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 x = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
      w[e] = *reinterpret_cast<const uint32_t*>(&x);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Vec<float> {
  static constexpr int kN = 4;
  __device__ static void load(const uint4& u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 store(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

// lanes_per_row = d / Vec<T>::kN divides 32; the output and every partial
// row are 16-byte aligned; P <= kMaxP.  Rows are visited token-fastest
// within a (batch, head), so that neighbouring rows' log-sum-exps are
// neighbours in memory, and every lane issues all loads of its row (the P
// log-sum-exps and the 16-byte pieces of every partial) before any
// arithmetic.  (Two rows per lane in flight were slower at every size
// measured, L2-resident or not.)
template <typename T, int kMaxP>
__global__ void __launch_bounds__(256) merge_vec_kernel(const uint4* __restrict__ outs,
                                                        const float* __restrict__ lses, int P,
                                                        int B, int S, int H, int lanes_per_row,
                                                        uint4* __restrict__ out,
                                                        float* __restrict__ lse) {
  constexpr int kN = Vec<T>::kN;
  const int lane = threadIdx.x & 31;
  const int rows_per_warp = 32 / lanes_per_row;
  const int sub = lane / lanes_per_row, piece = lane % lanes_per_row;
  const long long nrows = static_cast<long long>(B) * S * H;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long lse_pstride = static_cast<long long>(B) * H * S;
  const long long out_pstride = nrows * lanes_per_row;  // in 16-byte pieces
  const long long step = nwarps * rows_per_warp;        // rows per sweep of all warps
  for (long long r = warp * rows_per_warp + sub; r < nrows; r += step) {
    // r = (b, h, t), t fastest: the lse index
    const int t = static_cast<int>(r % S);
    const long long bh = r / S;
    const int h = static_cast<int>(bh % H);
    const long long b = bh / H;
    const long long src = ((b * S + t) * H + h) * lanes_per_row + piece;  // (b, t, h)
    float l[kMaxP];
    uint4 xv[kMaxP];
#pragma unroll
    for (int p = 0; p < kMaxP; ++p) {
      l[p] = p < P ? lses[p * lse_pstride + r] : -INFINITY;
      if (p < P) xv[p] = outs[p * out_pstride + src];
    }
    float m = -INFINITY, w = 0.f;
#pragma unroll
    for (int p = 0; p < kMaxP; ++p) m = fmaxf(m, l[p]);
    if (m == -INFINITY) {  // every partial empty
      out[src] = make_uint4(0u, 0u, 0u, 0u);
      if (lse && piece == 0) lse[r] = -INFINITY;
      continue;
    }
#pragma unroll
    for (int p = 0; p < kMaxP; ++p)
      if (p < P) w += expf(l[p] - m);
    const float inv_w = 1.f / w;
    float acc[kN];
#pragma unroll
    for (int e = 0; e < kN; ++e) acc[e] = 0.f;
#pragma unroll
    for (int p = 0; p < kMaxP; ++p) {
      if (p >= P) break;
      const float coef = (l[p] == -INFINITY) ? 0.f : expf(l[p] - m) * inv_w;
      float x[kN];
      Vec<T>::load(xv[p], x);
#pragma unroll
      for (int e = 0; e < kN; ++e) acc[e] = fmaf(coef, x[e], acc[e]);
    }
    out[src] = Vec<T>::store(acc);
    if (lse && piece == 0) lse[r] = m + logf(w);
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
  {
    const int vec = dtype == SP_BF16 ? 8 : 4;
    const int lanes = d / vec;
    if (P <= 8 && d % vec == 0 && lanes <= 32 && 32 % lanes == 0 && sp::aligned(outs, 16) &&
        sp::aligned(out, 16)) {
      // enough warps to keep every SM's loads in flight
      const long long warps = (nrows * lanes + 31) / 32;
      long long blocks = (warps + 7) / 8;
      const long long cap = static_cast<long long>(sp::device_sm_count()) * 32;
      if (blocks > cap) blocks = cap;
      const uint4* in = static_cast<const uint4*>(outs);
      uint4* o = static_cast<uint4*>(out);
      const unsigned g = static_cast<unsigned>(blocks);
      // the partial count fixes how many loads a lane keeps in flight
      if (dtype == SP_BF16) {
        if (P <= 2)
          sp::merge_vec_kernel<__nv_bfloat16, 2><<<g, 256, 0, st>>>(in, lses, P, B, S, H, lanes,
                                                                   o, lse);
        else if (P <= 4)
          sp::merge_vec_kernel<__nv_bfloat16, 4><<<g, 256, 0, st>>>(in, lses, P, B, S, H, lanes,
                                                                   o, lse);
        else
          sp::merge_vec_kernel<__nv_bfloat16, 8><<<g, 256, 0, st>>>(in, lses, P, B, S, H, lanes,
                                                                   o, lse);
      } else {
        if (P <= 2)
          sp::merge_vec_kernel<float, 2><<<g, 256, 0, st>>>(in, lses, P, B, S, H, lanes, o, lse);
        else if (P <= 4)
          sp::merge_vec_kernel<float, 4><<<g, 256, 0, st>>>(in, lses, P, B, S, H, lanes, o, lse);
        else
          sp::merge_vec_kernel<float, 8><<<g, 256, 0, st>>>(in, lses, P, B, S, H, lanes, o, lse);
      }
      if (cudaGetLastError() != cudaSuccess) return SP_ERR_CUDA;
      sp::g_last_launches = 1;
      return SP_OK;
    }
  }
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
