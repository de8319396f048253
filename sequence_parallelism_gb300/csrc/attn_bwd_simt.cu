// attn_bwd_simt.cu -- backward of blockwise ring attention on the CUDA cores.
//
// Training is what the pages use sequence parallelism for ("Ulysses SP:
// entrenar modelos con millones de tokens"); the ring keeps each query block
// resident while key/value blocks circulate ("Ring Attention", "Cómo funciona
// la atención en anillo").  The gradients are the derivatives of the forward:
//   P = exp(scale * Q K^T - lse)   (lse from the forward; masked pairs 0)
//   dP = dO V^T,  dS = P * (dP - D),  D_t = sum_c dO[t, c] O[t, c]
//   dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO
// Three kernels: D per query row; dQ with the query block resident and the
// key/value blocks in ring order j = (i - s) mod P; dK and dV with the
// key/value block resident and the query blocks in the order that block meets
// them on the ring, i = (j + s) mod P, every query head of the GQA group added
// inside the CTA (no atomics).  float32 arithmetic; inputs float32 or bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "attn_common.cuh"

namespace sp {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRows = kWarps * kRowsPerWarp;  // resident rows per CTA
constexpr int kChunk = 32;                    // streamed rows per step
constexpr int kMaxE = 8;                      // d <= 256: columns per lane

template <typename T>
__device__ __forceinline__ float ld(const T* p, long long i);
template <>
__device__ __forceinline__ float ld<float>(const float* p, long long i) { return p[i]; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p, long long i) {
  return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ void st(T* p, long long i, float v);
template <>
__device__ __forceinline__ void st<float>(float* p, long long i, float v) { p[i] = v; }
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, long long i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

// D[b][h][t] = sum_c dout[b][t][h][c] * out[b][t][h][c]; one warp per row.
template <typename T>
__global__ void __launch_bounds__(256) bwd_dot_kernel(const T* __restrict__ out,
                                                      const T* __restrict__ dout, int B, int S,
                                                      int H, int d, float* __restrict__ D) {
  const int lane = threadIdx.x & 31;
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (row >= static_cast<long long>(B) * S * H) return;
  const int h = static_cast<int>(row % H);
  const long long bt = row / H;
  const int t = static_cast<int>(bt % S);
  const int b = static_cast<int>(bt / S);
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) acc = fmaf(ld(dout, row * d + c), ld(out, row * d + c), acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) D[(static_cast<long long>(b) * H + h) * S + t] = acc;
}

__device__ __forceinline__ bool allowed(const BwdArgs& a, int b, long long tq, long long tk) {
  if (!a.doc_start) return true;
  return tk <= tq && a.doc_start[static_cast<long long>(b % a.pos_rows) * a.S + tq] <= tk;
}

// dQ: CTA = 16 query rows of block i for one (b, h); key/value chunks of 32
// in ring order.  Lane j scores key j; lanes own output columns lane + 32e.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) bwd_dq_kernel(BwdArgs a, int ntiles) {
  extern __shared__ float sm[];
  const int d = a.d;
  float* Qs = sm;                        // [kRows][d]
  float* dOs = Qs + kRows * d;           // [kRows][d]
  float* Ks = dOs + kRows * d;           // [kChunk][d + 1]
  float* Vs = Ks + kChunk * (d + 1);     // [kChunk][d + 1]
  const int tile = blockIdx.x % ntiles, i = blockIdx.x / ntiles;
  const int h = blockIdx.y, b = blockIdx.z, kvh = h / (a.Hq / a.Hkv);
  const int Lb = a.S / a.P, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* dout = static_cast<const T*>(a.dout);
  const long long qs = static_cast<long long>(a.Hq) * d, ks = static_cast<long long>(a.Hkv) * d;
  const long long qb = static_cast<long long>(b) * a.S * qs + static_cast<long long>(h) * d;
  const long long kb = static_cast<long long>(b) * a.S * ks + static_cast<long long>(kvh) * d;
  for (int idx = threadIdx.x; idx < kRows * d; idx += blockDim.x) {
    const int r = idx / d, c = idx % d;
    const long long u = static_cast<long long>(tile) * kRows + r;
    float qv = 0.f, dv = 0.f;
    if (u < Lb) {
      const long long off = qb + block_token(a.order, a.S, a.P, i, u) * qs + c;
      qv = ld(q, off);
      dv = ld(dout, off);
    }
    Qs[idx] = qv;
    dOs[idx] = dv;
  }
  float lse_r[kRowsPerWarp], D_r[kRowsPerWarp], acc[kRowsPerWarp][kMaxE];
  long long tq_r[kRowsPerWarp];
  bool live[kRowsPerWarp];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const long long u = static_cast<long long>(tile) * kRows + warp * kRowsPerWarp + rr;
    live[rr] = u < Lb;
    tq_r[rr] = live[rr] ? block_token(a.order, a.S, a.P, i, u) : 0;
    const long long li = (static_cast<long long>(b) * a.Hq + h) * a.S + tq_r[rr];
    lse_r[rr] = live[rr] ? a.lse[li] : 0.f;
    D_r[rr] = live[rr] ? a.Dsum[li] : 0.f;
#pragma unroll
    for (int e = 0; e < kMaxE; ++e) acc[rr][e] = 0.f;
  }
  for (int s = 0; s < a.P; ++s) {
    const int j = ((i - s) % a.P + a.P) % a.P;
    for (int w0 = 0; w0 < Lb; w0 += kChunk) {
      const int wn = min(kChunk, Lb - w0);
      __syncthreads();
      for (int idx = threadIdx.x; idx < kChunk * d; idx += blockDim.x) {
        const int r = idx / d, c = idx % d;
        float kv = 0.f, vv = 0.f;
        if (r < wn) {
          const long long off = kb + block_token(a.order, a.S, a.P, j, w0 + r) * ks + c;
          kv = ld(k, off);
          vv = ld(v, off);
        }
        Ks[r * (d + 1) + c] = kv;
        Vs[r * (d + 1) + c] = vv;
      }
      __syncthreads();
      const long long tk = block_token(a.order, a.S, a.P, j, w0 + lane);
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        if (!live[rr]) continue;
        const float* qr = Qs + (warp * kRowsPerWarp + rr) * d;
        const float* dr = dOs + (warp * kRowsPerWarp + rr) * d;
        const float* kr = Ks + lane * (d + 1);
        const float* vr = Vs + lane * (d + 1);
        float sdot = 0.f, pdot = 0.f;
        for (int c = 0; c < d; ++c) {
          sdot = fmaf(qr[c], kr[c], sdot);
          pdot = fmaf(dr[c], vr[c], pdot);
        }
        const bool ok = lane < wn && allowed(a, b, tq_r[rr], tk);
        const float p = ok ? expf(sdot * a.scale - lse_r[rr]) : 0.f;
        const float ds = p * (pdot - D_r[rr]);
        for (int jj = 0; jj < wn; ++jj) {
          const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
          for (int e = 0; e < kMaxE; ++e) {
            const int c = lane + 32 * e;
            if (c < d) acc[rr][e] = fmaf(dsj, Ks[jj * (d + 1) + c], acc[rr][e]);
          }
        }
      }
    }
  }
  T* dq = static_cast<T*>(a.dq);
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    if (!live[rr]) continue;
#pragma unroll
    for (int e = 0; e < kMaxE; ++e) {
      const int c = lane + 32 * e;
      if (c < d) st(dq, qb + tq_r[rr] * qs + c, acc[rr][e] * a.scale);
    }
  }
}

// dK, dV: CTA = 16 key rows of block j for one (b, kv head); for every query
// head of the group, query chunks of 32 in the order block j meets them.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) bwd_dkdv_kernel(BwdArgs a, int ntiles) {
  extern __shared__ float sm[];
  const int d = a.d;
  float* Ks = sm;                        // [kRows][d]
  float* Vs = Ks + kRows * d;            // [kRows][d]
  float* Qs = Vs + kRows * d;            // [kChunk][d + 1]
  float* dOs = Qs + kChunk * (d + 1);    // [kChunk][d + 1]
  const int tile = blockIdx.x % ntiles, j = blockIdx.x / ntiles;
  const int kvh = blockIdx.y, b = blockIdx.z, g = a.Hq / a.Hkv;
  const int Lb = a.S / a.P, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* dout = static_cast<const T*>(a.dout);
  const long long qs = static_cast<long long>(a.Hq) * d, ks = static_cast<long long>(a.Hkv) * d;
  const long long kb = static_cast<long long>(b) * a.S * ks + static_cast<long long>(kvh) * d;
  for (int idx = threadIdx.x; idx < kRows * d; idx += blockDim.x) {
    const int r = idx / d, c = idx % d;
    const long long u = static_cast<long long>(tile) * kRows + r;
    float kv = 0.f, vv = 0.f;
    if (u < Lb) {
      const long long off = kb + block_token(a.order, a.S, a.P, j, u) * ks + c;
      kv = ld(k, off);
      vv = ld(v, off);
    }
    Ks[idx] = kv;
    Vs[idx] = vv;
  }
  float dk[kRowsPerWarp][kMaxE], dv[kRowsPerWarp][kMaxE];
  long long tk_r[kRowsPerWarp];
  bool live[kRowsPerWarp];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const long long u = static_cast<long long>(tile) * kRows + warp * kRowsPerWarp + rr;
    live[rr] = u < Lb;
    tk_r[rr] = live[rr] ? block_token(a.order, a.S, a.P, j, u) : 0;
#pragma unroll
    for (int e = 0; e < kMaxE; ++e) dk[rr][e] = dv[rr][e] = 0.f;
  }
  for (int hh = 0; hh < g; ++hh) {
    const int h = kvh * g + hh;
    const long long qb = static_cast<long long>(b) * a.S * qs + static_cast<long long>(h) * d;
    for (int s = 0; s < a.P; ++s) {
      const int i = (j + s) % a.P;
      for (int w0 = 0; w0 < Lb; w0 += kChunk) {
        const int wn = min(kChunk, Lb - w0);
        __syncthreads();
        for (int idx = threadIdx.x; idx < kChunk * d; idx += blockDim.x) {
          const int r = idx / d, c = idx % d;
          float qv = 0.f, dv0 = 0.f;
          if (r < wn) {
            const long long off = qb + block_token(a.order, a.S, a.P, i, w0 + r) * qs + c;
            qv = ld(q, off);
            dv0 = ld(dout, off);
          }
          Qs[r * (d + 1) + c] = qv;
          dOs[r * (d + 1) + c] = dv0;
        }
        __syncthreads();
        // lane jq owns query w0 + jq of block i
        const long long tq = block_token(a.order, a.S, a.P, i, w0 + lane);
        const long long li = (static_cast<long long>(b) * a.Hq + h) * a.S + tq;
        const float lse_q = lane < wn ? a.lse[li] : 0.f;
        const float D_q = lane < wn ? a.Dsum[li] : 0.f;
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          if (!live[rr]) continue;
          const float* kr = Ks + (warp * kRowsPerWarp + rr) * d;
          const float* vr = Vs + (warp * kRowsPerWarp + rr) * d;
          const float* qr = Qs + lane * (d + 1);
          const float* dr = dOs + lane * (d + 1);
          float sdot = 0.f, pdot = 0.f;
          for (int c = 0; c < d; ++c) {
            sdot = fmaf(qr[c], kr[c], sdot);
            pdot = fmaf(dr[c], vr[c], pdot);
          }
          const bool ok = lane < wn && allowed(a, b, tq, tk_r[rr]);
          const float p = ok ? expf(sdot * a.scale - lse_q) : 0.f;
          const float ds = p * (pdot - D_q);
          for (int jj = 0; jj < wn; ++jj) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
            for (int e = 0; e < kMaxE; ++e) {
              const int c = lane + 32 * e;
              if (c < d) {
                dv[rr][e] = fmaf(pj, dOs[jj * (d + 1) + c], dv[rr][e]);
                dk[rr][e] = fmaf(dsj, Qs[jj * (d + 1) + c], dk[rr][e]);
              }
            }
          }
        }
      }
    }
  }
  T* dK = static_cast<T*>(a.dk);
  T* dV = static_cast<T*>(a.dv);
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    if (!live[rr]) continue;
#pragma unroll
    for (int e = 0; e < kMaxE; ++e) {
      const int c = lane + 32 * e;
      if (c < d) {
        st(dK, kb + tk_r[rr] * ks + c, dk[rr][e] * a.scale);
        st(dV, kb + tk_r[rr] * ks + c, dv[rr][e]);
      }
    }
  }
}

template <typename T>
int launch_all(const BwdArgs& a, cudaStream_t st) {
  const long long rows = static_cast<long long>(a.B) * a.S * a.Hq;
  bwd_dot_kernel<T><<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, st>>>(
      static_cast<const T*>(a.out), static_cast<const T*>(a.dout), a.B, a.S, a.Hq, a.d, a.Dsum);
  const int Lb = a.S / a.P, ntiles = (Lb + kRows - 1) / kRows;
  const size_t smem = sizeof(float) * (2 * static_cast<size_t>(kRows) * a.d +
                                       2 * static_cast<size_t>(kChunk) * (a.d + 1));
  if (cudaFuncSetAttribute(bwd_dq_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess ||
      cudaFuncSetAttribute(bwd_dkdv_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return -1;
  bwd_dq_kernel<T><<<dim3(ntiles * a.P, a.Hq, a.B), kWarps * 32, smem, st>>>(a, ntiles);
  bwd_dkdv_kernel<T><<<dim3(ntiles * a.P, a.Hkv, a.B), kWarps * 32, smem, st>>>(a, ntiles);
  return cudaGetLastError() == cudaSuccess ? 3 : -1;
}

}  // namespace

int launch_attn_bwd_simt(const BwdArgs& a, cudaStream_t stream) {
  return a.dtype == SP_F32 ? launch_all<float>(a, stream) : launch_all<__nv_bfloat16>(a, stream);
}

}  // namespace sp
