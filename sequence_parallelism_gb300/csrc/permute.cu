// permute.cu -- Ulysses sequence-shard <-> head-shard redistribution as a
// single-GPU layout permutation.
//
// "Ulysses SP: entrenar modelos con millones de tokens" (Keryc), "Cómo
// funciona Ulysses Sequence Parallelism (SP)": the first all-to-all leaves
// every GPU with all positions of a subset of the heads, the second one
// undoes it.  "DeepSpeed-Ulysses" (orangingq), "Method": (N/P, d) -> (N, d/P).
//
// x [B][S][H][d] is viewed as rows = B*S rows of P chunks, chunk r holding
// the C = (H/P)*d elements of head group r; y [P][B*S][C] stores chunk r of
// row n at y[r][n].  The copy is pure data movement, bound by HBM bandwidth:
// each warp moves one contiguous chunk at a time (2 KiB at the Ulysses shapes)
// with 16-byte vector loads, four in flight per lane before the stores, so
// both the read and the write side stream whole 128-byte lines.
#include <cuda_runtime.h>

#include "common.cuh"

namespace sp {
namespace {

template <typename V, bool kSeqToHead>
__global__ void __launch_bounds__(256) permute_kernel(const V* __restrict__ src,
                                                      V* __restrict__ dst, long long rows, int P,
                                                      int units_per_chunk, long long nchunks) {
  const int lane = threadIdx.x & 31;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int U = units_per_chunk;
  for (long long c = warp; c < nchunks; c += nwarps) {
    // c enumerates chunks in head-sharded order: c = r * rows + n
    const long long r = c / rows;
    const long long n = c - r * rows;
    const long long y_off = c * U;
    const long long x_off = (n * P + r) * U;
    const V* s = src + (kSeqToHead ? x_off : y_off);
    V* d = dst + (kSeqToHead ? y_off : x_off);
    for (int u0 = 0; u0 < U; u0 += 128) {
      V a[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int u = u0 + k * 32 + lane;
        if (u < U) a[k] = __ldcs(s + u);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int u = u0 + k * 32 + lane;
        if (u < U) __stcs(d + u, a[k]);
      }
    }
  }
}

template <typename V>
cudaError_t launch_permute(const void* src, void* dst, long long rows, int P, long long chunk_bytes,
                           bool seq_to_head, cudaStream_t stream) {
  const int U = static_cast<int>(chunk_bytes / sizeof(V));
  const long long nchunks = rows * P;
  // 8 CTAs x 256 threads per SM keeps 64 warps resident, each with four
  // 16-byte loads in flight.
  long long blocks = static_cast<long long>(device_sm_count()) * 8;
  const long long need = (nchunks + 7) / 8;
  if (blocks > need) blocks = need;
  if (blocks < 1) blocks = 1;
  if (seq_to_head)
    permute_kernel<V, true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const V*>(src), static_cast<V*>(dst), rows, P, U, nchunks);
  else
    permute_kernel<V, false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const V*>(src), static_cast<V*>(dst), rows, P, U, nchunks);
  return cudaGetLastError();
}

sp_status permute(const void* src, void* dst, int B, int S, int H, int d, int P, sp_dtype dtype,
                  sp_stream_t stream, bool seq_to_head) {
  g_last_launches = 0;
  if (!src || !dst) return SP_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || d < 1 || P < 1) return SP_ERR_INVALID_ARG;
  if (S % P != 0 || H % P != 0) return SP_ERR_INVALID_ARG;
  const size_t es = dtype_size(dtype);
  if (es == 0) return SP_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * S;
  const long long chunk_bytes = static_cast<long long>(H / P) * d * static_cast<long long>(es);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (chunk_bytes % 16 == 0 && aligned(src, 16) && aligned(dst, 16))
    e = launch_permute<uint4>(src, dst, rows, P, chunk_bytes, seq_to_head, st);
  else if (chunk_bytes % 4 == 0 && aligned(src, 4) && aligned(dst, 4))
    e = launch_permute<uint32_t>(src, dst, rows, P, chunk_bytes, seq_to_head, st);
  else
    e = launch_permute<uint16_t>(src, dst, rows, P, chunk_bytes, seq_to_head, st);
  if (e != cudaSuccess) return SP_ERR_CUDA;
  g_last_launches = 1;
  return SP_OK;
}

}  // namespace
}  // namespace sp

extern "C" sp_status sp_ulysses_seq_to_head(const void* x, void* y, int B, int S, int H, int d,
                                            int P, sp_dtype dtype, sp_stream_t stream) {
  return sp::permute(x, y, B, S, H, d, P, dtype, stream, true);
}

extern "C" sp_status sp_ulysses_head_to_seq(const void* y, void* x, int B, int S, int H, int d,
                                            int P, sp_dtype dtype, sp_stream_t stream) {
  return sp::permute(y, x, B, S, H, d, P, dtype, stream, false);
}
