// segments.cu -- document starts from position_ids, the O(n) carrier of the
// causal mask ("Ulysses SPで100万トークン学習", section 3: position_ids
// instead of a 4D mask that would reach ~1 TB at 128k tokens).
//
// A document starts at token 0 and at every t where position_ids does not
// continue by +1.  doc_start[t] = the last start at or before t, i.e. an
// inclusive max-scan of (t if t starts a document else 0).  Two launches:
//   1. per 1024-token chunk, the largest start index in it;
//   2. per chunk, the carry (max over earlier chunks) combined with a
//      block-wide max-scan of the chunk.
// Query t may then attend key j iff doc_start[t] <= j <= t.
#include <cuda_runtime.h>

#include "common.cuh"

namespace sp {
namespace {

constexpr int kChunk = 1024;

__device__ __forceinline__ int start_value(const int32_t* pos, int S, int t) {
  if (t >= S) return 0;
  if (t == 0) return 0;
  return (pos[t] != pos[t - 1] + 1) ? t : 0;
}

__global__ void __launch_bounds__(kChunk) chunk_max_kernel(const int32_t* __restrict__ pos_all,
                                                           int S, int nchunks,
                                                           int32_t* __restrict__ chunk_max) {
  const int b = blockIdx.y;
  const int c = blockIdx.x;
  const int32_t* pos = pos_all + static_cast<long long>(b) * S;
  int v = start_value(pos, S, c * kChunk + threadIdx.x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  __shared__ int warp_max[kChunk / 32];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    v = warp_max[threadIdx.x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) chunk_max[static_cast<long long>(b) * nchunks + c] = v;
  }
}

__global__ void __launch_bounds__(kChunk) doc_start_kernel(const int32_t* __restrict__ pos_all,
                                                           int S, int nchunks,
                                                           const int32_t* __restrict__ chunk_max,
                                                           int32_t* __restrict__ doc_start_all) {
  const int b = blockIdx.y;
  const int c = blockIdx.x;
  const int32_t* pos = pos_all + static_cast<long long>(b) * S;
  __shared__ int warp_scan[kChunk / 32];
  __shared__ int carry_s;
  // carry: largest start strictly before this chunk
  int carry = 0;
  for (int i = threadIdx.x; i < c; i += kChunk)
    carry = max(carry, chunk_max[static_cast<long long>(b) * nchunks + i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) carry = max(carry, __shfl_xor_sync(0xffffffffu, carry, o));
  if ((threadIdx.x & 31) == 0) warp_scan[threadIdx.x >> 5] = carry;
  __syncthreads();
  if (threadIdx.x < 32) {
    int v = warp_scan[threadIdx.x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) carry_s = v;
  }
  __syncthreads();
  carry = carry_s;
  // inclusive max-scan of the chunk
  const int t = c * kChunk + threadIdx.x;
  const int lane = threadIdx.x & 31;
  int v = start_value(pos, S, t);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = max(v, n);
  }
  __syncthreads();  // warp_scan reuse
  if (lane == 31) warp_scan[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    int w = warp_scan[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w = max(w, n);
    }
    warp_scan[lane] = w;
  }
  __syncthreads();
  const int wid = threadIdx.x >> 5;
  if (wid > 0) v = max(v, warp_scan[wid - 1]);
  v = max(v, carry);
  if (t < S) doc_start_all[static_cast<long long>(b) * S + t] = v;
}

}  // namespace

size_t segment_scratch_bytes(int B, int S) {
  const size_t nchunks = (static_cast<size_t>(S) + kChunk - 1) / kChunk;
  return round_up(static_cast<size_t>(B) * nchunks * sizeof(int32_t), 256);
}

int launch_segment_starts(const int32_t* position_ids, int32_t* doc_start, int B, int S,
                          void* scratch, cudaStream_t stream) {
  const int nchunks = (S + kChunk - 1) / kChunk;
  int32_t* cmax = static_cast<int32_t*>(scratch);
  dim3 grid(nchunks, B);
  chunk_max_kernel<<<grid, kChunk, 0, stream>>>(position_ids, S, nchunks, cmax);
  doc_start_kernel<<<grid, kChunk, 0, stream>>>(position_ids, S, nchunks, cmax, doc_start);
  return cudaGetLastError() == cudaSuccess ? 2 : -1;
}

}  // namespace sp

extern "C" size_t sp_segment_starts_workspace_bytes(int B, int S) {
  if (B < 1 || S < 1) return 0;
  return sp::segment_scratch_bytes(B, S);
}

extern "C" sp_status sp_segment_starts(const int32_t* position_ids, int32_t* doc_start, int B,
                                       int S, void* workspace, size_t workspace_bytes,
                                       sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_segment_starts");
  sp::g_last_launches = 0;
  if (!position_ids || !doc_start || B < 1 || S < 1) return SP_ERR_INVALID_ARG;
  if (B > 65535) return SP_ERR_UNSUPPORTED;
  if (!workspace || !sp::aligned(workspace, 256) ||
      workspace_bytes < sp::segment_scratch_bytes(B, S))
    return SP_ERR_WORKSPACE;
  const int n = sp::launch_segment_starts(position_ids, doc_start, B, S, workspace,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (n < 0) return SP_ERR_CUDA;
  sp::g_last_launches = n;
  return SP_OK;
}
