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
// both the read and the write side stream whole 128-byte lines.  q, k and v
// of a layer can go through one launch (sp_ulysses_seq_to_head_qkv), which
// spares two launch ramps on tensors that take ~10 us each.
#include <cuda_runtime.h>

#include "common.cuh"

namespace sp {
namespace {

// Up to three tensors permuted by one launch (q, k, v of an attention layer);
// their chunks form one concatenated index space.
struct PermSet {
  const void* src[3];
  void* dst[3];
  long long rows[3];       // B * S
  long long first[4];      // first global chunk of each tensor, first[n] = total
  int units[3];            // vector units per chunk
  int n;
  int P;
};

template <typename V, bool kSeqToHead>
__global__ void __launch_bounds__(256) permute_kernel(PermSet set) {
  const int lane = threadIdx.x & 31;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  // The tensor loop is unrolled so that the set's fields are read with
  // constant indices (no local-memory copy); warps keep one global stride
  // over the concatenated chunks, so the work stays balanced across tensors.
#pragma unroll
  for (int t = 0; t < 3; ++t) {
    if (t >= set.n) break;
    const V* src = static_cast<const V*>(set.src[t]);
    V* dst = static_cast<V*>(set.dst[t]);
    const long long rows = set.rows[t];
    const long long lo = set.first[t], hi = set.first[t + 1];
    const int U = set.units[t];
    long long off = (warp - lo) % nwarps;
    if (off < 0) off += nwarps;
    for (long long g = lo + off; g < hi; g += nwarps) {
      // c enumerates chunks in head-sharded order: c = r * rows + n
      const long long c = g - lo;
      const long long r = c / rows;
      const long long n = c - r * rows;
      const long long y_off = c * U;
      const long long x_off = (n * set.P + r) * U;
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
}

template <typename V>
cudaError_t launch_permute(PermSet set, bool seq_to_head, cudaStream_t stream) {
  const long long total = set.first[set.n];
  // Up to 8 CTAs x 8 warps per SM, each warp with four 16-byte loads in
  // flight per lane; the warp count is chosen so that every warp copies the
  // same number of chunks (no partly idle last pass).
  const long long max_warps = static_cast<long long>(device_sm_count()) * 8 * 8;
  const long long passes = (total + max_warps - 1) / max_warps;
  const long long warps = (total + passes - 1) / passes;
  long long blocks = (warps + 7) / 8;
  if (blocks < 1) blocks = 1;
  if (seq_to_head)
    permute_kernel<V, true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(set);
  else
    permute_kernel<V, false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(set);
  return cudaGetLastError();
}

// Fills `set` for n tensors with heads H[t]; returns false on a bad argument.
bool make_set(PermSet& set, int n, const void* const* src, void* const* dst, int B, int S,
              const int* H, int d, int P, sp_dtype dtype, size_t* unit) {
  if (B < 1 || S < 1 || d < 1 || P < 1 || S % P != 0) return false;
  const size_t es = dtype_size(dtype);
  if (es == 0) return false;
  // widest vector every tensor of the set allows
  size_t v = 16;
  for (int t = 0; t < n; ++t) {
    if (!src[t] || !dst[t] || H[t] < 1 || H[t] % P != 0) return false;
    const long long cb = static_cast<long long>(H[t] / P) * d * static_cast<long long>(es);
    while (v > es && (cb % v != 0 || !aligned(src[t], v) || !aligned(dst[t], v))) v /= 2;
  }
  if (v < es) v = es;
  set.n = n;
  set.P = P;
  set.first[0] = 0;
  for (int t = 0; t < n; ++t) {
    const long long cb = static_cast<long long>(H[t] / P) * d * static_cast<long long>(es);
    set.src[t] = src[t];
    set.dst[t] = dst[t];
    set.rows[t] = static_cast<long long>(B) * S;
    set.units[t] = static_cast<int>(cb / static_cast<long long>(v));
    set.first[t + 1] = set.first[t] + set.rows[t] * P;
  }
  for (int t = n; t < 3; ++t) {
    set.src[t] = nullptr;
    set.dst[t] = nullptr;
    set.rows[t] = 1;
    set.units[t] = 1;
    set.first[t + 1] = set.first[t];
  }
  *unit = v;
  return true;
}

sp_status permute_n(int n, const void* const* src, void* const* dst, int B, int S, const int* H,
                    int d, int P, sp_dtype dtype, sp_stream_t stream, bool seq_to_head) {
  g_last_launches = 0;
  PermSet set;
  size_t unit = 0;
  if (!make_set(set, n, src, dst, B, S, H, d, P, dtype, &unit)) return SP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (unit == 16)
    e = launch_permute<uint4>(set, seq_to_head, st);
  else if (unit == 8)
    e = launch_permute<uint2>(set, seq_to_head, st);
  else if (unit == 4)
    e = launch_permute<uint32_t>(set, seq_to_head, st);
  else
    e = launch_permute<uint16_t>(set, seq_to_head, st);
  if (e != cudaSuccess) return SP_ERR_CUDA;
  g_last_launches = 1;
  return SP_OK;
}

sp_status permute(const void* src, void* dst, int B, int S, int H, int d, int P, sp_dtype dtype,
                  sp_stream_t stream, bool seq_to_head) {
  const void* s[1] = {src};
  void* t[1] = {dst};
  return permute_n(1, s, t, B, S, &H, d, P, dtype, stream, seq_to_head);
}

}  // namespace
}  // namespace sp

extern "C" sp_status sp_ulysses_seq_to_head(const void* x, void* y, int B, int S, int H, int d,
                                            int P, sp_dtype dtype, sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_ulysses_seq_to_head");
  return sp::permute(x, y, B, S, H, d, P, dtype, stream, true);
}

extern "C" sp_status sp_ulysses_head_to_seq(const void* y, void* x, int B, int S, int H, int d,
                                            int P, sp_dtype dtype, sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_ulysses_head_to_seq");
  return sp::permute(y, x, B, S, H, d, P, dtype, stream, false);
}

extern "C" sp_status sp_ulysses_seq_to_head_qkv(const void* q, const void* k, const void* v,
                                                void* yq, void* yk, void* yv, int B, int S, int Hq,
                                                int Hkv, int d, int P, sp_dtype dtype,
                                                sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_ulysses_seq_to_head_qkv");
  const void* src[3] = {q, k, v};
  void* dst[3] = {yq, yk, yv};
  const int H[3] = {Hq, Hkv, Hkv};
  return sp::permute_n(3, src, dst, B, S, H, d, P, dtype, stream, true);
}
