// attn_f32.cu -- blockwise ring attention in float32 on the CUDA cores.
//
// The float32 path exists for exactness checks at float32 tolerance (bf16
// tensor cores cannot meet 1e-5).  It follows the same schedule as the
// tensor-core kernel: a CTA keeps 16 query rows of block i resident and walks
// the key/value blocks in ring order j = (i - s) mod P ("Ring Attention",
// "Cómo funciona la atención en anillo"), 32 keys at a time, merging them
// into running (max, sum, weighted-value sum) per row and dividing at the end.
//
// Layout of the work: 4 warps x 4 rows.  For a 32-key chunk lane j scores
// key j against the row (q row broadcast from shared memory, key row j read
// from a padded shared tile), the warp reduces max and sum with shuffles, and
// every lane then accumulates its d/32 output columns over the 32 keys.
#include <cuda_runtime.h>
#include <math.h>

#include "attn_common.cuh"

namespace sp {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRows = kWarps * kRowsPerWarp;  // query rows per CTA
constexpr int kKeys = 32;                     // keys per chunk
constexpr int kMaxD = 256;
constexpr int kMaxE = kMaxD / 32;             // output columns per lane

__global__ void __launch_bounds__(kWarps * 32) attn_f32_kernel(AttnArgs a, int ntiles) {
  extern __shared__ float smem[];
  const int d = a.d;
  float* Qs = smem;                      // [kRows][d]
  float* Ks = Qs + kRows * d;            // [kKeys][d + 1]
  float* Vs = Ks + kKeys * (d + 1);      // [kKeys][d]
  __shared__ long long hull_lo_s, hull_hi_s;

  const int tile = blockIdx.x % ntiles;
  const int i = a.q_block >= 0 ? a.q_block : static_cast<int>(blockIdx.x / ntiles);
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int kvh = h / (a.Hq / a.Hkv);
  const int Lb = a.S / a.P;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const float* q = static_cast<const float*>(a.q);
  const float* k = static_cast<const float*>(a.k);
  const float* v = static_cast<const float*>(a.v);
  const long long qrow_stride = static_cast<long long>(a.Hq) * d;
  const long long krow_stride = static_cast<long long>(a.Hkv) * d;
  // rows per batch and the row of (block, local row) in q/out and in k/v:
  // the token, or the local row when the tensor holds a single block
  const bool qb = a.q_block >= 0, kvb = a.kv_block >= 0;
  const long long q_rows = qb ? Lb : a.S, kv_rows = kvb ? Lb : a.S;
  auto q_row = [&](long long u) { return qb ? u : block_token(a.order, a.S, a.P, i, u); };
  auto kv_row = [&](int jb, long long w) { return kvb ? w : block_token(a.order, a.S, a.P, jb, w); };
  const long long qbase = static_cast<long long>(b) * q_rows * qrow_stride + static_cast<long long>(h) * d;
  const long long kbase = static_cast<long long>(b) * kv_rows * krow_stride + static_cast<long long>(kvh) * d;

  // resident query rows
  for (int idx = threadIdx.x; idx < kRows * d; idx += blockDim.x) {
    const int r = idx / d, c = idx % d;
    const long long u = static_cast<long long>(tile) * kRows + r;
    float val = 0.f;
    if (u < Lb) val = q[qbase + q_row(u) * qrow_stride + c];
    Qs[idx] = val;
  }
  // allowed key-token interval [lo, hi] of each of my rows
  long long lo[kRowsPerWarp], hi[kRowsPerWarp];
  bool live[kRowsPerWarp];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const long long u = static_cast<long long>(tile) * kRows + warp * kRowsPerWarp + rr;
    live[rr] = u < Lb;
    const long long t = live[rr] ? block_token(a.order, a.S, a.P, i, u) : 0;
    if (a.doc_start) {
      lo[rr] = live[rr] ? a.doc_start[static_cast<long long>(b % a.pos_rows) * a.S + t] : 0;
      hi[rr] = t;
    } else {
      lo[rr] = 0;
      hi[rr] = a.S - 1;
    }
  }
  if (threadIdx.x == 0) {  // hull of every row's interval, to skip empty chunks
    long long hl = a.S, hh = -1;
    for (int r = 0; r < kRows; ++r) {
      const long long u = static_cast<long long>(tile) * kRows + r;
      if (u >= Lb) break;
      const long long t = block_token(a.order, a.S, a.P, i, u);
      const long long l0 = a.doc_start ? a.doc_start[static_cast<long long>(b % a.pos_rows) * a.S + t] : 0;
      const long long h0 = a.doc_start ? t : a.S - 1;
      hl = l0 < hl ? l0 : hl;
      hh = h0 > hh ? h0 : hh;
    }
    hull_lo_s = hl;
    hull_hi_s = hh;
  }
  __syncthreads();
  const long long hull_lo = hull_lo_s, hull_hi = hull_hi_s;

  float m[kRowsPerWarp], l[kRowsPerWarp], o[kRowsPerWarp][kMaxE];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int e = 0; e < kMaxE; ++e) o[rr][e] = 0.f;
  }

  for (int s = a.step_begin; s < a.step_end; ++s) {
    const int j = ((i - s) % a.P + a.P) % a.P;
    for (int w0 = 0; w0 < Lb; w0 += kKeys) {
      const int wn = min(kKeys, Lb - w0);
      const long long t_first = block_token(a.order, a.S, a.P, j, w0);
      const long long t_last = block_token(a.order, a.S, a.P, j, w0 + wn - 1);
      if (t_last < hull_lo || t_first > hull_hi) continue;  // CTA-uniform skip
      __syncthreads();
      for (int idx = threadIdx.x; idx < kKeys * d; idx += blockDim.x) {
        const int r = idx / d, c = idx % d;
        float kv = 0.f, vv = 0.f;
        if (r < wn) {
          const long long off = kbase + kv_row(j, w0 + r) * krow_stride + c;
          kv = k[off];
          vv = v[off];
        }
        Ks[r * (d + 1) + c] = kv;
        Vs[r * d + c] = vv;
      }
      __syncthreads();
      const long long tk = block_token(a.order, a.S, a.P, j, w0 + lane);
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        if (!live[rr]) continue;
        const bool ok = lane < wn && tk >= lo[rr] && tk <= hi[rr];
        const float* qr = Qs + (warp * kRowsPerWarp + rr) * d;
        const float* kr = Ks + lane * (d + 1);
        float dot = 0.f;
        for (int c = 0; c < d; ++c) dot = fmaf(qr[c], kr[c], dot);
        const float sc = ok ? dot * a.scale : -INFINITY;
        float mx = sc;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m[rr], mx);
        if (m_new == -INFINITY) continue;  // nothing allowed yet for this row
        const float alpha = (m[rr] == -INFINITY) ? 0.f : expf(m[rr] - m_new);
        const float p = ok ? expf(sc - m_new) : 0.f;
        float ps = p;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l[rr] = l[rr] * alpha + ps;
#pragma unroll
        for (int e = 0; e < kMaxE; ++e) o[rr][e] *= alpha;
        for (int jj = 0; jj < wn; ++jj) {
          const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
          for (int e = 0; e < kMaxE; ++e) {
            const int c = lane + 32 * e;
            if (c < d) o[rr][e] = fmaf(pj, Vs[jj * d + c], o[rr][e]);
          }
        }
        m[rr] = m_new;
      }
    }
  }

  float* out = static_cast<float*>(a.out);
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    if (!live[rr]) continue;
    const long long u = static_cast<long long>(tile) * kRows + warp * kRowsPerWarp + rr;
    const long long t = q_row(u);
    const bool any = l[rr] > 0.f;
    const float inv = any ? 1.f / l[rr] : 0.f;
    float* orow = out + static_cast<long long>(b) * q_rows * qrow_stride + t * qrow_stride +
                  static_cast<long long>(h) * d;
#pragma unroll
    for (int e = 0; e < kMaxE; ++e) {
      const int c = lane + 32 * e;
      if (c < d) orow[c] = o[rr][e] * inv;
    }
    if (a.lse && lane == 0)
      a.lse[(static_cast<long long>(b) * a.Hq + h) * q_rows + t] = any ? m[rr] + logf(l[rr]) : -INFINITY;
  }
}

}  // namespace

int launch_attn_f32(const AttnArgs& a, cudaStream_t stream) {
  const int Lb = a.S / a.P;
  const int ntiles = (Lb + kRows - 1) / kRows;
  const size_t smem = sizeof(float) * (static_cast<size_t>(kRows) * a.d +
                                       static_cast<size_t>(kKeys) * (a.d + 1) +
                                       static_cast<size_t>(kKeys) * a.d);
  if (cudaFuncSetAttribute(attn_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return -1;
  dim3 grid(static_cast<unsigned>(ntiles) * (a.q_block >= 0 ? 1 : a.P), a.Hq, a.B);
  attn_f32_kernel<<<grid, kWarps * 32, smem, stream>>>(a, ntiles);
  return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace sp
