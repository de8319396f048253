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
// row n at y[r][n].  The copy is pure data movement, bound by HBM bandwidth.
//
// Two kernels, the same result:
//  * permute_bulk_kernel: the chunks are staged through shared memory by the
//    Tensor Memory Accelerator.  Consecutive rows of one head group form an
//    item of up to 8 KiB, contiguous on the head-sharded side and one chunk
//    per row on the sequence-sharded side; each side of an item moves as ONE
//    request (a tiled tensor copy gathers or scatters the rows, an untiled
//    bulk copy covers the contiguous run), and every warp keeps the loads of
//    four items in flight in a six-stage ring.  Measured on GB300 (CUDA
//    events, L2 flushed): the same asymptotic rate as the vector kernel
//    (~7.1 TB/s of read + write, part of the writes still in L2 at the end)
//    and 1.5-3% more with 1 KiB chunks at 256 MiB .. 1 GiB, but about 1 us
//    more fixed cost per launch (a TMA request's latency is longer than a
//    load's and only a long launch hides it).  Used when the launch moves at
//    least 128 MiB (sp_permute_set_bulk_min_bytes changes that) and the bulk rules hold (chunks of 256 B .. 8 KiB,
//    a multiple of 16 B; 16-byte aligned pointers).
//  * permute_kernel (every other launch): each warp moves one contiguous
//    chunk at a time with 16-, 8-, 4- or 2-byte vector loads, four in flight
//    per lane before the stores.
// q, k and v of a layer can go through one launch (sp_ulysses_seq_to_head_qkv),
// which spares two launch ramps on tensors that take ~10 us each.
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace sp {
namespace {

using namespace ptx;

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

// ---------------------------------------------------------- TMA-staged copy
// An item is g = kItemBytes / cb consecutive rows n0 .. n0+g-1 of one head
// group r: contiguous in y (bytes (r*rows + n0)*cb onwards) and one chunk per
// row in x.  The x side moves as ONE tiled tensor copy: x viewed as the 4-D
// tensor (W bytes, cb/W, P, rows) with the box (W, cb/W, 1, g) gathers the g
// chunks into consecutive shared memory (rows past the end read as zeros on a
// load and are not written on a store); the y side moves as ONE untiled bulk
// copy.  Two requests per item: the TMA unit is bound by its request count,
// so items are as large as the ring allows.  Every warp's lane 0 is an
// independent pipeline with its own ring of kRounds stages: in round j it
// loads its item j and stores its item j - kLag.
constexpr int kItemBytes = 8192;  // one stage
constexpr int kRounds = 6;        // stages per pipeline
constexpr int kLag = 4;           // items whose loads are in flight
constexpr int kBulkWarps = 4;     // pipelines per CTA, one CTA per SM
constexpr int kMinBulkChunk = 256;
constexpr long long kBulkMinBytesDefault = 128ll << 20;
// launches reading fewer bytes take the vector kernel (process-wide setting)
std::atomic<long long> g_bulk_min_bytes{kBulkMinBytesDefault};
constexpr size_t kBulkSmem = static_cast<size_t>(kBulkWarps) * kRounds * kItemBytes + 1024;

// Set by a bulk-permutation pipeline whose bounded wait gave up (0 = none).
__device__ int g_permute_error;

struct BulkMaps {
  CUtensorMap x[3];  // sequence-sharded side of each tensor
};

struct BulkSet {
  const unsigned char* y[3];  // head-sharded side (source or destination)
  unsigned rows[3];           // B * S
  unsigned cb[3];             // chunk bytes
  unsigned g[3];              // rows per item
  unsigned items_per_group[3];
  long long first_item[4];    // first global item of each tensor, first_item[n] = total
  int n;
};

template <bool kSeqToHead>
__global__ void __launch_bounds__(32 * kBulkWarps, 1)
    permute_bulk_kernel(const __grid_constant__ BulkMaps maps, BulkSet set) {
  extern __shared__ __align__(1024) unsigned char ring_raw[];
  __shared__ __align__(8) uint64_t bars[kBulkWarps * kRounds];
  __shared__ int abort_flag[kBulkWarps];
  if ((threadIdx.x & 31) != 0) return;  // lane 0 of every warp runs a pipeline
  const int warp = threadIdx.x >> 5;
  uint64_t* wbars = bars + warp * kRounds;
  for (int s = 0; s < kRounds; ++s) mbar_init(smem_u32(&wbars[s]), 1);
  abort_flag[warp] = 0;
  fence_mbar_init();
  if (warp == 0) {
    for (int t = 0; t < set.n; ++t) prefetch_tmap(&maps.x[t]);
  }

  const long long total = set.first_item[set.n];
  const long long pipes = static_cast<long long>(gridDim.x) * kBulkWarps;
  const long long pipe = static_cast<long long>(blockIdx.x) * kBulkWarps + warp;
  const long long mine = total > pipe ? (total - pipe + pipes - 1) / pipes : 0;
  const uint32_t base = (smem_u32(ring_raw) + 1023u) & ~1023u;
  const uint32_t stages0 = base + static_cast<uint32_t>(warp * kRounds * kItemBytes);

  // per-tensor fields read with constant indices (selects, no local copy)
  auto pick = [](int t, auto a0, auto a1, auto a2) { return t == 0 ? a0 : (t == 1 ? a1 : a2); };
  // item i: tensor t, head group r, first row n0, rows cnt, chunk bytes cb,
  // rows per item g, y byte offset
  struct Item {
    int t;
    unsigned r, n0, cnt, cb, g;
    unsigned long long y_off;
  };
  auto locate = [&](long long i) {
    Item it;
    it.t = (set.n > 2 && i >= set.first_item[2]) ? 2 : ((set.n > 1 && i >= set.first_item[1]) ? 1 : 0);
    const int t = it.t;
    const unsigned rows = pick(t, set.rows[0], set.rows[1], set.rows[2]);
    const unsigned ipg = pick(t, set.items_per_group[0], set.items_per_group[1],
                              set.items_per_group[2]);
    it.g = pick(t, set.g[0], set.g[1], set.g[2]);
    it.cb = pick(t, set.cb[0], set.cb[1], set.cb[2]);
    const unsigned li =
        static_cast<unsigned>(i - pick(t, set.first_item[0], set.first_item[1], set.first_item[2]));
    it.r = li / ipg;
    it.n0 = (li - it.r * ipg) * it.g;
    const unsigned left = rows - it.n0;
    it.cnt = left < it.g ? left : it.g;
    it.y_off = (static_cast<unsigned long long>(it.r) * rows + it.n0) * it.cb;
    return it;
  };
  auto ybase = [&](int t) { return pick(t, set.y[0], set.y[1], set.y[2]); };
  auto xmap = [&](int t) { return pick(t, &maps.x[0], &maps.x[1], &maps.x[2]); };

  long long loaded = 0;   // items whose loads were issued
  long long failed = -1;  // item whose wait gave up
#pragma unroll 1
  for (long long j = 0; j < mine + kLag; ++j) {
    if (j < mine) {
      // stage j % kRounds last held item j - kRounds, whose store was issued
      // kRounds - kLag rounds ago: all but the newest kRounds - kLag - 1
      // stores must have read their stages
      if (j >= kRounds) bulk_wait_group_read<kRounds - kLag - 1>();
      const int st = static_cast<int>(j % kRounds);
      const uint32_t bar = smem_u32(&wbars[st]);
      const uint32_t stage = stages0 + st * kItemBytes;
      const Item it = locate(pipe + j * pipes);
      if (kSeqToHead) {  // box of g rows (rows past the end zero-filled, counted)
        mbar_arrive_expect_tx(bar, it.g * it.cb);
        tma_load_4d(stage, xmap(it.t), bar, 0, 0, static_cast<int>(it.r),
                    static_cast<int>(it.n0));
      } else {
        mbar_arrive_expect_tx(bar, it.cnt * it.cb);
        bulk_load(stage, ybase(it.t) + it.y_off, it.cnt * it.cb, bar);
      }
      loaded = j + 1;
    }
    if (j >= kLag) {
      const long long jj = j - kLag;
      const int st = static_cast<int>(jj % kRounds);
      if (!mbar_wait(smem_u32(&wbars[st]), static_cast<uint32_t>((jj / kRounds) & 1),
                     &abort_flag[warp], &g_permute_error, 1)) {
        failed = jj;
        break;
      }
      fence_proxy_async_smem();  // order the landed bytes before the store reads them
      const uint32_t stage = stages0 + st * kItemBytes;
      const Item it = locate(pipe + jj * pipes);
      if (kSeqToHead) {
        bulk_store(const_cast<unsigned char*>(ybase(it.t)) + it.y_off, stage, it.cnt * it.cb);
      } else {  // box of g rows; rows past the end are not written
        tma_store_4d(xmap(it.t), stage, 0, 0, static_cast<int>(it.r), static_cast<int>(it.n0));
      }
      bulk_commit_group();
    }
  }
  if (failed >= 0) {
    // wait (bounded) for the loads still in flight before shared memory goes
    for (long long jj = failed; jj < loaded; ++jj) {
      abort_flag[warp] = 0;
      mbar_wait(smem_u32(&wbars[jj % kRounds]), static_cast<uint32_t>((jj / kRounds) & 1),
                &abort_flag[warp], nullptr, 0);
    }
  }
  bulk_wait_group0();
}

// Largest divisor of cb that is a multiple of 16 and at most 1024 bytes (the
// box's inner extent: 256 four-byte elements).
unsigned inner_width(unsigned cb) {
  for (unsigned w = 1024; w >= 16; w -= 16)
    if (cb % w == 0) return w;
  return 0;
}

// Bulk-copy geometry and tensor maps for n tensors; false when the launch
// reads fewer bytes than the set minimum or the bulk rules do not hold (then the vector
// kernel runs).
bool make_bulk_set(BulkSet& set, BulkMaps& maps, int n, const void* const* x,
                   const void* const* y, int B, int S, const int* H, int d, int P, size_t es) {
  long long bytes = 0;
  for (int t = 0; t < n; ++t)
    bytes += static_cast<long long>(B) * S * H[t] * d * static_cast<long long>(es);
  if (bytes < g_bulk_min_bytes.load(std::memory_order_relaxed)) return false;
  tmap::EncodeTiledFn enc = tmap::encode_fn();
  if (!enc) return false;
  set.n = n;
  set.first_item[0] = 0;
  for (int t = 0; t < n; ++t) {
    const long long cb = static_cast<long long>(H[t] / P) * d * static_cast<long long>(es);
    const long long rows = static_cast<long long>(B) * S;
    if (cb < kMinBulkChunk || cb > kItemBytes || cb % 16 != 0 || rows * P >= (1ll << 31) ||
        !aligned(x[t], 16) || !aligned(y[t], 16))
      return false;
    const unsigned w = inner_width(static_cast<unsigned>(cb));
    if (w == 0) return false;
    const unsigned g = static_cast<unsigned>(kItemBytes / cb);
    set.y[t] = static_cast<const unsigned char*>(y[t]);
    set.rows[t] = static_cast<unsigned>(rows);
    set.cb[t] = static_cast<unsigned>(cb);
    set.g[t] = g;
    set.items_per_group[t] = static_cast<unsigned>((rows + g - 1) / g);
    set.first_item[t + 1] = set.first_item[t] + static_cast<long long>(P) * set.items_per_group[t];
    // x as (w/4 four-byte elements, cb/w, P, rows); box (w/4, cb/w, 1, g)
    cuuint64_t dims[4] = {w / 4, static_cast<cuuint64_t>(cb / w), static_cast<cuuint64_t>(P),
                          static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[3] = {w, static_cast<cuuint64_t>(cb), static_cast<cuuint64_t>(cb) * P};
    cuuint32_t box[4] = {w / 4, static_cast<cuuint32_t>(cb / w), 1, g};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (enc(&maps.x[t], CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void*>(x[t]), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  for (int t = n; t < 3; ++t) {
    set.y[t] = nullptr;
    set.rows[t] = 1;
    set.cb[t] = 16;
    set.g[t] = 1;
    set.items_per_group[t] = 1;
    set.first_item[t + 1] = set.first_item[t];
    maps.x[t] = maps.x[0];
  }
  return true;
}

cudaError_t launch_bulk(const BulkMaps& maps, const BulkSet& set, bool seq_to_head,
                        cudaStream_t stream) {
  static thread_local int configured = -1;  // device whose attributes are set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured != dev) {
    e = cudaFuncSetAttribute(permute_bulk_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kBulkSmem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(permute_bulk_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kBulkSmem));
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  const long long total = set.first_item[set.n];
  long long grid = device_sm_count();
  const long long need = (total + kBulkWarps - 1) / kBulkWarps;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  if (seq_to_head)
    permute_bulk_kernel<true><<<static_cast<unsigned>(grid), 32 * kBulkWarps, kBulkSmem, stream>>>(
        maps, set);
  else
    permute_bulk_kernel<false><<<static_cast<unsigned>(grid), 32 * kBulkWarps, kBulkSmem,
                                 stream>>>(maps, set);
  return cudaGetLastError();
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
  BulkSet bset;
  BulkMaps bmaps;
  // x is the source of seq->head and the destination of head->seq
  const void* xs[3] = {nullptr, nullptr, nullptr};
  const void* ys[3] = {nullptr, nullptr, nullptr};
  for (int t = 0; t < n; ++t) {
    xs[t] = seq_to_head ? src[t] : dst[t];
    ys[t] = seq_to_head ? dst[t] : src[t];
  }
  if (make_bulk_set(bset, bmaps, n, xs, ys, B, S, H, d, P, dtype_size(dtype)))
    e = launch_bulk(bmaps, bset, seq_to_head, st);
  else if (unit == 16)
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

extern "C" sp_status sp_get_permute_error(int* code) {
  if (!code) return SP_ERR_INVALID_ARG;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, sp::g_permute_error, sizeof(int)) != cudaSuccess) return SP_ERR_CUDA;
  *code = v;
  if (v == 0) return SP_OK;
  const int zero = 0;
  if (cudaMemcpyToSymbol(sp::g_permute_error, &zero, sizeof(int)) != cudaSuccess)
    return SP_ERR_CUDA;
  return SP_ERR_DEVICE_TIMEOUT;
}

extern "C" size_t sp_permute_set_bulk_min_bytes(size_t min_bytes) {
  const long long v = min_bytes > static_cast<size_t>(1ll << 62) ? (1ll << 62)
                                                                 : static_cast<long long>(min_bytes);
  return static_cast<size_t>(sp::g_bulk_min_bytes.exchange(v));
}
