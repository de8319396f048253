// attn_bwd_bf16.cu -- backward of blockwise ring attention on the sm_103a
// tensor cores (bf16 operands, fp32 accumulation in TMEM, d = 128).
//
// The gradients are the derivatives of the forward (the pages train with
// sequence parallelism -- "Ulysses SP: entrenar modelos con millones de
// tokens" -- but print no backward):
//   P = exp(scale * Q K^T - lse), dP = dO V^T, dS = P * (dP - D),
//   dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO,
// D_t = sum_c dO[t, c] O[t, c].
//
// Two forms, sharing the prep kernel:
//  * prep: D per query row, and lse * log2(e), D and the document starts
//    rewritten in block order (each block padded to a multiple of 128 rows),
//    so that the key-stationary kernels fetch a query tile's per-column data
//    with three contiguous bulk copies.
//  * fused (default): key-stationary.  One CTA keeps a 128-key K tile and V
//    tile and walks, for every query head of the GQA group, the query
//    blocks in the order its key block meets them on the ring,
//    i = (j + s) mod P, in tiles of 128 queries; per tile S^T and dP^T are
//    multiplied once and give dV, dK and the tile's piece of dQ, which the
//    TMA adds into a float32 accumulator (bulk reductions); a last kernel
//    scales and rounds dq.  Per-device mode: one query block against one
//    key/value block from block tensors, one CTA per key tile and query
//    head, dK/dV added into float32 accumulators by reductions (the
//    backward of one ring step on one device).
//  * two kernels, no atomics (bit-reproducible): dQ query-stationary -- one
//    CTA keeps a 128-row Q tile and its dO tile and walks the key/value
//    blocks in ring order j = (i - s) mod P ("Ring Attention", "Cómo
//    funciona la atención en anillo"), S = Q K^T and dP = dO V^T (SS MMAs),
//    two elementwise warpgroups form dS into TMEM, dQ += dS K -- and dK/dV
//    key-stationary, like the fused kernel without dQ.
// Warp roles: elementwise warps (one thread per TMEM lane = tile row), a TMA
// producer warp, an MMA warp (TMEM owner) and, in the fused kernel, a warp
// that issues the dQ bulk reductions.  Every barrier wait is bounded.
#include <climits>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "attn_common.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace sp {
namespace {

using namespace ptx;

constexpr int kD = 128;
constexpr int kT = 128;                      // rows per resident tile
constexpr int kKSlots = 3;                   // dQ: streamed K tiles (held until dQ += dS K)
constexpr int kVSlots = 2;                   // dQ: streamed V tiles (held until dP = dO V^T)
constexpr int kTileBytes = kT * kD * 2;      // 32 KiB
constexpr int kHalfBytes = kTileBytes / 2;   // one 64-column half
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t kIdescKmaj = idesc_bf16_f32(kT, kT, false);  // both operands K-major
constexpr uint32_t kIdescBmn = idesc_bf16_f32(kT, kD, true);    // B MN-major

enum : int {
  kErrBwdQFull = 0x201, kErrBwdKvEmpty = 0x202, kErrBwdKvFull = 0x203, kErrBwdSFull = 0x204,
  kErrBwdSFree = 0x205, kErrBwdDsFull = 0x206, kErrBwdOut = 0x207, kErrBwdDrain = 0x208
};

struct BwdMaps {
  CUtensorMap q, k, v, dout;
};

__host__ __device__ __forceinline__ int floor_div_i(int a, int b) {
  return a >= 0 ? a / b : -((-a + b - 1) / b);
}

// Tiles [kt0, kt1] of `rows` local rows of block j that hold a token of the
// interval [lo, hi] (kt1 < kt0: none); local row w of block j holds token
// block_token(order, S, P, j, w).
__device__ __forceinline__ void block_tiles(int order, int S, int P, int j, int lo, int hi,
                                            int rows, int& kt0, int& kt1) {
  const int Lb = S / P;
  int w_lo, w_hi;
  if (order == SP_ORDER_STRIPED) {
    w_lo = -floor_div_i(-(lo - j), P);
    w_hi = floor_div_i(hi - j, P);
  } else {
    w_lo = lo - j * Lb;
    w_hi = hi - j * Lb;
  }
  if (w_lo < 0) w_lo = 0;
  if (w_hi > Lb - 1) w_hi = Lb - 1;
  if (w_lo > w_hi) {
    kt0 = 0;
    kt1 = -1;
    return;
  }
  kt0 = w_lo / rows;
  kt1 = w_hi / rows;
}

// Allowed local columns [c_lo, c_hi] (clamped to [0, 127] / [-1, 127]) of
// tile kt of block j for a row whose allowed token interval is [lo, hi].
__device__ __forceinline__ void col_bounds(int order, int S, int P, int j, int kt, int lo, int hi,
                                           int& c_lo, int& c_hi) {
  const int Lb = S / P;
  const int w_base = kt * kT;
  int a, b;
  if (order == SP_ORDER_STRIPED) {
    a = -floor_div_i(-(lo - j), P) - w_base;
    b = floor_div_i(hi - j, P) - w_base;
  } else {
    a = lo - j * Lb - w_base;
    b = hi - j * Lb - w_base;
  }
  const int valid = Lb - w_base - 1;
  if (b > valid) b = valid;
  c_lo = a < 0 ? 0 : (a > kT ? kT : a);
  c_hi = b < -1 ? -1 : (b > kT - 1 ? kT - 1 : b);
}

// One tile of rows from local row u of block p, head h: two 64-column boxes,
// the second `half` bytes after the first.
__device__ __forceinline__ void row_tma(uint32_t dst, const CUtensorMap* map, uint32_t bar, int h,
                                        int order, int p, int u, int b, int half = kHalfBytes) {
  const int c2 = order == SP_ORDER_STRIPED ? p : u;
  const int c3 = order == SP_ORDER_STRIPED ? u : p;
  tma_load_5d(dst, map, bar, 0, h, c2, c3, b);
  tma_load_5d(dst + half, map, bar, 64, h, c2, c3, b);
}

// K-major bf16 tile of 128 columns (two 64-column halves `half` bytes apart,
// 128-byte swizzle): descriptor of k-step kk (16 columns).
__device__ __forceinline__ uint64_t kmaj_desc(uint64_t base, int kk, int half = kHalfBytes) {
  return base + ((((kk >> 2) * half) + (kk & 3) * 32) >> 4);
}

// Wait that first tests without blocking: loads that usually landed long ago
// then cost the issuing thread little (a blocking wait costs ~150 cycles).
__device__ __forceinline__ bool wait_ready(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int* err, int code) {
  return mbar_test_wait(bar, parity) || mbar_wait(bar, parity, abort_flag, err, code);
}

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err, int code) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, err, code));
}

// Offset of local row u of block p in a block-ordered [outer][P][Lbp] array.
__device__ __forceinline__ long long blk_index(long long outer, int P, int Lbp, int p, int u) {
  return (outer * P + p) * Lbp + u;
}

// ------------------------------------------------------------------ prep
// Three index ranges in one launch:
//  [0, nA)        16 lanes per query row (b, t, h): D = dout . out (16-byte
//                 loads), written with lse * log2(e) at the row's block slot;
//  [nA, +nB)      the padding slots u in [Lb, Lbp): D = 0, lse2 = +inf;
//  [.., +nC)      doc_start in block order (INT_MAX in the padding), causal.
// nA is a multiple of 32 so that no warp straddles the first two ranges.
struct PrepArgs {
  const uint4* out;
  const uint4* dout;
  const float* lse;
  const int32_t* doc_start;
  float* D_blk;
  float* lse2_blk;
  int32_t* lo_blk;
  long long rows, nA, nB, nC;
  int S, H, P, Lbp, order;
  // geometry of the doc_start lookups (the whole sequence); lo_block >= 0:
  // the rows are those of that one block (per-device form)
  int lo_S, lo_P, lo_order, lo_block;
};

__global__ void __launch_bounds__(256) bwd_prep_kernel(PrepArgs pa) {
  long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int Lb = pa.S / pa.P;
  if (g < pa.nA) {
    const long long row = g >> 4;
    const bool live = row < pa.rows;
    float acc = 0.f;
    if (live) {
      const uint4 x = __ldcs(pa.out + g), y = __ldcs(pa.dout + g);
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
        const float2 yf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[e]));
        acc = fmaf(xf.x, yf.x, acc);
        acc = fmaf(xf.y, yf.y, acc);
      }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (live && (threadIdx.x & 15) == 0) {
      const int h = static_cast<int>(row % pa.H);
      const long long bt = row / pa.H;
      const int t = static_cast<int>(bt % pa.S);
      const long long b = bt / pa.S;
      const int p = pa.order == SP_ORDER_STRIPED ? t % pa.P : t / Lb;
      const int u = pa.order == SP_ORDER_STRIPED ? t / pa.P : t % Lb;
      const long long bh = b * pa.H + h;
      const long long idx = blk_index(bh, pa.P, pa.Lbp, p, u);
      pa.D_blk[idx] = acc;
      pa.lse2_blk[idx] = pa.lse[bh * pa.S + t] * kLog2e;
    }
    return;
  }
  g -= pa.nA;
  if (g < pa.nB) {
    const int w = pa.Lbp - Lb;
    const long long bhp = g / w;
    const long long idx = bhp * pa.Lbp + Lb + g % w;
    pa.D_blk[idx] = 0.f;
    pa.lse2_blk[idx] = INFINITY;
    return;
  }
  g -= pa.nB;
  if (g < pa.nC) {
    const int u = static_cast<int>(g % pa.Lbp);
    const long long rp = g / pa.Lbp;
    const int p = pa.lo_block >= 0 ? pa.lo_block : static_cast<int>(rp % pa.P);
    const long long r = pa.lo_block >= 0 ? rp : rp / pa.P;
    pa.lo_blk[g] = u < Lb ? pa.doc_start[r * pa.lo_S +
                                         block_token(pa.lo_order, pa.lo_S, pa.lo_P, p, u)]
                          : INT_MAX;
  }
}

// ------------------------------------------------------------------ dQ
constexpr int kQThreads = 320;  // warps 0-7 elementwise (two warpgroups), 8 TMA, 9 MMA
constexpr int kQProducer = 8;
constexpr int kQMma = 9;
constexpr int kQEw = 256;       // elementwise threads
constexpr int kQSmemBytes = (2 + kKSlots + kVSlots) * kTileBytes;

__global__ void __launch_bounds__(kQThreads, 1)
    bwd_dq_kernel(const __grid_constant__ BwdMaps tm, BwdArgs a, int n_tiles_q) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t q_full, s_full, s_free, dq_full, done;
  __shared__ uint64_t ds_full[2];  // per dS buffer
  __shared__ uint64_t k_full[kKSlots], k_empty[kKSlots], v_full[kVSlots], v_empty[kVSlots];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sq = smem_u32(smem), sdo = sq + kTileBytes, sks = sq + 2 * kTileBytes;
  const uint32_t svs = sks + kKSlots * kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work item: heavy query positions first, heads innermost
  const int BH = a.B * a.Hq;
  const int pos = blockIdx.x / BH, bh = blockIdx.x % BH;
  const int b = bh / a.Hq, h = bh % a.Hq, kvh = h / (a.Hq / a.Hkv);
  const int rev = a.P * n_tiles_q - 1 - pos;
  const int i = rev / n_tiles_q, qt = rev % n_tiles_q;
  const int Lb = a.S / a.P, u0 = qt * kT;
  int hull_lo, hull_hi;
  {
    const int u_last = min(u0 + kT, Lb) - 1;
    const int t_first = static_cast<int>(block_token(a.order, a.S, a.P, i, u0));
    const int t_last = static_cast<int>(block_token(a.order, a.S, a.P, i, u_last));
    if (a.doc_start) {
      hull_lo = a.doc_start[static_cast<long long>(b % a.pos_rows) * a.S + t_first];
      hull_hi = t_last;
    } else {
      hull_lo = 0;
      hull_hi = a.S - 1;
    }
  }
  int n_tiles = 0;
  for (int s = 0; s < a.P; ++s) {
    int kt0, kt1;
    block_tiles(a.order, a.S, a.P, ((i - s) % a.P + a.P) % a.P, hull_lo, hull_hi, kT, kt0, kt1);
    n_tiles += kt1 - kt0 + 1;
  }

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&q_full), 1);
    mbar_init(smem_u32(&s_full), 1);
    mbar_init(smem_u32(&s_free), kQEw);
    mbar_init(smem_u32(&ds_full[0]), kQEw);
    mbar_init(smem_u32(&ds_full[1]), kQEw);
    mbar_init(smem_u32(&dq_full), 1);
    mbar_init(smem_u32(&done), 1);
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
    }
    abort_s = 0;
    fence_mbar_init();
  }
  if (warp == kQMma) {
    tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  volatile int* abort_flag = &abort_s;
  // TMEM columns: S [0,128) dP [128,256) dQ [256,384) dS buffers [384,448) [448,512)
  const uint32_t cS = 0, cdP = 128, cdQ = 256, cdS = 384;

  if (warp == kQProducer) {
    if (lane == 0) {
      prefetch_tmap(&tm.q);
      prefetch_tmap(&tm.dout);
      prefetch_tmap(&tm.k);
      prefetch_tmap(&tm.v);
      const uint32_t qf = smem_u32(&q_full);
      mbar_arrive_expect_tx(qf, 2 * kTileBytes);
      row_tma(sq, &tm.q, qf, h, a.order, i, u0, b);
      row_tma(sdo, &tm.dout, qf, h, a.order, i, u0, b);
      int n = 0;  // tiles loaded
      bool ok = true;
      for (int s = 0; s < a.P && ok; ++s) {
        const int j = ((i - s) % a.P + a.P) % a.P;
        int kt0, kt1;
        block_tiles(a.order, a.S, a.P, j, hull_lo, hull_hi, kT, kt0, kt1);
        for (int kt = kt0; kt <= kt1; ++kt, ++n) {
          const int ks = n % kKSlots, vs = n % kVSlots;
          if (!mbar_wait(smem_u32(&k_empty[ks]), ((n / kKSlots) & 1) ^ 1, abort_flag, a.err,
                         kErrBwdKvEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_u32(&k_full[ks]), kTileBytes);
          row_tma(sks + ks * kTileBytes, &tm.k, smem_u32(&k_full[ks]), kvh, a.order, j, kt * kT, b);
          if (!mbar_wait(smem_u32(&v_empty[vs]), ((n / kVSlots) & 1) ^ 1, abort_flag, a.err,
                         kErrBwdKvEmpty)) {
            ok = false;
            ++n;  // K of this tile is in flight
            break;
          }
          mbar_arrive_expect_tx(smem_u32(&v_full[vs]), kTileBytes);
          row_tma(svs + vs * kTileBytes, &tm.v, smem_u32(&v_full[vs]), kvh, a.order, j, kt * kT, b);
        }
      }
      // copies still in flight land before the CTA can exit
      mbar_wait(qf, 0, abort_flag, a.err, kErrBwdDrain);
      for (int m = n - 1; m >= 0 && m >= n - kKSlots; --m)
        mbar_wait(smem_u32(&k_full[m % kKSlots]), (m / kKSlots) & 1, abort_flag, a.err,
                  kErrBwdDrain);
      for (int m = n - 1; m >= 0 && m >= n - kVSlots; --m)
        mbar_wait(smem_u32(&v_full[m % kVSlots]), (m / kVSlots) & 1, abort_flag, a.err,
                  kErrBwdDrain);
    }
  } else if (warp == kQMma) {
    if (lane == 0 && n_tiles > 0) {
      const uint64_t dq_ = smem_desc_sw128(sq, 16, 1024), ddo = smem_desc_sw128(sdo, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sks, 16, 1024);          // K-major K slots
      const uint64_t dkmn = smem_desc_sw128(sks, kHalfBytes, 1024);  // MN-major view (B of dS K)
      const uint64_t dv0 = smem_desc_sw128(svs, 16, 1024);          // K-major V slots
      // S = Q K^T, then dP = dO V^T for tile t, each as soon as its operand landed
      auto issue_sdp = [&](int t) -> bool {
        const int ks = t % kKSlots, vs = t % kVSlots;
        if (!wait_ready(smem_u32(&k_full[ks]), (t / kKSlots) & 1, abort_flag, a.err, kErrBwdKvFull))
          return false;
        // V_t has usually landed too: test it now, so that dP follows S
        // without a barrier access between the two batches of MMAs
        const bool v_ready = mbar_test_wait(smem_u32(&v_full[vs]), (t / kVSlots) & 1);
        tc_fence_after();
        const uint64_t kb = dk0 + ((ks * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(tmem + cS, kmaj_desc(dq_, kk), kmaj_desc(kb, kk), kIdescKmaj, kk > 0 ? 1u : 0u);
        if (!v_ready) {
          if (!wait_ready(smem_u32(&v_full[vs]), (t / kVSlots) & 1, abort_flag, a.err,
                          kErrBwdKvFull))
            return false;
          tc_fence_after();
        }
        const uint64_t vb = dv0 + ((vs * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(tmem + cdP, kmaj_desc(ddo, kk), kmaj_desc(vb, kk), kIdescKmaj, kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&s_full));
        mma_commit(smem_u32(&v_empty[vs]));  // V_t consumed once dP is done
        return true;
      };
      bool ok = mbar_wait(smem_u32(&q_full), 0, abort_flag, a.err, kErrBwdQFull);
      tc_fence_after();
      if (ok) ok = issue_sdp(0);
      for (int t = 0; t < n_tiles && ok; ++t) {
        if (!mbar_wait(smem_u32(&s_free), t & 1, abort_flag, a.err, kErrBwdSFree)) break;
        if (t + 1 < n_tiles && !issue_sdp(t + 1)) break;
        if (!mbar_wait(smem_u32(&ds_full[t & 1]), (t >> 1) & 1, abort_flag, a.err, kErrBwdDsFull))
          break;
        tc_fence_after();
        // dQ += dS K: dS (bf16 pairs) from TMEM, K_t as the MN-major B operand
        const uint64_t kmn = dkmn + (((t % kKSlots) * kTileBytes) >> 4);
        const uint32_t ds = tmem + cdS + (t & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_ts(tmem + cdQ, ds + kk * 8, kmn + ((kk * 16 * 128) >> 4), kIdescBmn,
                 (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(smem_u32(&k_empty[t % kKSlots]));  // K_t consumed
      }
      mma_commit(smem_u32(&dq_full));
      mma_commit(smem_u32(&done));
      mbar_wait(smem_u32(&done), 0, abort_flag, a.err, kErrBwdDrain);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------- elementwise warps
    // warpgroup `half` owns columns [64 half, 64 half + 64) of every tile
    const int half = warp >> 2;
    const int row = threadIdx.x & 127;  // TMEM lane == query row of the tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int u = u0 + row;
    const bool row_live = u < Lb;
    const int tq = row_live ? static_cast<int>(block_token(a.order, a.S, a.P, i, u)) : 0;
    const long long bi = blk_index(static_cast<long long>(b) * a.Hq + h, a.P, a.Lbp, i, u);
    const float lse2 = row_live ? a.lse2_blk[bi] : 0.f;
    const float Drow = row_live ? a.D_blk[bi] : 0.f;
    int lo = 0, hi = a.S - 1;
    if (a.doc_start && row_live) {
      lo = a.doc_start[static_cast<long long>(b % a.pos_rows) * a.S + tq];
      hi = tq;
    }
    const float sl2 = a.scale * kLog2e;
    const int col0 = half * 64;
    int t = 0;
    bool ok = true;
    for (int s = 0; s < a.P && ok; ++s) {
      const int j = ((i - s) % a.P + a.P) % a.P;
      int kt0, kt1;
      block_tiles(a.order, a.S, a.P, j, hull_lo, hull_hi, kT, kt0, kt1);
      for (int kt = kt0; kt <= kt1; ++kt, ++t) {
        if (!wait_warp(smem_u32(&s_full), t & 1, abort_flag, a.err, kErrBwdSFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sx[64], px[64];
        tmem_ld32_at(tmem + lane_base + cS + col0, sx, 0);
        tmem_ld32_at(tmem + lane_base + cS + col0 + 32, sx, 32);
        tmem_ld32_at(tmem + lane_base + cdP + col0, px, 0);
        tmem_ld32_at(tmem + lane_base + cdP + col0 + 32, px, 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(smem_u32(&s_free));  // S and dP read: the next tile's MMAs may start
        int c_lo, c_hi;
        col_bounds(a.order, a.S, a.P, j, kt, lo, hi, c_lo, c_hi);
        if (!row_live) {
          c_lo = 0;
          c_hi = -1;
        }
        c_lo -= col0;
        c_hi -= col0;
        // masked scores become -inf (p = 0), outside the exp loop
        if (c_lo > 0 || c_hi < 63) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < c_lo || c > c_hi) sx[c] = 0xff800000u;
        }
        uint32_t dsw[32];  // dS, bf16 pairs
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float x0, x1, p0, p1, d0, d1;
          ffma2(x0, x1, __uint_as_float(sx[c]), __uint_as_float(sx[c + 1]), sl2, sl2, -lse2,
                -lse2);
          p0 = ex2(x0);
          p1 = ex2(x1);
          fadd2(d0, d1, __uint_as_float(px[c]), __uint_as_float(px[c + 1]), -Drow, -Drow);
          fmul2(d0, d1, d0, d1, p0, p1);
          dsw[c >> 1] = pack_bf16(d0, d1);
        }
        tmem_st32(tmem + lane_base + cdS + (t & 1) * 64 + half * 32, dsw);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&ds_full[t & 1]));
      }
    }
    // epilogue: dQ * scale, this warpgroup's 64 columns
    const bool have = n_tiles > 0 && ok;
    if (have && !wait_warp(smem_u32(&dq_full), 0, abort_flag, a.err, kErrBwdOut)) ok = false;
    tc_fence_after();
    __nv_bfloat16* dq = static_cast<__nv_bfloat16*>(a.dq);
    uint4* orow = reinterpret_cast<uint4*>(
        dq + ((static_cast<long long>(b) * a.S + tq) * a.Hq + h) * kD + col0);
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      uint32_t r[32];
      if (have && ok) {
        tmem_ld32(tmem + lane_base + cdQ + col0 + c * 32, r);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = 0u;
      }
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pk[e] = pack_bf16(__uint_as_float(r[2 * e]) * a.scale,
                          __uint_as_float(r[2 * e + 1]) * a.scale);
      if (row_live) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          orow[c * 4 + e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kQMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------------------------------------- dK / dV
constexpr int kKvThreads = 192;             // warps 0-3 elementwise, 4 TMA, 5 MMA
constexpr int kKvProducer = 4;
constexpr int kKvMma = 5;
constexpr int kQT = 128;                     // query rows per streamed tile
constexpr int kQSlots = 2;                   // Q + dO tile pairs in flight
constexpr int kKvSmemBytes = 2 * kTileBytes + kQSlots * 2 * kTileBytes;
static_assert(kQT == kBwdRowPad, "query tiles are the block-order padding unit");

enum : int { kInfoEnd = 0, kInfoTile = 1, kInfoFull = 3 };

// Per-column data of one streamed query tile: three bulk copies from the
// block-ordered arrays, plus a header the producer writes.
struct alignas(16) ColData {
  float lse2[kQT];  // lse * log2(e); +inf for rows past the end of the block
  float D[kQT];
  int lo[kQT];      // doc_start of the column's query (causal); INT_MAX past the end
  int info;         // kInfoEnd, kInfoTile (masked per pair) or kInfoFull (every pair allowed)
  int i, u0;        // query block and first local row of the tile
  int h;            // query head
};

// One CTA per 128-key tile (K, V resident).  Per 128-query tile:
//   S^T = K Q^T, dP^T = V dO^T            (SS, into TMEM [0,128) / [128,256))
//   elementwise, in two 64-column halves:  P^T, dS^T (bf16 pairs) written over
//     the first 32 (half 0) / next 32 (half 1) columns of S^T / dP^T
//   dV += P^T dO, dK += dS^T Q            (TS, one 64-query half at a time:
//     half 0's products run while half 1 is being computed)
// TMEM is full (S^T, dP^T, dV, dK), so S^T of the next tile waits for the
// last dV/dK product of this one (tcgen05 MMAs of one thread run in order).
__global__ void __launch_bounds__(kKvThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ BwdMaps tm, BwdArgs a, int n_tiles_k) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t q_full[kQSlots], q_empty[kQSlots], kv_full, s_full, half_full[2], dkv_full,
      done;
  __shared__ ColData cols[kQSlots];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sk = smem_u32(smem), sv = sk + kTileBytes, sslot = sk + 2 * kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work item: earliest key tiles first (for causal calls they meet the most queries)
  const int BH = a.B * a.Hkv;
  const int pos = blockIdx.x / BH, bh = blockIdx.x % BH;
  const int b = bh / a.Hkv, hk = bh % a.Hkv;
  const int j = pos / n_tiles_k, kt = pos % n_tiles_k;
  const int Lb = a.S / a.P, w0 = kt * kT;
  const int k_first = static_cast<int>(block_token(a.order, a.S, a.P, j, w0));
  const int k_last = static_cast<int>(block_token(a.order, a.S, a.P, j, min(w0 + kT, Lb) - 1));
  const int32_t* ds_row =
      a.doc_start ? a.doc_start + static_cast<long long>(b % a.pos_rows) * a.S : nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQSlots; ++s) {
      mbar_init(smem_u32(&q_full[s]), 1);
      mbar_init(smem_u32(&q_empty[s]), 1);
    }
    mbar_init(smem_u32(&kv_full), 1);
    mbar_init(smem_u32(&s_full), 1);
    mbar_init(smem_u32(&half_full[0]), kT);
    mbar_init(smem_u32(&half_full[1]), kT);
    mbar_init(smem_u32(&dkv_full), 1);
    mbar_init(smem_u32(&done), 1);
    abort_s = 0;
    fence_mbar_init();
  }
  if (warp == kKvMma) {
    tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  volatile int* abort_flag = &abort_s;
  // TMEM columns: S^T [0,128), dP^T [128,256), dV [256,384), dK [384,512)
  const uint32_t cdP = 128, cdV = 256, cdK = 384;

  if (warp == kKvProducer) {
    // ------------------------------------------------------------ producer
    const int G = a.Hq / a.Hkv;
    if (lane == 0) {
      prefetch_tmap(&tm.k);
      prefetch_tmap(&tm.v);
      prefetch_tmap(&tm.q);
      prefetch_tmap(&tm.dout);
      const uint32_t kf = smem_u32(&kv_full);
      mbar_arrive_expect_tx(kf, 2 * kTileBytes);
      row_tma(sk, &tm.k, kf, hk, a.order, j, w0, b);
      row_tma(sv, &tm.v, kf, hk, a.order, j, w0, b);
    }
    const long long lo_row = static_cast<long long>(b % a.pos_rows);
    const uint32_t col_bytes = (ds_row ? 3 : 2) * kQT * 4;
    int n = 0;
    bool ok = true;
    for (int g = 0; g < G && ok; ++g) {
      const int h = hk * G + g;
      const long long bhq = static_cast<long long>(b) * a.Hq + h;
      for (int s = 0; s < a.P && ok; ++s) {
        const int i = (j + s) % a.P;
        int qt0, qt1;
        block_tiles(a.order, a.S, a.P, i, ds_row ? k_first : 0, a.S - 1, kQT, qt0, qt1);
        // flags of 32 tiles at a time, one per lane
        for (int base = qt0; base <= qt1 && ok; base += 32) {
          const int qt = base + lane;
          bool stop = false, full = true;
          if (ds_row && qt <= qt1) {
            const int u0 = qt * kQT;
            const int tq_first = static_cast<int>(block_token(a.order, a.S, a.P, i, u0));
            const int tq_last =
                static_cast<int>(block_token(a.order, a.S, a.P, i, min(u0 + kQT, Lb) - 1));
            // document starts do not decrease along the tokens of a block, so
            // once a tile starts past the keys' documents the rest do too
            stop = ds_row[tq_first] > k_last;
            full = k_last <= tq_first && ds_row[tq_last] <= k_first;
          }
          const unsigned stops = __ballot_sync(0xffffffffu, stop);
          const unsigned fulls = __ballot_sync(0xffffffffu, full);
          int cnt = min(32, qt1 - base + 1);
          if (stops) cnt = min(cnt, __ffs(static_cast<int>(stops)) - 1);
          for (int e = 0; e < cnt; ++e) {
            const int slot = n % kQSlots;
            if (!wait_warp(smem_u32(&q_empty[slot]), ((n / kQSlots) & 1) ^ 1, abort_flag, a.err,
                           kErrBwdKvEmpty)) {
              ok = false;
              break;
            }
            if (lane == 0) {
              const int u0 = (base + e) * kQT;
              ColData& cd = cols[slot];
              cd.info = (fulls >> e) & 1u ? kInfoFull : kInfoTile;
              cd.i = i;
              cd.u0 = u0;
              cd.h = h;
              const uint32_t bar = smem_u32(&q_full[slot]);
              const uint32_t dst = sslot + slot * 2 * kTileBytes;
              mbar_arrive_expect_tx(bar, 2 * kTileBytes + col_bytes);
              row_tma(dst, &tm.q, bar, h, a.order, i, u0, b);
              row_tma(dst + kTileBytes, &tm.dout, bar, h, a.order, i, u0, b);
              const long long off = blk_index(bhq, a.P, a.Lbp, i, u0);
              bulk_load(smem_u32(cd.lse2), a.lse2_blk + off, kQT * 4, bar);
              bulk_load(smem_u32(cd.D), a.D_blk + off, kQT * 4, bar);
              if (ds_row)
                bulk_load(smem_u32(cd.lo), a.lo_blk + blk_index(lo_row, a.P, a.Lbp, i, u0),
                          kQT * 4, bar);
            }
            ++n;
          }
          if (stops) break;
        }
      }
    }
    if (ok) {  // end of the list
      const int slot = n % kQSlots;
      if (wait_warp(smem_u32(&q_empty[slot]), ((n / kQSlots) & 1) ^ 1, abort_flag, a.err,
                    kErrBwdKvEmpty) &&
          lane == 0) {
        cols[slot].info = kInfoEnd;
        mbar_arrive(smem_u32(&q_full[slot]));
      }
    }
    // copies still in flight land before the CTA can exit
    if (lane == 0) {
      mbar_wait(smem_u32(&kv_full), 0, abort_flag, a.err, kErrBwdDrain);
      for (int m = n - 1; m >= 0 && m > n - kQSlots; --m)
        mbar_wait(smem_u32(&q_full[m % kQSlots]), (m / kQSlots) & 1, abort_flag, a.err,
                  kErrBwdDrain);
    }
    __syncwarp();
  } else if (warp == kKvMma) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint64_t dk0 = smem_desc_sw128(sk, 16, 1024), dv0 = smem_desc_sw128(sv, 16, 1024);
      const uint64_t dkq = smem_desc_sw128(sslot, 16, 1024);          // K-major Q / dO views
      const uint64_t dmn = smem_desc_sw128(sslot, kHalfBytes, 1024);  // MN-major Q / dO views
      // info of tile t once its slot is full; -1 when the wait gave up
      auto tile_info = [&](int t) -> int {
        const int slot = t % kQSlots;
        if (!wait_ready(smem_u32(&q_full[slot]), (t / kQSlots) & 1, abort_flag, a.err,
                        kErrBwdQFull))
          return -1;
        return cols[slot].info;
      };
      // S^T = K Q^T and dP^T = V dO^T for tile t (N = 128 queries)
      auto issue_sdp = [&](int t) {
        tc_fence_after();
        const uint64_t qb = dkq + (((t % kQSlots) * 2 * kTileBytes) >> 4);
        const uint64_t ob = qb + (kTileBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(tmem, kmaj_desc(dk0, kk), kmaj_desc(qb, kk), kIdescKmaj, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(tmem + cdP, kmaj_desc(dv0, kk), kmaj_desc(ob, kk), kIdescKmaj, kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&s_full));
      };
      // dV += P^T dO and dK += dS^T Q over the 64 queries of half h of tile t
      auto issue_grad = [&](int t, int h) {
        const uint64_t qb = dmn + (((t % kQSlots) * 2 * kTileBytes) >> 4);
        const uint64_t ob = qb + (kTileBytes >> 4);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = h * 4 + k4;  // 16-query step within the tile
          mma_ts(tmem + cdV, tmem + kk * 8, ob + ((kk * 16 * 128) >> 4), kIdescBmn,
                 (t > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = h * 4 + k4;
          mma_ts(tmem + cdK, tmem + cdP + kk * 8, qb + ((kk * 16 * 128) >> 4), kIdescBmn,
                 (t > 0 || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(smem_u32(&kv_full), 0, abort_flag, a.err, kErrBwdKvFull);
      int cur = ok ? tile_info(0) : -1;
      if (cur > 0) issue_sdp(0);
      for (int t = 0; cur > 0; ++t) {
        bool got = true;
        int nxt = -2;  // tile t+1's info, once known
        for (int h = 0; h < 2 && got; ++h) {
          got = mbar_wait(smem_u32(&half_full[h]), t & 1, abort_flag, a.err, kErrBwdDsFull);
          if (got) {
            // Tile t+1's Q and dO have usually landed by now: test it here,
            // where the thread has just woken, rather than after the
            // gradient MMAs, where a barrier access waits for the issue
            // queue to drain while the tensor pipe runs dry.
            if (h == 0) {
              const int ns = (t + 1) % kQSlots;
              if (mbar_test_wait(smem_u32(&q_full[ns]), ((t + 1) / kQSlots) & 1))
                nxt = cols[ns].info;
            }
            tc_fence_after();
            issue_grad(t, h);
          }
        }
        if (!got) break;
        mma_commit(smem_u32(&q_empty[t % kQSlots]));  // Q_t, dO_t consumed
        if (nxt == -2) nxt = tile_info(t + 1);
        if (nxt > 0) issue_sdp(t + 1);
        cur = nxt;
      }
      mma_commit(smem_u32(&dkv_full));
      mma_commit(smem_u32(&done));
      mbar_wait(smem_u32(&done), 0, abort_flag, a.err, kErrBwdDrain);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------- elementwise warps
    const int r = threadIdx.x;  // TMEM lane == key row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int w = w0 + r;
    const bool key_live = w < Lb;
    const int ktok = key_live ? static_cast<int>(block_token(a.order, a.S, a.P, j, w)) : -1;
    const float sl2 = a.scale * kLog2e;
    int t = 0;
    bool ok = true;
    for (;; ++t) {
      const int slot = t % kQSlots;
      if (!wait_warp(smem_u32(&q_full[slot]), (t / kQSlots) & 1, abort_flag, a.err,
                     kErrBwdQFull)) {
        ok = false;
        break;
      }
      const ColData& cd = cols[slot];
      const int info = cd.info;
      if (info == kInfoEnd) break;
      if (!wait_warp(smem_u32(&s_full), t & 1, abort_flag, a.err, kErrBwdSFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool full = info == kInfoFull;
      // causal part of the mask: column c holds a query token >= ktok iff c >= c_min
      int c_min = 0;
      if (!full) {
        c_min = a.order == SP_ORDER_STRIPED ? -floor_div_i(-(ktok - cd.i), a.P) - cd.u0
                                            : ktok - (cd.i * Lb + cd.u0);
      }
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t sx[64], px[64];
        tmem_ld32_at(tmem + lane_base + h * 64, sx, 0);
        tmem_ld32_at(tmem + lane_base + h * 64 + 32, sx, 32);
        tmem_ld32_at(tmem + lane_base + cdP + h * 64, px, 0);
        tmem_ld32_at(tmem + lane_base + cdP + h * 64 + 32, px, 32);
        tmem_wait_ld();
        if (!full) {  // masked scores become -inf (p = 0), outside the exp loop
#pragma unroll
          for (int c4 = 0; c4 < 64; c4 += 4) {
            const int c = h * 64 + c4;
            const int4 lo = *reinterpret_cast<const int4*>(&cd.lo[c]);
            if (c < c_min || lo.x > ktok) sx[c4] = 0xff800000u;
            if (c + 1 < c_min || lo.y > ktok) sx[c4 + 1] = 0xff800000u;
            if (c + 2 < c_min || lo.z > ktok) sx[c4 + 2] = 0xff800000u;
            if (c + 3 < c_min || lo.w > ktok) sx[c4 + 3] = 0xff800000u;
          }
        }
        uint32_t pk[32], dk[32];
#pragma unroll
        for (int c4 = 0; c4 < 64; c4 += 4) {
          const int c = h * 64 + c4;  // column of the tile
          const float4 l2 = *reinterpret_cast<const float4*>(&cd.lse2[c]);
          const float4 D = *reinterpret_cast<const float4*>(&cd.D[c]);
          float x0, x1, x2, x3;
          ffma2(x0, x1, __uint_as_float(sx[c4]), __uint_as_float(sx[c4 + 1]), sl2, sl2, -l2.x,
                -l2.y);
          ffma2(x2, x3, __uint_as_float(sx[c4 + 2]), __uint_as_float(sx[c4 + 3]), sl2, sl2, -l2.z,
                -l2.w);
          const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
          float d0, d1, d2, d3;
          fadd2(d0, d1, __uint_as_float(px[c4]), __uint_as_float(px[c4 + 1]), -D.x, -D.y);
          fadd2(d2, d3, __uint_as_float(px[c4 + 2]), __uint_as_float(px[c4 + 3]), -D.z, -D.w);
          fmul2(d0, d1, d0, d1, p0, p1);
          fmul2(d2, d3, d2, d3, p2, p3);
          pk[c4 >> 1] = pack_bf16(p0, p1);
          pk[(c4 >> 1) + 1] = pack_bf16(p2, p3);
          dk[c4 >> 1] = pack_bf16(d0, d1);
          dk[(c4 >> 1) + 1] = pack_bf16(d2, d3);
        }
        // half h's 64 queries as 32 bf16-pair columns; S^T / dP^T columns
        // [32h, 32h + 32) were read in half 0
        tmem_st32(tmem + lane_base + h * 32, pk);
        tmem_st32(tmem + lane_base + cdP + h * 32, dk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&half_full[h]));
      }
    }
    // epilogue: dK * scale and dV, rows of key token ktok
    const bool have = t > 0 && ok;
    if (have && !wait_warp(smem_u32(&dkv_full), 0, abort_flag, a.err, kErrBwdOut)) ok = false;
    tc_fence_after();
    const long long orow =
        ((static_cast<long long>(b) * a.S + (key_live ? ktok : 0)) * a.Hkv + hk) * kD;
    uint4* dk_row = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dk) + orow);
    uint4* dv_row = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dv) + orow);
#pragma unroll 1
    for (int m = 0; m < 2; ++m) {
      const float mul = m == 0 ? a.scale : 1.f;
      uint4* dst = m == 0 ? dk_row : dv_row;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t x[32];
        if (have && ok) {
          tmem_ld32(tmem + lane_base + (m == 0 ? cdK : cdV) + c * 32, x);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16(__uint_as_float(x[2 * e]) * mul, __uint_as_float(x[2 * e + 1]) * mul);
        if (key_live) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[c * 4 + e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kKvMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}


// ------------------------------------------------------ fused dK/dV + dQ
// The dK/dV walk with dQ folded in, so that S^T and dP^T are multiplied once
// per pair of tiles (10 d FLOPs per allowed pair instead of 14 d for the two
// kernels above).  dS^T goes to shared memory instead of tensor memory: read
// as a K-major operand it is the A of dK += dS^T Q, read MN-major it is the A
// of dQ_tile = dS K.  dQ_tile (128 queries x 128 columns, fp32) lands in the
// tensor-memory columns dP^T held; the elementwise warps read it and stage it
// in shared memory, and the TMA adds it into an fp32 accumulator in global
// memory (bulk reductions); bwd_dq_convert_kernel scales and rounds the sums
// to bf16.  The reductions arrive in no fixed order, so dQ is reproducible to fp32 rounding, not bit
// for bit (the two-kernel path is).
constexpr int kFThreads = 224;  // warps 0-3 elementwise, 4 TMA, 5 MMA, 6 dQ reductions
constexpr int kFProducer = 4;
constexpr int kFMma = 5;
constexpr int kFReducer = 6;
constexpr int kFSmemBytes = 6 * kTileBytes;  // K, V, Q slots 0 and 1, dO, dS^T
// A and B MN-major: dQ_tile = dS K reads dS from the key-row-major dS^T
// buffer and K from its key-row-major tile.
constexpr uint32_t kIdescAmnBmn = kIdescBmn | (1u << 15);

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t x, uint32_t y, uint32_t z,
                                       uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z),
               "r"(w)
               : "memory");
}

__device__ __forceinline__ void red_add_v4(float* addr, float x, float y, float z, float w) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(x),
               "f"(y), "f"(z), "f"(w)
               : "memory");
}

// dst[i] += src[i] for `bytes` / 4 floats, by the TMA unit (bulk group of the
// issuing thread; both addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                   dst),
               "r"(src), "r"(bytes)
               : "memory");
}


// Per-device form of the fused kernel: query block i against key/value block
// j, the block tensors [B][S/P][H][d] in local row order (their tensor maps
// hold one block); masks use the global tokens of both blocks.  q_block < 0:
// the whole sequence.
struct BwdBlock {
  int q_block, kv_block;
  float* dk_acc;  // [B][S/P][Hkv][d] float32: += scale * dS^T Q
  float* dv_acc;  // [B][S/P][Hkv][d] float32: += P^T dO
};

// One CTA per 128-key tile, walking the query tiles like bwd_dkdv_kernel.
// Per 128-query tile t:
//   S^T = K Q^T, dP^T = V dO^T                (SS, TMEM [0,128) / [128,256))
//   two 64-column halves: P^T (bf16 pairs) over S^T columns [32h, 32h+32),
//     dS^T (bf16) to the shared-memory buffer
//   dV += P^T dO (TS), dK += dS^T Q (SS)        half 0 while half 1 is computed
//   dQ_tile = dS K (SS, TMEM [128,256)) -> elementwise warps -> shared memory
//     (Q_t's slot and the dS^T buffer, both free once dQ_tile is complete)
//     -> two 32 KiB TMA bulk reductions into the global fp32 sums
// dO has one slot (released after the last dV product, reloaded while dK,
// dQ and the next S^T run); dP^T of the next tile waits until dQ_tile has
// been read out of tensor memory.  The reducer warp issues the two bulk
// reductions and, as the TMA finishes reading them, releases the dS^T buffer
// (to the next tile's dS^T stores) and Q_t's slot (to the producer, for
// Q_{t+2}), so the reductions drain while the next tile is computed.
//
// dQ accumulator layout: per (batch, query head, block, 128-row tile) a
// 64 KiB block ordered [column quad 32][row 128][4]: staged in the same
// order, its two halves are two contiguous bulk reductions, and a warp's
// shared-memory stores cover 512 contiguous bytes.
__global__ void __launch_bounds__(kFThreads, 1)
    bwd_fused_kernel(const __grid_constant__ BwdMaps tm, BwdArgs a, int n_tiles_k,
                     float* __restrict__ dq_acc, BwdBlock bb) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t q_full[kQSlots], q_empty[kQSlots], do_full, do_empty, kv_full, s_full,
      half_full[2], dq_full, dq_free, stage_full, stage_free, dkv_full, done;
  __shared__ ColData cols[kQSlots];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sk = smem_u32(smem), sv = sk + kTileBytes, sq = sk + 2 * kTileBytes;
  const uint32_t sdo = sk + 4 * kTileBytes, sds = sk + 5 * kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // per-device form: one block in the tensor maps, the per-query arrays and
  // the dQ accumulator
  // (in the per-device form every query head has its CTAs -- one block
  // pair alone gives too few CTAs per key/value head to fill the GPU -- and
  // the heads of a GQA group add into the accumulators by reductions)
  const bool per_dev = bb.q_block >= 0;
  const int P_arr = per_dev ? 1 : a.P;
  const int map_order = per_dev ? static_cast<int>(SP_ORDER_CONTIGUOUS) : a.order;
  const int G = a.Hq / a.Hkv;
  const int n_heads = per_dev ? a.Hq : a.Hkv;
  const int BH = a.B * n_heads;
  const int pos = blockIdx.x / BH, bh = blockIdx.x % BH;
  const int b = bh / n_heads;
  const int hk = per_dev ? (bh % n_heads) / G : bh % n_heads;
  const int g_begin = per_dev ? (bh % n_heads) % G : 0, g_end = per_dev ? g_begin + 1 : G;
  const int j = per_dev ? bb.kv_block : pos / n_tiles_k, kt = per_dev ? pos : pos % n_tiles_k;
  const int Lb = a.S / a.P, w0 = kt * kT;
  const int k_first = static_cast<int>(block_token(a.order, a.S, a.P, j, w0));
  const int k_last = static_cast<int>(block_token(a.order, a.S, a.P, j, min(w0 + kT, Lb) - 1));
  const int32_t* ds_row =
      a.doc_start ? a.doc_start + static_cast<long long>(b % a.pos_rows) * a.S : nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQSlots; ++s) {
      mbar_init(smem_u32(&q_full[s]), 1);
      mbar_init(smem_u32(&q_empty[s]), 1);
    }
    mbar_init(smem_u32(&do_full), 1);
    mbar_init(smem_u32(&do_empty), 1);
    mbar_init(smem_u32(&kv_full), 1);
    mbar_init(smem_u32(&s_full), 1);
    mbar_init(smem_u32(&half_full[0]), kT);
    mbar_init(smem_u32(&half_full[1]), kT);
    mbar_init(smem_u32(&dq_full), 1);
    mbar_init(smem_u32(&dq_free), kT);
    mbar_init(smem_u32(&stage_full), kT);
    mbar_init(smem_u32(&stage_free), 1);
    mbar_init(smem_u32(&dkv_full), 1);
    mbar_init(smem_u32(&done), 1);
    abort_s = 0;
    fence_mbar_init();
  }
  if (warp == kFMma) {
    tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  volatile int* abort_flag = &abort_s;
  // TMEM columns: S^T [0,128), dP^T then dQ_tile [128,256), dV [256,384), dK [384,512)
  const uint32_t cdP = 128, cdQ = 128, cdV = 256, cdK = 384;

  if (warp == kFProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm.k);
      prefetch_tmap(&tm.v);
      prefetch_tmap(&tm.q);
      prefetch_tmap(&tm.dout);
      const uint32_t kf = smem_u32(&kv_full);
      mbar_arrive_expect_tx(kf, 2 * kTileBytes);
      row_tma(sk, &tm.k, kf, hk, map_order, per_dev ? 0 : j, w0, b);
      row_tma(sv, &tm.v, kf, hk, map_order, per_dev ? 0 : j, w0, b);
    }
    const long long lo_row = static_cast<long long>(b % a.pos_rows);
    const uint32_t col_bytes = (ds_row ? 3 : 2) * kQT * 4;
    int n = 0, n_do = 0;  // Q tiles and dO tiles issued
    bool ok = true, ended = false;
    for (int g = g_begin; g < g_end && ok; ++g) {
      const int h = hk * G + g;
      const long long bhq = static_cast<long long>(b) * a.Hq + h;
      for (int s = 0; s < a.P && ok; ++s) {
        const int i = (j + s) % a.P;
        if (per_dev && i != bb.q_block) continue;
        int qt0, qt1;
        block_tiles(a.order, a.S, a.P, i, ds_row ? k_first : 0, a.S - 1, kQT, qt0, qt1);
        // Q, dO and the column data of query tile qt into the next slots
        auto issue_tile = [&](int qt, bool full) -> bool {
          const int slot = n % kQSlots;
          if (!wait_warp(smem_u32(&q_empty[slot]), ((n / kQSlots) & 1) ^ 1, abort_flag, a.err,
                         kErrBwdKvEmpty))
            return false;
          const int u0 = qt * kQT;
          if (lane == 0) {
            ColData& cd = cols[slot];
            cd.info = full ? kInfoFull : kInfoTile;
            cd.i = i;
            cd.u0 = u0;
            cd.h = h;
            const uint32_t bar = smem_u32(&q_full[slot]);
            mbar_arrive_expect_tx(bar, kTileBytes + col_bytes);
            row_tma(sq + slot * kTileBytes, &tm.q, bar, h, map_order, per_dev ? 0 : i, u0, b);
            const long long off = blk_index(bhq, P_arr, a.Lbp, per_dev ? 0 : i, u0);
            bulk_load(smem_u32(cd.lse2), a.lse2_blk + off, kQT * 4, bar);
            bulk_load(smem_u32(cd.D), a.D_blk + off, kQT * 4, bar);
            if (ds_row)
              bulk_load(smem_u32(cd.lo),
                        a.lo_blk + blk_index(lo_row, P_arr, a.Lbp, per_dev ? 0 : i, u0),
                        kQT * 4, bar);
          }
          ++n;
          if (!wait_warp(smem_u32(&do_empty), (n_do & 1) ^ 1, abort_flag, a.err,
                         kErrBwdKvEmpty))
            return false;
          if (lane == 0) {
            const uint32_t bar = smem_u32(&do_full);
            mbar_arrive_expect_tx(bar, kTileBytes);
            row_tma(sdo, &tm.dout, bar, h, map_order, per_dev ? 0 : i, u0, b);
          }
          ++n_do;
          return true;
        };
        // skip/full flags of query tile qt (lane-parallel, 32 tiles at a time)
        auto flags = [&](int qt, bool& stop, bool& full) {
          stop = false;
          full = true;
          if (ds_row) {
            const int u0 = qt * kQT;
            const int tq_first = static_cast<int>(block_token(a.order, a.S, a.P, i, u0));
            const int tq_last =
                static_cast<int>(block_token(a.order, a.S, a.P, i, min(u0 + kQT, Lb) - 1));
            stop = ds_row[tq_first] > k_last;
            full = k_last <= tq_first && ds_row[tq_last] <= k_first;
          }
        };
        if (!per_dev) {
          for (int base = qt0; base <= qt1 && ok; base += 32) {
            bool stop = false, full = true;
            if (base + lane <= qt1) flags(base + lane, stop, full);
            const unsigned stops = __ballot_sync(0xffffffffu, stop);
            const unsigned fulls = __ballot_sync(0xffffffffu, full);
            int cnt = min(32, qt1 - base + 1);
            if (stops) cnt = min(cnt, __ffs(static_cast<int>(stops)) - 1);
            for (int e = 0; e < cnt && ok; ++e) ok = issue_tile(base + e, (fulls >> e) & 1u);
            if (stops) break;
          }
          continue;
        }
        // Per-device form: the walk is trimmed at its first tile past the
        // keys' documents and starts at a tile that depends on the key tile
        // -- otherwise the key tiles of a head walk the same query tiles in
        // step and reduce into the same dQ tile at once.
        int n_walk = qt1 - qt0 + 1;
        for (int base = qt0; base <= qt1; base += 32) {
          bool stop = false, full = true;
          if (base + lane <= qt1) flags(base + lane, stop, full);
          const unsigned stops = __ballot_sync(0xffffffffu, stop);
          if (stops) {
            n_walk = base + __ffs(static_cast<int>(stops)) - 1 - qt0;
            break;
          }
        }
        const int rot = n_walk > 0 ? kt % n_walk : 0;
        for (int base = 0; base < n_walk && ok; base += 32) {
          const int idx = base + lane;
          bool stop = false, full = true;
          if (idx < n_walk) flags(qt0 + (idx + rot) % n_walk, stop, full);
          const unsigned fulls = __ballot_sync(0xffffffffu, full);
          const int cnt = min(32, n_walk - base);
          for (int e = 0; e < cnt && ok; ++e)
            ok = issue_tile(qt0 + (base + e + rot) % n_walk, (fulls >> e) & 1u);
        }
      }
    }
    if (ok) {  // end of the list
      const int slot = n % kQSlots;
      if (wait_warp(smem_u32(&q_empty[slot]), ((n / kQSlots) & 1) ^ 1, abort_flag, a.err,
                    kErrBwdKvEmpty)) {
        ended = true;
        if (lane == 0) {
          cols[slot].info = kInfoEnd;
          mbar_arrive(smem_u32(&q_full[slot]));
        }
      }
    }
    // copies still in flight land before the CTA can exit: K/V, the last dO,
    // the last Q tile, and the one before it unless the end marker's wait
    // for its slot already saw it consumed
    if (lane == 0) {
      mbar_wait(smem_u32(&kv_full), 0, abort_flag, a.err, kErrBwdDrain);
      if (n_do > 0)
        mbar_wait(smem_u32(&do_full), (n_do - 1) & 1, abort_flag, a.err, kErrBwdDrain);
      for (int m = n - 1; m >= 0 && m > n - 1 - (ended ? 1 : kQSlots); --m)
        mbar_wait(smem_u32(&q_full[m % kQSlots]), (m / kQSlots) & 1, abort_flag, a.err,
                  kErrBwdDrain);
    }
    __syncwarp();
  } else if (warp == kFMma) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint64_t dk0 = smem_desc_sw128(sk, 16, 1024), dv0 = smem_desc_sw128(sv, 16, 1024);
      const uint64_t dkq = smem_desc_sw128(sq, 16, 1024);          // K-major Q views
      const uint64_t dqmn = smem_desc_sw128(sq, kHalfBytes, 1024);  // MN-major Q views
      const uint64_t ddo = smem_desc_sw128(sdo, 16, 1024);          // K-major dO
      const uint64_t ddomn = smem_desc_sw128(sdo, kHalfBytes, 1024);
      const uint64_t dds = smem_desc_sw128(sds, 16, 1024);            // dS^T, K-major
      const uint64_t ddsmn = smem_desc_sw128(sds, kHalfBytes, 1024);  // dS, MN-major
      const uint64_t dkmn = smem_desc_sw128(sk, kHalfBytes, 1024);    // K, MN-major
      auto tile_info = [&](int t) -> int {
        const int slot = t % kQSlots;
        if (!wait_ready(smem_u32(&q_full[slot]), (t / kQSlots) & 1, abort_flag, a.err,
                        kErrBwdQFull))
          return -1;
        return cols[slot].info;
      };
      // S^T = K Q^T for tile t
      auto issue_s = [&](int t) {
        tc_fence_after();
        const uint64_t qb = dkq + (((t % kQSlots) * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(tmem, kmaj_desc(dk0, kk), kmaj_desc(qb, kk), kIdescKmaj, kk > 0 ? 1u : 0u);
      };
      // dP^T = V dO^T for tile t (its dO has landed), then publish S^T, dP^T
      auto issue_dp = [&]() {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(tmem + cdP, kmaj_desc(dv0, kk), kmaj_desc(ddo, kk), kIdescKmaj, kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&s_full));
      };
      auto issue_dv = [&](int t, int h) {
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = h * 4 + k4;  // 16-query step within the tile
          mma_ts(tmem + cdV, tmem + kk * 8, ddomn + ((kk * 16 * 128) >> 4), kIdescBmn,
                 (t > 0 || kk > 0) ? 1u : 0u);
        }
      };
      auto issue_dk = [&](int t, int h) {
        const uint64_t qb = dqmn + (((t % kQSlots) * kTileBytes) >> 4);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = h * 4 + k4;
          mma_ss(tmem + cdK, kmaj_desc(dds, kk), qb + ((kk * 16 * 128) >> 4), kIdescBmn,
                 (t > 0 || kk > 0) ? 1u : 0u);
        }
      };
      // dQ_tile = dS K over the 128 keys (16 per step)
      auto issue_dq = [&]() {
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_ss(tmem + cdQ, ddsmn + ((kk * 16 * 128) >> 4), dkmn + ((kk * 16 * 128) >> 4),
                 kIdescAmnBmn, kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&dq_full));
      };
      bool ok = mbar_wait(smem_u32(&kv_full), 0, abort_flag, a.err, kErrBwdKvFull);
      int cur = ok ? tile_info(0) : -1;
      if (cur > 0) {
        issue_s(0);
        if (wait_ready(smem_u32(&do_full), 0, abort_flag, a.err, kErrBwdQFull))
          issue_dp();
        else
          cur = -1;
      }
      for (int t = 0; cur > 0; ++t) {
        if (!mbar_wait(smem_u32(&half_full[0]), t & 1, abort_flag, a.err, kErrBwdDsFull)) break;
        tc_fence_after();
        issue_dv(t, 0);
        issue_dk(t, 0);
        if (!mbar_wait(smem_u32(&half_full[1]), t & 1, abort_flag, a.err, kErrBwdDsFull)) break;
        tc_fence_after();
        issue_dv(t, 1);
        mma_commit(smem_u32(&do_empty));  // dO_t consumed
        issue_dk(t, 1);
        issue_dq();  // Q_t's slot is released by the elementwise warps (dQ staging)
        const int nxt = tile_info(t + 1);
        if (nxt > 0) {
          issue_s(t + 1);
          if (!wait_ready(smem_u32(&dq_free), t & 1, abort_flag, a.err, kErrBwdSFree) ||
              !wait_ready(smem_u32(&do_full), (t + 1) & 1, abort_flag, a.err, kErrBwdQFull))
            break;
          issue_dp();
        }
        cur = nxt;
      }
      mma_commit(smem_u32(&dkv_full));
      mma_commit(smem_u32(&done));
      mbar_wait(smem_u32(&done), 0, abort_flag, a.err, kErrBwdDrain);
    }
    __syncwarp();
  } else if (warp == kFReducer) {
    // ------------------------------------------------------ dQ reductions
    if (lane == 0) {
      for (int t = 0;; ++t) {
        const int slot = t % kQSlots;
        // Q_t's column data stays put until this thread releases the slot
        if (!mbar_wait(smem_u32(&q_full[slot]), (t / kQSlots) & 1, abort_flag, a.err,
                       kErrBwdQFull))
          break;
        const ColData& cd = cols[slot];
        if (cd.info == kInfoEnd) break;
        const long long bhq = static_cast<long long>(b) * a.Hq + cd.h;
        float* blk = dq_acc + blk_index(bhq, P_arr, a.Lbp, per_dev ? 0 : cd.i, cd.u0) * kD;
        if (!mbar_wait(smem_u32(&stage_full), t & 1, abort_flag, a.err, kErrBwdOut)) break;
        // the dS^T half first: the next tile's dS^T stores need that buffer
        // soonest; Q_t's slot is needed again only for Q_{t+2}
        bulk_reduce_add_f32(blk + kTileBytes / 4, sds, kTileBytes);
        bulk_commit_group();
        bulk_reduce_add_f32(blk, sq + slot * kTileBytes, kTileBytes);
        bulk_commit_group();
        bulk_wait_group_read<1>();
        mbar_arrive(smem_u32(&stage_free));
        bulk_wait_group_read0();
        mbar_arrive(smem_u32(&q_empty[slot]));
      }
      bulk_wait_group0();  // the last reductions are complete
    }
    __syncwarp();
  } else {
    // --------------------------------------------------- elementwise warps
    const int r = threadIdx.x;  // TMEM lane: key row of S^T / dP^T, query row of dQ_tile
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int w = w0 + r;
    const bool key_live = w < Lb;
    const int ktok = key_live ? static_cast<int>(block_token(a.order, a.S, a.P, j, w)) : -1;
    const float sl2 = a.scale * kLog2e;
    const uint32_t ds_row_addr = sds + r * 128;
    const uint32_t swz = static_cast<uint32_t>(r & 7);
    int t = 0;
    bool ok = true;
    for (;; ++t) {
      const int slot = t % kQSlots;
      if (!wait_warp(smem_u32(&q_full[slot]), (t / kQSlots) & 1, abort_flag, a.err,
                     kErrBwdQFull)) {
        ok = false;
        break;
      }
      const ColData& cd = cols[slot];
      const int info = cd.info;
      if (info == kInfoEnd) break;
      const int ti = cd.i, tu0 = cd.u0;
      if (!wait_warp(smem_u32(&s_full), t & 1, abort_flag, a.err, kErrBwdSFull)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool full = info == kInfoFull;
      int c_min = 0;
      if (!full) {
        c_min = a.order == SP_ORDER_STRIPED ? -floor_div_i(-(ktok - ti), a.P) - tu0
                                            : ktok - (ti * Lb + tu0);
      }
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t sx[64], px[64];
        tmem_ld32_at(tmem + lane_base + h * 64, sx, 0);
        tmem_ld32_at(tmem + lane_base + h * 64 + 32, sx, 32);
        tmem_ld32_at(tmem + lane_base + cdP + h * 64, px, 0);
        tmem_ld32_at(tmem + lane_base + cdP + h * 64 + 32, px, 32);
        tmem_wait_ld();
        if (!full) {
#pragma unroll
          for (int c4 = 0; c4 < 64; c4 += 4) {
            const int c = h * 64 + c4;
            const int4 lo = *reinterpret_cast<const int4*>(&cd.lo[c]);
            if (c < c_min || lo.x > ktok) sx[c4] = 0xff800000u;
            if (c + 1 < c_min || lo.y > ktok) sx[c4 + 1] = 0xff800000u;
            if (c + 2 < c_min || lo.z > ktok) sx[c4 + 2] = 0xff800000u;
            if (c + 3 < c_min || lo.w > ktok) sx[c4 + 3] = 0xff800000u;
          }
        }
        uint32_t pk[32], dk[32];
#pragma unroll
        for (int c4 = 0; c4 < 64; c4 += 4) {
          const int c = h * 64 + c4;
          const float4 l2 = *reinterpret_cast<const float4*>(&cd.lse2[c]);
          const float4 D = *reinterpret_cast<const float4*>(&cd.D[c]);
          float x0, x1, x2, x3;
          ffma2(x0, x1, __uint_as_float(sx[c4]), __uint_as_float(sx[c4 + 1]), sl2, sl2, -l2.x,
                -l2.y);
          ffma2(x2, x3, __uint_as_float(sx[c4 + 2]), __uint_as_float(sx[c4 + 3]), sl2, sl2, -l2.z,
                -l2.w);
          const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
          float d0, d1, d2, d3;
          fadd2(d0, d1, __uint_as_float(px[c4]), __uint_as_float(px[c4 + 1]), -D.x, -D.y);
          fadd2(d2, d3, __uint_as_float(px[c4 + 2]), __uint_as_float(px[c4 + 3]), -D.z, -D.w);
          fmul2(d0, d1, d0, d1, p0, p1);
          fmul2(d2, d3, d2, d3, p2, p3);
          pk[c4 >> 1] = pack_bf16(p0, p1);
          pk[(c4 >> 1) + 1] = pack_bf16(p2, p3);
          dk[c4 >> 1] = pack_bf16(d0, d1);
          dk[(c4 >> 1) + 1] = pack_bf16(d2, d3);
        }
        // P^T of half h as 32 bf16-pair columns (S^T columns [32h, 32h + 32)
        // were read in half 0); dS^T row r, queries [64h, 64h + 64): one
        // 128-byte row of the half's swizzled 16 KiB block
        tmem_st32(tmem + lane_base + h * 32, pk);
        if (h == 0 && t > 0) {
          // the dS^T buffer held half of dQ_{t-1} until the TMA read it
          if (!wait_warp(smem_u32(&stage_free), (t - 1) & 1, abort_flag, a.err, kErrBwdOut)) {
            ok = false;
            break;
          }
        }
        const uint32_t row = ds_row_addr + h * kHalfBytes;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          sts128(row + ((static_cast<uint32_t>(c) ^ swz) << 4), dk[4 * c], dk[4 * c + 1],
                 dk[4 * c + 2], dk[4 * c + 3]);
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&half_full[h]));
      }
      if (!ok) break;
      // dQ_tile: this thread's query row, 128 fp32 columns
      if (!wait_warp(smem_u32(&dq_full), t & 1, abort_flag, a.err, kErrBwdOut)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t x[128];
      tmem_ld32_at(tmem + lane_base + cdQ, x, 0);
      tmem_ld32_at(tmem + lane_base + cdQ + 32, x, 32);
      tmem_ld32_at(tmem + lane_base + cdQ + 64, x, 64);
      tmem_ld32_at(tmem + lane_base + cdQ + 96, x, 96);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(smem_u32(&dq_free));
      // stage: column quads 0..15 in Q_t's slot, 16..31 in the dS^T buffer
      // (free: every product that read them is complete)
      const uint32_t stage0 = sq + slot * kTileBytes + r * 16, stage1 = sds + r * 16;
#pragma unroll
      for (int q4 = 0; q4 < 32; ++q4)
        sts128((q4 < 16 ? stage0 : stage1) + (q4 & 15) * (kQT * 16), x[4 * q4], x[4 * q4 + 1],
               x[4 * q4 + 2], x[4 * q4 + 3]);
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&stage_full));
    }
    // epilogue: dK * scale and dV, rows of key token ktok (bf16), or in the
    // per-device form added to the float32 accumulators at local row w
    const bool have = t > 0 && ok;
    if (have && !wait_warp(smem_u32(&dkv_full), 0, abort_flag, a.err, kErrBwdOut)) ok = false;
    tc_fence_after();
    const long long orow =
        ((static_cast<long long>(b) * a.S + (key_live ? ktok : 0)) * a.Hkv + hk) * kD;
    const long long lrow =
        ((static_cast<long long>(b) * Lb + (key_live ? w : 0)) * a.Hkv + hk) * kD;
#pragma unroll 1
    for (int m = 0; m < 2; ++m) {
      const float mul = m == 0 ? a.scale : 1.f;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t x[32];
        if (have && ok) {
          tmem_ld32(tmem + lane_base + (m == 0 ? cdK : cdV) + c * 32, x);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = 0u;
        }
        if (per_dev) {
          if (key_live && have && ok) {
            float* acc = (m == 0 ? bb.dk_acc : bb.dv_acc) + lrow + c * 32;
#pragma unroll
            for (int e = 0; e < 8; ++e)
              red_add_v4(acc + 4 * e, __uint_as_float(x[4 * e]) * mul,
                         __uint_as_float(x[4 * e + 1]) * mul, __uint_as_float(x[4 * e + 2]) * mul,
                         __uint_as_float(x[4 * e + 3]) * mul);
          }
          continue;
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16(__uint_as_float(x[2 * e]) * mul, __uint_as_float(x[2 * e + 1]) * mul);
        if (key_live) {
          uint4* dst = reinterpret_cast<uint4*>(
              static_cast<__nv_bfloat16*>(m == 0 ? a.dk : a.dv) + orow);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[c * 4 + e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kFMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One 64 KiB accumulator block ([column quad 32][row 128][4] floats: rows
// u0 .. u0 + 127 of one block and head) read into shared memory half a block
// (16 quads) at a time, so that both sides are contiguous: the reads in the
// block's own order, the writes along each row.  Padded to 129 rows per quad
// so that the 16 lanes reading one row from 16 quads hit distinct banks.
constexpr int kQuadsPerPass = 16;
struct AccHalf {
  float4 v[kQuadsPerPass][kQT + 1];
};

__device__ __forceinline__ void load_acc_half(AccHalf& sm, const float4* __restrict__ blk,
                                              int pass) {
  const float4* src = blk + pass * kQuadsPerPass * kQT;
#pragma unroll 4
  for (int e = threadIdx.x; e < kQuadsPerPass * kQT; e += 256)
    sm.v[e / kQT][e % kQT] = src[e];
}

// dq = scale * (the fp32 sums), bf16, in [B][S][Hq][d].  One CTA per
// accumulator block; per pass a half-warp writes 64 columns (128 bytes) of
// one row.
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float4* __restrict__ acc,
                                                             __nv_bfloat16* dq, int S, int Hq,
                                                             int P, int Lbp, int order,
                                                             float scale) {
  __shared__ AccHalf sm;
  const int tiles = Lbp / kQT;
  const long long blk = blockIdx.x;  // ((b * Hq + h) * P + i) * tiles + tile
  const int tile = static_cast<int>(blk % tiles);
  const long long bhp = blk / tiles;
  const int i = static_cast<int>(bhp % P);
  const long long bh = bhp / P;
  const int h = static_cast<int>(bh % Hq);
  const long long b = bh / Hq;
  const int Lb = S / P;
  const int l16 = threadIdx.x & 15, row0 = threadIdx.x >> 4;  // 16 rows per sweep
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    if (pass) __syncthreads();
    load_acc_half(sm, acc + blk * (kQT * kD / 4), pass);
    __syncthreads();
#pragma unroll 1
    for (int r = row0; r < kQT; r += 16) {
      const int u = tile * kQT + r;
      if (u >= Lb) break;
      const long long t = block_token(order, S, P, i, u);
      const float4 x = sm.v[l16][r];
      uint2* dst = reinterpret_cast<uint2*>(dq + ((b * S + t) * Hq + h) * kD +
                                            (pass * kQuadsPerPass + l16) * 4);
      *dst = make_uint2(pack_bf16(x.x * scale, x.y * scale), pack_bf16(x.z * scale, x.w * scale));
    }
  }
}

// Per-device form: dq_acc[b][u][h][:] += scale * (the fp32 sums of block i),
// float32, [B][S/P][Hq][d]; the blocked accumulator holds one block.  Same
// staging as bwd_dq_convert_kernel; a half-warp updates 64 columns (256
// bytes) of one row.
__global__ void __launch_bounds__(256) bwd_dq_add_kernel(const float4* __restrict__ acc,
                                                         float4* dq_acc, int Lb, int Hq, int Lbp,
                                                         float scale) {
  __shared__ AccHalf sm;
  const int tiles = Lbp / kQT;
  const long long blk = blockIdx.x;  // (b * Hq + h) * tiles + tile
  const int tile = static_cast<int>(blk % tiles);
  const long long bh = blk / tiles;
  const int h = static_cast<int>(bh % Hq);
  const long long b = bh / Hq;
  const int l16 = threadIdx.x & 15, row0 = threadIdx.x >> 4;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    if (pass) __syncthreads();
    load_acc_half(sm, acc + blk * (kQT * kD / 4), pass);
    __syncthreads();
#pragma unroll 1
    for (int r = row0; r < kQT; r += 16) {
      const int u = tile * kQT + r;
      if (u >= Lb) break;
      const float4 x = sm.v[l16][r];
      float4* dst = dq_acc + ((b * Lb + u) * Hq + h) * (kD / 4) + pass * kQuadsPerPass + l16;
      float4 y = *dst;
      y.x += x.x * scale;
      y.y += x.y * scale;
      y.z += x.z * scale;
      y.w += x.w * scale;
      *dst = y;
    }
  }
}

// Tensor maps and the prep kernel, shared by both backward forms.
bool launch_prep(const BwdArgs& a, BwdMaps& tm, cudaStream_t st) {
  if (!tmap::make_map(&tm.q, a.q, a.B, a.S, a.Hq, a.P, a.order) ||
      !tmap::make_map(&tm.dout, a.dout, a.B, a.S, a.Hq, a.P, a.order) ||
      !tmap::make_map(&tm.k, a.k, a.B, a.S, a.Hkv, a.P, a.order) ||
      !tmap::make_map(&tm.v, a.v, a.B, a.S, a.Hkv, a.P, a.order))
    return false;
  const int Lb = a.S / a.P;
  PrepArgs pa;
  pa.out = static_cast<const uint4*>(a.out);
  pa.dout = static_cast<const uint4*>(a.dout);
  pa.lse = a.lse;
  pa.doc_start = a.doc_start;
  pa.D_blk = a.D_blk;
  pa.lse2_blk = a.lse2_blk;
  pa.lo_blk = a.lo_blk;
  pa.rows = static_cast<long long>(a.B) * a.S * a.Hq;
  pa.nA = (pa.rows * 16 + 31) / 32 * 32;
  pa.nB = static_cast<long long>(a.B) * a.Hq * a.P * (a.Lbp - Lb);
  pa.nC = a.doc_start ? static_cast<long long>(a.pos_rows) * a.P * a.Lbp : 0;
  pa.S = a.S;
  pa.H = a.Hq;
  pa.P = a.P;
  pa.Lbp = a.Lbp;
  pa.order = a.order;
  pa.lo_S = a.S;
  pa.lo_P = a.P;
  pa.lo_order = a.order;
  pa.lo_block = -1;
  const long long n_prep = pa.nA + pa.nB + pa.nC;
  bwd_prep_kernel<<<static_cast<unsigned>((n_prep + 255) / 256), 256, 0, st>>>(pa);
  return true;
}

}  // namespace

// prep, then dQ and dK/dV (independent of each other) on the tensor cores.
int launch_attn_bwd_bf16(const BwdArgs& a, cudaStream_t st) {
  BwdMaps tm;  // 128-row boxes for both kernels
  if (!launch_prep(a, tm, st)) return -1;
  const int n_tiles = (a.S / a.P + kT - 1) / kT;
  const int dq_smem = kQSmemBytes + 1024, kv_smem = kKvSmemBytes + 1024;
  if (cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dq_smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kv_smem) != cudaSuccess)
    return -1;
  const unsigned n_q = static_cast<unsigned>(a.P) * n_tiles * a.B * a.Hq;
  bwd_dq_kernel<<<n_q, kQThreads, dq_smem, st>>>(tm, a, n_tiles);
  const unsigned n_kv = static_cast<unsigned>(a.P) * n_tiles * a.B * a.Hkv;
  bwd_dkdv_kernel<<<n_kv, kKvThreads, kv_smem, st>>>(tm, a, n_tiles);
  return cudaGetLastError() == cudaSuccess ? 3 : -1;
}

// prep, the fused kernel into a zeroed fp32 dQ accumulator
// (B * Hq * P * Lbp * 128 floats), then dq from the accumulator.
int launch_attn_bwd_bf16_fused(const BwdArgs& a, float* dq_acc, cudaStream_t st) {
  BwdMaps tm;
  const size_t acc_bytes =
      static_cast<size_t>(a.B) * a.Hq * a.P * a.Lbp * kD * sizeof(float);
  if (cudaMemsetAsync(dq_acc, 0, acc_bytes, st) != cudaSuccess) return -1;
  if (!launch_prep(a, tm, st)) return -1;
  const int n_tiles = (a.S / a.P + kT - 1) / kT;
  const int f_smem = kFSmemBytes + 1024;
  if (cudaFuncSetAttribute(bwd_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           f_smem) != cudaSuccess)
    return -1;
  const unsigned n_kv = static_cast<unsigned>(a.P) * n_tiles * a.B * a.Hkv;
  bwd_fused_kernel<<<n_kv, kFThreads, f_smem, st>>>(tm, a, n_tiles, dq_acc,
                                                     BwdBlock{-1, -1, nullptr, nullptr});
  const unsigned n_blk = static_cast<unsigned>(static_cast<long long>(a.B) * a.Hq * a.P *
                                               (a.Lbp / kQT));
  bwd_dq_convert_kernel<<<n_blk, 256, 0, st>>>(reinterpret_cast<const float4*>(dq_acc),
                                                static_cast<__nv_bfloat16*>(a.dq), a.S, a.Hq,
                                                a.P, a.Lbp, a.order, a.scale);
  return cudaGetLastError() == cudaSuccess ? 3 : -1;
}

// Per-device form: prep of block i's rows, the fused kernel over key/value
// block j's key tiles walking block i's query tiles, then dq_acc += the
// block's dQ sums.  a.q, a.out, a.dout, a.lse hold block i ([B][S/P][Hq][d],
// lse [B][Hq][S/P]); a.k, a.v block j; a.S, a.P, a.order the whole sequence;
// dq_blocked: B * Hq * Lbp * 128 floats of scratch.
int launch_attn_bwd_bf16_block(const BwdArgs& a, int qb, int kb, float* dq_blocked,
                               float* dq_acc, float* dk_acc, float* dv_acc, cudaStream_t st) {
  const int Lb = a.S / a.P;
  BwdMaps tm;  // one block of Lb rows in each map
  if (!tmap::make_map(&tm.q, a.q, a.B, Lb, a.Hq, 1, SP_ORDER_CONTIGUOUS) ||
      !tmap::make_map(&tm.dout, a.dout, a.B, Lb, a.Hq, 1, SP_ORDER_CONTIGUOUS) ||
      !tmap::make_map(&tm.k, a.k, a.B, Lb, a.Hkv, 1, SP_ORDER_CONTIGUOUS) ||
      !tmap::make_map(&tm.v, a.v, a.B, Lb, a.Hkv, 1, SP_ORDER_CONTIGUOUS))
    return -1;
  PrepArgs pa;
  pa.out = static_cast<const uint4*>(a.out);
  pa.dout = static_cast<const uint4*>(a.dout);
  pa.lse = a.lse;
  pa.doc_start = a.doc_start;
  pa.D_blk = a.D_blk;
  pa.lse2_blk = a.lse2_blk;
  pa.lo_blk = a.lo_blk;
  pa.rows = static_cast<long long>(a.B) * Lb * a.Hq;
  pa.nA = (pa.rows * 16 + 31) / 32 * 32;
  pa.nB = static_cast<long long>(a.B) * a.Hq * (a.Lbp - Lb);
  pa.nC = a.doc_start ? static_cast<long long>(a.pos_rows) * a.Lbp : 0;
  pa.S = Lb;  // the rows of one block, in local order
  pa.H = a.Hq;
  pa.P = 1;
  pa.Lbp = a.Lbp;
  pa.order = SP_ORDER_CONTIGUOUS;
  pa.lo_S = a.S;
  pa.lo_P = a.P;
  pa.lo_order = a.order;
  pa.lo_block = qb;
  const long long n_prep = pa.nA + pa.nB + pa.nC;
  bwd_prep_kernel<<<static_cast<unsigned>((n_prep + 255) / 256), 256, 0, st>>>(pa);
  const size_t acc_bytes = static_cast<size_t>(a.B) * a.Hq * a.Lbp * kD * sizeof(float);
  if (cudaMemsetAsync(dq_blocked, 0, acc_bytes, st) != cudaSuccess) return -1;
  const int n_tiles = (Lb + kT - 1) / kT;
  const int f_smem = kFSmemBytes + 1024;
  if (cudaFuncSetAttribute(bwd_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           f_smem) != cudaSuccess)
    return -1;
  const unsigned n_cta = static_cast<unsigned>(n_tiles) * a.B * a.Hq;  // one per query head
  bwd_fused_kernel<<<n_cta, kFThreads, f_smem, st>>>(tm, a, n_tiles, dq_blocked,
                                                      BwdBlock{qb, kb, dk_acc, dv_acc});
  const unsigned n_blk =
      static_cast<unsigned>(static_cast<long long>(a.B) * a.Hq * (a.Lbp / kQT));
  bwd_dq_add_kernel<<<n_blk, 256, 0, st>>>(reinterpret_cast<const float4*>(dq_blocked),
                                            reinterpret_cast<float4*>(dq_acc), Lb, a.Hq, a.Lbp,
                                            a.scale);
  return cudaGetLastError() == cudaSuccess ? 3 : -1;
}

}  // namespace sp
