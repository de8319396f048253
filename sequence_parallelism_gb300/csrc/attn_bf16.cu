// attn_bf16.cu -- blockwise ring attention on the sm_103a tensor cores.
//
// Method ("Ring Attention", "Cómo funciona la atención en anillo"): the
// sequence is cut into P blocks; query block i stays resident while the
// key/value blocks arrive in ring order j = (i - s) mod P; each arrival is
// folded into a running max m, a running sum of exponentiated scores l and a
// running weighted-value sum O (the cumulative softmax, with the running
// maximum subtracted as production kernels do), and O / l is written at the
// end.  The causal mask comes from O(n) position_ids ("Ulysses SPで100万
// トークン学習", section 3) through the doc_start array: query t may attend
// key j iff doc_start[t] <= j <= t, so each score row has one contiguous
// allowed interval per key tile and fully masked tiles are never visited.
//
// One CTA = one (batch, q head, query block i, 256 query rows) and keeps its
// two 128-row Q tiles in shared memory for the whole ring.  Warp roles:
//   warps 0-3   softmax group 0: one thread per row of Q tile 0
//   warps 4-7   softmax group 1: one thread per row of Q tile 1
//   warp  8     TMA producer: Q once, then K_t, V_t into a 4-slot ring
//   warp  9     TMEM owner + single-thread tcgen05.mma issuer
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128) S0   [128,256) S1   [256,384) O0   [384,512) O1
// P (bf16, two per column) overwrites the first 64 columns of its S tile and
// feeds the PV product straight from TMEM.  The MMA issue order
//   S0(t+1) after PV0(t), PV1(t) between, S1(t+1) after PV1(t)
// keeps the tensor pipe busy with one Q tile while the other tile's softmax
// runs.  O is rescaled in TMEM only when a row's max grows by more than
// 2^8 (exact after the final division; bf16 P stays far from overflow).
//
// Per-device form (what one device of a real ring holds): a fixed query
// block whose rows live in a block tensor, and optionally a single key/value
// block tensor for one ring step; tensor maps over those block tensors, masks
// and doc_start in global token indices (AttnArgs::q_block, ::kv_block).
//
// Operand layouts (all 128-byte swizzled, as TMA writes them):
//   Q, K tile: [2 halves of d][128 rows][64 elements]  K-major for S = Q K^T
//   V tile   : [2 halves of d][128 keys][64 elements]  MN-major B for O += P V
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
constexpr int kBM = 128;              // rows per Q tile
constexpr int kBN = 128;              // keys per K/V tile
constexpr int kQTiles = 2;            // Q tiles per CTA
constexpr int kRowsPerCta = kBM * kQTiles;
constexpr int kSlots = 4;             // K/V ring depth
constexpr int kTileBytes = kBN * kD * 2;          // 32 KiB
constexpr int kHalfBytes = kTileBytes / 2;        // one 64-column half
constexpr int kStageBytes = kBM * 64 * 2;    // one 64-column half of an output tile
constexpr int kSmemBytes = (kQTiles + kSlots) * kTileBytes + kQTiles * kStageBytes;
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kD, true);

// error codes recorded in the workspace error word (which wait gave up)
enum : int {
  kErrQFull = 0x101, kErrKvEmpty = 0x102, kErrKvFull = 0x103, kErrSFull = 0x104,
  kErrPFull = 0x105, kErrOFull = 0x106, kErrDrain = 0x107, kErrUnit = 0x108,
  kErrQEmpty = 0x109, kErrOFree = 0x10a, kErrAccFull = 0x10b
};

struct Tmaps {
  CUtensorMap q, k, v, o;
};

// Token indices fit in int (S is an int), so the schedule works in 32 bits.
__device__ __forceinline__ int floor_div(int a, int b) {
  return a >= 0 ? a / b : -((-a + b - 1) / b);
}

// The part of the ring schedule every role must agree on.  Tiles are
// numbered in visiting order (ring step, then key tile); a CTA processes the
// window [t_lo, t_hi) of that sequence (the whole sequence unless the item is
// split across several CTAs).
struct Schedule {
  int i, P, Lb, S, order, step_begin, step_end;
  int hull_lo, hull_hi;  // key-token interval any row of the CTA may use
  int t_lo, t_hi;

  // KV tiles [kt0, kt1] of block j that intersect the hull (kt1 < kt0: none)
  __device__ __forceinline__ void tiles(int s, int& j, int& kt0, int& kt1) const {
    j = ((i - s) % P + P) % P;
    int w_lo, w_hi;
    if (order == SP_ORDER_STRIPED) {
      w_lo = -floor_div(-(hull_lo - j), P);  // ceil((lo - j) / P)
      w_hi = floor_div(hull_hi - j, P);
    } else {
      const int base = j * Lb;
      w_lo = hull_lo - base;
      w_hi = hull_hi - base;
    }
    if (w_lo < 0) w_lo = 0;
    if (w_hi > Lb - 1) w_hi = Lb - 1;
    if (w_lo > w_hi) {
      kt0 = 0;
      kt1 = -1;
      return;
    }
    kt0 = static_cast<int>(w_lo / kBN);
    kt1 = static_cast<int>(w_hi / kBN);
  }

  // total number of tiles in the item's sequence
  __device__ __forceinline__ int total() const {
    int n = 0;
    for (int s = step_begin; s < step_end; ++s) {
      int j, a, b;
      tiles(s, j, a, b);
      n += b - a + 1;
    }
    return n;
  }
};

// Work item of linear index L: heavy query positions first (the causal work
// of a query block grows with its position), heads innermost so that the
// query heads sharing a key/value head run side by side.
// With a fixed query block (per-device form) only that block's items exist.
__device__ __forceinline__ void item_coords(int L, const AttnArgs& a, int n_pairs, int& b, int& hq,
                                            int& i, int& pair) {
  const int BH = a.B * a.Hq;
  const int pos = L / BH;
  const int bh = L % BH;
  b = bh / a.Hq;
  hq = bh % a.Hq;
  const int nqb = a.q_block >= 0 ? 1 : a.P;
  const int rev = nqb * n_pairs - 1 - pos;
  i = a.q_block >= 0 ? a.q_block : rev / n_pairs;
  pair = rev % n_pairs;
}

struct __align__(8) Barriers {
  uint64_t unit_full[2];   // producer -> all: work-unit index published
  uint64_t unit_empty[2];  // all -> producer: work-unit index read
  uint64_t q_full;         // Q tiles of a unit landed
  uint64_t q_empty;        // last S MMAs of a unit done: Q may be replaced
  uint64_t kv_full[kSlots];
  uint64_t kv_empty[kSlots];
  uint64_t s_full[kQTiles];
  uint64_t p_full[kQTiles];
  uint64_t o_full[kQTiles];
  uint64_t o_free[kQTiles];  // epilogue read O: the next unit may overwrite it
  uint64_t acc_full[kQTiles];  // accumulate form: a half of the running output landed
  uint64_t done;
};

// Everything a role derives from a work-unit index w: units [0, n_whole) are
// whole items, the units after them are split_k pieces (tile windows) of each
// remaining item, whose fp32 partials merge_split_kernel combines.
struct Unit {
  int w;  // unit index; -1: no more work
  int b, hq, i, kvh, u0, split, sidx;
  int n_tiles;
  Schedule sch;
};

__device__ __forceinline__ void make_unit(int w, const AttnArgs& a, int n_pairs, int n_whole,
                                          int split_k, Unit& U) {
  const bool whole = w < n_whole;
  U.w = w;
  U.split = whole ? 1 : split_k;
  U.sidx = whole ? 0 : w - n_whole;
  int pair;
  item_coords(whole ? w : n_whole + U.sidx / split_k, a, n_pairs, U.b, U.hq, U.i, pair);
  const int piece = whole ? 0 : U.sidx % split_k;
  U.kvh = U.hq / (a.Hq / a.Hkv);
  const int Lb = a.S / a.P;
  U.u0 = pair * kRowsPerCta;
  Schedule& sch = U.sch;
  sch.i = U.i;
  sch.P = a.P;
  sch.Lb = Lb;
  sch.S = a.S;
  sch.order = a.order;
  sch.step_begin = a.step_begin;
  sch.step_end = a.step_end;
  const int u_last = min(U.u0 + kRowsPerCta, Lb) - 1;
  const int t_first = static_cast<int>(block_token(a.order, a.S, a.P, U.i, U.u0));
  const int t_last = static_cast<int>(block_token(a.order, a.S, a.P, U.i, u_last));
  if (a.doc_start) {
    sch.hull_lo = a.doc_start[static_cast<long long>(U.b % a.pos_rows) * a.S + t_first];
    sch.hull_hi = t_last;
  } else {
    sch.hull_lo = 0;
    sch.hull_hi = a.S - 1;
  }
  const int tot = sch.total();
  sch.t_lo = static_cast<int>(static_cast<long long>(tot) * piece / U.split);
  sch.t_hi = static_cast<int>(static_cast<long long>(tot) * (piece + 1) / U.split);
  U.n_tiles = sch.t_hi - sch.t_lo;
}

// Persistent: each CTA runs work units until the counter passes n_work; the
// producer fetches the next unit (the first one is blockIdx.x, the others
// come from an atomic counter, so units start in heavy-first order) and
// publishes its decoded description in a two-slot shared-memory mailbox that
// the other roles read in place (a slot is released at the end of the unit).  The next unit's Q is loaded as
// soon as the current unit's last S MMAs are done, and its first S MMAs run
// while the softmax warps are still in the current unit's epilogue.
//
// kAcc (per-device form, one ring step): out / lse hold a running result on
// entry, and the epilogue folds this step's partial into it by the
// log-sum-exp merge instead of writing the partial.  The running output
// tile comes in through the same swizzled stage the stores use (one TMA load
// per 64-column half); a unit without tiles leaves its rows untouched.
template <bool kAcc>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bf16_kernel(const __grid_constant__ Tmaps tm, AttnArgs a, float scale_log2, int n_pairs,
                     int n_whole, int split_k, int n_work, float* __restrict__ part_o,
                     float* __restrict__ part_lse) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ Unit units_s[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;

  // 1024-byte alignment for the 128-byte swizzle atoms
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_q = smem_u32(smem);                         // Q0, Q1
  const uint32_t smem_kv = smem_q + kQTiles * kTileBytes;         // ring slots
  const uint32_t smem_stage = smem_kv + kSlots * kTileBytes;      // output staging, per tile

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Lb = a.S / a.P;

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&bars.unit_full[x]), 1);
      mbar_init(smem_u32(&bars.unit_empty[x]), 1 + 2 * kBM);
    }
    mbar_init(smem_u32(&bars.q_full), 1);
    mbar_init(smem_u32(&bars.q_empty), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_u32(&bars.kv_full[s]), 1);
      mbar_init(smem_u32(&bars.kv_empty[s]), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(smem_u32(&bars.s_full[t]), 1);
      mbar_init(smem_u32(&bars.p_full[t]), kBM);
      mbar_init(smem_u32(&bars.o_full[t]), 1);
      mbar_init(smem_u32(&bars.o_free[t]), kBM);
      mbar_init(smem_u32(&bars.acc_full[t]), 1);
    }
    mbar_init(smem_u32(&bars.done), 1);
    abort_s = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  volatile int* abort_flag = &abort_s;

  // coordinates of local row u of block p in the 5-D tensor maps; a tensor
  // that holds a single block (per-device form) is mapped as one contiguous
  // block
  auto coord_rows = [&](int p, int u, int& c2, int& c3) {
    if (a.order == SP_ORDER_STRIPED) {
      c2 = p;
      c3 = u;
    } else {
      c2 = u;
      c3 = p;
    }
  };
  auto coord_q = [&](int p, int u, int& c2, int& c3) {
    if (a.q_block >= 0) {
      c2 = u;
      c3 = 0;
    } else {
      coord_rows(p, u, c2, c3);
    }
  };
  auto coord_kv = [&](int p, int u, int& c2, int& c3) {
    if (a.kv_block >= 0) {
      c2 = u;
      c3 = 0;
    } else {
      coord_rows(p, u, c2, c3);
    }
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm.q);
      prefetch_tmap(&tm.k);
      prefetch_tmap(&tm.v);
      int w = static_cast<int>(blockIdx.x) < n_work ? static_cast<int>(blockIdx.x) : -1;
      int n = 0;   // K/V load index over the CTA's life: K, V of each tile in turn
      int qn = 0;  // units with tiles so far (Q loads)
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        const int x = seq & 1;
        if (!mbar_wait(smem_u32(&bars.unit_empty[x]), ((seq >> 1) & 1) ^ 1, abort_flag, a.err,
                       kErrUnit))
          break;
        Unit& U = units_s[x];
        if (w >= 0)
          make_unit(w, a, n_pairs, n_whole, split_k, U);
        else
          U.w = -1;
        mbar_arrive(smem_u32(&bars.unit_full[x]));
        if (w < 0) break;
        if (U.n_tiles > 0) {
          // this unit's Q replaces the previous one's once its S MMAs are done
          if (!mbar_wait(smem_u32(&bars.q_empty), (qn & 1) ^ 1, abort_flag, a.err, kErrQEmpty))
            break;
          const uint32_t qf = smem_u32(&bars.q_full);
          mbar_arrive_expect_tx(qf, kQTiles * kTileBytes);
          for (int t = 0; t < kQTiles; ++t) {
            int c2, c3;
            coord_q(U.i, U.u0 + t * kBM, c2, c3);
            for (int half = 0; half < 2; ++half)
              tma_load_5d(smem_q + t * kTileBytes + half * kHalfBytes, &tm.q, qf, half * 64, U.hq,
                          c2, c3, U.b);
          }
          ++qn;
          int ft = 0;  // position in the item's tile sequence
          for (int s = a.step_begin; s < a.step_end && ok && ft < U.sch.t_hi; ++s) {
            int j, kt0, kt1;
            U.sch.tiles(s, j, kt0, kt1);
            for (int kt = kt0; kt <= kt1 && ok; ++kt, ++ft) {
              if (ft < U.sch.t_lo) continue;
              if (ft >= U.sch.t_hi) break;
              int c2, c3;
              coord_kv(j, kt * kBN, c2, c3);
              for (int kv = 0; kv < 2; ++kv, ++n) {
                const int slot = n % kSlots;
                const uint32_t parity = ((n / kSlots) & 1) ^ 1;
                if (!mbar_wait(smem_u32(&bars.kv_empty[slot]), parity, abort_flag, a.err,
                               kErrKvEmpty)) {
                  ok = false;
                  break;
                }
                const uint32_t full = smem_u32(&bars.kv_full[slot]);
                mbar_arrive_expect_tx(full, kTileBytes);
                const CUtensorMap* map = kv == 0 ? &tm.k : &tm.v;
                for (int half = 0; half < 2; ++half)
                  tma_load_5d(smem_kv + slot * kTileBytes + half * kHalfBytes, map, full,
                              half * 64, U.kvh, c2, c3, U.b);
              }
            }
          }
        }
        w = static_cast<int>(gridDim.x) + atomicAdd(a.counter, 1);
        if (w >= n_work) w = -1;
      }
      // drain: every copy this CTA started has landed before it may exit
      if (qn > 0) mbar_wait(smem_u32(&bars.q_full), (qn - 1) & 1, abort_flag, a.err, kErrDrain);
      for (int m = n - 1; m >= 0 && m >= n - kSlots; --m)
        mbar_wait(smem_u32(&bars.kv_full[m % kSlots]), (m / kSlots) & 1, abort_flag, a.err,
                  kErrDrain);
    }
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // Descriptors are built once; a k-step only adds its byte offset >> 4
      // to the start-address field (all addresses stay below 256 KiB, so the
      // 14-bit field never carries).
      const uint64_t dq0 = smem_desc_sw128(smem_q, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_kv, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_kv, kHalfBytes, 1024);
      // S_t = Q_t K^T over d = 128: 8 k-steps of 16, 32 bytes apart inside a
      // 128-byte swizzled row, the second 64 columns in the next half tile.
      auto issue_s = [&](int t, int load_idx) {
        const uint64_t qa = dq0 + ((t * kTileBytes) >> 4);
        const uint64_t kb = dk0 + (((load_idx % kSlots) * kTileBytes) >> 4);
        const uint32_t d = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
          mma_ss(d, qa + off, kb + off, kIdescQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars.s_full[t]));
      };
      // O_t (+)= P_t V: P from TMEM (8 columns = 16 keys per k-step), V
      // MN-major: 16 keys = 2 swizzle atoms of 8 rows (stride 1024 B), the
      // two 64-column halves of d 16 KiB apart.
      auto issue_pv = [&](int t, bool first, int slot) {
        const uint64_t vb = dv0 + ((slot * kTileBytes) >> 4);
        const uint32_t d = tmem + 256 + t * 128;
        const uint32_t pa = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(d, pa + kk * 8, vb + ((kk * 16 * 128) >> 4), kIdescPV,
                 (!first || kk > 0) ? 1u : 0u);
      };
      int n = 0;   // K/V load index (the producer's sequence)
      int it = 0;  // tiles over the CTA's life (s_full / p_full phases)
      int qn = 0;  // units with tiles so far
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        const int x = seq & 1;
        if (!mbar_wait(smem_u32(&bars.unit_full[x]), (seq >> 1) & 1, abort_flag, a.err, kErrUnit))
          break;
        const int nt = units_s[x].w < 0 ? -1 : units_s[x].n_tiles;
        mbar_arrive(smem_u32(&bars.unit_empty[x]));  // everything it needs is in nt
        if (nt < 0) break;
        if (nt == 0) continue;
        // first tile: S of both Q tiles as soon as Q and K_0 landed (the
        // previous unit's PVs, issued before, read P from the same columns
        // and complete first: tcgen05 MMAs of one thread run in order)
        if (!mbar_wait(smem_u32(&bars.q_full), qn & 1, abort_flag, a.err, kErrQFull) ||
            !mbar_wait(smem_u32(&bars.kv_full[n % kSlots]), (n / kSlots) & 1, abort_flag, a.err,
                       kErrKvFull))
          break;
        tc_fence_after();
        issue_s(0, n);
        issue_s(1, n);
        mma_commit(smem_u32(&bars.kv_empty[n % kSlots]));  // K_0 consumed
        if (nt == 1) mma_commit(smem_u32(&bars.q_empty));
        for (int lt = 0; lt < nt; ++lt, ++it, n += 2) {
          const int v_idx = n + 1, k_next = n + 2;
          const int v_slot = v_idx % kSlots, k_slot = k_next % kSlots;
          const bool more = lt + 1 < nt;
          // V_lt and K_{lt+1} have usually landed long ago: test both at once
          // (each blocking wait costs the issuing thread ~150 cycles during
          // which the tensor pipe, fed one MMA deep, runs dry)
          const bool v_ready = mbar_test_wait(smem_u32(&bars.kv_full[v_slot]), (v_idx / kSlots) & 1);
          const bool k_ready =
              !more || mbar_test_wait(smem_u32(&bars.kv_full[k_slot]), (k_next / kSlots) & 1);
          if (!(v_ready && k_ready) &&
              (!mbar_wait(smem_u32(&bars.kv_full[v_slot]), (v_idx / kSlots) & 1, abort_flag, a.err,
                          kErrKvFull) ||
               (more && !mbar_wait(smem_u32(&bars.kv_full[k_slot]), (k_next / kSlots) & 1,
                                   abort_flag, a.err, kErrKvFull)))) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int t = 0; t < kQTiles; ++t) {
            // PV_t(lt) once its P is in TMEM; the unit's first PV overwrites
            // O_t, so it also waits for the previous unit's epilogue
            if (!mbar_wait(smem_u32(&bars.p_full[t]), it & 1, abort_flag, a.err, kErrPFull) ||
                (lt == 0 && !mbar_wait(smem_u32(&bars.o_free[t]), (qn & 1) ^ 1, abort_flag, a.err,
                                       kErrOFree))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(t, lt == 0, v_slot);
            if (t == kQTiles - 1) mma_commit(smem_u32(&bars.kv_empty[v_slot]));  // V_lt consumed
            if (!more) {
              mma_commit(smem_u32(&bars.o_full[t]));
            } else {
              issue_s(t, k_next);
              if (t == kQTiles - 1) {
                mma_commit(smem_u32(&bars.kv_empty[k_slot]));  // K_{lt+1} consumed
                if (lt + 2 == nt) mma_commit(smem_u32(&bars.q_empty));  // last S of the unit
              }
            }
          }
          if (!ok) break;
        }
        ++qn;
      }
      // every MMA issued has completed before TMEM is released
      mma_commit(smem_u32(&bars.done));
      mbar_wait(smem_u32(&bars.done), 0, abort_flag, a.err, kErrDrain);
    }
    __syncwarp();
  } else if (warp < 2 * 4) {
    // ------------------------------------------------- softmax warpgroups
    const int t = warp >> 2;           // Q tile of this group
    const int row = threadIdx.x & 127;  // TMEM lane == row of the tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + 256 + t * 128;
    int it = 0;  // tiles over the CTA's life
    int qn = 0;  // units with tiles so far
    int qa = 0;  // running-output loads so far (accumulate form)
    bool ok = true;
    for (int seq = 0; ok; ++seq) {
      const int xs = seq & 1;
      const bool got_unit =
          mbar_wait(smem_u32(&bars.unit_full[xs]), (seq >> 1) & 1, abort_flag, a.err, kErrUnit);
      if (!__all_sync(0xffffffffu, got_unit)) break;
      const Unit& U = units_s[xs];  // read in place; released after the epilogue
      if (U.w < 0) break;
      const Schedule& sch = U.sch;
      const int u = U.u0 + t * kBM + row;  // local row in block i
      const bool row_live = u < Lb;
      const int tq = row_live ? static_cast<int>(block_token(a.order, a.S, a.P, U.i, u)) : 0;
      int lo, hi;
      if (a.doc_start && row_live) {
        lo = a.doc_start[static_cast<long long>(U.b % a.pos_rows) * a.S + tq];
        hi = tq;
      } else {
        lo = 0;
        hi = a.S - 1;
      }
      float m_run = -INFINITY;   // running max (log2 units, scaled)
      float m_use = -INFINITY;   // exponent base actually applied
      float l = 0.f;
      int ft = 0;  // position in the item's tile sequence
      for (int s = a.step_begin; s < a.step_end && ok && ft < sch.t_hi; ++s) {
        int j, kt0, kt1;
        sch.tiles(s, j, kt0, kt1);
        for (int kt = kt0; kt <= kt1; ++kt, ++ft) {
          if (ft < sch.t_lo) continue;
          if (ft >= sch.t_hi) break;
          // warp-uniform outcome: the tcgen05.ld below is warp-collective
          const bool got =
              mbar_wait(smem_u32(&bars.s_full[t]), it & 1, abort_flag, a.err, kErrSFull);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // the whole score row: four 32-column loads in flight, one wait;
          // each load also returns the max of its 32 scores
          uint32_t x[kBN];
          float hm[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32_max_at(tS + c * 32, x, c * 32, hm[c]);
          tmem_wait_ld();
          // allowed columns [c_lo, c_hi] of this tile for this row
          int c_lo, c_hi;
          {
            int lo_c, hi_c;
            const int w_base = kt * kBN;
            if (a.order == SP_ORDER_STRIPED) {
              lo_c = -floor_div(-(lo - j), a.P) - w_base;
              hi_c = floor_div(hi - j, a.P) - w_base;
            } else {
              const int base = j * Lb + w_base;
              lo_c = lo - base;
              hi_c = hi - base;
            }
            const int c_valid = Lb - w_base - 1;
            if (hi_c > c_valid) hi_c = c_valid;
            c_lo = lo_c < 0 ? 0 : (lo_c > kBN ? kBN : lo_c);
            c_hi = hi_c < -1 ? -1 : (hi_c > kBN - 1 ? kBN - 1 : hi_c);
          }
          // row max: on a tile with every column allowed, the loads' own
          // maxima; on a masked tile, over the allowed columns only (8
          // independent chains of 3-input max)
          float mt = fmax3(hm[0], hm[1], fmaxf(hm[2], hm[3]));
          if (c_lo > 0 || c_hi < kBN - 1) {
#pragma unroll
            for (int c = 0; c < kBN; ++c)
              if (c < c_lo || c > c_hi) x[c] = 0xff800000u;  // -inf
            float mx[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = __uint_as_float(x[k]);
#pragma unroll
            for (int c = 8; c < kBN - 8; c += 16) {
#pragma unroll
              for (int k = 0; k < 8; ++k)
                mx[k] = fmax3(mx[k], __uint_as_float(x[c + k]), __uint_as_float(x[c + 8 + k]));
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], __uint_as_float(x[kBN - 8 + k]));
            mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                       fmaxf(mx[6], mx[7]));
          }
          m_run = fmaxf(m_run, mt * scale_log2);
          float alpha = 1.f;
          bool rescale = false;
          if (m_use == -INFINITY) {
            m_use = m_run;  // first allowed key: O and l are still zero
          } else if (m_run > m_use + kRescaleThreshold) {
            alpha = ex2(m_use - m_run);
            m_use = m_run;
            rescale = true;
          }
          const float nbase = (m_use == -INFINITY) ? 0.f : -m_use;
          // p = 2^(s * scale_log2 - base), two lanes per FFMA; 4 pair sums
          float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < kBN; c += 2) {
            float e0, e1;
            ffma2(e0, e1, __uint_as_float(x[c]), __uint_as_float(x[c + 1]), scale_log2,
                  scale_log2, nbase, nbase);
            e0 = ex2(e0);
            e1 = ex2(e1);
            const int k = (c >> 1) & 3;
            fadd2(sa[k], sb[k], sa[k], sb[k], e0, e1);
            x[c >> 1] = pack_bf16(e0, e1);  // P row, packed in place (c/2 <= c)
          }
          l = l * alpha + ((sa[0] + sb[0]) + (sa[1] + sb[1])) + ((sa[2] + sb[2]) + (sa[3] + sb[3]));
          tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
          tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
          // O *= alpha in TMEM (after the scores are dead, to keep registers
          // free); the PV MMA that adds this tile waits for p_full below.
          if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t r[32];
              tmem_ld32(tO + c * 32, r);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tmem_st32(tO + c * 32, r);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(smem_u32(&bars.p_full[t]));
          ++it;
        }
      }
      // ---------------------------------------------------------- epilogue
      if (kAcc && U.n_tiles == 0) {  // nothing to fold in: the running rows stay
        mbar_arrive(smem_u32(&bars.unit_empty[xs]));
        continue;
      }
      const uint32_t stage = smem_stage + t * kStageBytes;
      const bool leader = row == 0;
      int c2, c3;
      coord_q(U.i, U.u0 + t * kBM, c2, c3);
      float lse_run = -INFINITY;
      if (kAcc) {
        // the running output's first half and the running lse, in flight
        // while the last PV completes
        if (row_live) lse_run = a.lse[(static_cast<long long>(U.b) * a.Hq + U.hq) * Lb + u];
        if (leader) {
          bulk_wait_group_read0();  // the stage's previous store has read it
          mbar_arrive_expect_tx(smem_u32(&bars.acc_full[t]), kStageBytes);
          tma_load_5d(stage, &tm.o, smem_u32(&bars.acc_full[t]), 0, U.hq, c2, c3, U.b);
        }
      }
      const bool have = U.n_tiles > 0 && ok;
      if (have) {
        const bool got = mbar_wait(smem_u32(&bars.o_full[t]), qn & 1, abort_flag, a.err, kErrOFull);
        if (!__all_sync(0xffffffffu, got)) ok = false;
      }
      tc_fence_after();
      const bool any = have && ok && l > 0.f;
      const float inv = any ? 1.f / l : 0.f;
      const float row_lse = any ? (m_use + lg2(l)) * 0.69314718055994530942f : -INFINITY;
      // out = c_new * O + c_run * out_run, lse = lse_out (without kAcc: the
      // partial itself)
      float c_new = inv, c_run = 0.f, lse_out = row_lse;
      if (kAcc) {
        const float mx = fmaxf(row_lse, lse_run);
        if (mx == -INFINITY) {  // neither has a key: the row stays as it is
          c_new = 0.f;
          c_run = 1.f;
        } else {
          const float wn = expf(row_lse - mx), wr = expf(lse_run - mx);
          const float wsum = wn + wr;
          c_new = inv * (wn / wsum);
          c_run = wr / wsum;
          lse_out = mx + logf(wsum);
        }
        if (c_new == 0.f) lse_out = lse_run;  // nothing added: the row keeps its bits
      }
      // the whole O row in one round trip, then O goes back to the MMA warp
      // (the next unit's first PV overwrites it) before the stores
      uint32_t r[kD];
      if (have && ok) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_at(tO + c * 32, r, c * 32);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < kD; ++e) r[e] = 0u;
      }
      if (U.n_tiles > 0) {
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.o_free[t]));
        ++qn;
      }
      if (!kAcc && U.split > 1) {
        // one piece of a split item: normalized partial O and its lse (fp32),
        // combined afterwards by merge_split_kernel
        const long long prow = static_cast<long long>(U.sidx) * kRowsPerCta + t * kBM + row;
        float4* po = reinterpret_cast<float4*>(part_o + prow * kD);
#pragma unroll
        for (int e = 0; e < kD / 4; ++e)
          po[e] = make_float4(__uint_as_float(r[4 * e]) * inv, __uint_as_float(r[4 * e + 1]) * inv,
                              __uint_as_float(r[4 * e + 2]) * inv,
                              __uint_as_float(r[4 * e + 3]) * inv);
        part_lse[prow] = row_lse;
      } else {
        // bf16 rows through a swizzled 16 KiB stage (one 64-column half at a
        // time, the layout a 64 x 128-row TMA box with 128-byte swizzle has)
        // and one bulk tensor store per half: coalesced, and asynchronous
        // for the warpgroup
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (leader) {
            bulk_wait_group_read0();  // the stage's previous store has read it
            if (kAcc && h == 1) {
              mbar_arrive_expect_tx(smem_u32(&bars.acc_full[t]), kStageBytes);
              tma_load_5d(stage, &tm.o, smem_u32(&bars.acc_full[t]), 64, U.hq, c2, c3, U.b);
            }
          }
          if (kAcc) {
            // every thread passes both named barriers whatever the outcome
            // (a timeout is recorded in the error word)
            if (!mbar_wait(smem_u32(&bars.acc_full[t]), qa & 1, abort_flag, a.err, kErrAccFull))
              ok = false;
            ++qa;
          }
          named_bar_sync(1 + t, kBM);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int e = h * 64 + c * 8;
            const uint32_t addr = stage + row * 128 + ((c ^ (row & 7)) << 4);
            float y[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) y[k] = __uint_as_float(r[e + k]) * c_new;
            uint4 v = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]),
                                 pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7]));
            if (kAcc && c_run > 0.f) {  // c_run = 0: the running row is not read
              uint32_t o[4];
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
                           : "r"(addr)
                           : "memory");
              if (c_new == 0.f) {  // nothing to add (then c_run = 1): the bits stay
                v = make_uint4(o[0], o[1], o[2], o[3]);
              } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  y[2 * k] = fmaf(c_run, __uint_as_float(o[k] << 16), y[2 * k]);
                  y[2 * k + 1] = fmaf(c_run, __uint_as_float(o[k] & 0xffff0000u), y[2 * k + 1]);
                }
                v = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]),
                               pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7]));
              }
            }
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x),
                         "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
          }
          fence_proxy_async_smem();
          named_bar_sync(1 + t, kBM);
          if (leader) {
            tma_store_5d(&tm.o, stage, h * 64, U.hq, c2, c3, U.b);
            bulk_commit_group();
          }
        }
        if (row_live && a.lse) {
          const bool blk = a.q_block >= 0;  // per-device lse: [B][Hq][S/P]
          a.lse[(static_cast<long long>(U.b) * a.Hq + U.hq) * (blk ? Lb : a.S) + (blk ? u : tq)] =
              lse_out;
        }
      }
      mbar_arrive(smem_u32(&bars.unit_empty[xs]));
    }
    if (row == 0) bulk_wait_group0();  // output stores complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Combines the pieces of split items: for every row, the `split` partial
// results (each normalized by its own sum, with its own lse) are merged by
// their log-sum-exp weights -- the same combine ring attention applies to
// per-device partials ("Ring Attention", "Cómo funciona la atención en
// anillo").  One warp per row of an item; lane c handles columns 4c..4c+3.
__global__ void __launch_bounds__(256) merge_split_kernel(AttnArgs a, int n_pairs, int item_base,
                                                          int split, const float* __restrict__ part_o,
                                                          const float* __restrict__ part_lse) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int x = blockIdx.x / (kRowsPerCta / 8);            // split item
  const int r = (blockIdx.x % (kRowsPerCta / 8)) * 8 + warp;  // row within the item
  int b, hq, i, pair;
  item_coords(item_base + x, a, n_pairs, b, hq, i, pair);
  const int Lb = a.S / a.P;
  const int u = pair * kRowsPerCta + r;
  if (u >= Lb) return;
  // row of out / lse: the token, or the local row of a per-device query block
  const bool blk = a.q_block >= 0;
  const long long tq = blk ? u : block_token(a.order, a.S, a.P, i, u);
  const long long rows = blk ? Lb : a.S;
  float m = -INFINITY;
  for (int p = 0; p < split; ++p)
    m = fmaxf(m, part_lse[(static_cast<long long>(x) * split + p) * kRowsPerCta + r]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int p = 0; p < split; ++p) {
      const long long prow = (static_cast<long long>(x) * split + p) * kRowsPerCta + r;
      const float lp = part_lse[prow];
      if (lp == -INFINITY) continue;
      const float w = expf(lp - m);
      wsum += w;
      const float4 o = reinterpret_cast<const float4*>(part_o + prow * kD)[lane];
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  uint2* orow = reinterpret_cast<uint2*>(out + ((static_cast<long long>(b) * rows + tq) * a.Hq + hq) * kD);
  orow[lane] = make_uint2(pack_bf16(acc.x * inv, acc.y * inv), pack_bf16(acc.z * inv, acc.w * inv));
  if (a.lse && lane == 0)
    a.lse[(static_cast<long long>(b) * a.Hq + hq) * rows + tq] =
        wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

// ------------------------------------------------------------------ host
}  // namespace

int launch_attn_bf16(const AttnArgs& a, cudaStream_t stream) {
  Tmaps tm;
  const int Lb = a.S / a.P;
  // a tensor holding a single block is mapped as one contiguous block
  const bool qb = a.q_block >= 0, kvb = a.kv_block >= 0;
  if (!tmap::make_map(&tm.q, a.q, a.B, qb ? Lb : a.S, a.Hq, qb ? 1 : a.P,
                      qb ? SP_ORDER_CONTIGUOUS : a.order) ||
      !tmap::make_map(&tm.k, a.k, a.B, kvb ? Lb : a.S, a.Hkv, kvb ? 1 : a.P,
                      kvb ? SP_ORDER_CONTIGUOUS : a.order) ||
      !tmap::make_map(&tm.v, a.v, a.B, kvb ? Lb : a.S, a.Hkv, kvb ? 1 : a.P,
                      kvb ? SP_ORDER_CONTIGUOUS : a.order) ||
      !tmap::make_map(&tm.o, a.out, a.B, qb ? Lb : a.S, a.Hq, qb ? 1 : a.P,
                      qb ? SP_ORDER_CONTIGUOUS : a.order))
    return -1;
  const int n_pairs = (Lb + kRowsPerCta - 1) / kRowsPerCta;
  const long long items = static_cast<long long>(a.B) * a.Hq * (qb ? 1 : a.P) * n_pairs;
  const size_t smem = kSmemBytes + 1024;
  if (cudaFuncSetAttribute(attn_bf16_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess ||
      cudaFuncSetAttribute(attn_bf16_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return -1;
  const float scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);

  // Tail split (non-causal only, where every item has the same tile count):
  // the items of the last, partly filled wave are cut into `split` pieces
  // along their ring-ordered tile sequence so that the wave fills the GPU;
  // the pieces write fp32 partials that merge_split_kernel combines.
  const long long G = device_sm_count();
  const long long rem = items % G;
  const long long full = items - rem;
  int split = 1;
  if (!a.doc_start && a.scratch && rem > 0 && !a.accumulate) {
    const long long tiles = static_cast<long long>(a.step_end - a.step_begin) *
                            ((Lb + kBN - 1) / kBN);
    long long k = G / rem;
    if (k > tiles) k = tiles;
    if (k > 32) k = 32;
    if (rem * k > kMaxSplitPieces) k = kMaxSplitPieces / rem;
    const size_t need = static_cast<size_t>(rem * k) * kRowsPerCta * (kD + 1) * sizeof(float);
    if (k >= 2 && need <= a.scratch_bytes) split = static_cast<int>(k);
  }
  // persistent grid: one CTA per SM (fewer when there is less work)
  const long long n_work = split == 1 ? items : full + rem * split;
  const unsigned grid = static_cast<unsigned>(n_work < G ? n_work : G);
  if (split == 1) {
    if (a.accumulate)
      attn_bf16_kernel<true><<<grid, kThreads, smem, stream>>>(
          tm, a, scale_log2, n_pairs, static_cast<int>(items), 1, static_cast<int>(n_work),
          nullptr, nullptr);
    else
      attn_bf16_kernel<false><<<grid, kThreads, smem, stream>>>(
          tm, a, scale_log2, n_pairs, static_cast<int>(items), 1, static_cast<int>(n_work),
          nullptr, nullptr);
    return cudaGetLastError() == cudaSuccess ? 1 : -1;
  }
  float* part_o = static_cast<float*>(a.scratch);
  float* part_lse = part_o + static_cast<size_t>(rem * split) * kRowsPerCta * kD;
  attn_bf16_kernel<false><<<grid, kThreads, smem, stream>>>(tm, a, scale_log2, n_pairs,
                                                            static_cast<int>(full), split,
                                                            static_cast<int>(n_work), part_o,
                                                            part_lse);
  merge_split_kernel<<<static_cast<unsigned>(rem * (kRowsPerCta / 8)), 256, 0, stream>>>(
      a, n_pairs, static_cast<int>(full), split, part_o, part_lse);
  return cudaGetLastError() == cudaSuccess ? 2 : -1;
}

}  // namespace sp
