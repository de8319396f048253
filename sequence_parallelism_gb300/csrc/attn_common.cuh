// attn_common.cuh -- what the attention entry points hand to the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace sp {

// One blockwise-attention launch.  Ring steps [step_begin, step_end) are
// visited for every query block i: key/value block j = (i - s) mod P.
// Per-device form (what one rank of a real ring holds): with q_block >= 0,
// q and out hold only query block q_block ([B][S/P][Hq][d], rows in block
// order) and lse is [B][Hq][S/P]; with kv_block >= 0, k and v hold only
// key/value block kv_block ([B][S/P][Hkv][d]) and the steps visit only that
// block.  Masks and doc_start stay in global token indices either way.
struct AttnArgs {
  const void* q;               // [B][S][Hq][d]   ([B][S/P][Hq][d] when q_block >= 0)
  const void* k;               // [B][S][Hkv][d]  ([B][S/P][Hkv][d] when kv_block >= 0)
  const void* v;               // [B][S][Hkv][d]  (likewise)
  const int32_t* doc_start;    // [pos_rows][S] or nullptr (non-causal)
  void* out;                   // [B][S][Hq][d]   ([B][S/P][Hq][d] when q_block >= 0)
  float* lse;                  // [B][Hq][S] ([B][Hq][S/P] when q_block >= 0) or nullptr
  int q_block;                 // -1: every query block
  int kv_block;                // -1: k and v hold the whole sequence
  int* err;                    // device error word
  int* counter;                // work-unit counter of the persistent kernel (zeroed per call)
  int B, S, Hq, Hkv, d, P;
  int pos_rows;                // batch b reads doc_start row b % pos_rows
  int order;                   // sp_block_order
  int step_begin, step_end;
  float scale;                 // multiplies q.k (natural-log domain)
  void* scratch;               // optional workspace beyond the minimum (256-aligned)
  size_t scratch_bytes;
  int accumulate;              // 1: out / lse hold a running result that this call's
                               // partial is folded into (bf16 per-device form only)
};

// Scratch that lets a non-causal bf16 call split the items of its last,
// partly filled wave (fp32 partial rows for at most kMaxSplitPieces CTAs).
constexpr int kMaxSplitPieces = 160;
constexpr size_t kSplitScratchBytes =
    static_cast<size_t>(kMaxSplitPieces) * 256 * (128 + 1) * sizeof(float);

// One backward call: gradients of blockwise attention.
struct BwdArgs {
  const void* q;               // [B][S][Hq][d]
  const void* k;               // [B][S][Hkv][d]
  const void* v;               // [B][S][Hkv][d]
  const void* out;             // [B][S][Hq][d]  forward output
  const void* dout;            // [B][S][Hq][d]  upstream gradient
  const float* lse;            // [B][Hq][S]     forward log-sum-exp (natural)
  const int32_t* doc_start;    // [pos_rows][S] or nullptr (non-causal)
  float* Dsum;                 // [B][Hq][S] scratch: rowsum(dout * out) (f32 path)
  // bf16 path: per-query data in block order, each block padded to Lbp rows
  float* lse2_blk;             // [B][Hq][P][Lbp] lse * log2(e), +inf in the padding
  float* D_blk;                // [B][Hq][P][Lbp] rowsum(dout * out), 0 in the padding
  int32_t* lo_blk;             // [B][P][Lbp] doc_start of the row's token (causal), INT_MAX pad
  int Lbp;
  void* dq;                    // [B][S][Hq][d]
  void* dk;                    // [B][S][Hkv][d]
  void* dv;                    // [B][S][Hkv][d]
  int* err;
  int B, S, Hq, Hkv, d, P, pos_rows, order;
  sp_dtype dtype;
  float scale;
};

int launch_attn_bwd_simt(const BwdArgs& a, cudaStream_t stream);
int launch_attn_bwd_bf16(const BwdArgs& a, cudaStream_t stream);  // d == 128
constexpr int kBwdRowPad = 128;  // Lbp = S / P rounded up to a multiple of this

// Validates and runs one blockwise-attention call (doc_start scan when
// position_ids != NULL, then the f32 or bf16 kernel).  position_ids has
// pos_rows rows; attention batch b reads row b % pos_rows (pos_rows divides B).
// q_block / kv_block: the per-device form of AttnArgs (-1: whole sequence).
// accumulate: fold the partial into the running (out, lse) instead of
// writing it (a single ring step of the bf16 per-device form).
// Sets g_last_launches.
sp_status attn(const void* q, const void* k, const void* v, const int32_t* position_ids,
               int pos_rows, int B, int S, int Hq, int Hkv, int d, int P, sp_block_order order,
               int step_begin, int step_end, float scale, sp_dtype dtype, void* out, float* lse,
               void* workspace, size_t workspace_bytes, sp_stream_t stream, int q_block = -1,
               int kv_block = -1, bool accumulate = false);

// Both return the number of kernels launched, or -1 on a CUDA error.
int launch_attn_f32(const AttnArgs& a, cudaStream_t stream);
int launch_attn_bf16(const AttnArgs& a, cudaStream_t stream);

// Token index of local row u of block p (both orders).
__host__ __device__ __forceinline__ long long block_token(int order, int S, int P, int p,
                                                          long long u) {
  return order == SP_ORDER_STRIPED ? u * P + p : static_cast<long long>(p) * (S / P) + u;
}

}  // namespace sp
