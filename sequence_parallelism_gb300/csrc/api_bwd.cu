// api_bwd.cu -- entry point of the attention backward: checks, workspace
// layout, dispatch.
//
// Workspace layout (256-byte aligned, caller-owned; Lbp = S/P rounded up to
// a multiple of 64):
//   [0, 256)                      error word + reserved
//   D                             rowsum(dout * out), fp32: [B][Hq][S] (f32
//                                 path) or [B][Hq][P][Lbp] (bf16 path)
//   lse2                          [B][Hq][P][Lbp] lse * log2(e) (bf16 path)
//   lo                            [B][P][Lbp] doc_start in block order (causal)
//   doc_start                     [B][S] (causal only)
//   scan scratch                  doc_start scan (causal only)
//   dQ accumulator                fp32, B * Hq * P * Lbp * 128 floats (bf16
//                                 path with dQ by reductions)
#include <atomic>
#include <cuda_runtime.h>
#include <math.h>

#include "attn_common.cuh"
#include "common.cuh"

namespace sp {

int launch_attn_bwd_bf16_fused(const BwdArgs& a, float* dq_acc, cudaStream_t st);

namespace {

std::atomic<int> g_bwd_dq_reduction{1};

struct BwdLayout {
  size_t dsum, lse2, lo, doc, scan, acc, total;
  int Lbp;
};

BwdLayout bwd_layout(int B, int S, int Hq, int P, int causal) {
  BwdLayout L;
  L.Lbp = static_cast<int>(round_up(static_cast<size_t>(S / P), kBwdRowPad));
  const size_t blk = static_cast<size_t>(B) * Hq * P * L.Lbp * sizeof(float);
  const size_t tok = static_cast<size_t>(B) * Hq * S * sizeof(float);
  L.dsum = round_up(blk > tok ? blk : tok, 256);
  L.lse2 = round_up(blk, 256);
  L.lo = causal ? round_up(static_cast<size_t>(B) * P * L.Lbp * sizeof(int32_t), 256) : 0;
  L.doc = causal ? round_up(static_cast<size_t>(B) * S * sizeof(int32_t), 256) : 0;
  L.scan = causal ? segment_scratch_bytes(B, S) : 0;
  L.acc = round_up(static_cast<size_t>(B) * Hq * P * L.Lbp * 128 * sizeof(float), 256);
  L.total = kWsHeaderBytes + L.dsum + L.lse2 + L.lo + L.doc + L.scan + L.acc;
  return L;
}

}  // namespace
}  // namespace sp

extern "C" int sp_set_bwd_dq_reduction(int on) {
  return sp::g_bwd_dq_reduction.exchange(on ? 1 : 0);
}

extern "C" size_t sp_blockwise_attn_bwd_workspace_bytes(int B, int S, int Hq, int P,
                                                        int causal) {
  if (B < 1 || S < 1 || Hq < 1 || P < 1 || S % P != 0) return 0;
  return sp::bwd_layout(B, S, Hq, P, causal).total;
}

extern "C" sp_status sp_blockwise_attn_bwd(const void* q, const void* k, const void* v,
                                           const void* out, const void* dout, const float* lse,
                                           const int32_t* position_ids, int B, int S, int Hq,
                                           int Hkv, int d, int P, sp_block_order order,
                                           float scale, sp_dtype dtype, void* dq, void* dk,
                                           void* dv, void* workspace, size_t workspace_bytes,
                                           sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_blockwise_attn_bwd");
  sp::g_last_launches = 0;
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return SP_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || d < 1 || P < 1) return SP_ERR_INVALID_ARG;
  if (S % P != 0 || Hq % Hkv != 0) return SP_ERR_INVALID_ARG;
  if (order != SP_ORDER_CONTIGUOUS && order != SP_ORDER_STRIPED) return SP_ERR_INVALID_ARG;
  if (dtype != SP_BF16 && dtype != SP_F32) return SP_ERR_INVALID_ARG;
  if (!(scale == scale) || isinf(scale)) return SP_ERR_INVALID_ARG;
  if (d > 256) return SP_ERR_UNSUPPORTED;
  if (dtype == SP_BF16 && d != 128) return SP_ERR_UNSUPPORTED;
  if (B > 65535 || Hq > 65535) return SP_ERR_UNSUPPORTED;
  if (dtype == SP_BF16) {  // TMA bases and 16-byte vector accesses
    const void* ptrs[8] = {q, k, v, out, dout, dq, dk, dv};
    for (const void* p : ptrs)
      if (!sp::aligned(p, 16)) return SP_ERR_INVALID_ARG;
  }
  const int causal = position_ids != nullptr;
  const sp::BwdLayout L = sp::bwd_layout(B, S, Hq, P, causal);
  if (!workspace || !sp::aligned(workspace, 256) || workspace_bytes < L.total)
    return SP_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  sp::BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.dout = dout;
  a.lse = lse;
  a.err = reinterpret_cast<int*>(ws);
  a.Dsum = reinterpret_cast<float*>(ws + sp::kWsHeaderBytes);
  a.D_blk = a.Dsum;
  a.lse2_blk = reinterpret_cast<float*>(ws + sp::kWsHeaderBytes + L.dsum);
  a.lo_blk = causal ? reinterpret_cast<int32_t*>(ws + sp::kWsHeaderBytes + L.dsum + L.lse2)
                    : nullptr;
  a.Lbp = L.Lbp;
  a.doc_start = nullptr;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.S = S;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.P = P;
  a.pos_rows = B;
  a.order = order;
  a.dtype = dtype;
  a.scale = scale > 0.f ? scale : static_cast<float>(1.0 / sqrt(static_cast<double>(d)));
  int launches = 0;
  if (cudaMemsetAsync(a.err, 0, sizeof(int), st) != cudaSuccess) return SP_ERR_CUDA;
  if (causal) {
    uint8_t* base = ws + sp::kWsHeaderBytes + L.dsum + L.lse2 + L.lo;
    int32_t* doc = reinterpret_cast<int32_t*>(base);
    const int n = sp::launch_segment_starts(position_ids, doc, B, S, base + L.doc, st);
    if (n < 0) return SP_ERR_CUDA;
    launches += n;
    a.doc_start = doc;
  }
  float* dq_acc = reinterpret_cast<float*>(ws + sp::kWsHeaderBytes + L.dsum + L.lse2 + L.lo +
                                            L.doc + L.scan);
  const int n = dtype != SP_BF16 ? sp::launch_attn_bwd_simt(a, st)
                : sp::g_bwd_dq_reduction.load() ? sp::launch_attn_bwd_bf16_fused(a, dq_acc, st)
                                                : sp::launch_attn_bwd_bf16(a, st);
  if (n < 0) return SP_ERR_CUDA;
  sp::g_last_launches = launches + n;
  return SP_OK;
}

// ------------------------------------------------------------------------
// Per-device backward step (query block i against key/value block j).
//
// Workspace layout (256-byte aligned; Lbp = S/P rounded up to 128):
//   [0, 256)                      error word + reserved
//   D, lse2                       [B][Hq][Lbp] each, fp32 (block i's rows)
//   lo                            [B][Lbp] doc_start of block i's tokens (causal)
//   doc_start, scan scratch       [B][S] (causal)
//   dQ sums                       B * Hq * Lbp * 128 floats
namespace sp {

int launch_attn_bwd_bf16_block(const BwdArgs& a, int qb, int kb, float* dq_blocked,
                               float* dq_acc, float* dk_acc, float* dv_acc, cudaStream_t st);

namespace {

struct BlockBwdLayout {
  size_t d, lse2, lo, doc, scan, acc, total;
  int Lbp;
};

BlockBwdLayout block_bwd_layout(int B, int S, int Hq, int P, int causal) {
  BlockBwdLayout L;
  L.Lbp = static_cast<int>(round_up(static_cast<size_t>(S / P), kBwdRowPad));
  const size_t rows = static_cast<size_t>(B) * Hq * L.Lbp * sizeof(float);
  L.d = round_up(rows, 256);
  L.lse2 = round_up(rows, 256);
  L.lo = causal ? round_up(static_cast<size_t>(B) * L.Lbp * sizeof(int32_t), 256) : 0;
  L.doc = causal ? round_up(static_cast<size_t>(B) * S * sizeof(int32_t), 256) : 0;
  L.scan = causal ? segment_scratch_bytes(B, S) : 0;
  L.acc = round_up(static_cast<size_t>(B) * Hq * L.Lbp * 128 * sizeof(float), 256);
  L.total = kWsHeaderBytes + L.d + L.lse2 + L.lo + L.doc + L.scan + L.acc;
  return L;
}

}  // namespace
}  // namespace sp

extern "C" size_t sp_ring_block_step_bwd_workspace_bytes(int B, int S, int Hq, int P,
                                                         int causal) {
  if (B < 1 || S < 1 || Hq < 1 || P < 1 || S % P != 0) return 0;
  return sp::block_bwd_layout(B, S, Hq, P, causal).total;
}

extern "C" sp_status sp_ring_block_step_bwd(const void* q_blk, const void* k_blk,
                                            const void* v_blk, const void* out_blk,
                                            const void* dout_blk, const float* lse_blk,
                                            const int32_t* position_ids, int B, int S, int Hq,
                                            int Hkv, int d, int P, sp_block_order order, int i,
                                            int j, float scale, sp_dtype dtype, float* dq_acc,
                                            float* dk_acc, float* dv_acc, void* workspace,
                                            size_t workspace_bytes, sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_ring_block_step_bwd");
  sp::g_last_launches = 0;
  if (!q_blk || !k_blk || !v_blk || !out_blk || !dout_blk || !lse_blk || !dq_acc || !dk_acc ||
      !dv_acc)
    return SP_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || d < 1 || P < 1) return SP_ERR_INVALID_ARG;
  if (S % P != 0 || Hq % Hkv != 0 || i < 0 || i >= P || j < 0 || j >= P)
    return SP_ERR_INVALID_ARG;
  if (order != SP_ORDER_CONTIGUOUS && order != SP_ORDER_STRIPED) return SP_ERR_INVALID_ARG;
  if (dtype != SP_BF16 && dtype != SP_F32) return SP_ERR_INVALID_ARG;
  if (!(scale == scale) || isinf(scale)) return SP_ERR_INVALID_ARG;
  if (dtype != SP_BF16 || d != 128) return SP_ERR_UNSUPPORTED;
  if (B > 65535 || Hq > 65535) return SP_ERR_UNSUPPORTED;
  {
    const void* ptrs[8] = {q_blk, k_blk, v_blk, out_blk, dout_blk, dq_acc, dk_acc, dv_acc};
    for (const void* p : ptrs)
      if (!sp::aligned(p, 16)) return SP_ERR_INVALID_ARG;
  }
  const int causal = position_ids != nullptr;
  const sp::BlockBwdLayout L = sp::block_bwd_layout(B, S, Hq, P, causal);
  if (!workspace || !sp::aligned(workspace, 256) || workspace_bytes < L.total)
    return SP_ERR_WORKSPACE;
  // contiguous blocks under the causal mask: no query of block i may attend a
  // key of block j > i, so the pair's gradient parts are zero
  if (causal && order == SP_ORDER_CONTIGUOUS && j > i) return SP_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* p0 = ws + sp::kWsHeaderBytes;
  sp::BwdArgs a;
  a.q = q_blk;
  a.k = k_blk;
  a.v = v_blk;
  a.out = out_blk;
  a.dout = dout_blk;
  a.lse = lse_blk;
  a.err = reinterpret_cast<int*>(ws);
  a.Dsum = reinterpret_cast<float*>(p0);
  a.D_blk = a.Dsum;
  a.lse2_blk = reinterpret_cast<float*>(p0 + L.d);
  a.lo_blk = causal ? reinterpret_cast<int32_t*>(p0 + L.d + L.lse2) : nullptr;
  a.Lbp = L.Lbp;
  a.doc_start = nullptr;
  a.dq = nullptr;
  a.dk = nullptr;
  a.dv = nullptr;
  a.B = B;
  a.S = S;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.P = P;
  a.pos_rows = B;
  a.order = order;
  a.dtype = dtype;
  a.scale = scale > 0.f ? scale : static_cast<float>(1.0 / sqrt(static_cast<double>(d)));
  int launches = 0;
  if (cudaMemsetAsync(a.err, 0, sizeof(int), st) != cudaSuccess) return SP_ERR_CUDA;
  if (causal) {
    uint8_t* base = p0 + L.d + L.lse2 + L.lo;
    int32_t* doc = reinterpret_cast<int32_t*>(base);
    const int n = sp::launch_segment_starts(position_ids, doc, B, S, base + L.doc, st);
    if (n < 0) return SP_ERR_CUDA;
    launches += n;
    a.doc_start = doc;
  }
  float* dq_blocked =
      reinterpret_cast<float*>(p0 + L.d + L.lse2 + L.lo + L.doc + L.scan);
  const int n = sp::launch_attn_bwd_bf16_block(a, i, j, dq_blocked, dq_acc, dk_acc, dv_acc, st);
  if (n < 0) return SP_ERR_CUDA;
  sp::g_last_launches = launches + n;
  return SP_OK;
}
