// ulysses_ring.cu -- Ulysses + Ring hybrid for fewer heads than devices.
//
// Ulysses needs num_heads >= sp_size ("Ulysses SP: entrenar modelos con
// millones de tokens", "Comparación práctica: Ulysses vs Ring Attention";
// "Ulysses SPで100万トークン学習", section 6, which points to a Ulysses + Ring
// hybrid when GQA/MQA leaves too few heads).  With P = P_u * P_r devices the
// heads are split over P_u Ulysses groups and every group runs ring attention
// over P_r sequence blocks.  On one GPU this is: seq->head permutation with
// P_u groups, blockwise attention with P_r ring blocks on each head group
// (batch P_u * B), head->seq permutation of the output.
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "common.cuh"

namespace sp {
namespace {

struct HybridLayout {
  size_t attn, yq, ykv, total;
};

HybridLayout hybrid_layout(int B, int S, int Hq, int Hkv, int d, int causal, sp_dtype dtype) {
  HybridLayout L;
  const size_t es = dtype_size(dtype);
  L.attn = round_up(sp_blockwise_attn_split_workspace_bytes(B, S, causal), 256);
  L.yq = round_up(static_cast<size_t>(B) * S * Hq * d * es, 256);
  L.ykv = round_up(static_cast<size_t>(B) * S * Hkv * d * es, 256);
  L.total = L.attn + 2 * L.yq + 2 * L.ykv;
  return L;
}

}  // namespace
}  // namespace sp

extern "C" size_t sp_ulysses_ring_attn_workspace_bytes(int B, int S, int Hq, int Hkv, int d,
                                                       int causal, sp_dtype dtype) {
  if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || d < 1 || sp::dtype_size(dtype) == 0) return 0;
  return sp::hybrid_layout(B, S, Hq, Hkv, d, causal, dtype).total;
}

extern "C" sp_status sp_ulysses_ring_attn_fwd(const void* q, const void* k, const void* v,
                                              const int32_t* position_ids, int B, int S, int Hq,
                                              int Hkv, int d, int P_u, int P_r,
                                              sp_block_order order, float scale, sp_dtype dtype,
                                              void* out, float* lse, void* workspace,
                                              size_t workspace_bytes, sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_ulysses_ring_attn_fwd");
  sp::g_last_launches = 0;
  if (!q || !k || !v || !out) return SP_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || d < 1 || P_u < 1 || P_r < 1)
    return SP_ERR_INVALID_ARG;
  if (S % P_u != 0 || S % P_r != 0 || Hq % P_u != 0 || Hkv % P_u != 0 || Hq % Hkv != 0)
    return SP_ERR_INVALID_ARG;
  if (sp::dtype_size(dtype) == 0) return SP_ERR_INVALID_ARG;
  if (static_cast<long long>(P_u) * B > 65535) return SP_ERR_UNSUPPORTED;
  const int causal = position_ids != nullptr;
  const sp::HybridLayout L = sp::hybrid_layout(B, S, Hq, Hkv, d, causal, dtype);
  if (!workspace || !sp::aligned(workspace, 256) || workspace_bytes < L.total)
    return SP_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* yq = ws + L.attn;
  void* yo = ws + L.attn + L.yq;
  void* yk = ws + L.attn + 2 * L.yq;
  void* yv = ws + L.attn + 2 * L.yq + L.ykv;
  int launches = 0;
  sp_status st;
  // Ulysses all-to-all #1 (sequence shards -> P_u head groups)
  st = sp_ulysses_seq_to_head_qkv(q, k, v, yq, yk, yv, B, S, Hq, Hkv, d, P_u, dtype, stream);
  if (st != SP_OK) return st;
  launches += sp::g_last_launches;
  // ring attention over P_r blocks inside every head group (batch P_u * B);
  // all groups share the B rows of position_ids
  st = sp::attn(yq, yk, yv, position_ids, B, P_u * B, S, Hq / P_u, Hkv / P_u, d, P_r, order, 0,
                P_r, scale, dtype, yo, lse, ws, L.attn, stream);
  if (st != SP_OK) return st;
  launches += sp::g_last_launches;
  // Ulysses all-to-all #2 (head groups -> sequence shards)
  if ((st = sp_ulysses_head_to_seq(yo, out, B, S, Hq, d, P_u, dtype, stream)) != SP_OK) return st;
  launches += sp::g_last_launches;
  sp::g_last_launches = launches;
  return SP_OK;
}
