// api_bwd.cu -- entry point of the attention backward: checks, workspace
// layout, dispatch.
//
// Workspace layout (256-byte aligned, caller-owned):
//   [0, 256)                      error word + reserved
//   [256, +B*Hq*S*4)              D = rowsum(dout * out) per query row, fp32
//   [.., +B*S*4)                  doc_start (causal only)
//   [.., + scan scratch)          doc_start scan scratch (causal only)
#include <cuda_runtime.h>
#include <math.h>

#include "attn_common.cuh"
#include "common.cuh"

namespace sp {
namespace {

struct BwdLayout {
  size_t dsum, doc, scan, total;
};

BwdLayout bwd_layout(int B, int S, int Hq, int causal) {
  BwdLayout L;
  L.dsum = round_up(static_cast<size_t>(B) * Hq * S * sizeof(float), 256);
  L.doc = causal ? round_up(static_cast<size_t>(B) * S * sizeof(int32_t), 256) : 0;
  L.scan = causal ? segment_scratch_bytes(B, S) : 0;
  L.total = kWsHeaderBytes + L.dsum + L.doc + L.scan;
  return L;
}

}  // namespace
}  // namespace sp

extern "C" size_t sp_blockwise_attn_bwd_workspace_bytes(int B, int S, int Hq, int causal) {
  if (B < 1 || S < 1 || Hq < 1) return 0;
  return sp::bwd_layout(B, S, Hq, causal).total;
}

extern "C" sp_status sp_blockwise_attn_bwd(const void* q, const void* k, const void* v,
                                           const void* out, const void* dout, const float* lse,
                                           const int32_t* position_ids, int B, int S, int Hq,
                                           int Hkv, int d, int P, sp_block_order order,
                                           float scale, sp_dtype dtype, void* dq, void* dk,
                                           void* dv, void* workspace, size_t workspace_bytes,
                                           sp_stream_t stream) {
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
  const sp::BwdLayout L = sp::bwd_layout(B, S, Hq, causal);
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
    int32_t* doc = reinterpret_cast<int32_t*>(ws + sp::kWsHeaderBytes + L.dsum);
    const int n = sp::launch_segment_starts(position_ids, doc, B, S,
                                            ws + sp::kWsHeaderBytes + L.dsum + L.doc, st);
    if (n < 0) return SP_ERR_CUDA;
    launches += n;
    a.doc_start = doc;
  }
  const int n = dtype == SP_BF16 ? sp::launch_attn_bwd_bf16(a, st) : sp::launch_attn_bwd_simt(a, st);
  if (n < 0) return SP_ERR_CUDA;
  sp::g_last_launches = launches + n;
  return SP_OK;
}
