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
