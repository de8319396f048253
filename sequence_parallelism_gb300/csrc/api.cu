// api.cu -- the attention entry points of the C ABI: argument checks,
// workspace layout and dispatch to the float32 (CUDA core) or bf16 (tcgen05)
// kernels.  Layouts and semantics are documented in include/sp_gb300.h.
//
// Workspace layout (256-byte aligned, caller-owned):
//   [0, 256)                   error word (int32) + reserved
//   [256, 256 + R*S*4)         doc_start [R][S] int32     (causal only; R rows of
//                              position_ids, R = B except in the Ulysses+Ring call)
//   [.., + scan scratch)       per-chunk maxima of the doc_start scan
#include <cuda_runtime.h>
#include <math.h>

#include "attn_common.cuh"
#include "common.cuh"

namespace sp {

thread_local int g_last_launches = 0;

int device_sm_count() {
  static int n = [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
      return kNumSMs;
    return v;
  }();
  return n;
}

namespace {

size_t doc_start_bytes(int B, int S) {
  return round_up(static_cast<size_t>(B) * static_cast<size_t>(S) * sizeof(int32_t), 256);
}

}  // namespace

sp_status attn(const void* q, const void* k, const void* v, const int32_t* position_ids,
               int pos_rows, int B, int S, int Hq, int Hkv, int d, int P, sp_block_order order,
               int step_begin, int step_end, float scale, sp_dtype dtype, void* out, float* lse,
               void* workspace, size_t workspace_bytes, sp_stream_t stream, int q_block,
               int kv_block, bool accumulate) {
  g_last_launches = 0;
  if (!q || !k || !v || !out) return SP_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || d < 1 || P < 1) return SP_ERR_INVALID_ARG;
  if (S % P != 0 || Hq % Hkv != 0) return SP_ERR_INVALID_ARG;
  if (order != SP_ORDER_CONTIGUOUS && order != SP_ORDER_STRIPED) return SP_ERR_INVALID_ARG;
  // per-device form: a single query block, and with it at most one key/value
  // block, the one the (single) ring step visits
  if (q_block < -1 || q_block >= P || kv_block < -1 || kv_block >= P) return SP_ERR_INVALID_ARG;
  if (kv_block >= 0 && (q_block < 0 || step_end != step_begin + 1 ||
                        ((q_block - step_begin) % P + P) % P != kv_block))
    return SP_ERR_INVALID_ARG;
  if (dtype != SP_BF16 && dtype != SP_F32) return SP_ERR_INVALID_ARG;
  if (!(scale == scale) || isinf(scale)) return SP_ERR_INVALID_ARG;
  if (dtype == SP_BF16 && d != 128) return SP_ERR_UNSUPPORTED;
  if (dtype == SP_F32 && d > 256) return SP_ERR_UNSUPPORTED;
  if (B > 65535 || Hq > 65535) return SP_ERR_UNSUPPORTED;
  if (dtype == SP_BF16) {
    // TMA needs 16-byte aligned bases; the grid is one CTA per 256 rows.
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
      return SP_ERR_INVALID_ARG;
    const long long pairs = (S / P + 255) / 256;
    if (static_cast<long long>(B) * Hq * P * pairs > 0x7fffffffLL) return SP_ERR_UNSUPPORTED;
  }
  if (pos_rows < 1 || B % pos_rows != 0) return SP_ERR_INVALID_ARG;
  if (accumulate && (q_block < 0 || kv_block < 0 || !lse)) return SP_ERR_INVALID_ARG;
  if (accumulate && dtype != SP_BF16) return SP_ERR_UNSUPPORTED;
  const int causal = position_ids != nullptr;
  if (!workspace || !aligned(workspace, 256) ||
      workspace_bytes < sp_blockwise_attn_workspace_bytes(pos_rows, S, causal))
    return SP_ERR_WORKSPACE;
  // contiguous blocks under the causal mask: every key of block j > i comes
  // after every query of block i, so the pair adds nothing to a running result
  if (accumulate && causal && order == SP_ORDER_CONTIGUOUS && kv_block > q_block) return SP_OK;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* err = reinterpret_cast<int*>(ws);
  int32_t* doc_start = nullptr;
  int launches = 0;
  // error word and work-unit counter
  if (cudaMemsetAsync(err, 0, 2 * sizeof(int), st) != cudaSuccess) return SP_ERR_CUDA;
  if (causal) {
    doc_start = reinterpret_cast<int32_t*>(ws + kWsHeaderBytes);
    void* scan = ws + kWsHeaderBytes + doc_start_bytes(pos_rows, S);
    const int n = launch_segment_starts(position_ids, doc_start, pos_rows, S, scan, st);
    if (n < 0) return SP_ERR_CUDA;
    launches += n;
  }
  AttnArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.doc_start = doc_start;
  a.out = out;
  a.lse = lse;
  a.q_block = q_block;
  a.kv_block = kv_block;
  a.err = err;
  a.counter = err + 1;
  a.B = B;
  a.pos_rows = pos_rows;
  a.S = S;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.P = P;
  a.order = order;
  a.step_begin = step_begin;
  a.step_end = step_end;
  a.scale = scale > 0.f ? scale : static_cast<float>(1.0 / sqrt(static_cast<double>(d)));
  a.scratch = nullptr;
  a.scratch_bytes = 0;
  a.accumulate = accumulate ? 1 : 0;
  if (!causal && workspace_bytes > kWsHeaderBytes) {
    a.scratch = ws + kWsHeaderBytes;
    a.scratch_bytes = workspace_bytes - kWsHeaderBytes;
  }
  const int n = dtype == SP_BF16 ? launch_attn_bf16(a, st) : launch_attn_f32(a, st);
  if (n < 0) return SP_ERR_CUDA;
  g_last_launches = launches + n;
  return SP_OK;
}

}  // namespace sp

extern "C" const char* sp_status_string(sp_status s) {
  switch (s) {
    case SP_OK: return "SP_OK";
    case SP_ERR_INVALID_ARG: return "SP_ERR_INVALID_ARG: invalid argument";
    case SP_ERR_UNSUPPORTED: return "SP_ERR_UNSUPPORTED: unsupported size or type";
    case SP_ERR_WORKSPACE: return "SP_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case SP_ERR_CUDA: return "SP_ERR_CUDA: CUDA error at launch";
    case SP_ERR_DEVICE_TIMEOUT: return "SP_ERR_DEVICE_TIMEOUT: a kernel timed out on a barrier";
  }
  return "unknown sp_status";
}

extern "C" size_t sp_blockwise_attn_workspace_bytes(int B, int S, int causal) {
  if (B < 1 || S < 1) return 0;
  size_t n = sp::kWsHeaderBytes;
  if (causal) n += sp::doc_start_bytes(B, S) + sp::segment_scratch_bytes(B, S);
  return n;
}

extern "C" size_t sp_blockwise_attn_split_workspace_bytes(int B, int S, int causal) {
  const size_t n = sp_blockwise_attn_workspace_bytes(B, S, causal);
  if (n == 0 || causal) return n;
  return n + sp::kSplitScratchBytes;
}

extern "C" sp_status sp_blockwise_attn_fwd(const void* q, const void* k, const void* v,
                                           const int32_t* position_ids, int B, int S, int Hq,
                                           int Hkv, int d, int P, sp_block_order order,
                                           float scale, sp_dtype dtype, void* out, float* lse,
                                           void* workspace, size_t workspace_bytes,
                                           sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_blockwise_attn_fwd");
  return sp::attn(q, k, v, position_ids, B, B, S, Hq, Hkv, d, P, order, 0, P, scale, dtype, out,
                  lse, workspace, workspace_bytes, stream);
}

extern "C" sp_status sp_blockwise_attn_step(const void* q, const void* k, const void* v,
                                            const int32_t* position_ids, int B, int S, int Hq,
                                            int Hkv, int d, int P, sp_block_order order, int step,
                                            float scale, sp_dtype dtype, void* out, float* lse,
                                            void* workspace, size_t workspace_bytes,
                                            sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_blockwise_attn_step");
  sp::g_last_launches = 0;
  if (step < 0 || step >= P) return SP_ERR_INVALID_ARG;
  return sp::attn(q, k, v, position_ids, B, B, S, Hq, Hkv, d, P, order, step, step + 1, scale,
                  dtype, out, lse, workspace, workspace_bytes, stream);
}

extern "C" sp_status sp_ring_block_step(const void* q_blk, const void* k_blk, const void* v_blk,
                                        const int32_t* position_ids, int B, int S, int Hq, int Hkv,
                                        int d, int P, sp_block_order order, int i, int j,
                                        float scale, sp_dtype dtype, void* out_blk, float* lse_blk,
                                        void* workspace, size_t workspace_bytes,
                                        sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_ring_block_step");
  sp::g_last_launches = 0;
  if (P < 1 || i < 0 || i >= P || j < 0 || j >= P) return SP_ERR_INVALID_ARG;
  const int step = ((i - j) % P + P) % P;
  return sp::attn(q_blk, k_blk, v_blk, position_ids, B, B, S, Hq, Hkv, d, P, order, step,
                  step + 1, scale, dtype, out_blk, lse_blk, workspace, workspace_bytes, stream, i,
                  j);
}

extern "C" sp_status sp_ring_block_step_accumulate(
    const void* q_blk, const void* k_blk, const void* v_blk, const int32_t* position_ids, int B,
    int S, int Hq, int Hkv, int d, int P, sp_block_order order, int i, int j, float scale,
    sp_dtype dtype, void* out_blk, float* lse_blk, void* workspace, size_t workspace_bytes,
    sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_ring_block_step_accumulate");
  sp::g_last_launches = 0;
  if (P < 1 || i < 0 || i >= P || j < 0 || j >= P) return SP_ERR_INVALID_ARG;
  const int step = ((i - j) % P + P) % P;
  return sp::attn(q_blk, k_blk, v_blk, position_ids, B, B, S, Hq, Hkv, d, P, order, step,
                  step + 1, scale, dtype, out_blk, lse_blk, workspace, workspace_bytes, stream, i,
                  j, true);
}

extern "C" sp_status sp_query_block_attn_fwd(const void* q_blk, const void* k, const void* v,
                                             const int32_t* position_ids, int B, int S, int Hq,
                                             int Hkv, int d, int P, sp_block_order order, int i,
                                             float scale, sp_dtype dtype, void* out_blk,
                                             float* lse_blk, void* workspace,
                                             size_t workspace_bytes, sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_query_block_attn_fwd");
  sp::g_last_launches = 0;
  if (P < 1 || i < 0 || i >= P) return SP_ERR_INVALID_ARG;
  return sp::attn(q_blk, k, v, position_ids, B, B, S, Hq, Hkv, d, P, order, 0, P, scale, dtype,
                  out_blk, lse_blk, workspace, workspace_bytes, stream, i, -1);
}

extern "C" sp_status sp_get_device_error(void* workspace, int* code, sp_stream_t stream) {
  if (!workspace) return SP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SP_ERR_CUDA;
  if (code) *code = v;
  if (v != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return SP_ERR_CUDA;
    return SP_ERR_DEVICE_TIMEOUT;
  }
  return SP_OK;
}

extern "C" int sp_last_launch_count(void) { return sp::g_last_launches; }
