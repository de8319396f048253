// noalloc.cu -- blockwise attention for callers that cannot allocate device
// memory.
//
// sp_blockwise_attn_fwd needs a caller-provided workspace (the device error
// word, the doc_start array and the scratch of its scan).  Some callers have
// no way to provide one: code running where cudaMalloc is off limits (inside
// a host callback or a driver/plugin hook that must not allocate, under an
// allocator that only hands out the caller's own tensors, or a framework
// that forbids hidden allocations on its stream).  For them this file keeps
// the workspace in a fixed-size array with static storage on the device.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds kNoAllocScratchBytes of it until the process exits.  In host
// code its name is only a host-side stand-in for the symbol, so the device
// address is obtained once per device with cudaGetSymbolAddress (with that
// device current) and cached.  The first call on each device does that
// lookup, so make it before capturing any stream into a CUDA graph.
//
// Every call shares the one array per device and the array keeps the last
// call's contents: the error word is cleared by each call and doc_start is
// rewritten in full, so nothing stale is read -- but two calls whose kernels
// overlap on the GPU (different streams, no ordering between them) race on
// the array.  The device error word lives in the array as well and cannot be
// read back through this entry point.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace sp {
namespace {

// 256 B header (error word) + doc_start for up to 2^20 tokens (4 MiB) + the
// doc_start scan's per-chunk maxima, with room to spare.
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(5) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up on
// the first call for that device, then cached).  nullptr on failure.
void* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace sp

extern "C" sp_status sp_blockwise_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                                   const int32_t* position_ids, int B, int S,
                                                   int Hq, int Hkv, int d, int P,
                                                   sp_block_order order, float scale,
                                                   sp_dtype dtype, void* out, float* lse,
                                                   sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_blockwise_attn_fwd_noalloc");
  sp::g_last_launches = 0;
  if (B < 1 || S < 1) return SP_ERR_INVALID_ARG;
  const size_t need = sp_blockwise_attn_workspace_bytes(B, S, position_ids != nullptr);
  if (need == 0 || need > sp::kNoAllocScratchBytes) return SP_ERR_WORKSPACE;
  void* ws = sp::scratch_for_current_device();
  if (!ws) return SP_ERR_CUDA;
  return sp_blockwise_attn_fwd(q, k, v, position_ids, B, S, Hq, Hkv, d, P, order, scale, dtype,
                               out, lse, ws, sp::kNoAllocScratchBytes, stream);
}
