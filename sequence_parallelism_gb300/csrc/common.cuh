// common.cuh -- host-side helpers shared by the entry points of the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "sp_gb300.h"

namespace sp {

// Kernels enqueued by the last successful call on this host thread.
extern thread_local int g_last_launches;

constexpr int kNumSMs = 152;           // GB300: 2 dies x 76 SMs (queried at run time too)
constexpr size_t kWsHeaderBytes = 256;  // error word + reserved, keeps arrays 256-aligned

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline size_t dtype_size(sp_dtype t) { return t == SP_BF16 ? 2 : (t == SP_F32 ? 4 : 0); }

// NVTX range around an entry point, named after it, so that a timeline
// (Nsight Systems) shows each library call; without an attached tool a push
// or pop is a test of a null function pointer.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

inline sp_status launch_status() {
  return cudaPeekAtLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

// Number of SMs of the current device (cached per process; every GB300
// reports the same count).
int device_sm_count();

// doc_start computation shared by sp_segment_starts and the attention entry
// points: fills doc_start[B][S] from position_ids using `scratch`
// (segment_scratch_bytes(B, S) bytes).  Returns the number of launches or -1.
size_t segment_scratch_bytes(int B, int S);
int launch_segment_starts(const int32_t* position_ids, int32_t* doc_start, int B, int S,
                          void* scratch, cudaStream_t stream);

}  // namespace sp
