// mxq_noalloc.cu -- mx_quantize_rowcol_dbias_noalloc: the MXFP8 cast with
// dbias, taking its scratch from a device array the library owns instead of
// a caller-provided workspace.
//
// Some callers cannot hand the library a workspace: code that runs inside a
// framework which owns all device memory through its own pool (a cudaMalloc
// of ours would bypass that pool and synchronise the device), loops that
// forbid allocation once they have started, and plugin hosts that pass this
// library only the tensors it reads and writes.  For them this entry point
// keeps the dbias band sums in the array below, sized for a fixed maximum.
//
// Every GPU that loads the library holds the array (8 MiB) until the process
// exits.  All calls share it and it keeps the last call's contents; nothing
// in it needs clearing, because every word the kernels read from it was
// written earlier in the same call.  Calls that overlap on the GPU (on
// different streams, or on the same device from different threads without
// ordering) race on the array.

#include <cuda_runtime.h>

#include <cstdint>

#include "mxq.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;   // 8 MiB

// Device-side scratch.  In host code this name is only a handle for
// cudaGetSymbolAddress, never a device address.
static __device__ __align__(256) unsigned char g_dbias_scratch[kScratchBytes];

// Device address of the scratch array in the current context.  Looked up on
// every call, not cached: after cudaDeviceReset, or with another context
// current for the same device, the module is loaded again and the array may
// sit at another address.  The lookup is a host-side table search once the
// module is loaded; the first call on a device loads it, which is why that
// first call must come before any stream capture begins.
mxq_status scratch_on_current_device(void** addr) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_dbias_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();   // a failed lookup leaves no error behind for later calls
    return MXQ_ECUDA;
  }
  *addr = p;
  return MXQ_OK;
}

}  // namespace

extern "C" mxq_status mx_quantize_rowcol_dbias_noalloc(
    const void* x, int64_t M, int64_t K, int64_t ldx, uint32_t flags, uint8_t* q_row,
    uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, float* dbias, uint32_t* dev_err,
    mxq_stream_t stream) {
  if (flags & MXQ_ACT_GELU_TANH) return MXQ_EINVAL;
  const uint32_t f = flags | MXQ_DBIAS;
  // The band sums need mxq_workspace_bytes(...) bytes; larger shapes do not
  // fit the fixed array and are refused before anything is enqueued.
  if (mxq_workspace_bytes(MXQ_OP_ROWCOL, M, K, f) > kScratchBytes) return MXQ_EWORKSPACE;
  void* scratch = nullptr;
  const mxq_status st = scratch_on_current_device(&scratch);
  if (st != MXQ_OK) return st;
  return mx_quantize_rowcol(x, M, K, ldx, f, q_row, s_row, q_col, s_col, dbias, scratch,
                            kScratchBytes, dev_err, stream);
}
