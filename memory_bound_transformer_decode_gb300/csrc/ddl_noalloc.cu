// ddl_noalloc.cu -- ddl_stack_decode_noalloc: the decode step without a
// caller-supplied workspace, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a plugin whose host framework owns all
// device memory and hands it only the input and output buffers, or a loop that
// must not pay cudaMalloc's implicit device synchronization.  This entry point
// takes its scratch (barrier/status words, tile counters, partial sums, the
// residual hand-off between layers) from a file-scope device array of
// DDL_NOALLOC_SCRATCH_BYTES instead.  Every GPU that loads the library holds
// that array until the process exits.  All calls share the array: a call reuses
// whatever the previous call left there (the decode clears the words that must
// start at zero itself), and calls that overlap on the GPU race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "ddl_internal.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[DDL_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (in host code the array's name is only a stand-in, not a device
// address).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return ddl::cuda_status(e);
  if (dev < 0 || dev >= 64) return DDL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return ddl::cuda_status(e);
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return DDL_OK;
}

}  // namespace

extern "C" int ddl_stack_decode_noalloc(const ddl_shape* shape, ddl_wtype wtype,
                                        const ddl_layer_w* layers, const ddl_kv* kv, int32_t L,
                                        int32_t B, int64_t pos, const float* resid_in,
                                        const uint16_t* x_bf16, float* resid_out,
                                        uint16_t* out_bf16, void* stream) {
  if (!shape || !kv) return DDL_ERR_ARG;
  const size_t need = ddl_workspace_bytes(shape, B, kv[0].s_max);
  if (need > (size_t)DDL_NOALLOC_SCRATCH_BYTES) return DDL_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != DDL_OK) return st;
  return ddl_stack_decode(shape, wtype, layers, kv, L, B, pos, resid_in, x_bf16, resid_out, out_bf16,
                          scratch, (size_t)DDL_NOALLOC_SCRATCH_BYTES, stream);
}
