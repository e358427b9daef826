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

#include "ddl_internal.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[DDL_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device (in host code
// the array's name is only a stand-in, not a device address).  It is looked up
// on every call, not cached: after cudaDeviceReset the module loads again and
// the array may move, and once the module is loaded the lookup is cheap.  The
// first lookup on a device loads the module, which is why the first call
// should come before any stream capture.
int scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return ddl::cuda_status(e);
  *out = p;
  return DDL_OK;
}

}  // namespace

namespace ddl {
// The scratch array's address for ddl_read_device_status (workspace NULL).
int noalloc_scratch(void** out) { return scratch_address(out); }
}  // namespace ddl

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
