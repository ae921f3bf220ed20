// ssm_noalloc.cu -- the selective scan for callers that cannot allocate device memory.
//
// Some callers own only their inputs and outputs: a host framework's plugin interface that
// hands this library tensor pointers but no workspace, or a latency-critical serving loop
// that must not call cudaMalloc (an allocation can block on device-wide synchronisation).
// For them the scan's chunk-carry scratch lives in a fixed, file-scope device array instead
// of a caller-provided workspace.
//
// The array costs SSM_NOALLOC_SCRATCH_BYTES of memory on every GPU that loads the library,
// held until the process exits. In host code the array's name is only a host-side stand-in,
// so its device address is looked up with cudaGetSymbolAddress, with the caller's device
// current. The first call on a device is the set-up: it loads the library's device code
// into that device's context (which is why it should come before any stream capture).
// Later calls repeat the lookup, which is a table lookup in the CUDA runtime and allocates
// nothing; an address cached across calls could go stale once the context is destroyed
// (cudaDeviceReset) and the module is loaded again at another address.
#include <cuda_runtime.h>

#include "../../include/ssm.h"

namespace {

static __device__ __align__(256) unsigned char g_scan_scratch[SSM_NOALLOC_SCRATCH_BYTES];

// Device address of g_scan_scratch in the current device's context.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&p, g_scan_scratch);
  if (err != cudaSuccess) return err;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" ssm_status ssm_selective_scan_fwd_noalloc(
    const void* x, const void* delta, const float* A, const void* B, const void* C, const float* D, const void* z,
    const float* delta_bias, int delta_softplus, const float* conv_w, const float* conv_b, int d_conv,
    const void* conv_init, const float* h0, void* out, float* h_last, void* conv_state_out, int batch, int dim,
    int seqlen, int dstate, ssm_dtype io, int chunk_len, unsigned int flags, void* stream) {
  // An explicit chunk length whose carries do not fit the fixed scratch is refused before
  // anything runs; with chunk_len = 0 the scan lowers its chunk count to fit.
  if (chunk_len > 0 && batch > 0 && dim > 0 && seqlen > 0 &&
      ssm_scan_workspace_bytes(batch, dim, seqlen, dstate, chunk_len, io) > (size_t)SSM_NOALLOC_SCRATCH_BYTES)
    return SSM_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if ((long long)batch * dim > 0 && seqlen > 0) {
    if (scratch_address(&scratch) != cudaSuccess) {
      cudaGetLastError();
      return SSM_ERR_CUDA;
    }
  }
  return ssm_selective_scan_fwd(x, delta, A, B, C, D, z, delta_bias, delta_softplus, conv_w, conv_b, d_conv,
                                conv_init, h0, out, h_last, conv_state_out, batch, dim, seqlen, dstate, io,
                                chunk_len, scratch, scratch ? (size_t)SSM_NOALLOC_SCRATCH_BYTES : 0, flags, stream);
}
