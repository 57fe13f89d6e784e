// gdn_prefill_chunked_static_scratch: the chunked prefill with its scratch in
// a fixed device array of this library instead of a caller-supplied workspace.
//
// For callers that cannot allocate device memory: a serving engine whose pool
// has already claimed the free HBM and hands out only the tensors it manages,
// a C host program with no allocator of its own, or a latency-critical loop
// where a cudaMalloc could block, fail or synchronise the device.
//
// The scratch is one file-scope __device__ array of kStaticScratchBytes
// (64 MiB) per GPU. With lazy module loading (the CUDA default) the array is
// reserved on a GPU when this entry point first runs there and kept until the
// process exits; with CUDA_MODULE_LOADING=EAGER every GPU whose context the
// process creates reserves it at context creation, whether or not it ever
// calls this entry point. The cached device address stays valid for the life
// of the device's primary context: cudaDeviceReset must not be called while
// the library is in use. All calls on a device share it, and it keeps whatever
// the last call left there (the prefill overwrites every byte it reads, so
// nothing needs clearing). Two calls that overlap on the GPU (different
// streams, no ordering between them) race on it.
#include <mutex>

#include "gdn_launch.h"

namespace gdn {
namespace {

constexpr size_t kStaticScratchBytes = (size_t)64 << 20;

__device__ __align__(256) unsigned char g_prefill_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of this device's copy of the array. In host code the array's
// name is only a host-side stand-in, so the address comes from the runtime,
// once per device, with that device current.
gdn_status scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(GDN_ERR_CUDA, "no usable CUDA device");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_prefill_scratch);
    if (e != cudaSuccess || !p) return fail(GDN_ERR_CUDA, "cannot locate the static prefill scratch on this device");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GDN_OK;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_prefill_chunked_static_scratch(const gdn_dims *dims, const gdn_inputs *in,
                                                         void *conv_state, float *recurrent_state, void *out,
                                                         void *stream) {
  // the same host checks as gdn_prefill_chunked, before the array is touched:
  // a call that fails them, or has nothing to do, never loads it
  if (gdn_status st = validate_prefill(dims, in, conv_state, recurrent_state, out)) return st;
  if (dims->B == 0 || dims->T == 0) return GDN_OK;
  const size_t need =
      prefill_workspace_bytes(dims->B, dims->T, dims->nk, dims->nv, dims->dk, in->cu_seqlens != nullptr);
  if (need > kStaticScratchBytes)
    return fail(GDN_ERR_WORKSPACE,
                "this prefill needs more scratch than the 64 MiB static array holds; use gdn_prefill_chunked "
                "with a workspace");
  void *scratch = nullptr;
  if (gdn_status st = scratch_address(&scratch)) return st;
  return gdn_prefill_chunked(dims, in, conv_state, recurrent_state, out, scratch, kStaticScratchBytes, stream);
}
