// gdn_copy_overlapped: a few byte copies done by one kernel on the caller's
// stream, which starts while the kernel before it on that stream is still
// running (programmatic dependent launch) and completes only after it.
//
// The staging step of a decode loop fed from host memory: the next step's
// activations go up, and an earlier step's output rows come down, while the
// current step's kernel streams its state. Either side of a copy may be device
// memory or page-locked host memory mapped into the device's address space
// (read and written across NVLink-C2C on a Grace-Blackwell node). The copies
// are plain 16-byte loads and stores by all the CTAs, loads through L2 only
// (another SM may have written the source since this SM last cached it); no
// copy engine takes part, so nothing orders the stream's kernels against a
// copy engine's work.
#include "gdn_launch.h"

namespace gdn {

struct CopyList {
  const uint4 *src[GDN_MAX_OVERLAPPED_COPIES];
  uint4 *dst[GDN_MAX_OVERLAPPED_COPIES];
  size_t n16[GDN_MAX_OVERLAPPED_COPIES];  // 16-byte vectors of each copy
  int n;
};

__global__ void __launch_bounds__(256) overlapped_copy_kernel(const __grid_constant__ CopyList L) {
  griddep_trigger();  // the next kernel may launch; it still waits for this grid to complete
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t start = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int c = 0; c < L.n; ++c) {
    const uint4 *s = L.src[c];
    uint4 *d = L.dst[c];
    const size_t n = L.n16[c];
    size_t e = start;
    for (; e + 3 * stride < n; e += 4 * stride) {  // four loads in flight per thread
      const uint4 a0 = __ldcg(s + e), a1 = __ldcg(s + e + stride), a2 = __ldcg(s + e + 2 * stride),
                  a3 = __ldcg(s + e + 3 * stride);
      d[e] = a0;
      d[e + stride] = a1;
      d[e + 2 * stride] = a2;
      d[e + 3 * stride] = a3;
    }
    for (; e < n; e += stride) d[e] = __ldcg(s + e);
  }
  griddep_wait();  // this grid completes after the kernel before it on the stream
}

}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_copy_overlapped(const gdn_copy *copies, int32_t n, void *stream) {
  if (n < 0 || n > GDN_MAX_OVERLAPPED_COPIES) return fail(GDN_ERR_SHAPE, "copy count must be in [0, 8]");
  if (n > 0 && !copies) return fail(GDN_ERR_ARG, "copies is NULL");
  CopyList L = {};
  size_t most = 0;
  for (int c = 0; c < n; ++c) {
    const gdn_copy &cp = copies[c];
    if (cp.bytes == 0) continue;
    if (!cp.dst || !cp.src) return fail(GDN_ERR_ARG, "a copy's dst or src is NULL");
    if ((reinterpret_cast<uintptr_t>(cp.dst) | reinterpret_cast<uintptr_t>(cp.src) | cp.bytes) % 16 != 0)
      return fail(GDN_ERR_ARG, "copy addresses and sizes must be multiples of 16 bytes");
    L.src[L.n] = static_cast<const uint4 *>(cp.src);
    L.dst[L.n] = static_cast<uint4 *>(cp.dst);
    L.n16[L.n] = cp.bytes / 16;
    if (L.n16[L.n] > most) most = L.n16[L.n];
    ++L.n;
  }
  if (L.n == 0) return GDN_OK;
  const DeviceInfo *dev = nullptr;
  if (gdn_status st = current_device(&dev)) return st;
  // each thread moves about four vectors of the largest copy, at most one CTA per SM
  size_t grid = (most + 256 * 4 - 1) / (256 * 4);
  if (grid > (size_t)dev->sms) grid = (size_t)dev->sms;
  if (launch_pdl(overlapped_copy_kernel, dim3((unsigned)grid), dim3(256), 0, static_cast<cudaStream_t>(stream),
                 L) != cudaSuccess)
    return check_launch("copy_overlapped");
  return check_launch("copy_overlapped");
}
