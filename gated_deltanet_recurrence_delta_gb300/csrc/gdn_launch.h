// Host-side plumbing shared by the launchers of libgdn (not part of the C-ABI).
#pragma once

#include <atomic>
#include <utility>

#include "gdn_common.cuh"

namespace gdn {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int id;
  int sms;                 // streaming multiprocessors
  unsigned int *status;    // device address of this device's status word
};

// Per-device facts of the current device, set up on first use (SM count and
// the status word's device address). Returns GDN_OK or GDN_ERR_CUDA.
gdn_status current_device(const DeviceInfo **out);
// The current device's info; valid only after current_device() succeeded.
const DeviceInfo &device_info();

// Record `msg` as this thread's last error and return `code`.
gdn_status fail(gdn_status code, const char *msg);
// GDN_OK, or GDN_ERR_CUDA with the launch error of `what`.
gdn_status check_launch(const char *what);

// Launch with programmatic stream serialization: the kernel may start before
// its predecessor in the stream completes and calls griddep_wait() before it
// touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Host checks of a prefill call (dims, inputs, pointers, token count), as
// gdn_prefill_chunked runs them before anything else: GDN_OK or the error.
gdn_status validate_prefill(const gdn_dims *dims, const gdn_inputs *in, const void *conv_state,
                            const float *recurrent_state, const void *out);

gdn_status launch_decode(const LayerArgs &A, cudaStream_t stream);
gdn_status launch_verify(const LayerArgs &A, float *ckpt_state, bf16 *ckpt_conv, cudaStream_t stream);
size_t prefill_workspace_bytes(int B, int T, int nk, int nv, int D, bool packed);
gdn_status launch_prefill(const LayerArgs &A, void *workspace, size_t workspace_bytes, cudaStream_t stream);
size_t prefill_tc_workspace_bytes(int B, int T, int nk, int nv, bool packed);
gdn_status launch_prefill_tc(const LayerArgs &A, void *workspace, cudaStream_t stream);
gdn_status launch_commit(const float *ckpt_state, const bf16 *ckpt_conv, float *pool_state, bf16 *pool_conv,
                         const int32_t *accept_len, const int32_t *dst_slot, int32_t *winner, int B, int T,
                         int paths, int n_layers, int n_slots, size_t state_floats, size_t conv_elems,
                         cudaStream_t stream);
gdn_status launch_state_copy(const float *src_state, const bf16 *src_conv, float *dst_state, bf16 *dst_conv,
                             const int32_t *src_slot, const int32_t *dst_slot, int n, int n_src, int n_dst,
                             size_t state_floats, size_t conv_elems, cudaStream_t stream);

}  // namespace gdn
