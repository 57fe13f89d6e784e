// gdn_state_copy: dst[dst_slot[i]] <- src[src_slot[i]] for (state, conv tail)
// slot pairs, the commit of an accepted verify prefix (generate.py, sparkle:
// commit_tree_row) and the O(1) state bridge (uni_engine.py,
// Qwen3.5-9B-SpeedX9-GDN32: copy_cache_ copies in place, addresses preserved).
// A plain HBM copy: 16-byte vector loads and streaming stores, grid sized to
// the SM count. Slot indices are device data, so a commit chosen on the GPU
// needs no host round trip.
#include "gdn_launch.h"

namespace gdn {

// One slot pair: the state (state_vec float4) and, when given, the conv tail
// (conv_vec 16-byte vectors), copied by the gridDim.x CTAs of one grid row.
__device__ __forceinline__ void copy_slot(const float4 *__restrict__ s, float4 *__restrict__ d, size_t state_vec,
                                          const uint4 *__restrict__ sc, uint4 *__restrict__ dc, size_t conv_vec) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t start = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  size_t e = start;
  // four independent 16-byte loads in flight per thread
  for (; e + 3 * stride < state_vec; e += 4 * stride) {
    const float4 a0 = __ldg(s + e), a1 = __ldg(s + e + stride), a2 = __ldg(s + e + 2 * stride),
                 a3 = __ldg(s + e + 3 * stride);
    __stcs(d + e, a0);
    __stcs(d + e + stride, a1);
    __stcs(d + e + 2 * stride, a2);
    __stcs(d + e + 3 * stride, a3);
  }
  for (; e < state_vec; e += stride) __stcs(d + e, __ldg(s + e));
  if (sc)
    for (size_t c = start; c < conv_vec; c += stride) dc[c] = __ldg(sc + c);
}

__global__ void __launch_bounds__(256) state_copy_kernel(const float4 *__restrict__ src_state,
                                                         const uint4 *__restrict__ src_conv,
                                                         float4 *__restrict__ dst_state, uint4 *__restrict__ dst_conv,
                                                         const int32_t *src_slot, const int32_t *dst_slot, int n_src,
                                                         int n_dst, size_t state_vec, size_t conv_vec,
                                                         unsigned int *status) {
  griddep_wait();  // the kernel before this call (e.g. the verify that wrote the checkpoints) is complete
  griddep_trigger();
  const int i = blockIdx.y;
  const int ss = src_slot[i], ds = dst_slot[i];
  if (ss == -1) return;  // nothing to commit for this pair
  if (ss < 0 || ss >= n_src || ds < 0 || ds >= n_dst) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, GDN_ERR_INDEX);
    return;
  }
  copy_slot(src_state + (size_t)ss * state_vec, dst_state + (size_t)ds * state_vec, state_vec,
            src_conv ? src_conv + (size_t)ss * conv_vec : nullptr, dst_conv + (size_t)ds * conv_vec, conv_vec);
}

// The commit of a verify call for every layer of a stack: grid row (group g,
// layer l) finds its group's winner -- the first of its `paths` rows with the
// longest accept length -- and copies that row's checkpoint after its L
// accepted tokens (slot winner*T + L - 1 of layer l's checkpoints) into the
// group's pool slot of layer l. L = 0 copies nothing.
__global__ void __launch_bounds__(256) commit_kernel(const float4 *__restrict__ ckpt_state,
                                                     const uint4 *__restrict__ ckpt_conv, float4 *__restrict__ pool_state,
                                                     uint4 *__restrict__ pool_conv, const int32_t *accept_len,
                                                     const int32_t *dst_slot, int32_t *winner_out, int B, int T,
                                                     int paths, int n_groups, int n_slots, size_t state_vec,
                                                     size_t conv_vec, unsigned int *status) {
  griddep_wait();  // the verify calls that wrote the checkpoints are complete
  griddep_trigger();
  const int g = blockIdx.y % n_groups, l = blockIdx.y / n_groups;
  int win = -1, best = -1;
  bool bad = false;
  for (int p = 0; p < paths; ++p) {  // first maximum: ties go to the lower row
    const int L = accept_len[g * paths + p];
    if (L < 0 || L > T) bad = true;
    if (L > best) {
      best = L;
      win = p;
    }
  }
  const int ds = dst_slot[g];
  if (bad || ds < 0 || ds >= n_slots) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, GDN_ERR_INDEX);
    if (winner_out && l == 0 && blockIdx.x == 0 && threadIdx.x == 0) winner_out[g] = -1;
    return;
  }
  if (winner_out && l == 0 && blockIdx.x == 0 && threadIdx.x == 0) winner_out[g] = g * paths + win;
  if (best == 0) return;  // nothing accepted: the state stays as it was
  const size_t src = (size_t)l * B * T + (size_t)(g * paths + win) * T + (best - 1);
  const size_t dst = (size_t)l * n_slots + ds;
  copy_slot(ckpt_state + src * state_vec, pool_state + dst * state_vec, state_vec,
            ckpt_conv ? ckpt_conv + src * conv_vec : nullptr, pool_conv + dst * conv_vec, conv_vec);
}

gdn_status launch_commit(const float *ckpt_state, const bf16 *ckpt_conv, float *pool_state, bf16 *pool_conv,
                         const int32_t *accept_len, const int32_t *dst_slot, int32_t *winner, int B, int T,
                         int paths, int n_layers, int n_slots, size_t state_floats, size_t conv_elems,
                         cudaStream_t stream) {
  const DeviceInfo &dev = device_info();
  const size_t state_vec = state_floats / 4, conv_vec = conv_elems / 8;
  const int n_groups = B / paths, rows = n_groups * n_layers;
  // each grid row streams one slot pair; together about four CTAs per SM
  size_t want = (state_vec + 256 * 4 - 1) / (256 * 4);
  size_t cap = (size_t)dev.sms * 4 / (size_t)rows;
  if (cap < 1) cap = 1;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  if (launch_pdl(commit_kernel, dim3((unsigned)want, (unsigned)rows), dim3(256), 0, stream,
                 reinterpret_cast<const float4 *>(ckpt_state), reinterpret_cast<const uint4 *>(ckpt_conv),
                 reinterpret_cast<float4 *>(pool_state), reinterpret_cast<uint4 *>(pool_conv), accept_len, dst_slot,
                 winner, B, T, paths, n_groups, n_slots, state_vec, conv_vec, dev.status) != cudaSuccess)
    return check_launch("commit");
  return check_launch("commit");
}

gdn_status launch_state_copy(const float *src_state, const bf16 *src_conv, float *dst_state, bf16 *dst_conv,
                             const int32_t *src_slot, const int32_t *dst_slot, int n, int n_src, int n_dst,
                             size_t state_floats, size_t conv_elems, cudaStream_t stream) {
  const DeviceInfo &dev = device_info();
  const size_t state_vec = state_floats / 4, conv_vec = conv_elems / 8;
  // enough CTAs to keep every SM streaming; each thread moves >= 4 vectors
  size_t want = (state_vec + 256 * 4 - 1) / (256 * 4);
  size_t cap = (size_t)dev.sms * 4 / (size_t)n;
  if (cap < 1) cap = 1;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  dim3 grid((unsigned)want, (unsigned)n);
  if (launch_pdl(state_copy_kernel, grid, dim3(256), 0, stream, reinterpret_cast<const float4 *>(src_state),
                 reinterpret_cast<const uint4 *>(src_conv), reinterpret_cast<float4 *>(dst_state),
                 reinterpret_cast<uint4 *>(dst_conv), src_slot, dst_slot, n_src, n_dst, state_vec, conv_vec,
                 dev.status) != cudaSuccess)
    return check_launch("state_copy");
  return check_launch("state_copy");
}

}  // namespace gdn
