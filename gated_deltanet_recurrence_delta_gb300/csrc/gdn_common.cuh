// Shared device helpers of libgdn (sm_103a): argument bundle, status word,
// bf16 access, warp reductions, mbarrier / bulk-copy (TMA) wrappers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

using bf16 = __nv_bfloat16;

// MXFP8 token channels (decode variant): e4m3 elements, one E8M0 scale (a
// power of two, 2^(s-127)) per 32 consecutive channels of a token. All NULL
// for bf16 inputs.
struct MxInputs {
  const uint8_t *q, *k, *v, *z;          // [B][T][channels]
  const uint8_t *qs, *ks, *vs, *zs;      // [B][T][channels / 32]
};

// Everything a layer kernel needs, in device-pointer form.
struct LayerArgs {
  int B, T, nk, nv, D, G, C, n_slots;
  float scale, l2_eps, rms_eps;
  const bf16 *q, *k, *v, *z, *a, *b;
  const float *A_log, *dt_bias;
  const bf16 *conv_w, *norm_w;
  const float *mask;
  const int32_t *cu_seqlens;
  const int32_t *state_idx;
  bf16 *conv_state;     // [n_slots][3][C]
  float *state;         // [n_slots][nv][D][D]
  bf16 *out;
  unsigned int *status; // device status word (bit n = gdn_status n)
  MxInputs mx;          // MXFP8 q / k / v / z (decode variant); all NULL otherwise
  // prefill checkpoints: n_ckpt (row, position, slot) triples; the state and
  // conv tail of `row` after its first `position` tokens of the call go to
  // slot `slot` of ckpt_state [n_ckpt_slots][nv][D][D] / ckpt_conv
  // [n_ckpt_slots][3][C]. n_ckpt == 0: none.
  const int32_t *ckpt;
  int n_ckpt, n_ckpt_slots;
  float *ckpt_state;
  bf16 *ckpt_conv;
};

// Most checkpoints one row of a prefill call may request.
constexpr int kMaxRowCkpt = 64;

constexpr int KC = 3;  // saved conv rows (kernel width 4)

__device__ __forceinline__ void set_status(unsigned int *status, int code) {
  atomicOr(status, 1u << code);
}

__device__ __forceinline__ float ldbf(const bf16 *p) { return __bfloat162float(*p); }

// Slot of row r, or -1 (and a recorded error) when it is out of range.
__device__ __forceinline__ int row_slot(const LayerArgs &A, int r) {
  int s = A.state_idx ? A.state_idx[r] : r;
  if (s < 0 || s >= A.n_slots) return -1;
  return s;
}

// ---------------------------------------------------------------- warps

__device__ __forceinline__ float warp_sum_bcast(float x) {
  // Butterfly, then lane 0's value for everyone so that every consumer sees
  // the same bits whichever lane it reads.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
  return __shfl_sync(0xffffffffu, x, 0);
}

// ------------------------------------------------- mbarrier + bulk copy

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: returns false when the phase did not complete in time.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < (1u << 24); ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Wait for a phase with one polling thread: only `leader` spins on the
// mbarrier (many threads spinning would flood the shared-memory pipe the TMA
// and the other warps need); the rest sleep in the CTA barrier `sync_or`, then
// take one (immediately successful) acquire test of their own. Returns false,
// for every thread, when the leader's bounded wait expired.
template <class SyncOr>
__device__ __forceinline__ bool mbar_wait_leader(uint64_t *bar, uint32_t parity, bool leader, SyncOr sync_or) {
  bool ok = true;
  if (leader) ok = mbar_wait_bounded(bar, parity);
  if (sync_or(!ok)) return false;
  if (!leader) (void)mbar_try_wait(bar, parity);
  return true;
}

// One bulk global -> shared copy completing on `bar` (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Streaming (evict-first) 16-byte store.
// Bulk shared -> global copy (16-byte aligned, size % 16 == 0), tracked as a bulk group.
__device__ __forceinline__ void bulk_s2g(void *gmem_dst, const void *smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// The shared-memory sources of this thread's bulk stores may be overwritten.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void st_cs(float4 *p, float4 v) { __stcs(p, v); }

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before its predecessor in the stream completes;
// griddep_wait() blocks until the predecessor grid has completed and its memory
// is visible (a no-op for an ordinary launch). griddep_trigger() lets this
// grid's own dependent start once every CTA of this grid has issued it or
// exited. Each kernel here triggers only after its own wait, so a dependent's
// pre-wait code may rely on everything before this grid's predecessor.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace gdn
