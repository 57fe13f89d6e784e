// gdn_decode_step: one token for B rows, in place.
//
// The step is bound by HBM traffic on the fp32 state (2 x D*D*4 bytes per
// (row, value head)). Design:
//   * persistent grid, one CTA per SM; a CTA walks its units (row, key head)
//     round-robin; a unit is the G value heads that read one key head, so the
//     conv tail of the unit's q/k channels is read and rewritten by this CTA
//     alone (no cross-CTA hazard on the in-place tail);
//   * each value head's state (one contiguous D*D fp32 block) is streamed into
//     a ring of NS shared-memory stages by one bulk copy (cp.async.bulk, TMA
//     engine) completing on an mbarrier; thread 0 refills a stage as soon as
//     every thread has taken its slice into registers, so NS-1 heads are in
//     flight while one is computed;
//   * the new state goes straight from registers to HBM with streaming stores.
// The per-token arithmetic is the shared code of gdn_token.cuh.
#include "gdn_launch.h"
#include "gdn_token.cuh"

namespace gdn {

constexpr int kMaxG = 8;

template <int D, int NS>
struct DecodeSmem {
  static constexpr int kStage = D * D;                          // floats per stage
  static constexpr int kRed = 2 * 2 * StateLayout<D>::NG * D;   // [parity][k|q][NG][D]
  static constexpr int kFront = (2 + kMaxG) * D + 4 * kMaxG;    // q, k, v[G], gates
  static constexpr size_t kBytes = sizeof(float) * (size_t)(NS * kStage + kRed + kFront) + 8 * NS;
};

template <int D, int NS>
__global__ void __launch_bounds__(256, 1) decode_kernel(LayerArgs A) {
  using L = StateLayout<D>;
  using S = DecodeSmem<D, NS>;
  extern __shared__ __align__(128) float smem[];
  float *stage = smem;
  float *red = stage + NS * S::kStage;
  float *fq = red + S::kRed;
  float *fk = fq + D;
  float *fv = fk + D;                  // [G][D]
  float *fdecay = fv + kMaxG * D;      // [G]
  float *fbeta = fdecay + kMaxG;       // [G]
  float *fbkq = fbeta + kMaxG;         // [G]
  uint64_t *full = reinterpret_cast<uint64_t *>(fbkq + 2 * kMaxG);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = A.G, kd = A.nk * D;
  const int n_units = A.B * A.nk;
  if ((int)blockIdx.x >= n_units) return;
  const int my_units = (n_units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int n_tasks = my_units * G;

  // Task n of this CTA -> (row b, key head kh, value head h); -1 slot = skip.
  auto task = [&](int n, int &b, int &kh, int &h) {
    const int u = (int)blockIdx.x + (n / G) * (int)gridDim.x;
    b = u / A.nk;
    kh = u % A.nk;
    h = kh * G + n % G;
  };
  // Slot of an active row, else -1 (bad slot or bad mask value recorded; mask 0 = skip).
  auto active_slot = [&](int b, bool record) -> int {
    if (A.mask) {
      const float m = A.mask[b];
      if (m != 1.0f) {
        if (m != 0.0f && record) set_status(A.status, GDN_ERR_MASK);
        return -1;
      }
    }
    const int s = row_slot(A, b);
    if (s < 0 && record) set_status(A.status, GDN_ERR_INDEX);
    return s;
  };
  auto issue = [&](int n) {  // thread 0 only
    int b, kh, h;
    task(n, b, kh, h);
    const int slot = active_slot(b, false);
    uint64_t *bar = &full[n % NS];
    if (slot >= 0) {
      mbar_arrive_expect_tx(bar, D * D * 4);
      bulk_g2s(stage + (n % NS) * S::kStage, A.state + ((size_t)slot * A.nv + h) * D * D, D * D * 4, bar);
    } else {
      mbar_arrive(bar);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int n = 0; n < NS && n < n_tasks; ++n) issue(n);

  for (int n = 0; n < n_tasks; ++n) {
    int b, kh, h;
    task(n, b, kh, h);
    const int j = n % G;
    const int slot = active_slot(b, j == 0 && tid == 0);

    if (j == 0 && slot >= 0) {
      // ---- unit front end: conv (+ in-place tail shift), L2 norms, gates
      __syncthreads();  // the previous unit is done with fq / fk / fv
      bf16 *cs = A.conv_state + (size_t)slot * KC * A.C;
      const int nch = (2 + G) * D;
      for (int e = tid; e < nch; e += 256) {
        int ch;
        const bf16 *src;
        if (e < D) {
          ch = kh * D + e;
          src = A.q + (size_t)b * kd + ch;
        } else if (e < 2 * D) {
          ch = kd + kh * D + (e - D);
          src = A.k + (size_t)b * kd + (ch - kd);
        } else {
          ch = 2 * kd + kh * G * D + (e - 2 * D);
          src = A.v + (size_t)b * A.nv * D + (ch - 2 * kd);
        }
        const bf16 x0 = cs[ch], x1 = cs[A.C + ch], x2 = cs[2 * A.C + ch], x3 = *src;
        const bf16 *w = A.conv_w + (size_t)ch * 4;
        const float y = conv4_silu(ldbf(w), ldbf(w + 1), ldbf(w + 2), ldbf(w + 3), __bfloat162float(x0),
                                   __bfloat162float(x1), __bfloat162float(x2), __bfloat162float(x3));
        fq[e] = y;  // fq, fk, fv are contiguous
        cs[ch] = x1;
        cs[A.C + ch] = x2;
        cs[2 * A.C + ch] = x3;
      }
      __syncthreads();
      if (warp == 0) warp_l2norm<D>(fq, A.l2_eps, A.scale, lane);
      if (warp == 1) warp_l2norm<D>(fk, A.l2_eps, 1.0f, lane);
      __syncthreads();
      if (warp == 0) {
        const float kq = warp_dot<D>(fq, fk, lane);
        if (lane < G) {
          const int hh = kh * G + lane;
          float decay, beta;
          gdn_gates(ldbf(A.a + (size_t)b * A.nv + hh), ldbf(A.b + (size_t)b * A.nv + hh), A.A_log[hh],
                    A.dt_bias[hh], decay, beta);
          fdecay[lane] = decay;
          fbeta[lane] = beta;
          fbkq[lane] = __fmul_rn(beta, kq);
        }
      }
      __syncthreads();
    }

    // ---- the value head's state
    const bool ok = mbar_wait_bounded(&full[n % NS], (uint32_t)((n / NS) & 1));
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        set_status(A.status, GDN_ERR_TIMEOUT);
        for (int m = n; m < n + NS && m < n_tasks; ++m)
          (void)mbar_wait_bounded(&full[m % NS], (uint32_t)((m / NS) & 1));
      }
      return;
    }
    bf16 *out = A.out + ((size_t)b * A.nv + h) * D;
    if (slot >= 0) {
      const int cq = tid % L::TPR, grp = tid / L::TPR;
      const float4 *st = reinterpret_cast<const float4 *>(stage + (n % NS) * S::kStage);
      float4 s[L::RPT];
#pragma unroll
      for (int i = 0; i < L::RPT; ++i) s[i] = st[(grp + i * L::NG) * L::TPR + cq];
      float4 o;
      state_step<D>(s, fq, fk, fv + j * D, fdecay[j], fbeta[j], fbkq[j], red + (n & 1) * 2 * L::NG * D, tid, o);
      // every thread holds its slice: the stage may be refilled
      if (tid == 0 && n + NS < n_tasks) {
        fence_proxy_async_smem();
        issue(n + NS);
      }
      float4 *gs = reinterpret_cast<float4 *>(A.state + ((size_t)slot * A.nv + h) * D * D);
#pragma unroll
      for (int i = 0; i < L::RPT; ++i) st_cs(gs + (grp + i * L::NG) * L::TPR + cq, s[i]);
      if (warp == 0) rmsnorm_store<D>(o, lane, A.z + ((size_t)b * A.nv + h) * D, A.norm_w, A.rms_eps, out);
    } else {
      if (tid == 0 && n + NS < n_tasks) issue(n + NS);
      zero_head<D>(out, tid);
    }
  }
}

template <int D, int NS>
static gdn_status launch_decode_t(const LayerArgs &A, cudaStream_t stream) {
  using S = DecodeSmem<D, NS>;
  const DeviceInfo &dev = device_info();
  static bool attr_set[kMaxDevices] = {};
  if (!attr_set[dev.id]) {
    if (cudaFuncSetAttribute(decode_kernel<D, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::kBytes) !=
        cudaSuccess)
      return fail(GDN_ERR_CUDA, "decode: cannot reserve shared memory");
    attr_set[dev.id] = true;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<D, NS>, 256, S::kBytes) != cudaSuccess ||
      per_sm < 1)
    return fail(GDN_ERR_CUDA, "decode: kernel does not fit on an SM");
  const int n_units = A.B * A.nk;
  const int grid = n_units < dev.sms * per_sm ? n_units : dev.sms * per_sm;
  decode_kernel<D, NS><<<grid, 256, S::kBytes, stream>>>(A);
  return check_launch("decode");
}

gdn_status launch_decode(const LayerArgs &A, cudaStream_t stream) {
  switch (A.D) {
    case 128: return launch_decode_t<128, 3>(A, stream);
    case 64: return launch_decode_t<64, 4>(A, stream);
    case 32: return launch_decode_t<32, 4>(A, stream);
  }
  return fail(GDN_ERR_SHAPE, "decode: unsupported head size");
}

}  // namespace gdn
