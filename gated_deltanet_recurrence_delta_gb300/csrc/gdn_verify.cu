// gdn_verify_with_checkpoints: T <= 8 draft tokens per row from a read-only
// saved state, emitting the state and the conv tail after every token
// (generate.py, sparkle mlx_streaming/mtp: the verify forward keeps per-token
// gated-delta checkpoints so that an accepted prefix is committed directly).
//
// One CTA per (row, value head). The state slice lives in registers for all T
// tokens; each token's checkpoint (D*D fp32) streams to HBM from registers, so
// the kernel is bound by the checkpoint writes. The per-token arithmetic is the
// shared code of gdn_token.cuh, which makes checkpoint t bit-identical to the
// state after t+1 gdn_decode_step calls.
#include "gdn_launch.h"
#include "gdn_token.cuh"

namespace gdn {

constexpr int kMaxVerifyT = 8;

template <int D>
struct VerifySmem {
  static constexpr int kFront = kMaxVerifyT * 4 * D;          // [t][q|k|v|z][D]
  static constexpr int kRed = StepScratch<D>::kFloats;
  static constexpr int kGates = 3 * kMaxVerifyT;
  static constexpr size_t kBytes = sizeof(float) * (size_t)(kFront + kRed + kGates + D) + 16;
};

template <int D>
__global__ void __launch_bounds__(256, 2) verify_kernel(LayerArgs A, float *ckpt_state, bf16 *ckpt_conv) {
  using L = StateLayout<D>;
  using S = VerifySmem<D>;
  extern __shared__ __align__(128) float smem[];
  float *F = smem;                       // [T][3][D] conv outputs (q, k, v)
  float *Z = F + kMaxVerifyT * 3 * D;    // [T][D] output gate
  float *red = F + S::kFront;
  float *gdecay = red + S::kRed;         // [T]
  float *gbeta = gdecay + kMaxVerifyT;   // [T]
  float *gbkq = gbeta + kMaxVerifyT;     // [T]
  float *fw = gbkq + kMaxVerifyT;        // [D] norm weight
  __shared__ int s_Lr;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / A.nv, h = blockIdx.x % A.nv, kh = h / A.G;
  const int T = A.T, kd = A.nk * D, C = A.C;

  const int slot = row_slot(A, b);
  if (slot < 0) {
    if (tid == 0) set_status(A.status, GDN_ERR_INDEX);
    return;
  }
  // ---- the state slice, in flight while the front end runs
  const int cq = tid % L::TPR, grp = tid / L::TPR;
  const float4 *gs = reinterpret_cast<const float4 *>(A.state + ((size_t)slot * A.nv + h) * D * D);
  float4 s[L::RPT];
#pragma unroll
  for (int i = 0; i < L::RPT; ++i) s[i] = __ldg(gs + (grp + i * L::NG) * L::TPR + cq);

  // gates of token tid (they do not depend on the conv)
  if (tid < T) {
    const size_t gi = ((size_t)b * T + tid) * A.nv + h;
    float decay, beta;
    gdn_gates(ldbf(A.a + gi), ldbf(A.b + gi), A.A_log[h], A.dt_bias[h], decay, beta);
    gdecay[tid] = decay;
    gbeta[tid] = beta;
  }
  if (tid == 0) {
    // The mask row must be ones then zeros; Lr = number of leading ones.
    int Lr = T;
    bool bad = false;
    if (A.mask) {
      const float *m = A.mask + (size_t)b * T;
      Lr = 0;
      while (Lr < T && m[Lr] == 1.0f) ++Lr;
      for (int t = Lr; t < T; ++t) bad |= (m[t] != 0.0f);
    }
    if (bad) set_status(A.status, GDN_ERR_MASK);
    s_Lr = bad ? -1 : Lr;
  }
  __syncthreads();
  const int Lr = s_Lr;
  if (Lr < 0) return;

  // ---- front end for every token: conv over xin = [tail ; x], SiLU
  for (int e = tid; e < T * D; e += 256) Z[e] = ldbf(A.z + (((size_t)b * T + e / D) * A.nv + h) * D + e % D);
  for (int c = tid; c < D; c += 256) fw[c] = ldbf(A.norm_w + c);
  const bf16 *cs = A.conv_state + (size_t)slot * KC * C;
  const bool write_qk_tail = (h % A.G) == 0;  // one writer per key head's channels
  for (int e = tid; e < T * 3 * D; e += 256) {
    const int t = e / (3 * D), c = e % (3 * D), which = c / D, cc = c % D;
    int ch;
    const bf16 *src;
    size_t rstride;
    if (which == 0) {
      ch = kh * D + cc;
      src = A.q + (size_t)b * T * kd + ch;
      rstride = kd;
    } else if (which == 1) {
      ch = kd + kh * D + cc;
      src = A.k + (size_t)b * T * kd + (ch - kd);
      rstride = kd;
    } else {
      ch = 2 * kd + h * D + cc;
      src = A.v + (size_t)b * T * A.nv * D + (ch - 2 * kd);
      rstride = (size_t)A.nv * D;
    }
    // xin row r: r < 3 from the saved tail, else token r - 3
    float xr[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = t + j;
      xr[j] = r < KC ? ldbf(cs + (size_t)r * C + ch) : ldbf(src + (size_t)(r - KC) * rstride);
    }
    const bf16 *w = A.conv_w + (size_t)ch * 4;
    F[(t * 3 + which) * D + cc] =
        conv4_silu(ldbf(w), ldbf(w + 1), ldbf(w + 2), ldbf(w + 3), xr[0], xr[1], xr[2], xr[3]);
    // conv checkpoint after token t: xin rows min(t+1, Lr) .. +2
    if (which == 2 || write_qk_tail) {
      const int e0 = t + 1 < Lr ? t + 1 : Lr;
      bf16 *dst = ckpt_conv + ((size_t)b * T + t) * KC * C + ch;
#pragma unroll
      for (int r = 0; r < KC; ++r) {
        const int xi = e0 + r;
        dst[(size_t)r * C] = xi < KC ? cs[(size_t)xi * C + ch] : src[(size_t)(xi - KC) * rstride];
      }
    }
  }
  __syncthreads();
  for (int vec = warp; vec < 2 * T; vec += 8) {
    const int t = vec >> 1, which = vec & 1;
    warp_l2norm<D>(F + (t * 3 + which) * D, A.l2_eps, which == 0 ? A.scale : 1.0f, lane);
  }
  __syncthreads();
  for (int t = warp; t < T; t += 8) {
    const float kq = warp_dot<D>(F + (t * 3) * D, F + (t * 3 + 1) * D, lane);
    if (lane == 0) gbkq[t] = __fmul_rn(gbeta[t], kq);
  }
  __syncthreads();

  // ---- the state: registers for all T tokens, a checkpoint after each
  for (int t = 0; t < T; ++t) {
    bf16 *out = A.out + (((size_t)b * T + t) * A.nv + h) * D;
    if (t < Lr) {
      float4 o;
      state_step<D>(s, F + (t * 3) * D, F + (t * 3 + 1) * D, F + (t * 3 + 2) * D, gdecay[t], gbeta[t], gbkq[t],
                    red, tid, o, SyncAll());
      if (warp == 0) rmsnorm_store_smem<D>(o, lane, Z + t * D, fw, A.rms_eps, out);
    } else {
      zero_head<D>(out, tid);
    }
    float4 *ck = reinterpret_cast<float4 *>(ckpt_state + (((size_t)b * T + t) * A.nv + h) * D * D);
#pragma unroll
    for (int i = 0; i < L::RPT; ++i) st_cs(ck + (grp + i * L::NG) * L::TPR + cq, s[i]);
  }
}

template <int D>
static gdn_status launch_verify_t(const LayerArgs &A, float *ckpt_state, bf16 *ckpt_conv, cudaStream_t stream) {
  using S = VerifySmem<D>;
  const DeviceInfo &dev = device_info();
  static bool attr_set[kMaxDevices] = {};
  if (!attr_set[dev.id]) {
    if (cudaFuncSetAttribute(verify_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::kBytes) !=
        cudaSuccess)
      return fail(GDN_ERR_CUDA, "verify: cannot reserve shared memory");
    attr_set[dev.id] = true;
  }
  verify_kernel<D><<<A.B * A.nv, 256, S::kBytes, stream>>>(A, ckpt_state, ckpt_conv);
  return check_launch("verify");
}

gdn_status launch_verify(const LayerArgs &A, float *ckpt_state, bf16 *ckpt_conv, cudaStream_t stream) {
  switch (A.D) {
    case 128: return launch_verify_t<128>(A, ckpt_state, ckpt_conv, stream);
    case 64: return launch_verify_t<64>(A, ckpt_state, ckpt_conv, stream);
    case 32: return launch_verify_t<32>(A, ckpt_state, ckpt_conv, stream);
  }
  return fail(GDN_ERR_SHAPE, "verify: unsupported head size");
}

}  // namespace gdn
