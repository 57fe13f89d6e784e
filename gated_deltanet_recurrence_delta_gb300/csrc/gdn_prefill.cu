// gdn_prefill_chunked: B rows (dense or packed with cu_seqlens) continuing
// from their saved conv tail and fp32 state, in place.
// statecache.py (squad-0.8b): CacheQwen35._gdn inside StateCache's chunk
// graphs -- rows continue from a saved state, padding is masked by
// g = beta = 0 so the state stops at the real end, and the conv tail keeps the
// last K-1 real inputs.
//
// Head size 128 runs the chunked tensor-core path (gdn_prefill_tc.cu). Head
// sizes 32 and 64 run the kernels below:
//   1. front: depthwise conv + SiLU over [saved tail ; tokens] and the q/k L2
//      norm, for every (token block, head channel group); results to the
//      workspace (fp32). Reads the saved tail, writes nothing in place.
//   2. recur: one CTA per (row, value head): the delta rule token by token
//      with the state in registers, the gated RMSNorm epilogue, requested
//      checkpoints, the final state in place, then the conv-tail update of the
//      channels it owns.
// Kernel 2 starts only after kernel 1 has read every saved tail (stream order),
// so the in-place tail update cannot race with the conv.
#include "gdn_launch.h"
#include "gdn_token.cuh"

namespace gdn {

namespace {

constexpr int kFrontTB = 32;  // tokens per front-end CTA

struct PrefillWs {
  float *qn, *kn, *vv;  // [Ttot][nk][D], [Ttot][nk][D], [Ttot][nv][D]
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

PrefillWs carve(void *ws, size_t Ttot, int nk, int nv, int D) {
  char *p = static_cast<char *>(ws);
  PrefillWs w;
  w.qn = reinterpret_cast<float *>(p);
  p += align256(Ttot * nk * D * sizeof(float));
  w.kn = reinterpret_cast<float *>(p);
  p += align256(Ttot * nk * D * sizeof(float));
  w.vv = reinterpret_cast<float *>(p);
  return w;
}

}  // namespace

size_t prefill_workspace_bytes(int B, int T, int nk, int nv, int D, bool packed) {
  if (D == 128) return prefill_tc_workspace_bytes(B, T, nk, nv, packed);
  const size_t Ttot = packed ? (size_t)T : (size_t)B * T;
  return 2 * align256(Ttot * nk * D * sizeof(float)) + align256(Ttot * nv * D * sizeof(float));
}

// Row of packed token p: the largest r with start(r) <= p.
__device__ __forceinline__ int token_row(const LayerArgs &A, int p, int &start) {
  if (!A.cu_seqlens) {
    start = (p / A.T) * A.T;
    return p / A.T;
  }
  int lo = 0, hi = A.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (A.cu_seqlens[mid] <= p) lo = mid; else hi = mid - 1;
  }
  start = A.cu_seqlens[lo];
  return lo;
}

template <int D>
__global__ void __launch_bounds__(256) prefill_front_kernel(LayerArgs A, int Ttot, PrefillWs W) {
  __shared__ float Y[kFrontTB][D];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gi = blockIdx.y, kd = A.nk * D;
  const int which = gi < A.nk ? 0 : (gi < 2 * A.nk ? 1 : 2);
  const int head = which == 0 ? gi : (which == 1 ? gi - A.nk : gi - 2 * A.nk);
  const int ch0 = which == 0 ? head * D : (which == 1 ? kd + head * D : 2 * kd + head * D);
  const bf16 *src = which == 0 ? A.q + head * D : (which == 1 ? A.k + head * D : A.v + head * D);
  const size_t rstride = which == 2 ? (size_t)A.nv * D : (size_t)kd;
  const int t0 = blockIdx.x * kFrontTB;

  for (int e = tid; e < kFrontTB * D; e += 256) {
    const int tt = e / D, c = e % D, p = t0 + tt;
    float y = 0.0f;
    if (p < Ttot) {
      int start;
      const int r = token_row(A, p, start);
      const int pos = p - start;
      const int slot = row_slot(A, r);
      if (slot >= 0 && start >= 0 && pos >= 0) {
        const int ch = ch0 + c;
        const bf16 *cs = A.conv_state + (size_t)slot * KC * A.C + ch;
        float xr[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ip = pos - KC + j;  // position of tap j within the row
          xr[j] = ip >= 0 ? ldbf(src + (size_t)(start + ip) * rstride + c) : ldbf(cs + (size_t)(KC + ip) * A.C);
        }
        const bf16 *w = A.conv_w + (size_t)ch * 4;
        y = conv4_silu(ldbf(w), ldbf(w + 1), ldbf(w + 2), ldbf(w + 3), xr[0], xr[1], xr[2], xr[3]);
      }
    }
    Y[tt][c] = y;
  }
  __syncthreads();
  if (which < 2)
    for (int tt = warp; tt < kFrontTB; tt += 8) warp_l2norm<D>(Y[tt], A.l2_eps, which == 0 ? A.scale : 1.0f, lane);
  __syncthreads();
  float *dst = which == 0 ? W.qn : (which == 1 ? W.kn : W.vv);
  const int nh = which == 2 ? A.nv : A.nk;
  for (int e = tid; e < kFrontTB * D; e += 256) {
    const int tt = e / D, c = e % D, p = t0 + tt;
    if (p < Ttot) dst[((size_t)p * nh + head) * D + c] = Y[tt][c];
  }
}

template <int D>
__global__ void __launch_bounds__(256, 2) prefill_recur_kernel(LayerArgs A, int Ttot, PrefillWs W) {
  using L = StateLayout<D>;
  __shared__ __align__(16) float F[2][4][D];  // q, k, v, z of the current / next token
  __shared__ float fw[D];
  __shared__ __align__(16) float red[StepScratch<D>::kFloats];
  __shared__ float s_gate[3];
  __shared__ int s_min_zero, s_max_one, s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / A.nv, h = blockIdx.x % A.nv, kh = h / A.G;
  const int kd = A.nk * D, C = A.C;

  int start, len;
  if (A.cu_seqlens) {
    start = A.cu_seqlens[b];
    len = A.cu_seqlens[b + 1] - start;
  } else {
    start = b * A.T;
    len = A.T;
  }
  const int slot = row_slot(A, b);
  if (slot < 0 || start < 0 || len < 0 || start + len > Ttot) {
    if (tid == 0) set_status(A.status, GDN_ERR_INDEX);
    return;
  }
  // ---- real length: the mask row must be ones then zeros
  if (tid == 0) {
    s_min_zero = len;
    s_max_one = -1;
    s_bad = 0;
  }
  __syncthreads();
  if (A.mask) {
    for (int i = tid; i < len; i += 256) {
      const float m = A.mask[start + i];
      if (m == 1.0f) atomicMax(&s_max_one, i);
      else if (m == 0.0f) atomicMin(&s_min_zero, i);
      else s_bad = 1;
    }
  }
  __syncthreads();
  const int Lr = s_min_zero;
  if (s_bad || s_max_one >= Lr) {
    if (tid == 0) set_status(A.status, GDN_ERR_MASK);
    return;
  }

  __shared__ RowCkpts ck;  // checkpoints this row asked for (prefix-cache states inside the call)
  if (tid == 0) {
    ck.n = 0;
    if (A.n_ckpt > 0) gather_row_ckpts(A, b, h, Lr, ck);
  }
  bf16 *cs = A.conv_state + (size_t)slot * KC * C;

  // ---- the delta rule, token by token
  const int cq = tid % L::TPR, grp = tid / L::TPR;
  float4 *gs = reinterpret_cast<float4 *>(A.state + ((size_t)slot * A.nv + h) * D * D);
  float4 s[L::RPT];
#pragma unroll
  for (int i = 0; i < L::RPT; ++i) s[i] = gs[(grp + i * L::NG) * L::TPR + cq];

  for (int c = tid; c < D; c += 256) fw[c] = ldbf(A.norm_w + c);
  auto fetch = [&](int t, float (&reg)[2]) {
    const size_t p = (size_t)start + t;
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int e = tid + k2 * 256;
      if (e < 4 * D) {
        const int which = e / D, c = e % D;
        reg[k2] = which == 0   ? W.qn[(p * A.nk + kh) * D + c]
                  : which == 1 ? W.kn[(p * A.nk + kh) * D + c]
                  : which == 2 ? W.vv[(p * A.nv + h) * D + c]
                               : ldbf(A.z + (p * A.nv + h) * D + c);
      }
    }
  };
  float cur[2] = {0.f, 0.f};
  if (Lr > 0) fetch(0, cur);
  for (int t = 0; t < Lr; ++t) {
    const int par = t & 1;
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int e = tid + k2 * 256;
      if (e < 4 * D) F[par][e / D][e % D] = cur[k2];
    }
    if (t + 1 < Lr) fetch(t + 1, cur);
    __syncthreads();
    if (warp == 0) {
      const float kq = warp_dot<D>(F[par][0], F[par][1], lane);
      if (lane == 0) {
        const size_t gi = ((size_t)start + t) * A.nv + h;
        float decay, beta;
        gdn_gates(ldbf(A.a + gi), ldbf(A.b + gi), A.A_log[h], A.dt_bias[h], decay, beta);
        s_gate[0] = decay;
        s_gate[1] = beta;
        s_gate[2] = __fmul_rn(beta, kq);
      }
    }
    __syncthreads();
    float4 o;
    state_step<D>(s, F[par][0], F[par][1], F[par][2], s_gate[0], s_gate[1], s_gate[2], red, tid, o, SyncAll());
    if (warp == 0)
      rmsnorm_store_smem<D>(o, lane, F[par][3], fw, A.rms_eps, A.out + ((size_t)start + t) * A.nv * D + h * D);
    for (int e = 0; e < ck.n; ++e) {  // checkpoints after this token: the state and the conv tail there
      if (ck.pos[e] != t + 1) continue;
      float4 *cS = reinterpret_cast<float4 *>(A.ckpt_state + ((size_t)ck.slot[e] * A.nv + h) * D * D);
#pragma unroll
      for (int i = 0; i < L::RPT; ++i) cS[(grp + i * L::NG) * L::TPR + cq] = s[i];
      conv_tail_at<D>(A, start, h, t + 1, cs, A.ckpt_conv + (size_t)ck.slot[e] * KC * C);
    }
    __syncthreads();  // s_gate is rewritten by the next token
  }
  for (int t = Lr; t < len; ++t) zero_head<D>(A.out + ((size_t)start + t) * A.nv * D + h * D, tid);
#pragma unroll
  for (int i = 0; i < L::RPT; ++i) gs[(grp + i * L::NG) * L::TPR + cq] = s[i];
  // conv tail: xin rows Lr .. Lr+2 (old rows when Lr < 3), own channels only,
  // after the checkpoints have read the saved rows
  __syncthreads();
  conv_tail_at<D>(A, start, h, Lr, cs, cs);
}

template <int D>
static gdn_status launch_prefill_t(const LayerArgs &A, void *ws, cudaStream_t stream) {
  const int Ttot = A.cu_seqlens ? A.T : A.B * A.T;
  PrefillWs W = carve(ws, (size_t)Ttot, A.nk, A.nv, D);
  dim3 gf((Ttot + kFrontTB - 1) / kFrontTB, 2 * A.nk + A.nv);
  prefill_front_kernel<D><<<gf, 256, 0, stream>>>(A, Ttot, W);
  if (gdn_status st = check_launch("prefill front")) return st;
  prefill_recur_kernel<D><<<A.B * A.nv, 256, 0, stream>>>(A, Ttot, W);
  return check_launch("prefill recurrence");
}

gdn_status launch_prefill(const LayerArgs &A, void *ws, size_t, cudaStream_t stream) {
  switch (A.D) {
    case 128: return launch_prefill_tc(A, ws, stream);
    case 64: return launch_prefill_t<64>(A, ws, stream);
    case 32: return launch_prefill_t<32>(A, ws, stream);
  }
  return fail(GDN_ERR_SHAPE, "prefill: unsupported head size");
}

}  // namespace gdn
