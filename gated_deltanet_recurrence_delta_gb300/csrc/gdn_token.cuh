// Per-token arithmetic of the Gated DeltaNet layer shared by the decode and the
// verify kernels. Both kernels call exactly these functions with the same
// thread mapping, so a verify checkpoint after token t equals, bit for bit, the
// state after t+1 decode steps (generate.py, sparkle mlx_streaming/mtp: the
// per-token checkpoints of the verify forward are committed without replay).
//
// Every rounding step is explicit (__fmaf_rn / __fmul_rn / __fadd_rn cannot be
// contracted or reassociated by the compiler).
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Thread layout of a D x D fp32 state St[k][v] over 256 threads: each thread
// owns 4 consecutive value columns (one float4) of RPT key rows; rows are
// strided by NG so that a warp touches whole contiguous rows.
template <int D>
struct StateLayout {
  static constexpr int NT = 256;
  static constexpr int TPR = D / 4;     // threads per row
  static constexpr int NG = NT / TPR;   // row groups
  static constexpr int RPT = D / NG;    // rows per thread
  static_assert(TPR <= 32 && NG * TPR == NT && RPT * NG == D, "unsupported head size");
};

// __frcp_rn is the correctly rounded 1/x, the same value as __fdiv_rn(1, x).
__device__ __forceinline__ float sigmoid_f(float x) { return __frcp_rn(__fadd_rn(1.0f, expf(-x))); }
__device__ __forceinline__ float silu_f(float x) { return __fmul_rn(x, sigmoid_f(x)); }
// softplus(x) = log(1 + e^x); above 20 the correction is below 2.1e-9 and x is returned.
__device__ __forceinline__ float softplus_f(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

// Depthwise conv of one channel at one token over xin rows t..t+3 (tap 3 is the
// current token), then SiLU: statecache.py, CacheQwen35._gdn (fla_conv, no bias).
__device__ __forceinline__ float conv4_silu(float w0, float w1, float w2, float w3, float x0, float x1,
                                            float x2, float x3) {
  float acc = __fmul_rn(w0, x0);
  acc = __fmaf_rn(w1, x1, acc);
  acc = __fmaf_rn(w2, x2, acc);
  acc = __fmaf_rn(w3, x3, acc);
  return silu_f(acc);
}

// L2-normalise a D-vector in shared memory in place and multiply by `scale`
// (use_qk_l2norm_in_kernel: x / sqrt(sum x^2 + eps)). Called by one whole warp.
template <int D>
__device__ __forceinline__ void warp_l2norm(float *x, float eps, float scale, int lane) {
  float s = 0.0f;
#pragma unroll
  for (int i = lane; i < D; i += 32) s = __fmaf_rn(x[i], x[i], s);
  s = warp_sum_bcast(s);
  const float r = __fdiv_rn(scale, sqrtf(__fadd_rn(s, eps)));
#pragma unroll
  for (int i = lane; i < D; i += 32) x[i] = __fmul_rn(x[i], r);
  __syncwarp();
}

template <int D>
__device__ __forceinline__ float warp_dot(const float *x, const float *y, int lane) {
  float s = 0.0f;
#pragma unroll
  for (int i = lane; i < D; i += 32) s = __fmaf_rn(x[i], y[i], s);
  return warp_sum_bcast(s);
}

// Gates of one (token, head): g = -exp(A_log) softplus(a + dt_bias),
// beta = sigmoid(b) (gdn_gates). Returned as exp(g) and beta.
__device__ __forceinline__ void gdn_gates(float a, float b, float A_log, float dt_bias, float &decay,
                                          float &beta) {
  const float g = __fmul_rn(-expf(A_log), softplus_f(__fadd_rn(a, dt_bias)));
  decay = expf(g);
  beta = sigmoid_f(b);
}

// CTA-wide barrier over all threads.
struct SyncAll {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};
// Barrier 1 over the 256 compute threads only (a producer warp stays out).
struct SyncCompute {
  __device__ __forceinline__ void operator()() const { asm volatile("bar.sync 1, 256;" ::: "memory"); }
};

// Shared-memory floats state_step needs for its reductions.
template <int D>
struct StepScratch {
  static constexpr int kFloats = 2 * StateLayout<D>::NG * D + 2 * D;  // partials [k|q][NG][D], totals [k|q][D]
};

// One token of the delta rule on the thread's slice s[] of St (fla_gdr):
//   St <- decay St;  u = v - St^T k;  St += beta k u^T;  o = St^T q
// computed as  KS = St_old^T k, QS = St_old^T q  (one pass over the old state),
//   u = v - decay KS,  St_new = decay St_old + (beta k) u^T,
//   o = decay QS + (beta k.q) u          (bkq = beta * k.q)
// The column sums over the key rows run in two levels: per-thread partials
// over its rows, then one thread per (k|q, column) adds the NG row-group
// partials in order. qn, kn, vv: shared D-vectors (q already scaled). red:
// StepScratch<D>::kFloats shared floats. Two barriers (Sync). Every thread
// returns o for its 4 columns (threads with equal columns agree bit for bit).
template <int D, class Sync>
__device__ __forceinline__ void state_step(float4 (&s)[StateLayout<D>::RPT], const float *qn, const float *kn,
                                           const float *vv, float decay, float beta, float bkq, float *red,
                                           int tid, float4 &o, Sync sync) {
  using L = StateLayout<D>;
  const int cq = tid % L::TPR, grp = tid / L::TPR;
  float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
  for (int i = 0; i < L::RPT; ++i) {
    const int r = grp + i * L::NG;
    const float kr = kn[r], qr = qn[r];
    pk.x = __fmaf_rn(s[i].x, kr, pk.x);
    pk.y = __fmaf_rn(s[i].y, kr, pk.y);
    pk.z = __fmaf_rn(s[i].z, kr, pk.z);
    pk.w = __fmaf_rn(s[i].w, kr, pk.w);
    pq.x = __fmaf_rn(s[i].x, qr, pq.x);
    pq.y = __fmaf_rn(s[i].y, qr, pq.y);
    pq.z = __fmaf_rn(s[i].z, qr, pq.z);
    pq.w = __fmaf_rn(s[i].w, qr, pq.w);
  }
  float *part = red;                       // [2][NG][D]
  float *tot = red + 2 * L::NG * D;        // [2][D]
  reinterpret_cast<float4 *>(part)[grp * L::TPR + cq] = pk;
  reinterpret_cast<float4 *>(part + L::NG * D)[grp * L::TPR + cq] = pq;
  sync();
  if (tid < 2 * D) {
    const float *p = part + (tid / D) * L::NG * D + tid % D;
    float acc = p[0];
#pragma unroll
    for (int g2 = 1; g2 < L::NG; ++g2) acc = __fadd_rn(acc, p[g2 * D]);
    tot[tid] = acc;
  }
  sync();
  const float4 KS = reinterpret_cast<const float4 *>(tot)[cq];
  const float4 QS = reinterpret_cast<const float4 *>(tot + D)[cq];
  const float4 v4 = reinterpret_cast<const float4 *>(vv)[cq];
  float4 u;
  u.x = __fmaf_rn(-decay, KS.x, v4.x);
  u.y = __fmaf_rn(-decay, KS.y, v4.y);
  u.z = __fmaf_rn(-decay, KS.z, v4.z);
  u.w = __fmaf_rn(-decay, KS.w, v4.w);
#pragma unroll
  for (int i = 0; i < L::RPT; ++i) {
    const float bk = __fmul_rn(beta, kn[grp + i * L::NG]);
    s[i].x = __fmaf_rn(bk, u.x, __fmul_rn(decay, s[i].x));
    s[i].y = __fmaf_rn(bk, u.y, __fmul_rn(decay, s[i].y));
    s[i].z = __fmaf_rn(bk, u.z, __fmul_rn(decay, s[i].z));
    s[i].w = __fmaf_rn(bk, u.w, __fmul_rn(decay, s[i].w));
  }
  o.x = __fmaf_rn(bkq, u.x, __fmul_rn(decay, QS.x));
  o.y = __fmaf_rn(bkq, u.y, __fmul_rn(decay, QS.y));
  o.z = __fmaf_rn(bkq, u.z, __fmul_rn(decay, QS.z));
  o.w = __fmaf_rn(bkq, u.w, __fmul_rn(decay, QS.w));
}

// Gated RMSNorm of one head's o (gated_rmsnorm: o / sqrt(mean o^2 + eps) * w *
// silu(z)) and its bf16 store. z and w are the head's values staged in shared
// memory as fp32 (exact copies of the bf16 inputs). Called by one whole warp
// whose lanes < TPR hold o for columns 4*lane .. 4*lane+3.
template <int D>
__device__ __forceinline__ void rmsnorm_store_smem(float4 o, int lane, const float *z, const float *w, float eps,
                                                   bf16 *out) {
  using L = StateLayout<D>;
  float ss = 0.0f;
  if (lane < L::TPR) {
    ss = __fmul_rn(o.x, o.x);
    ss = __fmaf_rn(o.y, o.y, ss);
    ss = __fmaf_rn(o.z, o.z, ss);
    ss = __fmaf_rn(o.w, o.w, ss);
  }
  ss = warp_sum_bcast(ss);
  // D is a power of two: ss * (1/D) is exactly ss / D
  const float r = __frcp_rn(sqrtf(__fadd_rn(__fmul_rn(ss, 1.0f / D), eps)));
  if (lane < L::TPR) {
    const int c = 4 * lane;
    const float ov[4] = {o.x, o.y, o.z, o.w};
    __align__(8) bf16 res[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float y = __fmul_rn(__fmul_rn(__fmul_rn(ov[e], r), w[c + e]), silu_f(z[c + e]));
      res[e] = __float2bfloat16_rn(y);
    }
    *reinterpret_cast<uint2 *>(out + c) = *reinterpret_cast<const uint2 *>(res);
  }
}

// The conv tail of a prefill row after its first `pos` tokens of the call, for
// value head h's own channels: its value channels, and the q / k channels of
// its key head when h is the first value head of the group (so every channel
// has one writer). xin rows pos .. pos+2: rows of the saved tail `old`
// ([3][C]) while pos + r < 3, else tokens pos + r - 3 of the row (which starts
// at packed token `start`). Written to dst ([3][C]; may be `old` itself: each
// thread reads its channel's three rows before writing them). All threads of
// the CTA take part.
template <int D>
__device__ __forceinline__ void conv_tail_at(const LayerArgs &A, int start, int h, int pos, const bf16 *old,
                                             bf16 *dst) {
  const int kh = h / A.G, kd = A.nk * D, C = A.C;
  const bool qk = (h % A.G) == 0;
  const int nch = qk ? 3 * D : D;
  for (int e = threadIdx.x; e < nch; e += blockDim.x) {
    const int which = qk ? e / D : 2, cc = e % D;
    const int ch = which == 0 ? kh * D + cc : (which == 1 ? kd + kh * D + cc : 2 * kd + h * D + cc);
    const bf16 *src = which == 0 ? A.q + kh * D + cc : (which == 1 ? A.k + kh * D + cc : A.v + h * D + cc);
    const size_t rstride = which == 2 ? (size_t)A.nv * D : (size_t)kd;
    bf16 nv3[KC];
#pragma unroll
    for (int r = 0; r < KC; ++r) {
      const int xi = pos + r;
      nv3[r] = xi < KC ? old[(size_t)xi * C + ch] : src[(size_t)(start + xi - KC) * rstride];
    }
#pragma unroll
    for (int r = 0; r < KC; ++r) dst[(size_t)r * C + ch] = nv3[r];
  }
}

// The checkpoints a prefill row requested (A.ckpt triples naming row b), for
// the chain of (row b, value head h); built by thread 0 into shared memory.
// A triple is kept when 0 < position <= Lr, position is a multiple of 64 or
// Lr itself, and 0 <= slot < n_ckpt_slots; otherwise, or past kMaxRowCkpt
// per row, it is a recorded index error and skipped. The chain of (row 0,
// head 0) also records triples whose row lies outside [0, B).
struct RowCkpts {
  int n;
  int pos[kMaxRowCkpt], slot[kMaxRowCkpt];
};
__device__ __forceinline__ void gather_row_ckpts(const LayerArgs &A, int b, int h, int Lr, RowCkpts &L) {
  int n = 0;
  for (int i = 0; i < A.n_ckpt; ++i) {
    const int r = A.ckpt[3 * i], p = A.ckpt[3 * i + 1], sl = A.ckpt[3 * i + 2];
    if (r < 0 || r >= A.B) {
      if (b == 0 && h == 0) set_status(A.status, GDN_ERR_INDEX);
      continue;
    }
    if (r != b) continue;
    const bool ok = p > 0 && p <= Lr && (p % 64 == 0 || p == Lr) && sl >= 0 && sl < A.n_ckpt_slots;
    if (!ok || n == kMaxRowCkpt) {
      set_status(A.status, GDN_ERR_INDEX);
      continue;
    }
    L.pos[n] = p;
    L.slot[n] = sl;
    ++n;
  }
  L.n = n;
}

// Zero one head's bf16 output (padded tokens, skipped rows).
template <int D>
__device__ __forceinline__ void zero_head(bf16 *out, int tid) {
  if (tid < D / 8) reinterpret_cast<uint4 *>(out)[tid] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace gdn
