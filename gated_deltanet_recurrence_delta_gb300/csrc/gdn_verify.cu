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


// ---------------------------------------------------------------------------
// Head size 128: each head's 128 state columns are split over a cluster of two
// CTAs (128 threads each, 64 columns each), doubling the CTA count so the
// checkpoint stream spreads evenly over the SMs. A thread owns the same rows
// (grp + 8i) and 4 columns as in the one-CTA mapping, so every column sum is
// added in the same order; the RMSNorm's sum of squares is the same tree too:
// the 16 first-level pair sums s_l + s_{l+16} take one value from each CTA
// (exchanged through distributed shared memory), then the rest of the tree
// runs in one warp. Checkpoints and outputs are therefore bit-identical to
// gdn_decode_step's.
namespace {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Cluster barrier phases split in two: arrive (relaxed: orders nothing, only
// says "this CTA is running") and wait.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
// Store `v` into the partner CTA's copy of the shared variable at `p`.
__device__ __forceinline__ void st_partner_f32(float *p, uint32_t partner, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(partner));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 4)
    verify_split_kernel(LayerArgs A, float *ckpt_state, bf16 *ckpt_conv) {
  constexpr int D = 128, HALF = 64, NQ = 16, NG = 8, RPT = 16;  // NQ column quads, NG row groups
  constexpr int FW = 2 * D + HALF;                               // q, k, own v half per token
  constexpr int FC = D + HALF;                                   // channels convolved here
  __shared__ __align__(16) float F[kMaxVerifyT][FW];
  __shared__ __align__(16) bf16 XI[kMaxVerifyT + KC][FC];
  __shared__ __align__(16) bf16 WT[FC][4];
  __shared__ __align__(16) float Z[kMaxVerifyT][HALF];
  __shared__ __align__(16) float fw[HALF];
  __shared__ __align__(16) float part[2][NG][HALF];
  __shared__ __align__(16) float tot[2][HALF];
  __shared__ float gdecay[kMaxVerifyT], gbeta[kMaxVerifyT], gbkq[kMaxVerifyT];
  __shared__ __align__(16) float OS[kMaxVerifyT][HALF];  // o of every token (this CTA's columns)
  __shared__ float sqp[kMaxVerifyT][NQ], sqq[kMaxVerifyT][NQ];  // own / partner's sums of squares
  __shared__ float rrs[kMaxVerifyT];
  __shared__ int s_Lr;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t half = cluster_rank(), partner = half ^ 1u;
  const int unit = blockIdx.x >> 1;
  const int b = unit / A.nv, h = unit % A.nv, kh = h / A.G;
  const int T = A.T, kd = A.nk * D, C = A.C;
  const int c0 = HALF * (int)half;  // first state column of this CTA

  // ---- every global read issued before any is used. First what does not
  // depend on the row's slot: raw conv inputs of this CTA's channels at the T
  // tokens (half 0: the q block, half 1: the k block, plus its own 64 value
  // channels), taps, output gate, norm weight, mask, gates; then the slot and
  // the state slice and conv tail it selects.
  griddep_wait();  // the kernel before this call (e.g. the previous commit) is complete
  griddep_trigger();
  const int slot_raw = A.state_idx ? __ldg(A.state_idx + b) : b;  // used only after the loads below
  const int cq = tid % NQ, grp = tid / NQ;
  const int NR = T + KC;
  const int own = half == 0 ? 0 : D;  // offset of this CTA's q|k block in F
  auto chan = [&](int c) {             // c in [0, FC): own q|k block, then the v half
    return c < D ? (half == 0 ? kh * D + c : kd + kh * D + c) : 2 * kd + h * D + c0 + (c - D);
  };
  constexpr int NX = ((kMaxVerifyT + KC) * (FC / 8) + 127) / 128;
  uint4 xr[NX];
#pragma unroll
  for (int j = 0; j < NX; ++j) {
    const int e = tid + 128 * j, r = e / (FC / 8);
    if (e < NR * (FC / 8) && r >= KC) {
      const int ch = chan(8 * (e % (FC / 8)));
      const size_t tok = (size_t)b * T + (r - KC);
      const bf16 *src = ch < kd ? A.q + tok * kd + ch
                        : ch < 2 * kd ? A.k + tok * kd + (ch - kd)
                                      : A.v + tok * A.nv * D + (ch - 2 * kd);
      xr[j] = __ldg(reinterpret_cast<const uint4 *>(src));
    }
  }
  const uint2 wr0 = __ldg(reinterpret_cast<const uint2 *>(A.conv_w + (size_t)chan(tid) * 4));
  uint2 wr1 = make_uint2(0u, 0u);
  if (tid + 128 < FC) wr1 = __ldg(reinterpret_cast<const uint2 *>(A.conv_w + (size_t)chan(tid + 128) * 4));
  uint4 zr = make_uint4(0u, 0u, 0u, 0u);
  if (tid < T * (HALF / 8))
    zr = __ldg(reinterpret_cast<const uint4 *>(A.z + (((size_t)b * T + tid / 8) * A.nv + h) * D + c0) + tid % 8);
  const float fwv = tid < HALF ? ldbf(A.norm_w + c0 + tid) : 0.0f;
  if (warp == 0) {
    const float m = (A.mask && lane < T) ? A.mask[(size_t)b * T + lane] : 1.0f;
    const unsigned ones = __ballot_sync(0xffffffffu, lane < T && m == 1.0f);
    const unsigned zero = __ballot_sync(0xffffffffu, lane < T && m == 0.0f);
    const unsigned inrow = T >= 32 ? 0xffffffffu : ((1u << T) - 1u);
    const int Lr = min(T, __ffs(~ones) - 1 < 0 ? 32 : __ffs(~ones) - 1);
    const unsigned tail = inrow & ~((Lr >= 32) ? 0xffffffffu : ((1u << Lr) - 1u));
    const bool bad = (ones | zero) != inrow || (ones & tail) != 0;
    if (lane == 0) {
      if (bad && half == 0) set_status(A.status, GDN_ERR_MASK);
      s_Lr = bad ? -1 : Lr;
    }
    if (lane < T) {
      const size_t gi = ((size_t)b * T + lane) * A.nv + h;
      float decay, beta;
      gdn_gates(ldbf(A.a + gi), ldbf(A.b + gi), A.A_log[h], A.dt_bias[h], decay, beta);
      gdecay[lane] = decay;
      gbeta[lane] = beta;
    }
  }
  // both CTAs of the pair take the same early exits (same data), before any cluster barrier
  const int slot = (slot_raw < 0 || slot_raw >= A.n_slots) ? -1 : slot_raw;
  if (slot < 0) {
    if (tid == 0 && half == 0) set_status(A.status, GDN_ERR_INDEX);
    return;
  }
  const float4 *gs = reinterpret_cast<const float4 *>(A.state + ((size_t)slot * A.nv + h) * D * D + c0);
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = __ldg(gs + (grp + i * NG) * (D / 4) + cq);
  uint4 xt = make_uint4(0u, 0u, 0u, 0u);
  if (tid < KC * (FC / 8))  // the conv tail rows
    xt = __ldg(reinterpret_cast<const uint4 *>(A.conv_state + ((size_t)slot * KC + tid / (FC / 8)) * C +
                                                  chan(8 * (tid % (FC / 8)))));
#pragma unroll
  for (int j = 0; j < NX; ++j) {
    const int e = tid + 128 * j;
    if (e < NR * (FC / 8) && e >= KC * (FC / 8)) reinterpret_cast<uint4 *>(&XI[e / (FC / 8)][0])[e % (FC / 8)] = xr[j];
  }
  reinterpret_cast<uint2 *>(WT)[tid] = wr0;
  if (tid + 128 < FC) reinterpret_cast<uint2 *>(WT)[tid + 128] = wr1;
  if (tid < T * (HALF / 8)) {
    const uint32_t zs[4] = {zr.x, zr.y, zr.z, zr.w};
    float *zd = &Z[tid / 8][8 * (tid % 8)];
#pragma unroll
    for (int q2 = 0; q2 < 4; ++q2) {
      zd[2 * q2] = __uint_as_float(zs[q2] << 16);
      zd[2 * q2 + 1] = __uint_as_float(zs[q2] & 0xffff0000u);
    }
  }
  if (tid < HALF) fw[tid] = fwv;
  __syncthreads();
  const int Lr = s_Lr;
  if (Lr < 0) return;
  cluster_arrive_relaxed();  // this CTA runs: the partner may store into its shared memory

  // ---- own q|k block: a warp per token, lane holding channels lane + 32j (the
  // lane order of the L2 norm's sums), normalised here, then sent to the partner
  const float nscale = half == 0 ? A.scale : 1.0f;
  constexpr int TW = kMaxVerifyT / 4;  // tokens per warp
  static_assert(TW == 2 && KC <= 4, "token order below assumes two tokens per warp");
  float yb[TW][4];
#pragma unroll
  for (int it0 = 0; it0 < TW; ++it0) {
    const int it = TW - 1 - it0;  // tokens 4..7 first: they do not read the conv tail rows
    const int t = warp + 4 * it;
    if (it0 == 1) {
      if (tid < KC * (FC / 8)) reinterpret_cast<uint4 *>(&XI[tid / (FC / 8)][0])[tid % (FC / 8)] = xt;
      __syncthreads();
    }
    if (t < T) {
      float ss = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = lane + 32 * j;
        const bf16 *w = &WT[c][0];
        const float y = conv4_silu(__bfloat162float(w[0]), __bfloat162float(w[1]), __bfloat162float(w[2]),
                                   __bfloat162float(w[3]), __bfloat162float(XI[t][c]),
                                   __bfloat162float(XI[t + 1][c]), __bfloat162float(XI[t + 2][c]),
                                   __bfloat162float(XI[t + 3][c]));
        ss = __fmaf_rn(y, y, ss);
        yb[it][j] = y;
      }
      ss = warp_sum_bcast(ss);
      const float r = __fdiv_rn(nscale, sqrtf(__fadd_rn(ss, A.l2_eps)));
#pragma unroll
      for (int j = 0; j < 4; ++j) yb[it][j] = __fmul_rn(yb[it][j], r);
    }
  }
  cluster_wait();  // the partner runs
#pragma unroll
  for (int it = 0; it < TW; ++it) {
    const int t = warp + 4 * it;
    if (t < T) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float *dst = &F[t][own + lane + 32 * j];
        *dst = yb[it][j];
        st_partner_f32(dst, partner, yb[it][j]);
      }
    }
  }
  cluster_sync();  // both normalised q|k blocks are in both CTAs
  const int cfirst = (h % A.G) == 0 ? 0 : D;  // conv checkpoint: the q|k block from the group's first value head

  for (int t = 0; t < T; ++t) {
    if (t < Lr) {
      // this token's own value half, and beta * (k . q)
      if (tid < HALF) {
        const bf16 *w = &WT[D + tid][0];
        F[t][2 * D + tid] = conv4_silu(__bfloat162float(w[0]), __bfloat162float(w[1]), __bfloat162float(w[2]),
                                       __bfloat162float(w[3]), __bfloat162float(XI[t][D + tid]),
                                       __bfloat162float(XI[t + 1][D + tid]), __bfloat162float(XI[t + 2][D + tid]),
                                       __bfloat162float(XI[t + 3][D + tid]));
      } else if (warp == 2 + (t & 1)) {
        const float kq = warp_dot<D>(&F[t][0], &F[t][D], lane);
        if (lane == 0) gbkq[t] = __fmul_rn(gbeta[t], kq);
      } else {  // the other warp: silu of the output gate, in place
        Z[t][lane] = silu_f(Z[t][lane]);
        Z[t][lane + 32] = silu_f(Z[t][lane + 32]);
      }
      const float *qn = &F[t][0], *kn = &F[t][D];
      const float decay = gdecay[t], beta = gbeta[t];
      float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int r = grp + i * NG;
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
      reinterpret_cast<float4 *>(part[0][grp])[cq] = pk;
      reinterpret_cast<float4 *>(part[1][grp])[cq] = pq;
      __syncthreads();
      {
        const int kind = tid / HALF, col = tid % HALF;
        float acc = part[kind][0][col];
#pragma unroll
        for (int g2 = 1; g2 < NG; ++g2) acc = __fadd_rn(acc, part[kind][g2][col]);
        tot[kind][col] = acc;
      }
      __syncthreads();
      const float4 KS = reinterpret_cast<const float4 *>(tot[0])[cq];
      const float4 QS = reinterpret_cast<const float4 *>(tot[1])[cq];
      const float4 v4 = reinterpret_cast<const float4 *>(&F[t][2 * D])[cq];
      float4 u;
      u.x = __fmaf_rn(-decay, KS.x, v4.x);
      u.y = __fmaf_rn(-decay, KS.y, v4.y);
      u.z = __fmaf_rn(-decay, KS.z, v4.z);
      u.w = __fmaf_rn(-decay, KS.w, v4.w);
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float bk = __fmul_rn(beta, kn[grp + i * NG]);
        s[i].x = __fmaf_rn(bk, u.x, __fmul_rn(decay, s[i].x));
        s[i].y = __fmaf_rn(bk, u.y, __fmul_rn(decay, s[i].y));
        s[i].z = __fmaf_rn(bk, u.z, __fmul_rn(decay, s[i].z));
        s[i].w = __fmaf_rn(bk, u.w, __fmul_rn(decay, s[i].w));
      }
      const float bkq = gbkq[t];
      float4 o;
      o.x = __fmaf_rn(bkq, u.x, __fmul_rn(decay, QS.x));
      o.y = __fmaf_rn(bkq, u.y, __fmul_rn(decay, QS.y));
      o.z = __fmaf_rn(bkq, u.z, __fmul_rn(decay, QS.z));
      o.w = __fmaf_rn(bkq, u.w, __fmul_rn(decay, QS.w));
      if (grp == 0) {
        reinterpret_cast<float4 *>(OS[t])[cq] = o;
        float ss = __fmul_rn(o.x, o.x);  // this quad's share of the RMS sum, also sent to the partner
        ss = __fmaf_rn(o.y, o.y, ss);
        ss = __fmaf_rn(o.z, o.z, ss);
        ss = __fmaf_rn(o.w, o.w, ss);
        sqp[t][cq] = ss;
        st_partner_f32(&sqq[t][cq], partner, ss);
      }
    }
    float4 *ck = reinterpret_cast<float4 *>(ckpt_state + (((size_t)b * T + t) * A.nv + h) * D * D + c0);
#pragma unroll
    for (int i = 0; i < RPT; ++i) st_cs(ck + (grp + i * NG) * (D / 4) + cq, s[i]);
    // conv checkpoint after token t: xin rows min(t+1, Lr) .. +2 of this CTA's channels
    {
      const int e0 = t + 1 < Lr ? t + 1 : Lr;
      for (int e = tid; e < KC * (FC / 8); e += 128) {
        const int r = e / (FC / 8), c = 8 * (e % (FC / 8));
        if (c >= cfirst)
          *reinterpret_cast<uint4 *>(ckpt_conv + (((size_t)b * T + t) * KC + r) * C + chan(c)) =
              *reinterpret_cast<const uint4 *>(&XI[e0 + r][c]);
      }
    }
  }
  // ---- outputs, after the recurrence: gated RMSNorm per token. This CTA's 16
  // per-quad sums of squares are paired with the partner's, then reduced with
  // the same tree as a 32-lane warp over all 128 columns.
  cluster_sync();  // after this no CTA touches the partner's shared memory
  for (int t = warp; t < Lr; t += 4) {
    float x = 0.0f;
    if (lane < NQ) x = half == 0 ? __fadd_rn(sqp[t][lane], sqq[t][lane]) : __fadd_rn(sqq[t][lane], sqp[t][lane]);
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, off));
    x = __shfl_sync(0xffffffffu, x, 0);
    if (lane == 0) rrs[t] = __frcp_rn(sqrtf(__fadd_rn(__fmul_rn(x, 1.0f / D), A.rms_eps)));
  }
  __syncthreads();
  for (int e = tid; e < T * NQ; e += 128) {
    const int t = e / NQ, q4 = e % NQ, c = 4 * q4;
    bf16 *out = A.out + (((size_t)b * T + t) * A.nv + h) * D + c0 + c;
    __align__(8) bf16 res[4];
    if (t < Lr) {
      const float4 o = reinterpret_cast<const float4 *>(OS[t])[q4];
      const float ov[4] = {o.x, o.y, o.z, o.w};
      const float rr = rrs[t];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2)
        res[e2] = __float2bfloat16_rn(__fmul_rn(__fmul_rn(__fmul_rn(ov[e2], rr), fw[c + e2]), Z[t][c + e2]));
    } else {
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) res[e2] = __float2bfloat16_rn(0.0f);
    }
    *reinterpret_cast<uint2 *>(out) = *reinterpret_cast<const uint2 *>(res);
  }
}

template <int D>
static gdn_status launch_verify_t(const LayerArgs &A, float *ckpt_state, bf16 *ckpt_conv, cudaStream_t stream) {
  using S = VerifySmem<D>;
  const DeviceInfo &dev = device_info();
  // set once per device; concurrent first calls may both set it (idempotent)
  static std::atomic<bool> attr_set[kMaxDevices];
  if (!attr_set[dev.id].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(verify_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::kBytes) !=
        cudaSuccess)
      return fail(GDN_ERR_CUDA, "verify: cannot reserve shared memory");
    attr_set[dev.id].store(true, std::memory_order_release);
  }
  verify_kernel<D><<<A.B * A.nv, 256, S::kBytes, stream>>>(A, ckpt_state, ckpt_conv);
  return check_launch("verify");
}

gdn_status launch_verify(const LayerArgs &A, float *ckpt_state, bf16 *ckpt_conv, cudaStream_t stream) {
  switch (A.D) {
    case 128:
      if (launch_pdl(verify_split_kernel, dim3(2 * A.B * A.nv), dim3(128), 0, stream, A, ckpt_state, ckpt_conv) !=
          cudaSuccess)
        return check_launch("verify");
      return check_launch("verify");
    case 64: return launch_verify_t<64>(A, ckpt_state, ckpt_conv, stream);
    case 32: return launch_verify_t<32>(A, ckpt_state, ckpt_conv, stream);
  }
  return fail(GDN_ERR_SHAPE, "verify: unsupported head size");
}

}  // namespace gdn
