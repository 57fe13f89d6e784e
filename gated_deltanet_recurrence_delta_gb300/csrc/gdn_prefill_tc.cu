// Chunked (WY / UT) prefill on the tcgen05 tensor cores, head size 128.
//
// statecache.py (squad-0.8b, qev_fast): fla_gdr over chunks of 64 tokens
// ("fla's delta-rule chunk: 64"), continued from the saved fp32 state, padding
// masked by g = beta = 0. Within a chunk, with G the inclusive prefix of g,
// Gamma_ij = exp(G_i - G_j) (i >= j), gamma = exp(G), the state after token i is
//   S_i = gamma_i S_0 + sum_{j<=i} Gamma_ij k_j u_j^T,
// where the pseudo-values solve the unit-lower system (I + A) U' = diag(beta) V
// - diag(beta gamma) K S_0 with A = strict_lower(diag(beta) (K K^T * Gamma)).
// With T = (I + A)^-1, P = (Q K^T * Gamma) on and below the diagonal:
//   W = T diag(beta gamma) K,  U = T diag(beta) V,  U' = U - W S_0
//   O = diag(gamma) Q S_0 + P U' = Q' S_0 + P U,   Q' = diag(gamma) Q - P W
//   S_C = gamma_C S_0 + (K * exp(G_C - G))^T U'
// (S on the stored transpose St[k][v]). exp(-G) is never formed.
//
// Passes, stream ordered. Few (row, head) chains: front -> chunk + state in
// one grid -> output. Otherwise: front -> chunk -> state, the state pass
// forming the outputs itself:
//   front  conv + SiLU + q/k L2 norm per (chunk slot, q/k/v head), written
//          as split fp16 tiles, 128B-swizzled [token][d] images of Q, K and V
//          (K-major operands where d is the contraction, MN-major ones where
//          the tokens are).
//   chunk  per (chunk slot, value head) unit, all chunks in parallel, one
//          persistent CTA per SM walking its units: [K;Q] K^T on
//          tcgen05 (M=128,N=64,K=128); A and P in fp32 from TMEM; T by a
//          blocked fp32 triangular inverse; R = P T (tcgen05); then the
//          tcgen05 products [T; R] diag(beta gamma) K and [T; R] diag(beta) V
//          (M=128,N=128,K=64 each; the factors ride on the columns of two
//          [T; R] images) yield W, P W (-> Q'), U and P U (= O_local). Writes
//          W|Q' as one swizzled image, U in fp16, O_local in fp32, and
//          exp(G_C - G).
//   state  per (row, value head), sequential over its chunks with the state
//          in registers (fp32) and an fp16 copy in shared memory:
//          X = S_math W^T (tcgen05 M=128,N=64,K=128) -> U' = U - X,
//          dS = (U' exp(G_C - G))^T-image x K-image (tcgen05 M=128,N=128,
//          K=64, K read MN-major), S = gamma_C S + dS. With many chains the
//          same product also yields O_S = Q' S (N=128: [W; Q']) and, while
//          the tensor cores form dS, O = O_S + O_local, the gated RMSNorm
//          and the bf16 rows go out. With few chains the fp16 state image
//          at every chunk start is copied out instead, for
//   output per (chunk slot, value head), all chunks in parallel on the SMs
//          the chains leave idle: O = Q' S + O_local from that image
//          (tcgen05 M=128,N=64,K=128), gated RMSNorm, bf16 rows through the
//          TMA.
// Operand tiles move between HBM and shared memory with bulk copies (TMA).
// Precision: accumulators are fp32. The chunk kernel runs every product in
// split fp16 (x = hi + lo, hi = fp16(x), lo = fp16(x - hi); a*b ~ hi*hi +
// hi*lo + lo*hi, ~21 significant bits), so W, Q', O_local reach the state
// kernel nearly exact (U in fp16: it only enters U' = U - X, which the state
// product takes in fp16 anyway); the state kernel's two products take plain
// fp16 operands (10-bit mantissa; bf16 would leave the final state ~3e-3 off
// in relative Frobenius norm). With every product in plain fp16 the normalised
// outputs of badly conditioned tokens drift by ~1e-2.
#include "gdn_launch.h"
#include "gdn_token.cuh"
#include "gdn_umma.cuh"

namespace gdn {
namespace tc {

constexpr int CH = 64;   // chunk length
constexpr int HD = 128;  // head size handled here

// ------------------------------------------------------------ workspace

struct Ws {
  __half *kimg, *qimg;  // [S][nk][2 hi|lo][2][64][64]  K, Q as swizzled [token][dk] images (2 x 16 KiB)
  __half *vimg;         // [S][nv][2 hi|lo][2][64][64]  V as a swizzled [token][dv] image
  __half *wq;           // [S][nv][2][128][64]  W (rows 0-63) | Q' (rows 64-127) image (32 KiB)
  float *gate;          // [S][nv][324]         per token j < 64: g, beta, G (inclusive prefix of g), exp(G),
                        //                      exp(G_C - G); then gamma_C (and 3 pad). Written by the front
                        //                      kernel when the chunk and state passes are separate kernels
                        //                      (else the chunk unit forms the gates and writes the last 68,
                        //                      which the state pass reads)
  __half *ut;           // [S][nv][64][128]     U, token-major fp16, 16-byte chunk c of row i
                        //                      stored at c ^ (i % 8) (16 KiB)
  float *ot;            // [S][nv][64][128]     O_local, token-major fp32, the same chunk order (32 KiB)
  __half *simg;         // [S][nv][2][128][64]  fp16 image of the state at the chunk's start (32 KiB;
                        //                      dense rows only: the grid of few chains)
  int *lr;              // [B][nv]              real length of each row, per value head; -1 = the
                        //                      row was rejected or the head's chain stopped
  int *flag;            // [S][nv]              chunk unit published (chunk + state in one grid)
  int2 *slot_rc;        // [S]                  (row, chunk) of each slot from the front kernel, row -1 = none
};

constexpr size_t kImg = 64 * 128;    // halves in a 64x128 image
constexpr size_t kWQ = 128 * 128;    // halves in the W|Q' image
constexpr size_t kRowF = 128 * 64;   // floats in O_local (and halves in U)
constexpr int kGateRec = 324;        // floats in one gate record (a multiple of 16 bytes)
constexpr int kGateLd = 320;         // floats of it a chunk unit loads (g, beta, G, exp(G), exp(G_C - G))
constexpr int kSecOff = 256;         // exp(G_C - G) | gamma_C: the state pass's 68 floats
constexpr int kSecRec = 68;

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t slots_total(int B, int T, bool packed) {
  return packed ? (size_t)T / CH + (size_t)B + 1 : (size_t)B * (size_t)((T + CH - 1) / CH);
}

size_t ws_bytes(int B, int T, int nk, int nv, bool packed) {
  const size_t S = slots_total(B, T, packed);
  return 2 * a256(S * nk * kImg * 4) + a256(S * nv * kImg * 4) + a256(S * nv * kWQ * 2) +
         a256(S * nv * kGateRec * 4) + a256(S * nv * kRowF * 2) + a256(S * nv * kRowF * 4) +
         (packed ? 0 : a256(S * nv * kWQ * 2)) + a256((size_t)B * nv * 4) + a256(S * nv * 4) + a256(S * 8);
}

Ws carve(void *ws, int B, int T, int nk, int nv, bool packed) {
  const size_t S = slots_total(B, T, packed);
  char *p = static_cast<char *>(ws);
  Ws w;
  w.kimg = reinterpret_cast<__half *>(p);
  p += a256(S * nk * kImg * 4);
  w.qimg = reinterpret_cast<__half *>(p);
  p += a256(S * nk * kImg * 4);
  w.vimg = reinterpret_cast<__half *>(p);
  p += a256(S * nv * kImg * 4);
  w.wq = reinterpret_cast<__half *>(p);
  p += a256(S * nv * kWQ * 2);
  w.gate = reinterpret_cast<float *>(p);
  p += a256(S * nv * kGateRec * 4);
  w.ut = reinterpret_cast<__half *>(p);
  p += a256(S * nv * kRowF * 2);
  w.ot = reinterpret_cast<float *>(p);
  p += a256(S * nv * kRowF * 4);
  w.simg = packed ? nullptr : reinterpret_cast<__half *>(p);
  if (!packed) p += a256(S * nv * kWQ * 2);
  w.lr = reinterpret_cast<int *>(p);
  p += a256((size_t)B * nv * 4);
  w.flag = reinterpret_cast<int *>(p);
  p += a256(S * nv * 4);
  w.slot_rc = reinterpret_cast<int2 *>(p);
  return w;
}

// ------------------------------------------------------------ row / slot map
//
// Dense rows: row r owns slots [r*cpr, (r+1)*cpr), cpr = ceil(T/64).
// Packed rows: row r owns slots starting at floor(cu[r]/64) + r (one extra slot
// per row covers its partial chunk; rows never overlap).

struct Rows {
  int B, T, cpr;  // cpr > 0: dense
  const int32_t *cu;
  __device__ __forceinline__ int start(int r) const { return cu ? cu[r] : r * T; }
  __device__ __forceinline__ int len(int r) const { return cu ? cu[r + 1] - cu[r] : T; }
  __device__ __forceinline__ int slot0(int r) const { return cu ? cu[r] / CH + r : r * cpr; }
  // (row, chunk) of slot s, or row -1 when the slot holds no chunk. Packed
  // rows: called by whole warps. The first slots slot0(r) increase with r, so
  // the rows with slot0(r) <= s form a prefix; each warp reads the row offsets
  // 32 at a time (one coalesced load instead of a chain of dependent loads)
  // and counts that prefix with a ballot.
  __device__ __forceinline__ void locate(int s, int Ttot, int &r, int &c) const {
    int st, ln;
    if (!cu) {
      r = s / cpr;
      c = s % cpr;
      st = r * T;
      ln = T;
    } else {
      const int lane = threadIdx.x & 31;
      int n = 0;
      for (int base = 0; base < B; base += 32) {
        const int i = base + lane;
        const unsigned m = __ballot_sync(0xffffffffu, i < B && __ldg(cu + i) / CH + i <= s);
        n += __popc(m);
        if (m != 0xffffffffu) break;
      }
      r = n - 1;
      if (r < 0) {
        r = -1;
        c = 0;
        return;
      }
      st = __ldg(cu + r);
      ln = __ldg(cu + r + 1) - st;
      c = s - (st / CH + r);
    }
    if (r < 0 || r >= B || c < 0 || st < 0 || ln < 0 || st + ln > Ttot || c * CH >= ln) r = -1;
  }
};

// (row, chunk) of slot s after the front kernel of the same call: packed rows
// read the front kernel's map (one load through L2, and callable by a single
// thread, unlike the warp-wide search over the row offsets); dense rows
// compute it.
__device__ __forceinline__ void slot_row(const Rows &R, const Ws &W, int s, int Ttot, int &r, int &c) {
  if (R.cu) {
    const int2 v = __ldcg(W.slot_rc + s);
    r = v.x;
    c = v.y;
  } else {
    R.locate(s, Ttot, r, c);
  }
}

// Bounded mbarrier wait agreed across the CTA (thread 0 polls, the rest sleep
// in the barrier); false = give up. abort (thread 0): do not wait at all, the
// CTA leaves (thread 0 has already recorded why).
__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t parity, unsigned int *status, bool abort = false) {
  const bool lead = threadIdx.x == 0;
  bool ok = true;
  if (lead) ok = !abort && mbar_wait_bounded(bar, parity);
  if (__syncthreads_or(!ok)) {
    if (lead && !abort) set_status(status, GDN_ERR_TIMEOUT);
    return false;
  }
  if (!lead) (void)mbar_try_wait(bar, parity);
  return true;
}

// The same for two barriers at once (one CTA barrier instead of two).
__device__ __forceinline__ bool cta_wait2(uint64_t *b0, uint32_t p0, uint64_t *b1, uint32_t p1, unsigned int *status) {
  const bool lead = threadIdx.x == 0;
  bool ok = true;
  if (lead) ok = mbar_wait_bounded(b0, p0) && mbar_wait_bounded(b1, p1);
  if (__syncthreads_or(!ok)) {
    if (lead) set_status(status, GDN_ERR_TIMEOUT);
    return false;
  }
  if (!lead) {
    (void)mbar_try_wait(b0, p0);
    (void)mbar_try_wait(b1, p1);
  }
  return true;
}

// A chunk unit's completion flag: set with release semantics at GPU scope,
// read with acquire semantics (both through L2).
__device__ __forceinline__ void release_flag(int *flag) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
}
__device__ __forceinline__ bool acquire_flag(const int *flag) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
  return v != 0;
}
__device__ __forceinline__ bool relaxed_flag(const int *flag) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
  return v != 0;
}
// With a relaxed read of a flag before it, an acquire of what the flag's release published.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// Orders this thread's bulk (async-proxy) global accesses with its generic ones.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Named barrier `id` over `n` threads (whole warps).
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ------------------------------------------------------------ SiLU

// x / (1 + 2^(-x log2 e)) with the approximate base-2 exponential and
// reciprocal instructions (relative error of each ~2^-22; denormals flush to
// zero); for large negative x, 2^(...) is +inf and the result -0.
__device__ __forceinline__ float silu_approx(float x) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return x * r;
}
// the depthwise conv of one channel at one token (taps x0 .. x3, x3 the current token), then SiLU
__device__ __forceinline__ float conv4_silu_approx(float w0, float w1, float w2, float w3, float x0, float x1, float x2,
                                                   float x3) {
  return silu_approx(fmaf(w3, x3, fmaf(w2, x2, fmaf(w1, x1, w0 * x0))));
}

// ------------------------------------------------------------ split fp16

__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
  // paired conversions (each half rounded to nearest, as one at a time would be)
  const __half2 h2 = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h2);
  const __half2 l2 = __floats2half2_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h2);
  lo = *reinterpret_cast<const uint32_t *>(&l2);
}
__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo) {
  split2(x[0], x[1], hi.x, lo.x);
  split2(x[2], x[3], hi.y, lo.y);
  split2(x[4], x[5], hi.z, lo.z);
  split2(x[6], x[7], hi.w, lo.w);
}
// hi + lo of one fp16 pair of a split value
__device__ __forceinline__ float2 join2(uint32_t hi, uint32_t lo) {
  const float2 h = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
  const float2 l = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
  return make_float2(h.x + l.x, h.y + l.y);
}
// D = A B^T in split fp16: hi*hi + hi*lo + lo*hi (three accumulating tiles)
__device__ __forceinline__ void umma_tile_split(uint32_t tmem_d, uint32_t a_hi, uint32_t a_lo, int RA, uint32_t b_hi,
                                                uint32_t b_lo, int RB, int K, uint32_t idesc) {
  umma_tile(tmem_d, a_hi, RA, b_hi, RB, K, idesc, false);
  umma_tile(tmem_d, a_hi, RA, b_lo, RB, K, idesc, true);
  umma_tile(tmem_d, a_lo, RA, b_hi, RB, K, idesc, true);
}

// D = A B in split fp16 with B read MN-major (blocks lbo bytes apart)
__device__ __forceinline__ void umma_tile_split_bmn(uint32_t tmem_d, uint32_t a_hi, uint32_t a_lo, int RA,
                                                    uint32_t b_hi, uint32_t b_lo, uint32_t lbo, int K,
                                                    uint32_t idesc) {
  umma_tile_bmn(tmem_d, a_hi, RA, b_hi, lbo, K, idesc, false);
  umma_tile_bmn(tmem_d, a_hi, RA, b_lo, lbo, K, idesc, true);
  umma_tile_bmn(tmem_d, a_lo, RA, b_hi, lbo, K, idesc, true);
}

// ------------------------------------------------------------ front end

// One CTA per (chunk slot, q/k/v head): 256 threads, thread = 8 channels (cb)
// x 4 tokens (tb) in registers. A token's 128 channels sit in one half-warp,
// so its L2 norm is a 16-lane butterfly, and each thread's 16-byte chunks of
// the [token][d] image are stored straight from registers (a warp writes
// whole lines).
// GATES: the value-head CTAs also form the chunk's gates (for calls whose chunk
// pass runs as its own kernel, where the units are the critical path; a
// compile-time choice, so the other instantiation carries none of that code).
template <bool GATES>
__global__ void __launch_bounds__(256, 4) front_kernel(LayerArgs A, Rows R, int Ttot, Ws W) {
  griddep_wait();  // the kernel before this call (a previous layer call) is complete
  griddep_trigger();
  const int tid = threadIdx.x;
  const int s = blockIdx.x, gi = blockIdx.y, kd = A.nk * HD;
  if (tid == 0 && gi >= 2 * A.nk) W.flag[(size_t)s * A.nv + gi - 2 * A.nk] = 0;  // unit (s, h) not yet published
  int r, c;
  R.locate(s, Ttot, r, c);
  if (tid == 0 && gi == 0) W.slot_rc[s] = make_int2(r, c);
  if (r < 0) return;
  const int start = R.start(r), len = R.len(r);
  const int which = gi < A.nk ? 0 : (gi < 2 * A.nk ? 1 : 2);
  const int head = which == 0 ? gi : (which == 1 ? gi - A.nk : gi - 2 * A.nk);
  const int slot = row_slot(A, r);
  // value heads: warp 0 also forms the chunk's gates (gdn_gates: g = -exp(A_log)
  // softplus(a + dt_bias), beta = sigmoid(b); g = beta = 0 on padding and past
  // the row end), two tokens per lane. Their inputs are loaded now and used
  // after the images are stored: these CTAs skip the L2 norm, so they have the
  // time the q / k CTAs spend on it.
  const bool gate_warp = GATES && which == 2 && tid < 32;
  float ga[2] = {0.f, 0.f}, gb[2] = {0.f, 0.f};
  bool greal[2] = {false, false};
  if (gate_warp) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = 2 * tid + e;
      if (c * CH + i < len) {
        const size_t p = (size_t)start + c * CH + i;
        greal[e] = !A.mask || A.mask[p] == 1.0f;
        ga[e] = ldbf(A.a + p * A.nv + head);
        gb[e] = ldbf(A.b + p * A.nv + head);
      }
    }
  }
  const int cb = tid & 15, tb = tid >> 4, pos0 = c * CH + 4 * tb;
  const int ch0 = which == 0 ? head * HD : (which == 1 ? kd + head * HD : 2 * kd + head * HD);
  const bf16 *src = which == 0 ? A.q + head * HD : (which == 1 ? A.k + head * HD : A.v + head * HD);
  const size_t rstride = which == 2 ? (size_t)A.nv * HD : (size_t)kd;
  // 16-byte loads of the 7 input rows pos0-3 .. pos0+3 (8 channels each) and of the weights
  uint4 xv[7];
#pragma unroll
  for (int j = 0; j < 7; ++j) {
    const int ip = pos0 - KC + j;
    xv[j] = make_uint4(0u, 0u, 0u, 0u);
    if (slot >= 0 && ip < len) {
      if (ip >= 0)
        xv[j] = __ldg(reinterpret_cast<const uint4 *>(src + (size_t)(start + ip) * rstride) + cb);
      else
        xv[j] = *reinterpret_cast<const uint4 *>(A.conv_state + (size_t)slot * KC * A.C + (size_t)(KC + ip) * A.C +
                                                 ch0 + 8 * cb);
    }
  }
  uint4 wv[4];  // channel 8cb + 2q + (e>>1): taps in bf16 pairs
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) wv[q4] = __ldg(reinterpret_cast<const uint4 *>(A.conv_w + (size_t)(ch0 + 8 * cb) * 4) + q4);
  float y[4][8];  // [token][channel]
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t wp[4] = {wv[e >> 1].x, wv[e >> 1].y, wv[e >> 1].z, wv[e >> 1].w};
    const uint32_t w01 = wp[2 * (e & 1)], w23 = wp[2 * (e & 1) + 1];
    const float w0 = __uint_as_float(w01 << 16), w1 = __uint_as_float(w01 & 0xffff0000u);
    const float w2 = __uint_as_float(w23 << 16), w3 = __uint_as_float(w23 & 0xffff0000u);
    float x[7];
#pragma unroll
    for (int j = 0; j < 7; ++j) {
      const uint32_t xp[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
      x[j] = (e & 1) ? __uint_as_float(xp[e >> 1] & 0xffff0000u) : __uint_as_float(xp[e >> 1] << 16);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t)
      y[t][e] = (slot >= 0 && pos0 + t < len) ? conv4_silu_approx(w0, w1, w2, w3, x[t], x[t + 1], x[t + 2], x[t + 3])
                                              : 0.0f;
  }
  // q, k: L2 norm per token over the 16 lanes of the half-warp; then the
  // [token][d] image, each thread's chunks straight from registers
  const float sc = which == 0 ? A.scale : 1.0f;
  unsigned char *img = reinterpret_cast<unsigned char *>(
      which == 2 ? W.vimg + ((size_t)s * A.nv + head) * 2 * kImg
                 : (which == 0 ? W.qimg : W.kimg) + ((size_t)s * A.nk + head) * 2 * kImg);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    if (which < 2) {
      float ss = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = __fmaf_rn(y[t][e], y[t][e], ss);
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
      const float rn = sc * rsqrtf(ss + A.l2_eps);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[t][e] = __fmul_rn(y[t][e], rn);
    }
    uint4 hi, lo;
    split8(y[t], hi, lo);
    const uint32_t off = sw128_chunk(CH, 4 * tb + t, cb);
    *reinterpret_cast<uint4 *>(img + off) = hi;
    *reinterpret_cast<uint4 *>(img + kImg * 2 + off) = lo;
  }
  if (gate_warp) {
    // the gates, then G = the inclusive prefix of g, exp(G), exp(G_C - G) and
    // gamma_C = exp(G_C): the same arithmetic as the chunk unit's
    const int lane = tid;
    float g[2], be[2];
    const float eA = -expf(A.A_log[head]), dtb = A.dt_bias[head];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      g[e] = greal[e] ? __fmul_rn(eA, softplus_f(__fadd_rn(ga[e], dtb))) : 0.f;
      be[e] = greal[e] ? sigmoid_f(gb[e]) : 0.f;
    }
    const float v0 = g[0], v1 = v0 + g[1];
    float run = v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, run, o);
      if (lane >= o) run += t;
    }
    const float G0 = run - v1 + v0, G1 = run;
    const float GC = __shfl_sync(0xffffffffu, run, 31);
    float *rec = W.gate + ((size_t)s * A.nv + head) * kGateRec;
    reinterpret_cast<float2 *>(rec)[lane] = make_float2(g[0], g[1]);
    reinterpret_cast<float2 *>(rec + 64)[lane] = make_float2(be[0], be[1]);
    reinterpret_cast<float2 *>(rec + 128)[lane] = make_float2(G0, G1);
    const float gam1 = __expf(G1);
    reinterpret_cast<float2 *>(rec + 192)[lane] = make_float2(__expf(G0), gam1);
    reinterpret_cast<float2 *>(rec + 256)[lane] = make_float2(__expf(GC - G0), __expf(GC - G1));
    if (lane == 31) rec[320] = gam1;  // gamma_C
  }
}

// ------------------------------------------------------------ chunk-local

// Shared memory of a chunk unit (chunk_kernel, chunk_state_kernel; bytes from
// a 1024-aligned base). "hi"/"lo" are the two fp16 parts of a split operand.
// The K|Q region [0, 64 KiB) and the A / T / [T; R] / P region [128, 192 KiB)
// below are the layout of an even unit; an odd unit swaps the two.
constexpr int kOffKQH = 0;       // [2 kb][128 rows][128 B]: K rows 0-63 | Q rows 64-127 (hi); later W|Q'
constexpr int kOffKQL = 32768;   // the same, lo parts
constexpr int kOffB2H = 65536;   // V image [2 kb][64 rows][128 B] (hi), then the lo parts at +16 KiB;
                                 // at the end the U | O_local staging (64 KiB)
constexpr int kOffAF = 131072;   // fp32 [64][kLD]: A, then T in place; later the [T; R] image (hi)
constexpr int kLD = 68;          // padded row stride: 16-byte aligned rows, and a 16-byte chunk of rows
                                 // i .. i+7 in eight different bank groups (the 1 KiB past 16 KiB
                                 // overlaps the [T; R] lo image, unused until then)
constexpr int kOffTRL = 147456;  // [T; R] image (lo)
constexpr int kOffPTH = 163840;  // [128 rows][128 B]: P rows 0-63 | T^T rows 64-127 (hi)
constexpr int kOffPTL = 180224;  // the same, lo parts
constexpr int kOffSCR = 196608;  // fp32 [1024] solve scratch
constexpr int kOffSm = 200704;   // 2 x the unit's gates g, beta, G, exp(G), exp(G_C - G): fp32 [5][64]
                                 // (unit parity p uses buffer p); barriers; tmem base
constexpr int kOffBar = kOffSm + 2 * kGateLd * 4;  // chunk-local loads and products, TMEM base
constexpr int kChunkSmem = kOffBar + 64 + 1024;     // + alignment slack

__device__ __forceinline__ void store_split8(unsigned char *hi_img, unsigned char *lo_img, uint32_t off,
                                             const float *x) {
  uint4 hi, lo;
  split8(x, hi, lo);
  *reinterpret_cast<uint4 *>(hi_img + off) = hi;
  *reinterpret_cast<uint4 *>(lo_img + off) = lo;
}

// Parities of the next phase that each barrier of the chunk-local pass
// completes; a CTA that runs several chunk units carries them from one unit to
// the next.
struct UnitPhase {
  uint32_t ld0, ld1, mma;
};

// The chunk-local pass of one (chunk slot s, value head h) unit, slot s holding
// chunk c of row r (r >= 0). Two 64 KiB regions trade roles from one unit to
// the next (parity): one holds the unit's K|Q tiles, the other its A / T /
// [T; R] / P tiles; once the unit's last products are done the second is free
// and takes the next unit's K|Q tiles (thread 0 learns the next unit, slot and
// value head, from find_next() while the first product runs). kq_issued: this
// unit's K|Q tiles were requested that way by the unit before. The caller has
// initialised the barriers at kOffBar, holds 256 TMEM columns at `tmem`
// and has synchronised the CTA since any earlier use of shared memory or TMEM.
// bars: the unit's barriers (two loads, the products).
// gates_ready: the front kernel formed the gates; they arrive with the K|Q
// tiles (else the unit forms them and stores exp(G_C - G), gamma_C for the
// state pass).
// publish: once the unit's outputs are complete in global memory, set its
// flag (release, GPU scope) for a chain pass of the same grid. Without
// publish the unit returns with its output stores possibly still reading
// shared memory; the next unit waits for them before it reuses those regions,
// and the caller before the CTA exits. Returns false when a bounded wait ran
// out (the status word is set).
template <bool GATES_READY, class FindNext>
__device__ __forceinline__ bool chunk_unit(unsigned char *sm, const LayerArgs &A, const Rows &R, const Ws &W, int s,
                                           int h, int r, int c, int parity, bool kq_issued, FindNext find_next,
                                           uint32_t tmem, uint64_t *bars, UnitPhase &ph, bool publish) {
  constexpr bool gates_ready = GATES_READY;
  const int xo = parity ? kOffAF : kOffKQH, yo = parity ? kOffKQH : kOffAF;  // K|Q region, A/T/P region
  unsigned char *KQH = sm + xo, *KQL = sm + xo + (kOffKQL - kOffKQH);
  unsigned char *B2H = sm + kOffB2H;
  float *AF = reinterpret_cast<float *>(sm + yo);
  unsigned char *TRH = sm + yo, *TRL = sm + yo + (kOffTRL - kOffAF);
  unsigned char *PTH = sm + yo + (kOffPTH - kOffAF), *PTL = sm + yo + (kOffPTL - kOffAF);
  float *SCR = reinterpret_cast<float *>(sm + kOffSCR);
  float *sg = reinterpret_cast<float *>(sm + kOffSm) + parity * kGateLd;  // g
  float *sb = sg + 64;                                   // beta
  float *sG = sb + 64;                                   // inclusive prefix of g
  float *sgam = sG + 64;                                 // exp(G_j)
  float *sec = sgam + 64;                                // exp(G_C - G_j)
  uint64_t *bar_ld = bars;  // [0]: K|Q tiles, [1]: V tiles
  uint64_t *bar_mma = bars + 2;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kh = h / A.G;
  const int start = R.start(r), len = R.len(r);
  const int nvalid = min(CH, len - c * CH);

  // thread 0: the K|Q tiles of (slot s2, key head kh2) into the region at
  // dstH (hi) / dstH + 32 KiB (lo), and with gates_ready the gates of (slot
  // s2, value head h2) into the gate buffer of parity par2
  auto issue_kq = [&](int s2, int kh2, unsigned char *dstH, int h2, int par2) {
    mbar_arrive_expect_tx(&bar_ld[0], 65536 + (gates_ready ? kGateLd * 4 : 0));
    if (gates_ready)
      bulk_g2s(reinterpret_cast<float *>(sm + kOffSm) + par2 * kGateLd, W.gate + ((size_t)s2 * A.nv + h2) * kGateRec,
               kGateLd * 4, &bar_ld[0]);
    for (int part = 0; part < 2; ++part) {
      const __half *ki = W.kimg + ((size_t)s2 * A.nk + kh2) * 2 * kImg + part * kImg;
      const __half *qi = W.qimg + ((size_t)s2 * A.nk + kh2) * 2 * kImg + part * kImg;
      unsigned char *dst = dstH + part * (kOffKQL - kOffKQH);
      bulk_g2s(dst, ki, 8192, &bar_ld[0]);                 // K, column block 0
      bulk_g2s(dst + 8192, qi, 8192, &bar_ld[0]);          // Q, column block 0
      bulk_g2s(dst + 16384, ki + 4096, 8192, &bar_ld[0]);  // K, column block 1
      bulk_g2s(dst + 24576, qi + 4096, 8192, &bar_ld[0]);  // Q, column block 1
    }
  };
  int2 nx = make_int2(-1, 0);  // thread 0: the next unit (slot, value head), slot -1 = none
  auto issue_v = [&]() {  // thread 0
    mbar_arrive_expect_tx(&bar_ld[1], 32768);
    bulk_g2s(B2H, W.vimg + ((size_t)s * A.nv + h) * 2 * kImg, 32768, &bar_ld[1]);  // hi | lo
  };
  // Without publish, the unit before may still be storing its outputs from
  // the V region and from the region this unit's A / P tiles go to: V is
  // requested, and those tiles written, once its stores have read them.
  if (tid == 0) {  // the K|Q tiles first (the first product needs them), then V
    if (!kq_issued) issue_kq(s, kh, KQH, h, parity);
    if (publish) issue_v();
  }
  // gates of the chunk's tokens; padding and tokens past the row end get g = beta = 0
  if (!gates_ready && tid < CH) {
    float g = 0.f, beta = 0.f;
    if (tid < nvalid) {
      const size_t p = (size_t)start + c * CH + tid;
      if (!A.mask || A.mask[p] == 1.0f) {
        // gdn_gates: g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)
        g = __fmul_rn(-expf(A.A_log[h]), softplus_f(__fadd_rn(ldbf(A.a + p * A.nv + h), A.dt_bias[h])));
        beta = sigmoid_f(ldbf(A.b + p * A.nv + h));
      }
    }
    sg[tid] = g;
    sb[tid] = beta;
  }
  __syncthreads();
  if (!gates_ready && warp == 0) {  // inclusive prefix over 64 values, two per lane
    const float v0 = sg[2 * lane], v1 = v0 + sg[2 * lane + 1];
    float run = v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, run, o);
      if (lane >= o) run += t;
    }
    const float excl = run - v1;
    sG[2 * lane] = excl + v0;
    sG[2 * lane + 1] = run;
    __syncwarp();
    const float GC = sG[CH - 1];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int j = 2 * lane + e;
      sgam[j] = __expf(sG[j]);
      sec[j] = __expf(GC - sG[j]);
    }
  }
  if (!cta_wait(&bar_ld[0], ph.ld0, A.status)) return false;
  ph.ld0 ^= 1;

  // ---- [K; Q] K^T -> TMEM columns [0, 64)
  if (tid == 0) {
    tc_fence_after();
    umma_tile_split(tmem, smem_u32(KQH), smem_u32(KQL), 128, smem_u32(KQH), smem_u32(KQL), 128, 128,
                    umma_idesc_f16(128, 64));
    umma_commit(bar_mma);
    nx = find_next();
  }
  if (!gates_ready && tid < CH) {  // per-token factors for the state pass: exp(G_C - G_j)
    float *rec = W.gate + ((size_t)s * A.nv + h) * kGateRec + kSecOff;
    rec[tid] = sec[tid];
    if (tid == 0) rec[CH] = sgam[CH - 1];  // gamma_C
  }
  if (!publish && (tid == 0 || tid == 128)) bulk_wait_read_all();  // the unit before's stores (see above)
  if (!cta_wait(bar_mma, ph.mma, A.status)) return false;
  ph.mma ^= 1;
  tc_fence_after();
  if (!publish && tid == 0) issue_v();
  {
    // A (rows 0-63: strictly lower, beta_i KK_ij Gamma_ij) in fp32; P (rows
    // 64-127: QK_ij Gamma_ij for j <= i) as a split image
    // rolled over 8-column groups: this code runs once per CTA, so a compact
    // loop fetches far fewer instructions than a fully unrolled one
    const int q = warp & 3, hh = warp >> 2, row = 32 * q + lane;
    const bool arow = row < CH;
    const int i = row & (CH - 1);
    const float Gi = sG[i], bi = sb[i];
#pragma unroll 1
    for (int g8 = 0; g8 < 4; ++g8) {
      // G_j of the 8 columns first: their load overlaps the TMEM load's
      const float4 ga = *reinterpret_cast<const float4 *>(sG + 32 * hh + 8 * g8);
      const float4 gb = *reinterpret_cast<const float4 *>(sG + 32 * hh + 8 * g8 + 4);
      const float Gj[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
      float v[8], y[8];
      tmem_ld8(tmem_at(tmem, q, 32 * hh + 8 * g8), v);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = 32 * hh + 8 * g8 + e;
        const float gam = __expf(Gi - Gj[e]);
        y[e] = arow ? (j < i ? bi * v[e] * gam : 0.0f) : (j <= i ? v[e] * gam : 0.0f);
      }
      if (arow) {
        float4 *dst = reinterpret_cast<float4 *>(AF + i * kLD + 32 * hh + 8 * g8);
        dst[0] = make_float4(y[0], y[1], y[2], y[3]);
        dst[1] = make_float4(y[4], y[5], y[6], y[7]);
      } else {
        store_split8(PTH, PTL, sw128_chunk(128, i, 4 * hh + g8), y);
      }
    }
  }
  tc_fence_before();
  __syncthreads();

  // ---- T = (I + A)^-1 in place by recursive doubling on the 2x2 block form
  //      inv([[X, 0], [Y, Z]]) = [[X^-1, 0], [-Z^-1 Y X^-1, Z^-1]]:
  //      the four diagonal 16x16 blocks by forward substitution, then the two
  //      16x16 off-diagonal blocks of the 32x32 diagonal blocks, then the
  //      lower-left 32x32 block. The off-diagonal products run on two / four
  //      warps, each thread accumulating a register block of the result from
  //      16-byte loads (few shared-memory loads per FMA); the other warps wait.
  float t16[16];  // T row i = tid / 4, columns 16 (tid % 4) .. +15 (kept for the second image)
  {
    if (tid < 64) {
      const int bb = tid >> 4, cc = tid & 15;
      float x[16];
      const float *Ab = AF + (16 * bb) * kLD + 16 * bb;
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) {
        float acc = rr == cc ? 1.0f : 0.0f;
#pragma unroll
        for (int l = 0; l < rr; ++l) acc = fmaf(-Ab[rr * kLD + l], x[l], acc);
        x[rr] = acc;
      }
      named_sync(1, 64);  // every diagonal block has been read
      float *Tb = AF + (16 * bb) * kLD + 16 * bb;
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) Tb[rr * kLD + cc] = x[rr];
    }
    __syncthreads();
    if (tid < 64) {
      // level 1: blocks (1,0) and (3,2), one warp each: X = A_rc T_cc, then
      // T_rc = -T_rr X; thread = a 4x2 block (rows 4bi.., columns 2bm..)
      const int pr = tid >> 5, bi = (tid >> 3) & 3, bm = tid & 7;
      const int r0 = 16 + 32 * pr, c0 = 32 * pr;
      float x[4][2];
#pragma unroll
      for (int j = 0; j < 4; ++j) x[j][0] = x[j][1] = 0.0f;
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        float4 a[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = *reinterpret_cast<const float4 *>(AF + (r0 + 4 * bi + j) * kLD + c0 + 4 * k4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float2 t = *reinterpret_cast<const float2 *>(AF + (c0 + 4 * k4 + kk) * kLD + c0 + 2 * bm);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float av = kk == 0 ? a[j].x : kk == 1 ? a[j].y : kk == 2 ? a[j].z : a[j].w;
            x[j][0] = fmaf(av, t.x, x[j][0]);
            x[j][1] = fmaf(av, t.y, x[j][1]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<float2 *>(SCR + pr * 256 + (4 * bi + j) * 16 + 2 * bm) = make_float2(x[j][0], x[j][1]);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 4; ++j) x[j][0] = x[j][1] = 0.0f;
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        float4 t[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) t[j] = *reinterpret_cast<const float4 *>(AF + (r0 + 4 * bi + j) * kLD + r0 + 4 * k4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float2 xk = *reinterpret_cast<const float2 *>(SCR + pr * 256 + (4 * k4 + kk) * 16 + 2 * bm);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float tv = kk == 0 ? t[j].x : kk == 1 ? t[j].y : kk == 2 ? t[j].z : t[j].w;
            x[j][0] = fmaf(tv, xk.x, x[j][0]);
            x[j][1] = fmaf(tv, xk.y, x[j][1]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<float2 *>(AF + (r0 + 4 * bi + j) * kLD + c0 + 2 * bm) = make_float2(-x[j][0], -x[j][1]);
    }
    __syncthreads();
    if (tid < 128) {
      // level 2: block rows 32-63, columns 0-31: Y = A_BA T_A, then T_BA = -T_B Y;
      // thread = a 4x2 block (rows 4bi.., columns 2bm..) of each 32x32 product
      const int bi = tid >> 4, bm = tid & 15;
      float y[4][2];
#pragma unroll
      for (int j = 0; j < 4; ++j) y[j][0] = y[j][1] = 0.0f;
#pragma unroll 2
      for (int k4 = 0; k4 < 8; ++k4) {
        float4 a[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = *reinterpret_cast<const float4 *>(AF + (32 + 4 * bi + j) * kLD + 4 * k4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float2 t = *reinterpret_cast<const float2 *>(AF + (4 * k4 + kk) * kLD + 2 * bm);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float av = kk == 0 ? a[j].x : kk == 1 ? a[j].y : kk == 2 ? a[j].z : a[j].w;
            y[j][0] = fmaf(av, t.x, y[j][0]);
            y[j][1] = fmaf(av, t.y, y[j][1]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<float2 *>(SCR + (4 * bi + j) * 32 + 2 * bm) = make_float2(y[j][0], y[j][1]);
      named_sync(5, 128);  // Y complete; A_BA is read
#pragma unroll
      for (int j = 0; j < 4; ++j) y[j][0] = y[j][1] = 0.0f;
#pragma unroll 2
      for (int k4 = 0; k4 < 8; ++k4) {
        float4 t[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          t[j] = *reinterpret_cast<const float4 *>(AF + (32 + 4 * bi + j) * kLD + 32 + 4 * k4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float2 yk = *reinterpret_cast<const float2 *>(SCR + (4 * k4 + kk) * 32 + 2 * bm);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float tv = kk == 0 ? t[j].x : kk == 1 ? t[j].y : kk == 2 ? t[j].z : t[j].w;
            y[j][0] = fmaf(tv, yk.x, y[j][0]);
            y[j][1] = fmaf(tv, yk.y, y[j][1]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<float2 *>(AF + (32 + 4 * bi + j) * kLD + 2 * bm) = make_float2(-y[j][0], -y[j][1]);
    }
    __syncthreads();
    // T (fp32, in AF) -> rows 0-63 of the split image [T; R] diag(beta gamma)
    // (hi aliases AF) and the split T^T image (rows 64-127 of the P tiles,
    // row j = column j of T, gathered by column)
    const int i = tid >> 2, q4 = tid & 3;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const float4 t4 = *reinterpret_cast<const float4 *>(AF + i * kLD + 16 * q4 + 4 * c4);
      t16[4 * c4] = t4.x;
      t16[4 * c4 + 1] = t4.y;
      t16[4 * c4 + 2] = t4.z;
      t16[4 * c4 + 3] = t4.w;
    }
    const int jc = tid & 63, ip = tid >> 6;  // T^T row jc, tokens 16 ip .. +15
    float tc16[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) tc16[k] = AF[(16 * ip + k) * kLD + jc];
    float bg16[16];  // beta_j gamma_j of this thread's 16 columns
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const float4 b4 = *reinterpret_cast<const float4 *>(sb + 16 * q4 + 4 * c4);
      const float4 g4 = *reinterpret_cast<const float4 *>(sgam + 16 * q4 + 4 * c4);
      bg16[4 * c4] = b4.x * g4.x;
      bg16[4 * c4 + 1] = b4.y * g4.y;
      bg16[4 * c4 + 2] = b4.z * g4.z;
      bg16[4 * c4 + 3] = b4.w * g4.w;
    }
    __syncthreads();
    float y16[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) y16[k] = t16[k] * bg16[k];
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) store_split8(TRH, TRL, sw128_chunk(128, i, 2 * q4 + c2), y16 + 8 * c2);
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) store_split8(PTH, PTL, sw128_chunk(128, CH + jc, 2 * ip + c2), tc16 + 8 * c2);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();

  // ---- R = P T -> TMEM columns [0, 64) (lanes 64-127 of this product are unused)
  if (tid == 0) {
    tc_fence_after();
    umma_tile_split(tmem, smem_u32(PTH), smem_u32(PTL), 128, smem_u32(PTH) + CH * 128, smem_u32(PTL) + CH * 128,
                    128, 64, umma_idesc_f16(128, 64));
    umma_commit(bar_mma);
  }
  if (!cta_wait(bar_mma, ph.mma, A.status)) return false;
  ph.mma ^= 1;
  tc_fence_after();
  // the P tiles are free: they take the second image [T; R] diag(beta)
  {
    const int i = tid >> 2, q4 = tid & 3;
    float y16[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) y16[k] = t16[k] * sb[16 * q4 + k];
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) store_split8(PTH, PTL, sw128_chunk(128, i, 2 * q4 + c2), y16 + 8 * c2);
  }
  if ((warp & 3) < 2) {
    const int q = warp & 3, hh = warp >> 2, i = 32 * q + lane;
#pragma unroll 1
    for (int g8 = 0; g8 < 4; ++g8) {
      const int j0 = 32 * hh + 8 * g8;
      // beta_j and gamma_j first: their loads overlap the TMEM load's
      const float4 b0 = *reinterpret_cast<const float4 *>(sb + j0), b1 = *reinterpret_cast<const float4 *>(sb + j0 + 4);
      const float4 m0 = *reinterpret_cast<const float4 *>(sgam + j0);
      const float4 m1 = *reinterpret_cast<const float4 *>(sgam + j0 + 4);
      const float bj[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
      const float mj[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
      float v[8], y[8];
      tmem_ld8(tmem_at(tmem, q, j0), v);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = v[e] * (bj[e] * mj[e]);
      store_split8(TRH, TRL, sw128_chunk(128, CH + i, 4 * hh + g8), y);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = v[e] * bj[e];
      store_split8(PTH, PTL, sw128_chunk(128, CH + i, 4 * hh + g8), y);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();

  // ---- [T; R] diag(beta gamma) K -> TMEM columns [0, 128) (W | P W) and
  //      [T; R] diag(beta) V -> columns [128, 256) (U | P U)
  if (!cta_wait(&bar_ld[1], ph.ld1, A.status)) return false;  // long landed: loaded during the steps above
  ph.ld1 ^= 1;
  if (tid == 0) {
    tc_fence_after();
    // K (rows 0-63 of the K|Q tiles, column blocks 16 KiB apart) and V (its own
    // tiles, column blocks 8 KiB apart), both read MN-major: tokens contract
    umma_tile_split_bmn(tmem, smem_u32(TRH), smem_u32(TRL), 128, smem_u32(KQH), smem_u32(KQL), 16384, 64,
                        umma_idesc_f16_bmn(128, 128));
    umma_tile_split_bmn(tmem + 128, smem_u32(PTH), smem_u32(PTL), 128, smem_u32(B2H), smem_u32(B2H) + 16384, 8192,
                        64, umma_idesc_f16_bmn(128, 128));
    umma_commit(bar_mma);
  }
  if (!cta_wait(bar_mma, ph.mma, A.status)) return false;
  ph.mma ^= 1;
  tc_fence_after();
  // the A / T / [T; R] / P tiles are consumed: that region takes the next unit's K|Q
  if (tid == 0 && nx.x >= 0) issue_kq(nx.x, nx.y / A.G, sm + yo, nx.y, parity ^ 1);
  {
    // W / Q' into the K|Q image (plain fp16); U rows (fp16) and O_local rows
    // (fp32) staged in the free B2 tiles in the row-swizzled layout of the
    // workspace (16-byte chunk c of row i at c ^ (i % 8)), then bulk-stored
    const int q = warp & 3, hh = warp >> 2, row = 32 * q + lane, i = row & (CH - 1);
    const bool upper = row >= CH;
    const float gam = sgam[i];
    float4 *stage = reinterpret_cast<float4 *>(sm + kOffB2H + 32768) + (size_t)i * 32;  // O_local row i
    uint4 *stage_u = reinterpret_cast<uint4 *>(sm + kOffB2H) + (size_t)i * 16;          // U row i
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      // Q' rows: this block's Q (hi, lo) first, every read before the first
      // store and overlapping the TMEM load
      uint4 qhv[4], qlv[4];
      if (hh == 0 && upper) {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const uint32_t off = sw128_chunk(128, row, 4 * cb + c4);
          qhv[c4] = *reinterpret_cast<const uint4 *>(KQH + off);
          qlv[c4] = *reinterpret_cast<const uint4 *>(KQL + off);
        }
      }
      float v[32];
      tmem_ld32(tmem_at(tmem, q, 128 * hh + 32 * cb), v);
      if (hh == 0) {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const uint32_t off = sw128_chunk(128, row, 4 * cb + c4);
          uint4 *dst = reinterpret_cast<uint4 *>(KQH + off);
          float y[8];
          if (upper) {
            const uint4 qh = qhv[c4], ql = qlv[c4];
            const uint32_t hs[4] = {qh.x, qh.y, qh.z, qh.w}, ls[4] = {ql.x, ql.y, ql.z, ql.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = join2(hs[e], ls[e]);
              y[2 * e] = gam * f.x - v[8 * c4 + 2 * e];
              y[2 * e + 1] = gam * f.y - v[8 * c4 + 2 * e + 1];
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = v[8 * c4 + e];
          }
          *dst = make_uint4(pack_h2(y[0], y[1]), pack_h2(y[2], y[3]), pack_h2(y[4], y[5]), pack_h2(y[6], y[7]));
        }
      } else if (upper) {
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          stage[(8 * cb + c4) ^ (i & 7)] = make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
      } else {
#pragma unroll
        for (int c2 = 0; c2 < 4; ++c2)
          stage_u[(4 * cb + c2) ^ (i & 7)] =
              make_uint4(pack_h2(v[8 * c2], v[8 * c2 + 1]), pack_h2(v[8 * c2 + 2], v[8 * c2 + 3]),
                         pack_h2(v[8 * c2 + 4], v[8 * c2 + 5]), pack_h2(v[8 * c2 + 6], v[8 * c2 + 7]));
      }
    }
    fence_proxy_async_smem();
    // each warp group stores its own tiles as soon as its 4 warps are done:
    // group 0 the W|Q' image, group 1 the U and O_local rows
    named_sync(1 + hh, 128);
    if (tid == 128 * hh) {
      const size_t sh = (size_t)s * A.nv + h;
      if (hh == 0) {
        bulk_s2g(W.wq + sh * kWQ, KQH, 32768);
      } else {
        bulk_s2g(W.ut + sh * kRowF, sm + kOffB2H, 16384);
        bulk_s2g(W.ot + sh * kRowF, sm + kOffB2H + 32768, 32768);
      }
      bulk_commit();
      if (publish) {
        bulk_wait_all();  // the writes are complete: a chain pass of this grid reads them
        fence_proxy_async_global();
      }  // else the next unit, or the CTA's exit, waits for the stores to read shared memory
    }
  }
  if (publish) {
    __syncthreads();
    if (tid == 0) {
      __threadfence();  // the other threads' stores (exp(G_C - G), gamma_C) before the flag
      release_flag(W.flag + (size_t)s * A.nv + h);
    }
  }
  return true;
}

// Persistent: one CTA per SM runs units u = blockIdx.x, + gridDim.x, ...
// (unit u = slot u / nv, value head u % nv: the value heads of a key head run
// side by side and share its K|Q tiles in L2), each unit prefetching the next
// one's K|Q tiles. Slots without a chunk are skipped.
__global__ void __launch_bounds__(256, 1) chunk_kernel(LayerArgs A, Rows R, int Ttot, Ws W, int n_units) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 6);
  __shared__ int3 s_next;  // this CTA's next unit (u, row, chunk), u -1 = none; written by thread 0
  if (threadIdx.x == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // the front kernel's images and slot map are complete
  griddep_trigger();
  // thread 0: the first unit from `from` on (stride gridDim.x) whose slot holds a chunk
  auto first_unit = [&](int from) {
    for (int v = from; v < n_units; v += gridDim.x) {
      int r, c;
      slot_row(R, W, v / A.nv, Ttot, r, c);
      if (r >= 0) return make_int3(v, r, c);
    }
    return make_int3(-1, 0, 0);
  };
  if (threadIdx.x == 0) s_next = first_unit(blockIdx.x);
  __syncthreads();
  int3 cur = s_next;
  UnitPhase ph{0u, 0u, 0u};
  int parity = 0;
  bool kq = false;
  while (cur.x >= 0) {
    // thread 0: the (row, chunk) of the next candidate unit's slot, requested
    // now (packed rows: a load through L2) and used once the unit's first
    // product is issued
    const int cand = cur.x + (int)gridDim.x;
    int2 cand_rc = make_int2(-1, 0);
    if (threadIdx.x == 0 && R.cu && cand < n_units) cand_rc = __ldcg(W.slot_rc + cand / A.nv);
    auto find_next = [&]() {  // thread 0, during the unit: published for the CTA in s_next
      int3 n;
      if (R.cu && cand < n_units && cand_rc.x >= 0) n = make_int3(cand, cand_rc.x, cand_rc.y);
      else n = first_unit(cand);
      s_next = n;
      return make_int2(n.x < 0 ? -1 : n.x / A.nv, n.x < 0 ? 0 : n.x % A.nv);
    };
    const bool ok =
        chunk_unit<true>(sm, A, R, W, cur.x / A.nv, cur.x % A.nv, cur.y, cur.z, parity, kq, find_next, tmem, bar, ph,
                         false);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!ok) break;
    cur = s_next;
    kq = true;
    parity ^= 1;
  }
  if (threadIdx.x == 0 || threadIdx.x == 128) bulk_wait_read_all();  // the last unit's stores
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------ state pass
//
// The sequential part, per (row, value head) over its chunks, with the state
// in registers (fp32) and its fp16 image in shared memory:
//   [X | O_S] = S_math [W; Q']^T (tcgen05 M=128 v, N=128 tokens, K=128),
//   U' = U - X, dS = (U' * exp(G_C - G))^T-image x K-image (M=128, N=128,
//   K=64, K read MN-major), S = gamma_C S + dS,
// and the chunk's outputs O = O_S + O_local (O_S = Q' S from the state at the
// chunk's start) with the gated RMSNorm (statecache.py, gated_rmsnorm), formed
// while the tensor cores compute dS. Padded tokens of the row get zeros.

constexpr int kSOffS = 0;         // S_math fp16 image [2 kb][128 rows][128 B] (32 KiB)
constexpr int kSOffWQ = 32768;    // 2 x W|Q' image [2 kb][128 rows][128 B] (32 KiB each)
constexpr int kSOffKT = 98304;    // 2 x K image (hi) [2 kb][64 rows][128 B] (16 KiB each), read MN-major
constexpr int kSOffUT = 131072;   // 2 x U fp16 [64 tokens][128 v] (16 KiB each)
constexpr int kSOffOL = 163840;   // O_local fp32 [64 tokens][128 v] (32 KiB; one chunk at a time)
constexpr int kSOffUP = 196608;   // U'^T image [128 rows][128 B] (16 KiB)
constexpr int kSOffZ = 212992;    // z bf16 [64 tokens][128 v] of the chunk whose outputs are formed (16 KiB)
constexpr int kSOffSec = 229376;  // 2 x the exp(G_C - G_j) | gamma_C record, fp32 [68]
constexpr int kSOffBar = kSOffSec + 2 * kSecRec * 4;  // the chain's barriers (5), TMEM base
constexpr int kStateSmem = kSOffBar + 128 + 1024;
// The outputs of a chunk are formed in buffers free at that time: o (fp32
// [64 tokens][128 v], the O_local layout) in the state image, which the first
// product has read and the step rewrites at its end; the RMS partials (fp32
// [4][64], then [64] rstd) in the chunk's U buffer, consumed before them, whose
// next loads are requested after they are read.
// chunk + state in one grid: the units' layout below kOffBar, the chain's above; barriers past both
constexpr int kMOffBar = kSOffBar > kOffBar ? kSOffBar : kOffBar;  // [0..2] units, [3..7] the chain, TMEM base
constexpr int kMergedSmem = kMOffBar + 128 + 1024;
static_assert(kStateSmem + 1024 <= 232448 && kMergedSmem + 1024 <= 232448,
              "shared memory of one CTA (with room for the static shared variables)");

// Polls of a unit flag before a blocking wait gives up (about a quarter of a
// second with the 64 ns sleeps between polls).
#ifndef GDN_FLAG_WAIT_CAP
#define GDN_FLAG_WAIT_CAP (1u << 22)
#endif

// A chain's reads of the unit flags. The test build that checks the expiry of
// the chains' flag waits (GDN_TEST_CHAIN_FLAGS_UNSET) reads every flag as
// unset, as if no unit were ever published; nothing else changes.
__device__ __forceinline__ bool chain_flag_relaxed(const int *flag) {
#ifdef GDN_TEST_CHAIN_FLAGS_UNSET
  (void)flag;
  return false;
#else
  return relaxed_flag(flag);
#endif
}
__device__ __forceinline__ bool chain_flag_acquire(const int *flag) {
#ifdef GDN_TEST_CHAIN_FLAGS_UNSET
  (void)flag;
  return false;
#else
  return acquire_flag(flag);
#endif
}

// Thread 0: is the chunk unit behind `flag` published? With `block`, wait for
// it (bounded; false and a recorded timeout when it never comes). chain: the
// reader is a state chain (see chain_flag_acquire).
__device__ __forceinline__ bool unit_ready(const int *flag, bool block, unsigned int *status, bool chain) {
  for (uint32_t i = 0;; ++i) {
    if (chain ? chain_flag_acquire(flag) : acquire_flag(flag)) {
      fence_proxy_async_global();  // the unit's bulk writes, before this thread's bulk reads
      return true;
    }
    if (!block) return false;
    if (i >= (uint32_t)GDN_FLAG_WAIT_CAP) {
      set_status(status, GDN_ERR_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
}

// What the (row b, value head h) chain needs before its chunks, and nothing
// of theirs: the row's checks (slot, mask of ones then zeros -> real length
// Lr, recorded per head for an output pass). False when the row is rejected
// (its status is set). With prefetch_state the head's fp32 state is fetched
// into L2 for the chain.
__device__ __forceinline__ bool chain_prologue(const LayerArgs &A, const Rows &R, int Ttot, const Ws &W, int b, int h,
                                               bool prefetch_state, int &Lr_out) {
  __shared__ int s_min_zero, s_max_one, s_bad;
  const int tid = threadIdx.x;
  const int start = R.start(b), len = R.len(b);
  const int slot = row_slot(A, b);
  if (slot < 0 || start < 0 || len < 0 || start + len > Ttot) {
    if (tid == 0) {
      set_status(A.status, GDN_ERR_INDEX);
      W.lr[(size_t)b * A.nv + h] = -1;
    }
    return false;
  }
  // real length: the mask row must be ones then zeros
  if (tid == 0) {
    s_min_zero = len;
    s_max_one = -1;
    s_bad = 0;
  }
  __syncthreads();
  if (A.mask)
    for (int i = tid; i < len; i += 256) {
      const float m = A.mask[start + i];
      if (m == 1.0f) atomicMax(&s_max_one, i);
      else if (m == 0.0f) atomicMin(&s_min_zero, i);
      else s_bad = 1;
    }
  __syncthreads();
  const int Lr = s_min_zero;
  if (s_bad || s_max_one >= Lr) {
    if (tid == 0) {
      set_status(A.status, GDN_ERR_MASK);
      W.lr[(size_t)b * A.nv + h] = -1;
    }
    return false;
  }
  if (tid == 0) W.lr[(size_t)b * A.nv + h] = Lr;  // read by an output pass
  Lr_out = Lr;
  if (prefetch_state) {  // 64 KiB: two 128-byte lines per thread
    const char *gS = reinterpret_cast<const char *>(A.state + ((size_t)slot * A.nv + h) * HD * HD);
    prefetch_l2(gS + 256 * tid);
    prefetch_l2(gS + 256 * tid + 128);
  }
  return true;
}

// The end of an accepted (row b, value head h) chain: when it completed, the
// conv-tail update of the head's own channels, xin rows Lr .. Lr+2 (old rows
// when Lr < 3), in place; when it stopped (a wait expired, or this grid's
// units did not complete), the head is marked so that an output pass writes
// nothing for it, and its state and conv-tail channels stay as they were.
__device__ __forceinline__ void chain_finish(const LayerArgs &A, const Rows &R, const Ws &W, int b, int h, int Lr,
                                             bool completed) {
  if (completed) {
    bf16 *cs = A.conv_state + (size_t)row_slot(A, b) * KC * A.C;
    conv_tail_at<HD>(A, R.start(b), h, Lr, cs, cs);
  } else if (threadIdx.x == 0) {
    W.lr[(size_t)b * A.nv + h] = -1;
  }
}

// The sequential pass of one (row b, value head h) chain, after its
// chain_prologue accepted the row. bars: the chain's barriers (two loads, the
// products, O_local, z). zmap (with OUT): z viewed as [tokens][nv*dv] bf16,
// box [64 tokens][128]. The caller holds 256 TMEM columns at `tmem` and has
// synchronised the CTA since any earlier use of shared memory or TMEM.
// OUT: the chain forms the chunks' outputs (else it copies out the state image
// at every chunk start, for the output kernel). wait_units: the chunk units run
// in this grid, so each chunk's loads wait for its unit's flag. Returns false
// when a bounded wait ran out (with OUT the outputs of the chunks before it are
// written).
template <bool OUT>
__device__ __forceinline__ bool state_chain(unsigned char *sm, uint64_t *bars, const LayerArgs &A, const Rows &R,
                                            const Ws &W, int b, int h, int Lr, uint32_t tmem, bool wait_units,
                                            const CUtensorMap *zmap) {
  uint64_t *bar_ld = bars, *bar_mma = bars + 2, *bar_ol = bars + 3, *bar_z = bars + 4;
  unsigned char *SI = sm + kSOffS;
  unsigned char *UP = sm + kSOffUP;
  float *OL = reinterpret_cast<float *>(sm + kSOffOL);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kh = h / A.G;
  const int start = R.start(b), len = R.len(b), slot = row_slot(A, b);
  const int n_chunks = (len + CH - 1) / CH;
  const int s0 = R.slot0(b);
  __shared__ RowCkpts ck;  // checkpoints this row asked for (prefix-cache states inside the call)
  if (tid == 0) {
    ck.n = 0;
    if (A.n_ckpt > 0) gather_row_ckpts(A, b, h, Lr, ck);
  }

  // chunk ci's W|Q' image, the fp16 K image (hi) of the key head, U and exp(G_C - G)
  constexpr uint32_t kLdBytes = 32768 + 16384 + 16384 + kSecRec * 4;
  // copy `part` (0-3, or all four with -1) of chunk ci's loads
  auto issue_part = [&](int ci, int part) {
    const int buf = ci & 1, s = s0 + ci;
    const size_t sh = (size_t)s * A.nv + h;
    if (part < 0 || part == 0) bulk_g2s(sm + kSOffWQ + buf * 32768, W.wq + sh * kWQ, 32768, &bar_ld[buf]);
    if (part < 0 || part == 1)
      bulk_g2s(sm + kSOffKT + buf * 16384, W.kimg + ((size_t)s * A.nk + kh) * 2 * kImg, 16384, &bar_ld[buf]);
    if (part < 0 || part == 2) bulk_g2s(sm + kSOffUT + buf * 16384, W.ut + sh * kRowF, 16384, &bar_ld[buf]);
    if (part < 0 || part == 3)
      bulk_g2s(sm + kSOffSec + buf * kSecRec * 4, W.gate + sh * kGateRec + kSecOff, kSecRec * 4, &bar_ld[buf]);
  };
  auto issue_loads = [&](int ci) {  // thread 0
    mbar_arrive_expect_tx(&bar_ld[ci & 1], kLdBytes);
    issue_part(ci, -1);
  };
  // thread 0: the last chunk whose loads are issued, and the last chunk up to
  // which every unit is known published and acquired; gave_up: a unit's flag
  // wait expired (no load of that chunk is in flight), the chain stops
  int issued = -1, acquired = wait_units ? -1 : n_chunks - 1;
  bool gave_up = false;
  // thread 0: O_local has one buffer: chunk ci's is requested once chunk
  // ci - 1's outputs have read theirs and chunk ci's unit is acquired
  int ol_issued = -1, ol_done = -1;
  auto try_issue_ol = [&]() {
    const int ci = ol_issued + 1;
    if (OUT && ci < n_chunks && ol_done == ol_issued && issued >= ci) {
      mbar_arrive_expect_tx(bar_ol, 32768);
      bulk_g2s(sm + kSOffOL, W.ot + ((size_t)(s0 + ci) * A.nv + h) * kRowF, 32768, bar_ol);
      ol_issued = ci;
    }
  };
  auto issue_when_ready = [&](int ci, bool block) {  // thread 0
    if (gave_up) return;
    if (ci <= acquired || unit_ready(W.flag + (size_t)(s0 + ci) * A.nv + h, block, A.status, true)) {
      if (ci > acquired) acquired = ci;
      issue_loads(ci);
      issued = ci;
      try_issue_ol();
    } else if (block) {
      gave_up = true;
    }
  };
  // thread 0: the last chunk from `from` on up to which (consecutively) the units
  // read as published, with unordered reads of up to 8 flags at once; from - 1
  // when none
  auto scan_published = [&](int from) {
    bool f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      f[e] = from + e < n_chunks && chain_flag_relaxed(W.flag + (size_t)(s0 + from + e) * A.nv + h);
    int seen = from - 1;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (f[e] && seen == from + e - 1) seen = from + e;
    return seen;
  };
  // same grid: chunk 0's loads (one acquire of its flag) before the state's;
  // the later units are scanned by the first step, after its first product
  if (wait_units && tid == 0 && n_chunks > 0) issue_when_ready(0, true);
  // thread <-> (value row v = TMEM lane, key half / token half hh)
  const int q = warp & 3, hh = warp >> 2, v = 32 * q + lane;
  float Sv[64];
  float *gS = A.state + ((size_t)slot * A.nv + h) * HD * HD;
#pragma unroll
  for (int k = 0; k < 64; ++k) Sv[k] = gS[(size_t)(64 * hh + k) * HD + v];
  auto write_simg = [&]() {
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8)
      *reinterpret_cast<uint4 *>(SI + sw128_chunk(128, v, 8 * hh + c8)) =
          make_uint4(pack_h2(Sv[8 * c8], Sv[8 * c8 + 1]), pack_h2(Sv[8 * c8 + 2], Sv[8 * c8 + 3]),
                     pack_h2(Sv[8 * c8 + 4], Sv[8 * c8 + 5]), pack_h2(Sv[8 * c8 + 6], Sv[8 * c8 + 7]));
    fence_proxy_async_smem();
  };
  write_simg();
  griddep_wait();  // the chunk kernel's outputs are complete (a no-op when this grid makes them)
  griddep_trigger();
  if (!wait_units && tid == 0 && n_chunks > 0) issue_when_ready(0, true);
  tc_fence_before();
  __syncthreads();
  if (!OUT && tid == 0 && n_chunks > 0) {  // the state image at the start of chunk 0
    bulk_s2g(W.simg + ((size_t)s0 * A.nv + h) * kWQ, SI, 32768);
    bulk_commit();
  }
  // the output rows' layout: thread r = tid % 128 of warp group hh takes values
  // 8c .. 8c+7 (c = r % 16) of tokens 32hh + r / 16 + 8k, k = 0..3
  const int orow = 32 * hh + ((tid & 127) >> 4), oc = tid & 15;
  float wn[8];  // the RMSNorm weights of those values
#pragma unroll
  for (int e = 0; e < 8; ++e) wn[e] = OUT ? ldbf(A.norm_w + 8 * oc + e) : 0.0f;
  // thread 0: chunk ci's z tile (rows past the tensor read as zeros), once
  // chunk ci - 1's outputs have read theirs
  auto load_z = [&](int ci) {
    mbar_arrive_expect_tx(bar_z, 16384);
    tma_load_2d(sm + kSOffZ, zmap, h * HD, start + ci * CH, bar_z);
  };
  if (OUT && tid == 0 && n_chunks > 0) load_z(0);

  bool ok = true;
  for (int ci = 0; ci < n_chunks; ++ci) {
    const int buf = ci & 1, t0 = ci * CH;
    const int ntok = min(CH, len - t0), nreal = max(0, min(CH, Lr - t0));
    int seen = -1;  // thread 0: the last chunk up to which the units read as published (unordered reads)
    // without unit flags (every chunk published before this grid), the next
    // chunk's four copies are issued by four threads once the product below is
    // on its way (threads 0, 32, 64, 96), their byte count expected here first
    const bool split_next = !wait_units && ci + 1 < n_chunks;
    if (split_next && tid == 0) {
      mbar_arrive_expect_tx(&bar_ld[(ci + 1) & 1], kLdBytes);
      issued = ci + 1;
    }
    if (wait_units && tid == 0) {  // a chunk not prefetched is waited for; the next one is prefetched when ready
      if (issued < ci) issue_when_ready(ci, true);
      if (issued == ci && ci + 1 < n_chunks) {
        if (ci + 1 <= acquired) {
          issue_loads(ci + 1);
          issued = ci + 1;
        } else {
          seen = scan_published(ci + 1);
        }
      }
    }
    if (!cta_wait(&bar_ld[buf], (uint32_t)((ci >> 1) & 1), A.status, gave_up)) {
      ok = false;
      break;
    }
    const float gC = reinterpret_cast<const float *>(sm + kSOffSec + buf * kSecRec * 4)[CH];
    if (tid == 0) {
      tc_fence_after();
      // rows 0-63 of the W|Q' image are W (N=64), all 128 rows [W; Q'] (N=128)
      umma_tile(tmem, smem_u32(SI), 128, smem_u32(sm + kSOffWQ + buf * 32768), 128, 128,
                umma_idesc_f16(128, OUT ? 128 : 64), false);
      umma_commit(bar_mma);
      if (seen > ci) {  // published: one acquire for all of them (off the product's path), then the loads
        fence_acq_rel_gpu();
        fence_proxy_async_global();
        acquired = seen;
        issue_loads(ci + 1);
        issued = ci + 1;
      }
    }
    if (split_next && (tid & 31) == 0 && tid < 128) issue_part(ci + 1, tid >> 5);
    if (!cta_wait(bar_mma, 0, A.status)) {
      ok = false;
      break;
    }
    tc_fence_after();
    {
      // (U - W S) * exp(G_C - G) for tokens 32hh .. 32hh+31 of value row v -> fp16 image row v
      const __half *ut = reinterpret_cast<const __half *>(sm + kSOffUT + buf * 16384);
      const float *sec = reinterpret_cast<const float *>(sm + kSOffSec + buf * kSecRec * 4) + 32 * hh;
      float x[32];
      tmem_ld32(tmem_at(tmem, q, 32 * hh), x);
#pragma unroll
      for (int e = 0; e < 32; ++e) {  // every read before the first store (see the output rows)
        const int i = 32 * hh + e;     // token; element (i, v) sits in chunk (v / 8) ^ (i % 8) of row i
        x[e] = (__half2float(ut[i * HD + ((((v >> 3) ^ (i & 7))) << 3) + (v & 7)]) - x[e]) * sec[e];
      }
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
        *reinterpret_cast<uint4 *>(UP + sw128_chunk(128, v, 4 * hh + c4)) =
            make_uint4(pack_h2(x[8 * c4], x[8 * c4 + 1]), pack_h2(x[8 * c4 + 2], x[8 * c4 + 3]),
                       pack_h2(x[8 * c4 + 4], x[8 * c4 + 5]), pack_h2(x[8 * c4 + 6], x[8 * c4 + 7]));
      fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      umma_tile_bmn(tmem + 128, smem_u32(UP), 128, smem_u32(sm + kSOffKT + buf * 16384), 8192, 64,
                    umma_idesc_f16_bmn(128, 128), false);
      umma_commit(bar_mma);
      if (!OUT) bulk_wait_read_all();  // the copy of the previous state image has left shared memory
    }
    // ---- the chunk's outputs while dS forms: O = O_S + O_local (value row v =
    //      TMEM lane, tokens 32hh .. 32hh+31 = TMEM columns 64 + 32hh ..), then
    //      the gated RMSNorm over the 128 value rows of each token
    if (OUT && !cta_wait2(bar_ol, (uint32_t)(ci & 1), bar_z, (uint32_t)(ci & 1), A.status)) {
      ok = false;
      break;
    }
    if (OUT) {
      float *red = reinterpret_cast<float *>(sm + kSOffUT + buf * 16384);  // [4][64] (see kStateSmem)
      float *rstd = red + 256;                                            // [64]
      float *OS = reinterpret_cast<float *>(SI);                         // o, in the O_local layout
      float o[32];
      tmem_ld32(tmem_at(tmem, q, 64 + 32 * hh), o);
      // o += O_local (element (i, v) sits in chunk (v / 4) ^ (i % 8) of row i), kept in OS
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int i = 32 * hh + e;
        o[e] += OL[i * HD + ((((v >> 2) ^ (i & 7))) << 2) + (v & 3)];
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int i = 32 * hh + e;
        OS[i * HD + ((((v >> 2) ^ (i & 7))) << 2) + (v & 3)] = o[e];
      }
      // sum over the warp's 32 rows of o^2 for each of the 32 tokens: after the
      // transposing butterfly lane l holds token l's partial
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] *= o[e];
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int e = 0; e < w; ++e) {
          const float send = up ? o[e] : o[e + w];
          const float keep = up ? o[e + w] : o[e];
          o[e] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
      }
      red[q * 64 + 32 * hh + lane] = o[0];
      __syncthreads();
      if (tid == 0) {  // every thread has read this chunk's O_local: the next chunk's may come
        ol_done = ci;
        try_issue_ol();
      }
      if (q == 0) {
        const int t = 32 * hh + lane;
        const float ss = red[t] + red[64 + t] + red[128 + t] + red[192 + t];
        rstd[t] = rsqrtf(ss / (float)HD + A.rms_eps);
      }
      named_sync(3 + hh, 128);
      // the bf16 rows, 16 bytes per access; padded tokens of the row get zeros
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = orow + 8 * k;
        if (i < ntok) {
          uint4 res = make_uint4(0u, 0u, 0u, 0u);
          if (i < nreal) {
            const float4 oa = *reinterpret_cast<const float4 *>(OS + i * HD + (((2 * oc) ^ (i & 7)) << 2));
            const float4 ob = *reinterpret_cast<const float4 *>(OS + i * HD + (((2 * oc + 1) ^ (i & 7)) << 2));
            const float rs = rstd[i];
            const float ov[8] = {oa.x, oa.y, oa.z, oa.w, ob.x, ob.y, ob.z, ob.w};
            const uint4 zk = *reinterpret_cast<const uint4 *>(sm + kSOffZ + (size_t)(i * HD + 8 * oc) * 2);
            const uint32_t zw[4] = {zk.x, zk.y, zk.z, zk.w};
            uint32_t pw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float z0 = __uint_as_float(zw[e] << 16), z1 = __uint_as_float(zw[e] & 0xffff0000u);
              const float y0 = ov[2 * e] * rs * (wn[2 * e] * silu_approx(z0));
              const float y1 = ov[2 * e + 1] * rs * (wn[2 * e + 1] * silu_approx(z1));
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(y0, y1);
              pw[e] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            res = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          }
          reinterpret_cast<uint4 *>(A.out + ((size_t)(start + t0 + i) * A.nv + h) * HD)[oc] = res;
        }
      }
    }
    if (!cta_wait(bar_mma, 1, A.status)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (OUT && tid == 0 && ci + 1 < n_chunks) load_z(ci + 1);  // every thread has read this chunk's z
    // S = gamma_C S + dS
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float d[32];
      tmem_ld32(tmem_at(tmem, q, 128 + 64 * hh + 32 * half), d);
#pragma unroll
      for (int e = 0; e < 32; ++e) Sv[32 * half + e] = fmaf(gC, Sv[32 * half + e], d[e]);
    }
    // checkpoints inside this chunk: the state at a chunk end, or at the real
    // end Lr (the padded tokens after it change nothing), and the conv tail there
    for (int e = 0; e < ck.n; ++e) {
      if ((ck.pos[e] - 1) / CH != ci) continue;
      float *cS = A.ckpt_state + ((size_t)ck.slot[e] * A.nv + h) * HD * HD;
#pragma unroll
      for (int k = 0; k < 64; ++k) cS[(size_t)(64 * hh + k) * HD + v] = Sv[k];
      conv_tail_at<HD>(A, R.start(b), h, ck.pos[e], A.conv_state + (size_t)slot * KC * A.C,
                       A.ckpt_conv + (size_t)ck.slot[e] * KC * A.C);
    }
    write_simg();
    tc_fence_before();
    __syncthreads();
    if (!OUT && tid == 0 && ci + 1 < n_chunks) {  // the state image at the start of chunk ci + 1
      bulk_s2g(W.simg + ((size_t)(s0 + ci + 1) * A.nv + h) * kWQ, SI, 32768);
      bulk_commit();
    }
  }
  if (!OUT && tid == 0) bulk_wait_read_all();  // no bulk store may still read this CTA's shared memory
  if (!ok) return false;
#pragma unroll
  for (int k = 0; k < 64; ++k) gS[(size_t)(64 * hh + k) * HD + v] = Sv[k];
  return true;
}

__global__ void __launch_bounds__(256, 1) state_kernel(LayerArgs A, Rows R, int Ttot, Ws W,
                                                       const __grid_constant__ CUtensorMap zmap) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + kSOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 5);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int b = blockIdx.x / A.nv, h = blockIdx.x % A.nv;
  int Lr = 0;
  if (chain_prologue(A, R, Ttot, W, b, h, false, Lr))
    chain_finish(A, R, W, b, h, Lr, state_chain<true>(sm, bar, A, R, W, b, h, Lr, tmem, false, &zmap));
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------ chunk + state in one grid
//
// For calls with few (row, head) chains (a 512-token call of one row has 32):
// the grid is one CTA per SM. The last B*nv CTAs each run the unit of their
// own chain's first chunk, then the chain, loading every later chunk as soon
// as its unit is published; the other CTAs run the later chunks' units in
// chunk-major order (all chains' second chunks first) and publish each unit's
// flag. The chains' early chunks thus overlap the units of the late chunks.
// The chain CTAs are at most half the grid, and no CTA waits on another before
// its units are done, so the units always complete; every wait is bounded.
__global__ void __launch_bounds__(256, 1) chunk_state_kernel(LayerArgs A, Rows R, int Ttot, Ws W) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + kMOffBar);  // [0..2] units, [3..6] the chain
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 8);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // the front kernel's images and the zeroed flags are complete
  const int BH = A.B * A.nv, n_units = R.B * R.cpr * A.nv;
  const int j = (int)gridDim.x - 1 - (int)blockIdx.x;  // chain of this CTA when j < BH
  int Lr = 0;
  const bool chain = j < BH && chain_prologue(A, R, Ttot, W, j / A.nv, j % A.nv, true, Lr);
  UnitPhase ph{0u, 0u, 0u};
  bool ok = true;
  int parity = 0;
  // units in chunk-major order, u = chunk * BH + row * nv + head. A chain CTA
  // runs one unit, the first chunk of its own chain (u = j), so that its first
  // step waits for no other CTA; the other CTAs share the later chunks' units
  const int u0 = j < BH ? j : BH + (int)blockIdx.x;
  const int ustep = j < BH ? n_units : (int)gridDim.x - BH;
  for (int u = u0; ok && u < n_units; u += ustep, parity ^= 1) {
    const int c = u / BH, rh = u % BH, r = rh / A.nv;  // unit (chunk c, row r, head rh % nv)
    auto find_next = [&]() {
      const int v = u + ustep, c2 = v / BH, rh2 = v % BH;
      return v < n_units ? make_int2((rh2 / A.nv) * R.cpr + c2, rh2 % A.nv) : make_int2(-1, 0);
    };
    ok = chunk_unit<false>(sm, A, R, W, r * R.cpr + c, rh % A.nv, r, c, parity, u != u0, find_next, tmem, bar, ph,
                           true);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  // the output kernel may start once every CTA is past its units (it acquires
  // the units' flags itself and waits for this grid before the state images)
  griddep_trigger();
  if (chain)
    chain_finish(A, R, W, j / A.nv, j % A.nv, Lr,
                 ok && state_chain<false>(sm, bar + 3, A, R, W, j / A.nv, j % A.nv, Lr, tmem, true, nullptr));
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------ outputs
//
// For the grid of few chains. Per (chunk slot, value head), all chunks in
// parallel: O^T = S_img Q'^T
// (tcgen05 M=128 v, N=64 tokens, K=128) from the state image at the chunk's
// start, + O_local, then the gated RMSNorm (statecache.py, gated_rmsnorm)
// and bf16 rows out through the TMA. Padded tokens of the row get zeros.

constexpr int kOOffS = 0;         // state image (32 KiB)
constexpr int kOOffQ = 32768;     // Q' image [2 kb][64 rows][128 B] (16 KiB)
constexpr int kOOffOT = 49152;    // O_local fp32 [64 tokens][128 v] (32 KiB)
constexpr int kOOffZ = 81920;     // z bf16 [64 tokens][128], overwritten in place by the bf16 output rows
constexpr int kOOffRed = 98304;   // fp32 [4][64] RMS partials, [64] rstd
constexpr int kOOffBar = kOOffRed + 4 * 64 * 4 + 64 * 4;
constexpr int kOutSmem = kOOffBar + 64 + 1024;

// omap: out viewed as [Ttot][nv*dv] bf16, box [32 tokens][128 values];
// zmap: z viewed the same way, box [64 tokens][128 values].
// Q' and O_local come from the grid this one follows, which published each
// chunk unit with a flag: the unit's flag is acquired, then they load before
// the wait for that grid (the state images load after it). That grid triggers
// this launch only after all its units are published, so the flag is set when
// read: the acquire orders memory, it does not wait for a running producer.
__global__ void __launch_bounds__(256, 2) output_kernel(LayerArgs A, Rows R, int Ttot, Ws W,
                                                        const __grid_constant__ CUtensorMap omap,
                                                        const __grid_constant__ CUtensorMap zmap) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  float *red = reinterpret_cast<float *>(sm + kOOffRed);  // [4][64]
  float *rstd = red + 256;                                // [64]
  uint64_t *bar_ld = reinterpret_cast<uint64_t *>(sm + kOOffBar);
  uint64_t *bar_s = bar_ld + 1;
  uint64_t *bar_mma = bar_ld + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_mma + 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x, h = blockIdx.y;
  int r, c;
  slot_row(R, W, s, Ttot, r, c);  // the front kernel completed before the kernel this one follows started
  if (r < 0) return;
  const int start = R.start(r), len = R.len(r), t0 = c * CH;
  if (tid == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const size_t sh = (size_t)s * A.nv + h;
  // Q', O_local (from the chunk pass) and z (from the caller)
  auto issue_qoz = [&]() {
    const unsigned char *wq = reinterpret_cast<const unsigned char *>(W.wq + sh * kWQ);
    mbar_arrive_expect_tx(bar_ld, 16384 + 32768 + 16384);
    bulk_g2s(sm + kOOffQ, wq + 8192, 8192, bar_ld);           // Q' rows, column block 0
    bulk_g2s(sm + kOOffQ + 8192, wq + 24576, 8192, bar_ld);   // Q' rows, column block 1
    bulk_g2s(sm + kOOffOT, W.ot + sh * kRowF, 32768, bar_ld);
    tma_load_2d(sm + kOOffZ, &zmap, h * HD, start + t0, bar_ld);  // rows past the tensor read as zeros
  };
  bool issued = false;  // thread 0: Q', O_local and z were requested (else its flag wait expired)
  if (tid == 0) {
    issued = unit_ready(W.flag + sh, true, A.status, false);
    if (issued) issue_qoz();
  }
  griddep_wait();  // the state pass's images and row lengths are complete
  griddep_trigger();
  const int Lr = W.lr[(size_t)r * A.nv + h];  // < 0: rejected row or stopped chain (its status is set)
  const int ntok = min(CH, len - t0), nreal = Lr < 0 ? 0 : max(0, min(CH, Lr - t0));
  // padded tokens of this chunk: zeros
  if (Lr >= 0)
    for (int e = nreal * 16 + tid; e < ntok * 16; e += 256)
      reinterpret_cast<uint4 *>(A.out + ((size_t)(start + t0 + e / 16) * A.nv + h) * HD)[e % 16] =
          make_uint4(0u, 0u, 0u, 0u);
  if (nreal == 0) {  // nothing to compute: let the loads in flight land, then leave
    (void)cta_wait(bar_ld, 0, A.status, !issued);
    goto done;
  }
  if (tid == 0 && issued) {
    mbar_arrive_expect_tx(bar_s, 32768);
    bulk_g2s(sm + kOOffS, W.simg + sh * kWQ, 32768, bar_s);
  }
  if (!cta_wait(bar_ld, 0, A.status, !issued)) goto done;
  if (!cta_wait(bar_s, 0, A.status)) goto done;
  if (tid == 0) {
    tc_fence_after();
    umma_tile(tmem, smem_u32(sm + kOOffS), 128, smem_u32(sm + kOOffQ), 64, 128, umma_idesc_f16(128, 64), false);
    umma_commit(bar_mma);
  }
  if (!cta_wait(bar_mma, 0, A.status)) goto done;
  tc_fence_after();
  {
    // value row v = TMEM lane, tokens 32hh .. 32hh+31 (warp group hh); the
    // group's 4 warps hold all 128 v of its tokens
    const int q = warp & 3, hh = warp >> 2, v = 32 * q + lane, bar_id = 1 + hh, issuer = 128 * hh;
    float o[32];
    tmem_ld32(tmem_at(tmem, q, 32 * hh), o);
    const float *ol = reinterpret_cast<const float *>(sm + kOOffOT);
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int i = 32 * hh + e;  // element (i, v) sits in chunk (v / 4) ^ (i % 8) of row i
      o[e] += ol[i * HD + ((((v >> 2) ^ (i & 7))) << 2) + (v & 3)];
    }
    // sum over the warp's 32 rows of o^2 for each of the 32 tokens: after the
    // transposing butterfly lane l holds token l's partial
    float sq[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) sq[e] = o[e] * o[e];
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
      const bool up = (lane & w) != 0;
#pragma unroll
      for (int e = 0; e < w; ++e) {
        const float send = up ? sq[e] : sq[e + w];
        const float keep = up ? sq[e + w] : sq[e];
        sq[e] = keep + __shfl_xor_sync(0xffffffffu, send, w);
      }
    }
    red[q * 64 + 32 * hh + lane] = sq[0];
    named_sync(bar_id, 128);
    if (q == 0) {
      const int t = 32 * hh + lane;
      const float ss = red[t] + red[64 + t] + red[128 + t] + red[192 + t];
      rstd[t] = rsqrtf(ss / (float)HD + A.rms_eps);
    }
    named_sync(bar_id, 128);
    bf16 *os = reinterpret_cast<bf16 *>(sm + kOOffZ);  // each z is read, then overwritten, by one thread
    const float wv = ldbf(A.norm_w + v);
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int i = 32 * hh + e;
      const float gz = wv * silu_approx(__bfloat162float(os[i * HD + v]));
      os[i * HD + v] = __float2bfloat16_rn(o[e] * rstd[i] * gz);
    }
    fence_proxy_async_smem();
    named_sync(bar_id, 128);
    if (tid == issuer) {
      const int nout = min(32, nreal - 32 * hh);  // real tokens of this half
      if (nout == 32) {
        tma_store_2d(&omap, h * HD, start + t0 + 32 * hh, os + 32 * hh * HD);
      } else {
        bf16 *dst = A.out + ((size_t)(start + t0 + 32 * hh) * A.nv + h) * HD;
        for (int i = 0; i < nout; ++i) bulk_s2g(dst + (size_t)i * A.nv * HD, os + (32 * hh + i) * HD, HD * 2);
      }
      bulk_commit();
      bulk_wait_read_all();
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

// Tensor map of a bf16 [rows][cols] row-major tensor with [box_rows][128] boxes.
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

gdn_status encode_rows_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows) {
  // the driver entry point, looked up once (thread-safe static initialisation)
  static const EncodeTiled encode = []() -> EncodeTiled {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiled>(fn);
  }();
  if (!encode) return fail(GDN_ERR_CUDA, "prefill: cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)HD, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return fail(GDN_ERR_CUDA, "prefill: cannot encode a tensor map");
  return GDN_OK;
}

}  // namespace tc

size_t prefill_tc_workspace_bytes(int B, int T, int nk, int nv, bool packed) {
  return tc::ws_bytes(B, T, nk, nv, packed);
}

gdn_status launch_prefill_tc(const LayerArgs &A, void *ws, cudaStream_t stream) {
  const bool packed = A.cu_seqlens != nullptr;
  const int Ttot = packed ? A.T : A.B * A.T;
  const int S = (int)tc::slots_total(A.B, A.T, packed);
  tc::Rows R{A.B, A.T, packed ? 0 : (A.T + tc::CH - 1) / tc::CH, A.cu_seqlens};
  tc::Ws W = tc::carve(ws, A.B, A.T, A.nk, A.nv, packed);
  const DeviceInfo &dev = device_info();
  // set once per device; concurrent first calls may both set it (idempotent)
  static std::atomic<bool> attr_set[kMaxDevices];
  if (!attr_set[dev.id].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(tc::chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kChunkSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(tc::state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kStateSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(tc::output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kOutSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(tc::chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tc::kMergedSmem) != cudaSuccess)
      return fail(GDN_ERR_CUDA, "prefill: cannot reserve shared memory");
    attr_set[dev.id].store(true, std::memory_order_release);
  }
  // Few chains (dense rows, at most half a grid of one CTA per SM): chunk units
  // and chains in one grid, so that the chains start while late chunks are
  // still being prepared; the chains are that grid's critical path and the
  // units form their own gates. Otherwise two kernels, and the front kernel
  // forms the gates (the chunk pass is the critical path there). Every kernel
  // starts early (programmatic dependent launch) and waits for its
  // predecessor inside the kernel.
  const int n_units = S * A.nv, grid = n_units < dev.sms ? n_units : dev.sms;
  const bool merged = !packed && 2 * A.B * A.nv <= grid;
  if (launch_pdl(merged ? tc::front_kernel<false> : tc::front_kernel<true>, dim3(S, 2 * A.nk + A.nv), dim3(256), 0,
                 stream, A, R, Ttot, W) != cudaSuccess)
    return check_launch("prefill front");
  if (merged) {
    CUtensorMap omap, zmap;
    if (gdn_status st = tc::encode_rows_map(&omap, A.out, Ttot, A.nv * tc::HD, tc::CH / 2)) return st;
    if (gdn_status st = tc::encode_rows_map(&zmap, A.z, Ttot, A.nv * tc::HD, tc::CH)) return st;
    if (launch_pdl(tc::chunk_state_kernel, dim3(grid), dim3(256), tc::kMergedSmem, stream, A, R, Ttot, W) !=
        cudaSuccess)
      return check_launch("prefill chunk+state");
    if (launch_pdl(tc::output_kernel, dim3(S, A.nv), dim3(256), tc::kOutSmem, stream, A, R, Ttot, W, omap, zmap) !=
        cudaSuccess)
      return check_launch("prefill output");
    return check_launch("prefill output");
  }
  if (launch_pdl(tc::chunk_kernel, dim3(grid), dim3(256), tc::kChunkSmem, stream, A, R, Ttot, W, n_units) !=
      cudaSuccess)
    return check_launch("prefill chunk");
  CUtensorMap zmap;
  if (gdn_status st = tc::encode_rows_map(&zmap, A.z, Ttot, A.nv * tc::HD, tc::CH)) return st;
  if (launch_pdl(tc::state_kernel, dim3(A.B * A.nv), dim3(256), tc::kStateSmem, stream, A, R, Ttot, W, zmap) !=
      cudaSuccess)
    return check_launch("prefill state");
  return check_launch("prefill state");
}

}  // namespace gdn
