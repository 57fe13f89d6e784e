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
//     engine) completing on a "full" mbarrier; the 8 compute warps write the
//     updated state back into the same stage and arrive on its "empty"
//     mbarrier; a dedicated producer warp then bulk-stores the stage to the
//     state slot and, once that copy has read it, refills the stage, so NS-1
//     heads are in flight while one is computed and the compute warps never
//     issue the 64 KiB of global stores themselves; the compute warps
//     synchronise among themselves only (barrier 1), never with the producer;
//   * the small per-unit inputs (token channels, conv tail, conv taps, z,
//     gates) are loaded into registers one unit ahead, so their latency hides
//     behind the current unit's state stream; row slots are resolved once
//     into a shared table.
// The per-token arithmetic is the shared code of gdn_token.cuh.

#include "gdn_launch.h"
#include "gdn_token.cuh"

namespace gdn {

constexpr int kMaxG = 8;
constexpr int kPre = 3;        // channels per thread prefetched one unit ahead
constexpr int kZPre = 4;       // z values per thread prefetched one unit ahead
constexpr int kSlotTable = 64; // units per CTA whose slots are tabulated

template <int D, int NS>
struct DecodeSmem {
  static constexpr int kStage = D * D;                          // floats per stage
  static constexpr int kRed = StepScratch<D>::kFloats;
  static constexpr int kFront = (2 + kMaxG) * D + kMaxG * D + D + 4 * kMaxG;  // q,k,v[G], z[G], norm_w, gates
  static constexpr size_t kBytes =
      sizeof(float) * (size_t)(NS * kStage + kRed + kFront) + sizeof(int) * kSlotTable + 16 * NS;
};

// One unit's raw inputs, loaded a unit ahead of their use.
struct FrontRegs {
  uint2 w[kPre];                    // 4 conv taps (bf16) per channel
  bf16 x[kPre], t0[kPre], t1[kPre], t2[kPre];
  bf16 z[kZPre];
  // MXFP8 inputs: the raw element and scale bytes, dequantized only where they
  // are used (converting at load time would wait for the loads a unit early)
  uint8_t xe[kPre], xs[kPre], ze[kZPre], zs[kZPre];
  bf16 ga, gb;
  float alog, dtb;
};

struct UnitGeom {
  int D, G, kd, nv, C;
  // channel (global index) and token source of unit-local channel e
  __device__ __forceinline__ int chan(int e, int kh) const {
    return e < D ? kh * D + e : (e < 2 * D ? kd + kh * D + (e - D) : 2 * kd + kh * G * D + (e - 2 * D));
  }
  __device__ __forceinline__ const bf16 *src(const LayerArgs &A, int b, int ch) const {
    return ch < kd ? A.q + (size_t)b * kd + ch
                   : (ch < 2 * kd ? A.k + (size_t)b * kd + (ch - kd) : A.v + (size_t)b * nv * D + (ch - 2 * kd));
  }
};

// One MXFP8 element: e4m3 times its block's scale
// 2^(s-127) (s = 0: 2^-127; s = 255: NaN, the format's NaN code). The product
// is exact in fp32 and, inside bf16's normal range, in bf16, so the conv and
// the saved conv tail see exactly the dequantized input.
// e4m3 (OCP FP8): sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0
// holds the subnormals m * 2^-9; S.1111.111 is NaN (no infinities). Decoded
// exactly into fp32 with integer operations.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t sgn = (b & 0x80u) << 24, ex = (b >> 3) & 15u, m = b & 7u;
  float v;
  if ((b & 0x7Fu) == 0x7Fu) v = __int_as_float(0x7fc00000);
  else if (ex == 0u) v = (float)m * 0.001953125f;  // m * 2^-9, exact
  else v = __uint_as_float(((ex + 120u) << 23) | (m << 20));
  return __uint_as_float(__float_as_uint(v) | sgn);
}

__device__ __forceinline__ bf16 mx_dequant(uint8_t e, uint8_t s) {
  const float f = e4m3_to_f32(e);
  const float scale = s == 255 ? __int_as_float(0x7fc00000) : (s == 0 ? __int_as_float(0x00400000)
                                                                       : __int_as_float((int)s << 23));
  return __float2bfloat16_rn(f * scale);
}

// Addresses of the MXFP8 element and scale of token channel ch of row b.
__device__ __forceinline__ void mx_x_at(const LayerArgs &A, const UnitGeom &U, int b, int ch, const uint8_t *&e,
                                        const uint8_t *&sc) {
  const int kd = U.kd, vd = U.nv * U.D;
  if (ch < kd) {
    e = A.mx.q + (size_t)b * kd + ch;
    sc = A.mx.qs + (size_t)b * (kd / 32) + ch / 32;
  } else if (ch < 2 * kd) {
    const int c = ch - kd;
    e = A.mx.k + (size_t)b * kd + c;
    sc = A.mx.ks + (size_t)b * (kd / 32) + c / 32;
  } else {
    const int c = ch - 2 * kd;
    e = A.mx.v + (size_t)b * vd + c;
    sc = A.mx.vs + (size_t)b * (vd / 32) + c / 32;
  }
}
// ... and of z value e of the G value heads of key head kh, row b.
__device__ __forceinline__ void mx_z_at(const LayerArgs &A, const UnitGeom &U, int b, int kh, int e,
                                        const uint8_t *&el, const uint8_t *&sc) {
  const int vd = U.nv * U.D, c = kh * U.G * U.D + e;
  el = A.mx.z + (size_t)b * vd + c;
  sc = A.mx.zs + (size_t)b * (vd / 32) + c / 32;
}

// Token channel ch of row b (one decode token per row): the bf16 input, or the
// dequantized MXFP8 one.
template <bool MX>
__device__ __forceinline__ bf16 load_x(const LayerArgs &A, const UnitGeom &U, int b, int ch) {
  if (!MX) return *U.src(A, b, ch);
  const uint8_t *e, *sc;
  mx_x_at(A, U, b, ch, e, sc);
  return mx_dequant(*e, *sc);
}

// z value e of the G value heads of key head kh, row b.
template <bool MX>
__device__ __forceinline__ bf16 load_z(const LayerArgs &A, const UnitGeom &U, int b, int kh, int e) {
  if (!MX) return A.z[((size_t)b * A.nv + kh * U.G) * U.D + e];
  const uint8_t *el, *sc;
  mx_z_at(A, U, b, kh, e, el, sc);
  return mx_dequant(*el, *sc);
}

template <bool MX>
__device__ __forceinline__ void load_front(FrontRegs &R, const LayerArgs &A, const UnitGeom &U, int b, int kh,
                                           int slot, int tid) {
  const int nch = (2 + U.G) * U.D;
  const bf16 *cs = A.conv_state + (size_t)slot * KC * U.C;
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int e = tid + 256 * i;
    if (e < nch) {
      const int ch = U.chan(e, kh);
      if (MX) {
        const uint8_t *e8, *s8;
        mx_x_at(A, U, b, ch, e8, s8);
        R.xe[i] = *e8;
        R.xs[i] = *s8;
      } else {
        R.x[i] = *U.src(A, b, ch);
      }
      R.t0[i] = cs[ch];
      R.t1[i] = cs[U.C + ch];
      R.t2[i] = cs[2 * U.C + ch];
      R.w[i] = *reinterpret_cast<const uint2 *>(A.conv_w + (size_t)ch * 4);
    }
  }
#pragma unroll
  for (int i = 0; i < kZPre; ++i) {
    const int e = tid + 256 * i;
    if (e < U.G * U.D) {
      if (MX) {
        const uint8_t *e8, *s8;
        mx_z_at(A, U, b, kh, e, e8, s8);
        R.ze[i] = *e8;
        R.zs[i] = *s8;
      } else {
        R.z[i] = A.z[((size_t)b * A.nv + kh * U.G) * U.D + e];
      }
    }
  }
  if (tid < U.G) {
    const int hh = kh * U.G + tid;
    R.ga = A.a[(size_t)b * A.nv + hh];
    R.gb = A.b[(size_t)b * A.nv + hh];
    R.alog = A.A_log[hh];
    R.dtb = A.dt_bias[hh];
  }
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Barrier 1 over the compute threads with an OR reduction of `pred`.
__device__ __forceinline__ bool compute_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// MX: the token channels q / k / v / z arrive as MXFP8 (A.mx) instead of bf16.
template <int D, int NS, bool MX>
__global__ void __launch_bounds__(288, 1) decode_kernel(LayerArgs A) {
  using L = StateLayout<D>;
  using S = DecodeSmem<D, NS>;
  extern __shared__ __align__(128) float smem[];
  float *stage = smem;
  float *red = stage + NS * S::kStage;
  float *fq = red + S::kRed;
  float *fk = fq + D;
  float *fv = fk + D;                  // [G][D]
  float *fz = fv + kMaxG * D;          // [G][D]
  float *fw = fz + kMaxG * D;          // [D] norm weight
  float *fdecay = fw + D;              // [G]
  float *fbeta = fdecay + kMaxG;       // [G]
  float *fbkq = fbeta + kMaxG;         // [G]
  int *slot_tab = reinterpret_cast<int *>(fbkq + 2 * kMaxG);
  uint64_t *full = reinterpret_cast<uint64_t *>(slot_tab + kSlotTable);
  uint64_t *empty = full + NS;
  const SyncCompute csync;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = A.G;
  const UnitGeom U{D, G, A.nk * D, A.nv, A.C};
  const int n_units = A.B * A.nk;
  if ((int)blockIdx.x >= n_units) return;
  const int my_units = (n_units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int n_tasks = my_units * G;
  const int nch = (2 + G) * D;

  // Slot of unit i's row, or -1 (mask 0 = skip; a bad mask value or slot is recorded).
  auto resolve = [&](int i, bool record) -> int {
    const int b = ((int)blockIdx.x + i * (int)gridDim.x) / A.nk;
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
  auto unit_slot = [&](int i) -> int { return i < kSlotTable ? slot_tab[i] : resolve(i, false); };
  auto issue = [&](int n) {  // producer lane only
    const int i = n / G;
    const int u = (int)blockIdx.x + i * (int)gridDim.x;
    const int h = (u % A.nk) * G + n % G;
    const int slot = unit_slot(i);
    uint64_t *bar = &full[n % NS];
    if (slot >= 0) {
      mbar_arrive_expect_tx(bar, D * D * 4);
      bulk_g2s(stage + (n % NS) * S::kStage, A.state + ((size_t)slot * A.nv + h) * D * D, D * D * 4, bar);
    } else {
      mbar_arrive(bar);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);  // one arrival per compute warp
    }
    fence_mbar_init();
  }
  // Before the wait: the first NS tasks' states are requested into L2. The
  // slot index read here is only a hint; the loads after the wait use the one
  // read then.
  for (int n = 0; n < NS && n < n_tasks; ++n) {
    const int u = (int)blockIdx.x + (n / G) * (int)gridDim.x, b = u / A.nk, h = (u % A.nk) * G + n % G;
    const int s = A.state_idx ? __ldcg(A.state_idx + b) : b;
    if (s >= 0 && s < A.n_slots) {
      const char *p = reinterpret_cast<const char *>(A.state + ((size_t)s * A.nv + h) * D * D);
      for (int off = 128 * tid; off < D * D * 4; off += 128 * (int)blockDim.x)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off));
    }
  }
  griddep_wait();  // the kernel before this call (e.g. the previous layer's) is complete
  griddep_trigger();
  for (int i = tid; i < my_units && i < kSlotTable; i += blockDim.x) slot_tab[i] = resolve(i, true);
  for (int i = kSlotTable + tid; i < my_units; i += blockDim.x) (void)resolve(i, true);
  for (int c = tid; c < D; c += blockDim.x) fw[c] = ldbf(A.norm_w + c);
  __syncthreads();

  if (warp == 8) {
    // ---- producer: stream every task's state into the stage ring
    if (lane == 0) {
      // task m's updated state is back in its stage: bulk-store it to the slot
      auto store_back = [&](int m) -> bool {
        if (!mbar_wait_bounded(&empty[m % NS], (uint32_t)((m / NS) & 1))) return false;
        const int u = (int)blockIdx.x + (m / G) * (int)gridDim.x;
        const int h = (u % A.nk) * G + m % G;
        const int slot = unit_slot(m / G);
        if (slot >= 0) {
          bulk_s2g(A.state + ((size_t)slot * A.nv + h) * D * D, stage + (m % NS) * S::kStage, D * D * 4);
          bulk_commit();
        }
        return true;
      };
      bool ok = true;
      for (int n = 0; n < n_tasks && ok; ++n) {
        if (n >= NS) {
          ok = store_back(n - NS);
          bulk_wait_read_all();  // the stage may be refilled
        }
        if (ok) issue(n);
      }
      for (int m = n_tasks - NS < 0 ? 0 : n_tasks - NS; m < n_tasks && ok; ++m) ok = store_back(m);
      if (!ok) set_status(A.status, GDN_ERR_TIMEOUT);
      bulk_wait_read_all();  // shared memory stays valid until every store has read it
    }
    return;
  }

  FrontRegs R;
  {
    const int s0 = unit_slot(0);
    const int u0 = (int)blockIdx.x;
    if (s0 >= 0) load_front<MX>(R, A, U, u0 / A.nk, u0 % A.nk, s0, tid);
  }

  for (int n = 0; n < n_tasks; ++n) {
    const int i = n / G, j = n % G;
    const int u = (int)blockIdx.x + i * (int)gridDim.x;
    const int b = u / A.nk, kh = u % A.nk, h = kh * G + j;
    const int slot = unit_slot(i);

    if (j == 0 && slot >= 0) {
      // ---- unit front end from the prefetched registers
      csync();  // the previous unit is done with fq / fk / fv / fz / gates
      bf16 *cs = A.conv_state + (size_t)slot * KC * A.C;
#pragma unroll
      for (int p = 0; p < kPre; ++p) {
        const int e = tid + 256 * p;
        if (e < nch) {
          const int ch = U.chan(e, kh);
          const bf16 xv = MX ? mx_dequant(R.xe[p], R.xs[p]) : R.x[p];
          fq[e] = conv4_silu(bf_lo(R.w[p].x), bf_hi(R.w[p].x), bf_lo(R.w[p].y), bf_hi(R.w[p].y),
                             __bfloat162float(R.t0[p]), __bfloat162float(R.t1[p]), __bfloat162float(R.t2[p]),
                             __bfloat162float(xv));
          cs[ch] = R.t1[p];
          cs[A.C + ch] = R.t2[p];
          cs[2 * A.C + ch] = xv;
        }
      }
      for (int e = tid + 256 * kPre; e < nch; e += 256) {  // groups wider than the prefetch
        const int ch = U.chan(e, kh);
        const bf16 x0 = cs[ch], x1 = cs[A.C + ch], x2 = cs[2 * A.C + ch], x3 = load_x<MX>(A, U, b, ch);
        const bf16 *w = A.conv_w + (size_t)ch * 4;
        fq[e] = conv4_silu(ldbf(w), ldbf(w + 1), ldbf(w + 2), ldbf(w + 3), __bfloat162float(x0),
                           __bfloat162float(x1), __bfloat162float(x2), __bfloat162float(x3));
        cs[ch] = x1;
        cs[A.C + ch] = x2;
        cs[2 * A.C + ch] = x3;
      }
#pragma unroll
      for (int p = 0; p < kZPre; ++p) {
        const int e = tid + 256 * p;
        if (e < G * D) fz[e] = __bfloat162float(MX ? mx_dequant(R.ze[p], R.zs[p]) : R.z[p]);
      }
      for (int e = tid + 256 * kZPre; e < G * D; e += 256)
        fz[e] = __bfloat162float(load_z<MX>(A, U, b, kh, e));
      float decay = 0.f, beta = 0.f;
      if (tid < G) gdn_gates(__bfloat162float(R.ga), __bfloat162float(R.gb), R.alog, R.dtb, decay, beta);
      csync();
      if (warp == 0) warp_l2norm<D>(fq, A.l2_eps, A.scale, lane);
      if (warp == 1) warp_l2norm<D>(fk, A.l2_eps, 1.0f, lane);
      csync();
      if (warp == 0) {
        const float kq = warp_dot<D>(fq, fk, lane);
        if (lane < G) {
          fdecay[lane] = decay;
          fbeta[lane] = beta;
          fbkq[lane] = __fmul_rn(beta, kq);
        }
      }
      csync();
      // next unit's inputs, in flight while this unit's heads stream: issued
      // after this unit's front end, whose shared-memory work would otherwise
      // queue behind the global loads and wait out their latency
      if (i + 1 < my_units) {
        const int s1 = unit_slot(i + 1);
        const int u1 = u + (int)gridDim.x;
        if (s1 >= 0) load_front<MX>(R, A, U, u1 / A.nk, u1 % A.nk, s1, tid);
      }
    } else if (j == 0 && i + 1 < my_units) {
      // skipped unit: still prefetch the next one
      const int s1 = unit_slot(i + 1);
      const int u1 = u + (int)gridDim.x;
      if (s1 >= 0) load_front<MX>(R, A, U, u1 / A.nk, u1 % A.nk, s1, tid);
    }

    // ---- the value head's state
    const bool ok = mbar_wait_leader(&full[n % NS], (uint32_t)((n / NS) & 1), tid == 0, compute_sync_or);
    if (!ok) {
      if (tid == 0) set_status(A.status, GDN_ERR_TIMEOUT);
      // let copies already in flight land before the CTA's memory is released
      if (tid < NS && n + tid < n_tasks) (void)mbar_wait_bounded(&full[(n + tid) % NS], (uint32_t)(((n + tid) / NS) & 1));
      return;
    }
    bf16 *out = A.out + ((size_t)b * A.nv + h) * D;
    if (slot >= 0) {
      const int cq = tid % L::TPR, grp = tid / L::TPR;
      const float4 *st = reinterpret_cast<const float4 *>(stage + (n % NS) * S::kStage);
      float4 s[L::RPT];
#pragma unroll
      for (int r = 0; r < L::RPT; ++r) s[r] = st[(grp + r * L::NG) * L::TPR + cq];
      float4 o;
      state_step<D>(s, fq, fk, fv + j * D, fdecay[j], fbeta[j], fbkq[j], red, tid, o, csync);
      // the updated slice back into the stage; the producer stores the stage
      float4 *sw = reinterpret_cast<float4 *>(stage + (n % NS) * S::kStage);
#pragma unroll
      for (int r = 0; r < L::RPT; ++r) sw[(grp + r * L::NG) * L::TPR + cq] = s[r];
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[n % NS]);
      if (warp == 7) rmsnorm_store_smem<D>(o, lane, fz + j * D, fw, A.rms_eps, out);
    } else {
      if (lane == 0) mbar_arrive(&empty[n % NS]);
      zero_head<D>(out, tid);
    }
  }
}

template <int D, int NS, bool MX>
static gdn_status launch_decode_t(const LayerArgs &A, cudaStream_t stream) {
  using S = DecodeSmem<D, NS>;
  const DeviceInfo &dev = device_info();
  // set once per device; concurrent first calls may both set it (idempotent)
  static std::atomic<bool> attr_set[kMaxDevices];
  if (!attr_set[dev.id].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(decode_kernel<D, NS, MX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::kBytes) !=
        cudaSuccess)
      return fail(GDN_ERR_CUDA, "decode: cannot reserve shared memory");
    attr_set[dev.id].store(true, std::memory_order_release);
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<D, NS, MX>, 288, S::kBytes) != cudaSuccess ||
      per_sm < 1)
    return fail(GDN_ERR_CUDA, "decode: kernel does not fit on an SM");
  const int n_units = A.B * A.nk;
  const int grid = n_units < dev.sms * per_sm ? n_units : dev.sms * per_sm;
  if (launch_pdl(decode_kernel<D, NS, MX>, dim3(grid), dim3(288), S::kBytes, stream, A) != cudaSuccess)
    return check_launch("decode");
  return check_launch("decode");
}

gdn_status launch_decode(const LayerArgs &A, cudaStream_t stream) {
  const bool mx = A.mx.q != nullptr;
  switch (A.D) {
    case 128: return mx ? launch_decode_t<128, 3, true>(A, stream) : launch_decode_t<128, 3, false>(A, stream);
    case 64: return mx ? launch_decode_t<64, 4, true>(A, stream) : launch_decode_t<64, 4, false>(A, stream);
    case 32: return mx ? launch_decode_t<32, 4, true>(A, stream) : launch_decode_t<32, 4, false>(A, stream);
  }
  return fail(GDN_ERR_SHAPE, "decode: unsupported head size");
}

}  // namespace gdn
