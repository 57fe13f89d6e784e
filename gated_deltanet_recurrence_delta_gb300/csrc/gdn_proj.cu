// The layer's projections on the tcgen05 tensor cores: the in-projection whose
// output is split, in the epilogue, straight into the q | k | v, z, b and a
// tensors the layer's calls read, and the out-projection after the gated
// RMSNorm.
//
// statecache.py (squad-0.8b, qev_fast), CacheQwen35._gdn: the hidden state goes
// through in_proj, whose output is split into the mixed q|k|v channels (the
// conv's input), z, b and a, in that order; the gated RMSNorm's output goes
// through the out-projection.
//
// One GEMM kernel, Y = X W^T with bf16 operands and fp32 accumulation, computed
// as Y^T = W X^T: the weight rows (output features) are the MMA's M = 128 rows
// in TMEM lanes and the tokens its N columns, so a decode step's 64 tokens fill
// one N tile and the 128-row weight tiles stream once. Per CTA one 128 x BN
// tile: a producer thread loads K-slices of 64 (one 128-byte swizzled row per
// operand row) with the TMA into a ring of STAGES stages; one thread issues
// the MMAs (kind::f16, bf16) and releases each stage when its products have
// read it; then all four warps read the accumulator from TMEM (a warp's lane
// quarter = 32 features) and write bf16 rows: for each token, a warp's 32
// consecutive features. Every wait is bounded.
#include <mutex>

#include "gdn_launch.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace proj {

constexpr int BM = 128;     // output features per tile (TMEM lanes)
constexpr int kGroupF = 16;  // feature tiles per group of the grouped tile order
constexpr int BK = 64;      // K elements per stage: one 128-byte swizzled row per operand row
// Stages of the K ring: decode-sized calls stream their weights and want many
// bytes in flight per SM; prefill-sized ones keep two CTAs per SM (each one's
// epilogue then runs under the other's products).
template <int BN>
struct Stages {
  static constexpr int value = BN <= 64 ? 8 : (BN == 128 ? 3 : 2);
};

// Output features [n0, n1) go to dst[token * ld + (feature - n0)].
struct Seg {
  int n0, n1;
  bf16 *dst;
  long long ld;
};
struct Epi {
  int nseg;
  Seg seg[6];
};

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <int BN>
struct Smem {
  static constexpr int STAGES = Stages<BN>::value;
  static constexpr int kA = BM * 128;                // bytes of one stage's weight tile
  static constexpr int kB = BN * 128;                // bytes of one stage's token tile
  static constexpr int kStage = kA + kB;
  static constexpr int kBar = STAGES * kStage;       // full[STAGES], empty[STAGES], done, tmem base
  static constexpr int kBytes = kBar + 8 * (2 * STAGES + 1) + 16 + 1024;  // + alignment slack
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The copy of shared address `p` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const float *p, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  return remote;
}
// A load from another CTA's shared memory. No memory clobber: the loads of a
// group issue back to back (the cluster barrier before them orders them after
// the partners' stores).
__device__ __forceinline__ float ld_cluster_f32(uint32_t remote) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote));
  return v;
}

// SPLIT > 1: a cluster of SPLIT CTAs shares one output tile, each taking an
// equal share of the K-slices; the partial tiles meet in distributed shared
// memory (each CTA parks its tile in its own stage ring, free by then, and
// CTA r sums every CTA's columns [r BN/SPLIT, (r+1) BN/SPLIT) and writes them).
// For calls with too few output tiles to occupy the GPU.
// GROUPED (SPLIT 1, weights far larger than a share of L2): the tiles are
// visited in groups of kGroupF feature tiles by all token tiles.
template <int BN, int SPLIT, bool GROUPED>
__global__ void __launch_bounds__(128, 1) gemm_kernel(const __grid_constant__ CUtensorMap wmap,
                                                      const __grid_constant__ CUtensorMap xmap, int Nout, int M,
                                                      int K, Epi epi, unsigned int *status) {
  using S = Smem<BN>;
  constexpr int STAGES = S::STAGES;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  unsigned char *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + S::kBar);
  uint64_t *empty = full + STAGES;
  uint64_t *done = empty + STAGES;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = SPLIT > 1 ? cluster_rank() : 0u;
  int fb = blockIdx.x / SPLIT, tb = blockIdx.y;  // feature tile, token tile
  if (GROUPED) {
    // consecutive CTAs take kGroupF feature tiles by all token tiles, feature
    // tile fastest, so the CTAs resident at one time share their weight and
    // token tiles in L2 (in row-major order the 101 MB in-projection weights
    // streamed from DRAM once per ~3 token tiles)
    const int nf = (int)gridDim.x, nt = (int)gridDim.y;
    const int pid = (int)blockIdx.y * nf + (int)blockIdx.x, per_group = kGroupF * nt;
    const int g = pid / per_group, f_first = g * kGroupF, gsize = min(nf - f_first, kGroupF);
    const int r = pid - g * per_group;
    fb = f_first + r % gsize;
    tb = r / gsize;
  }
  const int f0 = fb * BM, t0 = tb * BN;
  const int nkt = K / BK, kb0 = (int)(nkt * (long long)rank / SPLIT), kb1 = (int)(nkt * (long long)(rank + 1) / SPLIT);
  const int nk = kb1 - kb0;  // this CTA's K-slices: kb0 + 0 .. kb0 + nk - 1
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(tmem_slot, BN < 32 ? 32 : BN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // the kernel before this call (which may have written X) is complete
  griddep_trigger();

  if (tid == 0) {
    // ---- producer: K-slices into the stage ring
    int issued = 0;
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % STAGES;
      if (kb >= STAGES && !mbar_wait_bounded(&empty[st], (uint32_t)(((kb / STAGES) - 1) & 1))) {
        set_status(status, GDN_ERR_TIMEOUT);
        atomicExch(&s_abort, 1);
        break;
      }
      unsigned char *a = sm + st * S::kStage;
      mbar_arrive_expect_tx(&full[st], S::kStage);
      tma_load_2d(a, &wmap, (kb0 + kb) * BK, f0, &full[st]);          // rows past Nout read as zeros
      tma_load_2d(a + S::kA, &xmap, (kb0 + kb) * BK, t0, &full[st]);  // tokens past M read as zeros
      issued = kb + 1;
    }
    // the copies this thread issued have landed before the CTA's memory is released
    for (int kb = issued - STAGES < 0 ? 0 : issued - STAGES; kb < issued; ++kb)
      (void)mbar_wait_bounded(&full[kb % STAGES], (uint32_t)((kb / STAGES) & 1));
  } else if (tid == 32) {
    // ---- MMA issuer
    const uint32_t idesc = idesc_bf16(BM, BN);
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % STAGES;
      if (!mbar_wait_bounded(&full[st], (uint32_t)((kb / STAGES) & 1))) {
        set_status(status, GDN_ERR_TIMEOUT);
        atomicExch(&s_abort, 1);
        break;
      }
      tc_fence_after();
      const uint32_t a = smem_u32(sm + st * S::kStage), b = a + S::kA;
#pragma unroll
      for (int ks = 0; ks < BK / 16; ++ks)
        umma_f16(tmem, umma_desc(a + ks * 32), umma_desc(b + ks * 32), idesc, kb > 0 || ks > 0);
      umma_commit(&empty[st]);  // the stage is free once these products have read it
    }
    umma_commit(done);  // every product issued so far is complete
  }
  // ---- epilogue: lane quarter `warp` = features f0 + 32 warp + lane. Thread 0
  // polls the product barrier, the rest wait in the CTA barrier.
  const bool ok = mbar_wait_leader(done, 0u, tid == 0, [](bool p) { return __syncthreads_or(p) != 0; });
  if (!ok && tid == 0) set_status(status, GDN_ERR_TIMEOUT);
  tc_fence_after();
  if (SPLIT > 1) {
    // every CTA parks its partial tile [token][feature] (feature-contiguous: a
    // warp's accesses to one token column are one 128-byte line, locally and
    // across the cluster) in its own stage ring
    float *part = reinterpret_cast<float *>(sm);
    const int row = 32 * warp + lane;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float v[32];
      tmem_ld32(tmem_at(tmem, warp, 32 * c), v);
#pragma unroll
      for (int e = 0; e < 32; ++e) part[(32 * c + e) * BM + row] = (ok && !s_abort) ? v[e] : 0.0f;
    }
    cluster_sync_all();  // every CTA's partial tile is in place
    const int f = f0 + row;
    bf16 *dst = nullptr;
    long long ld = 0;
    if (f < Nout)
      for (int i = 0; i < epi.nseg; ++i)
        if (f >= epi.seg[i].n0 && f < epi.seg[i].n1) {
          dst = epi.seg[i].dst + (f - epi.seg[i].n0);
          ld = epi.seg[i].ld;
        }
    constexpr int CW = BN / SPLIT;  // token columns this CTA writes
    if (dst && ok && !s_abort) {
      uint32_t base[SPLIT];
#pragma unroll
      for (int p = 0; p < SPLIT; ++p) base[p] = cluster_addr(part + (int)rank * CW * BM + row, (uint32_t)p);
      constexpr int G = 8;  // columns whose SPLIT loads are in flight together
      static_assert(CW % G == 0, "column groups");
#pragma unroll 1
      for (int c0 = 0; c0 < CW; c0 += G) {
        float v[G][SPLIT];
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
          for (int p = 0; p < SPLIT; ++p) v[j][p] = ld_cluster_f32(base[p] + 4u * (uint32_t)((c0 + j) * BM));
#pragma unroll
        for (int j = 0; j < G; ++j) {
          float acc = 0.0f;
#pragma unroll
          for (int p = 0; p < SPLIT; ++p) acc += v[j][p];
          const int t = t0 + (int)rank * CW + c0 + j;
          if (t < M) dst[(long long)t * ld] = __float2bfloat16_rn(acc);
        }
      }
    }
    cluster_sync_all();  // no CTA leaves while another reads its shared memory
  } else if (ok && !s_abort) {
    const int f = f0 + 32 * warp + lane;
    bf16 *dst = nullptr;
    long long ld = 0;
    if (f < Nout)
      for (int i = 0; i < epi.nseg; ++i)
        if (f >= epi.seg[i].n0 && f < epi.seg[i].n1) {
          dst = epi.seg[i].dst + (f - epi.seg[i].n0);
          ld = epi.seg[i].ld;
        }
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float v[32];
      tmem_ld32(tmem_at(tmem, warp, 32 * c), v);
      if (dst) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int t = t0 + 32 * c + e;
          if (t < M) dst[(long long)t * ld] = __float2bfloat16_rn(v[e]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, BN < 32 ? 32 : BN);
}

// A bf16 [rows][cols] row-major tensor map with [box_rows][64] boxes and the
// 128-byte swizzle (the K-major operand layout of the MMA).
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

gdn_status encode_operand(CUtensorMap *map, const void *base, long long rows, long long cols, int box_rows) {
  static const EncodeTiled encode = []() -> EncodeTiled {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiled>(fn);
  }();
  if (!encode) return fail(GDN_ERR_CUDA, "projection: cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return fail(GDN_ERR_CUDA, "projection: cannot encode a tensor map");
  return GDN_OK;
}

template <int BN, int SPLIT, bool GROUPED = false>
gdn_status launch_t(const void *w, const void *x, int Nout, int M, int K, const Epi &epi, cudaStream_t stream) {
  static_assert(SPLIT == 1 || BN * BM * 4 <= Smem<BN>::kBar, "the partial tile fits in the stage ring");
  static_assert(!GROUPED || SPLIT == 1, "grouped order for unsplit tiles");
  const DeviceInfo &dev = device_info();
  static std::atomic<bool> attr_set[kMaxDevices];
  if (!attr_set[dev.id].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(gemm_kernel<BN, SPLIT, GROUPED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<BN>::kBytes) != cudaSuccess)
      return fail(GDN_ERR_CUDA, "projection: cannot reserve shared memory");
    attr_set[dev.id].store(true, std::memory_order_release);
  }
  CUtensorMap wmap, xmap;
  if (gdn_status st = encode_operand(&wmap, w, Nout, K, BM)) return st;
  if (gdn_status st = encode_operand(&xmap, x, M, K, BN)) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(SPLIT * ((Nout + BM - 1) / BM), (M + BN - 1) / BN);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = Smem<BN>::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = SPLIT;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, gemm_kernel<BN, SPLIT, GROUPED>, wmap, xmap, Nout, M, K, epi, dev.status) != cudaSuccess)
    return check_launch("projection");
  return check_launch("projection");
}

// Token tile: 64 for decode-sized calls (one tile), 128 up to 128 tokens, 256
// beyond. Calls with too few output tiles for the GPU split K over a cluster
// (2 or 4 CTAs).
gdn_status launch(const void *w, const void *x, int Nout, int M, int K, const Epi &epi, cudaStream_t stream) {
  const int sms = device_info().sms;
  const long long tiles = (long long)((Nout + BM - 1) / BM) * ((M + (M <= 64 ? 64 : 128) - 1) / (M <= 64 ? 64 : 128));
  const int nkt = K / BK;
  if (M <= 64) {
    if (4 * tiles <= sms && nkt >= 4) return launch_t<64, 4>(w, x, Nout, M, K, epi, stream);
    if (2 * tiles <= sms && nkt >= 2) return launch_t<64, 2>(w, x, Nout, M, K, epi, stream);
    return launch_t<64, 1>(w, x, Nout, M, K, epi, stream);
  }
  // weights beyond half of L2 would stream from DRAM once per few token tiles in row-major order
  const bool grouped = (long long)Nout * K * 2 > (64LL << 20);
  if (M <= 128) return grouped ? launch_t<128, 1, true>(w, x, Nout, M, K, epi, stream)
                               : launch_t<128, 1>(w, x, Nout, M, K, epi, stream);
  // 256-token tiles: a quarter less shared-memory traffic per product than 128
  return grouped ? launch_t<256, 1, true>(w, x, Nout, M, K, epi, stream) : launch_t<256, 1>(w, x, Nout, M, K, epi, stream);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace proj
}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status gdn_in_proj(const gdn_dims *dims, int32_t M, int32_t H, const void *hidden, const void *w_in, void *q,
                       void *k, void *v, void *z, void *a, void *b, void *stream) {
  if (!dims) return fail(GDN_ERR_ARG, "dims is NULL");
  if (dims->nk <= 0 || dims->nv <= 0 || dims->dk <= 0 || dims->dv <= 0)
    return fail(GDN_ERR_SHAPE, "bad head dimensions");
  if (M < 0 || H <= 0 || H % proj::BK != 0) return fail(GDN_ERR_SHAPE, "M must be >= 0 and H a multiple of 64");
  const void *ptrs[] = {hidden, w_in, q, k, v, z, a, b};
  for (const void *p : ptrs)
    if (!p || !proj::aligned16(p)) return fail(GDN_ERR_ARG, "a pointer is NULL or not 16-byte aligned");
  const long long kd = (long long)dims->nk * dims->dk, vd = (long long)dims->nv * dims->dv, nv = dims->nv;
  const long long N = 2 * kd + vd + vd + 2 * nv;
  if (N > (1LL << 30) || (long long)M * H > (1LL << 40)) return fail(GDN_ERR_SHAPE, "projection too large");
  if (M == 0) return GDN_OK;
  const DeviceInfo *dev;
  if (gdn_status st = current_device(&dev)) return st;
  proj::Epi epi;
  epi.nseg = 6;
  // in_proj output columns: the mixed q | k | v channels, then z, b, a
  const long long C = 2 * kd + vd;
  epi.seg[0] = {0, (int)kd, static_cast<bf16 *>(q), kd};
  epi.seg[1] = {(int)kd, (int)(2 * kd), static_cast<bf16 *>(k), kd};
  epi.seg[2] = {(int)(2 * kd), (int)C, static_cast<bf16 *>(v), vd};
  epi.seg[3] = {(int)C, (int)(C + vd), static_cast<bf16 *>(z), vd};
  epi.seg[4] = {(int)(C + vd), (int)(C + vd + nv), static_cast<bf16 *>(b), nv};
  epi.seg[5] = {(int)(C + vd + nv), (int)N, static_cast<bf16 *>(a), nv};
  return proj::launch(w_in, hidden, (int)N, M, H, epi, static_cast<cudaStream_t>(stream));
}

gdn_status gdn_out_proj(int32_t M, int32_t H, int32_t V, const void *o, const void *w_out, void *y, void *stream) {
  if (M < 0 || H <= 0 || V <= 0 || V % proj::BK != 0)
    return fail(GDN_ERR_SHAPE, "M must be >= 0, H > 0 and V a multiple of 64");
  const void *ptrs[] = {o, w_out, y};
  for (const void *p : ptrs)
    if (!p || !proj::aligned16(p)) return fail(GDN_ERR_ARG, "a pointer is NULL or not 16-byte aligned");
  if ((long long)H * 2 % 16 != 0) return fail(GDN_ERR_SHAPE, "H must be a multiple of 8");
  if (M == 0) return GDN_OK;
  const DeviceInfo *dev;
  if (gdn_status st = current_device(&dev)) return st;
  proj::Epi epi;
  epi.nseg = 1;
  epi.seg[0] = {0, H, static_cast<bf16 *>(y), H};
  return proj::launch(w_out, o, H, M, V, epi, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
