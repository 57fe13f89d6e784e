// The C-ABI of libgdn (declared in include/gdn.h): host-side validation, the
// per-device status word, and dispatch to the kernels' launchers.
#include <stdio.h>

#include <mutex>
#include <string>

#include "gdn_launch.h"

namespace gdn {

// Device-detected errors: bit n set = gdn_status n was recorded.
__device__ unsigned int g_status_word;

namespace {

thread_local std::string t_last_error = "no error";

struct DeviceTable {
  std::mutex mu;
  bool ready[kMaxDevices] = {};
  DeviceInfo info[kMaxDevices];
};
DeviceTable &table() {
  static DeviceTable t;
  return t;
}
thread_local int t_device = -1;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

gdn_status fail(gdn_status code, const char *msg) {
  t_last_error = msg;
  return code;
}

gdn_status check_launch(const char *what) {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return GDN_OK;
  t_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return GDN_ERR_CUDA;
}

gdn_status current_device(const DeviceInfo **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(GDN_ERR_CUDA, "no usable CUDA device");
  DeviceTable &T = table();
  std::lock_guard<std::mutex> lock(T.mu);
  if (!T.ready[dev]) {
    DeviceInfo d;
    d.id = dev;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return fail(GDN_ERR_CUDA, "cannot query the SM count");
    void *p = nullptr;
    // The symbol's host-side name is not a device address: ask the runtime
    // for this device's copy.
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess)
      return fail(GDN_ERR_CUDA, "cannot locate the device status word");
    d.status = static_cast<unsigned int *>(p);
    T.info[dev] = d;
    T.ready[dev] = true;
  }
  t_device = dev;
  *out = &T.info[dev];
  return GDN_OK;
}

const DeviceInfo &device_info() { return table().info[t_device]; }

}  // namespace gdn

using namespace gdn;

namespace {

gdn_status check_dims(const gdn_dims *d, bool /*packed_ok*/) {
  if (!d) return fail(GDN_ERR_ARG, "dims is NULL");
  if (d->B < 0 || d->T < 0) return fail(GDN_ERR_SHAPE, "B and T must be >= 0");
  if (d->nk <= 0 || d->nv <= 0 || d->nv % d->nk != 0)
    return fail(GDN_ERR_SHAPE, "nk, nv must be > 0 with nv a multiple of nk");
  if (d->nv / d->nk > 8) return fail(GDN_ERR_SHAPE, "GQA group nv/nk must be <= 8");
  if (d->dk != d->dv || (d->dk != 32 && d->dk != 64 && d->dk != 128))
    return fail(GDN_ERR_SHAPE, "dk must equal dv and be 32, 64 or 128");
  if (d->conv_k != 4) return fail(GDN_ERR_SHAPE, "conv_k must be 4");
  if (d->n_slots < 1) return fail(GDN_ERR_SHAPE, "n_slots must be >= 1");
  const long long C = 2LL * d->nk * d->dk + (long long)d->nv * d->dv;
  if (C % 8 != 0 || C > (1LL << 24)) return fail(GDN_ERR_SHAPE, "channel count must be a multiple of 8");
  if (!(d->scale == d->scale) || !(d->l2_eps >= 0.0f) || !(d->rms_eps >= 0.0f))
    return fail(GDN_ERR_ARG, "scale must be a number and eps values >= 0");
  return GDN_OK;
}

gdn_status check_ptr(const void *p, const char *name, size_t align = 16) {
  static thread_local char buf[160];
  if (!p) {
    snprintf(buf, sizeof buf, "%s is NULL", name);
    return fail(GDN_ERR_ARG, buf);
  }
  if (!aligned(p, align)) {
    snprintf(buf, sizeof buf, "%s is not %zu-byte aligned", name, align);
    return fail(GDN_ERR_ARG, buf);
  }
  return GDN_OK;
}

#define GDN_TRY(x)                      \
  do {                                  \
    const gdn_status _s = (x);          \
    if (_s != GDN_OK) return _s;        \
  } while (0)

gdn_status check_inputs(const gdn_inputs *in, bool packed_ok) {
  if (!in) return fail(GDN_ERR_ARG, "inputs is NULL");
  GDN_TRY(check_ptr(in->q, "q"));
  GDN_TRY(check_ptr(in->k, "k"));
  GDN_TRY(check_ptr(in->v, "v"));
  GDN_TRY(check_ptr(in->z, "z"));
  GDN_TRY(check_ptr(in->a, "a", 2));
  GDN_TRY(check_ptr(in->b, "b", 2));
  GDN_TRY(check_ptr(in->A_log, "A_log", 4));
  GDN_TRY(check_ptr(in->dt_bias, "dt_bias", 4));
  GDN_TRY(check_ptr(in->conv_w, "conv_w"));
  GDN_TRY(check_ptr(in->norm_w, "norm_w"));
  if (in->mask && !aligned(in->mask, 4)) return fail(GDN_ERR_ARG, "mask is not 4-byte aligned");
  if (in->state_idx && !aligned(in->state_idx, 4)) return fail(GDN_ERR_ARG, "state_idx is not 4-byte aligned");
  if (in->cu_seqlens) {
    if (!packed_ok) return fail(GDN_ERR_ARG, "cu_seqlens is only accepted by prefill");
    if (!aligned(in->cu_seqlens, 4)) return fail(GDN_ERR_ARG, "cu_seqlens is not 4-byte aligned");
  }
  return GDN_OK;
}

LayerArgs make_args(const gdn_dims *d, const gdn_inputs *in, void *conv_state, float *state, void *out,
                    unsigned int *status) {
  LayerArgs A;
  A.B = d->B;
  A.T = d->T;
  A.nk = d->nk;
  A.nv = d->nv;
  A.D = d->dk;
  A.G = d->nv / d->nk;
  A.C = 2 * d->nk * d->dk + d->nv * d->dv;
  A.n_slots = d->n_slots;
  A.scale = d->scale;
  A.l2_eps = d->l2_eps;
  A.rms_eps = d->rms_eps;
  A.q = static_cast<const bf16 *>(in->q);
  A.k = static_cast<const bf16 *>(in->k);
  A.v = static_cast<const bf16 *>(in->v);
  A.z = static_cast<const bf16 *>(in->z);
  A.a = static_cast<const bf16 *>(in->a);
  A.b = static_cast<const bf16 *>(in->b);
  A.A_log = in->A_log;
  A.dt_bias = in->dt_bias;
  A.conv_w = static_cast<const bf16 *>(in->conv_w);
  A.norm_w = static_cast<const bf16 *>(in->norm_w);
  A.mask = in->mask;
  A.cu_seqlens = in->cu_seqlens;
  A.state_idx = in->state_idx;
  A.conv_state = static_cast<bf16 *>(conv_state);
  A.state = state;
  A.out = static_cast<bf16 *>(out);
  A.status = status;
  A.mx = MxInputs{};
  A.ckpt = nullptr;
  A.n_ckpt = 0;
  A.n_ckpt_slots = 0;
  A.ckpt_state = nullptr;
  A.ckpt_conv = nullptr;
  return A;
}

}  // namespace

namespace gdn {
gdn_status validate_prefill(const gdn_dims *dims, const gdn_inputs *in, const void *conv_state,
                            const float *recurrent_state, const void *out) {
  GDN_TRY(check_dims(dims, true));
  GDN_TRY(check_inputs(in, true));
  GDN_TRY(check_ptr(conv_state, "conv_state"));
  GDN_TRY(check_ptr(recurrent_state, "recurrent_state"));
  GDN_TRY(check_ptr(out, "out"));
  if ((long long)(in->cu_seqlens ? 1 : dims->B) * dims->T > (1LL << 31) - 1)
    return fail(GDN_ERR_SHAPE, "too many tokens in one call");
  return GDN_OK;
}
}  // namespace gdn

extern "C" {

gdn_status gdn_decode_step(const gdn_dims *dims, const gdn_inputs *in, void *conv_state, float *recurrent_state,
                           void *out, void *stream) {
  GDN_TRY(check_dims(dims, false));
  if (dims->T != 1) return fail(GDN_ERR_SHAPE, "decode needs T == 1");
  GDN_TRY(check_inputs(in, false));
  GDN_TRY(check_ptr(conv_state, "conv_state"));
  GDN_TRY(check_ptr(recurrent_state, "recurrent_state"));
  GDN_TRY(check_ptr(out, "out"));
  if (dims->B == 0) return GDN_OK;
  const DeviceInfo *dev;
  GDN_TRY(current_device(&dev));
  LayerArgs A = make_args(dims, in, conv_state, recurrent_state, out, dev->status);
  return launch_decode(A, static_cast<cudaStream_t>(stream));
}

gdn_status gdn_decode_step_mxfp8(const gdn_dims *dims, const gdn_inputs_mxfp8 *in, void *conv_state,
                                 float *recurrent_state, void *out, void *stream) {
  GDN_TRY(check_dims(dims, false));
  if (dims->T != 1) return fail(GDN_ERR_SHAPE, "decode needs T == 1");
  if (!in) return fail(GDN_ERR_ARG, "inputs is NULL");
  GDN_TRY(check_ptr(in->q, "q"));
  GDN_TRY(check_ptr(in->k, "k"));
  GDN_TRY(check_ptr(in->v, "v"));
  GDN_TRY(check_ptr(in->z, "z"));
  GDN_TRY(check_ptr(in->q_scale, "q_scale", 1));
  GDN_TRY(check_ptr(in->k_scale, "k_scale", 1));
  GDN_TRY(check_ptr(in->v_scale, "v_scale", 1));
  GDN_TRY(check_ptr(in->z_scale, "z_scale", 1));
  // the bf16 / fp32 members are checked as in gdn_decode_step (token channels
  // stand in for q / k / v / z there: they are not read as bf16)
  gdn_inputs rest = {};
  rest.q = in->q;
  rest.k = in->k;
  rest.v = in->v;
  rest.z = in->z;
  rest.a = in->a;
  rest.b = in->b;
  rest.A_log = in->A_log;
  rest.dt_bias = in->dt_bias;
  rest.conv_w = in->conv_w;
  rest.norm_w = in->norm_w;
  rest.mask = in->mask;
  rest.state_idx = in->state_idx;
  GDN_TRY(check_inputs(&rest, false));
  GDN_TRY(check_ptr(conv_state, "conv_state"));
  GDN_TRY(check_ptr(recurrent_state, "recurrent_state"));
  GDN_TRY(check_ptr(out, "out"));
  if (dims->B == 0) return GDN_OK;
  const DeviceInfo *dev;
  GDN_TRY(current_device(&dev));
  LayerArgs A = make_args(dims, &rest, conv_state, recurrent_state, out, dev->status);
  A.q = A.k = A.v = A.z = nullptr;  // read through A.mx only
  A.mx.q = static_cast<const uint8_t *>(in->q);
  A.mx.k = static_cast<const uint8_t *>(in->k);
  A.mx.v = static_cast<const uint8_t *>(in->v);
  A.mx.z = static_cast<const uint8_t *>(in->z);
  A.mx.qs = static_cast<const uint8_t *>(in->q_scale);
  A.mx.ks = static_cast<const uint8_t *>(in->k_scale);
  A.mx.vs = static_cast<const uint8_t *>(in->v_scale);
  A.mx.zs = static_cast<const uint8_t *>(in->z_scale);
  return launch_decode(A, static_cast<cudaStream_t>(stream));
}

gdn_status gdn_verify_with_checkpoints(const gdn_dims *dims, const gdn_inputs *in, const void *conv_state,
                                       const float *recurrent_state, void *out, float *ckpt_state, void *ckpt_conv,
                                       void *stream) {
  GDN_TRY(check_dims(dims, false));
  if (dims->T < 1 || dims->T > 8) return fail(GDN_ERR_SHAPE, "verify needs 1 <= T <= 8");
  GDN_TRY(check_inputs(in, false));
  GDN_TRY(check_ptr(conv_state, "conv_state"));
  GDN_TRY(check_ptr(recurrent_state, "recurrent_state"));
  GDN_TRY(check_ptr(out, "out"));
  GDN_TRY(check_ptr(ckpt_state, "ckpt_state"));
  GDN_TRY(check_ptr(ckpt_conv, "ckpt_conv"));
  if (dims->B == 0) return GDN_OK;
  const DeviceInfo *dev;
  GDN_TRY(current_device(&dev));
  LayerArgs A = make_args(dims, in, const_cast<void *>(conv_state), const_cast<float *>(recurrent_state), out,
                          dev->status);
  return launch_verify(A, ckpt_state, static_cast<bf16 *>(ckpt_conv), static_cast<cudaStream_t>(stream));
}

size_t gdn_prefill_workspace_size(const gdn_dims *dims, int packed) {
  if (check_dims(dims, true) != GDN_OK) return 0;
  const int B = dims->B > 1 ? dims->B : 1;
  return prefill_workspace_bytes(B, dims->T, dims->nk, dims->nv, dims->dk, packed != 0);
}

gdn_status gdn_prefill_chunked(const gdn_dims *dims, const gdn_inputs *in, void *conv_state, float *recurrent_state,
                               void *out, void *workspace, size_t workspace_bytes, void *stream) {
  GDN_TRY(validate_prefill(dims, in, conv_state, recurrent_state, out));
  const bool packed = in->cu_seqlens != nullptr;
  if (dims->B == 0 || dims->T == 0) return GDN_OK;
  const size_t need = prefill_workspace_bytes(dims->B, dims->T, dims->nk, dims->nv, dims->dk, packed);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(GDN_ERR_WORKSPACE, "workspace missing, not 256-byte aligned, or too small");
  const DeviceInfo *dev;
  GDN_TRY(current_device(&dev));
  LayerArgs A = make_args(dims, in, conv_state, recurrent_state, out, dev->status);
  return launch_prefill(A, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

gdn_status gdn_prefill_chunked_ckpt(const gdn_dims *dims, const gdn_inputs *in, void *conv_state,
                                    float *recurrent_state, void *out, void *workspace, size_t workspace_bytes,
                                    const int32_t *ckpt, int32_t n_ckpt, float *ckpt_state, void *ckpt_conv,
                                    int32_t n_ckpt_slots, void *stream) {
  GDN_TRY(validate_prefill(dims, in, conv_state, recurrent_state, out));
  if (n_ckpt < 0 || n_ckpt > (1 << 20)) return fail(GDN_ERR_SHAPE, "n_ckpt must be in [0, 2^20]");
  if (n_ckpt > 0) {
    GDN_TRY(check_ptr(ckpt, "ckpt", 4));
    GDN_TRY(check_ptr(ckpt_state, "ckpt_state"));
    GDN_TRY(check_ptr(ckpt_conv, "ckpt_conv"));
    if (n_ckpt_slots < 1) return fail(GDN_ERR_SHAPE, "n_ckpt_slots must be >= 1");
  }
  const bool packed = in->cu_seqlens != nullptr;
  if (dims->B == 0 || dims->T == 0) return GDN_OK;
  const size_t need = prefill_workspace_bytes(dims->B, dims->T, dims->nk, dims->nv, dims->dk, packed);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(GDN_ERR_WORKSPACE, "workspace missing, not 256-byte aligned, or too small");
  const DeviceInfo *dev;
  GDN_TRY(current_device(&dev));
  LayerArgs A = make_args(dims, in, conv_state, recurrent_state, out, dev->status);
  if (n_ckpt > 0) {
    A.ckpt = ckpt;
    A.n_ckpt = n_ckpt;
    A.n_ckpt_slots = n_ckpt_slots;
    A.ckpt_state = ckpt_state;
    A.ckpt_conv = static_cast<bf16 *>(ckpt_conv);
  }
  return launch_prefill(A, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

gdn_status gdn_state_copy(const gdn_dims *dims, const float *src_state, const void *src_conv, float *dst_state,
                          void *dst_conv, const int32_t *src_slot, const int32_t *dst_slot, int32_t n,
                          int32_t n_src_slots, int32_t n_dst_slots, void *stream) {
  if (!dims) return fail(GDN_ERR_ARG, "dims is NULL");
  if (dims->nk <= 0 || dims->nv <= 0 || dims->dk <= 0 || dims->dv <= 0 || dims->conv_k < 2)
    return fail(GDN_ERR_SHAPE, "bad head dimensions");
  if (n < 0 || n > 65535) return fail(GDN_ERR_SHAPE, "n must be in [0, 65535]");
  if (n_src_slots < 1 || n_dst_slots < 1) return fail(GDN_ERR_SHAPE, "slot counts must be >= 1");
  GDN_TRY(check_ptr(src_state, "src_state"));
  GDN_TRY(check_ptr(dst_state, "dst_state"));
  GDN_TRY(check_ptr(src_slot, "src_slot", 4));
  GDN_TRY(check_ptr(dst_slot, "dst_slot", 4));
  if ((src_conv == nullptr) != (dst_conv == nullptr))
    return fail(GDN_ERR_ARG, "src_conv and dst_conv must both be given or both be NULL");
  if (src_conv) {
    GDN_TRY(check_ptr(src_conv, "src_conv"));
    GDN_TRY(check_ptr(dst_conv, "dst_conv"));
  }
  const size_t state_floats = (size_t)dims->nv * dims->dk * dims->dv;
  const size_t C = 2 * (size_t)dims->nk * dims->dk + (size_t)dims->nv * dims->dv;
  const size_t conv_elems = (size_t)(dims->conv_k - 1) * C;
  if (state_floats % 4 != 0 || (src_conv && conv_elems % 8 != 0))
    return fail(GDN_ERR_SHAPE, "slot sizes must be multiples of 16 bytes");
  if (n == 0) return GDN_OK;
  const DeviceInfo *dev;
  GDN_TRY(current_device(&dev));
  return launch_state_copy(src_state, static_cast<const bf16 *>(src_conv), dst_state, static_cast<bf16 *>(dst_conv),
                           src_slot, dst_slot, n, n_src_slots, n_dst_slots, state_floats, conv_elems,
                           static_cast<cudaStream_t>(stream));
}

gdn_status gdn_commit_accepted(const gdn_dims *dims, int32_t n_layers, int32_t paths, const float *ckpt_state,
                               const void *ckpt_conv, float *state_pool, void *conv_pool, const int32_t *accept_len,
                               const int32_t *dst_slot, int32_t *winner, void *stream) {
  if (!dims) return fail(GDN_ERR_ARG, "dims is NULL");
  if (dims->nk <= 0 || dims->nv <= 0 || dims->dk <= 0 || dims->dv <= 0 || dims->conv_k < 2)
    return fail(GDN_ERR_SHAPE, "bad head dimensions");
  if (dims->B < 0 || dims->T < 1 || dims->T > 8) return fail(GDN_ERR_SHAPE, "B must be >= 0 and 1 <= T <= 8");
  if (dims->n_slots < 1) return fail(GDN_ERR_SHAPE, "n_slots must be >= 1");
  if (paths < 1 || dims->B % paths != 0) return fail(GDN_ERR_SHAPE, "B must be a multiple of paths >= 1");
  if (n_layers < 1) return fail(GDN_ERR_SHAPE, "n_layers must be >= 1");
  if ((long long)(dims->B / paths) * n_layers > 65535) return fail(GDN_ERR_SHAPE, "too many (group, layer) pairs");
  GDN_TRY(check_ptr(ckpt_state, "ckpt_state"));
  GDN_TRY(check_ptr(state_pool, "state_pool"));
  GDN_TRY(check_ptr(accept_len, "accept_len", 4));
  GDN_TRY(check_ptr(dst_slot, "dst_slot", 4));
  if (winner && !aligned(winner, 4)) return fail(GDN_ERR_ARG, "winner is not 4-byte aligned");
  if ((ckpt_conv == nullptr) != (conv_pool == nullptr))
    return fail(GDN_ERR_ARG, "ckpt_conv and conv_pool must both be given or both be NULL");
  if (ckpt_conv) {
    GDN_TRY(check_ptr(ckpt_conv, "ckpt_conv"));
    GDN_TRY(check_ptr(conv_pool, "conv_pool"));
  }
  const size_t state_floats = (size_t)dims->nv * dims->dk * dims->dv;
  const size_t C = 2 * (size_t)dims->nk * dims->dk + (size_t)dims->nv * dims->dv;
  const size_t conv_elems = (size_t)(dims->conv_k - 1) * C;
  if (state_floats % 4 != 0 || (ckpt_conv && conv_elems % 8 != 0))
    return fail(GDN_ERR_SHAPE, "slot sizes must be multiples of 16 bytes");
  if (dims->B == 0) return GDN_OK;
  const DeviceInfo *dev;
  GDN_TRY(current_device(&dev));
  return launch_commit(ckpt_state, static_cast<const bf16 *>(ckpt_conv), state_pool, static_cast<bf16 *>(conv_pool),
                       accept_len, dst_slot, winner, dims->B, dims->T, paths, n_layers, dims->n_slots, state_floats,
                       conv_elems, static_cast<cudaStream_t>(stream));
}

gdn_status gdn_check_status(void *stream) {
  const DeviceInfo *dev;
  GDN_TRY(current_device(&dev));
  const cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, cudaGetErrorString(e));
  unsigned int word = 0;
  if (cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return fail(GDN_ERR_CUDA, "cannot read the device status word");
  if (word == 0) return GDN_OK;
  const unsigned int zero = 0;
  if (cudaMemcpy(dev->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return fail(GDN_ERR_CUDA, "cannot clear the device status word");
  for (int code = 1; code < 32; ++code) {
    if (word & (1u << code)) {
      switch (code) {
        case GDN_ERR_MASK: return fail(GDN_ERR_MASK, "a mask row was not ones followed by zeros (row skipped)");
        case GDN_ERR_INDEX: return fail(GDN_ERR_INDEX, "a slot index or row range was out of bounds (row skipped)");
        case GDN_ERR_TIMEOUT: return fail(GDN_ERR_TIMEOUT, "a bounded wait inside a kernel expired");
        default: return fail(static_cast<gdn_status>(code), "device error");
      }
    }
  }
  return GDN_OK;
}

const char *gdn_last_error(void) { return t_last_error.c_str(); }

}  // extern "C"
