// abi.cu -- the extern "C" entry points of libgdn.so: host-side validation (on any error
// nothing is launched), kernel-parameter packing and dispatch.  Declarations and the
// contract of every entry point are in include/gdn.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>

#include "kernels.h"

namespace gdn {

constexpr int kMaxDevices = 64;

int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    return 1;
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

cudaError_t launch_prefill_sequential(const PrefillParams& p, int dtype, cudaStream_t stream);
cudaError_t launch_conv_state_update(const ConvParams& p, int dtype, cudaStream_t stream);
cudaError_t launch_seqlens_check(const int32_t* cu, int n, int total, int32_t* status,
                                 cudaStream_t stream);

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t esize(int dtype) { return dtype == GDN_DTYPE_BF16 ? 2 : 4; }

int conv_dim_of(const gdn_dims& d) { return 2 * d.n_k_heads * d.d_k + d.n_v_heads * d.d_v; }

gdn_status check_dims(const gdn_dims* d) {
  if (!d) return GDN_ERR_NULL_POINTER;
  if (d->n_k_heads <= 0 || d->n_v_heads <= 0 || d->n_v_heads > 1024)
    return GDN_ERR_INVALID_ARGUMENT;
  if (!((d->d_k == 16 && d->d_v == 16) || (d->d_k == 128 && d->d_v == 128)))
    return GDN_ERR_UNSUPPORTED_DIMS;
  if (d->d_conv != 4) return GDN_ERR_UNSUPPORTED_DIMS;
  if (d->n_v_heads % d->n_k_heads != 0) return GDN_ERR_UNSUPPORTED_DIMS;
  if (d->n_v_heads / d->n_k_heads > kMaxG) return GDN_ERR_UNSUPPORTED_DIMS;
  if (!std::isfinite(d->q_scale) || !std::isfinite(d->l2_eps) || !std::isfinite(d->norm_eps) ||
      d->l2_eps < 0.f || d->norm_eps < 0.f)
    return GDN_ERR_INVALID_ARGUMENT;
  if (d->norm_gate != GDN_NORM_GATE_SILU && d->norm_gate != GDN_NORM_GATE_SIGMOID)
    return GDN_ERR_INVALID_ARGUMENT;
  if (d->prefill_precision != GDN_PREFILL_TENSOR_FP16 && d->prefill_precision != GDN_PREFILL_F32)
    return GDN_ERR_INVALID_ARGUMENT;
  return GDN_OK;
}

gdn_status check_weights(const gdn_weights* w) {
  if (!w) return GDN_ERR_NULL_POINTER;
  if (!w->conv_w || !w->A_log || !w->dt_bias || !w->norm_w) return GDN_ERR_NULL_POINTER;
  if (!aligned(w->conv_w, 16) || !aligned(w->norm_w, 16) || !aligned(w->A_log, 4) ||
      !aligned(w->dt_bias, 4))
    return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

// rows: tokens the call reads; 0 skips the pointer checks.
gdn_status check_inputs(const gdn_inputs* in, const gdn_dims& d, int64_t rows) {
  if (!in) return GDN_ERR_NULL_POINTER;
  if (in->dtype != GDN_DTYPE_F32 && in->dtype != GDN_DTYPE_BF16) return GDN_ERR_INVALID_ARGUMENT;
  if (rows == 0) return GDN_OK;
  if (!in->qkv || !in->z || !in->a || !in->b) return GDN_ERR_NULL_POINTER;
  const size_t es = esize(in->dtype);
  if (in->qkv_stride < conv_dim_of(d) || in->z_stride < int64_t(d.n_v_heads) * d.d_v ||
      in->ab_stride < d.n_v_heads)
    return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned(in->qkv, 16) || !aligned(in->z, 16) || (in->qkv_stride * es) % 16 != 0 ||
      (in->z_stride * es) % 16 != 0 || !aligned(in->a, es) || !aligned(in->b, es))
    return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

gdn_status check_out(const void* y, const float* core_out, const int32_t* status) {
  if (!y || !status) return GDN_ERR_NULL_POINTER;
  if (!aligned(y, 16) || (core_out && !aligned(core_out, 16)) || !aligned(status, 4))
    return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

gdn_status check_pools(const void* conv_pool, int32_t n_slots, const int32_t* slots) {
  if (!conv_pool || !slots) return GDN_ERR_NULL_POINTER;
  if (n_slots <= 0) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned(conv_pool, 16) || !aligned(slots, 4)) return GDN_ERR_MISALIGNED;
  return GDN_OK;
}

// A launcher refuses a shape whose shared-memory plan does not fit with
// cudaErrorInvalidConfiguration before launching anything.
gdn_status status_of(cudaError_t e) {
  if (e == cudaSuccess) return GDN_OK;
  if (e == cudaErrorInvalidConfiguration) return GDN_ERR_UNSUPPORTED_DIMS;
  return GDN_ERR_CUDA;
}

#define GDN_TRY(expr)                \
  do {                               \
    const gdn_status s_ = (expr);    \
    if (s_ != GDN_OK) return s_;     \
  } while (0)

void fill_common(RecParams& p, const gdn_dims& d, const gdn_weights& w, const gdn_inputs& in) {
  std::memset(&p, 0, sizeof(p));
  p.Hk = d.n_k_heads;
  p.Hv = d.n_v_heads;
  p.G = d.n_v_heads / d.n_k_heads;
  p.conv_dim = conv_dim_of(d);
  p.q_scale = d.q_scale;
  p.l2_eps = d.l2_eps;
  p.norm_eps = d.norm_eps;
  p.norm_gate = d.norm_gate;
  p.conv_w = w.conv_w;
  p.A_log = w.A_log;
  p.dt_bias = w.dt_bias;
  p.norm_w = w.norm_w;
  p.qkv = in.qkv;
  p.qkv_stride = in.qkv_stride;
  p.z = in.z;
  p.z_stride = in.z_stride;
  p.a = in.a;
  p.b = in.b;
  p.ab_stride = in.ab_stride;
}

gdn_status gated_rmsnorm_impl(const float* o, const void* z, int64_t z_stride, const float* w,
                              float eps, int32_t T, int32_t n_v_heads, int32_t d_v,
                              int32_t dtype, int gate, void* y, gdn_stream_t stream) {
  if (T < 0 || n_v_heads <= 0 || !std::isfinite(eps) || eps < 0.f)
    return GDN_ERR_INVALID_ARGUMENT;
  if (d_v != 16 && d_v != 128) return GDN_ERR_UNSUPPORTED_DIMS;
  if (dtype != GDN_DTYPE_F32 && dtype != GDN_DTYPE_BF16) return GDN_ERR_INVALID_ARGUMENT;
  if (T == 0) return GDN_OK;
  if (!o || !z || !w || !y) return GDN_ERR_NULL_POINTER;
  if (z_stride < int64_t(n_v_heads) * d_v) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned(o, 16) || !aligned(z, 16) || !aligned(w, 16) || !aligned(y, 16) ||
      (z_stride * esize(dtype)) % 16 != 0)
    return GDN_ERR_MISALIGNED;
  const cudaError_t e = launch_gated_rmsnorm(o, false, z, z_stride, w, eps, T, n_v_heads, d_v,
                                             dtype, gate, y, stream);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

int32_t gdn_version(void) { return 100; }

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARGUMENT: return "invalid argument";
    case GDN_ERR_UNSUPPORTED_DIMS: return "unsupported dims";
    case GDN_ERR_NULL_POINTER: return "null pointer";
    case GDN_ERR_MISALIGNED: return "misaligned pointer or stride";
    case GDN_ERR_BAD_K: return "verify k outside 2..16";
    case GDN_ERR_TOO_MANY_SEQS: return "too many sequences";
    case GDN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case GDN_ERR_CUDA: return "CUDA runtime error";
    case GDN_ERR_SCRATCH_TOO_SMALL: return "call needs more than the library's static scratch";
    case GDN_ERR_BAD_TABLE_ENTRY: return "null or misaligned state pointer";
    case GDN_ERR_BAD_SLOT: return "slot out of range";
    case GDN_ERR_BAD_SEQLENS: return "bad cu_seqlens";
    case GDN_ERR_TIMEOUT: return "device wait timed out";
    case GDN_ERR_BAD_ACCEPTED: return "accepted count outside 1..k";
    default: return "unknown status";
  }
}

static gdn_status decode_impl(const gdn_dims* dims, const gdn_weights* weights,
                              const gdn_inputs* inputs, int32_t n, void* h_pool,
                              void* conv_pool, int32_t n_slots, const int32_t* slots_dev,
                              void* y, float* core_out, int32_t* status_dev,
                              gdn_stream_t stream, bool h16) {
  GDN_TRY(check_dims(dims));
  GDN_TRY(check_weights(weights));
  if (n < 0) return GDN_ERR_INVALID_ARGUMENT;
  if (n > GDN_MAX_SEQS) return GDN_ERR_TOO_MANY_SEQS;
  GDN_TRY(check_inputs(inputs, *dims, n));
  if (n == 0) return GDN_OK;
  GDN_TRY(check_out(y, core_out, status_dev));
  GDN_TRY(check_pools(conv_pool, n_slots, slots_dev));
  if (!h_pool) return GDN_ERR_NULL_POINTER;
  if (!aligned(h_pool, 16)) return GDN_ERR_MISALIGNED;
  RecParams p;
  fill_common(p, *dims, *weights, *inputs);
  p.n = n;
  p.n_slots = n_slots;
  p.h_pool = h_pool;
  p.conv_pool = conv_pool;
  p.slots = slots_dev;
  p.y = y;
  p.core_out = core_out;
  p.status = status_dev;
  p.n_items = n * p.Hk;
  const cudaError_t e = launch_recurrent(p, inputs->dtype, dims->d_k, false, h16, stream);
  return status_of(e);
}

gdn_status gdn_decode_batched(const gdn_dims* dims, const gdn_weights* weights,
                              const gdn_inputs* inputs, int32_t n, float* h_pool,
                              void* conv_pool, int32_t n_slots, const int32_t* slots_dev,
                              void* y, float* core_out, int32_t* status_dev,
                              gdn_stream_t stream) {
  return decode_impl(dims, weights, inputs, n, h_pool, conv_pool, n_slots, slots_dev, y,
                     core_out, status_dev, stream, false);
}

gdn_status gdn_decode_batched_h16(const gdn_dims* dims, const gdn_weights* weights,
                                  const gdn_inputs* inputs, int32_t n, void* h_pool,
                                  void* conv_pool, int32_t n_slots, const int32_t* slots_dev,
                                  void* y, float* core_out, int32_t* status_dev,
                                  gdn_stream_t stream) {
  return decode_impl(dims, weights, inputs, n, h_pool, conv_pool, n_slots, slots_dev, y,
                     core_out, status_dev, stream, true);
}

static gdn_status verify_impl(const gdn_dims* dims, const gdn_weights* weights,
                            const gdn_inputs* inputs, int32_t n, const int32_t* ks_host,
                            const uint64_t* wy_tables_dev, void* conv_pool, int32_t n_slots,
                            const int32_t* slots_dev, void* conv_inter, void* y,
                            float* core_out, int32_t* status_dev, gdn_stream_t stream,
                              bool h16, void* woa_stash = nullptr, int32_t woa_seqs = 0,
                              uint32_t* woa_flag = nullptr) {
  GDN_TRY(check_dims(dims));
  GDN_TRY(check_weights(weights));
  if (n <= 0) return GDN_ERR_INVALID_ARGUMENT;
  if (n > GDN_MAX_SEQS) return GDN_ERR_TOO_MANY_SEQS;
  if (!ks_host) return GDN_ERR_NULL_POINTER;
  int64_t rows = 0;
  for (int i = 0; i < n; ++i) {
    if (ks_host[i] < GDN_VERIFY_K_MIN || ks_host[i] > GDN_VERIFY_K_MAX) return GDN_ERR_BAD_K;
    rows += ks_host[i];
  }
  GDN_TRY(check_inputs(inputs, *dims, rows));
  GDN_TRY(check_out(y, core_out, status_dev));
  GDN_TRY(check_pools(conv_pool, n_slots, slots_dev));
  if (!wy_tables_dev) return GDN_ERR_NULL_POINTER;
  if (!aligned(wy_tables_dev, 8) || (conv_inter && !aligned(conv_inter, 16)))
    return GDN_ERR_MISALIGNED;
  if (woa_stash) {
    if (!woa_flag) return GDN_ERR_NULL_POINTER;
    if (!aligned(woa_stash, 16) || !aligned(woa_flag, 4)) return GDN_ERR_MISALIGNED;
    if (woa_seqs < n) return GDN_ERR_INVALID_ARGUMENT;
  }
  RecParams p;
  fill_common(p, *dims, *weights, *inputs);
  if (woa_stash) {
    const WoaLayout l = woa_layout(dims->n_k_heads, dims->n_v_heads, dims->d_k, dims->d_v,
                                   conv_dim_of(*dims), int(esize(inputs->dtype)));
    p.woa_stash = static_cast<unsigned char*>(woa_stash);
    p.woa_flag = woa_flag;
    p.woa_seq_bytes = l.seq_bytes;
    p.woa_alpha = int32_t(l.alpha);
    p.woa_khat = int32_t(l.khat);
    p.woa_delta = int32_t(l.delta);
    p.woa_raw = int32_t(l.raw);
  }
  p.n = n;
  p.n_slots = n_slots;
  p.tables = wy_tables_dev;
  p.conv_pool = conv_pool;
  p.slots = slots_dev;
  p.conv_inter = conv_inter;
  p.y = y;
  p.core_out = core_out;
  p.status = status_dev;
  p.n_items = n * p.Hk;
  int order[GDN_MAX_SEQS];
  int off = 0;
  for (int i = 0; i < n; ++i) {
    p.ks[i] = uint8_t(ks_host[i]);
    p.row_off[i] = uint16_t(off);
    off += ks_host[i];
    order[i] = i;
  }
  // Longest verify first, so the zig-zag deal balances the ragged work.
  std::stable_sort(order, order + n, [&](int a, int b) { return ks_host[a] > ks_host[b]; });
  for (int i = 0; i < n; ++i) p.order[i] = uint8_t(order[i]);
  const cudaError_t e = launch_recurrent(p, inputs->dtype, dims->d_k, true, h16, stream);
  return status_of(e);
}

gdn_status gdn_verify_multi(const gdn_dims* dims, const gdn_weights* weights,
                            const gdn_inputs* inputs, int32_t n, const int32_t* ks_host,
                            const uint64_t* wy_tables_dev, void* conv_pool, int32_t n_slots,
                            const int32_t* slots_dev, void* conv_inter, void* y,
                            float* core_out, int32_t* status_dev, gdn_stream_t stream) {
  return verify_impl(dims, weights, inputs, n, ks_host, wy_tables_dev, conv_pool, n_slots,
                     slots_dev, conv_inter, y, core_out, status_dev, stream, false);
}

size_t gdn_woa_stash_seq_floats(const gdn_dims* dims, int32_t dtype) {
  if (check_dims(dims) != GDN_OK) return 0;
  if (dtype != GDN_DTYPE_F32 && dtype != GDN_DTYPE_BF16) return 0;
  const WoaLayout l = woa_layout(dims->n_k_heads, dims->n_v_heads, dims->d_k, dims->d_v,
                                 conv_dim_of(*dims), int(esize(dtype)));
  return size_t(l.seq_bytes / 4);
}

gdn_status gdn_verify_woa(const gdn_dims* dims, const gdn_weights* weights,
                          const gdn_inputs* inputs, int32_t n, const int32_t* ks_host,
                          const uint64_t* wy_tables_dev, void* conv_pool, int32_t n_slots,
                          const int32_t* slots_dev, void* stash, int32_t stash_seqs,
                          uint32_t* flag_dev, void* y, float* core_out, int32_t* status_dev,
                          gdn_stream_t stream) {
  if (!stash) return GDN_ERR_NULL_POINTER;
  return verify_impl(dims, weights, inputs, n, ks_host, wy_tables_dev, conv_pool, n_slots,
                     slots_dev, nullptr, y, core_out, status_dev, stream, false, stash,
                     stash_seqs, flag_dev);
}

gdn_status gdn_woa_fold(const gdn_dims* dims, int32_t n, const int32_t* accepted_dev,
                        const uint64_t* wy_tables_dev, void* conv_pool, int32_t n_slots,
                        const int32_t* slots_dev, const void* stash, const uint32_t* flag_dev,
                        int32_t dtype, int32_t* status_dev, gdn_stream_t stream) {
  GDN_TRY(check_dims(dims));
  if (n <= 0) return GDN_ERR_INVALID_ARGUMENT;
  if (n > GDN_MAX_SEQS) return GDN_ERR_TOO_MANY_SEQS;
  if (dtype != GDN_DTYPE_F32 && dtype != GDN_DTYPE_BF16) return GDN_ERR_INVALID_ARGUMENT;
  if (!accepted_dev || !wy_tables_dev || !stash || !flag_dev || !status_dev)
    return GDN_ERR_NULL_POINTER;
  GDN_TRY(check_pools(conv_pool, n_slots, slots_dev));
  if (!aligned(accepted_dev, 4) || !aligned(wy_tables_dev, 8) || !aligned(stash, 16) ||
      !aligned(flag_dev, 4) || !aligned(status_dev, 4))
    return GDN_ERR_MISALIGNED;
  WoaFoldParams p;
  std::memset(&p, 0, sizeof(p));
  p.Hk = dims->n_k_heads;
  p.Hv = dims->n_v_heads;
  p.d = dims->d_k;
  p.conv_dim = conv_dim_of(*dims);
  p.esize = int32_t(esize(dtype));
  p.n = n;
  p.n_slots = n_slots;
  p.accepted = accepted_dev;
  p.tables = wy_tables_dev;
  p.conv_pool = conv_pool;
  p.slots = slots_dev;
  p.stash = static_cast<const unsigned char*>(stash);
  p.flag = flag_dev;
  p.status = status_dev;
  p.lay = woa_layout(p.Hk, p.Hv, dims->d_k, dims->d_v, p.conv_dim, p.esize);
  return status_of(launch_woa_fold(p, stream));
}

gdn_status gdn_woa_clear(uint32_t* flag_dev, gdn_stream_t stream) {
  if (!flag_dev) return GDN_ERR_NULL_POINTER;
  if (!aligned(flag_dev, 4)) return GDN_ERR_MISALIGNED;
  return status_of(launch_woa_clear(flag_dev, stream));
}

gdn_status gdn_verify_multi_h16(const gdn_dims* dims, const gdn_weights* weights,
                                const gdn_inputs* inputs, int32_t n, const int32_t* ks_host,
                                const uint64_t* wy_tables_dev, void* conv_pool,
                                int32_t n_slots, const int32_t* slots_dev, void* conv_inter,
                                void* y, float* core_out, int32_t* status_dev,
                                gdn_stream_t stream) {
  return verify_impl(dims, weights, inputs, n, ks_host, wy_tables_dev, conv_pool, n_slots,
                     slots_dev, conv_inter, y, core_out, status_dev, stream, true);
}

gdn_status gdn_state_convert(const void* src, int32_t src_dtype, void* dst, int32_t dst_dtype,
                             int64_t count, gdn_stream_t stream) {
  const bool widen = src_dtype == GDN_DTYPE_F16 && dst_dtype == GDN_DTYPE_F32;
  const bool narrow = src_dtype == GDN_DTYPE_F32 && dst_dtype == GDN_DTYPE_F16;
  if (!widen && !narrow) return GDN_ERR_INVALID_ARGUMENT;
  if (count < 0) return GDN_ERR_INVALID_ARGUMENT;
  if (count == 0) return GDN_OK;
  if (!src || !dst) return GDN_ERR_NULL_POINTER;
  if (!aligned(src, 16) || !aligned(dst, 16)) return GDN_ERR_MISALIGNED;
  return status_of(launch_state_convert(src, src_dtype, dst, dst_dtype, size_t(count), stream));
}

gdn_status gdn_fold_accepted(const gdn_dims* dims, int32_t n, const int32_t* ks_host,
                             const int32_t* accepted_dev, const uint64_t* wy_tables_dev,
                             void* conv_pool, int32_t n_slots, const int32_t* slots_dev,
                             const void* conv_inter, int32_t dtype, int32_t h_dtype,
                             int32_t* status_dev, gdn_stream_t stream) {
  GDN_TRY(check_dims(dims));
  if (n <= 0) return GDN_ERR_INVALID_ARGUMENT;
  if (n > GDN_MAX_SEQS) return GDN_ERR_TOO_MANY_SEQS;
  if (dtype != GDN_DTYPE_F32 && dtype != GDN_DTYPE_BF16) return GDN_ERR_INVALID_ARGUMENT;
  if (h_dtype != GDN_DTYPE_F32 && h_dtype != GDN_DTYPE_F16) return GDN_ERR_INVALID_ARGUMENT;
  if (!ks_host || !accepted_dev || !wy_tables_dev || !conv_inter || !status_dev)
    return GDN_ERR_NULL_POINTER;
  for (int i = 0; i < n; ++i)
    if (ks_host[i] < GDN_VERIFY_K_MIN || ks_host[i] > GDN_VERIFY_K_MAX) return GDN_ERR_BAD_K;
  GDN_TRY(check_pools(conv_pool, n_slots, slots_dev));
  if (!aligned(accepted_dev, 4) || !aligned(wy_tables_dev, 8) || !aligned(conv_inter, 16) ||
      !aligned(status_dev, 4))
    return GDN_ERR_MISALIGNED;
  FoldParams p;
  std::memset(&p, 0, sizeof(p));
  p.Hv = dims->n_v_heads;
  p.d_k = dims->d_k;
  p.d_v = dims->d_v;
  p.conv_dim = conv_dim_of(*dims);
  p.d_conv = dims->d_conv;
  p.esize = int32_t(esize(dtype));
  p.h_esize = h_dtype == GDN_DTYPE_F16 ? 2 : 4;
  p.n = n;
  p.n_slots = n_slots;
  p.accepted = accepted_dev;
  p.tables = wy_tables_dev;
  p.conv_pool = conv_pool;
  p.slots = slots_dev;
  p.conv_inter = conv_inter;
  p.status = status_dev;
  for (int i = 0; i < n; ++i) p.ks[i] = uint8_t(ks_host[i]);
  return status_of(launch_fold(p, stream));
}

gdn_status gdn_conv_step(const gdn_dims* dims, const gdn_weights* weights,
                         const gdn_inputs* inputs, int32_t n, const int32_t* cu_seqlens_dev,
                         int32_t total_tokens, void* conv_pool, int32_t n_slots,
                         const int32_t* slots_dev, float* qkv_out, int32_t* status_dev,
                         gdn_stream_t stream) {
  GDN_TRY(check_dims(dims));
  GDN_TRY(check_weights(weights));
  if (n < 0 || total_tokens < 0) return GDN_ERR_INVALID_ARGUMENT;
  if (n == 0) return total_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARGUMENT;
  if (!inputs) return GDN_ERR_NULL_POINTER;
  if (inputs->dtype != GDN_DTYPE_F32 && inputs->dtype != GDN_DTYPE_BF16)
    return GDN_ERR_INVALID_ARGUMENT;
  if (total_tokens > 0) {
    if (!inputs->qkv || !qkv_out) return GDN_ERR_NULL_POINTER;
    if (inputs->qkv_stride < conv_dim_of(*dims)) return GDN_ERR_INVALID_ARGUMENT;
    if (!aligned(inputs->qkv, 16) || (inputs->qkv_stride * esize(inputs->dtype)) % 16 != 0 ||
        !aligned(qkv_out, 16))
      return GDN_ERR_MISALIGNED;
  }
  if (!cu_seqlens_dev || !status_dev) return GDN_ERR_NULL_POINTER;
  GDN_TRY(check_pools(conv_pool, n_slots, slots_dev));
  ConvParams p;
  std::memset(&p, 0, sizeof(p));
  p.Hk = dims->n_k_heads;
  p.Hv = dims->n_v_heads;
  p.D = dims->d_k;
  p.conv_dim = conv_dim_of(*dims);
  p.n = n;
  p.n_slots = n_slots;
  p.total_tokens = total_tokens;
  p.q_scale = dims->q_scale;
  p.l2_eps = dims->l2_eps;
  p.conv_w = weights->conv_w;
  p.qkv = inputs->qkv;
  p.qkv_stride = inputs->qkv_stride;
  p.cu_seqlens = cu_seqlens_dev;
  p.conv_pool = conv_pool;
  p.slots = slots_dev;
  p.out = qkv_out;
  p.out_bf16 = 0;
  p.status = status_dev;
  const cudaError_t e = launch_conv_step(p, inputs->dtype, stream);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

size_t gdn_prefill_workspace_bytes(const gdn_dims* dims, int32_t n, int32_t total_tokens,
                                   int32_t max_seqlen, int32_t chunk) {
  if (check_dims(dims) != GDN_OK || n < 0 || total_tokens < 0 || max_seqlen < 0 ||
      chunk != GDN_PREFILL_CHUNK)
    return 0;
  if (dims->prefill_precision == GDN_PREFILL_F32) return 0;  // the sequential form needs none
  return prefill_workspace_bytes(dims->n_k_heads, dims->n_v_heads, dims->d_k, n, total_tokens,
                                 max_seqlen);
}

gdn_status gdn_prefill_chunked(const gdn_dims* dims, const gdn_weights* weights,
                               const gdn_inputs* inputs, int32_t n,
                               const int32_t* cu_seqlens_dev, int32_t total_tokens,
                               int32_t max_seqlen, int32_t chunk,
                               const uint64_t* h_state_ptrs_dev, void* conv_pool,
                               int32_t n_slots, const int32_t* slots_dev, void* y,
                               float* core_out, void* workspace, size_t workspace_bytes,
                               int32_t* status_dev, gdn_stream_t stream) {
  GDN_TRY(check_dims(dims));
  GDN_TRY(check_weights(weights));
  if (chunk != GDN_PREFILL_CHUNK) return GDN_ERR_INVALID_ARGUMENT;
  if (n < 0 || n > 65535 / 32 || total_tokens < 0 || max_seqlen < 0)
    return GDN_ERR_INVALID_ARGUMENT;
  if (n == 0) return total_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARGUMENT;
  GDN_TRY(check_inputs(inputs, *dims, total_tokens));
  GDN_TRY(check_out(y, core_out, status_dev));
  GDN_TRY(check_pools(conv_pool, n_slots, slots_dev));
  if (!cu_seqlens_dev || !h_state_ptrs_dev) return GDN_ERR_NULL_POINTER;
  if (!aligned(cu_seqlens_dev, 4) || !aligned(h_state_ptrs_dev, 8)) return GDN_ERR_MISALIGNED;
  const size_t need = dims->prefill_precision == GDN_PREFILL_F32
                          ? 0
                          : prefill_workspace_bytes(dims->n_k_heads, dims->n_v_heads, dims->d_k,
                                                    n, total_tokens, max_seqlen);
  if (need > 0) {
    if (!workspace) return GDN_ERR_NULL_POINTER;
    if (!aligned(workspace, 256)) return GDN_ERR_MISALIGNED;
    if (workspace_bytes < need) return GDN_ERR_WORKSPACE_TOO_SMALL;
  }
  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  p.Hk = dims->n_k_heads;
  p.Hv = dims->n_v_heads;
  p.G = p.Hv / p.Hk;
  p.D = dims->d_k;
  p.conv_dim = conv_dim_of(*dims);
  p.n = n;
  p.n_slots = n_slots;
  p.total_tokens = total_tokens;
  p.max_seqlen = max_seqlen;
  p.max_chunks = (max_seqlen + GDN_PREFILL_CHUNK - 1) / GDN_PREFILL_CHUNK;
  p.q_scale = dims->q_scale;
  p.l2_eps = dims->l2_eps;
  p.norm_eps = dims->norm_eps;
  p.norm_gate = dims->norm_gate;
  p.f32_path = dims->prefill_precision == GDN_PREFILL_F32;
  p.conv_w = weights->conv_w;
  p.A_log = weights->A_log;
  p.dt_bias = weights->dt_bias;
  p.norm_w = weights->norm_w;
  p.qkv = inputs->qkv;
  p.qkv_stride = inputs->qkv_stride;
  p.z = inputs->z;
  p.z_stride = inputs->z_stride;
  p.a = inputs->a;
  p.b = inputs->b;
  p.ab_stride = inputs->ab_stride;
  p.cu_seqlens = cu_seqlens_dev;
  p.h_ptrs = h_state_ptrs_dev;
  p.conv_pool = conv_pool;
  p.slots = slots_dev;
  p.y = y;
  p.core_out = core_out;
  p.status = status_dev;
  p.workspace = workspace;
  p.workspace_bytes = workspace_bytes;
  cudaError_t e = launch_seqlens_check(cu_seqlens_dev, n, total_tokens, status_dev, stream);
  if (e == cudaSuccess) e = launch_prefill(p, inputs->dtype, stream);
  if (e == cudaSuccess) {
    // The conv state moves to each sequence's last d_conv inputs only after the prefill
    // kernels have read the old one.
    ConvParams c;
    std::memset(&c, 0, sizeof(c));
    c.conv_dim = p.conv_dim;
    c.n = n;
    c.n_slots = n_slots;
    c.total_tokens = total_tokens;
    c.qkv = inputs->qkv;
    c.qkv_stride = inputs->qkv_stride;
    c.cu_seqlens = cu_seqlens_dev;
    c.conv_pool = conv_pool;
    c.slots = slots_dev;
    c.status = status_dev;
    e = launch_conv_state_update(c, inputs->dtype, stream);
  }
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}


gdn_status gdn_gated_rmsnorm(const float* o, const void* z, int64_t z_stride, const float* w,
                             float eps, int32_t T, int32_t n_v_heads, int32_t d_v,
                             int32_t dtype, void* y, gdn_stream_t stream) {
  return gated_rmsnorm_impl(o, z, z_stride, w, eps, T, n_v_heads, d_v, dtype,
                            GDN_NORM_GATE_SILU, y, stream);
}

gdn_status gdn_gated_rmsnorm_sigmoid(const float* o, const void* z, int64_t z_stride,
                                     const float* w, float eps, int32_t T, int32_t n_v_heads,
                                     int32_t d_v, int32_t dtype, void* y, gdn_stream_t stream) {
  return gated_rmsnorm_impl(o, z, z_stride, w, eps, T, n_v_heads, d_v, dtype,
                            GDN_NORM_GATE_SIGMOID, y, stream);
}

namespace {
// b_weights: B is a weight matrix no kernel writes (in_proj / out_proj), which the GEMM
// fetches before the previous kernel in the stream has finished.
gdn_status proj_gemm_impl(const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                          int64_t ldc, int32_t M, int32_t N, int32_t K, int32_t* status_dev,
                          gdn_stream_t stream, bool b_weights) {
  if (M < 0 || N < 8 || K < 8 || N % 8 != 0 || K % 8 != 0 || lda < K || ldb < K || ldc < N)
    return GDN_ERR_INVALID_ARGUMENT;
  if (M == 0) return GDN_OK;
  if (!A || !B || !C || !status_dev) return GDN_ERR_NULL_POINTER;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(status_dev, 4) ||
      lda % 8 != 0 || ldb % 8 != 0 || ldc % 8 != 0)
    return GDN_ERR_MISALIGNED;
  ProjParams p;
  std::memset(&p, 0, sizeof(p));
  p.A = A;
  p.lda = lda;
  p.B = B;
  p.ldb = ldb;
  p.C = C;
  p.ldc = ldc;
  p.M = M;
  p.N = N;
  p.K = K;
  p.b_weights = b_weights ? 1 : 0;
  p.status = status_dev;
  return launch_proj(p, stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
}  // namespace

gdn_status gdn_proj_gemm(const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                         int64_t ldc, int32_t M, int32_t N, int32_t K, int32_t* status_dev,
                         gdn_stream_t stream) {
  return proj_gemm_impl(A, lda, B, ldb, C, ldc, M, N, K, status_dev, stream, false);
}

int32_t gdn_in_proj_width(const gdn_dims* dims) {
  if (check_dims(dims) != GDN_OK) return 0;
  const int32_t w = conv_dim_of(*dims) + dims->n_v_heads * dims->d_v + 2 * dims->n_v_heads;
  return (w + 7) / 8 * 8;
}

gdn_status gdn_in_proj(const gdn_dims* dims, int32_t hidden_size, const void* hidden,
                       int64_t hidden_stride, int32_t T, const void* w_in, void* out,
                       int32_t* status_dev, gdn_stream_t stream) {
  GDN_TRY(check_dims(dims));
  if (T < 0) return GDN_ERR_INVALID_ARGUMENT;
  const int32_t width = gdn_in_proj_width(dims);
  return proj_gemm_impl(hidden, hidden_stride, w_in, hidden_size, out, width, T, width,
                        hidden_size, status_dev, stream, true);
}

gdn_status gdn_out_proj(const gdn_dims* dims, int32_t hidden_size, const void* y, int32_t T,
                        const void* w_out, void* out, int64_t out_stride, int32_t* status_dev,
                        gdn_stream_t stream) {
  GDN_TRY(check_dims(dims));
  if (T < 0) return GDN_ERR_INVALID_ARGUMENT;
  const int32_t vd = dims->n_v_heads * dims->d_v;
  return proj_gemm_impl(y, vd, w_out, vd, out, out_stride, T, hidden_size, vd, status_dev,
                        stream, true);
}

gdn_status gdn_selftest_wait(int64_t budget_ns, int32_t* status_dev, gdn_stream_t stream) {
  if (budget_ns < 1 || budget_ns > 1000000000LL) return GDN_ERR_INVALID_ARGUMENT;
  if (!status_dev) return GDN_ERR_NULL_POINTER;
  if (!aligned(status_dev, 4)) return GDN_ERR_MISALIGNED;
  return launch_wait_selftest(uint64_t(budget_ns), status_dev, stream) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

gdn_status gdn_wy_tables_fill(uint64_t* host_tables, int32_t n, const int32_t* ks,
                              const uint64_t* h_ptrs, const uint64_t* inter_ptrs) {
  if (!host_tables) return GDN_ERR_NULL_POINTER;
  std::memset(host_tables, 0, GDN_VERIFY_WY_LAYER_STRIDE_BYTES);
  if (n < 0) return GDN_ERR_INVALID_ARGUMENT;
  if (n > GDN_VERIFY_WY_TABLE_SEQS) return GDN_ERR_TOO_MANY_SEQS;
  if (n == 0) return GDN_OK;
  if (!ks || !h_ptrs || !inter_ptrs) return GDN_ERR_NULL_POINTER;
  for (int i = 0; i < n; ++i)
    if (ks[i] < GDN_VERIFY_K_MIN || ks[i] > GDN_VERIFY_WY_TABLES_PER_LAYER) return GDN_ERR_BAD_K;
  for (int i = 0; i < n; ++i) {
    host_tables[i] = h_ptrs[i];
    for (int t = 0; t + 1 < ks[i]; ++t)
      host_tables[size_t(t + 1) * GDN_VERIFY_WY_TABLE_SEQS + i] =
          inter_ptrs[size_t(i) * (GDN_VERIFY_WY_TABLES_PER_LAYER - 1) + t];
  }
  return GDN_OK;
}

}  // extern "C"
