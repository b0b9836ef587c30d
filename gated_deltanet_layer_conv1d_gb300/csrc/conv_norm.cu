// conv_norm.cu -- standalone conv + SiLU + L2 norm over many tokens, the conv-state
// update that follows it, and the Z-gated RMSNorm (sm_103a).
//
// gdn_conv_kernel: one CTA per token; each thread takes 4 consecutive channels, so a
//   warp covers 128 channels = one head at d = 128 and the per-head L2 norm of q and k
//   is a shuffle reduction over the lanes of that head (layer_struct.rs,
//   conv1d_l2norm_f32_strided_k / conv1d_prefill_k).  Inputs before a sequence's first
//   token come from its conv state, which this kernel only reads.
// gdn_prefill_tiles_kernel: the same conv, SiLU and L2 norms for the tensor-core prefill,
//   one CTA per (half of a 64-token chunk, 8 heads): the raw rows arrive in shared memory
//   by bulk copies, then each warp walks one head's tokens in order with the conv window
//   in registers; rows go to the fp16 tile images of the workspace and the gates next to
//   them.
// gdn_conv_state_kernel: afterwards, each sequence's conv state becomes its last d_conv
//   raw inputs (exact copies).  Running it as a second launch keeps every read of the
//   old state ordered before the write of the new one.
// gdn_gated_rmsnorm_kernel: one warp per (token, value head) (layer_struct.rs,
//   gated_rms_norm_f32_k / gated_rms_norm_prefill_k); GATE 1 takes sigmoid(z) in place of
//   SiLU(z) (gated_rms_norm_f32_strided_k of the gdn_norm_sigmoid models).
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "prefill_layout.cuh"
#include "tcgen05.cuh"

namespace gdn {
namespace {

constexpr int kW = 4;
constexpr int kConvThreads = 256;

// Sequence of token t: the last s with cu[s] <= t (cu has n+1 entries).
__device__ __forceinline__ int seq_of(const int32_t* cu, int n, int t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <typename T, int D>
__global__ void __launch_bounds__(kConvThreads) gdn_conv_kernel(const __grid_constant__ ConvParams p) {
  using A = Act<T>;
  const int t = blockIdx.x;
  const int seq = seq_of(p.cu_seqlens, p.n, t);
  const int t0 = p.cu_seqlens[seq], t1 = p.cu_seqlens[seq + 1];
  const int pos = t - t0;
  if (t0 < 0 || t < t0 || t >= t1 || t1 > p.total_tokens) {
    if (threadIdx.x == 0) report(p.status, GDN_ERR_BAD_SEQLENS);
    return;
  }
  const int slot = p.slots[seq];
  if (slot < 0 || slot >= p.n_slots) {
    if (threadIdx.x == 0) report(p.status, GDN_ERR_BAD_SLOT);
    return;
  }
  const T* qkv = reinterpret_cast<const T*>(p.qkv);
  const T* cs = reinterpret_cast<const T*>(p.conv_pool) + size_t(slot) * p.conv_dim * kW;
  const int nq = p.conv_dim / 4;          // channel quads
  const int qk_quads = 2 * p.Hk * D / 4;  // quads of q and k (normalised)
  const int nq_pad = (nq + 31) & ~31;     // whole warps take part in the shuffles
  constexpr int kHeadLanes = D / 4;       // lanes of one head

  for (int qd = threadIdx.x; qd < nq_pad; qd += kConvThreads) {
    const bool live = qd < nq;
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
      const int c = qd * 4;
      float4 win[kW];
#pragma unroll
      for (int j = 0; j < kW; ++j) {
        const int sp = pos - (kW - 1) + j;  // sequence position of window entry j
        if (sp >= 0) {
          win[j] = A::load4(qkv + size_t(t0 + sp) * p.qkv_stride + c);
        } else {
          // entry kW + sp of the conv state of channels c .. c+3
          win[j].x = A::to_f(cs[size_t(c + 0) * kW + kW + sp]);
          win[j].y = A::to_f(cs[size_t(c + 1) * kW + kW + sp]);
          win[j].z = A::to_f(cs[size_t(c + 2) * kW + kW + sp]);
          win[j].w = A::to_f(cs[size_t(c + 3) * kW + kW + sp]);
        }
      }
      const float4 w0 = *reinterpret_cast<const float4*>(p.conv_w + size_t(c + 0) * kW);
      const float4 w1 = *reinterpret_cast<const float4*>(p.conv_w + size_t(c + 1) * kW);
      const float4 w2 = *reinterpret_cast<const float4*>(p.conv_w + size_t(c + 2) * kW);
      const float4 w3 = *reinterpret_cast<const float4*>(p.conv_w + size_t(c + 3) * kW);
      y.x = silu_f(w0.x * win[0].x + w0.y * win[1].x + w0.z * win[2].x + w0.w * win[3].x);
      y.y = silu_f(w1.x * win[0].y + w1.y * win[1].y + w1.z * win[2].y + w1.w * win[3].y);
      y.z = silu_f(w2.x * win[0].z + w2.y * win[1].z + w2.z * win[2].z + w2.w * win[3].z);
      y.w = silu_f(w3.x * win[0].w + w3.y * win[1].w + w3.z * win[2].w + w3.w * win[3].w);
    }
    // L2 norm of each q / k head over its D channels (kHeadLanes lanes).
    float ss = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
#pragma unroll
    for (int off = 1; off < kHeadLanes; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (live) {
      if (qd < qk_quads) {
        const bool is_q = qd < qk_quads / 2;
        const float r = (is_q ? p.q_scale : 1.f) * rsqrtf(ss + p.l2_eps);
        y.x *= r; y.y *= r; y.z *= r; y.w *= r;
      }
      const size_t o = size_t(t) * p.conv_dim + qd * 4;
      if (p.out_bf16) Act<__nv_bfloat16>::store4(reinterpret_cast<__nv_bfloat16*>(p.out) + o, y);
      else *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o) = y;
    }
  }
}

// Pre-pass of the tensor-core prefill (bf16 activations, d = 128).  One CTA per (chunk
// slot, half of the chunk, group of kTileWarps heads), heads numbered as the qkv channels
// are laid out: q heads, then k heads, then v heads.  The CTA's 32 rows of the group's raw
// channels, and the 3 rows before them, arrive in shared memory by one bulk copy per row,
// all issued at once; then warp w walks head w's rows in order with the conv window of its
// lane's 4 channels in registers.  q and k rows are L2-normalised (a shuffle sum over the
// warp, q also scaled by q_scale) and every row lands in its fp16 tile image.  CTAs whose
// group holds value heads also write log(alpha) and beta of those heads.
constexpr int kTileWarps = 8;
constexpr int kTileRows = 32;  // rows per CTA: half a chunk
constexpr uint32_t kTileRowBytes = kTileWarps * 128 * 2;
constexpr uint32_t kTileSmem = (kTileRows + kW - 1) * kTileRowBytes + 16;  // rows + mbarrier

__global__ void __launch_bounds__(kTileWarps * 32)
    gdn_prefill_tiles_kernel(const __grid_constant__ ConvParams p) {
  using A = Act<__nv_bfloat16>;
  constexpr int D = 128, kC = PrefillLayout::kC;
  extern __shared__ __align__(16) unsigned char tsm[];
  const int n_heads = 2 * p.Hk + p.Hv;
  const int groups = (n_heads + kTileWarps - 1) / kTileWarps;
  const int grp = blockIdx.x % groups, hf = (blockIdx.x / groups) & 1;
  const int cs = blockIdx.x / (2 * groups);
  int seq = 0;
  {
    int lo = 0, hi = p.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (PrefillLayout::base(p.cu_seqlens[mid], mid) <= size_t(cs)) lo = mid;
      else hi = mid - 1;
    }
    seq = lo;
  }
  const int t0 = p.cu_seqlens[seq], t1 = p.cu_seqlens[seq + 1];
  if (t0 < 0 || t1 < t0 || t1 > p.total_tokens) {
    if (threadIdx.x == 0) report(p.status, GDN_ERR_BAD_SEQLENS);
    return;
  }
  const size_t slot0 = PrefillLayout::base(t0, seq);
  const int len = t1 - t0, nc = (len + kC - 1) / kC;
  if (size_t(cs) < slot0 || size_t(cs) - slot0 >= size_t(nc)) return;  // an unused slot
  const int pos0 = int(size_t(cs) - slot0) * kC;
  const int L = (len - pos0) < kC ? (len - pos0) : kC;
  const int r_begin = hf * kTileRows;
  if (r_begin >= L) return;  // a short last chunk has no second half
  const int nrows = (L - r_begin) < kTileRows ? (L - r_begin) : kTileRows;
  const int slot = p.slots[seq];
  if (slot < 0 || slot >= p.n_slots) {
    if (threadIdx.x == 0) report(p.status, GDN_ERR_BAD_SLOT);
    return;
  }
  const int nh = (n_heads - grp * kTileWarps) < kTileWarps ? (n_heads - grp * kTileWarps)
                                                          : kTileWarps;
  const __nv_bfloat16* qkv = reinterpret_cast<const __nv_bfloat16*>(p.qkv);
  // shared row j holds sequence position pos0 + r_begin - 3 + j (j < nrows + 3)
  const int p_first = pos0 + r_begin - (kW - 1);
  uint64_t* bar = reinterpret_cast<uint64_t*>(tsm + (kTileRows + kW - 1) * kTileRowBytes);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int j0 = p_first < 0 ? -p_first : 0;  // rows before the sequence: conv state
    const uint32_t bytes = uint32_t(nh) * D * 2;
    mbar_arrive_expect_tx(bar, uint32_t(nrows + kW - 1 - j0) * bytes);
    for (int j = j0; j < nrows + kW - 1; ++j)
      bulk_g2s(tsm + j * kTileRowBytes,
               qkv + size_t(t0 + p_first + j) * p.qkv_stride + size_t(grp) * kTileWarps * D,
               bytes, bar);
  }
  const PrefillLayout lay{p.Hk, p.Hv};
  unsigned char* ws = reinterpret_cast<unsigned char*>(p.workspace);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = grp * kTileWarps + warp;

  // log(alpha) and beta of this group's value heads, while the rows arrive
  for (int idx = threadIdx.x; idx < kTileRows * kTileWarps; idx += kTileWarps * 32) {
    const int r = r_begin + idx / kTileWarps, hh = grp * kTileWarps + idx % kTileWarps;
    if (r >= r_begin + nrows || hh < 2 * p.Hk || hh >= n_heads) continue;
    const int h = hh - 2 * p.Hk;
    const size_t ro = size_t(t0 + pos0 + r) * p.ab_stride + h;
    const float av = A::to_f(reinterpret_cast<const __nv_bfloat16*>(p.a)[ro]);
    const float bv = A::to_f(reinterpret_cast<const __nv_bfloat16*>(p.b)[ro]);
    float* g = reinterpret_cast<float*>(ws + lay.gate(cs, h));
    g[r] = -expf(p.A_log[h]) * softplus_f(av + p.dt_bias[h]);
    g[kC + r] = sigmoid_f(bv);
  }
  if (warp >= nh) return;

  const int c = head * D + lane * 4;  // first channel of this lane
  size_t tile;
  float scale = 0.f;  // 0: v (not normalised)
  if (head < p.Hk) {
    tile = lay.qk(cs, head, 1);
    scale = p.q_scale;
  } else if (head < 2 * p.Hk) {
    tile = lay.qk(cs, head - p.Hk, 0);
    scale = 1.f;
  } else {
    tile = lay.v(cs, head - 2 * p.Hk);
  }
  const float4 w0 = *reinterpret_cast<const float4*>(p.conv_w + size_t(c + 0) * kW);
  const float4 w1 = *reinterpret_cast<const float4*>(p.conv_w + size_t(c + 1) * kW);
  const float4 w2 = *reinterpret_cast<const float4*>(p.conv_w + size_t(c + 2) * kW);
  const float4 w3 = *reinterpret_cast<const float4*>(p.conv_w + size_t(c + 3) * kW);
  float4 win[kW - 1];
  if (p_first < 0) {
    const __nv_bfloat16* cst =
        reinterpret_cast<const __nv_bfloat16*>(p.conv_pool) + size_t(slot) * p.conv_dim * kW;
#pragma unroll
    for (int j = 0; j < kW - 1; ++j) {  // positions -3 .. -1: conv state entries 1 .. 3
      win[j].x = A::to_f(cst[size_t(c + 0) * kW + 1 + j]);
      win[j].y = A::to_f(cst[size_t(c + 1) * kW + 1 + j]);
      win[j].z = A::to_f(cst[size_t(c + 2) * kW + 1 + j]);
      win[j].w = A::to_f(cst[size_t(c + 3) * kW + 1 + j]);
    }
  }
  if (!mbar_wait_bounded(bar, 0)) {
    report(p.status, GDN_ERR_TIMEOUT);
    return;
  }
  const unsigned char* col = tsm + warp * (D * 2) + lane * 8;
  if (p_first >= 0) {
#pragma unroll
    for (int j = 0; j < kW - 1; ++j)
      win[j] = A::load4(reinterpret_cast<const __nv_bfloat16*>(col + j * kTileRowBytes));
  }
  // Four tokens per pass: their inputs are loaded first, the window rotates through
  // registers, and the four L2 sums reduce side by side.
  unsigned char* dst = ws + tile + (lane >> 4) * (kC * 128) + (lane * 4 & 7) * 2;
  const int piece = (lane & 15) >> 1;  // 16-byte piece of the lane's 4 channels in a row
  for (int r0 = 0; r0 < nrows; r0 += 4) {
    float4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      x[u] = (r0 + u < nrows) ? A::load4(reinterpret_cast<const __nv_bfloat16*>(
                                    col + (r0 + u + kW - 1) * kTileRowBytes))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 y[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 a = u >= 3 ? x[u - 3] : win[u];
      const float4 b = u >= 2 ? x[u - 2] : win[u + 1];
      const float4 c = u >= 1 ? x[u - 1] : win[u + 2];
      y[u].x = silu_fast(w0.x * a.x + w0.y * b.x + w0.z * c.x + w0.w * x[u].x);
      y[u].y = silu_fast(w1.x * a.y + w1.y * b.y + w1.z * c.y + w1.w * x[u].y);
      y[u].z = silu_fast(w2.x * a.z + w2.y * b.z + w2.z * c.z + w2.w * x[u].z);
      y[u].w = silu_fast(w3.x * a.w + w3.y * b.w + w3.z * c.w + w3.w * x[u].w);
    }
    win[0] = x[1];
    win[1] = x[2];
    win[2] = x[3];
    if (scale != 0.f) {
      float ss[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        ss[u] = y[u].x * y[u].x + y[u].y * y[u].y + y[u].z * y[u].z + y[u].w * y[u].w;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int u = 0; u < 4; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], o);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float rn = scale * rsqrtf(ss[u] + p.l2_eps);
        y[u].x *= rn;
        y[u].y *= rn;
        y[u].z *= rn;
        y[u].w *= rn;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (r0 + u >= nrows) break;
      const int row = r_begin + r0 + u;
      const __half2 lo = __floats2half2_rn(y[u].x, y[u].y), hi = __floats2half2_rn(y[u].z, y[u].w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&lo);
      pk.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(dst + row * 128 + ((piece ^ (row & 7)) << 4)) = pk;
    }
  }
}

// New conv state of each (sequence, channel): its last kW raw inputs.
template <typename T>
__global__ void gdn_conv_state_kernel(const __grid_constant__ ConvParams p) {
  using A = Act<T>;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.n * p.conv_dim) return;
  const int seq = idx / p.conv_dim, c = idx - seq * p.conv_dim;
  const int t0 = p.cu_seqlens[seq], len = p.cu_seqlens[seq + 1] - t0;
  const int slot = p.slots[seq];
  if (len <= 0 || t0 < 0 || t0 + len > p.total_tokens || slot < 0 || slot >= p.n_slots) return;
  T* cs = reinterpret_cast<T*>(p.conv_pool) + (size_t(slot) * p.conv_dim + c) * kW;
  const float4 old = A::load4(cs);
  const float o[kW] = {old.x, old.y, old.z, old.w};
  const T* qkv = reinterpret_cast<const T*>(p.qkv);
  float nw[kW];
#pragma unroll
  for (int j = 0; j < kW; ++j) {
    const int sp = len - kW + j;  // sequence position of the new entry j
    nw[j] = sp >= 0 ? A::to_f(qkv[size_t(t0 + sp) * p.qkv_stride + c]) : o[kW + sp];
  }
  A::store4(cs, make_float4(nw[0], nw[1], nw[2], nw[3]));
}

// Validates cu_seqlens once (device-side) for the conv launches.
__global__ void gdn_seqlens_check_kernel(const int32_t* cu, int n, int total, int32_t* status) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int a = cu[i], b = cu[i + 1];
    if (a < 0 || b < a || b > total || (i == 0 && a != 0) || (i == n - 1 && b != total))
      report(status, GDN_ERR_BAD_SEQLENS);
  }
}

// kRows rows per warp per pass, all their loads issued before any use, so each warp keeps
// several independent rows in flight.
__device__ __forceinline__ float4 load_o4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 load_o4(const __half* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename T, int D, int GATE, typename OT = float>
__global__ void gdn_gated_rmsnorm_kernel(const OT* __restrict__ o, const T* __restrict__ z,
                                         int64_t z_stride, const float* __restrict__ w,
                                         float eps, int T_, int Hv, T* __restrict__ y) {
  using A = Act<T>;
  constexpr int kRows = 8;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  const bool live = lane * 4 < D;
  const int j = live ? lane * 4 : 0;  // a lane past D reads (and discards) column 0
  const float4 w4 = live ? *reinterpret_cast<const float4*>(w + j) : make_float4(0.f, 0.f, 0.f, 0.f);
  const int rows = T_ * Hv;
  for (int r0 = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * kRows; r0 < rows;
       r0 += warps * kRows) {
    // a row past the end reads row 0: no branch between the loads, so all of them issue
    // before the first use
    float4 ov[kRows], z4[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      const int r = r0 + k < rows ? r0 + k : 0, t = r / Hv, h = r - t * Hv;
      ov[k] = load_o4(o + size_t(r) * D + j);
      z4[k] = A::load4(z + size_t(t) * z_stride + h * D + j);
    }
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      if (!live) {
        ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        z4[k] = ov[k];
      }
    }
    // the rows' sums side by side
    float ss[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k)
      ss[k] = ov[k].x * ov[k].x + ov[k].y * ov[k].y + ov[k].z * ov[k].z + ov[k].w * ov[k].w;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
#pragma unroll
      for (int k = 0; k < kRows; ++k) ss[k] += __shfl_xor_sync(0xffffffffu, ss[k], m);
    }
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      const int r = r0 + k, t = r / Hv, h = r - t * Hv;
      if (live && r < rows) {
        const float inv = rsqrtf(ss[k] / float(D) + eps);
        float4 yv;
        yv.x = ov[k].x * inv * w4.x * zgate_fast(z4[k].x, GATE);
        yv.y = ov[k].y * inv * w4.y * zgate_fast(z4[k].y, GATE);
        yv.z = ov[k].z * inv * w4.z * zgate_fast(z4[k].z, GATE);
        yv.w = ov[k].w * inv * w4.w * zgate_fast(z4[k].w, GATE);
        A::store4(y + size_t(t) * Hv * D + h * D + j, yv);
      }
    }
  }
}

template <typename T>
cudaError_t conv_typed(const ConvParams& p, cudaStream_t stream) {
  gdn_seqlens_check_kernel<<<1, 128, 0, stream>>>(p.cu_seqlens, p.n, p.total_tokens, p.status);
  if (p.total_tokens > 0) {
    if (p.D == 128) gdn_conv_kernel<T, 128><<<p.total_tokens, kConvThreads, 0, stream>>>(p);
    else gdn_conv_kernel<T, 16><<<p.total_tokens, kConvThreads, 0, stream>>>(p);
  }
  const int total = p.n * p.conv_dim;
  gdn_conv_state_kernel<T><<<(total + 255) / 256, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv_step(const ConvParams& p, int dtype, cudaStream_t stream) {
  if (dtype == GDN_DTYPE_BF16) return conv_typed<__nv_bfloat16>(p, stream);
  return conv_typed<float>(p, stream);
}

cudaError_t launch_prefill_prep(const ConvParams& p, cudaStream_t stream) {
  if (p.total_tokens == 0 || p.n == 0) return cudaSuccess;
  const int groups = (2 * p.Hk + p.Hv + kTileWarps - 1) / kTileWarps;
  const size_t slots = PrefillLayout::slots(p.n, p.total_tokens);
  cudaError_t e = cudaFuncSetAttribute(gdn_prefill_tiles_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(kTileSmem));
  if (e != cudaSuccess) return e;
  gdn_prefill_tiles_kernel<<<unsigned(slots * 2 * groups), kTileWarps * 32, kTileSmem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_conv_state_update(const ConvParams& p, int dtype, cudaStream_t stream) {
  const int total = p.n * p.conv_dim;
  if (dtype == GDN_DTYPE_BF16)
    gdn_conv_state_kernel<__nv_bfloat16><<<(total + 255) / 256, 256, 0, stream>>>(p);
  else
    gdn_conv_state_kernel<float><<<(total + 255) / 256, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_seqlens_check(const int32_t* cu, int n, int total, int32_t* status,
                                 cudaStream_t stream) {
  gdn_seqlens_check_kernel<<<1, 128, 0, stream>>>(cu, n, total, status);
  return cudaGetLastError();
}

namespace {

template <int GATE, typename OT>
void gated_rmsnorm_gate(const OT* o, const void* z, int64_t z_stride, const float* w, float eps,
                        int T, int Hv, int D, int dtype, void* y, int blocks, int threads,
                        cudaStream_t stream) {
  if (dtype == GDN_DTYPE_BF16) {
    auto zp = reinterpret_cast<const __nv_bfloat16*>(z);
    auto yp = reinterpret_cast<__nv_bfloat16*>(y);
    if (D == 128) gdn_gated_rmsnorm_kernel<__nv_bfloat16, 128, GATE, OT><<<blocks, threads, 0, stream>>>(o, zp, z_stride, w, eps, T, Hv, yp);
    else gdn_gated_rmsnorm_kernel<__nv_bfloat16, 16, GATE, OT><<<blocks, threads, 0, stream>>>(o, zp, z_stride, w, eps, T, Hv, yp);
  } else {
    auto zp = reinterpret_cast<const float*>(z);
    auto yp = reinterpret_cast<float*>(y);
    if (D == 128) gdn_gated_rmsnorm_kernel<float, 128, GATE, OT><<<blocks, threads, 0, stream>>>(o, zp, z_stride, w, eps, T, Hv, yp);
    else gdn_gated_rmsnorm_kernel<float, 16, GATE, OT><<<blocks, threads, 0, stream>>>(o, zp, z_stride, w, eps, T, Hv, yp);
  }
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const void* o, bool o_half, const void* z, int64_t z_stride,
                                 const float* w, float eps, int T, int Hv, int D, int dtype,
                                 int gate, void* y, cudaStream_t stream) {
  const int rows = T * Hv;
  if (rows == 0) return cudaSuccess;
  const int threads = 256, per_block = threads / 32;
  int blocks = (rows + per_block - 1) / per_block;
  const int cap = sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (o_half) {
    const __half* oh = reinterpret_cast<const __half*>(o);
    if (gate) gated_rmsnorm_gate<1>(oh, z, z_stride, w, eps, T, Hv, D, dtype, y, blocks, threads, stream);
    else gated_rmsnorm_gate<0>(oh, z, z_stride, w, eps, T, Hv, D, dtype, y, blocks, threads, stream);
  } else {
    const float* of = reinterpret_cast<const float*>(o);
    if (gate) gated_rmsnorm_gate<1>(of, z, z_stride, w, eps, T, Hv, D, dtype, y, blocks, threads, stream);
    else gated_rmsnorm_gate<0>(of, z, z_stride, w, eps, T, Hv, D, dtype, y, blocks, threads, stream);
  }
  return cudaGetLastError();
}

}  // namespace gdn
