// woa.cu -- the write-on-accept verify's stash layout, its deferred fold and the flag clear
// (trait_layer.rs LayerWriteOnAccept: gdn_woa_stash_seq_floats, gdn_woa_bind;
// layer_struct.rs, the gdn_wy4_woa_k / gdn_wy4_fold_k / gdn_wy4_clear_k handles and the
// woa_flag / woa_stash bindings).
//
// A write-on-accept verify writes no state.  Per sequence it leaves k, and per token t and
// head the factors of that token's rank-1 state update, in the stash:
//   S_t = alpha_t S_{t-1} + delta_t k_hat_t^T,   delta_t = beta_t (v_t - alpha_t S_{t-1} k_hat_t)
// (stored as H = S^T: H_t[i][j] = alpha_t H_{t-1}[i][j] + k_hat_t[i] delta_t[j]), together
// with the raw qkv row of every token, and sets the engaged word.  Once the number m of
// accepted drafts is known, the fold replays tokens 0 .. m-1 on the state in one pass (one
// read and one write of it, against k - 1 intermediate states written by the copy form),
// and rolls the conv state forward to the last d_conv raw inputs up to token m - 1.  The
// clear kernel then zeroes the engaged word, so a second fold changes nothing.
#include "common.cuh"
#include "kernels.h"

namespace gdn {

WoaLayout woa_layout(int Hk, int Hv, int dk, int dv, int conv_dim, int esize) {
  auto up16 = [](int64_t x) { return (x + 15) / 16 * 16; };
  constexpr int K = GDN_VERIFY_K_MAX;
  WoaLayout l;
  l.alpha = 128;                                         // [K][Hv] f32 (after k, an i32)
  l.khat = up16(l.alpha + int64_t(K) * Hv * 4);          // [K][Hk][dk] f32
  l.delta = up16(l.khat + int64_t(K) * Hk * dk * 4);     // [K][Hv][dv] f32
  l.raw = up16(l.delta + int64_t(K) * Hv * dv * 4);      // [K][conv_dim], activation dtype
  l.seq_bytes = (l.raw + int64_t(K) * conv_dim * esize + 255) / 256 * 256;
  return l;
}

namespace {

constexpr int kFoldThreads = 256;
constexpr int kW = 4;

// One CTA per (sequence, value head) replays the accepted tokens on that head's state tile;
// one more CTA per sequence rolls its conv state.
template <int D, typename E>
__global__ void __launch_bounds__(kFoldThreads)
    gdn_woa_fold_kernel(const __grid_constant__ WoaFoldParams p) {
  if (*p.flag == 0u) return;  // no verify is waiting to be folded
  const int seq = blockIdx.x / (p.Hv + 1), h = blockIdx.x % (p.Hv + 1);
  const int tid = threadIdx.x;
  const unsigned char* st = p.stash + size_t(seq) * p.lay.seq_bytes;
  const int k = *reinterpret_cast<const int32_t*>(st);
  const int m = p.accepted[seq];
  if (k < GDN_VERIFY_K_MIN || k > GDN_VERIFY_K_MAX || m < 1 || m > k) {
    if (tid == 0 && h == 0) report(p.status, GDN_ERR_BAD_ACCEPTED);
    return;
  }
  if (h < p.Hv) {
    const uint64_t e = p.tables[seq];  // table 0: the sequence's state
    if (e == 0 || (e & 15u) != 0) {
      if (tid == 0 && h == 0) report(p.status, GDN_ERR_BAD_TABLE_ENTRY);
      return;
    }
    __shared__ float al_s[GDN_VERIFY_K_MAX];
    __shared__ __align__(16) float kh_s[GDN_VERIFY_K_MAX][D];
    __shared__ __align__(16) float dl_s[GDN_VERIFY_K_MAX][D];
    const int kh = h / (p.Hv / p.Hk);
    const float* alpha = reinterpret_cast<const float*>(st + p.lay.alpha);
    const float* khat = reinterpret_cast<const float*>(st + p.lay.khat);
    const float* delta = reinterpret_cast<const float*>(st + p.lay.delta);
    for (int idx = tid; idx < m * D; idx += kFoldThreads) {
      const int t = idx / D, i = idx - t * D;
      kh_s[t][i] = khat[(size_t(t) * p.Hk + kh) * D + i];
      dl_s[t][i] = delta[(size_t(t) * p.Hv + h) * D + i];
    }
    if (tid < m) al_s[tid] = alpha[tid * p.Hv + h];
    __syncthreads();
    // H[i][j0..j0+3] for every fourth column: a warp covers one row (D = 128) or two (16)
    float4* H4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(e) + size_t(h) * D * D);
    constexpr int kPer = (D * D / 4 + kFoldThreads - 1) / kFoldThreads;
    float4 x[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int e4 = tid + r * kFoldThreads;
      if (e4 < D * D / 4) x[r] = H4[e4];
    }
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int e4 = tid + r * kFoldThreads;
      if (e4 >= D * D / 4) continue;
      const int i = e4 / (D / 4), j0 = (e4 % (D / 4)) * 4;
      for (int t = 0; t < m; ++t) {
        const float a = al_s[t], ki = kh_s[t][i];
        const float4 d4 = *reinterpret_cast<const float4*>(&dl_s[t][j0]);
        x[r].x = a * x[r].x + ki * d4.x;
        x[r].y = a * x[r].y + ki * d4.y;
        x[r].z = a * x[r].z + ki * d4.z;
        x[r].w = a * x[r].w + ki * d4.w;
      }
      H4[e4] = x[r];
    }
  } else {
    const int slot = p.slots[seq];
    if (slot < 0 || slot >= p.n_slots) {
      if (tid == 0) report(p.status, GDN_ERR_BAD_SLOT);
      return;
    }
    // entry e of the new conv state is sequence position m - 4 + e: from the old state
    // below position 0, else the stashed raw input (both exact copies)
    E* cs = reinterpret_cast<E*>(p.conv_pool) + size_t(slot) * p.conv_dim * kW;
    const E* raw = reinterpret_cast<const E*>(st + p.lay.raw);
    for (int c = tid; c < p.conv_dim; c += kFoldThreads) {
      E old[kW], nw[kW];
#pragma unroll
      for (int e = 0; e < kW; ++e) old[e] = cs[size_t(c) * kW + e];
#pragma unroll
      for (int e = 0; e < kW; ++e) {
        const int pos = m - kW + e;
        nw[e] = pos < 0 ? old[kW + pos] : raw[size_t(pos) * p.conv_dim + c];
      }
#pragma unroll
      for (int e = 0; e < kW; ++e) cs[size_t(c) * kW + e] = nw[e];
    }
  }
}

__global__ void gdn_woa_clear_kernel(uint32_t* flag) { *flag = 0u; }

}  // namespace

cudaError_t launch_woa_fold(const WoaFoldParams& p, cudaStream_t stream) {
  const unsigned grid = unsigned(p.n * (p.Hv + 1));
  if (p.d == 128) {
    if (p.esize == 2) gdn_woa_fold_kernel<128, uint16_t><<<grid, kFoldThreads, 0, stream>>>(p);
    else gdn_woa_fold_kernel<128, uint32_t><<<grid, kFoldThreads, 0, stream>>>(p);
  } else {
    if (p.esize == 2) gdn_woa_fold_kernel<16, uint16_t><<<grid, kFoldThreads, 0, stream>>>(p);
    else gdn_woa_fold_kernel<16, uint32_t><<<grid, kFoldThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_woa_clear(uint32_t* flag, cudaStream_t stream) {
  gdn_woa_clear_kernel<<<1, 1, 0, stream>>>(flag);
  return cudaGetLastError();
}

}  // namespace gdn
