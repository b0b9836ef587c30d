// fold.cu -- the accepted-draft fold after a ragged verify (sm_103a).
//
// trait_layer.rs, LayerWriteOnAccept::gdn_fold_accepted (the h-state table plus a device
// table of accepted counts); layer_struct.rs, gdn_wy4_fold_k.  Sequence i verified k_i
// drafts and kept the first m_i: its state after m_i tokens is intermediate m_i - 1, which
// the verify wrote through table m_i, and its conv state after m_i tokens is the conv
// intermediate m_i - 1.  The fold copies both over the after-k_i states.  It is a pure copy
// (HBM-bound: 2 x the state bytes of every rolled-back sequence), one CTA per (sequence,
// value head) for the state tiles plus one per sequence for the conv state; every thread
// issues all of its 16-byte loads before its stores.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int kFoldThreads = 256;
constexpr int kFoldUnroll = 8;  // 16-byte pieces in flight per thread

// Copies `bytes` (a multiple of 16, both ends 16-B aligned) with the CTA's threads.
__device__ __forceinline__ void copy_block(unsigned char* dst, const unsigned char* src,
                                           size_t bytes) {
  const size_t pieces = bytes / 16;
  for (size_t base = size_t(threadIdx.x); base < pieces; base += size_t(kFoldThreads) * kFoldUnroll) {
    uint4 v[kFoldUnroll];
#pragma unroll
    for (int u = 0; u < kFoldUnroll; ++u) {
      const size_t q = base + size_t(u) * kFoldThreads;
      if (q < pieces) v[u] = reinterpret_cast<const uint4*>(src)[q];
    }
#pragma unroll
    for (int u = 0; u < kFoldUnroll; ++u) {
      const size_t q = base + size_t(u) * kFoldThreads;
      if (q < pieces) reinterpret_cast<uint4*>(dst)[q] = v[u];
    }
  }
}

__global__ void __launch_bounds__(kFoldThreads) gdn_fold_kernel(const __grid_constant__ FoldParams p) {
  const int i = blockIdx.x / (p.Hv + 1), part = blockIdx.x % (p.Hv + 1);
  const int k = p.ks[i];
  const int m = p.accepted[i];
  if (m < 1 || m > k) {
    if (threadIdx.x == 0 && part == 0) report(p.status, GDN_ERR_BAD_ACCEPTED);
    return;
  }
  if (m == k) return;  // the verify already left the state after all k tokens
  if (part < p.Hv) {
    const uint64_t dst = p.tables[i];
    const uint64_t src = p.tables[size_t(m) * GDN_VERIFY_WY_TABLE_SEQS + i];
    if (dst == 0 || src == 0 || (dst & 15u) != 0 || (src & 15u) != 0) {
      if (threadIdx.x == 0 && part == 0) report(p.status, GDN_ERR_BAD_TABLE_ENTRY);
      return;
    }
    const size_t tile = size_t(p.d_k) * p.d_v * p.h_esize;
    copy_block(reinterpret_cast<unsigned char*>(dst) + size_t(part) * tile,
               reinterpret_cast<const unsigned char*>(src) + size_t(part) * tile, tile);
  } else {
    const int slot = p.slots[i];
    if (slot < 0 || slot >= p.n_slots) {
      if (threadIdx.x == 0) report(p.status, GDN_ERR_BAD_SLOT);
      return;
    }
    const size_t bytes = size_t(p.conv_dim) * p.d_conv * p.esize;
    copy_block(reinterpret_cast<unsigned char*>(p.conv_pool) + size_t(slot) * bytes,
               reinterpret_cast<const unsigned char*>(p.conv_inter) +
                   (size_t(i) * (GDN_VERIFY_K_MAX - 1) + size_t(m - 1)) * bytes,
               bytes);
  }
}

}  // namespace

cudaError_t launch_fold(const FoldParams& p, cudaStream_t stream) {
  if (p.n <= 0) return cudaSuccess;
  gdn_fold_kernel<<<p.n * (p.Hv + 1), kFoldThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
