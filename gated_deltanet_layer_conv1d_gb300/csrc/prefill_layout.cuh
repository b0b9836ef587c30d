// prefill_layout.cuh -- workspace layout of the tensor-core chunked prefill, shared by its
// kernels: the pre-pass writes the q/k/v tiles and gates, the chunk-parallel prep kernel
// reads those and writes W, U, P and the decay sums, the state spine reads all of it and
// writes the core outputs O, and the gated norm turns O into y.
//
// Per 64-token "chunk slot" (each tile an exact shared-memory image, so it moves with one
// bulk copy; "swizzled" = fp16, K-major, 128-byte swizzle, [64][128] = two [64][64] blocks):
//   for every key head:   k_hat tile, q_hat tile                 (swizzled [64][128])
//   for every value head: v tile                                 (swizzled [64][128])
//                         log(alpha)[64], beta[64]               (f32, from the pre-pass)
//                         W  = T diag(beta e^g) K                (swizzled [64][128])
//                         K~ = diag(e^{g_L - g}) K               (swizzled [64][128])
//                         P  = lower_incl(Q K^T e^{g_r - g_s})   (swizzled [64][64])
//                         g  = cumulative log2 decay [64]        (f32; rows past the end
//                                                                 repeat the last value)
//                         U  = T diag(beta) V                    (fp16, [4][64][32]: the
//                               value columns in groups of 32, each group [r][32] with its
//                               16-byte pieces swizzled, piece p of row r at
//                               p ^ ((r / 2) % 4))
// Sequence s owns slots base(s) .. base(s) + ceil(len_s / 64) - 1 with
// base(s) = floor(cu_seqlens[s] / 64) + s, which never overlap and need at most
// floor(total_tokens / 64) + n + 1 slots.  Rows of a slot past the end of its sequence are
// never written by the pre-pass; the prep kernel clears them in shared memory.
// After the slots: O, the f32 core output [total_tokens][H_v][128], used when the caller
// passes no buffer of its own for it.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace gdn {

constexpr int kCountStride = 32;  // int32 words between the spine's progress counters

struct PrefillLayout {
  static constexpr int kC = 64;                          // chunk length
  static constexpr size_t kTile = size_t(64) * 128 * 2;  // one fp16 [64][128] tile
  static constexpr size_t kPTile = size_t(64) * 64 * 2;  // one fp16 [64][64] tile
  static constexpr size_t kGate = size_t(2) * kC * 4;    // log(alpha), beta
  static constexpr size_t kDecay = size_t(kC) * 4;       // g
  static constexpr size_t kU = size_t(kC) * 128 * 2;     // U, fp16
  // per value head: W | K~ | P | g | U  (every part 256-byte aligned)
  static constexpr size_t kHeadPrep = kTile + kTile + kPTile + kDecay + kU;
  int Hk, Hv;
  __host__ __device__ size_t slot_bytes() const {
    return size_t(Hk) * 2 * kTile + size_t(Hv) * (kTile + kGate + kHeadPrep);
  }
  // which: 0 = k_hat, 1 = q_hat
  __host__ __device__ size_t qk(size_t cs, int kh, int which) const {
    return cs * slot_bytes() + (size_t(kh) * 2 + which) * kTile;
  }
  __host__ __device__ size_t v(size_t cs, int h) const {
    return cs * slot_bytes() + size_t(Hk) * 2 * kTile + size_t(h) * kTile;
  }
  __host__ __device__ size_t gate(size_t cs, int h) const {
    return cs * slot_bytes() + size_t(Hk) * 2 * kTile + size_t(Hv) * kTile + size_t(h) * kGate;
  }
  __host__ __device__ size_t prep(size_t cs, int h) const {
    return cs * slot_bytes() + size_t(Hk) * 2 * kTile + size_t(Hv) * (kTile + kGate) +
           size_t(h) * kHeadPrep;
  }
  __host__ __device__ size_t w(size_t cs, int h) const { return prep(cs, h); }
  __host__ __device__ size_t kt(size_t cs, int h) const { return prep(cs, h) + kTile; }
  __host__ __device__ size_t p(size_t cs, int h) const { return prep(cs, h) + 2 * kTile; }
  __host__ __device__ size_t g(size_t cs, int h) const {
    return prep(cs, h) + 2 * kTile + kPTile;
  }
  __host__ __device__ size_t u(size_t cs, int h) const {
    return prep(cs, h) + 2 * kTile + kPTile + kDecay;
  }
  __host__ __device__ static size_t base(int cu_seq, int seq) {
    return size_t(cu_seq / kC) + size_t(seq);
  }
  static size_t slots(int n, int total_tokens) {
    return size_t(total_tokens) / kC + size_t(n) + 1;
  }
  // byte offset of O, after every slot (256-byte aligned)
  size_t o_offset(int n, int total_tokens) const {
    return (slots(n, total_tokens) * slot_bytes() + 255) / 256 * 256;
  }
  // byte offset of the two-slice spine's progress counters: int32 [n][Hv][2], each in a
  // 128-byte line of its own (kCountStride words apart), after O
  size_t count_offset(int n, int total_tokens) const {
    return o_offset(n, total_tokens) + (size_t(total_tokens) * Hv * 128 * 4 + 255) / 256 * 256;
  }
  size_t total_bytes(int n, int total_tokens) const {
    return count_offset(n, total_tokens) + size_t(n) * Hv * 2 * kCountStride * 4;
  }
};

}  // namespace gdn
