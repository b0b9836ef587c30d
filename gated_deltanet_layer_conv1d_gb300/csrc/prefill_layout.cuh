// prefill_layout.cuh -- workspace layout shared by the chunked-prefill pre-pass (writer)
// and the tensor-core chunk kernel (reader).
//
// The workspace holds, per 64-token "chunk slot", the operand tiles of that chunk exactly
// as the chunk kernel wants them in shared memory, so each arrives with one bulk copy:
//   for every key head:   k_hat tile, q_hat tile  ([64 tokens][128] fp16, 128B-swizzled,
//                         K-major, i.e. two [64][64] column blocks)
//   for every value head: v tile (same layout)
//   for every value head: log(alpha)[64], beta[64] (f32)
// Sequence s owns slots base(s) .. base(s) + ceil(len_s / 64) - 1 with
// base(s) = floor(cu_seqlens[s] / 64) + s, which never overlap and need at most
// floor(total_tokens / 64) + n + 1 slots.  Rows of a slot past the end of its sequence
// are never written; the chunk kernel clears them in shared memory.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace gdn {

struct PrefillLayout {
  static constexpr int kC = 64;                       // chunk length
  static constexpr size_t kTile = size_t(64) * 128 * 2;  // one fp16 [64][128] tile
  int Hk, Hv;
  __host__ __device__ size_t slot_bytes() const {
    return size_t(Hk) * 2 * kTile + size_t(Hv) * kTile + size_t(Hv) * 2 * kC * 4;
  }
  // which: 0 = k_hat, 1 = q_hat
  __host__ __device__ size_t qk(size_t cs, int kh, int which) const {
    return cs * slot_bytes() + (size_t(kh) * 2 + which) * kTile;
  }
  __host__ __device__ size_t v(size_t cs, int h) const {
    return cs * slot_bytes() + size_t(Hk) * 2 * kTile + size_t(h) * kTile;
  }
  __host__ __device__ size_t gate(size_t cs, int h) const {
    return cs * slot_bytes() + size_t(Hk) * 2 * kTile + size_t(Hv) * kTile +
           size_t(h) * 2 * kC * 4;
  }
  __host__ __device__ static size_t base(int cu_seq, int seq) {
    return size_t(cu_seq / kC) + size_t(seq);
  }
  static size_t slots(int n, int total_tokens) {
    return size_t(total_tokens) / kC + size_t(n) + 1;
  }
};

}  // namespace gdn
