// recurrent.cu -- token-sequential GDN mixer kernels (sm_103a): fused batched decode,
// ragged batched verify, and the token-sequential prefill.
//
// gdn_recurrent_kernel runs, for every (sequence, key head) "item":
//   conv + SiLU over the item's channels (q and k of the key head, v of its G value
//   heads) for the sequence's tokens, the conv-state update, the L2 norms of q and k,
//   the gates, then for each value head the token-sequential gated delta rule on its
//   f32 state and the Z-gated RMSNorm of the outputs
//   (layer_struct.rs: conv1d_l2norm_f32_strided_k, gdn_f32_strided_norm_k,
//   gdn_f32_strided_norm_smem_k, gated_rms_norm_f32_strided_k for decode;
//   gdn_wyn_table_k, gdn_f32_strided_norm_snap_k and gdn_verify_fused_conv_kn_batched_k
//   for the batched verify, which writes every intermediate state through the WY
//   pointer tables of transformer_layer.rs, VERIFY_WY_TABLE_SEQS).
// Decode is verify with one token per sequence, its state addressed through the slot
// pool instead of table 0 and no intermediates.
//
// Design (HBM-bound: the state tile is read once, and written once per token kept):
//   * persistent grid: one CTA per SM (two on fp16 decode pools; decode takes the fewest
//     CTAs that need no more rounds, so its last round is full too); items are dealt to CTAs
//     in a zig-zag over the item list (most tokens first), so ragged k balances;
//   * threads: NT compute threads (16 warps for verify, 8 for decode); decode adds one
//     producer warp and one norm warp;
//   * the state tile of each (item, value head) streams into a shared-memory ring with
//     bulk async copies completing on mbarriers; the tile is moved to registers and its
//     stage refilled -- by decode's producer thread at once, by verify's thread 0 after
//     the head's first barrier -- so STAGES tiles are in flight while one is computed;
//     decode also prefetches the next item's raw prologue inputs;
//   * thread (warp w, lane l) owns rows rb*RS*M + (l/8) + 4m and columns
//     cb*32 + (l%8)*4 .. +3 of the [d_k][d_v] tile (rb = w/4, cb = w%4): every
//     shared-memory read is conflict-free and every 128-bit global store of a warp
//     covers four whole 128-byte lines; fp16 decode holds its tile packed, two values
//     per register;
//   * per token, the column sums u = S k and p = S q are reduced in registers, across
//     the row-lanes with warp shuffles and across the row-block warps through shared
//     memory, then
//       delta = beta (v - alpha u),  S <- alpha S + k delta^T,  o = alpha p + delta (k.q)
//     which is S_t = alpha S (I - beta k k^T) + beta v k^T, o = S_t q regrouped; decode
//     does this once (one barrier) and applies the L2 norms of q and k there as scales
//     (their sums come from the conv pass); verify takes its tokens in pairs, one barrier
//     per pair, the second token seeing the first's update through k_0.k_1 and k_0.q_1
//     (verify_head);
//   * the gated RMSNorm of a head's outputs: decode hands o to the norm warp through a
//     two-slot buffer; verify runs it one warp per token after each head, with z staged
//     in shared memory by the item prologue.
//
// gdn_prefill_seq_kernel is the same per-token update run over a whole sequence, one CTA
// per (sequence, value head), in segments of 16 tokens (layer_struct.rs,
// gdn_prefill_k: the sequential prefill recurrence).  It serves head sizes and dtypes
// the tensor-core chunked prefill does not take.
#include <cuda_fp16.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int kW = 4;  // conv width
constexpr size_t kMaxSmemPerBlock = 232448;  // 227 KiB opt-in shared memory per CTA

template <int D, int NT>
struct RecMap {
  static constexpr int CQ = (D / 4 < 8) ? D / 4 : 8;  // lanes across a row segment
  static constexpr int RS = 32 / CQ;                  // rows per warp instruction
  static constexpr int NW = NT / 32;
  static constexpr int CB = D / (4 * CQ);             // column blocks
  static constexpr int RB = NW / CB;                  // row blocks
  static constexpr int M = D / (RB * RS);             // rows per thread
  static_assert(CB * RB == NW, "warps must tile the columns");
  static_assert(RB * RS * M == D, "threads must tile the rows");
};

// Thread coordinates inside a [D][D] tile.
template <int D, int NT>
struct Lane {
  using Map = RecMap<D, NT>;
  int warp, lane, rb, rs, col0, rowb;
  __device__ __forceinline__ Lane(int tid) {
    warp = tid >> 5;
    lane = tid & 31;
    const int cb = warp % Map::CB;
    rb = warp / Map::CB;
    const int cq = lane % Map::CQ;
    rs = lane / Map::CQ;
    col0 = cb * 4 * Map::CQ + cq * 4;
    rowb = rb * (Map::RS * Map::M) + rs;  // row of m = 0; row m is rowb + RS*m
    xrow = rb * (Map::RS * Map::M) + rs * Map::M;
  }
  __device__ __forceinline__ int row(int m) const { return rowb + Map::RS * m; }
  // xrow: where the thread's M rows start in a vector held in qk_pos order
  int xrow;
};

// Position of element i of a d_k vector held in shared memory in "row-block order": each
// thread's M rows (rowb + RS*m, strided so that a warp's 128-bit stores cover whole
// lines of consecutive rows) sit at xrow .. xrow + M - 1, so it reads them with vector
// loads.  q and k of the verify and decode prologues are staged this way.
template <int D, int NT>
__device__ __forceinline__ int qk_pos(int i) {
  using Map = RecMap<D, NT>;
  constexpr int B = Map::RS * Map::M;
  const int b = i / B, r = i - b * B;
  return b * B + (r % Map::RS) * Map::M + r / Map::RS;
}

// The thread's M elements x[0 .. M - 1] of a shared-memory vector in row-block order
// (x = vector + xrow, 16-byte aligned when M is a multiple of 4).
template <int M>
__device__ __forceinline__ void load_rows(const float* x, float (&out)[M]) {
  if constexpr (M % 4 == 0) {
#pragma unroll
    for (int m = 0; m < M; m += 4) {
      const float4 v = *reinterpret_cast<const float4*>(x + m);
      out[m] = v.x;
      out[m + 1] = v.y;
      out[m + 2] = v.z;
      out[m + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int m = 0; m < M; ++m) out[m] = x[m];
  }
}

// A thread's four state elements of one tile row in registers: f32 (float4), or packed
// fp16 (uint2) where the tile is read from and written back to an fp16 pool after a single
// token, so holding it at storage width rounds exactly where the store would.
__device__ __forceinline__ float4 sr_get(const float4& s) { return s; }
__device__ __forceinline__ float4 sr_get(const uint2& s) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&s.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&s.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void sr_set(float4& s, float4 v) { s = v; }
__device__ __forceinline__ void sr_set(uint2& s, float4 v) {
  const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
  s.x = *reinterpret_cast<const uint32_t*>(&a);
  s.y = *reinterpret_cast<const uint32_t*>(&b);
}

// One token of the gated delta rule on the register tile S (rows L.row(m), columns
// L.col0..+3).  xq, xk: the normalised q, k of the token in shared memory; xv: its v;
// red: this token's reduction buffer [2][RB][D] (alternate per token); orow: where the
// (rb == 0, rs == 0) threads put o.  Contains one __syncthreads.
//
// NAMED selects the barrier: named barrier 1 over the NT compute threads (kernels with a
// separate producer warp) or __syncthreads.  `flag` is OR-reduced by that barrier; if any
// thread raised it, every thread gets true back and the update is not applied.
// PERM: xq and xk hold q and k in row-block order (qk_pos), else in natural order.
// rq, rk: the L2 scales of q and k when xq, xk hold them unnormalised (decode), else 1:
// S k_hat = rk (S k), S q_hat = rq (S q), and k_hat delta^T = k (rk delta)^T.
template <int D, int NT, bool NAMED = false, typename SR = float4, bool PERM = false>
__device__ __forceinline__ bool token_update(SR (&S)[RecMap<D, NT>::M], const Lane<D, NT>& L,
                                             const float* xq, const float* xk, const float* xv,
                                             float al, float be, float kq, float* red,
                                             float* orow, bool flag = false, float rq = 1.f,
                                             float rk = 1.f) {
  using Map = RecMap<D, NT>;
  // packed tiles run at a tighter register budget: k is read again rather than kept, and
  // q and k are read one element at a time
  constexpr bool kReloadK = std::is_same<SR, uint2>::value;
  constexpr bool kVecLoad = PERM && !kReloadK;
  auto at = [&](const float* x, int m) { return PERM ? x[L.xrow + m] : x[L.row(m)]; };
  float kr[Map::M], qr[Map::M];
  if constexpr (kVecLoad) {
    load_rows(xk + L.xrow, kr);
    load_rows(xq + L.xrow, qr);
  }
  float4 u = make_float4(0.f, 0.f, 0.f, 0.f), pp = u;
#pragma unroll
  for (int m = 0; m < Map::M; ++m) {
    const float ki = kVecLoad ? kr[m] : at(xk, m), qi = kVecLoad ? qr[m] : at(xq, m);
    const float4 sm = sr_get(S[m]);
    kr[m] = ki;
    u.x += sm.x * ki; u.y += sm.y * ki; u.z += sm.z * ki; u.w += sm.w * ki;
    pp.x += sm.x * qi; pp.y += sm.y * qi; pp.z += sm.z * qi; pp.w += sm.w * qi;
  }
#pragma unroll
  for (int off = Map::CQ; off < 32; off <<= 1) {
    u.x += __shfl_xor_sync(0xffffffffu, u.x, off);
    u.y += __shfl_xor_sync(0xffffffffu, u.y, off);
    u.z += __shfl_xor_sync(0xffffffffu, u.z, off);
    u.w += __shfl_xor_sync(0xffffffffu, u.w, off);
    pp.x += __shfl_xor_sync(0xffffffffu, pp.x, off);
    pp.y += __shfl_xor_sync(0xffffffffu, pp.y, off);
    pp.z += __shfl_xor_sync(0xffffffffu, pp.z, off);
    pp.w += __shfl_xor_sync(0xffffffffu, pp.w, off);
  }
  if (L.rs == 0) {
    *reinterpret_cast<float4*>(red + L.rb * D + L.col0) = u;
    *reinterpret_cast<float4*>(red + (Map::RB + L.rb) * D + L.col0) = pp;
  }
  const bool abort = NAMED ? named_sync_or(1, NT, flag) : (__syncthreads_or(flag) != 0);
  if (abort) return true;
  float4 U = make_float4(0.f, 0.f, 0.f, 0.f), PP = U;
#pragma unroll
  for (int b = 0; b < Map::RB; ++b) {
    const float4 a4 = *reinterpret_cast<const float4*>(red + b * D + L.col0);
    const float4 p4 = *reinterpret_cast<const float4*>(red + (Map::RB + b) * D + L.col0);
    U.x += a4.x; U.y += a4.y; U.z += a4.z; U.w += a4.w;
    PP.x += p4.x; PP.y += p4.y; PP.z += p4.z; PP.w += p4.w;
  }
  U.x *= rk; U.y *= rk; U.z *= rk; U.w *= rk;
  PP.x *= rq; PP.y *= rq; PP.z *= rq; PP.w *= rq;
  const float4 v4 = *reinterpret_cast<const float4*>(xv + L.col0);
  float4 dl;
  dl.x = be * (v4.x - al * U.x);
  dl.y = be * (v4.y - al * U.y);
  dl.z = be * (v4.z - al * U.z);
  dl.w = be * (v4.w - al * U.w);
  if (L.rb == 0 && L.rs == 0) {
    float4 o;
    o.x = al * PP.x + dl.x * kq;
    o.y = al * PP.y + dl.y * kq;
    o.z = al * PP.z + dl.z * kq;
    o.w = al * PP.w + dl.w * kq;
    *reinterpret_cast<float4*>(orow + L.col0) = o;
  }
  dl.x *= rk; dl.y *= rk; dl.z *= rk; dl.w *= rk;
#pragma unroll
  for (int m = 0; m < Map::M; ++m) {
    const float ki = kReloadK ? at(xk, m) : kr[m];
    float4 sm = sr_get(S[m]);
    sm.x = al * sm.x + ki * dl.x;
    sm.y = al * sm.y + ki * dl.y;
    sm.z = al * sm.z + ki * dl.z;
    sm.w = al * sm.w + ki * dl.w;
    sr_set(S[m], sm);
  }
  return false;
}

// State elements: f32, or fp16 in a half-width pool (the arithmetic stays f32; a tile
// is widened when it is read and rounded to nearest even when it is written).
__device__ __forceinline__ float4 load_state4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 load_state4(const __half* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store_state4(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
__device__ __forceinline__ void store_state4(__half* p, float4 v) {
  const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&a);
  u.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// Tile element (row, col0..+3) into a register of either kind, and back out.
__device__ __forceinline__ void load_sr(float4& r, const float* p) { r = load_state4(p); }
__device__ __forceinline__ void load_sr(float4& r, const __half* p) { r = load_state4(p); }
__device__ __forceinline__ void load_sr(uint2& r, const __half* p) {
  r = *reinterpret_cast<const uint2*>(p);
}
__device__ __forceinline__ void store_sr(float* p, const float4& r) { store_state4(p, r); }
__device__ __forceinline__ void store_sr(__half* p, const float4& r) { store_state4(p, r); }
__device__ __forceinline__ void store_sr(__half* p, const uint2& r) {
  *reinterpret_cast<uint2*>(p) = r;
}

template <int D, int NT, typename SH = float, typename SR = float4>
__device__ __forceinline__ void store_tile(SH* dst, const SR (&S)[RecMap<D, NT>::M],
                                           const Lane<D, NT>& L) {
#pragma unroll
  for (int m = 0; m < RecMap<D, NT>::M; ++m) store_sr(dst + L.row(m) * D + L.col0, S[m]);
}

// L2-normalises q and k of `k` tokens held in shared memory (q at x + t*stride, k right
// after it) and records kq[t] = q.k; one warp per token.
template <int D, int NW>
__device__ __forceinline__ void l2norm_tokens(float* x, int stride, int k, float q_scale,
                                              float eps, float* kq_s, int warp, int lane) {
  for (int t = warp; t < k; t += NW) {
    float* xq = x + t * stride;
    float* xk = xq + D;
    float sq = 0.f, sk = 0.f;
    for (int i = lane; i < D; i += 32) {
      sq += xq[i] * xq[i];
      sk += xk[i] * xk[i];
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    const float rq = q_scale * rsqrtf(sq + eps);
    const float rk = rsqrtf(sk + eps);
    float kq = 0.f;
    for (int i = lane; i < D; i += 32) {
      const float qn = xq[i] * rq, kn = xk[i] * rk;
      xq[i] = qn;
      xk[i] = kn;
      kq += qn * kn;
    }
    kq = warp_sum(kq);
    if (lane == 0) kq_s[t] = kq;
  }
}

// Verify: for each token t (one warp each) the sums q.q, k.k and q.k of its q and k as
// staged (not normalised) and, for the second token of a pair (t odd), k_{t-1}.k_t and
// k_{t-1}.q_t.  The L2 scales r_q = q_scale / |q| and r_k = 1 / |k| go to scl_s[t][2],
// q_hat.k_hat to kq_s[t], the unscaled pair dots to pair_s[t-1], pair_s[t] (the pair loop
// scales them: k_hat_0.k_hat_1 = r_k0 r_k1 k_0.k_1, ...).  Order-independent, so it reads
// q and k in their staged (row-block) order.
template <int D, int NW>
__device__ __forceinline__ void qk_scales_tokens(const float* x, int stride, int k, float q_scale,
                                                 float eps, float* kq_s, float* scl_s,
                                                 float* pair_s, int warp, int lane) {
  for (int t = warp; t < k; t += NW) {
    const float* xq = x + t * stride;
    const float* xk = xq + D;
    const bool second = (t & 1) != 0;  // warp-uniform
    float sq = 0.f, sk = 0.f, sqk = 0.f, skk = 0.f, skq = 0.f;
    for (int i = lane; i < D; i += 32) {
      const float qv = xq[i], kv = xk[i];
      sq += qv * qv;
      sk += kv * kv;
      sqk += qv * kv;
      if (second) {
        const float pv = xk[i - stride];  // k of token t - 1
        skk += pv * kv;
        skq += pv * qv;
      }
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    sqk = warp_sum(sqk);
    if (second) {
      skk = warp_sum(skk);
      skq = warp_sum(skq);
    }
    if (lane == 0) {
      const float rq = q_scale * rsqrtf(sq + eps), rk = rsqrtf(sk + eps);
      scl_s[2 * t] = rq;
      scl_s[2 * t + 1] = rk;
      kq_s[t] = rq * rk * sqk;
      if (second) {
        pair_s[t - 1] = skk;
        pair_s[t] = skq;
      }
    }
  }
}

// Gated RMSNorm of one value head's outputs for `k` tokens, one warp per token.
// o: [k][D] f32 in shared memory; z: [k][zstride] f32 in shared memory (this head's
// slice); y row r = row0 + t.
template <typename T, int D, int NW>
__device__ __forceinline__ void norm_tokens(const float* o, const float* z, int zstride, int k,
                                            int row0, int h, const float* norm_w, float eps,
                                            int gate, int Hv, T* y, float* core_out, int warp,
                                            int lane) {
  using A = Act<T>;
  for (int t = warp; t < k; t += NW) {
    const int row = row0 + t;
    const int j = lane * 4;
    float4 ov = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < D) ov = *reinterpret_cast<const float4*>(o + t * D + j);
    const float ss = warp_sum(ov.x * ov.x + ov.y * ov.y + ov.z * ov.z + ov.w * ov.w);
    if (j < D) {
      const float inv = rsqrtf(ss / float(D) + eps);
      const float4 w4 = *reinterpret_cast<const float4*>(norm_w + j);
      const float4 z4 = *reinterpret_cast<const float4*>(z + t * zstride + j);
      float4 yv;
      yv.x = ov.x * inv * w4.x * zgate(z4.x, gate);
      yv.y = ov.y * inv * w4.y * zgate(z4.y, gate);
      yv.z = ov.z * inv * w4.z * zgate(z4.z, gate);
      yv.w = ov.w * inv * w4.w * zgate(z4.w, gate);
      A::store4(y + size_t(row) * Hv * D + h * D + j, yv);
      if (core_out) *reinterpret_cast<float4*>(core_out + (size_t(row) * Hv + h) * D + j) = ov;
    }
  }
}

// ======================================================================================
// decode / verify
// ======================================================================================
template <int D, int NT, int KMAX, int STAGES, typename T, typename SH = float,
          bool RAWPF = false>
struct RecSmem {
  using Map = RecMap<D, NT>;
  // Decode prefetches the next item's raw inputs into shared memory while the current
  // item runs; verify (k tokens per item) amortises the prologue and skips it.
  static constexpr bool kPrefetch = (KMAX == 1);
  static constexpr size_t kTile = size_t(D) * D * sizeof(SH);
  static constexpr size_t kStage = 0;
  static constexpr size_t kRed = kStage + STAGES * kTile;                  // [2][2][RB][D]
  // Verify reduces a head's column sums two tokens at a time: red is then two buffers of
  // [RB][4][D] (the k and q sums of a pair of tokens).
  static constexpr bool kPairs = (KMAX > 1);
  static constexpr size_t kRedBytes =
      kPairs ? size_t(2) * Map::RB * 4 * D * 4 : size_t(2) * 2 * Map::RB * D * 4;
  // Decode hands each head's output to a norm warp through a two-slot obuf.
  static constexpr bool kNormWarp = (KMAX == 1);
  static constexpr int kObufRows = KMAX > 2 ? KMAX : 2;
  static constexpr size_t kObuf = kRed + kRedBytes;                        // [kObufRows][D]
  static constexpr size_t kNw = kObuf + size_t(kObufRows) * D * 4;         // [D] norm_w
  // mbarriers: full[STAGES] | empty[STAGES] | raw_full | raw_empty | nfull[2] | nfree[2],
  // then two counters (tiles and raw blocks the producer has started), read only when a
  // wait gives up.
  static constexpr size_t kBar = kNw + size_t(D) * 4;
  static constexpr size_t kIssued = kBar + 8 * (2 * STAGES + 6);           // [2] i32
  static constexpr size_t kGate = kIssued + 16;                            // [KMAX][kMaxG][2]
  static constexpr size_t kKq = kGate + size_t(KMAX) * kMaxG * 2 * 4;      // [KMAX]
  // Per-launch staging so no global load sits on the per-head critical path:
  // slot of each sequence, whether its item can run (0 = yes, else the GDN_ERR_* code),
  // its table-0 pointer (verify), and the current item's 16 table entries (verify).
  // decode: per-warp partial sums q.q, k.k, q.k of the item's q and k, [D / 32][3]
  // verify: (k_t0.k_t1, k_t0.q_t1) of each pair of tokens [KMAX/2][2], unscaled; the L2
  // scales (r_q, r_k) of every token [KMAX][2]
  static constexpr size_t kPair = kKq + ((size_t(KMAX) * 4 + 15) / 16) * 16;
  static constexpr size_t kScl = kPair + (kPairs ? ((size_t(KMAX) * 4 + 15) / 16) * 16 : 0);
  static constexpr size_t kL2 = kScl + (kPairs ? size_t(KMAX) * 2 * 4 : 0);
  static constexpr size_t kSlots = kL2 + ((size_t(D + 31) / 32 * 12 + 15) / 16) * 16;  // [128] i32
  static constexpr size_t kValid = kSlots + GDN_MAX_SEQS * 4;                  // [128] i32
  static constexpr size_t kTab0 = kValid + GDN_MAX_SEQS * 4;                   // [128] u64
  static constexpr size_t kTabItem = kTab0 + GDN_MAX_SEQS * 8;                 // [16] u64
  static constexpr size_t kXs = kTabItem + GDN_VERIFY_WY_TABLES_PER_LAYER * 8;
  // xs: [KMAX][(2 + 2G) D] f32 = q | k | v of G heads | z of G heads, per token
  __host__ __device__ static size_t xs_bytes(int G) { return size_t(KMAX) * (2 + 2 * G) * D * 4; }
  // RAWPF: verify prefetches each next item's raw inputs as decode does (where shared memory
  // has room beside the stages), without the conv weights (read from global, where every
  // item of a key head finds them in L2).
  static constexpr bool kRawPF = (KMAX > 1) && RAWPF;
  // raw (decode, kRawPF): conv state [CH][4] T | conv_w [CH][4] f32 (decode) |
  // x [KMAX][CH] T | z [KMAX][G D] T, CH = (2 + G) D
  __host__ __device__ static size_t raw_cs(int) { return 0; }
  __host__ __device__ static size_t raw_w(int G) { return raw_cs(G) + size_t(2 + G) * D * 4 * sizeof(T); }
  __host__ __device__ static size_t raw_x(int G) {
    return raw_w(G) + (kPrefetch ? size_t(2 + G) * D * 4 * 4 : 0);
  }
  __host__ __device__ static size_t raw_z(int G) { return raw_x(G) + size_t(KMAX) * (2 + G) * D * sizeof(T); }
  __host__ __device__ static size_t raw_bytes(int G) {
    return (kPrefetch || kRawPF) ? raw_z(G) + size_t(KMAX) * G * D * sizeof(T) : 0;
  }
  __host__ __device__ static size_t kRaw(int G) { return kXs + xs_bytes(G); }
  __host__ __device__ static size_t bytes(int G) { return kRaw(G) + raw_bytes(G); }
};

// The item this CTA owns in round r: a zig-zag over the item list.
__device__ __forceinline__ int item_at(int cta, int r, int P) {
  return r * P + ((r & 1) ? (P - 1 - cta) : cta);
}

struct Item {
  int seq, kh, k, row0, slot;
};

// Checks a sequence before any of its memory is touched: 0 if it can run, else the
// GDN_ERR_* code (slot out of range; a needed table entry NULL or misaligned).
template <bool VERIFY>
__device__ __forceinline__ int seq_check(const RecParams& p, int seq) {
  const int slot = p.slots[seq];
  if (slot < 0 || slot >= p.n_slots) return GDN_ERR_BAD_SLOT;
  if (VERIFY) {
    const int k = p.woa_stash ? 1 : p.ks[seq];  // write-on-accept reads table 0 only
    for (int t = 0; t < k; ++t) {
      const uint64_t e = p.tables[t * GDN_VERIFY_WY_TABLE_SEQS + seq];
      if (e == 0 || (e & 15u) != 0) return GDN_ERR_BAD_TABLE_ENTRY;
    }
  }
  return 0;
}

// Decodes item j from the launch's staged per-sequence data (shared memory only).
// Returns 0 if the item can run, else its GDN_ERR_* code.
template <bool VERIFY>
__device__ __forceinline__ int item_decode(const RecParams& p, int j, const int32_t* slots_s,
                                           const int32_t* valid_s, Item& it) {
  const int rank = j / p.Hk;
  it.kh = j - rank * p.Hk;
  it.seq = VERIFY ? int(p.order[rank]) : rank;
  it.k = VERIFY ? int(p.ks[it.seq]) : 1;
  it.row0 = VERIFY ? int(p.row_off[it.seq]) : it.seq;
  it.slot = slots_s[it.seq];
  return valid_s[it.seq];
}

// The state of value head h of an item, written after token t (t = k-1: final state).
// tab_item: the item's 16 table entries (verify).
template <int D, bool VERIFY, typename SH>
__device__ __forceinline__ SH* state_dst(const RecParams& p, const Item& it,
                                         const uint64_t* tab_item, int h, int t) {
  if (VERIFY) {
    const int table = (t == it.k - 1) ? 0 : t + 1;
    return reinterpret_cast<SH*>(tab_item[table]) + size_t(h) * D * D;
  }
  return reinterpret_cast<SH*>(p.h_pool) + (size_t(it.slot) * p.Hv + h) * D * D;
}

// The state of value head h of an item as read at its start.
template <int D, bool VERIFY, typename SH>
__device__ __forceinline__ const SH* state_src(const RecParams& p, const Item& it,
                                               const uint64_t* tab0_s, int h) {
  if (VERIFY) return reinterpret_cast<const SH*>(tab0_s[it.seq]) + size_t(h) * D * D;
  return reinterpret_cast<const SH*>(p.h_pool) + (size_t(it.slot) * p.Hv + h) * D * D;
}

__device__ __forceinline__ void fma4(float4& acc, const float4& s, float x) {
  acc.x += s.x * x;
  acc.y += s.y * x;
  acc.z += s.z * x;
  acc.w += s.w * x;
}
// acc += the value of `send` held by lane (lane ^ off)
__device__ __forceinline__ void add_xor4(float4& acc, const float4& send, int off) {
  const float4 r = make_float4(__shfl_xor_sync(0xffffffffu, send.x, off),
                               __shfl_xor_sync(0xffffffffu, send.y, off),
                               __shfl_xor_sync(0xffffffffu, send.z, off),
                               __shfl_xor_sync(0xffffffffu, send.w, off));
  acc.x += r.x;
  acc.y += r.y;
  acc.z += r.z;
  acc.w += r.w;
}

// One value head of a verify item, two tokens per barrier: the column sums of a pair are
// taken from the state before the pair, and the pair's second token sees the first's
// update through two scalars.  In the tile's orientation (H = S^T: rows d_k, columns d_v),
// with A_t = H^T k_t and B_t = H^T q_t of the state H before the pair (t0, t1):
//   delta_0 = beta_0 (v_0 - alpha_0 A_0),       o_0 = alpha_0 B_0 + (q_0.k_0) delta_0
//   H' = alpha_0 H + k_0 delta_0^T,  so  H'^T k_1 = alpha_0 A_1 + (k_0.k_1) delta_0  and
//   H'^T q_1 = alpha_0 B_1 + (k_0.q_1) delta_0, which give delta_1 and o_1 by the same rule
// (the token-by-token delta rule, Gated DeltaNet paper, the gated delta rule's recurrence;
// the pair is its chunkwise form with chunks of two).  The four sums of a pair come out of
// the register tile in one pass: each warp reduce-scatters them over its rows (lane bits 4
// and 3 pick the vector a lane keeps), the warps' partials go through one of two buffers
// [RB][4][D] in turn, and every thread adds the RB partials of its own four columns.  The
// state updates and stores follow in the same step, so stores go out between reductions.
// After the barrier each lane adds up only the vector it kept (RB loads) and takes the
// other three from its neighbours by shuffles.
// q and k are staged unnormalised; scl_s: [KMAX][2] their L2 scales (r_q with the q
// scale); pair_s: [KMAX/2][2] = (k_0.k_1, k_0.q_1) of each pair, unscaled; kq_s:
// q_hat_t.k_hat_t.  after_first()
// runs once, on every thread, after the head's first barrier (every thread holds the tile
// in registers by then).
// Returns true if the first barrier saw `abort` raised by any thread (nothing written).
template <typename T, int D, int NT, int KMAX, typename SH, typename SR, bool WOA, typename F>
__device__ __forceinline__ bool verify_head(const RecParams& p, const Item& it, int h, int g,
                                            int k, SR (&S)[RecMap<D, NT>::M],
                                            const Lane<D, NT>& L, const float* xs, int CHX,
                                            const float* gate, const float* kq_s,
                                            const float* pair_s, const float* scl_s,
                                            float* red, float* obuf,
                                            const uint64_t* tab_item, unsigned char* woa_seq,
                                            bool abort, F&& after_first) {
  using Map = RecMap<D, NT>;
  static_assert(Map::CQ == 4 || Map::CQ == 8, "the reduce-scatter splits lane bits 3 and 4");
  // after the reduce-scatter a lane holds vector 2 hi + mid of (A_0, B_0, A_1, B_1)
  const bool hi = (L.lane >> 4) & 1, mid = (L.lane >> 3) & 1;
  const bool writer = ((L.lane / Map::CQ) & (8 / Map::CQ - 1)) == 0;
  float* woa_d = WOA ? reinterpret_cast<float*>(woa_seq + p.woa_delta) + size_t(h) * D + L.col0
                     : nullptr;
  // The state after a pair's second token is stored row by row inside the next pair's
  // partial sums (which read the same registers), and the state after its first token row
  // by row inside the second token's update, so stores leave between arithmetic rather
  // than in bursts.  pend: where the registers' state still has to go (null: nowhere).
  SH* pend = nullptr;
  for (int t0 = 0; t0 < k; t0 += 2) {
    const bool has1 = t0 + 1 < k;
    const int t1 = has1 ? t0 + 1 : t0;  // odd k: the last pair's second token is a copy
    const float* x0 = xs + t0 * CHX;
    const float* x1 = xs + t1 * CHX;
    float4 K0, K1;  // the k sums of the pair, then its q sums, each halved across lane bit 4
#pragma unroll
    for (int qk = 0; qk < 2; ++qk) {
      const int off = qk ? 0 : D;
      float4 Pa = make_float4(0.f, 0.f, 0.f, 0.f), Pb = Pa;
      float xa[Map::M], xb[Map::M];
      load_rows(x0 + off + L.xrow, xa);
      load_rows(x1 + off + L.xrow, xb);
#pragma unroll
      for (int m = 0; m < Map::M; ++m) {
        const float4 sm = sr_get(S[m]);
        if (!WOA && qk == 0 && pend) store_sr(pend + L.row(m) * D + L.col0, S[m]);
        fma4(Pa, sm, xa[m]);
        fma4(Pb, sm, xb[m]);
      }
      float4 Kx = hi ? Pb : Pa;
      add_xor4(Kx, hi ? Pa : Pb, 16);
      if (qk) K1 = Kx; else K0 = Kx;
    }
    float4 R = mid ? K1 : K0;
    add_xor4(R, mid ? K0 : K1, 8);
#pragma unroll
    for (int off = Map::CQ; off < 8; off <<= 1) {
      const float4 mine = R;
      add_xor4(R, mine, off);
    }
    float* rbuf = red + ((t0 >> 1) & 1) * Map::RB * 4 * D;
    if (writer)
      *reinterpret_cast<float4*>(rbuf + (L.rb * 4 + 2 * hi + mid) * D + L.col0) = R;
    if (t0 == 0) {
      if (named_sync_or(1, NT, abort)) return true;
      after_first();
    } else {
      named_sync(1, NT);
    }
    // each lane adds the RB partials of the vector it holds, for its four columns; the
    // others come from the lanes that hold them
    float4 V = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int b = 0; b < Map::RB; ++b) {
      const float4 a = *reinterpret_cast<const float4*>(rbuf + (b * 4 + 2 * hi + mid) * D + L.col0);
      V.x += a.x; V.y += a.y; V.z += a.z; V.w += a.w;
    }
    auto vec_of = [&](int v) {  // the lane with this lane's columns holding vector v
      const int src = (L.lane & 7) | ((v & 1) << 3) | ((v >> 1) << 4);
      return make_float4(__shfl_sync(0xffffffffu, V.x, src), __shfl_sync(0xffffffffu, V.y, src),
                         __shfl_sync(0xffffffffu, V.z, src), __shfl_sync(0xffffffffu, V.w, src));
    };
    // q and k are staged unnormalised: the sums and the pair dots take their L2 scales here,
    // and k_hat delta^T = k (r_k delta)^T in the updates
    const float rq0 = scl_s[2 * t0], rk0 = scl_s[2 * t0 + 1];
    const float rq1 = scl_s[2 * t1], rk1 = scl_s[2 * t1 + 1];
    float4 A0 = vec_of(0), A1 = vec_of(2);
    A0.x *= rk0; A0.y *= rk0; A0.z *= rk0; A0.w *= rk0;
    A1.x *= rk1; A1.y *= rk1; A1.z *= rk1; A1.w *= rk1;
    const float al0 = gate[(t0 * kMaxG + g) * 2], be0 = gate[(t0 * kMaxG + g) * 2 + 1];
    const float al1 = gate[(t1 * kMaxG + g) * 2], be1 = gate[(t1 * kMaxG + g) * 2 + 1];
    const float kk = pair_s[t0] * rk0 * rk1, kq01 = pair_s[t0 + 1] * rk0 * rq1;
    const float kq0 = kq_s[t0], kq1 = kq_s[t1];
    const float4 v0 = *reinterpret_cast<const float4*>(x0 + (2 + g) * D + L.col0);
    const float4 v1 = *reinterpret_cast<const float4*>(x1 + (2 + g) * D + L.col0);
    float4 d0, d1;
    d0.x = be0 * (v0.x - al0 * A0.x);
    d0.y = be0 * (v0.y - al0 * A0.y);
    d0.z = be0 * (v0.z - al0 * A0.z);
    d0.w = be0 * (v0.w - al0 * A0.w);
    d1.x = be1 * (v1.x - al1 * (al0 * A1.x + kk * d0.x));
    d1.y = be1 * (v1.y - al1 * (al0 * A1.y + kk * d0.y));
    d1.z = be1 * (v1.z - al1 * (al0 * A1.z + kk * d0.z));
    d1.w = be1 * (v1.w - al1 * (al0 * A1.w + kk * d0.w));
    if (L.rb == 0) {  // warp-uniform: o of t0 on row block 0, of t1 on row block 1
      float4 B0 = vec_of(1);
      B0.x *= rq0; B0.y *= rq0; B0.z *= rq0; B0.w *= rq0;
      float4 o0;
      o0.x = al0 * B0.x + kq0 * d0.x;
      o0.y = al0 * B0.y + kq0 * d0.y;
      o0.z = al0 * B0.z + kq0 * d0.z;
      o0.w = al0 * B0.w + kq0 * d0.w;
      if (L.rs == 0) {
        *reinterpret_cast<float4*>(obuf + t0 * D + L.col0) = o0;
        if (WOA) *reinterpret_cast<float4*>(woa_d + size_t(t0) * p.Hv * D) = d0;
      }
    } else if (L.rb == 1 && has1) {
      float4 B1 = vec_of(3);
      B1.x *= rq1; B1.y *= rq1; B1.z *= rq1; B1.w *= rq1;
      float4 o1;
      o1.x = al1 * (al0 * B1.x + kq01 * d0.x) + kq1 * d1.x;
      o1.y = al1 * (al0 * B1.y + kq01 * d0.y) + kq1 * d1.y;
      o1.z = al1 * (al0 * B1.z + kq01 * d0.z) + kq1 * d1.z;
      o1.w = al1 * (al0 * B1.w + kq01 * d0.w) + kq1 * d1.w;
      if (L.rs == 0) {
        *reinterpret_cast<float4*>(obuf + t1 * D + L.col0) = o1;
        if (WOA) *reinterpret_cast<float4*>(woa_d + size_t(t1) * p.Hv * D) = d1;
      }
    }
    SH* dst0 = WOA ? nullptr : state_dst<D, true, SH>(p, it, tab_item, h, t0);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u == 1 && !has1) break;
      const float al = u ? al1 : al0;
      const float rk = u ? rk1 : rk0;
      const float4 dd = u ? make_float4(d1.x * rk, d1.y * rk, d1.z * rk, d1.w * rk)
                          : make_float4(d0.x * rk, d0.y * rk, d0.z * rk, d0.w * rk);
      float kr[Map::M];
      load_rows((u ? x1 : x0) + D + L.xrow, kr);
#pragma unroll
      for (int m = 0; m < Map::M; ++m) {
        const float ki = kr[m];
        float4 sm = sr_get(S[m]);
        if (!WOA && u == 1) store_sr(dst0 + L.row(m) * D + L.col0, S[m]);  // the state after t0
        sm.x = al * sm.x + ki * dd.x;
        sm.y = al * sm.y + ki * dd.y;
        sm.z = al * sm.z + ki * dd.z;
        sm.w = al * sm.w + ki * dd.w;
        sr_set(S[m], sm);
      }
    }
    if (!WOA) pend = has1 ? state_dst<D, true, SH>(p, it, tab_item, h, t1) : dst0;
  }
  if (!WOA && pend) store_tile<D, NT, SH, SR>(pend, S, L);
  return false;
}

// Thread roles: threads [0, NT) compute (at d = 128, 16 warps for verify and 8 for
// decode).  State tiles stream into a ring of stages by bulk async copies, each landing on
// the stage's full mbarrier.  Decode has a producer warp after the compute threads: its
// lane 0 issues the tiles (a stage is released by one mbarrier arrive per compute warp on
// its empty mbarrier) and each item's raw prologue inputs into a staging block
// (raw_full/raw_empty).  Verify has no producer warp: once every compute thread has a
// head's tile in registers (its first barrier), thread 0 issues the tile STAGES heads
// ahead into the stage it came from -- sixteen warps, so 128 registers a thread.  Compute
// threads synchronise only with named barrier 1.
// Decode has one more warp, which applies the gated RMSNorm to each head's output: the
// compute warps that write a head's o arrive on nfull[slot], the norm warp copies o and z
// to registers and arrives on nfree[slot], so the norm never sits on the chain of heads.
template <int NT, int KMAX>
__host__ __device__ constexpr int rec_threads() {
  return NT + (KMAX == 1 ? 64 : 0);
}
// Decode on fp16 pools holds its tile packed (half the registers) and runs two CTAs per
// SM, so one CTA's per-head chain (reduction, barrier, update) overlaps the other's.
template <int KMAX, typename SH>
__host__ __device__ constexpr int rec_min_blocks() {
  return (KMAX == 1 && sizeof(SH) == 2) ? 2 : 1;
}

template <typename T, int D, int NT, int KMAX, int STAGES, bool VERIFY, typename SH,
          bool WOA = false, bool RAWPF = false>
__global__ void __launch_bounds__(rec_threads<NT, KMAX>(), (rec_min_blocks<KMAX, SH>()))
    gdn_recurrent_kernel(const __grid_constant__ RecParams p) {
  using Map = RecMap<D, NT>;
  using SL = RecSmem<D, NT, KMAX, STAGES, T, SH, RAWPF>;
  using A = Act<T>;
  constexpr int NWC = NT / 32;  // compute warps
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* stage = smem + SL::kStage;
  float* red = reinterpret_cast<float*>(smem + SL::kRed);
  float* obuf = reinterpret_cast<float*>(smem + SL::kObuf);
  float* nw_s = reinterpret_cast<float*>(smem + SL::kNw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SL::kBar);
  uint64_t* empty = full + STAGES;
  uint64_t* raw_full = full + 2 * STAGES;
  uint64_t* raw_empty = raw_full + 1;
  uint64_t* nfull = raw_full + 2;  // [2] (decode)
  uint64_t* nfree = raw_full + 4;  // [2] (decode)
  constexpr int kThreads = rec_threads<NT, KMAX>();
  volatile int32_t* issued_s = reinterpret_cast<volatile int32_t*>(smem + SL::kIssued);
  float* gate = reinterpret_cast<float*>(smem + SL::kGate);
  float* kq_s = reinterpret_cast<float*>(smem + SL::kKq);
  float* pair_s = reinterpret_cast<float*>(smem + SL::kPair);
  float* scl_s = reinterpret_cast<float*>(smem + SL::kScl);
  float* l2_s = reinterpret_cast<float*>(smem + SL::kL2);
  float* xs = reinterpret_cast<float*>(smem + SL::kXs);
  int32_t* slots_s = reinterpret_cast<int32_t*>(smem + SL::kSlots);
  int32_t* valid_s = reinterpret_cast<int32_t*>(smem + SL::kValid);
  uint64_t* tab0_s = reinterpret_cast<uint64_t*>(smem + SL::kTab0);
  uint64_t* tab_item = reinterpret_cast<uint64_t*>(smem + SL::kTabItem);

  const int tid = threadIdx.x;
  const int G = p.G, Hk = p.Hk;
  const int CH = (2 + G) * D;   // conv channels of one item
  const int CHX = CH + G * D;   // plus the z channels
  const int P = gridDim.x, cta = blockIdx.x;
  const int rounds = (p.n_items + P - 1) / P;
  unsigned char* raw = smem + SL::kRaw(G);
  T* raw_cs = reinterpret_cast<T*>(raw + SL::raw_cs(G));
  float* raw_w = reinterpret_cast<float*>(raw + SL::raw_w(G));
  T* raw_x = reinterpret_cast<T*>(raw + SL::raw_x(G));
  T* raw_z = reinterpret_cast<T*>(raw + SL::raw_z(G));

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NWC);
    }
    mbar_init(raw_full, 1);
    mbar_init(raw_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&nfull[b], Map::CB);  // the warps that write o: row block 0
      mbar_init(&nfree[b], 1);
    }
    issued_s[0] = 0;
    issued_s[1] = 0;
    fence_mbar_init();
  }
  for (int j = tid; j < D; j += kThreads) nw_s[j] = p.norm_w[j];  // weights: no kernel writes them
  // Everything below may read what the previous kernel in the stream wrote (slots, tables,
  // states, inputs); once past that, the next kernel may start on SMs this grid leaves.
  pdl_wait();
  pdl_launch_dependents();
  for (int i = tid; i < p.n; i += kThreads) {
    slots_s[i] = p.slots[i];
    valid_s[i] = seq_check<VERIFY>(p, i);
    if (VERIFY) tab0_s[i] = p.tables[i];
  }
  __syncthreads();  // the only CTA-wide barrier: barriers initialised, staging done

  // Global channel of item-local conv channel lc: q | k | v of the G value heads.
  auto global_channel = [&](int kh, int lc) -> int {
    if (lc < D) return kh * D + lc;
    if (lc < 2 * D) return Hk * D + kh * D + (lc - D);
    return 2 * Hk * D + kh * G * D + (lc - 2 * D);
  };
  // Position in a token's row of xs of item-local channel lc: q and k in row-block order.
  auto xpos = [&](int lc) -> int {
    if (lc < D) return qk_pos<D, NT>(lc);
    if (lc < 2 * D) return D + qk_pos<D, NT>(lc - D);
    return lc;
  };
  // First round at or after r whose item can run (rounds if none).
  auto next_valid = [&](int r, Item& it) -> int {
    for (; r < rounds; ++r) {
      const int j = item_at(cta, r, P);
      if (j < p.n_items && item_decode<VERIFY>(p, j, slots_s, valid_s, it) == 0) return r;
    }
    return rounds;
  };

  // Tile of value head g of item `it` into stage s (one thread).
  auto issue_tile = [&](int s, const Item& it, int g) {
    const SH* src = state_src<D, VERIFY, SH>(p, it, tab0_s, it.kh * G + g);
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&full[s], uint32_t(SL::kTile));
    constexpr uint32_t kPiece = SL::kTile >= 16384 ? 16384u : uint32_t(SL::kTile);
#pragma unroll
    for (uint32_t off = 0; off < SL::kTile; off += kPiece)
      bulk_g2s(stage + s * SL::kTile + off,
               reinterpret_cast<const unsigned char*>(src) + off, kPiece, &full[s]);
    issued_s[0] = issued_s[0] + 1;
  };
  // The next (item, head) after (r, g).
  auto advance = [&](int& r, int& g, Item& it) {
    if (++g == G) {
      g = 0;
      r = next_valid(r + 1, it);
    }
  };

  // Verify with kRawPF: the raw inputs of item `it` into the raw block -- its conv state
  // and, per token, its q | k | v raw channel ranges and its z row range -- issued by the
  // lanes of warp 0 (lane t: token t; lanes 16..18: the three conv-state ranges).
  auto issue_raw_verify = [&](const Item& it) {
    static_assert(KMAX <= 16, "one lane per token");
    const int lane = tid & 31, k = it.k;
    // channel range seg: q [0, D), k [D, 2D), v [2D, (2 + G) D)
    auto len = [&](int seg) { return seg < 2 ? D : G * D; };
    if (lane == 0) {
      mbar_arrive_expect_tx(raw_full, uint32_t(CH) * kW * sizeof(T) +
                                          uint32_t(k) * (CH + G * D) * sizeof(T));
      issued_s[1] = issued_s[1] + 1;
    }
    __syncwarp();
    fence_proxy_async_smem();
    if (lane < k) {
      const T* row = reinterpret_cast<const T*>(p.qkv) + size_t(it.row0 + lane) * p.qkv_stride;
#pragma unroll
      for (int seg = 0; seg < 3; ++seg)
        bulk_g2s(raw_x + size_t(lane) * CH + seg * D, row + global_channel(it.kh, seg * D),
                 uint32_t(len(seg)) * sizeof(T), raw_full);
      bulk_g2s(raw_z + size_t(lane) * G * D,
               reinterpret_cast<const T*>(p.z) + size_t(it.row0 + lane) * p.z_stride + it.kh * G * D,
               uint32_t(G) * D * sizeof(T), raw_full);
    } else if (lane >= 16 && lane < 19) {
      const int seg = lane - 16;
      bulk_g2s(raw_cs + size_t(seg) * D * kW,
               reinterpret_cast<const T*>(p.conv_pool) +
                   (size_t(it.slot) * p.conv_dim + global_channel(it.kh, seg * D)) * kW,
               uint32_t(len(seg)) * kW * sizeof(T), raw_full);
    }
  };

  // =========================================================================== norm (decode)
  if (SL::kNormWarp && tid >= NT + 32) {
    using A = Act<T>;
    const int lane = tid & 31, j = lane * 4;
    int hq = 0;
    Item it;
    for (int r = next_valid(0, it); r < rounds; r = next_valid(r + 1, it)) {
      for (int g = 0; g < G; ++g, ++hq) {
        const int b = hq & 1;
        if (!mbar_wait_bounded(&nfull[b], uint32_t(hq >> 1) & 1u)) {
          if (lane == 0) report(p.status, GDN_ERR_TIMEOUT);
          return;
        }
        float4 ov = make_float4(0.f, 0.f, 0.f, 0.f), z4 = ov;
        if (j < D) {
          ov = *reinterpret_cast<const float4*>(obuf + b * D + j);
          z4 = *reinterpret_cast<const float4*>(xs + CH + g * D + j);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&nfree[b]);  // o and z are in registers
        const float ss = warp_sum(ov.x * ov.x + ov.y * ov.y + ov.z * ov.z + ov.w * ov.w);
        if (j < D) {
          const int h = it.kh * G + g;
          const float inv = rsqrtf(ss / float(D) + p.norm_eps);
          const float4 w4 = *reinterpret_cast<const float4*>(nw_s + j);
          float4 yv;
          yv.x = ov.x * inv * w4.x * zgate(z4.x, p.norm_gate);
          yv.y = ov.y * inv * w4.y * zgate(z4.y, p.norm_gate);
          yv.z = ov.z * inv * w4.z * zgate(z4.z, p.norm_gate);
          yv.w = ov.w * inv * w4.w * zgate(z4.w, p.norm_gate);
          A::store4(reinterpret_cast<T*>(p.y) + size_t(it.row0) * p.Hv * D + h * D + j, yv);
          if (p.core_out)
            *reinterpret_cast<float4*>(p.core_out + (size_t(it.row0) * p.Hv + h) * D + j) = ov;
        }
      }
    }
    return;
  }

  // =========================================================================== producer
  if (tid >= NT) {
    if (tid != NT) return;
    // The raw prologue inputs of one item as contiguous blocks: conv state, conv
    // weights and raw qkv of its q | k | v channel ranges, and z of its value heads.
    auto issue_raw = [&](const Item& it) {
      const int k = it.k;
      const int lens[3] = {D, D, G * D};
      const int lstart[3] = {0, D, 2 * D};
      uint32_t total = uint32_t(CH) * kW * sizeof(T) + uint32_t(CH) * kW * 4 +
                       uint32_t(k) * CH * sizeof(T) + uint32_t(k) * G * D * sizeof(T);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(raw_full, total);
      for (int seg = 0; seg < 3; ++seg) {
        const int gc = global_channel(it.kh, lstart[seg]);
        bulk_g2s(reinterpret_cast<unsigned char*>(raw_cs) + size_t(lstart[seg]) * kW * sizeof(T),
                 reinterpret_cast<const T*>(p.conv_pool) + (size_t(it.slot) * p.conv_dim + gc) * kW,
                 uint32_t(lens[seg]) * kW * sizeof(T), raw_full);
        bulk_g2s(raw_w + size_t(lstart[seg]) * kW, p.conv_w + size_t(gc) * kW,
                 uint32_t(lens[seg]) * kW * 4, raw_full);
        for (int t = 0; t < k; ++t)
          bulk_g2s(raw_x + size_t(t) * CH + lstart[seg],
                   reinterpret_cast<const T*>(p.qkv) + size_t(it.row0 + t) * p.qkv_stride + gc,
                   uint32_t(lens[seg]) * sizeof(T), raw_full);
      }
      for (int t = 0; t < k; ++t)
        bulk_g2s(raw_z + size_t(t) * G * D,
                 reinterpret_cast<const T*>(p.z) + size_t(it.row0 + t) * p.z_stride + it.kh * G * D,
                 uint32_t(G) * D * sizeof(T), raw_full);
      issued_s[1] = issued_s[1] + 1;
    };
    Item it_raw, it_i, it_x;
    int r_raw = next_valid(0, it_raw);
    if (SL::kPrefetch && r_raw < rounds) {
      issue_raw(it_raw);
      r_raw = next_valid(r_raw + 1, it_raw);
    }
    int r_i = next_valid(0, it_i), g_i = 0;  // next tile to issue
    for (int s = 0; s < STAGES && r_i < rounds; ++s) {
      issue_tile(s, it_i, g_i);
      advance(r_i, g_i, it_i);
    }
    int r_x = next_valid(0, it_x), g_x = 0;  // tile the consumers take next
    int x = 0, items = 0;
    while (r_x < rounds) {
      if (SL::kPrefetch && g_x == 0) {
        // the consumers read raw inputs of item `items` before its first tile
        if (!mbar_wait_bounded(raw_empty, uint32_t(items) & 1u)) {
          report(p.status, GDN_ERR_TIMEOUT);
          return;
        }
        if (r_raw < rounds) {
          issue_raw(it_raw);
          r_raw = next_valid(r_raw + 1, it_raw);
        }
        ++items;
      }
      if (r_i < rounds) {
        const int s = x % STAGES;
        if (!mbar_wait_bounded(&empty[s], uint32_t(x / STAGES) & 1u)) {
          report(p.status, GDN_ERR_TIMEOUT);
          return;
        }
        issue_tile(s, it_i, g_i);
        advance(r_i, g_i, it_i);
      }
      ++x;
      advance(r_x, g_x, it_x);
    }
    return;
  }

  // =========================================================================== compute
  const Lane<D, NT> L(tid);
  // Bad items are reported once, here.
  if (tid == 0) {
    for (int r = 0; r < rounds; ++r) {
      const int j = item_at(cta, r, P);
      Item it;
      if (j < p.n_items) {
        const int bad = item_decode<VERIFY>(p, j, slots_s, valid_s, it);
        if (bad) report(p.status, bad);
      }
    }
  }
  int q = 0, m = 0;  // tiles and items consumed by this CTA
  // verify: thread 0 issues the tiles, the first STAGES now and then one per finished head
  Item it_i;
  int r_i = rounds, g_i = 0;  // next tile to issue
  if (SL::kPairs && tid == 0) {
    r_i = next_valid(0, it_i);
    for (int s = 0; s < STAGES && r_i < rounds; ++s) {
      issue_tile(s, it_i, g_i);
      advance(r_i, g_i, it_i);
    }
  }
  // A bounded wait gave up: let this CTA's copies still in flight land, then stop.
  auto drain = [&](int q_from) {
    if (tid != 0) return;
    report(p.status, GDN_ERR_TIMEOUT);
    const int nt = issued_s[0], nr = issued_s[1];
    for (int x = q_from; x < nt; ++x)
      mbar_wait_bounded(&full[x % STAGES], uint32_t(x / STAGES) & 1u, kWaitBudgetNs / 8);
    if (nr > m) mbar_wait_bounded(raw_full, uint32_t(m) & 1u, kWaitBudgetNs / 8);
  };
  // Gate logits and per-head gate parameters of an item, loaded ahead into registers
  // (threads < k*G; decode).
  float ra = 0.f, rbv = 0.f, rAl = 0.f, rDt = 0.f;
  auto load_scalars = [&](const Item& it) {
    if (tid < it.k * G) {
      const int t = tid / G, g = tid - t * G;
      const size_t ro = size_t(it.row0 + t) * p.ab_stride + it.kh * G + g;
      ra = A::to_f(reinterpret_cast<const T*>(p.a)[ro]);
      rbv = A::to_f(reinterpret_cast<const T*>(p.b)[ro]);
      rAl = p.A_log[it.kh * G + g];
      rDt = p.dt_bias[it.kh * G + g];
    }
  };

  Item nxt;
  int r_next = next_valid(0, nxt);
  if (SL::kPrefetch && r_next < rounds) load_scalars(nxt);
  if (SL::kRawPF && L.warp == 0 && r_next < rounds) issue_raw_verify(nxt);
  while (r_next < rounds) {
    const Item it = nxt;
    const int k = it.k;
    // write-on-accept (a verify built for it): the stash of this item's sequence
    constexpr bool woa = VERIFY && WOA;
    unsigned char* woa_seq = woa ? p.woa_stash + size_t(it.seq) * p.woa_seq_bytes : nullptr;
    r_next = next_valid(r_next + 1, nxt);

    // ---------------- item prologue: conv + SiLU (+ state update), z, gates, L2 norms
    if constexpr (SL::kPrefetch) {
      const bool ok = mbar_wait_bounded(raw_full, uint32_t(m) & 1u);
      if (tid < k * G) {  // gates from the prefetched logits
        const int t = tid / G, g = tid - t * G;
        float al, be;
        gates_f(ra, rbv, rAl, rDt, &al, &be);
        gate[(t * kMaxG + g) * 2 + 0] = al;
        gate[(t * kMaxG + g) * 2 + 1] = be;
      }
      // the norm warp has taken the previous item's z (and every earlier o) out of xs
      const bool okn =
          q == 0 || mbar_wait_bounded(&nfree[(q - 1) & 1], uint32_t((q - 1) >> 1) & 1u);
      if (named_sync_or(1, NT, !ok || !okn)) {
        drain(q);
        return;
      }
      // One token per item: conv + SiLU of channel lc into xs, the conv state shifted by
      // the new raw input (exact copies); returns the channel's output.
      auto conv_channel = [&](int lc) -> float {
        const float4 w4 = *reinterpret_cast<const float4*>(raw_w + size_t(lc) * kW);
        const float4 s4 = A::load4(raw_cs + size_t(lc) * kW);
        const float x = A::to_f(raw_x[lc]);
        const float y = silu_f(w4.x * s4.y + w4.y * s4.z + w4.z * s4.w + w4.w * x);
        xs[xpos(lc)] = y;
        T* cs = reinterpret_cast<T*>(p.conv_pool) +
                (size_t(it.slot) * p.conv_dim + global_channel(it.kh, lc)) * kW;
        A::store4(cs, make_float4(s4.y, s4.z, s4.w, x));
        return y;
      };
      // Threads below D take q_i and k_i together and sum q.q, k.k and q.k for the L2
      // norms, which the head updates apply as scales (no normalising pass, no barrier
      // for it); the others take the v channels; everyone stages one z channel.
      float sq = 0.f, sk = 0.f, sqk = 0.f;
      for (int i = tid; i < D; i += NT) {
        const float qv = conv_channel(i), kv = conv_channel(D + i);
        sq += qv * qv;
        sk += kv * kv;
        sqk += qv * kv;
      }
      for (int vi = tid - D; vi >= 0 && vi < G * D; vi += NT - D) conv_channel(2 * D + vi);
      for (int zi = tid; zi < G * D; zi += NT) xs[CH + zi] = A::to_f(raw_z[zi]);
      if (L.warp < (D + 31) / 32) {
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        sqk = warp_sum(sqk);
        if (L.lane == 0) {
          l2_s[3 * L.warp + 0] = sq;
          l2_s[3 * L.warp + 1] = sk;
          l2_s[3 * L.warp + 2] = sqk;
        }
      }
      named_sync(1, NT);  // raw block consumed; xs and the sums complete
      if (tid == 0) mbar_arrive(raw_empty);
      if (r_next < rounds) load_scalars(nxt);
    } else {
      // every warp is done with the previous item's xs, gates, tables (and, kRawPF, this
      // item's raw block has landed)
      const bool rok = !SL::kRawPF || mbar_wait_bounded(raw_full, uint32_t(m) & 1u);
      if (named_sync_or(1, NT, !rok)) {
        drain(q);
        return;
      }
      // Every load of the prologue is issued before any of its results is used: the
      // item's table entries and gate inputs, then a thread's channels two at a time.
      static_assert(NT >= KMAX * kMaxG, "one thread per (token, value head) for the gates");
      uint64_t tab_v = 0;
      if (VERIFY && tid < k) tab_v = p.tables[tid * GDN_VERIFY_WY_TABLE_SEQS + it.seq];
      float g_a = 0.f, g_b = 0.f, g_Al = 0.f, g_Dt = 0.f;
      if (tid < k * G) {
        const int t = tid / G, h = it.kh * G + (tid - t * G);
        const size_t ro = size_t(it.row0 + t) * p.ab_stride + h;
        g_a = A::to_f(reinterpret_cast<const T*>(p.a)[ro]);
        g_b = A::to_f(reinterpret_cast<const T*>(p.b)[ro]);
        g_Al = p.A_log[h];
        g_Dt = p.dt_bias[h];
      }
      // Pass 1, loads: a thread's channels two at a time, every raw input of both (z
      // inputs for lc >= CH; else the k raw conv inputs, the conv state -- the last kW raw
      // inputs, oldest first -- and the weights) in registers before any is stored; the raw
      // values are parked in xs.  Pass 2 runs the conv + SiLU of each conv channel over
      // xs in place, each token shifting its raw input into the window; the window after
      // the last token is the new conv state.
      constexpr int kG = KMAX < 8 ? KMAX : 8;  // tokens per round of loads
      auto channel_src = [&](int lc, size_t& stride) -> const T* {
        if (lc >= CH) {
          stride = p.z_stride;
          return reinterpret_cast<const T*>(p.z) + size_t(it.row0) * p.z_stride +
                 it.kh * G * D + (lc - CH);
        }
        stride = p.qkv_stride;
        return reinterpret_cast<const T*>(p.qkv) + size_t(it.row0) * p.qkv_stride +
               global_channel(it.kh, lc);
      };
      auto load_state = [&](int lc, float4& win, float4& w4) {
        if (lc >= CH) return;
        const int gc = global_channel(it.kh, lc);
        win = A::load4(reinterpret_cast<const T*>(p.conv_pool) +
                       (size_t(it.slot) * p.conv_dim + gc) * kW);
        w4 = *reinterpret_cast<const float4*>(p.conv_w + size_t(gc) * kW);
      };
      auto conv_channel = [&](int lc, float4 win, const float4& w4) {
        const int gc = global_channel(it.kh, lc);
        const int xl = xpos(lc);
        for (int t = 0; t < k; ++t) {
          const float x = xs[t * CHX + xl];
          win = make_float4(win.y, win.z, win.w, x);
          if (VERIFY && woa)  // the raw input, an exact copy, for the deferred fold
            reinterpret_cast<T*>(woa_seq + p.woa_raw)[size_t(t) * p.conv_dim + gc] = A::from_f(x);
          xs[t * CHX + xl] = silu_f(w4.x * win.x + w4.y * win.y + w4.z * win.z + w4.w * win.w);
          if (VERIFY && p.conv_inter && t < k - 1) {
            T* ci = reinterpret_cast<T*>(p.conv_inter) +
                    ((size_t(it.seq) * (GDN_VERIFY_WY_TABLES_PER_LAYER - 1) + t) * p.conv_dim + gc) * kW;
            A::store4(ci, win);
          }
        }
        if (!woa)  // exact copies of the last kW raw inputs
          A::store4(reinterpret_cast<T*>(p.conv_pool) + (size_t(it.slot) * p.conv_dim + gc) * kW,
                    win);
      };
      if constexpr (SL::kRawPF) {
        // the raw inputs are in the raw block: z staged as f32; each conv channel's raw
        // column parked in xs, then run with the weights (global, L2) and its conv state
        for (int lc = tid; lc < CHX; lc += NT) {
          if (lc >= CH) {
            for (int t = 0; t < k; ++t) xs[t * CHX + lc] = A::to_f(raw_z[t * G * D + (lc - CH)]);
            continue;
          }
          const float4 w4 =
              *reinterpret_cast<const float4*>(p.conv_w + size_t(global_channel(it.kh, lc)) * kW);
          const float4 win = A::load4(raw_cs + size_t(lc) * kW);
          const int xl = xpos(lc);
          for (int t = 0; t < k; ++t) xs[t * CHX + xl] = A::to_f(raw_x[t * CH + lc]);
          conv_channel(lc, win, w4);
        }
      } else
      for (int lc = tid; lc < CHX; lc += 2 * NT) {
        const int lc1 = lc + NT;
        const bool two = lc1 < CHX;
        float4 wina, w4a, winb, w4b;
        size_t sa, sb = 0;
        const T* pa = channel_src(lc, sa);
        const T* pb = two ? channel_src(lc1, sb) : pa;
        load_state(lc, wina, w4a);
        if (two) load_state(lc1, winb, w4b);
        const int xla = xpos(lc), xlb = xpos(lc1);
        for (int t0 = 0; t0 < k; t0 += kG) {
          float xa[kG], xb[kG];
#pragma unroll
          for (int u = 0; u < kG; ++u)
            if (t0 + u < k) xa[u] = A::to_f(pa[size_t(t0 + u) * sa]);
          if (two) {
#pragma unroll
            for (int u = 0; u < kG; ++u)
              if (t0 + u < k) xb[u] = A::to_f(pb[size_t(t0 + u) * sb]);
          }
#pragma unroll
          for (int u = 0; u < kG; ++u)
            if (t0 + u < k) xs[(t0 + u) * CHX + xla] = xa[u];
          if (two) {
#pragma unroll
            for (int u = 0; u < kG; ++u)
              if (t0 + u < k) xs[(t0 + u) * CHX + xlb] = xb[u];
          }
        }
        if (lc < CH) conv_channel(lc, wina, w4a);
        if (two && lc1 < CH) conv_channel(lc1, winb, w4b);
      }
      if (VERIFY && tid < k) tab_item[tid] = tab_v;
      if (tid < k * G) {
        const int t = tid / G, g = tid - t * G;
        float al, be;
        gates_f(g_a, g_b, g_Al, g_Dt, &al, &be);
        gate[(t * kMaxG + g) * 2 + 0] = al;
        gate[(t * kMaxG + g) * 2 + 1] = be;
        if (VERIFY && woa) reinterpret_cast<float*>(woa_seq + p.woa_alpha)[t * p.Hv + it.kh * G + g] = al;
      }
      named_sync(1, NT);
      // kRawPF: every thread is done with the raw block; the next item's inputs stream in
      // while this item's heads run
      if (SL::kRawPF && L.warp == 0 && r_next < rounds) issue_raw_verify(nxt);
    }
    ++m;
    float rq = 1.f, rk = 1.f, kq1 = 0.f;  // decode: L2 scales of q and k, q_hat.k_hat
    if constexpr (SL::kPrefetch) {
      float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
      for (int w = 0; w < (D + 31) / 32; ++w) {
        sq += l2_s[3 * w];
        sk += l2_s[3 * w + 1];
        sqk += l2_s[3 * w + 2];
      }
      rq = p.q_scale * rsqrtf(sq + p.l2_eps);
      rk = rsqrtf(sk + p.l2_eps);
      kq1 = rq * rk * sqk;
    } else {
      qk_scales_tokens<D, Map::NW>(xs, CHX, k, p.q_scale, p.l2_eps, kq_s, scl_s, pair_s,
                                   L.warp, L.lane);
      named_sync(1, NT);
      if (VERIFY && woa) {  // k, and the normalised k of every token, for the deferred fold
        float* kh_out = reinterpret_cast<float*>(woa_seq + p.woa_khat);
        for (int idx = tid; idx < k * D; idx += NT) {
          const int t = idx / D, i = idx - t * D;
          kh_out[(size_t(t) * p.Hk + it.kh) * D + i] =
              xs[t * CHX + D + qk_pos<D, NT>(i)] * scl_s[2 * t + 1];
        }
        if (tid == 0 && it.kh == 0) *reinterpret_cast<int32_t*>(woa_seq) = k;
      }
    }

    // ---------------- value heads of the item
    for (int g = 0; g < G; ++g) {
      const int h = it.kh * G + g;
      const int s = q % STAGES;
      const int hq = q;  // this head's index in the CTA's sequence of heads
      bool ok = mbar_wait_bounded(&full[s], uint32_t(q / STAGES) & 1u);
      // decode: obuf slot hq & 1 is free once the norm warp has taken head hq - 2
      if (SL::kNormWarp && hq >= 2)
        ok &= mbar_wait_bounded(&nfree[hq & 1], uint32_t((hq - 2) >> 1) & 1u);
      using SR = std::conditional_t<(KMAX == 1 && sizeof(SH) == 2), uint2, float4>;
      SR S[Map::M];
      const SH* tile = reinterpret_cast<const SH*>(stage + size_t(s) * SL::kTile);
#pragma unroll
      for (int mm = 0; mm < Map::M; ++mm) load_sr(S[mm], tile + L.row(mm) * D + L.col0);
      if constexpr (!SL::kPairs) {
        __syncwarp();
        if (L.lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
      }
      ++q;
      if constexpr (SL::kPairs) {
        // stage s is free once every thread has its tile in registers: after the first
        // barrier of the head, thread 0 issues the tile STAGES heads ahead into it
        auto refill = [&]() {
          if (tid == 0 && r_i < rounds) {
            issue_tile(s, it_i, g_i);
            advance(r_i, g_i, it_i);
          }
        };
        if (verify_head<T, D, NT, KMAX, SH, SR, VERIFY && WOA>(p, it, h, g, k, S, L, xs, CHX,
                                                               gate, kq_s, pair_s, scl_s, red,
                                                               obuf,
                                                               tab_item, woa_seq, !ok, refill)) {
          drain(q - 1);
          return;
        }
        named_sync(1, NT);  // obuf complete
        norm_tokens<T, D, Map::NW>(obuf, xs + CH + g * D, CHX, k, it.row0, h, nw_s,
                                   p.norm_eps, p.norm_gate, p.Hv, reinterpret_cast<T*>(p.y),
                                   p.core_out, L.warp, L.lane);
      } else {  // decode: one token; the norm warp takes o from obuf slot hq & 1
        static_assert(KMAX == 1 && !VERIFY, "verify runs in pairs of tokens");
        // slots alternate by head: no barrier separates one head's reduction reads from
        // the next's writes
        if (token_update<D, NT, true, SR, true>(S, L, xs, xs + D, xs + (2 + g) * D, gate[g * 2],
                                          gate[g * 2 + 1], kq1,
                                          red + (hq & 1) * 2 * Map::RB * D,
                                          obuf + (hq & 1) * D, !ok, rq, rk)) {
          drain(q - 1);
          return;
        }
        store_tile<D, NT, SH, SR>(state_dst<D, VERIFY, SH>(p, it, tab_item, h, 0), S, L);
        if (L.rb == 0) {  // this warp wrote part of o
          __syncwarp();
          if (L.lane == 0) mbar_arrive(&nfull[hq & 1]);
        }
      }
    }
  }
  // write-on-accept: the stash holds a verify the fold has not applied yet
  if (VERIFY && WOA && tid == 0) *p.woa_flag = 1u;
}

template <typename T, int D, int NT, int KMAX, int STAGES, bool VERIFY, typename SH,
          bool WOA = false, bool RAWPF = false>
cudaError_t launch_rec(const RecParams& p, cudaStream_t stream) {
  using SL = RecSmem<D, NT, KMAX, STAGES, T, SH, RAWPF>;
  auto kern = gdn_recurrent_kernel<T, D, NT, KMAX, STAGES, VERIFY, SH, WOA, RAWPF>;
  const size_t smem = SL::bytes(p.G);
  if (smem > kMaxSmemPerBlock) return cudaErrorInvalidConfiguration;  // shape not supported
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  // persistent: as many CTAs as fit at once (every CTA's producer and consumers wait only
  // on one another, so a CTA that had to wait for a free SM would still finish)
  int per_sm = 1;
  if (rec_min_blocks<KMAX, SH>() > 1) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, rec_threads<NT, KMAX>(),
                                                      smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    if (per_sm > rec_min_blocks<KMAX, SH>()) per_sm = rec_min_blocks<KMAX, SH>();
  }
  const int cap = sm_count() * per_sm;
  int P = p.n_items < cap ? p.n_items : cap;
  if (KMAX == 1) {
    // decode items all cost the same: the fewest CTAs that still need only as many rounds
    // as a full grid, so the last round is (nearly) full too -- 2048 items on 152 SMs run
    // as 147 CTAs x 14 rounds instead of 152 CTAs with 72 of them busy in the 14th
    // (128-sequence decode 91.6 -> 90.2 us; fp16 pools, 2 CTAs per SM: 59.4 -> 59.1 us)
    const int rounds = (p.n_items + P - 1) / P;
    P = (p.n_items + rounds - 1) / rounds;
  }
  return launch_pdl(kern, dim3(unsigned(P)), dim3(unsigned(rec_threads<NT, KMAX>())), smem, stream,
                    1u, p);
}

// Verify prefetches raw inputs where the raw block fits beside the rest: fp16 pools with
// two stages; f32 pools with one (its tile is issued a whole head ahead, after the
// previous head's first barrier, which measured as enough).
template <typename T, int D, int NT, typename SH>
cudaError_t launch_verify(const RecParams& p, cudaStream_t stream) {
  if constexpr (sizeof(SH) == 2) {
    if (RecSmem<D, NT, GDN_VERIFY_K_MAX, 2, T, SH, true>::bytes(p.G) <= kMaxSmemPerBlock)
      return launch_rec<T, D, NT, GDN_VERIFY_K_MAX, 2, true, SH, false, true>(p, stream);
  } else {
    if (RecSmem<D, NT, GDN_VERIFY_K_MAX, 1, T, SH, true>::bytes(p.G) <= kMaxSmemPerBlock)
      return launch_rec<T, D, NT, GDN_VERIFY_K_MAX, 1, true, SH, false, true>(p, stream);
  }
  return launch_rec<T, D, NT, GDN_VERIFY_K_MAX, 2, true, SH>(p, stream);
}

template <typename T, typename SH>
cudaError_t launch_rec_typed(const RecParams& p, int D, bool verify, cudaStream_t stream) {
  if (D == 128) {
    // Verify keeps sixteen compute warps (k updates per head tile); decode does better
    // with eight, each thread holding sixteen rows of the tile: half as many warps meet at
    // each head's barrier (measured: f32 pools 0.0997 -> 0.0968 ms, fp16 0.0772 -> 0.0735
    // ms per 128-sequence step; verify with eight 0.469 -> 0.523 ms).
    // Decode on fp16 pools: two stages of 32 KiB tiles, so two CTAs share an SM.
    constexpr int kDecodeStages = sizeof(SH) == 2 ? 2 : 3;
    if (verify) return launch_verify<T, 128, 512, SH>(p, stream);
    return launch_rec<T, 128, 256, 1, kDecodeStages, false, SH>(p, stream);
  }
  if (verify) return launch_verify<T, 16, 64, SH>(p, stream);
  return launch_rec<T, 16, 64, 1, 3, false, SH>(p, stream);
}

// The write-on-accept verify (f32 state pools only).
template <typename T>
cudaError_t launch_rec_woa(const RecParams& p, int D, cudaStream_t stream) {
  if (D == 128) {
    if (RecSmem<128, 512, GDN_VERIFY_K_MAX, 1, T, float, true>::bytes(p.G) <= kMaxSmemPerBlock)
      return launch_rec<T, 128, 512, GDN_VERIFY_K_MAX, 1, true, float, true, true>(p, stream);
    return launch_rec<T, 128, 512, GDN_VERIFY_K_MAX, 2, true, float, true>(p, stream);
  }
  return launch_rec<T, 16, 64, GDN_VERIFY_K_MAX, 2, true, float, true>(p, stream);
}

// ======================================================================================
// token-sequential prefill: one CTA per (sequence, value head)
// ======================================================================================
constexpr int kSeg = 16;  // tokens per segment

template <int D, int NT>
struct SeqSmem {
  using Map = RecMap<D, NT>;
  static constexpr int kCHX = 4 * D;  // q | k | v | z of one value head
  static constexpr size_t kRed = 0;
  static constexpr size_t kObuf = kRed + size_t(2) * 2 * Map::RB * D * 4;
  static constexpr size_t kGate = kObuf + size_t(kSeg) * D * 4;
  static constexpr size_t kKq = kGate + kSeg * 2 * 4;
  static constexpr size_t kXs = kKq + kSeg * 4;
  static constexpr size_t kBytes = kXs + size_t(kSeg) * kCHX * 4;
};

template <typename T, int D, int NT>
__global__ void __launch_bounds__(NT, 1)
    gdn_prefill_seq_kernel(const __grid_constant__ PrefillParams p) {
  using Map = RecMap<D, NT>;
  using SL = SeqSmem<D, NT>;
  using A = Act<T>;
  extern __shared__ __align__(128) unsigned char smem[];
  float* red = reinterpret_cast<float*>(smem + SL::kRed);
  float* obuf = reinterpret_cast<float*>(smem + SL::kObuf);
  float* gate = reinterpret_cast<float*>(smem + SL::kGate);
  float* kq_s = reinterpret_cast<float*>(smem + SL::kKq);
  float* xs = reinterpret_cast<float*>(smem + SL::kXs);
  constexpr int CHX = SL::kCHX;

  const int tid = threadIdx.x;
  const Lane<D, NT> L(tid);
  const int seq = blockIdx.x / p.Hv, h = blockIdx.x % p.Hv;
  const int kh = h / p.G;
  const int t_begin = p.cu_seqlens[seq], t_end = p.cu_seqlens[seq + 1];
  const int len = t_end - t_begin;
  const int slot = p.slots[seq];
  const uint64_t hp = p.h_ptrs[seq];
  {
    int bad = 0;
    if (t_begin < 0 || len < 0 || t_end > p.total_tokens || len > p.max_seqlen)
      bad = GDN_ERR_BAD_SEQLENS;
    else if (slot < 0 || slot >= p.n_slots) bad = GDN_ERR_BAD_SLOT;
    else if (hp == 0 || (hp & 15u) != 0) bad = GDN_ERR_BAD_TABLE_ENTRY;
    if (bad) {
      if (tid == 0) report(p.status, bad);
      return;
    }
  }
  float* Hg = reinterpret_cast<float*>(hp) + size_t(h) * D * D;
  float4 S[Map::M];
#pragma unroll
  for (int m = 0; m < Map::M; ++m)
    S[m] = *reinterpret_cast<const float4*>(Hg + L.row(m) * D + L.col0);
  const T* cs = reinterpret_cast<const T*>(p.conv_pool) + size_t(slot) * p.conv_dim * kW;
  const T* qkv = reinterpret_cast<const T*>(p.qkv);

  for (int t0 = 0; t0 < len; t0 += kSeg) {
    const int k = (len - t0) < kSeg ? (len - t0) : kSeg;
    for (int lc = tid; lc < CHX; lc += NT) {
      if (lc >= 3 * D) {  // z
        const T* zp = reinterpret_cast<const T*>(p.z) + size_t(t_begin + t0) * p.z_stride +
                      h * D + (lc - 3 * D);
        for (int t = 0; t < k; ++t) xs[t * CHX + lc] = A::to_f(zp[size_t(t) * p.z_stride]);
        continue;
      }
      int gc;
      if (lc < D) gc = kh * D + lc;
      else if (lc < 2 * D) gc = p.Hk * D + kh * D + (lc - D);
      else gc = 2 * p.Hk * D + h * D + (lc - 2 * D);
      const float4 w4 = *reinterpret_cast<const float4*>(p.conv_w + size_t(gc) * kW);
      // raw input at sequence position pos: pos < 0 reads the conv state (entry kW + pos)
      auto raw = [&](int pos) -> float {
        return pos < 0 ? A::to_f(cs[size_t(gc) * kW + kW + pos])
                       : A::to_f(qkv[size_t(t_begin + pos) * p.qkv_stride + gc]);
      };
      float w0 = raw(t0 - 3), w1 = raw(t0 - 2), w2 = raw(t0 - 1);
      for (int t = 0; t < k; ++t) {
        const float w3 = raw(t0 + t);
        xs[t * CHX + lc] = silu_f(w4.x * w0 + w4.y * w1 + w4.z * w2 + w4.w * w3);
        w0 = w1; w1 = w2; w2 = w3;
      }
    }
    for (int t = tid; t < k; t += NT) {
      const size_t ro = size_t(t_begin + t0 + t) * p.ab_stride + h;
      float al, be;
      gates_f(A::to_f(reinterpret_cast<const T*>(p.a)[ro]),
              A::to_f(reinterpret_cast<const T*>(p.b)[ro]), p.A_log[h], p.dt_bias[h], &al, &be);
      gate[2 * t] = al;
      gate[2 * t + 1] = be;
    }
    __syncthreads();
    l2norm_tokens<D, Map::NW>(xs, CHX, k, p.q_scale, p.l2_eps, kq_s, L.warp, L.lane);
    __syncthreads();
    for (int t = 0; t < k; ++t) {
      const float* xq = xs + t * CHX;
      token_update<D, NT>(S, L, xq, xq + D, xq + 2 * D, gate[2 * t], gate[2 * t + 1], kq_s[t],
                          red + (t & 1) * 2 * Map::RB * D, obuf + t * D);
    }
    __syncthreads();
    norm_tokens<T, D, Map::NW>(obuf, xs + 3 * D, CHX, k, t_begin + t0, h, p.norm_w, p.norm_eps,
                               p.norm_gate, p.Hv, reinterpret_cast<T*>(p.y), p.core_out, L.warp,
                               L.lane);
    __syncthreads();  // xs, obuf and gate are rewritten by the next segment
  }
  store_tile<D, NT>(Hg, S, L);
}

template <typename T, int D, int NT>
cudaError_t launch_seq(const PrefillParams& p, cudaStream_t stream) {
  using SL = SeqSmem<D, NT>;
  auto kern = gdn_prefill_seq_kernel<T, D, NT>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SL::kBytes));
  if (e != cudaSuccess) return e;
  kern<<<p.n * p.Hv, NT, SL::kBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(const RecParams& p, int dtype, int D, bool verify, bool h16,
                             cudaStream_t stream) {
  if (verify && p.woa_stash) {
    if (h16) return cudaErrorInvalidConfiguration;  // write-on-accept keeps f32 pools only
    return dtype == GDN_DTYPE_BF16 ? launch_rec_woa<__nv_bfloat16>(p, D, stream)
                                   : launch_rec_woa<float>(p, D, stream);
  }
  if (h16) {
    if (dtype == GDN_DTYPE_BF16)
      return launch_rec_typed<__nv_bfloat16, __half>(p, D, verify, stream);
    return launch_rec_typed<float, __half>(p, D, verify, stream);
  }
  if (dtype == GDN_DTYPE_BF16) return launch_rec_typed<__nv_bfloat16, float>(p, D, verify, stream);
  return launch_rec_typed<float, float>(p, D, verify, stream);
}

cudaError_t launch_prefill_sequential(const PrefillParams& p, int dtype, cudaStream_t stream) {
  if (dtype == GDN_DTYPE_BF16) {
    if (p.D == 128) return launch_seq<__nv_bfloat16, 128, 512>(p, stream);
    return launch_seq<__nv_bfloat16, 16, 64>(p, stream);
  }
  if (p.D == 128) return launch_seq<float, 128, 512>(p, stream);
  return launch_seq<float, 16, 64>(p, stream);
}

}  // namespace gdn
