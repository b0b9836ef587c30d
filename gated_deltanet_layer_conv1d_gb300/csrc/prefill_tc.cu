// prefill_tc.cu -- chunked (WY / UT-transform) prefill of the gated delta rule on the
// 5th-generation tensor cores (tcgen05, accumulators in TMEM), d_k = d_v = 128, chunk 64.
//
// The method (layer_struct.rs, the FLA chunked prefill: gdn_prefill_fla_recompute_wu_k ->
// the chunk_delta_h state spine -> gdn_prefill_fla_chunk_fwd_o_k).  Inside a chunk of L
// tokens, with g_r = sum_{s<=r} log alpha_s:
//   A   = strict_lower(beta_r (k_r . k_s) e^{g_r - g_s}),   T = (I + A)^{-1}
//   W   = T diag(beta e^g) K,   U = T diag(beta) V,   Delta = U - W H0      (H0 = S0^T)
//   O   = diag(e^g) Q H0 + P Delta,    P  = lower_incl(Q K^T e^{g_r - g_s})
//   H_L = e^{g_L} H0 + K~^T Delta,     K~ = diag(e^{g_L - g}) K
//
// Two kernels follow the pre-pass (which leaves the normalised q, k, v tiles and the gates
// in the workspace):
//
// gdn_prefill_chunk_kernel -- everything that does not depend on the state, for every
//   (chunk, value head) at once:
//     MMA0  [K;Q] K^T            (M 128 = 64 keys + 64 queries, N 64, K 128) -> A and P
//     T = (I + A)^{-1} on CUDA cores (16 x 16 diagonal blocks, then the blocks below them
//       level by level with warp-level TF32 MMAs)
//     MMA_W W^T = K^T (T diag(beta e^g))^T,  MMA_U U^T = V^T (T diag(beta))^T  (N 64, K 64)
//   and writes W, K~, P, g and U to the workspace.
// gdn_prefill_spine_kernel<NCOL> -- the state recurrence, chunk after chunk, for one
//   (sequence, value head) and NCOL of its 128 value columns (columns of H never mix, so
//   the 128 / NCOL slices run in separate CTAs).  Per chunk, two MMAs:
//     MMA_a [Q;W] H0             (M 128 = 64 query rows + 64 W rows, N NCOL, K 128)
//     MMA_b K~^T Delta and [P;*] Delta  (M 128, N NCOL, K 64; rows past P are ignored)
//   with Delta and the new H written back between them as fp16 MN-major operands (each
//   thread stores its own row, 16 bytes at a time).  The next chunk's operands arrive by
//   bulk copy into the other of two buffers meanwhile.  With whole rows (NCOL = 128) the
//   spine applies the gated RMSNorm to O itself and writes y; with two column slices it
//   writes O (fp16 unless the caller asked for the f32 core output), counts the chunks it
//   has stored, and the launch's remaining CTAs (a cooperative launch over the SMs the
//   chains leave free) apply the gated norm to each chunk behind the chains.
//
// Operands are fp16 (kind::f16, f32 accumulation): every operand here is bounded
// (normalised q and k, O(1) v, T, P, Delta and state), and fp16's 11-bit significand
// keeps the rounding of the inputs and of T, P and Delta eight times below bf16's.  The
// state itself stays f32 in registers from the first chunk to the last.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "prefill_layout.cuh"
#include "tcgen05.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kD = 128;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint4 pack8_h(const float* v) {
  uint4 u;
  __half2 a = __floats2half2_rn(v[0], v[1]), b = __floats2half2_rn(v[2], v[3]);
  __half2 c = __floats2half2_rn(v[4], v[5]), d = __floats2half2_rn(v[6], v[7]);
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  u.z = *reinterpret_cast<uint32_t*>(&c);
  u.w = *reinterpret_cast<uint32_t*>(&d);
  return u;
}

// Warp-level TF32 MMA (m16n8k8, row-major A, column-major B, f32 accumulate) for the small
// 16 x 16 block products of the triangular inverse.  Fragment of lane l (g = l / 4,
// t = l % 4): A (16 x 8) a0 (g, t), a1 (g + 8, t), a2 (g, t + 4), a3 (g + 8, t + 4);
// B (8 x 8) b0 (t, g), b1 (t + 4, g); D (16 x 8) d0 (g, 2t), d1 (g, 2t + 1), d2 (g + 8, 2t),
// d3 (g + 8, 2t + 1).
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Both kernels check their sequence's token range and state pointer the same way.
__device__ __forceinline__ int check_seq(const PrefillParams& p, int t_begin, int t_end,
                                         uint64_t hp) {
  const int len = t_end - t_begin;
  if (t_begin < 0 || len < 0 || t_end > p.total_tokens || len > p.max_seqlen)
    return GDN_ERR_BAD_SEQLENS;
  if (hp == 0 || (hp & 15u) != 0) return GDN_ERR_BAD_TABLE_ENTRY;
  return 0;
}

// ------------------------------------------------------------------------------------
// Chunk kernel: one CTA of 256 threads per (chunk slot, value head).

constexpr int kPrepThreads = 256;

struct PrepSmem {
  static constexpr uint32_t kAQK = 0;        // [128][128] f16: rows 0-63 k_hat, 64-127 q_hat;
                                             // later K~ in the k rows, P in q block 0 and,
                                             // once P is out, v in the two q blocks
  static constexpr uint32_t kP = 8192;       // [64][64] f16 P (q block 0, dead after MMA0)
  static constexpr uint32_t kV = 8192;       // v, MN-major A of MMA_U: column blocks at
                                             // 8192 and 24576 (16384 apart)
  static constexpr int kAS = 65;             // row stride of A: odd, so column writes from
                                             // 32 lanes hit 32 banks
  static constexpr uint32_t kAm = 32768;     // [64][65] f32 A
  static constexpr uint32_t kTw = kAm;       // [64][64] f16 T diag(beta e^g) (A is dead)
  static constexpr uint32_t kTu = kAm + 8192;  // [64][64] f16 T diag(beta)
  static constexpr int kTS = 72;             // row stride of T: the TF32 fragment reads of
                                             // 8 rows x 4 columns hit distinct banks
  static constexpr uint32_t kTf = 50176;     // [64][72] f32 T
  static constexpr uint32_t kWi = kTf;       // [64][128] f16 W image (T is dead)
  static constexpr uint32_t kY = 68608;      // [3][16][16] f32 scratch of the inverse
  static constexpr uint32_t kGate = 71680;   // [2][64] f32 log(alpha), beta (bulk copied)
  static constexpr uint32_t kG = 72192;      // [64] f32 cumulative log2 decay g
  static constexpr uint32_t kB = 72448;      // [64] f32 beta (0 past the chunk end)
  static constexpr uint32_t kMisc = 72704;   // bars, tmem slot, scan carry
  static constexpr uint32_t kBytes = 72832;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // room to align the base to 1024
};
static_assert(PrepSmem::kAm + 64 * PrepSmem::kAS * 4 <= PrepSmem::kTf, "A fits");
static_assert(PrepSmem::kTf + 64 * PrepSmem::kTS * 4 <= PrepSmem::kY, "T fits");
static_assert(PrepSmem::kY + 3 * 256 * 4 <= PrepSmem::kGate, "inverse scratch fits");

// TMEM columns of the chunk kernel (128 allocated, so three CTAs share an SM); MMA_W
// reuses MMA0's columns, which are read before it is issued.
constexpr uint32_t kT0 = 0;     // MMA0: [K;Q] K^T   (64 cols)
constexpr uint32_t kTW = 0;     // MMA_W: W^T        (64)
constexpr uint32_t kTU = 64;    // MMA_U: U^T        (64)
constexpr uint32_t kPrepTmem = 128;

__global__ void __launch_bounds__(kPrepThreads, 3)
    gdn_prefill_chunk_kernel(const __grid_constant__ PrefillParams p) {
  using S = PrepSmem;
  // the two-slice spine's progress counters start from zero on every call
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < 2 * p.n * p.Hv; i += blockDim.x) p.counts[i * kCountStride] = 0;
  const int cs = blockIdx.x / p.Hv, h = blockIdx.x % p.Hv, kh = h / p.G;
  // The sequence that owns chunk slot cs: the last s with base(s) <= cs.
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
  const int t_begin = p.cu_seqlens[seq], t_end = p.cu_seqlens[seq + 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    const int bad = check_seq(p, t_begin, t_end, p.h_ptrs[seq]);
    if (bad) {
      if (tid == 0) report(p.status, bad);
      return;
    }
  }
  const size_t slot0 = PrefillLayout::base(t_begin, seq);
  const int len = t_end - t_begin, nc = (len + kC - 1) / kC;
  if (size_t(cs) < slot0 || size_t(cs) - slot0 >= size_t(nc)) return;  // an unused slot
  const int c = int(size_t(cs) - slot0);
  const int L = (len - c * kC) < kC ? (len - c * kC) : kC;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  float* Am = reinterpret_cast<float*>(sm + S::kAm);
  float* Tf = reinterpret_cast<float*>(sm + S::kTf);
  float* Ys = reinterpret_cast<float*>(sm + S::kY);
  float* gate = reinterpret_cast<float*>(sm + S::kGate);
  float* G_s = reinterpret_cast<float*>(sm + S::kG);
  float* B_s = reinterpret_cast<float*>(sm + S::kB);
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(sm + S::kMisc);
  uint64_t* bar_mma = bar_load + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  float* carry = reinterpret_cast<float*>(tslot + 1);

  const PrefillLayout lay{p.Hk, p.Hv};
  unsigned char* ws = reinterpret_cast<unsigned char*>(p.workspace);

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, kPrepTmem);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  if (tid == 0) {
    const unsigned char* kimg = ws + lay.qk(cs, kh, 0);
    const unsigned char* qimg = ws + lay.qk(cs, kh, 1);
    mbar_arrive_expect_tx(bar_load, 2u * 16384u + 512u);
    bulk_g2s(sm + S::kAQK, kimg, 8192, bar_load);
    bulk_g2s(sm + S::kAQK + 16384, kimg + 8192, 8192, bar_load);
    bulk_g2s(sm + S::kAQK + 8192, qimg, 8192, bar_load);
    bulk_g2s(sm + S::kAQK + 24576, qimg + 8192, 8192, bar_load);
    bulk_g2s(gate, ws + lay.gate(cs, h), 512, bar_load);
  }
  const int q4 = warp & 3, half = warp >> 2;
  const uint32_t tl = uint32_t(32 * q4) << 16;  // this warp's TMEM lane quarter
  bool bad = !mbar_wait_bounded(bar_load, 0);
  uint32_t mma_phase = 0;
  auto mma_wait = [&]() {
    bad |= !mbar_wait_bounded(bar_mma, mma_phase);
    mma_phase ^= 1u;
    tc::fence_after_sync();
  };
  auto sync_or_stop = [&]() -> bool {
    tc::fence_before_sync();
    const bool stop = __syncthreads_or(bad) != 0;
    tc::fence_after_sync();
    return stop;
  };

  bool v_issued = false;  // (thread 128)
  do {
    // ---- rows past the end of the sequence are zero; decay prefix sums
    if (L < kC) {
      const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
      for (int idx = tid; idx < (kC - L) * 16; idx += kPrepThreads) {
        const int row = L + idx / 16, ch = idx % 16, blk = ch / 8, c16 = ch % 8;
        *reinterpret_cast<uint4*>(sm + S::kAQK + blk * 16384 + row * 128 + c16 * 16) = zero;
        *reinterpret_cast<uint4*>(sm + S::kAQK + blk * 16384 + (kC + row) * 128 + c16 * 16) =
            zero;
      }
    }
    if (tid < kC) {
      // g in log2 units, so each decay factor below is one exp2; rows past the end of the
      // sequence add nothing, so they repeat g_{L-1}
      float v = tid < L ? gate[tid] * kLog2e : 0.f;
      const float be = tid < L ? gate[kC + tid] : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
      }
      if (tid == 31) carry[0] = v;
      named_sync(2, kC);
      if (tid >= 32) v += carry[0];
      G_s[tid] = v;
      B_s[tid] = be;
      reinterpret_cast<float*>(ws + lay.g(cs, h))[tid] = v;
    }
    fence_proxy_async_smem();
    if (sync_or_stop()) break;
    const float gL = G_s[kC - 1];

    // ---- MMA0: [K;Q] K^T
    if (tid == 0) {
#pragma unroll
      for (int k0 = 0; k0 < kD; k0 += 16)
        tc::mma_f16(tmem + kT0, tc::desc_at(sb + S::kAQK, 128, k0),
                     tc::desc_at(sb + S::kAQK, 128, k0), tc::idesc_f16(128, 64), k0 > 0);
      tc::commit(bar_mma);
    }
    mma_wait();

    // ---- A (f32) from the K K^T rows, P (fp16, over q block 0) from the Q K^T rows
    {
      float v[32];
      tc::ld32(tmem + tl + kT0 + 32 * half, v);
      const int row = 32 * q4 + lane;
      if (row < kC) {
        const int r = row;
        const float gr = G_s[r], br = B_s[r];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int s = 32 * half + u;
          Am[r * S::kAS + s] = (s < r && r < L) ? br * v[u] * exp2_fast(gr - G_s[s]) : 0.f;
        }
      } else {
        const int r = row - kC;
        const float gr = G_s[r];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int s = 32 * half + u;
          v[u] = (s <= r && r < L) ? v[u] * exp2_fast(gr - G_s[s]) : 0.f;
        }
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8)
          *reinterpret_cast<uint4*>(sm + S::kP + tc::sw128_offset(64, r, 32 * half + 8 * c8)) =
              pack8_h(v + 8 * c8);
      }
    }
    fence_proxy_async_smem();
    if (sync_or_stop()) break;
    // P goes out; once it has been read, v comes into the q blocks (MMA0 is done with them)
    if (tid == 128) {
      v_issued = true;
      bulk_s2g(ws + lay.p(cs, h), sm + S::kP, 8192);
      bulk_commit();
      bulk_wait_read();
      mbar_arrive_expect_tx(bar_load, 16384u);
      bulk_g2s(sm + S::kV, ws + lay.v(cs, h), 8192, bar_load);
      bulk_g2s(sm + S::kV + 16384, ws + lay.v(cs, h) + 8192, 8192, bar_load);
    }

    // ---- T = (I + A)^{-1}: diagonal 16 x 16 blocks, then the blocks below them
    if (warp < 4) {
      if (lane < 16) {
        const int b0 = 16 * warp;
        float X[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
          float acc0 = (rr == lane) ? 1.f : 0.f, acc1 = 0.f;
#pragma unroll
          for (int ss = 0; ss + 1 < rr; ss += 2) {
            acc0 -= Am[(b0 + rr) * S::kAS + b0 + ss] * X[ss];
            acc1 -= Am[(b0 + rr) * S::kAS + b0 + ss + 1] * X[ss + 1];
          }
          if (rr & 1) acc0 -= Am[(b0 + rr) * S::kAS + b0 + rr - 1] * X[rr - 1];
          X[rr] = acc0 + acc1;
        }
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) Tf[(b0 + rr) * S::kTS + b0 + lane] = X[rr];
      }
    } else {
      // blocks above the diagonal are zero
      for (int e = tid - 128; e < 6 * 256; e += 128) {
        const int blk = e / 256, a = (e % 256) / 16, bb = e % 16;
        const int I = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int J = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        Tf[(16 * I + a) * S::kTS + 16 * J + bb] = 0.f;
      }
    }
    __syncthreads();
    // Block (I, J = I - d) of T: T_IJ = -T_II sum_{K=J}^{I-1} A_IK T_KJ, one warp per block,
    // as TF32 warp MMAs over 16 x 8 output halves.
    for (int d = 1; d < 4; ++d) {
      if (warp < 4 - d) {
        const int I = d + warp, J = I - d;
        const int g = lane >> 2, t = lane & 3;
        float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        for (int k0 = 16 * J; k0 < 16 * I; k0 += 8) {
          const float* ar = Am + (16 * I + g) * S::kAS + k0 + t;
          const uint32_t a[4] = {to_tf32(ar[0]), to_tf32(ar[8 * S::kAS]), to_tf32(ar[4]),
                                 to_tf32(ar[8 * S::kAS + 4])};
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const float* br = Tf + (k0 + t) * S::kTS + 16 * J + 8 * nt + g;
            mma_tf32(y[nt], a, to_tf32(br[0]), to_tf32(br[4 * S::kTS]));
          }
        }
        float* Yw = Ys + warp * 256;  // Y of this block, [16][16]
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          Yw[g * 16 + 8 * nt + 2 * t] = y[nt][0];
          Yw[g * 16 + 8 * nt + 2 * t + 1] = y[nt][1];
          Yw[(g + 8) * 16 + 8 * nt + 2 * t] = y[nt][2];
          Yw[(g + 8) * 16 + 8 * nt + 2 * t + 1] = y[nt][3];
        }
        __syncwarp();
        float tt[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int k0 = 0; k0 < 16; k0 += 8) {
          const float* ar = Tf + (16 * I + g) * S::kTS + 16 * I + k0 + t;
          const uint32_t a[4] = {to_tf32(ar[0]), to_tf32(ar[8 * S::kTS]), to_tf32(ar[4]),
                                 to_tf32(ar[8 * S::kTS + 4])};
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
            mma_tf32(tt[nt], a, to_tf32(Yw[(k0 + t) * 16 + 8 * nt + g]),
                     to_tf32(Yw[(k0 + t + 4) * 16 + 8 * nt + g]));
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          float* tr = Tf + (16 * I + g) * S::kTS + 16 * J + 8 * nt + 2 * t;
          tr[0] = -tt[nt][0];
          tr[1] = -tt[nt][1];
          tr[8 * S::kTS] = -tt[nt][2];
          tr[8 * S::kTS + 1] = -tt[nt][3];
        }
      }
      __syncthreads();
    }
    // v has arrived; its rows past the end of the sequence are zero
    bad |= !mbar_wait_bounded(bar_load, 1);
    if (L < kC) {
      const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
      for (int idx = tid; idx < (kC - L) * 16; idx += kPrepThreads) {
        const int row = L + idx / 16, ch = idx % 16, blk = ch / 8, c16 = ch % 8;
        *reinterpret_cast<uint4*>(sm + S::kV + blk * 16384 + row * 128 + c16 * 16) = zero;
      }
    }
    // T diag(beta e^g) and T diag(beta), fp16, [r][s] (over A, which is dead now)
    for (int cid = tid; cid < kC * 8; cid += kPrepThreads) {
      const int r = cid / 8, s0 = (cid % 8) * 8;
      float tw[8], tu[8];
      const float4 t0 = *reinterpret_cast<const float4*>(Tf + r * S::kTS + s0);
      const float4 t1 = *reinterpret_cast<const float4*>(Tf + r * S::kTS + s0 + 4);
      const float tv8[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        tu[u] = tv8[u] * B_s[s0 + u];
        tw[u] = tu[u] * exp2_fast(G_s[s0 + u]);
      }
      *reinterpret_cast<uint4*>(sm + S::kTw + tc::sw128_offset(64, r, s0)) = pack8_h(tw);
      *reinterpret_cast<uint4*>(sm + S::kTu + tc::sw128_offset(64, r, s0)) = pack8_h(tu);
    }
    fence_proxy_async_smem();
    if (sync_or_stop()) break;

    // ---- W^T = K^T (T diag(beta e^g))^T, U^T = V^T (T diag(beta))^T
    if (tid == 0) {
#pragma unroll
      for (int s0 = 0; s0 < kC; s0 += 16) {
        tc::mma_f16(tmem + kTW, tc::desc_mn_sw128(sb + S::kAQK + s0 * 128, 16384),
                     tc::desc_at(sb + S::kTw, 64, s0), tc::idesc_f16(128, 64, true, false),
                     s0 > 0);
        tc::mma_f16(tmem + kTU, tc::desc_mn_sw128(sb + S::kV + s0 * 128, 16384),
                     tc::desc_at(sb + S::kTu, 64, s0), tc::idesc_f16(128, 64, true, false),
                     s0 > 0);
      }
      tc::commit(bar_mma);
    }
    mma_wait();
    if (sync_or_stop()) break;

    // ---- W [r][i] (fp16 image, over T) from W^T (lane i); U [r][j] (f32, straight to the
    // workspace) from U^T (lane j); K~ in place of the k rows, which no MMA reads any more
    {
      const int i = 32 * q4 + lane;
      float v[32];
      tc::ld32(tmem + tl + kTW + 32 * half, v);
#pragma unroll
      for (int u = 0; u < 32; ++u)
        *reinterpret_cast<__half*>(sm + S::kWi + tc::sw128_offset(64, 32 * half + u, i)) =
            __float2half_rn(v[u]);
      tc::ld32(tmem + tl + kTU + 32 * half, v);
      // U (fp16) column group q4 (= i / 32), row r, column i % 32 = lane: 16-byte piece
      // lane / 8 of the row at piece (lane / 8) ^ ((r / 2) % 4), so that the spine's
      // row-per-thread reads of a piece are free of bank conflicts
      __half* Ug = reinterpret_cast<__half*>(ws + lay.u(cs, h)) + q4 * (kC * 32);
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const int r = 32 * half + u;
        Ug[r * 32 + (((lane >> 3) ^ ((r >> 1) & 3)) << 3) + (lane & 7)] = __float2half_rn(v[u]);
      }
    }
    for (int idx = tid; idx < kC * 16; idx += kPrepThreads) {
      const int blk = idx >> 9, row = (idx >> 3) & 63, c16 = idx & 7;
      uint4* q = reinterpret_cast<uint4*>(sm + S::kAQK + blk * 16384 + row * 128 + c16 * 16);
      const float sc = exp2_fast(gL - G_s[row]);
      const uint4 raw = *q;
      const __half2* hv = reinterpret_cast<const __half2*>(&raw);
      float f[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __half22float2(hv[e]);
        f[2 * e] = x.x * sc;
        f[2 * e + 1] = x.y * sc;
      }
      *q = pack8_h(f);
    }
    fence_proxy_async_smem();
    if (sync_or_stop()) break;
    if (tid == 0) {
      bulk_s2g(ws + lay.w(cs, h), sm + S::kWi, 16384);
      bulk_s2g(ws + lay.kt(cs, h), sm + S::kAQK, 8192);
      bulk_s2g(ws + lay.kt(cs, h) + 8192, sm + S::kAQK + 16384, 8192);
      bulk_commit();
    }
  } while (false);

  if (tid == 0) {
    bulk_wait_read();  // the shared memory the stores read is released with the CTA
    if (bad) report(p.status, GDN_ERR_TIMEOUT);
  }
  // after a stop, the v copy still lands before the shared memory is released
  if (tid == 128 && v_issued) mbar_wait_bounded(bar_load, 1);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, kPrepTmem);
}

// ------------------------------------------------------------------------------------
// State spine: one CTA of 4 * NCOL threads per (sequence, value head, column slice).
// Warp w serves TMEM lanes 32 (w % 4) .. + 31 and the 32 columns 32 (w / 4) .. + 31 of
// its slice; lane l of it owns H row i = 32 (w % 4) + l over those columns.

template <int NCOL>
struct SpineSmem {
  // One chunk's operands (two such buffers):
  static constexpr uint32_t kQW = 0;       // [128][128] f16: rows 0-63 q_hat, 64-127 W
  static constexpr uint32_t kP = 32768;    // [64][64] f16 P; an M = 128 operand starting
                                           // here reads its rows 64-127 from K~ (unused)
  static constexpr uint32_t kKt = 40960;   // [64][128] f16 K~ (MN-major A of K~^T Delta)
  static constexpr uint32_t kGd = 57344;   // [64] f32 g
  // The two-slice spine also keeps U in each buffer (one chunk ahead, like the rest); the
  // whole-row spine has room for one U buffer only, refilled after each chunk's read.
  static constexpr bool kUInStage = NCOL == 64;
  static constexpr uint32_t kUst = 58368;  // [NCOL / 32][64][32] fp16 U (swizzled), kUInStage
  static constexpr uint32_t kStage = kUInStage ? kUst + NCOL * 128 : 58368;
  static constexpr uint32_t kTx = 4 * 8192 + 8192 + 16384 + 256 + (kUInStage ? NCOL * 128 : 0);
  static constexpr uint32_t kHT = 2 * kStage;          // [128][NCOL] f16 H slice (MN-major B)
  static constexpr uint32_t kDT = kHT + NCOL * 256;    // [64][NCOL] f16 Delta (MN-major B)
  static constexpr uint32_t kUs = kDT + NCOL * 128;    // the single U buffer, !kUInStage
  // Gated norm in the spine (whole rows, NCOL = 128 only):
  static constexpr bool kNorm = NCOL == 128;
  // Two column slices: O goes out as it is, counted per chunk, and the launch's last CTAs
  // apply the norm.
  static constexpr bool kCounted = NCOL == 64;
  static constexpr uint32_t kZ = kUs + (kUInStage ? 0 : NCOL * 128);  // [64][128] bf16 z rows
  static constexpr uint32_t kRed = kZ + (kNorm ? 16384 : 0);   // [4][64] f32 partial sums
  static constexpr uint32_t kNW = kRed + (kNorm ? 1024 : 0);   // [128] f32 norm weight
  static constexpr uint32_t kMisc = kNW + (kNorm ? 512 : 0);   // bars, tmem slot
  static constexpr uint32_t kBytes = kMisc + 128;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemCols = NCOL == 64 ? 256 : 512;
  static_assert(NCOL == 64 || NCOL == 128, "whole 64-column blocks of the MN-major operands");
};

constexpr int kOrderMax = 512;  // sequences the spine orders by length (more: call order)
constexpr int kCountStop = 1 << 30;  // counted by a chain that stopped early

// A column slice's count of stored chunks of O: written after a CTA barrier that follows
// the stores, behind a device-scope fence (so it releases every thread's stores); read
// relaxed and followed by a fence before the reader's CTA barrier.
__device__ __forceinline__ void publish_count(int32_t* cnt, int v) {
  __threadfence();
  asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(cnt), "r"(v) : "memory");
}
__device__ __forceinline__ int load_count(const int32_t* cnt) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
  return v;
}

// The gated RMSNorm behind the two-slice spine, y = O / rms(O) * w * gate(z), run by the
// launch's last CTAs on the SMs the chains leave free (the launch is cooperative, so the
// chains they wait for are resident; it has at least two such CTAs per head).  Units of
// work are (sequence, head, 8-row part of a chunk); norm CTA k follows units k, k + nr, ...
// (at most kNormUnits of them) chunk by chunk.  Each round waits until both column slices
// of every one of its heads have stored past the next chunk, then normalises every chunk
// that has become ready, so a CTA that falls behind catches up in one round.  Warp w of NW
// takes rows w, w + NW, ... of the round, eight at a time, lane l columns 4l .. 4l + 3.
constexpr int kNormUnits = 4;
constexpr int kNormRows = 8;  // rows of a chunk per unit

__device__ void spine_norm_ctas(const PrefillParams& p, int k, int nr) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  constexpr int kParts = kC / kNormRows;
  const int units = p.n * p.Hv * kParts;
  const int nwu = k < units ? (units - 1 - k) / nr + 1 : 0;
  if (nwu == 0 || nwu > kNormUnits) return;  // the launch keeps nwu <= kNormUnits
  __shared__ int uh_s[kNormUnits], r0_s[kNormUnits], tb_s[kNormUnits], len_s[kNormUnits],
      upto_s;
  if (tid < nwu) {
    const int w = k + tid * nr, u = w / kParts, seq = u / p.Hv;
    const int tb = p.cu_seqlens[seq], te = p.cu_seqlens[seq + 1];
    uh_s[tid] = u;                         // (sequence, head)
    r0_s[tid] = (w % kParts) * kNormRows;  // first row of the part within a chunk
    tb_s[tid] = tb;
    // the chains skip what this skips: a bad range or state pointer
    len_s[tid] = check_seq(p, tb, te, p.h_ptrs[seq]) != 0 ? 0 : te - tb;
  }
  __syncthreads();
  int ncmax = 0;
  for (int i = 0; i < nwu; ++i) ncmax = max(ncmax, (len_s[i] + kC - 1) / kC);
  // floor(q / nwu) as (q * ceil(2^32 / nwu)) >> 32, exact for q < 2^32 / nwu
  const uint64_t inv_nwu = (0x100000000ull + nwu - 1) / nwu;
  const float4 w4 = *reinterpret_cast<const float4*>(p.norm_w + 4 * lane);
  const __nv_bfloat16* zg = reinterpret_cast<const __nv_bfloat16*>(p.z);
  __nv_bfloat16* yg = reinterpret_cast<__nv_bfloat16*>(p.y);
  int c0 = 0;
  while (c0 < ncmax) {
    if (tid == 0) {
      // chunks below `ready` are stored in both slices of every head still running
      int ready = 0;
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
        ready = ncmax;
        for (int i = 0; i < nwu; ++i) {
          const int nc = (len_s[i] + kC - 1) / kC;
          if (nc <= c0) continue;
          const int32_t* cnt = p.counts + 2 * uh_s[i] * kCountStride;
          const int v = min(load_count(cnt), load_count(cnt + kCountStride));
          if (v < nc) ready = min(ready, v);
        }
        if (ready > c0) break;
        if (globaltimer_ns() - t0 > kWaitBudgetNs) {
          report(p.status, GDN_ERR_TIMEOUT);
          ready = -1;
          break;
        }
        __nanosleep(512);
      }
      __threadfence();
      upto_s = ready;
    }
    __syncthreads();
    const int c1 = upto_s;
    __syncthreads();  // upto_s is rewritten next round
    if (c1 < 0) return;
    // rows of this round in (chunk, unit, row) order
    const int X = (c1 - c0) * nwu * kNormRows;
    for (int x0 = warp; x0 < X; x0 += 8 * nw) {
      // eight rows' addresses (a dead row reads row 0, which exists: X > 0 means some
      // sequence has tokens), then every load before any use
      size_t orow[8], zrow[8];
      bool live[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int x = x0 + j * nw, q = x / kNormRows;
        const int cc = int((uint64_t(q) * inv_nwu) >> 32), i = q - cc * nwu;
        const int r = (c0 + cc) * kC + r0_s[i] + x % kNormRows;  // row within the sequence
        live[j] = x < X && r < len_s[i];
        const int t = tb_s[i] + r, h = uh_s[i] % p.Hv;
        orow[j] = live[j] ? size_t(t) * p.Hv + h : 0;
        zrow[j] = live[j] ? size_t(t) * p.z_stride + size_t(h) * kD : 0;
      }
      float4 ov[8];
      uint2 zr[8];
      if (p.o_half) {
        const __half* oh = reinterpret_cast<const __half*>(p.o_half) + 4 * lane;
        uint2 oraw[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) oraw[j] = __ldcg(reinterpret_cast<const uint2*>(oh + orow[j] * kD));
#pragma unroll
        for (int j = 0; j < 8; ++j) zr[j] = __ldg(reinterpret_cast<const uint2*>(zg + zrow[j] + 4 * lane));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&oraw[j].x));
          const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&oraw[j].y));
          ov[j] = make_float4(a.x, a.y, b.x, b.y);
        }
      } else {
        const float* of = p.core_out + 4 * lane;
#pragma unroll
        for (int j = 0; j < 8; ++j) ov[j] = __ldcg(reinterpret_cast<const float4*>(of + orow[j] * kD));
#pragma unroll
        for (int j = 0; j < 8; ++j) zr[j] = __ldg(reinterpret_cast<const uint2*>(zg + zrow[j] + 4 * lane));
      }
      // the eight rows side by side (dead rows too; only their stores are skipped)
      float ss[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        ss[j] = ov[j].x * ov[j].x + ov[j].y * ov[j].y + ov[j].z * ov[j].z + ov[j].w * ov[j].w;
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], m);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 o = ov[j];
        const float inv = rsqrtf(ss[j] / float(kD) + p.norm_eps);
        const float2 za = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zr[j].x));
        const float2 zb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zr[j].y));
        const __nv_bfloat162 y01 =
            __floats2bfloat162_rn(o.x * inv * w4.x * zgate_bf16(za.x, p.norm_gate),
                                  o.y * inv * w4.y * zgate_bf16(za.y, p.norm_gate));
        const __nv_bfloat162 y23 =
            __floats2bfloat162_rn(o.z * inv * w4.z * zgate_bf16(zb.x, p.norm_gate),
                                  o.w * inv * w4.w * zgate_bf16(zb.y, p.norm_gate));
        if (live[j])
          *reinterpret_cast<uint2*>(yg + orow[j] * kD + 4 * lane) =
              make_uint2(*reinterpret_cast<const uint32_t*>(&y01),
                         *reinterpret_cast<const uint32_t*>(&y23));
      }
    }
    c0 = c1;
  }
}

template <int NCOL>
__global__ void __launch_bounds__(4 * NCOL + (SpineSmem<NCOL>::kCounted ? 32 : 0), 1)
    gdn_prefill_spine_kernel(const __grid_constant__ PrefillParams p) {
  using S = SpineSmem<NCOL>;
  constexpr int kNS = kD / NCOL;  // slices per head
  if (S::kCounted && int(blockIdx.x) >= p.n * p.Hv * kNS) {
    const int chains = p.n * p.Hv * kNS;
    spine_norm_ctas(p, int(blockIdx.x) - chains, int(gridDim.x) - chains);
    return;
  }
  constexpr int kIssuer = 64;     // warp 2, lane 0: issues the MMAs
  constexpr int kLoader = 96;     // warp 3, lane 0: issues the bulk copies
  // (neither is in an output warp, whose work trails the chain)
  constexpr int kChain = 4 * NCOL;  // the chain's threads; a two-slice CTA has one more warp,
                                    // which only turns progress into the device-wide count
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slice = blockIdx.x % kNS, unit = blockIdx.x / kNS;
  // Units are handed out longest sequence first (ties: lower index first): CTAs start in
  // block order, so the long chains start early and the short ones fill in behind them.
  __shared__ int len_s[kOrderMax], order_s[kOrderMax];
  int seq = unit / p.Hv;
  if (p.n > 1 && p.n <= kOrderMax) {
    for (int i = tid; i < p.n; i += blockDim.x) len_s[i] = p.cu_seqlens[i + 1] - p.cu_seqlens[i];
    __syncthreads();
    for (int i = tid; i < p.n; i += blockDim.x) {
      const int li = len_s[i];
      int r = 0;
      for (int j = 0; j < p.n; ++j) r += (len_s[j] > li) || (len_s[j] == li && j < i);
      order_s[r] = i;
    }
    __syncthreads();
    seq = order_s[seq];
  }
  const int h = unit % p.Hv, kh = h / p.G;
  const int t_begin = p.cu_seqlens[seq], t_end = p.cu_seqlens[seq + 1];
  const uint64_t hp = p.h_ptrs[seq];
  {
    const int bad = check_seq(p, t_begin, t_end, hp);
    if (bad) {
      if (tid == 0) report(p.status, bad);
      return;
    }
  }
  const int len = t_end - t_begin;
  if (len == 0) return;  // nothing to do: the state stays as it is
  const int nc = (len + kC - 1) / kC;
  int32_t* cnt = p.counts + (2 * (size_t(seq) * p.Hv + h) + slice) * kCountStride;
  // chunks whose O rows this CTA has stored (set by kLoader after a chain barrier)
  __shared__ int stored_s;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  // full[b]: q_hat, W, g (and U) of buffer b; fullB[b]: P and K~ of buffer b, which only
  // MMA_b reads
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + S::kMisc);  // [2]
  uint64_t* fullB = full + 2;                                    // [2]
  uint64_t* bar_mma = full + 4;  // MMA_a, then K~^T Delta: the chain
  uint64_t* bar_o = full + 5;    // [P;*] Delta: only the outputs wait for it
  uint64_t* ufull = full + 6;    // U of the current chunk (whole-row spine)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(full + 7);

  const PrefillLayout lay{p.Hk, p.Hv};
  const unsigned char* ws = reinterpret_cast<const unsigned char*>(p.workspace);
  const size_t slot0 = PrefillLayout::base(t_begin, seq);

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&fullB[0], 1);
    mbar_init(&fullB[1], 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_o, 1);
    mbar_init(ufull, 1);
    fence_mbar_init();
    stored_s = 0;
  }
  if (warp == 0) tc::alloc(tslot, S::kTmemCols);
  if (S::kCounted && tid >= kChain) {
    // The counting warp: polls stored_s (acquire: the chain barrier before kLoader's
    // release store ordered every output thread's stores before it) and publishes each
    // new value behind a device-scope fence, off the chain's path.
    __syncthreads();
    int done = 0;
    uint64_t t0 = globaltimer_ns();
    for (;;) {
      int v;
      asm volatile("ld.acquire.cta.shared.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(&stored_s))
                   : "memory");
      if (v != done) {
        if (lane == 0) publish_count(cnt, v);
        done = v;
        t0 = globaltimer_ns();
      }
      if (v >= nc) break;  // all stored, or kCountStop
      if (globaltimer_ns() - t0 > kWaitBudgetNs) {  // the chain reports its own stop
        if (lane == 0) publish_count(cnt, kCountStop);
        break;
      }
    }
    __syncthreads();
    return;
  }

  const int q4 = warp & 3, cg = warp >> 2;
  const int row = 32 * q4 + lane;       // TMEM lane; the H row i of this thread
  const int jl0 = 32 * cg;              // first column of this warp within the slice
  const int col0 = NCOL * slice + jl0;  // ... and within the head
  float* Hg = reinterpret_cast<float*>(hp) + size_t(h) * kD * kD;
  float Hr[32];
#pragma unroll
  for (int u = 0; u < 32; u += 4) {
    const float4 x = *reinterpret_cast<const float4*>(Hg + size_t(row) * kD + col0 + u);
    Hr[u] = x.x;
    Hr[u + 1] = x.y;
    Hr[u + 2] = x.z;
    Hr[u + 3] = x.w;
  }
  // fp16 H rows as the MN-major B operand of MMA_a: [K = i][N = j] in 64-column blocks
  auto write_HT = [&]() {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(sm + S::kHT + tc::sw128_offset(128, row, jl0 + 8 * q)) =
          pack8_h(Hr + 8 * q);
  };
  write_HT();
  if (S::kNorm && tid < kD) reinterpret_cast<float*>(sm + S::kNW)[tid] = p.norm_w[tid];
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tl = uint32_t(32 * q4) << 16;
  constexpr uint32_t kTA = 0, kTH = NCOL, kTO = 2 * NCOL;

  // Chunk c's operands into buffer c & 1 (issued by kIssuer, completing on full[c & 1]).
  auto issue_loads = [&](int c) {
    const size_t cs = slot0 + size_t(c);
    unsigned char* st = sm + (c & 1) * S::kStage;
    const unsigned char* qimg = ws + lay.qk(cs, kh, 1);
    const unsigned char* wimg = ws + lay.w(cs, h);
    mbar_arrive_expect_tx(&full[c & 1], S::kTx - 8192 - 16384);
    bulk_g2s(st + S::kQW, qimg, 8192, &full[c & 1]);
    bulk_g2s(st + S::kQW + 8192, wimg, 8192, &full[c & 1]);
    bulk_g2s(st + S::kQW + 16384, qimg + 8192, 8192, &full[c & 1]);
    bulk_g2s(st + S::kQW + 24576, wimg + 8192, 8192, &full[c & 1]);
    bulk_g2s(st + S::kGd, ws + lay.g(cs, h), 256, &full[c & 1]);
    if constexpr (S::kUInStage)
      bulk_g2s(st + S::kUst, ws + lay.u(cs, h) + size_t(slice) * NCOL * 128, NCOL * 128,
               &full[c & 1]);
    mbar_arrive_expect_tx(&fullB[c & 1], 8192 + 16384);
    bulk_g2s(st + S::kP, ws + lay.p(cs, h), 8192, &fullB[c & 1]);
    bulk_g2s(st + S::kKt, ws + lay.kt(cs, h), 16384, &fullB[c & 1]);
  };
  // Chunk c's U columns of this slice into the single U buffer (completing on ufull).
  auto issue_u = [&](int c) {
    mbar_arrive_expect_tx(ufull, NCOL * 128);
    bulk_g2s(sm + S::kUs, ws + lay.u(slot0 + size_t(c), h) + size_t(slice) * NCOL * 128,
             NCOL * 128, ufull);
  };
  if (tid == kLoader) {
    issue_loads(0);
    if (!S::kUInStage) issue_u(0);
  }
  int issued = 0;    // last chunk whose loads were issued (meaningful in kLoader)
  int u_issued = 0;  // ... and whose U was
  // The z rows of chunk c (bf16, this head's 128 columns; 16-byte piece k of row r at
  // k ^ (r % 16)): each output thread copies its own 64 bytes.
  const __nv_bfloat16* zg = reinterpret_cast<const __nv_bfloat16*>(p.z);
  auto issue_z = [&](int c) {
    const int r = row, t0 = c * kC;
    if (r < ((len - t0) < kC ? (len - t0) : kC)) {
      const unsigned char* src = reinterpret_cast<const unsigned char*>(
          zg + size_t(t_begin + t0 + r) * p.z_stride + size_t(h) * kD + jl0);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        cp_async16(sm + S::kZ + r * 256 + (((cg * 4 + k) ^ (r & 15)) << 4), src + 16 * k);
    }
    cp_async_commit();
  };

  uint32_t mma_phase = 0;
  bool bad = false;
  auto mma_wait = [&]() {
    bad |= !mbar_wait_bounded(bar_mma, mma_phase);
    mma_phase ^= 1u;
    tc::fence_after_sync();
  };
  auto sync_or_stop = [&]() -> bool {
    tc::fence_before_sync();
    const bool stop = S::kCounted ? named_sync_or(3, kChain, bad) : __syncthreads_or(bad) != 0;
    tc::fence_after_sync();
    return stop;
  };
  auto set_stored = [&](int v) {
    asm volatile("st.release.cta.shared.s32 [%0], %1;" ::"r"(smem_u32(&stored_s)), "r"(v)
                 : "memory");
  };

  bool aborted = false;
  int consumed = -1;
  for (int c = 0; c < nc; ++c) {
    const int t0 = c * kC;
    const int L = (len - t0) < kC ? (len - t0) : kC;
    const uint32_t st = uint32_t(c & 1) * S::kStage;
    // The other buffer was last read by chunk c - 1's MMAs (complete) and by this CTA's
    // threads before the last barrier: refill it for chunk c + 1.
    if (tid == kLoader && c + 1 < nc) {
      issue_loads(c + 1);
      issued = c + 1;
    }
    if (S::kNorm && q4 < 2) issue_z(c);
    bad |= !mbar_wait_bounded(&full[c & 1], uint32_t(c >> 1) & 1u);
    consumed = c;
    const float* gd = reinterpret_cast<const float*>(sm + st + S::kGd);
    // U rows of this thread (W-row lanes 64..127) into registers: while MMA_a runs when U
    // came with the chunk's operands (two-slice spine), else once its own copy has landed
    float X[32];
    auto read_u = [&]() {
      const int r = row - kC;
      if (!S::kUInStage) bad |= !mbar_wait_bounded(ufull, uint32_t(c) & 1u);
      const __half* Us = reinterpret_cast<const __half*>(
                             sm + (S::kUInStage ? st + S::kUst : S::kUs)) +
                         cg * (kC * 32) + r * 32;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 x = *reinterpret_cast<const uint4*>(Us + ((k ^ ((r >> 1) & 3)) << 3));
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          X[8 * k + 2 * e] = f.x;
          X[8 * k + 2 * e + 1] = f.y;
        }
      }
    };
    if (S::kUInStage && q4 >= 2) read_u();

    // ---- MMA_a: [Q;W] H0
    if (tid == kIssuer) {
      if (!bad) {
#pragma unroll
        for (int k0 = 0; k0 < kD; k0 += 16)
          tc::mma_f16(tmem + kTA, tc::desc_at(sb + st + S::kQW, 128, k0),
                       tc::desc_mn_sw128(sb + S::kHT + k0 * 128, 16384),
                       tc::idesc_f16(128, NCOL, false, true), k0 > 0);
      }
      tc::commit(bar_mma);
    }
    mma_wait();

    // ---- Delta = U - W H0 (fp16 Delta^T for MMA_b); the Q H0 rows stay in registers
    float eg = 0.f;
    const float eL = exp2_fast(gd[kC - 1]);
    {
      float v[32];
      tc::ld32(tmem + tl + kTA + jl0, v);
      if (q4 >= 2) {
        const int r = row - kC;
        if (!S::kUInStage) read_u();
#pragma unroll
        for (int u = 0; u < 32; ++u) v[u] = X[u] - v[u];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(sm + S::kDT + tc::sw128_offset(64, r, jl0 + 8 * q)) =
              pack8_h(v + 8 * q);
      } else {
#pragma unroll
        for (int u = 0; u < 32; ++u) X[u] = v[u];
        eg = exp2_fast(gd[row]);
      }
    }
    fence_proxy_async_smem();
    if (sync_or_stop()) { aborted = true; break; }
    // chunk c - 1's O rows were stored before that barrier
    if (S::kCounted && tid == kLoader && c > 0) set_stored(c);

    // ---- MMA_b: K~^T Delta (the chain), then [P;*] Delta (the outputs)
    if (tid == kIssuer) {
      bad |= !mbar_wait_bounded(&fullB[c & 1], uint32_t(c >> 1) & 1u);
      if (!bad) {
#pragma unroll
        for (int s0 = 0; s0 < kC; s0 += 16)
          tc::mma_f16(tmem + kTH, tc::desc_mn_sw128(sb + st + S::kKt + s0 * 128, 8192),
                       tc::desc_mn_sw128(sb + S::kDT + s0 * 128, 8192),
                       tc::idesc_f16(128, NCOL, true, true), s0 > 0);
      }
      tc::commit(bar_mma);
      if (!bad) {
#pragma unroll
        for (int s0 = 0; s0 < kC; s0 += 16)
          tc::mma_f16(tmem + kTO, tc::desc_at(sb + st + S::kP, 128, s0),
                       tc::desc_mn_sw128(sb + S::kDT + s0 * 128, 8192),
                       tc::idesc_f16(128, NCOL, false, true), s0 > 0);
      }
      tc::commit(bar_o);
    }
    // this chunk's U has been read (before the barrier): fetch the next chunk's
    if (!S::kUInStage && tid == kLoader && c + 1 < nc) {
      issue_u(c + 1);
      u_issued = c + 1;
    }
    mma_wait();

    // ---- H = e^{g_L} H + K~^T Delta (f32 registers, fp16 copy for the next MMA_a)
    {
      float v[32];
      tc::ld32(tmem + tl + kTH + jl0, v);
#pragma unroll
      for (int u = 0; u < 32; ++u) Hr[u] = eL * Hr[u] + v[u];
      write_HT();
    }
    fence_proxy_async_smem();
    if (sync_or_stop()) { aborted = true; break; }

    // ---- O = e^g (Q H0) + P Delta for the query rows (lanes 0..63), behind the next MMA_a
    if (q4 < 2) {
      bad |= !mbar_wait_bounded(bar_o, uint32_t(c) & 1u);
      tc::fence_after_sync();
      float v[32];
      tc::ld32(tmem + tl + kTO + jl0, v);
#pragma unroll
      for (int u = 0; u < 32; ++u) v[u] = eg * X[u] + v[u];
      const size_t orow = size_t(t_begin + t0 + row) * p.Hv + h;
      if (p.o_half && row < L) {  // the norm kernel's fp16 copy of O
        __half* o = reinterpret_cast<__half*>(p.o_half) + orow * kD + col0;
#pragma unroll
        for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(o + 8 * q) = pack8_h(v + 8 * q);
      } else if (p.core_out && row < L) {
        float* o = p.core_out + orow * kD + col0;
#pragma unroll
        for (int u = 0; u < 32; u += 4)
          *reinterpret_cast<float4*>(o + u) = make_float4(v[u], v[u + 1], v[u + 2], v[u + 3]);
      }
      if constexpr (S::kNorm) {
        // y = O / rms(O) * w * silu(z), the row's sum of squares over the 4 column groups
        float* red = reinterpret_cast<float*>(sm + S::kRed);
        const float* nw = reinterpret_cast<const float*>(sm + S::kNW) + jl0;
        float ss = 0.f;
#pragma unroll
        for (int u = 0; u < 32; ++u) ss += v[u] * v[u];
        red[cg * kC + row] = ss;
        named_sync(1, 8 * 32);
        ss = red[row] + red[kC + row] + red[2 * kC + row] + red[3 * kC + row];
        const float inv = rsqrtf(ss / float(kD) + p.norm_eps);
        cp_async_wait_all();
        if (row < L) {
          __nv_bfloat16* yo = reinterpret_cast<__nv_bfloat16*>(p.y) + orow * kD + jl0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 zr = *reinterpret_cast<const uint4*>(
                sm + S::kZ + row * 256 + (((cg * 4 + k) ^ (row & 15)) << 4));
            const __nv_bfloat162* z2 = reinterpret_cast<const __nv_bfloat162*>(&zr);
            uint32_t out[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 zf = __bfloat1622float2(z2[e]);
              const int u = 8 * k + 2 * e;
              const __nv_bfloat162 yy = __floats2bfloat162_rn(
                  v[u] * inv * nw[u] * zgate_bf16(zf.x, p.norm_gate),
                  v[u + 1] * inv * nw[u + 1] * zgate_bf16(zf.y, p.norm_gate));
              out[e] = *reinterpret_cast<const uint32_t*>(&yy);
            }
            *reinterpret_cast<uint4*>(yo + 8 * k) = make_uint4(out[0], out[1], out[2], out[3]);
          }
        }
      }
    }
  }
  if (S::kNorm) cp_async_wait_all();

  if (aborted) {
    if (tid == kLoader) {
      report(p.status, GDN_ERR_TIMEOUT);
      // fills still in flight land before this CTA's shared memory is released
      if (issued > consumed) {
        mbar_wait_bounded(&full[issued & 1], uint32_t(issued >> 1) & 1u);
        mbar_wait_bounded(&fullB[issued & 1], uint32_t(issued >> 1) & 1u);
      }
      if (consumed >= 0) mbar_wait_bounded(&fullB[consumed & 1], uint32_t(consumed >> 1) & 1u);
      if (!S::kUInStage && u_issued > consumed) mbar_wait_bounded(ufull, uint32_t(u_issued) & 1u);
    }
  } else {
#pragma unroll
    for (int u = 0; u < 32; u += 4)
      *reinterpret_cast<float4*>(Hg + size_t(row) * kD + col0 + u) =
          make_float4(Hr[u], Hr[u + 1], Hr[u + 2], Hr[u + 3]);
  }
  if constexpr (S::kCounted) {
    named_sync(3, kChain);  // the last chunk's O rows are stored
    if (tid == kLoader) set_stored(aborted ? kCountStop : nc);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, S::kTmemCols);
}

template <int NCOL>
cudaError_t launch_spine(const PrefillParams& p, cudaStream_t stream) {
  auto kern = gdn_prefill_spine_kernel<NCOL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(SpineSmem<NCOL>::kAlloc));
  if (e != cudaSuccess) return e;
  const int chains = p.n * p.Hv * (kD / NCOL);
  if (!SpineSmem<NCOL>::kCounted) {
    kern<<<chains, 4 * NCOL, SpineSmem<NCOL>::kAlloc, stream>>>(p);
    return cudaGetLastError();
  }
  // Cooperative, so that every norm CTA's chains are resident: as many CTAs as fit at once.
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 4 * NCOL + 32,
                                                    SpineSmem<NCOL>::kAlloc);
  if (e != cudaSuccess) return e;
  const int grid = per_sm * sm_count();
  if (grid - chains >= 2 * p.n * p.Hv) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(4 * NCOL + 32);
    cfg.dynamicSmemBytes = SpineSmem<NCOL>::kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeCooperative;
    attr.val.cooperative = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaErrorCooperativeLaunchTooLarge) return e != cudaSuccess ? e : cudaGetLastError();
    // fewer SMs than the device has are open to this context (an MPS limit, say)
    (void)cudaGetLastError();
  }
  {
    // fewer than two spare SMs per head (the norm CTAs would trail the chains): the chains
    // alone, then the norm kernel
    kern<<<chains, 4 * NCOL + 32, SpineSmem<NCOL>::kAlloc, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_gated_rmsnorm(p.o_half ? p.o_half : static_cast<const void*>(p.core_out),
                                p.o_half != nullptr, p.z, p.z_stride, p.norm_w, p.norm_eps,
                                p.total_tokens, p.Hv, kD, GDN_DTYPE_BF16, p.norm_gate, p.y,
                                stream);
  }
}

}  // namespace

// Chunk kernel, the spine and the gated norm.  o_work: f32 [total_tokens][Hv][128] room for
// the core output when the caller passes none and the norm runs as its own kernel.
cudaError_t launch_prefill_tc(const PrefillParams& p, float* o_work, cudaStream_t stream) {
  if (p.n <= 0) return cudaSuccess;
  {
    auto kern = gdn_prefill_chunk_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(PrepSmem::kAlloc));
    if (e != cudaSuccess) return e;
    const size_t slots = PrefillLayout::slots(p.n, p.total_tokens);
    kern<<<unsigned(slots * p.Hv), kPrepThreads, PrepSmem::kAlloc, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // Column slices per (sequence, head): as many as one wave of CTAs holds, since the
  // spine's time is its chain of chunks, not its arithmetic.
  // A whole-row spine (128 columns) applies the gated norm itself; two column slices per
  // head double the chains when one wave would otherwise leave SMs idle, and leave the norm
  // to the CTAs of the same launch on the SMs still free.
  const int units = p.n * p.Hv, sms = sm_count();
  if (units * 2 > sms) return launch_spine<128>(p, stream);
  // Without an f32 core output to fill, O reaches the norm as fp16 (2^-11 relative, far
  // below the bf16 rounding of y), which halves that hand-off's bytes.
  PrefillParams q = p;
  q.o_half = p.core_out ? nullptr : static_cast<void*>(o_work);
  return launch_spine<64>(q, stream);
}

}  // namespace gdn
