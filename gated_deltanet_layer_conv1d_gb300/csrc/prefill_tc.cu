// prefill_tc.cu -- chunked (WY / UT-transform) prefill of the gated delta rule on the
// 5th-generation tensor cores (tcgen05, accumulators in TMEM), d_k = d_v = 128, chunk 64.
//
// The method (layer_struct.rs, the FLA chunked prefill: gdn_prefill_fla_recompute_wu_k ->
// the chunk_delta_h state spine -> gdn_prefill_fla_chunk_fwd_o_k; here one fused kernel per
// (sequence, value head)).  Inside a chunk of L tokens, with g_r = sum_{s<=r} log alpha_s:
//   A   = strict_lower(beta_r (k_r . k_s) e^{g_r - g_s}),   T = (I + A)^{-1}
//   W   = T diag(beta e^g) K,   U = T diag(beta) V,   Delta = U - W H0      (H0 = S0^T)
//   O   = diag(e^g) Q H0 + lower_incl(Q K^T e^{g_r - g_s}) Delta
//   H_L = e^{g_L} H0 + (diag(e^{g_L - g}) K)^T Delta
// Every product is computed transposed so that M = 128 (one TMEM lane per accumulator row):
//   MMA0  [K;Q] K^T            (M 128 = 64 keys + 64 queries, N 64, K 128)
//   MMA_W W^T = K^T (T diag(beta e^g))^T      (A = K MN-major, N 64, K 64)
//   MMA_U U^T = V^T (T diag(beta))^T          (A = V MN-major)
//   MMA1  (W H0)^T = H0^T W^T,   MMA2  (Q H0)^T = H0^T Q^T     (N 64, K 128)
//   MMA3  (P Delta)^T = Delta^T P^T           (N 64, K 64)
//   MMA4  (K~^T Delta)^T = (Delta^T diag(e^{g_L - g})) K        (B = K MN-major, N 128, K 64)
// All per-token scalings are folded into T's columns, Delta's columns or the epilogue, so
// the q, k, v tiles come straight from the pre-pass workspace (one bulk copy each).
// Operands are fp16 (kind::f16, f32 accumulation): every operand here is bounded
// (normalised q and k, O(1) v, T, P, Delta and state), and fp16's 11-bit significand
// keeps the rounding of the inputs and of T, P and Delta eight times below bf16's.
// H0 lives in registers (f32) of the 8 warps: thread (w, l) owns row j = 32 (w % 4) + l of
// H^T and columns i in [64 (w / 4), +64); its fp16 copy is the A operand of MMA1/MMA2.
// T = (I + A)^{-1} is computed on CUDA cores by blocked forward substitution (16 x 16
// diagonal blocks, then the off-diagonal blocks level by level).
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "prefill_layout.cuh"
#include "tcgen05.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 256;

// Shared memory (offsets from a 1024-aligned base).
struct TcSmem {
  static constexpr uint32_t kAQK = 0;            // [128][128] f16: rows 0-63 k_hat, 64-127 q_hat
  static constexpr uint32_t kV = 32768;          // [64][128] f16 v (MN-major A of MMA_U)
  static constexpr uint32_t kHT = 49152;         // [128][128] f16 H^T
  static constexpr uint32_t kW = 81920;          // [64][128] f16 W
  static constexpr uint32_t kTw = 98304;         // [64][64] f16 T diag(beta e^g)
  static constexpr uint32_t kTu = 106496;        // [64][64] f16 T diag(beta)
  static constexpr uint32_t kP = 114688;         // [64][64] f16 P
  static constexpr uint32_t kDT = 122880;        // [128][64] f16 Delta^T
  static constexpr uint32_t kDTs = 139264;       // [128][64] f16 Delta^T diag(e^{g_L - g})
  static constexpr int kAS = 65;                 // row stride of A: odd, so column writes
                                                 // from 32 lanes hit 32 banks
  static constexpr uint32_t kAm = 155648;        // [64][65] f32 A
  static constexpr uint32_t kTf = 172288;        // [64][64] f32 T
  static constexpr uint32_t kOs = kAm;           // [64][128] f32 outputs (A and T are dead then)
  static constexpr uint32_t kY = 188672;         // [3][16][16] f32 scratch of the inverse
  static constexpr uint32_t kZ = 191744;         // [2][64][128] bf16 z rows, double-buffered
  static constexpr uint32_t kNW = 224512;        // [128] f32 norm weight
  static constexpr uint32_t kGate = 225024;      // [2][64] f32 log(alpha), beta (bulk copied)
  static constexpr uint32_t kG = 225536;         // [64] f32 cumulative log decay g
  static constexpr uint32_t kB = 225792;         // [64] f32 beta (0 past the chunk end)
  static constexpr uint32_t kMisc = 226048;      // bars, tmem slot, scan carry
  static constexpr uint32_t kBytes = 226176;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // room to align the base to 1024
};
static_assert(TcSmem::kOs + 64 * 128 * 4 <= TcSmem::kY, "output staging fits in A and T");
static_assert(TcSmem::kAm + 64 * TcSmem::kAS * 4 <= TcSmem::kTf, "A fits");

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

// TMEM columns of the accumulators (512 allocated).
constexpr uint32_t kT0 = 0;     // MMA0: [K;Q] K^T          (64 cols)
constexpr uint32_t kTW = 64;    // MMA_W: W^T               (64)
constexpr uint32_t kTU = 128;   // MMA_U: U^T               (64)
constexpr uint32_t kTD = 192;   // MMA1: (W H0)^T           (64)
constexpr uint32_t kT2 = 256;   // MMA2: (Q H0)^T           (64)
constexpr uint32_t kT3 = 320;   // MMA3: (P Delta)^T        (64)
constexpr uint32_t kT4 = 384;   // MMA4: (K~^T Delta)^T     (128)

__global__ void __launch_bounds__(kThreads, 1)
    gdn_prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
  using S = TcSmem;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  float* Am = reinterpret_cast<float*>(sm + S::kAm);
  float* Tf = reinterpret_cast<float*>(sm + S::kTf);
  float* Ys = reinterpret_cast<float*>(sm + S::kY);
  float* gate = reinterpret_cast<float*>(sm + S::kGate);
  float* G_s = reinterpret_cast<float*>(sm + S::kG);  // cumulative log2 decay
  float* B_s = reinterpret_cast<float*>(sm + S::kB);
  float* NW = reinterpret_cast<float*>(sm + S::kNW);
  float* Os = reinterpret_cast<float*>(sm + S::kOs);  // output staging, after the inverse
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(sm + S::kMisc);
  uint64_t* bar_mma = bar_load + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  float* carry = reinterpret_cast<float*>(tslot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seq = blockIdx.x / p.Hv, h = blockIdx.x % p.Hv, kh = h / p.G;
  const int t_begin = p.cu_seqlens[seq], t_end = p.cu_seqlens[seq + 1];
  const int len = t_end - t_begin;
  const uint64_t hp = p.h_ptrs[seq];
  {
    int bad = 0;
    if (t_begin < 0 || len < 0 || t_end > p.total_tokens || len > p.max_seqlen)
      bad = GDN_ERR_BAD_SEQLENS;
    else if (hp == 0 || (hp & 15u) != 0)
      bad = GDN_ERR_BAD_TABLE_ENTRY;
    if (bad) {
      if (tid == 0) report(p.status, bad);
      return;
    }
  }
  if (len == 0) return;  // nothing to do: the state stays as it is

  const PrefillLayout lay{p.Hk, p.Hv};
  const size_t slot0 = PrefillLayout::base(t_begin, seq);
  const unsigned char* ws = reinterpret_cast<const unsigned char*>(p.workspace);
  const int nc = (len + kC - 1) / kC;

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, 512);

  // H0 (f32) into registers: H^T row j, columns i0 .. i0 + 63.
  const int q4 = warp & 3, half = warp >> 2;
  const int j = 32 * q4 + lane;
  const int i0 = 64 * half;
  float* Hg = reinterpret_cast<float*>(hp) + size_t(h) * kD * kD;
  float Hr[64];
#pragma unroll
  for (int ii = 0; ii < 64; ++ii) Hr[ii] = Hg[(i0 + ii) * kD + j];
  auto write_HT = [&]() {
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8)
      *reinterpret_cast<uint4*>(sm + S::kHT + tc::sw128_offset(128, j, i0 + 8 * c8)) =
          pack8_h(Hr + 8 * c8);
  };
  write_HT();
  if (tid < kD) NW[tid] = p.norm_w[tid];
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  // The q_hat / k_hat / v tiles and gates of chunk c into shared memory: bulk copies issued
  // by thread 0, completing on bar_load.
  auto issue_loads = [&](int c) {
    const size_t cs = slot0 + size_t(c);
    const unsigned char* kimg = ws + lay.qk(cs, kh, 0);
    const unsigned char* qimg = ws + lay.qk(cs, kh, 1);
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar_load, 3u * 16384u + 512u);
    bulk_g2s(sm + S::kAQK, kimg, 8192, bar_load);
    bulk_g2s(sm + S::kAQK + 16384, kimg + 8192, 8192, bar_load);
    bulk_g2s(sm + S::kAQK + 8192, qimg, 8192, bar_load);
    bulk_g2s(sm + S::kAQK + 24576, qimg + 8192, 8192, bar_load);
    bulk_g2s(sm + S::kV, ws + lay.v(cs, h), 16384, bar_load);
    bulk_g2s(gate, ws + lay.gate(cs, h), 512, bar_load);
  };
  // The z rows of chunk c (bf16, this value head's 128 columns) into z buffer c & 1: every
  // thread copies 16-byte pieces with cp.async; each waits for its own before the barrier
  // that precedes the norm.
  auto issue_z = [&](int c) {
    const int t0 = c * kC;
    const int L = (len - t0) < kC ? (len - t0) : kC;
    unsigned char* zdst = sm + S::kZ + (c & 1) * 16384;
    const unsigned char* zsrc = reinterpret_cast<const unsigned char*>(
        reinterpret_cast<const __nv_bfloat16*>(p.z) + size_t(t_begin + t0) * p.z_stride +
        size_t(h) * kD);
    for (int e = tid; e < L * 16; e += kThreads) {
      const int r = e / 16, piece = e % 16;
      cp_async16(zdst + r * 256 + piece * 16, zsrc + size_t(r) * p.z_stride * 2 + piece * 16);
    }
    cp_async_commit();
  };
  if (tid == 0) issue_loads(0);
  issue_z(0);
  const uint32_t tl = uint32_t(32 * q4) << 16;  // this warp's TMEM lane quarter
  uint32_t load_phase = 0, mma_phase = 0;
  bool bad = false;
  // Every thread waits for the MMAs committed so far.
  auto mma_wait = [&]() {
    bad |= !mbar_wait_bounded(bar_mma, mma_phase);
    mma_phase ^= 1u;
    tc::fence_after_sync();
  };
  // Barrier that also agrees on a failed wait; true means stop.
  auto sync_or_stop = [&]() -> bool {
    tc::fence_before_sync();
    const bool stop = __syncthreads_or(bad) != 0;
    tc::fence_after_sync();
    return stop;
  };

  bool aborted = false;
  for (int c = 0; c < nc; ++c) {
    const int t0 = c * kC;
    const int L = (len - t0) < kC ? (len - t0) : kC;

    // ---- 1. this chunk's tiles, gates and z rows (issued during the previous chunk)
    bad |= !mbar_wait_bounded(bar_load, load_phase);
    load_phase ^= 1u;

    // ---- 2. rows past the end of the sequence are zero; decay prefix sums
    if (L < kC) {
      const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
      for (int idx = tid; idx < (kC - L) * 16; idx += kThreads) {
        const int row = L + idx / 16, ch = idx % 16, blk = ch / 8, c16 = ch % 8;
        *reinterpret_cast<uint4*>(sm + S::kAQK + blk * 16384 + row * 128 + c16 * 16) = zero;
        *reinterpret_cast<uint4*>(sm + S::kAQK + blk * 16384 + (kC + row) * 128 + c16 * 16) = zero;
        *reinterpret_cast<uint4*>(sm + S::kV + blk * 8192 + row * 128 + c16 * 16) = zero;
      }
    }
    if (tid < kC) {
      // g in log2 units (log(alpha) * log2(e)), so each decay factor below is one exp2f
      float v = tid < L ? gate[tid] * 1.4426950408889634f : 0.f;
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
    }
    fence_proxy_async_smem();
    if (sync_or_stop()) { aborted = true; break; }
    const float gL = G_s[L - 1];

    // ---- 3. MMA0: [K;Q] K^T
    if (tid == 0) {
#pragma unroll
      for (int k0 = 0; k0 < kD; k0 += 16)
        tc::mma_f16(tmem + kT0, tc::desc_at(sb + S::kAQK, 128, k0),
                     tc::desc_at(sb + S::kAQK, 128, k0), tc::idesc_f16(128, 64), k0 > 0);
      tc::commit(bar_mma);
    }
    mma_wait();

    // ---- 4. A (f32) from the K K^T rows, P (fp16) from the Q K^T rows
    {
      float v[32];
      tc::ld16(tmem + tl + kT0 + 32 * half, *reinterpret_cast<float(*)[16]>(v));
      tc::ld16(tmem + tl + kT0 + 32 * half + 16, *reinterpret_cast<float(*)[16]>(v + 16));
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
    if (sync_or_stop()) { aborted = true; break; }

    // ---- 5. T = (I + A)^{-1}: diagonal 16 x 16 blocks, then the blocks below them
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
        for (int rr = 0; rr < 16; ++rr) Tf[(b0 + rr) * kC + b0 + lane] = X[rr];
      }
    } else {
      // blocks above the diagonal are zero
      for (int e = tid - 128; e < 6 * 256; e += 128) {
        const int blk = e / 256, a = (e % 256) / 16, bb = e % 16;
        const int I = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int J = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        Tf[(16 * I + a) * kC + 16 * J + bb] = 0.f;
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
            const float* br = Tf + (k0 + t) * kC + 16 * J + 8 * nt + g;
            mma_tf32(y[nt], a, to_tf32(br[0]), to_tf32(br[4 * kC]));
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
          const float* ar = Tf + (16 * I + g) * kC + 16 * I + k0 + t;
          const uint32_t a[4] = {to_tf32(ar[0]), to_tf32(ar[8 * kC]), to_tf32(ar[4]),
                                 to_tf32(ar[8 * kC + 4])};
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
            mma_tf32(tt[nt], a, to_tf32(Yw[(k0 + t) * 16 + 8 * nt + g]),
                     to_tf32(Yw[(k0 + t + 4) * 16 + 8 * nt + g]));
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          float* tr = Tf + (16 * I + g) * kC + 16 * J + 8 * nt + 2 * t;
          tr[0] = -tt[nt][0];
          tr[1] = -tt[nt][1];
          tr[8 * kC] = -tt[nt][2];
          tr[8 * kC + 1] = -tt[nt][3];
        }
      }
      __syncthreads();
    }
    // T diag(beta e^g) and T diag(beta), fp16, [r][s]
    for (int cid = tid; cid < kC * 8; cid += kThreads) {
      const int r = cid / 8, s0 = (cid % 8) * 8;
      float tw[8], tu[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float tv = Tf[r * kC + s0 + u];
        tu[u] = tv * B_s[s0 + u];
        tw[u] = tu[u] * exp2_fast(G_s[s0 + u]);
      }
      *reinterpret_cast<uint4*>(sm + S::kTw + tc::sw128_offset(64, r, s0)) = pack8_h(tw);
      *reinterpret_cast<uint4*>(sm + S::kTu + tc::sw128_offset(64, r, s0)) = pack8_h(tu);
    }
    fence_proxy_async_smem();
    if (sync_or_stop()) { aborted = true; break; }

    // ---- 6. W^T = K^T (T diag(beta e^g))^T, U^T = V^T (T diag(beta))^T
    if (tid == 0) {
#pragma unroll
      for (int s0 = 0; s0 < kC; s0 += 16) {
        tc::mma_f16(tmem + kTW, tc::desc_mn_sw128(sb + S::kAQK + s0 * 128, 16384),
                     tc::desc_at(sb + S::kTw, 64, s0), tc::idesc_f16(128, 64, true, false),
                     s0 > 0);
        tc::mma_f16(tmem + kTU, tc::desc_mn_sw128(sb + S::kV + s0 * 128, 8192),
                     tc::desc_at(sb + S::kTu, 64, s0), tc::idesc_f16(128, 64, true, false),
                     s0 > 0);
      }
      tc::commit(bar_mma);
    }
    mma_wait();

    // ---- 7. W [r][i] from W^T (lane i)
    {
      float v[32];
      tc::ld16(tmem + tl + kTW + 32 * half, *reinterpret_cast<float(*)[16]>(v));
      tc::ld16(tmem + tl + kTW + 32 * half + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      const int i = 32 * q4 + lane;
#pragma unroll
      for (int u = 0; u < 32; ++u)
        *reinterpret_cast<__half*>(sm + S::kW + tc::sw128_offset(64, 32 * half + u, i)) =
            __float2half_rn(v[u]);
    }
    fence_proxy_async_smem();
    if (sync_or_stop()) { aborted = true; break; }

    // ---- 8. (W H0)^T = H0^T W^T and (Q H0)^T = H0^T Q^T
    if (tid == 0) {
#pragma unroll
      for (int k0 = 0; k0 < kD; k0 += 16) {
        tc::mma_f16(tmem + kTD, tc::desc_at(sb + S::kHT, 128, k0),
                     tc::desc_at(sb + S::kW, 64, k0), tc::idesc_f16(128, 64), k0 > 0);
        tc::mma_f16(tmem + kT2, tc::desc_at(sb + S::kHT, 128, k0),
                     tc::desc_at(sb + S::kAQK + 8192, 128, k0), tc::idesc_f16(128, 64),
                     k0 > 0);
      }
      tc::commit(bar_mma);
    }
    mma_wait();

    // ---- 9. Delta^T = U^T - (W H0)^T, and its decay-weighted copy
    {
      float du[32], dd[32];
      tc::ld16(tmem + tl + kTU + 32 * half, *reinterpret_cast<float(*)[16]>(du));
      tc::ld16(tmem + tl + kTU + 32 * half + 16, *reinterpret_cast<float(*)[16]>(du + 16));
      tc::ld16(tmem + tl + kTD + 32 * half, *reinterpret_cast<float(*)[16]>(dd));
      tc::ld16(tmem + tl + kTD + 32 * half + 16, *reinterpret_cast<float(*)[16]>(dd + 16));
      float ds[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        du[u] -= dd[u];
        ds[u] = du[u] * exp2_fast(gL - G_s[32 * half + u]);
      }
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        const uint32_t off = tc::sw128_offset(128, j, 32 * half + 8 * c8);
        *reinterpret_cast<uint4*>(sm + S::kDT + off) = pack8_h(du + 8 * c8);
        *reinterpret_cast<uint4*>(sm + S::kDTs + off) = pack8_h(ds + 8 * c8);
      }
    }
    fence_proxy_async_smem();
    if (sync_or_stop()) { aborted = true; break; }

    // ---- 10. (P Delta)^T = Delta^T P^T and (K~^T Delta)^T = (Delta^T e^{g_L - g}) K
    if (tid == 0) {
#pragma unroll
      for (int s0 = 0; s0 < kC; s0 += 16) {
        tc::mma_f16(tmem + kT3, tc::desc_at(sb + S::kDT, 128, s0),
                     tc::desc_at(sb + S::kP, 64, s0), tc::idesc_f16(128, 64), s0 > 0);
        tc::mma_f16(tmem + kT4, tc::desc_at(sb + S::kDTs, 128, s0),
                     tc::desc_mn_sw128(sb + S::kAQK + s0 * 128, 16384),
                     tc::idesc_f16(128, 128, false, true), s0 > 0);
      }
      tc::commit(bar_mma);
    }
    mma_wait();
    // Every MMA of this chunk has completed and the q/k, v and gate buffers are no longer
    // read: start the next chunk's loads now, behind this chunk's epilogue.
    if (c + 1 < nc) {
      if (tid == 0) issue_loads(c + 1);
      issue_z(c + 1);
    }

    // ---- 11. H update (registers + fp16 copy) and the chunk outputs
    {
      const float eL = exp2_fast(gL);
#pragma unroll
      for (int c16 = 0; c16 < 4; ++c16) {
        float v[16];
        tc::ld16(tmem + tl + kT4 + i0 + 16 * c16, v);
#pragma unroll
        for (int u = 0; u < 16; ++u) Hr[16 * c16 + u] = eL * Hr[16 * c16 + u] + v[u];
      }
      write_HT();
      float d2[32], d3[32];
      tc::ld16(tmem + tl + kT2 + 32 * half, *reinterpret_cast<float(*)[16]>(d2));
      tc::ld16(tmem + tl + kT2 + 32 * half + 16, *reinterpret_cast<float(*)[16]>(d2 + 16));
      tc::ld16(tmem + tl + kT3 + 32 * half, *reinterpret_cast<float(*)[16]>(d3));
      tc::ld16(tmem + tl + kT3 + 32 * half + 16, *reinterpret_cast<float(*)[16]>(d3 + 16));
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const int r = 32 * half + u;
        Os[r * kD + j] = exp2_fast(G_s[r]) * d2[u] + d3[u];
      }
    }
    // this chunk's z rows: the last group of this thread's own copies still in flight is
    // the next chunk's, so wait until at most one group remains
    if (c + 1 < nc) asm volatile("cp.async.wait_group 1;" ::: "memory");
    else asm volatile("cp.async.wait_group 0;" ::: "memory");
    fence_proxy_async_smem();
    if (sync_or_stop()) { aborted = true; break; }

    // ---- 12. gated RMSNorm of the chunk's outputs, one warp per token
#pragma unroll
    for (int rr = 0; rr < kC / (kThreads / 32); ++rr) {
      const int r = warp + rr * (kThreads / 32);
      if (r >= L) break;
      const int row = t_begin + t0 + r;
      const int jj = lane * 4;
      const float4 o = *reinterpret_cast<const float4*>(Os + r * kD + jj);
      const float ss = warp_sum(o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w);
      const float inv = rsqrtf(ss / float(kD) + p.norm_eps);
      const float4 w4 = *reinterpret_cast<const float4*>(NW + jj);
      const float4 z4 = Act<__nv_bfloat16>::load4(
          reinterpret_cast<const __nv_bfloat16*>(sm + S::kZ + (c & 1) * 16384) + r * kD + jj);
      float4 yv;
      yv.x = o.x * inv * w4.x * silu_fast(z4.x);
      yv.y = o.y * inv * w4.y * silu_fast(z4.y);
      yv.z = o.z * inv * w4.z * silu_fast(z4.z);
      yv.w = o.w * inv * w4.w * silu_fast(z4.w);
      Act<__nv_bfloat16>::store4(
          reinterpret_cast<__nv_bfloat16*>(p.y) + size_t(row) * p.Hv * kD + h * kD + jj, yv);
      if (p.core_out)
        *reinterpret_cast<float4*>(p.core_out + (size_t(row) * p.Hv + h) * kD + jj) = o;
    }
    __syncthreads();  // Os and this chunk's z buffer are read
  }

  if (aborted) {
    if (tid == 0) report(p.status, GDN_ERR_TIMEOUT);
  } else {
#pragma unroll
    for (int ii = 0; ii < 64; ++ii) Hg[(i0 + ii) * kD + j] = Hr[ii];
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, 512);
}

}  // namespace

size_t prefill_tc_smem_bytes() { return TcSmem::kAlloc; }

cudaError_t launch_prefill_tc(const PrefillParams& p, cudaStream_t stream) {
  auto kern = gdn_prefill_tc_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(TcSmem::kAlloc));
  if (e != cudaSuccess) return e;
  if (p.n > 0) kern<<<p.n * p.Hv, kThreads, TcSmem::kAlloc, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
