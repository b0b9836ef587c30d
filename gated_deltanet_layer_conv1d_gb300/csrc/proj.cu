// proj.cu -- the bf16 projections on either side of the GDN mixer (sm_103a).
//
// layer_struct.rs, Qwen3SsmLayer: the layer projects the hidden row to [Q | K | V | Z]
// (the sequential QKVZ layout) and to the b, a gate inputs (ba_gates_k reads them), runs
// the mixer, and projects the gated-norm output y back to the hidden width (out_proj; the
// dense_gemm / dense_gemm_pipelined fields are the layer's bf16 GEMMs).  Both are one
// C[M][N] = A[M][K] B[N][K]^T with bf16 operands, f32 accumulation and a bf16 result:
//   in_proj:  A = hidden [T][H], B = [W_qkvz ; W_ba] [conv_dim + H_v d_v + 2 H_v][H]
//             -> one row [Q | K | V | Z | b | a] per token, the row layout the mixer's
//             entry points read (qkv, z, b, a are column offsets of that row);
//   out_proj: A = y [T][H_v d_v], B = W_out [H][H_v d_v] -> [T][H].
//
// gdn_proj_gemm_kernel is persistent (one CTA per SM, tiles strided over the grid) and
// warp-specialized:
//   warp 0, one lane   -- TMA producer: 128 x 64 tiles of A and BN x 64 tiles of B into a
//                         ring of STAGES shared-memory stages (128-byte swizzle, the layout
//                         the MMA descriptors read), completion on full[s];
//   warp 1, one lane   -- MMA issuer: four M128 x BN x K16 tcgen05.mma per stage into one
//                         of two TMEM accumulators, commit -> empty[s] frees the stage,
//                         commit -> tfull[acc] hands the finished tile to the epilogue;
//   warps 2..5         -- epilogue: TMEM -> registers (one row per thread), bf16, global
//                         stores, then tempty[acc] returns the accumulator.
// With two accumulators the epilogue of one tile runs under the main loop of the next.
// Rows past M and columns past N of the tiles are zero-filled by TMA and never stored;
// K past the end is zero-filled too, so K needs only 16-byte rows.
//
// Calls with two row blocks or more that take 256-wide tiles run on SM pairs instead (the
// pair kernel further down: 256 x 256 tiles, tcgen05.mma.cta_group::2).
//
// Calls with fewer tiles than SMs (a decode step's 128 tokens) split K instead: a cluster
// of `splits` CTAs per tile, each over its own run of K blocks.  Each CTA keeps an inbox
// beside its stage ring for the partial rows of the slice of the tile it sums; as soon as
// its accumulator is complete it writes every row of its f32 partial tile from TMEM into
// the inbox of the CTA that owns the row (remote async stores that complete on that CTA's
// inbox barrier; its own rows with plain stores), and every CTA sums its slice once its
// barrier has counted every peer's bytes -- no cluster barrier after the main loop.
//
// Every wait is bounded: a wait that runs out sets a shared abort flag, every role leaves
// its loop when it sees the flag, the producer waits for the copies it issued, the issuer
// for its MMAs, and the CTA reports GDN_ERR_TIMEOUT before freeing its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace gdn {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;                     // one 128-byte swizzle row of bf16
constexpr int kProjThreads = 192;
constexpr uint32_t kATileBytes = kBM * kBK * 2;

template <int BN, bool SPLIT = false>
struct ProjCfg {
  static constexpr uint32_t kBTileBytes = uint32_t(BN) * kBK * 2;
  static constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes;
  // split-K inbox: f32 [splits][rows][BN + 4] (splits * rows <= 128 + 7): the partial rows
  // of this CTA's slice from every CTA of the cluster, its own included
  static constexpr int kRedStride = BN + 4;
  static constexpr uint32_t kInbox =
      SPLIT ? ((uint32_t(kBM + 7) * kRedStride * 4 + 1023u) / 1024u) * 1024u : 0u;
  static constexpr int kStages = int((196u * 1024u - kInbox) / kStageBytes);
  static constexpr uint32_t kRing = uint32_t(kStages) * kStageBytes;
  static constexpr uint32_t kBar = kRing + kInbox;
  // full[S], empty[S], tfull[2], tempty[2], drain, inbox; then the TMEM slot and the abort
  // flag
  static constexpr uint32_t kTmemSlot = kBar + 8u * uint32_t(2 * kStages + 6);
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kBytes = kAbort + 4 + 1024;  // + slack to align the base
  // two accumulators of BN columns, rounded up to the power of two TMEM allocates
  static constexpr uint32_t kTmemCols =
      2u * BN <= 32u ? 32u : (2u * BN <= 64u ? 64u : (2u * BN <= 128u ? 128u : (2u * BN <= 256u ? 256u : 512u)));
  static_assert(kStages >= 3, "a ring of at least three stages");
  static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "M = 128 MMA: N in 16..256, step 16");
  static_assert((kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation: a power of two");
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
        "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Waits for the phase of `bar` with the given parity; false once the CTA aborts (another
// role gave up) or this wait runs past the budget (then it raises the abort itself).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitBudgetNs) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

// All threads of all CTAs of the cluster; release / acquire orders shared memory.
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The work of one CTA: tiles first, first + stride, ... below end, each over the K blocks
// [kb0, kb1).  Without a split that is every grid-stride tile over all of K; with one it
// is tile blockIdx.x / splits over the K run of rank blockIdx.x % splits (the host makes
// every run non-empty).
struct Work {
  int first, stride, end, kb0, kb1, rank;
};
__device__ __forceinline__ Work work_of(const ProjParams& p, int tiles, int kblocks) {
  if (p.splits <= 1) return {int(blockIdx.x), int(gridDim.x), tiles, 0, kblocks, 0};
  const int r = int(blockIdx.x) % p.splits, t = int(blockIdx.x) / p.splits;
  const int kc = (kblocks + p.splits - 1) / p.splits;
  const int kb1 = (r + 1) * kc < kblocks ? (r + 1) * kc : kblocks;
  return {t, 1, t + 1, r * kc, kb1, r};
}

// Tile t's row and column block.  Tiles are walked M-fastest (the CTAs in flight share a
// weight tile and the activations stay in L2) unless the activation operand is the larger
// one (n_fast: the CTAs in flight share an activation tile and the weights stay in L2).
__device__ __forceinline__ int tile_m(const ProjParams& p, int t, int tiles_m, int tiles_n) {
  return p.n_fast ? t / tiles_n : t % tiles_m;
}
__device__ __forceinline__ int tile_n(const ProjParams& p, int t, int tiles_m, int tiles_n) {
  return p.n_fast ? t % tiles_n : t / tiles_m;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int BN, bool SPLIT>
__global__ void __launch_bounds__(kProjThreads, 1)
    gdn_proj_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                         const __grid_constant__ CUtensorMap map_b,
                         const __grid_constant__ ProjParams p) {
  using C = ProjCfg<BN, SPLIT>;
  constexpr int S = C::kStages;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::kBar);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* inbox_full = drain + 1;
  float* inbox = reinterpret_cast<float*>(sm + C::kRing);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + C::kAbort);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_m = (p.M + kBM - 1) / kBM, tiles_n = (p.N + BN - 1) / BN;
  const int tiles = tiles_m * tiles_n, kblocks = (p.K + kBK - 1) / kBK;
  const Work wk = work_of(p, tiles, kblocks);
  constexpr bool split = SPLIT;  // launched with p.splits > 1 in clusters of p.splits
  const int rows = (kBM + p.splits - 1) / p.splits;  // split: rows per CTA's slice
  const int r0 = wk.rank * rows, nr = (r0 + rows < kBM ? r0 + rows : kBM) - r0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);  // one arrive per epilogue warp
    }
    mbar_init(drain, 1);
    mbar_init(inbox_full, 1);
    // split: every other CTA of the cluster sends this CTA's nr rows of its partial tile
    if (split) mbar_arrive_expect_tx(inbox_full, uint32_t(p.splits - 1) * nr * BN * 4);
    *abort = 0;
    fence_mbar_init();
    prefetch_map(&map_a);
    prefetch_map(&map_b);
  }
  if (warp == 1) tc::alloc(tslot, C::kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  // split: this CTA's barriers are initialised; a CTA sends to a peer only after the
  // cluster barrier this arrive belongs to has completed
  if (split) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  // Every thread but the producer waits for the previous kernel in the stream at once (the
  // epilogue's stores must not overtake its reads); the producer first fetches weights.
  const bool producer = warp == 0 && lane == 0;
  if (!producer) {
    pdl_wait();
    pdl_launch_dependents();
  }

  if (producer) {
    // ---------------------------------------------------------------- TMA producer
    int s = 0;
    uint32_t ph = 0;
    uint32_t issued_mask = 0, issued_par = 0;  // per stage: a copy issued, its phase parity
    bool ok = true;
    // A weight operand: the B tiles of the first `pre` stages are on their way before the
    // wait (their stages expect both halves); every A tile waits.
    int pre = 0;
    if (p.b_weights) {
      int t = wk.first, kb = wk.kb0;
      for (; pre < S && t < wk.end; ++pre) {
        mbar_arrive_expect_tx(&full[pre], C::kStageBytes);
        tma_load_2d(sm + uint32_t(pre) * C::kStageBytes + kATileBytes, &map_b, kb * kBK,
                    tile_n(p, t, tiles_m, tiles_n) * BN, &full[pre]);
        if (++kb == wk.kb1) {
          kb = wk.kb0;
          t += wk.stride;
        }
      }
    }
    pdl_wait();
    pdl_launch_dependents();
    int idx = 0;  // loads issued, in order
    for (int t = wk.first; t < wk.end && ok; t += wk.stride) {
      const int m0 = tile_m(p, t, tiles_m, tiles_n) * kBM;
      const int n0 = tile_n(p, t, tiles_m, tiles_n) * BN;
      for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++idx) {
        unsigned char* st = sm + uint32_t(s) * C::kStageBytes;
        if (idx < pre) {  // stage s = idx: fresh, its B half already issued
          tma_load_2d(st, &map_a, kb * kBK, m0, &full[s]);
        } else {
          if (!wait_or_abort(&empty[s], ph ^ 1u, abort)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], C::kStageBytes);
          tma_load_2d(st, &map_a, kb * kBK, m0, &full[s]);
          tma_load_2d(st + kATileBytes, &map_b, kb * kBK, n0, &full[s]);
        }
        issued_mask |= 1u << s;
        issued_par = (issued_par & ~(1u << s)) | (ph << s);
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
    if (!ok) {
      // copies still in flight land before this CTA's shared memory is released
      for (int q = 0; q < S; ++q)
        if (issued_mask & (1u << q)) mbar_wait_bounded(&full[q], (issued_par >> q) & 1u);
    }

  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = tc::idesc_bf16(kBM, BN);
    int s = 0;
    uint32_t ph = 0;
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    for (int t = wk.first; t < wk.end && ok; t += wk.stride) {
      if (!wait_or_abort(&tempty[acc], aph ^ 1u, abort)) break;
      tc::fence_after_sync();
      const uint32_t d = tmem + uint32_t(acc * BN);
      for (int kb = wk.kb0; kb < wk.kb1; ++kb) {
        if (!wait_or_abort(&full[s], ph, abort)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t a = smem_u32(sm + uint32_t(s) * C::kStageBytes);
        const uint32_t b = a + kATileBytes;
#pragma unroll
        for (int k0 = 0; k0 < kBK; k0 += 16)
          tc::mma_f16(d, tc::desc_at(a, kBM, k0), tc::desc_at(b, BN, k0), idesc,
                      kb > wk.kb0 || k0 > 0);
        tc::commit(&empty[s]);
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
      tc::commit(&tfull[acc]);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    // every MMA issued above has completed before the tensor memory is freed
    tc::commit(drain);
    mbar_wait_bounded(drain, 0);
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lanes 32q .. 32q + 31
    int acc = 0;
    uint32_t aph = 0;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.C);
    for (int t = wk.first; t < wk.end; t += wk.stride) {
      const int m0 = tile_m(p, t, tiles_m, tiles_n) * kBM;
      const int n0 = tile_n(p, t, tiles_m, tiles_n) * BN;
      if (!wait_or_abort(&tfull[acc], aph, abort)) break;
      tc::fence_after_sync();
      if (split) break;  // one tile per CTA: its partial stays in TMEM for now
      const int row = m0 + 32 * q + lane;
      __nv_bfloat16* orow = out + size_t(row) * size_t(p.ldc) + n0;
      const uint32_t taddr = tmem + (uint32_t(32 * q) << 16) + uint32_t(acc * BN);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float v[32];
        tc::ld32(taddr + uint32_t(c0), v);
        if (row < p.M) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            if (n0 + c0 + 8 * g < p.N) {
              const uint4 w = make_uint4(pack_bf16x2(v[8 * g], v[8 * g + 1]),
                                         pack_bf16x2(v[8 * g + 2], v[8 * g + 3]),
                                         pack_bf16x2(v[8 * g + 4], v[8 * g + 5]),
                                         pack_bf16x2(v[8 * g + 6], v[8 * g + 7]));
              *reinterpret_cast<uint4*>(orow + c0 + 8 * g) = w;
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }

  if (split) {
    // Rows are dealt to the CTAs of the cluster in slices of `rows`.  Each epilogue thread
    // sends its row of the partial tile from TMEM to the CTA that owns the row's slice --
    // into slot [this rank] of that CTA's inbox, by remote async stores that complete on
    // the owner's inbox barrier, or by plain stores into its own inbox -- and then every
    // CTA sums its slice over the slots once its barrier says every peer's rows landed.
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // peers initialised
    if (warp >= 2) {
      const int q = warp & 3, row = 32 * q + lane, owner = row / rows;
      float* dst = inbox + (wk.rank * rows + (row - owner * rows)) * C::kRedStride;
      const bool mine = owner == wk.rank;
      uint32_t rdst = 0, rbar = 0;
      if (!mine) {
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                     : "=r"(rdst) : "r"(smem_u32(dst)), "r"(uint32_t(owner)));
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                     : "=r"(rbar) : "r"(smem_u32(inbox_full)), "r"(uint32_t(owner)));
      }
      const bool have = !*abort;  // the accumulator is complete unless the CTA aborted
      const uint32_t taddr = tmem + (uint32_t(32 * q) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BN && have; c0 += 32) {
        float v[32];
        tc::ld32(taddr + uint32_t(c0), v);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (mine) {
            *reinterpret_cast<float4*>(dst + c0 + 4 * j) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
            asm volatile(
                "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], "
                "{%1, %2, %3, %4}, [%5];"
                ::"r"(rdst + uint32_t(4 * (c0 + 4 * j))), "f"(v[4 * j]), "f"(v[4 * j + 1]),
                  "f"(v[4 * j + 2]), "f"(v[4 * j + 3]), "r"(rbar)
                : "memory");
          }
        }
      }
      named_sync(1, 128);  // this CTA's own rows are in its inbox
      if (wait_or_abort(inbox_full, 0u, abort)) {
        const int t = wk.first;
        const int m0 = tile_m(p, t, tiles_m, tiles_n) * kBM;
        const int n0 = tile_n(p, t, tiles_m, tiles_n) * BN;
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.C);
        constexpr int kQ = BN / 4;  // float4 groups per row
        for (int e = int(threadIdx.x) - 64; e < nr * kQ; e += kProjThreads - 64) {
          const int lr = e / kQ, c = 4 * (e % kQ);
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int f = 0; f < p.splits; ++f) {
            const float4 x =
                *reinterpret_cast<const float4*>(inbox + (f * rows + lr) * C::kRedStride + c);
            acc.x += x.x;
            acc.y += x.y;
            acc.z += x.z;
            acc.w += x.w;
          }
          if (m0 + r0 + lr < p.M && n0 + c < p.N)
            *reinterpret_cast<uint2*>(out + size_t(m0 + r0 + lr) * size_t(p.ldc) + n0 + c) =
                make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort) report(p.status, GDN_ERR_TIMEOUT);
  if (warp == 1) tc::dealloc(tmem, C::kTmemCols);
}

// ------------------------------------------------------------------ SM pairs
// Large calls (two row blocks or more, 256-wide tiles) run on SM pairs: a cluster of two
// CTAs computes one 256 x 256 tile with tcgen05.mma.cta_group::2.  CTA r of the pair loads
// rows r*128 .. r*128+127 of the tile's A block and of its B block into its own shared
// memory; both copies complete on the even (leader) CTA's full barrier, the leader's one
// thread issues the M = 256 MMAs that read both CTAs' halves, and its commits arrive on
// the stage and accumulator barriers of both CTAs at once.  Each CTA's TMEM holds its 128
// rows of the 256 x 256 accumulator, which its own epilogue warps store; they report back
// to the leader's tempty barrier.  Per SM and K block that is 32 KB of operands for a
// 128 x 256 x 64 product instead of 48 KB, and six stages fit where four did.
struct PairCfg {
  static constexpr uint32_t kHalfTile = 128u * kBK * 2;      // 128 rows x 64 bf16
  static constexpr uint32_t kStageBytes = 2 * kHalfTile;     // this CTA's A and B halves
  static constexpr int kStages = 6;
  static constexpr uint32_t kBar = uint32_t(kStages) * kStageBytes;
  static constexpr uint32_t kTmemSlot = kBar + 8u * uint32_t(2 * kStages + 5);
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kBytes = kAbort + 4 + 1024;
  static constexpr int kAccs = 2;             // 256-column accumulators in TMEM
  static constexpr uint32_t kTmemCols = 256u * kAccs;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  return ra;
}
// A tile into this CTA's shared memory, completing on a barrier of either CTA of the pair
// (bar: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// Arrives on the barrier at this offset in both CTAs of the pair once the MMAs issued
// before have completed.
__device__ __forceinline__ void commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)), "h"(uint16_t(3))
      : "memory");
}
__device__ __forceinline__ void commit_pair_local(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
      ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void arrive_remote(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
               : "memory");
}

__global__ void __launch_bounds__(kProjThreads, 1)
    gdn_proj_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a,
                              const __grid_constant__ CUtensorMap map_b,
                              const __grid_constant__ ProjParams p) {
  using C = PairCfg;
  constexpr int S = C::kStages;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::kBar);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + C::kAbort);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int tiles_m = (p.M + 255) / 256, tiles_n = (p.N + 255) / 256;
  const int tiles = tiles_m * tiles_n, kblocks = (p.K + kBK - 1) / kBK;
  const int pair = int(blockIdx.x) >> 1, pairs = int(gridDim.x) >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);  // the four epilogue warps of each CTA of the pair
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
    prefetch_map(&map_a);
    prefetch_map(&map_b);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tslot)), "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either signals the other's
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  pdl_wait();  // everything below may read what the previous kernel in the stream wrote
  pdl_launch_dependents();

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = pair; t < tiles && ok; t += pairs) {
      const int mb = p.n_fast ? t / tiles_n : t % tiles_m;
      const int nb = p.n_fast ? t % tiles_n : t / tiles_m;
      const int m0 = mb * 256 + int(rank) * 128, n0 = nb * 256 + int(rank) * 128;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_or_abort(&empty[s], ph ^ 1u, abort)) { ok = false; break; }
        unsigned char* st = sm + uint32_t(s) * C::kStageBytes;
        if (leader) mbar_arrive_expect_tx(&full[s], 2 * C::kStageBytes);
        const uint32_t fb = peer_addr(&full[s], 0);
        tma_load_2d_pair(st, &map_a, kb * kBK, m0, fb);
        tma_load_2d_pair(st + C::kHalfTile, &map_b, kb * kBK, n0, fb);
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
    if (!ok && leader) {
      // the pair's copies still in flight land before shared memory is released
      for (int q = 0; q < S; ++q) mbar_wait_bounded(&full[q], 0, kWaitBudgetNs / 8);
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ---------------------------------------------------------------- MMA issuer (leader)
    constexpr uint32_t idesc = tc::idesc_bf16(256, 256);
    int s = 0;
    uint32_t ph = 0;
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    for (int t = pair; t < tiles && ok; t += pairs) {
      if (!wait_or_abort(&tempty[acc], aph ^ 1u, abort)) break;
      tc::fence_after_sync();
      const uint32_t d = tmem + uint32_t(acc * 256);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_or_abort(&full[s], ph, abort)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t a = smem_u32(sm + uint32_t(s) * C::kStageBytes);
        const uint32_t b = a + C::kHalfTile;
#pragma unroll
        for (int k0 = 0; k0 < kBK; k0 += 16)
          mma_pair(d, tc::desc_at(a, 128, k0), tc::desc_at(b, 128, k0), idesc, kb > 0 || k0 > 0);
        commit_pair(&empty[s]);
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
      commit_pair(&tfull[acc]);
      if (++acc == C::kAccs) {
        acc = 0;
        aph ^= 1u;
      }
    }
    commit_pair_local(drain);
    mbar_wait_bounded(drain, 0);
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lanes 32q .. 32q + 31 of this CTA's 128 rows
    int acc = 0;
    uint32_t aph = 0;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.C);
    for (int t = pair; t < tiles; t += pairs) {
      const int mb = p.n_fast ? t / tiles_n : t % tiles_m;
      const int nb = p.n_fast ? t % tiles_n : t / tiles_m;
      const int n0 = nb * 256;
      if (!wait_or_abort(&tfull[acc], aph, abort)) break;
      tc::fence_after_sync();
      const int row = mb * 256 + int(rank) * 128 + 32 * q + lane;
      __nv_bfloat16* orow = out + size_t(row) * size_t(p.ldc) + n0;
      const uint32_t taddr = tmem + (uint32_t(32 * q) << 16) + uint32_t(acc * 256);
#pragma unroll 1
      for (int c0 = 0; c0 < 256; c0 += 32) {
        float v[32];
        tc::ld32(taddr + uint32_t(c0), v);
        if (row < p.M) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            if (n0 + c0 + 8 * g < p.N) {
              const uint4 w = make_uint4(pack_bf16x2(v[8 * g], v[8 * g + 1]),
                                         pack_bf16x2(v[8 * g + 2], v[8 * g + 3]),
                                         pack_bf16x2(v[8 * g + 4], v[8 * g + 5]),
                                         pack_bf16x2(v[8 * g + 6], v[8 * g + 7]));
              *reinterpret_cast<uint4*>(orow + c0 + 8 * g) = w;
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive_remote(peer_addr(&tempty[acc], 0));
      if (++acc == C::kAccs) {
        acc = 0;
        aph ^= 1u;
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  cluster_sync();  // the pair's MMAs, copies and remote arrivals are done
  tc::fence_after_sync();
  if (threadIdx.x == 0 && *abort) report(p.status, GDN_ERR_TIMEOUT);
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kTmemCols)
                 : "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // the driver's entry point, looked up once per process (calls may come from any thread)
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
  if (!f) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    fn.store(f, std::memory_order_release);
  }
  return f;
}

// A row-major bf16 matrix [rows][cols] (row stride ld elements) read in boxes of
// box_rows x 64 with the 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int rows, int cols, int64_t ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(ld) * 2};
  const cuuint32_t box[2] = {cuuint32_t(kBK), cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int BN, bool SPLIT>
cudaError_t launch_bn(const ProjParams& p, cudaStream_t stream) {
  using C = ProjCfg<BN, SPLIT>;
  CUtensorMap ma, mb;
  if (!make_map(&ma, p.A, p.M, p.K, p.lda, kBM) || !make_map(&mb, p.B, p.N, p.K, p.ldb, BN))
    return cudaErrorInvalidValue;
  auto kern = gdn_proj_gemm_kernel<BN, SPLIT>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kBytes));
  if (e != cudaSuccess) return e;
  const int tiles = ((p.M + kBM - 1) / kBM) * ((p.N + BN - 1) / BN);
  if (!SPLIT) {
    const int grid = tiles < sm_count() ? tiles : sm_count();
    return launch_pdl(kern, dim3(unsigned(grid)), dim3(kProjThreads), C::kBytes, stream, 1u, ma,
                      mb, p);
  }
  return launch_pdl(kern, dim3(unsigned(tiles * p.splits)), dim3(kProjThreads), C::kBytes,
                    stream, unsigned(p.splits), ma, mb, p);
}

// Clusters of s CTAs of the split kernel of width BN the current GPU holds at once.
template <int BN>
int query_active_clusters(int s) {
  int n = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(s));
  cfg.blockDim = dim3(kProjThreads);
  cfg.dynamicSmemBytes = ProjCfg<BN, true>::kBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(s);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaFuncSetAttribute(gdn_proj_gemm_kernel<BN, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(ProjCfg<BN, true>::kBytes));
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, gdn_proj_gemm_kernel<BN, true>, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  return n;
}

// How many clusters of `s` CTAs of the BN-wide split kernel the current GPU holds at once
// (a cluster stays inside one GPC, so this is below SMs / s); cached per device and shape.
// Splits run at widths 128, 96 and 64 (a 256-wide split leaves no room for a ring).
constexpr int kProjMaxDevices = 64;
int max_active_clusters(int bn, int s) {
  static std::atomic<int> cache[kProjMaxDevices][3][9];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kProjMaxDevices) return -1;
  if (bn != 128 && bn != 96 && bn != 64) return -1;
  const int i = bn == 128 ? 0 : (bn == 96 ? 1 : 2);
  int cached = cache[dev][i][s].load(std::memory_order_relaxed);
  if (cached == 0) {
    const int n = bn == 128 ? query_active_clusters<128>(s)
                            : (bn == 96 ? query_active_clusters<96>(s) : query_active_clusters<64>(s));
    cached = n > 0 ? n : -1;  // -1: this split is not available
    cache[dev][i][s].store(cached, std::memory_order_relaxed);
  }
  return cached;
}

// How many SM pairs of the pair kernel the current GPU holds at once; cached per device.
int max_active_pairs() {
  static std::atomic<int> cache[kProjMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kProjMaxDevices) return -1;
  int cached = cache[dev].load(std::memory_order_relaxed);
  if (cached == 0) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kProjThreads);
    cfg.dynamicSmemBytes = PairCfg::kBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaFuncSetAttribute(gdn_proj_gemm_pair_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(PairCfg::kBytes));
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, gdn_proj_gemm_pair_kernel, &cfg);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    cached = n > 0 ? n : -1;
    cache[dev].store(cached, std::memory_order_relaxed);
  }
  return cached;
}

cudaError_t launch_pair(const ProjParams& p, cudaStream_t stream) {
  using C = PairCfg;
  CUtensorMap ma, mb;
  if (!make_map(&ma, p.A, p.M, p.K, p.lda, 128) || !make_map(&mb, p.B, p.N, p.K, p.ldb, 128))
    return cudaErrorInvalidValue;
  auto kern = gdn_proj_gemm_pair_kernel;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kBytes));
  if (e != cudaSuccess) return e;
  const int tiles = ((p.M + 255) / 256) * ((p.N + 255) / 256);
  const int max_pairs = max_active_pairs();
  if (max_pairs <= 0) return cudaErrorInvalidConfiguration;
  const int pairs = tiles < max_pairs ? tiles : max_pairs;
  return launch_pdl(kern, dim3(unsigned(2 * pairs)), dim3(kProjThreads), C::kBytes, stream, 2u,
                    ma, mb, p);
}

}  // namespace

ProjShape proj_shape(int M, int N, int K) {
  // Cost of a choice, in operand rows x K blocks through the busiest SM: a tile of BN
  // columns streams 128 + BN rows per K block.  Whole-K tiles run in waves over the SMs;
  // a split of S (one wave of tiles x S CTAs, at most 8 to a cluster, every K run
  // non-empty) pays ceil(K blocks / S) blocks plus its partial-tile round trip through
  // shared memory, measured at about 32 BN; every cluster of it has to be resident at once
  // (a cluster stays inside one GPC).  Least cost wins; on a tie the wider tile, then no
  // split.
  const int sms = sm_count();
  const int tm = (M + kBM - 1) / kBM, kblocks = (K + kBK - 1) / kBK;
  ProjShape best{256, 1};
  long best_cost = -1;
  auto consider = [&](int bn, int s, long cost) {
    if (best_cost < 0 || cost < best_cost) {
      best = {bn, s};
      best_cost = cost;
    }
  };
  for (int bn : {256, 128, 96, 64}) {
    const long tiles = long(tm) * ((N + bn - 1) / bn);
    consider(bn, 1, ((tiles + sms - 1) / sms) * (kBM + bn) * long(kblocks));
    for (int s = 2; s <= 8 && tiles * s <= sms; ++s) {
      const int kc = (kblocks + s - 1) / s;
      if ((s - 1) * kc >= kblocks || tiles > max_active_clusters(bn, s)) continue;
      consider(bn, s, long(kBM + bn) * kc + 32L * bn);
    }
  }
  return best;
}

cudaError_t launch_proj(const ProjParams& p_in, cudaStream_t stream) {
  if (p_in.M == 0 || p_in.N == 0) return cudaSuccess;
  ProjParams p = p_in;
  if (p.bn == 0) {
    const ProjShape sh = proj_shape(p.M, p.N, p.K);
    p.bn = sh.bn;
    p.splits = sh.splits;
  }
  if (p.splits < 1 || p.splits > 8) return cudaErrorInvalidValue;
  p.n_fast = p.M > p.N ? 1 : 0;  // A (M x K) larger than B (N x K)
  if (p.bn == 256 && p.splits == 1 && p.M > kBM && max_active_pairs() > 0)
    return launch_pair(p, stream);
  if (p.splits > 1) {
    switch (p.bn) {
      case 128: return launch_bn<128, true>(p, stream);
      case 96: return launch_bn<96, true>(p, stream);
      case 64: return launch_bn<64, true>(p, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (p.bn) {
    case 256: return launch_bn<256, false>(p, stream);
    case 128: return launch_bn<128, false>(p, stream);
    case 96: return launch_bn<96, false>(p, stream);
    case 64: return launch_bn<64, false>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
