// kernels.h -- host-side declarations of the GDN kernel launchers (internal to libgdn.so).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr int kMaxG = 4;  // value heads per key head a launch supports

// Parameters of the fused decode / verify kernel (by value, in the constant bank).
struct RecParams {
  int32_t Hk, Hv, G, conv_dim, n, n_slots;
  float q_scale, l2_eps, norm_eps;
  int32_t norm_gate;  // 0: SiLU(z), 1: sigmoid(z)
  const float* conv_w;
  const float* A_log;
  const float* dt_bias;
  const float* norm_w;
  const void* qkv;
  int64_t qkv_stride;
  const void* z;
  int64_t z_stride;
  const void* a;
  const void* b;
  int64_t ab_stride;
  void* h_pool;            // decode: [n_slots][Hv][D][D], f32 or fp16 elements
  const uint64_t* tables;  // verify: [16][128]
  void* conv_pool;         // [n_slots][conv_dim][4]
  const int32_t* slots;    // [n]
  void* conv_inter;        // verify, nullable: [n][15][conv_dim][4]
  void* y;
  float* core_out;
  int32_t* status;
  int32_t n_items;         // n * Hk
  // Write-on-accept verify (woa_stash non-null): no state is written; sequence i's stash
  // at woa_stash + i * woa_seq_bytes receives k, and per token alpha, k_hat, delta and the
  // raw qkv row (byte offsets below); every CTA sets *woa_flag to 1 at its end.
  unsigned char* woa_stash;
  uint32_t* woa_flag;
  int64_t woa_seq_bytes;
  int32_t woa_alpha, woa_khat, woa_delta, woa_raw;
  uint8_t ks[GDN_MAX_SEQS];       // tokens of sequence i (original index)
  uint8_t order[GDN_MAX_SEQS];    // sequence indices, most tokens first
  uint16_t row_off[GDN_MAX_SEQS]; // first token row of sequence i
};

// Fused conv + L2 + gates + recurrence + gated norm, one launch for all sequences.
// h16: the state pool / tables hold fp16 elements (f32 arithmetic).
cudaError_t launch_recurrent(const RecParams& p, int dtype, int D, bool verify, bool h16,
                             cudaStream_t stream);
// Element-wise conversion between f32 and fp16 state pools (round to nearest even).
cudaError_t launch_state_convert(const void* src, int src_dtype, void* dst, int dst_dtype,
                                 size_t count, cudaStream_t stream);

// Conv + SiLU + L2 norm over T tokens of n sequences -> f32 [T][conv_dim]
// (or bf16 when out_bf16), then the conv-state update.
struct ConvParams {
  int32_t Hk, Hv, D, conv_dim, n, n_slots, total_tokens;
  float q_scale, l2_eps;
  const float* conv_w;
  const void* qkv;
  int64_t qkv_stride;
  const int32_t* cu_seqlens;
  void* conv_pool;
  const int32_t* slots;
  void* out;
  int32_t out_bf16;
  int32_t* status;
  // Chunked-prefill pre-pass only: gates and the workspace tiles.
  const float* A_log;
  const float* dt_bias;
  const void* a;
  const void* b;
  int64_t ab_stride;
  void* workspace;
};
cudaError_t launch_conv_step(const ConvParams& p, int dtype, cudaStream_t stream);
// Pre-pass of the tensor-core prefill: conv, SiLU, L2 norms and gates of every token into
// the workspace tiles (bf16 activations, d = 128).
cudaError_t launch_prefill_prep(const ConvParams& p, cudaStream_t stream);

// o: f32, or fp16 when o_half (the prefill's internal hand-off of O to the norm).
cudaError_t launch_gated_rmsnorm(const void* o, bool o_half, const void* z, int64_t z_stride,
                                 const float* w, float eps, int T, int Hv, int D, int dtype,
                                 int gate, void* y, cudaStream_t stream);

// Chunked prefill.
struct PrefillParams {
  int32_t Hk, Hv, G, D, conv_dim, n, n_slots, total_tokens, max_seqlen, max_chunks;
  void* o_half;  // internal: fp16 [T][Hv][128] room for O when no f32 core output is wanted
  int32_t* counts;  // internal: [n][Hv][2] chunks of O each column slice has stored
  float q_scale, l2_eps, norm_eps;
  int32_t norm_gate;  // 0: SiLU(z), 1: sigmoid(z)
  int32_t f32_path;   // 1: the token-sequential f32 form even where the tensor-core form runs
  const float* conv_w;
  const float* A_log;
  const float* dt_bias;
  const float* norm_w;
  const void* qkv;
  int64_t qkv_stride;
  const void* z;
  int64_t z_stride;
  const void* a;
  const void* b;
  int64_t ab_stride;
  const int32_t* cu_seqlens;
  const uint64_t* h_ptrs;
  void* conv_pool;
  const int32_t* slots;
  void* y;
  float* core_out;
  int32_t* status;
  void* workspace;
  size_t workspace_bytes;
};
size_t prefill_workspace_bytes(int Hk, int Hv, int D, int n, int total_tokens,
                               int max_seqlen);
cudaError_t launch_prefill(const PrefillParams& p, int dtype, cudaStream_t stream);

// Accepted-draft fold after a ragged verify.
struct FoldParams {
  int32_t Hv, d_k, d_v, conv_dim, d_conv, esize, h_esize, n, n_slots;
  const int32_t* accepted;  // [n] device
  const uint64_t* tables;   // [16][128]
  void* conv_pool;
  const int32_t* slots;
  const void* conv_inter;   // [n][15][conv_dim][d_conv]
  int32_t* status;
  uint8_t ks[GDN_MAX_SEQS];
};
cudaError_t launch_fold(const FoldParams& p, cudaStream_t stream);

// Write-on-accept stash of one sequence (byte offsets; see RecParams), sized for
// GDN_VERIFY_K_MAX tokens.
struct WoaLayout {
  int64_t alpha, khat, delta, raw, seq_bytes;
};
WoaLayout woa_layout(int Hk, int Hv, int dk, int dv, int conv_dim, int esize);

// The deferred fold of a write-on-accept verify: sequence i's state (table 0 entry i) takes
// the first accepted[i] tokens' updates from its stash, and its conv state the last d_conv
// raw inputs up to that token; nothing happens while *flag is 0.
struct WoaFoldParams {
  int32_t Hk, Hv, d, conv_dim, esize, n, n_slots;
  const int32_t* accepted;   // [n] device
  const uint64_t* tables;    // [16][128]; table 0 only
  void* conv_pool;
  const int32_t* slots;
  const unsigned char* stash;
  const uint32_t* flag;
  int32_t* status;
  WoaLayout lay;
};
cudaError_t launch_woa_fold(const WoaFoldParams& p, cudaStream_t stream);
cudaError_t launch_woa_clear(uint32_t* flag, cudaStream_t stream);

// bf16 projection GEMM: C[M][N] = A[M][K] B[N][K]^T (f32 accumulation, bf16 result).
struct ProjParams {
  const void* A;
  int64_t lda;
  const void* B;
  int64_t ldb;
  void* C;
  int64_t ldc;
  int32_t M, N, K;
  int32_t bn;      // output tile width 256 / 128 / 96 / 64; 0: the launcher picks bn and splits
  int32_t splits;  // CTAs (one cluster) per tile splitting K, 1..8
  int32_t n_fast;  // tile order: 1 walks N fastest, 0 walks M fastest
  // 1: B is a weight matrix that no kernel writes, so its first tiles are fetched before
  // the previous kernel in the stream has finished (programmatic dependent launch)
  int32_t b_weights;
  int32_t* status;
};
struct ProjShape {
  int bn, splits;
};
cudaError_t launch_proj(const ProjParams& p, cudaStream_t stream);
ProjShape proj_shape(int M, int N, int K);

cudaError_t launch_wait_selftest(uint64_t budget_ns, int32_t* status, cudaStream_t stream);

int sm_count();

}  // namespace gdn
