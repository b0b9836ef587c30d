/*
 * gdn.h -- C ABI of libgdn.so, the Gated DeltaNet (GDN) token mixer for GB300 (sm_103a).
 *
 * One GDN layer's token mixer, as the `qwen3_ssm` layer of the reference engine runs it:
 *   causal depthwise conv over the raw [Q|K|V] channels, SiLU, per-key-head L2 norm of
 *   q and k (layer_struct.rs, Qwen3SsmLayer::conv1d_l2norm_f32_k);
 *   gates alpha = exp(-exp(A_log) * softplus(a + dt_bias)), beta = sigmoid(b)
 *   (layer_struct.rs, ba_gates_k / compute_gdn_gates_k);
 *   the gated delta rule on an f32 state S (d_v x d_k) per value head,
 *       S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t
 *   (layer_struct.rs, gdn_f32_k and its strided / WY / prefill variants);
 *   the Z-gated RMSNorm y = o / sqrt(mean(o^2) + eps) * w * SiLU(z)
 *   (layer_struct.rs, gated_rms_norm_f32_k).
 *
 * Conventions shared by every entry point
 *   - Ownership: the caller owns every buffer.  The library allocates nothing, keeps no
 *     state between calls and never synchronises; every GPU call is enqueued on `stream`.
 *   - Errors: arguments are validated on the host first; on any error the call returns
 *     a nonzero gdn_status and launches nothing (trait_layer.rs, the module invariant
 *     that a refused mode "returns an error and launches nothing").  Problems only the
 *     device can see (a NULL or misaligned table entry, a slot out of range, bad
 *     cu_seqlens, a bounded wait that ran out) are written by the kernel to the
 *     caller's device status word `*status_dev` -- the first error wins, the kernel
 *     skips the affected work and returns normally; it never traps.  The caller zeroes
 *     the word before the call and reads it afterwards.
 *   - Stream order: the decode / verify kernels and the projection GEMMs are launched with
 *     programmatic stream serialization.  Each one lets the next kernel in the stream
 *     start on the SMs it leaves once it has itself waited for the kernel before it, and
 *     reads nothing another kernel may have written until that kernel has finished --
 *     except read-only weights: the gated-norm weight (decode / verify) and the weight
 *     operand of gdn_in_proj / gdn_out_proj, which may be fetched while the previous
 *     kernel in the stream is still running.  A caller that rewrites those weights does so
 *     with a kernel or copy that is not the last work before the call (any kernel of its
 *     own does: it does not trigger early) -- in practice nothing changes for a caller.
 *     The tensor-core prefill of few sequences (2 n H_v <= half the SMs) ends in one
 *     cooperative launch that takes every SM for its length (the state chains and, beside
 *     them, the gated norm); kernels on other streams share the GPU with it only before
 *     and after.  Where the context may not use every SM, it runs as two plain launches.
 *   - Pointers marked "device" are CUDA device (or managed) memory; "host" is host memory.
 *   - Row strides are in ELEMENTS of the activation dtype.
 *   - Supported shapes: (d_k, d_v) in {(16, 16), (128, 128)}, d_conv = 4,
 *     n_v_heads a multiple of n_k_heads with G = n_v_heads / n_k_heads <= 4 (<= 3 for
 *     gdn_verify_multi, whose per-token staging must fit in shared memory).
 *
 * Layouts (readings of the reference pages; the design notes list each one)
 *   raw QKV row  [conv_dim] = [Q: n_k_heads*d_k | K: n_k_heads*d_k | V: n_v_heads*d_v],
 *                each head's channels contiguous (layer_struct.rs, Qwen3SsmLayer doc:
 *                the QKVZ projection is brought into [Q | K | V | Z] order);
 *   Z row        [n_v_heads*d_v];   a, b rows [n_v_heads];
 *   value head h reads key head h / G;
 *   h state of one sequence [n_v_heads][d_k][d_v] f32, element (i, j) = S[j][i]
 *                (layer_struct.rs, h_state_bytes = nv * kd * vd values);
 *   conv state of one sequence [conv_dim][d_conv] in the activation dtype, the last
 *                d_conv raw inputs of each channel, oldest first (layer_struct.rs,
 *                conv_state_bytes = conv_dim * d_conv values); conv_w[c][d_conv-1]
 *                multiplies the newest input;
 *   y row        [n_v_heads*d_v] in the activation dtype.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

/* A CUDA stream: the same type as cudaStream_t.  NULL is the legacy default stream. */
typedef struct CUstream_st* gdn_stream_t;

typedef int32_t gdn_status;

/* Host-side status codes (returned). */
#define GDN_OK 0
#define GDN_ERR_INVALID_ARGUMENT 1   /* a count, size, stride, eps or enum out of range */
#define GDN_ERR_UNSUPPORTED_DIMS 2   /* head dims / conv width / G not built (see above) */
#define GDN_ERR_NULL_POINTER 3       /* a required pointer is NULL */
#define GDN_ERR_MISALIGNED 4         /* a pointer or stride breaks the alignment rule */
#define GDN_ERR_BAD_K 5              /* a verify k outside 2..16 */
#define GDN_ERR_TOO_MANY_SEQS 6      /* more than GDN_MAX_SEQS sequences in one call */
#define GDN_ERR_WORKSPACE_TOO_SMALL 7
#define GDN_ERR_CUDA 8               /* a CUDA runtime call (launch, attribute) failed */
#define GDN_ERR_SCRATCH_TOO_SMALL 9  /* the call needs more than the library's static scratch */
/* Device-side codes (written to *status_dev by a kernel). */
#define GDN_ERR_BAD_TABLE_ENTRY 16   /* verify: a needed table entry is NULL or not 16-B aligned */
#define GDN_ERR_BAD_SLOT 17          /* a slot index outside [0, n_slots) */
#define GDN_ERR_BAD_SEQLENS 18       /* cu_seqlens not monotone / not matching the sizes */
#define GDN_ERR_TIMEOUT 19           /* a bounded device-side wait ran out */
#define GDN_ERR_BAD_ACCEPTED 20      /* fold: an accepted count outside 1..k */

/* Activation dtypes (raw QKV, Z, a, b, the conv state and the output y). */
#define GDN_DTYPE_F32 0
#define GDN_DTYPE_BF16 1
#define GDN_DTYPE_F16 2   /* h-state pools only (the *_h16 entry points, gdn_state_convert) */

/* Most sequences one batched decode or verify call holds, and the WY pointer-table
 * layout of the batched verify (transformer_layer.rs, VERIFY_WY_TABLE_SEQS = 128,
 * VERIFY_WY_TABLES_PER_LAYER = 16, VERIFY_WY_TABLE_STRIDE_BYTES = SEQS * 8,
 * VERIFY_WY_LAYER_STRIDE_BYTES = TABLES * TABLE_STRIDE): per layer, 16 tables of 128
 * u64 entries lie back to back; table 0 holds each sequence's h state, table t + 1 its
 * intermediate t; entries a call does not use stay zero; strides do not depend on k. */
#define GDN_MAX_SEQS 128
#define GDN_VERIFY_WY_TABLE_SEQS 128
#define GDN_VERIFY_WY_TABLES_PER_LAYER 16
#define GDN_VERIFY_WY_TABLE_STRIDE_BYTES (GDN_VERIFY_WY_TABLE_SEQS * 8)
#define GDN_VERIFY_WY_LAYER_STRIDE_BYTES \
  (GDN_VERIFY_WY_TABLES_PER_LAYER * GDN_VERIFY_WY_TABLE_STRIDE_BYTES)
#define GDN_VERIFY_K_MIN 2
#define GDN_VERIFY_K_MAX 16
#define GDN_PREFILL_CHUNK 64

typedef struct {
  int32_t n_k_heads; /* H_k */
  int32_t n_v_heads; /* H_v, a multiple of H_k */
  int32_t d_k;
  int32_t d_v;
  int32_t d_conv;    /* conv width; 4 */
  float q_scale;     /* q <- q / sqrt(sum q^2 + l2_eps) * q_scale */
  float l2_eps;      /* >= 0 */
  float norm_eps;    /* gated RMSNorm epsilon, >= 0 */
  int32_t norm_gate; /* GDN_NORM_GATE_SILU (0): y = norm(o) w SiLU(z);
                        GDN_NORM_GATE_SIGMOID (1): y = norm(o) w sigmoid(z), the gate of the
                        gdn_norm_sigmoid models (layer_struct.rs, gated_rms_norm_f32_strided_k) */
  int32_t prefill_precision; /* gdn_prefill_chunked at d = 128 with bf16 activations:
                        GDN_PREFILL_TENSOR_FP16 (0): the chunked WY form on the tensor cores,
                        fp16 operands (state error ~4e-4 relative);
                        GDN_PREFILL_F32 (1): the token-sequential f32 form on CUDA cores (the
                        1e-4 class of the decode and verify paths; no workspace), far slower.
                        Every other entry point ignores it. */
} gdn_dims;

#define GDN_NORM_GATE_SILU 0
#define GDN_NORM_GATE_SIGMOID 1
#define GDN_PREFILL_TENSOR_FP16 0
#define GDN_PREFILL_F32 1

/* Layer parameters, all f32 device memory. */
typedef struct {
  const float* conv_w;  /* [conv_dim][d_conv] */
  const float* A_log;   /* [n_v_heads] */
  const float* dt_bias; /* [n_v_heads] */
  const float* norm_w;  /* [d_v], shared by all value heads */
} gdn_weights;

/* Per-token activations, device memory, rows in token order (sequence-major when a call
 * holds several sequences).  Base pointers of qkv and z are 16-byte aligned and their
 * row strides (in elements) are multiples of 16 bytes; a and b are element aligned. */
typedef struct {
  const void* qkv;    /* [T][qkv_stride], the first conv_dim elements of a row are used */
  int64_t qkv_stride;
  const void* z;      /* [T][z_stride], the first n_v_heads*d_v elements are used */
  int64_t z_stride;
  const void* a;      /* [T][ab_stride], decay logits (first n_v_heads elements) */
  const void* b;      /* [T][ab_stride], write-strength logits */
  int64_t ab_stride;
  int32_t dtype;      /* GDN_DTYPE_*: dtype of qkv, z, a, b, the conv state and y */
} gdn_inputs;

/* Batched single-token decode across n sequences (trait_layer.rs,
 * TransformerLayer::decode_batched / decode_multi_seq; layer_struct.rs, the strided
 * conv1d_l2norm_f32_strided_k, gdn_f32_strided_norm_k and
 * gated_rms_norm_f32_strided_k, here fused into one launch).
 *   inputs    : n rows, row i is sequence i's token.
 *   h_pool    : device [n_slots][n_v_heads][d_k][d_v] f32, 16-B aligned; the state of
 *               sequence i is slot slots_dev[i], read and written in place.
 *   conv_pool : device [n_slots][conv_dim][d_conv] in inputs->dtype, updated in place.
 *   slots_dev : device int32 [n]; distinct slots (a repeated slot races).
 *   y         : device [n][n_v_heads*d_v] in inputs->dtype.
 *   core_out  : device f32 [n][n_v_heads][d_v] (o before the norm), or NULL.
 *   status_dev: device int32 status word (see conventions).
 * Returns GDN_ERR_TOO_MANY_SEQS for n > GDN_MAX_SEQS; n == 0 is a no-op. */
GDN_API gdn_status gdn_decode_batched(const gdn_dims* dims, const gdn_weights* weights,
                              const gdn_inputs* inputs, int32_t n, float* h_pool,
                              void* conv_pool, int32_t n_slots, const int32_t* slots_dev,
                              void* y, float* core_out, int32_t* status_dev,
                              gdn_stream_t stream);

/* Ragged speculative verify: sequence i runs ks_host[i] draft tokens in one launch
 * (trait_layer.rs, TransformerLayer::decode_verify_multi; layer_struct.rs, the
 * pointer-table wyN kernels gdn_wyn_table_k and the snapshot-writing
 * gdn_f32_strided_norm_snap_k).  Sequence i starts from the state that table 0 entry i
 * points to, and after its t+1-th token (t = 0 .. k_i-2) writes the state to table t+1
 * entry i ("intermediate t"); the state after all k_i tokens is written back to table 0
 * entry i.  Intermediate t equals t+1 sequential decode steps.
 *   n          : 1 .. GDN_MAX_SEQS sequences.
 *   ks_host    : host int32 [n], each in 2..16; rows are sequence-major, sequence i
 *                owns rows sum(ks[:i]) .. + ks[i] of inputs, y and core_out.
 *   wy_tables_dev: device u64 [16][128], this layer's slice.  Each entry used points to
 *                a [n_v_heads][d_k][d_v] f32 state, 16-B aligned.  Entries the call does
 *                not use are never read.  A NULL or misaligned needed entry sets
 *                GDN_ERR_BAD_TABLE_ENTRY and that sequence is skipped.  The tables
 *                themselves are never written.
 *   conv_pool, n_slots, slots_dev: as in decode; the conv state ends after all k_i
 *                tokens.
 *   conv_inter : device [n][15][conv_dim][d_conv] in inputs->dtype, or NULL: the conv
 *                state after token t+1 (t = 0 .. k_i-2), for rolling back to an
 *                accepted prefix.
 *   y, core_out, status_dev: as in decode, with sum(ks) rows. */
GDN_API gdn_status gdn_verify_multi(const gdn_dims* dims, const gdn_weights* weights,
                            const gdn_inputs* inputs, int32_t n, const int32_t* ks_host,
                            const uint64_t* wy_tables_dev, void* conv_pool, int32_t n_slots,
                            const int32_t* slots_dev, void* conv_inter, void* y,
                            float* core_out, int32_t* status_dev, gdn_stream_t stream);

/* Folds the accepted drafts of a ragged verify into each sequence's state (trait_layer.rs,
 * LayerWriteOnAccept::gdn_fold_accepted over the h-state table and a device table of
 * accepted counts; layer_struct.rs, the fold kernel gdn_wy4_fold_k).  After
 * gdn_verify_multi ran sequence i over k_i draft tokens, the caller accepted the first
 * m_i = accepted_dev[i] of them (1 <= m_i <= k_i).  When m_i < k_i the state after m_i
 * tokens replaces the state after all k_i: table 0 entry i receives a copy of the state
 * table m_i entry i points to (intermediate m_i - 1), and the conv state of slot
 * slots_dev[i] receives conv_inter[i][m_i - 1].  When m_i == k_i nothing is written.
 *   n, ks_host  : the verify's sequence count and draft counts (each 2..16).
 *   accepted_dev: device int32 [n]; a count outside 1..k_i sets GDN_ERR_BAD_ACCEPTED and
 *                 that sequence is left as it is.
 *   wy_tables_dev, conv_pool, n_slots, slots_dev: as passed to gdn_verify_multi; a NULL or
 *                 misaligned table entry it needs sets GDN_ERR_BAD_TABLE_ENTRY.
 *   conv_inter  : the conv intermediates that gdn_verify_multi wrote (required here),
 *                 [n][15][conv_dim][d_conv] in `dtype`.
 *   dtype       : the activation dtype of the verify (GDN_DTYPE_BF16 or GDN_DTYPE_F32).
 *   h_dtype     : the states' element type: GDN_DTYPE_F32, or GDN_DTYPE_F16 after
 *                 gdn_verify_multi_h16. */
GDN_API gdn_status gdn_fold_accepted(const gdn_dims* dims, int32_t n, const int32_t* ks_host,
                                     const int32_t* accepted_dev,
                                     const uint64_t* wy_tables_dev, void* conv_pool,
                                     int32_t n_slots, const int32_t* slots_dev,
                                     const void* conv_inter, int32_t dtype, int32_t h_dtype,
                                     int32_t* status_dev, gdn_stream_t stream);

/* Write-on-accept verify and its deferred fold (trait_layer.rs, LayerWriteOnAccept:
 * gdn_woa_stash_seq_floats and gdn_woa_bind; layer_struct.rs, the gdn_wy4_woa_k,
 * gdn_wy4_fold_k and gdn_wy4_clear_k handles and the woa_flag / woa_stash bindings).
 * gdn_verify_woa computes the same outputs as gdn_verify_multi but writes no state: the
 * state (table 0 entry i) and the conv state stay as they were, and sequence i's stash
 * receives k_i and, for each draft token t, the factors of its state update
 * (S_t = alpha_t S_{t-1} + delta_t k_hat_t^T, with delta_t = beta_t (v_t - alpha_t S_{t-1}
 * k_hat_t)) and its raw qkv row; then the engaged word is set to 1.  Once the caller knows
 * how many drafts m_i it accepts, gdn_woa_fold replays tokens 0 .. m_i - 1 on the state in
 * one pass and moves the conv state to the last d_conv raw inputs up to token m_i - 1, and
 * gdn_woa_clear zeroes the engaged word (a fold while it is 0 changes nothing).  The
 * verify writes k_i x (a few KiB) per sequence instead of k_i - 1 intermediate states of
 * H_v d_k d_v floats each; the fold reads and writes each state once.  f32 state pools only.
 *   gdn_woa_stash_seq_floats: 4-byte words of stash per sequence (room for
 *     GDN_VERIFY_K_MAX tokens) for these dims and activation dtype; 0 on invalid input.
 *   stash      : device, [stash_seqs][gdn_woa_stash_seq_floats] 4-byte words, 16-B aligned,
 *                caller-owned; sequence i (the verify's i) uses row i; stash_seqs >= n.
 *   flag_dev   : device uint32, the engaged word (4-B aligned).
 * gdn_verify_woa: the arguments and errors of gdn_verify_multi without conv_inter; only
 *   table 0 is read (the intermediate tables may be zero).
 * gdn_woa_fold: n, accepted_dev, wy_tables_dev, conv_pool, n_slots, slots_dev as for
 *   gdn_fold_accepted (1 <= accepted_dev[i] <= k_i, else GDN_ERR_BAD_ACCEPTED and that
 *   sequence is left as it is); stash and flag_dev as passed to gdn_verify_woa; dtype is
 *   the verify's activation dtype. */
GDN_API size_t gdn_woa_stash_seq_floats(const gdn_dims* dims, int32_t dtype);
GDN_API gdn_status gdn_verify_woa(const gdn_dims* dims, const gdn_weights* weights,
                                  const gdn_inputs* inputs, int32_t n, const int32_t* ks_host,
                                  const uint64_t* wy_tables_dev, void* conv_pool,
                                  int32_t n_slots, const int32_t* slots_dev, void* stash,
                                  int32_t stash_seqs, uint32_t* flag_dev, void* y,
                                  float* core_out, int32_t* status_dev, gdn_stream_t stream);
GDN_API gdn_status gdn_woa_fold(const gdn_dims* dims, int32_t n, const int32_t* accepted_dev,
                                const uint64_t* wy_tables_dev, void* conv_pool,
                                int32_t n_slots, const int32_t* slots_dev, const void* stash,
                                const uint32_t* flag_dev, int32_t dtype, int32_t* status_dev,
                                gdn_stream_t stream);
GDN_API gdn_status gdn_woa_clear(uint32_t* flag_dev, gdn_stream_t stream);

/* Half-width h-state pools (layer_struct.rs: the FP16 h-state variants gdn_f16_norm_k,
 * gdn_f16_strided_norm_half_k and gdn_wyn_f16_table_k, and the width converters
 * ssm_h_f16_to_f32_k / ssm_h_f32_to_f16_k).  The same mixer on states stored as fp16
 * [n_v_heads][d_k][d_v] (element (i, j) = S[j][i]), which halves the state traffic that
 * dominates decode and verify.  The arithmetic stays f32: each head's state is widened when
 * it is read and rounded to the nearest fp16 (ties to even) when it is written, once per
 * token kept, so every stored state is the f32 update of the previous stored state,
 * rounded.  Arguments and errors are those of gdn_decode_batched / gdn_verify_multi, with
 * h_pool an fp16 pool and every table entry pointing to an fp16 state (16-B aligned).
 * Prefill stays f32: widen a sequence's state with gdn_state_convert before
 * gdn_prefill_chunked and narrow it after. */
GDN_API gdn_status gdn_decode_batched_h16(const gdn_dims* dims, const gdn_weights* weights,
                                          const gdn_inputs* inputs, int32_t n, void* h_pool,
                                          void* conv_pool, int32_t n_slots,
                                          const int32_t* slots_dev, void* y, float* core_out,
                                          int32_t* status_dev, gdn_stream_t stream);
GDN_API gdn_status gdn_verify_multi_h16(const gdn_dims* dims, const gdn_weights* weights,
                                        const gdn_inputs* inputs, int32_t n,
                                        const int32_t* ks_host, const uint64_t* wy_tables_dev,
                                        void* conv_pool, int32_t n_slots,
                                        const int32_t* slots_dev, void* conv_inter, void* y,
                                        float* core_out, int32_t* status_dev,
                                        gdn_stream_t stream);

/* Converts `count` state elements between an f32 and an fp16 pool (src_dtype / dst_dtype =
 * GDN_DTYPE_F32 and GDN_DTYPE_F16 in either order; round to nearest even when narrowing).
 * src and dst are device memory, 16-B aligned, and must not overlap. */
GDN_API gdn_status gdn_state_convert(const void* src, int32_t src_dtype, void* dst,
                                     int32_t dst_dtype, int64_t count, gdn_stream_t stream);

/* Conv + SiLU + L2 norm of q and k (q also scaled) for T tokens of n sequences in one
 * launch, updating each sequence's conv state to its last d_conv raw inputs
 * (layer_struct.rs, conv1d_l2norm_f32_strided_k; trait_layer.rs,
 * LayerSplitPrefill::prefill_phase1_conv1d_one / prefill_phase1_l2_batched).
 *   cu_seqlens_dev: device int32 [n+1], cu[0] = 0, non-decreasing, cu[n] = total_tokens.
 *   qkv_out    : device f32 [total_tokens][conv_dim]: normalised q, normalised k, raw
 *                conv+SiLU v, in the [Q|K|V] channel order. */
GDN_API gdn_status gdn_conv_step(const gdn_dims* dims, const gdn_weights* weights,
                         const gdn_inputs* inputs, int32_t n, const int32_t* cu_seqlens_dev,
                         int32_t total_tokens, void* conv_pool, int32_t n_slots,
                         const int32_t* slots_dev, float* qkv_out, int32_t* status_dev,
                         gdn_stream_t stream);

/* Chunked (WY-form) prefill of n variable-length sequences (trait_layer.rs,
 * LayerSplitPrefill::prefill_gdn_full_batched_fla_varlen; layer_struct.rs, the FLA
 * chunked prefill gdn_prefill_fla_recompute_wu_k -> state spine chunk_delta_h ->
 * chunk_fwd_o, and gated_rms_norm_prefill_k).  Chunk length 64.
 *   cu_seqlens_dev : device int32 [n+1] (as in gdn_conv_step); total_tokens = cu[n],
 *                    max_seqlen >= every length.
 *   h_state_ptrs_dev: device u64 [n], each a 16-B aligned [n_v_heads][d_k][d_v] f32
 *                    state, read as the initial state and overwritten with the final.
 *   conv_pool, n_slots, slots_dev: as in decode.
 *   y, core_out    : [total_tokens] rows, as in decode.
 *   workspace      : device scratch of at least gdn_prefill_workspace_bytes(...) bytes,
 *                    256-B aligned; its contents on entry do not matter. */
GDN_API gdn_status gdn_prefill_chunked(const gdn_dims* dims, const gdn_weights* weights,
                               const gdn_inputs* inputs, int32_t n,
                               const int32_t* cu_seqlens_dev, int32_t total_tokens,
                               int32_t max_seqlen, int32_t chunk,
                               const uint64_t* h_state_ptrs_dev, void* conv_pool,
                               int32_t n_slots, const int32_t* slots_dev, void* y,
                               float* core_out, void* workspace, size_t workspace_bytes,
                               int32_t* status_dev, gdn_stream_t stream);

/* Bytes of workspace gdn_prefill_chunked needs for these sizes (0 on invalid input). */
GDN_API size_t gdn_prefill_workspace_bytes(const gdn_dims* dims, int32_t n, int32_t total_tokens,
                                   int32_t max_seqlen, int32_t chunk);

/* Allocation-free variant of gdn_prefill_chunked (the reference pages have no counterpart).
 * Some callers cannot allocate device memory at the time they prefill: a serving engine that
 * reserved nearly all of HBM at start-up for its own state and KV pools (a cudaMalloc would
 * fail, or fragment memory the engine manages), or a plug-in running under a host runtime
 * that owns every allocation and hands out no scratch.  This entry point takes the same
 * arguments as gdn_prefill_chunked minus the workspace and uses instead a scratch array the
 * library keeps in device memory: GDN_NOALLOC_SCRATCH_BYTES (64 MiB) per GPU, held by every
 * GPU that loads the library until the process exits.  It calls no allocator.
 *   - Sizes: a call whose gdn_prefill_workspace_bytes(...) exceeds the scratch returns
 *     GDN_ERR_SCRATCH_TOO_SMALL and launches nothing.  At H_k = 16, H_v = 32, d = 128 each
 *     64-token chunk slot takes 2.8 MiB (tiles, W, K~, P, U) and each token 16 KiB of
 *     core output, so the scratch holds one sequence of up to 1,023 tokens, or several
 *     shorter ones.
 *   - Set-up: the first call on a device, with that device current, looks up the scratch's
 *     device address (cudaGetSymbolAddress); make that first call before any stream capture.
 *     Its failure returns GDN_ERR_CUDA.  Under CUDA's lazy module loading (the default since
 *     CUDA 12.2; CUDA_MODULE_LOADING=EAGER changes it) the array is reserved by that first
 *     call, not when the library loads, so make it before reserving the rest of the device's
 *     memory: a call with n = 0 and total_tokens = 0 (valid dims and weights, every other
 *     pointer may be NULL) does only this set-up.  The cached address does not survive a
 *     cudaDeviceReset of that device; do not use this entry point after one.
 *   - Sharing: every call on a device uses the same array and leaves its contents behind;
 *     nothing in it needs to start at zero.  Calls that overlap on the GPU (other streams,
 *     other host threads) race on it: serialise them.
 *   - Results are the same as gdn_prefill_chunked's for the same arguments. */
GDN_API gdn_status gdn_prefill_chunked_noalloc(const gdn_dims* dims, const gdn_weights* weights,
                                               const gdn_inputs* inputs, int32_t n,
                                               const int32_t* cu_seqlens_dev,
                                               int32_t total_tokens, int32_t max_seqlen,
                                               int32_t chunk, const uint64_t* h_state_ptrs_dev,
                                               void* conv_pool, int32_t n_slots,
                                               const int32_t* slots_dev, void* y,
                                               float* core_out, int32_t* status_dev,
                                               gdn_stream_t stream);
#define GDN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* Z-gated RMSNorm of T rows (layer_struct.rs, gated_rms_norm_f32_k: f32 input):
 *   y[t][h*d_v + j] = o[t][h][j] / sqrt(mean_j o[t][h][:]^2 + eps) * w[j] * SiLU(z[t][h*d_v + j])
 *   o : device f32 [T][n_v_heads][d_v];  z : device [T][z_stride] in `dtype`;
 *   w : device f32 [d_v];  y : device [T][n_v_heads*d_v] in `dtype`.  d_v in {16, 128}. */
GDN_API gdn_status gdn_gated_rmsnorm(const float* o, const void* z, int64_t z_stride, const float* w,
                             float eps, int32_t T, int32_t n_v_heads, int32_t d_v,
                             int32_t dtype, void* y, gdn_stream_t stream);

/* The same with the sigmoid gate: y = o / sqrt(mean o^2 + eps) * w * sigmoid(z) (the
 * gdn_norm_sigmoid models of layer_struct.rs; gdn_dims.norm_gate selects it in the fused
 * entry points). */
GDN_API gdn_status gdn_gated_rmsnorm_sigmoid(const float* o, const void* z, int64_t z_stride,
                                             const float* w, float eps, int32_t T,
                                             int32_t n_v_heads, int32_t d_v, int32_t dtype,
                                             void* y, gdn_stream_t stream);

/* The bf16 projections on either side of the mixer (layer_struct.rs, Qwen3SsmLayer: the
 * sequential [Q | K | V | Z] QKVZ projection, the b / a inputs that ba_gates_k reads, and
 * out_proj; the dense_gemm fields are the layer's bf16 GEMMs).  One GEMM on the tcgen05
 * tensor cores: C[M][N] = A[M][K] * B[N][K]^T, bf16 operands, f32 accumulation, the result
 * rounded to the nearest bf16 (ties to even).
 *   A          : device bf16 [M][lda], lda >= K.
 *   B          : device bf16 [N][ldb], ldb >= K; row n holds output feature n (the layout
 *                of a linear layer's weight).
 *   C          : device bf16 [M][ldc], ldc >= N; must not overlap A or B.
 *   M >= 0 (0 does nothing, and no pointer is read); N >= 8 and K >= 8, both multiples
 *   of 8; lda, ldb, ldc multiples of 8 and A, B, C 16-byte aligned (else
 *   GDN_ERR_MISALIGNED).
 *   status_dev : device int32; a device-side wait that runs out sets GDN_ERR_TIMEOUT.
 * Nothing is allocated; the call is asynchronous on `stream`. */
GDN_API gdn_status gdn_proj_gemm(const void* A, int64_t lda, const void* B, int64_t ldb,
                                 void* C, int64_t ldc, int32_t M, int32_t N, int32_t K,
                                 int32_t* status_dev, gdn_stream_t stream);

/* Width of one in_proj output row: conv_dim + H_v d_v + 2 H_v rounded up to a multiple of
 * 8, so that rows start on 16-byte boundaries as the mixer's entry points require (0 for
 * invalid dims).  Columns past the b / a inputs are padding: their weight rows are the
 * caller's and nothing reads their outputs.  12352 for H_k = 16, H_v = 32, d = 128. */
GDN_API int32_t gdn_in_proj_width(const gdn_dims* dims);

/* in_proj: hidden [T][hidden_size] bf16 (row stride hidden_stride) times
 * w_in [gdn_in_proj_width(dims)][hidden_size] bf16 -> out [T][width] bf16 with the row
 * [Q | K | V | Z | b | a] per token.  The mixer's entry points read it directly as
 * qkv = out, z = out + conv_dim, b = out + conv_dim + H_v d_v, a = b + H_v, every row
 * stride = width, dtype GDN_DTYPE_BF16.  Same rules as gdn_proj_gemm. */
GDN_API gdn_status gdn_in_proj(const gdn_dims* dims, int32_t hidden_size, const void* hidden,
                               int64_t hidden_stride, int32_t T, const void* w_in, void* out,
                               int32_t* status_dev, gdn_stream_t stream);

/* out_proj: y [T][H_v d_v] bf16 (the mixer's output rows) times
 * w_out [hidden_size][H_v d_v] bf16 -> out [T][hidden_size] bf16 (row stride out_stride).
 * Same rules as gdn_proj_gemm. */
GDN_API gdn_status gdn_out_proj(const gdn_dims* dims, int32_t hidden_size, const void* y,
                                int32_t T, const void* w_out, void* out, int64_t out_stride,
                                int32_t* status_dev, gdn_stream_t stream);

/* Host helper: fills one layer's WY pointer tables in HOST memory
 * (transformer_layer.rs, the VERIFY_WY_* layout; the engine's upload_verify_wy_tables
 * stages them only for k in 2..16).  Zero-fills all 16 x 128 entries, then sets
 * table 0 entry i = h_ptrs[i] and table t+1 entry i = inter_ptrs[i*15 + t] for
 * t < ks[i] - 1.  Returns GDN_ERR_BAD_K for a k outside 2..16 (tables left zero). */
GDN_API gdn_status gdn_wy_tables_fill(uint64_t* host_tables, int32_t n, const int32_t* ks,
                              const uint64_t* h_ptrs, const uint64_t* inter_ptrs);

/* Self-test of the bounded device-side wait every kernel uses: one thread waits, for at
 * most budget_ns (1 .. 1e9 ns), on an mbarrier that nothing arrives on, then writes
 * GDN_ERR_TIMEOUT to *status_dev (first error wins) and returns.  The context stays usable;
 * nothing faults or traps.  Used by the tests to show that a wait which never completes
 * ends with a status the host can read. */
GDN_API gdn_status gdn_selftest_wait(int64_t budget_ns, int32_t* status_dev, gdn_stream_t stream);

/* A static, human-readable name of a status code. */
GDN_API const char* gdn_status_string(gdn_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
GDN_API int32_t gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
