// prefill.cu -- dispatch of the GDN prefill (sm_103a).
//
// d_k = d_v = 128 with bf16 activations: the tensor-core chunked path -- a pre-pass
// (conv, SiLU, L2 norms, gates of every token into the workspace tiles), the chunk kernel
// (every chunk's W, U, P and K~ at once), the state spine (chunk after chunk per sequence
// and value head, writing the core output O) and the gated RMSNorm of O.  Every other
// shape or dtype, and any call whose dims ask for GDN_PREFILL_F32: the token-sequential
// kernel, f32 throughout.  The conv-state update runs after either (see abi.cu).
#include "common.cuh"
#include "kernels.h"
#include "prefill_layout.cuh"

namespace gdn {

cudaError_t launch_prefill_sequential(const PrefillParams& p, int dtype, cudaStream_t stream);
cudaError_t launch_prefill_tc(const PrefillParams& p, float* o_work, cudaStream_t stream);

size_t prefill_workspace_bytes(int Hk, int Hv, int D, int n, int total_tokens, int max_seqlen) {
  (void)max_seqlen;
  if (D != 128) return 0;
  const PrefillLayout lay{Hk, Hv};
  return lay.total_bytes(n, total_tokens);
}

cudaError_t launch_prefill(const PrefillParams& p, int dtype, cudaStream_t stream) {
  if (p.D == 128 && dtype == GDN_DTYPE_BF16 && !p.f32_path) {
    ConvParams c{};
    c.Hk = p.Hk;
    c.Hv = p.Hv;
    c.D = p.D;
    c.conv_dim = p.conv_dim;
    c.n = p.n;
    c.n_slots = p.n_slots;
    c.total_tokens = p.total_tokens;
    c.q_scale = p.q_scale;
    c.l2_eps = p.l2_eps;
    c.conv_w = p.conv_w;
    c.qkv = p.qkv;
    c.qkv_stride = p.qkv_stride;
    c.cu_seqlens = p.cu_seqlens;
    c.conv_pool = p.conv_pool;
    c.slots = p.slots;
    c.status = p.status;
    c.A_log = p.A_log;
    c.dt_bias = p.dt_bias;
    c.a = p.a;
    c.b = p.b;
    c.ab_stride = p.ab_stride;
    c.workspace = p.workspace;
    cudaError_t e = launch_prefill_prep(c, stream);
    if (e != cudaSuccess) return e;
    const PrefillLayout lay{p.Hk, p.Hv};
    unsigned char* ws = static_cast<unsigned char*>(p.workspace);
    PrefillParams q = p;
    q.counts = reinterpret_cast<int32_t*>(ws + lay.count_offset(p.n, p.total_tokens));
    return launch_prefill_tc(q, reinterpret_cast<float*>(ws + lay.o_offset(p.n, p.total_tokens)),
                             stream);
  }
  return launch_prefill_sequential(p, dtype, stream);
}

}  // namespace gdn
