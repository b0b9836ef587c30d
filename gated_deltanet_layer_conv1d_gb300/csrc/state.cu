// state.cu -- conversion between f32 and fp16 state pools (sm_103a).
//
// layer_struct.rs, ssm_h_f16_to_f32_k / ssm_h_f32_to_f16_k: under a half-width h-state
// pool the prefill widens a sequence's state to f32 before it runs and narrows it after.
// Plain element-wise copy with 16-byte loads where the pointers allow, round to nearest
// even when narrowing.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

__global__ void gdn_h_widen_kernel(const __half* __restrict__ src, float* __restrict__ dst,
                                   size_t count) {
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i * 8 < count; i += stride) {
    if (i * 8 + 8 <= count) {
      const uint4 u = reinterpret_cast<const uint4*>(src)[i];
      const __half2* h = reinterpret_cast<const __half2*>(&u);
      float2 f[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) f[e] = __half22float2(h[e]);
      reinterpret_cast<float4*>(dst)[2 * i] = make_float4(f[0].x, f[0].y, f[1].x, f[1].y);
      reinterpret_cast<float4*>(dst)[2 * i + 1] = make_float4(f[2].x, f[2].y, f[3].x, f[3].y);
    } else {
      for (size_t j = i * 8; j < count; ++j) dst[j] = __half2float(src[j]);
    }
  }
}

__global__ void gdn_h_narrow_kernel(const float* __restrict__ src, __half* __restrict__ dst,
                                    size_t count) {
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i * 8 < count; i += stride) {
    if (i * 8 + 8 <= count) {
      const float4 a = reinterpret_cast<const float4*>(src)[2 * i];
      const float4 b = reinterpret_cast<const float4*>(src)[2 * i + 1];
      const __half2 h[4] = {__floats2half2_rn(a.x, a.y), __floats2half2_rn(a.z, a.w),
                            __floats2half2_rn(b.x, b.y), __floats2half2_rn(b.z, b.w)};
      reinterpret_cast<uint4*>(dst)[i] = *reinterpret_cast<const uint4*>(h);
    } else {
      for (size_t j = i * 8; j < count; ++j) dst[j] = __float2half_rn(src[j]);
    }
  }
}

}  // namespace

cudaError_t launch_state_convert(const void* src, int src_dtype, void* dst, int dst_dtype,
                                 size_t count, cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  const size_t vec = (count + 7) / 8;
  size_t blocks = (vec + 255) / 256;
  const size_t cap = size_t(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (src_dtype == GDN_DTYPE_F16 && dst_dtype == GDN_DTYPE_F32)
    gdn_h_widen_kernel<<<unsigned(blocks), 256, 0, stream>>>(
        static_cast<const __half*>(src), static_cast<float*>(dst), count);
  else
    gdn_h_narrow_kernel<<<unsigned(blocks), 256, 0, stream>>>(
        static_cast<const float*>(src), static_cast<__half*>(dst), count);
  return cudaGetLastError();
}

}  // namespace gdn
