// AdamW for the parameters Muon does not take (one-dimensional and scalar
// tensors: norm gains, biases; HyperParallel-FSDP section 6.3 delegates them
// to AdamW through a chained optimizer, DMuon-2 section 2.1 names the
// embeddings, the output head and the normalization gains and biases).
//
// One launch updates every tensor of the call: the tensors are cut into
// units of 8 elements, numbered across tensors, and a grid-stride loop over
// the units does, per element, in fp32,
//     m = b1 m + (1 - b1) g,   v = b2 v + (1 - b2) g^2,
//     p = p (1 - lr wd) - (lr / (1 - b1^t)) m / (sqrt(v) / sqrt(1 - b2^t) + eps),
// which is AdamW with bias correction and decoupled decay.  HBM-bound:
// 16-byte loads and stores where the tensor is 16-byte aligned, element-wise
// at the tails.
#include <algorithm>

#include "muon_internal.h"

namespace muon {

namespace {

__device__ __forceinline__ void ld8(const void* base, int dtype, int64_t e, bool vec, int n,
                                    float* d) {
  if (dtype == 0) {
    const float* p = static_cast<const float*>(base) + e;
    if (vec) {
      const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
      const float4 b = __ldcs(reinterpret_cast<const float4*>(p + 4));
      d[0] = a.x; d[1] = a.y; d[2] = a.z; d[3] = a.w;
      d[4] = b.x; d[5] = b.y; d[6] = b.z; d[7] = b.w;
    } else {
      for (int j = 0; j < 8; ++j) d[j] = j < n ? p[j] : 0.f;
    }
  } else {
    const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(base) + e;
    if (vec) {
      const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(h[j]);
        d[2 * j] = f.x;
        d[2 * j + 1] = f.y;
      }
    } else {
      for (int j = 0; j < 8; ++j) d[j] = j < n ? __bfloat162float(p[j]) : 0.f;
    }
  }
}

__device__ __forceinline__ void st8(void* base, int dtype, int64_t e, bool vec, int n,
                                    const float* d) {
  if (dtype == 0) {
    float* p = static_cast<float*>(base) + e;
    if (vec) {
      __stcs(reinterpret_cast<float4*>(p), make_float4(d[0], d[1], d[2], d[3]));
      __stcs(reinterpret_cast<float4*>(p + 4), make_float4(d[4], d[5], d[6], d[7]));
    } else {
      for (int j = 0; j < n; ++j) p[j] = d[j];
    }
  } else {
    __nv_bfloat16* p = static_cast<__nv_bfloat16*>(base) + e;
    if (vec) {
      uint4 u;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(d[2 * j], d[2 * j + 1]);
      __stcs(reinterpret_cast<uint4*>(p), u);
    } else {
      for (int j = 0; j < n; ++j) p[j] = __float2bfloat16_rn(d[j]);
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(256) adamw_kernel(const __grid_constant__ AdamwParams p) {
  const float b1 = p.beta1, b2 = p.beta2;
  const float decay = 1.f - p.lr * p.wd;
  for (int64_t u = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; u < p.total_units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int si = 0;
    while (si + 1 < p.n_slices && u >= p.s[si + 1].unit_base) ++si;
    const AdamwSlice& s = p.s[si];
    const int64_t e = (u - s.unit_base) * 8;
    const int n = static_cast<int>(min(static_cast<int64_t>(8), s.numel - e));
    const bool vec = s.vec && n == 8;
    float pv[8], gv[8], mv[8], vv[8];
    ld8(s.p, s.p_dtype, e, vec, n, pv);
    ld8(s.g, s.g_dtype, e, vec, n, gv);
    ld8(s.m, 0, e, vec, n, mv);
    ld8(s.v, 0, e, vec, n, vv);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float g = gv[j];
      mv[j] = fmaf(b1, mv[j], (1.f - b1) * g);
      vv[j] = fmaf(b2, vv[j], (1.f - b2) * g * g);
      const float denom = fmaf(__fsqrt_rn(vv[j]), p.inv_sqrt_bc2, p.eps);
      pv[j] = fmaf(decay, pv[j], -p.step_size * __fdiv_rn(mv[j], denom));
    }
    st8(s.p, s.p_dtype, e, vec, n, pv);
    st8(s.m, 0, e, vec, n, mv);
    st8(s.v, 0, e, vec, n, vv);
  }
}

cudaError_t launch_adamw(const AdamwParams& p, int sms, cudaStream_t s) {
  if (p.total_units <= 0) return cudaSuccess;
  const int64_t want = (p.total_units + 255) / 256;
  const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sms) * 8));
  adamw_kernel<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace muon
