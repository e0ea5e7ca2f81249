// Rotary re-alignment of cached keys (RedKnot summary page, section "Elastic
// Sparsity（弹性稀疏恢复）": reusing a cached segment at another position starts
// by aligning its RoPE positions). Each kept key of the selected heads turns
// every dimension pair i by delta * theta_i in place; V is untouched.
//
// HBM bound: every rotated bf16 pair is read once and written once. One CTA
// per run of consecutive rows of one page; the cos/sin of delta * theta_i
// come with the plan, formed in fp64 on the host and rounded once to fp32.
#include <cuda_bf16.h>

#include "segkv_internal.h"

namespace skv {

template <class T>
__device__ __forceinline__ const T* rope_plan_ptr(const T* p, const AppendBlob& blob, int inl) {
  return inl ? reinterpret_cast<const T*>(blob.data + reinterpret_cast<uintptr_t>(p)) : p;
}

__device__ __forceinline__ void rot8(uint4& a, uint4& b, const float2* cs, bool interleaved) {
  // eight pairs: interleaved -> (a.x lo, a.x hi), ... spread over a then b;
  // split-half -> element e of a pairs with element e of b
  __nv_bfloat16* pa = reinterpret_cast<__nv_bfloat16*>(&a);
  __nv_bfloat16* pb = reinterpret_cast<__nv_bfloat16*>(&b);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    __nv_bfloat16* x = interleaved ? (e < 4 ? pa + 2 * e : pb + 2 * (e - 4)) : pa + e;
    __nv_bfloat16* y = interleaved ? x + 1 : pb + e;
    const float xa = __bfloat162float(*x), xb = __bfloat162float(*y);
    const float2 c = cs[e];
    *x = __float2bfloat16_rn(fmaf(xa, c.x, -xb * c.y));
    *y = __float2bfloat16_rn(fmaf(xa, c.y, xb * c.x));
  }
}

__global__ void __launch_bounds__(256)
    rope_kernel(RopeParams p, const __grid_constant__ AppendBlob blob) {
  const RopeRun* runs = rope_plan_ptr(p.runs, blob, p.plan_inline);
  const float2* cs_g = rope_plan_ptr(p.cos_sin, blob, p.plan_inline);
  __shared__ float2 cs[128];
  const int half = p.rotary_dim / 2;
  for (int i = threadIdx.x; i < half; i += blockDim.x) cs[i] = cs_g[i];
  __syncthreads();
  const bool vec = (half % 8) == 0;  // whole 16-byte chunks of eight pairs
  const int per_row = vec ? half / 8 : half;
  for (int r = blockIdx.x; r < p.n_runs; r += gridDim.x) {
    const RopeRun run = runs[r];
    __nv_bfloat16* base =
        static_cast<__nv_bfloat16*>(p.kpool) +
        (static_cast<int64_t>(run.page) * p.page_size + run.slot0) * p.head_dim;
    const int items = run.nrows * per_row;
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
      const int row = it / per_row, j = it - row * per_row;
      __nv_bfloat16* v = base + static_cast<int64_t>(row) * p.head_dim;
      if (vec) {
        uint4* pa = reinterpret_cast<uint4*>(v + (p.style == 0 ? 16 * j : 8 * j));
        uint4* pb = reinterpret_cast<uint4*>(v + (p.style == 0 ? 16 * j + 8 : half + 8 * j));
        uint4 a = *pa, b = *pb;
        rot8(a, b, cs + 8 * j, p.style == 0);
        *pa = a;
        *pb = b;
      } else {
        const int i = j;
        const int ia = p.style == 0 ? 2 * i : i;
        const int ib = p.style == 0 ? 2 * i + 1 : i + half;
        const float xa = __bfloat162float(v[ia]), xb = __bfloat162float(v[ib]);
        const float2 c = cs[i];
        v[ia] = __float2bfloat16_rn(fmaf(xa, c.x, -xb * c.y));
        v[ib] = __float2bfloat16_rn(fmaf(xa, c.y, xb * c.x));
      }
    }
  }
}

cudaError_t launch_rope(const RopeParams& p, const AppendBlob* blob, int grid, cudaStream_t s) {
  static const AppendBlob empty_blob{};
  rope_kernel<<<grid, 256, 0, s>>>(p, blob ? *blob : empty_blob);
  return cudaGetLastError();
}

}  // namespace skv
