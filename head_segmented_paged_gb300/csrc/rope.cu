// Rotary re-alignment of cached keys (RedKnot summary page, section "Elastic
// Sparsity（弹性稀疏恢复）": reusing a cached segment at another position starts
// by aligning its RoPE positions). Each kept key of the selected heads turns
// every dimension pair i by delta * theta_i in place; V is untouched.
//
// HBM bound: every rotated bf16 pair is read once and written once. The CTAs
// stride over (head, page) chunks, finding each page through the block
// table one chunk ahead; the plan (one entry per head) and the cos/sin of
// delta * theta_i, formed in fp64 on the host and rounded once to fp32,
// travel in the kernel's parameters, so a call uploads nothing.
#include <cuda_bf16.h>

#include "segkv_internal.h"

namespace skv {

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

__global__ void __launch_bounds__(256) rope_kernel(const __grid_constant__ RopeParams p, int chunks_per_head) {
  const int half = p.rotary_dim / 2;
  // cos/sin to shared memory: the lanes of a warp read eight different pairs
  // at a time, which the parameter (constant) cache would serve one by one
  __shared__ float2 cs[128];
  for (int i = threadIdx.x; i < half; i += blockDim.x) cs[i] = p.cos_sin[i];
  __syncthreads();
  // launched as a programmatic dependent of the previous kernel: the block
  // table and the keys are read only after it has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __nv_bfloat16* kp = static_cast<__nv_bfloat16*>(p.kpool);
  const int n_chunks = chunks_per_head * p.n_heads;
  // chunk c: head c / chunks_per_head, rows [P * (c % chunks_per_head), + P) of
  // its kept range counted from the first kept page's start; the next
  // chunk's page id is fetched while this one streams
  auto page_of = [&](int c, int* pos0, int* nrows) -> int32_t {
    const RopeHead H = p.heads[c / chunks_per_head];
    const int k = H.s0 / p.page_size + c % chunks_per_head;
    const int lo = max(H.s0, k * p.page_size), hi = min(H.n, (k + 1) * p.page_size);
    *pos0 = lo;
    *nrows = hi - lo;
    return hi > lo ? p.table[static_cast<int64_t>(H.table_row) * p.R + k] : 0;
  };
  int c = blockIdx.x, pos0 = 0, nrows = 0;
  int32_t page = c < n_chunks ? page_of(c, &pos0, &nrows) : 0;
  for (; c < n_chunks; c += gridDim.x) {
    int npos0 = 0, nnrows = 0;
    const int32_t npage = c + gridDim.x < n_chunks ? page_of(c + gridDim.x, &npos0, &nnrows) : 0;
    __nv_bfloat16* base =
        kp + (static_cast<int64_t>(page) * p.page_size + (pos0 - (pos0 / p.page_size) * p.page_size)) * p.head_dim;
    if (half % 8 == 0) {
      const int per_row = half / 8;
      const int items = nrows * per_row;
      for (int it = threadIdx.x; it < items; it += 2 * blockDim.x) {
        const int it2 = it + blockDim.x;
        const bool two = it2 < items;
        const int row = it / per_row, j = it - row * per_row;
        const int row2 = two ? it2 / per_row : row, j2 = two ? it2 - row2 * per_row : j;
        __nv_bfloat16* v = base + static_cast<int64_t>(row) * p.head_dim;
        __nv_bfloat16* v2 = base + static_cast<int64_t>(row2) * p.head_dim;
        uint4* pa = reinterpret_cast<uint4*>(v + (p.style == 0 ? 16 * j : 8 * j));
        uint4* pb = reinterpret_cast<uint4*>(v + (p.style == 0 ? 16 * j + 8 : half + 8 * j));
        uint4* pa2 = reinterpret_cast<uint4*>(v2 + (p.style == 0 ? 16 * j2 : 8 * j2));
        uint4* pb2 = reinterpret_cast<uint4*>(v2 + (p.style == 0 ? 16 * j2 + 8 : half + 8 * j2));
        uint4 a = *pa, b = *pb, a2 = make_uint4(0, 0, 0, 0), b2 = a2;
        if (two) {
          a2 = *pa2;
          b2 = *pb2;
        }
        rot8(a, b, cs + 8 * j, p.style == 0);
        *pa = a;
        *pb = b;
        if (two) {
          rot8(a2, b2, cs + 8 * j2, p.style == 0);
          *pa2 = a2;
          *pb2 = b2;
        }
      }
    } else {
      for (int it = threadIdx.x; it < nrows * half; it += blockDim.x) {
        const int row = it / half, i = it - row * half;
        __nv_bfloat16* v = base + static_cast<int64_t>(row) * p.head_dim;
        const int ia = p.style == 0 ? 2 * i : i;
        const int ib = p.style == 0 ? 2 * i + 1 : i + half;
        const float xa = __bfloat162float(v[ia]), xb = __bfloat162float(v[ib]);
        const float2 cc = cs[i];
        v[ia] = __float2bfloat16_rn(fmaf(xa, cc.x, -xb * cc.y));
        v[ib] = __float2bfloat16_rn(fmaf(xa, cc.y, xb * cc.x));
      }
    }
    page = npage;
    pos0 = npos0;
    nrows = nnrows;
  }
}

cudaError_t launch_rope(const RopeParams& p, int chunks_per_head, int grid, cudaStream_t s) {
  return launch_pdl(rope_kernel, dim3(grid), dim3(256), 0, s, p, chunks_per_head);
}

}  // namespace skv
