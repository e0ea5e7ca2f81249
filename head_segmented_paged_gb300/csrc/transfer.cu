// Segment transfer: gather a sequence's kept K/V rows out of its pages into
// one contiguous buffer, or scatter such a buffer into freshly taken pages
// (RedKnot summary page, section "系统收益": with prefill and decode on
// different GPUs only each head's kept tokens need to cross the link).
// HBM bound: every kept row is read once and written once.
#include "segkv_internal.h"

namespace skv {

template <class T>
__device__ __forceinline__ const T* xfer_plan_ptr(const T* p, const AppendBlob& blob, int inl) {
  return inl ? reinterpret_cast<const T*>(blob.data + reinterpret_cast<uintptr_t>(p)) : p;
}

constexpr int kXferUnroll = 4;  // 16-byte chunks of K and of V in flight per thread

// Grid-stride over the 16-byte chunks of all kept rows; each chunk moves its
// K and its V. The heads' descriptors sit in shared memory.
__global__ void __launch_bounds__(256)
    transfer_kernel(TransferParams p, const __grid_constant__ AppendBlob blob) {
  extern __shared__ XferHead hs[];  // [n_heads]
  // launched as a programmatic dependent of the previous kernel: the plan (it
  // may come from the upload kernel), the tables and the pools are read only
  // after it has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const XferHead* heads = xfer_plan_ptr(p.heads, blob, p.plan_inline);
  const int32_t* page_list = xfer_plan_ptr(p.page_list, blob, p.plan_inline);
  for (int i = threadIdx.x; i < p.n_heads; i += blockDim.x) hs[i] = heads[i];
  __syncthreads();
  if (p.to_pool) {  // an import's block-table entries: head h, logical page first_k + i
    int h = 0;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < p.n_pages; e += gridDim.x * blockDim.x) {
      while (h + 1 < p.n_heads && e >= hs[h + 1].page_off) ++h;
      p.table[static_cast<int64_t>(hs[h].table_row) * p.R + hs[h].first_k + (e - hs[h].page_off)] =
          page_list[e];
    }
  }
  const int vec = p.vec_per_row;
  const int64_t items = p.total_rows * vec;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < items;
       base += stride * kXferUnroll) {
    int64_t src_k[kXferUnroll], dst_k[kXferUnroll], src_v[kXferUnroll], dst_v[kXferUnroll];
    uint4 kx[kXferUnroll], vx[kXferUnroll];
#pragma unroll
    for (int u = 0; u < kXferUnroll; ++u) {
      const int64_t it = base + u * stride;
      src_k[u] = -1;
      if (it >= items) continue;
      const int64_t rg = it / vec;
      const int c = static_cast<int>(it - rg * vec);
      int h = 0;
      while (h + 1 < p.n_heads && rg >= hs[h + 1].row_begin) ++h;
      const XferHead& H = hs[h];
      const int32_t i = static_cast<int32_t>(rg - H.row_begin), pos = H.s0 + i;
      const int32_t k = pos / p.page_size;
      const int64_t pool = (static_cast<int64_t>(page_list[H.page_off + k - H.first_k]) * p.page_size +
                            (pos - k * p.page_size)) * vec + c;
      const int64_t bk = (static_cast<int64_t>(H.out_row) + i) * vec + c;
      const int64_t bv = bk + static_cast<int64_t>(H.len) * vec;
      if (p.to_pool) {
        src_k[u] = bk; src_v[u] = bv; dst_k[u] = pool; dst_v[u] = pool;
      } else {
        src_k[u] = pool; src_v[u] = pool; dst_k[u] = bk; dst_v[u] = bv;
      }
    }
#pragma unroll
    for (int u = 0; u < kXferUnroll; ++u)
      if (src_k[u] >= 0) {
        kx[u] = p.to_pool ? __ldg(p.buf + src_k[u]) : __ldg(p.kpool + src_k[u]);
        vx[u] = p.to_pool ? __ldg(p.buf + src_v[u]) : __ldg(p.vpool + src_v[u]);
      }
#pragma unroll
    for (int u = 0; u < kXferUnroll; ++u)
      if (src_k[u] >= 0) {
        if (p.to_pool) {
          p.kpool[dst_k[u]] = kx[u];
          p.vpool[dst_v[u]] = vx[u];
        } else {
          p.buf_out[dst_k[u]] = kx[u];
          p.buf_out[dst_v[u]] = vx[u];
        }
      }
  }
}

cudaError_t launch_transfer(const TransferParams& p, const AppendBlob* blob, int grid,
                            cudaStream_t s) {
  static const AppendBlob empty_blob{};
  return launch_pdl(transfer_kernel, dim3(grid), dim3(256), p.n_heads * sizeof(XferHead), s, p,
                    blob ? *blob : empty_blob);
}

}  // namespace skv
