// Append / scatter: write each new token's K and V rows into the page that
// holds its position in every head's segment (RedKnot summary page, section
// "SegPagedAttention": the store is paged per (layer, head), and each head
// keeps only the tokens it needs; section "SegPaged Attention(段页注意力）":
// storage per head). Page ids were chosen on the host; this kernel also
// writes the new ids into the device block table.
//
// HBM bound: every 16-byte vector of K and V is read once and written once.
#include <algorithm>

#include "segkv_internal.h"

namespace skv {

template <class T>
__device__ __forceinline__ const T* plan_ptr(const T* p, const AppendBlob& blob, int inl) {
  return inl ? reinterpret_cast<const T*>(blob.data + reinterpret_cast<uintptr_t>(p)) : p;
}

__global__ void __launch_bounds__(256)
    append_kernel(AppendParams p, const __grid_constant__ AppendBlob blob) {
  // a kernel launched as a programmatic dependent of this one (decode) may
  // start its prologue now; it waits for this grid's completion before it
  // reads anything this grid writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  p.seqs = plan_ptr(p.seqs, blob, p.plan_inline);
  p.tiles = plan_ptr(p.tiles, blob, p.plan_inline);
  p.page_list = plan_ptr(p.page_list, blob, p.plan_inline);
  p.table_idx = plan_ptr(p.table_idx, blob, p.plan_inline);
  // block-table entries for the pages this call uses
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < p.n_entries;
       e += gridDim.x * blockDim.x)
    p.table[p.table_idx[e]] = p.page_list[e];

  const int row_vecs = p.hkv * p.vec_per_row;  // 16-byte vectors per token
  for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x) {
    const AppendTile tile = p.tiles[t];
    const AppendSeq sq = p.seqs[tile.seq];
    const int total = tile.ntok * row_vecs;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
      const int tl = i / row_vecs;
      const int rem = i - tl * row_vecs;
      const int h = rem / p.vec_per_row;
      const int c = rem - h * p.vec_per_row;
      const int tok = tile.tok0 + tl;
      const int pos = sq.pos0 + (tok - sq.tok0);
      const int k = pos / p.page_size;
      const int id = p.page_list[sq.list_off + h * sq.n_pages + (k - sq.first_k)];
      const int64_t src = (static_cast<int64_t>(tok) * p.hkv + h) * p.vec_per_row + c;
      const int64_t dst =
          (static_cast<int64_t>(id) * p.page_size + (pos - k * p.page_size)) * p.vec_per_row + c;
      const uint4 kv = __ldg(p.k + src);
      const uint4 vv = __ldg(p.v + src);
      p.kpool[dst] = kv;
      p.vpool[dst] = vv;
    }
  }
}

cudaError_t launch_append(const AppendParams& p, const AppendBlob* blob, int grid, cudaStream_t s) {
  static const AppendBlob empty_blob{};
  append_kernel<<<grid, 256, 0, s>>>(p, blob ? *blob : empty_blob);
  return cudaGetLastError();
}

// Plan upload on the SMs: copies a plan from mapped pinned host memory into
// device memory. A copy-engine transfer would queue behind the caller's own
// large host-to-device copies; this kernel only shares the link's bandwidth.
__global__ void plan_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n) {
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n;
       i += size_t(gridDim.x) * blockDim.x)
    dst[i] = src[i];
}

cudaError_t launch_plan_copy(const void* src, void* dst, size_t bytes, cudaStream_t s) {
  const size_t n = (bytes + 15) / 16;
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const size_t blocks = std::min<size_t>((n + threads - 1) / threads, 1024);
  plan_copy_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(static_cast<const uint4*>(src),
                                                                static_cast<uint4*>(dst), n);
  return cudaGetLastError();
}

}  // namespace skv
