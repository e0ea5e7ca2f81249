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

__global__ void __launch_bounds__(256)
    transfer_kernel(TransferParams p, const __grid_constant__ AppendBlob blob) {
  const TransferRun* runs = xfer_plan_ptr(p.runs, blob, p.plan_inline);
  const int32_t* page_list = xfer_plan_ptr(p.page_list, blob, p.plan_inline);
  const int64_t* table_idx = xfer_plan_ptr(p.table_idx, blob, p.plan_inline);
  // block-table entries of the pages an import takes
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < p.n_entries;
       e += gridDim.x * blockDim.x)
    p.table[table_idx[e]] = page_list[e];
  const int vec = p.vec_per_row;
  for (int r = blockIdx.x; r < p.n_runs; r += gridDim.x) {
    const TransferRun run = runs[r];
    const int64_t pool_row = static_cast<int64_t>(run.page) * p.page_size + run.slot0;
    const int items = run.nrows * vec;
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
      const int row = it / vec, c = it - row * vec;
      const int64_t pk = (pool_row + row) * vec + c;
      const int64_t bk = (static_cast<int64_t>(run.k_row) + row) * vec + c;
      const int64_t bv = (static_cast<int64_t>(run.v_row) + row) * vec + c;
      if (p.to_pool) {
        p.kpool[pk] = __ldg(p.buf + bk);
        p.vpool[pk] = __ldg(p.buf + bv);
      } else {
        p.buf_out[bk] = __ldg(p.kpool + pk);
        p.buf_out[bv] = __ldg(p.vpool + pk);
      }
    }
  }
}

cudaError_t launch_transfer(const TransferParams& p, const AppendBlob* blob, int grid,
                            cudaStream_t s) {
  static const AppendBlob empty_blob{};
  transfer_kernel<<<grid, 256, 0, s>>>(p, blob ? *blob : empty_blob);
  return cudaGetLastError();
}

}  // namespace skv
