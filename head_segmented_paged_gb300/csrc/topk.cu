// Token choice for sparse FFN routing (RedKnot summary page, section "稀疏 FFN
// （Sparse FFN）": the dense FFN runs on the top-k tokens by attention score).
//   score[t] = sum over KV heads h (in order) of mass[h, t], fp32;
//   per sequence, the k tokens with the largest score, ties to the lower
//   position, written in ascending position order.
// Selection is exact on the fp32 bit patterns: scores are non-negative, so
// their IEEE bits order like the values. One 1024-thread block per sequence
// finds the k-th largest pattern with four 8-bit radix passes (shared-memory
// histograms), then two ordered block scans place every chosen position.
#include <cuda_runtime.h>

#include <algorithm>

#include "segkv_internal.h"

namespace skv {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kTopkSmemValues = 11 * 1024;  // scores staged in shared memory up to this length

__global__ void score_sum_kernel(const float* __restrict__ mass, float* __restrict__ score,
                                 int64_t total, int hkv) {
  for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < total;
       t += int64_t(gridDim.x) * blockDim.x) {
    float s = mass[t];
    for (int h = 1; h < hkv; ++h) s += mass[h * total + t];
    score[t] = s;
  }
}

// Exclusive prefix sum over the block; *total receives the sum of all values.
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
  *total = warp_tot[31];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const float* __restrict__ score, TopkParams p, const __grid_constant__ AppendBlob blob) {
  const TopkSeq* seqs =
      p.plan_inline ? reinterpret_cast<const TopkSeq*>(blob.data + reinterpret_cast<uintptr_t>(p.seqs))
                    : p.seqs;
  const TopkSeq S = seqs[blockIdx.x];
  if (S.k <= 0) return;
  const int n = S.ntok, tid = threadIdx.x;
  __shared__ int hist[256];
  __shared__ int warp_tot[32];
  __shared__ int sel_digit, sel_need;
  __shared__ uint32_t staged[kTopkSmemValues];
  // the four passes read the scores from shared memory when they fit
  const uint32_t* bits = reinterpret_cast<const uint32_t*>(score + S.tok0);
  if (n <= kTopkSmemValues) {
    for (int t = tid; t < n; t += kTopkThreads) staged[t] = bits[t];
    __syncthreads();
    bits = staged;
  }
  // k-th largest bit pattern, 8 bits at a time from the top
  uint32_t prefix = 0, mask = 0;
  int need = S.k;  // how many to take from the bucket that matches prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    for (int t = tid; t < n; t += kTopkThreads) {
      const uint32_t b = bits[t];
      if ((b & mask) == prefix) atomicAdd(&hist[(b >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 32) {
      // digits from the top: lane l holds digits 255-8l .. 248-8l; the lane
      // whose bins cross `need` picks the digit
      int c[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[255 - 8 * tid - i];
        sum += c[i];
      }
      int before = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, before, o);
        if (tid >= o) before += y;
      }
      before -= sum;  // count of patterns in higher lanes' digits
      if (before < need && before + sum >= need) {
        int above = before, i = 0;
        for (; i < 7; ++i) {
          if (above + c[i] >= need) break;
          above += c[i];
        }
        sel_digit = 255 - 8 * tid - i;
        sel_need = need - above;
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sel_digit) << shift;
    mask |= 255u << shift;
    need = sel_need;
    __syncthreads();
  }
  // chosen: every pattern above the threshold, and the first `need` equal to it
  const int chunk = (n + kTopkThreads - 1) / kTopkThreads;
  const int t0 = min(n, tid * chunk), t1 = min(n, t0 + chunk);
  int eq = 0, gt = 0;
  for (int t = t0; t < t1; ++t) {
    const uint32_t b = bits[t];
    eq += b == prefix;
    gt += b > prefix;
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, warp_tot, &tot);
  const int take_eq = max(0, min(eq, need - eq_before));
  const int out_before = block_exclusive_scan(gt + take_eq, warp_tot, &tot);
  int o = S.out0 + out_before, eq_seen = eq_before;
  for (int t = t0; t < t1; ++t) {
    const uint32_t b = bits[t];
    bool take = b > prefix;
    if (b == prefix) take = eq_seen++ < need;
    if (take) p.idx[o++] = S.tok0 + t;
  }
}

}  // namespace

cudaError_t launch_topk(const float* mass, float* score, int64_t total, int hkv,
                        const TopkParams& p, const AppendBlob* blob, int n_seqs, cudaStream_t s) {
  static const AppendBlob empty_blob{};
  if (total > 0) {
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((total + threads - 1) / threads, 4096);
    score_sum_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(mass, score, total, hkv);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (n_seqs <= 0) return cudaSuccess;
  topk_kernel<<<n_seqs, kTopkThreads, 0, s>>>(score, p, blob ? *blob : empty_blob);
  return cudaGetLastError();
}

}  // namespace skv
