// Sparse FFN routing, compute side (RedKnot summary page, section "稀疏 FFN
// （Sparse FFN）": only the tokens with the highest attention scores go
// through the dense FFN, every other token takes the residual identity
// path). For the m chosen rows:
//   X   = x[idx]                               (gather, HBM bound)
//   H   = silu(X W_gate^T) * (X W_up^T)        (GEMM 1, SwiGLU fused in its epilogue)
//   residual[idx] += H W_down^T                (GEMM 2, scatter-add fused in its epilogue)
// Rows not chosen are never read or written.
//
// Both GEMMs run on one persistent tcgen05 kernel (cta_group::1, M = 128
// rows, N = 256 accumulator columns, K steps of 64, both operands
// K-major in 128-byte-swizzled shared memory, fed by TMA through a 4-stage
// ring). TMEM holds two 256-column accumulators, so the epilogue of one tile
// overlaps the MMAs of the next. Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer (A tile 128 x 64, B tile 256 x 64 as two 128-row boxes);
//   warp 1      TMEM owner and MMA issuer;
//   warps 2..5  epilogue, one thread per accumulator row (TMEM lane).
// In GEMM 1 the B tile stacks 128 rows of W_gate over the same 128 rows of
// W_up, so one accumulator holds gate (columns 0..127) and up (128..255) of
// 128 hidden features and the epilogue forms h = silu(g) * u directly.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "segkv_internal.h"

namespace skv {
using namespace ptx;

namespace {

constexpr int GM = 128, GN = 256, GK = 64;
constexpr int kStages = 4;
constexpr int kThreadsG = 192;
constexpr uint32_t kABytes = GM * GK * 2;  // 16 KB
constexpr uint32_t kBHalf = 128 * GK * 2;  // 16 KB
constexpr uint32_t kStageBytes = kABytes + 2 * kBHalf;
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;

enum {
  G_FULL = 0,                    // +stage
  G_EMPTY = kStages,             // +stage
  G_ACC_FULL = 2 * kStages,      // +buffer
  G_ACC_EMPTY = 2 * kStages + 2, // +buffer
  G_DRAIN = 2 * kStages + 4,
  G_NUM = 2 * kStages + 5
};
constexpr uint32_t OFF_BAR = kStages * kStageBytes;
constexpr uint32_t OFF_MISC = OFF_BAR + G_NUM * 8;
constexpr uint32_t GEMM_SMEM = OFF_MISC + 16 + 1024;  // + slack to align the ring to 1 KB

struct GCtx {
  uint32_t sbase;
  uint32_t tmem;
  WaitCtx wc;
  __device__ uint32_t bar(int i) const { return sbase + OFF_BAR + 8u * i; }
  __device__ uint32_t a(int st) const { return sbase + st * kStageBytes; }
  __device__ uint32_t b(int st) const { return sbase + st * kStageBytes + kABytes; }
};

__device__ __forceinline__ void tile_of(const FfnGemmParams& p, int t, int* tm, int* tn) {
  *tn = t / p.tiles_m;  // consecutive CTAs share a B column, which stays in L2
  *tm = t - *tn * p.tiles_m;
}

template <int EPI>
__device__ void g_producer(const CUtensorMap* ta, const CUtensorMap* tb0, const CUtensorMap* tb1,
                           const FfnGemmParams& p, const GCtx& c, int lane) {
  const int nk = p.K / GK, tiles = p.tiles_m * p.tiles_n;
  int armed[kStages];
  for (int s = 0; s < kStages; ++s) armed[s] = -1;
  bool ok = true;
  int it = 0;
  for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
    int tm, tn;
    tile_of(p, t, &tm, &tn);
    // GEMM 1: gate rows f0.., up rows f0..; GEMM 2: W_down rows n0.. and n0+128..
    const int r0 = EPI == 0 ? tn * 128 : tn * GN;
    const int r1 = EPI == 0 ? tn * 128 : tn * GN + 128;
    for (int ks = 0; ks < nk; ++ks, ++it) {
      const int st = it % kStages;
      const uint32_t ph = (it / kStages) & 1;
      if (!waitw(c.bar(G_EMPTY + st), ph ^ 1, c.wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(c.bar(G_FULL + st), kStageBytes);
        tma_load_2d(c.a(st), ta, ks * GK, tm * GM, c.bar(G_FULL + st));
        tma_load_2d(c.b(st), tb0, ks * GK, r0, c.bar(G_FULL + st));
        tma_load_2d(c.b(st) + kBHalf, tb1, ks * GK, r1, c.bar(G_FULL + st));
      }
      armed[st] = static_cast<int>(ph);
    }
  }
  if (!ok && lane == 0)
    for (int s = 0; s < kStages; ++s)
      if (armed[s] >= 0) wait_drain(c.bar(G_FULL + s), armed[s], kDrainNs);
}

__device__ void g_mma(const FfnGemmParams& p, const GCtx& c) {
  constexpr uint32_t IDESC = idesc_bf16(GM, GN, 0);
  const int nk = p.K / GK, tiles = p.tiles_m * p.tiles_n;
  bool ok = true;
  int it = 0, tc = 0;
  for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++tc) {
    const int buf = tc & 1;
    if (!wait1(c.bar(G_ACC_EMPTY + buf), ((tc >> 1) & 1) ^ 1, c.wc)) { ok = false; break; }
    tc_fence_after();
    for (int ks = 0; ks < nk; ++ks, ++it) {
      const int st = it % kStages;
      if (!wait1(c.bar(G_FULL + st), (it / kStages) & 1, c.wc)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < GK / 16; ++kk)
        mma_bf16(c.tmem + buf * GN, sdesc_sw128(c.a(st) + kk * 32, 16, 1024),
                 sdesc_sw128(c.b(st) + kk * 32, 16, 1024), IDESC, (ks | kk) ? 1u : 0u);
      mma_commit(c.bar(G_EMPTY + st));
    }
    if (ok) mma_commit(c.bar(G_ACC_FULL + buf));
  }
  if (!ok) {  // aborting: let issued MMAs finish before TMEM is freed
    mma_commit(c.bar(G_DRAIN));
    wait_drain(c.bar(G_DRAIN), 0, kDrainNs);
  }
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  // silu(g) * u = g * u / (1 + e^-g), e^-g = 2^(-g log2 e)
  return g * u * __frcp_rn(1.0f + ex2(-1.4426950408889634f * g));
}

template <int EPI>
__device__ void g_epilogue(const FfnGemmParams& p, const GCtx& c, int warp, int lane) {
  const int tiles = p.tiles_m * p.tiles_n;
  const int wq = warp & 3;  // the TMEM lane quarter this warp may access
  const int row = wq * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  int tc = 0;
  for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++tc) {
    const int buf = tc & 1;
    if (!waitw(c.bar(G_ACC_FULL + buf), (tc >> 1) & 1, c.wc)) break;
    tc_fence_after();
    int tm, tn;
    tile_of(p, t, &tm, &tn);
    const int m = tm * GM + row;
    const uint32_t tacc = c.tmem + lane_off + buf * GN;
    if constexpr (EPI == 0) {
      __nv_bfloat16* hrow = static_cast<__nv_bfloat16*>(p.out) +
                            static_cast<int64_t>(m) * p.n_out + tn * 128;
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t g[32], u[32];
        tmem_ld32(tacc + c0, g);
        tmem_ld32(tacc + 128 + c0, u);
        tmem_wait_ld();
        if (m < p.M) {
          uint4* dst = reinterpret_cast<uint4*>(hrow + c0);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 w;
            w.x = pack_bf16x2(silu_mul(__uint_as_float(g[8 * e + 0]), __uint_as_float(u[8 * e + 0])),
                              silu_mul(__uint_as_float(g[8 * e + 1]), __uint_as_float(u[8 * e + 1])));
            w.y = pack_bf16x2(silu_mul(__uint_as_float(g[8 * e + 2]), __uint_as_float(u[8 * e + 2])),
                              silu_mul(__uint_as_float(g[8 * e + 3]), __uint_as_float(u[8 * e + 3])));
            w.z = pack_bf16x2(silu_mul(__uint_as_float(g[8 * e + 4]), __uint_as_float(u[8 * e + 4])),
                              silu_mul(__uint_as_float(g[8 * e + 5]), __uint_as_float(u[8 * e + 5])));
            w.w = pack_bf16x2(silu_mul(__uint_as_float(g[8 * e + 6]), __uint_as_float(u[8 * e + 6])),
                              silu_mul(__uint_as_float(g[8 * e + 7]), __uint_as_float(u[8 * e + 7])));
            dst[e] = w;
          }
        }
      }
    } else {
      // the output row: idx[m], or m itself for the dense FFN (idx NULL)
      int dst_row = -1;
      if (m < p.M) {
        dst_row = p.idx ? p.idx[m] : m;
        if (dst_row < 0 || dst_row >= p.n_rows) {
          atomicExch(p.status, kStatusBadIndex);
          dst_row = -1;
        }
      }
      __nv_bfloat16* rrow = static_cast<__nv_bfloat16*>(p.out) +
                            static_cast<int64_t>(dst_row < 0 ? 0 : dst_row) * p.n_out + tn * GN;
#pragma unroll 1
      for (int c0 = 0; c0 < GN; c0 += 32) {
        if (tn * GN + c0 >= p.n_out) break;  // uniform over the warp
        uint32_t a[32];
        tmem_ld32(tacc + c0, a);
        tmem_wait_ld();
        if (dst_row >= 0) {
          uint4* ptr = reinterpret_cast<uint4*>(rrow + c0);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint4 r = ptr[e];
            const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
            uint32_t ow[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float lo = __uint_as_float(rw[q] << 16) + __uint_as_float(a[8 * e + 2 * q]);
              const float hi = __uint_as_float(rw[q] & 0xffff0000u) + __uint_as_float(a[8 * e + 2 * q + 1]);
              ow[q] = pack_bf16x2(lo, hi);
            }
            ptr[e] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(G_ACC_EMPTY + buf));
  }
}

template <int EPI>
__global__ void __launch_bounds__(kThreadsG, 1)
    ffn_gemm_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb0,
                    const __grid_constant__ CUtensorMap tb1, const FfnGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  GCtx c;
  c.sbase = smem_addr(smem);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(c.bar(G_FULL + s), 1);
      mbar_init(c.bar(G_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.bar(G_ACC_FULL + b), 1);
      mbar_init(c.bar(G_ACC_EMPTY + b), 4);  // one arrival per epilogue warp
    }
    mbar_init(c.bar(G_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&ta);
    prefetch_tmap(&tb0);
    prefetch_tmap(&tb1);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tmem = *tmem_slot;
  c.wc.abort = abort_flag;
  c.wc.status = p.status;
  c.wc.limit_ns = p.timeout_ns;
  if (warp == 0) {
    g_producer<EPI>(&ta, &tb0, &tb1, p, c, lane);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) g_mma(p, c);
    __syncwarp();
  } else {
    g_epilogue<EPI>(p, c, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(c.tmem, 512);
  }
}

// out[r] = x[idx[r]] for r < m; one warp per row, 16-byte vectors.
__global__ void gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ idx,
                                   uint4* __restrict__ out, int m, int row_vec, int64_t n_rows,
                                   int* status) {
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= m) return;
  const int src = idx[r];
  const int lane = threadIdx.x & 31;
  if (src < 0 || src >= n_rows) {  // leave the row as it is and report
    if (lane == 0) atomicExch(status, kStatusBadIndex);
    return;
  }
  const uint4* s = x + static_cast<int64_t>(src) * row_vec;
  uint4* d = out + static_cast<int64_t>(r) * row_vec;
  for (int i = lane; i < row_vec; i += 32) d[i] = s[i];
}

template <int EPI>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb0, const CUtensorMap& tb1,
                        const FfnGemmParams& p, int grid, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= kMaxDevices || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(ffn_gemm_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) attr_set[dev] = true;
  }
  ffn_gemm_kernel<EPI><<<grid, kThreadsG, GEMM_SMEM, s>>>(ta, tb0, tb1, p);
  return cudaGetLastError();
}

}  // namespace

int ffn_tile_rows() { return GM; }

cudaError_t launch_gather_rows(const void* x, const int32_t* idx, void* out, int m, int d_model,
                               int64_t n_rows, int* status, cudaStream_t s) {
  if (m <= 0) return cudaSuccess;
  const int warps = 8;
  gather_rows_kernel<<<(m + warps - 1) / warps, warps * 32, 0, s>>>(
      static_cast<const uint4*>(x), idx, static_cast<uint4*>(out), m, d_model / 8, n_rows, status);
  return cudaGetLastError();
}

cudaError_t launch_ffn_gemm(int epilogue, const CUtensorMap& ta, const CUtensorMap& tb0,
                            const CUtensorMap& tb1, const FfnGemmParams& p, int grid,
                            cudaStream_t s) {
  return epilogue == 0 ? launch_gemm<0>(ta, tb0, tb1, p, grid, s)
                       : launch_gemm<1>(ta, tb0, tb1, p, grid, s);
}

}  // namespace skv
