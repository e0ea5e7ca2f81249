// Attention mass each token of a prefill chunk receives as a key: the score
// by which sparse FFN routing picks its tokens (RedKnot summary page, section
// "稀疏 FFN（Sparse FFN）": the dense FFN runs on the tokens with the highest
// attention scores). For key j of the chunk and KV head h:
//   mass[h, j] = sum over the chunk's query tokens q that see j, and over the
//                G query heads of h, of exp(scale q.k_j - lse_q)
// with lse_q the natural-log softmax denominator the prefill wrote.
//
// Keys are the stationary operand: a work unit is one KV head x one tile of
// 128 keys, and the query tiles that see any of them stream past it. The
// tensor core forms S^T = K Q^T (M = 128 keys in TMEM lanes, N = 128 packed
// query rows), so each thread owns one key and sums its 128 columns without
// any cross-thread reduction; a key's total is built inside one unit, in a
// fixed order, so the result does not depend on scheduling.
//
// Warp roles (320 threads, persistent over an LPT-sorted unit list):
//   warp 0      producer: the unit's K tile through the block table, then the
//               query tiles (TMA, 2 stages) with each row's position and
//               log2-domain lse staged beside them;
//   warp 1      TMEM owner (256 columns) and MMA issuer: S^T of query tile g
//               into TMEM buffer g % 2;
//   warps 2..5  consumer group 0 (even query tiles), warps 6..9 group 1
//               (odd tiles): one thread per key, p = 2^(s c - lse2) over the
//               visible (key, row) pairs; the groups add their sums at the end
//               of a unit and group 0 stores them.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "segkv_internal.h"

namespace skv {
using namespace ptx;

namespace {

constexpr int MT = 128;           // keys per unit, rows per query tile
constexpr int kThreadsM = 320;
constexpr uint32_t kAtomM = MT * 128;  // one 64-column, 128-row swizzle block
constexpr uint64_t kDrainNsM = 200ull * 1000 * 1000;
constexpr float kLog2e = 1.4426950408889634f;

enum {
  M_K_FULL = 0,
  M_K_EMPTY = 1,
  M_Q_FULL = 2,   // +stage
  M_Q_EMPTY = 4,  // +stage
  M_S_FULL = 6,   // +buffer
  M_S_EMPTY = 8,  // +buffer
  M_RED_FULL = 10,
  M_RED_EMPTY = 11,
  M_DRAIN = 12,
  M_NUM = 13
};

template <int D>
struct MLayout {
  static constexpr uint32_t TILE = MT * D * 2;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_Q = TILE;                 // 2 stages
  static constexpr uint32_t OFF_ROW = OFF_Q + 2 * TILE;   // per stage: lse2[128], pos[128], meta[4]
  static constexpr uint32_t ROW_BYTES = MT * 8 + 16;
  static constexpr uint32_t OFF_RED = OFF_ROW + 2 * ROW_BYTES;  // float [128]
  static constexpr uint32_t OFF_BAR = (OFF_RED + MT * 4 + 7) & ~7u;
  static constexpr uint32_t OFF_MISC = OFF_BAR + M_NUM * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16 + 1024;  // + slack to align to 1 KB
};

struct MCtx {
  uint8_t* smem;
  uint32_t sbase;
  uint32_t tmem;
  uint32_t off_bar;
  WaitCtx wc;
  __device__ uint32_t bar(int i) const { return sbase + off_bar + 8u * i; }
};

template <int D>
__device__ void m_producer(const CUtensorMap* tmq, const CUtensorMap* tmk, const MassParams& p,
                           const MCtx& c, int lane) {
  using L = MLayout<D>;
  constexpr int NC = D / 64;
  const int box_rows = p.page_size <= MT ? p.page_size : MT;
  const int boxes = MT / box_rows;
  int armed_k = -1, armed_q[2] = {-1, -1};
  bool ok = true;
  int g = 0, ui = 0;
  for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x, ++ui) {
    const MassUnit U = p.units[u];
    // the unit's key tile, page by page through the block table
    if (!waitw(c.bar(M_K_EMPTY), (ui & 1) ^ 1, c.wc)) { ok = false; break; }
    if (lane == 0) mbar_expect_tx(c.bar(M_K_FULL), L::TILE);
    armed_k = ui & 1;
    const int32_t* trow = p.table + static_cast<int64_t>(U.table_row) * p.R;
    for (int bi = 0; bi < boxes; ++bi) {
      const int pos = U.kt * MT + bi * box_rows;
      const int k = pos / p.page_size;
      int id = 0;
      if (k >= U.first_page && k <= U.last_page && lane == 0) id = trow[k];
      if (lane == 0) {
        const int y = (k >= U.first_page && k <= U.last_page)
                          ? id * p.page_size + (pos - k * p.page_size)
                          : p.oob_row;  // not held by the segment: zero fill
        for (int cc = 0; cc < NC; ++cc)
          tma_load_2d(c.sbase + L::OFF_K + bi * box_rows * 128 + cc * kAtomM, tmk, cc * 64, y,
                      c.bar(M_K_FULL));
      }
    }
    // the query tiles that see any key of the tile
    for (int qt = U.qt0; qt <= U.qt1; ++qt, ++g) {
      const int st = g & 1;
      const uint32_t ph = (g >> 1) & 1;
      if (!waitw(c.bar(M_Q_EMPTY + st), ph ^ 1, c.wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(c.bar(M_Q_FULL + st), L::TILE);
        for (int cc = 0; cc < NC; ++cc)
          tma_load_3d(c.sbase + L::OFF_Q + st * L::TILE + cc * kAtomM, tmq, cc * 64,
                      U.head * p.G, U.tok0 + qt * p.tpt, c.bar(M_Q_FULL + st));
      }
      armed_q[st] = static_cast<int>(ph);
      // row r = token (r / G) x head (r % G): position (-1: no such token) and lse in log2 units
      float* lse2 = reinterpret_cast<float*>(c.smem + L::OFF_ROW + st * L::ROW_BYTES);
      int* rpos = reinterpret_cast<int*>(lse2 + MT);
      int* meta = rpos + MT;
      int pmin = 1 << 30, pmax = -1, all_valid = 1;
#pragma unroll
      for (int e = 0; e < MT / 32; ++e) {
        const int r = lane + 32 * e;
        const int t = qt * p.tpt + r / p.G;
        int pos = -1;
        float l2 = 0.f;
        if (t < U.ntok) {
          pos = U.a + t;
          l2 = p.lse[static_cast<int64_t>(U.head * p.G + r % p.G) * p.total_q + U.tok0 + t] * kLog2e;
          pmin = min(pmin, pos);
          pmax = max(pmax, pos);
        } else {
          all_valid = 0;
        }
        lse2[r] = l2;
        rpos[r] = pos;
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, o));
        pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
      }
      all_valid = __all_sync(0xffffffffu, all_valid);
      if (lane == 0) {
        meta[0] = pmin;
        meta[1] = pmax;
        meta[2] = all_valid;
      }
      mbar_arrive(c.bar(M_Q_FULL + st));  // every lane: its rows are written
    }
  }
  if (!ok && lane == 0) {  // aborting: let our own copies land before the block exits
    if (armed_k >= 0) wait_drain(c.bar(M_K_FULL), armed_k, kDrainNsM);
    for (int st = 0; st < 2; ++st)
      if (armed_q[st] >= 0) wait_drain(c.bar(M_Q_FULL + st), armed_q[st], kDrainNsM);
  }
}

template <int D>
__device__ void m_mma(const MassParams& p, const MCtx& c) {
  using L = MLayout<D>;
  constexpr uint32_t IDESC = idesc_bf16(MT, MT, 0);
  bool ok = true;
  int g = 0, ui = 0;
  for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x, ++ui) {
    const MassUnit U = p.units[u];
    if (!wait1(c.bar(M_K_FULL), ui & 1, c.wc)) { ok = false; break; }
    for (int qt = U.qt0; qt <= U.qt1; ++qt, ++g) {
      const int st = g & 1;
      const uint32_t ph = (g >> 1) & 1;
      if (!wait1(c.bar(M_S_EMPTY + st), ph ^ 1, c.wc)) { ok = false; break; }
      if (!wait1(c.bar(M_Q_FULL + st), ph, c.wc)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t a = c.sbase + L::OFF_K + (kk >> 2) * kAtomM + (kk & 3) * 32;
        const uint32_t b = c.sbase + L::OFF_Q + st * L::TILE + (kk >> 2) * kAtomM + (kk & 3) * 32;
        mma_bf16(c.tmem + st * MT, sdesc_sw128(a, 16, 1024), sdesc_sw128(b, 16, 1024), IDESC,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit(c.bar(M_S_FULL + st));
      mma_commit(c.bar(M_Q_EMPTY + st));
    }
    if (ok) mma_commit(c.bar(M_K_EMPTY));
  }
  if (!ok) {  // aborting: let issued MMAs finish before TMEM is freed
    mma_commit(c.bar(M_DRAIN));
    wait_drain(c.bar(M_DRAIN), 0, kDrainNsM);
  }
}

template <int D>
__device__ void m_consumer(const MassParams& p, const MCtx& c, int grp, int warp, int lane) {
  using L = MLayout<D>;
  const int wq = warp & 3;  // TMEM lane quarter this warp may access
  const int jl = wq * 32 + lane;
  const uint32_t t_s = c.tmem + (static_cast<uint32_t>(wq * 32) << 16) + grp * MT;
  float* red = reinterpret_cast<float*>(c.smem + L::OFF_RED);
  const float sc = p.scale_log2;
  int g = 0, ui = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++ui) {
    const MassUnit U = p.units[u];
    const int j = U.kt * MT + jl;           // this thread's key
    const int jw = U.kt * MT + wq * 32;     // the warp's first key
    float acc = 0.f;
    for (int qt = U.qt0; ok && qt <= U.qt1; ++qt, ++g) {
      if ((g & 1) != grp) continue;
      const uint32_t ph = (g >> 1) & 1;
      if (!waitw(c.bar(M_Q_FULL + grp), ph, c.wc) || !waitw(c.bar(M_S_FULL + grp), ph, c.wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(c.smem + L::OFF_ROW + grp * L::ROW_BYTES);
      const int* rpos = reinterpret_cast<const int*>(lse2 + MT);
      const int* meta = rpos + MT;
      // every (key, row) pair of this warp visible: no per-element test
      const bool whole = meta[2] && jw + 31 <= meta[0] &&
                         (!U.local || meta[1] - p.window + 1 <= jw);
      float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // 64 columns at a time keeps s in registers
        float s[MT / 2];
        tmem_ld32(t_s + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(t_s + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_wait_ld();
        if (half == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(c.bar(M_S_EMPTY + grp));
        }
        const int e0 = half * 64;
        if (whole) {
#pragma unroll
          for (int e = 0; e < MT / 2; e += 2) {
            const float2 l2 = *reinterpret_cast<const float2*>(lse2 + e0 + e);
            const float2 x = __ffma2_rn(make_float2(s[e], s[e + 1]), make_float2(sc, sc),
                                        make_float2(-l2.x, -l2.y));
            part[(e >> 1) & 3] += ex2(x.x) + ex2(x.y);
          }
        } else {
#pragma unroll
          for (int e = 0; e < MT / 2; ++e) {
            const int pe = rpos[e0 + e];
            const bool vis = j <= pe && (!U.local || j >= pe - p.window + 1);
            const float x = fmaf(s[e], sc, -lse2[e0 + e]);
            part[e & 3] += vis ? ex2(x) : 0.f;
          }
        }
      }
      acc += (part[0] + part[1]) + (part[2] + part[3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(M_Q_EMPTY + grp));
    }
    if (!ok) break;
    // group 1 hands its sums to group 0, which adds them and stores
    if (grp == 1) {
      if (!waitw(c.bar(M_RED_EMPTY), (ui & 1) ^ 1, c.wc)) break;
      red[jl] = acc;
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(M_RED_FULL));
    } else {
      if (!waitw(c.bar(M_RED_FULL), ui & 1, c.wc)) break;
      const float tot = acc + red[jl];
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(M_RED_EMPTY));
      if (j >= U.a && j < U.a + U.ntok)
        p.mass[static_cast<int64_t>(U.head) * p.total_q + U.tok0 + (j - U.a)] = tot;
    }
  }
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreadsM, 1)
    mass_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                const MassParams p) {
  using L = MLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  MCtx c;
  c.smem = smem;
  c.sbase = smem_addr(smem);
  c.off_bar = L::OFF_BAR;
  if (threadIdx.x == 0) {
    mbar_init(c.bar(M_K_FULL), 1);
    mbar_init(c.bar(M_K_EMPTY), 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(c.bar(M_Q_FULL + x), 1 + 32);  // the copy's arrival + every producer lane
      mbar_init(c.bar(M_Q_EMPTY + x), 1 + 4);  // the MMA commit + the group's four warps
      mbar_init(c.bar(M_S_FULL + x), 1);
      mbar_init(c.bar(M_S_EMPTY + x), 4);
    }
    mbar_init(c.bar(M_RED_FULL), 4);
    mbar_init(c.bar(M_RED_EMPTY), 4);
    mbar_init(c.bar(M_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 2 * MT);
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
    m_producer<D>(&tmq, &tmk, p, c, lane);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) m_mma<D>(p, c);
    __syncwarp();
  } else {
    m_consumer<D>(p, c, (warp - 2) >> 2, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(c.tmem, 2 * MT);
  }
}

cudaError_t launch_mass(const MassParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                        int head_dim, int grid, cudaStream_t s) {
  if (head_dim == 64) {
    const int bytes = MLayout<64>::BYTES;
    cudaError_t e =
        cudaFuncSetAttribute(mass_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    mass_kernel<64><<<grid, kThreadsM, bytes, s>>>(tq, tk, p);
  } else {
    const int bytes = MLayout<128>::BYTES;
    cudaError_t e =
        cudaFuncSetAttribute(mass_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    mass_kernel<128><<<grid, kThreadsM, bytes, s>>>(tq, tk, p);
  }
  return cudaGetLastError();
}

}  // namespace skv
