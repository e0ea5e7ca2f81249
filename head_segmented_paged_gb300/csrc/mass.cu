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
// Warp roles (320 threads; each CTA runs its own list of units from an LPT
// schedule):
//   warp 0      producer: the unit's K tile through the block table, then the
//               query tiles (TMA, 4 stages) with each row's position and
//               log2-domain lse staged beside them;
//   warp 1      TMEM owner (256 columns) and MMA issuer: S^T of query tile g
//               into TMEM buffer g % 2;
//   warps 2..9  two consumer groups of four warps, group x taking the
//               query tiles g with g % 2 == x: one thread per key,
//               p = 2^(s c - lse2) over the visible (key, row) pairs; the
//               groups add their sums at the end of a unit and group 0
//               stores them.
// A key tile seen by many query tiles (a global head's first keys) is cut
// into pieces that run as separate units; their partial sums meet in a
// scratch buffer and the last piece to finish adds them in piece order, so
// the total is still formed in one fixed order.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "segkv_internal.h"

namespace skv {
using namespace ptx;

namespace {

constexpr int MT = 128;           // keys per unit, rows per query tile
constexpr int NQ = 4;             // query-tile stages
constexpr int NG = 2;             // consumer groups; group x takes query tiles g with g % NG == x
constexpr int kThreadsM = 32 * (2 + 4 * NG);
constexpr uint32_t kAtomM = MT * 128;  // one 64-column, 128-row swizzle block
constexpr uint64_t kDrainNsM = 200ull * 1000 * 1000;
constexpr float kLog2e = 1.4426950408889634f;

enum {
  M_K_FULL = 0,
  M_K_EMPTY = 1,
  M_Q_FULL = 2,        // +stage
  M_Q_EMPTY = 2 + NQ,  // +stage
  M_S_FULL = 2 + 2 * NQ,        // +buffer (one per group)
  M_S_EMPTY = 2 + 2 * NQ + NG,  // +buffer
  M_RED_FULL = 2 + 2 * NQ + 2 * NG,
  M_RED_EMPTY = 3 + 2 * NQ + 2 * NG,
  M_DRAIN = 4 + 2 * NQ + 2 * NG,
  M_NUM = 5 + 2 * NQ + 2 * NG
};

template <int D>
struct MLayout {
  static constexpr uint32_t TILE = MT * D * 2;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_Q = TILE;                 // NQ stages
  static constexpr uint32_t OFF_ROW = OFF_Q + NQ * TILE;  // per stage: lse2[128], pos[128], meta[4]
  static constexpr uint32_t ROW_BYTES = MT * 8 + 16;
  static constexpr uint32_t OFF_RED = OFF_ROW + NQ * ROW_BYTES;  // float [NG - 1][128]
  static constexpr uint32_t OFF_BAR = (OFF_RED + (NG - 1) * MT * 4 + 7) & ~7u;
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
  int armed_k = -1, armed_q[NQ];
  for (int st = 0; st < NQ; ++st) armed_q[st] = -1;
  bool ok = true;
  int g = 0, ui = 0;
  for (int u = p.cta_begin[blockIdx.x]; ok && u < p.cta_begin[blockIdx.x + 1]; ++u, ++ui) {
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
    // the query tiles that see any key of the tile. Row r = token (r / G) x
    // head (r % G); each row's lse (log2 units) is loaded one tile ahead so
    // its latency overlaps the wait for a free stage.
    auto load_lse = [&](int qt, float (&l2)[MT / 32]) {
#pragma unroll
      for (int e = 0; e < MT / 32; ++e) {
        const int r = lane + 32 * e;
        const int t = qt * p.tpt + r / p.G;
        l2[e] = t < U.ntok ? __ldg(p.lse + static_cast<int64_t>(U.head * p.G + r % p.G) * p.total_q +
                                   U.tok0 + t)
                           : 0.f;
      }
    };
    float l_next[MT / 32];
    load_lse(U.qt0, l_next);
    for (int qt = U.qt0; qt <= U.qt1; ++qt, ++g) {
      float l_cur[MT / 32];
#pragma unroll
      for (int e = 0; e < MT / 32; ++e) l_cur[e] = l_next[e];
      if (qt < U.qt1) load_lse(qt + 1, l_next);
      const int st = g % NQ;
      const uint32_t ph = (g / NQ) & 1;
      if (!waitw(c.bar(M_Q_EMPTY + st), ph ^ 1, c.wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(c.bar(M_Q_FULL + st), L::TILE);
        for (int cc = 0; cc < NC; ++cc)
          tma_load_3d(c.sbase + L::OFF_Q + st * L::TILE + cc * kAtomM, tmq, cc * 64,
                      U.head * p.G, U.tok0 + qt * p.tpt, c.bar(M_Q_FULL + st));
      }
      armed_q[st] = static_cast<int>(ph);
      float* lse2 = reinterpret_cast<float*>(c.smem + L::OFF_ROW + st * L::ROW_BYTES);
      int* rpos = reinterpret_cast<int*>(lse2 + MT);
      int* meta = rpos + MT;
      const int tq0 = qt * p.tpt;  // first token of the tile; position -1: no such token
      const int last = min(U.ntok, tq0 + p.tpt) - 1;
#pragma unroll
      for (int e = 0; e < MT / 32; ++e) {
        const int r = lane + 32 * e;
        const int t = tq0 + r / p.G;
        lse2[r] = l_cur[e] * kLog2e;
        rpos[r] = t < U.ntok ? U.a + t : -1;
      }
      if (lane == 0) {
        meta[0] = U.a + tq0;             // smallest position of the tile
        meta[1] = U.a + last;            // largest
        meta[2] = tq0 + p.tpt <= U.ntok;  // every row is a token
      }
      __syncwarp();  // every lane's rows are written
      if (lane == 0) mbar_arrive(c.bar(M_Q_FULL + st));
    }
  }
  if (!ok && lane == 0) {  // aborting: let our own copies land before the block exits
    if (armed_k >= 0) wait_drain(c.bar(M_K_FULL), armed_k, kDrainNsM);
    for (int st = 0; st < NQ; ++st)
      if (armed_q[st] >= 0) wait_drain(c.bar(M_Q_FULL + st), armed_q[st], kDrainNsM);
  }
}

template <int D>
__device__ void m_mma(const MassParams& p, const MCtx& c) {
  using L = MLayout<D>;
  constexpr uint32_t IDESC = idesc_bf16(MT, MT, 0);
  bool ok = true;
  int g = 0, ui = 0;
  for (int u = p.cta_begin[blockIdx.x]; ok && u < p.cta_begin[blockIdx.x + 1]; ++u, ++ui) {
    const MassUnit U = p.units[u];
    if (!wait1(c.bar(M_K_FULL), ui & 1, c.wc)) { ok = false; break; }
    for (int qt = U.qt0; qt <= U.qt1; ++qt, ++g) {
      const int sb = g % NG, qs = g % NQ;
      if (!wait1(c.bar(M_S_EMPTY + sb), ((g / NG) & 1) ^ 1, c.wc)) { ok = false; break; }
      if (!wait1(c.bar(M_Q_FULL + qs), (g / NQ) & 1, c.wc)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t a = c.sbase + L::OFF_K + (kk >> 2) * kAtomM + (kk & 3) * 32;
        const uint32_t b = c.sbase + L::OFF_Q + qs * L::TILE + (kk >> 2) * kAtomM + (kk & 3) * 32;
        mma_bf16(c.tmem + sb * MT, sdesc_sw128(a, 16, 1024), sdesc_sw128(b, 16, 1024), IDESC,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit(c.bar(M_S_FULL + sb));
      mma_commit(c.bar(M_Q_EMPTY + qs));
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
  for (int u = p.cta_begin[blockIdx.x]; u < p.cta_begin[blockIdx.x + 1]; ++u, ++ui) {
    const MassUnit U = p.units[u];
    const int j = U.kt * MT + jl;           // this thread's key
    const int jw = U.kt * MT + wq * 32;     // the warp's first key
    float acc = 0.f;
    for (int qt = U.qt0; ok && qt <= U.qt1; ++qt, ++g) {
      if (g % NG != grp) continue;
      const int qs = g % NQ;
      if (!waitw(c.bar(M_Q_FULL + qs), (g / NQ) & 1, c.wc) ||
          !waitw(c.bar(M_S_FULL + grp), (g / NG) & 1, c.wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(c.smem + L::OFF_ROW + qs * L::ROW_BYTES);
      const int* rpos = reinterpret_cast<const int*>(lse2 + MT);
      const int* meta = rpos + MT;
      // every (key, row) pair of this warp visible: no per-element test
      const bool whole = meta[2] && jw + 31 <= meta[0] &&
                         (!U.local || meta[1] - p.window + 1 <= jw);
      float part[4] = {0.f, 0.f, 0.f, 0.f};
      // 32 columns at a time; the next quarter's TMEM load is in flight while
      // this one is summed
      auto quarter = [&](const uint32_t (&b)[32], int e0) {
        if (whole) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 l2 = *reinterpret_cast<const float2*>(lse2 + e0 + e);
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(b[e]), __uint_as_float(b[e + 1])),
                                        make_float2(sc, sc), make_float2(-l2.x, -l2.y));
            part[(e >> 1) & 3] += ex2(x.x) + ex2(x.y);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int pe = rpos[e0 + e];
            const bool vis = j <= pe && (!U.local || j >= pe - p.window + 1);
            const float x = fmaf(__uint_as_float(b[e]), sc, -lse2[e0 + e]);
            part[e & 3] += vis ? ex2(x) : 0.f;
          }
        }
      };
      uint32_t bA[32], bB[32];
      tmem_ld32(t_s, bA);
      tmem_wait_ld_dep(bA);
      tmem_ld32(t_s + 32, bB);
      quarter(bA, 0);
      tmem_wait_ld_dep(bB);
      tmem_ld32(t_s + 64, bA);
      quarter(bB, 32);
      tmem_wait_ld_dep(bA);
      tmem_ld32(t_s + 96, bB);
      quarter(bA, 64);
      tmem_wait_ld_dep(bB);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(M_S_EMPTY + grp));  // the S buffer is read
      quarter(bB, 96);
      acc += (part[0] + part[1]) + (part[2] + part[3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(M_Q_EMPTY + qs));
    }
    if (!ok) break;
    // the other groups hand their sums to group 0, which adds them in group
    // order and stores
    if (grp > 0) {
      if (!waitw(c.bar(M_RED_EMPTY), (ui & 1) ^ 1, c.wc)) break;
      red[(grp - 1) * MT + jl] = acc;
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(M_RED_FULL));
    } else {
      if (!waitw(c.bar(M_RED_FULL), ui & 1, c.wc)) break;
      float tot = acc;
#pragma unroll
      for (int x = 0; x < NG - 1; ++x) tot += red[x * MT + jl];
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(M_RED_EMPTY));
      if (U.n_pieces == 1) {
        if (j >= U.a && j < U.a + U.ntok)
          p.mass[static_cast<int64_t>(U.head) * p.total_q + U.tok0 + (j - U.a)] = tot;
      } else {
        // a split key tile: each warp posts its 32 sums; the warp that
        // finishes the tile last adds every piece in piece order
        p.part[static_cast<int64_t>(U.part0 + U.piece) * MT + jl] = tot;
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(p.tile_cnt + U.tile_id, 1) == 4 * U.n_pieces - 1;
        if (__shfl_sync(0xffffffffu, last, 0)) {
          __threadfence();
          for (int k = lane; k < MT; k += 32) {
            float sum = 0.f;
            for (int pc = 0; pc < U.n_pieces; ++pc)
              sum += __ldcg(p.part + static_cast<int64_t>(U.part0 + pc) * MT + k);
            const int jk = U.kt * MT + k;
            if (jk >= U.a && jk < U.a + U.ntok)
              p.mass[static_cast<int64_t>(U.head) * p.total_q + U.tok0 + (jk - U.a)] = sum;
          }
        }
      }
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
    for (int x = 0; x < NQ; ++x) {
      mbar_init(c.bar(M_Q_FULL + x), 2);  // the copy's arrival + the rows written
      mbar_init(c.bar(M_Q_EMPTY + x), 1 + 4);  // the MMA commit + the reading group's four warps
    }
    for (int x = 0; x < NG; ++x) {
      mbar_init(c.bar(M_S_FULL + x), 1);
      mbar_init(c.bar(M_S_EMPTY + x), 4);
    }
    mbar_init(c.bar(M_RED_FULL), 4 * (NG - 1));
    mbar_init(c.bar(M_RED_EMPTY), 4);
    mbar_init(c.bar(M_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), NG * MT);  // NG S buffers of 128 columns
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
    tmem_dealloc(c.tmem, NG * MT);
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
