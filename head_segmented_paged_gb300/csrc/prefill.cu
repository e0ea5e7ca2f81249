// Prefill attention over head-segmented pages on the 5th-generation tensor
// core (RedKnot summary page, section "SegPagedAttention（存储与执行底座）": one
// fused varlen attention kernel over per-(layer, head) paged segments, every
// head on the fast path, no attn_mask). Online softmax with a running maximum
// (KV-cache architecture page, section 5.2).
//
// One work unit = one KV head x one tile of 128 query rows. Rows pack the G
// query heads that share the KV head: row r = token (r / G) x head (r % G), so
// one K/V tile feeds every head of the group (GQA packing). Keys are visited
// in tiles of 128 positions; each tile's pages are fetched by TMA through the
// segment's block table. Pages outside the segment are read as zeros (an
// out-of-range TMA coordinate), and per-row masks keep every row to its own
// key set: j <= p, and j >= p-W+1 for a local head.
//
// Warp roles (192 threads, one CTA per SM, persistent over an LPT-sorted
// unit list):
//   warp 0      TMA producer: Q tile, then K and V tiles into a 2-stage ring;
//   warp 1      TMEM owner and MMA issuer: S = Q K^T into a double-buffered
//               TMEM accumulator, then O += P V into a TMEM accumulator;
//   warps 2..5  softmax (one thread per row): read S from TMEM, mask, update
//               the running max (O is rescaled in TMEM only when the max grows
//               by more than 2^8, which is exact), write P as bf16 to shared
//               memory; after the last tile, normalise O and store it.
// TMEM columns: S buffers [0,128) and [128,256), O [256, 256+D).
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "segkv_internal.h"

namespace skv {
using namespace ptx;

namespace {

constexpr int BM = kRowsPerTile;
constexpr int BN = kKeyTile;
constexpr int kThreads = 192;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kAtom = BM * 128;  // one 64-column, 128-row swizzle block (16 KB)
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;
constexpr uint64_t kDebugWaitNs = 20ull * 1000 * 1000;

enum {
  B_Q_FULL = 0,
  B_Q_EMPTY = 1,
  B_K_FULL = 2,    // +stage
  B_V_FULL = 4,    // +stage
  B_KV_EMPTY = 6,  // +stage
  B_S_FULL = 8,    // +buffer
  B_S_EMPTY = 10,  // +buffer
  B_P_FULL = 12,
  B_O_DONE = 13,
  B_O_EMPTY = 14,
  B_NEVER = 15,
  B_DRAIN = 16,
  NUM_BARS = 17
};

template <int D>
struct Layout {
  static constexpr uint32_t Q_BYTES = BM * D * 2;
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr uint32_t P_BYTES = BM * BN * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + 2 * KV_BYTES;
  static constexpr uint32_t OFF_P = OFF_V + 2 * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_P + P_BYTES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  // + slack to align to 1 KB; at least 116 KB so that one CTA holds an SM (and
  // its 512 TMEM columns) alone
  static constexpr uint32_t RAW = OFF_MISC + 16 + 1024;
  static constexpr uint32_t BYTES = RAW > 116u * 1024 ? RAW : 116u * 1024;
};

struct Ctx {
  uint8_t* smem;
  uint32_t sbase;
  uint32_t tmem;
  WaitCtx wc;
  __device__ uint32_t bar(int i, uint32_t off_bar) const { return sbase + off_bar + 8u * i; }
};

// ---------------------------------------------------------------- producer
template <int D>
__device__ void producer(const CUtensorMap* tmq, const CUtensorMap* tmk, const CUtensorMap* tmv,
                         const PrefillParams& p, const Ctx& c) {
  using L = Layout<D>;
  constexpr int NC = D / 64;
  const int box_rows = p.page_size <= BN ? p.page_size : BN;
  const int boxes = BN / box_rows;
  int armed_q = -1, armed_kv[2] = {-1, -1};
  bool ok = true;
  int g = 0, ui = 0;
  for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x, ++ui) {
    const PrefillUnit U = p.units[u];
    if (!wait1(c.bar(B_Q_EMPTY, L::OFF_BAR), (ui & 1) ^ 1, c.wc)) { ok = false; break; }
    mbar_expect_tx(c.bar(B_Q_FULL, L::OFF_BAR), L::Q_BYTES);
    for (int cc = 0; cc < NC; ++cc)
      tma_load_3d(c.sbase + L::OFF_Q + cc * kAtom, tmq, cc * 64, U.head * p.G, U.tok0,
                  c.bar(B_Q_FULL, L::OFF_BAR));
    armed_q = ui & 1;
    const int32_t* trow = p.table + static_cast<int64_t>(U.table_row) * p.R;
    for (int kt = U.kt0; kt <= U.kt1; ++kt, ++g) {
      const int st = g & 1;
      const uint32_t ph = (g >> 1) & 1;
      if (!wait1(c.bar(B_KV_EMPTY + st, L::OFF_BAR), ph ^ 1, c.wc)) { ok = false; break; }
      mbar_expect_tx(c.bar(B_K_FULL + st, L::OFF_BAR), L::KV_BYTES);
      mbar_expect_tx(c.bar(B_V_FULL + st, L::OFF_BAR), L::KV_BYTES);
      armed_kv[st] = static_cast<int>(ph);
      for (int bi = 0; bi < boxes; ++bi) {
        const int pos = kt * BN + bi * box_rows;
        const int k = pos / p.page_size;
        int y = p.oob_row;  // zero fill: page not held by this segment
        if (k >= U.first_page && k <= U.last_page) y = trow[k] * p.page_size + (pos - k * p.page_size);
        const uint32_t off = st * L::KV_BYTES + bi * box_rows * 128;
        for (int cc = 0; cc < NC; ++cc) {
          tma_load_2d(c.sbase + L::OFF_K + off + cc * kAtom, tmk, cc * 64, y,
                      c.bar(B_K_FULL + st, L::OFF_BAR));
          tma_load_2d(c.sbase + L::OFF_V + off + cc * kAtom, tmv, cc * 64, y,
                      c.bar(B_V_FULL + st, L::OFF_BAR));
        }
      }
    }
  }
  if (!ok) {  // aborting: let our own copies land before the block exits
    if (armed_q >= 0) wait_drain(c.bar(B_Q_FULL, L::OFF_BAR), armed_q, kDrainNs);
    for (int st = 0; st < 2; ++st)
      if (armed_kv[st] >= 0) {
        wait_drain(c.bar(B_K_FULL + st, L::OFF_BAR), armed_kv[st], kDrainNs);
        wait_drain(c.bar(B_V_FULL + st, L::OFF_BAR), armed_kv[st], kDrainNs);
      }
  }
}

// ---------------------------------------------------------------- MMA issuer
template <int D>
__device__ bool issue_pv(const Ctx& c, int gj, bool first, int ui) {
  using L = Layout<D>;
  constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, 1);
  if (first && !wait1(c.bar(B_O_EMPTY, L::OFF_BAR), (ui & 1) ^ 1, c.wc)) return false;
  if (!wait1(c.bar(B_P_FULL, L::OFF_BAR), gj & 1, c.wc)) return false;
  const int st = gj & 1;
  if (!wait1(c.bar(B_V_FULL + st, L::OFF_BAR), (gj >> 1) & 1, c.wc)) return false;
  tc_fence_after();
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    const uint32_t a = c.sbase + L::OFF_P + (kk >> 2) * kAtom + (kk & 3) * 32;
    const uint32_t b = c.sbase + L::OFF_V + st * L::KV_BYTES + kk * 2048;
    mma_bf16(c.tmem + 256, sdesc_sw128(a, 16, 1024), sdesc_sw128(b, kAtom, 1024), IDESC_PV,
             (first && kk == 0) ? 0u : 1u);
  }
  mma_commit(c.bar(B_O_DONE, L::OFF_BAR));
  mma_commit(c.bar(B_KV_EMPTY + st, L::OFF_BAR));
  return true;
}

template <int D>
__device__ void mma_issuer(const PrefillParams& p, const Ctx& c) {
  using L = Layout<D>;
  constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, 0);
  bool ok = true;
  if (p.debug & 1) {  // test hook: one wait on a barrier nothing signals
    WaitCtx w = c.wc;
    w.limit_ns = kDebugWaitNs;
    wait1(c.bar(B_NEVER, L::OFF_BAR), 0, w);
    ok = false;
  }
  int g = 0, ui = 0;
  for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x, ++ui) {
    const PrefillUnit U = p.units[u];
    const int nt = U.kt1 - U.kt0 + 1;
    if (!wait1(c.bar(B_Q_FULL, L::OFF_BAR), ui & 1, c.wc)) { ok = false; break; }
    tc_fence_after();
    for (int i = 0; i < nt; ++i) {
      const int gi = g + i, st = gi & 1;
      const uint32_t ph = (gi >> 1) & 1;
      if (!wait1(c.bar(B_K_FULL + st, L::OFF_BAR), ph, c.wc) ||
          !wait1(c.bar(B_S_EMPTY + st, L::OFF_BAR), ph ^ 1, c.wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t a = c.sbase + L::OFF_Q + (kk >> 2) * kAtom + (kk & 3) * 32;
        const uint32_t b = c.sbase + L::OFF_K + st * L::KV_BYTES + (kk >> 2) * kAtom + (kk & 3) * 32;
        mma_bf16(c.tmem + st * BN, sdesc_sw128(a, 16, 1024), sdesc_sw128(b, 16, 1024), IDESC_QK,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit(c.bar(B_S_FULL + st, L::OFF_BAR));
      if (i > 0 && !issue_pv<D>(c, gi - 1, i == 1, ui)) { ok = false; break; }
    }
    if (!ok || !issue_pv<D>(c, g + nt - 1, nt == 1, ui)) { ok = false; break; }
    mma_commit(c.bar(B_Q_EMPTY, L::OFF_BAR));
    g += nt;
  }
  if (!ok) {  // aborting: let issued MMAs finish before TMEM is freed
    mma_commit(c.bar(B_DRAIN, L::OFF_BAR));
    wait_drain(c.bar(B_DRAIN, L::OFF_BAR), 0, kDrainNs);
  }
}

// ---------------------------------------------------------------- softmax
template <int D>
__device__ void softmax_epilogue(const PrefillParams& p, const Ctx& c, int warp, int lane) {
  using L = Layout<D>;
  constexpr int NC = D / 64;
  const int wq = warp & 3;  // TMEM lane quarter this warp may access
  const int r = wq * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t t_o = c.tmem + lane_off + 256;
  int g = 0, ui = 0;
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++ui) {
    const PrefillUnit U = p.units[u];
    const int nt = U.kt1 - U.kt0 + 1;
    const int t = r / p.G, gg = r - t * p.G;
    const bool row_ok = t < U.ntok;
    const int tok = U.tok0 + t;
    int hi = -1, lo = 1 << 30;  // an invalid row sees no key
    if (row_ok) {
      hi = p.q_pos[tok];
      lo = U.local ? max(0, hi - p.window + 1) : 0;
    }
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < nt; ++i) {
      const int gi = g + i, st = gi & 1;
      const uint32_t ph = (gi >> 1) & 1;
      const int j0 = (U.kt0 + i) * BN;
      if (!waitw(c.bar(B_S_FULL + st, L::OFF_BAR), ph, c.wc)) { ok = false; break; }
      tc_fence_after();
      float s[BN];
#pragma unroll
      for (int q = 0; q < BN / 32; ++q) {
        uint32_t v[32];
        tmem_ld32(c.tmem + lane_off + st * BN + q * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) s[q * 32 + x] = __uint_as_float(v[x]);
      }
      tc_fence_before();
      mbar_arrive(c.bar(B_S_EMPTY + st, L::OFF_BAR));

      float mx = -INFINITY;
#pragma unroll
      for (int x = 0; x < BN; ++x) {
        const int j = j0 + x;
        const float y = (j >= lo && j <= hi) ? s[x] * p.scale_log2 : -INFINITY;
        s[x] = y;
        mx = fmaxf(mx, y);
      }
      const float m_new = fmaxf(m_used, mx);
      const bool resc = m_new > m_used + kRescaleLog2;
      const float m_tgt = resc ? m_new : m_used;
      const float alpha = resc ? ex2(m_used - m_new) : 1.f;
      const float m_sub = (m_tgt == -INFINITY) ? 0.f : m_tgt;

      if (i > 0) {  // P buffer and O are free once the previous P V finished
        if (!waitw(c.bar(B_O_DONE, L::OFF_BAR), (gi - 1) & 1, c.wc)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t v[32];
            tmem_ld32(t_o + q * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) v[x] = __float_as_uint(__uint_as_float(v[x]) * alpha);
            tmem_st32(t_o + q * 32, v);
          }
          tmem_wait_st();
        }
      }
      l *= alpha;

      float rs = 0.f;
      uint8_t* prow = c.smem + L::OFF_P + r * 128;
#pragma unroll
      for (int q = 0; q < BN / 8; ++q) {
        float e[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          e[x] = ex2(s[q * 8 + x] - m_sub);
          rs += e[x];
        }
        uint4 w;
        w.x = pack_bf16x2(e[0], e[1]);
        w.y = pack_bf16x2(e[2], e[3]);
        w.z = pack_bf16x2(e[4], e[5]);
        w.w = pack_bf16x2(e[6], e[7]);
        const int half = q >> 3, cq = q & 7;
        *reinterpret_cast<uint4*>(prow + half * kAtom + ((cq ^ (r & 7)) << 4)) = w;
      }
      l += rs;

      if (i == 0 || i == nt - 1) {
        // Edge tiles: zero the V rows of keys outside every row's range
        // (stale page heads, unwritten page tails) so P = 0 never meets NaN.
        if (!waitw(c.bar(B_V_FULL + st, L::OFF_BAR), ph, c.wc)) { ok = false; break; }
        const int jr = j0 + r;
        if (jr < U.klo || jr > U.khi) {
          uint8_t* vrow = c.smem + L::OFF_V + st * L::KV_BYTES + r * 128;
#pragma unroll
          for (int cc = 0; cc < NC; ++cc)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(vrow + cc * kAtom + q * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(c.bar(B_P_FULL, L::OFF_BAR));
      m_used = m_tgt;
    }
    if (!ok) break;

    if (!waitw(c.bar(B_O_DONE, L::OFF_BAR), (g + nt - 1) & 1, c.wc)) break;
    tc_fence_after();
    const float inv_l = row_ok ? 1.f / l : 0.f;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) +
                          (static_cast<int64_t>(tok) * p.hq + U.head * p.G + gg) * D;
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
      uint32_t v[32];
      tmem_ld32(t_o + q * 32, v);
      tmem_wait_ld();
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[8 * x + 0]) * inv_l, __uint_as_float(v[8 * x + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(v[8 * x + 2]) * inv_l, __uint_as_float(v[8 * x + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(v[8 * x + 4]) * inv_l, __uint_as_float(v[8 * x + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(v[8 * x + 6]) * inv_l, __uint_as_float(v[8 * x + 7]) * inv_l);
          dst[x] = w;
        }
      }
    }
    if (row_ok && p.lse != nullptr)
      p.lse[static_cast<int64_t>(U.head * p.G + gg) * p.total_q + tok] =
          (m_used + log2f(l)) * 0.69314718055994530942f;
    tc_fence_before();
    mbar_arrive(c.bar(B_O_EMPTY, L::OFF_BAR));
    g += nt;
  }
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  Ctx c;
  c.smem = smem;
  c.sbase = smem_addr(smem);
  if (threadIdx.x == 0) {
    mbar_init(c.bar(B_Q_FULL, L::OFF_BAR), 1);
    mbar_init(c.bar(B_Q_EMPTY, L::OFF_BAR), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(c.bar(B_K_FULL + s, L::OFF_BAR), 1);
      mbar_init(c.bar(B_V_FULL + s, L::OFF_BAR), 1);
      mbar_init(c.bar(B_KV_EMPTY + s, L::OFF_BAR), 1);
      mbar_init(c.bar(B_S_FULL + s, L::OFF_BAR), 1);
      mbar_init(c.bar(B_S_EMPTY + s, L::OFF_BAR), 128);
    }
    mbar_init(c.bar(B_P_FULL, L::OFF_BAR), 128);
    mbar_init(c.bar(B_O_DONE, L::OFF_BAR), 1);
    mbar_init(c.bar(B_O_EMPTY, L::OFF_BAR), 128);
    mbar_init(c.bar(B_NEVER, L::OFF_BAR), 1);
    mbar_init(c.bar(B_DRAIN, L::OFF_BAR), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
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
    if (lane == 0) producer<D>(&tmq, &tmk, &tmv, p, c);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<D>(p, c);
    __syncwarp();
  } else {
    softmax_epilogue<D>(p, c, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(c.tmem, 512);
  }
}

int prefill_smem_bytes(int head_dim) {
  return head_dim == 64 ? static_cast<int>(Layout<64>::BYTES) : static_cast<int>(Layout<128>::BYTES);
}

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, int head_dim, int grid, cudaStream_t s) {
  if (head_dim == 64) {
    const int bytes = Layout<64>::BYTES;
    cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    prefill_kernel<64><<<grid, kThreads, bytes, s>>>(tq, tk, tv, p);
  } else {
    const int bytes = Layout<128>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<128>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    prefill_kernel<128><<<grid, kThreads, bytes, s>>>(tq, tk, tv, p);
  }
  return cudaGetLastError();
}

}  // namespace skv
