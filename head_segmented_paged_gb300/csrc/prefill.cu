// Prefill attention over head-segmented pages on the 5th-generation tensor
// core (RedKnot summary page, section "SegPagedAttention（存储与执行底座）": one
// fused varlen attention kernel over per-(layer, head) paged segments, every
// head on the fast path, no attn_mask). Online softmax with a running maximum
// (KV-cache architecture page, section 5.2).
//
// Work unit: one KV head x two tiles (A, B) of 128 query rows. Rows pack the
// G query heads that share the KV head: row r of a tile = token (r / G) x head
// (r % G), so each K/V tile feeds every head of the group (GQA packing), and
// the two Q tiles share every K/V tile fetched. Keys are visited in tiles of
// 128 positions whose pages TMA fetches through the segment's block table;
// pages outside the segment are read as zeros (out-of-range TMA coordinate)
// and per-row masks keep every row to its own key set: j <= p, and j >= p-W+1
// for a local head.
//
// Warp roles (320 threads, one CTA per SM). The units form one list, in
// descending key tiles; CTA c starts with unit c and then claims the next
// unclaimed unit from a counter in global memory, so a CTA on a slower SM runs
// fewer units (greedy list scheduling with the measured rather than the
// estimated unit times):
//   warp 0      TMA producer: claims the units (one ahead of the one it
//               publishes), then Q tiles A and B, then K and V tiles (2
//               stages), block-table entries fetched 32 at a time by the
//               whole warp;
//   warp 1      TMEM owner and MMA issuer: S_X = Q_X K^T (X = A, B) into TMEM,
//               then O_X += P_X V with P_X read back from TMEM, as one stream
//               across the CTA's units; every MMA is issued from descriptors
//               computed once, because the issuing thread shares its
//               sub-partition with two softmax warps and the tensor pipe
//               drains whenever it is starved of issue slots;
//   warps 2..5  softmax of tile A, warps 6..9 softmax of tile B (one thread
//               per row): read S from TMEM, mask only on edge tiles, update
//               the running max (O is rescaled in TMEM only when the max grows
//               by more than 2^8, which is exact), write P as bf16 over S; a
//               unit's O is normalised and stored after the next unit's first
//               P is written (the first P of a unit is on the tensor pipe's
//               critical path, the output is not). Unit descriptors
//               come from the producer through a shared-memory ring, which
//               the MMA issuer reads too; a descriptor with no key tiles ends
//               the CTA's work.
// TMEM columns: S_A [0,128), S_B [128,256) (P_X aliases the first 64 columns
// of S_X), O_A [256, 256+D), O_B [384, 384+D).
//
// Ordering: the MMA issuer issues S_X of tile j+1 after P_X V of tile j, and
// tcgen05 operations of one thread complete in order, so when the softmax sees
// S_X(j+1) complete, P_X(j) has been consumed and O_X is stable (across a unit
// boundary: the last O_X of the old unit is final).
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "segkv_internal.h"

namespace skv {
using namespace ptx;

namespace {

constexpr int BM = kRowsPerTile;
constexpr int BN = kKeyTile;
constexpr int kThreads = 320;
constexpr float kRescaleLog2 = 8.0f;
// Of every 8 score columns, how many use exp2_poly instead of the MUFU unit.
// GB300's MUFU exp rate keeps up with the D=128 MMAs, so there all use MUFU;
// at D=64 the MMAs per key tile halve and a quarter go to the FMA pipe.
template <int D>
constexpr int kEmuPer8 = D == 64 ? 2 : 0;
constexpr uint32_t kAtom = BM * 128;  // one 64-column, 128-row swizzle block (16 KB)
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;
constexpr uint64_t kDebugWaitNs = 20ull * 1000 * 1000;

enum {
  B_Q_FULL = 0,    // +X
  B_Q_EMPTY = 2,   // +X
  B_K_FULL = 4,    // +stage
  B_V_FULL = 6,    // +stage
  B_KV_EMPTY = 8,  // +stage
  B_S_FULL = 10,   // +X
  B_P_FULL = 12,   // +X
  B_O_FULL = 14,   // +X
  B_O_EMPTY = 16,  // +X
  B_NEVER = 18,
  B_DRAIN = 19,
  B_DESC = 20,     // +slot: the producer has written that slot's unit descriptor
  NUM_BARS = 24
};
// Unit descriptors reach the MMA issuer and the softmax warps through a ring
// of kDescSlots shared-memory slots written by the producer; a slot is
// rewritten four units later. The producer publishes unit u+4 only after it
// has loaded unit u+3's Q tiles, which waits for the last S MMAs of unit
// u+2. The issuer issues those after it has read unit u+2's descriptor and
// after P of a tile of unit u+1 or u+2, so every reader is past unit u.
constexpr int kDescSlots = 4;

template <int D>
struct Layout {
  static constexpr uint32_t Q_BYTES = BM * D * 2;  // one Q tile
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr uint32_t OFF_Q = 0;              // tiles A, B
  static constexpr uint32_t OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + 2 * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + 2 * KV_BYTES;
  static constexpr uint32_t OFF_DESC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t OFF_MISC = OFF_DESC + kDescSlots * sizeof(PrefillUnit);
  // O staging for the bulk tensor stores: 32 rows x 64 columns per softmax warp
  static constexpr uint32_t OFF_STAGE = (OFF_MISC + 16 + 1023) / 1024 * 1024;
  static constexpr uint32_t STAGE_WARP = 32 * 128;
  // + slack to align to 1 KB; at least 116 KB so that one CTA holds an SM (and
  // its 512 TMEM columns) alone
  static constexpr uint32_t RAW = OFF_STAGE + 8 * STAGE_WARP + 1024;
  static constexpr uint32_t BYTES = RAW > 116u * 1024 ? RAW : 116u * 1024;
  static constexpr uint32_t TM_O = 256;             // TMEM column of O_A
  static constexpr uint32_t TM_O_STRIDE = 128;      // O_B = O_A + this
};

struct Ctx {
  uint8_t* smem;
  uint32_t sbase;
  uint32_t tmem;
  uint32_t off_bar;
  WaitCtx wc;
  __device__ uint32_t bar(int i) const { return sbase + off_bar + 8u * i; }
};

// ---------------------------------------------------------------- producer
// Run by the whole warp: lanes fetch 32 block-table entries at a time (one
// coalesced load instead of a dependent load per key tile); lane 0 issues the
// TMA copies.
template <int D>
__device__ void producer(const CUtensorMap* tmq, const CUtensorMap* tmk, const CUtensorMap* tmv,
                         const PrefillParams& p, const Ctx& c, int lane) {
  using L = Layout<D>;
  constexpr int NC = D / 64;
  const int box_rows = p.page_size <= BN ? p.page_size : BN;
  const int boxes = BN / box_rows;
  int armed_q[2] = {-1, -1}, armed_kv[2] = {-1, -1};
  bool ok = true;
  int g = 0, ui = 0;
  // CTA c starts with unit c. Lane 0 claims every later unit one unit ahead
  // of its use, so the atomic's round trip hides behind a unit's loads.
  const int n = p.n_units;
  int u = static_cast<int>(blockIdx.x), claim = 0;
  if (lane == 0 && u < n) claim = atomicAdd(p.next_unit, 1);
  PrefillUnit U{};
  if (u < n) U = p.units[u];
  for (; ok && u < n; ++ui) {
    const int un = __shfl_sync(0xffffffffu, claim, 0) + static_cast<int>(gridDim.x);
    const bool has_next = un < n;
    PrefillUnit Un{};
    if (has_next) Un = p.units[un];
    if (lane == 0 && has_next) claim = atomicAdd(p.next_unit, 1);
    if (lane == 0) {  // publish the descriptor (arrive = release)
      reinterpret_cast<PrefillUnit*>(c.smem + L::OFF_DESC)[ui % kDescSlots] = U;
      mbar_arrive(c.bar(B_DESC + ui % kDescSlots));
    }
    for (int x = 0; x < 2; ++x) {
      if (!waitw(c.bar(B_Q_EMPTY + x), (ui & 1) ^ 1, c.wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(c.bar(B_Q_FULL + x), L::Q_BYTES);
        for (int cc = 0; cc < NC; ++cc)
          tma_load_3d(c.sbase + L::OFF_Q + x * L::Q_BYTES + cc * kAtom, tmq, cc * 64,
                      U.head * p.G, U.tok0 + x * p.tpt, c.bar(B_Q_FULL + x));
      }
      armed_q[x] = ui & 1;
    }
    if (!ok) break;
    const int32_t* trow = p.table + static_cast<int64_t>(U.table_row) * p.R;
    const int first_page = U.vlo / p.page_size, last_page = U.vhi / p.page_size;
    int kbase = -(1 << 30), my_id = 0;
    for (int kt = U.kt0; kt <= U.kt1; ++kt, ++g) {
      const int st = g & 1;
      const uint32_t ph = (g >> 1) & 1;
      if (!waitw(c.bar(B_KV_EMPTY + st), ph ^ 1, c.wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(c.bar(B_K_FULL + st), L::KV_BYTES);
        mbar_expect_tx(c.bar(B_V_FULL + st), L::KV_BYTES);
      }
      armed_kv[st] = static_cast<int>(ph);
      int yv = 0;  // lane bi keeps box bi's row
      for (int bi = 0; bi < boxes; ++bi) {
        const int pos = kt * BN + bi * box_rows;
        const int k = pos / p.page_size;
        int y = p.oob_row;  // zero fill: page not held by this segment
        if (k >= first_page && k <= last_page) {
          if (k >= kbase + 32) {
            kbase = k;
            my_id = (k + lane < p.R) ? trow[k + lane] : 0;
          }
          y = __shfl_sync(0xffffffffu, my_id, k - kbase) * p.page_size + (pos - k * p.page_size);
        }
        if (lane == bi) yv = y;
        if (lane == 0) {
          const uint32_t off = st * L::KV_BYTES + bi * box_rows * 128;
          for (int cc = 0; cc < NC; ++cc)
            tma_load_2d(c.sbase + L::OFF_K + off + cc * kAtom, tmk, cc * 64, y, c.bar(B_K_FULL + st));
        }
      }
      // V boxes after every K box: the tile's S MMAs wait for K only, and V
      // is needed half a key tile later
      for (int bi = 0; bi < boxes; ++bi) {
        const int y = __shfl_sync(0xffffffffu, yv, bi);
        if (lane == 0) {
          const uint32_t off = st * L::KV_BYTES + bi * box_rows * 128;
          for (int cc = 0; cc < NC; ++cc)
            tma_load_2d(c.sbase + L::OFF_V + off + cc * kAtom, tmv, cc * 64, y, c.bar(B_V_FULL + st));
        }
      }
    }
    U = Un;
    u = un;
  }
  if (ok && lane == 0) {  // no unit left: a descriptor with no key tiles ends the readers' loops
    PrefillUnit E{};
    E.kt1 = -1;
    reinterpret_cast<PrefillUnit*>(c.smem + L::OFF_DESC)[ui % kDescSlots] = E;
    mbar_arrive(c.bar(B_DESC + ui % kDescSlots));
  }
  if (!ok && lane == 0) {  // aborting: let our own copies land before the block exits
    for (int x = 0; x < 2; ++x)
      if (armed_q[x] >= 0) wait_drain(c.bar(B_Q_FULL + x), armed_q[x], kDrainNs);
    for (int st = 0; st < 2; ++st)
      if (armed_kv[st] >= 0) {
        wait_drain(c.bar(B_K_FULL + st), armed_kv[st], kDrainNs);
        wait_drain(c.bar(B_V_FULL + st), armed_kv[st], kDrainNs);
      }
  }
}

// ---------------------------------------------------------------- MMA issuer
// The issuing thread shares its sub-partition with a softmax warp, so each
// MMA is issued from precomputed descriptors: the descriptors of the six
// shared-memory operands (Q tiles A and B, K and V of both stages) are built
// once, and an MMA's own descriptor adds its compile-time offset (in 16-byte
// units, which never carries out of the 14-bit address field) to the low
// word.
struct MmaDescs {
  uint64_t q[2], k[2], v[2];
};

__device__ __forceinline__ uint64_t desc_add(uint64_t base, uint32_t off16) {
  return base + off16;  // the address field is the low 14 bits; no carry out
}

template <int D>
__device__ __forceinline__ MmaDescs mma_descs(const Ctx& c) {
  using L = Layout<D>;
  MmaDescs m;
  for (int i = 0; i < 2; ++i) {
    m.q[i] = sdesc_sw128(c.sbase + L::OFF_Q + i * L::Q_BYTES, 16, 1024);
    m.k[i] = sdesc_sw128(c.sbase + L::OFF_K + i * L::KV_BYTES, 16, 1024);
    m.v[i] = sdesc_sw128(c.sbase + L::OFF_V + i * L::KV_BYTES, kAtom, 1024);
  }
  return m;
}

template <int D>
__device__ __forceinline__ void issue_s(const Ctx& c, const MmaDescs& m, int x, int st) {
  constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, 0);
  const uint64_t qa = x ? m.q[1] : m.q[0], kb = st ? m.k[1] : m.k[0];
  const uint32_t d = c.tmem + x * BN;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off16 = ((kk >> 2) * kAtom + (kk & 3) * 32) >> 4;
    mma_bf16(d, desc_add(qa, off16), desc_add(kb, off16), IDESC_QK, kk > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void issue_pv(const Ctx& c, const MmaDescs& m, int x, int st,
                                         bool first) {
  using L = Layout<D>;
  constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, 1);
  const uint64_t vb = st ? m.v[1] : m.v[0];
  const uint32_t d = c.tmem + L::TM_O + x * L::TM_O_STRIDE, a = c.tmem + x * BN;
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk)
    mma_bf16_ts(d, a + kk * 8, desc_add(vb, kk * 2048 / 16), IDESC_PV,
                (first && kk == 0) ? 0u : 1u);
}

template <int D>
__device__ void mma_issuer(const PrefillParams& p, const Ctx& c) {
  const MmaDescs md = mma_descs<D>(c);
  bool ok = true;
  if (p.debug & 1) {  // test hook: one wait on a barrier nothing signals
    WaitCtx w = c.wc;
    w.limit_ns = kDebugWaitNs;
    wait1(c.bar(B_NEVER), 0, w);
    ok = false;
  }
  // The MMAs run as one stream across the CTA's units: S_A and S_B of the
  // next unit's first key tile follow this unit's last P V MMAs directly
  // (S_A already between P_A V and P_B V when its operands are there).
  // A unit's key-tile count comes from the producer's descriptor ring, where
  // the producer has published it a key tile or more before it is needed;
  // zero tiles means no unit is left.
  const PrefillUnit* ring = reinterpret_cast<const PrefillUnit*>(c.smem + Layout<D>::OFF_DESC);
  auto tiles_of = [&](int ui, int* nt) {
    if (!wait1(c.bar(B_DESC + ui % kDescSlots), (ui / kDescSlots) & 1, c.wc)) return false;
    const PrefillUnit& d = ring[ui % kDescSlots];
    *nt = max(0, d.kt1 - d.kt0 + 1);
    return true;
  };
  int g = 0, nt_next = 0;
  if (ok && !tiles_of(0, &nt_next)) ok = false;
  // S_A and S_B of the first unit's first key tile
  if (ok && nt_next > 0) {
    if (!wait1(c.bar(B_K_FULL + 0), 0, c.wc)) ok = false;
    for (int x = 0; ok && x < 2; ++x) {
      if (!wait1(c.bar(B_Q_FULL + x), 0, c.wc)) { ok = false; break; }
      tc_fence_after();
      issue_s<D>(c, md, x, 0);
      mma_commit(c.bar(B_S_FULL + x));
      if (nt_next == 1) mma_commit(c.bar(B_Q_EMPTY + x));
    }
  }
  for (int ui = 0; ok && nt_next > 0; ++ui) {
    const int nt = nt_next;
    const uint32_t qpar = ui & 1;
    bool early_a = false;
    for (int i = 0; i < nt && ok; ++i) {
      const int gi = g + i, st = gi & 1, gn = gi + 1;
      const uint32_t ph = (gi >> 1) & 1;
      const bool last = (i + 1 == nt);
      for (int x = 0; x < 2; ++x) {
        if (i == 0 && !wait1(c.bar(B_O_EMPTY + x), qpar ^ 1, c.wc)) { ok = false; break; }
        if (!wait1(c.bar(B_P_FULL + x), gi & 1, c.wc)) { ok = false; break; }
        if (x == 0 && !wait1(c.bar(B_V_FULL + st), ph, c.wc)) { ok = false; break; }
        tc_fence_after();
        issue_pv<D>(c, md, x, st, i == 0);
        if (x == 1) mma_commit(c.bar(B_KV_EMPTY + st));
        if (last) {
          mma_commit(c.bar(B_O_FULL + x));
          // The next unit's S_A right behind this unit's last P_A V, if its
          // descriptor, K tile and Q_A tile are already there (tested, not
          // waited for: a wait here would hold up P_B V): tile A's first
          // softmax of the next unit then runs while the pipe does P_B V
          // and S_B, instead of both tiles' first softmax running with the
          // pipe idle.
          if (x == 0) {
            const int un = ui + 1, gn2 = g + nt;
            if (mbar_peek(c.bar(B_DESC + un % kDescSlots), (un / kDescSlots) & 1)) {
              const PrefillUnit& d = ring[un % kDescSlots];
              const int ntn = d.kt1 - d.kt0 + 1;
              if (ntn > 0 && mbar_peek(c.bar(B_K_FULL + (gn2 & 1)), (gn2 >> 1) & 1) &&
                  mbar_peek(c.bar(B_Q_FULL + 0), qpar ^ 1)) {
                tc_fence_after();
                issue_s<D>(c, md, 0, gn2 & 1);
                mma_commit(c.bar(B_S_FULL + 0));
                if (ntn == 1) mma_commit(c.bar(B_Q_EMPTY + 0));
                early_a = true;
              }
            }
          }
          continue;
        }
        if (x == 0 && !wait1(c.bar(B_K_FULL + (gn & 1)), (gn >> 1) & 1, c.wc)) { ok = false; break; }
        tc_fence_after();
        issue_s<D>(c, md, x, gn & 1);
        mma_commit(c.bar(B_S_FULL + x));
        if (i + 2 == nt) mma_commit(c.bar(B_Q_EMPTY + x));  // the unit's last S MMAs
      }
    }
    // S_A and S_B of the next unit's first key tile, issued behind this
    // unit's last P V MMAs
    if (ok && !tiles_of(ui + 1, &nt_next)) ok = false;
    if (ok && nt_next > 0) {
      const int gn = g + nt;
      if (!wait1(c.bar(B_K_FULL + (gn & 1)), (gn >> 1) & 1, c.wc)) { ok = false; break; }
      for (int x = 0; x < 2; ++x) {
        if (x == 0 && early_a) continue;
        if (!wait1(c.bar(B_Q_FULL + x), qpar ^ 1, c.wc)) { ok = false; break; }
        tc_fence_after();
        issue_s<D>(c, md, x, gn & 1);
        mma_commit(c.bar(B_S_FULL + x));
        if (nt_next == 1) mma_commit(c.bar(B_Q_EMPTY + x));
      }
    }
    g += nt;
  }
  if (!ok) {  // aborting: let issued MMAs finish before TMEM is freed
    mma_commit(c.bar(B_DRAIN));
    wait_drain(c.bar(B_DRAIN), 0, kDrainNs);
  }
}

// ---------------------------------------------------------------- softmax
// What the output of a finished unit needs, kept in registers while the warp
// runs the next unit's first softmax tile.
struct Pending {
  int ui;        // the unit's index in this CTA (O_FULL parity)
  int head, tok0, ntok;
  int tok;       // this row's token (valid when row_ok)
  bool row_ok;
  float inv_l;   // 1 / O's normaliser (0 for an invalid row)
  float lse;     // natural-log LSE of the row
};

// O / l of a finished unit as bf16: read O_X from TMEM (after its last P V),
// free O_X for the next unit's P V, then store the rows and the LSE.
template <int D>
__device__ __forceinline__ bool write_output(const CUtensorMap* tmo, const PrefillParams& p, const Ctx& c,
                                             int x, int wq, int lane, uint32_t t_o, const Pending& e) {
  using L = Layout<D>;
  constexpr int NC = D / 64;
  if (!waitw(c.bar(B_O_FULL + x), e.ui & 1, c.wc)) return false;
  tc_fence_after();
  if (lane == 0) bulk_wait_read();  // the last unit's stores have read the staging rows
  uint32_t ob[D / 2];
#pragma unroll
  for (int q = 0; q < D / 32; ++q) {
    uint32_t v[32];
    tmem_ld32(t_o + q * 32, v);
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < 16; ++k)
      ob[q * 16 + k] = pack_bf16x2(__uint_as_float(v[2 * k]) * e.inv_l, __uint_as_float(v[2 * k + 1]) * e.inv_l);
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(c.bar(B_O_EMPTY + x));
  const int gg = (wq * 32 + lane) % p.G;
  if (e.ntok >= x * p.tpt + (wq + 1) * 32 / p.G) {
    // The warp's 32 rows are 32 / G whole tokens: they go to the warp's
    // 128B-swizzled staging rows, 64 columns at a time, and lane 0 writes
    // them with one bulk tensor store each (the rows are one box of the O
    // tensor map). Per-thread row stores would touch 32 rows per
    // instruction and hold this SM's shared-memory and barrier operations
    // up behind them.
    uint8_t* stg = c.smem + L::OFF_STAGE + (x * 4 + wq) * L::STAGE_WARP;
#pragma unroll
    for (int cc = 0; cc < NC; ++cc) {
      if (cc > 0) {  // the previous store has read the staging rows
        if (lane == 0) bulk_wait_read();
        __syncwarp();
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
            make_uint4(ob[cc * 32 + 4 * j], ob[cc * 32 + 4 * j + 1], ob[cc * 32 + 4 * j + 2],
                       ob[cc * 32 + 4 * j + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(tmo, smem_addr(stg), cc * 64, e.head * p.G, e.tok0 + x * p.tpt + wq * 32 / p.G);
        bulk_commit();
      }
    }
  } else if (e.row_ok) {  // rows of a sequence's last, partial tile: row stores
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) +
                                          (static_cast<int64_t>(e.tok) * p.hq + e.head * p.G + gg) * D);
#pragma unroll
    for (int k = 0; k < D / 8; ++k)
      dst[k] = make_uint4(ob[4 * k], ob[4 * k + 1], ob[4 * k + 2], ob[4 * k + 3]);
  }
  if (e.row_ok && p.lse != nullptr)
    p.lse[static_cast<int64_t>(e.head * p.G + gg) * p.total_q + e.tok] = e.lse;
  return true;
}

template <int D>
__device__ void softmax_epilogue(const CUtensorMap* tmo, const PrefillParams& p, const Ctx& c, int x,
                                 int warp, int lane) {
  using L = Layout<D>;
  constexpr int NC = D / 64;
  const int wq = warp & 3;  // TMEM lane quarter this warp may access
  const int r = wq * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t t_s = c.tmem + lane_off + x * BN;
  const uint32_t t_o = c.tmem + lane_off + L::TM_O + x * L::TM_O_STRIDE;
  const float scale = p.scale_log2;
  int g = 0;
  Pending pend{};
  bool have = false;  // pend holds a finished unit whose output is not written yet
  for (int ui = 0;; ++ui) {
    // the unit's descriptor, from the producer's ring (no key tiles: no unit
    // is left); consecutive query positions come with it (pos0), so no
    // per-row load of q_pos is needed
    if (!waitw(c.bar(B_DESC + ui % kDescSlots), (ui / kDescSlots) & 1, c.wc)) break;
    const PrefillUnit U = reinterpret_cast<const PrefillUnit*>(c.smem + L::OFF_DESC)[ui % kDescSlots];
    const int nt = U.kt1 - U.kt0 + 1;
    if (nt <= 0) break;
    const int t = x * p.tpt + r / p.G;
    const bool row_ok = t < U.ntok;
    const int tok = U.tok0 + t;
    int hi = -1, lo = 1 << 30;  // an invalid row sees no key
    if (row_ok) {
      hi = U.pos0 >= 0 ? U.pos0 + t : p.q_pos[tok];
      lo = U.local ? max(0, hi - p.window + 1) : 0;
    }
    float m_used = -INFINITY, l = 0.f, lc = 0.f;
    bool ok = true;
    for (int i = 0; i < nt; ++i) {
      const int gi = g + i, st = gi & 1;
      const uint32_t ph = (gi >> 1) & 1;
      const int j0 = (U.kt0 + i) * BN;
      if (!waitw(c.bar(B_S_FULL + x), gi & 1, c.wc)) { ok = false; break; }
      tc_fence_after();
      float s[BN];
      tmem_ld32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
      tmem_ld32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
      tmem_wait_ld();
      // mask only where some row of this warp does not see the whole tile;
      // where every row of the warp sees one end of it (the diagonal tile of
      // a causal row, the first tile of a window), test only the other bound
      const bool whole = (j0 >= lo) && (j0 + BN - 1 <= hi);
      if (!__all_sync(0xffffffffu, whole)) {
        const int c_lo = lo - j0, c_hi = hi - j0;
        if (__all_sync(0xffffffffu, c_lo <= 0)) {
#pragma unroll
          for (int e = 0; e < BN; ++e) s[e] = e <= c_hi ? s[e] : -INFINITY;
        } else if (__all_sync(0xffffffffu, c_hi >= BN - 1)) {
#pragma unroll
          for (int e = 0; e < BN; ++e) s[e] = e >= c_lo ? s[e] : -INFINITY;
        } else {
#pragma unroll
          for (int e = 0; e < BN; ++e) s[e] = (e >= c_lo && e <= c_hi) ? s[e] : -INFINITY;
        }
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < BN; e += 8) {
        m4[0] = max3(m4[0], s[e + 0], s[e + 1]);
        m4[1] = max3(m4[1], s[e + 2], s[e + 3]);
        m4[2] = max3(m4[2], s[e + 4], s[e + 5]);
        m4[3] = max3(m4[3], s[e + 6], s[e + 7]);
      }
      const float smax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      const float mx = smax * scale;
      const float m_new = fmaxf(m_used, mx);
      const bool resc = m_new > m_used + kRescaleLog2;
      const float m_tgt = resc ? m_new : m_used;
      const float alpha = resc ? ex2(m_used - m_new) : 1.f;
      const float neg_m = (m_tgt == -INFINITY) ? 0.f : -m_tgt;

      l *= alpha;
      lc *= alpha;

      // p = 2^(s * scale - m), two columns per packed FMA/add
      const float2 sc2 = make_float2(scale, scale), nm2 = make_float2(neg_m, neg_m);
      float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int q = 0; q < BN / 32; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = q * 32 + 2 * e;
          const float2 xx = __ffma2_rn(make_float2(s[col], s[col + 1]), sc2, nm2);
          const float p0 = ((col & 7) >= 8 - kEmuPer8<D>) ? exp2_poly(xx.x) : ex2(xx.x);
          const float p1 = (((col + 1) & 7) >= 8 - kEmuPer8<D>) ? exp2_poly(xx.y) : ex2(xx.y);
          rs[e & 1] = __fadd2_rn(rs[e & 1], make_float2(p0, p1));
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(t_s + q * 16, pk);
      }
      l += (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y);
      {
        // P is rounded to bf16 for the P V MMA while l sums the fp32 values.
        // Where attention concentrates on a few keys, the rounding of the
        // largest P dominates the error of O, so O's normaliser also adds the
        // rounding error of each tile's largest P (same FMA and ex2 as its
        // column above); the LSE keeps the exact sum.
        const float pm = ex2(fmaf(smax, scale, neg_m));
        lc += __bfloat162float(__float2bfloat16_rn(pm)) - pm;
      }

      if (i > 0 && __any_sync(0xffffffffu, resc)) {  // O_X is stable: P V of tile i-1 is done
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t v[32];
          tmem_ld32(t_o + q * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st32(t_o + q * 32, v);
        }
      }

      if (x == 0 && (i == 0 || i == nt - 1) && (j0 < U.vlo || j0 + BN - 1 > U.vhi)) {
        // An edge tile that reaches past the segment's written keys: zero
        // those V rows (a stale page head, an unwritten page tail) so that
        // P = 0 never meets NaN. Keys of the segment that a row does not see
        // hold finite values and meet P = 0 as they are.
        if (!waitw(c.bar(B_V_FULL + st), ph, c.wc)) { ok = false; break; }
        const int jr = j0 + r;
        if (jr < U.vlo || jr > U.vhi) {
          uint8_t* vrow = c.smem + L::OFF_V + st * L::KV_BYTES + r * 128;
#pragma unroll
          for (int cc = 0; cc < NC; ++cc)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              // chunk q ^ (r % 8): the warp's 32 rows spread over all banks
              *reinterpret_cast<uint4*>(vrow + cc * kAtom + ((q ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();  // one arrival per warp: the barrier is on the softmax -> P V path
      if (lane == 0) mbar_arrive(c.bar(B_P_FULL + x));
      m_used = m_tgt;
      // The previous unit's output, now that this unit's first P is in TMEM:
      // its S MMAs were issued after that unit's last P V, so the wait for
      // O_FULL returns at once, and the next P V waits for O_EMPTY.
      if (i == 0 && have) {
        if (!write_output<D>(tmo, p, c, x, wq, lane, t_o, pend)) { ok = false; break; }
        have = false;
      }
    }
    if (!ok) break;
    pend.ui = ui;
    pend.head = U.head;
    pend.tok0 = U.tok0;
    pend.ntok = U.ntok;
    pend.tok = tok;
    pend.row_ok = row_ok;
    pend.inv_l = row_ok ? 1.f / (l + lc) : 0.f;
    pend.lse = (m_used + log2f(l)) * 0.69314718055994530942f;
    have = true;
    g += nt;
  }
  if (have) write_output<D>(tmo, p, c, x, wq, lane, t_o, pend);
  if (lane == 0) bulk_wait();  // this warp's bulk stores are complete
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                   const PrefillParams p) {
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
  c.off_bar = L::OFF_BAR;
  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(c.bar(B_Q_FULL + x), 1);
      mbar_init(c.bar(B_Q_EMPTY + x), 1);
      mbar_init(c.bar(B_S_FULL + x), 1);
      mbar_init(c.bar(B_P_FULL + x), 4);  // one arrival per softmax warp
      mbar_init(c.bar(B_O_FULL + x), 1);
      mbar_init(c.bar(B_O_EMPTY + x), 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(c.bar(B_K_FULL + s), 1);
      mbar_init(c.bar(B_V_FULL + s), 1);
      mbar_init(c.bar(B_KV_EMPTY + s), 1);
    }
    mbar_init(c.bar(B_NEVER), 1);
    mbar_init(c.bar(B_DRAIN), 1);
    for (int d = 0; d < kDescSlots; ++d) mbar_init(c.bar(B_DESC + d), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
    prefetch_tmap(&tmo);
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
    producer<D>(&tmq, &tmk, &tmv, p, c, lane);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<D>(p, c);
    __syncwarp();
  } else {
    softmax_epilogue<D>(&tmo, p, c, (warp - 2) >> 2, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(c.tmem, 512);
  }
}

// The two base-2 exponentials of the softmax, elementwise over an array, so
// that they can be checked against 2^x outside any attention call.
__global__ void exp2_check_kernel(const float* x, float* y_poly, float* y_mufu, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    y_poly[i] = exp2_poly(x[i]);
    y_mufu[i] = ex2(x[i]);
  }
}

cudaError_t launch_exp2_check(const float* x, float* y_poly, float* y_mufu, int n, cudaStream_t s) {
  exp2_check_kernel<<<(n + 255) / 256, 256, 0, s>>>(x, y_poly, y_mufu, n);
  return cudaGetLastError();
}

int prefill_smem_bytes(int head_dim) {
  return head_dim == 64 ? static_cast<int>(Layout<64>::BYTES) : static_cast<int>(Layout<128>::BYTES);
}

int prefill_unit_tokens(int G) { return 2 * (kRowsPerTile / G); }

template <class K>
cudaError_t launch_kernel(K kernel, int smem, int grid, cudaStream_t s, const CUtensorMap& tq,
                          const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                          const PrefillParams& p) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, smem, s>>>(tq, tk, tv, to, p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to, int head_dim, int grid,
                           cudaStream_t s) {
  if (head_dim == 64)
    return launch_kernel(prefill_kernel<64>, Layout<64>::BYTES, grid, s, tq, tk, tv, to, p);
  return launch_kernel(prefill_kernel<128>, Layout<128>::BYTES, grid, s, tq, tk, tv, to, p);
}

}  // namespace skv
