// Decode attention on the 5th-generation tensor core for 8 or 16 query rows
// per KV head: several query tokens per sequence (T tokens x Gm heads, as in
// speculative or chunked decoding) or wide GQA groups (RedKnot summary page,
// section "SegPagedAttention（存储与执行底座）": attention over the per-head
// segments; online softmax merge from the KV-cache architecture page, section
// 5.2). On the CUDA cores these rows make decode FMA-bound; here both
// contractions run on tcgen05 and the kernel stays bound by the K/V stream.
//
// Keys go to the TMEM lanes. Per stage of 128 keys the tensor core forms
// S^T = K Q^T (M = 128 keys, N = 16 rows, K = D = 128). Each softmax thread
// owns one key; a row's maximum over the stage comes from a warp redux and an
// exchange among the four softmax warps. P^T (16 rows x 128 keys, bf16) is
// written to shared memory in the 128-byte swizzled layout and the tensor core
// accumulates O^T += V^T P^T (M = 128 dimensions, N = 16 rows, K = 128 keys)
// in TMEM, with V read as an MN-major operand straight from its TMA tile. O is
// rescaled only when a row's maximum grows by more than 2^8, which is exact.
//
// Work comes from the split-KV decode's stream-K plan. A unit whose (sequence,
// KV head) pair lies in one unit writes O directly; otherwise it writes fp32
// partials and decode_combine_kernel merges each split pair afterwards, one
// CTA per (pair, row), with the running-maximum rule.
//
// Warp roles (320 threads, one CTA per SM):
//   warp 0      producer: the unit's query rows (TMA), then K and V tiles of
//               128 keys, page by page through the block table (3 stages);
//   warp 1      TMEM owner (64 columns: two S^T buffers and O^T) and MMA
//               issuer;
//   warps 2..5, 6..9  two softmax groups working on every stage together,
//               each on its own query rows (rows 0..7 and 8..15; with 8 rows
//               group 0 takes them all), with their own running maxima and row
//               sums; thread t holds key t of a stage and dimension t of O^T.
//               At the end of a unit each group writes its own rows.
// Ordering: S and P have two buffers by stage parity; O^T is one accumulator.
// S of stage i+1 is issued before P V of stage i, so the tensor core forms it
// while the groups work on stage i. A thread's tcgen05 operations complete in
// order: when S(i) is complete, P V(i-2) is too, so P buffer i % 2 is free. A
// group that must rescale O^T at stage i first waits for P V(i-1).
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "segkv_internal.h"

namespace skv {
using namespace ptx;

namespace {

constexpr int KT = 128;  // keys per stage
constexpr int NST = 3;   // K/V stages
constexpr int MN = 16;   // MMA N: query rows (8 or 16 used)
constexpr int kThreadsMD = 320;
constexpr uint32_t kAtomKV = KT * 128;     // 64 dims x 128 keys: 16 KB
constexpr uint32_t KV_TILE = 2 * kAtomKV;  // D = 128
constexpr uint32_t kAtomR = MN * 128;      // 64 columns x 16 rows: 2 KB
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_V = NST * KV_TILE;
constexpr uint32_t OFF_Q = 2 * NST * KV_TILE;          // Q [2 buffers, by unit parity]: 2 atoms (dims 0..63, 64..127)
constexpr uint32_t OFF_P = OFF_Q + 4 * kAtomR;         // P^T [2 buffers]: 2 atoms (keys 0..63, 64..127)
constexpr uint32_t OFF_XCH = OFF_P + 4 * kAtomR;          // int [group][2][4][16]: per-warp row maxima
constexpr uint32_t OFF_LS = OFF_XCH + 2 * 2 * 4 * MN * 4;  // float [group][2][4][16]: per-warp row sums
constexpr uint32_t OFF_BAR = OFF_LS + 2 * 2 * 4 * MN * 4;
enum {
  Y_Q_FULL = 0,                 // +Q buffer (unit parity)
  Y_Q_EMPTY = 2,                // +Q buffer
  Y_K_FULL = 4,                 // +stage
  Y_V_FULL = 4 + NST,           // +stage
  Y_KV_EMPTY = 4 + 2 * NST,     // +stage
  Y_S_FULL = 4 + 3 * NST,       // +stage parity: S buffer
  Y_P_FULL = Y_S_FULL + 2,      // +stage parity: P buffer
  Y_O_FULL = Y_S_FULL + 4,
  Y_O_EMPTY = Y_S_FULL + 5,
  Y_MX = Y_S_FULL + 6,          // +group * 2 + stage parity
  Y_LS = Y_S_FULL + 10,         // +group * 2 + unit parity
  Y_PV_DONE = Y_S_FULL + 14,    // the last P V issued is complete
  Y_DRAIN = Y_S_FULL + 16,
  Y_NUM = Y_S_FULL + 17
};
constexpr uint32_t OFF_MISC = OFF_BAR + Y_NUM * 8;
constexpr uint32_t MD_BYTES = OFF_MISC + 16 + 1024;  // + slack to align to 1 KB
constexpr uint32_t TM_S = 0, TM_O = 32, TM_COLS = 64;  // S^T at 0 and 16 (by stage parity), O^T at 32
constexpr int RG = 8;  // query rows per softmax group (TMEM columns 8 * group ..)
constexpr uint64_t kDrainNsMD = 200ull * 1000 * 1000;
static_assert(MD_BYTES <= 227 * 1024, "decode_mma shared memory");

struct MdCtx {
  uint8_t* smem;
  uint32_t sbase;
  uint32_t tmem;
  WaitCtx wc;
  __device__ uint32_t bar(int i) const { return sbase + OFF_BAR + 8u * i; }
};

// 16 rows: each softmax group takes 8; 8 rows: group 0 takes them all
__device__ __forceinline__ int n_groups(const DecodeMmaParams& p) { return p.R_rows > RG ? 2 : 1; }

template <typename T>
__device__ __forceinline__ const T* plan_ptr(const T* p, const PlanBlob& blob, int inl) {
  return inl ? reinterpret_cast<const T*>(blob.data + reinterpret_cast<uintptr_t>(p)) : p;
}

__device__ void md_producer(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                            const DecodeMmaParams& p, const DecodeUnit* units,
                            const int32_t* cta_begin, const MdCtx& c, int lane) {
  const int box_rows = p.page_size <= KT ? p.page_size : KT;
  const int boxes = KT / box_rows;
  int armed_q[2] = {-1, -1}, armed_kv[NST];
  for (int s = 0; s < NST; ++s) armed_kv[s] = -1;
  bool ok = true;
  int g = 0, ui = 0;
  for (int u = cta_begin[blockIdx.x]; ok && u < cta_begin[blockIdx.x + 1]; ++u, ++ui) {
    const DecodeUnit U = units[u];
    // the unit's query rows: token t of the sequence, heads head*Gm .. +Gm-1 -> row t*Gm + j.
    // Two buffers by unit parity, so they load while the previous unit runs.
    const int qb = ui & 1;
    const uint32_t qph = (ui >> 1) & 1;
    if (!waitw(c.bar(Y_Q_EMPTY + qb), qph ^ 1, c.wc)) { ok = false; break; }
    if (lane == 0) {
      mbar_expect_tx(c.bar(Y_Q_FULL + qb), 2u * p.R_rows * 128);
      for (int cc = 0; cc < 2; ++cc)
        tma_load_3d(c.sbase + OFF_Q + (qb * 2 + cc) * kAtomR, tq, cc * 64, U.head * p.Gm,
                    U.req * p.T, c.bar(Y_Q_FULL + qb));
    }
    armed_q[qb] = static_cast<int>(qph);
    const int32_t* trow = p.table + static_cast<int64_t>(U.table_row) * p.R;
    const int kfirst = U.k0 / p.page_size, klast = (U.k1 - 1) / p.page_size;
    int kbase = -(1 << 30), my_id = 0;
    for (int kt = U.k0 / KT; kt <= (U.k1 - 1) / KT; ++kt, ++g) {
      const int st = g % NST;
      const uint32_t ph = (g / NST) & 1;
      if (!waitw(c.bar(Y_KV_EMPTY + st), ph ^ 1, c.wc)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(c.bar(Y_K_FULL + st), KV_TILE);
        mbar_expect_tx(c.bar(Y_V_FULL + st), KV_TILE);
      }
      armed_kv[st] = static_cast<int>(ph);
      for (int bi = 0; bi < boxes; ++bi) {
        const int pos = kt * KT + bi * box_rows;
        const int k = pos / p.page_size;
        int y = p.oob_row;  // a page the unit does not use: zero fill
        if (k >= kfirst && k <= klast) {
          if (k >= kbase + 32) {
            kbase = k;
            my_id = (k + lane < p.R) ? trow[k + lane] : 0;
          }
          y = __shfl_sync(0xffffffffu, my_id, k - kbase) * p.page_size + (pos - k * p.page_size);
        }
        if (lane == 0) {
          const uint32_t off = st * KV_TILE + bi * box_rows * 128;
          for (int cc = 0; cc < 2; ++cc) {
            tma_load_2d(c.sbase + OFF_K + off + cc * kAtomKV, tk, cc * 64, y, c.bar(Y_K_FULL + st));
            tma_load_2d(c.sbase + OFF_V + off + cc * kAtomKV, tv, cc * 64, y, c.bar(Y_V_FULL + st));
          }
        }
      }
    }
  }
  if (!ok && lane == 0) {  // aborting: let our own copies land before the block exits
    for (int b = 0; b < 2; ++b)
      if (armed_q[b] >= 0) wait_drain(c.bar(Y_Q_FULL + b), armed_q[b], kDrainNsMD);
    for (int s = 0; s < NST; ++s)
      if (armed_kv[s] >= 0) {
        wait_drain(c.bar(Y_K_FULL + s), armed_kv[s], kDrainNsMD);
        wait_drain(c.bar(Y_V_FULL + s), armed_kv[s], kDrainNsMD);
      }
  }
}

__device__ void md_mma(const DecodeMmaParams& p, const DecodeUnit* units, const int32_t* cta_begin,
                       const MdCtx& c) {
  constexpr uint32_t IDESC_S = idesc_bf16_ab(KT, MN, 0, 0);   // K (keys x D) . Q^T
  constexpr uint32_t IDESC_PV = idesc_bf16_ab(128, MN, 1, 0); // V^T (D x keys, MN-major) . P^T
  // The issuing thread shares its sub-partition with softmax warps, so each
  // MMA is issued from descriptors built once: one per shared-memory operand
  // buffer (K and V stages, Q and P buffers); an MMA adds its compile-time
  // offset, in 16-byte units, which never carries out of the 14-bit address
  // field.
  uint64_t dk[NST], dv[NST], dq[2], dp[2];
  for (int i = 0; i < NST; ++i) {
    dk[i] = sdesc_sw128(c.sbase + OFF_K + i * KV_TILE, 16, 1024);
    dv[i] = sdesc_sw128(c.sbase + OFF_V + i * KV_TILE, kAtomKV, 1024);
  }
  for (int i = 0; i < 2; ++i) {
    dq[i] = sdesc_sw128(c.sbase + OFF_Q + i * 2 * kAtomR, 16, 1024);
    dp[i] = sdesc_sw128(c.sbase + OFF_P + i * 2 * kAtomR, 16, 1024);
  }
  // S(g) = K(g) Q^T into S buffer g % 2, with Q buffer qb
  auto issue_s = [&](int g, int qb) -> bool {
    const int st = g % NST;
    if (!wait1(c.bar(Y_K_FULL + st), (g / NST) & 1, c.wc)) return false;
    tc_fence_after();
    const uint64_t ka = st == 0 ? dk[0] : (st == 1 ? dk[1] : dk[2]);
    const uint64_t qb_desc = qb ? dq[1] : dq[0];
    const uint32_t d = c.tmem + TM_S + (g & 1) * MN;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(d, ka + (((kk >> 2) * kAtomKV + (kk & 3) * 32) >> 4),
               qb_desc + (((kk >> 2) * kAtomR + (kk & 3) * 32) >> 4), IDESC_S, kk > 0 ? 1u : 0u);
    mma_commit(c.bar(Y_S_FULL + (g & 1)));
    return true;
  };
  bool ok = true;
  int g = 0, ui = 0;
  for (int u = cta_begin[blockIdx.x]; ok && u < cta_begin[blockIdx.x + 1]; ++u, ++ui) {
    const DecodeUnit U = units[u];
    const int kt0 = U.k0 / KT, kt1 = (U.k1 - 1) / KT;
    const int qb = ui & 1;
    if (!wait1(c.bar(Y_Q_FULL + qb), (ui >> 1) & 1, c.wc)) { ok = false; break; }
    // S of the next stage is issued before P V of this one, so the tensor core
    // works on it while the softmax warps handle this stage
    if (!issue_s(g, qb)) { ok = false; break; }
    if (kt0 == kt1) mma_commit(c.bar(Y_Q_EMPTY + qb));
    const int g0 = g;
    for (int kt = kt0; kt <= kt1; ++kt, ++g) {
      const int st = g % NST;
      if (kt < kt1) {
        if (!issue_s(g + 1, qb)) { ok = false; break; }
        if (kt + 1 == kt1) mma_commit(c.bar(Y_Q_EMPTY + qb));
      }
      if (!wait1(c.bar(Y_P_FULL + (g & 1)), (g >> 1) & 1, c.wc)) { ok = false; break; }
      if (!wait1(c.bar(Y_V_FULL + st), (g / NST) & 1, c.wc)) { ok = false; break; }
      if (kt == kt0 && !wait1(c.bar(Y_O_EMPTY), (ui & 1) ^ 1, c.wc)) { ok = false; break; }
      tc_fence_after();
      {
        const uint64_t va = st == 0 ? dv[0] : (st == 1 ? dv[1] : dv[2]);
        const uint64_t pb = (g & 1) ? dp[1] : dp[0];
        const uint32_t d = c.tmem + TM_O;
        const bool fresh = g == g0;
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk)
          // the unit's first stage starts O^T afresh
          mma_bf16(d, va + kk * 2048 / 16, pb + (((kk >> 2) * kAtomR + (kk & 3) * 32) >> 4),
                   IDESC_PV, (!fresh || kk > 0) ? 1u : 0u);
      }
      mma_commit(c.bar(Y_PV_DONE));
      mma_commit(c.bar(Y_KV_EMPTY + st));
      if (kt == kt1) mma_commit(c.bar(Y_O_FULL));
    }
  }
  if (!ok) {  // aborting: let issued MMAs finish before TMEM is freed
    mma_commit(c.bar(Y_DRAIN));
    wait_drain(c.bar(Y_DRAIN), 0, kDrainNsMD);
  }
}

__device__ void md_softmax(const DecodeMmaParams& p, const DecodeUnit* units,
                           const int32_t* cta_begin, const MdCtx& c, int grp, int warp, int lane) {
  // rows of this group: with 16 rows each group takes 8 (TMEM columns
  // 8 * grp ..); with 8 rows group 0 takes them all and group 1 has no work
  if (grp >= n_groups(p)) return;
  const int r0 = grp * RG;  // first row (and S^T / O^T column) of the group
  const int nr = p.R_rows - r0 < RG ? p.R_rows - r0 : RG;
  const int wq = warp & 3;  // the TMEM lane quarter this warp may access
  const int t = wq * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const float sc = p.scale_log2;
  const bool multi = p.T > 1;
  int g = 0, ui = 0;
  for (int u = cta_begin[blockIdx.x]; u < cta_begin[blockIdx.x + 1]; ++u, ++ui) {
    const DecodeUnit U = units[u];
    const int kt0 = U.k0 / KT, kt1 = (U.k1 - 1) / KT;
    const int g0 = g;
    float m_ref[RG], l_part[RG];
#pragma unroll
    for (int r = 0; r < RG; ++r) {
      m_ref[r] = -INFINITY;
      l_part[r] = 0.f;
    }
    bool ok = true;
    for (int kt = kt0; kt <= kt1; ++kt, ++g) {
      const int sb = g & 1;  // S and P buffers, exchange slot: by stage parity
      if (!waitw(c.bar(Y_S_FULL + sb), (g >> 1) & 1, c.wc)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[RG];
      tmem_ld8(c.tmem + lane_off + TM_S + sb * MN + r0, sv);
      tmem_wait_ld();
      const int j = kt * KT + t;  // this thread's key
      const bool in_unit = j >= U.k0 && j < U.k1;
      float s[RG];
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        bool vis = in_unit && r < nr;
        if (multi) {  // row r0 + r = token (r0 + r) / Gm sees keys up to its own position (and its window)
          const int pr = U.q_last - (p.T - 1) + (r0 + r) / p.Gm;
          vis = vis && j <= pr && (!U.local || j >= pr - p.window + 1);
        }
        s[r] = vis ? __uint_as_float(sv[r]) * sc : -INFINITY;
      }
      // each row's maximum over the stage's 128 keys, shared by the group's warps
      int* xch = reinterpret_cast<int*>(c.smem + OFF_XCH) + (grp * 2 + sb) * 4 * MN;
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const int wm = warp_max_s32(f32_ordered(s[r]));
        if (lane == 0) xch[wq * MN + r] = wm;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(Y_MX + grp * 2 + sb));
      if (!waitw(c.bar(Y_MX + grp * 2 + sb), (g >> 1) & 1, c.wc)) { ok = false; break; }
      bool resc = false;
      float alpha[RG];
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        float mst = f32_from_ordered(xch[r]);
#pragma unroll
        for (int w = 1; w < 4; ++w) mst = fmaxf(mst, f32_from_ordered(xch[w * MN + r]));
        alpha[r] = 1.f;
        if (mst > m_ref[r] + 8.0f) {  // the same decision in every thread of the group
          alpha[r] = ex2(m_ref[r] - mst);
          m_ref[r] = mst;
          resc = true;
        }
      }
      if (resc) {
#pragma unroll
        for (int r = 0; r < RG; ++r) l_part[r] *= alpha[r];
        if (g > g0) {
          // O^T holds the unit's earlier stages. S(g) was issued after P V(g-2)
          // but before P V(g-1): wait for P V(g-1), then scale this group's rows
          if (!waitw(c.bar(Y_PV_DONE), (g - 1) & 1, c.wc)) { ok = false; break; }
          tc_fence_after();
          uint32_t ov[RG];
          tmem_ld8(c.tmem + lane_off + TM_O + r0, ov);
          tmem_wait_ld();
#pragma unroll
          for (int r = 0; r < RG; ++r) ov[r] = __float_as_uint(__uint_as_float(ov[r]) * alpha[r]);
          tmem_st8(c.tmem + lane_off + TM_O + r0, ov);
          tmem_wait_st();
        }
      }
      // P^T[r][t] in bf16, 128-byte swizzled: atom t / 64, 16-byte chunk ((t % 64) / 8) ^ (r % 8).
      // S(g) was issued after P V(g-2), so P buffer g % 2 is free once S(g) is complete.
      uint8_t* pb = c.smem + OFF_P + sb * 2 * kAtomR + (t >> 6) * kAtomR + (t & 7) * 2;
      const int chunk = (t & 63) >> 3;
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const int row = r0 + r;
        const float mu = (m_ref[r] == -INFINITY) ? 0.f : m_ref[r];
        const float pr = ex2(s[r] - mu);
        l_part[r] += pr;
        const __nv_bfloat16 hb = __float2bfloat16_rn(pr);
        *reinterpret_cast<__nv_bfloat16*>(pb + row * 128 + ((chunk ^ (row & 7)) << 4)) = hb;
      }
      if (grp == 0 && (kt == kt0 || kt == kt1)) {
        // edge stage: zero the V rows of keys outside the unit (stale or
        // unwritten slots), once their tile has landed, so P = 0 never meets NaN
        const int st = g % NST;
        if (!waitw(c.bar(Y_V_FULL + st), (g / NST) & 1, c.wc)) { ok = false; break; }
        if (!in_unit) {
          uint8_t* vrow = c.smem + OFF_V + st * KV_TILE + t * 128;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              // chunk q ^ (t % 8): the warp's 32 rows spread over all banks
              *reinterpret_cast<uint4*>(vrow + cc * kAtomKV + ((q ^ (t & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();  // P (and zeroed V rows) are read by the tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(Y_P_FULL + sb));
    }
    if (!ok) break;

    // the group's row sums over the stage's keys
    float* ls = reinterpret_cast<float*>(c.smem + OFF_LS) + (grp * 2 + (ui & 1)) * 4 * MN;
#pragma unroll
    for (int r = 0; r < RG; ++r) {
      float v = l_part[r];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) ls[wq * MN + r] = v;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(Y_LS + grp * 2 + (ui & 1)));
    if (!waitw(c.bar(Y_LS + grp * 2 + (ui & 1)), (ui >> 1) & 1, c.wc)) break;
    float L[RG];
#pragma unroll
    for (int r = 0; r < RG; ++r) L[r] = ((ls[r] + ls[MN + r]) + ls[2 * MN + r]) + ls[3 * MN + r];

    // this group's rows of O^T (thread t = dimension t), then its output
    if (!waitw(c.bar(Y_O_FULL), ui & 1, c.wc)) break;
    tc_fence_after();
    uint32_t ov[RG];
    tmem_ld8(c.tmem + lane_off + TM_O + r0, ov);
    tmem_wait_ld();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(Y_O_EMPTY));
    if (U.pair_units == 1) {
      __nv_bfloat16 ob[RG];
#pragma unroll
      for (int r = 0; r < RG; ++r) ob[r] = __float2bfloat16_rn(__uint_as_float(ov[r]) / L[r]);
      __nv_bfloat16* obase = static_cast<__nv_bfloat16*>(p.o) +
                             (static_cast<int64_t>(U.req) * p.T * p.hq + U.head * p.Gm) * 128 + t;
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        if (r >= nr) break;
        const int tk = (r0 + r) / p.Gm, gm = (r0 + r) - tk * p.Gm;
        obase[(static_cast<int64_t>(tk) * p.hq + gm) * 128] = ob[r];
      }
      if (p.lse != nullptr && t == 0) {
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          if (r >= nr) break;
          const int tk = (r0 + r) / p.Gm, gm = (r0 + r) - tk * p.Gm;
          p.lse[static_cast<int64_t>(U.head * p.Gm + gm) * p.n_rows + U.req * p.T + tk] =
              (m_ref[r] + log2f(L[r])) * 0.6931471805599453f;
        }
      }
    } else {
      float* acc = p.part_acc + (static_cast<int64_t>(u) * p.R_rows + r0) * 128 + t;
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        if (r >= nr) break;
        acc[r * 128] = __uint_as_float(ov[r]);
      }
      if (t == 0) {
        float* ml = p.part_ml + (static_cast<int64_t>(u) * p.R_rows + r0) * 2;
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          if (r >= nr) break;
          ml[2 * r] = m_ref[r];
          ml[2 * r + 1] = L[r];
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreadsMD, 1)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const DecodeMmaParams p,
                      const __grid_constant__ PlanBlob blob) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  MdCtx c;
  c.smem = smem;
  c.sbase = smem_addr(smem);
  const DecodeUnit* units = plan_ptr(p.units, blob, p.plan_inline);
  const int32_t* cta_begin = plan_ptr(p.cta_begin, blob, p.plan_inline);
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.bar(Y_Q_FULL + b), 1);
      mbar_init(c.bar(Y_Q_EMPTY + b), 1);
    }
    for (int s = 0; s < NST; ++s) {
      mbar_init(c.bar(Y_K_FULL + s), 1);
      mbar_init(c.bar(Y_V_FULL + s), 1);
      mbar_init(c.bar(Y_KV_EMPTY + s), 1);
    }
    const uint32_t softmax_warps = 4u * n_groups(p);
    for (int x = 0; x < 2; ++x) {
      mbar_init(c.bar(Y_S_FULL + x), 1);
      mbar_init(c.bar(Y_P_FULL + x), softmax_warps);  // one arrival per softmax warp
    }
    mbar_init(c.bar(Y_PV_DONE), 1);
    mbar_init(c.bar(Y_O_FULL), 1);
    mbar_init(c.bar(Y_O_EMPTY), softmax_warps);  // each group reads its rows of O^T
    for (int x = 0; x < 4; ++x) {
      mbar_init(c.bar(Y_MX + x), 4);
      mbar_init(c.bar(Y_LS + x), 4);
    }
    mbar_init(c.bar(Y_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tmem = *tmem_slot;
  // launched as a programmatic dependent of the previous kernel on the stream:
  // the setup above overlaps its tail; nothing the previous kernels wrote is
  // read before this wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the merge kernel may be scheduled now: it waits for this whole grid to
  // complete (griddepcontrol.wait) before it reads a partial
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  c.wc.abort = abort_flag;
  c.wc.status = p.status;
  c.wc.limit_ns = p.timeout_ns;
  if (warp == 0) {
    md_producer(&tmq, &tmk, &tmv, p, units, cta_begin, c, lane);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) md_mma(p, units, cta_begin, c);
    __syncwarp();
  } else {
    md_softmax(p, units, cta_begin, c, (warp - 2) >> 2, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(c.tmem, TM_COLS);
  }
}

// Merge the partials of split pairs: block (pair, row), thread = dimension.
__global__ void __launch_bounds__(128)
    decode_combine_kernel(const DecodeMmaParams p, const __grid_constant__ PlanBlob blob) {
  // launched as a programmatic dependent of decode_mma_kernel: wait until
  // that grid is complete and its partials are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const DecodeCombine* cmb = plan_ptr(p.combine, blob, p.plan_inline);
  const DecodeCombine C = cmb[blockIdx.x / p.R_rows];
  const int r = blockIdx.x % p.R_rows;
  const int d = threadIdx.x;
  // running-maximum merge over the pair's pieces, eight at a time with all
  // their loads issued together: one round trip to L2 for up to eight pieces
  constexpr int CH = 8;
  float M = -INFINITY, Ls = 0.f, o = 0.f;
  for (int x0 = 0; x0 < C.units; x0 += CH) {
    float mm[CH], ll[CH], aa[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int64_t ur = static_cast<int64_t>(C.unit0 + min(x0 + j, C.units - 1)) * p.R_rows + r;
      mm[j] = x0 + j < C.units ? __ldg(p.part_ml + ur * 2) : -INFINITY;
      ll[j] = __ldg(p.part_ml + ur * 2 + 1);
      aa[j] = __ldg(p.part_acc + ur * 128 + d);
    }
    float Mn = M;
#pragma unroll
    for (int j = 0; j < CH; ++j) Mn = fmaxf(Mn, mm[j]);
    const float Mr = (Mn == -INFINITY) ? 0.f : Mn;  // a piece that sees no key has weight 0
    const float sc = ex2(M - Mr);
    Ls *= sc;
    o *= sc;
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const float wgt = ex2(mm[j] - Mr);
      Ls = fmaf(wgt, ll[j], Ls);
      o = fmaf(wgt, aa[j], o);
    }
    M = Mn;
  }
  const int tk = r / p.Gm, gm = r - tk * p.Gm;
  static_cast<__nv_bfloat16*>(p.o)[(static_cast<int64_t>(C.req * p.T + tk) * p.hq + C.head * p.Gm + gm) * 128 + d] =
      __float2bfloat16_rn(o / Ls);
  if (p.lse != nullptr && d == 0)
    p.lse[static_cast<int64_t>(C.head * p.Gm + gm) * p.n_rows + C.req * p.T + tk] =
        (M + log2f(Ls)) * 0.6931471805599453f;
}

}  // namespace

cudaError_t launch_decode_mma(const DecodeMmaParams& p, const PlanBlob* blob, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                              cudaStream_t s) {
  static const PlanBlob empty_blob{};
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= kMaxDevices || !attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MD_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) attr_set[dev] = true;
  }
  const PlanBlob& b = blob ? *blob : empty_blob;
  cudaError_t e = launch_pdl(decode_mma_kernel, dim3(grid), dim3(kThreadsMD), MD_BYTES, s, tq, tk, tv, p, b);
  if (e != cudaSuccess || p.n_combine == 0) return e;
  // the merge's launch overlaps the tail of the attention kernel
  return launch_pdl(decode_combine_kernel, dim3(p.n_combine * p.R_rows), dim3(128), 0, s, p, b);
}

}  // namespace skv
