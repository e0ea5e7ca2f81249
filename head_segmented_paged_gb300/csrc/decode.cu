// Decode attention over head-segmented pages: one query token per sequence
// (or a few: T tokens x Gm heads form the G query rows of a KV head) against
// every KV head's kept keys (RedKnot summary page, section
// "SegPagedAttention": each head keeps only the keys it needs; "系统收益": many
// concurrent long sessions per GPU). Split-KV with a running-maximum merge of
// the pieces (KV-cache architecture page, section 5.2).
//
// HBM bound. Work is split stream-K style: the (sequence, KV head, key)
// sequence is cut into slices of equal cost, one per CTA and one CTA per SM;
// a slice may hold the tail of one (sequence, head) pair and the head of the
// next. In each CTA a producer lane streams page runs into a shared-memory
// ring with bulk copies. Twelve consumer warps at G = 4 (eight or four
// otherwise) each own a fixed share of every stage and keep their own online
// softmax state, so a stage needs no block-wide synchronisation:
//   scores: 16-byte K chunk reads (lane i of a group of 8 takes chunks i and
//           i+8 of a row, so every read is free of bank conflicts), packed
//           f32x2 FMAs for the G query heads that share the KV head, an
//           8-lane reduce-scatter;
//   softmax: max and sum over the lanes holding one head (shuffles);
//   P V:    8-byte V row reads, packed f32x2 FMAs into per-lane accumulators.
// At the end of a slice the warps merge in shared memory. A pair that
// lies inside one slice writes O directly; otherwise each slice writes fp32
// partials and the last slice to finish (an atomic count per pair) merges
// them and writes O.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "segkv_internal.h"

namespace skv {
using namespace ptx;

namespace {

constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;

// One CTA per SM. With two smaller CTAs per SM, measured per-CTA timestamps
// showed the pair sharing the SM's memory stream unevenly: on 96 % of the SMs
// one CTA of the two (nearly always the higher block index) finished about
// 8 us later than the other, after about 4x longer waits for data, although
// both streamed the same bytes. A static plan cannot balance that. One CTA
// with twice the consumer warps streams a single slice per SM instead
// (ragged decode, G = 4: 66.9 -> 62.6 us per call).
template <int D, int G>
struct DCfg {
  // consumer warps: 12 for G = 4; 8 for G = 2, and for 8 or 16 rows of 64
  // dims; 4 for G = 1 (32 keys per warp and stage) and for 8 or 16 rows of
  // 128 dims (register-heavy, and run on the tensor-core kernel instead)
  static constexpr int NW = G == 4 ? 12 : (G == 2 || (D == 64 && G >= 8)) ? 8 : 4;
  static constexpr int THREADS = 32 * (NW + 1);            // + one producer warp
  static constexpr int LG = G > 8 ? G : 8;                 // lanes per score group
  static constexpr int KPG = LG / G;                       // keys per group per round
  static constexpr int KR = (32 / LG) * KPG;               // keys per warp per round (= 32/G)
  static constexpr int KW = KR > 8 ? KR : 8;               // keys per consumer warp per stage
  static constexpr int ROUNDS = KW / KR;
  static constexpr int SK = NW * KW;                       // keys per stage
  static constexpr int DPL = D / LG;                       // score dims per lane
  static constexpr int DPV = D / 32;                       // P V dims per lane
  static constexpr int ROW = D * 2;
  static constexpr int STAGE = SK * ROW;                   // bytes of K (or V) per stage
  // stages: as many K + V stages as fit in 192 KB, between 2 and 8
  static constexpr int NS_FIT = 192 * 1024 / (2 * STAGE);
  static constexpr int NS = NS_FIT < 2 ? 2 : (NS_FIT > 8 ? 8 : NS_FIT);
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NS * STAGE;
  static constexpr int OFF_P = OFF_V + NS * STAGE;         // float [NW][KW][G]
  static constexpr int OFF_MRG = OFF_P + NW * KW * G * 4;  // float [NW/2][G][D]
  static constexpr int OFF_ML = OFF_MRG + (NW / 2) * G * D * 4;  // float [NW/2][G][2]
  static constexpr int META = sizeof(DecodeUnit);
  static constexpr int OFF_META = (OFF_ML + (NW / 2) * G * 2 * 4 + 31) & ~31;  // DecodeUnit [NS]
  static constexpr int OFF_QB = OFF_META + NS * META;                          // bf16 [NS][G][D]
  static constexpr int OFF_BAR = (OFF_QB + NS * G * D * 2 + 15) & ~15;
  static constexpr int OFF_MISC = OFF_BAR + 2 * NS * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static_assert(BYTES <= 227 * 1024, "decode shared memory");
  static constexpr int MIN_BLOCKS = 1;
};

template <int N>
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// Sum LG per-lane values over each group of LG consecutive lanes; lane
// (lane % LG) ends with the total of value index lane % LG. Each level sends
// the half of the values the partner keeps and adds the half it receives.
template <int LG>
__device__ __forceinline__ float reduce_scatter(float (&v)[LG], int sub) {
#pragma unroll
  for (int w = LG / 2; w >= 1; w >>= 1) {
    const bool up = sub & w;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

}  // namespace

// MQ: several query tokens per sequence (T > 1), each row with its own key limits
template <int D, int G, bool MQ>
__global__ void __launch_bounds__(DCfg<D, G>::THREADS, DCfg<D, G>::MIN_BLOCKS)
    decode_split_kernel(const DecodeParams p, const __grid_constant__ PlanBlob blob) {
  using C = DCfg<D, G>;
  constexpr int NCONS = 32 * C::NW;
  constexpr int HALF = C::NW / 2;
  constexpr int CPL = C::DPL >= 8 ? C::DPL / 8 : 1;  // 16-byte K chunks per lane
  extern __shared__ __align__(128) uint8_t sm[];
  const uint32_t sbase = smem_addr(sm);
  float* pbuf = reinterpret_cast<float*>(sm + C::OFF_P);
  float* mrg = reinterpret_cast<float*>(sm + C::OFF_MRG);
  float* mls = reinterpret_cast<float*>(sm + C::OFF_ML);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC);
  int* last_flag = reinterpret_cast<int*>(sm + C::OFF_MISC + 4);
  auto full = [&](int s) { return sbase + C::OFF_BAR + 8u * s; };
  constexpr int NS = C::NS;
  auto empty = [&](int s) { return sbase + C::OFF_BAR + 8u * (NS + s); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), C::NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // launched as a programmatic dependent of the previous kernel on the stream:
  // everything above overlaps its tail; nothing the previous kernels wrote
  // (plan, block table, q, K/V, partials, counters) is read before this wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  const DecodeUnit* units =
      p.plan_inline ? reinterpret_cast<const DecodeUnit*>(blob.data + reinterpret_cast<uintptr_t>(p.units))
                    : p.units;
  const int32_t* cta_begin =
      p.plan_inline ? reinterpret_cast<const int32_t*>(blob.data + reinterpret_cast<uintptr_t>(p.cta_begin))
                    : p.cta_begin;
  const int u_begin = cta_begin[blockIdx.x], u_end = cta_begin[blockIdx.x + 1];

  if (warp == C::NW) {
    // The whole warp runs the loop: its lanes fetch 32 block-table entries at
    // a time (one coalesced load instead of a dependent load per page run) and
    // lane 0 issues the copies.
    int armed[NS];
    for (int s = 0; s < NS; ++s) armed[s] = -1;
    bool ok = true;
    int gs = 0;
    for (int u = u_begin; ok && u < u_end; ++u) {
      const DecodeUnit U = units[u];
      const int32_t* trow = p.table + static_cast<int64_t>(U.table_row) * p.R;
      int kbase = -(1 << 30), my_id = 0;
      // stages start at the unit's first key, so only its last stage is partial
      for (int w = 0; U.k0 + w * C::SK < U.k1; ++w, ++gs) {
        const int st = gs % NS;
        const uint32_t ph = (gs / NS) & 1;
        if (!waitw(empty(st), ph ^ 1, wc)) { ok = false; break; }
        const int vlo = U.k0 + w * C::SK, vhi = min(U.k1, vlo + C::SK);
        const bool first = (w == 0);
        if (lane == 0) {
          uint32_t bytes = static_cast<uint32_t>((vhi - vlo) * C::ROW * 2);
          if (first) {  // the unit's descriptor and its G query rows travel with its first stage
            *reinterpret_cast<DecodeUnit*>(sm + C::OFF_META + st * C::META) = U;
            bytes += G * D * 2;
          }
          mbar_expect_tx(full(st), bytes);
          if (first) {
            if constexpr (MQ) {  // row t * Gm + j = token t, query head head * Gm + j
              for (int t = 0; t < p.T; ++t)
                bulk_g2s(sbase + C::OFF_QB + (st * G + t * p.Gm) * D * 2,
                         static_cast<const __nv_bfloat16*>(p.q) +
                             (static_cast<int64_t>(U.req * p.T + t) * p.hq + U.head * p.Gm) * D,
                         p.Gm * D * 2, full(st));
            } else {
              bulk_g2s(sbase + C::OFF_QB + st * G * D * 2,
                       static_cast<const __nv_bfloat16*>(p.q) +
                           (static_cast<int64_t>(U.req) * p.hq + U.head * G) * D,
                       G * D * 2, full(st));
            }
          }
        }
        armed[st] = static_cast<int>(ph);
        for (int pos = vlo; pos < vhi;) {
          const int k = pos / p.page_size;
          if (k >= kbase + 32) {
            kbase = k;
            my_id = (k + lane < p.R) ? trow[k + lane] : 0;
          }
          const int id = __shfl_sync(0xffffffffu, my_id, k - kbase);
          const int pend = min(vhi, (k + 1) * p.page_size);
          if (lane == 0) {
            const int64_t src =
                (static_cast<int64_t>(id) * p.page_size + (pos - k * p.page_size)) * C::ROW;
            const uint32_t dst = st * C::STAGE + (pos - vlo) * C::ROW;
            const uint32_t n = static_cast<uint32_t>((pend - pos) * C::ROW);
            bulk_g2s(sbase + C::OFF_K + dst, static_cast<const uint8_t*>(p.kpool) + src, n, full(st));
            bulk_g2s(sbase + C::OFF_V + dst, static_cast<const uint8_t*>(p.vpool) + src, n, full(st));
          }
          pos = pend;
        }
      }
    }
    if (!ok && lane == 0)
      for (int s = 0; s < NS; ++s)
        if (armed[s] >= 0) wait_drain(full(s), armed[s], kDrainNs);
    __syncwarp();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int sub = lane % C::LG, grp = lane / C::LG;
  const int g_own = lane % G;  // the query head whose softmax state this lane keeps
  float* my_p = pbuf + warp * C::KW * G;
  int gs = 0;
  for (int u = u_begin; u < u_end; ++u) {
    // the unit's descriptor and query rows arrive with its first stage
    if (!waitw(full(gs % NS), (gs / NS) & 1, wc)) break;
    const DecodeUnit U = *reinterpret_cast<const DecodeUnit*>(sm + C::OFF_META + (gs % NS) * C::META);
    // the keys this lane's query row may see: up to its own position, and for
    // a local head no further back than its window (with one query token per
    // sequence the unit's key range holds exactly these)
    int p_own = 0, lo_own = 0;
    if constexpr (MQ) {
      p_own = U.q_last - (p.T - 1) + g_own / p.Gm;
      lo_own = U.local ? p_own - p.window + 1 : 0;
    }
    // this lane's dims of the G query rows (chunks sub, sub+LG, ... of 8 dims,
    // or 4 dims at sub*4 when D/LG = 4), pre-scaled to log2 units
    float2 q2[G][C::DPL / 2];
    {
      const __nv_bfloat16* qb =
          reinterpret_cast<const __nv_bfloat16*>(sm + C::OFF_QB + (gs % NS) * G * D * 2);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if constexpr (C::DPL >= 8) {
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const uint4 x = *reinterpret_cast<const uint4*>(qb + g * D + (sub + C::LG * c) * 8);
            const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = bf16x2_to_float2(w4[e]);
              q2[g][c * 4 + e] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
            }
          }
        } else {
          const uint2 x = *reinterpret_cast<const uint2*>(qb + g * D + sub * 4);
          const float2 f0 = bf16x2_to_float2(x.x), f1 = bf16x2_to_float2(x.y);
          q2[g][0] = make_float2(f0.x * p.scale_log2, f0.y * p.scale_log2);
          q2[g][1] = make_float2(f1.x * p.scale_log2, f1.y * p.scale_log2);
        }
      }
    }
    float2 acc[G][C::DPV / 2];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < C::DPV / 2; ++e) acc[g][e] = make_float2(0.f, 0.f);
    float m = -INFINITY, l = 0.f;

    bool ok = true;
    for (int w = 0; U.k0 + w * C::SK < U.k1; ++w, ++gs) {
      const int st = gs % NS;
      const uint32_t ph = (gs / NS) & 1;
      if (!waitw(full(st), ph, wc)) { ok = false; break; }
      const int base = U.k0 + w * C::SK;  // first key of the stage
      const int vlo = max(U.k0, base) - base, vhi = min(U.k1, base + C::SK) - base;
      // the keys of this stage the lane's query row sees
      const int vlo_own = MQ ? max(vlo, lo_own - base) : vlo;
      const int vhi_own = MQ ? min(vhi, p_own + 1 - base) : vhi;
      const int mine0 = warp * C::KW;
      if (mine0 < vhi && mine0 + C::KW > vlo) {
        const uint8_t* sK = sm + C::OFF_K + st * C::STAGE;
        const uint8_t* sV = sm + C::OFF_V + st * C::STAGE;
        // scores for this warp's keys
        float sr[C::ROUNDS];
#pragma unroll
        for (int r = 0; r < C::ROUNDS; ++r) {
          const int key0 = mine0 + r * C::KR + grp * C::KPG;
          float part[C::LG];
#pragma unroll
          for (int kk = 0; kk < C::KPG; ++kk) {
            const uint8_t* krow = sK + (key0 + kk) * C::ROW;
            float2 k2[C::DPL / 2];
            if constexpr (C::DPL >= 8) {
#pragma unroll
              for (int c = 0; c < CPL; ++c) {
                const uint4 x = *reinterpret_cast<const uint4*>(krow + (sub + C::LG * c) * 16);
                k2[c * 4 + 0] = bf16x2_to_float2(x.x);
                k2[c * 4 + 1] = bf16x2_to_float2(x.y);
                k2[c * 4 + 2] = bf16x2_to_float2(x.z);
                k2[c * 4 + 3] = bf16x2_to_float2(x.w);
              }
            } else {
              const uint2 x = *reinterpret_cast<const uint2*>(krow + sub * 8);
              k2[0] = bf16x2_to_float2(x.x);
              k2[1] = bf16x2_to_float2(x.y);
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float2 a = make_float2(0.f, 0.f);
#pragma unroll
              for (int e = 0; e < C::DPL / 2; ++e) a = __ffma2_rn(q2[g][e], k2[e], a);
              part[kk * G + g] = a.x + a.y;
            }
          }
          const float tot = reduce_scatter<C::LG>(part, sub);
          const int kidx = key0 + sub / G;
          sr[r] = (kidx >= vlo_own && kidx < vhi_own) ? tot : -INFINITY;
        }
        // online softmax for head g_own over this warp's keys
        float mx = sr[0];
#pragma unroll
        for (int r = 1; r < C::ROUNDS; ++r) mx = fmaxf(mx, sr[r]);
#pragma unroll
        for (int o = G; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_new = fmaxf(m, mx);
        const float msub = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2(m - msub);
        float psum = 0.f;
#pragma unroll
        for (int r = 0; r < C::ROUNDS; ++r) {
          const float pr = ex2(sr[r] - msub);
          psum += pr;
          my_p[(r * C::KR + grp * C::KPG + sub / G) * G + g_own] = pr;
        }
#pragma unroll
        for (int o = G; o < 32; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
        l = l * alpha + psum;
        m = m_new;
        __syncwarp();
        // acc = acc * alpha + P V over this warp's valid keys
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float ag = __shfl_sync(0xffffffffu, alpha, g);
          const float2 a2 = make_float2(ag, ag);
#pragma unroll
          for (int e = 0; e < C::DPV / 2; ++e) acc[g][e] = __fmul2_rn(acc[g][e], a2);
        }
        auto pv_key = [&](int kl) {
          const uint8_t* vrow = sV + (mine0 + kl) * C::ROW + lane * C::DPV * 2;
          float2 v2[C::DPV / 2];
          if constexpr (C::DPV == 4) {
            const uint2 x = *reinterpret_cast<const uint2*>(vrow);
            v2[0] = bf16x2_to_float2(x.x);
            v2[1] = bf16x2_to_float2(x.y);
          } else {
            v2[0] = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(vrow));
          }
          const float* pk = my_p + kl * G;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float2 pg = make_float2(pk[g], pk[g]);
#pragma unroll
            for (int e = 0; e < C::DPV / 2; ++e) acc[g][e] = __ffma2_rn(pg, v2[e], acc[g][e]);
          }
        };
        const int kl0 = max(vlo - mine0, 0), kl1 = min(vhi - mine0, C::KW);
        if (kl0 == 0 && kl1 == C::KW) {
#pragma unroll
          for (int kl = 0; kl < C::KW; ++kl) pv_key(kl);
        } else {
          for (int kl = kl0; kl < kl1; ++kl) pv_key(kl);
        }
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(empty(st));
    }
    if (!ok) break;

    // merge the warps' states: the upper half hands its state to the lower half,
    // which folds it into its own, then every thread combines the lower half's
    if (warp >= HALF) {
      const int slot = warp - HALF;
      if (lane < G) {
        mls[(slot * G + lane) * 2 + 0] = m;
        mls[(slot * G + lane) * 2 + 1] = l;
      }
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < C::DPV / 2; ++e)
          *reinterpret_cast<float2*>(mrg + (slot * G + g) * D + lane * C::DPV + 2 * e) = acc[g][e];
    }
    consumer_sync<NCONS>();
    if (warp < HALF) {
      const int slot = warp;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float m1 = __shfl_sync(0xffffffffu, m, g), l1 = __shfl_sync(0xffffffffu, l, g);
        const float m2 = mls[(slot * G + g) * 2], l2 = mls[(slot * G + g) * 2 + 1];
        const float M = fmaxf(m1, m2);
        const float ms = (M == -INFINITY) ? 0.f : M;
        const float a1 = ex2(m1 - ms), a2 = ex2(m2 - ms);
        const float2 w1 = make_float2(a1, a1), w2 = make_float2(a2, a2);
#pragma unroll
        for (int e = 0; e < C::DPV / 2; ++e) {
          float2* dst = reinterpret_cast<float2*>(mrg + (slot * G + g) * D + lane * C::DPV + 2 * e);
          *dst = __ffma2_rn(acc[g][e], w1, __fmul2_rn(*dst, w2));
        }
        __syncwarp();
        if (lane == 0) {
          mls[(slot * G + g) * 2] = M;
          mls[(slot * G + g) * 2 + 1] = l1 * a1 + l2 * a2;
        }
      }
    }
    consumer_sync<NCONS>();
    const bool single = U.pair_units == 1;
    const int pair = U.req * p.hkv + U.head;
    // query row g is token g / Gm of the sequence, query head head * Gm + g % Gm
    auto out_at = [&](int g) -> __nv_bfloat16* {
      if constexpr (!MQ)
        return static_cast<__nv_bfloat16*>(p.o) + (static_cast<int64_t>(U.req) * p.hq + U.head * G + g) * D;
      const int t = g / p.Gm;
      return static_cast<__nv_bfloat16*>(p.o) +
             (static_cast<int64_t>(U.req * p.T + t) * p.hq + U.head * p.Gm + g - t * p.Gm) * D;
    };
    auto put_lse = [&](int g, float M, float Ls) {  // natural-log LSE of row g
      const int t = g / p.Gm;
      p.lse[static_cast<int64_t>(U.head * p.Gm + g - t * p.Gm) * p.n_rows + U.req * p.T + t] =
          (M + log2f(Ls)) * 0.6931471805599453f;
    };
    for (int idx = tid; idx < G * D; idx += NCONS) {
      const int g = idx / D, d = idx - g * D;
      float M = -INFINITY;
#pragma unroll
      for (int x = 0; x < HALF; ++x) M = fmaxf(M, mls[(x * G + g) * 2]);
      const float ms = (M == -INFINITY) ? 0.f : M;
      float Ls = 0.f, o = 0.f;
#pragma unroll
      for (int x = 0; x < HALF; ++x) {
        const float wgt = ex2(mls[(x * G + g) * 2] - ms);
        Ls = fmaf(wgt, mls[(x * G + g) * 2 + 1], Ls);
        o = fmaf(wgt, mrg[(x * G + g) * D + d], o);
      }
      if (single) {
        out_at(g)[d] = __float2bfloat16_rn(o / Ls);
        if (MQ && p.lse != nullptr && d == 0) put_lse(g, M, Ls);
      } else {
        p.part_acc[(static_cast<int64_t>(u) * G + g) * D + d] = o;
        if (d == 0) {
          p.part_ml[(static_cast<int64_t>(u) * G + g) * 2] = M;
          p.part_ml[(static_cast<int64_t>(u) * G + g) * 2 + 1] = Ls;
        }
      }
    }
    if (!single) {
      __threadfence();
      consumer_sync<NCONS>();
      if (tid == 0) *last_flag = atomicAdd(p.pair_cnt + pair, 1) == U.pair_units - 1;
      consumer_sync<NCONS>();
      if (*last_flag) {
        // the last slice of the pair merges every slice's partials. Each
        // thread owns EPT output elements; the loads of CH slices for all of
        // them are issued together, so a pair of n slices costs about n / CH
        // dependent L2 round trips instead of n / 4 per element.
        constexpr int EPT = (G * D + NCONS - 1) / NCONS;
        constexpr int CH = (16 / EPT) > 8 ? 8 : ((16 / EPT) < 1 ? 1 : 16 / EPT);
        __threadfence();
        float M[EPT], Ls[EPT], o[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
          M[e] = -INFINITY;
          Ls[e] = 0.f;
          o[e] = 0.f;
        }
        for (int c0 = 0; c0 < U.pair_units; c0 += CH) {
          float mm[EPT][CH], ll[EPT][CH], aa[EPT][CH];
#pragma unroll
          for (int e = 0; e < EPT; ++e) {
            const int idx = min(tid + e * NCONS, G * D - 1);
            const int g = idx / D, d = idx - g * D;
#pragma unroll
            for (int j = 0; j < CH; ++j) {
              const int64_t uu = U.pair_unit0 + min(c0 + j, U.pair_units - 1);
              mm[e][j] = (c0 + j < U.pair_units) ? __ldcg(p.part_ml + (uu * G + g) * 2) : -INFINITY;
              ll[e][j] = __ldcg(p.part_ml + (uu * G + g) * 2 + 1);
              aa[e][j] = __ldcg(p.part_acc + (uu * G + g) * D + d);
            }
          }
#pragma unroll
          for (int e = 0; e < EPT; ++e) {
            // a slice may hold no key a row sees (several query tokens per
            // sequence): its maximum is -inf and its weight 0
            float Mn = M[e];
#pragma unroll
            for (int j = 0; j < CH; ++j) Mn = fmaxf(Mn, mm[e][j]);
            const float Mr = (Mn == -INFINITY) ? 0.f : Mn;
            const float sc = ex2(M[e] - Mr);
            Ls[e] *= sc;
            o[e] *= sc;
#pragma unroll
            for (int j = 0; j < CH; ++j) {
              const float wgt = ex2(mm[e][j] - Mr);
              Ls[e] = fmaf(wgt, ll[e][j], Ls[e]);
              o[e] = fmaf(wgt, aa[e][j], o[e]);
            }
            M[e] = Mn;
          }
        }
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
          const int idx = tid + e * NCONS;
          if (idx < G * D) {
            const int g = idx / D, d = idx - g * D;
            out_at(g)[d] = __float2bfloat16_rn(o[e] / Ls[e]);
            if (MQ && p.lse != nullptr && d == 0) put_lse(g, M[e], Ls[e]);
          }
        }
        if (tid == 0) p.pair_cnt[pair] = 0;  // ready for the next call
      }
    }
    consumer_sync<NCONS>();  // merge buffers are free again
  }
}

template <int D, int G, bool MQ>
static cudaError_t launch_dgm(const DecodeParams& p, const PlanBlob* blob, int grid, cudaStream_t s) {
  using C = DCfg<D, G>;
  static const PlanBlob empty_blob{};
  static bool attr_set[kMaxDevices] = {};  // the attribute outlives the launch
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= kMaxDevices || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, G, MQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) attr_set[dev] = true;
  }
  return launch_pdl(decode_split_kernel<D, G, MQ>, dim3(grid), dim3(C::THREADS), C::BYTES, s, p,
                    blob ? *blob : empty_blob);
}

template <int D, int G>
static cudaError_t launch_dg(const DecodeParams& p, const PlanBlob* blob, int grid, cudaStream_t s) {
  // the single-token variant skips the per-row limits and writes no LSE
  return (p.T > 1 || p.lse != nullptr) ? launch_dgm<D, G, true>(p, blob, grid, s)
                                       : launch_dgm<D, G, false>(p, blob, grid, s);
}

template <int D>
static cudaError_t launch_d(const DecodeParams& p, const PlanBlob* blob, int grid, cudaStream_t s) {
  switch (p.G) {
    case 1: return launch_dg<D, 1>(p, blob, grid, s);
    case 2: return launch_dg<D, 2>(p, blob, grid, s);
    case 4: return launch_dg<D, 4>(p, blob, grid, s);
    case 8: return launch_dg<D, 8>(p, blob, grid, s);
    case 16: return launch_dg<D, 16>(p, blob, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

int decode_stage_keys(int G) {
  switch (G) {
    case 1: return DCfg<128, 1>::SK;
    case 2: return DCfg<128, 2>::SK;
    case 4: return DCfg<128, 4>::SK;
    case 8: return DCfg<128, 8>::SK;
    default: return DCfg<128, 16>::SK;
  }
}

int decode_ctas_per_sm(int head_dim, int G) {
  if (head_dim == 64) {
    switch (G) {
      case 1: return DCfg<64, 1>::MIN_BLOCKS;
      case 2: return DCfg<64, 2>::MIN_BLOCKS;
      case 4: return DCfg<64, 4>::MIN_BLOCKS;
      case 8: return DCfg<64, 8>::MIN_BLOCKS;
      default: return DCfg<64, 16>::MIN_BLOCKS;
    }
  }
  switch (G) {
    case 1: return DCfg<128, 1>::MIN_BLOCKS;
    case 2: return DCfg<128, 2>::MIN_BLOCKS;
    case 4: return DCfg<128, 4>::MIN_BLOCKS;
    case 8: return DCfg<128, 8>::MIN_BLOCKS;
    default: return DCfg<128, 16>::MIN_BLOCKS;
  }
}

cudaError_t launch_decode(const DecodeParams& p, const PlanBlob* blob, int head_dim, int grid,
                          cudaStream_t s) {
  return head_dim == 64 ? launch_d<64>(p, blob, grid, s) : launch_d<128>(p, blob, grid, s);
}

}  // namespace skv
