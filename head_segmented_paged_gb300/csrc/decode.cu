// Decode attention over head-segmented pages: one query token per sequence
// against every KV head's kept keys (RedKnot summary page, section
// "SegPagedAttention": each head keeps only the keys it needs; "系统收益": many
// concurrent long sessions per GPU). Split-KV with a running-maximum merge of
// the pieces (KV-cache architecture page, section 5.2).
//
// HBM bound. Work is split stream-K style: the (sequence, KV head, key)
// sequence is cut into equal slices, one per CTA, so every CTA streams the
// same number of K/V bytes; a slice may hold the tail of one (sequence, head)
// pair and the head of the next. In each CTA a producer lane streams page
// runs into a 3-stage shared-memory ring with bulk copies. Four consumer
// warps each own a fixed quarter of every stage and keep their own online
// softmax state, so a stage needs no block-wide synchronisation:
//   scores: 16-byte K row reads, packed f32x2 FMAs for the G query heads that
//           share the KV head, a 16-lane reduce-scatter;
//   softmax: max and sum over the lanes holding one head (shuffles);
//   P V:    8-byte V row reads, packed f32x2 FMAs into per-lane accumulators.
// At the end of a slice the four warps merge in shared memory. A pair that
// lies inside one slice writes O directly; otherwise each slice writes fp32
// partials and the last slice to finish (an atomic count per pair) merges
// them and writes O.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "segkv_internal.h"

namespace skv {
using namespace ptx;

namespace {

constexpr int kConsumers = 128;
constexpr int kThreadsSplit = kConsumers + 32;
constexpr int NS = 3;
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;

template <int D, int G>
struct DCfg {
  static constexpr int KW = (32 / G > 16) ? 32 / G : 16;  // keys per consumer warp per stage
  static constexpr int SK = 4 * KW;                       // keys per stage
  static constexpr int KPG = 16 / G;                      // keys per half-warp per round
  static constexpr int ROUNDS = KW / (2 * KPG);
  static constexpr int DPL = D / 16;                      // score dims per lane
  static constexpr int DPV = D / 32;                      // P V dims per lane
  static constexpr int ROW = D * 2;
  static constexpr int STAGE = SK * ROW;                  // bytes of K (or V) per stage
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NS * STAGE;
  static constexpr int OFF_P = OFF_V + NS * STAGE;        // float [4][KW][G]
  static constexpr int OFF_MRG = OFF_P + 4 * KW * G * 4;  // float [4][G][D]
  static constexpr int OFF_ML = OFF_MRG + 4 * G * D * 4;  // float [4][G][2]
  static constexpr int OFF_BAR = (OFF_ML + 4 * G * 2 * 4 + 15) & ~15;
  static constexpr int OFF_MISC = OFF_BAR + 2 * NS * 8;
  static constexpr int BYTES = OFF_MISC + 16;
};

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// Sum 16 per-lane values over the 16 lanes of a half-warp; lane (sub) ends
// with the total of value index sub.
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int sub) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool up = sub & 8;
    const float send = up ? v[i] : v[i + 8];
    const float keep = up ? v[i + 8] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool up = sub & 4;
    const float send = up ? v[i] : v[i + 4];
    const float keep = up ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool up = sub & 2;
    const float send = up ? v[i] : v[i + 2];
    const float keep = up ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  {
    const bool up = sub & 1;
    const float send = up ? v[0] : v[1];
    const float keep = up ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
  }
  return v[0];
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kThreadsSplit)
    decode_split_kernel(const DecodeParams p) {
  using C = DCfg<D, G>;
  extern __shared__ __align__(128) uint8_t sm[];
  const uint32_t sbase = smem_addr(sm);
  float* pbuf = reinterpret_cast<float*>(sm + C::OFF_P);
  float* mrg = reinterpret_cast<float*>(sm + C::OFF_MRG);
  float* mls = reinterpret_cast<float*>(sm + C::OFF_ML);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC);
  int* last_flag = reinterpret_cast<int*>(sm + C::OFF_MISC + 4);
  auto full = [&](int s) { return sbase + C::OFF_BAR + 8u * s; };
  auto empty = [&](int s) { return sbase + C::OFF_BAR + 8u * (NS + s); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kConsumers / 32);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  const int u_begin = p.cta_begin[blockIdx.x], u_end = p.cta_begin[blockIdx.x + 1];

  if (warp == kConsumers / 32) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int armed[NS];
      for (int s = 0; s < NS; ++s) armed[s] = -1;
      bool ok = true;
      int gs = 0;
      for (int u = u_begin; ok && u < u_end; ++u) {
        const DecodeUnit U = p.units[u];
        const int32_t* trow = p.table + static_cast<int64_t>(U.table_row) * p.R;
        for (int w = U.k0 / C::SK; w <= (U.k1 - 1) / C::SK; ++w, ++gs) {
          const int st = gs % NS;
          const uint32_t ph = (gs / NS) & 1;
          if (!wait1(empty(st), ph ^ 1, wc)) { ok = false; break; }
          const int vlo = max(U.k0, w * C::SK), vhi = min(U.k1, w * C::SK + C::SK);
          mbar_expect_tx(full(st), static_cast<uint32_t>((vhi - vlo) * C::ROW * 2));
          armed[st] = static_cast<int>(ph);
          for (int pos = vlo; pos < vhi;) {
            const int k = pos / p.page_size;
            const int pend = min(vhi, (k + 1) * p.page_size);
            const int64_t src =
                (static_cast<int64_t>(trow[k]) * p.page_size + (pos - k * p.page_size)) * C::ROW;
            const uint32_t dst = st * C::STAGE + (pos - w * C::SK) * C::ROW;
            const uint32_t n = static_cast<uint32_t>((pend - pos) * C::ROW);
            bulk_g2s(sbase + C::OFF_K + dst, static_cast<const uint8_t*>(p.kpool) + src, n, full(st));
            bulk_g2s(sbase + C::OFF_V + dst, static_cast<const uint8_t*>(p.vpool) + src, n, full(st));
            pos = pend;
          }
        }
      }
      if (!ok)
        for (int s = 0; s < NS; ++s)
          if (armed[s] >= 0) wait_drain(full(s), armed[s], kDrainNs);
    }
    __syncwarp();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int sub = lane & 15, half = lane >> 4;
  const int g_own = lane % G;  // the query head whose softmax state this lane keeps
  float* my_p = pbuf + warp * C::KW * G;
  int gs = 0;
  for (int u = u_begin; u < u_end; ++u) {
    const DecodeUnit U = p.units[u];
    // this lane's slice of the G query rows, pre-scaled to log2 units
    float2 q2[G][C::DPL / 2];
    {
      const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(p.q) +
                                (static_cast<int64_t>(U.req) * p.hq + U.head * G) * D + sub * C::DPL;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        uint32_t w[C::DPL / 2];
        if constexpr (C::DPL == 8) {
          const uint4 x = *reinterpret_cast<const uint4*>(qb + g * D);
          w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
        } else {
          const uint2 x = *reinterpret_cast<const uint2*>(qb + g * D);
          w[0] = x.x; w[1] = x.y;
        }
#pragma unroll
        for (int e = 0; e < C::DPL / 2; ++e) {
          const float2 f = bf16x2_to_float2(w[e]);
          q2[g][e] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
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
    for (int w = U.k0 / C::SK; w <= (U.k1 - 1) / C::SK; ++w, ++gs) {
      const int st = gs % NS;
      const uint32_t ph = (gs / NS) & 1;
      if (!waitw(full(st), ph, wc)) { ok = false; break; }
      const int base = w * C::SK;
      const int vlo = max(U.k0, base) - base, vhi = min(U.k1, base + C::SK) - base;
      const int mine0 = warp * C::KW;
      if (mine0 < vhi && mine0 + C::KW > vlo) {
        const uint8_t* sK = sm + C::OFF_K + st * C::STAGE;
        const uint8_t* sV = sm + C::OFF_V + st * C::STAGE;
        // scores for this warp's keys
        float sr[C::ROUNDS];
#pragma unroll
        for (int r = 0; r < C::ROUNDS; ++r) {
          const int key0 = mine0 + r * 2 * C::KPG + half * C::KPG;
          float part[16];
#pragma unroll
          for (int kk = 0; kk < C::KPG; ++kk) {
            const uint8_t* krow = sK + (key0 + kk) * C::ROW + sub * C::DPL * 2;
            float2 k2[C::DPL / 2];
            if constexpr (C::DPL == 8) {
              const uint4 x = *reinterpret_cast<const uint4*>(krow);
              k2[0] = bf16x2_to_float2(x.x); k2[1] = bf16x2_to_float2(x.y);
              k2[2] = bf16x2_to_float2(x.z); k2[3] = bf16x2_to_float2(x.w);
            } else {
              const uint2 x = *reinterpret_cast<const uint2*>(krow);
              k2[0] = bf16x2_to_float2(x.x); k2[1] = bf16x2_to_float2(x.y);
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float2 a = make_float2(0.f, 0.f);
#pragma unroll
              for (int e = 0; e < C::DPL / 2; ++e) a = __ffma2_rn(q2[g][e], k2[e], a);
              part[kk * G + g] = a.x + a.y;
            }
          }
          const float tot = reduce_scatter16(part, sub);
          const int kidx = key0 + sub / G;
          sr[r] = (kidx >= vlo && kidx < vhi) ? tot : -INFINITY;
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
          const int kl = r * 2 * C::KPG + half * C::KPG + sub / G;
          my_p[kl * G + g_own] = pr;
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
        const int kl0 = max(vlo - mine0, 0), kl1 = min(vhi - mine0, C::KW);
        for (int kl = kl0; kl < kl1; ++kl) {
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
        }
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(empty(st));
    }
    if (!ok) break;

    // merge the four warps' states
    if (lane < G) {
      mls[(warp * G + lane) * 2 + 0] = m;
      mls[(warp * G + lane) * 2 + 1] = l;
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < C::DPV / 2; ++e)
        *reinterpret_cast<float2*>(mrg + (warp * G + g) * D + lane * C::DPV + 2 * e) = acc[g][e];
    consumer_sync();
    const DecodePair pr = p.pairs[U.pair];
    const bool single = pr.n_units == 1;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) +
                          (static_cast<int64_t>(pr.req) * p.hq + pr.head * G) * D;
    for (int idx = tid; idx < G * D; idx += kConsumers) {
      const int g = idx / D, d = idx - g * D;
      float M = -INFINITY;
#pragma unroll
      for (int x = 0; x < 4; ++x) M = fmaxf(M, mls[(x * G + g) * 2]);
      float Ls = 0.f, o = 0.f;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float wgt = ex2(mls[(x * G + g) * 2] - M);
        Ls = fmaf(wgt, mls[(x * G + g) * 2 + 1], Ls);
        o = fmaf(wgt, mrg[(x * G + g) * D + d], o);
      }
      if (single) {
        orow[g * D + d] = __float2bfloat16_rn(o / Ls);
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
      consumer_sync();
      if (tid == 0) *last_flag = atomicAdd(p.pair_cnt + U.pair, 1) == pr.n_units - 1;
      consumer_sync();
      if (*last_flag) {
        __threadfence();
        for (int idx = tid; idx < G * D; idx += kConsumers) {
          const int g = idx / D, d = idx - g * D;
          float M = -INFINITY;
          for (int c = 0; c < pr.n_units; ++c)
            M = fmaxf(M, __ldcg(p.part_ml + (static_cast<int64_t>(pr.unit0 + c) * G + g) * 2));
          float Ls = 0.f, o = 0.f;
          for (int c = 0; c < pr.n_units; ++c) {
            const int64_t uu = pr.unit0 + c;
            const float wgt = ex2(__ldcg(p.part_ml + (uu * G + g) * 2) - M);
            Ls = fmaf(wgt, __ldcg(p.part_ml + (uu * G + g) * 2 + 1), Ls);
            o = fmaf(wgt, __ldcg(p.part_acc + (uu * G + g) * D + d), o);
          }
          orow[g * D + d] = __float2bfloat16_rn(o / Ls);
        }
      }
    }
    consumer_sync();  // merge buffers are free again
  }
}

template <int D, int G>
static cudaError_t launch_dg(const DecodeParams& p, int grid, cudaStream_t s) {
  using C = DCfg<D, G>;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES);
  if (e != cudaSuccess) return e;
  decode_split_kernel<D, G><<<grid, kThreadsSplit, C::BYTES, s>>>(p);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_d(const DecodeParams& p, int grid, cudaStream_t s) {
  switch (p.G) {
    case 1: return launch_dg<D, 1>(p, grid, s);
    case 2: return launch_dg<D, 2>(p, grid, s);
    case 4: return launch_dg<D, 4>(p, grid, s);
    case 8: return launch_dg<D, 8>(p, grid, s);
    case 16: return launch_dg<D, 16>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

int decode_stage_keys(int G) { return G == 1 ? 128 : 64; }

cudaError_t launch_decode(const DecodeParams& p, int head_dim, int grid, cudaStream_t s) {
  return head_dim == 64 ? launch_d<64>(p, grid, s) : launch_d<128>(p, grid, s);
}

}  // namespace skv
