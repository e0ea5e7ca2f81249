// Decode attention over head-segmented pages: one query token per sequence
// against every KV head's kept keys (RedKnot summary page, section
// "SegPagedAttention": each head keeps only the keys it needs; "系统收益": many
// concurrent long sessions per GPU). Split-KV: each unit reduces one key chunk
// of one (sequence, KV head) to partial (m, l, acc) per query head; a combine
// pass merges the chunks with the running-maximum rule (KV-cache architecture
// page, section 5.2).
//
// HBM bound. The G query heads of a KV head share each K/V byte. Keys stream
// through a 3-stage shared-memory ring filled by bulk copies of whole page
// runs (one producer lane); four consumer warps compute scores with 16-byte
// row reads and a 16-lane reduce-scatter, then P V with 4-byte reads.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "segkv_internal.h"

namespace skv {
using namespace ptx;

namespace {

constexpr int SK = kDecodeStageKeys;  // keys per stage
constexpr int NS = 3;                 // stages
constexpr int kConsumers = 128;
constexpr int kThreadsSplit = kConsumers + 32;
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;

template <int D, int G>
struct DLayout {
  static constexpr int ROW = D * 2;
  static constexpr int STAGE = SK * ROW;  // bytes of K (or V) per stage
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NS * STAGE;
  static constexpr int OFF_SC = OFF_V + NS * STAGE;          // float [SK][G]
  static constexpr int OFF_RED = OFF_SC + SK * G * 4;        // float [G][D] reduction
  static constexpr int OFF_ML = OFF_RED + G * D * 4;         // float m[G], l[G], alpha[G]
  static constexpr int OFF_BAR = (OFF_ML + 3 * G * 4 + 15) & ~15;
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

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kThreadsSplit)
    decode_split_kernel(const DecodeParams p) {
  using L = DLayout<D, G>;
  constexpr int DPL = D / 16;     // dims per lane in the score phase
  constexpr int KPG = 16 / G;     // keys per half-warp per round
  constexpr int NPAIR = D / 2;    // bf16 pairs per row
  constexpr int KH = kConsumers / NPAIR;  // key phases in P V
  extern __shared__ __align__(128) uint8_t sm[];
  const uint32_t sbase = smem_addr(sm);
  float* sc = reinterpret_cast<float*>(sm + L::OFF_SC);
  float* red = reinterpret_cast<float*>(sm + L::OFF_RED);
  float* s_m = reinterpret_cast<float*>(sm + L::OFF_ML);
  float* s_l = s_m + G;
  float* s_alpha = s_l + G;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::OFF_MISC);
  auto full = [&](int s) { return sbase + L::OFF_BAR + 8u * s; };
  auto empty = [&](int s) { return sbase + L::OFF_BAR + 8u * (NS + s); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (tid < G) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  __syncthreads();
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  if (warp == kConsumers / 32) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int armed[NS];
      for (int s = 0; s < NS; ++s) armed[s] = -1;
      bool ok = true;
      int gs = 0;
      for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
        const DecodeUnit U = p.units[u];
        const int32_t* trow = p.table + static_cast<int64_t>(U.table_row) * p.R;
        for (int w = U.k0 / SK; w <= (U.k1 - 1) / SK; ++w, ++gs) {
          const int st = gs % NS;
          const uint32_t ph = (gs / NS) & 1;
          if (!wait1(empty(st), ph ^ 1, wc)) { ok = false; break; }
          const int vlo = max(U.k0, w * SK), vhi = min(U.k1, w * SK + SK);
          mbar_expect_tx(full(st), static_cast<uint32_t>((vhi - vlo) * L::ROW * 2));
          armed[st] = static_cast<int>(ph);
          for (int pos = vlo; pos < vhi;) {
            const int k = pos / p.page_size;
            const int pend = min(vhi, (k + 1) * p.page_size);
            const int64_t src =
                (static_cast<int64_t>(trow[k]) * p.page_size + (pos - k * p.page_size)) * L::ROW;
            const uint32_t dst = st * L::STAGE + (pos - w * SK) * L::ROW;
            const uint32_t n = static_cast<uint32_t>((pend - pos) * L::ROW);
            bulk_g2s(sbase + L::OFF_K + dst, static_cast<const uint8_t*>(p.kpool) + src, n, full(st));
            bulk_g2s(sbase + L::OFF_V + dst, static_cast<const uint8_t*>(p.vpool) + src, n, full(st));
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
  const int kh = tid / NPAIR, dp = tid - kh * NPAIR;
  int gs = 0;
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const DecodeUnit U = p.units[u];
    // this lane's slice of the G query rows, pre-scaled to log2 units
    float qr[G][DPL];
    {
      const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(p.q) +
                                (static_cast<int64_t>(U.req) * p.hq + U.head * G) * D + sub * DPL;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        uint32_t w[DPL / 2];
        if constexpr (DPL == 8) {
          const uint4 x = *reinterpret_cast<const uint4*>(qb + g * D);
          w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
        } else {
          const uint2 x = *reinterpret_cast<const uint2*>(qb + g * D);
          w[0] = x.x; w[1] = x.y;
        }
#pragma unroll
        for (int e = 0; e < DPL / 2; ++e) {
          qr[g][2 * e] = bf16lo(w[e]) * p.scale_log2;
          qr[g][2 * e + 1] = bf16hi(w[e]) * p.scale_log2;
        }
      }
    }
    float acc[G][2];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g][0] = acc[g][1] = 0.f;

    bool ok = true;
    for (int w = U.k0 / SK; w <= (U.k1 - 1) / SK; ++w, ++gs) {
      const int st = gs % NS;
      const uint32_t ph = (gs / NS) & 1;
      if (!waitw(full(st), ph, wc)) { ok = false; break; }
      const int base = w * SK;
      const int vlo = max(U.k0, base) - base, vhi = min(U.k1, base + SK) - base;
      const uint8_t* sK = sm + L::OFF_K + st * L::STAGE;
      const uint8_t* sV = sm + L::OFF_V + st * L::STAGE;

      // scores: each half-warp takes KPG keys per round
#pragma unroll
      for (int r0 = 0; r0 < SK; r0 += 8 * KPG) {
        const int key0 = r0 + (warp * 2 + half) * KPG;
        float part[16];
#pragma unroll
        for (int kk = 0; kk < KPG; ++kk) {
          const int key = min(key0 + kk, SK - 1);
          float kf[DPL];
          const uint8_t* krow = sK + key * L::ROW + sub * DPL * 2;
          if constexpr (DPL == 8) {
            const uint4 x = *reinterpret_cast<const uint4*>(krow);
            kf[0] = bf16lo(x.x); kf[1] = bf16hi(x.x); kf[2] = bf16lo(x.y); kf[3] = bf16hi(x.y);
            kf[4] = bf16lo(x.z); kf[5] = bf16hi(x.z); kf[6] = bf16lo(x.w); kf[7] = bf16hi(x.w);
          } else {
            const uint2 x = *reinterpret_cast<const uint2*>(krow);
            kf[0] = bf16lo(x.x); kf[1] = bf16hi(x.x); kf[2] = bf16lo(x.y); kf[3] = bf16hi(x.y);
          }
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float a = 0.f;
#pragma unroll
            for (int d = 0; d < DPL; ++d) a = fmaf(qr[g][d], kf[d], a);
            part[kk * G + g] = a;
          }
        }
        const float tot = reduce_scatter16(part, sub);
        const int kidx = key0 + sub / G;
        if (kidx < SK) sc[kidx * G + (sub % G)] = (kidx >= vlo && kidx < vhi) ? tot : -INFINITY;
      }
      consumer_sync();

      // running max / sum per query head
      for (int g = warp; g < G; g += kConsumers / 32) {
        const float a = sc[lane * G + g], b = sc[(lane + 32) * G + g];
        float mx = fmaxf(a, b);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_old = s_m[g];
        const float m_new = fmaxf(m_old, mx);
        const float msub = (m_new == -INFINITY) ? 0.f : m_new;
        const float pa = ex2(a - msub), pb = ex2(b - msub);
        sc[lane * G + g] = pa;
        sc[(lane + 32) * G + g] = pb;
        float sum = pa + pb;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) {
          const float al = ex2(m_old - msub);
          s_l[g] = s_l[g] * al + sum;
          s_m[g] = m_new;
          s_alpha[g] = al;
        }
      }
      consumer_sync();

      // acc = acc * alpha + P V over this stage's valid keys
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float al = s_alpha[g];
        acc[g][0] *= al;
        acc[g][1] *= al;
      }
      for (int kidx = vlo + kh; kidx < vhi; kidx += KH) {
        const uint32_t vv = *reinterpret_cast<const uint32_t*>(sV + kidx * L::ROW + dp * 4);
        const float v0 = bf16lo(vv), v1 = bf16hi(vv);
        const float* pk = sc + kidx * G;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pg = pk[g];
          acc[g][0] = fmaf(pg, v0, acc[g][0]);
          acc[g][1] = fmaf(pg, v1, acc[g][1]);
        }
      }
      consumer_sync();  // sc and the stage are free
      mbar_arrive(empty(st));
    }
    if (!ok) break;

    // reduce the KH key phases and write this unit's partials
    for (int x = 0; x < KH; ++x) {
      if (kh == x) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float* rr = red + g * D + 2 * dp;
          if (x == 0) {
            rr[0] = acc[g][0];
            rr[1] = acc[g][1];
          } else {
            rr[0] += acc[g][0];
            rr[1] += acc[g][1];
          }
        }
      }
      consumer_sync();
    }
    float* pa = p.part_acc + static_cast<int64_t>(u) * G * D;
    for (int i = tid; i < G * D; i += kConsumers) pa[i] = red[i];
    if (tid < G) {
      p.part_ml[(static_cast<int64_t>(u) * G + tid) * 2 + 0] = s_m[tid];
      p.part_ml[(static_cast<int64_t>(u) * G + tid) * 2 + 1] = s_l[tid];
    }
    consumer_sync();
    if (tid < G) {
      s_m[tid] = -INFINITY;
      s_l[tid] = 0.f;
    }
    consumer_sync();
  }
}

// One block per (sequence, KV head); warp g merges query head g's chunks.
template <int D, int G>
__global__ void __launch_bounds__(G * 32) decode_combine_kernel(const DecodeParams p) {
  constexpr int PER = D / 32;
  const DecodePair pr = p.pairs[blockIdx.x];
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float M = -INFINITY;
  for (int c = 0; c < pr.n_units; ++c)
    M = fmaxf(M, p.part_ml[(static_cast<int64_t>(pr.unit0 + c) * G + g) * 2]);
  float Lsum = 0.f, acc[PER];
#pragma unroll
  for (int x = 0; x < PER; ++x) acc[x] = 0.f;
  for (int c = 0; c < pr.n_units; ++c) {
    const int64_t uu = pr.unit0 + c;
    const float m = p.part_ml[(uu * G + g) * 2];
    const float l = p.part_ml[(uu * G + g) * 2 + 1];
    const float w = ex2(m - M);
    Lsum = fmaf(w, l, Lsum);
    const float* a = p.part_acc + (uu * G + g) * D;
#pragma unroll
    for (int x = 0; x < PER; ++x) acc[x] = fmaf(w, a[lane + 32 * x], acc[x]);
  }
  const float inv = 1.f / Lsum;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o) +
                     (static_cast<int64_t>(pr.req) * p.hq + pr.head * G + g) * D;
#pragma unroll
  for (int x = 0; x < PER; ++x) o[lane + 32 * x] = __float2bfloat16_rn(acc[x] * inv);
}

template <int D, int G>
static cudaError_t launch_dg(const DecodeParams& p, int grid, cudaStream_t s) {
  using L = DLayout<D, G>;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
  if (e != cudaSuccess) return e;
  decode_split_kernel<D, G><<<grid, kThreadsSplit, L::BYTES, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<D, G><<<p.n_pairs, G * 32, 0, s>>>(p);
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

cudaError_t launch_decode(const DecodeParams& p, int head_dim, int grid, cudaStream_t s) {
  return head_dim == 64 ? launch_d<64>(p, grid, s) : launch_d<128>(p, grid, s);
}

}  // namespace skv
