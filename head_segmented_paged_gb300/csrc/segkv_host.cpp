// Host side of segkv: segment allocator and page-table builder, work
// planners for the kernels, the upload ring, and the C ABI (include/segkv.h).
//
// The page model follows the RedKnot summary page ("让 KV Cache「按头分家」"):
// section "头分类稀疏" (global heads keep the causal context, local heads a
// sliding window) and section "SegPagedAttention" (KV paged per (layer, head)
// segment, each head keeps only what it needs). Readings where the page is
// silent: window W includes the query; eviction is lazy and frees whole pages
// k with (k+1)P <= kept start; one pool, lowest free id first, K and V share
// an id; evictions before allocations, in (seq_ids order, head, page) order.
// All planning is host-only and never waits on the device.
#include <algorithm>
#include <cassert>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <functional>
#include <memory>
#include <new>
#include <queue>
#include <string>
#include <vector>

#include "../../include/segkv.h"
#include "segkv_internal.h"

using namespace skv;

namespace {

constexpr unsigned long long kTimeoutNs = 2000ull * 1000 * 1000;  // 2 s per wait
constexpr size_t kRingInitial = size_t(8) << 20;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// Pinned, device-mapped host staging buffer mirrored by a device buffer of
// the same size. Each call takes the next region, fills it on the host, has a
// small kernel copy it to the device (upload) and records an event after its
// own kernels; a region is reused only once its event has completed. The
// copy runs on the SMs: a copy-engine transfer would wait behind the caller's
// own large host-to-device copies and serialise them with the compute.
struct UploadRing {
  uint8_t* host = nullptr;
  uint8_t* hmap = nullptr;  // device address of the host buffer
  uint8_t* dev = nullptr;
  size_t cap = 0, head = 0;
  struct Chunk {
    size_t off, len;
    cudaEvent_t ev;
  };
  std::deque<Chunk> live;
  std::vector<cudaEvent_t> spare;

  cudaError_t init(size_t bytes) {
    cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&host), bytes, cudaHostAllocMapped);
    if (e != cudaSuccess) return e;
    e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&hmap), host, 0);
    if (e != cudaSuccess) return e;
    e = cudaMalloc(reinterpret_cast<void**>(&dev), bytes);
    if (e != cudaSuccess) return e;
    cap = bytes;
    head = 0;
    return cudaSuccess;
  }
  void release() {
    for (auto& c : live) {
      cudaEventSynchronize(c.ev);
      cudaEventDestroy(c.ev);
    }
    live.clear();
    for (auto ev : spare) cudaEventDestroy(ev);
    spare.clear();
    if (host) cudaFreeHost(host);
    if (dev) cudaFree(dev);
    host = hmap = dev = nullptr;
    cap = head = 0;
  }
  void retire_front() {
    cudaEventSynchronize(live.front().ev);
    spare.push_back(live.front().ev);
    live.pop_front();
  }
  // Reserve len bytes; returns the offset or an error.
  cudaError_t reserve(size_t len, size_t* off) {
    len = align_up(std::max<size_t>(len, 256), 256);
    if (len > cap) {
      size_t ncap = std::max(len, cap * 2);
      while (!live.empty()) retire_front();
      cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) return e;
      for (auto ev : spare) cudaEventDestroy(ev);
      spare.clear();
      cudaFreeHost(host);
      cudaFree(dev);
      host = hmap = dev = nullptr;
      e = init(ncap);
      if (e != cudaSuccess) return e;
    }
    if (head + len > cap) head = 0;
    // the oldest live region is the next one in ring order
    while (!live.empty()) {
      const Chunk& c = live.front();
      const bool overlap = c.off < head + len && head < c.off + c.len;
      if (!overlap) break;
      retire_front();
    }
    *off = head;
    head += len;
    return cudaSuccess;
  }
  // Copy len bytes of a reserved region to the device, on stream s.
  cudaError_t upload(size_t off, size_t len, cudaStream_t s) {
    return launch_plan_copy(hmap + off, dev + off, len, s);
  }
  cudaError_t commit(size_t off, size_t len, cudaStream_t s) {
    cudaEvent_t ev;
    if (!spare.empty()) {
      ev = spare.back();
      spare.pop_back();
    } else {
      cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaEventRecord(ev, s);
    if (e != cudaSuccess) {
      spare.push_back(ev);
      return e;
    }
    live.push_back({off, align_up(std::max<size_t>(len, 256), 256), ev});
    return cudaSuccess;
  }
};

// Bump allocator over one staging region.
struct Pack {
  std::vector<uint8_t> buf;
  template <class T>
  size_t add(const T* data, size_t count) {
    size_t off = align_up(buf.size(), 16);
    buf.resize(off + sizeof(T) * count);
    if (count) std::memcpy(buf.data() + off, data, sizeof(T) * count);
    return off;
  }
};

// The least-loaded list of an LPT schedule: a winner tree over the lists'
// keys (load << 16 | list), its leaves padded to a power of two with the
// largest key, so the root is the least loaded list (the lowest index on
// ties). add() raises one list's load and redoes the path above its leaf,
// keeping the running minimum in a register. Lists < 65,536, loads < 2^47.
constexpr int kMaxPlanCtas = 65535;  // LeastLoaded packs a list index into 16 bits

// The free pages, handed out lowest id first. A bit per page and a bit per
// 64-page word that has any free page: push and pop touch one or two words,
// and the lowest free page is found from a cursor that only moves down when
// a lower page is freed, so a run of allocations costs O(1) per page.
class PagePool {
 public:
  void reset(int64_t n) {
    bits_.assign(static_cast<size_t>((n + 63) / 64), 0);
    sum_.assign((bits_.size() + 63) / 64, 0);
    count_ = 0;
    cursor_ = 0;
    for (int64_t i = 0; i < n; ++i) push(static_cast<int32_t>(i));
  }
  int64_t size() const { return count_; }
  void push(int32_t id) {
    const size_t w = static_cast<size_t>(id) >> 6;
    if (bits_[w] == 0) sum_[w >> 6] |= 1ull << (w & 63);
    bits_[w] |= 1ull << (id & 63);
    cursor_ = std::min(cursor_, w >> 6);
    ++count_;
  }
  int32_t take() {  // remove and return the lowest free page; the pool must not be empty
    while (sum_[cursor_] == 0) ++cursor_;
    const size_t w = cursor_ * 64 + static_cast<size_t>(__builtin_ctzll(sum_[cursor_]));
    const uint64_t b = bits_[w];
    bits_[w] = b & (b - 1);  // clear the lowest set bit
    if (bits_[w] == 0) sum_[cursor_] &= ~(1ull << (w & 63));
    --count_;
    return static_cast<int32_t>(w * 64 + static_cast<size_t>(__builtin_ctzll(b)));
  }
  // the n lowest free pages into out[0..n), ascending, a bitmap word at a time;
  // the pool must hold n pages
  void take(int32_t* out, int64_t n) {
    int64_t k = 0;
    while (k < n) {
      while (sum_[cursor_] == 0) ++cursor_;
      const size_t w = cursor_ * 64 + static_cast<size_t>(__builtin_ctzll(sum_[cursor_]));
      uint64_t b = bits_[w];
      while (b != 0 && k < n) {
        out[k++] = static_cast<int32_t>(w * 64 + static_cast<size_t>(__builtin_ctzll(b)));
        b &= b - 1;
      }
      bits_[w] = b;
      if (b == 0) sum_[cursor_] &= ~(1ull << (w & 63));
    }
    count_ -= n;
  }

 private:
  std::vector<uint64_t> bits_, sum_;
  int64_t count_ = 0;
  size_t cursor_ = 0;
};

class LeastLoaded {
 public:
  void reset(int lists) {
    assert(lists >= 1 && lists <= kMaxPlanCtas);
    leaves_ = 1;
    while (leaves_ < static_cast<size_t>(lists)) leaves_ <<= 1;
    tree_.assign(2 * leaves_, ~0ull);
    for (int c = 0; c < lists; ++c) tree_[leaves_ + c] = static_cast<uint64_t>(c);
    for (size_t i = leaves_ - 1; i >= 1; --i) tree_[i] = std::min(tree_[2 * i], tree_[2 * i + 1]);
  }
  int least() const { return static_cast<int>(tree_[1] & 0xffffu); }
  void add(int c, int64_t load) {
    uint64_t* t = tree_.data();
    size_t i = leaves_ + static_cast<size_t>(c);
    uint64_t v = t[i] + (static_cast<uint64_t>(load) << 16);
    t[i] = v;
    for (; i > 1; i >>= 1) {  // each node on the path: the smaller of its two children
      v = std::min(v, t[i ^ 1]);
      t[i >> 1] = v;
    }
  }

 private:
  std::vector<uint64_t> tree_;
  size_t leaves_ = 1;
};

}  // namespace

// One (sequence, KV head) key range of a decode call, and the plan cut from
// them. A handle keeps one plan and reuses its storage from call to call.
struct DecodeRange { int32_t req, head, lo, n, row, local; };
struct DecodePlan {
  std::vector<DecodeRange> ranges;
  std::vector<int64_t> keys;  // per range: its key count, n - lo
  std::vector<DecodeUnit> units;
  std::vector<int32_t> cta_begin;
  std::vector<int32_t> pair_unit0, pair_units;  // per range
  int grid = 0, rows = 0;
  bool mma = false;
};

// The prefill plan and its scratch; a handle keeps one and reuses its storage.
struct PrefillPlan {
  std::vector<PrefillUnit> units;  // in building order
  std::vector<PrefillUnit> claim;  // the plan: the order in which the kernel's CTAs claim units
  int grid = 0;                    // CTAs of the launch: min(units, CTAs asked for)
  std::vector<int32_t> count;
};

struct segkv {
  int L = 0, Hq = 0, Hkv = 0, D = 0, G = 0, P = 0, S = 0, max_len = 0, R = 0;
  int64_t num_pages = 0;
  float scale = 0.f;
  bool host_only = true;
  std::vector<uint8_t> cls;   // [L][Hkv]
  std::vector<int32_t> win;   // [L]
  void* kpool = nullptr;
  void* vpool = nullptr;

  // host page tables
  std::vector<int32_t> len;    // [L][S]
  std::vector<int32_t> start;  // [L][Hkv][S]
  std::vector<int32_t> table;  // [L][Hkv][S][R], -1 = not held
  PagePool free_ids;  // lowest id first

  // device
  int device = 0, num_sms = 0;
  int32_t* d_table = nullptr;
  int* d_status = nullptr;
  int* d_pair_cnt = nullptr;  // decode merge counters, [max_seqs * Hkv], kept at zero
  CUtensorMap tm_k{}, tm_v{};
  UploadRing ring;
  PlanBlob blob;  // staging for plans small enough to travel as kernel parameters
  int debug = 0;
  bool window_fa = false;  // win[] holds W+1 for the FlashAttention convention
  int64_t upload_bytes = 0;
  DecodePlan dplan;   // the last decode plan (storage reused)
  PrefillPlan pplan;  // the last prefill plan (storage reused)
  Pack pack;          // staging of a plan upload (storage reused)
  std::vector<XferHead> xfer_heads;  // a transfer's plan (storage reused)
  std::vector<int32_t> xfer_pages;
  std::string err;

  size_t seg(int l, int h, int b) const { return (static_cast<size_t>(l) * Hkv + h) * S + b; }
  size_t lidx(int l, int b) const { return static_cast<size_t>(l) * S + b; }
  bool local(int l, int h) const { return cls[l * Hkv + h] != SEGKV_GLOBAL; }
  int32_t* row(int l, int h, int b) { return table.data() + seg(l, h, b) * R; }
};

namespace {

std::string g_create_error;

int fail(segkv* h, int code, const char* fmt, ...) {
  char msg[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(msg, sizeof msg, fmt, ap);
  va_end(ap);
  if (h) h->err = msg; else g_create_error = msg;
  return code;
}

int cuda_fail(segkv* h, cudaError_t e, const char* what) {
  return fail(h, SEGKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool ids_valid(const segkv* h, const int32_t* ids, int n) {
  if (n < 0 || (n > 0 && ids == nullptr)) return false;
  std::vector<uint8_t> seen(h->S, 0);
  for (int i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= h->S || seen[ids[i]]) return false;
    seen[ids[i]] = 1;
  }
  return true;
}

// First position a head must keep for queries starting at q0.
int32_t needed_start(const segkv* h, int l, int hd, int32_t cur, int64_t q0) {
  if (!h->local(l, hd)) return cur;
  int64_t need = q0 - h->win[l] + 1;
  if (need < 0) need = 0;
  return need > cur ? static_cast<int32_t>(need) : cur;
}

// Free every held page k with (k+1) P <= new_s.
void evict_below(segkv* h, int l, int hd, int b, int32_t new_s) {
  int32_t* r = h->row(l, hd, b);
  const int32_t old_s = h->start[h->seg(l, hd, b)];
  const int32_t n = h->len[h->lidx(l, b)];
  if (n > 0) {
    const int k_first = old_s / h->P;
    const int k_stop = new_s / h->P;  // pages below this are wholly before new_s
    for (int k = k_first; k < k_stop && k < h->R; ++k)
      if (r[k] >= 0) {
        h->free_ids.push(r[k]);
        r[k] = -1;
      }
  }
  h->start[h->seg(l, hd, b)] = new_s;
}

int count_evictions(const segkv* h, int l, int hd, int b, int32_t new_s) {
  const int32_t old_s = h->start[h->seg(l, hd, b)];
  const int32_t n = h->len[h->lidx(l, b)];
  if (n == 0) return 0;
  const int32_t* r = h->table.data() + h->seg(l, hd, b) * h->R;
  int c = 0;
  for (int k = old_s / h->P; k < new_s / h->P && k < h->R; ++k) c += r[k] >= 0;
  return c;
}

CUresult encode_2d(CUtensorMap* m, void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

extern "C" {

int segkv_create(segkv_t* out, int num_layers, int num_q_heads, int num_kv_heads, int head_dim,
                 const uint8_t* head_class, const int32_t* window, int page_size, int max_seqs,
                 int max_seq_len, void* k_pool, void* v_pool, int64_t num_pages,
                 float softmax_scale) {
  if (!out) return fail(nullptr, SEGKV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (num_layers <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
    return fail(nullptr, SEGKV_ERR_INVALID_ARG, "bad head counts");
  const int G = num_q_heads / num_kv_heads;
  if (G > 16 || 128 % G) return fail(nullptr, SEGKV_ERR_INVALID_ARG, "G=%d must divide 16", G);
  if (head_dim != 64 && head_dim != 128)
    return fail(nullptr, SEGKV_ERR_INVALID_ARG, "head_dim must be 64 or 128");
  if (page_size < 8 || page_size % 8 || (page_size < 128 && 128 % page_size) ||
      (page_size > 128 && page_size % 128))
    return fail(nullptr, SEGKV_ERR_INVALID_ARG, "bad page_size %d", page_size);
  if (max_seqs <= 0 || max_seq_len <= 0 || num_pages <= 0 || !head_class || !window)
    return fail(nullptr, SEGKV_ERR_INVALID_ARG, "bad sizes");
  if (num_pages * page_size >= (int64_t(1) << 31) - 256 || num_pages >= (int64_t(1) << 31))
    return fail(nullptr, SEGKV_ERR_INVALID_ARG, "pool too large for 32-bit rows");
  if ((k_pool == nullptr) != (v_pool == nullptr))
    return fail(nullptr, SEGKV_ERR_INVALID_ARG, "k_pool and v_pool must both be set or NULL");
  for (int l = 0; l < num_layers; ++l) {
    if (window[l] < 1) return fail(nullptr, SEGKV_ERR_INVALID_ARG, "window[%d] < 1", l);
    for (int x = 0; x < num_kv_heads; ++x)
      if (head_class[l * num_kv_heads + x] > 1)
        return fail(nullptr, SEGKV_ERR_INVALID_ARG, "bad head_class");
  }
  const int64_t R = (static_cast<int64_t>(max_seq_len) + page_size - 1) / page_size;
  const int64_t entries = int64_t(num_layers) * num_kv_heads * max_seqs * R;
  if (entries > (int64_t(1) << 33)) return fail(nullptr, SEGKV_ERR_INVALID_ARG, "table too large");

  std::unique_ptr<segkv> h(new (std::nothrow) segkv());
  if (!h) return fail(nullptr, SEGKV_ERR_INVALID_ARG, "out of host memory");
  h->L = num_layers; h->Hq = num_q_heads; h->Hkv = num_kv_heads; h->D = head_dim; h->G = G;
  h->P = page_size; h->S = max_seqs; h->max_len = max_seq_len; h->R = static_cast<int>(R);
  h->num_pages = num_pages;
  h->scale = softmax_scale > 0.f ? softmax_scale : 1.f / std::sqrt(static_cast<float>(head_dim));
  h->cls.assign(head_class, head_class + num_layers * num_kv_heads);
  h->win.assign(window, window + num_layers);
  h->len.assign(static_cast<size_t>(num_layers) * max_seqs, 0);
  h->start.assign(static_cast<size_t>(num_layers) * num_kv_heads * max_seqs, 0);
  h->table.assign(static_cast<size_t>(entries), -1);
  h->free_ids.reset(num_pages);
  h->host_only = (k_pool == nullptr);
  h->kpool = k_pool;
  h->vpool = v_pool;
  if (!h->host_only) {
    if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 15)
      return fail(nullptr, SEGKV_ERR_INVALID_ARG, "pools must be 16-byte aligned");
    if (!encode_fn()) return fail(nullptr, SEGKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDevice");
    e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaDeviceGetAttribute");
    e = cudaMalloc(reinterpret_cast<void**>(&h->d_table), sizeof(int32_t) * entries);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaMalloc(table)");
    e = cudaMemset(h->d_table, 0xff, sizeof(int32_t) * entries);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&h->d_status), sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, sizeof(int));
    const size_t cnt_bytes = sizeof(int) * static_cast<size_t>(max_seqs) * num_kv_heads;
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&h->d_pair_cnt), cnt_bytes);
    if (e == cudaSuccess) e = cudaMemset(h->d_pair_cnt, 0, cnt_bytes);
    if (e == cudaSuccess) e = h->ring.init(kRingInitial);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      h->ring.release();
      cudaFree(h->d_table);
      cudaFree(h->d_status);
      cudaFree(h->d_pair_cnt);
      return cuda_fail(nullptr, e, "device setup");
    }
    const uint64_t rows = static_cast<uint64_t>(num_pages) * page_size;
    const uint32_t box_rows = page_size <= 128 ? page_size : 128;
    if (encode_2d(&h->tm_k, k_pool, head_dim, rows, box_rows) != CUDA_SUCCESS ||
        encode_2d(&h->tm_v, v_pool, head_dim, rows, box_rows) != CUDA_SUCCESS) {
      h->ring.release();
      cudaFree(h->d_table);
      cudaFree(h->d_status);
      cudaFree(h->d_pair_cnt);
      return fail(nullptr, SEGKV_ERR_CUDA, "tensor map encode failed for the pools");
    }
  }
  *out = h.release();
  return SEGKV_OK;
}

int segkv_destroy(segkv_t h) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (!h->host_only) {
    cudaDeviceSynchronize();
    h->ring.release();
    cudaFree(h->d_table);
    cudaFree(h->d_status);
    cudaFree(h->d_pair_cnt);
  }
  delete h;
  return SEGKV_OK;
}

const char* segkv_last_error(segkv_t h) {
  return h ? h->err.c_str() : g_create_error.c_str();
}

int segkv_exp2_check(const float* x, float* y_poly, float* y_mufu, int n, segkv_stream_t stream) {
  if (n < 0 || (n > 0 && (!x || !y_poly || !y_mufu))) return SEGKV_ERR_INVALID_ARG;
  if (n == 0) return SEGKV_OK;
  const cudaError_t e = skv::launch_exp2_check(x, y_poly, y_mufu, n, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SEGKV_OK : SEGKV_ERR_CUDA;
}

int segkv_set_debug(segkv_t h, int flags) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  h->debug = flags;
  return SEGKV_OK;
}

// ---------------------------------------------------------------- append
int segkv_append(segkv_t h, int layer, const void* k, const void* v, const int32_t* cu_seqlens,
                 const int32_t* seq_ids, int n, segkv_stream_t stream) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->L) return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer %d", layer);
  if (!ids_valid(h, seq_ids, n)) return fail(h, SEGKV_ERR_INVALID_ARG, "bad seq_ids");
  if (n == 0) return SEGKV_OK;
  if (!cu_seqlens || cu_seqlens[0] != 0) return fail(h, SEGKV_ERR_INVALID_ARG, "cu_seqlens[0] != 0");
  for (int i = 0; i < n; ++i) {
    const int64_t T = int64_t(cu_seqlens[i + 1]) - cu_seqlens[i];
    if (T < 0) return fail(h, SEGKV_ERR_INVALID_ARG, "cu_seqlens decreases at %d", i);
    if (h->len[h->lidx(layer, seq_ids[i])] + T > h->max_len)
      return fail(h, SEGKV_ERR_INVALID_ARG, "seq %d would exceed max_seq_len", seq_ids[i]);
  }
  const int64_t total = cu_seqlens[n];
  if (total > 0 && !h->host_only && (!k || !v))
    return fail(h, SEGKV_ERR_INVALID_ARG, "k/v are NULL");

  // plan: evictions (all), then allocations, in (seq_ids order, head, page) order
  std::vector<int32_t> new_s(static_cast<size_t>(n) * h->Hkv);
  int64_t freed = 0, need = 0;
  for (int i = 0; i < n; ++i) {
    const int b = seq_ids[i];
    const int32_t a = h->len[h->lidx(layer, b)];
    const int32_t T = cu_seqlens[i + 1] - cu_seqlens[i];
    for (int hd = 0; hd < h->Hkv; ++hd) {
      const int32_t s0 = h->start[h->seg(layer, hd, b)];
      const int32_t ns = needed_start(h, layer, hd, s0, a);
      new_s[i * h->Hkv + hd] = ns;
      freed += count_evictions(h, layer, hd, b, ns);
      if (T > 0) {
        const int32_t* r = h->table.data() + h->seg(layer, hd, b) * h->R;
        for (int kk = a / h->P; kk <= (a + T - 1) / h->P; ++kk) need += r[kk] < 0;
      }
    }
  }
  if (static_cast<int64_t>(h->free_ids.size()) + freed < need)
    return fail(h, SEGKV_ERR_OUT_OF_PAGES, "append needs %lld pages, %lld free after eviction",
                static_cast<long long>(need),
                static_cast<long long>(h->free_ids.size() + freed));

  for (int i = 0; i < n; ++i)
    for (int hd = 0; hd < h->Hkv; ++hd)
      evict_below(h, layer, hd, seq_ids[i], new_s[i * h->Hkv + hd]);

  std::vector<AppendSeq> seqs;
  std::vector<AppendTile> tiles;
  std::vector<int32_t> plist;
  std::vector<int64_t> tidx;
  for (int i = 0; i < n; ++i) {
    const int b = seq_ids[i];
    const int32_t a = h->len[h->lidx(layer, b)];
    const int32_t T = cu_seqlens[i + 1] - cu_seqlens[i];
    if (T == 0) continue;
    AppendSeq sq{};
    sq.tok0 = cu_seqlens[i];
    sq.pos0 = a;
    sq.first_k = a / h->P;
    sq.n_pages = (a + T - 1) / h->P - sq.first_k + 1;
    sq.list_off = static_cast<int32_t>(plist.size());
    for (int hd = 0; hd < h->Hkv; ++hd) {
      int32_t* r = h->row(layer, hd, b);
      for (int kk = sq.first_k; kk < sq.first_k + sq.n_pages; ++kk) {
        if (r[kk] < 0) r[kk] = h->free_ids.take();
        plist.push_back(r[kk]);
        tidx.push_back(static_cast<int64_t>(h->seg(layer, hd, b)) * h->R + kk);
      }
    }
    const int seq_index = static_cast<int>(seqs.size());
    seqs.push_back(sq);
    constexpr int kTileTok = 16;
    for (int t0 = 0; t0 < T; t0 += kTileTok)
      tiles.push_back({seq_index, sq.tok0 + t0, std::min(kTileTok, T - t0), 0});
  }
  for (int i = 0; i < n; ++i)
    h->len[h->lidx(layer, seq_ids[i])] += cu_seqlens[i + 1] - cu_seqlens[i];

  if (h->host_only || tiles.empty()) return SEGKV_OK;

  Pack pk;
  const size_t o_seq = pk.add(seqs.data(), seqs.size());
  const size_t o_tile = pk.add(tiles.data(), tiles.size());
  const size_t o_pl = pk.add(plist.data(), plist.size());
  const size_t o_ti = pk.add(tidx.data(), tidx.size());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool inl = pk.buf.size() <= sizeof(AppendBlob);
  size_t off = 0;
  uintptr_t d = 0;  // device address of the plan; 0 (offsets alone) when it is inline
  cudaError_t e;
  if (inl) {
    std::memcpy(h->blob.data, pk.buf.data(), pk.buf.size());
  } else {
    e = h->ring.reserve(pk.buf.size(), &off);
    if (e != cudaSuccess) return cuda_fail(h, e, "upload ring");
    std::memcpy(h->ring.host + off, pk.buf.data(), pk.buf.size());
    e = h->ring.upload(off, pk.buf.size(), s);
    if (e != cudaSuccess) return cuda_fail(h, e, "plan upload (append)");
    d = reinterpret_cast<uintptr_t>(h->ring.dev + off);
  }
  h->upload_bytes += static_cast<int64_t>(pk.buf.size());
  AppendParams p{};
  p.plan_inline = inl ? 1 : 0;
  p.k = static_cast<const uint4*>(k);
  p.v = static_cast<const uint4*>(v);
  p.kpool = static_cast<uint4*>(h->kpool);
  p.vpool = static_cast<uint4*>(h->vpool);
  p.seqs = reinterpret_cast<const AppendSeq*>(d + o_seq);
  p.tiles = reinterpret_cast<const AppendTile*>(d + o_tile);
  p.page_list = reinterpret_cast<const int32_t*>(d + o_pl);
  p.table_idx = reinterpret_cast<const int64_t*>(d + o_ti);
  p.table = h->d_table;
  p.n_tiles = static_cast<int>(tiles.size());
  p.n_entries = static_cast<int>(plist.size());
  p.hkv = h->Hkv;
  p.vec_per_row = h->D / 8;
  p.page_size = h->P;
  const int grid = static_cast<int>(std::min<int64_t>(tiles.size(), int64_t(h->num_sms) * 8));
  e = launch_append(p, inl ? reinterpret_cast<const AppendBlob*>(&h->blob) : nullptr,
                    std::max(grid, 1), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "append kernel launch");
  if (!inl) {
    e = h->ring.commit(off, pk.buf.size(), s);
    if (e != cudaSuccess) return cuda_fail(h, e, "event record");
  }
  return SEGKV_OK;
}

// ---------------------------------------------------------------- prefill
// Positions and kept keys of a prefill call (host): every query position lies
// in its sequence, and every key it sees is still kept.
static int prefill_validate(segkv* h, int layer, const int32_t* cu_seqlens, const int32_t* q_pos,
                            const int32_t* seq_ids, int n) {
  const int W = h->win[layer];
  for (int i = 0; i < n; ++i) {
    const int b = seq_ids[i];
    const int32_t nlen = h->len[h->lidx(layer, b)];
    if (cu_seqlens[i + 1] == cu_seqlens[i]) continue;
    // positions in range; the lowest one needs the oldest keys
    int32_t pmin = q_pos[cu_seqlens[i]];
    int32_t tmin = cu_seqlens[i];
    for (int32_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) {
      const int32_t p = q_pos[t];
      if (p < 0 || p >= nlen)
        return fail(h, SEGKV_ERR_INVALID_ARG, "q_pos[%d]=%d outside [0,%d) of seq %d", t, p, nlen, b);
      if (p < pmin) {
        pmin = p;
        tmin = t;
      }
    }
    (void)tmin;
    for (int hd = 0; hd < h->Hkv; ++hd) {
      const int32_t need = h->local(layer, hd) ? std::max(0, pmin - W + 1) : 0;
      if (need < h->start[h->seg(layer, hd, b)])
        return fail(h, SEGKV_ERR_EVICTED, "seq %d head %d: key %d already evicted", b, hd, need);
    }
  }
  return SEGKV_OK;
}

// The prefill work plan (host): units of one KV head x the Q tiles of a
// chunk of tokens, in the order the kernel's CTAs claim them, and the grid
// for `ctas` CTAs, into h->pplan (claim, grid).
static void prefill_plan(segkv* h, int layer, const int32_t* cu_seqlens, const int32_t* q_pos,
                         const int32_t* seq_ids, int n, int ctas) {
  PrefillPlan& P = h->pplan;
  const int W = h->win[layer];
  // units: (KV head, two Q tiles of 128/G tokens each)
  const int unit_tok = prefill_unit_tokens(h->G);
  std::vector<PrefillUnit>& units = P.units;
  units.clear();
  {
    int64_t count = 0;
    for (int i = 0; i < n; ++i) count += (cu_seqlens[i + 1] - cu_seqlens[i] + unit_tok - 1) / unit_tok;
    units.reserve(static_cast<size_t>(count) * h->Hkv);
  }
  for (int i = 0; i < n; ++i) {
    const int b = seq_ids[i];
    const int32_t nlen = h->len[h->lidx(layer, b)];
    for (int32_t t0 = cu_seqlens[i]; t0 < cu_seqlens[i + 1]; t0 += unit_tok) {
      const int32_t t1 = std::min<int32_t>(t0 + unit_tok, cu_seqlens[i + 1]);
      int32_t pmin = q_pos[t0], pmax = q_pos[t0];
      bool consecutive = true;
      for (int32_t t = t0; t < t1; ++t) {
        pmin = std::min(pmin, q_pos[t]);
        pmax = std::max(pmax, q_pos[t]);
        consecutive = consecutive && q_pos[t] == q_pos[t0] + (t - t0);
      }
      for (int hd = 0; hd < h->Hkv; ++hd) {
        PrefillUnit u{};
        u.tok0 = t0;
        u.ntok = t1 - t0;
        u.head = hd;
        u.local = h->local(layer, hd) ? 1 : 0;
        u.klo = u.local ? std::max(0, pmin - W + 1) : 0;
        u.khi = pmax;
        u.kt0 = u.klo / kKeyTile;
        u.kt1 = u.khi / kKeyTile;
        u.vlo = h->start[h->seg(layer, hd, b)];
        u.vhi = nlen - 1;
        u.table_row = static_cast<int32_t>(h->seg(layer, hd, b));
        u.pos0 = consecutive ? q_pos[t0] : -1;
        units.push_back(u);
      }
    }
  }
  const size_t nu = units.size();
  // Claim order: descending key tiles, stable (a counting sort on the tile
  // count). The kernel's CTA c runs unit c first; each CTA that finishes a
  // unit claims the next unit of this order, so the longest units start
  // first and every CTA stays busy until the list runs out, whatever the
  // speed of its SM.
  int32_t max_tiles = 0;
  for (const PrefillUnit& u : units) max_tiles = std::max(max_tiles, u.kt1 - u.kt0);
  std::vector<int32_t>& start = P.count;
  start.assign(static_cast<size_t>(max_tiles) + 2, 0);
  for (const PrefillUnit& u : units) ++start[max_tiles - (u.kt1 - u.kt0) + 1];
  for (size_t c = 1; c < start.size(); ++c) start[c] += start[c - 1];
  std::vector<PrefillUnit>& claim = P.claim;
  claim.resize(nu);
  for (size_t x = 0; x < nu; ++x) claim[start[max_tiles - (units[x].kt1 - units[x].kt0)]++] = units[x];
  P.grid = static_cast<int>(std::min<int64_t>(static_cast<int64_t>(nu), ctas));
}

int segkv_prefill_attn(segkv_t h, int layer, const void* q, const int32_t* cu_seqlens,
                       const int32_t* q_pos, const int32_t* seq_ids, int n, void* o, float* lse,
                       void* workspace, size_t workspace_bytes, segkv_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (h->host_only) return fail(h, SEGKV_ERR_INVALID_ARG, "host-only handle has no pools");
  if (layer < 0 || layer >= h->L) return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer %d", layer);
  if (!ids_valid(h, seq_ids, n)) return fail(h, SEGKV_ERR_INVALID_ARG, "bad seq_ids");
  if (n == 0) return SEGKV_OK;
  if (!cu_seqlens || cu_seqlens[0] != 0) return fail(h, SEGKV_ERR_INVALID_ARG, "cu_seqlens[0] != 0");
  for (int i = 0; i < n; ++i)
    if (cu_seqlens[i + 1] < cu_seqlens[i])
      return fail(h, SEGKV_ERR_INVALID_ARG, "cu_seqlens decreases at %d", i);
  const int64_t total = cu_seqlens[n];
  if (total == 0) return SEGKV_OK;
  if (!q || !o || !q_pos) return fail(h, SEGKV_ERR_INVALID_ARG, "q/o/q_pos NULL");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(o)) & 15)
    return fail(h, SEGKV_ERR_INVALID_ARG, "q and o must be 16-byte aligned");
  {
    const int vrc = prefill_validate(h, layer, cu_seqlens, q_pos, seq_ids, n);
    if (vrc != SEGKV_OK) return vrc;
  }
  const int W = h->win[layer];
  const int tpt = kRowsPerTile / h->G;
  prefill_plan(h, layer, cu_seqlens, q_pos, seq_ids, n, h->num_sms);
  const std::vector<PrefillUnit>& claim = h->pplan.claim;
  const int grid = h->pplan.grid;
  const size_t n_units = claim.size();

  Pack& pk = h->pack;
  pk.buf.clear();
  const size_t o_units = pk.add(claim.data(), claim.size());
  const int32_t zero = 0;  // the claim counter, fresh for every launch
  const size_t o_next = pk.add(&zero, 1);
  const size_t o_pos = pk.add(q_pos, static_cast<size_t>(total));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  size_t off;
  cudaError_t e = h->ring.reserve(pk.buf.size(), &off);
  if (e != cudaSuccess) return cuda_fail(h, e, "upload ring");
  std::memcpy(h->ring.host + off, pk.buf.data(), pk.buf.size());
  e = h->ring.upload(off, pk.buf.size(), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "plan upload (prefill)");
  h->upload_bytes += static_cast<int64_t>(pk.buf.size());

  CUtensorMap tq, to;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(h->D), static_cast<cuuint64_t>(h->Hq),
                          static_cast<cuuint64_t>(total)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(h->D) * 2,
                             static_cast<cuuint64_t>(h->Hq) * h->D * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(h->G), static_cast<cuuint32_t>(tpt)};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode_fn()(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return fail(h, SEGKV_ERR_CUDA, "tensor map encode failed for q");
    // O has Q's shape; a box is one softmax warp's 32 rows (32 / G tokens)
    cuuint32_t obox[3] = {64, static_cast<cuuint32_t>(h->G), static_cast<cuuint32_t>(32 / h->G)};
    if (encode_fn()(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o, dims, strides, obox, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return fail(h, SEGKV_ERR_CUDA, "tensor map encode failed for o");
  }
  uint8_t* d = h->ring.dev + off;
  PrefillParams p{};
  p.units = reinterpret_cast<const PrefillUnit*>(d + o_units);
  p.next_unit = reinterpret_cast<int*>(d + o_next);
  p.q_pos = reinterpret_cast<const int32_t*>(d + o_pos);
  p.table = h->d_table;
  p.o = o;
  p.lse = lse;
  p.total_q = total;
  p.n_units = static_cast<int>(n_units);
  p.R = h->R;
  p.hq = h->Hq;
  p.G = h->G;
  p.tpt = tpt;
  p.window = W;
  p.page_size = h->P;
  p.oob_row = static_cast<int>(h->num_pages * h->P);
  p.scale_log2 = h->scale * 1.4426950408889634f;
  p.status = h->d_status;
  p.debug = h->debug;
  p.timeout_ns = kTimeoutNs;
  h->debug = 0;
  e = launch_prefill(p, tq, h->tm_k, h->tm_v, to, h->D, grid, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "prefill kernel launch");
  e = h->ring.commit(off, pk.buf.size(), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "event record");
  return SEGKV_OK;
}

int segkv_plan_prefill(segkv_t h, int layer, const int32_t* cu_seqlens, const int32_t* q_pos,
                       const int32_t* seq_ids, int n, int num_ctas, int32_t* units_out, int max_units,
                       int* n_units, int* n_ctas) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->L) return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer %d", layer);
  if (n < 0 || max_units < 0 || !n_units || !n_ctas)
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad n or output sizes");
  if (!ids_valid(h, seq_ids, n)) return fail(h, SEGKV_ERR_INVALID_ARG, "bad seq_ids");
  *n_units = 0;
  *n_ctas = 0;
  if (n == 0) return SEGKV_OK;
  if (!cu_seqlens || cu_seqlens[0] != 0) return fail(h, SEGKV_ERR_INVALID_ARG, "cu_seqlens[0] != 0");
  for (int i = 0; i < n; ++i)
    if (cu_seqlens[i + 1] < cu_seqlens[i])
      return fail(h, SEGKV_ERR_INVALID_ARG, "cu_seqlens decreases at %d", i);
  if (cu_seqlens[n] == 0) return SEGKV_OK;
  if (!q_pos) return fail(h, SEGKV_ERR_INVALID_ARG, "q_pos NULL");
  const int vrc = prefill_validate(h, layer, cu_seqlens, q_pos, seq_ids, n);
  if (vrc != SEGKV_OK) return vrc;
  if (num_ctas > kMaxPlanCtas)
    return fail(h, SEGKV_ERR_INVALID_ARG, "num_ctas %d above %d", num_ctas, kMaxPlanCtas);
  const int ctas = num_ctas > 0 ? num_ctas : (h->num_sms > 0 ? h->num_sms : 1);
  prefill_plan(h, layer, cu_seqlens, q_pos, seq_ids, n, ctas);
  const std::vector<PrefillUnit>& claim = h->pplan.claim;
  *n_units = static_cast<int>(claim.size());
  *n_ctas = h->pplan.grid;
  if (*n_units > max_units || (max_units && !units_out))
    return fail(h, SEGKV_ERR_INVALID_ARG, "plan needs %d units", *n_units);
  for (size_t x = 0; x < claim.size(); ++x) {
    const PrefillUnit& u = claim[x];
    int32_t* o = units_out + 8 * x;
    o[0] = u.tok0;
    o[1] = u.ntok;
    o[2] = u.head;
    o[3] = u.local;
    o[4] = u.kt0;
    o[5] = u.kt1;
    o[6] = u.klo;
    o[7] = u.khi;
  }
  return SEGKV_OK;
}

// ---------------------------------------------------------------- decode
// Split units: at most one per (sequence, KV head) pair plus one per CTA slice
// boundary.
static int decode_max_grid(const segkv* h) { return h->num_sms > 0 ? 2 * h->num_sms : 1024; }

// rows = query rows per KV head (T * G)
static size_t decode_ws_bytes(const segkv* h, int64_t units, int rows, size_t* acc_bytes,
                              size_t* ml_bytes) {
  *acc_bytes = align_up(static_cast<size_t>(units) * rows * h->D * 4, 256);
  *ml_bytes = align_up(static_cast<size_t>(units) * rows * 2 * 4, 256);
  return *acc_bytes + *ml_bytes;
}

// The split-KV decode kernel takes up to 16 query rows per KV head.
static bool decode_kernel_rows(int rows) {
  return rows == 1 || rows == 2 || rows == 4 || rows == 8 || rows == 16;
}

int segkv_workspace_size(segkv_t h, int kind, int64_t n_tokens, int n_seqs, size_t* bytes) {
  if (!h || !bytes || n_seqs < 0 || n_tokens < 0) return SEGKV_ERR_INVALID_ARG;
  if (kind == SEGKV_WS_PREFILL) {
    *bytes = 0;
    return SEGKV_OK;
  }
  if (kind != SEGKV_WS_DECODE) return fail(h, SEGKV_ERR_INVALID_ARG, "bad workspace kind");
  // T = n_tokens / n_seqs query tokens per sequence (at least 1)
  const int64_t T = n_seqs > 0 ? std::max<int64_t>(1, (n_tokens + n_seqs - 1) / n_seqs) : 1;
  const int64_t rows = T * h->G;
  if (rows > 16 || !decode_kernel_rows(static_cast<int>(rows))) {
    *bytes = 0;  // served by the prefill kernel, which needs none
    return SEGKV_OK;
  }
  const int64_t pairs = int64_t(n_seqs) * h->Hkv;
  size_t a, m;
  *bytes = decode_ws_bytes(h, pairs + decode_max_grid(h), static_cast<int>(rows), &a, &m);
  return SEGKV_OK;
}

// Tensor-core decode (8 or 16 query rows per KV head, D = 128) of a plan made
// by decode_core, plus the merge of split pairs.
static int decode_mma_launch(segkv* h, int layer, const void* q, int T, int n, void* o, float* lse,
                             const std::vector<DecodeUnit>& units,
                             const std::vector<int32_t>& cta_begin,
                             const std::vector<DecodeCombine>& comb, void* workspace,
                             size_t acc_bytes, int grid, cudaStream_t s) {
  Pack pk;
  const size_t o_units = pk.add(units.data(), units.size());
  const size_t o_cta = pk.add(cta_begin.data(), cta_begin.size());
  const size_t o_comb = pk.add(comb.data(), comb.size());
  const bool inl = pk.buf.size() <= sizeof(PlanBlob);
  size_t off_ring = 0;
  uintptr_t d = 0;  // device address of the plan; 0 (offsets alone) when it is inline
  cudaError_t e;
  if (inl) {
    std::memcpy(h->blob.data, pk.buf.data(), pk.buf.size());
  } else {
    e = h->ring.reserve(pk.buf.size(), &off_ring);
    if (e != cudaSuccess) return cuda_fail(h, e, "upload ring");
    std::memcpy(h->ring.host + off_ring, pk.buf.data(), pk.buf.size());
    e = h->ring.upload(off_ring, pk.buf.size(), s);
    if (e != cudaSuccess) return cuda_fail(h, e, "plan upload (decode)");
    d = reinterpret_cast<uintptr_t>(h->ring.dev + off_ring);
  }
  h->upload_bytes += static_cast<int64_t>(pk.buf.size());
  const int rows = T * h->G;
  CUtensorMap tq;  // the T tokens x Gm heads of one (sequence, KV head): box {64, Gm, T}
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(h->D), static_cast<cuuint64_t>(h->Hq),
                          static_cast<cuuint64_t>(n) * T};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(h->D) * 2,
                             static_cast<cuuint64_t>(h->Hq) * h->D * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(h->G), static_cast<cuuint32_t>(T)};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode_fn()(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return fail(h, SEGKV_ERR_CUDA, "tensor map encode failed for q");
  }
  DecodeMmaParams p{};
  p.units = reinterpret_cast<const DecodeUnit*>(d + o_units);
  p.cta_begin = reinterpret_cast<const int32_t*>(d + o_cta);
  p.combine = reinterpret_cast<const DecodeCombine*>(d + o_comb);
  p.plan_inline = inl ? 1 : 0;
  p.n_combine = static_cast<int>(comb.size());
  p.o = o;
  p.lse = lse;
  p.table = h->d_table;
  p.part_acc = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + acc_bytes);
  p.n_rows = n * T;
  p.R = h->R;
  p.hq = h->Hq;
  p.hkv = h->Hkv;
  p.page_size = h->P;
  p.R_rows = rows;
  p.T = T;
  p.Gm = h->G;
  p.window = h->win[layer];
  p.oob_row = static_cast<int>(h->num_pages * h->P);
  p.scale_log2 = h->scale * 1.4426950408889634f;
  p.status = h->d_status;
  p.timeout_ns = kTimeoutNs;
  e = launch_decode_mma(p, inl ? &h->blob : nullptr, tq, h->tm_k, h->tm_v, grid, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "decode kernel launch");
  if (!inl) {
    e = h->ring.commit(off_ring, pk.buf.size(), s);
    if (e != cudaSuccess) return cuda_fail(h, e, "event record");
  }
  return SEGKV_OK;
}

// Whether the greedy stream-K cut of decode_plan, with per-CTA budget B, fits
// in max_grid CTAs. The same walk as the cut that emits the units, over the
// ranges' key counts alone, given up as soon as the grid is full.
static bool decode_cut_fits(const int64_t* keys, int64_t nr, int64_t B, int64_t unit_cost,
                            int64_t split_cost, int64_t max_grid, int64_t quantum) {
  int64_t used = 0, r = 0, off = 0;
  while (r < nr) {
    if (++used > max_grid) return false;
    int64_t cost = 0;
    bool any = false;
    while (r < nr) {
      const int64_t avail = keys[r] - off;  // >= 1
      int64_t room = B - cost - unit_cost;
      const bool whole = off == 0 && avail <= room;
      if (!whole) room -= split_cost;
      if (room < quantum) {
        if (!any) return false;  // B cannot hold even one key (or tile)
        break;
      }
      const int64_t take = avail <= room ? avail : room / quantum * quantum;
      cost += unit_cost + (whole ? 0 : split_cost) + take;
      any = true;
      if (take == avail) {
        ++r;
        off = 0;
      } else {
        off += take;
        break;  // this CTA's budget is spent
      }
    }
  }
  return true;
}

// The split-KV decode plan of the T newest tokens of n sequences (host only):
// the (sequence, KV head) key ranges cut into units, grouped by CTA. ctas > 0
// plans for that many CTAs instead of the device's.
static int decode_plan(segkv* h, int layer, int T, const int32_t* seq_lens, const int32_t* seq_ids,
                       int n, int64_t ctas_override, DecodePlan& P) {
  const int W = h->win[layer];
  const int rows = T * h->G;
  // 8 or 16 query rows of 128 dims run on the tensor-core decode kernel
  // (128-key stages, one CTA per SM); the rest on the CUDA-core kernel
  const bool mma = h->D == 128 && (rows == 8 || rows == 16);
  // pairs (req, head) with their key ranges [lo, n)
  std::vector<DecodeRange>& ranges = P.ranges;
  std::vector<int64_t>& keys = P.keys;
  ranges.clear();
  keys.clear();
  ranges.reserve(static_cast<size_t>(n) * h->Hkv);
  keys.reserve(static_cast<size_t>(n) * h->Hkv);
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {
    const int b = seq_ids[i];
    const int32_t nlen = h->len[h->lidx(layer, b)];
    if (seq_lens[i] != nlen || nlen < T)
      return fail(h, SEGKV_ERR_INVALID_ARG, "seq_lens[%d]=%d but seq %d has %d tokens (T=%d)", i,
                  seq_lens[i], b, nlen, T);
    const int32_t p0 = nlen - T;  // the oldest query token's position
    for (int hd = 0; hd < h->Hkv; ++hd) {
      const int local = h->local(layer, hd) ? 1 : 0;
      const int32_t lo = local ? std::max(0, p0 - W + 1) : 0;
      if (lo < h->start[h->seg(layer, hd, b)])
        return fail(h, SEGKV_ERR_EVICTED, "seq %d head %d: key %d already evicted", b, hd, lo);
      ranges.push_back({i, hd, lo, nlen, static_cast<int32_t>(h->seg(layer, hd, b)), local});
      // the tensor-core kernel streams whole 128-key tiles: its work is priced in tiles
      const int64_t work = mma ? (int64_t((nlen - 1) / 128) - lo / 128 + 1) * 128 : int64_t(nlen - lo);
      keys.push_back(work);
      total += work;
    }
  }
  // Stream-K split with a cost model: the concatenated key ranges are cut into
  // one slice per CTA so that keys + kDecodeUnitCost per unit (+
  // kDecodeSplitCost per piece of a split pair) is the same for every CTA. A
  // unit's epilogue (the warps' merge, the output or partials) pauses its
  // CTA's memory stream; a piece of a split pair also writes partials, takes
  // a ticket and may merge. Per-CTA timestamps on the ragged-decode workload
  // priced a unit at about the time a CTA streams 128 keys in; the split
  // surcharge was tuned on the same workload (0 -> 256 keys: 62.4 -> 61.6 us).
  // On the tensor-core kernel, with the rows split between its two softmax
  // groups, a sweep on the four-token ragged decode priced a unit at 64 keys
  // (0: 71.3-71.8 us, 64: 70.2-70.5, 128: 70.8-71.1, 384: 73.6, 512: 75.6-75.9)
  // and a split piece at 128 (70.5 us; 512: 72.0).
  // The smallest per-CTA budget whose greedy cut fits the grid is found by
  // bisection.
  // On the tensor-core kernel, work and cuts are in whole 128-key tiles: a cut
  // inside a tile would make both neighbours stream that whole tile.
  const int64_t quantum = mma ? 128 : 1;
  const int64_t kDecodeUnitCost = mma ? 64 : 128;
  const int64_t kDecodeSplitCost = mma ? 128 : 256;
  const int64_t sk = mma ? 128 : decode_stage_keys(rows);
  const int64_t ctas = ctas_override > 0 ? ctas_override
                       : h->num_sms <= 0 ? decode_max_grid(h)
                       : mma ? int64_t(h->num_sms)
                             : int64_t(h->num_sms) * decode_ctas_per_sm(h->D, rows);
  const int max_grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(
      std::min<int64_t>(ctas, ctas_override > 0 ? ctas_override : decode_max_grid(h)),
      (total + sk - 1) / sk)));
  std::vector<DecodeUnit>& units = P.units;
  std::vector<int32_t>& pair_unit0 = P.pair_unit0;
  std::vector<int32_t>& pair_units = P.pair_units;
  std::vector<int32_t>& cta_begin = P.cta_begin;
  const int64_t nr = static_cast<int64_t>(ranges.size());
  // Every CTA costs at most the budget, so the budget is at least the total
  // cost over the grid; the greedy cut leaves each CTA short of the budget by
  // less than a unit and a split surcharge, so a budget a little above that
  // bound usually fits. Probing it first narrows the bisection to a few steps.
  int64_t lo = std::max<int64_t>(1, (total + kDecodeUnitCost * nr) / max_grid);
  int64_t hi = total + kDecodeUnitCost * (nr + 1);  // one CTA holds everything
  auto fits = [&](int64_t B) {
    return decode_cut_fits(keys.data(), nr, B, kDecodeUnitCost, kDecodeSplitCost, max_grid, quantum);
  };
  const int64_t probe = lo + lo / 8 + 2 * (kDecodeUnitCost + kDecodeSplitCost);
  if (probe < hi && fits(probe)) hi = probe;
  while (lo < hi) {  // smallest budget that fits max_grid CTAs
    const int64_t mid = lo + (hi - lo) / 2;
    if (fits(mid)) hi = mid;
    else lo = mid + 1;
  }
  // The greedy cut with that budget, emitting the units. A CTA takes whole
  // ranges while they fit, then a piece of the next one, which pays the split
  // surcharge (a piece also writes partials and may merge).
  units.clear();
  cta_begin.clear();
  units.reserve(static_cast<size_t>(nr + max_grid));
  cta_begin.reserve(static_cast<size_t>(max_grid) + 1);
  pair_unit0.resize(static_cast<size_t>(nr));
  pair_units.resize(static_cast<size_t>(nr));
  {
    const int64_t B = lo;
    int64_t r = 0, off = 0;
    while (r < nr) {
      cta_begin.push_back(static_cast<int32_t>(units.size()));
      int64_t cost = 0;
      while (r < nr) {
        const DecodeRange& R = ranges[r];
        const int64_t avail = keys[r] - off;
        int64_t room = B - cost - kDecodeUnitCost;
        const bool whole = off == 0 && avail <= room;
        if (!whole) room -= kDecodeSplitCost;
        if (room < quantum) {
          if (cost == 0)  // cannot happen: B was found to fit
            return fail(h, SEGKV_ERR_INVALID_ARG, "decode plan: budget %lld holds no key",
                        static_cast<long long>(B));
          break;
        }
        const int64_t take = avail <= room ? avail : room / quantum * quantum;
        if (off == 0) pair_unit0[r] = static_cast<int32_t>(units.size());
        DecodeUnit u{};
        u.req = R.req;
        u.head = static_cast<int16_t>(R.head);
        u.local = static_cast<int16_t>(R.local);
        // work offsets are keys from lo, or from lo's tile start when quantum = 128
        const int64_t base = quantum > 1 ? R.lo / quantum * quantum : R.lo;
        u.k0 = static_cast<int32_t>(std::max<int64_t>(R.lo, base + off));
        u.k1 = static_cast<int32_t>(std::min<int64_t>(R.n, base + off + take));
        u.table_row = R.row;
        u.q_last = R.n - 1;
        units.push_back(u);
        cost += kDecodeUnitCost + (whole ? 0 : kDecodeSplitCost) + take;
        if (take == avail) {  // the pair is complete: its units learn their count
          const int32_t u0 = pair_unit0[r], cnt = static_cast<int32_t>(units.size()) - u0;
          pair_units[r] = cnt;
          for (int32_t x = u0; x < u0 + cnt; ++x) {
            units[x].pair_unit0 = u0;
            units[x].pair_units = cnt;
          }
          ++r;
          off = 0;
        } else {
          off += take;
          break;  // this CTA's budget is spent
        }
      }
    }
  }
  const int grid = static_cast<int>(cta_begin.size());
  cta_begin.push_back(static_cast<int32_t>(units.size()));
  P.grid = grid;
  P.rows = rows;
  P.mma = mma;
  return SEGKV_OK;
}

// Split-KV decode of the T newest tokens of n sequences: T * G query rows per
// KV head, each with its own causal (and window) limit.
static int decode_core(segkv* h, int layer, const void* q, int T, const int32_t* seq_lens,
                       const int32_t* seq_ids, int n, void* o, float* lse, void* workspace,
                       size_t workspace_bytes, cudaStream_t s) {
  const int W = h->win[layer];
  DecodePlan& P = h->dplan;
  const int prc = decode_plan(h, layer, T, seq_lens, seq_ids, n, 0, P);
  if (prc != SEGKV_OK) return prc;
  const std::vector<DecodeRange>& ranges = P.ranges;
  const std::vector<DecodeUnit>& units = P.units;
  const std::vector<int32_t>& cta_begin = P.cta_begin;
  const std::vector<int32_t>& pair_unit0 = P.pair_unit0;
  const std::vector<int32_t>& pair_units = P.pair_units;
  const int rows = P.rows, grid = P.grid;
  const bool mma = P.mma;
  size_t acc_bytes, ml_bytes;
  const size_t need =
      decode_ws_bytes(h, static_cast<int64_t>(units.size()), rows, &acc_bytes, &ml_bytes);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return fail(h, SEGKV_ERR_INVALID_ARG, "workspace needs %zu bytes (256-aligned), got %zu", need,
                workspace_bytes);

  if (mma) {
    std::vector<DecodeCombine> comb;  // pairs split over several units
    for (size_t r = 0; r < ranges.size(); ++r)
      if (pair_units[r] > 1) comb.push_back({pair_unit0[r], pair_units[r], ranges[r].req, ranges[r].head});
    return decode_mma_launch(h, layer, q, T, n, o, lse, units, cta_begin, comb, workspace, acc_bytes,
                             grid, s);
  }
  Pack pk;
  const size_t o_units = pk.add(units.data(), units.size());
  const size_t o_cta = pk.add(cta_begin.data(), cta_begin.size());
  const bool inl = pk.buf.size() <= sizeof(PlanBlob);
  size_t off_ring = 0;
  uintptr_t d = 0;  // device address of the plan; 0 (offsets alone) when it is inline
  cudaError_t e;
  if (inl) {
    std::memcpy(h->blob.data, pk.buf.data(), pk.buf.size());
  } else {
    e = h->ring.reserve(pk.buf.size(), &off_ring);
    if (e != cudaSuccess) return cuda_fail(h, e, "upload ring");
    std::memcpy(h->ring.host + off_ring, pk.buf.data(), pk.buf.size());
    e = h->ring.upload(off_ring, pk.buf.size(), s);
    if (e != cudaSuccess) return cuda_fail(h, e, "plan upload (decode)");
    d = reinterpret_cast<uintptr_t>(h->ring.dev + off_ring);
  }
  h->upload_bytes += static_cast<int64_t>(pk.buf.size());
  DecodeParams p{};
  p.plan_inline = inl ? 1 : 0;
  p.units = reinterpret_cast<const DecodeUnit*>(d + o_units);
  p.cta_begin = reinterpret_cast<const int32_t*>(d + o_cta);
  p.q = q;
  p.o = o;
  p.table = h->d_table;
  p.kpool = h->kpool;
  p.vpool = h->vpool;
  p.part_acc = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + acc_bytes);
  p.pair_cnt = h->d_pair_cnt;
  p.lse = lse;
  p.n_rows = n * T;
  p.n_units = static_cast<int>(units.size());
  p.n_pairs = static_cast<int>(ranges.size());
  p.R = h->R;
  p.hq = h->Hq;
  p.hkv = h->Hkv;
  p.G = rows;
  p.T = T;
  p.Gm = h->G;
  p.window = W;
  p.page_size = h->P;
  p.scale_log2 = h->scale * 1.4426950408889634f;
  p.status = h->d_status;
  p.timeout_ns = kTimeoutNs;
  e = launch_decode(p, inl ? &h->blob : nullptr, h->D, grid, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "decode kernel launch");
  if (!inl) {
    e = h->ring.commit(off_ring, pk.buf.size(), s);
    if (e != cudaSuccess) return cuda_fail(h, e, "event record");
  }
  return SEGKV_OK;
}

int segkv_decode_attn(segkv_t h, int layer, const void* q, const int32_t* seq_lens,
                      const int32_t* seq_ids, int n, void* o, void* workspace,
                      size_t workspace_bytes, segkv_stream_t stream) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (h->host_only) return fail(h, SEGKV_ERR_INVALID_ARG, "host-only handle has no pools");
  if (layer < 0 || layer >= h->L) return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer %d", layer);
  if (!ids_valid(h, seq_ids, n)) return fail(h, SEGKV_ERR_INVALID_ARG, "bad seq_ids");
  if (n == 0) return SEGKV_OK;
  if (!q || !o || !seq_lens) return fail(h, SEGKV_ERR_INVALID_ARG, "q/o/seq_lens NULL");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(o)) & 15)
    return fail(h, SEGKV_ERR_INVALID_ARG, "q and o must be 16-byte aligned");
  return decode_core(h, layer, q, 1, seq_lens, seq_ids, n, o, nullptr, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- rope shift
int segkv_rope_shift(segkv_t h, int layer, int seq, int32_t delta, double base, int rotary_dim,
                     int style, uint64_t head_mask, segkv_stream_t stream) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (h->host_only) return fail(h, SEGKV_ERR_INVALID_ARG, "host-only handle has no pools");
  if (layer < 0 || layer >= h->L || seq < 0 || seq >= h->S)
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer or seq");
  if (rotary_dim < 2 || rotary_dim > h->D || rotary_dim % 2 || (style != 0 && style != 1) ||
      !(base > 1.0))
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad rotary parameters");
  const int32_t nlen = h->len[h->lidx(layer, seq)];
  // the plan is one entry per selected KV head, passed in the kernel's
  // parameters; the kernel walks each head's block-table row itself
  RopeParams p{};
  int32_t max_pages = 0;
  for (int hd = 0; hd < h->Hkv && hd < 64; ++hd) {
    if (!((head_mask >> hd) & 1u)) continue;
    const int32_t s0 = h->start[h->seg(layer, hd, seq)];
    if (s0 >= nlen) continue;
    p.heads[p.n_heads++] = {static_cast<int32_t>(h->seg(layer, hd, seq)), s0, nlen, 0};
    max_pages = std::max(max_pages, (nlen - 1) / h->P - s0 / h->P + 1);
  }
  if (p.n_heads == 0 || delta == 0) return SEGKV_OK;
  for (int i = 0; i < rotary_dim / 2; ++i) {
    const double ang = static_cast<double>(delta) * std::pow(base, -2.0 * i / rotary_dim);
    p.cos_sin[i] = make_float2(static_cast<float>(std::cos(ang)), static_cast<float>(std::sin(ang)));
  }
  p.table = h->d_table;
  p.kpool = h->kpool;
  p.R = h->R;
  p.page_size = h->P;
  p.head_dim = h->D;
  p.rotary_dim = rotary_dim;
  p.style = style;
  const int64_t chunks = int64_t(max_pages) * p.n_heads;
  const int grid = static_cast<int>(std::min<int64_t>(chunks, int64_t(std::max(1, h->num_sms)) * 8));
  cudaError_t e = launch_rope(p, max_pages, grid, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "rope kernel launch");
  return SEGKV_OK;
}

// ---------------------------------------------------------------- variants
int segkv_set_window_convention(segkv_t h, int convention) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (convention != SEGKV_WINDOW_INCLUSIVE && convention != SEGKV_WINDOW_FA)
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad window convention %d", convention);
  for (int32_t n : h->len)
    if (n != 0) return fail(h, SEGKV_ERR_INVALID_ARG, "the handle already holds tokens");
  // the FA window (W, 0) covers W+1 keys: the same as an inclusive window of W+1
  const int add = (convention == SEGKV_WINDOW_FA) - (h->window_fa ? 1 : 0);
  for (int32_t& w : h->win) w += add;
  h->window_fa = convention == SEGKV_WINDOW_FA;
  return SEGKV_OK;
}

int segkv_plan_decode(segkv_t h, int layer, int T, const int32_t* seq_lens, const int32_t* seq_ids,
                      int n, int num_ctas, int32_t* units_out, int max_units, int32_t* cta_begin_out,
                      int max_ctas, int* n_units, int* n_ctas) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->L) return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer %d", layer);
  if (T < 1 || n < 0 || max_units < 0 || max_ctas < 0 || !n_units || !n_ctas)
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad T, n or output sizes");
  if (!ids_valid(h, seq_ids, n)) return fail(h, SEGKV_ERR_INVALID_ARG, "bad seq_ids");
  *n_units = 0;
  *n_ctas = 0;
  if (n == 0) return SEGKV_OK;
  if (!seq_lens) return fail(h, SEGKV_ERR_INVALID_ARG, "seq_lens NULL");
  DecodePlan& P = h->dplan;
  const int rc = decode_plan(h, layer, T, seq_lens, seq_ids, n, num_ctas, P);
  if (rc != SEGKV_OK) return rc;
  *n_units = static_cast<int>(P.units.size());
  *n_ctas = P.grid;
  if (static_cast<int>(P.units.size()) > max_units || P.grid > max_ctas || (max_units && !units_out) ||
      !cta_begin_out)
    return fail(h, SEGKV_ERR_INVALID_ARG, "plan needs %d units and %d CTAs", *n_units, *n_ctas);
  for (size_t x = 0; x < P.units.size(); ++x) {
    const DecodeUnit& u = P.units[x];
    int32_t* o = units_out + 8 * x;
    o[0] = u.req;
    o[1] = u.head;
    o[2] = u.local;
    o[3] = u.k0;
    o[4] = u.k1;
    o[5] = u.pair_unit0;
    o[6] = u.pair_units;
    o[7] = u.q_last;
  }
  for (int c = 0; c <= P.grid; ++c) cta_begin_out[c] = P.cta_begin[c];
  return SEGKV_OK;
}

int segkv_decode_attn_multi(segkv_t h, int layer, const void* q, int T, const int32_t* seq_lens,
                            const int32_t* seq_ids, int n, void* o, float* lse, void* workspace,
                            size_t workspace_bytes, segkv_stream_t stream) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (T < 1 || n < 0 || (n > 0 && !seq_lens))
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad T or seq_lens");
  if (layer < 0 || layer >= h->L) return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer %d", layer);
  if (!ids_valid(h, seq_ids, n)) return fail(h, SEGKV_ERR_INVALID_ARG, "bad seq_ids");
  if (decode_kernel_rows(T * h->G) && !h->host_only) {
    if (n == 0) return SEGKV_OK;
    if (!q || !o) return fail(h, SEGKV_ERR_INVALID_ARG, "q/o NULL");
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(o)) & 15)
      return fail(h, SEGKV_ERR_INVALID_ARG, "q and o must be 16-byte aligned");
    return decode_core(h, layer, q, T, seq_lens, seq_ids, n, o, lse, workspace, workspace_bytes,
                       static_cast<cudaStream_t>(stream));
  }
  // more than 16 query rows per KV head: the tensor-core prefill kernel
  std::vector<int32_t> cu(n + 1), pos(static_cast<size_t>(n) * T);
  for (int i = 0; i < n; ++i) {
    const int32_t nlen = h->len[h->lidx(layer, seq_ids[i])];
    if (seq_lens[i] != nlen || nlen < T)
      return fail(h, SEGKV_ERR_INVALID_ARG, "seq_lens[%d]=%d but seq %d has %d tokens (T=%d)", i,
                  seq_lens[i], seq_ids[i], nlen, T);
    cu[i] = i * T;
    for (int t = 0; t < T; ++t) pos[static_cast<size_t>(i) * T + t] = nlen - T + t;
  }
  cu[n] = n * T;
  return segkv_prefill_attn(h, layer, q, cu.data(), pos.data(), seq_ids, n, o, lse, nullptr, 0,
                            stream);
}

// ---------------------------------------------------------------- transfer
// A packed plan goes inside the kernel parameters when it fits, else through
// the upload ring. base is the plan's device address, 0 when it is inline.
struct PlanPlace {
  bool inl = false;
  size_t off = 0;
  uintptr_t base = 0;
};

static int place_small_plan(segkv* h, const Pack& pk, cudaStream_t s, PlanPlace* pp) {
  pp->inl = pk.buf.size() <= sizeof(AppendBlob);
  if (pp->inl) {
    std::memcpy(h->blob.data, pk.buf.data(), pk.buf.size());
  } else {
    cudaError_t e = h->ring.reserve(pk.buf.size(), &pp->off);
    if (e != cudaSuccess) return cuda_fail(h, e, "upload ring");
    std::memcpy(h->ring.host + pp->off, pk.buf.data(), pk.buf.size());
    e = h->ring.upload(pp->off, pk.buf.size(), s);
    if (e != cudaSuccess) return cuda_fail(h, e, "plan upload");
    pp->base = reinterpret_cast<uintptr_t>(h->ring.dev + pp->off);
  }
  h->upload_bytes += static_cast<int64_t>(pk.buf.size());
  return SEGKV_OK;
}

static int finish_small_plan(segkv* h, const PlanPlace& pp, const Pack& pk, cudaStream_t s) {
  if (pp.inl) return SEGKV_OK;
  cudaError_t e = h->ring.commit(pp.off, pk.buf.size(), s);
  return e == cudaSuccess ? SEGKV_OK : cuda_fail(h, e, "event record");
}

// Transfer grid: enough CTAs for about 4 chunks per thread, at most 8 per SM.
static int transfer_grid(const segkv* h, int64_t rows) {
  const int64_t chunks = rows * (h->D / 8);
  const int64_t want = (chunks + 256 * 4 - 1) / (256 * 4);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(std::max(1, h->num_sms)) * 8)));
}

int segkv_export_size(segkv_t h, int layer, int seq, size_t* bytes) {
  if (!h || !bytes) return SEGKV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->L || seq < 0 || seq >= h->S)
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer or seq");
  const int32_t n = h->len[h->lidx(layer, seq)];
  size_t rows = 0;
  for (int hd = 0; hd < h->Hkv; ++hd) rows += n - h->start[h->seg(layer, hd, seq)];
  *bytes = rows * h->D * 2 * 2;
  return SEGKV_OK;
}

int segkv_export(segkv_t h, int layer, int seq, void* out, size_t out_bytes, int32_t* header,
                 segkv_stream_t stream) {
  size_t need = 0;
  int rc = segkv_export_size(h, layer, seq, &need);
  if (rc != SEGKV_OK) return rc;
  if (!header) return fail(h, SEGKV_ERR_INVALID_ARG, "header is NULL");
  const int32_t n = h->len[h->lidx(layer, seq)];
  header[0] = n;
  for (int hd = 0; hd < h->Hkv; ++hd) header[1 + hd] = h->start[h->seg(layer, hd, seq)];
  if (!out && out_bytes == 0) return SEGKV_OK;  // header and size only
  if (h->host_only) return fail(h, SEGKV_ERR_INVALID_ARG, "host-only handle has no pools");
  if (!out || out_bytes < need || (reinterpret_cast<uintptr_t>(out) & 15))
    return fail(h, SEGKV_ERR_INVALID_ARG, "export needs %zu bytes (16-aligned), got %zu", need,
                out_bytes);
  std::vector<XferHead>& hv = h->xfer_heads;
  std::vector<int32_t>& pl = h->xfer_pages;
  hv.clear();
  pl.clear();
  int32_t row = 0, rows = 0;
  for (int hd = 0; hd < h->Hkv; ++hd) {
    const int64_t sg = h->seg(layer, hd, seq);
    const int32_t s0 = h->start[sg], len = n - s0;
    const int32_t* r = h->table.data() + sg * h->R;
    XferHead H{};
    H.s0 = s0;
    H.len = len;
    H.out_row = row;
    H.first_k = s0 / h->P;
    H.page_off = static_cast<int32_t>(pl.size());
    H.table_row = static_cast<int32_t>(sg);
    H.row_begin = rows;
    if (len > 0)
      for (int k = s0 / h->P; k <= (n - 1) / h->P; ++k) pl.push_back(r[k]);
    hv.push_back(H);
    row += 2 * len;
    rows += len;
  }
  if (rows == 0) return SEGKV_OK;
  Pack& pk = h->pack;
  pk.buf.clear();
  const size_t o_heads = pk.add(hv.data(), hv.size());
  const size_t o_pages = pk.add(pl.data(), pl.size());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PlanPlace pp;
  rc = place_small_plan(h, pk, s, &pp);
  if (rc != SEGKV_OK) return rc;
  TransferParams p{};
  p.heads = reinterpret_cast<const XferHead*>(pp.base + o_heads);
  p.page_list = reinterpret_cast<const int32_t*>(pp.base + o_pages);
  p.kpool = static_cast<uint4*>(h->kpool);
  p.vpool = static_cast<uint4*>(h->vpool);
  p.buf_out = static_cast<uint4*>(out);
  p.table = h->d_table;
  p.plan_inline = pp.inl ? 1 : 0;
  p.to_pool = 0;
  p.n_heads = h->Hkv;
  p.n_pages = static_cast<int>(pl.size());
  p.vec_per_row = h->D / 8;
  p.page_size = h->P;
  p.R = h->R;
  p.total_rows = rows;
  cudaError_t e = launch_transfer(p, pp.inl ? reinterpret_cast<const AppendBlob*>(&h->blob) : nullptr,
                                  transfer_grid(h, rows), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "export kernel launch");
  return finish_small_plan(h, pp, pk, s);
}

int segkv_import(segkv_t h, int layer, int seq, const void* in, size_t in_bytes,
                 const int32_t* header, segkv_stream_t stream) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->L || seq < 0 || seq >= h->S || !header)
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer, seq or header");
  if (h->len[h->lidx(layer, seq)] != 0)
    return fail(h, SEGKV_ERR_INVALID_ARG, "seq %d is not empty in layer %d", seq, layer);
  const int32_t n = header[0];
  if (n < 0 || n > h->max_len) return fail(h, SEGKV_ERR_INVALID_ARG, "bad length %d", n);
  int64_t need = 0;
  size_t rows = 0;
  for (int hd = 0; hd < h->Hkv; ++hd) {
    const int32_t s0 = header[1 + hd];
    if (s0 < 0 || s0 > n) return fail(h, SEGKV_ERR_INVALID_ARG, "bad kept start %d", s0);
    rows += n - s0;
    if (n > 0 && (n - 1) / h->P >= s0 / h->P) need += (n - 1) / h->P - s0 / h->P + 1;
  }
  const size_t bytes = rows * h->D * 2 * 2;
  if (!h->host_only && bytes > 0 &&
      (!in || in_bytes < bytes || (reinterpret_cast<uintptr_t>(in) & 15)))
    return fail(h, SEGKV_ERR_INVALID_ARG, "import needs %zu bytes (16-aligned), got %zu", bytes,
                in_bytes);
  if (static_cast<int64_t>(h->free_ids.size()) < need)
    return fail(h, SEGKV_ERR_OUT_OF_PAGES, "import needs %lld pages, %lld free",
                static_cast<long long>(need), static_cast<long long>(h->free_ids.size()));
  std::vector<XferHead>& hv = h->xfer_heads;
  std::vector<int32_t>& pl = h->xfer_pages;
  hv.clear();
  pl.clear();
  int32_t row = 0, nrows = 0;
  for (int hd = 0; hd < h->Hkv; ++hd) {
    const int64_t sg = h->seg(layer, hd, seq);
    const int32_t s0 = header[1 + hd], len = n - s0;
    h->start[sg] = s0;
    int32_t* r = h->row(layer, hd, seq);
    XferHead H{};
    H.s0 = s0;
    H.len = len;
    H.out_row = row;
    H.first_k = s0 / h->P;
    H.page_off = static_cast<int32_t>(pl.size());
    H.table_row = static_cast<int32_t>(sg);
    H.row_begin = nrows;
    if (n > 0) {
      const int k0 = s0 / h->P, np = (n - 1) / h->P - k0 + 1;
      h->free_ids.take(r + k0, np);
      pl.insert(pl.end(), r + k0, r + k0 + np);
    }
    hv.push_back(H);
    row += 2 * len;
    nrows += len;
  }
  h->len[h->lidx(layer, seq)] = n;
  if (h->host_only || pl.empty()) return SEGKV_OK;
  Pack& pk = h->pack;
  pk.buf.clear();
  const size_t o_heads = pk.add(hv.data(), hv.size());
  const size_t o_pages = pk.add(pl.data(), pl.size());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PlanPlace pp;
  int rc = place_small_plan(h, pk, s, &pp);
  if (rc != SEGKV_OK) return rc;
  TransferParams p{};
  p.heads = reinterpret_cast<const XferHead*>(pp.base + o_heads);
  p.page_list = reinterpret_cast<const int32_t*>(pp.base + o_pages);
  p.kpool = static_cast<uint4*>(h->kpool);
  p.vpool = static_cast<uint4*>(h->vpool);
  p.buf = static_cast<const uint4*>(in);
  p.table = h->d_table;
  p.plan_inline = pp.inl ? 1 : 0;
  p.to_pool = 1;
  p.n_heads = h->Hkv;
  p.n_pages = static_cast<int>(pl.size());
  p.vec_per_row = h->D / 8;
  p.page_size = h->P;
  p.R = h->R;
  p.total_rows = nrows;
  cudaError_t e = launch_transfer(p, pp.inl ? reinterpret_cast<const AppendBlob*>(&h->blob) : nullptr,
                                  transfer_grid(h, std::max<int64_t>(nrows, static_cast<int64_t>(pl.size()))), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "import kernel launch");
  return finish_small_plan(h, pp, pk, s);
}

// ---------------------------------------------------------------- trim / free
int segkv_trim(segkv_t h, int layer, const int32_t* seq_ids, int n) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (layer < -1 || layer >= h->L) return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer %d", layer);
  if (!ids_valid(h, seq_ids, n)) return fail(h, SEGKV_ERR_INVALID_ARG, "bad seq_ids");
  const int l0 = layer < 0 ? 0 : layer, l1 = layer < 0 ? h->L : layer + 1;
  for (int l = l0; l < l1; ++l)
    for (int i = 0; i < n; ++i) {
      const int b = seq_ids[i];
      const int32_t nlen = h->len[h->lidx(l, b)];
      for (int hd = 0; hd < h->Hkv; ++hd)
        evict_below(h, l, hd, b, needed_start(h, l, hd, h->start[h->seg(l, hd, b)], nlen));
    }
  return SEGKV_OK;
}

int segkv_free_seq(segkv_t h, int seq_id) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (seq_id < 0 || seq_id >= h->S) return fail(h, SEGKV_ERR_INVALID_ARG, "bad seq %d", seq_id);
  for (int l = 0; l < h->L; ++l) {
    for (int hd = 0; hd < h->Hkv; ++hd) {
      int32_t* r = h->row(l, hd, seq_id);
      for (int k = 0; k < h->R; ++k)
        if (r[k] >= 0) {
          h->free_ids.push(r[k]);
          r[k] = -1;
        }
      h->start[h->seg(l, hd, seq_id)] = 0;
    }
    h->len[h->lidx(l, seq_id)] = 0;
  }
  return SEGKV_OK;
}

// ---------------------------------------------------------------- queries
int segkv_get_segment(segkv_t h, int layer, int head, int seq, int32_t* start, int32_t* len,
                      int32_t* first_page, int32_t* ids, int max_ids, int32_t* n_ids) {
  if (!h || !start || !len || !first_page || !n_ids) return SEGKV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->L || head < 0 || head >= h->Hkv || seq < 0 || seq >= h->S)
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad segment index");
  const int32_t s0 = h->start[h->seg(layer, head, seq)];
  const int32_t nlen = h->len[h->lidx(layer, seq)];
  *start = s0;
  *len = nlen - s0;
  const int32_t* r = h->table.data() + h->seg(layer, head, seq) * h->R;
  int c = 0, first = -1;
  for (int k = 0; k < h->R; ++k)
    if (r[k] >= 0) {
      if (first < 0) first = k;
      if (ids && c < max_ids) ids[c] = r[k];
      ++c;
    }
  *first_page = first < 0 ? 0 : first;
  *n_ids = c;
  return c <= max_ids || !ids ? SEGKV_OK : fail(h, SEGKV_ERR_INVALID_ARG, "ids buffer too small");
}

int segkv_seq_len(segkv_t h, int layer, int seq, int32_t* len) {
  if (!h || !len || layer < 0 || layer >= h->L || seq < 0 || seq >= h->S)
    return SEGKV_ERR_INVALID_ARG;
  *len = h->len[h->lidx(layer, seq)];
  return SEGKV_OK;
}

int segkv_stats(segkv_t h, segkv_stats_t* out) {
  if (!h || !out) return SEGKV_ERR_INVALID_ARG;
  segkv_stats_t st{};
  st.num_pages = h->num_pages;
  for (int l = 0; l < h->L; ++l)
    for (int hd = 0; hd < h->Hkv; ++hd)
      for (int b = 0; b < h->S; ++b) {
        const int32_t* r = h->table.data() + h->seg(l, hd, b) * h->R;
        int64_t c = 0;
        for (int k = 0; k < h->R; ++k) c += r[k] >= 0;
        (h->local(l, hd) ? st.pages_local : st.pages_global) += c;
        st.kept_tokens += h->len[h->lidx(l, b)] - h->start[h->seg(l, hd, b)];
      }
  st.pages_in_use = st.pages_local + st.pages_global;
  st.upload_bytes = h->upload_bytes;
  *out = st;
  return SEGKV_OK;
}

// ---------------------------------------------------------------- attention mass
// One prefill chunk per sequence, its attention mass per key: the work plan
// (host). A unit is one KV head x one key tile of 128 positions, over the
// query tiles that see some of its keys; a key tile seen by many query tiles
// is cut into pieces (partial sums in slots part0 .. part0 + n_pieces - 1, a
// finished-piece counter tile_id). Units are dealt to `ctas` lists by LPT.
struct MassPlan {
  std::vector<MassUnit> units;     // grouped by CTA
  std::vector<int32_t> cta_begin;  // [grid + 1]
  int32_t slots = 0, tiles = 0;
  int grid = 0;
};

static int mass_plan(segkv* h, int layer, const int32_t* cu_seqlens, const int32_t* q_pos,
                     const int32_t* seq_ids, int n, int ctas, MassPlan& M) {
  const int W = h->win[layer];
  const int tpt = kRowsPerTile / h->G;
  std::vector<MassUnit>& units = M.units;
  units.clear();
  M.cta_begin.assign(1, 0);
  M.slots = M.tiles = 0;
  M.grid = 0;
  for (int i = 0; i < n; ++i) {
    const int b = seq_ids[i];
    const int32_t nlen = h->len[h->lidx(layer, b)];
    const int32_t T = cu_seqlens[i + 1] - cu_seqlens[i];
    if (T == 0) continue;
    const int32_t a = q_pos[cu_seqlens[i]];
    for (int32_t t = 0; t < T; ++t)
      if (q_pos[cu_seqlens[i] + t] != a + t)
        return fail(h, SEGKV_ERR_INVALID_ARG, "q_pos of seq %d are not consecutive", b);
    if (a < 0 || a + T > nlen)
      return fail(h, SEGKV_ERR_INVALID_ARG, "chunk [%d,%d) outside seq %d of length %d", a, a + T,
                  b, nlen);
    for (int hd = 0; hd < h->Hkv; ++hd) {
      const int32_t s0 = h->start[h->seg(layer, hd, b)];
      const bool local = h->local(layer, hd);
      const int32_t need = local ? std::max(0, a - W + 1) : 0;
      if (need < s0)
        return fail(h, SEGKV_ERR_EVICTED, "seq %d head %d: key %d already evicted", b, hd, need);
      for (int32_t kt = a / kKeyTile; kt <= (a + T - 1) / kKeyTile; ++kt) {
        const int32_t j0 = std::max(a, kt * kKeyTile);
        const int32_t j1 = std::min(a + T, (kt + 1) * kKeyTile) - 1;
        // query tokens that see some key of [j0, j1]
        const int32_t tlo = j0 - a;
        const int32_t thi = local ? std::min(T - 1, j1 + W - 1 - a) : T - 1;
        MassUnit u{};
        u.tok0 = cu_seqlens[i];
        u.ntok = T;
        u.a = a;
        u.head = hd;
        u.local = local ? 1 : 0;
        u.kt = kt;
        u.qt0 = tlo / tpt;
        u.qt1 = thi / tpt;
        u.first_page = s0 / h->P;
        u.last_page = (nlen - 1) / h->P;
        u.table_row = static_cast<int32_t>(h->seg(layer, hd, b));
        units.push_back(u);
      }
    }
  }
  if (units.empty()) return SEGKV_OK;
  // Cut key tiles seen by many query tiles into pieces of at most `cap`
  // query tiles, so that no unit is much longer than a CTA's fair share.
  int64_t steps = 0;
  for (const MassUnit& u : units) steps += u.qt1 - u.qt0 + 1;
  const int32_t cap = static_cast<int32_t>(std::max<int64_t>(8, (steps + 2 * ctas - 1) / (2 * ctas)));
  std::vector<MassUnit> cut;
  int32_t slots = 0, tiles = 0;
  for (const MassUnit& u : units) {
    const int32_t len = u.qt1 - u.qt0 + 1;
    const int32_t np = (len + cap - 1) / cap;
    for (int32_t pc = 0; pc < np; ++pc) {
      MassUnit v = u;
      v.qt0 = u.qt0 + static_cast<int32_t>(int64_t(len) * pc / np);
      v.qt1 = u.qt0 + static_cast<int32_t>(int64_t(len) * (pc + 1) / np) - 1;
      v.piece = pc;
      v.n_pieces = np;
      v.part0 = np > 1 ? slots : 0;
      v.tile_id = np > 1 ? tiles : 0;
      cut.push_back(v);
    }
    if (np > 1) {
      slots += np;
      ++tiles;
    }
  }
  units.swap(cut);
  // LPT schedule: longest first, each to the least-loaded CTA
  std::stable_sort(units.begin(), units.end(), [](const MassUnit& x, const MassUnit& y) {
    return (x.qt1 - x.qt0) > (y.qt1 - y.qt0);
  });
  const int grid = static_cast<int>(std::min<int64_t>(units.size(), ctas));
  std::vector<int32_t>& cta_begin = M.cta_begin;
  cta_begin.assign(grid + 1, 0);
  std::vector<int32_t> cta_of(units.size());
  {
    LeastLoaded lpt;
    lpt.reset(grid);
    for (size_t x = 0; x < units.size(); ++x) {
      const int c = lpt.least();
      cta_of[x] = c;
      ++cta_begin[c + 1];
      lpt.add(c, units[x].qt1 - units[x].qt0 + 2);  // + the unit's key-tile load and hand-off
    }
    for (int c = 0; c < grid; ++c) cta_begin[c + 1] += cta_begin[c];
    std::vector<MassUnit> by_cta(units.size());
    std::vector<int32_t> fill(cta_begin.begin(), cta_begin.end() - 1);
    for (size_t x = 0; x < units.size(); ++x) by_cta[fill[cta_of[x]]++] = units[x];
    units.swap(by_cta);
  }
  M.slots = slots;
  M.tiles = tiles;
  M.grid = grid;
  return SEGKV_OK;
}

int segkv_attn_mass(segkv_t h, int layer, const void* q, const int32_t* cu_seqlens,
                    const int32_t* q_pos, const int32_t* seq_ids, int n, const float* lse,
                    float* mass, segkv_stream_t stream) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (h->host_only) return fail(h, SEGKV_ERR_INVALID_ARG, "host-only handle has no pools");
  if (layer < 0 || layer >= h->L) return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer %d", layer);
  if (!ids_valid(h, seq_ids, n)) return fail(h, SEGKV_ERR_INVALID_ARG, "bad seq_ids");
  if (n == 0) return SEGKV_OK;
  if (!cu_seqlens || cu_seqlens[0] != 0) return fail(h, SEGKV_ERR_INVALID_ARG, "cu_seqlens[0] != 0");
  for (int i = 0; i < n; ++i)
    if (cu_seqlens[i + 1] < cu_seqlens[i])
      return fail(h, SEGKV_ERR_INVALID_ARG, "cu_seqlens decreases at %d", i);
  const int64_t total = cu_seqlens[n];
  if (total == 0) return SEGKV_OK;
  if (!q || !lse || !mass || !q_pos) return fail(h, SEGKV_ERR_INVALID_ARG, "q/lse/mass/q_pos NULL");
  if (reinterpret_cast<uintptr_t>(q) & 15)
    return fail(h, SEGKV_ERR_INVALID_ARG, "q must be 16-byte aligned");
  const int W = h->win[layer];
  const int tpt = kRowsPerTile / h->G;
  MassPlan M;
  {
    const int prc = mass_plan(h, layer, cu_seqlens, q_pos, seq_ids, n, std::max(1, h->num_sms), M);
    if (prc != SEGKV_OK) return prc;
  }
  if (M.units.empty()) return SEGKV_OK;
  const std::vector<MassUnit>& units = M.units;
  const std::vector<int32_t>& cta_begin = M.cta_begin;
  const int32_t slots = M.slots, tiles = M.tiles;
  const int grid = M.grid;
  Pack pk;
  const size_t o_units = pk.add(units.data(), units.size());
  const size_t o_cta = pk.add(cta_begin.data(), cta_begin.size());
  const std::vector<int32_t> zeros(std::max(tiles, 1), 0);
  const size_t o_cnt = pk.add(zeros.data(), zeros.size());  // counters travel as zeros
  // partial sums live after the plan in the same ring region; they are not uploaded
  const size_t o_part = align_up(pk.buf.size(), 256);
  const size_t region = o_part + static_cast<size_t>(slots) * kKeyTile * 4;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  size_t off;
  cudaError_t e = h->ring.reserve(region, &off);
  if (e != cudaSuccess) return cuda_fail(h, e, "upload ring");
  std::memcpy(h->ring.host + off, pk.buf.data(), pk.buf.size());
  e = h->ring.upload(off, pk.buf.size(), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "plan upload (mass)");
  h->upload_bytes += static_cast<int64_t>(pk.buf.size());
  CUtensorMap tq;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(h->D), static_cast<cuuint64_t>(h->Hq),
                          static_cast<cuuint64_t>(total)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(h->D) * 2,
                             static_cast<cuuint64_t>(h->Hq) * h->D * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(h->G), static_cast<cuuint32_t>(tpt)};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode_fn()(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return fail(h, SEGKV_ERR_CUDA, "tensor map encode failed for q");
  }
  MassParams p{};
  p.units = reinterpret_cast<const MassUnit*>(h->ring.dev + off + o_units);
  p.cta_begin = reinterpret_cast<const int32_t*>(h->ring.dev + off + o_cta);
  p.tile_cnt = reinterpret_cast<int*>(h->ring.dev + off + o_cnt);
  p.part = reinterpret_cast<float*>(h->ring.dev + off + o_part);
  p.table = h->d_table;
  p.lse = lse;
  p.mass = mass;
  p.total_q = total;
  p.n_units = static_cast<int>(units.size());
  p.R = h->R;
  p.hq = h->Hq;
  p.G = h->G;
  p.tpt = tpt;
  p.window = W;
  p.page_size = h->P;
  p.oob_row = static_cast<int>(h->num_pages * h->P);
  p.scale_log2 = h->scale * 1.4426950408889634f;
  p.status = h->d_status;
  p.timeout_ns = kTimeoutNs;
  e = launch_mass(p, tq, h->tm_k, h->D, grid, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "mass kernel launch");
  e = h->ring.commit(off, region, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "event record");
  return SEGKV_OK;
}

int segkv_plan_mass(segkv_t h, int layer, const int32_t* cu_seqlens, const int32_t* q_pos,
                    const int32_t* seq_ids, int n, int num_ctas, int32_t* units_out, int max_units,
                    int32_t* cta_begin_out, int max_ctas, int* n_units, int* n_ctas) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->L) return fail(h, SEGKV_ERR_INVALID_ARG, "bad layer %d", layer);
  if (n < 0 || max_units < 0 || max_ctas < 0 || !n_units || !n_ctas)
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad n or output sizes");
  if (!ids_valid(h, seq_ids, n)) return fail(h, SEGKV_ERR_INVALID_ARG, "bad seq_ids");
  *n_units = 0;
  *n_ctas = 0;
  if (n == 0) return SEGKV_OK;
  if (!cu_seqlens || cu_seqlens[0] != 0) return fail(h, SEGKV_ERR_INVALID_ARG, "cu_seqlens[0] != 0");
  for (int i = 0; i < n; ++i)
    if (cu_seqlens[i + 1] < cu_seqlens[i])
      return fail(h, SEGKV_ERR_INVALID_ARG, "cu_seqlens decreases at %d", i);
  if (cu_seqlens[n] == 0) return SEGKV_OK;
  if (!q_pos) return fail(h, SEGKV_ERR_INVALID_ARG, "q_pos NULL");
  if (num_ctas > kMaxPlanCtas)
    return fail(h, SEGKV_ERR_INVALID_ARG, "num_ctas %d above %d", num_ctas, kMaxPlanCtas);
  const int ctas = num_ctas > 0 ? num_ctas : std::max(1, h->num_sms);
  MassPlan M;
  const int rc = mass_plan(h, layer, cu_seqlens, q_pos, seq_ids, n, ctas, M);
  if (rc != SEGKV_OK) return rc;
  if (M.units.empty()) return SEGKV_OK;
  *n_units = static_cast<int>(M.units.size());
  *n_ctas = M.grid;
  if (*n_units > max_units || *n_ctas > max_ctas || (max_units && !units_out) || !cta_begin_out)
    return fail(h, SEGKV_ERR_INVALID_ARG, "plan needs %d units and %d CTAs", *n_units, *n_ctas);
  for (size_t x = 0; x < M.units.size(); ++x) {
    const MassUnit& u = M.units[x];
    int32_t* o = units_out + 12 * x;
    o[0] = u.tok0;
    o[1] = u.ntok;
    o[2] = u.a;
    o[3] = u.head;
    o[4] = u.local;
    o[5] = u.kt;
    o[6] = u.qt0;
    o[7] = u.qt1;
    o[8] = u.piece;
    o[9] = u.n_pieces;
    o[10] = u.part0;
    o[11] = u.tile_id;
  }
  for (int c = 0; c <= M.grid; ++c) cta_begin_out[c] = M.cta_begin[c];
  return SEGKV_OK;
}

int segkv_topk_tokens(segkv_t h, const float* mass, const int32_t* cu_seqlens, int n,
                      const int32_t* k, float* score, int32_t* idx, segkv_stream_t stream) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (h->host_only) return fail(h, SEGKV_ERR_INVALID_ARG, "host-only handle has no device");
  if (n < 0 || (n > 0 && (!cu_seqlens || !k || cu_seqlens[0] != 0)))
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad n, cu_seqlens or k");
  if (n == 0) return SEGKV_OK;
  std::vector<TopkSeq> seqs(n);
  int64_t out = 0;
  for (int i = 0; i < n; ++i) {
    const int32_t T = cu_seqlens[i + 1] - cu_seqlens[i];
    if (T < 0 || k[i] < 0 || k[i] > T)
      return fail(h, SEGKV_ERR_INVALID_ARG, "k[%d]=%d outside [0, %d]", i, k[i], T);
    seqs[i] = {cu_seqlens[i], T, k[i], static_cast<int32_t>(out)};
    out += k[i];
  }
  const int64_t total = cu_seqlens[n];
  if (total > 0 && (!mass || !score)) return fail(h, SEGKV_ERR_INVALID_ARG, "mass/score NULL");
  if (out > 0 && !idx) return fail(h, SEGKV_ERR_INVALID_ARG, "idx NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Pack pk;
  const size_t o_seqs = pk.add(seqs.data(), seqs.size());
  PlanPlace pp;
  int rc = place_small_plan(h, pk, s, &pp);
  if (rc != SEGKV_OK) return rc;
  TopkParams p{};
  p.seqs = reinterpret_cast<const TopkSeq*>(pp.base + o_seqs);
  p.idx = idx;
  p.plan_inline = pp.inl ? 1 : 0;
  cudaError_t e = launch_topk(mass, score, total, h->Hkv, p,
                              pp.inl ? reinterpret_cast<const AppendBlob*>(&h->blob) : nullptr, n, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "top-k kernel launch");
  return finish_small_plan(h, pp, pk, s);
}

// ---------------------------------------------------------------- sparse FFN
static size_t ffn_ws_parts(int64_t m, int d_model, int d_ff, bool gather, size_t* h_off) {
  const size_t xs = gather ? align_up(static_cast<size_t>(m) * d_model * 2, 1024) : 0;
  *h_off = xs;
  return xs + align_up(static_cast<size_t>(m) * d_ff * 2, 1024);
}

int segkv_ffn_workspace_size(int m, int d_model, int d_ff, size_t* bytes) {
  if (m < 0 || d_model <= 0 || d_ff <= 0 || !bytes) return SEGKV_ERR_INVALID_ARG;
  size_t off;
  *bytes = ffn_ws_parts(m, d_model, d_ff, true, &off);
  return SEGKV_OK;
}

int segkv_sparse_ffn(segkv_t h, const void* x, void* residual, int64_t n_rows, const int32_t* idx,
                     int m, const void* w_gate, const void* w_up, const void* w_down, int d_model,
                     int d_ff, void* workspace, size_t workspace_bytes, segkv_stream_t stream) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (h->host_only) return fail(h, SEGKV_ERR_INVALID_ARG, "host-only handle has no device");
  if (m < 0 || n_rows < 0 || n_rows > INT32_MAX || m > n_rows || (!idx && m != n_rows))
    return fail(h, SEGKV_ERR_INVALID_ARG, "bad m=%d / n_rows=%lld (idx NULL needs m = n_rows)", m,
                static_cast<long long>(n_rows));
  if (d_model < 64 || d_model % 64 || d_ff < 128 || d_ff % 128)
    return fail(h, SEGKV_ERR_INVALID_ARG, "d_model must be a multiple of 64, d_ff of 128");
  if (m == 0) return SEGKV_OK;
  const uintptr_t al = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(residual) |
                       reinterpret_cast<uintptr_t>(w_gate) | reinterpret_cast<uintptr_t>(w_up) |
                       reinterpret_cast<uintptr_t>(w_down) | reinterpret_cast<uintptr_t>(workspace);
  if (!x || !residual || !w_gate || !w_up || !w_down || !workspace || (al & 255))
    return fail(h, SEGKV_ERR_INVALID_ARG, "x, residual, weights and workspace: 256-byte aligned");
  size_t h_off;
  const size_t need = ffn_ws_parts(m, d_model, d_ff, idx != nullptr, &h_off);
  if (workspace_bytes < need)
    return fail(h, SEGKV_ERR_INVALID_ARG, "workspace needs %zu bytes, got %zu", need,
                workspace_bytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* hbuf = ws + h_off;
  const void* a1 = x;
  cudaError_t e;
  if (idx) {
    e = launch_gather_rows(x, idx, ws, m, d_model, n_rows, h->d_status, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "gather kernel launch");
    a1 = ws;
  }
  CUtensorMap ta1, tg, tu, ta2, td;
  if (encode_2d(&ta1, const_cast<void*>(a1), d_model, m, 128) != CUDA_SUCCESS ||
      encode_2d(&tg, const_cast<void*>(w_gate), d_model, d_ff, 128) != CUDA_SUCCESS ||
      encode_2d(&tu, const_cast<void*>(w_up), d_model, d_ff, 128) != CUDA_SUCCESS ||
      encode_2d(&ta2, hbuf, d_ff, m, 128) != CUDA_SUCCESS ||
      encode_2d(&td, const_cast<void*>(w_down), d_ff, d_model, 128) != CUDA_SUCCESS)
    return fail(h, SEGKV_ERR_CUDA, "tensor map encode failed for the FFN operands");
  const int tr = ffn_tile_rows();
  FfnGemmParams p{};
  p.M = m;
  p.K = d_model;
  p.tiles_m = (m + tr - 1) / tr;
  p.tiles_n = d_ff / 128;
  p.n_out = d_ff;
  p.n_rows = n_rows;
  p.out = hbuf;
  p.idx = nullptr;
  p.status = h->d_status;
  p.timeout_ns = kTimeoutNs;
  const int sms = h->num_sms > 0 ? h->num_sms : 1;
  e = launch_ffn_gemm(0, ta1, tg, tu, p,
                      static_cast<int>(std::min<int64_t>(int64_t(p.tiles_m) * p.tiles_n, sms)), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "FFN gate/up GEMM launch");
  p.K = d_ff;
  p.tiles_n = (d_model + 255) / 256;
  p.n_out = d_model;
  p.out = residual;
  p.idx = idx;
  e = launch_ffn_gemm(1, ta2, td, td, p,
                      static_cast<int>(std::min<int64_t>(int64_t(p.tiles_m) * p.tiles_n, sms)), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "FFN down GEMM launch");
  return SEGKV_OK;
}

int segkv_status(segkv_t h, segkv_stream_t stream) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  if (h->host_only) return SEGKV_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, h->d_status, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "status read");
  if (v == kStatusBadIndex) {
    e = cudaMemset(h->d_status, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(h, e, "status clear");
    return fail(h, SEGKV_ERR_INVALID_ARG, "a device row index was out of range");
  }
  if (v != 0) {
    // a launch that gave up may have left decode merge counters non-zero
    e = cudaMemset(h->d_pair_cnt, 0, sizeof(int) * static_cast<size_t>(h->S) * h->Hkv);
    if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(h, e, "status clear");
    return fail(h, SEGKV_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait expired (code %d)", v);
  }
  return SEGKV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- helpers for
// the no-allocation decode entry point (decode_noalloc.cu)
namespace skv {

// Bytes of fp32 partials segkv_decode_attn would need for this call; 0 when
// the arguments are not valid (the decode call itself then reports why).
size_t decode_partials_bytes(segkv* h, int layer, const int32_t* seq_lens,
                             const int32_t* seq_ids, int n) {
  if (!h || layer < 0 || layer >= h->L || !seq_lens || !ids_valid(h, seq_ids, n)) return 0;
  const int64_t pairs = int64_t(n) * h->Hkv;
  size_t a, m;
  return decode_ws_bytes(h, pairs + decode_max_grid(h), h->G, &a, &m);
}

int set_error(segkv* h, int code, const char* msg) { return fail(h, code, "%s", msg); }

int handle_device(const segkv* h) { return h->host_only ? -1 : h->device; }

}  // namespace skv
