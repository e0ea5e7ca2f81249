// Oracle for head-segmented paged attention. TEST INFRASTRUCTURE ONLY.
//
// A plain, slow CPU restatement of what the library computes, used by the
// tests, by the smoke check and by the CPU-baseline leg of the benchmark to
// check the CUDA path. It shares no code, header or constant with the library
// and is never linked into it.
//
// Sources (RedKnot summary page, "让 KV Cache「按头分家」：小红书 RedKnot 如何重做
// 长文本推理新引擎"):
//  * section "头分类稀疏（Head-Class Sparsification）": each (layer, KV head) is
//    either global (needs the whole causal context) or local (needs only a
//    sliding window).
//  * section "SegPagedAttention（存储与执行底座）": the KV cache is paged per
//    (layer, head) segment, each head physically keeps only the tokens it
//    needs, and attention is the ordinary softmax attention over them with no
//    mask materialised.
//  * section "SegPaged Attention(段页注意力）": storage is per head, not per token.
// and the online softmax merge of the KV-cache architecture page ("KV Cache管理
// 架构演进概述", section 5.2): per-block softmax with the running maximum kept
// as an offset.
//
// Readings where the pages are silent (each is also listed in the design notes):
//  * window W counts the query itself: a local head at position p sees keys
//    max(0, p-W+1) .. p;
//  * eviction is lazy and page-granular: on an append of [a, a+T) a local
//    head keeps [max(0, a-W+1), a+T); a trim keeps [max(0, n-W+1), n); a page
//    k (positions [kP, (k+1)P)) is freed once (k+1)P <= s;
//  * one pool of page ids, lowest free id first; K and V use the same id;
//    within one call all evictions happen before all allocations, both in the
//    order (seq_ids order, head ascending, logical page ascending);
//  * query head hq reads KV head hq / (Hq/Hkv); softmax scale 1/sqrt(D).
//
// Everything here is fp64 on exactly widened bf16 inputs.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <map>
#include <set>
#include <vector>

namespace {

constexpr int OK = 0;
constexpr int INVALID_ARG = -1;
constexpr int OUT_OF_PAGES = -2;
constexpr int EVICTED = -3;
constexpr int GLOBAL_HEAD = 0;

double bf16_to_double(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// ---------------------------------------------------------------------------
// Part 1: kept sets and page tables.

struct Segment {
  int s = 0;                        // first kept position
  std::map<int, int> page_of;       // logical page k -> physical page id
};

struct State {
  int L, H, P, S, max_len;
  int num_pages;
  std::vector<uint8_t> head_class;  // [L][H]
  std::vector<int> window;          // [L]
  std::vector<int> n;               // [L][S] tracked length per layer
  std::vector<Segment> seg;         // [L][H][S]
  std::set<int> free_ids;           // ordered: begin() is the lowest free id

  Segment& at(int l, int h, int b) { return seg[(static_cast<size_t>(l) * H + h) * S + b]; }
  bool is_local(int l, int h) const { return head_class[l * H + h] != GLOBAL_HEAD; }
};

// New kept start of a head whose pending queries start at position q0: a
// global head keeps everything; a local head needs keys from q0-W+1 on.
int kept_start(const State& st, int l, int h, int old_s, int q0) {
  if (!st.is_local(l, h)) return old_s;
  int need = q0 - st.window[l] + 1;
  if (need < 0) need = 0;
  return need > old_s ? need : old_s;
}

bool seq_ids_valid(const State& st, const int32_t* seq_ids, int n) {
  std::set<int> seen;
  for (int i = 0; i < n; ++i) {
    if (seq_ids[i] < 0 || seq_ids[i] >= st.S) return false;
    if (!seen.insert(seq_ids[i]).second) return false;
  }
  return true;
}

// One eviction pass: which pages go when the kept start moves to new_s.
void pages_to_evict(const State& st, Segment& g, int new_s, std::vector<int>* out_k) {
  for (const auto& kv : g.page_of)
    if ((kv.first + 1) * st.P <= new_s) out_k->push_back(kv.first);
}

}  // namespace

extern "C" {

void* orc_state_create(int num_layers, int num_kv_heads, const uint8_t* head_class,
                       const int32_t* window, int page_size, int max_seqs, int max_seq_len,
                       int num_pages) {
  if (num_layers <= 0 || num_kv_heads <= 0 || page_size <= 0 || max_seqs <= 0 ||
      max_seq_len <= 0 || num_pages < 0)
    return nullptr;
  State* st = new State();
  st->L = num_layers; st->H = num_kv_heads; st->P = page_size; st->S = max_seqs;
  st->max_len = max_seq_len; st->num_pages = num_pages;
  st->head_class.assign(head_class, head_class + num_layers * num_kv_heads);
  st->window.assign(window, window + num_layers);
  for (int l = 0; l < num_layers; ++l) {
    if (st->window[l] < 1) { delete st; return nullptr; }
  }
  st->n.assign(static_cast<size_t>(num_layers) * max_seqs, 0);
  st->seg.assign(static_cast<size_t>(num_layers) * num_kv_heads * max_seqs, Segment());
  for (int i = 0; i < num_pages; ++i) st->free_ids.insert(i);
  return st;
}

void orc_state_destroy(void* h) { delete static_cast<State*>(h); }

int orc_free_pages(void* h) { return static_cast<int>(static_cast<State*>(h)->free_ids.size()); }

int orc_seq_len(void* h, int layer, int seq) {
  State* st = static_cast<State*>(h);
  return st->n[static_cast<size_t>(layer) * st->S + seq];
}

// Append tokens [a, a+T) of each listed sequence (a = its tracked length in
// this layer). Transactional: on any error nothing changes.
int orc_append(void* hnd, int layer, const int32_t* cu_seqlens, const int32_t* seq_ids, int n) {
  State& st = *static_cast<State*>(hnd);
  if (layer < 0 || layer >= st.L || n < 0) return INVALID_ARG;
  if (!seq_ids_valid(st, seq_ids, n)) return INVALID_ARG;
  if (n > 0 && cu_seqlens[0] != 0) return INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    int T = cu_seqlens[i + 1] - cu_seqlens[i];
    if (T < 0) return INVALID_ARG;
    int a = st.n[static_cast<size_t>(layer) * st.S + seq_ids[i]];
    if (static_cast<int64_t>(a) + T > st.max_len) return INVALID_ARG;
  }

  // Plan: evictions, then allocations, in (seq_ids order, head, page) order.
  struct Evict { int b, h, new_s; std::vector<int> ks; };
  struct Alloc { int b, h, k; };
  std::vector<Evict> ev;
  std::vector<Alloc> al;
  size_t freed = 0;
  for (int i = 0; i < n; ++i) {
    int b = seq_ids[i];
    int a = st.n[static_cast<size_t>(layer) * st.S + b];
    int T = cu_seqlens[i + 1] - cu_seqlens[i];
    for (int h = 0; h < st.H; ++h) {
      Segment& g = st.at(layer, h, b);
      Evict e{b, h, kept_start(st, layer, h, g.s, a), {}};
      pages_to_evict(st, g, e.new_s, &e.ks);
      freed += e.ks.size();
      ev.push_back(e);
    }
  }
  for (int i = 0; i < n; ++i) {
    int b = seq_ids[i];
    int a = st.n[static_cast<size_t>(layer) * st.S + b];
    int T = cu_seqlens[i + 1] - cu_seqlens[i];
    if (T == 0) continue;
    for (int h = 0; h < st.H; ++h) {
      const Segment& g = st.at(layer, h, b);
      for (int k = a / st.P; k <= (a + T - 1) / st.P; ++k)
        if (!g.page_of.count(k)) al.push_back({b, h, k});
    }
  }
  if (st.free_ids.size() + freed < al.size()) return OUT_OF_PAGES;

  for (const Evict& e : ev) {
    Segment& g = st.at(layer, e.h, e.b);
    for (int k : e.ks) {
      st.free_ids.insert(g.page_of[k]);
      g.page_of.erase(k);
    }
    g.s = e.new_s;
  }
  for (const Alloc& x : al) {
    int id = *st.free_ids.begin();
    st.free_ids.erase(st.free_ids.begin());
    st.at(layer, x.h, x.b).page_of[x.k] = id;
  }
  for (int i = 0; i < n; ++i)
    st.n[static_cast<size_t>(layer) * st.S + seq_ids[i]] += cu_seqlens[i + 1] - cu_seqlens[i];
  return OK;
}

// Local heads drop to the W-1 newest tokens (what the next query needs).
int orc_trim(void* hnd, int layer, const int32_t* seq_ids, int n) {
  State& st = *static_cast<State*>(hnd);
  if (layer < -1 || layer >= st.L || n < 0) return INVALID_ARG;
  if (!seq_ids_valid(st, seq_ids, n)) return INVALID_ARG;
  int l0 = layer < 0 ? 0 : layer, l1 = layer < 0 ? st.L : layer + 1;
  for (int l = l0; l < l1; ++l)
    for (int i = 0; i < n; ++i) {
      int b = seq_ids[i];
      int len = st.n[static_cast<size_t>(l) * st.S + b];
      for (int h = 0; h < st.H; ++h) {
        Segment& g = st.at(l, h, b);
        int new_s = kept_start(st, l, h, g.s, len);
        std::vector<int> ks;
        pages_to_evict(st, g, new_s, &ks);
        for (int k : ks) { st.free_ids.insert(g.page_of[k]); g.page_of.erase(k); }
        g.s = new_s;
      }
    }
  return OK;
}

int orc_free_seq(void* hnd, int seq) {
  State& st = *static_cast<State*>(hnd);
  if (seq < 0 || seq >= st.S) return INVALID_ARG;
  for (int l = 0; l < st.L; ++l) {
    for (int h = 0; h < st.H; ++h) {
      Segment& g = st.at(l, h, seq);
      for (const auto& kv : g.page_of) st.free_ids.insert(kv.second);
      g.page_of.clear();
      g.s = 0;
    }
    st.n[static_cast<size_t>(l) * st.S + seq] = 0;
  }
  return OK;
}

// Install a transferred segment set into an empty (layer, seq): every head
// gets length n and its own kept start s[h]; pages floor(s/P) .. floor((n-1)/P)
// are taken lowest id first, in (head ascending, page ascending) order.
// Transactional: on any error nothing changes.
int orc_import(void* hnd, int layer, int seq, int n, const int32_t* starts) {
  State& st = *static_cast<State*>(hnd);
  if (layer < 0 || layer >= st.L || seq < 0 || seq >= st.S || n < 0 || n > st.max_len)
    return INVALID_ARG;
  if (st.n[static_cast<size_t>(layer) * st.S + seq] != 0) return INVALID_ARG;
  size_t need = 0;
  for (int h = 0; h < st.H; ++h) {
    if (starts[h] < 0 || starts[h] > n) return INVALID_ARG;
    if (n > 0 && (n - 1) / st.P >= starts[h] / st.P) need += (n - 1) / st.P - starts[h] / st.P + 1;
  }
  if (st.free_ids.size() < need) return OUT_OF_PAGES;
  for (int h = 0; h < st.H; ++h) {
    Segment& g = st.at(layer, h, seq);
    g.s = starts[h];
    if (n == 0) continue;
    for (int k = starts[h] / st.P; k <= (n - 1) / st.P; ++k) {
      g.page_of[k] = *st.free_ids.begin();
      st.free_ids.erase(st.free_ids.begin());
    }
  }
  st.n[static_cast<size_t>(layer) * st.S + seq] = n;
  return OK;
}

// Segment (layer, head, seq): kept start, kept length, first logical page and
// the ids of its pages in logical order.
int orc_segment(void* hnd, int layer, int head, int seq, int32_t* start, int32_t* len,
                int32_t* first_page, int32_t* ids, int max_ids, int32_t* n_ids) {
  State& st = *static_cast<State*>(hnd);
  if (layer < 0 || layer >= st.L || head < 0 || head >= st.H || seq < 0 || seq >= st.S)
    return INVALID_ARG;
  const Segment& g = st.at(layer, head, seq);
  int n = st.n[static_cast<size_t>(layer) * st.S + seq];
  *start = g.s;
  *len = n - g.s;
  *first_page = g.page_of.empty() ? 0 : g.page_of.begin()->first;
  int c = 0;
  for (const auto& kv : g.page_of) {
    if (c < max_ids) ids[c] = kv.second;
    ++c;
  }
  *n_ids = c;
  return c <= max_ids ? OK : INVALID_ARG;
}

// ---------------------------------------------------------------------------
// Part 2: attention over explicit per-head key sets.
//
// Q: [q_tokens, hq, d]; token t belongs to sequence row_seq[t] at position
// row_pos[t]. K, V: [sum kv_len, hkv, d], sequence b at rows kv_off[b] ..
// kv_off[b]+kv_len[b]-1 (the logical sequence, not pages). seg_start[b*hkv+h]
// is the first key the segment still keeps. Only the tokens listed in rows[]
// are computed; o: [nrows, hq, d], lse (natural log): [nrows, hq].

static int visible_keys(int p, int n, int s, bool local, int window, std::vector<int>* keys) {
  if (p < 0 || p >= n) return INVALID_ARG;
  int need = local ? p - window + 1 : 0;
  if (need < 0) need = 0;
  if (need < s) return EVICTED;
  keys->clear();
  for (int j = s; j < n; ++j) {       // walk the kept set [s, n)
    if (j > p) continue;              // causal
    if (local && j < p - window + 1) continue;  // outside the window
    keys->push_back(j);
  }
  return OK;
}

int orc_attention(int hq, int hkv, int d, double scale, const uint16_t* q,
                  const int32_t* row_seq, const int32_t* row_pos, const int64_t* kv_off,
                  const int32_t* kv_len, const uint16_t* k, const uint16_t* v,
                  const uint8_t* head_class, int window, const int32_t* seg_start,
                  const int64_t* rows, int64_t nrows, double* o, double* lse) {
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || window < 1) return INVALID_ARG;
  const int G = hq / hkv;
  int status = OK;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int64_t r = 0; r < nrows; ++r) {
    for (int qh = 0; qh < hq; ++qh) {
      const int64_t t = rows[r];
      const int b = row_seq[t], p = row_pos[t], h = qh / G;
      const bool local = head_class[h] != GLOBAL_HEAD;
      std::vector<int> keys;
      int rc = visible_keys(p, kv_len[b], seg_start[b * hkv + h], local, window, &keys);
      double* orow = o + (r * hq + qh) * d;
      if (rc != OK) {
#pragma omp critical
        status = rc;
        continue;
      }
      std::vector<double> qv(d), sc(keys.size());
      for (int c = 0; c < d; ++c) qv[c] = bf16_to_double(q[(t * hq + qh) * d + c]);
      double m = -std::numeric_limits<double>::infinity();
      for (size_t i = 0; i < keys.size(); ++i) {
        const uint16_t* kr = k + ((kv_off[b] + keys[i]) * hkv + h) * d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += qv[c] * bf16_to_double(kr[c]);
        sc[i] = scale * dot;
        if (sc[i] > m) m = sc[i];
      }
      double denom = 0.0;
      for (int c = 0; c < d; ++c) orow[c] = 0.0;
      for (size_t i = 0; i < keys.size(); ++i) {
        double w = std::exp(sc[i] - m);
        denom += w;
        const uint16_t* vr = v + ((kv_off[b] + keys[i]) * hkv + h) * d;
        for (int c = 0; c < d; ++c) orow[c] += w * bf16_to_double(vr[c]);
      }
      for (int c = 0; c < d; ++c) orow[c] /= denom;
      lse[r * hq + qh] = m + std::log(denom);
    }
  }
  return status;
}

// ---------------------------------------------------------------------------
// Part 3: the same attention computed block by block, each block reduced to
// (m, l, acc) and the blocks merged with the running-maximum offset. Used to
// check that splitting the key set changes nothing (the identity split-KV
// decode relies on).

int orc_attention_blocked(int hq, int hkv, int d, double scale, const uint16_t* q,
                          const int32_t* row_seq, const int32_t* row_pos, const int64_t* kv_off,
                          const int32_t* kv_len, const uint16_t* k, const uint16_t* v,
                          const uint8_t* head_class, int window, const int32_t* seg_start,
                          const int64_t* rows, int64_t nrows, int block, double* o, double* lse) {
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || window < 1 || block < 1) return INVALID_ARG;
  const int G = hq / hkv;
  int status = OK;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int64_t r = 0; r < nrows; ++r) {
    for (int qh = 0; qh < hq; ++qh) {
      const int64_t t = rows[r];
      const int b = row_seq[t], p = row_pos[t], h = qh / G;
      const bool local = head_class[h] != GLOBAL_HEAD;
      std::vector<int> keys;
      int rc = visible_keys(p, kv_len[b], seg_start[b * hkv + h], local, window, &keys);
      double* orow = o + (r * hq + qh) * d;
      if (rc != OK) {
#pragma omp critical
        status = rc;
        continue;
      }
      std::vector<double> qv(d);
      for (int c = 0; c < d; ++c) qv[c] = bf16_to_double(q[(t * hq + qh) * d + c]);
      // running state over the blocks merged so far
      double M = -std::numeric_limits<double>::infinity(), Lsum = 0.0;
      std::vector<double> acc(d, 0.0), bacc(d);
      for (size_t b0 = 0; b0 < keys.size(); b0 += block) {
        size_t b1 = b0 + block < keys.size() ? b0 + block : keys.size();
        std::vector<double> sc(b1 - b0);
        double m = -std::numeric_limits<double>::infinity();
        for (size_t i = b0; i < b1; ++i) {
          const uint16_t* kr = k + ((kv_off[b] + keys[i]) * hkv + h) * d;
          double dot = 0.0;
          for (int c = 0; c < d; ++c) dot += qv[c] * bf16_to_double(kr[c]);
          sc[i - b0] = scale * dot;
          if (sc[i - b0] > m) m = sc[i - b0];
        }
        double l = 0.0;
        for (int c = 0; c < d; ++c) bacc[c] = 0.0;
        for (size_t i = b0; i < b1; ++i) {
          double w = std::exp(sc[i - b0] - m);
          l += w;
          const uint16_t* vr = v + ((kv_off[b] + keys[i]) * hkv + h) * d;
          for (int c = 0; c < d; ++c) bacc[c] += w * bf16_to_double(vr[c]);
        }
        // merge block (m, l, bacc) into (M, Lsum, acc)
        double Mn = m > M ? m : M;
        double a_old = std::exp(M - Mn), a_new = std::exp(m - Mn);
        Lsum = Lsum * a_old + l * a_new;
        for (int c = 0; c < d; ++c) acc[c] = acc[c] * a_old + bacc[c] * a_new;
        M = Mn;
      }
      for (int c = 0; c < d; ++c) orow[c] = acc[c] / Lsum;
      lse[r * hq + qh] = M + std::log(Lsum);
    }
  }
  return status;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Part 4: rotary position re-alignment of cached keys (RedKnot summary page,
// section "Elastic Sparsity（弹性稀疏恢复）": reuse starts by aligning RoPE
// positions). A key rotated for position p becomes the key for position
// p + delta by rotating every dimension pair i by delta * theta_i, with
// theta_i = base^(-2i / rotary_dim). Pairs are (2i, 2i+1) for the interleaved
// layout (style 0) or (i, i + rotary_dim/2) for the split-half layout
// (style 1); dimensions at or beyond rotary_dim are left unchanged.
// x: rows x d values (fp64), rotated in place by pos[row] positions.
extern "C" int orc_rope(double* x, int64_t rows, int d, int rotary_dim, int style, double base,
                        const double* pos) {
  if (d <= 0 || rotary_dim <= 0 || rotary_dim > d || rotary_dim % 2 || style < 0 || style > 1)
    return INVALID_ARG;
  const int half = rotary_dim / 2;
  for (int64_t r = 0; r < rows; ++r) {
    double* v = x + r * d;
    for (int i = 0; i < half; ++i) {
      const double theta = std::pow(base, -2.0 * i / rotary_dim);
      const double ang = pos[r] * theta;
      const double c = std::cos(ang), s = std::sin(ang);
      const int a = style == 0 ? 2 * i : i;
      const int b = style == 0 ? 2 * i + 1 : i + half;
      const double xa = v[a], xb = v[b];
      v[a] = xa * c - xb * s;
      v[b] = xa * s + xb * c;
    }
  }
  return OK;
}

// ---------------------------------------------------------------------------
// Part 5: attention mass received by each key (RedKnot summary page, section
// "稀疏 FFN（Sparse FFN）": the dense FFN runs only on the tokens with the
// highest attention scores, the others take the residual identity path).
// Reading: a token's score is the softmax probability it receives as a key,
// summed over the listed query rows and over every query head. Per KV head h
// the sum over its query heads goes to mass[h * nkeys + kv_off[b] + j] for
// key j of sequence b. The probabilities are those of the attention above:
// each query's softmax over exactly its visible keys.
extern "C" int orc_attn_mass(int hq, int hkv, int d, double scale, const uint16_t* q,
                             const int32_t* row_seq, const int32_t* row_pos,
                             const int64_t* kv_off, const int32_t* kv_len, int nseq,
                             const uint16_t* k, const uint8_t* head_class, int window,
                             const int32_t* seg_start, int64_t nq, int64_t nkeys, double* mass) {
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || window < 1 || nseq < 0) return INVALID_ARG;
  const int G = hq / hkv;
  for (int64_t i = 0; i < int64_t(hkv) * nkeys; ++i) mass[i] = 0.0;
  int status = OK;
  // one (sequence, KV head) per task: each task owns its slice of mass
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int b = 0; b < nseq; ++b) {
    for (int h = 0; h < hkv; ++h) {
      const bool local = head_class[h] != GLOBAL_HEAD;
      double* mrow = mass + int64_t(h) * nkeys + kv_off[b];
      std::vector<int> keys;
      std::vector<double> qv(d), sc;
      for (int64_t t = 0; t < nq; ++t) {
        if (row_seq[t] != b) continue;
        int rc = visible_keys(row_pos[t], kv_len[b], seg_start[b * hkv + h], local, window, &keys);
        if (rc != OK) {
#pragma omp critical
          status = rc;
          continue;
        }
        for (int qh = h * G; qh < (h + 1) * G; ++qh) {
          for (int c = 0; c < d; ++c) qv[c] = bf16_to_double(q[(t * hq + qh) * d + c]);
          sc.assign(keys.size(), 0.0);
          double m = -std::numeric_limits<double>::infinity();
          for (size_t i = 0; i < keys.size(); ++i) {
            const uint16_t* kr = k + ((kv_off[b] + keys[i]) * hkv + h) * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += qv[c] * bf16_to_double(kr[c]);
            sc[i] = scale * dot;
            if (sc[i] > m) m = sc[i];
          }
          double denom = 0.0;
          for (size_t i = 0; i < keys.size(); ++i) {
            sc[i] = std::exp(sc[i] - m);
            denom += sc[i];
          }
          for (size_t i = 0; i < keys.size(); ++i) mrow[keys[i]] += sc[i] / denom;
        }
      }
    }
  }
  return status;
}
