/*
 * segkv — head-segmented paged KV attention for one GB300 (sm_103a).
 *
 * The KV cache is paged per (layer, KV head) segment. Each head keeps only
 * the keys it needs: a global head the whole causal context, a local head a
 * sliding window. Attention runs over those segments with no mask ever
 * materialised. Sources (RedKnot summary page, "让 KV Cache「按头分家」：小红书
 * RedKnot 如何重做长文本推理新引擎"):
 *   - section "头分类稀疏（Head-Class Sparsification）": offline global/local
 *     classification of every (layer, head);
 *   - section "SegPagedAttention（存储与执行底座）": paged KV store segmented per
 *     (layer, head), one fused varlen attention kernel over it, each head keeps
 *     only the tokens it needs, no attn_mask;
 *   - section "SegPaged Attention(段页注意力）": storage per head, not per token;
 * and the KV-cache architecture page ("KV Cache管理架构演进概述"), section 3.1
 * (pages of a fixed token count mapped through a logical-to-physical table)
 * and section 5.2 (block-wise softmax merged with a running maximum).
 *
 * Conventions shared by every call:
 *   - Shapes. Lq query heads per KV head: G = num_q_heads / num_kv_heads;
 *     query head hq reads KV head hq / G. D = head_dim (64 or 128).
 *     P = page_size tokens per page.
 *   - Readings where the pages are silent. Window W counts the query: a
 *     local head at position p sees keys max(0, p-W+1) .. p. Eviction is lazy
 *     and page-granular: an append of positions [a, a+T) lets a local head
 *     drop keys below a-W+1 (what the new tokens' queries still need); a
 *     trim drops them below n-W+1 (what the next token needs); a page k
 *     (positions [kP, (k+1)P)) is freed once (k+1)P <= kept start. Page ids
 *     come from one pool, lowest free id first; K and V of a page share its
 *     id; within one call all evictions precede all allocations, both in the
 *     order (seq_ids order, head ascending, logical page ascending).
 *   - Memory. Pointers named "device" are device memory owned by the caller;
 *     arrays named "host" are host memory read during the call only, so the
 *     host never waits on the device to plan work. K/V pools are bf16
 *     [num_pages, P, D] each, owned by the caller for the handle's lifetime.
 *   - Streams. Every device-side effect is ordered on the stream passed in
 *     (NULL = legacy default stream). Host-side state (lengths, page tables)
 *     changes when the call returns, so calls must be made in stream order
 *     and all calls on one handle must use one stream (or the caller orders
 *     them). A handle is not thread-safe.
 *   - Errors. Every call returns SEGKV_OK or a negative SEGKV_ERR_* code and
 *     records a message (segkv_last_error). A failing call changes no state.
 *     Device-side faults that the kernels catch themselves (a bounded wait
 *     that timed out) are reported by segkv_status.
 */
#ifndef SEGKV_H_
#define SEGKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct segkv* segkv_t;
/* A cudaStream_t passed as an opaque pointer (NULL = legacy default stream). */
typedef void* segkv_stream_t;

enum { SEGKV_GLOBAL = 0, SEGKV_LOCAL = 1 };

enum {
  SEGKV_OK = 0,
  SEGKV_ERR_INVALID_ARG = -1,   /* bad argument or shape; nothing changed */
  SEGKV_ERR_OUT_OF_PAGES = -2,  /* the pool cannot hold the append; nothing changed */
  SEGKV_ERR_EVICTED = -3,       /* a query needs a key its head no longer keeps */
  SEGKV_ERR_CUDA = -4,          /* a CUDA runtime call failed */
  SEGKV_ERR_DEVICE_TIMEOUT = -5 /* a kernel's bounded wait expired (segkv_status) */
};

enum { SEGKV_WS_PREFILL = 0, SEGKV_WS_DECODE = 1 };

typedef struct segkv_stats {
  int64_t num_pages;         /* pool size */
  int64_t pages_in_use;      /* pages held by any segment */
  int64_t pages_global;      /* held by global-head segments */
  int64_t pages_local;       /* held by local-head segments */
  int64_t kept_tokens;       /* sum over segments of kept length */
  int64_t upload_bytes;      /* bytes of plans uploaded so far (host -> device) */
} segkv_stats_t;

/*
 * segkv_create — set up the segment tables over caller-owned page pools.
 * Defines the head classes (summary page, section "头分类稀疏") and the paged
 * per-(layer, head) store (section "SegPagedAttention").
 *   head_class  host uint8 [num_layers * num_kv_heads], SEGKV_GLOBAL/LOCAL.
 *   window      host int32 [num_layers], W >= 1, used by local heads.
 *   page_size   P, a multiple of 8 that divides 128 or is a multiple of 128.
 *   max_seqs    sequence slots; seq ids are 0 .. max_seqs-1.
 *   max_seq_len longest sequence (positions 0 .. max_seq_len-1).
 *   k_pool, v_pool  device bf16 [num_pages, P, D], 16-byte aligned. Both
 *               NULL (with num_pages > 0) gives a host-only handle that plans
 *               and tracks pages but launches nothing (attention calls then
 *               return SEGKV_ERR_INVALID_ARG).
 *   softmax_scale  <= 0 selects 1/sqrt(D).
 * Allocates the device block table int32 [L][Hkv][max_seqs][ceil(max_seq_len/P)],
 * a device status word and pinned/device upload rings. The current CUDA
 * device at create is the handle's device.
 * Errors: INVALID_ARG for bad shapes (G must divide 128; D in {64, 128}),
 * CUDA if an allocation fails.
 */
int segkv_create(segkv_t* out, int num_layers, int num_q_heads, int num_kv_heads, int head_dim,
                 const uint8_t* head_class, const int32_t* window, int page_size, int max_seqs,
                 int max_seq_len, void* k_pool, void* v_pool, int64_t num_pages,
                 float softmax_scale);

/* segkv_destroy — synchronises the device and frees what segkv_create made. */
int segkv_destroy(segkv_t h);

/*
 * segkv_append — write new tokens into every head's segment (BUILDSTATE).
 * Each head physically keeps only the keys its pending queries need (summary
 * page, section "SegPagedAttention"): first the local heads' pages that fell
 * out of the window are freed, then pages for the new tokens are taken, then
 * the append kernel scatters K/V rows into them.
 *   k, v        device bf16 [cu_seqlens[n], Hkv, D], token-major.
 *   cu_seqlens  host int32 [n+1], cu_seqlens[0] = 0, non-decreasing; sequence
 *               i appends tokens cu_seqlens[i] .. cu_seqlens[i+1]-1 at its
 *               positions a_i .. a_i+T_i-1, a_i = its tracked length in layer.
 *   seq_ids     host int32 [n], distinct.
 * Errors: INVALID_ARG (bad ids, length beyond max_seq_len), OUT_OF_PAGES.
 */
int segkv_append(segkv_t h, int layer, const void* k, const void* v, const int32_t* cu_seqlens,
                 const int32_t* seq_ids, int n, segkv_stream_t stream);

/*
 * segkv_prefill_attn — varlen attention of packed queries over the segments
 * (EXECUTE; summary page, section "SegPagedAttention": one fused varlen
 * kernel, no attn_mask). For query token t of sequence i at position
 * p = q_pos[t] and query head hq (KV head h = hq / G):
 *   O[t, hq] = softmax_j(scale * q . k_j) v_j over kept keys j <= p, and for a
 *   local head also j >= p-W+1;  lse[hq, t] = log sum_j exp(scale * q . k_j).
 *   q       device bf16 [cu_seqlens[n], Hq, D].
 *   cu_seqlens host int32 [n+1]; q_pos host int32 [cu_seqlens[n]], each < the
 *           sequence's tracked length (append first); seq_ids host int32 [n].
 *   o       device bf16 [cu_seqlens[n], Hq, D]; lse device fp32 [Hq, cu_seqlens[n]]
 *           (natural log) or NULL.
 *   workspace, workspace_bytes  unused by this call (pass NULL, 0).
 * The kernel's CTAs claim work units at run time (from a counter in the
 * call's own uploaded plan), but every unit is computed in a fixed order, so
 * repeated calls return the same bits.
 * Errors: INVALID_ARG, EVICTED (a local head already dropped a needed key).
 */
int segkv_prefill_attn(segkv_t h, int layer, const void* q, const int32_t* cu_seqlens,
                       const int32_t* q_pos, const int32_t* seq_ids, int n, void* o, float* lse,
                       void* workspace, size_t workspace_bytes, segkv_stream_t stream);

/*
 * segkv_decode_attn — one query token per sequence at position seq_len-1
 * against its segments: split-KV partials over key chunks, then a combine
 * pass that merges them with the running-maximum rule (KV-cache architecture
 * page, section 5.2).
 *   q         device bf16 [n, Hq, D]; o device bf16 [n, Hq, D].
 *   seq_lens  host int32 [n], must equal each sequence's tracked length.
 *   seq_ids   host int32 [n], distinct.
 *   workspace device, >= segkv_workspace_size(SEGKV_WS_DECODE, n, n) bytes,
 *             256-byte aligned; holds the fp32 partials.
 * Errors: INVALID_ARG (length mismatch, small workspace), EVICTED.
 */
int segkv_decode_attn(segkv_t h, int layer, const void* q, const int32_t* seq_lens,
                      const int32_t* seq_ids, int n, void* o, void* workspace,
                      size_t workspace_bytes, segkv_stream_t stream);

/*
 * segkv_trim — let local heads of the listed sequences drop every key the
 * next token's query will not see (keep the W-1 newest); layer -1 = all
 * layers. Host-only bookkeeping: freed pages are reused by later appends,
 * which are stream-ordered after earlier reads.
 */
int segkv_trim(segkv_t h, int layer, const int32_t* seq_ids, int n);

/* segkv_free_seq — return every page of a sequence in every layer; its
 * tracked lengths become 0. */
int segkv_free_seq(segkv_t h, int seq_id);

/* segkv_workspace_size — device workspace a call needs. kind SEGKV_WS_DECODE:
 * n_seqs sequences with n_tokens query tokens in all (n_tokens = n_seqs for
 * segkv_decode_attn, n*T for segkv_decode_attn_multi); SEGKV_WS_PREFILL: 0. */
int segkv_workspace_size(segkv_t h, int kind, int64_t n_tokens, int n_seqs, size_t* bytes);

/*
 * segkv_rope_shift — re-align the cached keys of one sequence to a position
 * offset (RedKnot summary page, section "Elastic Sparsity（弹性稀疏恢复）": reuse
 * of a cached segment at another position starts with RoPE position
 * alignment). Every kept key of the selected KV heads of (layer, seq) is
 * rotated in place: dimension pair i turns by delta * base^(-2i/rotary_dim),
 * which maps a key encoded for position p to the key for position p + delta.
 *   style       SEGKV_ROPE_INTERLEAVED: pairs (2i, 2i+1);
 *               SEGKV_ROPE_HALF: pairs (i, i + rotary_dim/2).
 *   rotary_dim  even, 2 .. head_dim; dimensions beyond it are unchanged.
 *   head_mask   bit h selects KV head h.
 * Angles are formed in fp64 on the host; the rotation runs in fp32 and each
 * key is rounded once to bf16. V, page tables and tracked lengths are
 * unchanged. Errors: INVALID_ARG.
 */
enum { SEGKV_ROPE_INTERLEAVED = 0, SEGKV_ROPE_HALF = 1 };
int segkv_rope_shift(segkv_t h, int layer, int seq, int32_t delta, double base, int rotary_dim,
                     int style, uint64_t head_mask, segkv_stream_t stream);

/*
 * segkv_export — pack one sequence's kept K/V of a layer into a contiguous
 * buffer for transfer (RedKnot summary page, section "系统收益": with prefill
 * and decode disaggregated, only each head's kept tokens need to move).
 * Layout: for KV head h = 0 .. Hkv-1: K rows [s_h, n) then V rows [s_h, n),
 * each bf16 [n - s_h, D]; heads back to back.
 *   header   host int32 [1 + Hkv], written: n, then s_h for every head.
 *   out      device, 16-byte aligned, >= segkv_export_size bytes. out = NULL
 *            with out_bytes = 0 only fills the header.
 * The segment itself is unchanged. Errors: INVALID_ARG.
 */
int segkv_export_size(segkv_t h, int layer, int seq, size_t* bytes);
int segkv_export(segkv_t h, int layer, int seq, void* out, size_t out_bytes, int32_t* header,
                 segkv_stream_t stream);

/*
 * segkv_import — install an exported sequence as (layer, seq), which must be
 * empty in that layer: tracked length n and kept start s_h per head from the
 * header; pages floor(s_h/P) .. floor((n-1)/P) are taken lowest id first in
 * (head ascending, page ascending) order and the rows are scattered into
 * them. The exporter must have had the same Hkv and D.
 *   in       device buffer from segkv_export (NULL on a host-only handle).
 *   header   host int32 [1 + Hkv] from segkv_export.
 * Errors: INVALID_ARG (seq not empty, bad header, short buffer),
 * OUT_OF_PAGES; both change nothing.
 */
int segkv_import(segkv_t h, int layer, int seq, const void* in, size_t in_bytes,
                 const int32_t* header, segkv_stream_t stream);

/*
 * segkv_set_window_convention — choose what a local head's window W covers.
 *   SEGKV_WINDOW_INCLUSIVE (default): W keys including the query,
 *     p-W+1 .. p (the reading this library takes of the summary page's
 *     "sliding window", section "头分类稀疏").
 *   SEGKV_WINDOW_FA: W+1 keys p-W .. p, the convention of FlashAttention's
 *     window_size = (W, 0).
 * Allowed only while the handle holds no tokens (every tracked length 0);
 * kept sets, eviction and attention all follow the chosen convention.
 * Errors: INVALID_ARG.
 */
enum { SEGKV_WINDOW_INCLUSIVE = 0, SEGKV_WINDOW_FA = 1 };
int segkv_set_window_convention(segkv_t h, int convention);

/*
 * segkv_decode_attn_multi — decode with T query tokens per sequence
 * (speculative or chunked decoding): the T newest tokens of each sequence,
 * at positions seq_len-T .. seq_len-1, attend causally over their segments
 * (each also to the earlier of the T; a local head's token at p to keys
 * p-W+1 .. p). When T * (Hq/Hkv) is 1, 2, 4, 8 or 16 the T*G query rows of
 * a KV head share every K/V read in the split-KV decode kernel; otherwise
 * the call runs on the prefill tensor-core kernel.
 *   q         device bf16 [n*T, Hq, D], sequence i's tokens at rows i*T .. i*T+T-1.
 *   seq_lens  host int32 [n], must equal each sequence's tracked length (>= T).
 *   o         device bf16 [n*T, Hq, D]; lse device fp32 [Hq, n*T] or NULL
 *             (natural log of each row's softmax denominator, scaled scores).
 *   workspace device, >= segkv_workspace_size(SEGKV_WS_DECODE, n*T, n) bytes,
 *             256-byte aligned (may be NULL when that size is 0).
 * Errors: INVALID_ARG, EVICTED.
 */
int segkv_decode_attn_multi(segkv_t h, int layer, const void* q, int T, const int32_t* seq_lens,
                            const int32_t* seq_ids, int n, void* o, float* lse, void* workspace,
                            size_t workspace_bytes, segkv_stream_t stream);

/*
 * segkv_attn_mass — the attention score of every token of a prefill chunk:
 * the softmax mass it receives as a key (RedKnot summary page, section
 * "稀疏 FFN（Sparse FFN）": the dense FFN runs only on the tokens with the
 * highest attention scores; the page does not define the score, and this
 * library reads it as the mass a token receives). For sequence i of the
 * call, the chunk is its tokens cu_seqlens[i] .. cu_seqlens[i+1]-1 at
 * consecutive positions a_i .. a_i+T_i-1 (q_pos), already appended; for each
 * key j of the chunk and KV head h:
 *   mass[h, t(j)] = sum over the chunk's queries p >= j that see j (local
 *                   heads: j >= p-W+1) and over the G query heads of h of
 *                   exp(scale q.k_j - lse_q)
 *   q         device bf16 [Σq, Hq, D], the chunk's queries (as for prefill).
 *   lse       device fp32 [Hq, Σq]: the LSE segkv_prefill_attn wrote for them.
 *   mass      device fp32 [Hkv, Σq], written for every token.
 * Summation order is fixed, so results repeat bit for bit.
 * Errors: INVALID_ARG (positions not consecutive, chunk beyond the tracked
 * length), EVICTED.
 */
int segkv_attn_mass(segkv_t h, int layer, const void* q, const int32_t* cu_seqlens,
                    const int32_t* q_pos, const int32_t* seq_ids, int n, const float* lse,
                    float* mass, segkv_stream_t stream);

/*
 * segkv_topk_tokens — choose the tokens that go through the FFN (section
 * "稀疏 FFN（Sparse FFN）"): score[t] = sum over h of mass[h, t] (fp32, in
 * head order); for sequence i, the k[i] tokens of cu_seqlens[i] ..
 * cu_seqlens[i+1]-1 with the largest score, ties to the lower position.
 *   mass      device fp32 [Hkv, Σq] from segkv_attn_mass (scores must be >= 0).
 *   k         host int32 [n], 0 <= k[i] <= the sequence's tokens.
 *   score     device fp32 [Σq], receives the summed score.
 *   idx       device int32 [Σ k]: sequence i's chosen token rows (global
 *             rows, cu_seqlens[i] + t) at idx[Σ_{j<i} k[j] ...], ascending.
 * Errors: INVALID_ARG.
 */
int segkv_topk_tokens(segkv_t h, const float* mass, const int32_t* cu_seqlens, int n,
                      const int32_t* k, float* score, int32_t* idx, segkv_stream_t stream);

/*
 * segkv_sparse_ffn — the dense FFN on chosen rows only (RedKnot summary page,
 * section "稀疏 FFN（Sparse FFN）": the tokens with the highest attention
 * scores go through the dense FFN, every other token takes the residual
 * identity path). The FFN is the gated SwiGLU MLP of the models the page
 * names (a reading; the page gives no formula):
 *   for r < m:  residual[idx[r]] += W_down (silu(W_gate x[idx[r]]) * (W_up x[idx[r]]))
 * with silu(g) = g / (1 + e^-g). Rows not in idx are neither read nor written.
 *   x         device bf16 [n_rows, d_model], the FFN input (normalised hidden state).
 *   residual  device bf16 [n_rows, d_model], updated in place (one rounding per element).
 *   idx       device int32 [m], distinct row ids in [0, n_rows); NULL = every row
 *             (the dense FFN; then m must equal n_rows). An id out of range is
 *             skipped and segkv_status reports SEGKV_ERR_INVALID_ARG.
 *   w_gate, w_up  device bf16 [d_ff, d_model]; w_down device bf16 [d_model, d_ff].
 *   d_model   a multiple of 64; d_ff a multiple of 128.
 *   workspace device, >= segkv_ffn_workspace_size(m, d_model, d_ff) bytes; it
 *             holds the gathered rows and the bf16 hidden activations h.
 * Pointers 256-byte aligned. The caller owns every buffer. fp32 accumulation
 * on the tensor cores; h is rounded to bf16 before W_down.
 * Errors: INVALID_ARG, CUDA.
 */
int segkv_sparse_ffn(segkv_t h, const void* x, void* residual, int64_t n_rows, const int32_t* idx,
                     int m, const void* w_gate, const void* w_up, const void* w_down, int d_model,
                     int d_ff, void* workspace, size_t workspace_bytes, segkv_stream_t stream);
int segkv_ffn_workspace_size(int m, int d_model, int d_ff, size_t* bytes);

/*
 * segkv_get_segment — host copy of one segment's table: kept start, kept
 * length, first logical page and the page ids in logical order (at most
 * max_ids written; *n_ids gets the count).
 */
int segkv_get_segment(segkv_t h, int layer, int head, int seq, int32_t* start, int32_t* len,
                      int32_t* first_page, int32_t* ids, int max_ids, int32_t* n_ids);

/* segkv_seq_len — tracked length of a sequence in a layer (host). */
int segkv_seq_len(segkv_t h, int layer, int seq, int32_t* len);

/* segkv_stats — page and token counts (host). */
int segkv_stats(segkv_t h, segkv_stats_t* out);

/*
 * segkv_status — synchronise the stream, read and clear the device status
 * word. Returns SEGKV_OK, SEGKV_ERR_DEVICE_TIMEOUT if a kernel's bounded wait
 * expired (that launch's outputs are undefined; the context stays usable),
 * or SEGKV_ERR_CUDA.
 */
int segkv_status(segkv_t h, segkv_stream_t stream);

/* segkv_last_error — message of the last failing call on h (or of a failed
 * create when h is NULL). */
const char* segkv_last_error(segkv_t h);

/*
 * segkv_decode_attn_noalloc — segkv_decode_attn without a caller workspace,
 * for callers that cannot allocate device memory when they decode (runtimes
 * that forbid cudaMalloc on the serving path, or that cannot size a
 * workspace per call). The paper has no counterpart; this is a packaging
 * choice of the library.
 *   The split partials live in a fixed device array inside the library,
 *   SEGKV_NOALLOC_SCRATCH_BYTES (8 MiB) per GPU, held by every GPU that loads
 *   the library until the process exits. A call whose partials could exceed
 *   it (a decode plan has at most n*Hkv + 2*SMs split units of G*(D+2)*4
 *   bytes each: about 3,700 (sequence, KV head) pairs at G=4, D=128) returns
 *   SEGKV_ERR_INVALID_ARG with a message; use segkv_decode_attn then.
 *   The call allocates no memory. Its first call on a device looks up the
 *   array's device address (cudaGetSymbolAddress) with the handle's device
 *   current, so make that first call before any stream capture. The address
 *   is kept for the life of the process: after a cudaDeviceReset (which also
 *   invalidates every handle on that device) this entry point may not be
 *   used again in the same process.
 *   Every call shares the one array: calls that overlap on the GPU (other
 *   streams, other handles) race. The caller clears nothing: each call
 *   resets, on its stream, the counters it keeps there.
 *   Other arguments, errors and results are those of segkv_decode_attn; the
 *   handle's device must be the current device.
 */
#define SEGKV_NOALLOC_SCRATCH_BYTES (8u << 20)
int segkv_decode_attn_noalloc(segkv_t h, int layer, const void* q, const int32_t* seq_lens,
                              const int32_t* seq_ids, int n, void* o, segkv_stream_t stream);

/* segkv_plan_prefill — the work plan that segkv_prefill_attn would use,
 * computed on the host only (no device work; host-only handles work too), for
 * tests and tools. A unit is one KV head x the query rows of two 128-row tiles
 * (2 x 128 / G tokens of one sequence). The units are listed in claim order:
 * descending key tiles, ties in building order (sequence, first token, KV
 * head). The kernel's CTA c runs unit c first; each CTA that finishes a unit
 * claims the next unclaimed unit of the list, so which CTA runs a later unit
 * is decided on the GPU.
 *   num_ctas    > 0: plan for that many CTAs (at most 65,535, else
 *               SEGKV_ERR_INVALID_ARG); otherwise one per SM.
 *   units       host int32 [max_units][8], out: first token (index into the
 *               call's packed tokens), tokens, KV head, 1 if local, key tiles
 *               kt0 .. kt1 (128 keys each), lowest and highest key any of
 *               its rows sees.
 *   n_units     out: the number of units, written even when the array is
 *               too small (then SEGKV_ERR_INVALID_ARG).
 *   n_ctas      out: the grid, min(n_units, num_ctas).
 * Errors: those of segkv_prefill_attn for the same arguments. */
int segkv_plan_prefill(segkv_t h, int layer, const int32_t* cu_seqlens, const int32_t* q_pos,
                       const int32_t* seq_ids, int n, int num_ctas, int32_t* units, int max_units,
                       int* n_units, int* n_ctas);

/* segkv_plan_mass — the work plan that segkv_attn_mass would use for the same
 * chunks, computed on the host only (host-only handles work too), for tests
 * and tools. A unit is one KV head x one key tile of 128 positions of one
 * chunk, over the query tiles (128 / G tokens each, chunk-relative) that see
 * some of its keys; a key tile seen by many query tiles is cut into pieces.
 * Units are dealt to num_ctas lists by longest-processing-time-first.
 *   num_ctas    > 0: plan for that many CTAs (at most 65,535, else
 *               SEGKV_ERR_INVALID_ARG); otherwise one per SM.
 *   units       host int32 [max_units][12], out: first token of the chunk
 *               (index into the call's packed tokens), chunk length, position
 *               of its first token, KV head, 1 if local, key tile, query
 *               tiles qt0 .. qt1, piece, pieces of its key tile, first
 *               partial-sum slot of the key tile, the key tile's counter
 *               (the last two 0 for a key tile in one piece).
 *   cta_begin   host int32 [max_ctas + 1], out: list c holds units
 *               cta_begin[c] .. cta_begin[c + 1] - 1.
 *   n_units, n_ctas  out: the plan's sizes, written even when an output
 *               array is too small (then SEGKV_ERR_INVALID_ARG).
 * Errors: those of segkv_attn_mass for the same arguments. */
int segkv_plan_mass(segkv_t h, int layer, const int32_t* cu_seqlens, const int32_t* q_pos,
                    const int32_t* seq_ids, int n, int num_ctas, int32_t* units, int max_units,
                    int32_t* cta_begin, int max_ctas, int* n_units, int* n_ctas);

/* segkv_plan_decode — the work plan that segkv_decode_attn (T = 1) or
 * segkv_decode_attn_multi would use for the T newest tokens of n sequences,
 * computed on the host only (no device work; host-only handles work too), for
 * tests and tools. The plan is the stream-K cut of the (sequence, KV head) key
 * ranges into units, grouped by CTA.
 *   num_ctas    > 0: plan for that many CTAs; otherwise for the device's grid.
 *   units       host int32 [max_units][8], out: sequence index i of the call,
 *               KV head, 1 if local, keys [k0, k1), first unit of the unit's
 *               (sequence, head) pair, units of that pair, position of the
 *               sequence's newest query token.
 *   cta_begin   host int32 [max_ctas + 1], out: CTA c runs units
 *               cta_begin[c] .. cta_begin[c + 1] - 1.
 *   n_units, n_ctas  out: the plan's sizes, written even when an output
 *               array is too small (then SEGKV_ERR_INVALID_ARG).
 * Errors: those of segkv_decode_attn_multi for the same arguments. */
int segkv_plan_decode(segkv_t h, int layer, int T, const int32_t* seq_lens, const int32_t* seq_ids,
                      int n, int num_ctas, int32_t* units, int max_units, int32_t* cta_begin,
                      int max_ctas, int* n_units, int* n_ctas);

/* segkv_exp2_check — test hook for the two base-2 exponentials that the
 * prefill softmax uses to form p = 2^(s*scale*log2(e) - m) (online softmax
 * with the running maximum kept as an offset: KV-cache architecture page,
 * section 5.2). For i < n it writes
 *   y_poly[i] = the cubic on the FMA pipe (2^x = 2^i * 2^f, f in [-1/2, 1/2],
 *               2^f by the minimax cubic on relative error, max 7.48e-5;
 *               inputs below -125, -inf included, are clamped to -125, so
 *               they give 2^-125 within the same bound; the softmax never
 *               passes more than 8, and inputs above 127 are outside the
 *               domain),
 *   y_mufu[i] = the hardware ex2.approx.ftz (2^-inf = 0).
 * x, y_poly, y_mufu are device fp32 [n]; stream-ordered on stream.
 * Errors: SEGKV_ERR_INVALID_ARG (n < 0 or a NULL array), SEGKV_ERR_CUDA. */
int segkv_exp2_check(const float* x, float* y_poly, float* y_mufu, int n, segkv_stream_t stream);

/* segkv_set_debug — test hook. Bit 0: the next prefill launch makes one wait
 * on a barrier that nothing signals, with a short limit, so the timeout path
 * runs (status becomes SEGKV_ERR_DEVICE_TIMEOUT). Bits are cleared on use. */
int segkv_set_debug(segkv_t h, int flags);

#ifdef __cplusplus
}
#endif

#endif /* SEGKV_H_ */
