// Work descriptors shared by the host planner and the kernels, and the
// kernel launchers. Host code fills these structs into a pinned staging
// buffer; one cudaMemcpyAsync per call moves them next to the kernel.
#pragma once

#include <utility>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace skv {

// Launch a kernel as a programmatic dependent of the previous kernel on the
// stream: its CTAs may start while that kernel drains. The kernel must execute
// griddepcontrol.wait before it reads anything an earlier kernel wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kKeyTile = 128;     // prefill: keys per tile (one MMA N)
constexpr int kRowsPerTile = 128; // prefill: query rows per tile (MMA M)

// A small plan travels inside the kernel's parameters (no separate copy
// before the launch); larger ones go through the upload ring.
template <int N>
struct alignas(16) Blob {
  unsigned char data[N];
};
using PlanBlob = Blob<30 * 1024>;  // decode plans
using AppendBlob = Blob<8 * 1024>; // append plans (kernel parameters cost launch time)
constexpr int kMaxDevices = 64;

// ---- append -------------------------------------------------------------
struct AppendSeq {
  int32_t tok0;      // first packed token of this sequence's chunk
  int32_t pos0;      // its position (tracked length before the append)
  int32_t first_k;   // logical page of pos0
  int32_t n_pages;   // logical pages the chunk touches
  int32_t list_off;  // offset of this sequence's [Hkv][n_pages] page ids
  int32_t pad;
};
struct AppendTile {
  int32_t seq;   // index into AppendSeq
  int32_t tok0;  // first packed token of the tile
  int32_t ntok;
  int32_t pad;
};
struct AppendParams {
  const uint4* k;
  const uint4* v;
  uint4* kpool;
  uint4* vpool;
  const AppendSeq* seqs;
  const AppendTile* tiles;
  const int32_t* page_list;   // page ids, per sequence [Hkv][n_pages]
  const int64_t* table_idx;   // block-table slot of each page_list entry
  int32_t* table;
  int plan_inline;            // 1: the four arrays above are offsets into the AppendBlob
  int n_tiles;
  int n_entries;
  int hkv, vec_per_row, page_size;
};

// ---- prefill --------------------------------------------------------------
struct PrefillUnit {
  int32_t tok0;        // first packed query token of the tile
  int32_t ntok;        // tokens in the unit (<= 2 * 128 / G: two Q tiles)
  int32_t head;        // KV head
  int32_t local;       // 1 = local head
  int32_t kt0, kt1;    // key tiles kt0 .. kt1 (inclusive), tile = 128 positions
  int32_t klo, khi;    // union of the rows' visible keys
  int32_t vlo, vhi;    // the segment's written keys [vlo, vhi]: its start, its length - 1
  int32_t table_row;   // (layer * Hkv + head) * max_seqs + seq
  int32_t pos0;        // position of token tok0 + t is pos0 + t; -1: read q_pos
};
static_assert(sizeof(PrefillUnit) == 48, "prefill units are staged in 48-byte slots");
struct PrefillParams {
  const PrefillUnit* units;    // [n_units], in claim order (descending key tiles)
  int* next_unit;              // claim counter, 0 at launch: CTA c runs unit c first, and
                               // each later claim k gets unit grid + k
  const int32_t* q_pos;
  const int32_t* table;
  void* o;        // bf16 [total_q, Hq, D]
  float* lse;     // fp32 [Hq, total_q] or null
  int64_t total_q;
  int n_units;
  int R;          // block-table row length
  int hq, G, tpt, window;  // tpt = tokens per 128-row Q tile
  int page_size;
  int oob_row;    // a K/V row coordinate past the end of the pools
  float scale_log2;
  int* status;
  int debug;
  unsigned long long timeout_ns;
};

// ---- decode ---------------------------------------------------------------
struct DecodeUnit {
  int32_t req;         // sequence index i of the call (row i*T of q / o)
  int16_t head;        // KV head; the unit's pair (req, head) is req * Hkv + head
  int16_t local;       // 1: local head, each query row sees only its window
  int32_t k0, k1;      // keys [k0, k1)
  int32_t table_row;
  int32_t pair_unit0;  // first unit of that pair
  int32_t pair_units;  // units of that pair
  int32_t q_last;      // position of the sequence's newest query token (length - 1)
};
static_assert(sizeof(DecodeUnit) == 32, "decode units are staged in 32-byte slots");
struct DecodeParams {
  const DecodeUnit* units;   // grouped by CTA
  const int32_t* cta_begin;  // [grid + 1]: CTA c runs units cta_begin[c] .. cta_begin[c+1]-1
  int plan_inline;           // 1: units and cta_begin are offsets into the PlanBlob
  const void* q;             // bf16 [n * T, Hq, D]
  void* o;                   // bf16 [n * T, Hq, D]
  const int32_t* table;
  const void* kpool;
  const void* vpool;
  float* part_acc;           // [n_units, G, D]
  float* part_ml;            // [n_units, G, 2]
  int* pair_cnt;             // [>= n_pairs]: zero before the launch, left zero after it
  float* lse;                // fp32 [Hq, n_rows] or null
  int n_rows;                // n * T query tokens
  int n_units, n_pairs;
  int R, hq, hkv, page_size;
  int G;                     // query rows per KV head, T * Gm: 1, 2, 4, 8 or 16
  int T, Gm;                 // query tokens per sequence; query heads per KV head
  int window;                // keys a local head's query sees
  float scale_log2;
  int* status;
  unsigned long long timeout_ns;
};

// ---- rotary re-alignment ------------------------------------------------------
// One KV head of the rotated sequence: its kept keys [s0, n), in the pages of
// block-table row table_row.
struct RopeHead {
  int32_t table_row, s0, n, pad;
};
constexpr int kRopeMaxHeads = 64;
struct RopeParams {
  RopeHead heads[kRopeMaxHeads];
  float2 cos_sin[128];    // cos and sin of delta * theta_i, i < rotary_dim / 2
  const int32_t* table;   // device block table
  void* kpool;
  int n_heads, R, page_size, head_dim, rotary_dim, style;
};
// chunks_per_head: pages spanned by the longest head's kept range
cudaError_t launch_rope(const RopeParams& p, int chunks_per_head, int grid, cudaStream_t s);

// ---- segment transfer -------------------------------------------------------
// One KV head of a transferred (layer, sequence): its kept rows [s0, s0 + len)
// in pages page_list[page_off ..] (logical pages first_k ..), and where they
// sit in the buffer (K rows from out_row, V rows from out_row + len).
struct XferHead {
  int32_t s0, len, out_row, first_k;
  int32_t page_off, table_row, row_begin;  // row_begin: sum of the earlier heads' len
  int32_t pad;
};
static_assert(sizeof(XferHead) == 32, "transfer heads are staged in 32-byte slots");
struct TransferParams {
  const XferHead* heads;
  const int32_t* page_list;
  uint4* kpool;
  uint4* vpool;
  const uint4* buf;          // import source
  uint4* buf_out;            // export destination
  int32_t* table;            // import: the heads' block-table rows get their new pages
  int plan_inline;           // 1: the plan arrays are offsets into the AppendBlob
  int to_pool;               // 1: import (buffer -> pages), 0: export
  int n_heads, n_pages, vec_per_row, page_size, R;
  int64_t total_rows;        // sum of the heads' len
};
cudaError_t launch_transfer(const TransferParams& p, const AppendBlob* blob, int grid,
                            cudaStream_t s);

// ---- attention mass per key ---------------------------------------------------
struct MassUnit {
  int32_t tok0;        // first token row of the chunk (its cu_seqlens entry)
  int32_t ntok;        // chunk length T
  int32_t a;           // position of the chunk's first token
  int32_t head;        // KV head
  int32_t local;       // 1 = local head
  int32_t kt;          // key tile: positions [kt * 128, kt * 128 + 128)
  int32_t qt0, qt1;    // query tiles (chunk-relative, tpt tokens each), inclusive
  int32_t first_page;  // first held logical page of the segment
  int32_t last_page;   // last held logical page
  int32_t table_row;
  int32_t piece;       // a long key tile's query range is cut into n_pieces pieces
  int32_t n_pieces;
  int32_t part0;       // partial-sum slot of piece 0 (slots part0 .. part0 + n_pieces - 1)
  int32_t tile_id;     // counter of the key tile's finished pieces
};
struct MassParams {
  const MassUnit* units;       // grouped by CTA
  const int32_t* cta_begin;    // [grid + 1]: CTA c runs units cta_begin[c] .. cta_begin[c+1]-1
  float* part;         // [slots][128] partial sums of split key tiles
  int* tile_cnt;       // [tiles] finished pieces, zero at launch
  const int32_t* table;
  const float* lse;    // fp32 [Hq, total_q], natural log, from the prefill of the chunk
  float* mass;         // fp32 [Hkv, total_q]
  int64_t total_q;
  int n_units;
  int R, hq, G, tpt, window, page_size;
  int oob_row;         // a K row coordinate past the end of the pool
  float scale_log2;
  int* status;
  unsigned long long timeout_ns;
};
cudaError_t launch_mass(const MassParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                        int head_dim, int grid, cudaStream_t s);

// ---- top-k token choice ------------------------------------------------------
struct TopkSeq {
  int32_t tok0;  // first token row of the sequence
  int32_t ntok;  // its tokens
  int32_t k;     // how many to choose
  int32_t out0;  // first output slot
};
struct TopkParams {
  const TopkSeq* seqs;
  int32_t* idx;      // chosen token rows
  int plan_inline;   // 1: seqs is an offset into the AppendBlob
};
cudaError_t launch_topk(const float* mass, float* score, int64_t total, int hkv,
                        const TopkParams& p, const AppendBlob* blob, int n_seqs, cudaStream_t s);

// ---- sparse FFN ------------------------------------------------------------
constexpr int kStatusBadIndex = 6;  // device status word: a row index was out of range
struct FfnGemmParams {
  int M;          // rows (chosen tokens)
  int K;          // reduction length (d_model for GEMM 1, d_ff for GEMM 2)
  int tiles_m, tiles_n;
  int n_out;      // row length of out: d_ff (GEMM 1, H) or d_model (GEMM 2, residual)
  int64_t n_rows; // GEMM 2: rows of the residual stream
  void* out;      // GEMM 1: H bf16 [M, d_ff]; GEMM 2: residual bf16 [n_rows, d_model]
  const int32_t* idx;  // GEMM 2: output row of each accumulator row, or null (row m)
  int* status;
  unsigned long long timeout_ns;
};
cudaError_t launch_gather_rows(const void* x, const int32_t* idx, void* out, int m, int d_model,
                               int64_t n_rows, int* status, cudaStream_t s);
// epilogue 0: H = silu(gate) * up; 1: residual[idx] += acc
cudaError_t launch_ffn_gemm(int epilogue, const CUtensorMap& ta, const CUtensorMap& tb0,
                            const CUtensorMap& tb1, const FfnGemmParams& p, int grid,
                            cudaStream_t s);
int ffn_tile_rows();

cudaError_t launch_append(const AppendParams& p, const AppendBlob* blob, int grid, cudaStream_t s);
// copy a plan (16-byte aligned, size rounded up to 16) from mapped host memory to the device
cudaError_t launch_plan_copy(const void* src, void* dst, size_t bytes, cudaStream_t s);
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to, int head_dim, int grid,
                           cudaStream_t s);
int prefill_smem_bytes(int head_dim);
cudaError_t launch_exp2_check(const float* x, float* y_poly, float* y_mufu, int n, cudaStream_t s);
int prefill_unit_tokens(int G);  // query tokens per prefill work unit
cudaError_t launch_decode(const DecodeParams& p, const PlanBlob* blob, int head_dim, int grid,
                          cudaStream_t s);

// Tensor-core decode for 8 or 16 query rows per KV head (D = 128).
struct DecodeCombine {  // one (sequence, KV head) pair split over several units
  int32_t unit0, units;
  int32_t req, head;
};
struct DecodeMmaParams {
  const DecodeUnit* units;     // grouped by CTA (offsets into the PlanBlob when plan_inline)
  const int32_t* cta_begin;    // [grid + 1]
  const DecodeCombine* combine;
  int plan_inline;
  int n_combine;
  void* o;                     // bf16 [n * T, Hq, D]
  float* lse;                  // fp32 [Hq, n_rows] or null
  const int32_t* table;
  float* part_acc;             // [units, R, D]
  float* part_ml;              // [units, R, 2]
  int n_rows;
  int R, hq, hkv, page_size;
  int R_rows;                  // query rows per KV head: T * Gm (8 or 16)
  int T, Gm, window;
  int oob_row;                 // a K/V row coordinate past the end of the pools
  float scale_log2;
  int* status;
  unsigned long long timeout_ns;
};
cudaError_t launch_decode_mma(const DecodeMmaParams& p, const PlanBlob* blob, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                              cudaStream_t s);
int decode_stage_keys(int G);  // keys per decode pipeline stage
int decode_ctas_per_sm(int head_dim, int G);  // resident decode CTAs per SM

}  // namespace skv
