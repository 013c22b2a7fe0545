// launch.h -- internal host interface between the C-ABI layer (vsd_api.cu) and the
// translation units that hold the kernels.  Arguments arrive here already checked.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace vsd {

// ---------------------------------------------------------------- verify
struct VerifyPlan {
  int pairs;     // B * Hkv
  int t_max;     // tiles of 128 keys per pair for the longest admissible sequence
  int ctas;      // persistent grid size
  int max_chunks;  // partial-result slots per pair
  int nq;        // verify rows of one KV group (R * G) rounded up to 16
};

VerifyPlan plan_verify(int B, int Hkv, int R, int G, int P_max, int num_sms);
size_t verify_workspace_bytes(const VerifyPlan& plan, int head_dim);

struct VerifyArgs {
  CUtensorMap kmap, vmap;  // 4-D maps over the caches: {d, page, Hkv, num_blocks}
  const void* q;
  const int32_t* block_table;
  const int32_t* prefix_len;
  float* logits;
  float* partial;
  void* out;
  float* ws;  // partial results: m, l, o per (pair, chunk) slot
  unsigned* status;
  int B, Hq, Hkv, G, R, d, max_blocks, num_blocks, P_max;
  int row0, row1;
  int collect_all;  // 1: every verify row's logits, partial summed over all rows
  const uint8_t* head_mask = nullptr;  // [Hq] or NULL: collected heads
  // fused aggregation (both or neither): score[b][j] = sum over groups of partial[b][g][j]
  // in group order, j < P_b; hist[b][bin] counts the top 12 bits of the order-preserving
  // keys of those scores (zeroed by the call)
  float* score = nullptr;
  uint32_t* hist = nullptr;
  // the histogram counts positions [min(hist_sink, P), max(P - hist_recent, that)) only
  int hist_sink = 0, hist_recent = 0;
  int early = 0;  // producers issue their first prefix tiles before the dependency wait
  // the verify block's keys / values ([B][R][Hkv][D]) stored into the caches (k_store,
  // v_store: the same memory as the maps) at P_b .. P_b + R - 1 before those tiles are
  // copied; null: nothing stored
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  void* k_store = nullptr;
  void* v_store = nullptr;
  float scale;
};

cudaError_t launch_verify(const VerifyArgs& a, const VerifyPlan& plan, cudaStream_t stream);

// ---------------------------------------------------------------- select
struct SelectArgs {
  const float* partial;
  const int32_t* prefix_len;
  int32_t* idx;
  int32_t* n_sel;
  float* scores_out;
  unsigned* status;
  int n_rows, Hkv, P_max, k, n_sink, n_recent;
  // hybrid budget passes (all optional; see select_topk.cu)
  int m_limit = -1;
  const uint32_t* pre_bitmap = nullptr;
  const int32_t* pre_count = nullptr;
  uint32_t* out_bitmap = nullptr;
  int32_t* out_count = nullptr;
  // scored input (Hkv = 1, partial = the aggregated score): [n_rows][4096] counts of
  // the top 12 key bits over every prefix position, as the fused verification writes
  const uint32_t* hist = nullptr;
};

// Scored input (select_scored.cu; Hkv = 1, hist given): CTAs per row for P_max, or -1
// above 16 x 32768 positions.
int select_scored_cluster(int P_max);
cudaError_t launch_select_scored(const SelectArgs& a, cudaStream_t stream);

int select_cluster_size(int P_max, int n_rows);
int select_chunk(int P_max, int cs);  // prefix positions per CTA, or -1 if unsupported
cudaError_t launch_select(const SelectArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- sparse decode
struct SparseArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* k_new = nullptr;  // [B][Hkv][d] the step's input token, or null
  const void* v_new = nullptr;
  void* k_store = nullptr;      // the caches, written at position seq_len - 1
  void* v_store = nullptr;
  int32_t* sel_rows = nullptr;  // [B][k_max] cache row bases of the selection
  int rows_mode = 0;            // 0 unused, 1 resolve and write, 2 read
  int early = 0;                // gather before waiting for the preceding kernel
  const int32_t* block_table;
  const int32_t* idx;
  const int32_t* n_sel;
  const int32_t* tail_start;
  const int32_t* seq_len;
  void* out;
  float* ws;  // per-split partial results (m, l, o); NULL when one split suffices
  unsigned* counters;  // per (sequence, KV head): zero between calls (self-resetting)
  unsigned* status;
  int B, Hq, Hkv, G, d, max_blocks, num_blocks, k_max, max_tail;
  float scale;
};

struct SparsePlan {
  int split_len;   // attended positions per CTA
  int max_splits;  // CTAs (and workspace slots) per (sequence, KV head) pair
};

SparsePlan plan_sparse(int k_max, int max_tail);
// Workspace layout: per-pair counters (sparse_counter_bytes), then the partials.
size_t sparse_counter_bytes(const SparsePlan& plan, int B, int Hkv);
size_t sparse_workspace_bytes(const SparsePlan& plan, int B, int Hkv, int G, int head_dim);
cudaError_t launch_sparse(const SparseArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- sparse verification
// The compressed cache: sequence b's compact position p holds token idx[b][p]
// (p < n_sel[b]) or P_b + p - n_sel[b] (the R verify rows), as a paged cache of
// sparse_verify_pages(k_max, R) pages per sequence with its own block table and
// prefix lengths (n_sel).
struct SparseVerifyArgs {
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* idx;
  const int32_t* n_sel;
  uint16_t* compact_k;        // [B * pages][Hkv][16][d]
  uint16_t* compact_v;
  int32_t* compact_table;     // [B][pages]
  int32_t* compact_prefix;    // [B]
  unsigned* status;
  int B, Hkv, d, R, max_blocks, num_blocks, k_max;
};

int sparse_verify_pages(int k_max, int R);
cudaError_t launch_sparse_verify_gather(const SparseVerifyArgs& a, cudaStream_t stream);

// Fused sparse verification (sparse_decode.cu): the draft step's tensor-core kernel with
// the R * G verify rows of a group as its queries, when R * G <= 32 (power-of-two G) and
// the list (k_max + R) fits 1024 batches; 0 / no bytes otherwise.  SparseArgs as for the
// draft step with tail_start = the prefix lengths, seq_len and counters unused,
// max_tail = R; ws holds the split partials (a second kernel merges them).
int sparse_verify_fused_nq(int R, int G, int k_max);
size_t sparse_verify_fused_bytes(int B, int Hkv, int R, int G, int k_max, int head_dim);
cudaError_t launch_sparse_verify_fused(const SparseArgs& a, int R, cudaStream_t stream);

// ---------------------------------------------------------------- cache bookkeeping
// K/V rows [B][n_new][Hkv][d] stored at positions pos_base[b] + pos_offset + t.
struct AppendArgs {
  const void* k_new;
  const void* v_new;
  const int32_t* block_table;
  const int32_t* pos_base;
  void* k_cache;
  void* v_cache;
  unsigned* status;
  int B, n_new, Hkv, d, max_blocks, num_blocks, pos_offset;
};

cudaError_t launch_append_kv(const AppendArgs& a, cudaStream_t stream);

// prefix_len[b] += accepted[b] + 1; tail_start[b] = old prefix; seq_len[i][b] = old
// prefix + accepted[b] + 2 + i; prefix_copies[r][b] = new prefix.
struct AdvanceArgs {
  const int32_t* accepted;
  int32_t* prefix_len;
  int32_t* tail_start;
  int32_t* seq_len;
  int32_t* prefix_copies;
  unsigned* status;
  int B, gamma, max_prefix, n_copies;
};

cudaError_t launch_advance(const AdvanceArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- copies
// dst <- src, `bytes` a multiple of 16, both 16-byte aligned; either may be pinned host
// memory (addressable from the device).
cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, cudaStream_t stream);

// ---------------------------------------------------------------- per-query block top-k
// Page mean keys kbar [B][Hkv][nblk_max][d] fp32, page scores [B][R][Hq][nblk_max] fp32,
// kept pages [B][R][Hq][kb] int32 (ascending, padded with -1).
struct BlockTopkArgs {
  const void* k_cache;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* page_begin;  // [B] first page to (re)compute, or null for 0
  const void* q;              // bf16 [B][R][Hq][d]
  float* kbar;
  float* scores;
  int32_t* blocks;
  unsigned* status;
  int B, R, Hq, Hkv, G, d, max_blocks, num_blocks, nblk_max, kb;
  float scale;
};

// Threads' item count of the selection kernel for nblk_max pages, -1 above 16384.
int block_select_items(int nblk_max);
cudaError_t launch_page_means(const BlockTopkArgs& a, cudaStream_t stream);
// kbar_map: 2-D fp32 tensor map over the page means {d, B * Hkv * nblk_max}, box
// {32, 128}, 128-byte swizzle.
cudaError_t launch_block_topk(const CUtensorMap& kbar_map, const BlockTopkArgs& a,
                              cudaStream_t stream);

}  // namespace vsd
