/*
 * vsd.h -- C ABI of libvsd: the data-parallel hot path of verification-guided
 * sparse self-speculative decoding on one GB300 GPU (sm_103a).
 *
 * One decoding iteration of the method has three steps, each one call here:
 *
 *   1. vsd_verify_attn_collect -- the target model's verification pass: the gamma+1
 *      verify rows attend the whole paged KV cache with full (causal) attention
 *      and, in the same pass, the pre-softmax logits of two rows (the first draft
 *      token and the bonus token) are written to memory ("Collect-2-Query").
 *      Source: "Vegas - verification-guided sparse attention for self-speculative
 *      decoding" (technical summary), sec. 2 (verification phase, KV selection),
 *      sec. 2.B (Collect-2-Query), sec. 3 (kernel instrumentation).
 *   2. vsd_select_topk -- the collected logits summed over both rows and all query
 *      heads give one score per prefix position; the selected set keeps the
 *      attention-sink prefix and the recent window and fills the rest of the budget
 *      k with the highest scores.  Source: Vegas summary sec. 2.A (the selection
 *      equation: argmax over |T| = k of the summed logits); "Dustin" (technical
 *      summary), Methodology sec. 1 (sink and recent-window protection).
 *   3. vsd_sparse_decode_attn -- a draft step: one query row per head attends only
 *      the selected positions plus the tokens appended after the selection.
 *      Source: Vegas summary sec. 2 (drafting phase) and sec. 3 (sparse execution:
 *      paged attention with page size 1 whose page indices are the selected
 *      token indices).
 *
 * Conventions shared by every call
 *   - All pointers named as device data are CUDA device pointers; the caller owns
 *     every buffer, including the workspace.  The library allocates no memory and
 *     keeps no state between calls except the device status word (below).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  A non-OK return means nothing was launched.
 *   - bf16 tensors hold IEEE bfloat16 values; fp32 tensors IEEE binary32.
 *   - Device pointers must be 16-byte aligned; workspace 256-byte aligned.
 *   - Geometry: G = Hq / Hkv query heads share one KV head; query head h reads KV
 *     head h / G.  head_dim is 64 or 128; page_size is 16.
 *   - KV cache layout: k_cache and v_cache are bf16 [num_blocks][Hkv][page_size]
 *     [head_dim]; logical token j of sequence b is stored in physical block
 *     block_table[b * max_blocks_per_seq + j / page_size] at row j % page_size.
 *   - Host-side argument errors return VSD_ERR_INVALID_ARG / VSD_ERR_UNSUPPORTED /
 *     VSD_ERR_WORKSPACE synchronously.  Data errors found on the device (a block-table
 *     entry outside [0, num_blocks), an index outside its sequence, a length beyond
 *     the declared maximum) never trap: the offending entry is skipped (treated as
 *     masked) and a bit is set in the device status word, read with
 *     vsd_read_device_status.  Every wait inside a kernel is bounded; a wait that
 *     gives up sets VSD_DEV_TIMEOUT and the kernel returns.
 *   - The library looks up the device addresses of its own device variables (the
 *     status word, the no-alloc scratch) once per device and keeps them: do not use it
 *     across a cudaDeviceReset or anything else that destroys and recreates the
 *     device's primary context (the kept addresses would be stale).
 */
#ifndef VSD_H_
#define VSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vsd_status {
  VSD_OK = 0,
  VSD_ERR_INVALID_ARG = -1, /* null pointer, bad size, inconsistent geometry */
  VSD_ERR_UNSUPPORTED = -2, /* valid but not implemented: head_dim, page_size, rows */
  VSD_ERR_CUDA = -3,        /* a CUDA runtime call failed (no GPU, launch failure) */
  VSD_ERR_WORKSPACE = -4,   /* workspace missing, too small or misaligned */
  VSD_ERR_TIMEOUT = -5      /* reserved: a bounded device wait gave up */
} vsd_status;

/* Bits of the device status word. */
#define VSD_DEV_BAD_BLOCK 0x1u  /* block-table entry outside [0, num_blocks) */
#define VSD_DEV_BAD_INDEX 0x2u  /* selected index outside [0, tail_start) or a bad count */
#define VSD_DEV_BAD_LENGTH 0x4u /* a sequence length outside the declared bounds */
#define VSD_DEV_TIMEOUT 0x8u    /* a bounded wait inside a kernel gave up */

/* Shape of a batch over a paged KV cache. */
typedef struct vsd_geom {
  int B;                  /* sequences */
  int Hq;                 /* query heads */
  int Hkv;                /* KV heads; Hq % Hkv == 0 */
  int head_dim;           /* 64 or 128 */
  int page_size;          /* tokens per cache page; 16 */
  int max_blocks_per_seq; /* row length of block_table */
  int num_blocks;         /* physical blocks in k_cache / v_cache */
} vsd_geom;

/* ------------------------------------------------------------------------------
 * Verification attention with Collect-2-Query (Vegas summary sec. 2 verification
 * phase; sec. 2.B; sec. 3 kernel instrumentation).
 *
 * For sequence b with prefix length P_b (tokens before the verify block), verify
 * row t in [0, R) sits at position P_b + t and attends keys 0 .. P_b + t; the cache
 * must already hold the keys and values of the verify block (length P_b + R).
 *   z[b,t,h,j] = scale * <q[b,t,h,:], K[b, j, h/G, :]>
 *   out[b,t,h,:] = sum_j softmax_j(z[b,t,h,:]) * V[b, j, h/G, :]
 *   logits[b,c,h,j] = z[b, row_c, h, j]        c in {0,1}, j < P_b
 *   partial_scores[b,g,j] = sum_{c in {0,1}} sum_{h in group g} logits[b,c,h,j]
 *
 *   q              bf16 [B][R][Hq][head_dim]
 *   block_table    int32 [B][max_blocks_per_seq]
 *   prefix_len     int32 [B]; 0 <= P_b <= P_max and P_b + R <= max_blocks*page_size
 *   collect_row0/1 verify rows whose logits are collected (0 and R-1 = gamma for
 *                  the first draft token and the bonus token); in [0, R).  They may
 *                  be equal: with R = 1 (no drafts) both are row 0 and the scores are
 *                  twice that row's logits, which ranks positions exactly as the one
 *                  row does
 *   P_max          row stride of logits / partial_scores (upper bound of P_b); a
 *                  multiple of 32 keeps every row on a 128-byte boundary, which the
 *                  stores need to cover whole 32-byte sectors (rows that start inside
 *                  a sector cost DRAM read-modify-writes: about 15 % of the call on a
 *                  64K-position batch of 4)
 *   scale          softmax scale (1/sqrt(head_dim) normally)
 *   logits         fp32 [B][2][Hq][P_max] or NULL; only j < P_b are written
 *   partial_scores fp32 [B][Hkv][P_max] or NULL; only j < P_b are written
 *   out            bf16 [B][R][Hq][head_dim]
 *   workspace      >= vsd_verify_workspace_size(...) bytes (0 bytes: may be NULL);
 *                  contents on entry are ignored and on exit unspecified
 * Supported: head_dim in {64, 128}, page_size 16, G <= 16, 1 <= R <= 16, R * G <= 64.
 * ------------------------------------------------------------------------------ */
vsd_status vsd_verify_workspace_size(const vsd_geom* geom, int R, int P_max, size_t* bytes);

vsd_status vsd_verify_attn_collect(const vsd_geom* geom, int R, const void* q,
                                   const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, const int32_t* prefix_len,
                                   int collect_row0, int collect_row1, int P_max, float scale,
                                   float* logits, float* partial_scores, void* out,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------
 * Verification with the collected importance restricted to a set of query heads
 * (Dustin summary, Methodology sec. 2: online, the importance computation is limited
 * to the semantic retrieval heads identified offline).
 *
 * Same as vsd_verify_attn_collect, except that only heads h with head_mask[h] != 0
 * are collected:
 *   partial_scores[b,g,j] = sum_{c in {0,1}} sum_{h in group g, head_mask[h]} logits[b,c,h,j]
 * and the logits of the other heads are not written.
 *   head_mask  uint8 [Hq], device memory (not NULL)
 * ------------------------------------------------------------------------------ */
vsd_status vsd_verify_attn_collect_srh(const vsd_geom* geom, int R, const void* q,
                                       const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, const int32_t* prefix_len,
                                       int collect_row0, int collect_row1,
                                       const uint8_t* head_mask, int P_max, float scale,
                                       float* logits, float* partial_scores, void* out,
                                       void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------
 * Verification attention collecting every verify row (Vegas summary sec. 2.A: the
 * selection equation sums the logits over all gamma+1 rows of the verification
 * block and over the query heads; Collect-2-Query, sec. 2.B, keeps two of them).
 * This is the reference against which Collect-2-Query's savings are measured.
 *
 * Same attention, arguments and workspace as vsd_verify_attn_collect, except:
 *   logits[b,t,h,j] = z[b,t,h,j]                          t in [0, R), j < P_b
 *   partial_scores[b,g,j] = sum_{t < R} sum_{h in group g} logits[b,t,h,j]
 *
 *   logits         fp32 [B][R][Hq][P_max] or NULL; only j < P_b are written
 *   partial_scores fp32 [B][Hkv][P_max] or NULL; only j < P_b are written
 * Supported: as vsd_verify_attn_collect with R * G <= 48 (VSD_ERR_UNSUPPORTED
 * otherwise).
 * ------------------------------------------------------------------------------ */
vsd_status vsd_verify_attn_collect_all(const vsd_geom* geom, int R, const void* q,
                                       const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, const int32_t* prefix_len,
                                       int P_max, float scale, float* logits,
                                       float* partial_scores, void* out, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------
 * Verification attention without a caller-provided workspace.  The pages have no
 * counterpart: this is a convenience of this library.
 *
 * Same operation, arguments and results as vsd_verify_attn_collect, minus the
 * workspace.  It is meant for callers that cannot allocate device memory on the
 * decode path: an engine that has reserved all free HBM for its paged KV cache up
 * front, or a host program that forbids cudaMalloc there because cudaMalloc can
 * synchronize the whole device.  The scratch it needs lives instead in a fixed
 * device array of VSD_NOALLOC_SCRATCH_BYTES that every GPU using this library holds
 * until the process exits; this call allocates nothing.
 *   - Returns VSD_ERR_WORKSPACE when vsd_verify_workspace_size reports more than
 *     VSD_NOALLOC_SCRATCH_BYTES for this geometry (use the regular call then).
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call before any stream
 *     capture.
 *   - Every call on a device shares the one array: calls whose kernels overlap on
 *     the GPU (different streams without ordering) race and give wrong results.
 *     Nothing in the array needs to start at zero.
 * ------------------------------------------------------------------------------ */
#define VSD_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB */

vsd_status vsd_verify_attn_collect_noalloc(const vsd_geom* geom, int R, const void* q,
                                           const void* k_cache, const void* v_cache,
                                           const int32_t* block_table,
                                           const int32_t* prefix_len, int collect_row0,
                                           int collect_row1, int P_max, float scale,
                                           float* logits, float* partial_scores, void* out,
                                           void* stream);

/* ------------------------------------------------------------------------------
 * Aggregated-logit top-k with a protected sink and recent window (Vegas summary
 * sec. 2.A selection equation; Dustin summary Methodology sec. 1).
 *
 * For row r (one (layer, sequence) pair) with prefix length P = prefix_len[r]:
 *   s[j] = sum_g partial_scores[r,g,j]                  for j < P
 *   S    = [0, min(n_sink, P)) U [max(0, P - n_recent), P)
 *   n    = min(k, P); the n - |S| highest s outside S are added (equal scores:
 *          the lower position first)
 *   idx[r, 0..n) = S U added, ascending; idx[r, n..k) = -1; n_sel[r] = n
 *
 *   partial_scores fp32 [n_rows][Hkv][P_max]
 *   prefix_len     int32 [n_rows], 0 <= P <= P_max
 *   idx            int32 [n_rows][k]
 *   n_sel          int32 [n_rows]
 *   scores_out     fp32 [n_rows][P_max] or NULL: the aggregated s (j < P written)
 *   workspace      >= vsd_select_workspace_size(...) bytes (may be 0)
 * Requires n_sink + n_recent <= k.  One launch covers all rows.
 * Supported: P_max <= 262144 for up to 7 rows, P_max <= 131072 for more rows
 * (VSD_ERR_UNSUPPORTED otherwise).  The kernel is launched as a programmatic
 * dependent of the preceding kernel on the stream: it waits for that kernel's
 * results before reading anything.
 * ------------------------------------------------------------------------------ */
vsd_status vsd_select_workspace_size(int n_rows, int Hkv, int P_max, int k, size_t* bytes);

vsd_status vsd_select_topk(int n_rows, int Hkv, const float* partial_scores,
                           const int32_t* prefix_len, int P_max, int k, int n_sink,
                           int n_recent, int32_t* idx, int32_t* n_sel, float* scores_out,
                           void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------
 * Fused aggregation (Vegas summary sec. 2.A: the selection objective sums the
 * collected logits over every query head; here the verification call finishes that
 * sum and the first histogram level of the selection, so the selection starts from
 * one score per position).
 *
 * vsd_verify_attn_collect_scored: vsd_verify_attn_collect (same arguments; logits may
 * be NULL, partial_scores may not) that also writes, for every sequence b,
 *   score[b][j] = sum_g partial_scores[b][g][j]   (fp32, groups in order from zero;
 *                                                  j < P_b; later entries not written)
 *   score_hist[b][i] = #{ j in C_b : key(score[b][j]) >> 20 == i },  i < 4096
 * over the selection's candidates C_b = [s, max(P_b - n_recent, s)), s = min(n_sink,
 * P_b): the selection's protected sinks and recent window are left out (n_sink =
 * n_recent = 0 counts every prefix position).
 * flags: 0 or VSD_VERIFY_EARLY_PREFETCH (any other bit: VSD_ERR_INVALID_ARG): the
 * kernel's K and V producers issue their first stages of cache tiles that lie wholly
 * below P_b before the call waits for the preceding kernel on the stream (which hides
 * the pipeline's start behind that kernel).  The caller promises that the preceding
 * kernel writes none of block_table and prefix_len nor any cache row below P_b -- a
 * decode loop's append of the verify block (rows P_b and beyond) qualifies -- and that
 * it is a kernel of this library or one launched without programmatic dependent launch
 * (every kernel of this library lets its dependents start only after its own wait, so
 * what was written two launches earlier is complete).  q, the outputs, the workspace
 * and score_hist are touched after the wait.
 * k_new, v_new: bf16 [B][R][Hkv][head_dim] (16-byte aligned, both or neither) or NULL:
 * the verify block's keys and values, stored into the caches at positions P_b .. P_b +
 * R - 1 through the block table (what vsd_append_kv with pos_offset 0 stores) by the
 * kernel itself, before it reads those rows; a block-table entry outside the cache is
 * flagged VSD_DEV_BAD_BLOCK and its rows are not stored.  With them the caches are
 * written (hence not const); without them they are only read.
 * where key(x) maps the fp32 bits order-preservingly to uint32 (sign bit set for
 * x >= +0: bits | 0x80000000; else ~bits).  score fp32 [B][P_max] and score_hist
 * uint32 [B][4096] are caller-owned (4-byte aligned; the rows of several calls may
 * share one buffer); score_hist is overwritten (no zeroing needed).  The selection
 * reads a score buffer with 16-byte loads: its base must be 16-byte aligned.
 *
 * vsd_select_topk_scored: vsd_select_topk on n_rows = B rows of such a score
 * (Hkv = 1) and its histogram (of the candidates for the same n_sink and n_recent, or
 * of every prefix position, whose protected positions the kernel then takes out itself
 * at the cost of one more round trip) -- the same index sets, bit for bit, as
 * vsd_select_topk on the partial scores (NaN scores excepted: their order among
 * themselves is unspecified).  Its own kernel: a cluster of up to 16 CTAs per row,
 * each holding a slice of the row in registers; the boundary bin's keys are exchanged
 * once between the CTAs.  A histogram that does not match the scores (its counts are
 * not the scores') raises VSD_DEV_BAD_LENGTH and the row's selection is unspecified;
 * a prefix length outside [0, P_max] raises it too and leaves the row empty
 * (n_sel = 0, all -1).  Supported: P_max <= 524288, n_rows <= 65535
 * (VSD_ERR_UNSUPPORTED otherwise).
 * ------------------------------------------------------------------------------ */
vsd_status vsd_verify_attn_collect_scored(const vsd_geom* geom, int R, const void* q,
                                          void* k_cache, void* v_cache,
                                          const int32_t* block_table, const int32_t* prefix_len,
                                          int collect_row0, int collect_row1, int P_max,
                                          float scale, float* logits, float* partial_scores,
                                          float* score, uint32_t* score_hist, int n_sink,
                                          int n_recent, unsigned flags, const void* k_new,
                                          const void* v_new, void* out, void* workspace,
                                          size_t workspace_bytes, void* stream);

#define VSD_VERIFY_EARLY_PREFETCH 0x4u

vsd_status vsd_select_topk_scored(int n_rows, const float* score, const uint32_t* score_hist,
                                  const int32_t* prefix_len, int P_max, int k, int n_sink,
                                  int n_recent, int32_t* idx, int32_t* n_sel, void* stream);

/* ------------------------------------------------------------------------------
 * Hybrid budget with two signals (Dustin summary, Methodology sec. 1: after the
 * protected sinks and recent window, the top-m tokens by the draft-lookahead signal,
 * then the most relevant remaining tokens by the target-historical signal).
 *
 * For row r with prefix length P (n = min(k, P), S as in vsd_select_topk):
 *   s_t[j] = sum_g partial_target[r,g,j],  s_d[j] = sum_g partial_draft[r,g,j]
 *   D  = the min(m, n - |S|) positions outside S with the highest s_d
 *   T' = the n - |S| - |D| positions outside S and D with the highest s_t
 *   (equal scores: the lower position first)
 *   idx[r, 0..n) = S U D U T', ascending; idx[r, n..k) = -1; n_sel[r] = n
 *
 *   partial_target fp32 [n_rows][Hkv_target][P_max]; partial_draft fp32
 *   [n_rows][Hkv_draft][P_max] (any per-group decomposition of the draft score)
 *   workspace      >= vsd_select_hybrid_workspace_size(...) bytes, 256-byte aligned;
 *                  contents on entry are ignored
 * Two launches of the selection kernel; supported sizes as vsd_select_topk.
 * ------------------------------------------------------------------------------ */
vsd_status vsd_select_hybrid_workspace_size(int n_rows, int P_max, size_t* bytes);

vsd_status vsd_select_topk_hybrid(int n_rows, int Hkv_target, const float* partial_target,
                                  int Hkv_draft, const float* partial_draft,
                                  const int32_t* prefix_len, int P_max, int k, int m,
                                  int n_sink, int n_recent, int32_t* idx, int32_t* n_sel,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------
 * Sparse draft-step attention (Vegas summary sec. 2 drafting phase; sec. 3 sparse
 * execution, page size 1 over the selected indices).
 *
 * For sequence b the attended positions are idx[b, 0..n_sel[b]) followed by the
 * dense tail tail_start[b] .. seq_len[b]-1 (tokens written after the selection):
 *   out[b,h,:] = sum_{j attended} softmax_j(scale * <q[b,h,:], K[b,j,h/G,:]>) V[b,j,h/G,:]
 * A position listed twice is attended twice; selected indices are expected to be
 * below tail_start[b] (the select step guarantees it).  An index outside
 * [0, seq_len[b]) is skipped and flagged VSD_DEV_BAD_INDEX.
 *
 *   q          bf16 [B][Hq][head_dim]
 *   idx        int32 [B][k_max] (may be NULL when k_max == 0)
 *   n_sel      int32 [B] (may be NULL when k_max == 0), 0 <= n_sel[b] <= k_max
 *   tail_start int32 [B]; seq_len int32 [B]; tail_start <= seq_len
 *   max_tail   host-side upper bound of seq_len[b] - tail_start[b]; it sizes
 *              the split of the work (results do not depend on it); a sequence
 *              whose list is longer than k_max + max_tail allows is flagged
 *              VSD_DEV_BAD_LENGTH and gets a zero output
 *   out        bf16 [B][Hq][head_dim]
 *   workspace  >= vsd_sparse_workspace_size(...) bytes (0 bytes: may be NULL),
 *              256-byte aligned.  It starts with per-(sequence, KV head) counters
 *              that must be zero before the first use; every call returns them to
 *              zero, so the buffer can be reused by later calls of this entry point
 *              with the same B and Hkv (with others the counters sit where this call
 *              wrote partials).  Zero it again before a call with other B or Hkv and
 *              after a call that raised VSD_DEV_TIMEOUT, and do not share it with
 *              other entry points or with calls that may run concurrently.
 * Supported: head_dim in {64, 128}, page_size 16, G <= 16.
 * ------------------------------------------------------------------------------ */
vsd_status vsd_sparse_workspace_size(const vsd_geom* geom, int k_max, int max_tail,
                                     size_t* bytes);

vsd_status vsd_sparse_decode_attn(const vsd_geom* geom, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_table,
                                  const int32_t* idx, const int32_t* n_sel, int k_max,
                                  const int32_t* tail_start, const int32_t* seq_len,
                                  int max_tail, float scale, void* out, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------
 * A draft step of a decode loop (Vegas summary, sec. 2 drafting phase and sec. 3
 * integration: the drafts come from repeated forward passes of the target model with
 * sparse attention; each pass processes one new token, whose keys and values join the
 * cache before its attention reads them).
 *
 * The same attention as vsd_sparse_decode_attn, with these options:
 *   k_new, v_new   bf16 [B][Hkv][head_dim] or both NULL: the keys and values of the
 *                  step's input token, stored at position seq_len[b] - 1 of the cache
 *                  (the last position of the dense tail, so tail_start[b] < seq_len[b]
 *                  is required for it) and attended from these buffers; the result is
 *                  the call on the cache after the store.  k_cache / v_cache are
 *                  written at that position only.
 *   sel_rows       int32 [B][k_max] (device) or NULL; with flags:
 *     VSD_STEP_RECORD_ROWS  the call also writes, for every selected position
 *                  i < n_sel[b], the cache row base of idx[b][i] (block * Hkv *
 *                  page_size + offset within the page; -1 for an invalid index or block)
 *     VSD_STEP_REUSE_ROWS   the call reads those row bases instead of resolving idx
 *                  through the block table: the later steps of one selection (the same
 *                  idx, n_sel and block table as the recording call); an entry outside
 *                  the cache is skipped and flagged VSD_DEV_BAD_INDEX
 *   flags          also:
 *     VSD_STEP_EARLY_GATHER  the selection and the tail are resolved and gathered before
 *                  the call waits for the preceding kernel on the stream (which hides the
 *                  gather behind that kernel's last microseconds).  The caller promises
 *                  that the preceding kernel writes none of idx, n_sel, tail_start,
 *                  seq_len, block_table and sel_rows, nor any cache row this call reads
 *                  except at seq_len[b] - 1, and that it is a kernel of this library or a
 *                  kernel launched without programmatic dependent launch.  (Every kernel
 *                  of this library lets its dependents start only after its own wait for
 *                  its predecessor, so anything written two launches earlier is complete.)
 *                  q, k_new / v_new, the workspace and out are always touched after the
 *                  wait.
 * Every other argument, result and rule as vsd_sparse_decode_attn (the workspace may be
 * shared with it).  Supported: as vsd_sparse_decode_attn, with num_blocks * Hkv *
 * page_size < 2^31 (VSD_ERR_UNSUPPORTED otherwise); RECORD and REUSE together, or an
 * unknown flag, are VSD_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------------ */
#define VSD_STEP_RECORD_ROWS 0x1u
#define VSD_STEP_REUSE_ROWS 0x2u
#define VSD_STEP_EARLY_GATHER 0x4u

vsd_status vsd_sparse_decode_attn_step(const vsd_geom* geom, const void* q, const void* k_new,
                                       const void* v_new, void* k_cache, void* v_cache,
                                       const int32_t* block_table, const int32_t* idx,
                                       const int32_t* n_sel, int k_max,
                                       const int32_t* tail_start, const int32_t* seq_len,
                                       int max_tail, int32_t* sel_rows, unsigned flags,
                                       float scale, void* out, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------
 * Sparse verification (Dustin summary, "Verification workflow", steps 3-4: a
 * compressed target KV cache is formed from the selected tokens only and the draft
 * block is verified against it).
 *
 * For sequence b with prefix length P_b, verify row t in [0, R) attends
 *   J_bt = idx[b, 0 .. n_sel[b])  followed by  P_b .. P_b + t
 *   out[b,t,h,:] = sum_{j in J_bt} softmax_j(scale * <q[b,t,h,:], K[b,j,h/G,:]>) V[b,j,h/G,:]
 * The cache must hold the verify block (positions P_b .. P_b + R - 1).  No logits are
 * collected.  When R * G <= 32 (and the list k_max + R spans at most 1024 batches of
 * 128) one kernel gathers the attended rows straight into shared memory, a split of
 * 128 list positions per CTA with the R * G verify rows of a KV group as the tensor-core
 * product's N side, the verify block masked causally, and a second kernel merges the
 * splits; otherwise the call writes the compressed cache into the workspace and runs
 * the verification kernel on it.
 *
 *   q          bf16 [B][R][Hq][head_dim]
 *   flags      0 or VSD_SPARSE_VERIFY_EARLY_GATHER (any other bit: VSD_ERR_INVALID_ARG):
 *              the fused kernel resolves and gathers the selected positions' rows before
 *              it waits for the preceding kernel on the stream, and the verify block's
 *              rows and q after the wait.  The caller promises that the preceding kernel
 *              writes none of idx, n_sel, prefix_len and block_table, nor the selected
 *              positions' cache rows, and that it is a kernel of this library or a
 *              kernel launched without programmatic dependent launch (every kernel of
 *              this library lets its dependents start only after its own wait, so what
 *              was written two launches earlier is complete).  The gathered path
 *              ignores the flag.
 *   prefix_len int32 [B]; P_b + R <= max_blocks_per_seq * page_size
 *   idx        int32 [B][k_max] selected prefix positions (< P_b), n_sel int32 [B]
 *              (0 <= n_sel[b] <= k_max); a position outside [0, P_b + R) is flagged
 *              VSD_DEV_BAD_INDEX and that sequence's output is unspecified
 *   out        bf16 [B][R][Hq][head_dim]
 *   workspace  >= vsd_sparse_verify_workspace_size(...) bytes, 256-byte aligned
 *              (the compressed cache, about 2 * B * Hkv * (k_max + R) * head_dim * 2
 *              bytes, or the fused kernel's split partials, B * Hkv * splits *
 *              R * G * (head_dim + 2) floats); contents on entry are ignored
 * Supported: as vsd_verify_attn_collect with P_max = k_max.
 * ------------------------------------------------------------------------------ */
vsd_status vsd_sparse_verify_workspace_size(const vsd_geom* geom, int R, int k_max,
                                            size_t* bytes);

#define VSD_SPARSE_VERIFY_EARLY_GATHER 0x4u

vsd_status vsd_sparse_verify_attn(const vsd_geom* geom, int R, const void* q,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, const int32_t* prefix_len,
                                  const int32_t* idx, const int32_t* n_sel, int k_max,
                                  unsigned flags, float scale, void* out, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------
 * Per-query block top-k (the sparse-verification summary, "Sparse Verification
 * Engine", attention sparsity: each query keeps only its top-k key/value blocks in
 * structured block sparsity, chosen by a cheap relevance score).  A contrasting
 * selector to the aggregated one above: the kept set differs per head and verify row.
 * Blocks are the 16-token pages of the prefix; the cheap score of a page is the
 * query's scaled dot product with the page's mean key.
 *
 * vsd_page_key_means: for every sequence b and page beta in
 * [page_begin[b], ceil(P_b / 16)),
 *   page_means[b][g][beta][:] = mean of K[b, j, g, :] over j in [16 beta, 16 beta + 16),
 *                               j < P_b          (fp32)
 *   page_means  fp32 [B][Hkv][page_blocks_max][head_dim], caller-owned; pages outside
 *               the range are not written (a decode loop passes page_begin to refresh
 *               only the pages that changed)
 *   page_begin  int32 [B] or NULL (all pages); a negative entry is flagged
 *               VSD_DEV_BAD_LENGTH
 *   prefix_len  int32 [B]; P_b <= max_blocks_per_seq * 16 and
 *               ceil(P_b / 16) <= page_blocks_max, else VSD_DEV_BAD_LENGTH and the
 *               sequence is skipped
 * A block-table entry outside [0, num_blocks) is flagged VSD_DEV_BAD_BLOCK and that
 * page's mean is written as zeros.
 *
 * vsd_block_topk: for every b, verify row t < R and query head h,
 *   scores[b][t][h][beta] = scale * <q[b,t,h,:], page_means[b][h/G][beta][:]>
 *                           for beta < ceil(P_b / 16) (fp32; later entries not written)
 *   blocks[b][t][h][0 .. min(kb, nblk_b)) = the kb pages with the highest score,
 *                           ties to the lower page, ascending; the rest -1
 *   q           bf16 [B][R][Hq][head_dim]
 *   scores      fp32 [B][R][Hq][page_blocks_max], caller-owned (also the selection's
 *               input, read back on the same stream)
 *   blocks      int32 [B][R][Hq][kb], caller-owned
 * Supported: head_dim 64 or 128, G a power of two, R * G <= 64, page_size 16,
 * 0 <= page_blocks_max <= 16384 (prefixes up to 262144 tokens), kb >= 1,
 * B * R * Hq <= 2^31 - 1.  Pointers 16-byte aligned (int32 arrays 4-byte).
 * ------------------------------------------------------------------------------ */
vsd_status vsd_page_key_means(const vsd_geom* geom, const void* k_cache,
                              const int32_t* block_table, const int32_t* prefix_len,
                              const int32_t* page_begin, int page_blocks_max,
                              float* page_means, void* stream);

vsd_status vsd_block_topk(const vsd_geom* geom, int R, const void* q, const float* page_means,
                          const int32_t* prefix_len, int page_blocks_max, int kb, float scale,
                          float* scores, int32_t* blocks, void* stream);

/* ------------------------------------------------------------------------------
 * Cache bookkeeping of a decode iteration (Vegas summary, sec. 2 core mechanism: each
 * iteration verifies the drafts with a full forward pass, selects from it and drafts
 * from the selection; sec. 3 integration: the drafts come from repeated forward passes
 * of the target model).  Every forward pass stores the keys and values of the tokens
 * it processes in the paged cache before their attention reads them, and the number of
 * drafts a verification accepts moves each sequence's prefix forward.
 *
 * vsd_append_kv: for every sequence b, token t < n_new and KV head g,
 *   K[b, p, g, :] = k_new[b][t][g][:],  V[b, p, g, :] = v_new[b][t][g][:],
 *   p = pos_base[b] + pos_offset + t   (stored through the block table)
 *   k_new, v_new  bf16 [B][n_new][Hkv][head_dim]
 *   pos_base      int32 [B] (device); pos_offset a host integer (e.g. 0 with
 *                 pos_base = prefix_len for the verify block, or -1 with pos_base =
 *                 seq_len for the newest token of a draft step)
 *   k_cache, v_cache written in place; nothing else is read or written
 * A position outside [0, max_blocks_per_seq * page_size) is skipped and flagged
 * VSD_DEV_BAD_LENGTH; a block-table entry outside [0, num_blocks), VSD_DEV_BAD_BLOCK.
 *
 * vsd_advance_lengths: after a verification that accepted a_b = accepted[b] of the
 * gamma drafts of sequence b (0 <= a_b <= gamma), with P = prefix_len[b]:
 *   prefix_len[b]        = P + a_b + 1   (the verify block's first token and the
 *                                          accepted drafts join the prefix)
 *   tail_start[b]        = P
 *   seq_len[i * B + b]   = P + a_b + 2 + i   for draft step i < gamma (the attended
 *                          dense tail of step i: the accepted tokens, the bonus token
 *                          and the inputs of steps 0 .. i)
 *   prefix_copies[r * B + b] = P + a_b + 1   for r < n_copies (e.g. the per-(layer,
 *                          sequence) prefix lengths of a multi-layer selection)
 *   accepted int32 [B]; prefix_len, tail_start int32 [B]; seq_len int32 [gamma][B];
 *   prefix_copies int32 [n_copies][B] or NULL when n_copies == 0 (all device memory)
 * A count outside [0, gamma], a negative prefix or a new prefix above max_prefix
 * (a host integer: the longest prefix the caches can take) is flagged
 * VSD_DEV_BAD_LENGTH and that sequence keeps its prefix (tail_start = P, seq_len
 * P + 1 + i, prefix_len and its copies P).
 *
 * Both are programmatic dependents of the preceding kernel on the stream: they wait
 * for its results before reading or writing anything.
 * ------------------------------------------------------------------------------ */
vsd_status vsd_append_kv(const vsd_geom* geom, int n_new, const void* k_new, const void* v_new,
                         const int32_t* block_table, const int32_t* pos_base, int pos_offset,
                         void* k_cache, void* v_cache, void* stream);

vsd_status vsd_advance_lengths(int B, int gamma, const int32_t* accepted, int max_prefix,
                               int32_t* prefix_len, int32_t* tail_start, int32_t* seq_len,
                               int n_copies, int32_t* prefix_copies, void* stream);

/* ------------------------------------------------------------------------------
 * vsd_copy: dst <- src as a kernel on `stream` (a programmatic dependent of the
 * preceding kernel).  Either pointer may be pinned host memory, which the device
 * addresses directly; a decode loop moves its inputs in and its results out this way.
 * bytes a multiple of 16, both pointers 16-byte aligned (VSD_ERR_INVALID_ARG
 * otherwise); the ranges must not overlap.
 * ------------------------------------------------------------------------------ */
vsd_status vsd_copy(void* dst, const void* src, size_t bytes, void* stream);

/* ------------------------------------------------------------------------------
 * Device status word and errors.
 * vsd_read_device_status synchronizes `stream`, returns the accumulated
 * VSD_DEV_* bits of every kernel of this library on the current device since the
 * last read, and clears them.
 * ------------------------------------------------------------------------------ */
vsd_status vsd_read_device_status(void* stream, unsigned* flags);

const char* vsd_get_error_string(vsd_status status);

/* The CUDA error behind the most recent VSD_ERR_CUDA of the calling thread
 * (a cudaError_t value; 0 if none). */
int vsd_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* VSD_H_ */
