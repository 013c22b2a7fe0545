// vsd_api.cu -- the C ABI of libvsd (declared in include/vsd.h): argument checks,
// launch planning, TMA descriptor encoding and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/vsd.h"
#include "launch.h"

namespace {

// Accumulated VSD_DEV_* bits of every kernel of this library on a device.
__device__ unsigned g_vsd_device_status = 0u;

thread_local int t_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned* g_status_ptr[kMaxDevices] = {nullptr};
int g_num_sms[kMaxDevices] = {0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

vsd_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return VSD_ERR_CUDA;
}

// Per-device constants: the status word's device address and the SM count.
vsd_status device_info(unsigned** status, int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return VSD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_vsd_device_status);
    if (e != cudaSuccess) return cuda_fail(e);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    g_status_ptr[dev] = static_cast<unsigned*>(p);
    g_num_sms[dev] = sms;
  }
  if (status) *status = g_status_ptr[dev];
  if (num_sms) *num_sms = g_num_sms[dev];
  return VSD_OK;
}

vsd_status encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &qr);
    if (e != cudaSuccess) return cuda_fail(e);
    if (qr != cudaDriverEntryPointSuccess || fn == nullptr) return VSD_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = g_encode;
  return VSD_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Shared checks of a paged-cache geometry.
vsd_status check_geom(const vsd_geom* g) {
  if (g == nullptr) return VSD_ERR_INVALID_ARG;
  if (g->B < 0 || g->Hq <= 0 || g->Hkv <= 0 || g->Hq % g->Hkv != 0) return VSD_ERR_INVALID_ARG;
  if (g->max_blocks_per_seq <= 0 || g->num_blocks <= 0) return VSD_ERR_INVALID_ARG;
  if (g->head_dim != 64 && g->head_dim != 128) return VSD_ERR_UNSUPPORTED;
  if (g->page_size != 16) return VSD_ERR_UNSUPPORTED;
  if (!is_pow2(g->Hq / g->Hkv)) return VSD_ERR_UNSUPPORTED;
  return VSD_OK;
}

// 4-D tiled map over a cache [num_blocks][Hkv][page][d]: box = 64 dims x one page.
vsd_status make_cache_map(CUtensorMap* map, const void* cache, const vsd_geom* g) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  vsd_status st = encoder(&enc);
  if (st != VSD_OK) return st;
  const cuuint64_t d = static_cast<cuuint64_t>(g->head_dim);
  cuuint64_t dims[4] = {d, 16, static_cast<cuuint64_t>(g->Hkv),
                        static_cast<cuuint64_t>(g->num_blocks)};
  cuuint64_t strides[3] = {d * 2, 16 * d * 2, static_cast<cuuint64_t>(g->Hkv) * 16 * d * 2};
  cuuint32_t box[4] = {64, 16, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = static_cast<int>(r);
    return VSD_ERR_CUDA;
  }
  return VSD_OK;
}

// 2-D fp32 map over page means [rows][d]: box = 32 columns (128 bytes) x 128 rows.
vsd_status make_means_map(CUtensorMap* map, const float* means, int d, long long rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  vsd_status st = encoder(&enc);
  if (st != VSD_OK) return st;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(means), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = static_cast<int>(r);
    return VSD_ERR_CUDA;
  }
  return VSD_OK;
}

vsd_status verify_checks(const vsd_geom* geom, int R, int P_max) {
  vsd_status st = check_geom(geom);
  if (st != VSD_OK) return st;
  if (R < 1 || P_max < 0) return VSD_ERR_INVALID_ARG;
  const int G = geom->Hq / geom->Hkv;
  if (R > 16 || G > 16 || R * G > 64) return VSD_ERR_UNSUPPORTED;
  return VSD_OK;
}

}  // namespace

extern "C" {

const char* vsd_get_error_string(vsd_status s) {
  switch (s) {
    case VSD_OK: return "success";
    case VSD_ERR_INVALID_ARG: return "invalid argument";
    case VSD_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case VSD_ERR_CUDA: return "CUDA runtime error (see vsd_last_cuda_error)";
    case VSD_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case VSD_ERR_TIMEOUT: return "a bounded device wait gave up";
  }
  return "unknown status";
}

int vsd_last_cuda_error(void) { return t_last_cuda_error; }

vsd_status vsd_read_device_status(void* stream, unsigned* flags) {
  if (flags == nullptr) return VSD_ERR_INVALID_ARG;
  unsigned* dptr = nullptr;
  vsd_status st = device_info(&dptr, nullptr);
  if (st != VSD_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned v = 0u;
  e = cudaMemcpy(&v, dptr, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemset(dptr, 0, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e);
  *flags = v;
  return VSD_OK;
}

vsd_status vsd_verify_workspace_size(const vsd_geom* geom, int R, int P_max, size_t* bytes) {
  if (bytes == nullptr) return VSD_ERR_INVALID_ARG;
  vsd_status st = verify_checks(geom, R, P_max);
  if (st != VSD_OK) return st;
  int sms = 0;
  st = device_info(nullptr, &sms);
  if (st != VSD_OK) return st;
  const vsd::VerifyPlan plan =
      vsd::plan_verify(geom->B, geom->Hkv, R, geom->Hq / geom->Hkv, P_max, sms);
  *bytes = vsd::verify_workspace_bytes(plan, geom->head_dim);
  return VSD_OK;
}

namespace {

vsd_status verify_call(const vsd_geom* geom, int R, const void* q, const void* k_cache,
                       const void* v_cache, const int32_t* block_table,
                       const int32_t* prefix_len, bool collect_all, int collect_row0,
                       int collect_row1, const uint8_t* head_mask, int P_max, float scale,
                       float* logits, float* partial_scores, void* out, void* workspace,
                       size_t workspace_bytes, void* stream, float* score = nullptr,
                       uint32_t* hist = nullptr, int hist_sink = 0, int hist_recent = 0,
                       int early = 0, const void* k_new = nullptr, const void* v_new = nullptr) {
  vsd_status st = verify_checks(geom, R, P_max);
  if (st != VSD_OK) return st;
  // all rows: the two halves of every key's columns meet in the part of the Q
  // staging area that 64 query rows would need and 48 leave free
  if (collect_all && R * (geom->Hq / geom->Hkv) > 48) return VSD_ERR_UNSUPPORTED;
  if (geom->B == 0) return VSD_OK;
  if (!q || !k_cache || !v_cache || !block_table || !prefix_len || !out)
    return VSD_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(logits, 16) || !aligned(partial_scores, 16) || !aligned(block_table, 4) ||
      !aligned(prefix_len, 4))
    return VSD_ERR_INVALID_ARG;
  if (!collect_all && (logits || partial_scores) &&
      (collect_row0 < 0 || collect_row0 >= R || collect_row1 < 0 || collect_row1 >= R))
    return VSD_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return VSD_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  int sms = 0;
  st = device_info(&status, &sms);
  if (st != VSD_OK) return st;
  const int G = geom->Hq / geom->Hkv;
  const vsd::VerifyPlan plan = vsd::plan_verify(geom->B, geom->Hkv, R, G, P_max, sms);
  const size_t need = vsd::verify_workspace_bytes(plan, geom->head_dim);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)))
    return VSD_ERR_WORKSPACE;
  vsd::VerifyArgs va;
  st = make_cache_map(&va.kmap, k_cache, geom);
  if (st != VSD_OK) return st;
  st = make_cache_map(&va.vmap, v_cache, geom);
  if (st != VSD_OK) return st;
  va.q = q;
  va.block_table = block_table;
  va.prefix_len = prefix_len;
  va.logits = logits;
  va.partial = partial_scores;
  va.out = out;
  va.ws = static_cast<float*>(workspace);
  va.status = status;
  va.B = geom->B;
  va.Hq = geom->Hq;
  va.Hkv = geom->Hkv;
  va.G = G;
  va.R = R;
  va.d = geom->head_dim;
  va.max_blocks = geom->max_blocks_per_seq;
  va.num_blocks = geom->num_blocks;
  va.P_max = P_max;
  va.row0 = collect_all ? 0 : collect_row0;
  va.row1 = collect_all ? 0 : collect_row1;
  va.collect_all = collect_all ? 1 : 0;
  va.head_mask = head_mask;
  va.score = score;
  va.hist = hist;
  va.hist_sink = hist_sink;
  va.hist_recent = hist_recent;
  va.early = early;
  va.k_new = k_new;
  va.v_new = v_new;
  va.k_store = const_cast<void*>(k_cache);  // written only when k_new is given
  va.v_store = const_cast<void*>(v_cache);
  va.scale = scale;
  cudaError_t e = vsd::launch_verify(va, plan, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return VSD_OK;
}

}  // namespace

vsd_status vsd_verify_attn_collect(const vsd_geom* geom, int R, const void* q,
                                   const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, const int32_t* prefix_len,
                                   int collect_row0, int collect_row1, int P_max, float scale,
                                   float* logits, float* partial_scores, void* out,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  return verify_call(geom, R, q, k_cache, v_cache, block_table, prefix_len, false,
                     collect_row0, collect_row1, nullptr, P_max, scale, logits,
                     partial_scores, out, workspace, workspace_bytes, stream);
}

vsd_status vsd_verify_attn_collect_srh(const vsd_geom* geom, int R, const void* q,
                                       const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, const int32_t* prefix_len,
                                       int collect_row0, int collect_row1,
                                       const uint8_t* head_mask, int P_max, float scale,
                                       float* logits, float* partial_scores, void* out,
                                       void* workspace, size_t workspace_bytes, void* stream) {
  if (head_mask == nullptr) return VSD_ERR_INVALID_ARG;
  return verify_call(geom, R, q, k_cache, v_cache, block_table, prefix_len, false,
                     collect_row0, collect_row1, head_mask, P_max, scale, logits,
                     partial_scores, out, workspace, workspace_bytes, stream);
}

vsd_status vsd_verify_attn_collect_scored(const vsd_geom* geom, int R, const void* q,
                                          void* k_cache, void* v_cache,
                                          const int32_t* block_table, const int32_t* prefix_len,
                                          int collect_row0, int collect_row1, int P_max,
                                          float scale, float* logits, float* partial_scores,
                                          float* score, uint32_t* score_hist, int n_sink,
                                          int n_recent, unsigned flags, const void* k_new,
                                          const void* v_new, void* out, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  if (n_sink < 0 || n_recent < 0) return VSD_ERR_INVALID_ARG;
  if ((flags & ~VSD_VERIFY_EARLY_PREFETCH) != 0u) return VSD_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr) || !aligned(k_new, 16) || !aligned(v_new, 16))
    return VSD_ERR_INVALID_ARG;
  if (partial_scores == nullptr || score == nullptr || score_hist == nullptr)
    return geom != nullptr && geom->B == 0 ? VSD_OK : VSD_ERR_INVALID_ARG;
  // the aggregation writes the score one float at a time: 4-byte alignment suffices
  if (!aligned(score, 4) || !aligned(score_hist, 4)) return VSD_ERR_INVALID_ARG;
  return verify_call(geom, R, q, k_cache, v_cache, block_table, prefix_len, false,
                     collect_row0, collect_row1, nullptr, P_max, scale, logits,
                     partial_scores, out, workspace, workspace_bytes, stream, score,
                     score_hist, n_sink, n_recent,
                     (flags & VSD_VERIFY_EARLY_PREFETCH) ? 1 : 0, k_new, v_new);
}

vsd_status vsd_verify_attn_collect_all(const vsd_geom* geom, int R, const void* q,
                                       const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, const int32_t* prefix_len,
                                       int P_max, float scale, float* logits,
                                       float* partial_scores, void* out, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  return verify_call(geom, R, q, k_cache, v_cache, block_table, prefix_len, true, 0, 0,
                     nullptr, P_max, scale, logits, partial_scores, out, workspace,
                     workspace_bytes, stream);
}

namespace {

// Workspace of sparse verification: compact K, compact V, compact block table and
// prefix lengths, then the verification kernel's own workspace (all 256-byte aligned).
// The workspace of a sparse verification: the compressed cache and the verification
// kernel's partials (gather path), or the split partials (fused path).
struct SparseVerifyLayout {
  size_t off_k, off_v, off_table, off_prefix, off_verify, total;
  int pages;
  int fused_nq;  // > 0: the fused kernel runs
  vsd::VerifyPlan plan;
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

vsd_status sparse_verify_layout(const vsd_geom* geom, int R, int k_max, int sms,
                                SparseVerifyLayout* L) {
  L->pages = vsd::sparse_verify_pages(k_max, R);
  const size_t cache = static_cast<size_t>(geom->B) * L->pages * geom->Hkv * 16 *
                       geom->head_dim * 2;
  L->off_k = 0;
  L->off_v = round256(cache);
  L->off_table = L->off_v + round256(cache);
  L->off_prefix = L->off_table + round256(static_cast<size_t>(geom->B) * L->pages * 4);
  L->off_verify = L->off_prefix + round256(static_cast<size_t>(geom->B) * 4);
  L->plan = vsd::plan_verify(geom->B, geom->Hkv, R, geom->Hq / geom->Hkv, k_max, sms);
  const size_t gathered = L->off_verify + round256(vsd::verify_workspace_bytes(L->plan, geom->head_dim));
  const int G = geom->Hq / geom->Hkv;
  L->fused_nq = vsd::sparse_verify_fused_nq(R, G, k_max);
  const size_t fused = round256(vsd::sparse_verify_fused_bytes(geom->B, geom->Hkv, R, G, k_max,
                                                              geom->head_dim));
  L->total = L->fused_nq > 0 ? fused : gathered;
  return VSD_OK;
}

vsd_status sparse_verify_checks(const vsd_geom* geom, int R, int k_max) {
  vsd_status st = verify_checks(geom, R, k_max);
  if (st != VSD_OK) return st;
  if (k_max < 0) return VSD_ERR_INVALID_ARG;
  if (static_cast<long long>(geom->B) * vsd::sparse_verify_pages(k_max, R) > (1ll << 30))
    return VSD_ERR_UNSUPPORTED;
  return VSD_OK;
}

}  // namespace

vsd_status vsd_sparse_verify_workspace_size(const vsd_geom* geom, int R, int k_max,
                                            size_t* bytes) {
  if (bytes == nullptr) return VSD_ERR_INVALID_ARG;
  vsd_status st = sparse_verify_checks(geom, R, k_max);
  if (st != VSD_OK) return st;
  int sms = 0;
  st = device_info(nullptr, &sms);
  if (st != VSD_OK) return st;
  SparseVerifyLayout L;
  sparse_verify_layout(geom, R, k_max, sms, &L);
  *bytes = L.total;
  return VSD_OK;
}

vsd_status vsd_sparse_verify_attn(const vsd_geom* geom, int R, const void* q,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, const int32_t* prefix_len,
                                  const int32_t* idx, const int32_t* n_sel, int k_max,
                                  unsigned flags, float scale, void* out, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  vsd_status st = sparse_verify_checks(geom, R, k_max);
  if (st != VSD_OK) return st;
  if ((flags & ~VSD_SPARSE_VERIFY_EARLY_GATHER) != 0u) return VSD_ERR_INVALID_ARG;
  if (geom->B == 0) return VSD_OK;
  if (!q || !k_cache || !v_cache || !block_table || !prefix_len || !out || !workspace)
    return workspace ? VSD_ERR_INVALID_ARG : VSD_ERR_WORKSPACE;
  if (k_max > 0 && (!idx || !n_sel)) return VSD_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(block_table, 4) || !aligned(prefix_len, 4) || !aligned(idx, 4) ||
      !aligned(n_sel, 4))
    return VSD_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return VSD_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  int sms = 0;
  st = device_info(&status, &sms);
  if (st != VSD_OK) return st;
  SparseVerifyLayout L;
  sparse_verify_layout(geom, R, k_max, sms, &L);
  if (workspace_bytes < L.total || !aligned(workspace, 256)) return VSD_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  if (L.fused_nq > 0) {
    // the draft step's tensor-core kernel with the verify rows as its queries
    vsd::SparseArgs sa;
    sa.q = q;
    sa.k_cache = k_cache;
    sa.v_cache = v_cache;
    sa.block_table = block_table;
    sa.idx = k_max > 0 ? idx : nullptr;
    sa.n_sel = k_max > 0 ? n_sel : nullptr;
    sa.tail_start = prefix_len;
    sa.seq_len = nullptr;
    sa.out = out;
    sa.ws = reinterpret_cast<float*>(ws);
    sa.counters = nullptr;
    sa.status = status;
    sa.B = geom->B;
    sa.Hq = geom->Hq;
    sa.Hkv = geom->Hkv;
    sa.G = geom->Hq / geom->Hkv;
    sa.d = geom->head_dim;
    sa.max_blocks = geom->max_blocks_per_seq;
    sa.num_blocks = geom->num_blocks;
    sa.k_max = k_max;
    sa.max_tail = R;
    sa.scale = scale;
    sa.early = (flags & VSD_SPARSE_VERIFY_EARLY_GATHER) ? 1 : 0;
    cudaError_t e = vsd::launch_sparse_verify_fused(sa, R, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return VSD_OK;
  }
  vsd::SparseVerifyArgs ga;
  ga.k_cache = k_cache;
  ga.v_cache = v_cache;
  ga.block_table = block_table;
  ga.prefix_len = prefix_len;
  ga.idx = k_max > 0 ? idx : nullptr;
  ga.n_sel = k_max > 0 ? n_sel : nullptr;
  ga.compact_k = reinterpret_cast<uint16_t*>(ws + L.off_k);
  ga.compact_v = reinterpret_cast<uint16_t*>(ws + L.off_v);
  ga.compact_table = reinterpret_cast<int32_t*>(ws + L.off_table);
  ga.compact_prefix = reinterpret_cast<int32_t*>(ws + L.off_prefix);
  ga.status = status;
  ga.B = geom->B;
  ga.Hkv = geom->Hkv;
  ga.d = geom->head_dim;
  ga.R = R;
  ga.max_blocks = geom->max_blocks_per_seq;
  ga.num_blocks = geom->num_blocks;
  ga.k_max = k_max;
  // the compressed cache as a paged cache of its own
  vsd_geom cg = *geom;
  cg.max_blocks_per_seq = L.pages;
  cg.num_blocks = geom->B * L.pages;
  vsd::VerifyArgs va;
  st = make_cache_map(&va.kmap, ga.compact_k, &cg);
  if (st != VSD_OK) return st;
  st = make_cache_map(&va.vmap, ga.compact_v, &cg);
  if (st != VSD_OK) return st;
  cudaError_t e = vsd::launch_sparse_verify_gather(ga, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  va.q = q;
  va.block_table = ga.compact_table;
  va.prefix_len = ga.compact_prefix;
  va.logits = nullptr;
  va.partial = nullptr;
  va.out = out;
  va.ws = reinterpret_cast<float*>(ws + L.off_verify);
  va.status = status;
  va.B = geom->B;
  va.Hq = geom->Hq;
  va.Hkv = geom->Hkv;
  va.G = geom->Hq / geom->Hkv;
  va.R = R;
  va.d = geom->head_dim;
  va.max_blocks = L.pages;
  va.num_blocks = geom->B * L.pages;
  va.P_max = k_max;
  va.row0 = 0;
  va.row1 = 0;
  va.collect_all = 0;
  va.scale = scale;
  e = vsd::launch_verify(va, L.plan, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return VSD_OK;
}

vsd_status vsd_select_workspace_size(int n_rows, int Hkv, int P_max, int k, size_t* bytes) {
  if (bytes == nullptr || n_rows < 0 || Hkv < 1 || P_max < 0 || k < 1)
    return VSD_ERR_INVALID_ARG;
  if (vsd::select_chunk(P_max, vsd::select_cluster_size(P_max, n_rows)) < 0)
    return VSD_ERR_UNSUPPORTED;
  *bytes = 0;
  return VSD_OK;
}

vsd_status vsd_select_topk(int n_rows, int Hkv, const float* partial_scores,
                           const int32_t* prefix_len, int P_max, int k, int n_sink,
                           int n_recent, int32_t* idx, int32_t* n_sel, float* scores_out,
                           void* workspace, size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (n_rows < 0 || Hkv < 1 || P_max < 0 || k < 1 || n_sink < 0 || n_recent < 0)
    return VSD_ERR_INVALID_ARG;
  if (static_cast<long long>(n_sink) + n_recent > k) return VSD_ERR_INVALID_ARG;
  if (vsd::select_chunk(P_max, vsd::select_cluster_size(P_max, n_rows)) < 0)
    return VSD_ERR_UNSUPPORTED;
  if (n_rows == 0) return VSD_OK;
  if (!partial_scores || !prefix_len || !idx || !n_sel) return VSD_ERR_INVALID_ARG;
  if (!aligned(partial_scores, 16) || !aligned(idx, 4) || !aligned(n_sel, 4) ||
      !aligned(prefix_len, 4) || !aligned(scores_out, 4))
    return VSD_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  vsd_status st = device_info(&status, nullptr);
  if (st != VSD_OK) return st;
  vsd::SelectArgs sa;
  sa.partial = partial_scores;
  sa.prefix_len = prefix_len;
  sa.idx = idx;
  sa.n_sel = n_sel;
  sa.scores_out = scores_out;
  sa.status = status;
  sa.n_rows = n_rows;
  sa.Hkv = Hkv;
  sa.P_max = P_max;
  sa.k = k;
  sa.n_sink = n_sink;
  sa.n_recent = n_recent;
  cudaError_t e = vsd::launch_select(sa, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return VSD_OK;
}

vsd_status vsd_select_topk_scored(int n_rows, const float* score, const uint32_t* score_hist,
                                  const int32_t* prefix_len, int P_max, int k, int n_sink,
                                  int n_recent, int32_t* idx, int32_t* n_sel, void* stream) {
  if (n_rows < 0 || P_max < 0 || k < 1 || n_sink < 0 || n_recent < 0)
    return VSD_ERR_INVALID_ARG;
  if (static_cast<long long>(n_sink) + n_recent > k) return VSD_ERR_INVALID_ARG;
  if (vsd::select_scored_cluster(P_max) < 0 || n_rows > 65535) return VSD_ERR_UNSUPPORTED;
  if (n_rows == 0) return VSD_OK;
  if (!score || !score_hist || !prefix_len || !idx || !n_sel) return VSD_ERR_INVALID_ARG;
  if (!aligned(score, 16) || !aligned(score_hist, 4) || !aligned(idx, 4) ||
      !aligned(n_sel, 4) || !aligned(prefix_len, 4))
    return VSD_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  vsd_status st = device_info(&status, nullptr);
  if (st != VSD_OK) return st;
  vsd::SelectArgs sa;
  sa.partial = score;
  sa.prefix_len = prefix_len;
  sa.idx = idx;
  sa.n_sel = n_sel;
  sa.scores_out = nullptr;
  sa.status = status;
  sa.n_rows = n_rows;
  sa.Hkv = 1;
  sa.P_max = P_max;
  sa.k = k;
  sa.n_sink = n_sink;
  sa.n_recent = n_recent;
  sa.hist = score_hist;
  cudaError_t e = vsd::launch_select_scored(sa, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return VSD_OK;
}

namespace {
size_t hybrid_bitmap_bytes(int n_rows, int P_max) {
  return (static_cast<size_t>(n_rows) * ((P_max + 31) / 32) * 4 + 255) / 256 * 256;
}
}  // namespace

vsd_status vsd_select_hybrid_workspace_size(int n_rows, int P_max, size_t* bytes) {
  if (bytes == nullptr || n_rows < 0 || P_max < 0) return VSD_ERR_INVALID_ARG;
  if (vsd::select_chunk(P_max, vsd::select_cluster_size(P_max, n_rows)) < 0)
    return VSD_ERR_UNSUPPORTED;
  *bytes = hybrid_bitmap_bytes(n_rows, P_max) + (static_cast<size_t>(n_rows) * 4 + 255) / 256 * 256;
  return VSD_OK;
}

vsd_status vsd_select_topk_hybrid(int n_rows, int Hkv_target, const float* partial_target,
                                  int Hkv_draft, const float* partial_draft,
                                  const int32_t* prefix_len, int P_max, int k, int m,
                                  int n_sink, int n_recent, int32_t* idx, int32_t* n_sel,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (n_rows < 0 || Hkv_target < 1 || Hkv_draft < 1 || P_max < 0 || k < 1 || m < 0 ||
      n_sink < 0 || n_recent < 0)
    return VSD_ERR_INVALID_ARG;
  if (static_cast<long long>(n_sink) + n_recent > k) return VSD_ERR_INVALID_ARG;
  if (vsd::select_chunk(P_max, vsd::select_cluster_size(P_max, n_rows)) < 0)
    return VSD_ERR_UNSUPPORTED;
  if (n_rows == 0) return VSD_OK;
  if (!partial_target || !partial_draft || !prefix_len || !idx || !n_sel)
    return VSD_ERR_INVALID_ARG;
  if (!aligned(partial_target, 16) || !aligned(partial_draft, 16) || !aligned(idx, 4) ||
      !aligned(n_sel, 4) || !aligned(prefix_len, 4))
    return VSD_ERR_INVALID_ARG;
  size_t need = 0;
  vsd_status st = vsd_select_hybrid_workspace_size(n_rows, P_max, &need);
  if (st != VSD_OK) return st;
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
    return VSD_ERR_WORKSPACE;
  unsigned* status = nullptr;
  st = device_info(&status, nullptr);
  if (st != VSD_OK) return st;
  uint32_t* bitmap = static_cast<uint32_t*>(workspace);
  int32_t* counts = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) +
                                               hybrid_bitmap_bytes(n_rows, P_max));
  // pass 1: the draft signal, at most m candidates; their bitmap and count
  vsd::SelectArgs sa;
  sa.partial = partial_draft;
  sa.prefix_len = prefix_len;
  sa.idx = idx;
  sa.n_sel = n_sel;
  sa.scores_out = nullptr;
  sa.status = status;
  sa.n_rows = n_rows;
  sa.Hkv = Hkv_draft;
  sa.P_max = P_max;
  sa.k = k;
  sa.n_sink = n_sink;
  sa.n_recent = n_recent;
  sa.m_limit = m;
  sa.out_bitmap = bitmap;
  sa.out_count = counts;
  cudaError_t e = vsd::launch_select(sa, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  // pass 2: the target signal over the rest of the budget
  sa.partial = partial_target;
  sa.Hkv = Hkv_target;
  sa.m_limit = -1;
  sa.out_bitmap = nullptr;
  sa.out_count = nullptr;
  sa.pre_bitmap = bitmap;
  sa.pre_count = counts;
  e = vsd::launch_select(sa, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return VSD_OK;
}

vsd_status vsd_sparse_workspace_size(const vsd_geom* geom, int k_max, int max_tail,
                                     size_t* bytes) {
  if (bytes == nullptr || k_max < 0 || max_tail < 0) return VSD_ERR_INVALID_ARG;
  vsd_status st = check_geom(geom);
  if (st != VSD_OK) return st;
  if (geom->Hq / geom->Hkv > 16) return VSD_ERR_UNSUPPORTED;
  *bytes = vsd::sparse_workspace_bytes(vsd::plan_sparse(k_max, max_tail), geom->B, geom->Hkv,
                                       geom->Hq / geom->Hkv, geom->head_dim);
  return VSD_OK;
}

}  // extern "C"

namespace {

// The draft step with its options (see vsd_sparse_decode_attn_step); the plain call
// passes none of them.
vsd_status sparse_step(const vsd_geom* geom, const void* q, const void* k_new, const void* v_new,
                       const void* k_cache, const void* v_cache, void* k_store, void* v_store,
                       const int32_t* block_table, const int32_t* idx, const int32_t* n_sel,
                       int k_max, const int32_t* tail_start, const int32_t* seq_len,
                       int max_tail, int32_t* sel_rows, unsigned flags, float scale, void* out,
                       void* workspace, size_t workspace_bytes, void* stream) {
  const unsigned kKnown = VSD_STEP_RECORD_ROWS | VSD_STEP_REUSE_ROWS | VSD_STEP_EARLY_GATHER;
  if ((flags & ~kKnown) != 0u) return VSD_ERR_INVALID_ARG;
  const int rows_mode = (flags & VSD_STEP_RECORD_ROWS) ? 1 : (flags & VSD_STEP_REUSE_ROWS) ? 2 : 0;
  if ((flags & VSD_STEP_RECORD_ROWS) && (flags & VSD_STEP_REUSE_ROWS)) return VSD_ERR_INVALID_ARG;
  vsd_status st = check_geom(geom);
  if (st != VSD_OK) return st;
  if (geom->Hq / geom->Hkv > 16) return VSD_ERR_UNSUPPORTED;
  if (k_max < 0 || max_tail < 0) return VSD_ERR_INVALID_ARG;
  if (geom->B > 65535) return VSD_ERR_UNSUPPORTED;
  // cache rows are 32-bit: block * Hkv * page_size + offset
  if (static_cast<long long>(geom->num_blocks) * geom->Hkv * geom->page_size > 0x7FFFFFFFll)
    return VSD_ERR_UNSUPPORTED;
  if ((k_new == nullptr) != (v_new == nullptr)) return VSD_ERR_INVALID_ARG;
  if (rows_mode != 0 && k_max > 0 && sel_rows == nullptr) return VSD_ERR_INVALID_ARG;
  if (geom->B == 0) return VSD_OK;
  const vsd::SparsePlan splan = vsd::plan_sparse(k_max, max_tail);
  const size_t need = vsd::sparse_workspace_bytes(splan, geom->B, geom->Hkv,
                                                  geom->Hq / geom->Hkv, geom->head_dim);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256)))
    return VSD_ERR_WORKSPACE;
  if (!q || !k_cache || !v_cache || !block_table || !tail_start || !seq_len || !out)
    return VSD_ERR_INVALID_ARG;
  if (k_max > 0 && (!idx || !n_sel)) return VSD_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(idx, 4) || !aligned(n_sel, 4) || !aligned(block_table, 4) ||
      !aligned(tail_start, 4) || !aligned(seq_len, 4) || !aligned(k_new, 16) ||
      !aligned(v_new, 16) || !aligned(sel_rows, 4))
    return VSD_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return VSD_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  st = device_info(&status, nullptr);
  if (st != VSD_OK) return st;
  vsd::SparseArgs sa;
  sa.q = q;
  sa.k_cache = k_cache;
  sa.v_cache = v_cache;
  sa.k_new = k_new;
  sa.v_new = v_new;
  sa.k_store = k_store;
  sa.v_store = v_store;
  sa.sel_rows = k_max > 0 ? sel_rows : nullptr;
  sa.rows_mode = k_max > 0 ? rows_mode : 0;
  sa.early = (flags & VSD_STEP_EARLY_GATHER) ? 1 : 0;
  sa.block_table = block_table;
  sa.idx = k_max > 0 ? idx : nullptr;
  sa.n_sel = k_max > 0 ? n_sel : nullptr;
  sa.tail_start = tail_start;
  sa.seq_len = seq_len;
  sa.out = out;
  sa.counters = need > 0 ? static_cast<unsigned*>(workspace) : nullptr;
  sa.ws = need > 0 ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                               vsd::sparse_counter_bytes(splan, geom->B,
                                                                         geom->Hkv))
                   : nullptr;
  sa.status = status;
  sa.B = geom->B;
  sa.Hq = geom->Hq;
  sa.Hkv = geom->Hkv;
  sa.G = geom->Hq / geom->Hkv;
  sa.d = geom->head_dim;
  sa.max_blocks = geom->max_blocks_per_seq;
  sa.num_blocks = geom->num_blocks;
  sa.k_max = k_max;
  sa.max_tail = max_tail;
  sa.scale = scale;
  cudaError_t e = vsd::launch_sparse(sa, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return VSD_OK;
}

}  // namespace

extern "C" {

vsd_status vsd_sparse_decode_attn(const vsd_geom* geom, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_table,
                                  const int32_t* idx, const int32_t* n_sel, int k_max,
                                  const int32_t* tail_start, const int32_t* seq_len,
                                  int max_tail, float scale, void* out, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return sparse_step(geom, q, nullptr, nullptr, k_cache, v_cache, nullptr, nullptr, block_table,
                     idx, n_sel, k_max, tail_start, seq_len, max_tail, nullptr, 0u, scale, out,
                     workspace, workspace_bytes, stream);
}

vsd_status vsd_sparse_decode_attn_step(const vsd_geom* geom, const void* q, const void* k_new,
                                       const void* v_new, void* k_cache, void* v_cache,
                                       const int32_t* block_table, const int32_t* idx,
                                       const int32_t* n_sel, int k_max,
                                       const int32_t* tail_start, const int32_t* seq_len,
                                       int max_tail, int32_t* sel_rows, unsigned flags,
                                       float scale, void* out, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  return sparse_step(geom, q, k_new, v_new, k_cache, v_cache, k_cache, v_cache, block_table, idx,
                     n_sel, k_max, tail_start, seq_len, max_tail, sel_rows, flags, scale, out,
                     workspace, workspace_bytes, stream);
}

vsd_status vsd_copy(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return VSD_OK;
  if (!dst || !src || bytes % 16 != 0 || !aligned(dst, 16) || !aligned(src, 16))
    return VSD_ERR_INVALID_ARG;
  cudaError_t e = vsd::launch_copy16(dst, src, bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return VSD_OK;
}

vsd_status vsd_append_kv(const vsd_geom* geom, int n_new, const void* k_new, const void* v_new,
                         const int32_t* block_table, const int32_t* pos_base, int pos_offset,
                         void* k_cache, void* v_cache, void* stream) {
  vsd_status st = check_geom(geom);
  if (st != VSD_OK) return st;
  if (n_new < 0) return VSD_ERR_INVALID_ARG;
  if (geom->B == 0 || n_new == 0) return VSD_OK;
  if (!k_new || !v_new || !block_table || !pos_base || !k_cache || !v_cache)
    return VSD_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(block_table, 4) || !aligned(pos_base, 4))
    return VSD_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  st = device_info(&status, nullptr);
  if (st != VSD_OK) return st;
  vsd::AppendArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.block_table = block_table;
  a.pos_base = pos_base;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.status = status;
  a.B = geom->B;
  a.n_new = n_new;
  a.Hkv = geom->Hkv;
  a.d = geom->head_dim;
  a.max_blocks = geom->max_blocks_per_seq;
  a.num_blocks = geom->num_blocks;
  a.pos_offset = pos_offset;
  cudaError_t e = vsd::launch_append_kv(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return VSD_OK;
}

vsd_status vsd_advance_lengths(int B, int gamma, const int32_t* accepted, int max_prefix,
                               int32_t* prefix_len, int32_t* tail_start, int32_t* seq_len,
                               int n_copies, int32_t* prefix_copies, void* stream) {
  if (B < 0 || gamma < 0 || n_copies < 0 || max_prefix < 0) return VSD_ERR_INVALID_ARG;
  if (B == 0) return VSD_OK;
  if (!accepted || !prefix_len || !tail_start || (gamma > 0 && !seq_len) ||
      (n_copies > 0 && !prefix_copies))
    return VSD_ERR_INVALID_ARG;
  if (!aligned(accepted, 4) || !aligned(prefix_len, 4) || !aligned(tail_start, 4) ||
      !aligned(seq_len, 4) || !aligned(prefix_copies, 4))
    return VSD_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  vsd_status st = device_info(&status, nullptr);
  if (st != VSD_OK) return st;
  vsd::AdvanceArgs a;
  a.accepted = accepted;
  a.prefix_len = prefix_len;
  a.tail_start = tail_start;
  a.seq_len = seq_len;
  a.prefix_copies = n_copies > 0 ? prefix_copies : nullptr;
  a.status = status;
  a.B = B;
  a.gamma = gamma;
  a.max_prefix = max_prefix;
  a.n_copies = n_copies;
  cudaError_t e = vsd::launch_advance(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return VSD_OK;
}

vsd_status vsd_page_key_means(const vsd_geom* geom, const void* k_cache,
                              const int32_t* block_table, const int32_t* prefix_len,
                              const int32_t* page_begin, int page_blocks_max,
                              float* page_means, void* stream) {
  vsd_status st = check_geom(geom);
  if (st != VSD_OK) return st;
  if (page_blocks_max < 0) return VSD_ERR_INVALID_ARG;
  if (vsd::block_select_items(page_blocks_max) < 0 || geom->B > 65535 || geom->Hkv > 65535)
    return VSD_ERR_UNSUPPORTED;
  if (geom->B == 0 || page_blocks_max == 0) return VSD_OK;
  if (!k_cache || !block_table || !prefix_len || !page_means) return VSD_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(page_means, 16) || !aligned(block_table, 4) ||
      !aligned(prefix_len, 4) || !aligned(page_begin, 4))
    return VSD_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  st = device_info(&status, nullptr);
  if (st != VSD_OK) return st;
  vsd::BlockTopkArgs a = {};
  a.k_cache = k_cache;
  a.block_table = block_table;
  a.prefix_len = prefix_len;
  a.page_begin = page_begin;
  a.kbar = page_means;
  a.status = status;
  a.B = geom->B;
  a.Hq = geom->Hq;
  a.Hkv = geom->Hkv;
  a.G = geom->Hq / geom->Hkv;
  a.d = geom->head_dim;
  a.max_blocks = geom->max_blocks_per_seq;
  a.num_blocks = geom->num_blocks;
  a.nblk_max = page_blocks_max;
  cudaError_t e = vsd::launch_page_means(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return VSD_OK;
}

vsd_status vsd_block_topk(const vsd_geom* geom, int R, const void* q, const float* page_means,
                          const int32_t* prefix_len, int page_blocks_max, int kb, float scale,
                          float* scores, int32_t* blocks, void* stream) {
  vsd_status st = check_geom(geom);
  if (st != VSD_OK) return st;
  if (R < 1 || kb < 1 || page_blocks_max < 0) return VSD_ERR_INVALID_ARG;
  const int G = geom->Hq / geom->Hkv;
  if (R * G > 64 || vsd::block_select_items(page_blocks_max) < 0 || geom->B > 65535 ||
      geom->Hkv > 65535)
    return VSD_ERR_UNSUPPORTED;
  if (static_cast<long long>(geom->B) * R * geom->Hq > 0x7FFFFFFFll ||
      static_cast<long long>(geom->B) * geom->Hkv * page_blocks_max > 0x7FFFFFFFll)
    return VSD_ERR_UNSUPPORTED;
  if (geom->B == 0) return VSD_OK;
  if (!q || !prefix_len || !blocks || (page_blocks_max > 0 && (!page_means || !scores)))
    return VSD_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(page_means, 16) || !aligned(scores, 16) ||
      !aligned(prefix_len, 4) || !aligned(blocks, 4))
    return VSD_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return VSD_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  st = device_info(&status, nullptr);
  if (st != VSD_OK) return st;
  vsd::BlockTopkArgs a = {};
  a.prefix_len = prefix_len;
  a.q = q;
  a.kbar = const_cast<float*>(page_means);
  a.scores = scores;
  a.blocks = blocks;
  a.status = status;
  a.B = geom->B;
  a.R = R;
  a.Hq = geom->Hq;
  a.Hkv = geom->Hkv;
  a.G = G;
  a.d = geom->head_dim;
  a.max_blocks = geom->max_blocks_per_seq;
  a.num_blocks = geom->num_blocks;
  a.nblk_max = page_blocks_max;
  a.kb = kb;
  a.scale = scale;
  CUtensorMap map;
  if (page_blocks_max > 0) {
    st = make_means_map(&map, page_means, geom->head_dim,
                        static_cast<long long>(geom->B) * geom->Hkv * page_blocks_max);
    if (st != VSD_OK) return st;
  }
  cudaError_t e = vsd::launch_block_topk(map, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return VSD_OK;
}

}  // extern "C"
