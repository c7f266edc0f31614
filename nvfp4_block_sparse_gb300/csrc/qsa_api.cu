// qsa_api.cu -- the library's C ABI (declared in include/qsa.h): host-side
// argument validation, the sm_103 gate and the launches on the caller's
// stream.  Nothing here allocates, synchronises (except the diagnostic
// qsa_workspace_status) or reads device data.
//
// TensorRT-LLM PR #20937 ("GB300 perf work on
// qwen3_8_flash_next_nvfp4__sm_103__tp1"), review of the grouped-verify
// tests: the grouped NVFP4 path runs on SM 10.3 only; callers pass their own
// buffers (Per-File QA: caller-provided buffers).
#include "qsa_common.cuh"

#include <math.h>
#include <stdint.h>

#include <atomic>

namespace {

using qsa::Geom;

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// max_rows: 8 for the decode / verify attention and the rollback; the index
// scores, the selection, the prologue and the context row-tile attention also
// take long context row groups.
qsa_status_t check_geom(const qsa_geom_t* g, int max_rows = qsa::kMaxRows) {
  if (!g) return QSA_ERR_INVALID_ARG;
  if (g->batch < 1 || g->batch > 65535) return QSA_ERR_INVALID_ARG;
  if (g->rows_per_req < 1) return QSA_ERR_INVALID_ARG;
  if (g->num_q_heads < 1 || g->num_kv_heads < 1) return QSA_ERR_INVALID_ARG;
  if (g->num_q_heads % g->num_kv_heads != 0) return QSA_ERR_INVALID_ARG;
  if (g->max_blocks < 1 || g->num_pages < 1) return QSA_ERR_INVALID_ARG;
  // head_dim 128 with 64/128-token pages; head_dim 256 (PR #20276, Performance,
  // shared code touched: the target's 24 q / 2 KV heads at head_dim 256) with
  // 32-token pages (Known limitations: tokens_per_block 32) or 64.
  if (g->index_dim != qsa::kIndexDim) return QSA_ERR_UNSUPPORTED;
  if (g->head_dim == 128) {
    if (g->page_size != 64 && g->page_size != 128) return QSA_ERR_UNSUPPORTED;
  } else if (g->head_dim == 256) {
    if (g->page_size != 32 && g->page_size != 64) return QSA_ERR_UNSUPPORTED;
  } else {
    return QSA_ERR_UNSUPPORTED;
  }
  if (g->rows_per_req > max_rows) return QSA_ERR_UNSUPPORTED;
  if (g->num_q_heads > qsa::kMaxQHeads) return QSA_ERR_UNSUPPORTED;
  if (g->max_blocks > qsa::kMaxBlocks) return QSA_ERR_UNSUPPORTED;
  if ((long long)g->batch * g->rows_per_req > (1LL << 24)) return QSA_ERR_UNSUPPORTED;
  return QSA_OK;
}

Geom to_geom(const qsa_geom_t* g) {
  Geom r;
  r.B = g->batch;
  r.R = g->rows_per_req;
  r.Hq = g->num_q_heads;
  r.Hkv = g->num_kv_heads;
  r.D = g->head_dim;
  r.Di = g->index_dim;
  r.P = g->page_size;
  r.MB = g->max_blocks;
  r.NP = g->num_pages;
  return r;
}

// The kernels use sm_103a instructions (tcgen05-era conversions, bulk copies).
qsa_status_t check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return QSA_ERR_UNSUPPORTED;
  return QSA_OK;
}

qsa_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) e = cudaGetLastError();
  else cudaGetLastError();
  return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

qsa_status_t check_decode_args(const qsa_geom_t* geom, int k) {
  qsa_status_t st = check_geom(geom);
  if (st != QSA_OK) return st;
  if (k < 1) return QSA_ERR_INVALID_ARG;
  if (k > qsa::kMaxK) return QSA_ERR_UNSUPPORTED;
  if ((long long)geom->rows_per_req * k > qsa::kMaxUnion) return QSA_ERR_UNSUPPORTED;
  return QSA_OK;
}

}  // namespace

namespace qsa {
unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
}  // namespace qsa

extern "C" {

void qsa_debug_set_wait_ns(unsigned long long ns) {
  g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
}

int qsa_debug_bounds_status(void) {
#ifdef QSA_DEBUG_BOUNDS
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  int first = 0;
  for (int v : {qsa::bounds_word_attend(), qsa::bounds_word_decode(), qsa::bounds_word_index(),
                qsa::bounds_word_select(), qsa::bounds_word_store(), qsa::bounds_word_rollback(),
                qsa::bounds_word_prefill()}) {
    if (v < 0) return -1;
    if (first == 0) first = v;
  }
  return first;
#else
  return -1;
#endif
}

const char* qsa_status_string(qsa_status_t s) {
  switch (s) {
    case QSA_OK: return "ok";
    case QSA_ERR_INVALID_ARG: return "invalid argument";
    case QSA_ERR_UNSUPPORTED: return "unsupported shape or device (needs sm_103)";
    case QSA_ERR_CUDA: return "CUDA error";
    case QSA_ERR_WORKSPACE: return "workspace missing or too small";
    case QSA_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
  }
  return "unknown status";
}

qsa_status_t qsa_store_kv_tokens(const qsa_geom_t* geom, const void* k_new_bf16,
                                 const void* v_new_bf16, const int8_t* ik_new, float k_scale,
                                 float v_scale, const int32_t* page_table,
                                 const int32_t* seqlens, uint8_t* k_pool, uint8_t* k_sf,
                                 uint8_t* v_pool, uint8_t* v_sf, int8_t* ik_pool,
                                 cudaStream_t stream) {
  qsa_status_t st = check_geom(geom, qsa::kMaxContextRows);
  if (st != QSA_OK) return st;
  if (!k_new_bf16 || !v_new_bf16 || !ik_new || !page_table || !seqlens || !k_pool || !k_sf ||
      !v_pool || !v_sf || !ik_pool)
    return QSA_ERR_INVALID_ARG;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale))
    return QSA_ERR_INVALID_ARG;
  // A lane moves D/32 values: 8 or 16 bytes of bf16 in, 2 or 4 code bytes out.
  const uintptr_t in_al = geom->head_dim / 16, out_al = geom->head_dim / 64;
  if (!aligned(k_new_bf16, in_al) || !aligned(v_new_bf16, in_al) || !aligned(ik_new, 4) ||
      !aligned(ik_pool, 4) || !aligned(k_pool, out_al) || !aligned(v_pool, out_al))
    return QSA_ERR_INVALID_ARG;
  st = check_device();
  if (st != QSA_OK) return st;
  return from_cuda(qsa::launch_store_tokens(to_geom(geom), k_new_bf16, v_new_bf16, ik_new,
                                            k_scale, v_scale, page_table, seqlens, k_pool, k_sf,
                                            v_pool, v_sf, ik_pool, true, stream));
}

size_t qsa_rollback_state_bytes(const qsa_geom_t* geom) {
  if (check_geom(geom) != QSA_OK) return 0;
  return (size_t)geom->batch * geom->rows_per_req * qsa::rollback_row_bytes(geom->num_kv_heads, geom->head_dim);
}

qsa_status_t qsa_rollback_gather(const qsa_geom_t* geom, const int32_t* page_table,
                                 const int32_t* seqlens, const uint8_t* k_pool,
                                 const uint8_t* k_sf, const uint8_t* v_pool, const uint8_t* v_sf,
                                 const int8_t* ik_pool, void* saved, cudaStream_t stream) {
  qsa_status_t st = check_geom(geom);
  if (st != QSA_OK) return st;
  if (!page_table || !seqlens || !k_pool || !k_sf || !v_pool || !v_sf || !ik_pool || !saved)
    return QSA_ERR_INVALID_ARG;
  if (!aligned(k_pool, 4) || !aligned(k_sf, 4) || !aligned(v_pool, 4) || !aligned(v_sf, 4) ||
      !aligned(ik_pool, 4) || !aligned(saved, 4))
    return QSA_ERR_INVALID_ARG;
  st = check_device();
  if (st != QSA_OK) return st;
  return from_cuda(qsa::launch_rollback(
      to_geom(geom), false, page_table, seqlens, nullptr, const_cast<uint8_t*>(k_pool),
      const_cast<uint8_t*>(k_sf), const_cast<uint8_t*>(v_pool), const_cast<uint8_t*>(v_sf),
      const_cast<int8_t*>(ik_pool), reinterpret_cast<uint8_t*>(saved), true, stream));
}

qsa_status_t qsa_rollback_restore(const qsa_geom_t* geom, const int32_t* page_table,
                                  const int32_t* seqlens, const int32_t* rejected,
                                  const void* saved, uint8_t* k_pool, uint8_t* k_sf,
                                  uint8_t* v_pool, uint8_t* v_sf, int8_t* ik_pool,
                                  cudaStream_t stream) {
  qsa_status_t st = check_geom(geom);
  if (st != QSA_OK) return st;
  if (!page_table || !seqlens || !rejected || !saved || !k_pool || !k_sf || !v_pool || !v_sf ||
      !ik_pool)
    return QSA_ERR_INVALID_ARG;
  if (!aligned(k_pool, 4) || !aligned(k_sf, 4) || !aligned(v_pool, 4) || !aligned(v_sf, 4) ||
      !aligned(ik_pool, 4) || !aligned(saved, 4))
    return QSA_ERR_INVALID_ARG;
  st = check_device();
  if (st != QSA_OK) return st;
  return from_cuda(qsa::launch_rollback(to_geom(geom), true, page_table, seqlens, rejected,
                                        k_pool, k_sf, v_pool, v_sf, ik_pool,
                                        const_cast<uint8_t*>(reinterpret_cast<const uint8_t*>(saved)),
                                        true, stream));
}

qsa_status_t qsa_index_scores(const qsa_geom_t* geom, const int8_t* iq, const int8_t* ik_pool,
                              const int32_t* page_table, const int32_t* seqlens,
                              int32_t* scores, cudaStream_t stream) {
  qsa_status_t st = check_geom(geom, qsa::kMaxContextRows);
  if (st != QSA_OK) return st;
  if (!iq || !ik_pool || !page_table || !seqlens || !scores) return QSA_ERR_INVALID_ARG;
  if (!aligned(ik_pool, 16) || !aligned(iq, 16)) return QSA_ERR_INVALID_ARG;
  st = check_device();
  if (st != QSA_OK) return st;
  return from_cuda(qsa::launch_index_scores(to_geom(geom), iq, ik_pool, page_table, seqlens,
                                            scores, true, stream));
}

qsa_status_t qsa_select_topk(const qsa_geom_t* geom, const int32_t* scores,
                             const int32_t* seqlens, int k, int window, int32_t* sel,
                             int32_t* nsel, cudaStream_t stream) {
  qsa_status_t st = check_geom(geom, qsa::kMaxContextRows);
  if (st != QSA_OK) return st;
  if (!scores || !seqlens || !sel || !nsel) return QSA_ERR_INVALID_ARG;
  if (k < 1 || window < 0 || window > k) return QSA_ERR_INVALID_ARG;
  if (k > qsa::kMaxK) return QSA_ERR_UNSUPPORTED;
  st = check_device();
  if (st != QSA_OK) return st;
  return from_cuda(qsa::launch_select_topk(to_geom(geom), scores, seqlens, k, window, sel, nsel,
                                           true, stream));
}

size_t qsa_sparse_decode_workspace_bytes_ex(const qsa_geom_t* geom, int k, int num_splits) {
  if (check_decode_args(geom, k) != QSA_OK || num_splits < 0) return 0;
  return qsa::plan_sparse_decode(to_geom(geom), k, num_splits).ws_bytes;
}

size_t qsa_sparse_decode_workspace_bytes(const qsa_geom_t* geom, int k) {
  return qsa_sparse_decode_workspace_bytes_ex(geom, k, 0);
}

qsa_status_t qsa_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!workspace || workspace_bytes == 0) return QSA_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(workspace, 0, workspace_bytes, stream));
}

qsa_status_t qsa_sparse_decode_ex(const qsa_geom_t* geom, const void* q_bf16,
                                  const uint8_t* k_pool, const uint8_t* k_sf,
                                  const uint8_t* v_pool, const uint8_t* v_sf, float k_scale,
                                  float v_scale, float sm_scale, const int32_t* page_table,
                                  const int32_t* seqlens, const int32_t* sel, int k,
                                  void* out_bf16, float* lse, void* workspace,
                                  size_t workspace_bytes, int num_splits, cudaStream_t stream) {
  qsa_status_t st = check_decode_args(geom, k);
  if (st != QSA_OK) return st;
  if (num_splits < 0) return QSA_ERR_INVALID_ARG;
  if (!q_bf16 || !k_pool || !k_sf || !v_pool || !v_sf || !page_table || !seqlens || !sel ||
      !out_bf16 || !lse)
    return QSA_ERR_INVALID_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(k_sf, 16) || !aligned(v_sf, 16) ||
      !aligned(q_bf16, 8))
    return QSA_ERR_INVALID_ARG;
  const Geom g = to_geom(geom);
  const qsa::DecodePlan plan = qsa::plan_sparse_decode(g, k, num_splits);
  if (!workspace || workspace_bytes < plan.ws_bytes || !aligned(workspace, 256))
    return QSA_ERR_WORKSPACE;
  st = check_device();
  if (st != QSA_OK) return st;
  // Verify rows launch without programmatic dependent launch: their grid is
  // planned to fill every CTA slot of the GPU in one wave, and CTAs placed
  // early (while the selection kernel still holds its SMs) left clusters
  // for a second wave (wide aggregated verify: 139.5 us per step with it,
  // 102.8 us without).  Decode rows keep the overlap.
  return from_cuda(qsa::launch_sparse_decode(g, plan, q_bf16, k_pool, k_sf, v_pool, v_sf, k_scale,
                                             v_scale, sm_scale, page_table, seqlens, sel, k,
                                             out_bf16, lse, workspace, g.R == 1, stream));
}

// Context row groups: head_dim 128 or 256, a head group of at most 128 heads,
// and a tile's selections + union within the CTA's shared memory.
qsa_status_t check_prefill_args(const qsa_geom_t* geom, int k) {
  qsa_status_t st = check_geom(geom, qsa::kMaxContextRows);
  if (st != QSA_OK) return st;
  if (k < 1) return QSA_ERR_INVALID_ARG;
  if (k > qsa::kMaxK || (geom->head_dim != 128 && geom->head_dim != 256))
    return QSA_ERR_UNSUPPORTED;
  const Geom g = to_geom(geom);
  if (qsa::prefill_rows_per_tile(g) < 1) return QSA_ERR_UNSUPPORTED;
  if (qsa::prefill_smem_bytes(g, k) > 227 * 1024) return QSA_ERR_UNSUPPORTED;
  return QSA_OK;
}

size_t qsa_sparse_prefill_workspace_bytes(const qsa_geom_t* geom, int k) {
  return check_prefill_args(geom, k) == QSA_OK ? 256 : 0;
}

qsa_status_t qsa_sparse_prefill(const qsa_geom_t* geom, const void* q_bf16,
                                const uint8_t* k_pool, const uint8_t* k_sf,
                                const uint8_t* v_pool, const uint8_t* v_sf, float k_scale,
                                float v_scale, float sm_scale, const int32_t* page_table,
                                const int32_t* seqlens, const int32_t* sel, int k,
                                void* out_bf16, float* lse, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  qsa_status_t st = check_prefill_args(geom, k);
  if (st != QSA_OK) return st;
  if (!q_bf16 || !k_pool || !k_sf || !v_pool || !v_sf || !page_table || !seqlens || !sel ||
      !out_bf16 || !lse)
    return QSA_ERR_INVALID_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(k_sf, 16) || !aligned(v_sf, 16) ||
      !aligned(q_bf16, 16) || !aligned(out_bf16, 16))
    return QSA_ERR_INVALID_ARG;
  if (!(k_scale > 0.f) || !(sm_scale > 0.f) || !isfinite(k_scale) || !isfinite(sm_scale) ||
      !isfinite(v_scale))
    return QSA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < 256 || !aligned(workspace, 256)) return QSA_ERR_WORKSPACE;
  st = check_device();
  if (st != QSA_OK) return st;
  return from_cuda(qsa::launch_sparse_prefill(to_geom(geom), q_bf16, k_pool, k_sf, v_pool, v_sf,
                                              k_scale, v_scale, sm_scale, page_table, seqlens,
                                              sel, k, out_bf16, lse,
                                              reinterpret_cast<int*>(workspace), stream));
}

int qsa_select_sparse_decode_fused(const qsa_geom_t* geom) {
  if (check_geom(geom) != QSA_OK) return 0;
  return qsa::decode_can_fuse_select(to_geom(geom)) ? 1 : 0;
}

qsa_status_t qsa_select_sparse_decode(const qsa_geom_t* geom, const int32_t* scores, int window,
                                      const void* q_bf16, const uint8_t* k_pool,
                                      const uint8_t* k_sf, const uint8_t* v_pool,
                                      const uint8_t* v_sf, float k_scale, float v_scale,
                                      float sm_scale, const int32_t* page_table,
                                      const int32_t* seqlens, int k, int32_t* sel, int32_t* nsel,
                                      void* out_bf16, float* lse, void* workspace,
                                      size_t workspace_bytes, int num_splits,
                                      cudaStream_t stream) {
  qsa_status_t st = check_decode_args(geom, k);
  if (st != QSA_OK) return st;
  if (window < 0 || window > k || num_splits < 0) return QSA_ERR_INVALID_ARG;
  if (!scores || !q_bf16 || !k_pool || !k_sf || !v_pool || !v_sf || !page_table || !seqlens ||
      !sel || !nsel || !out_bf16 || !lse)
    return QSA_ERR_INVALID_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(k_sf, 16) || !aligned(v_sf, 16) ||
      !aligned(q_bf16, 8))
    return QSA_ERR_INVALID_ARG;
  const Geom g = to_geom(geom);
  const qsa::DecodePlan plan = qsa::plan_sparse_decode(g, k, num_splits);
  if (!workspace || workspace_bytes < plan.ws_bytes || !aligned(workspace, 256))
    return QSA_ERR_WORKSPACE;
  st = check_device();
  if (st != QSA_OK) return st;
  if (qsa::decode_can_fuse_select(g))
    return from_cuda(qsa::launch_sparse_decode(g, plan, q_bf16, k_pool, k_sf, v_pool, v_sf,
                                               k_scale, v_scale, sm_scale, page_table, seqlens,
                                               nullptr, k, out_bf16, lse, workspace, true, stream,
                                               scores, window, sel, nsel));
  cudaError_t e = qsa::launch_select_topk(g, scores, seqlens, k, window, sel, nsel, true, stream);
  if (e != cudaSuccess) return from_cuda(e);
  // Verify rows launch without programmatic dependent launch: their grid is
  // planned to fill every CTA slot of the GPU in one wave, and CTAs placed
  // early (while the selection kernel still holds its SMs) left clusters
  // for a second wave (wide aggregated verify: 139.5 us per step with it,
  // 102.8 us without).  Decode rows keep the overlap.
  return from_cuda(qsa::launch_sparse_decode(g, plan, q_bf16, k_pool, k_sf, v_pool, v_sf, k_scale,
                                             v_scale, sm_scale, page_table, seqlens, sel, k,
                                             out_bf16, lse, workspace, g.R == 1, stream));
}

qsa_status_t qsa_sparse_decode(const qsa_geom_t* geom, const void* q_bf16, const uint8_t* k_pool,
                               const uint8_t* k_sf, const uint8_t* v_pool, const uint8_t* v_sf,
                               float k_scale, float v_scale, float sm_scale,
                               const int32_t* page_table, const int32_t* seqlens,
                               const int32_t* sel, int k, void* out_bf16, float* lse,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return qsa_sparse_decode_ex(geom, q_bf16, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale,
                              sm_scale, page_table, seqlens, sel, k, out_bf16, lse, workspace,
                              workspace_bytes, 0, stream);
}

qsa_status_t qsa_workspace_status(const void* workspace, int* device_code, cudaStream_t stream) {
  if (!workspace || !device_code) return QSA_ERR_INVALID_ARG;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  *device_code = v;
  return v == 0 ? QSA_OK : QSA_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
