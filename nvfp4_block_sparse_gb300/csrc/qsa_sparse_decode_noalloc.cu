// qsa_sparse_decode_noalloc.cu -- qsa_sparse_decode for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a workspace: code running
// where cudaMalloc is unavailable or forbidden once the process is serving
// (a pre-reserved memory pool that must not grow, an allocator-free runtime,
// a plugin that only ever receives input and output pointers).  This entry
// point runs the same sparse decode kernel, but takes its scratch (the split
// tickets, the status word and the split partials) from a fixed array that is
// compiled into the library.  It calls no cudaMalloc, cudaFree or allocating
// library routine.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it until the process exits, and every call on that GPU shares
// it: calls that overlap on the GPU (two streams, or two threads) race on it
// and must be serialised by the caller.  Its split tickets start at zero (a
// __device__ array is zero-filled when the module loads) and every call leaves
// them at zero again, so nothing is cleared between calls and the call keeps
// the programmatic-launch overlap with the kernel before it.  Its status word
// is sticky: a bounded device wait that gives up in any call sets it, and
// qsa_sparse_decode_noalloc_status() reads and clears it.
#include "qsa_common.cuh"

namespace {

// 4 MiB: the status word and tickets always fit; the number of KV splits is
// reduced until the split partials fit as well.
constexpr size_t kNoAllocBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// The device address of the scratch array on the current device.  The name
// g_noalloc_scratch is only a host-side handle; kernels and copies must be
// given the address cudaGetSymbolAddress returns.  It is looked up on every
// call (host-only and cheap), so a context created anew on the device (after
// cudaDeviceReset, say) gets its own array's address.
qsa_status_t scratch_for_current_device(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  *out = p;
  return QSA_OK;
}

}  // namespace

extern "C" qsa_status_t qsa_sparse_decode_noalloc(
    const qsa_geom_t* geom, const void* q_bf16, const uint8_t* k_pool, const uint8_t* k_sf,
    const uint8_t* v_pool, const uint8_t* v_sf, float k_scale, float v_scale, float sm_scale,
    const int32_t* page_table, const int32_t* seqlens, const int32_t* sel, int k,
    void* out_bf16, float* lse, cudaStream_t stream) {
  // Argument checks mirror qsa_sparse_decode's; the workspace size check is
  // replaced by the fit against the built-in array.
  if (!geom) return QSA_ERR_INVALID_ARG;
  const size_t auto_bytes = qsa_sparse_decode_workspace_bytes(geom, k);
  if (auto_bytes == 0) {
    // Invalid or unsupported geometry / k: let the regular entry point report
    // which, without launching (its workspace check fails first otherwise).
    return qsa_sparse_decode_ex(geom, q_bf16, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale,
                                sm_scale, page_table, seqlens, sel, k, out_bf16, lse, nullptr,
                                0, 0, stream);
  }
  if (!q_bf16 || !k_pool || !k_sf || !v_pool || !v_sf || !page_table || !seqlens || !sel ||
      !out_bf16 || !lse)
    return QSA_ERR_INVALID_ARG;
  qsa::Geom g;
  g.B = geom->batch; g.R = geom->rows_per_req; g.Hq = geom->num_q_heads;
  g.Hkv = geom->num_kv_heads; g.D = geom->head_dim; g.Di = geom->index_dim;
  g.P = geom->page_size; g.MB = geom->max_blocks; g.NP = geom->num_pages;
  // Largest split count (at most the automatic one) whose scratch fits.
  qsa::DecodePlan plan = qsa::plan_sparse_decode(g, k, 0);
  while (plan.ws_bytes > kNoAllocBytes && plan.splits > 1)
    plan = qsa::plan_sparse_decode(g, k, plan.splits - 1);
  if (plan.ws_bytes > kNoAllocBytes) return QSA_ERR_WORKSPACE;   // too large for the array

  void* scratch = nullptr;
  qsa_status_t st = scratch_for_current_device(&scratch);
  if (st != QSA_OK) return st;
  return qsa_sparse_decode_ex(geom, q_bf16, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale,
                              sm_scale, page_table, seqlens, sel, k, out_bf16, lse, scratch,
                              kNoAllocBytes, plan.splits, stream);
}

extern "C" qsa_status_t qsa_sparse_decode_noalloc_status(int* device_code, cudaStream_t stream) {
  if (!device_code) return QSA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  qsa_status_t st = scratch_for_current_device(&scratch);
  if (st != QSA_OK) return st;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, scratch, sizeof(int), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, sizeof(int), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  *device_code = v;
  return v == 0 ? QSA_OK : QSA_ERR_DEVICE_TIMEOUT;
}
