// qsa_common.cuh -- device helpers shared by the QSA kernels (sm_103a only):
// inline-PTX wrappers for mbarriers, bulk (TMA) copies, NVFP4 element
// conversion, legacy warp MMA and the 8x8 fragment transpose, plus the
// internal launch interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qsa.h"

namespace qsa {

constexpr int kIndexDim = 64;
constexpr int kMaxRows = 8;           // rows per request (1 + drafts)
constexpr int kMaxContextRows = 4096; // rows per request of a context (prefill) row group
constexpr int kMaxQHeads = 256;
constexpr int kMaxK = 1024;
constexpr int kMaxUnion = 2048;       // R * k bound for the decode union
constexpr int kMaxBlocks = 32768;     // page-table width bound
constexpr int kSentinel = (int)0x80000000;

// Device status codes written to the workspace status word.
constexpr int kStatusWaitTimeout = 1;

// Visible tokens of row j of a request with L cached tokens.
__host__ __device__ __forceinline__ int visible_tokens(int L, int R, int j, int cap) {
  long long n = (long long)L - R + 1 + j;
  if (n < 0) n = 0;
  if (n > cap) n = cap;
  return (int)n;
}

// ---------------------------------------------------------------------------
// Bounds-checked builds.  Built with QSA_DEBUG_BOUNDS, every kernel checks the
// indices it derives from data (page ids, token offsets, list and record
// slots, output rows) before the access: a failed check records its code in
// the translation unit's bounds word (the first failure wins) and the access
// is skipped -- never a trap.  QSA_IN_BOUNDS(cond, code) is an invariant the
// code relies on (plain `true` in normal builds, cond not evaluated);
// QSA_GUARD(cond, code) is a test that normal builds also make, and that
// bounds-checked builds also report.
// ---------------------------------------------------------------------------
#ifdef QSA_DEBUG_BOUNDS
static __device__ int qsa_bounds_word = 0;
__device__ __forceinline__ bool qsa_bounds_fail(int code) {
  atomicCAS(&qsa_bounds_word, 0, code);
  return false;
}
#define QSA_IN_BOUNDS(cond, code) ((cond) ? true : ::qsa::qsa_bounds_fail(code))
#define QSA_GUARD(cond, code) ((cond) ? true : ::qsa::qsa_bounds_fail(code))
// Defines `int fn()` reading and clearing this translation unit's word.
#define QSA_BOUNDS_READER(fn)                                                    \
  namespace qsa {                                                                \
  int fn() {                                                                     \
    int v = 0, z = 0;                                                            \
    if (cudaMemcpyFromSymbol(&v, qsa_bounds_word, sizeof(int)) != cudaSuccess)   \
      v = -1;                                                                    \
    else if (cudaMemcpyToSymbol(qsa_bounds_word, &z, sizeof(int)) != cudaSuccess) \
      v = -1;                                                                    \
    cudaGetLastError();                                                          \
    return v;                                                                    \
  }                                                                              \
  }
#else
#define QSA_IN_BOUNDS(cond, code) true
#define QSA_GUARD(cond, code) (cond)
#define QSA_BOUNDS_READER(fn)
#endif

// ---------------------------------------------------------------------------
// mbarrier + bulk copy (TMA engine, non-tensor form)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// One non-blocking probe of phase `parity`; true when that phase completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// One probe of phase `parity` that never suspends the thread.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Contiguous global -> shared copy on the TMA engine; completion is signalled
// as transaction bytes on `bar`.  dst, src and bytes must be 16-byte aligned.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// NVFP4 element conversion
// ---------------------------------------------------------------------------

// Two e4m3 bytes (low byte -> low half) to two fp16 values.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(two_bytes));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Selects bytes of {b:a} (8 bytes) into a 32-bit word per `sel`.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// ---------------------------------------------------------------------------
// Warp-level MMA and fragment transpose
// ---------------------------------------------------------------------------

// D = A(16x16, row) * B(16x8, col) + D, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4],
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transposes an 8x8 16-bit matrix held one 32-bit pair per lane (lane holds
// row lane/4, columns 2*(lane%4) and 2*(lane%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------

// Waits until the preceding kernel in the stream has completed (or triggered)
// and its memory is visible; a no-op when launched without the PDL attribute.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allows the next kernel in the stream to begin launching.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace qsa

// ---------------------------------------------------------------------------
// Internal launch interface (host side), implemented by each kernel file.
// ---------------------------------------------------------------------------
namespace qsa {

struct Geom {
  int B, R, Hq, Hkv, D, Di, P, MB, NP;
};

size_t rollback_row_bytes(int hkv, int d);
cudaError_t launch_rollback(const Geom& g, bool restore, const int32_t* page_table,
                            const int32_t* seqlens, const int32_t* rejected, uint8_t* k_pool,
                            uint8_t* k_sf, uint8_t* v_pool, uint8_t* v_sf, int8_t* ik_pool,
                            uint8_t* saved, bool pdl, cudaStream_t stream);
cudaError_t launch_store_tokens(const Geom& g, const void* k_new, const void* v_new,
                                const int8_t* ik_new, float k_scale, float v_scale,
                                const int32_t* page_table, const int32_t* seqlens,
                                uint8_t* k_pool, uint8_t* k_sf, uint8_t* v_pool, uint8_t* v_sf,
                                int8_t* ik_pool, bool pdl, cudaStream_t stream);
cudaError_t launch_index_scores(const Geom& g, const int8_t* iq, const int8_t* ik_pool,
                                const int32_t* page_table, const int32_t* seqlens,
                                int32_t* scores, bool pdl, cudaStream_t stream);

cudaError_t launch_select_topk(const Geom& g, const int32_t* scores, const int32_t* seqlens,
                               int k, int window, int32_t* sel, int32_t* nsel, bool pdl,
                               cudaStream_t stream);

struct DecodePlan {
  int splits;        // KV splits per (request, KV head, query group)
  int qgroups;       // query-column groups per (request, KV head)
  int cols;          // query columns per (request, KV head) = G * R
  size_t ws_bytes;   // workspace bytes
};

DecodePlan plan_sparse_decode(const Geom& g, int k, int num_splits);
bool decode_can_fuse_select(const Geom& g);

#ifdef QSA_DEBUG_BOUNDS
// Each file's bounds word, read and cleared (0 = no failed check).
int bounds_word_attend();
int bounds_word_decode();
int bounds_word_index();
int bounds_word_select();
int bounds_word_store();
int bounds_word_rollback();
int bounds_word_prefill();
#endif

// Bound of the attention kernels' waits for their chunk copies, in ns
// (qsa_debug_set_wait_ns; 2 s unless a diagnostic changed it).
unsigned long long wait_limit_ns();

// head_dim 128 attention with one dequantisation per chunk for all of a
// request's query columns (qsa_attend.cu).
bool attend_supports(const Geom& g);
DecodePlan plan_attend(const Geom& g, int k, int num_splits);
cudaError_t launch_attend(const Geom& g, const DecodePlan& plan, const void* q,
                          const uint8_t* k_pool, const uint8_t* k_sf, const uint8_t* v_pool,
                          const uint8_t* v_sf, float k_scale, float v_scale, float sm_scale,
                          const int32_t* page_table, const int32_t* seqlens, const int32_t* sel,
                          int k, void* out, float* lse, void* workspace, bool pdl,
                          cudaStream_t stream);

// Context row groups (qsa_sparse_prefill): rows per 128-vector tile, dynamic
// shared memory of a CTA, and the launch.
int prefill_rows_per_tile(const Geom& g);
size_t prefill_smem_bytes(const Geom& g, int k);
cudaError_t launch_sparse_prefill(const Geom& g, const void* q, const uint8_t* k_pool,
                                  const uint8_t* k_sf, const uint8_t* v_pool, const uint8_t* v_sf,
                                  float k_scale, float v_scale, float sm_scale,
                                  const int32_t* page_table, const int32_t* seqlens,
                                  const int32_t* sel, int k, void* out, float* lse,
                                  int* status, cudaStream_t stream);

cudaError_t launch_sparse_decode(const Geom& g, const DecodePlan& plan, const void* q,
                                 const uint8_t* k_pool, const uint8_t* k_sf,
                                 const uint8_t* v_pool, const uint8_t* v_sf, float k_scale,
                                 float v_scale, float sm_scale, const int32_t* page_table,
                                 const int32_t* seqlens, const int32_t* sel, int k,
                                 void* out, float* lse, void* workspace, bool pdl,
                                 cudaStream_t stream,
                                 const int32_t* scores = nullptr, int window = 0,
                                 int32_t* sel_out = nullptr, int32_t* nsel_out = nullptr);

}  // namespace qsa
