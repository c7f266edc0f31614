// qsa_rollback.cu -- speculative rollback of the cache planes for rejected
// draft rows: gather the slots a verify step is about to overwrite, restore
// them for the rows the step rejects.
//
// TensorRT-LLM PR #20937 ("GB300 perf work on
// qwen3_8_flash_next_nvfp4__sm_103__tp1"), What changes (Rollback and PLE):
// batched rollback of the QSA index planes; Per-File QA: rollback
// gather/restore of the QSA planes, state restoration; review of the
// rollback-planes test: rejected rows get their old values back and kept rows
// stay untouched.
//
// Row j of request b owns the slot at position L_b - R + j (block / P, slot
// % P of its page); rows whose position is negative, at or past MB*P, or
// whose page is invalid own no slot and are skipped.  A row's saved state is
// rollback_row_bytes(Hkv, D) contiguous bytes:
//   for each KV head: K codes (D/2) | K scales (D/16) | V codes (D/2) |
//   V scales (D/16)
//   then the index key (64)
// One warp per (row, KV head) moves its 9D/8 bytes as 9D/32 words; the
// KV-head-0 warp also moves the 64-byte index key.
#include "qsa_common.cuh"

namespace qsa {
namespace {

// Bounds-check code (reported by bounds-checked builds only): pool row out of range.
[[maybe_unused]] constexpr int kChkRow = 0x601;
constexpr int kWarpsPerCta = 8;
constexpr int kIkWords = kIndexDim / 4;                              // 16

// Words of one (row, KV head) state: K codes, K scales, V codes, V scales.
__host__ __device__ __forceinline__ int kv_words(int d) { return 2 * (d / 8 + d / 64); }

// Word w of the (row, KV head) state: its address in the pools (cw = D/8 code
// words, sw = D/64 scale words per pool row).
__device__ __forceinline__ uint32_t* pool_word(int w, int cw, int sw, size_t row, uint8_t* k_pool,
                                               uint8_t* k_sf, uint8_t* v_pool, uint8_t* v_sf) {
  if (w < cw) return reinterpret_cast<uint32_t*>(k_pool + row * 4 * cw) + w;
  w -= cw;
  if (w < sw) return reinterpret_cast<uint32_t*>(k_sf + row * 4 * sw) + w;
  w -= sw;
  if (w < cw) return reinterpret_cast<uint32_t*>(v_pool + row * 4 * cw) + w;
  w -= cw;
  return reinterpret_cast<uint32_t*>(v_sf + row * 4 * sw) + w;
}

template <bool RESTORE>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
rollback_kernel(Geom g, const int32_t* __restrict__ page_table, const int32_t* __restrict__ seqlens,
                const int32_t* __restrict__ rejected, uint8_t* k_pool, uint8_t* k_sf,
                uint8_t* v_pool, uint8_t* v_sf, int8_t* ik_pool, uint8_t* saved) {
  const int lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  pdl_wait();
  pdl_trigger();
  if (item >= (long long)g.B * g.R * g.Hkv) return;
  const int kvh = (int)(item % g.Hkv);
  const int r = (int)(item / g.Hkv);
  if (RESTORE && rejected[r] == 0) return;
  const int b = r / g.R, j = r % g.R;
  const long long pos = (long long)seqlens[b] - g.R + j;
  if (pos < 0 || pos >= (long long)g.MB * g.P) return;
  const int page = page_table[(size_t)b * g.MB + pos / g.P];
  if (page < 0 || page >= g.NP) return;
  const int slot = (int)(pos % g.P);
  const size_t row = ((size_t)page * g.Hkv + kvh) * g.P + slot;
  if (!QSA_IN_BOUNDS(b < g.B && slot >= 0 && slot < g.P && row < (size_t)g.NP * g.Hkv * g.P,
                     kChkRow))
    return;
  const int kw = kv_words(g.D), cw = g.D / 8, sw = g.D / 64;
  const size_t row_bytes = (size_t)g.Hkv * kw * 4 + kIkWords * 4;
  uint32_t* sv = reinterpret_cast<uint32_t*>(saved + (size_t)r * row_bytes) + kvh * kw;
  for (int w = lane; w < kw; w += 32) {
    uint32_t* p = pool_word(w, cw, sw, row, k_pool, k_sf, v_pool, v_sf);
    if (RESTORE) *p = sv[w]; else sv[w] = *p;
  }
  if (kvh == 0 && lane < kIkWords) {
    uint32_t* p = reinterpret_cast<uint32_t*>(ik_pool + ((size_t)page * g.P + slot) * kIndexDim) + lane;
    uint32_t* s = reinterpret_cast<uint32_t*>(saved + (size_t)r * row_bytes) + g.Hkv * kw + lane;
    if (RESTORE) *p = *s; else *s = *p;
  }
}

}  // namespace

size_t rollback_row_bytes(int hkv, int d) { return (size_t)hkv * kv_words(d) * 4 + kIkWords * 4; }

cudaError_t launch_rollback(const Geom& g, bool restore, const int32_t* page_table,
                            const int32_t* seqlens, const int32_t* rejected, uint8_t* k_pool,
                            uint8_t* k_sf, uint8_t* v_pool, uint8_t* v_sf, int8_t* ik_pool,
                            uint8_t* saved, bool pdl, cudaStream_t stream) {
  const long long items = (long long)g.B * g.R * g.Hkv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((items + kWarpsPerCta - 1) / kWarpsPerCta));
  cfg.blockDim = dim3(kWarpsPerCta * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (restore)
    return cudaLaunchKernelEx(&cfg, rollback_kernel<true>, g, page_table, seqlens, rejected,
                              k_pool, k_sf, v_pool, v_sf, ik_pool, saved);
  return cudaLaunchKernelEx(&cfg, rollback_kernel<false>, g, page_table, seqlens, rejected, k_pool,
                            k_sf, v_pool, v_sf, ik_pool, saved);
}

}  // namespace qsa

QSA_BOUNDS_READER(bounds_word_rollback)
