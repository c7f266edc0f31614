// qsa_store_tokens.cu -- decode prologue: the step's new tokens into the NVFP4
// K/V pages and the index-key pool.
//
// TensorRT-LLM PR #20937 ("GB300 perf work on
// qwen3_8_flash_next_nvfp4__sm_103__tp1"), What changes (NVFP4 sparse GQA
// decode): a decode prologue over the NVFP4 KV cache that also serves verify
// steps; Walkthrough, changes table: NVFP4 storage in the decode prologue.
// PR #20276 ("Qwen3.8-Flash-Next NVFP4 target"), Features table: uint8 e2m1
// pages with e4m3 block scales; the QSA index plane uses the same page index.
//
// Row j of request b is the token at position pos = L_b - R + j; it goes to
// block pos / P, slot pos % P of page page_table[b][pos / P] (skipped when
// pos < 0, pos >= MB*P or the page is invalid).  Each 16-element block of a
// K or V row (one KV head) is quantised with the per-tensor scale s:
//   a   = max |x| over the block          (x: the bf16 value, exact in fp32)
//   sf  = e4m3_rne_satfinite((a / 6) / s)
//   c_i = e2m1_rne_satfinite(x_i / (e4m3(sf) * s)), all zero when e4m3(sf)*s
//         is zero; a code whose magnitude rounds to zero is stored as +0
// with every division and product an IEEE fp32 operation in that order.
// The row's int8 index key is copied into the index pool at the same slot.
//
// One warp per (row, KV head, K|V): lane l holds the E = D/32 elements
// E*l..E*l+E-1 (4 at head_dim 128, 8 at 256), so the 16/E lanes of a
// 16-element block reduce its maximum with shuffles and each lane writes E/2
// code bytes; the first lane of block g writes its scale byte.
#include "qsa_common.cuh"

namespace qsa {
namespace {

constexpr int kWarpsPerCta = 8;
// Bounds-check code (reported by bounds-checked builds only): pool row out of range.
[[maybe_unused]] constexpr int kChkRow = 0x501;

__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(lo), "f"(hi));
  return r;   // low nibble: lo, high nibble: hi
}

__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(x));
  return r & 0xFFu;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t h2 = e4m3x2_to_f16x2(b & 0xFFu);
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// A nibble whose magnitude bits are zero is stored as +0.
__device__ __forceinline__ uint32_t canon_zero(uint32_t byte) {
  if ((byte & 0x07u) == 0) byte &= 0xF0u;
  if ((byte & 0x70u) == 0) byte &= 0x0Fu;
  return byte;
}

template <int D>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
store_tokens_kernel(Geom g, const __nv_bfloat16* __restrict__ k_new,
                    const __nv_bfloat16* __restrict__ v_new, const int8_t* __restrict__ ik_new,
                    float k_scale, float v_scale, const int32_t* __restrict__ page_table,
                    const int32_t* __restrict__ seqlens, uint8_t* __restrict__ k_pool,
                    uint8_t* __restrict__ k_sf, uint8_t* __restrict__ v_pool,
                    uint8_t* __restrict__ v_sf, int8_t* __restrict__ ik_pool) {
  const int lane = threadIdx.x & 31;
  // (row, KV head, K|V) of this warp
  const long long item = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const long long T = (long long)g.B * g.R;
  pdl_wait();   // earlier kernels of the stream may still read these pages
  pdl_trigger();
  if (item >= T * g.Hkv * 2) return;
  const int is_v = (int)(item & 1);
  const int kvh = (int)((item >> 1) % g.Hkv);
  const int r = (int)((item >> 1) / g.Hkv);
  const int b = r / g.R, j = r % g.R;
  const long long pos = (long long)seqlens[b] - g.R + j;
  if (pos < 0 || pos >= (long long)g.MB * g.P) return;
  const int beta = (int)(pos / g.P), slot = (int)(pos % g.P);
  const int page = page_table[(size_t)b * g.MB + beta];
  if (page < 0 || page >= g.NP) return;

  constexpr int E = D / 32;        // elements per lane
  constexpr int LPB = 16 / E;      // lanes per 16-element block
  const __nv_bfloat16* src = (is_v ? v_new : k_new) + ((size_t)r * g.Hkv + kvh) * D;
  const float s = is_v ? v_scale : k_scale;
  float x[E];
#pragma unroll
  for (int u = 0; u < E / 4; ++u) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src + E * lane + 4 * u);
    const __nv_bfloat162 p01 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 p23 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    x[4 * u + 0] = __low2float(p01); x[4 * u + 1] = __high2float(p01);
    x[4 * u + 2] = __low2float(p23); x[4 * u + 3] = __high2float(p23);
  }
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) a = fmaxf(a, fabsf(x[i]));
#pragma unroll
  for (int o = 1; o < LPB; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const uint32_t sf = f32_to_e4m3(__fdiv_rn(__fdiv_rn(a, 6.0f), s));
  const float den = __fmul_rn(e4m3_to_f32(sf), s);
  uint32_t codes = 0;   // E/2 code bytes, element 2i in the low nibble of byte i
  if (den != 0.f) {
#pragma unroll
    for (int i = 0; i < E / 2; ++i)
      codes |= canon_zero(f32x2_to_e2m1x2(__fdiv_rn(x[2 * i], den),
                                          __fdiv_rn(x[2 * i + 1], den))) << (8 * i);
  }
  const size_t row = ((size_t)page * g.Hkv + kvh) * g.P + slot;   // token row in the pool
  if (!QSA_IN_BOUNDS(b < g.B && slot >= 0 && slot < g.P && row < (size_t)g.NP * g.Hkv * g.P,
                     kChkRow))
    return;
  uint8_t* pool = is_v ? v_pool : k_pool;
  uint8_t* sfp = is_v ? v_sf : k_sf;
  if constexpr (E == 4)
    *reinterpret_cast<uint16_t*>(pool + row * (D / 2) + 2 * lane) = (uint16_t)codes;
  else
    *reinterpret_cast<uint32_t*>(pool + row * (D / 2) + 4 * lane) = codes;
  if (lane % LPB == 0) sfp[row * (D / 16) + lane / LPB] = (uint8_t)sf;
  // The index key: one warp per row (K side of KV head 0), 16 lanes x 4 B.
  if (!is_v && kvh == 0 && lane < kIndexDim / 4) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(ik_new + (size_t)r * kIndexDim + 4 * lane);
    *reinterpret_cast<uint32_t*>(ik_pool + ((size_t)page * g.P + slot) * kIndexDim + 4 * lane) = w;
  }
}

}  // namespace

cudaError_t launch_store_tokens(const Geom& g, const void* k_new, const void* v_new,
                                const int8_t* ik_new, float k_scale, float v_scale,
                                const int32_t* page_table, const int32_t* seqlens,
                                uint8_t* k_pool, uint8_t* k_sf, uint8_t* v_pool, uint8_t* v_sf,
                                int8_t* ik_pool, bool pdl, cudaStream_t stream) {
  const long long items = (long long)g.B * g.R * g.Hkv * 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((items + kWarpsPerCta - 1) / kWarpsPerCta));
  cfg.blockDim = dim3(kWarpsPerCta * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  auto* kern = g.D == 256 ? store_tokens_kernel<256> : store_tokens_kernel<128>;
  return cudaLaunchKernelEx(&cfg, kern, g, reinterpret_cast<const __nv_bfloat16*>(k_new),
                            reinterpret_cast<const __nv_bfloat16*>(v_new), ik_new, k_scale,
                            v_scale, page_table, seqlens, k_pool, k_sf, v_pool, v_sf, ik_pool);
}

}  // namespace qsa

QSA_BOUNDS_READER(bounds_word_store)
