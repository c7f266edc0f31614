// qsa_sparse_prefill.cu -- context (prefill) rows: row-tile sparse GQA on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// TensorRT-LLM PR #20276 ("Qwen3.8-Flash-Next NVFP4 target"), Performance /
// what runs on the fast paths: context and mixed steps run a row-tile sparse
// GQA on tcgen05 whose K/V tiles are read once per group of rows of one
// request; Known limitations: the context rows read NVFP4 pages dequantised
// to bf16 through the row-tile pass.  PR #20937 ("GB300 perf work on
// qwen3_8_flash_next_nvfp4__sm_103__tp1"), What changes: the NVFP4 page
// conversion and the row-tile planning and scheduling.
//
// One CTA = (request b, KV head g, row tile): TR = floor(128 / G) consecutive
// rows of the request, whose TR*G query vectors (row j, head h) are the 128
// rows of the MMA tile (padding rows are zero and never stored).  The tile
// visits the union of its rows' selected blocks in 64-token chunks; every
// query vector takes the logits of a chunk only if its row selected the
// block and only for tokens it sees (causal, n_j = L - R + 1 + j).
//
// Per chunk (one pipeline step; the NVFP4 bytes of the next chunk are in
// flight on the bulk-copy engine meanwhile):
//   1. dequantise K (64 tokens x 128 dims) and V^T (128 dims x 64 tokens)
//      from the staged NVFP4 bytes into fp16 tiles in shared memory, K-major
//      with the 128-byte swizzle; e2m1 x e4m3 is exact in fp16 and the
//      per-tensor scales are applied in fp32 outside the MMAs, so the tiles
//      hold the cache's values exactly (the page conversion, on chip);
//   2. S = Q . K^T     tcgen05.mma kind::f16, M = 128, N = 64, K = 128,
//                      fp32 accumulator in tensor memory;
//   3. each thread owns one query vector (one tensor-memory lane): masks,
//      log2-domain online softmax with a lazy rescale (the running base only
//      moves when the maximum grows by more than 2^8; O and l are then
//      rescaled), P = exp2(z - base) as fp16 into a swizzled P tile;
//   4. O += P . V      tcgen05.mma kind::f16, M = 128, N = 128, K = 64.
// After the last chunk every thread reads its O row from tensor memory,
// divides by l, applies the V tensor scale and writes out (bf16) and lse.
//
// Queries enter as fp16 pre-scaled by a power of two per vector (|q|max in
// [256, 512)); the scale is undone in fp32 with the logit scale.  Every wait
// is bounded (2 s); a wait that gives up records a status word in the
// workspace, lets the copies and MMAs in flight finish and frees tensor memory.
#include "qsa_common.cuh"

namespace qsa {
namespace {

// Bounds-check codes (reported by bounds-checked builds only).
[[maybe_unused]] constexpr int kChkUnion = 0x701;   // union slot past its capacity
[[maybe_unused]] constexpr int kChkChunk = 0x702;   // chunk: union slot or page id out of range
[[maybe_unused]] constexpr int kChkOut = 0x703;     // output row out of range
constexpr int kThreads = 128;           // four warps: one thread per tile row
constexpr int kStage = 9216;            // NVFP4 bytes of one chunk (8192 K and V values)

// Per head dim D: a chunk is 8192 / D tokens (64 at D = 128, 32 at D = 256).
// Every fp16 tile is K-major in 64-element (128-byte) column blocks of rows.
template <int D>
struct PT {
  static_assert(D == 128 || D == 256, "head_dim 128 or 256");
  static constexpr int kTok = 8192 / D;           // tokens per chunk
  static constexpr int kQBytes = 128 * D * 2;     // Q: D/64 blocks of 128 rows x 128 B
  static constexpr int kKBlk = kTok * 128;        // one 64-dim block of the K tile
  static constexpr int kKBytes = (D / 64) * kKBlk;
  static constexpr int kVBytes = D * 128;         // V^T: D rows of 64 tokens (zero-padded)
  static constexpr int kPBytes = 128 * 128;       // P: 128 rows of 64 tokens (zero-padded)
  static constexpr uint32_t kTmemCols = D == 128 ? 256 : 512;
  static constexpr uint32_t kOCol = D == 128 ? 64 : 256;   // S at column 0, O here
};
static_assert(2 * PT<128>::kTok * 128 / 2 + 2 * PT<128>::kTok * 128 / 16 == kStage, "stage");
static_assert(2 * PT<256>::kTok * 256 / 2 + 2 * PT<256>::kTok * 256 / 16 == kStage, "stage");
constexpr unsigned long long kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleGap = 8.f;      // log2 units the base may trail the maximum

struct Params {
  Geom g;
  const __nv_bfloat16* q;
  const uint8_t* k_pool;
  const uint8_t* k_sf;
  const uint8_t* v_pool;
  const uint8_t* v_sf;
  float k_scale, v_scale, sm_scale;
  const int32_t* page_table;
  const int32_t* seqlens;
  const int32_t* sel;
  int k;
  int tr;                 // rows per tile
  int ucap;               // union capacity (blocks)
  __nv_bfloat16* out;
  float* lse;
  int* status;
};

// Byte offset of (row r, element e) of a K-major fp16 tile whose rows are 64
// elements (128 B), in 8-row atoms of 1024 B with the 128-byte swizzle (the
// 16-byte chunk index is xor-ed with the row within the atom).
__host__ __device__ __forceinline__ int sw128(int r, int chunk16) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((chunk16 ^ (r & 7)) << 4);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 B apart (the leading offset is unused in this layout).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;                 // leading byte offset 16 B (unused)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1 << 46;                 // descriptor version
  d |= (uint64_t)2 << 61;                 // 128-byte swizzle
  return d;
}

// The same for an MN-major operand: rows of 64 N-elements (128 B, swizzled)
// along K in 8-row groups 1024 B apart; consecutive 64-element groups along
// N `lbo` bytes apart.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t lbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;   // leading byte offset: along N
  d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset: along K
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t f16_idesc(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
constexpr uint32_t kIdescBMn = 1u << 16;   // instruction descriptor: B is MN-major

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = now_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (now_ns() - t0 > kWaitNs) return false;
  }
}

// A CTA-wide bounded wait on one mbarrier phase: every thread polls, then
// the CTA agrees on the outcome.  True when the wait gave up, in every thread.
__device__ __forceinline__ bool cta_wait_failed(uint64_t* bar, uint32_t parity) {
  return __syncthreads_or(!wait_bounded(bar, parity));
}

// 2^x, hardware approximation (flushes subnormal results to zero).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// tcgen05.mma with A (M x 16, fp16) in tensor memory reads lane m as row m,
// column j as the elements 2j (low half) and 2j + 1.
// The same MMAs issued by one elected lane of a converged warp (warp-uniform
// operands), and their commit from that lane.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ void mma_f16_elect(uint32_t d_tmem, uint64_t a, uint64_t b,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_f16_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

// 16 words into 16 consecutive columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Eight e2m1 codes (one word, element 2i in the low nibble of byte i) times
// one fp16 scale pair -> four fp16 pairs.
__device__ __forceinline__ uint4 dequant8(uint32_t w, uint32_t s2) {
  uint32_t o[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
  return make_uint4(hmul2_u32(o[0], s2), hmul2_u32(o[1], s2), hmul2_u32(o[2], s2),
                    hmul2_u32(o[3], s2));
}

__device__ __forceinline__ void ws_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Lower bound of beta in an ascending selection row padded with -1 (+inf).
__device__ __forceinline__ bool row_holds(const int32_t* row, int k, int beta) {
  int lo = 0, hi = k;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int x = row[mid] < 0 ? 0x7FFFFFFF : row[mid];
    if (x < beta) lo = mid + 1; else hi = mid;
  }
  return lo < k && row[lo] == beta;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
sparse_prefill_kernel(Params p) {
  using T = PT<D>;
  constexpr int kTok = T::kTok;
  const Geom& g = p.g;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = g.Hq / g.Hkv;
  const int TR = p.tr;
  const int tile = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int r0 = tile * TR;                   // first row of the tile
  const int rows = min(TR, g.R - r0);
  const int k = p.k;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The swizzle atoms need 1024-byte alignment (one spare KB is allocated).
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                           // 32 / 64 KB
  uint8_t* sK = sQ + T::kQBytes;                // 16 KB
  uint8_t* sV = sK + T::kKBytes;                // 16 / 32 KB
  uint8_t* sP = sV + T::kVBytes;                // 16 KB
  uint8_t* sStage = sP + T::kPBytes;            // 2 x 9216 B
  uint64_t* full = reinterpret_cast<uint64_t*>(sStage + 2 * kStage);
  uint64_t* barS = full + 2;                    // S = Q K^T complete
  uint64_t* barO = full + 3;                    // O += P V complete
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(full + 4);
  int* s_misc = reinterpret_cast<int*>(s_tmem + 1);            // [8]
  int32_t* s_sel = s_misc + 8;                                  // [TR][k]
  int32_t* s_union = s_sel + TR * k;                            // [ucap]
  int32_t* s_upage = s_union + p.ucap;                          // [ucap]
  uint32_t* s_bits = reinterpret_cast<uint32_t*>(s_upage + p.ucap);   // [ceil(MB/32)]
  const int nwords = (g.MB + 31) >> 5;

  // ---- barriers, tensor memory ---------------------------------------------
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(barS, 1);
    mbar_init(barO, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(s_tmem)),
                 "r"(T::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }

  // ---- this thread's query vector: Q row into the swizzled tile -------------
  const int jj = tid / G, hh = tid % G;
  const bool vec = jj < rows;                   // a real (row, head) vector
  const int j = r0 + jj;
  const int L = p.seqlens[b];
  const int cap = g.MB * g.P;
  const int nrow = vec ? visible_tokens(L, g.R, j, cap) : 0;
  float cq = 0.f;                               // logit scale, log2 domain
  {
    // Two passes over the row (L1/L2-resident the second time): the maximum,
    // then the scaled fp16 copy into 16-byte chunks of the swizzled tile.
    const size_t qrow = ((size_t)b * g.R + j) * g.Hq + (size_t)kvh * G + hh;
    const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow * D);
    float amax = 0.f;
    if (vec) {
#pragma unroll 4
      for (int i = 0; i < D / 8; ++i) {
        const uint4 r = src[i];
        const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          amax = fmaxf(amax, fabsf(__uint_as_float(w4[u] << 16)));
          amax = fmaxf(amax, fabsf(__uint_as_float(w4[u] & 0xFFFF0000u)));
        }
      }
    }
    const int ebits = (int)((__float_as_uint(amax) >> 23) & 0xFF);
    int sq = (amax > 0.f) ? 135 - ebits : 0;
    sq = sq > 126 ? 126 : (sq < -126 ? -126 : sq);
    const float up = __uint_as_float((uint32_t)(sq + 127) << 23);
    const float down = __uint_as_float((uint32_t)(127 - sq) << 23);
    cq = p.k_scale * p.sm_scale * kLog2e * down;
#pragma unroll 4
    for (int i = 0; i < D / 8; ++i) {
      uint4 h = make_uint4(0u, 0u, 0u, 0u);
      if (vec) {
        const uint4 r = src[i];
        const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
        uint32_t o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          o[u] = pack_half2(__uint_as_float(w4[u] << 16) * up,
                            __uint_as_float(w4[u] & 0xFFFF0000u) * up);
        h = make_uint4(o[0], o[1], o[2], o[3]);
      }
      // dims 8i..8i+7: column block i / 8, 16-byte chunk i % 8 of row tid
      *reinterpret_cast<uint4*>(sQ + (i >> 3) * 16384 + sw128(tid, i & 7)) = h;
    }
  }
  // Tokens past a chunk (D = 256: 32 of the 64 token slots of the P and V^T
  // tiles) stay zero: the tiles are cleared once and those slots never written.
  if (kTok < 64) {
    for (int i = tid; i < (T::kVBytes + T::kPBytes) / 16; i += kThreads)
      reinterpret_cast<uint4*>(sV)[i] = make_uint4(0u, 0u, 0u, 0u);
  }

  // ---- the tile's rows' selections and their union ----------------------------
  for (int i = tid; i < TR * k; i += kThreads) {
    const int jr = i / k;
    int v = -1;
    if (jr < rows) {
      v = p.sel[((size_t)b * g.R + r0 + jr) * k + (i - jr * k)];
      if (v < 0 || v >= g.MB) v = -1;
    }
    s_sel[i] = v;
  }
  for (int i = tid; i < nwords; i += kThreads) s_bits[i] = 0u;
  __syncthreads();
  for (int i = tid; i < rows * k; i += kThreads) {
    const int v = s_sel[i];
    if (v >= 0) atomicOr(&s_bits[v >> 5], 1u << (v & 31));
  }
  __syncthreads();
  {
    // Blocks with a valid page, ascending: thread t scans words [t*per, ...).
    const int per = (nwords + kThreads - 1) / kThreads;
    const int w0 = min(nwords, tid * per), w1 = min(nwords, w0 + per);
    const int32_t* pt = p.page_table + (size_t)b * g.MB;
    int cnt = 0;
    for (int w = w0; w < w1; ++w) {
      uint32_t m = s_bits[w];
      while (m) {
        const int beta = (w << 5) + __ffs(m) - 1;
        m &= m - 1;
        const int pg = pt[beta];
        if (pg >= 0 && pg < g.NP) ++cnt; else s_bits[w] &= ~(1u << (beta & 31));
      }
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if ((tid & 31) >= o) x += y;
    }
    if ((tid & 31) == 31) s_misc[warp] = x;
    __syncthreads();
    int pos = x - cnt;
    for (int w = 0; w < warp; ++w) pos += s_misc[w];
    for (int w = w0; w < w1; ++w) {
      uint32_t m = s_bits[w];
      while (m) {
        const int beta = (w << 5) + __ffs(m) - 1;
        m &= m - 1;
        if (QSA_IN_BOUNDS(pos < p.ucap, kChkUnion)) {
          s_union[pos] = beta;
          s_upage[pos] = pt[beta];
        }
        ++pos;
      }
    }
    if (tid == kThreads - 1) s_misc[4] = pos;
  }
  fence_proxy_async_smem();       // Q tile (generic stores) before the MMAs read it
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int U = s_misc[4];
  const int csh = (g.P == 2 * kTok) ? 1 : 0;    // chunks per block: 1 << csh
  const int C = U << csh;
  const int32_t* myrow = s_sel + jj * k;

  const uint64_t pol = policy_evict_first();
  // Chunk c's four bulk copies (K codes, V codes, K scales, V scales).
  auto issue = [&](int c) {
    uint8_t* dst = sStage + (c & 1) * kStage;
    const int u = c >> csh, sub = c & csh;
    if (!QSA_IN_BOUNDS(u < U && u < p.ucap && s_upage[u] >= 0 && s_upage[u] < g.NP, kChkChunk))
      return;
    const size_t row0 = ((size_t)s_upage[u] * g.Hkv + kvh) * g.P + (size_t)sub * kTok;
    mbar_arrive_expect_tx(&full[c & 1], kStage);
    bulk_g2s(dst, p.k_pool + row0 * (D / 2), kTok * D / 2, &full[c & 1], pol);
    bulk_g2s(dst + kTok * D / 2, p.v_pool + row0 * (D / 2), kTok * D / 2, &full[c & 1], pol);
    bulk_g2s(dst + kTok * D, p.k_sf + row0 * (D / 16), kTok * D / 16, &full[c & 1], pol);
    bulk_g2s(dst + kTok * D + kTok * D / 16, p.v_sf + row0 * (D / 16), kTok * D / 16,
             &full[c & 1], pol);
  };
  const uint32_t tS = tmem, tO = tmem + T::kOCol;
  const uint32_t lane_off = (uint32_t)(32 * warp) << 16;

  // ---- stage helpers ---------------------------------------------------------
  // K rows = tokens (two 64-dim halves), V^T rows = dims; 8 pieces per thread.
  auto dequant_k = [&](const uint8_t* st) {
    const uint8_t* kc = st;
    const uint8_t* ks = st + kTok * D;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int pc = tid + kThreads * i;      // (token, 8-dim group)
      const int t = pc / (D / 8), c8 = pc % (D / 8);
      const uint32_t w = *reinterpret_cast<const uint32_t*>(kc + t * (D / 2) + c8 * 4);
      const uint32_t s = e4m3x2_to_f16x2(ks[t * (D / 16) + (c8 >> 1)]);
      *reinterpret_cast<uint4*>(sK + (c8 >> 3) * T::kKBlk + sw128(t, c8 & 7)) =
          dequant8(w, prmt(s, 0, 0x1010));
    }
  };
  auto dequant_v = [&](const uint8_t* st) {
    const uint8_t* vc = st + kTok * D / 2;
    const uint8_t* vs = st + kTok * D + kTok * D / 16;
    // 8 tokens x 8 dims per thread.  D = 128: lane = dim group (16) +
    // half-warp bit, the two half-warps on neighbouring 8-token groups; the
    // upper half loads each token pair in swapped order, so that one load
    // instruction touches tokens of both parities (32 distinct banks: token
    // rows are 64 B apart).  D = 256: warp w takes dim groups 8w..8w+7, lane
    // bits 3-4 the 8-token group.
    const int lane = tid & 31;
    const int hw = D == 128 ? lane >> 4 : 0;
    const int c8 = D == 128 ? lane & 15 : 8 * warp + (lane & 7);
    const int tg = D == 128 ? 2 * warp + hw : lane >> 3;
    uint32_t X[8], sf[8];   // X[u]: token 8*tg + (u ^ hw)
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = 8 * tg + (u ^ hw);
      X[u] = *reinterpret_cast<const uint32_t*>(vc + t * (D / 2) + c8 * 4);
      sf[u] = vs[t * (D / 16) + (c8 >> 1)];
    }
    uint32_t rowv[8][4];   // [dim e][token pair]
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      const uint32_t x0 = hw ? X[2 * pr + 1] : X[2 * pr];        // token 8*tg + 2*pr
      const uint32_t x1 = hw ? X[2 * pr] : X[2 * pr + 1];        // token 8*tg + 2*pr + 1
      const uint32_t f0 = hw ? sf[2 * pr + 1] : sf[2 * pr];
      const uint32_t f1 = hw ? sf[2 * pr] : sf[2 * pr + 1];
      const uint32_t s2 = e4m3x2_to_f16x2(f0 | (f1 << 8));
      const uint32_t LO = (x0 & 0x0F0F0F0Fu) | ((x1 << 4) & 0xF0F0F0F0u);    // even dims
      const uint32_t HI = ((x0 >> 4) & 0x0F0F0F0Fu) | (x1 & 0xF0F0F0F0u);    // odd dims
      const uint4 el = dequant8(LO, s2), od = dequant8(HI, s2);
      rowv[0][pr] = el.x; rowv[2][pr] = el.y; rowv[4][pr] = el.z; rowv[6][pr] = el.w;
      rowv[1][pr] = od.x; rowv[3][pr] = od.y; rowv[5][pr] = od.z; rowv[7][pr] = od.w;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
      *reinterpret_cast<uint4*>(sV + sw128(8 * c8 + e, tg)) =
          make_uint4(rowv[e][0], rowv[e][1], rowv[e][2], rowv[e][3]);
  };
  // Generic-proxy shared-memory writes become visible to the tensor core and
  // every thread's tensor-memory accesses are ordered around the barrier.
  auto publish = [&]() {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  auto issue_s = [&]() {       // S = Q . K^T, then the S barrier
    const uint32_t id = f16_idesc(128, kTok);
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
#pragma unroll
      for (int ks2 = 0; ks2 < 4; ++ks2)
        mma_f16(tS, sw128_desc(smem_u32(sQ + h * 16384) + 32 * ks2),
                sw128_desc(smem_u32(sK + h * T::kKBlk) + 32 * ks2), id,
                (h | ks2) ? 1u : 0u);
    mma_commit(barS);
  };
  auto issue_o = [&](int c) {  // O += P . V (64 token slots), then the O barrier
    const uint32_t id = f16_idesc(128, D);
#pragma unroll
    for (int ks2 = 0; ks2 < 4; ++ks2)
      mma_f16(tO, sw128_desc(smem_u32(sP) + 32 * ks2), sw128_desc(smem_u32(sV) + 32 * ks2), id,
              (c | ks2) ? 1u : 0u);
    mma_commit(barO);
  };

  // ---- pipeline ----------------------------------------------------------------
  // Chunk c:  softmax(c) -> [O += P(c) V(c)  ||  dequantise K(c+1)]
  //           -> [S(c+1) = Q K(c+1)^T  ||  dequantise V(c+1) once O(c) is done]
  // The NVFP4 bytes of chunk c+2 are requested when chunk c's stage is free.
  float m_base = -INFINITY, l_run = 0.f;
  uint32_t phS = 0, phO = 0;
  bool dead = false;
  int issued = 0;
  if (tid == 0) {
    for (int c = 0; c < min(C, 2); ++c) issue(c);
  }
  issued = min(C, 2);
  if (C > 0) {
    if (cta_wait_failed(&full[0], 0)) {
      dead = true;
    } else {
      dequant_k(sStage);
      dequant_v(sStage);
      publish();
      if (tid == 0) issue_s();
    }
  }

  for (int c = 0; c < C && !dead; ++c) {
    if (cta_wait_failed(barS, phS & 1)) { dead = true; break; }   // S(c) and all before it
    ++phS;
    tc_fence_after();
    // Every thread is past V(c) (the barrier above), so chunk c's stage is
    // free: request chunk c + 2 now, a whole chunk ahead of its use.
    if (tid == 0 && c + 2 < C) {
      fence_proxy_async_smem();
      issue(c + 2);
      issued = c + 3;
    }

    // ---- softmax(c): masks, online softmax, P tile, O rescale ------------------
    const int ue = s_union[c >> csh];
    const int tok0 = ue * g.P + (c & csh) * kTok;
    const bool member = vec && tok0 < nrow && row_holds(myrow, k, ue);
    float z[kTok];
#pragma unroll
    for (int q4 = 0; q4 < kTok / 16; ++q4) {
      float v16[16];
      tmem_ld16(tS + lane_off + 16 * q4, v16);
#pragma unroll
      for (int i = 0; i < 16; ++i) z[16 * q4 + i] = v16[i];
    }
    tmem_wait_ld();
    float cmax = -INFINITY;   // log2 units
    if (member) {
      if (tok0 + kTok > nrow) {
#pragma unroll
        for (int i = 0; i < kTok; ++i)
          if (tok0 + i >= nrow) z[i] = -INFINITY;
      }
      float mx8[8];           // eight independent chains, then a tree
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = z[i];
#pragma unroll
      for (int i = 8; i < kTok; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], z[i]);
#pragma unroll
      for (int h = 4; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) mx8[i] = fmaxf(mx8[i], mx8[i + h]);
      cmax = mx8[0] * cq;     // cq > 0: the scale keeps the order
    }
    bool rescale = false;
    float alpha = 1.f;
    if (cmax != -INFINITY) {
      if (m_base == -INFINITY) {
        m_base = cmax;
      } else if (cmax > m_base + kRescaleGap) {
        alpha = exp2_approx(m_base - cmax);
        m_base = cmax;
        rescale = true;
      }
    }
    uint32_t pk[kTok / 2];
    if (member) {
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kTok / 2; ++i) {
        const float p0 = exp2_approx(fmaf(z[2 * i], cq, -m_base));
        const float p1 = exp2_approx(fmaf(z[2 * i + 1], cq, -m_base));
        ls4[i & 3] += p0 + p1;
        pk[i] = pack_half2(p0, p1);
      }
      l_run = l_run * alpha + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
    } else {
#pragma unroll
      for (int i = 0; i < kTok / 2; ++i) pk[i] = 0u;
    }
#pragma unroll
    for (int c16 = 0; c16 < kTok / 8; ++c16)
      *reinterpret_cast<uint4*>(sP + sw128(tid, c16)) =
          make_uint4(pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
    // O (complete: O(c-1) finished before V(c) was dequantised).  Tensor-memory
    // loads and stores are warp-wide: a warp rescales when any of its lanes
    // must (alpha = 1 for the others).
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int q8 = 0; q8 < D / 16; ++q8) {
        float o16[16];
        tmem_ld16(tO + lane_off + 16 * q8, o16);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) o16[i] *= alpha;
        tmem_st16(tO + lane_off + 16 * q8, o16);
      }
      tmem_wait_st();
    }
    publish();   // P(c), V(c), the rescaled O; S(c) has been read

    if (tid == 0) issue_o(c);
    if (c + 1 < C) {
      // K(c+1) while O(c) runs (S(c) is done, so sK is free).
      if (cta_wait_failed(&full[(c + 1) & 1], ((c + 1) >> 1) & 1)) { dead = true; break; }
      dequant_k(sStage + ((c + 1) & 1) * kStage);
      publish();
      if (tid == 0) issue_s();
      // V(c+1) once O(c) has read sV; S(c+1) runs meanwhile.
      if (cta_wait_failed(barO, phO & 1)) { dead = true; break; }
      ++phO;
      dequant_v(sStage + ((c + 1) & 1) * kStage);
    } else {
      if (cta_wait_failed(barO, phO & 1)) { dead = true; break; }
      ++phO;
    }
  }
  tc_fence_after();

  if (dead) {
    if (tid == 0) atomicExch(p.status, kStatusWaitTimeout);
    // Let this CTA's copies in flight land before the CTA's memory goes away.
    if (tid == 0)
      for (int c = max(0, issued - 2); c < issued; ++c) wait_bounded(&full[c & 1], (c >> 1) & 1);
  }

  // ---- epilogue: out = O / l * v_scale, lse -------------------------------------
  // (tensor-memory loads by every lane of every warp; O holds no value when no
  // chunk was visited, and rows without a token write zeros)
  if (!dead) {
    const size_t orow = ((size_t)b * g.R + j) * g.Hq + (size_t)kvh * G + hh;
    const bool out_ok = !vec || QSA_IN_BOUNDS(b < g.B && j < g.R && kvh * G + hh < g.Hq, kChkOut);
    uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D);
    const bool has = l_run > 0.f && C > 0;
    const float sc = has ? p.v_scale / l_run : 0.f;
#pragma unroll 4
    for (int q8 = 0; q8 < D / 16; ++q8) {
      float o16[16];
      if (C > 0) {
        tmem_ld16(tO + lane_off + 16 * q8, o16);
        tmem_wait_ld();
      }
      uint32_t h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        __nv_bfloat162 x = __floats2bfloat162_rn(has ? o16[2 * i] * sc : 0.f,
                                                 has ? o16[2 * i + 1] * sc : 0.f);
        h[i] = *reinterpret_cast<uint32_t*>(&x);
      }
      if (vec && out_ok) {
        dst[2 * q8] = make_uint4(h[0], h[1], h[2], h[3]);
        dst[2 * q8 + 1] = make_uint4(h[4], h[5], h[6], h[7]);
      }
    }
    if (vec && out_ok) p.lse[orow] = has ? (m_base + log2f(l_run)) * kLn2 : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(T::kTmemCols));
}

// ---------------------------------------------------------------------------
// Warp-specialised row tiles.  Per query tile four softmax warps own its 128
// tensor-memory lanes (queries, softmax, epilogue); two warps issue the MMAs
// (one per tile with two tiles; with one tile one issues S and the other O);
// ND warps dequantise the NVFP4 chunks into double-buffered fp16 K and V
// tiles in shared memory (both with token rows; with eight warps four convert
// K and four V), and one thread issues the bulk copies.  P goes from the softmax into tensor memory (double-buffered)
// and feeds O += P V as the A operand from there, with V as an MN-major B
// operand, so shared memory carries only the K and V operands.  S is
// double-buffered in tensor memory at head_dim 256 and single-buffered at
// head_dim 128 (two tiles' O fill half of it); the softmax releases its S
// buffer as soon as it has loaded S into registers.  For chunk c the softmax
// of c, the dequantisation of c + 1 and the MMAs S(c + 1) and O(c - 1) overlap.
// Hand-overs are mbarriers (all waits bounded):
//   full[z]      copy of a chunk into stage z landed         (1 arrival + bytes)
//   empty[z]     the dequant warps are done with stage z      (ND arrivals)
//   kready[x]    K tile x written                             (its converting threads)
//   vready[x]    V tile x written                             (its converting threads)
//   kfree[x]     every tile's S MMAs that read K tile x done  (commit)
//   vfree[x]     every tile's O MMAs that read V tile x done  (commit)
//   barS[t][y]   S of tile t into its buffer y complete       (commit)
//   sfree[t][y]  tile t's softmax has loaded S buffer y       (128 arrivals)
//   pready[t][x] P buffer x of tile t written, O rescaled     (128 arrivals)
//   barO[t][x]   O_t += P_t(x) V(x) complete                  (commit)
//   mdone[w]     every MMA of MMA warp w complete             (commit)
//   qbar         the CTA's query rows landed                  (1 arrival + bytes)
//   qready       Q in tensor memory (head_dim 256)            (128 arrivals)
// Chunk c uses stage z = c % 4 (phase c / 4), tile buffer x = c & 1 (phase
// c >> 1) and S buffer y = c % SB (phase c / SB), SB the S buffers per tile.
// Each tile has its own S, P and O hand-overs, so one tile's MMAs issue
// while the other tile's softmax runs.
// At head_dim 128 a CTA holds two query tiles (NTL = 2: eight softmax warps,
// 2 x TR consecutive rows) that share every dequantised chunk of the union of
// their rows' selections; at head_dim 256 one (two Q tiles would not fit).
// Tensor memory (512 columns): S buffers from column 0, then the P buffers
// (kTok / 2 columns each: two fp16 per column), at head_dim 256 Q at 128
// (D / 2 columns), O of tile t at 256 + t D.
constexpr int kWsStages = 4;   // NVFP4 chunk stages of the warp-specialised kernel
constexpr int kWsBars = 32;    // its mbarriers

// Words of a row's membership bitmap over the union (odd, so the rows of one
// warp fall on different banks).
__host__ __device__ __forceinline__ int ws_member_words(int ucap) {
  return ((ucap + 31) >> 5) | 1;
}

template <int D>
struct WT {
  using T = PT<D>;
  static constexpr int kNtl = D == 128 ? 2 : 1;       // query tiles per CTA
  static constexpr int kDeq = D == 128 ? 4 : 8;       // dequantisation warps (registers)
  static constexpr int kThreads = 128 * kNtl + 32 * kDeq + 96;   // softmax, dequant, 2 MMA, copy
  static constexpr int kSBuf = D == 128 ? 1 : 2;      // S buffers per tile
  static constexpr uint32_t kPBase = kNtl * kSBuf * T::kTok;   // P of (t, x) after S
  static constexpr uint32_t kOBase = 256;             // O of tile t at kOBase + t * D
  static constexpr uint32_t kTmemCols = 512;
  // At head_dim 256 (one tile) Q also lives in tensor memory, so the S MMAs
  // read only K from shared memory; at 128 two tiles' O leave no room.
  static constexpr bool kQTmem = D == 256;
  static constexpr uint32_t kQBase = 128;
  static_assert(!kQTmem || (kPBase + 2 * kNtl * T::kTok / 2 <= kQBase && kQBase + D / 2 <= kOBase),
                "tensor-memory columns for Q");
  static constexpr size_t kTiles = (size_t)kNtl * T::kQBytes + 4 * (size_t)T::kKBytes;   // Q, K, V
  static_assert(kPBase + 2 * kNtl * T::kTok / 2 <= kOBase, "tensor-memory columns");
};

template <int D>
__global__ void __launch_bounds__(WT<D>::kThreads, 1)
sparse_prefill_ws_kernel(Params p) {
  using T = PT<D>;
  using W = WT<D>;
  constexpr int NTL = W::kNtl;
  constexpr int kTok = T::kTok;
  constexpr int SB = W::kSBuf;
  const Geom& g = p.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = g.Hq / g.Hkv;
  const int TR = p.tr;
  const int tile = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int r0 = tile * NTL * TR;             // first row of the CTA's tiles
  const int rows = min(NTL * TR, g.R - r0);   // rows of the CTA
  const int k = p.k;
  constexpr int ND = W::kDeq;
  const bool soft = warp < 4 * NTL, deq = warp >= 4 * NTL && warp < 4 * NTL + ND;
  // Two MMA warps: one per tile (S and O) with two tiles; with one tile, one
  // issues S and the other O.
  const bool mmaw = warp >= 4 * NTL + ND && warp < 4 * NTL + ND + 2;
  const int mw = warp - (4 * NTL + ND);
  const int mt = NTL == 2 ? mw : 0;                                 // its tile
  const bool does_s = NTL == 2 || mw == 0, does_o = NTL == 2 || mw == 1;
  const bool cpy = warp == 4 * NTL + ND + 2 && lane == 0;           // the copy thread
  const int tt = soft ? warp >> 2 : 0;        // a softmax thread's tile
  const int vi = tid & 127;                   // its query vector (tile row)

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ0 = smem;                                  // [NTL][kQBytes]
  uint8_t* sK0 = sQ0 + NTL * T::kQBytes;                // [2][kKBytes]
  uint8_t* sV0 = sK0 + 2 * T::kKBytes;                  // [2][kKBytes] (V in K's layout)
  uint8_t* sStage = sV0 + 2 * T::kKBytes;               // [kWsStages][kStage]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + kWsStages * kStage);
  uint64_t* full = bars;                 // [kWsStages]
  uint64_t* empty = bars + 4;            // [kWsStages]
  uint64_t* kready = bars + 8;           // [2]
  uint64_t* vready = bars + 10;          // [2]
  uint64_t* kfree = bars + 12;           // [2]
  uint64_t* vfree = bars + 14;           // [2]
  uint64_t* barS = bars + 16;            // [NTL][SB]
  uint64_t* sfree = bars + 18;           // [NTL][SB]
  uint64_t* pready = bars + 20;          // [NTL][2]
  uint64_t* barO = bars + 24;            // [NTL][2]
  uint64_t* mdone = bars + 28;           // [NTL] every MMA of tile t's warp completed
  uint64_t* qbar = bars + 30;            // the CTA's query rows landed
  uint64_t* qready = bars + 31;          // Q in tensor memory (head_dim 256)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + kWsBars);
  int* s_misc = reinterpret_cast<int*>(s_tmem + 1);            // [12]: warp counts, total
  int32_t* s_sel = s_misc + 12;                                 // [NTL * TR][k]
  int32_t* s_union = s_sel + NTL * TR * k;                      // [ucap]
  int32_t* s_upage = s_union + p.ucap;                          // [ucap]
  const int nwords = (g.MB + 31) >> 5;
  const int mwords = ws_member_words(p.ucap);
  uint32_t* s_bits = reinterpret_cast<uint32_t*>(s_upage + p.ucap);   // [nwords]
  int* s_wpre = reinterpret_cast<int*>(s_bits + nwords);              // [nwords]
  uint32_t* s_mem = reinterpret_cast<uint32_t*>(s_wpre + nwords);     // [NTL * TR][mwords]
  int32_t* s_pt = reinterpret_cast<int32_t*>(s_mem + NTL * TR * mwords);   // [MB] page row
  // The CTA's query rows (bf16, [tile][vector][D]) land in the K and V tiles,
  // which stay unused until the chunk loop.
  uint8_t* sQst = sK0;
  float* s_cq = reinterpret_cast<float*>(s_pt + g.MB);   // [NTL * 128] logit scales
  static_assert(NTL * 128 * D * 2 <= 4 * T::kKBytes, "query staging");

  if (tid == 0) {
    for (int z = 0; z < kWsStages; ++z) {
      mbar_init(&full[z], 1);
      mbar_init(&empty[z], ND);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&kready[x], ND >= 8 ? 16 * ND : 32 * ND);   // the threads converting K
      mbar_init(&vready[x], ND >= 8 ? 16 * ND : 32 * ND);   // ... and V
      mbar_init(&kfree[x], NTL);   // one commit per MMA warp
      mbar_init(&vfree[x], NTL);
      mbar_init(&barS[x], 1);
      mbar_init(&sfree[x], 128);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&pready[i], 128);
      mbar_init(&barO[i], 1);
    }
    mbar_init(&mdone[0], 1);
    mbar_init(&mdone[1], 1);
    mbar_init(qbar, 1);
    mbar_init(qready, 128 * NTL);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(s_tmem)),
                 "r"(W::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  bool dead = false;
  __syncthreads();   // the barriers are initialised

  // ---- the CTA's query rows: one bulk copy per row (its G heads, contiguous) ---
  if (cpy) {
    const uint32_t row_bytes = (uint32_t)(G * D * 2);
    mbar_arrive_expect_tx(qbar, (uint32_t)rows * row_bytes);
    for (int jr = 0; jr < rows; ++jr) {
      const int t = jr / TR, jq = jr - t * TR;
      const size_t qrow = ((size_t)b * g.R + r0 + jr) * g.Hq + (size_t)kvh * G;
      bulk_g2s(sQst + ((size_t)t * 128 + (size_t)jq * G) * D * 2, p.q + qrow * D, row_bytes, qbar,
               policy_evict_first());
    }
  }

  // ---- each softmax thread's query vector: its row, head and visible tokens ----
  const int jj = tt * TR + vi / G, hh = vi % G; // row of the CTA, head
  const bool vec = soft && vi / G < TR && jj < rows;   // a real (row, head) vector
  const int j = r0 + jj;
  const int L = p.seqlens[b];
  const int cap = g.MB * g.P;
  const int nrow = vec ? visible_tokens(L, g.R, j, cap) : 0;
  float cq = 0.f;                               // logit scale, log2 domain
  // ---- the tile's rows' selections and their union (softmax warps) ------------
  if (soft) {
    auto soft_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(128 * NTL) : "memory"); };
    // Selections and the page-table row, eight loads in flight per thread.
    constexpr int kNs = 128 * NTL, kLd = 8;
    for (int i0 = tid; i0 < NTL * TR * k; i0 += kLd * kNs) {
      int v[kLd];
#pragma unroll
      for (int u = 0; u < kLd; ++u) {
        const int i = i0 + u * kNs, jr = i / k;
        v[u] = (i < NTL * TR * k && jr < rows) ? p.sel[((size_t)b * g.R + r0 + jr) * k + (i - jr * k)]
                                                : -1;
      }
#pragma unroll
      for (int u = 0; u < kLd; ++u) {
        const int i = i0 + u * kNs;
        if (i < NTL * TR * k) s_sel[i] = (v[u] < 0 || v[u] >= g.MB) ? -1 : v[u];
      }
    }
    for (int i0 = tid; i0 < g.MB; i0 += kLd * kNs) {
      int v[kLd];
#pragma unroll
      for (int u = 0; u < kLd; ++u) {
        const int i = i0 + u * kNs;
        v[u] = i < g.MB ? p.page_table[(size_t)b * g.MB + i] : -1;
      }
#pragma unroll
      for (int u = 0; u < kLd; ++u)
        if (i0 + u * kNs < g.MB) s_pt[i0 + u * kNs] = v[u];
    }
    for (int i = tid; i < nwords; i += 128 * NTL) s_bits[i] = 0u;
    for (int i = tid; i < NTL * TR * mwords; i += 128 * NTL) s_mem[i] = 0u;
    soft_sync();
    for (int i = tid; i < rows * k; i += 128 * NTL) {
      const int v = s_sel[i];
      if (v >= 0) atomicOr(&s_bits[v >> 5], 1u << (v & 31));
    }
    soft_sync();
    // Blocks with a valid page, ascending: thread t scans words [t*per, ...).
    const int per = (nwords + 128 * NTL - 1) / (128 * NTL);
    const int w0 = min(nwords, tid * per), w1 = min(nwords, w0 + per);
    const int32_t* pt = s_pt;
    int cnt = 0;
    for (int w = w0; w < w1; ++w) {
      uint32_t m = s_bits[w];
      while (m) {
        const int beta = (w << 5) + __ffs(m) - 1;
        m &= m - 1;
        const int pg = pt[beta];
        if (pg >= 0 && pg < g.NP) ++cnt; else s_bits[w] &= ~(1u << (beta & 31));
      }
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_misc[warp] = x;
    soft_sync();
    int pos = x - cnt;
    for (int w = 0; w < warp; ++w) pos += s_misc[w];
    for (int w = w0; w < w1; ++w) {
      s_wpre[w] = pos;   // union position of the word's first block
      uint32_t m = s_bits[w];
      while (m) {
        const int beta = (w << 5) + __ffs(m) - 1;
        m &= m - 1;
        if (QSA_IN_BOUNDS(pos < p.ucap, kChkUnion)) {
          s_union[pos] = beta;
          s_upage[pos] = pt[beta];
        }
        ++pos;
      }
    }
    if (tid == 128 * NTL - 1) s_misc[10] = pos;
    soft_sync();
    // Each row's membership bitmap over the union positions.
    for (int i = tid; i < rows * k; i += 128 * NTL) {
      const int v = s_sel[i];
      if (v < 0 || !((s_bits[v >> 5] >> (v & 31)) & 1u)) continue;
      const int u = s_wpre[v >> 5] + __popc(s_bits[v >> 5] & ((1u << (v & 31)) - 1u));
      if (QSA_IN_BOUNDS(u < p.ucap, kChkUnion))
        atomicOr(&s_mem[(i / k) * mwords + (u >> 5)], 1u << (u & 31));
    }
  }

  // ---- the query vectors into the swizzled fp16 Q tiles ------------------------
  // By the dequantisation warps (idle until the chunk loop) while the softmax
  // warps build the union: a per-vector power-of-two scale (the largest
  // magnitude near 2^8), with one or two threads per vector.  Lanes start at
  // different 16-byte pieces of their rows, so the staging reads avoid bank
  // conflicts.
  if (deq) {
    const int dt = tid - 128 * NTL;
    constexpr int kNv = NTL * 128;                       // the CTA's vectors
    constexpr int kGs = 32 * ND >= 2 * kNv ? 2 : 1;      // threads per vector
    constexpr int kPer = D / 8 / kGs;                    // 16-byte pieces per thread
    constexpr int kStride = 32 * ND / kGs;
    const bool qok = __all_sync(0xffffffffu, wait_bounded(qbar, 0));
    if (!qok) dead = true;
    const int half = dt % kGs;
    for (int v = dt / kGs; v < kNv; v += kStride) {
      const int t = v >> 7, vv = v & 127, jr = t * TR + vv / G;
      const bool valid = qok && vv / G < TR && jr < rows;
      const uint8_t* src = sQst + (size_t)v * D * 2;
      float amax = 0.f;
      if (valid) {
#pragma unroll 4
        for (int i = 0; i < kPer; ++i) {
          const int ii = half * kPer + ((i + lane) & (kPer - 1));
          const uint4 r = *reinterpret_cast<const uint4*>(src + ii * 16);
          const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[u] << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(w4[u] & 0xFFFF0000u)));
          }
        }
      }
      if (kGs == 2) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      const int ebits = (int)((__float_as_uint(amax) >> 23) & 0xFF);
      int sq = (amax > 0.f) ? 135 - ebits : 0;
      sq = sq > 126 ? 126 : (sq < -126 ? -126 : sq);
      const float up = __uint_as_float((uint32_t)(sq + 127) << 23);
      const float down = __uint_as_float((uint32_t)(127 - sq) << 23);
      if (half == 0) s_cq[v] = valid ? p.k_scale * p.sm_scale * kLog2e * down : 0.f;
#pragma unroll 4
      for (int i = 0; i < kPer; ++i) {
        const int ii = half * kPer + ((i + lane) & (kPer - 1));
        uint4 h = make_uint4(0u, 0u, 0u, 0u);
        if (valid) {
          const uint4 r = *reinterpret_cast<const uint4*>(src + ii * 16);
          const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
          uint32_t o[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            o[u] = pack_half2(__uint_as_float(w4[u] << 16) * up,
                              __uint_as_float(w4[u] & 0xFFFF0000u) * up);
          h = make_uint4(o[0], o[1], o[2], o[3]);
        }
        *reinterpret_cast<uint4*>(sQ0 + t * T::kQBytes + (ii >> 3) * 16384 + sw128(vv, ii & 7)) = h;
      }
    }
  }
  fence_proxy_async_smem();       // Q and zero tiles (generic stores) before the MMAs
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int U = s_misc[10];
  if (soft) cq = s_cq[tt * 128 + vi];
  if constexpr (W::kQTmem) {
    // Each softmax thread copies its Q row (fp16, dims in order, two per
    // column: the A-operand layout) into its tensor-memory lane.
    if (soft) {
      const uint32_t lane_q = (uint32_t)(32 * (warp & 3)) << 16;
#pragma unroll
      for (int q16 = 0; q16 < D / 32; ++q16) {   // 16 columns = 32 dims = 4 pieces
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int pc = 4 * q16 + i;   // 8-dim piece
          const uint4 r = *reinterpret_cast<const uint4*>(sQ0 + (pc >> 3) * 16384 + sw128(vi, pc & 7));
          v[4 * i] = r.x; v[4 * i + 1] = r.y; v[4 * i + 2] = r.z; v[4 * i + 3] = r.w;
        }
        tmem_st16u(tmem + W::kQBase + lane_q + 16 * q16, v);
      }
      tmem_wait_st();
      tc_fence_before();
      ws_arrive(qready);
    }
  }
  const int csh = (g.P == 2 * kTok) ? 1 : 0;    // chunks per block: 1 << csh
  const int C = U << csh;
  const uint32_t* mymem = s_mem + (vec ? jj : 0) * mwords;
  auto tO = [&](int t) { return tmem + W::kOBase + (uint32_t)(t * D); };
  auto tS = [&](int t, int c) { return tmem + (uint32_t)((t * SB + c % SB) * kTok); };
  auto tP = [&](int t, int x) { return tmem + W::kPBase + (uint32_t)((2 * t + x) * (kTok / 2)); };
  auto sQ = [&](int t) { return sQ0 + t * T::kQBytes; };
  auto sK = [&](int x) { return sK0 + x * T::kKBytes; };
  auto sV = [&](int x) { return sV0 + x * T::kKBytes; };

  // ---- bulk copies (lane 0 of the copy warp) ----------------------------------
  // Stage c % 4 is refilled with chunk c + 4 once the dequantisation warps
  // are done with chunk c.
  if (cpy) {
    const uint64_t pol = policy_evict_first();
    auto issue_copy = [&](int c) {
      const int z = c % kWsStages;
      uint8_t* dst = sStage + z * kStage;
      const int u = c >> csh, sub = c & csh;
      if (!QSA_IN_BOUNDS(u < U && u < p.ucap && s_upage[u] >= 0 && s_upage[u] < g.NP,
                         kChkChunk))
        return;
      const size_t row0 = ((size_t)s_upage[u] * g.Hkv + kvh) * g.P + (size_t)sub * kTok;
      mbar_arrive_expect_tx(&full[z], kStage);
      bulk_g2s(dst, p.k_pool + row0 * (D / 2), kTok * D / 2, &full[z], pol);
      bulk_g2s(dst + kTok * D / 2, p.v_pool + row0 * (D / 2), kTok * D / 2, &full[z], pol);
      bulk_g2s(dst + kTok * D, p.k_sf + row0 * (D / 16), kTok * D / 16, &full[z], pol);
      bulk_g2s(dst + kTok * D + kTok * D / 16, p.v_sf + row0 * (D / 16), kTok * D / 16,
               &full[z], pol);
    };
    int ncopy = min(C, kWsStages);
    for (int c = 0; c < ncopy; ++c) issue_copy(c);
    for (int c = kWsStages; c < C; ++c) {
      const int cp = c - kWsStages;   // the chunk that last used stage c % kWsStages
      if (!wait_bounded(&empty[cp % kWsStages], (cp / kWsStages) & 1)) {
        dead = true;
        break;
      }
      fence_proxy_async_smem();   // the dequant warps' reads of the stage come first
      issue_copy(c);
      ncopy = c + 1;
    }
    // Every copy issued lands before shared memory is released.
    for (int c = max(0, ncopy - kWsStages); c < ncopy; ++c)
      wait_bounded(&full[c % kWsStages], (c / kWsStages) & 1);
    wait_bounded(qbar, 0);
  }

  // ---- MMA issue (two warps; one elected lane of each issues) -----------------
  // S(c) once K(c) is dequantised and the tile's softmax(c - SB) has loaded
  // S buffer c % SB; O(c) once P(c) and V(c) are ready.  The whole warp runs
  // the loop so descriptors stay warp-uniform.
  if (mmaw) {
    const int t = mt;
    // S: Q (A) and K (B) K-major.  O: P from tensor memory, V (B) MN-major:
    // 64-dim blocks kKBlk bytes apart, 8-token row groups 1024 bytes apart.
    const uint32_t id_s = f16_idesc(128, kTok), id_o = f16_idesc(128, D) | kIdescBMn;
    const uint64_t dq = sw128_desc(smem_u32(sQ(t)));
    const uint64_t dk0 = sw128_desc(smem_u32(sK(0))), dk1 = sw128_desc(smem_u32(sK(1)));
    const uint64_t dv0 = sw128_mn_desc(smem_u32(sV(0)), T::kKBlk);
    const uint64_t dv1 = sw128_mn_desc(smem_u32(sV(1)), T::kKBlk);
    auto issue_s = [&](int c) {   // the tile's S(c); then its S buffer and K tile x commits
      const int x = c & 1;
      const uint64_t dk = x ? dk1 : dk0;
#pragma unroll
      for (int h = 0; h < D / 64; ++h)
#pragma unroll
        for (int ks2 = 0; ks2 < 4; ++ks2) {
          const uint64_t bk = dk + (uint64_t)((h * T::kKBlk + 32 * ks2) >> 4);
          if constexpr (W::kQTmem)   // Q columns: 16 dims (one K step) per 8
            mma_f16_ts_elect(tS(t, c), tmem + W::kQBase + 8 * (4 * h + ks2), bk, id_s,
                             (h | ks2) ? 1u : 0u);
          else
            mma_f16_elect(tS(t, c), dq + (uint64_t)((h * 16384 + 32 * ks2) >> 4), bk, id_s,
                          (h | ks2) ? 1u : 0u);
        }
      mma_commit_elect(&barS[t * SB + c % SB]);
      mma_commit_elect(&kfree[x]);
    };
    // The tile's O += P(c) V(c): P from tensor memory (kTok / 16 steps of 16
    // tokens, eight columns each), V from shared memory (16 token rows per
    // step); then the O and V tile x commits.
    auto issue_o = [&](int c) {
      const int x = c & 1;
      const uint64_t dv = x ? dv1 : dv0;
#pragma unroll
      for (int ks2 = 0; ks2 < kTok / 16; ++ks2)
        mma_f16_ts_elect(tO(t), tP(t, x) + 8 * ks2, dv + (uint64_t)((2048 * ks2) >> 4), id_o,
                         (c | ks2) ? 1u : 0u);
      mma_commit_elect(&barO[t * 2 + x]);
      mma_commit_elect(&vfree[x]);
    };
    // Each pass probes every barrier the next O and the next S wait on (the
    // probes overlap), then issues O(no) and S(ns) if they are ready: O(no)
    // needs V(no) and P(no); S(ns) needs K(ns) and the softmax's release of
    // S buffer ns % SB.  Neither barrier can run a phase ahead of the waiter
    // (each next phase needs an MMA this warp has not issued yet).
    int ns = does_s ? 0 : C, no = does_o ? 0 : C;
    if (W::kQTmem && does_s && ns < C) {
      if (!__all_sync(0xffffffffu, wait_bounded(qready, 0))) {
        dead = true;
        ns = no = C;
      }
      tc_fence_after();
    }
    unsigned long long spin0 = 0;
    bool spinning = false;
    while (no < C || ns < C) {
      bool s_ok = false, o_ok = false;
      if (ns < C) {
        const int cf = max(ns - SB, 0);   // the chunk whose S buffer S(ns) reuses
        const bool k_ok = mbar_test_wait(&kready[ns & 1], (ns >> 1) & 1);
        const bool f_ok = ns < SB || mbar_test_wait(&sfree[t * SB + cf % SB], (cf / SB) & 1);
        s_ok = k_ok && f_ok;
      }
      if (no < C && (no < ns || !does_s)) {   // (P(no) implies S(no) was issued)
        const bool v_ok = mbar_test_wait(&vready[no & 1], (no >> 1) & 1);
        const bool p_ok = mbar_test_wait(&pready[t * 2 + (no & 1)], (no >> 1) & 1);
        o_ok = v_ok && p_ok;
      }
      o_ok = __all_sync(0xffffffffu, o_ok);
      s_ok = __all_sync(0xffffffffu, s_ok);
      if (o_ok || s_ok) {
        tc_fence_after();
        if (o_ok) issue_o(no++);
        if (s_ok) issue_s(ns++);
        spinning = false;
      } else if (!spinning) {
        spin0 = now_ns();
        spinning = true;
      } else if (__any_sync(0xffffffffu, now_ns() - spin0 > kWaitNs)) {
        dead = true;
        break;
      }
    }
    // Every MMA this warp issued completes before the tiles and tensor memory
    // are read or released (at once when nothing went wrong).
    mma_commit_elect(&mdone[mw]);
    wait_bounded(&mdone[mw], 0);
    __syncwarp();
  }

  // ---- dequantisation (ND warps) -----------------------------------------------
  // K and V alike: rows = tokens, D/64 blocks of 64 dims (128-byte swizzled
  // rows); a thread converts pieces of eight values (one code word, one
  // scale).  K feeds S as a K-major B operand, V feeds O as an MN-major one.
  // With eight warps, four convert K and four V, each group waiting only on
  // its own tile's release; with four, every warp converts both.
  if (deq) {
    const int dt = tid - 128 * NTL;
    constexpr bool kSplitKV = ND >= 8;
    constexpr int kOpThreads = kSplitKV ? 16 * ND : 32 * ND;   // threads per operand
    constexpr int kPieces = kTok * D / 8 / kOpThreads;
    const bool do_k = !kSplitKV || dt < kOpThreads, do_v = !kSplitKV || dt >= kOpThreads;
    const int ot = kSplitKV ? dt % kOpThreads : dt;            // thread within its operand
    auto rows_tile = [&](const uint8_t* codes, const uint8_t* scales, uint8_t* tile) {
#pragma unroll
      for (int i = 0; i < kPieces; ++i) {
        const int pc = ot + kOpThreads * i;   // (token, 8-dim group)
        const int t = pc / (D / 8), c8 = pc % (D / 8);
        const uint32_t w = *reinterpret_cast<const uint32_t*>(codes + t * (D / 2) + c8 * 4);
        const uint32_t sc = e4m3x2_to_f16x2(scales[t * (D / 16) + (c8 >> 1)]);
        *reinterpret_cast<uint4*>(tile + (c8 >> 3) * T::kKBlk + sw128(t, c8 & 7)) =
            dequant8(w, prmt(sc, 0, 0x1010));
      }
    };
    for (int c = 0; c < C; ++c) {
      const int x = c & 1, z = c % kWsStages;
      const uint8_t* st = sStage + z * kStage;
      // First probes of the stage, the K tile and the V tile overlap; then
      // warp-uniform give-ups (the warp syncs below).  kfree / vfree: every
      // S(c - 2) / O(c - 2) has read tile x.
      const bool f_now = mbar_test_wait(&full[z], (c / kWsStages) & 1);
      const bool k_now = !do_k || c < 2 || mbar_test_wait(&kfree[x], ((c - 2) >> 1) & 1);
      const bool v_now = !do_v || c < 2 || mbar_test_wait(&vfree[x], ((c - 2) >> 1) & 1);
      if (__any_sync(0xffffffffu,
                     !((f_now || wait_bounded(&full[z], (c / kWsStages) & 1)) &&
                       (k_now || wait_bounded(&kfree[x], ((c - 2) >> 1) & 1))))) {
        dead = true;
        break;
      }
      if (do_k) {
        rows_tile(st, st + kTok * D, sK(x));
        fence_proxy_async_smem();
        ws_arrive(&kready[x]);
      }
      if (do_v) {
        if (__any_sync(0xffffffffu, !(v_now || wait_bounded(&vfree[x], ((c - 2) >> 1) & 1)))) {
          dead = true;
          break;
        }
        rows_tile(st + kTok * D / 2, st + kTok * D + kTok * D / 16, sV(x));
        fence_proxy_async_smem();
        ws_arrive(&vready[x]);
      }
      __syncwarp();
      if (lane == 0) ws_arrive(&empty[z]);   // this warp is done with the stage
    }
  }

  // ---- softmax (four warps per tile: thread = query vector = tensor-memory lane)
  float m_base = -INFINITY, l_run = 0.f;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  if (soft) {
    for (int c = 0; c < C; ++c) {
      const int x = c & 1;
      const int u = c >> csh;                      // union position of the chunk
      const uint32_t mword = mymem[u >> 5];
      const int ue = s_union[u];
      // First probes of S(c) and of O(c - 2) (P buffer x free) overlap; then a
      // warp-uniform give-up (tensor-memory loads and stores are warp-wide).
      const bool s_now = mbar_test_wait(&barS[tt * SB + c % SB], (c / SB) & 1);
      const bool p_now = c < 2 || mbar_test_wait(&barO[tt * 2 + x], ((c - 2) >> 1) & 1);
      if (__any_sync(0xffffffffu,
                     !(s_now || wait_bounded(&barS[tt * SB + c % SB], (c / SB) & 1)))) {
        dead = true;
        break;
      }
      tc_fence_after();
      const int tok0 = ue * g.P + (c & csh) * kTok;
      const bool member = vec && tok0 < nrow && ((mword >> (u & 31)) & 1u);
      float z[kTok];
      if (__any_sync(0xffffffffu, member)) {   // a warp with no member skips the load
#pragma unroll
        for (int q4 = 0; q4 < kTok / 16; ++q4) {
          float v16[16];
          tmem_ld16(tS(tt, c) + lane_off + 16 * q4, v16);
#pragma unroll
          for (int i = 0; i < 16; ++i) z[16 * q4 + i] = v16[i];
        }
        tmem_wait_ld();
      }
      tc_fence_before();
      ws_arrive(&sfree[tt * SB + c % SB]);   // S buffer loaded: S(c + SB) may overwrite it
      float cmax = -INFINITY;   // log2 units
      if (member) {
        if (tok0 + kTok > nrow) {
#pragma unroll
          for (int i = 0; i < kTok; ++i)
            if (tok0 + i >= nrow) z[i] = -INFINITY;
        }
        float mx8[8];   // three-input maxima: eight running maxima, then a tree
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = z[i];
#pragma unroll
        for (int i = 8; i < kTok; i += 2) mx8[(i >> 1) & 7] = fmax3(mx8[(i >> 1) & 7], z[i], z[i + 1]);
        const float m3 = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7]));
        cmax = m3 * cq;     // cq > 0: the scale keeps the order
      }
      bool rescale = false;
      float alpha = 1.f;
      if (cmax != -INFINITY) {
        if (m_base == -INFINITY) {
          m_base = cmax;
        } else if (cmax > m_base + kRescaleGap) {
          alpha = exp2_approx(m_base - cmax);
          m_base = cmax;
          rescale = true;
        }
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O holds every chunk before c once O(c - 1) completed (O(c) waits for
        // this chunk's P); a warp rescales when any of its lanes must.
        if (c >= 1 &&
            __any_sync(0xffffffffu,
                       !wait_bounded(&barO[tt * 2 + ((c - 1) & 1)], ((c - 1) >> 1) & 1))) {
          dead = true;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int q8 = 0; q8 < D / 16; ++q8) {
          float o16[16];
          tmem_ld16(tO(tt) + lane_off + 16 * q8, o16);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) o16[i] *= alpha;
          tmem_st16(tO(tt) + lane_off + 16 * q8, o16);
        }
        tmem_wait_st();
      }
      // P buffer x is free once O(c - 2) completed.
      if (__any_sync(0xffffffffu,
                     !(p_now || wait_bounded(&barO[tt * 2 + x], ((c - 2) >> 1) & 1)))) {
        dead = true;
        break;
      }
      tc_fence_after();
      // This lane's P row, 32 tokens at a time: token pair i in column i (the
      // A-operand layout); the row sum from the same fp32 values.
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < kTok / 32; ++q) {
        uint32_t pk[16];
        if (member) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float p0 = exp2_approx(fmaf(z[32 * q + 2 * i], cq, -m_base));
            const float p1 = exp2_approx(fmaf(z[32 * q + 2 * i + 1], cq, -m_base));
            ls4[i & 3] += p0 + p1;
            pk[i] = pack_half2(p0, p1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = 0u;
        }
        tmem_st16u(tP(tt, x) + lane_off + 16 * q, pk);
      }
      if (member) l_run = l_run * alpha + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
      tmem_wait_st();
      tc_fence_before();
      ws_arrive(&pready[tt * 2 + x]);   // P(c) written, O rescaled
    }
  }

  // ---- epilogue: out = O / l * v_scale, lse -------------------------------------
  // The issuer has seen its last O complete; the barrier publishes that.
  if (dead) atomicExch(p.status, kStatusWaitTimeout);
  tc_fence_before();
  const bool any_dead = __syncthreads_or(dead);
  tc_fence_after();
  if (soft && !any_dead) {
    const size_t orow = ((size_t)b * g.R + j) * g.Hq + (size_t)kvh * G + hh;
    const bool out_ok = !vec || QSA_IN_BOUNDS(b < g.B && j < g.R && kvh * G + hh < g.Hq, kChkOut);
    uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D);
    const bool has = l_run > 0.f && C > 0;
    const float sc = has ? p.v_scale / l_run : 0.f;
#pragma unroll 4
    for (int q8 = 0; q8 < D / 16; ++q8) {
      float o16[16];
      if (C > 0) {
        tmem_ld16(tO(tt) + lane_off + 16 * q8, o16);
        tmem_wait_ld();
      }
      uint32_t h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        __nv_bfloat162 x2 = __floats2bfloat162_rn(has ? o16[2 * i] * sc : 0.f,
                                                  has ? o16[2 * i + 1] * sc : 0.f);
        h[i] = *reinterpret_cast<uint32_t*>(&x2);
      }
      if (vec && out_ok) {
        dst[2 * q8] = make_uint4(h[0], h[1], h[2], h[3]);
        dst[2 * q8 + 1] = make_uint4(h[4], h[5], h[6], h[7]);
      }
    }
    if (vec && out_ok) p.lse[orow] = has ? (m_base + log2f(l_run)) * kLn2 : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(W::kTmemCols));
}

}  // namespace

int prefill_rows_per_tile(const Geom& g) {
  const int G = g.Hq / g.Hkv;
  return G <= 128 ? 128 / G : 0;
}

size_t prefill_smem_bytes(const Geom& g, int k) {
  const int tr = prefill_rows_per_tile(g);
  const int ucap = min(g.MB, tr * k);
  const size_t tiles = g.D == 256
                           ? (size_t)PT<256>::kQBytes + PT<256>::kKBytes + PT<256>::kVBytes + PT<256>::kPBytes
                           : (size_t)PT<128>::kQBytes + PT<128>::kKBytes + PT<128>::kVBytes + PT<128>::kPBytes;
  return (size_t)1024 + tiles + 2 * kStage + 4 * 8 + 4 + 8 * 4 +
         (size_t)tr * k * 4 + (size_t)ucap * 8 + (size_t)((g.MB + 31) / 32) * 4;
}

// The warp-specialised kernel's shared memory (double-buffered tiles); the
// four-warp kernel (single tiles) serves geometries where it does not fit.
int prefill_ws_tiles(const Geom& g) { return g.D == 256 ? WT<256>::kNtl : WT<128>::kNtl; }

// Rows per tile of the warp-specialised kernel (one CTA per SM): at most
// 128 / G; among the heights down to half of that whose grid takes as many
// waves as the tallest, the shortest, so that each CTA walks the smallest
// union of selected blocks the wave count allows.
int prefill_ws_rows_per_tile(const Geom& g) {
  const int trmax = prefill_rows_per_tile(g);
  if (trmax < 1) return trmax;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int ntl = prefill_ws_tiles(g);
  auto waves = [&](int tr) {
    const long long ctas = (long long)((g.R + ntl * tr - 1) / (ntl * tr)) * g.Hkv * g.B;
    return (ctas + sms - 1) / sms;
  };
  const long long w0 = waves(trmax);
  int tr = trmax;
  while (tr - 1 >= (trmax + 1) / 2 && waves(tr - 1) == w0) --tr;
  return tr;
}

size_t prefill_ws_smem_bytes(const Geom& g, int k) {
  const int rows = prefill_ws_tiles(g) * prefill_ws_rows_per_tile(g);   // rows per CTA
  const int ucap = min(g.MB, rows * k);
  const size_t tiles = g.D == 256 ? WT<256>::kTiles : WT<128>::kTiles;
  return (size_t)1024 + tiles + kWsStages * kStage + kWsBars * 8 + 4 + 12 * 4 + (size_t)rows * k * 4 +
         (size_t)ucap * 8 + (size_t)((g.MB + 31) / 32) * 8 + (size_t)rows * ws_member_words(ucap) * 4 +
         (size_t)g.MB * 4 + (size_t)prefill_ws_tiles(g) * 128 * 4;
}

cudaError_t launch_sparse_prefill(const Geom& g, const void* q, const uint8_t* k_pool,
                                  const uint8_t* k_sf, const uint8_t* v_pool, const uint8_t* v_sf,
                                  float k_scale, float v_scale, float sm_scale,
                                  const int32_t* page_table, const int32_t* seqlens,
                                  const int32_t* sel, int k, void* out, float* lse,
                                  int* status, cudaStream_t stream) {
  Params prm;
  prm.g = g;
  prm.q = reinterpret_cast<const __nv_bfloat16*>(q);
  prm.k_pool = k_pool; prm.k_sf = k_sf; prm.v_pool = v_pool; prm.v_sf = v_sf;
  prm.k_scale = k_scale; prm.v_scale = v_scale; prm.sm_scale = sm_scale;
  prm.page_table = page_table; prm.seqlens = seqlens; prm.sel = sel; prm.k = k;
  prm.out = reinterpret_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.status = status;
#ifdef QSA_PREFILL_FOUR_WARPS
  const bool ws = false;
#else
  const bool ws = prefill_ws_smem_bytes(g, k) <= 227 * 1024;
#endif
  const size_t smem = ws ? prefill_ws_smem_bytes(g, k) : prefill_smem_bytes(g, k);
  prm.tr = ws ? prefill_ws_rows_per_tile(g) : prefill_rows_per_tile(g);
  const int rows_per_cta = (ws ? prefill_ws_tiles(g) : 1) * prm.tr;
  prm.ucap = min(g.MB, rows_per_cta * k);
  auto* kern = ws ? (g.D == 256 ? sparse_prefill_ws_kernel<256> : sparse_prefill_ws_kernel<128>)
                  : (g.D == 256 ? sparse_prefill_kernel<256> : sparse_prefill_kernel<128>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((g.R + rows_per_cta - 1) / rows_per_cta, g.Hkv, g.B);
  cfg.blockDim = dim3(ws ? (g.D == 256 ? WT<256>::kThreads : WT<128>::kThreads) : kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace qsa

QSA_BOUNDS_READER(bounds_word_prefill)
