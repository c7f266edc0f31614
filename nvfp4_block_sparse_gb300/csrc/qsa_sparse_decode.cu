// qsa_sparse_decode.cu -- A3: split-KV sparse GQA over the selected NVFP4
// pages, dequantised in registers, partials merged by log-sum-exp.
//
// TensorRT-LLM PR #20937 ("GB300 perf work on
// qwen3_8_flash_next_nvfp4__sm_103__tp1"), What changes: NVFP4 sparse GQA
// decode as a split-K + merge kernel with a lean one-split variant, and verify
// as request-grouped NVFP4 sparse GQA with a per-row merge; Per-File QA:
// invalid-page handling and masking.  PR #20276 ("Qwen3.8-Flash-Next NVFP4
// target"), Features table: uint8 e2m1 pages + e4m3 block scales.
//
// One CTA = (request b, KV head g, head slice, KV split s).  Its query columns
// are the (row j, head) pairs of the request's R rows for a slice of up to
// 8*NTR of the G query heads that read KV head g.  The pages it reads are the
// union of the rows' selections (each page carries a mask of the rows that
// selected it), so each page is read from HBM once per KV head; the split
// takes a contiguous share of that union's 64-token chunks.
//
// Warp roles.  A producer warp streams the chunks (K 4 KB + K scales 512 B +
// V 4 KB + V scales 512 B, contiguous in the pools) into shared-memory stages
// with TMA bulk copies and full/empty mbarriers.  Each consumer warp owns one
// row's columns and processes a chunk completely and alone: with one row
// (decode) the consumers take chunks round-robin; with R rows (verify) there
// is one consumer per row and it processes exactly the chunks its row
// selected.  No warp waits on another inside a chunk.
//
// Per chunk the consumer dequantises straight into mma.sync fragments:
//   S^T = K . Q^T     A = K tile (tokens x dims) from e2m1 bytes * e4m3 scale,
//                     B = Q^T (fp16, pre-scaled by a power of two per column)
//   O^T += V^T . P^T  A = V^T tile (dims x tokens) built from two tokens'
//                     nibbles per byte, B = P^T from S^T by an 8x8 transpose
// e2m1 x e4m3 products are exact in fp16, so the only roundings are the fp16
// P and fp32 accumulation.  Dims and tokens are permuted inside each MMA so
// that each thread reads whole 16-byte (K) and 8-byte (V) runs of a token row
// and shared-memory wavefronts stay conflict-free; the contraction is
// invariant under those permutations and the output un-permutes them.
//
// Every wait is bounded: a wait that gives up records a status word in the
// workspace and the kernel still finishes.
#include "qsa_common.cuh"
#include "qsa_select_row.cuh"

#include <cooperative_groups.h>
#include <math.h>

#include <mutex>
#include <vector>

namespace cg = cooperative_groups;

namespace qsa {
namespace {

// Per head dimension D (128 or 256): a stage holds 8192 elements of K and of
// V, i.e. 64 tokens at D = 128 and 32 tokens at D = 256, so every stage is
// K codes 4 KB | V codes 4 KB | K scales 512 B | V scales 512 B.
template <int D>
struct Hd {
  static_assert(D == 128 || D == 256, "head_dim 128 or 256");
  static constexpr int kChunk = 8192 / D;            // tokens per pipeline stage
  static constexpr int kRow = D / 2;                 // code bytes per token row
  static constexpr int kSfRow = D / 16;              // scale bytes per token row
  static constexpr int kKBytes = kChunk * kRow;      // 4096
  static constexpr int kSfBytes = kChunk * kSfRow;   // 512
  static constexpr int kPartStride = 4 + D;          // m, l, pad, pad, O[D] per column
  static constexpr int kMt = kChunk / 16;            // 16-token tiles per stage
  static constexpr int kDt = D / 16;                 // 16-dim tiles
  static constexpr int kRuns = D / 128;              // 16-byte runs of a row per lane
};
// Bounds-check codes (reported by bounds-checked builds only).
[[maybe_unused]] constexpr int kChkList = 0x201;    // decode warp list slot past its capacity
[[maybe_unused]] constexpr int kChkUnion = 0x202;   // verify union slot out of range
[[maybe_unused]] constexpr int kChkChunk = 0x203;   // chunk: slot, page id or token offset out of range
[[maybe_unused]] constexpr int kChkOut = 0x204;     // output row or dims out of range
[[maybe_unused]] constexpr int kChkUnit = 0x205;    // workspace unit or split out of range
constexpr int kStageBytes = 9216;
static_assert(2 * Hd<128>::kKBytes + 2 * Hd<128>::kSfBytes == kStageBytes, "stage size");
static_assert(2 * Hd<256>::kKBytes + 2 * Hd<256>::kSfBytes == kStageBytes, "stage size");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s per bounded wait
constexpr int kMaxCluster = 8;               // portable cluster size
constexpr int kPtRowMax = 4096;              // page-table rows up to this stay in smem

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
  __nv_bfloat16* out;
  float* lse;
  int* status;          // workspace status word
  int* tickets;         // [units]
  float* partials;      // [units][splits][R * 8 * NTR][4 + D]
  int splits;           // KV splits per unit
  int slices;           // head slices per KV head
  int cluster;          // 1: ticket merge through partials; >1: cluster (DSMEM) merge
  // Fused selection (decode rows only): when scores is set, each CTA selects
  // its row from the scores itself instead of reading sel; the CTA of split
  // 0, KV head 0, slice 0 writes the row's sel_out / nsel_out.
  const int32_t* scores;
  int window;
  int32_t* sel_out;
  int32_t* nsel_out;
};

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitNs) return false;
  }
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Four bytes of e2m1 pairs -> four fp16 pairs (byte i -> o[i], low nibble in
// the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

// Chunks a decode warp can own: the row's k entries of up to two stages
// each, dealt over splits * W warps.
__host__ __device__ inline int decode_list_cap(int k, int splits, int W) {
  return (2 * k + splits * W - 1) / (splits * W);
}

// Rows of its request one CTA takes: all of them, except for self-issued
// variants with fewer warps than rows (one warp per row, R / W CTAs per
// request).
__host__ __device__ inline int rows_per_cta(bool one, int W, int R) {
  return (one && W < R) ? W : R;
}

// Shared-memory layout (bytes), shared by host sizing and the kernel.  ONE:
// the single-row specialisation (no producer warp; W consumer warps).
template <int NTR, int W, int S, bool ONE, int D>
struct Layout {
  static constexpr int kHsp = 8 * NTR;                            // padded head slice
  static constexpr int kWarps = ONE ? W : W + 1;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kStagesSz = S * kStageBytes;
  static constexpr int kPartStride = Hd<D>::kPartStride;
  // After the main loop the stage region holds the consumers' partials (co,
  // cm, cl), the CTA partial (cp) and the cluster merge's receive buffer
  // (rb); the ticket merge instead reuses it for its weights.  Before the
  // main loop it holds the union's temporaries.  With one consumer per row
  // (direct) each consumer writes its row's partial straight into cp and co,
  // cm, cl are not used.
  static constexpr int kCoSz = W * kHsp * D * 4;
  static constexpr int kCmSz = W * kHsp * 4;
  static constexpr int kClSz = W * kHsp * 4;
  __host__ __device__ static bool direct(int R) { return W == R; }
  __host__ __device__ static int cp_off(int R) { return direct(R) ? 0 : kCoSz + kCmSz + kClSz; }
  __host__ __device__ static int cp_bytes(int R) { return R * kHsp * kPartStride * 4; }
  __host__ __device__ static int rb_off(int R) { return (cp_off(R) + cp_bytes(R) + 15) & ~15; }
  __host__ __device__ static int region_bytes(int R, int k, int splits) {
    const int combine = rb_off(R) + rb_bytes(R, splits);
    const int merge = R * kHsp * (splits + 2) * 4;
    const int uni = R * k * 4 * 2;
    int r = kStagesSz;
    r = r > combine ? r : combine;
    r = r > merge ? r : merge;
    r = r > uni ? r : uni;
    const int qtile = R * kHsp * D * 2;   // the queries, before the main loop
    r = r > qtile ? r : qtile;
    return (r + 15) & ~15;
  }
  // Receive buffer of the cluster merge: [splits][ceil(ncols / splits)] partials.
  __host__ __device__ static int rb_bytes(int R, int splits) {
    if (splits < 2 || splits > kMaxCluster) return 0;
    const int per = (R * kHsp + splits - 1) / splits;
    return splits * per * kPartStride * 4;
  }
  static size_t bytes(int R, int k, int mb, int splits) {
    size_t off = (size_t)region_bytes(R, k, splits);
    off += 2 * S * 8;                                   // full + empty barriers
    off += (size_t)R * kHsp * 4 * 2;                    // cq, n per column
    off += 64 * 4;                                      // scalars
    // union variants: sel rows, union ids, pages, scan; self-issued: the
    // per-warp chunk lists, then the fused selection's row
    off += ONE ? ((size_t)W * 2 * decode_list_cap(k, splits, W / R) + k) * 4
               : (size_t)R * k * 4 * 4 + 16;
    off += mb <= kPtRowMax ? (size_t)mb * 4 : 0;        // page-table row
    return off;
  }
};

// Register budget: at D = 128, 128 per thread for single-row 8-column CTAs
// (two CTAs of 256 threads or four of 128 per SM), about 136 for 8-column
// verify CTAs with up to four row consumers, unconstrained otherwise; at
// D = 256 (twice the output and query fragments) two CTAs per SM of up to
// five warps, unconstrained for wider ones.
#ifndef QSA_SELF_MIN_BLOCKS
#define QSA_SELF_MIN_BLOCKS 4
#endif
template <int NTR, int W, bool ONE, int D>
constexpr int decode_min_blocks() {
  return NTR != 1 ? 1
                  : (D != 128 ? (W <= 4 ? 2 : 1)
                              : (ONE ? (W <= 4 ? QSA_SELF_MIN_BLOCKS : 2) : (W <= 4 ? 3 : 2)));
}

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One stage (K, V and their scales at sk, contiguous) into the online-softmax
// state of 8*NTR columns.  tok0: the stage's first token; tokens at or past
// nrow are masked.
//
// Lane (gid, tig) reads, for QK, bytes [D/8 * tig, D/8 * (tig+1)) of two token
// rows per 16-token tile (D/4 dims, in D/128 runs of 16 bytes): k-step kk
// covers dims D/4 * tig + 4*kk + {0..3} on both operands.  For PV it reads
// bytes [D/16 * gid, D/16 * (gid+1)) of four token rows per k-step: dim tile
// dt holds dims D/8 * gid + 2*dt (+1 in the upper eight rows).
//
// The work is two halves: consume_qk reads only the stage's K codes and
// scales and leaves P^T in registers (pf), consume_pv reads only the V codes
// and scales, so a warp that owns its stage can refill the K half while it
// still works on the V half.
template <int NTR, int D>
__device__ __forceinline__ void consume_qk(const uint8_t* __restrict__ sk, int tok0, int nrow,
                                           const uint32_t (&qf)[NTR][D / 8],
                                           const float (&cq)[NTR][2], float (&m_run)[NTR][2],
                                           float (&l_run)[NTR][2],
                                           float (&o_acc)[D / 16][NTR][4],
                                           uint32_t (&pf)[Hd<D>::kMt][NTR][2]) {
  using H = Hd<D>;
  constexpr int kMt = H::kMt;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const bool partial = tok0 + H::kChunk > nrow;
  const uint8_t* sks = sk + 2 * H::kKBytes;

  // ---- S^T = K . Q^T over the stage's 16-token tiles -----------------
  // Tiles go in pairs: k-steps outside and the pair inside, so
  // consecutive MMAs feed different accumulators.
  float sacc[kMt][NTR][4];
#pragma unroll
  for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
    for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = 0.f;
#pragma unroll
  for (int m0 = 0; m0 < kMt; m0 += 2) {
#pragma unroll
    for (int run = 0; run < H::kRuns; ++run) {
      uint32_t wA[2][4], wB[2][4], scA[2][2], scB[2][2];
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        const int mt = m0 + gi;
        const int rA = 16 * mt + (gid >> 1) + 4 * (gid & 1);
        const int rB = rA + 8;
        const int kb = (D / 8) * tig + 16 * run;          // byte of the run in a row
        const uint4 kA = *reinterpret_cast<const uint4*>(sk + rA * H::kRow + kb);
        const uint4 kB = *reinterpret_cast<const uint4*>(sk + rB * H::kRow + kb);
        const uint32_t sA =
            e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sks + rA * H::kSfRow + kb / 8));
        const uint32_t sB =
            e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sks + rB * H::kSfRow + kb / 8));
        scA[gi][0] = prmt(sA, 0, 0x1010); scA[gi][1] = prmt(sA, 0, 0x3232);
        scB[gi][0] = prmt(sB, 0, 0x1010); scB[gi][1] = prmt(sB, 0, 0x3232);
        wA[gi][0] = kA.x; wA[gi][1] = kA.y; wA[gi][2] = kA.z; wA[gi][3] = kA.w;
        wB[gi][0] = kB.x; wB[gi][1] = kB.y; wB[gi][2] = kB.z; wB[gi][3] = kB.w;
      }
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        uint32_t fa[2][4], fb[2][4];
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
          e2m1x8_to_f16x2x4(wA[gi][wd], fa[gi]);
          e2m1x8_to_f16x2x4(wB[gi][wd], fb[gi]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int kk = 8 * run + 2 * wd + h;
#pragma unroll
          for (int gi = 0; gi < 2; ++gi) {
            const uint32_t sa = scA[gi][wd >> 1], sb = scB[gi][wd >> 1];
            uint32_t a[4];
            a[0] = hmul2_u32(fa[gi][2 * h], sa);
            a[2] = hmul2_u32(fa[gi][2 * h + 1], sa);
            a[1] = hmul2_u32(fb[gi][2 * h], sb);
            a[3] = hmul2_u32(fb[gi][2 * h + 1], sb);
#pragma unroll
            for (int nt = 0; nt < NTR; ++nt)
              mma_f16_16816(sacc[m0 + gi][nt], a, qf[nt][2 * kk], qf[nt][2 * kk + 1]);
          }
        }
      }
    }
  }

  // ---- logits, causal mask, chunk max --------------------------------
  float cmax[NTR][2];
#pragma unroll
  for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) cmax[nt][e] = -INFINITY;
#pragma unroll
  for (int mt = 0; mt < kMt; ++mt) {
    const int tA = tok0 + 16 * mt + (gid >> 1) + 4 * (gid & 1);
    const int tB = tA + 8;
#pragma unroll
    for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float zA = sacc[mt][nt][e] * cq[nt][e];
        float zB = sacc[mt][nt][2 + e] * cq[nt][e];
        if (partial) {
          if (tA >= nrow) zA = -INFINITY;
          if (tB >= nrow) zB = -INFINITY;
        }
        sacc[mt][nt][e] = zA;
        sacc[mt][nt][2 + e] = zB;
        cmax[nt][e] = fmaxf(cmax[nt][e], fmaxf(zA, zB));
      }
  }
#pragma unroll
  for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = cmax[nt][e];
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
      cmax[nt][e] = v;
    }

  // ---- online softmax update -----------------------------------------
  float base[NTR][2];
  bool rescale = false;
#pragma unroll
  for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float mn = fmaxf(m_run[nt][e], cmax[nt][e]);
      rescale |= (mn != m_run[nt][e]) && (m_run[nt][e] != -INFINITY);
      base[nt][e] = (mn == -INFINITY) ? 0.f : mn;
    }
  if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
    for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float alpha = exp2f(m_run[nt][e] - base[nt][e]);
        l_run[nt][e] *= alpha;
#pragma unroll
        for (int dt = 0; dt < H::kDt; ++dt) {
          o_acc[dt][nt][e] *= alpha;
          o_acc[dt][nt][2 + e] *= alpha;
        }
      }
  }
#pragma unroll
  for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) m_run[nt][e] = fmaxf(m_run[nt][e], cmax[nt][e]);

  // P = exp2(z - base) -> fp16 -> transposed B fragments for P^T.
#pragma unroll
  for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
    for (int nt = 0; nt < NTR; ++nt) {
      const float p0 = exp2f(sacc[mt][nt][0] - base[nt][0]);
      const float p1 = exp2f(sacc[mt][nt][1] - base[nt][1]);
      const float p2 = exp2f(sacc[mt][nt][2] - base[nt][0]);
      const float p3 = exp2f(sacc[mt][nt][3] - base[nt][1]);
      l_run[nt][0] += p0 + p2;
      l_run[nt][1] += p1 + p3;
      pf[mt][nt][0] = movmatrix_trans(pack_half2(p0, p1));
      pf[mt][nt][1] = movmatrix_trans(pack_half2(p2, p3));
    }
}

template <int NTR, int D>
__device__ __forceinline__ void consume_pv(const uint8_t* __restrict__ sk,
                                           const uint32_t (&pf)[Hd<D>::kMt][NTR][2],
                                           float (&o_acc)[D / 16][NTR][4]) {
  using H = Hd<D>;
  constexpr int kMt = H::kMt;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const uint8_t* sv = sk + H::kKBytes;
  const uint8_t* svs = sk + 2 * H::kKBytes + H::kSfBytes;

  // ---- O^T += V^T . P^T over the 16-dim tiles -------------------------
#pragma unroll
  for (int ks = 0; ks < kMt; ++ks) {
    const int t0 = 16 * ks + tig;
#pragma unroll
    for (int run = 0; run < H::kRuns; ++run) {
      // scale block of bytes [D/16 * gid + 8 * run, +8) of the four token rows
      const int blk = (D / 128) * gid + run;
      const uint32_t sv01 = e4m3x2_to_f16x2((uint32_t)svs[t0 * H::kSfRow + blk] |
                                            ((uint32_t)svs[(t0 + 4) * H::kSfRow + blk] << 8));
      const uint32_t sv23 = e4m3x2_to_f16x2((uint32_t)svs[(t0 + 8) * H::kSfRow + blk] |
                                            ((uint32_t)svs[(t0 + 12) * H::kSfRow + blk] << 8));
#pragma unroll
      for (int w4 = 0; w4 < 2; ++w4) {
        // bytes [D/16 * gid + 8 * run + 4 * w4, +4) of the four token rows
        const int boff = (D / 16) * gid + 8 * run + 4 * w4;
        const uint32_t X = *reinterpret_cast<const uint32_t*>(sv + t0 * H::kRow + boff);
        const uint32_t Y = *reinterpret_cast<const uint32_t*>(sv + (t0 + 4) * H::kRow + boff);
        const uint32_t X2 = *reinterpret_cast<const uint32_t*>(sv + (t0 + 8) * H::kRow + boff);
        const uint32_t Y2 = *reinterpret_cast<const uint32_t*>(sv + (t0 + 12) * H::kRow + boff);
        const uint32_t LO = (X & 0x0F0F0F0Fu) | ((Y << 4) & 0xF0F0F0F0u);
        const uint32_t HI = ((X >> 4) & 0x0F0F0F0Fu) | (Y & 0xF0F0F0F0u);
        const uint32_t LO2 = (X2 & 0x0F0F0F0Fu) | ((Y2 << 4) & 0xF0F0F0F0u);
        const uint32_t HI2 = ((X2 >> 4) & 0x0F0F0F0Fu) | (Y2 & 0xF0F0F0F0u);
        uint32_t f0[4], f1[4], f2[4], f3[4];
        e2m1x8_to_f16x2x4(LO, f0);
        e2m1x8_to_f16x2x4(HI, f1);
        e2m1x8_to_f16x2x4(LO2, f2);
        e2m1x8_to_f16x2x4(HI2, f3);
#pragma unroll
        for (int bi = 0; bi < 4; ++bi) {
          const int dt = 8 * run + 4 * w4 + bi;
          uint32_t a[4];
          a[0] = hmul2_u32(f0[bi], sv01);
          a[1] = hmul2_u32(f1[bi], sv01);
          a[2] = hmul2_u32(f2[bi], sv23);
          a[3] = hmul2_u32(f3[bi], sv23);
#pragma unroll
          for (int nt = 0; nt < NTR; ++nt)
            mma_f16_16816(o_acc[dt][nt], a, pf[ks][nt][0], pf[ks][nt][1]);
        }
      }
    }
  }
}

template <int NTR, int D>
__device__ __forceinline__ void consume_chunk(const uint8_t* __restrict__ sk, int tok0, int nrow,
                                              const uint32_t (&qf)[NTR][D / 8],
                                              const float (&cq)[NTR][2], float (&m_run)[NTR][2],
                                              float (&l_run)[NTR][2],
                                              float (&o_acc)[D / 16][NTR][4]) {
  uint32_t pf[Hd<D>::kMt][NTR][2];
  consume_qk<NTR, D>(sk, tok0, nrow, qf, cq, m_run, l_run, o_acc, pf);
  consume_pv<NTR, D>(sk, pf, o_acc);
}

template <int NTR, int W, int S, bool ONE, int D>
__global__ void __launch_bounds__(Layout<NTR, W, S, ONE, D>::kThreads,
                                  (decode_min_blocks<NTR, W, ONE, D>()))
sparse_decode_kernel(Params p) {
  using Lay = Layout<NTR, W, S, ONE, D>;
  using H = Hd<D>;
  constexpr int kPartStride = H::kPartStride;
  constexpr int kChunk = H::kChunk;
  constexpr int kHsp = Lay::kHsp;
  constexpr int kWarps = Lay::kWarps;
  constexpr int kThreads = Lay::kThreads;
  static_assert(!ONE || S % W == 0, "a single-row stage must always belong to one consumer");

  const Geom& g = p.g;
  const int R = g.R;
  const int G = g.Hq / g.Hkv;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const bool producer = !ONE && warp == W;
  // A CTA takes RC consecutive rows of its request (all R rows, except for
  // self-issued variants with fewer warps than rows: RC = W, one warp per
  // row, and the request's rows are spread over R / RC CTAs).  Self-issued
  // (ONE) variants: warp w owns row w % RC and, of that row's chunks of this
  // split, every (W / RC)-th starting at the (w / RC)-th; it lists, requests
  // and consumes them itself.  Union variants: a producer warp streams the
  // union and consumer w owns row w % R.
  const int RC = rows_per_cta(ONE, W, R);
  const int nrg = R / RC;                       // row groups per request
  const int gper = W / RC;                      // consumers per row
  const int jw = warp % RC;                     // the row (of the CTA's) this warp owns
  const int gw = warp / RC;

  const int s = blockIdx.x;                           // KV split (= cluster rank)
  const int kvh = blockIdx.y / p.slices, slice = blockIdx.y % p.slices;
  const int b = blockIdx.z / nrg;
  const int rgi = blockIdx.z - b * nrg;               // row group of the request
  const int r0 = rgi * RC;                            // its first row
  const int hs0 = slice * kHsp;                       // first head of the slice
  const int hs = min(kHsp, G - hs0);                  // real heads in the slice
  const int ncols = RC * kHsp;                        // padded columns (j, hh)
  const int k = p.k;

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* region = smem;
  size_t off = (size_t)Lay::region_bytes(RC, k, p.splits);
  float* rb = reinterpret_cast<float*>(region + Lay::rb_off(RC));   // cluster merge receive buffer
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + off);
  uint64_t* empty = full + S;
  off += 2 * S * 8;
  // The fp16 query tile sits in the stage region: every warp takes its
  // fragments into registers before the region is first written.
  __half* qs = reinterpret_cast<__half*>(region);
  float* col_cq = reinterpret_cast<float*>(smem + off);
  int* col_n = reinterpret_cast<int*>(col_cq + ncols);
  off += (size_t)ncols * 4 * 2;
  int* misc = reinterpret_cast<int*>(smem + off);
  off += 64 * 4;
  int32_t* s_sel = reinterpret_cast<int32_t*>(smem + off);
  int32_t* s_union = s_sel + RC * k;                  // (union variants: RC = R)
  int32_t* s_upage = s_union + RC * k;
  int32_t* s_scan = s_upage + RC * k;                 // [R * k + 1]
  const int list_ints = ONE ? W * 2 * decode_list_cap(k, p.splits, gper) + k : 0;
  int32_t* s_pt = s_sel + (ONE ? list_ints : RC * k * 4 + 4);

  // full[st]: one arrival (the copy issuer) plus the copies' bytes.  empty[st]
  // (verify only): every row consumer arrives, so stage reuse waits for all.
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      // ONE: empty[st] is the V half's full barrier (see the consumers).
      mbar_init(&empty[i], ONE ? 1 : W);
    }
    fence_mbar_init();
  }

  // ---- before the dependency wait: what does not depend on the selection ---
  // The queries, the request's page-table row and its length are step inputs
  // that no kernel of the step writes; the selection kernel triggers its
  // dependents only after its own wait returned, so they are complete here.
  const bool pt_in_smem = g.MB <= kPtRowMax;
  if (pt_in_smem)
    for (int i = tid; i < g.MB; i += kThreads) s_pt[i] = p.page_table[(size_t)b * g.MB + i];
  const int L = p.seqlens[b];
  const int cap = g.MB * g.P;
  {
    // Queries -> fp16 pre-scaled by a power of two per column, one warp per
    // column.  The scale maps |q|max into [256, 512): exact, and keeps bf16
    // queries of any magnitude inside fp16 range.  2^sq and its inverse are
    // built from exponent bits (|sq| <= 126 keeps both normal).
    // Lane holds D/32 consecutive dims (4 or 8), read as D/128 8-byte words.
    // Columns in passes of kQPerWarp per warp (one pass for decode rows).
    constexpr int kQPerWarp = ONE ? (kHsp + kWarps - 1) / kWarps : (kMaxRows * kHsp + kWarps - 1) / kWarps;
    constexpr int kQw = D / 128;
    for (int cb = 0; cb < ncols; cb += kQPerWarp * kWarps) {
    uint2 raw[kQPerWarp][kQw];
#pragma unroll
    for (int ci = 0; ci < kQPerWarp; ++ci) {
      const int c = cb + warp + ci * kWarps;
#pragma unroll
      for (int u = 0; u < kQw; ++u) raw[ci][u] = make_uint2(0u, 0u);
      if (c < ncols && (c % kHsp) < hs) {
        const int j = c / kHsp;
        const int h = kvh * G + hs0 + c % kHsp;
        const uint2* src = reinterpret_cast<const uint2*>(
            p.q + ((size_t)(b * R + r0 + j) * g.Hq + h) * D + lane * (D / 32));
#pragma unroll
        for (int u = 0; u < kQw; ++u) raw[ci][u] = src[u];
      }
    }
#pragma unroll
    for (int ci = 0; ci < kQPerWarp; ++ci) {
      const int c = cb + warp + ci * kWarps;
      if (c >= ncols) break;
      float v[4 * kQw];
#pragma unroll
      for (int u = 0; u < kQw; ++u) {
        const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw[ci][u].x);
        const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw[ci][u].y);
        v[4 * u + 0] = __low2float(lo); v[4 * u + 1] = __high2float(lo);
        v[4 * u + 2] = __low2float(hi); v[4 * u + 3] = __high2float(hi);
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 4 * kQw; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
      for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const int ebits = (int)((__float_as_uint(amax) >> 23) & 0xFF);
      int sq = (amax > 0.f) ? 135 - ebits : 0;
      sq = sq > 126 ? 126 : (sq < -126 ? -126 : sq);
      const float up = __uint_as_float((uint32_t)(sq + 127) << 23);
      const float down = __uint_as_float((uint32_t)(127 - sq) << 23);
      __half2* dst = reinterpret_cast<__half2*>(qs + c * D + lane * (D / 32));
#pragma unroll
      for (int i = 0; i < 2 * kQw; ++i) dst[i] = __floats2half2_rn(v[2 * i] * up, v[2 * i + 1] * up);
      if (lane == 0) {
        col_cq[c] = ((c % kHsp) < hs) ? p.k_scale * p.sm_scale * kLog2e * down : 0.f;
        col_n[c] = visible_tokens(L, R, r0 + c / kHsp, cap);
      }
    }
    }
  }

  __syncthreads();   // barriers, page-table row and queries visible to every warp

  // Each consumer's query fragments and column constants, into registers.
  const int cbase = jw * kHsp;
  float cq[NTR][2];
  int nrow = 0;                                 // tokens this row sees
  // Q^T fragments: column nt*8+gid of the row, dims [D/4*tig, D/4*(tig+1)).
  uint32_t qf[NTR][D / 8];
  if (!producer) {
#pragma unroll
    for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) cq[nt][e] = col_cq[cbase + nt * 8 + 2 * tig + e];
    nrow = col_n[cbase];
#pragma unroll
    for (int nt = 0; nt < NTR; ++nt) {
      const uint4* src =
          reinterpret_cast<const uint4*>(qs + (cbase + nt * 8 + gid) * D + (D / 4) * tig);
#pragma unroll
      for (int v4 = 0; v4 < D / 32; ++v4) {
        const uint4 x = src[v4];
        qf[nt][4 * v4 + 0] = x.x; qf[nt][4 * v4 + 1] = x.y;
        qf[nt][4 * v4 + 2] = x.z; qf[nt][4 * v4 + 3] = x.w;
      }
    }
  }
  __syncthreads();   // the query tile (in the stage region) is no longer read
  pdl_wait();        // the selections come from the preceding kernel

  const int csh = (g.P == 2 * kChunk) ? 1 : 0;  // stages per page: 1 << csh
  // Self-issued: each warp lists its own chunks straight from its row's
  // selection (no union and no CTA-wide barrier before the first copies).
  // Candidate chunk c of the row (entry c >> csh, part c & csh) belongs to
  // split c mod splits and, within it, to the row's warp (c / splits) mod
  // (W / R).  An entry equal to its predecessor (the selection is ascending)
  // or on an invalid page is dropped.
  const int wcap = ONE ? decode_list_cap(k, p.splits, gper) : 0;
  int* wl = s_sel + warp * 2 * wcap;            // (page, tok0) pairs
  int wcnt = 0;
  if constexpr (ONE) {
    const int nc = k << csh;
    const int32_t* selrow = p.sel + (size_t)(b * R + r0 + jw) * k;
    if (p.scores) {
      // Fused selection (one row per request): this CTA selects its row from
      // the scores, with the (still idle) stage region as the selection's
      // scratch.
      int32_t* s_row = s_sel + W * 2 * wcap;
      const int n = visible_tokens(L, 1, 0, cap);
      select_row<kThreads>(p.scores + (size_t)b * g.MB, (n + g.P - 1) / g.P, p.window, k, s_row,
                           misc + 20, region);
      __syncthreads();   // the row is complete and the scratch is free
      if (s == 0 && kvh == 0 && slice == 0) {
        for (int i = tid; i < k; i += kThreads) p.sel_out[(size_t)b * k + i] = s_row[i];
        if (tid == 0) p.nsel_out[b] = misc[20];
      }
      selrow = s_row;
    }
    for (int t0 = 0;; t0 += 32) {
      if (s + (long long)p.splits * (gw + (long long)gper * t0) >= nc) break;
      const long long c = s + (long long)p.splits * (gw + (long long)gper * (t0 + lane));
      int page = -1, tok0 = 0;
      if (c < nc) {
        const int e = (int)(c >> csh);
        const int beta = selrow[e];
        const int prev = e > 0 ? selrow[e - 1] : -1;
        if (beta >= 0 && beta < g.MB && beta != prev) {
          const int pg = pt_in_smem ? s_pt[beta] : p.page_table[(size_t)b * g.MB + beta];
          if (pg >= 0 && pg < g.NP) {
            page = pg;
            tok0 = beta * g.P + (int)(c & csh) * kChunk;
          }
        }
      }
      const unsigned vm = __ballot_sync(0xffffffffu, page >= 0);
      if (page >= 0) {
        const int q = wcnt + __popc(vm & ((1u << lane) - 1u));
        if (QSA_IN_BOUNDS(q < wcap, kChkList)) {
          wl[2 * q] = page;
          wl[2 * q + 1] = tok0;
        }
      }
      wcnt += __popc(vm);
    }
    __syncwarp();
  } else {
  for (int i = tid; i < R * k; i += kThreads) {
    const int v = p.sel[(size_t)b * R * k + i];
    s_sel[i] = (v >= 0 && v < g.MB) ? v : -1;
  }
  __syncthreads();

  // ---- union of the rows' selections: distinct valid pages, ascending ------
  // Entry e = (row jj, block beta) is kept when no earlier row holds beta and
  // its page is valid; its mask marks every row that holds beta.  Rows are
  // ascending (padding last), so a kept entry's union position is the number
  // of kept entries, over all rows, with smaller blocks: per row, a prefix
  // count of kept entries up to the binary-search bound.  The union is thus
  // in block order and each row's pages spread across the whole of it.
  // Each thread takes a contiguous run of entries; flags and pages wait in
  // the (still idle) stage region.  Verify rows whose page-table row fits in
  // shared memory use a per-block row mask instead (below).
  if (!ONE && pt_in_smem) {
    // Row mask per block (one byte per block, four per word): every entry
    // ors its row bit in; the union is then the blocks with a mask and a
    // valid page, compacted in block order.
    uint32_t* s_rm = reinterpret_cast<uint32_t*>(region);   // [ceil(MB / 4)]
    const int nw = (g.MB + 3) >> 2;
    for (int i = tid; i < nw; i += kThreads) s_rm[i] = 0u;
    __syncthreads();
    const int ne = R * k;
    const int per_e = (ne + kThreads - 1) / kThreads;
    const int e_lo = min(ne, tid * per_e), e_hi = min(ne, e_lo + per_e);
    for (int e = e_lo, jj = e_lo / k, ii = e_lo - (e_lo / k) * k; e < e_hi; ++e) {
      const int beta = s_sel[e];
      if (beta >= 0) atomicOr(&s_rm[beta >> 2], (1u << jj) << (8 * (beta & 3)));
      if (++ii == k) { ii = 0; ++jj; }
    }
    __syncthreads();
    const uint8_t* rm = reinterpret_cast<const uint8_t*>(s_rm);
    const int per_b = (g.MB + kThreads - 1) / kThreads;
    const int b_lo = min(g.MB, tid * per_b), b_hi = min(g.MB, b_lo + per_b);
    int cnt = 0;
    for (int beta = b_lo; beta < b_hi; ++beta) {
      const int page = s_pt[beta];
      cnt += (rm[beta] != 0 && page >= 0 && page < g.NP) ? 1 : 0;
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) misc[warp] = x;
    __syncthreads();
    int pos = x - cnt;
    for (int w = 0; w < warp; ++w) pos += misc[w];
    for (int beta = b_lo; beta < b_hi; ++beta) {
      const int mask = rm[beta];
      const int page = s_pt[beta];
      if (mask != 0 && page >= 0 && page < g.NP && QSA_IN_BOUNDS(pos < R * k, kChkUnion)) {
        s_union[pos] = beta | (mask << 24);
        s_upage[pos] = page;
        ++pos;
      }
    }
    if (tid == kThreads - 1) s_scan[R * k] = pos;   // the last thread's end is the total
  } else {
    const int ne = R * k;
    const int per = (ne + kThreads - 1) / kThreads;
    const int e_lo = min(ne, tid * per), e_hi = min(ne, e_lo + per);
    int32_t* t_flag = reinterpret_cast<int32_t*>(region);   // [ne]
    int32_t* t_page = t_flag + ne;                          // [ne]
    // lower bound of beta in row j2 (padding counts as +inf)
    auto lower = [&](int j2, int beta) {
      const int32_t* row = s_sel + j2 * k;
      int lo2 = 0, hi2 = k;
      while (lo2 < hi2) {
        const int mid = (lo2 + hi2) >> 1;
        const int x = row[mid] < 0 ? 0x7FFFFFFF : row[mid];
        if (x < beta) lo2 = mid + 1; else hi2 = mid;
      }
      return lo2;
    };
    const int jj0 = e_lo / k, ii0 = e_lo - jj0 * k;
    int keep_cnt = 0;
    for (int e = e_lo, jj = jj0, ii = ii0; e < e_hi; ++e) {
      int flag = 0, page = 0;
      const int beta = s_sel[e];
      if (beta >= 0) {
        bool first = true;
        int mask = 1 << jj;
        if (!ONE) {
          for (int j2 = 0; j2 < R; ++j2) {
            if (j2 == jj) continue;
            const int lb = lower(j2, beta);
            if (lb < k && s_sel[j2 * k + lb] == beta) {
              mask |= 1 << j2;
              if (j2 < jj) first = false;
            }
          }
        }
        if (first) {
          page = pt_in_smem ? s_pt[beta] : p.page_table[(size_t)b * g.MB + beta];
          if (page >= 0 && page < g.NP) {
            flag = 0x100 | (mask & 0xFF);
            ++keep_cnt;
          }
        }
      }
      t_flag[e] = flag;
      t_page[e] = page;
      if (++ii == k) { ii = 0; ++jj; }
    }
    // exclusive prefix of kept entries over the flat entry order
    int x = keep_cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) misc[warp] = x;
    __syncthreads();
    int run = x - keep_cnt;
    for (int w = 0; w < warp; ++w) run += misc[w];
    for (int e = e_lo; e < e_hi; ++e) {
      s_scan[e] = run;
      run += t_flag[e] ? 1 : 0;
    }
    if (tid == kThreads - 1) s_scan[ne] = run;   // the last thread's run is the total
    __syncthreads();
    for (int e = e_lo, jj = jj0, ii = ii0; e < e_hi; ++e) {
      const int flag = t_flag[e];
      if (flag) {
        const int beta = s_sel[e];
        int pos = s_scan[e] - s_scan[jj * k];
        if (!ONE)
          for (int j2 = 0; j2 < R; ++j2)
            if (j2 != jj) pos += s_scan[j2 * k + lower(j2, beta)] - s_scan[j2 * k];
        if (QSA_IN_BOUNDS(pos >= 0 && pos < R * k, kChkUnion)) {
          s_union[pos] = beta | ((flag & 0xFF) << 24);
          s_upage[pos] = t_page[e];
        }
      }
      if (++ii == k) { ii = 0; ++jj; }
    }
  }
  __syncthreads();
  }   // verify union
  pdl_trigger();

  const int U = ONE ? 0 : s_scan[R * k];
  const int C = U << csh;
  // Split s takes union chunks s, s + splits, ... so every split gets an even
  // share of every row's pages.
  const int n_ch = (C > s) ? (C - s + p.splits - 1) / p.splits : 0;

  // Chunks read by one warp only are evicted first; a verify row's chunk may
  // be read again by another row's warp, so self-issued verify copies keep
  // the normal policy.
  const uint64_t pol = ((ONE && R == 1) || producer) ? policy_evict_first()
                                                     : (ONE ? policy_evict_normal() : 0ull);
  // Chunk i of this split into stage i % S (one lane).
  auto issue = [&](int i) {
    const int st = i % S;
    const int c = s + i * p.splits;
    const int u = c >> csh, sub = c & csh;
    if (!QSA_IN_BOUNDS(u < U && s_upage[u] >= 0 && s_upage[u] < g.NP, kChkChunk)) return;
    const size_t row0 = ((size_t)s_upage[u] * g.Hkv + kvh) * g.P + (size_t)sub * kChunk;
    uint8_t* dst = region + st * kStageBytes;
    mbar_arrive_expect_tx(&full[st], kStageBytes);
    bulk_g2s(dst, p.k_pool + row0 * H::kRow, H::kKBytes, &full[st], pol);
    bulk_g2s(dst + H::kKBytes, p.v_pool + row0 * H::kRow, H::kKBytes, &full[st], pol);
    bulk_g2s(dst + 2 * H::kKBytes, p.k_sf + row0 * H::kSfRow, H::kSfBytes, &full[st], pol);
    bulk_g2s(dst + 2 * H::kKBytes + H::kSfBytes, p.v_sf + row0 * H::kSfRow, H::kSfBytes,
             &full[st], pol);
  };

  // ---- producer (verify): stream this split's chunks through the stages ----
  if (producer) {
    if (lane == 0) {
      fence_proxy_async_smem();   // after the union's temporaries in the stage region
      int dead = 0, issued = 0;
      for (int i = 0; i < n_ch; ++i) {
        if (i >= S) {
          if (!wait_bounded(&empty[i % S], ((i / S) - 1) & 1)) {
            dead = 1;
            break;
          }
          fence_proxy_async_smem();   // consumers' reads of the stage come first
        }
        issue(i);
        issued = i + 1;
      }
      if (dead) atomicExch(p.status, kStatusWaitTimeout);
      // Every issued copy lands before the stage memory is reused below (older
      // ones were consumed before their stage was refilled).
      for (int i = max(0, issued - S); i < issued; ++i)
        if (!wait_bounded(&full[i % S], (i / S) & 1)) atomicExch(p.status, kStatusWaitTimeout);
    }
    __syncwarp();
  }

  // ---- consumers -------------------------------------------------------------
  // Decode: consumer w takes chunks w, w + W, ... and itself refills the stage
  // it has just read with its chunk S further on (S % W == 0 keeps a stage
  // with one consumer), so no warp waits on another.  Verify: consumer w owns
  // row w % R and, of the chunks of this split that its row selected, every
  // (W / R)-th starting at the (w / R)-th.
  float m_run[NTR][2], l_run[NTR][2];
  float o_acc[H::kDt][NTR][4];
#pragma unroll
  for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) { m_run[nt][e] = -INFINITY; l_run[nt][e] = 0.f; }
#pragma unroll
  for (int dt = 0; dt < H::kDt; ++dt)
#pragma unroll
    for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o_acc[dt][nt][e] = 0.f;

  // Self-issued: this warp's q-th chunk goes to stage warp + W * (q mod S/W).
  // Its K half (codes and scales) completes on full[st] and its V half on
  // empty[st], so the K half of chunk q + S/W is requested as soon as the
  // logits of chunk q are done, and its V half once P.V is: one stage per
  // warp is then already double-buffered by halves.
  constexpr int kSpw = ONE ? S / W : 1;          // stages per self-issuing warp
  auto chunk_row0 = [&](int q, size_t& row0) -> bool {
    const int page = wl[2 * q], tok0 = wl[2 * q + 1];
    if (!QSA_IN_BOUNDS(q < wcap && page >= 0 && page < g.NP && tok0 >= 0 && tok0 < cap &&
                           (tok0 & (g.P - 1)) + kChunk <= g.P,
                       kChkChunk))
      return false;
    row0 = ((size_t)page * g.Hkv + kvh) * g.P + (size_t)(tok0 & (g.P - 1));
    return true;
  };
  auto issue_k = [&](int q) {
    const int st = warp + W * (q % kSpw);
    size_t row0;
    if (!chunk_row0(q, row0)) return;
    uint8_t* dst = region + st * kStageBytes;
    mbar_arrive_expect_tx(&full[st], H::kKBytes + H::kSfBytes);
    bulk_g2s(dst, p.k_pool + row0 * H::kRow, H::kKBytes, &full[st], pol);
    bulk_g2s(dst + 2 * H::kKBytes, p.k_sf + row0 * H::kSfRow, H::kSfBytes, &full[st], pol);
  };
  auto issue_v = [&](int q) {
    const int st = warp + W * (q % kSpw);
    size_t row0;
    if (!chunk_row0(q, row0)) return;
    uint8_t* dst = region + st * kStageBytes;
    mbar_arrive_expect_tx(&empty[st], H::kKBytes + H::kSfBytes);
    bulk_g2s(dst + H::kKBytes, p.v_pool + row0 * H::kRow, H::kKBytes, &empty[st], pol);
    bulk_g2s(dst + 2 * H::kKBytes + H::kSfBytes, p.v_sf + row0 * H::kSfRow, H::kSfBytes,
             &empty[st], pol);
  };
  const int n_first = ONE ? min(kSpw, wcnt) : 0;
  if (ONE && lane == 0) {
    fence_proxy_async_smem();   // after the fused selection's scratch in the region
    for (int q = 0; q < n_first; ++q) {
      issue_k(q);
      issue_v(q);
    }
  }

  if (!producer) {
    if (ONE) {
      // K and V halves requested so far (chunks [0, nk) and [0, nv)) and the
      // first ones not yet seen complete (a stage has at most one of each in
      // flight: its next half is requested only after this one completed).
      int nk = n_first, nv = n_first, k_seen = 0, v_seen = 0;
      bool dead = false;
      for (int q = 0; q < wcnt; ++q) {
        const int st = warp + W * (q % kSpw);
        const uint32_t ph = (q / kSpw) & 1;
        const uint8_t* stage = region + st * kStageBytes;
        if (!wait_bounded(&full[st], ph)) { dead = true; break; }
        k_seen = q + 1;
        uint32_t pf[H::kMt][NTR][2];
        consume_qk<NTR, D>(stage, wl[2 * q + 1], nrow, qf, cq, m_run, l_run, o_acc, pf);
        __syncwarp();   // every lane's reads of the K half are done
        if (q + kSpw < wcnt) {
          if (lane == 0) {
            fence_proxy_async_smem();
            issue_k(q + kSpw);
          }
          ++nk;
        }
        if (!wait_bounded(&empty[st], ph)) { dead = true; break; }
        v_seen = q + 1;
        consume_pv<NTR, D>(stage, pf, o_acc);
        __syncwarp();   // every lane's reads of the V half are done
        if (q + kSpw < wcnt) {
          if (lane == 0) {
            fence_proxy_async_smem();
            issue_v(q + kSpw);
          }
          ++nv;
        }
      }
      // After a wait gave up, let this warp's copies still in flight land
      // before the stage memory is reused.
      if (dead && lane == 0) {
        atomicExch(p.status, kStatusWaitTimeout);
        for (int q = k_seen; q < nk; ++q)
          if (!wait_bounded(&full[warp + W * (q % kSpw)], (q / kSpw) & 1)) break;
        for (int q = v_seen; q < nv; ++q)
          if (!wait_bounded(&empty[warp + W * (q % kSpw)], (q / kSpw) & 1)) break;
      }
    } else {
      bool dead = false;
      int rc = 0;                               // this row's chunks seen so far
      for (int i = 0; i < n_ch; ++i) {
        const int st = i % S;
        const int c = s + i * p.splits;
        const int ue = s_union[c >> csh];
        const bool rowbit = (ue >> (24 + jw)) & 1;
        const bool mine = rowbit && (rc % gper) == gw;
        rc += rowbit ? 1 : 0;
        if (!dead && !wait_bounded(&full[st], (i / S) & 1)) {
          dead = true;
          if (lane == 0) atomicExch(p.status, kStatusWaitTimeout);
        }
        if (mine && !dead)
          consume_chunk<NTR, D>(region + st * kStageBytes, (ue & 0xFFFFFF) * g.P + (c & csh) * kChunk,
                             nrow, qf, cq, m_run, l_run, o_acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
    }
  }

  // Row sums over the 8 token lanes of the warp.
#pragma unroll
  for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = l_run[nt][e];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l_run[nt][e] = v;
    }

  // ---- combine the consumers of this CTA ------------------------------------
  __syncthreads();   // every copy landed and was consumed: reuse the stage region

  const bool direct = Lay::direct(RC);
  float* co = reinterpret_cast<float*>(region);                  // [W][kHsp][D]
  float* cm = co + W * kHsp * D;                                  // [W][kHsp]
  float* cl = cm + W * kHsp;                                      // [W][kHsp]
  float* cp = reinterpret_cast<float*>(region + Lay::cp_off(RC));  // [ncols][kPartStride]
  if (!producer) {
    // Direct: consumer `warp` is row `warp`'s only consumer, and its state is
    // the CTA partial of the row's columns.
    float* dsto = direct ? cp + (size_t)warp * kHsp * kPartStride + 4 : co + (size_t)warp * kHsp * D;
    const int cstride = direct ? kPartStride : D;
    if (gid == 0) {
#pragma unroll
      for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int cc = nt * 8 + 2 * tig + e;
          if (direct) {
            float* pc = cp + ((size_t)warp * kHsp + cc) * kPartStride;
            pc[0] = (l_run[nt][e] > 0.f) ? m_run[nt][e] : -INFINITY;
            pc[1] = l_run[nt][e];
          } else {
            cm[warp * kHsp + cc] = m_run[nt][e];
            cl[warp * kHsp + cc] = l_run[nt][e];
          }
        }
    }
    // O^T accumulators: dim D/8*gid + 2*dt (+1 for c2/c3), column nt*8+2*tig+e.
#pragma unroll
    for (int dt = 0; dt < H::kDt; ++dt)
#pragma unroll
      for (int nt = 0; nt < NTR; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int cc = nt * 8 + 2 * tig + e;
          *reinterpret_cast<float2*>(dsto + (size_t)cc * cstride + (D / 8) * gid + 2 * dt) =
              make_float2(o_acc[dt][nt][e], o_acc[dt][nt][2 + e]);
        }
  }
  __syncthreads();

  auto store_out = [&](int c, int d4, float4 O, float Lsum, float M) {
    const int j = c / kHsp, hh = c % kHsp;
    if (hh >= hs) return;   // padding column
    const int h = kvh * G + hs0 + hh;
    const size_t orow = (size_t)(b * R + r0 + j) * g.Hq + h;
    if (!QSA_IN_BOUNDS(r0 + j < R && b < g.B && h < g.Hq && d4 + 4 <= D, kChkOut)) return;
    const float sc = Lsum > 0.f ? p.v_scale / Lsum : 0.f;
    __nv_bfloat162 o01 = __floats2bfloat162_rn(O.x * sc, O.y * sc);
    __nv_bfloat162 o23 = __floats2bfloat162_rn(O.z * sc, O.w * sc);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&o01);
    packed.y = *reinterpret_cast<uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(p.out + orow * D + d4) = packed;
    if (d4 == 0) p.lse[orow] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
  };

  if (direct) {
    if (p.splits == 1) {
      for (int idx = tid; idx < ncols * (D / 4); idx += kThreads) {
        const int c = idx / (D / 4), d4 = (idx % (D / 4)) * 4;
        const float* pc = cp + (size_t)c * kPartStride;
        store_out(c, d4, *reinterpret_cast<const float4*>(pc + 4 + d4), pc[1], pc[0]);
      }
    }
  } else {
  // CTA partial per column (j, hh): m (log2 domain, -inf when empty), l, O,
  // merged over the consumers of row j (warps j, j + RC, ...).  With one split
  // it is the result.
  for (int idx = tid; idx < ncols * (D / 4); idx += kThreads) {
    const int c = idx / (D / 4), d4 = (idx % (D / 4)) * 4;
    const int j = c / kHsp, cc = c % kHsp;
    float mv[W];
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      mv[w] = (w % RC == j) ? cm[w * kHsp + cc] : -INFINITY;
      mx = fmaxf(mx, mv[w]);
    }
    const float M = (mx == -INFINITY) ? 0.f : mx;
    float Lsum = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < W; ++w) {
      if (w % RC == j) {
        const float wt = exp2f(mv[w] - M);
        Lsum += cl[w * kHsp + cc] * wt;
        const float4 v =
            *reinterpret_cast<const float4*>(co + ((size_t)w * kHsp + cc) * D + d4);
        O.x += v.x * wt; O.y += v.y * wt; O.z += v.z * wt; O.w += v.w * wt;
      }
    }
    const float Mc = (Lsum > 0.f) ? M : -INFINITY;
    if (p.splits == 1) {
      store_out(c, d4, O, Lsum, Mc);
    } else {
      float* pc = cp + (size_t)c * kPartStride;
      *reinterpret_cast<float4*>(pc + 4 + d4) = O;
      if (d4 == 0) {
        pc[0] = Mc;
        pc[1] = Lsum;
      }
    }
  }
  }
  if (p.splits == 1) return;
  __syncthreads();

  if (p.cluster > 1) {
    // The splits of this unit form one thread-block cluster.  Column c is
    // merged by rank c % CL: every CTA pushes its partial of c into that
    // rank's receive buffer (slot [split][c / CL]), one cluster barrier
    // publishes the writes, and each rank merges its columns from local
    // shared memory in split order (deterministic).
    cg::cluster_group cluster = cg::this_cluster();
    const int CL = p.cluster;
    const int per = (ncols + CL - 1) / CL;
    // The receive buffers live in the stage regions: the first barrier lets
    // every CTA of the cluster finish its main loop before any remote write.
    cluster_arrive_release();
    cluster_wait_acquire();
    for (int idx = tid; idx < ncols * (kPartStride / 4); idx += kThreads) {
      const int c = idx / (kPartStride / 4), w4 = (idx % (kPartStride / 4)) * 4;
      float* dst = cluster.map_shared_rank(rb, c % CL) +
                   ((size_t)s * per + c / CL) * kPartStride + w4;
      *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(cp + c * kPartStride + w4);
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    for (int idx = tid; idx < per * (D / 4); idx += kThreads) {
      const int q = idx / (D / 4), d4 = (idx % (D / 4)) * 4;
      const int c = q * CL + s;
      if (c >= ncols) continue;
      float mr[kMaxCluster];
      float mx = -INFINITY;
#pragma unroll
      for (int r2 = 0; r2 < kMaxCluster; ++r2) {
        mr[r2] = (r2 < CL) ? rb[((size_t)r2 * per + q) * kPartStride] : -INFINITY;
        mx = fmaxf(mx, mr[r2]);
      }
      const float M = (mx == -INFINITY) ? 0.f : mx;
      float Lsum = 0.f;
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r2 = 0; r2 < kMaxCluster; ++r2) {
        if (r2 < CL) {
          const float* pr = rb + ((size_t)r2 * per + q) * kPartStride;
          const float w = exp2f(mr[r2] - M);
          Lsum += pr[1] * w;
          const float4 v = *reinterpret_cast<const float4*>(pr + 4 + d4);
          O.x += v.x * w; O.y += v.y * w; O.z += v.z * w; O.w += v.w * w;
        }
      }
      store_out(c, d4, O, Lsum, M);
    }
    return;
  }

  // Ticket merge: partials go to the workspace; the last split of this
  // (request, KV head, slice) to arrive merges them in split order
  // (deterministic) and resets the ticket.
  const int units_idx = ((b * g.Hkv + kvh) * p.slices + slice) * nrg + rgi;
  if (!QSA_IN_BOUNDS(b < g.B && kvh < g.Hkv && slice < p.slices && s < p.splits, kChkUnit))
    return;
  const size_t split_floats = (size_t)ncols * kPartStride;
  float* part = p.partials + ((size_t)units_idx * p.splits + s) * split_floats;
  for (int idx = tid; idx < ncols * (kPartStride / 4); idx += kThreads)
    reinterpret_cast<float4*>(part)[idx] = reinterpret_cast<const float4*>(cp)[idx];
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&p.tickets[units_idx], 1);
    misc[17] = (prev == p.splits - 1);
  }
  __syncthreads();
  if (!misc[17]) return;
  __threadfence();

  // Merge: per-column max and weights first, then float4 sums over splits.
  const float* parts = p.partials + (size_t)units_idx * p.splits * split_floats;
  float* wsplit = reinterpret_cast<float*>(region);                 // [ncols][splits]
  float* lcol = wsplit + (size_t)ncols * p.splits;                  // [ncols]
  float* mcol = lcol + ncols;                                       // [ncols]
  for (int c = warp; c < ncols; c += kWarps) {
    float mloc = -INFINITY;
    for (int t = lane; t < p.splits; t += 32)
      mloc = fmaxf(mloc, __ldcg(parts + t * split_floats + (size_t)c * kPartStride));
#pragma unroll
    for (int o = 16; o; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    const float base = (mloc == -INFINITY) ? 0.f : mloc;
    float lsum = 0.f;
    for (int t = lane; t < p.splits; t += 32) {
      const float* pc = parts + t * split_floats + (size_t)c * kPartStride;
      const float wgt = exp2f(__ldcg(pc) - base);
      wsplit[c * p.splits + t] = wgt;
      lsum += __ldcg(pc + 1) * wgt;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    if (lane == 0) {
      lcol[c] = lsum;
      mcol[c] = base;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < ncols * (D / 4); idx += kThreads) {
    const int c = idx / (D / 4), d4 = (idx % (D / 4)) * 4;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    const float* src = parts + (size_t)c * kPartStride + 4 + d4;
    const float* wrow = wsplit + c * p.splits;
    int t = 0;
    for (; t + 4 <= p.splits; t += 4) {
      float4 v[4];
#pragma unroll
      for (int u2 = 0; u2 < 4; ++u2)
        v[u2] = __ldcg(reinterpret_cast<const float4*>(src + (t + u2) * split_floats));
#pragma unroll
      for (int u2 = 0; u2 < 4; ++u2) {
        const float wgt = wrow[t + u2];
        O.x += v[u2].x * wgt; O.y += v[u2].y * wgt; O.z += v[u2].z * wgt; O.w += v[u2].w * wgt;
      }
    }
    for (; t < p.splits; ++t) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(src + t * split_floats));
      const float wgt = wrow[t];
      O.x += v.x * wgt; O.y += v.y * wgt; O.z += v.z * wgt; O.w += v.w * wgt;
    }
    store_out(c, d4, O, lcol[c], mcol[c]);
  }
  if (tid == 0) atomicExch(&p.tickets[units_idx], 0);
}

constexpr size_t kWsHeader = 256;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int NTR, int W, int S, bool ONE, int D>
cudaLaunchConfig_t make_config(dim3 grid, size_t smem, cudaStream_t stream,
                               cudaLaunchAttribute* attr, bool pdl, int cluster) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Layout<NTR, W, S, ONE, D>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cfg;
}

// Whether a cluster of `cl` CTAs of this variant can be resident at all.
template <int NTR, int W, int S, bool ONE, int D>
bool cluster_fits(int cl, size_t smem, dim3 grid) {
  struct Entry { int dev, cl; size_t smem; bool ok; };
  static std::mutex mu;
  static std::vector<Entry> cache;
  if (cl < 2 || cl > kMaxCluster) return false;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
      if (e.dev == dev && e.cl == cl && e.smem == smem) return e.ok;
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_config<NTR, W, S, ONE, D>(grid, smem, 0, attr, false, cl);
  int n = 0;
  const bool ok = cudaOccupancyMaxActiveClusters(&n, sparse_decode_kernel<NTR, W, S, ONE, D>,
                                                 &cfg) == cudaSuccess && n > 0;
  cudaGetLastError();
  std::lock_guard<std::mutex> lock(mu);
  cache.push_back({dev, cl, smem, ok});
  return ok;
}

template <int NTR, int W, int S, bool ONE, int D>
cudaError_t launch_t(Params prm, dim3 grid, int R, int k, int mb, bool pdl,
                     cudaStream_t stream) {
  const size_t smem = Layout<NTR, W, S, ONE, D>::bytes(R, k, mb, prm.splits);
  cudaError_t e = cudaFuncSetAttribute(sparse_decode_kernel<NTR, W, S, ONE, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  prm.cluster = 1;
  if (prm.splits > 1 && cluster_fits<NTR, W, S, ONE, D>(prm.splits, smem, grid))
    prm.cluster = prm.splits;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg =
      make_config<NTR, W, S, ONE, D>(grid, smem, stream, attr, pdl, prm.cluster);
  return cudaLaunchKernelEx(&cfg, sparse_decode_kernel<NTR, W, S, ONE, D>, prm);
}

// Resident CTAs per SM of a variant, for split sizing.
template <int NTR, int W, int S, bool ONE, int D>
int resident_ctas(int R, int k, int mb, int splits) {
  const size_t smem = Layout<NTR, W, S, ONE, D>::bytes(R, k, mb, splits);
  cudaFuncSetAttribute(sparse_decode_kernel<NTR, W, S, ONE, D>,
                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sparse_decode_kernel<NTR, W, S, ONE, D>,
                                                    Layout<NTR, W, S, ONE, D>::kThreads,
                                                    smem) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  return n < 1 ? 1 : n;
}

// Variant by (tiles per row, rows, head_dim).  Self-issued variants (ONE =
// true): W warps, each owning one row (two per row for two-row requests at
// head_dim 128), S / W stages per warp; decode rows at head_dim 256 use four
// warps per row.  Built with QSA_VERIFY_UNION, verify rows run the union
// variants instead (ONE = false: a producer warp streams the union of the
// rows' chunks through S stages, W / R consumers per row take the chunks
// their row selected), kept for comparison.
#ifndef QSA_DECODE_STAGES_R1
#define QSA_DECODE_STAGES_R1 8
#endif
#ifndef QSA_DECODE_WARPS_R1
#define QSA_DECODE_WARPS_R1 8
#endif
#ifndef QSA_DECODE_STAGES_RN
#define QSA_DECODE_STAGES_RN 4
#endif
#ifndef QSA_VERIFY_STAGES_PER_WARP
#define QSA_VERIFY_STAGES_PER_WARP 1
#endif
// Warps per verify CTA (0 = one per row, two per row for two-row requests at
// head_dim 128; n > 0 = n warps, one row each, the request's rows spread over
// R / n CTAs where n divides R).
#ifndef QSA_VERIFY_CTA_WARPS
#define QSA_VERIFY_CTA_WARPS 0
#endif
#define QSA_VSPW QSA_VERIFY_STAGES_PER_WARP
#define QSA_VW(R_, DEF_) \
  ((QSA_VERIFY_CTA_WARPS > 0 && (R_) % (QSA_VERIFY_CTA_WARPS > 0 ? QSA_VERIFY_CTA_WARPS : 1) == 0) \
       ? QSA_VERIFY_CTA_WARPS                                                        \
       : (DEF_))
#ifdef QSA_VERIFY_UNION
#define QSA_V128(NTR_, R_, DEF_) X(NTR_, R_, (R_) == 2 ? 4 : (R_), QSA_DECODE_STAGES_RN, false, 128)
#define QSA_V256(R_, W_) X(1, R_, W_, QSA_DECODE_STAGES_RN, false, 256)
#else
#define QSA_V128(NTR_, R_, DEF_) \
  X(NTR_, R_, QSA_VW(R_, DEF_), QSA_VW(R_, DEF_) * QSA_VSPW, true, 128)
#define QSA_V256(R_, W_) X(1, R_, QSA_VW(R_, R_), QSA_VW(R_, R_) * QSA_VSPW, true, 256)
#endif
#define QSA_DECODE_VARIANTS(X)                                                        \
  X(1, 1, QSA_DECODE_WARPS_R1, QSA_DECODE_STAGES_R1, true, 128)                       \
  X(2, 1, QSA_DECODE_WARPS_R1, QSA_DECODE_STAGES_R1, true, 128)                       \
  QSA_V128(1, 2, 4) QSA_V128(2, 2, 4) QSA_V128(1, 3, 3) QSA_V128(2, 3, 3)             \
  QSA_V128(1, 4, 4) QSA_V128(2, 4, 4) QSA_V128(1, 5, 5) QSA_V128(2, 5, 5)             \
  QSA_V128(1, 6, 6) QSA_V128(2, 6, 6) QSA_V128(1, 7, 7) QSA_V128(2, 7, 7)             \
  QSA_V128(1, 8, 8) QSA_V128(2, 8, 8)                                                 \
  X(1, 1, 4, 8, true, 256)                                                            \
  QSA_V256(2, 4) QSA_V256(3, 6) QSA_V256(4, 4) QSA_V256(5, 5) QSA_V256(6, 6)          \
  QSA_V256(7, 7) QSA_V256(8, 8)

int tiles_per_row(const Geom& g) {
  const int G = g.Hq / g.Hkv;
  return (G <= 8 || g.D != 128) ? 1 : 2;
}

int stage_tokens(const Geom& g) { return 8192 / g.D; }

// Rows per CTA of the variant that serves (tiles per row, R, D).
int variant_rows(int ntr, int R, int d) {
#define X(NTR_, R_, W_, S_, ONE_, D_) \
  if (ntr == NTR_ && R == R_ && d == D_) return rows_per_cta(ONE_, W_, R_);
  QSA_DECODE_VARIANTS(X)
#undef X
  return R;
}

int variant_resident(int ntr, int R, int d, int k, int mb, int splits) {
  const int rc = variant_rows(ntr, R, d);
#define X(NTR_, R_, W_, S_, ONE_, D_) \
  if (ntr == NTR_ && R == R_ && d == D_) return resident_ctas<NTR_, W_, S_, ONE_, D_>(rc, k, mb, splits);
  QSA_DECODE_VARIANTS(X)
#undef X
  return 1;
}

}  // namespace

// The per-row-warp variant (head_dim 256) can select its row itself when the
// selection's scratch fits in its stage region; head_dim 128 runs the shared-
// dequantisation kernel, which reads a finished selection.
bool decode_can_fuse_select(const Geom& g) {
  if (g.R != 1 || attend_supports(g)) return false;
  const int ntr = tiles_per_row(g);
#define X(NTR_, R_, W_, S_, ONE_, D_)                                                 \
  if (ONE_ && ntr == NTR_ && R_ == 1 && g.D == D_)                                      \
    return select_row_smem<Layout<NTR_, W_, S_, ONE_, D_>::kThreads>(g.MB) <=           \
           (size_t)Layout<NTR_, W_, S_, ONE_, D_>::kStagesSz;
  QSA_DECODE_VARIANTS(X)
#undef X
  return false;
}

DecodePlan plan_legacy_decode(const Geom& g, int k, int num_splits) {
  DecodePlan pl;
  const int G = g.Hq / g.Hkv;
  const int ntr = tiles_per_row(g);
  pl.qgroups = (G + 8 * ntr - 1) / (8 * ntr);           // head slices per KV head
  const int rc = variant_rows(ntr, g.R, g.D);            // rows per CTA
  pl.cols = rc * 8 * ntr;                                // padded columns per CTA
  // units: (request, KV head, head slice, row group)
  const long long units = (long long)g.B * g.Hkv * pl.qgroups * (g.R / rc);
  const int max_union = min(g.R * k, g.MB);
  const int max_chunks = max(1, max_union * (g.P / stage_tokens(g)));
  int splits = num_splits;
  if (splits <= 0) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaGetLastError();
    const int resident = variant_resident(ntr, g.R, g.D, k, g.MB, kMaxCluster);
    const long long slots = (long long)sms * resident;
    // One wave: the most splits up to a portable cluster (whose splits
    // merge in distributed shared memory) with units * splits within
    // the resident CTA slots.  Each CTA carries a fixed cost (prologue, union,
    // merge), so more waves of smaller CTAs lose.  Only when even a full
    // cluster per unit fills under a quarter of the slots (a handful of
    // requests) do more splits, merged by ticket, pay.
    splits = 1;
    while (splits + 1 <= kMaxCluster && units * (splits + 1) <= slots) ++splits;
    if (units * kMaxCluster * 4 < slots) splits = (int)min(64LL, slots / units);
    splits = min(splits, max(1, max_chunks / 2));
    splits = max(1, splits);
  }
  pl.splits = splits;
  size_t ws = kWsHeader + align256((size_t)units * sizeof(int));
  if (splits > 1) ws += (size_t)units * splits * pl.cols * (4 + g.D) * sizeof(float);
  pl.ws_bytes = ws;
  return pl;
}

cudaError_t launch_legacy_decode(const Geom& g, const DecodePlan& plan, const void* q,
                                 const uint8_t* k_pool, const uint8_t* k_sf,
                                 const uint8_t* v_pool, const uint8_t* v_sf, float k_scale,
                                 float v_scale, float sm_scale, const int32_t* page_table,
                                 const int32_t* seqlens, const int32_t* sel, int k, void* out,
                                 float* lse, void* workspace, bool pdl, cudaStream_t stream,
                                 const int32_t* scores, int window, int32_t* sel_out,
                                 int32_t* nsel_out) {
  Params prm;
  prm.scores = scores;
  prm.window = window;
  prm.sel_out = sel_out;
  prm.nsel_out = nsel_out;
  prm.g = g;
  prm.q = reinterpret_cast<const __nv_bfloat16*>(q);
  prm.k_pool = k_pool; prm.k_sf = k_sf; prm.v_pool = v_pool; prm.v_sf = v_sf;
  prm.k_scale = k_scale; prm.v_scale = v_scale; prm.sm_scale = sm_scale;
  prm.page_table = page_table; prm.seqlens = seqlens; prm.sel = sel; prm.k = k;
  prm.out = reinterpret_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  const int ntr = tiles_per_row(g);
  const int rc = variant_rows(ntr, g.R, g.D);
  const long long units = (long long)g.B * g.Hkv * plan.qgroups * (g.R / rc);
  prm.status = reinterpret_cast<int*>(ws);
  prm.tickets = reinterpret_cast<int*>(ws + kWsHeader);
  prm.partials = reinterpret_cast<float*>(ws + kWsHeader + align256((size_t)units * sizeof(int)));
  prm.splits = plan.splits;
  prm.slices = plan.qgroups;
  prm.cluster = 1;
  dim3 grid(plan.splits, g.Hkv * plan.qgroups, g.B * (g.R / rc));
#define X(NTR_, R_, W_, S_, ONE_, D_)                                \
  if (ntr == NTR_ && g.R == R_ && g.D == D_)                           \
    return launch_t<NTR_, W_, S_, ONE_, D_>(prm, grid, rc, k, g.MB, pdl, stream);
  QSA_DECODE_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

// head_dim 128: the shared-dequantisation kernel (qsa_attend.cu); head_dim
// 256: the per-row-warp kernel above.
DecodePlan plan_sparse_decode(const Geom& g, int k, int num_splits) {
  return attend_supports(g) ? plan_attend(g, k, num_splits) : plan_legacy_decode(g, k, num_splits);
}

cudaError_t launch_sparse_decode(const Geom& g, const DecodePlan& plan, const void* q,
                                 const uint8_t* k_pool, const uint8_t* k_sf,
                                 const uint8_t* v_pool, const uint8_t* v_sf, float k_scale,
                                 float v_scale, float sm_scale, const int32_t* page_table,
                                 const int32_t* seqlens, const int32_t* sel, int k, void* out,
                                 float* lse, void* workspace, bool pdl, cudaStream_t stream,
                                 const int32_t* scores, int window, int32_t* sel_out,
                                 int32_t* nsel_out) {
  if (!scores && attend_supports(g))
    return launch_attend(g, plan, q, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale, sm_scale,
                         page_table, seqlens, sel, k, out, lse, workspace, pdl, stream);
  return launch_legacy_decode(g, plan, q, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale, sm_scale,
                              page_table, seqlens, sel, k, out, lse, workspace, pdl, stream,
                              scores, window, sel_out, nsel_out);
}

}  // namespace qsa

QSA_BOUNDS_READER(bounds_word_decode)
