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
// One CTA = (request b, KV head g, query-column group, KV split s).  Its
// query columns are the G*R query vectors (row j, head g*G + hh) of the
// request that read KV head g, so every page is read once per KV head for all
// of them.  The pages are the union of the rows' selections (each page carries
// a mask of the rows that selected it); the split takes a contiguous share of
// that union's 64-token chunks.
//
// Per chunk (K 4 KB + K scales 512 B + V 4 KB + V scales 512 B, contiguous in
// the pools) a TMA bulk copy lands it in shared memory; the consuming warp
// dequantises straight into mma.sync fragments:
//   S^T = K . Q^T   A = K tile (tokens x dims) from e2m1 bytes * e4m3 scale,
//                   B = Q^T (fp16, pre-scaled by a power of two per column)
//   O^T += V^T . P^T  A = V^T tile (dims x tokens) built from two tokens'
//                   nibbles per byte, B = P^T from S^T by an 8x8 transpose
// e2m1 x e4m3 products are exact in fp16, so the only roundings are the fp16
// P and fp32 accumulation.  Dims and tokens are permuted inside each MMA so
// that each thread reads whole 16-byte (K) and 8-byte (V) runs of a token row
// and every shared-memory wavefront is conflict-free; the contraction is
// invariant under those permutations and the output un-permutes them.
//
// Teams: with up to 16 columns a warp owns a whole chunk; with 17..32 a pair
// of warps shares one chunk (QK split by tokens, PV split by dims, max and P
// exchanged through shared memory) so no dequantised element is produced
// twice and accumulators stay in registers.
#include "qsa_common.cuh"

#include <math.h>

namespace qsa {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;                   // tokens per pipeline stage
constexpr int kMaxCols = 32;                 // query columns per CTA
constexpr int kKBytes = kChunk * kHeadDim / 2;     // 4096
constexpr int kSfBytes = kChunk * kHeadDim / 16;   // 512
constexpr int kStageBytes = 2 * kKBytes + 2 * kSfBytes;  // 9216
constexpr int kStages = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s per bounded wait

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
  int* tickets;         // [B * Hkv * QG]
  float* partials;      // [B * Hkv * QG][S][kMaxCols][2 + D]
  int splits, qgroups, cols;
};

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_stage(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitNs) return false;
  }
}

// Shared-memory layout (bytes), shared by host sizing and the kernel.
template <int NT, int TEAM>
struct Layout {
  static constexpr int kTeams = kWarps / TEAM;
  static constexpr int kStagesOff = 0;
  static constexpr int kStagesSz = kTeams * kStages * kStageBytes;
  static constexpr int kBarOff = kStagesSz;
  static constexpr int kBarSz = kTeams * kStages * 8;
  static constexpr int kQOff = kBarOff + kBarSz;                 // half [kMaxCols][128]
  static constexpr int kQSz = kMaxCols * kHeadDim * 2;
  static constexpr int kColOff = kQOff + kQSz;                   // cq, lim-n, row bit
  static constexpr int kColSz = 3 * kMaxCols * 4;
  static constexpr int kXmaxOff = kColOff + kColSz;              // [teams][2][32] float
  static constexpr int kXmaxSz = (TEAM == 2) ? kTeams * 2 * kMaxCols * 4 : 0;
  static constexpr int kXpOff = kXmaxOff + kXmaxSz;              // [teams][2][32 lanes][4*NT]
  static constexpr int kXpSz = (TEAM == 2) ? kTeams * 2 * 32 * 4 * NT * 4 : 0;
  static constexpr int kMiscOff = kXpOff + kXpSz;                // scan scratch + scalars
  static constexpr int kMiscSz = 64 * 4;
  static constexpr int kSelOff = kMiscOff + kMiscSz;             // [rows][k] int32, then union
  // Combine region (reuses stages after the main loop): m, l, O per team.
  static constexpr int kCombineSz = kTeams * kMaxCols * (2 + kHeadDim) * 4;
  static_assert(kCombineSz <= kStagesSz, "combine buffers must fit in the stage region");
  static size_t bytes(int rows, int k) {
    return (size_t)kSelOff + (size_t)rows * k * 4 * 3;  // sel rows + union ids + union pages
  }
};

template <int NT, int TEAM>
__global__ void __launch_bounds__(kThreads)
sparse_decode_kernel(Params p) {
  using Lay = Layout<NT, TEAM>;
  constexpr int kTeams = Lay::kTeams;
  constexpr int kMtPerWarp = 4 / TEAM;   // QK m-tiles (16 tokens) per warp per chunk
  constexpr int kDtPerWarp = 8 / TEAM;   // PV m-tiles (16 dims) per warp

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem + Lay::kStagesOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
  __half* qs = reinterpret_cast<__half*>(smem + Lay::kQOff);
  float* col_cq = reinterpret_cast<float*>(smem + Lay::kColOff);
  int* col_n = reinterpret_cast<int*>(smem + Lay::kColOff + kMaxCols * 4);
  int* col_bit = reinterpret_cast<int*>(smem + Lay::kColOff + 2 * kMaxCols * 4);
  float* xmax = reinterpret_cast<float*>(smem + Lay::kXmaxOff);
  uint32_t* xp = reinterpret_cast<uint32_t*>(smem + Lay::kXpOff);
  int* misc = reinterpret_cast<int*>(smem + Lay::kMiscOff);
  int32_t* s_sel = reinterpret_cast<int32_t*>(smem + Lay::kSelOff);

  const Geom& g = p.g;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int team = warp / TEAM, rank = warp % TEAM;

  const int s = blockIdx.x;
  const int gq = blockIdx.y;
  const int kvh = gq / p.qgroups, qg = gq % p.qgroups;
  const int b = blockIdx.z;
  const int G = g.Hq / g.Hkv;
  const int R = g.R;
  const int c0 = qg * kMaxCols;
  const int ncols = min(kMaxCols, p.cols - c0);
  const int j_lo = c0 / G, j_hi = (c0 + ncols - 1) / G;
  const int nrows = j_hi - j_lo + 1;
  const int k = p.k;
  int32_t* s_union = s_sel + nrows * k;
  int32_t* s_upage = s_union + nrows * k;

  if (tid == 0) {
    for (int i = 0; i < kTeams * kStages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }

  pdl_wait();   // every global read below may depend on the preceding kernel

  // Column metadata and pre-scaled fp16 queries.
  const int L = p.seqlens[b];
  const int cap = g.MB * g.P;
  for (int c = warp; c < kMaxCols; c += kWarps) {
    float amax = 0.f;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    int jrow = 0;
    if (c < ncols) {
      const int col = c0 + c;
      jrow = col / G;
      const int h = kvh * G + col % G;
      const __nv_bfloat16* src = p.q + ((size_t)(b * R + jrow) * g.Hq + h) * kHeadDim + lane * 4;
      const uint2 raw = *reinterpret_cast<const uint2*>(src);
      const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
      const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
      v[0] = __low2float(lo); v[1] = __high2float(lo);
      v[2] = __low2float(hi); v[3] = __high2float(hi);
      amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    // Power-of-two pre-scale mapping |q|max into [256, 512): exact, and keeps
    // bf16 queries of any magnitude inside fp16 range.
    int e = 0;
    if (amax > 0.f) frexpf(amax, &e);
    const int sq = (amax > 0.f) ? 9 - e : 0;
    __half2* dst = reinterpret_cast<__half2*>(qs + c * kHeadDim + lane * 4);
    dst[0] = __floats2half2_rn(ldexpf(v[0], sq), ldexpf(v[1], sq));
    dst[1] = __floats2half2_rn(ldexpf(v[2], sq), ldexpf(v[3], sq));
    if (lane == 0) {
      col_cq[c] = (c < ncols) ? p.k_scale * p.sm_scale * kLog2e * ldexpf(1.f, -sq) : 0.f;
      col_n[c] = (c < ncols) ? visible_tokens(L, R, jrow, cap) : 0;
      col_bit[c] = (c < ncols) ? (jrow - j_lo) : 31;
    }
  }

  // Union of the selections of rows j_lo..j_hi, in (row, position) order of
  // first occurrence, restricted to blocks with a valid page.
  for (int i = tid; i < nrows * k; i += kThreads) {
    int v = p.sel[(size_t)(b * R + j_lo + i / k) * k + (i % k)];
    s_sel[i] = (v >= 0 && v < g.MB) ? v : -1;
  }
  __syncthreads();
  const int ne = nrows * k;
  const int per = (ne + kThreads - 1) / kThreads;
  const int e_lo = min(ne, tid * per), e_hi = min(ne, e_lo + per);
  int keep_cnt = 0;
  for (int e = e_lo; e < e_hi; ++e) {
    const int beta = s_sel[e];
    if (beta < 0) continue;
    const int jj = e / k;
    bool first = true;
    int mask = 0;
    for (int j2 = 0; j2 < nrows; ++j2) {
      // binary search beta in row j2 (ascending, -1 padding treated as +inf)
      const int32_t* row = s_sel + j2 * k;
      int lo2 = 0, hi2 = k;
      while (lo2 < hi2) {
        const int mid = (lo2 + hi2) >> 1;
        const int x = row[mid] < 0 ? 0x7FFFFFFF : row[mid];
        if (x < beta) lo2 = mid + 1; else hi2 = mid;
      }
      if (lo2 < k && row[lo2] == beta) {
        mask |= 1 << j2;
        if (j2 < jj) first = false;
      }
    }
    if (!first) continue;
    const int page = p.page_table[(size_t)b * g.MB + beta];
    if (page < 0 || page >= g.NP) continue;
    ++keep_cnt;
  }
  // Exclusive scan of keep counts (thread order = entry order).
  {
    int x = keep_cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) misc[warp] = x;
    __syncthreads();
    int base = 0, tot = 0;
    for (int w = 0; w < kWarps; ++w) {
      base += (w < warp) ? misc[w] : 0;
      tot += misc[w];
    }
    int pos = base + x - keep_cnt;
    for (int e = e_lo; e < e_hi; ++e) {
      const int beta = s_sel[e];
      if (beta < 0) continue;
      const int jj = e / k;
      bool first = true;
      int mask = 0;
      for (int j2 = 0; j2 < nrows; ++j2) {
        const int32_t* row = s_sel + j2 * k;
        int lo2 = 0, hi2 = k;
        while (lo2 < hi2) {
          const int mid = (lo2 + hi2) >> 1;
          const int xv = row[mid] < 0 ? 0x7FFFFFFF : row[mid];
          if (xv < beta) lo2 = mid + 1; else hi2 = mid;
        }
        if (lo2 < k && row[lo2] == beta) {
          mask |= 1 << j2;
          if (j2 < jj) first = false;
        }
      }
      if (!first) continue;
      const int page = p.page_table[(size_t)b * g.MB + beta];
      if (page < 0 || page >= g.NP) continue;
      s_union[pos] = beta | (mask << 24);
      s_upage[pos] = page;
      ++pos;
    }
    if (tid == 0) misc[8] = tot;
  }
  __syncthreads();
  pdl_trigger();

  const int U = misc[8];
  const int cpp = g.P / kChunk;               // chunks per page
  const int C = U * cpp;
  const int per_split = (C + p.splits - 1) / p.splits;
  const int ch_lo = min(C, s * per_split);
  const int ch_hi = min(C, ch_lo + per_split);
  const int all_rows = (1 << nrows) - 1;

  // Per-thread column scale factors (the mask limits stay in shared memory).
  float cq[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) cq[nt][e] = col_cq[nt * 8 + 2 * tig + e];
  int min_n = 0x7FFFFFFF;
  for (int c = 0; c < ncols; ++c) min_n = min(min_n, col_n[c]);

  // Q^T fragments: column nt*8+gid, dims [32*tig, 32*tig+32) as 16 half2.
  uint32_t qf[NT][16];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint4* src = reinterpret_cast<const uint4*>(qs + (nt * 8 + gid) * kHeadDim + 32 * tig);
#pragma unroll
    for (int v4 = 0; v4 < 4; ++v4) {
      const uint4 x = src[v4];
      qf[nt][4 * v4 + 0] = x.x; qf[nt][4 * v4 + 1] = x.y;
      qf[nt][4 * v4 + 2] = x.z; qf[nt][4 * v4 + 3] = x.w;
    }
  }

  // Online-softmax state (log2 domain) for the thread's columns.
  float m_run[NT][2], l_run[NT][2];
  float o_acc[kDtPerWarp][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) { m_run[nt][e] = -INFINITY; l_run[nt][e] = 0.f; }
#pragma unroll
  for (int dt = 0; dt < kDtPerWarp; ++dt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o_acc[dt][nt][e] = 0.f;

  const uint64_t pol = policy_evict_first();
  const bool leader = (rank == 0) && (lane == 0);
  uint8_t* my_stages = stages + team * kStages * kStageBytes;
  uint64_t* my_bars = bars + team * kStages;
  const int first_ch = ch_lo + team;
  const int n_my = (ch_hi > first_ch) ? (ch_hi - first_ch + kTeams - 1) / kTeams : 0;

  auto issue = [&](int i) {   // chunk i of this team into stage i % kStages
    const int c = first_ch + i * kTeams;
    const int u = c / cpp, sub = c % cpp;
    const size_t row0 = ((size_t)s_upage[u] * g.Hkv + kvh) * g.P + (size_t)sub * kChunk;
    uint8_t* st = my_stages + (i % kStages) * kStageBytes;
    uint64_t* bar = &my_bars[i % kStages];
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, kStageBytes);
    bulk_g2s(st, p.k_pool + row0 * (kHeadDim / 2), kKBytes, bar, pol);
    bulk_g2s(st + kKBytes, p.v_pool + row0 * (kHeadDim / 2), kKBytes, bar, pol);
    bulk_g2s(st + 2 * kKBytes, p.k_sf + row0 * (kHeadDim / 16), kSfBytes, bar, pol);
    bulk_g2s(st + 2 * kKBytes + kSfBytes, p.v_sf + row0 * (kHeadDim / 16), kSfBytes, bar, pol);
  };

  if (leader)
    for (int i = 0; i < kStages && i < n_my; ++i) issue(i);

  bool dead = false;
  int i = 0;
  for (; i < n_my; ++i) {
    const int c = first_ch + i * kTeams;
    const int u = c / cpp, sub = c % cpp;
    const int ue = s_union[u];
    const int beta = ue & 0xFFFFFF;
    const int rmask = (ue >> 24) & 0xFF;
    const int tok0 = beta * g.P + sub * kChunk;
    const bool full = (rmask == all_rows) && (tok0 + kChunk <= min_n);
    uint8_t* st = my_stages + (i % kStages) * kStageBytes;
    const bool ok = wait_stage(&my_bars[i % kStages], (i / kStages) & 1);
    if constexpr (TEAM == 2) {
      // Both warps of the team leave together, so neither is left waiting at
      // a named barrier for a partner that gave up.
      int* xdead = misc + 16 + team * 2;
      if (lane == 0) xdead[rank] = ok ? 0 : 1;
      asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(64) : "memory");
      dead = (xdead[0] | xdead[1]) != 0;
      asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(64) : "memory");
      if (dead) break;
    } else {
      if (!ok) {
        dead = true;
        break;
      }
    }
    const uint8_t* sk = st;
    const uint8_t* sv = st + kKBytes;
    const uint8_t* sks = st + 2 * kKBytes;
    const uint8_t* svs = st + 2 * kKBytes + kSfBytes;

    // ---- S^T = K . Q^T over this warp's m-tiles --------------------------
    float sacc[kMtPerWarp][NT][4];
#pragma unroll
    for (int mi = 0; mi < kMtPerWarp; ++mi) {
      const int mt = rank * kMtPerWarp + mi;
      const int rA = 16 * mt + (gid >> 1) + 4 * (gid & 1);
      const int rB = rA + 8;
      const uint4 kA = *reinterpret_cast<const uint4*>(sk + rA * 64 + 16 * tig);
      const uint4 kB = *reinterpret_cast<const uint4*>(sk + rB * 64 + 16 * tig);
      const uint32_t sA = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sks + rA * 8 + 2 * tig));
      const uint32_t sB = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sks + rB * 8 + 2 * tig));
      const uint32_t sA0 = prmt(sA, 0, 0x1010), sA1 = prmt(sA, 0, 0x3232);
      const uint32_t sB0 = prmt(sB, 0, 0x1010), sB1 = prmt(sB, 0, 0x3232);
      const uint32_t wA[4] = {kA.x, kA.y, kA.z, kA.w};
      const uint32_t wB[4] = {kB.x, kB.y, kB.z, kB.w};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mi][nt][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t scA = (kk < 4) ? sA0 : sA1;
        const uint32_t scB = (kk < 4) ? sB0 : sB1;
        const int wd = kk >> 1, sh = (kk & 1) * 16;
        uint32_t a[4];
        a[0] = hmul2_u32(e2m1x2_to_f16x2((wA[wd] >> sh) & 0xFF), scA);
        a[2] = hmul2_u32(e2m1x2_to_f16x2((wA[wd] >> (sh + 8)) & 0xFF), scA);
        a[1] = hmul2_u32(e2m1x2_to_f16x2((wB[wd] >> sh) & 0xFF), scB);
        a[3] = hmul2_u32(e2m1x2_to_f16x2((wB[wd] >> (sh + 8)) & 0xFF), scB);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_f16_16816(sacc[mi][nt], a, qf[nt][2 * kk], qf[nt][2 * kk + 1]);
      }
    }

    // ---- logits, masking, chunk max --------------------------------------
    float cmax[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) cmax[nt][e] = -INFINITY;
#pragma unroll
    for (int mi = 0; mi < kMtPerWarp; ++mi) {
      const int mt = rank * kMtPerWarp + mi;
      const int tA = tok0 + 16 * mt + (gid >> 1) + 4 * (gid & 1);
      const int tB = tA + 8;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float zA = sacc[mi][nt][e] * cq[nt][e];
          float zB = sacc[mi][nt][2 + e] * cq[nt][e];
          if (!full) {
            const int c = nt * 8 + 2 * tig + e;
            const int lim = ((rmask >> col_bit[c]) & 1) ? col_n[c] : 0;
            if (tA >= lim) zA = -INFINITY;
            if (tB >= lim) zB = -INFINITY;
          }
          sacc[mi][nt][e] = zA;
          sacc[mi][nt][2 + e] = zB;
          cmax[nt][e] = fmaxf(cmax[nt][e], fmaxf(zA, zB));
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = cmax[nt][e];
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        cmax[nt][e] = v;
      }
    if constexpr (TEAM == 2) {
      float* xm = xmax + team * 2 * kMaxCols;
      if (gid == 0)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) xm[rank * kMaxCols + nt * 8 + 2 * tig + e] = cmax[nt][e];
      asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(64) : "memory");
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          cmax[nt][e] = fmaxf(cmax[nt][e], xm[(1 - rank) * kMaxCols + nt * 8 + 2 * tig + e]);
    }

    // ---- online softmax update -------------------------------------------
    float base[NT][2];
    bool rescale = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float mn = fmaxf(m_run[nt][e], cmax[nt][e]);
        rescale |= (mn != m_run[nt][e]) && (m_run[nt][e] != -INFINITY);
        base[nt][e] = (mn == -INFINITY) ? 0.f : mn;
      }
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float alpha = exp2f(m_run[nt][e] - base[nt][e]);
          l_run[nt][e] *= alpha;
#pragma unroll
          for (int dt = 0; dt < kDtPerWarp; ++dt) {
            o_acc[dt][nt][e] *= alpha;
            o_acc[dt][nt][2 + e] *= alpha;
          }
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) m_run[nt][e] = fmaxf(m_run[nt][e], cmax[nt][e]);

    // P = exp2(z - base) -> fp16 -> transposed B fragments for P^T.  Slot q
    // holds m-tile mt_of(q): this warp's own m-tiles first, then the partner's.
    uint32_t pf[4][NT][2];
#pragma unroll
    for (int mi = 0; mi < kMtPerWarp; ++mi) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float p0 = exp2f(sacc[mi][nt][0] - base[nt][0]);
        const float p1 = exp2f(sacc[mi][nt][1] - base[nt][1]);
        const float p2 = exp2f(sacc[mi][nt][2] - base[nt][0]);
        const float p3 = exp2f(sacc[mi][nt][3] - base[nt][1]);
        l_run[nt][0] += p0 + p2;
        l_run[nt][1] += p1 + p3;
        pf[mi][nt][0] = movmatrix_trans(pack_half2(p0, p1));
        pf[mi][nt][1] = movmatrix_trans(pack_half2(p2, p3));
      }
    }
    if constexpr (TEAM == 2) {
      uint32_t* mine = xp + ((team * 2 + rank) * 32 + lane) * (4 * NT);
#pragma unroll
      for (int mi = 0; mi < kMtPerWarp; ++mi)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mine[(mi * NT + nt) * 2 + 0] = pf[mi][nt][0];
          mine[(mi * NT + nt) * 2 + 1] = pf[mi][nt][1];
        }
      asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(64) : "memory");
      const uint32_t* theirs = xp + ((team * 2 + (1 - rank)) * 32 + lane) * (4 * NT);
#pragma unroll
      for (int mi = 0; mi < kMtPerWarp; ++mi)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          pf[kMtPerWarp + mi][nt][0] = theirs[(mi * NT + nt) * 2 + 0];
          pf[kMtPerWarp + mi][nt][1] = theirs[(mi * NT + nt) * 2 + 1];
        }
    }

    // ---- O^T += V^T . P^T over this warp's dim tiles -----------------------
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int ks = (q < kMtPerWarp) ? rank * kMtPerWarp + q : (1 - rank) * kMtPerWarp + q - kMtPerWarp;
      const int t0 = 16 * ks + tig;
      const uint32_t sv01 = e4m3x2_to_f16x2((uint32_t)svs[t0 * 8 + gid] |
                                            ((uint32_t)svs[(t0 + 4) * 8 + gid] << 8));
      const uint32_t sv23 = e4m3x2_to_f16x2((uint32_t)svs[(t0 + 8) * 8 + gid] |
                                            ((uint32_t)svs[(t0 + 12) * 8 + gid] << 8));
#pragma unroll
      for (int w4 = 0; w4 < kDtPerWarp / 4; ++w4) {
        const int boff = 8 * gid + 4 * (rank * (kDtPerWarp / 4) + w4);
        const uint32_t X = *reinterpret_cast<const uint32_t*>(sv + t0 * 64 + boff);
        const uint32_t Y = *reinterpret_cast<const uint32_t*>(sv + (t0 + 4) * 64 + boff);
        const uint32_t X2 = *reinterpret_cast<const uint32_t*>(sv + (t0 + 8) * 64 + boff);
        const uint32_t Y2 = *reinterpret_cast<const uint32_t*>(sv + (t0 + 12) * 64 + boff);
        const uint32_t LO = (X & 0x0F0F0F0Fu) | ((Y << 4) & 0xF0F0F0F0u);
        const uint32_t HI = ((X >> 4) & 0x0F0F0F0Fu) | (Y & 0xF0F0F0F0u);
        const uint32_t LO2 = (X2 & 0x0F0F0F0Fu) | ((Y2 << 4) & 0xF0F0F0F0u);
        const uint32_t HI2 = ((X2 >> 4) & 0x0F0F0F0Fu) | (Y2 & 0xF0F0F0F0u);
#pragma unroll
        for (int bi = 0; bi < 4; ++bi) {
          const int dt = w4 * 4 + bi;
          uint32_t a[4];
          a[0] = hmul2_u32(e2m1x2_to_f16x2((LO >> (8 * bi)) & 0xFF), sv01);
          a[1] = hmul2_u32(e2m1x2_to_f16x2((HI >> (8 * bi)) & 0xFF), sv01);
          a[2] = hmul2_u32(e2m1x2_to_f16x2((LO2 >> (8 * bi)) & 0xFF), sv23);
          a[3] = hmul2_u32(e2m1x2_to_f16x2((HI2 >> (8 * bi)) & 0xFF), sv23);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_f16_16816(o_acc[dt][nt], a, pf[q][nt][0], pf[q][nt][1]);
        }
      }
    }

    // Release the stage and refill it with this team's chunk i + kStages.
    if constexpr (TEAM == 2) {
      asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(64) : "memory");
    } else {
      __syncwarp();
    }
    if (leader && i + kStages < n_my) issue(i + kStages);
  }

  if (dead) {
    // A copy never completed: record it, then drain this team's other
    // in-flight copies (bounded) before the stage memory is reused.
    if (lane == 0) atomicExch(p.status, kStatusWaitTimeout);
    for (int i2 = i; i2 < n_my && i2 < i + kStages; ++i2)
      (void)wait_stage(&my_bars[i2 % kStages], (i2 / kStages) & 1);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) { m_run[nt][e] = -INFINITY; l_run[nt][e] = 0.f; }
  }

  // Row sums: reduce the per-lane partials over the 8 token lanes.
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = l_run[nt][e];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l_run[nt][e] = v;
    }

  // ---- combine the teams of this CTA -----------------------------------
  __syncthreads();  // every stage consumed; reuse the stage region
  float* cm = reinterpret_cast<float*>(stages);            // [teams][32]
  float* cl = cm + kTeams * kMaxCols;                       // [teams][32]
  float* co = cl + kTeams * kMaxCols;                       // [teams][32][128]
  if (gid == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = nt * 8 + 2 * tig + e;
        if (rank == 0) cm[team * kMaxCols + c] = m_run[nt][e];
        if (rank == 0) cl[team * kMaxCols + c] = l_run[nt][e];
      }
  }
  if constexpr (TEAM == 2) {
    __syncthreads();
    if (gid == 0 && rank == 1)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) cl[team * kMaxCols + nt * 8 + 2 * tig + e] += l_run[nt][e];
  }
  // O^T accumulators: dim 16*gid + 2*dt (+1 for c2/c3), column nt*8 + 2*tig + e.
#pragma unroll
  for (int dl = 0; dl < kDtPerWarp; ++dl) {
    const int dt = rank * kDtPerWarp + dl;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = nt * 8 + 2 * tig + e;
        float* dst = co + ((size_t)team * kMaxCols + c) * kHeadDim + 16 * gid + 2 * dt;
        dst[0] = o_acc[dl][nt][e];
        dst[1] = o_acc[dl][nt][2 + e];
      }
  }
  __syncthreads();

  const int units_idx = (b * g.Hkv + kvh) * p.qgroups + qg;
  if (p.splits == 1) {
    for (int idx = tid; idx < ncols * kHeadDim; idx += kThreads) {
      const int c = idx / kHeadDim, d = idx % kHeadDim;
      float M = -INFINITY;
      for (int t = 0; t < kTeams; ++t) M = fmaxf(M, cm[t * kMaxCols + c]);
      const float base = (M == -INFINITY) ? 0.f : M;
      float Lsum = 0.f, O = 0.f;
      for (int t = 0; t < kTeams; ++t) {
        const float w = exp2f(cm[t * kMaxCols + c] - base);
        Lsum += cl[t * kMaxCols + c] * w;
        O += co[((size_t)t * kMaxCols + c) * kHeadDim + d] * w;
      }
      const int col = c0 + c;
      const int jrow = col / G, h = kvh * G + col % G;
      const size_t orow = (size_t)(b * R + jrow) * g.Hq + h;
      p.out[orow * kHeadDim + d] = __float2bfloat16_rn(Lsum > 0.f ? O / Lsum * p.v_scale : 0.f);
      if (d == 0) p.lse[orow] = Lsum > 0.f ? (base + log2f(Lsum)) * kLn2 : -INFINITY;
    }
    return;
  }

  // Split partial: (m, l, O) in the log2 domain, then a ticket; the last split
  // of this (request, KV head, group) to arrive merges all of them in split
  // order (deterministic) and resets the ticket.
  float* part = p.partials + ((size_t)units_idx * p.splits + s) * kMaxCols * (2 + kHeadDim);
  for (int idx = tid; idx < ncols * kHeadDim; idx += kThreads) {
    const int c = idx / kHeadDim, d = idx % kHeadDim;
    float M = -INFINITY;
    for (int t = 0; t < kTeams; ++t) M = fmaxf(M, cm[t * kMaxCols + c]);
    const float base = (M == -INFINITY) ? 0.f : M;
    float Lsum = 0.f, O = 0.f;
    for (int t = 0; t < kTeams; ++t) {
      const float w = exp2f(cm[t * kMaxCols + c] - base);
      Lsum += cl[t * kMaxCols + c] * w;
      O += co[((size_t)t * kMaxCols + c) * kHeadDim + d] * w;
    }
    float* pc = part + (size_t)c * (2 + kHeadDim);
    pc[2 + d] = O;
    if (d == 0) { pc[0] = M; pc[1] = Lsum; }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&p.tickets[units_idx], 1);
    misc[9] = (prev == p.splits - 1);
  }
  __syncthreads();
  if (!misc[9]) return;
  __threadfence();
  const float* parts = p.partials + (size_t)units_idx * p.splits * kMaxCols * (2 + kHeadDim);
  for (int idx = tid; idx < ncols * kHeadDim; idx += kThreads) {
    const int c = idx / kHeadDim, d = idx % kHeadDim;
    float M = -INFINITY;
    for (int t = 0; t < p.splits; ++t)
      M = fmaxf(M, __ldcg(parts + ((size_t)t * kMaxCols + c) * (2 + kHeadDim)));
    const float base = (M == -INFINITY) ? 0.f : M;
    float Lsum = 0.f, O = 0.f;
    for (int t = 0; t < p.splits; ++t) {
      const float* pc = parts + ((size_t)t * kMaxCols + c) * (2 + kHeadDim);
      const float w = exp2f(__ldcg(pc) - base);
      Lsum += __ldcg(pc + 1) * w;
      O += __ldcg(pc + 2 + d) * w;
    }
    const int col = c0 + c;
    const int jrow = col / G, h = kvh * G + col % G;
    const size_t orow = (size_t)(b * R + jrow) * g.Hq + h;
    p.out[orow * kHeadDim + d] = __float2bfloat16_rn(Lsum > 0.f ? O / Lsum * p.v_scale : 0.f);
    if (d == 0) p.lse[orow] = Lsum > 0.f ? (base + log2f(Lsum)) * kLn2 : -INFINITY;
  }
  if (tid == 0) atomicExch(&p.tickets[units_idx], 0);
}

constexpr size_t kWsHeader = 256;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int NT, int TEAM>
cudaError_t launch_t(const Params& prm, dim3 grid, size_t smem, bool pdl, cudaStream_t stream) {
  static bool configured = false;  // per-process; the attribute is per device
  (void)configured;
  cudaError_t e = cudaFuncSetAttribute(sparse_decode_kernel<NT, TEAM>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, sparse_decode_kernel<NT, TEAM>, prm);
}

}  // namespace

DecodePlan plan_sparse_decode(const Geom& g, int k, int num_splits) {
  DecodePlan pl;
  const int G = g.Hq / g.Hkv;
  pl.cols = G * g.R;
  pl.qgroups = (pl.cols + kMaxCols - 1) / kMaxCols;
  const long long units = (long long)g.B * g.Hkv * pl.qgroups;
  const int rows_per_group = pl.qgroups == 1 ? g.R : (kMaxCols + G - 1) / G + 1;
  int max_union = min(rows_per_group * k, g.MB);
  const int max_chunks = max(1, max_union * (g.P / kChunk));
  int splits = num_splits;
  if (splits <= 0) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long target = 2LL * sms;          // two CTAs per SM
    splits = (int)((target + units - 1) / units);
    const int min_chunks_per_cta = kWarps;      // at least one chunk per warp
    splits = min(splits, max(1, max_chunks / min_chunks_per_cta));
    splits = max(1, min(splits, 64));
  }
  pl.splits = splits;
  size_t ws = kWsHeader + align256((size_t)units * sizeof(int));
  if (splits > 1) ws += (size_t)units * splits * kMaxCols * (2 + kHeadDim) * sizeof(float);
  pl.ws_bytes = ws;
  return pl;
}

cudaError_t launch_sparse_decode(const Geom& g, const DecodePlan& plan, const void* q,
                                 const uint8_t* k_pool, const uint8_t* k_sf,
                                 const uint8_t* v_pool, const uint8_t* v_sf, float k_scale,
                                 float v_scale, float sm_scale, const int32_t* page_table,
                                 const int32_t* seqlens, const int32_t* sel, int k, void* out,
                                 float* lse, void* workspace, bool pdl, cudaStream_t stream) {
  Params prm;
  prm.g = g;
  prm.q = reinterpret_cast<const __nv_bfloat16*>(q);
  prm.k_pool = k_pool; prm.k_sf = k_sf; prm.v_pool = v_pool; prm.v_sf = v_sf;
  prm.k_scale = k_scale; prm.v_scale = v_scale; prm.sm_scale = sm_scale;
  prm.page_table = page_table; prm.seqlens = seqlens; prm.sel = sel; prm.k = k;
  prm.out = reinterpret_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  const long long units = (long long)g.B * g.Hkv * plan.qgroups;
  prm.status = reinterpret_cast<int*>(ws);
  prm.tickets = reinterpret_cast<int*>(ws + kWsHeader);
  prm.partials = reinterpret_cast<float*>(ws + kWsHeader + align256((size_t)units * sizeof(int)));
  prm.splits = plan.splits;
  prm.qgroups = plan.qgroups;
  prm.cols = plan.cols;
  const int G = g.Hq / g.Hkv;
  const int cols_cta = min(plan.cols, kMaxCols);
  const int nt = (cols_cta + 7) / 8;
  const int rows = plan.qgroups == 1 ? g.R : min(g.R, (kMaxCols + G - 1) / G + 1);
  dim3 grid(plan.splits, g.Hkv * plan.qgroups, g.B);
  switch (nt) {
    case 1: return launch_t<1, 1>(prm, grid, Layout<1, 1>::bytes(rows, k), pdl, stream);
    case 2: return launch_t<2, 1>(prm, grid, Layout<2, 1>::bytes(rows, k), pdl, stream);
    case 3: return launch_t<3, 2>(prm, grid, Layout<3, 2>::bytes(rows, k), pdl, stream);
    default: return launch_t<4, 2>(prm, grid, Layout<4, 2>::bytes(rows, k), pdl, stream);
  }
}

}  // namespace qsa
