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
// the pools) a TMA bulk copy lands it in shared memory; the consuming warps
// dequantise straight into mma.sync fragments:
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
// A team of TEAM warps shares each chunk: QK is split by 16-token tiles and
// PV by 16-dim tiles, the chunk max and P fragments are exchanged through
// shared memory, so no element is dequantised twice and each warp keeps only
// its share of the accumulators.  Query-column tiles whose rows did not select
// the chunk's page are skipped (verify rows mostly select different pages).
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
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s per bounded wait
constexpr int kPartStride = 4 + kHeadDim;    // m, l, pad, pad, O[128] per column

#ifndef QSA_DECODE_TEAM_NT1
#define QSA_DECODE_TEAM_NT1 4
#endif
#ifndef QSA_DECODE_STAGES_NT1
#define QSA_DECODE_STAGES_NT1 4
#endif

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
  float* partials;      // [B * Hkv * QG][S][kMaxCols][kPartStride]
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

// Four bytes of e2m1 pairs -> four fp16 pairs (byte i -> o[i], low nibble in
// the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

template <int TEAM>
__device__ __forceinline__ void team_sync(int team) {
  if constexpr (TEAM == 1) {
    __syncwarp();
  } else if constexpr (TEAM == kWarps) {
    __syncthreads();
  } else {
    named_bar(1 + team, TEAM * 32);
  }
}

// Shared-memory layout (bytes), shared by host sizing and the kernel.
template <int NT, int TEAM, int STAGES>
struct Layout {
  static constexpr int kTeams = kWarps / TEAM;
  static constexpr int kMtPerWarp = 4 / TEAM;
  static constexpr int kStagesSz = kTeams * STAGES * kStageBytes;
  // After the main loop the stage region holds the team partials, and in the
  // merging CTA the split weights.
  static constexpr int kCombineSz = kTeams * kMaxCols * kHeadDim * 4 + kTeams * kMaxCols * 4 +
                                    kWarps * kMaxCols * 4;
  static constexpr int kMergeSz = kMaxCols * 64 * 4 + kMaxCols * 8;
  static constexpr int kRegion0 = kStagesSz > kCombineSz ? kStagesSz : kCombineSz;
  static constexpr int kRegionSz = kRegion0 > kMergeSz ? kRegion0 : kMergeSz;
  static constexpr int kBarOff = kRegionSz;
  static constexpr int kBarSz = kTeams * STAGES * 8;
  static constexpr int kQOff = kBarOff + kBarSz;                 // half [NT*8][128]
  static constexpr int kQSz = NT * 8 * kHeadDim * 2;
  static constexpr int kColOff = kQOff + kQSz;                   // cq, n, row bit, tile rows
  static constexpr int kColSz = 3 * kMaxCols * 4 + 4 * 4;
  static constexpr int kXmaxOff = kColOff + kColSz;              // [teams][TEAM][32] float
  static constexpr int kXmaxSz = (TEAM > 1) ? kTeams * TEAM * kMaxCols * 4 : 0;
  static constexpr int kXpSlots = kMtPerWarp * NT * 2;
  static constexpr int kXpOff = kXmaxOff + kXmaxSz;              // [teams][TEAM][slots][32]
  static constexpr int kXpSz = (TEAM > 1) ? kTeams * TEAM * kXpSlots * 32 * 4 : 0;
  static constexpr int kMiscOff = kXpOff + kXpSz;
  static constexpr int kMiscSz = 64 * 4;
  static constexpr int kSelOff = kMiscOff + kMiscSz;             // sel rows, union, pages
  static size_t bytes(int rows, int k) { return (size_t)kSelOff + (size_t)rows * k * 4 * 3; }
};

template <int NT, int TEAM, int STAGES>
__global__ void __launch_bounds__(kThreads)
sparse_decode_kernel(Params p) {
  using Lay = Layout<NT, TEAM, STAGES>;
  constexpr int kTeams = Lay::kTeams;
  constexpr int kMtPerWarp = 4 / TEAM;   // QK 16-token tiles per warp per chunk
  constexpr int kDtPerWarp = 8 / TEAM;   // PV 16-dim tiles per warp
  constexpr int kSlots = Lay::kXpSlots;

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* region = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
  __half* qs = reinterpret_cast<__half*>(smem + Lay::kQOff);
  float* col_cq = reinterpret_cast<float*>(smem + Lay::kColOff);
  int* col_n = reinterpret_cast<int*>(smem + Lay::kColOff + kMaxCols * 4);
  int* col_bit = reinterpret_cast<int*>(smem + Lay::kColOff + 2 * kMaxCols * 4);
  int* tile_rows = reinterpret_cast<int*>(smem + Lay::kColOff + 3 * kMaxCols * 4);
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
    for (int i = 0; i < kTeams * STAGES; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }

  pdl_wait();   // every global read below may depend on the preceding kernel

  // ---- union of the rows' selections (first occurrence, valid pages) -------
  for (int i = tid; i < nrows * k; i += kThreads) {
    const int v = p.sel[(size_t)(b * R + j_lo + i / k) * k + (i % k)];
    s_sel[i] = (v >= 0 && v < g.MB) ? v : -1;
  }
  __syncthreads();
  const int ne = nrows * k;
  const int per = (ne + kThreads - 1) / kThreads;   // <= 16 (union bound 2048)
  const int e_lo = min(ne, tid * per), e_hi = min(ne, e_lo + per);
  // Each thread marks its entries: kept (first occurrence, valid page) with
  // the mask of rows that selected the block.
  int flags[16];
  int keep_cnt = 0;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int e = e_lo + q;
    int flag = 0;
    if (e < e_hi) {
      const int beta = s_sel[e];
      if (beta >= 0) {
        const int jj = e / k;
        bool first = true;
        int mask = 1 << jj;
        for (int j2 = 0; j2 < nrows; ++j2) {
          if (j2 == jj) continue;
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
        if (first) {
          const int page = p.page_table[(size_t)b * g.MB + beta];
          if (page >= 0 && page < g.NP) {
            flag = 0x100 | (mask & 0xFF);
            s_upage[e] = page;   // staged at the entry index, compacted below
            ++keep_cnt;
          }
        }
      }
    }
    flags[q] = flag;
  }
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
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      base += (w < warp) ? misc[w] : 0;
      tot += misc[w];
    }
    int pos = base + x - keep_cnt;
    int pages[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) pages[q] = flags[q] ? s_upage[e_lo + q] : 0;
    __syncthreads();   // every staged page read before compaction overwrites
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      if (!flags[q]) continue;
      const int beta = s_sel[e_lo + q];
      s_union[pos] = beta | ((flags[q] & 0xFF) << 24);
      s_upage[pos] = pages[q];
      ++pos;
    }
    if (tid == 0) misc[8] = tot;
  }
  __syncthreads();

  const int U = misc[8];
  const int cpp = g.P / kChunk;               // chunks per page
  const int C = U * cpp;
  const int per_split = (C + p.splits - 1) / p.splits;
  const int ch_lo = min(C, s * per_split);
  const int ch_hi = min(C, ch_lo + per_split);
  const int all_rows = (1 << nrows) - 1;

  const uint64_t pol = policy_evict_first();
  const bool leader = (rank == 0) && (lane == 0);
  uint8_t* my_stages = region + team * STAGES * kStageBytes;
  uint64_t* my_bars = bars + team * STAGES;
  const int first_ch = ch_lo + team;
  const int n_my = (ch_hi > first_ch) ? (ch_hi - first_ch + kTeams - 1) / kTeams : 0;

  auto issue = [&](int i) {   // this team's chunk i into stage i % STAGES
    const int c = first_ch + i * kTeams;
    const int u = c / cpp, sub = c % cpp;
    const size_t row0 = ((size_t)s_upage[u] * g.Hkv + kvh) * g.P + (size_t)sub * kChunk;
    uint8_t* st = my_stages + (i % STAGES) * kStageBytes;
    uint64_t* bar = &my_bars[i % STAGES];
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, kStageBytes);
    bulk_g2s(st, p.k_pool + row0 * (kHeadDim / 2), kKBytes, bar, pol);
    bulk_g2s(st + kKBytes, p.v_pool + row0 * (kHeadDim / 2), kKBytes, bar, pol);
    bulk_g2s(st + 2 * kKBytes, p.k_sf + row0 * (kHeadDim / 16), kSfBytes, bar, pol);
    bulk_g2s(st + 2 * kKBytes + kSfBytes, p.v_sf + row0 * (kHeadDim / 16), kSfBytes, bar, pol);
  };
  if (leader)
    for (int i = 0; i < STAGES && i < n_my; ++i) issue(i);

  // ---- queries (overlapping the first copies) -----------------------------
  const int L = p.seqlens[b];
  const int cap = g.MB * g.P;
  for (int c = warp; c < NT * 8; c += kWarps) {
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
  __syncthreads();
  if (tid < NT) {
    int m = 0;
    for (int c = tid * 8; c < tid * 8 + 8; ++c)
      if (c < ncols) m |= 1 << col_bit[c];
    tile_rows[tid] = m;
  }
  int min_n = 0x7FFFFFFF;
  for (int c = 0; c < ncols; ++c) min_n = min(min_n, col_n[c]);
  __syncthreads();
  pdl_trigger();

  float cq[NT][2];
  int trows[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    trows[nt] = tile_rows[nt];
#pragma unroll
    for (int e = 0; e < 2; ++e) cq[nt][e] = col_cq[nt * 8 + 2 * tig + e];
  }
  int all_tiles = 0;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) all_tiles |= (trows[nt] != 0) << nt;

  // Q^T fragments (column nt*8+gid, dims [32*tig, 32*tig+32)) in registers for
  // up to two column tiles; wider tiles are read from shared memory per use.
  constexpr bool kQInRegs = NT <= 2;
  uint32_t qf[kQInRegs ? NT : 1][16];
  if constexpr (kQInRegs) {
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
    int act = 0;   // column tiles with a row that selected this page
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) act |= ((trows[nt] & rmask) != 0) << nt;
    if (full) act = all_tiles;
    const uint8_t* st = my_stages + (i % STAGES) * kStageBytes;
    const bool ok = wait_stage(&my_bars[i % STAGES], (i / STAGES) & 1);
    if constexpr (TEAM == 1) {
      if (!ok) { dead = true; break; }
    } else {
      if (lane == 0) misc[16 + warp] = ok ? 0 : 1;
    }
    const uint8_t* sk = st;
    const uint8_t* sv = st + kKBytes;
    const uint8_t* sks = st + 2 * kKBytes;
    const uint8_t* svs = st + 2 * kKBytes + kSfBytes;

    // ---- S^T = K . Q^T over this warp's 16-token tiles ---------------------
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
      const uint32_t scA[2] = {prmt(sA, 0, 0x1010), prmt(sA, 0, 0x3232)};
      const uint32_t scB[2] = {prmt(sB, 0, 0x1010), prmt(sB, 0, 0x3232)};
      const uint32_t wA[4] = {kA.x, kA.y, kA.z, kA.w};
      const uint32_t wB[4] = {kB.x, kB.y, kB.z, kB.w};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mi][nt][e] = 0.f;
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        uint32_t fa[4], fb[4];
        e2m1x8_to_f16x2x4(wA[wd], fa);
        e2m1x8_to_f16x2x4(wB[wd], fb);
        const uint32_t sa = scA[wd >> 1], sb = scB[wd >> 1];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int kk = 2 * wd + h;
          uint32_t a[4];
          a[0] = hmul2_u32(fa[2 * h], sa);
          a[2] = hmul2_u32(fa[2 * h + 1], sa);
          a[1] = hmul2_u32(fb[2 * h], sb);
          a[3] = hmul2_u32(fb[2 * h + 1], sb);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (act & (1 << nt)) {
              uint32_t b0, b1;
              if constexpr (kQInRegs) {
                b0 = qf[kQInRegs ? nt : 0][2 * kk];
                b1 = qf[kQInRegs ? nt : 0][2 * kk + 1];
              } else {
                const uint2 qv = *reinterpret_cast<const uint2*>(
                    qs + (nt * 8 + gid) * kHeadDim + 32 * tig + 4 * kk);
                b0 = qv.x;
                b1 = qv.y;
              }
              mma_f16_16816(sacc[mi][nt], a, b0, b1);
            }
          }
        }
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
      for (int nt = 0; nt < NT; ++nt) {
        if (!(act & (1 << nt))) continue;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float zA = sacc[mi][nt][e] * cq[nt][e];
          float zB = sacc[mi][nt][2 + e] * cq[nt][e];
          if (!full) {
            const int cc = nt * 8 + 2 * tig + e;
            const int lim = ((rmask >> col_bit[cc]) & 1) ? col_n[cc] : 0;
            if (tA >= lim) zA = -INFINITY;
            if (tB >= lim) zB = -INFINITY;
          }
          sacc[mi][nt][e] = zA;
          sacc[mi][nt][2 + e] = zB;
          cmax[nt][e] = fmaxf(cmax[nt][e], fmaxf(zA, zB));
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (!(act & (1 << nt))) continue;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = cmax[nt][e];
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
        cmax[nt][e] = v;
      }
    }
    if constexpr (TEAM > 1) {
      float* xm = xmax + team * TEAM * kMaxCols;
      if (gid == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) xm[rank * kMaxCols + nt * 8 + 2 * tig + e] = cmax[nt][e];
      }
      team_sync<TEAM>(team);
      int dead_any = 0;
#pragma unroll
      for (int r2 = 0; r2 < TEAM; ++r2) dead_any |= misc[16 + team * TEAM + r2];
      if (dead_any) { dead = true; break; }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (!(act & (1 << nt))) continue;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = -INFINITY;
#pragma unroll
          for (int r2 = 0; r2 < TEAM; ++r2) v = fmaxf(v, xm[r2 * kMaxCols + nt * 8 + 2 * tig + e]);
          cmax[nt][e] = v;
        }
      }
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
    // holds 16-token tile ((q / kMtPerWarp + rank) % TEAM) * kMtPerWarp +
    // q % kMtPerWarp: this warp's own tiles first.
    uint32_t pf[4][NT][2];
#pragma unroll
    for (int mi = 0; mi < kMtPerWarp; ++mi) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (!(act & (1 << nt))) continue;
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
    if constexpr (TEAM > 1) {
      uint32_t* mine = xp + ((team * TEAM + rank) * kSlots) * 32 + lane;
#pragma unroll
      for (int mi = 0; mi < kMtPerWarp; ++mi)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (!(act & (1 << nt))) continue;
          mine[((mi * NT + nt) * 2 + 0) * 32] = pf[mi][nt][0];
          mine[((mi * NT + nt) * 2 + 1) * 32] = pf[mi][nt][1];
        }
      team_sync<TEAM>(team);
#pragma unroll
      for (int r2 = 1; r2 < TEAM; ++r2) {
        const int other = (rank + r2) % TEAM;
        const uint32_t* theirs = xp + ((team * TEAM + other) * kSlots) * 32 + lane;
#pragma unroll
        for (int mi = 0; mi < kMtPerWarp; ++mi)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (!(act & (1 << nt))) continue;
            pf[r2 * kMtPerWarp + mi][nt][0] = theirs[((mi * NT + nt) * 2 + 0) * 32];
            pf[r2 * kMtPerWarp + mi][nt][1] = theirs[((mi * NT + nt) * 2 + 1) * 32];
          }
      }
    }

    // ---- O^T += V^T . P^T over this warp's 16-dim tiles ---------------------
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int ks = ((q / kMtPerWarp + rank) % TEAM) * kMtPerWarp + q % kMtPerWarp;
      const int t0 = 16 * ks + tig;
      const uint32_t sv01 = e4m3x2_to_f16x2((uint32_t)svs[t0 * 8 + gid] |
                                            ((uint32_t)svs[(t0 + 4) * 8 + gid] << 8));
      const uint32_t sv23 = e4m3x2_to_f16x2((uint32_t)svs[(t0 + 8) * 8 + gid] |
                                            ((uint32_t)svs[(t0 + 12) * 8 + gid] << 8));
#pragma unroll
      for (int w4 = 0; w4 < (kDtPerWarp + 3) / 4; ++w4) {
        // bytes [8*gid + dbase, +kNb) of the four token rows of this k-step
        constexpr int kNb = kDtPerWarp < 4 ? kDtPerWarp : 4;
        const int dbase = rank * kDtPerWarp + 4 * w4;
        uint32_t X, Y, X2, Y2;
        if constexpr (kNb == 4) {
          X = *reinterpret_cast<const uint32_t*>(sv + t0 * 64 + 8 * gid + dbase);
          Y = *reinterpret_cast<const uint32_t*>(sv + (t0 + 4) * 64 + 8 * gid + dbase);
          X2 = *reinterpret_cast<const uint32_t*>(sv + (t0 + 8) * 64 + 8 * gid + dbase);
          Y2 = *reinterpret_cast<const uint32_t*>(sv + (t0 + 12) * 64 + 8 * gid + dbase);
        } else {
          X = *reinterpret_cast<const uint16_t*>(sv + t0 * 64 + 8 * gid + dbase);
          Y = *reinterpret_cast<const uint16_t*>(sv + (t0 + 4) * 64 + 8 * gid + dbase);
          X2 = *reinterpret_cast<const uint16_t*>(sv + (t0 + 8) * 64 + 8 * gid + dbase);
          Y2 = *reinterpret_cast<const uint16_t*>(sv + (t0 + 12) * 64 + 8 * gid + dbase);
        }
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
        for (int bi = 0; bi < kNb; ++bi) {
          const int dl = 4 * w4 + bi;
          uint32_t a[4];
          a[0] = hmul2_u32(f0[bi], sv01);
          a[1] = hmul2_u32(f1[bi], sv01);
          a[2] = hmul2_u32(f2[bi], sv23);
          a[3] = hmul2_u32(f3[bi], sv23);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            if (act & (1 << nt)) mma_f16_16816(o_acc[dl][nt], a, pf[q][nt][0], pf[q][nt][1]);
        }
      }
    }

    // Release the stage and refill it with this team's chunk i + STAGES.
    team_sync<TEAM>(team);
    if (leader && i + STAGES < n_my) issue(i + STAGES);
  }

  if (dead) {
    // A copy never completed: record it, then drain this team's other
    // in-flight copies (bounded) before the stage memory is reused.
    if (lane == 0) atomicExch(p.status, kStatusWaitTimeout);
    for (int i2 = i; i2 < n_my && i2 < i + STAGES; ++i2)
      (void)wait_stage(&my_bars[i2 % STAGES], (i2 / STAGES) & 1);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) { m_run[nt][e] = -INFINITY; l_run[nt][e] = 0.f; }
  }

  // Row sums over the 8 token lanes of this warp.
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

  // ---- combine the warps and teams of this CTA ----------------------------
  __syncthreads();   // every stage consumed: the region holds the partials now
  float* co = reinterpret_cast<float*>(region);                  // [teams][32][128]
  float* cm = co + kTeams * kMaxCols * kHeadDim;                  // [teams][32]
  float* cl = cm + kTeams * kMaxCols;                             // [warps][32]
  if (gid == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int cc = nt * 8 + 2 * tig + e;
        if (rank == 0) cm[team * kMaxCols + cc] = m_run[nt][e];
        cl[warp * kMaxCols + cc] = l_run[nt][e];
      }
  }
  // O^T accumulators: dim 16*gid + 2*dt (+1 for c2/c3), column nt*8 + 2*tig + e.
#pragma unroll
  for (int dl = 0; dl < kDtPerWarp; ++dl) {
    const int dt = rank * kDtPerWarp + dl;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int cc = nt * 8 + 2 * tig + e;
        const float2 v2 = make_float2(o_acc[dl][nt][e], o_acc[dl][nt][2 + e]);
        *reinterpret_cast<float2*>(co + ((size_t)team * kMaxCols + cc) * kHeadDim + 16 * gid +
                                   2 * dt) = v2;
      }
  }
  __syncthreads();

  const int units_idx = (b * g.Hkv + kvh) * p.qgroups + qg;
  // Team weights exp2(m_team - M) for column cc; returns M (0 when empty) and
  // the combined row sum.
  auto team_weights = [&](int cc, float& M, float& Lsum, float (&wt)[kTeams]) {
    float mx = -INFINITY;
#pragma unroll
    for (int t = 0; t < kTeams; ++t) mx = fmaxf(mx, cm[t * kMaxCols + cc]);
    M = (mx == -INFINITY) ? 0.f : mx;
    Lsum = 0.f;
#pragma unroll
    for (int t = 0; t < kTeams; ++t) {
      wt[t] = exp2f(cm[t * kMaxCols + cc] - M);
      float lt = 0.f;
#pragma unroll
      for (int r2 = 0; r2 < TEAM; ++r2) lt += cl[(t * TEAM + r2) * kMaxCols + cc];
      Lsum += lt * wt[t];
    }
  };
  auto store_out = [&](int cc, int d4, float4 O, float Lsum, float M) {
    const int col = c0 + cc;
    const int jrow = col / G, h = kvh * G + col % G;
    const size_t orow = (size_t)(b * R + jrow) * g.Hq + h;
    const float sc = Lsum > 0.f ? p.v_scale / Lsum : 0.f;
    __nv_bfloat162 o01 = __floats2bfloat162_rn(O.x * sc, O.y * sc);
    __nv_bfloat162 o23 = __floats2bfloat162_rn(O.z * sc, O.w * sc);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&o01);
    packed.y = *reinterpret_cast<uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(p.out + orow * kHeadDim + d4) = packed;
    if (d4 == 0) p.lse[orow] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
  };

  if (p.splits == 1) {
    for (int idx = tid; idx < ncols * (kHeadDim / 4); idx += kThreads) {
      const int cc = idx / (kHeadDim / 4), d4 = (idx % (kHeadDim / 4)) * 4;
      float M, Lsum, wt[kTeams];
      team_weights(cc, M, Lsum, wt);
      float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int t = 0; t < kTeams; ++t) {
        const float4 v = *reinterpret_cast<const float4*>(co + ((size_t)t * kMaxCols + cc) * kHeadDim + d4);
        O.x += v.x * wt[t]; O.y += v.y * wt[t]; O.z += v.z * wt[t]; O.w += v.w * wt[t];
      }
      store_out(cc, d4, O, Lsum, M);
    }
    return;
  }

  // Split partial (log2 domain), then a ticket: the last split of this
  // (request, KV head, group) to arrive merges all of them in split order
  // (deterministic) and resets the ticket.
  float* part = p.partials + ((size_t)units_idx * p.splits + s) * kMaxCols * kPartStride;
  for (int idx = tid; idx < ncols * (kHeadDim / 4); idx += kThreads) {
    const int cc = idx / (kHeadDim / 4), d4 = (idx % (kHeadDim / 4)) * 4;
    float M, Lsum, wt[kTeams];
    team_weights(cc, M, Lsum, wt);
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int t = 0; t < kTeams; ++t) {
      const float4 v = *reinterpret_cast<const float4*>(co + ((size_t)t * kMaxCols + cc) * kHeadDim + d4);
      O.x += v.x * wt[t]; O.y += v.y * wt[t]; O.z += v.z * wt[t]; O.w += v.w * wt[t];
    }
    float* pc = part + (size_t)cc * kPartStride;
    *reinterpret_cast<float4*>(pc + 4 + d4) = O;
    if (d4 == 0) {
      pc[0] = (Lsum > 0.f) ? M : -INFINITY;
      pc[1] = Lsum;
    }
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

  // Merge: per-column max and weights first, then float4 sums over splits.
  const float* parts = p.partials + (size_t)units_idx * p.splits * kMaxCols * kPartStride;
  float* wsplit = reinterpret_cast<float*>(region);                 // [32][splits]
  float* lcol = wsplit + kMaxCols * p.splits;                       // [32]
  float* mcol = lcol + kMaxCols;                                    // [32]
  for (int cc = warp; cc < ncols; cc += kWarps) {
    float mloc = -INFINITY;
    for (int t = lane; t < p.splits; t += 32)
      mloc = fmaxf(mloc, __ldcg(parts + ((size_t)t * kMaxCols + cc) * kPartStride));
#pragma unroll
    for (int o = 16; o; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    const float base = (mloc == -INFINITY) ? 0.f : mloc;
    float lsum = 0.f;
    for (int t = lane; t < p.splits; t += 32) {
      const float* pc = parts + ((size_t)t * kMaxCols + cc) * kPartStride;
      const float wgt = exp2f(__ldcg(pc) - base);
      wsplit[cc * p.splits + t] = wgt;
      lsum += __ldcg(pc + 1) * wgt;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    if (lane == 0) {
      lcol[cc] = lsum;
      mcol[cc] = base;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < ncols * (kHeadDim / 4); idx += kThreads) {
    const int cc = idx / (kHeadDim / 4), d4 = (idx % (kHeadDim / 4)) * 4;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    const float* src = parts + (size_t)cc * kPartStride + 4 + d4;
    const float* wrow = wsplit + cc * p.splits;
    int t = 0;
    for (; t + 4 <= p.splits; t += 4) {
      float4 v[4];
#pragma unroll
      for (int u2 = 0; u2 < 4; ++u2)
        v[u2] = __ldcg(reinterpret_cast<const float4*>(src + (size_t)(t + u2) * kMaxCols * kPartStride));
#pragma unroll
      for (int u2 = 0; u2 < 4; ++u2) {
        const float wgt = wrow[t + u2];
        O.x += v[u2].x * wgt; O.y += v[u2].y * wgt; O.z += v[u2].z * wgt; O.w += v[u2].w * wgt;
      }
    }
    for (; t < p.splits; ++t) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(src + (size_t)t * kMaxCols * kPartStride));
      const float wgt = wrow[t];
      O.x += v.x * wgt; O.y += v.y * wgt; O.z += v.z * wgt; O.w += v.w * wgt;
    }
    store_out(cc, d4, O, lcol[cc], mcol[cc]);
  }
  if (tid == 0) atomicExch(&p.tickets[units_idx], 0);
}

constexpr size_t kWsHeader = 256;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int NT, int TEAM, int STAGES>
cudaError_t launch_t(const Params& prm, dim3 grid, int rows, int k, bool pdl,
                     cudaStream_t stream) {
  const size_t smem = Layout<NT, TEAM, STAGES>::bytes(rows, k);
  cudaError_t e = cudaFuncSetAttribute(sparse_decode_kernel<NT, TEAM, STAGES>,
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
  return cudaLaunchKernelEx(&cfg, sparse_decode_kernel<NT, TEAM, STAGES>, prm);
}

// Resident CTAs per SM of a variant, for split sizing.
template <int NT, int TEAM, int STAGES>
int resident_ctas(int rows, int k) {
  const size_t smem = Layout<NT, TEAM, STAGES>::bytes(rows, k);
  cudaFuncSetAttribute(sparse_decode_kernel<NT, TEAM, STAGES>,
                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sparse_decode_kernel<NT, TEAM, STAGES>,
                                                    kThreads, smem) != cudaSuccess) {
    cudaGetLastError();
    n = 2;
  }
  return n < 1 ? 1 : n;
}

int cols_tiles(const Geom& g) {
  const int cols = (g.Hq / g.Hkv) * g.R;
  const int cta_cols = cols < kMaxCols ? cols : kMaxCols;
  return (cta_cols + 7) / 8;
}

int rows_per_cta(const Geom& g, int qgroups) {
  const int G = g.Hq / g.Hkv;
  return qgroups == 1 ? g.R : min(g.R, (kMaxCols + G - 1) / G + 1);
}

#define QSA_DECODE_VARIANTS(X)                     \
  X(1, QSA_DECODE_TEAM_NT1, QSA_DECODE_STAGES_NT1) \
  X(2, 2, 4)                                       \
  X(3, 4, 4)                                       \
  X(4, 4, 4)

int variant_resident(int nt, int rows, int k) {
#define X(NT_, TEAM_, ST_) \
  if (nt == NT_) return resident_ctas<NT_, TEAM_, ST_>(rows, k);
  QSA_DECODE_VARIANTS(X)
#undef X
  return 1;
}

}  // namespace

DecodePlan plan_sparse_decode(const Geom& g, int k, int num_splits) {
  DecodePlan pl;
  const int G = g.Hq / g.Hkv;
  pl.cols = G * g.R;
  pl.qgroups = (pl.cols + kMaxCols - 1) / kMaxCols;
  const long long units = (long long)g.B * g.Hkv * pl.qgroups;
  const int rows = rows_per_cta(g, pl.qgroups);
  const int max_union = min(rows * k, g.MB);
  const int max_chunks = max(1, max_union * (g.P / kChunk));
  int splits = num_splits;
  if (splits <= 0) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaGetLastError();
    const int resident = variant_resident(cols_tiles(g), rows, k);
    const long long slots = (long long)sms * resident;
    // Fill every resident slot once; a CTA keeps at least 2 chunks.
    splits = (int)((slots + units - 1) / units);
    splits = min(splits, max(1, max_chunks / 2));
    splits = max(1, min(splits, 64));
  }
  pl.splits = splits;
  size_t ws = kWsHeader + align256((size_t)units * sizeof(int));
  if (splits > 1) ws += (size_t)units * splits * kMaxCols * kPartStride * sizeof(float);
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
  const int rows = rows_per_cta(g, plan.qgroups);
  dim3 grid(plan.splits, g.Hkv * plan.qgroups, g.B);
  const int nt = cols_tiles(g);
#define X(NT_, TEAM_, ST_) \
  if (nt == NT_) return launch_t<NT_, TEAM_, ST_>(prm, grid, rows, k, pdl, stream);
  QSA_DECODE_VARIANTS(X)
#undef X
  return cudaErrorInvalidValue;
}

}  // namespace qsa
