// qsa_attend.cu -- A3 for decode rows at head_dim 128: split-KV sparse GQA
// over the selected NVFP4 pages, each 64-token chunk shared by a group of
// four warps, partials merged by log-sum-exp.
//
// TensorRT-LLM PR #20937 ("GB300 perf work on
// qwen3_8_flash_next_nvfp4__sm_103__tp1"), What changes: NVFP4 sparse GQA
// decode as split-K + merge with a lean one-split variant; Per-File QA:
// invalid-page handling and masking.  PR #20276 ("Qwen3.8-Flash-Next NVFP4
// target"), Features table: uint8 e2m1 pages + e4m3 block scales.
//
// One CTA = (request b, KV head g, head slice, KV split s); its query columns
// are the slice's query heads (up to 32, padded to NT tiles of 8).  Split s
// takes the row's selected chunks s, s + splits, ...  One CTA per SM: the
// split count is planned so that the grid is one wave of clusters.
//
// Warp groups.  A group of four warps processes one chunk at a time:
//   S^T = K . Q^T   warp w takes tokens [16w, 16w + 16) of the chunk, every
//                   column; K is dequantised straight into mma.sync fragments
//   P               fp16, written to a shared tile [column][token] (stmatrix)
//   O^T += V^T.P^T  warp w takes dims [32w, 32w + 32) over all 64 tokens; V^T
//                   fragments are built from two tokens' nibbles per byte
// so a chunk's last arrival is turned around by four warps, not one.  All
// warps of a group share one softmax base per column, so O can be split by
// dims.  The base moves only when a logit exceeds it by more than 2^8 (log2
// domain): the common chunk costs one group barrier (a barrier-reduction
// that also tells whether any warp saw such a logit); the rare chunk that
// moves the base exchanges the group's column maxima, rescales O and
// rewrites P.
//
// Chunks stream in with TMA bulk copies (K codes 4 KB, V codes 4 KB, K and V
// scales 512 B each, contiguous in the pools) into per-group stages under
// mbarriers; every group requests all of its stages before its first chunk
// (four copy issuers per SM), and refills a stage as soon as it has finished
// it.  Waits sleep in hardware instead of spinning.
//
// Merge: each group's state (m, l per warp, O) is a partial record.  Up to 16
// splits form a thread-block cluster and push their records into the merging
// rank's shared memory (column c is merged by rank c mod splits); otherwise
// records go to the workspace and the last CTA of the unit to take its ticket
// merges them.  Every merge runs in a fixed order (deterministic).
//
// Every wait is bounded (2 s): a wait that gives up records a status word in
// the workspace, stops further copies, lets the copies in flight land and the
// kernel finishes.
#include "qsa_common.cuh"

#include <cooperative_groups.h>
#include <math.h>

#include <mutex>
#include <vector>

namespace cg = cooperative_groups;

namespace qsa {
namespace att {

constexpr int kD = 128;
constexpr int kChunk = 64;                    // tokens per stage
constexpr int kRowB = kD / 2;                 // code bytes per token row
constexpr int kSfB = kD / 16;                 // scale bytes per token row
constexpr int kKB = kChunk * kRowB;           // 4096
constexpr int kSB = kChunk * kSfB;            // 512
constexpr int kStage = 2 * kKB + 2 * kSB;     // 9216
constexpr int kGW = 4;                        // warps per group
constexpr int kGT = kGW * 32;                 // threads per group
constexpr int kPRow = 72;                     // halfs per P-tile row (64 tokens + pad)
constexpr int kRec = 8 + kD;                  // record: m, l[4 warps], pad[3], O[D]
constexpr int kMaxCols = 32;
// Bounds-check codes (reported by bounds-checked builds only).
[[maybe_unused]] constexpr int kChkList = 0x101;     // chunk-list slot past the list capacity
[[maybe_unused]] constexpr int kChkChunk = 0x102;    // listed chunk: slot, page id or token offset out of range
[[maybe_unused]] constexpr int kChkOut = 0x103;      // output row or dims out of range
[[maybe_unused]] constexpr int kChkRecord = 0x104;   // cluster record slot out of range
[[maybe_unused]] constexpr int kChkUnit = 0x105;     // workspace unit or split out of range
constexpr int kMaxCl = 16;                    // cluster size (non-portable above 8)
constexpr int kPtMax = 4096;                  // page-table rows up to this stay in smem
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazy = 8.f;                  // log2-domain headroom of the softmax base
constexpr unsigned long long kWaitNs = 2000000000ull;

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
  float* partials;      // [units][splits][NG][cols][kRec]
  int splits;           // KV splits per unit
  int slices;           // head slices per KV head
  int hs;               // heads per slice (column stride of a row)
  int cluster;          // >1: cluster merge over `cluster` = splits CTAs
  int list_cap;         // decode rows: chunk-list capacity per CTA
  unsigned long long wait_ns;   // bound of the waits for chunks (the drain keeps 2 s)
};

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// One wait for phase `parity` during which the thread sleeps in hardware
// until the phase completes or about 20 us pass (no spinning that would take
// issue slots from the warps that compute).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` for at most limit_ns; a bound below 1 us
// (a diagnostic setting) is a single probe that never suspends.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             unsigned long long limit_ns = kWaitNs) {
  if (limit_ns < 1000ull) return mbar_test_wait(bar, parity);
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Group barrier (named barrier 1 + group, the group's 128 threads).
__device__ __forceinline__ void group_sync(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(kGT) : "memory");
}
// Group barrier that also returns whether any participating thread passed p.
__device__ __forceinline__ bool group_sync_or(int id, bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
      "bar.red.or.pred b, %2, %3, a;\n\tselp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "r"(id), "r"(kGT)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Four e2m1 pairs (bytes of w) -> four fp16 pairs (byte i -> o[i], low nibble
// in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}
// Two e2m1 pairs (the low 16 bits of w) -> two fp16 pairs.
__device__ __forceinline__ void e2m1x4_to_f16x2x2(uint32_t w, uint32_t& o0, uint32_t& o1) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t}"
      : "=r"(o0), "=r"(o1)
      : "r"(w));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
__device__ __forceinline__ void stsm_x2_trans(uint32_t addr, uint32_t r0, uint32_t r1) {
  asm volatile("stmatrix.sync.aligned.m8n8.x2.trans.shared.b16 [%0], {%1,%2};" ::"r"(addr),
               "r"(r0), "r"(r1)
               : "memory");
}

// Position of 16-byte unit j (dims 8j .. 8j + 7) in row c of the query tile:
// a lane (gid, tig) reads unit 4 tig + wd of row nt*8 + gid, and the swizzle
// gives the eight rows' reads of one quarter-warp distinct bank groups.
__device__ __forceinline__ int qunit(int c, int j) {
  return j ^ ((j >> 3) & 1) ^ (2 * (c & 1));
}

// Shared-memory layout (bytes), shared by host sizing and the kernel.
template <int NT, int NG, int SG>
struct Lay {
  static constexpr int kCols = NT * 8;
  static constexpr int kThreads = NG * kGT;
  static constexpr int kStagesB = NG * SG * kStage;
  static constexpr int kBarB = NG * SG * 8;
  static constexpr int kQB = kCols * kD * 2;                  // q, fp16
  static constexpr int kPB = NG * 2 * kCols * kPRow * 2;      // P tiles, double-buffered
  static constexpr int kRedB = NG * 2 * kGW * kCols * 4;      // column maxima
  static constexpr int kColB = kCols * 4 * 3;                 // cq, n, row per column
  static constexpr int kMiscB = 64 * 4;
  static_assert(NG * SG * kStage >= 32768, "the row-mask scratch lives in the stages");
  // merge receive buffer: sources (CL splits x NG groups) x columns per rank
  __host__ __device__ static int rb_floats(int cl) {
    const int per = (kCols + cl - 1) / cl;
    return cl * NG * per * kRec;
  }
  // this CTA's chunk list: (page, first token) pairs
  __host__ __device__ static int list_ints(int list_cap) { return 2 * list_cap + 4; }
  static size_t bytes(int mb, int cl, int list_cap) {
    size_t off = (size_t)kStagesB + kBarB + kQB + kPB + kRedB + kColB + kMiscB;
    off += (size_t)rb_floats(cl) * 4;
    off += (size_t)list_ints(list_cap) * 4;
    off += mb <= kPtMax ? (size_t)mb * 4 : 0;
    return (off + 127) & ~(size_t)127;
  }
};


// One (request b, KV head kvh, head slice, split s) unit of work by the whole
// CTA.  wait_before_list() runs after the prologue (the queries, the page-table
// row and the length are in shared memory), before the row's selection is
// read; after_list() once this CTA's chunk list is built.
template <int NT, int NG, int SG, class Wait, class After>
__device__ __forceinline__ void attend_cta(const Params& p, int s, int kvh, int slice, int b,
                                           Wait&& wait_before_list, After&& after_list) {
  using L = Lay<NT, NG, SG>;
  constexpr int kCols = L::kCols;
  constexpr int kThreads = L::kThreads;

  const Geom& g = p.g;
  const int R = g.R;
  const int G = g.Hq / g.Hkv;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int grp = warp / kGW, wg = warp % kGW;
  const int hs = p.hs;
  const int h0 = slice * hs;
  const int hreal = min(hs, G - h0);
  const int k = p.k;
  const int csh = g.P == 2 * kChunk ? 1 : 0;           // chunks per page: 1 << csh
  const int CL = p.splits == 1 ? 1 : (p.cluster > 1 ? p.cluster : 0);

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  size_t off = L::kStagesB;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + off);
  off += L::kBarB;
  __half* qs = reinterpret_cast<__half*>(smem + off);
  off += L::kQB;
  __half* ptile = reinterpret_cast<__half*>(smem + off);   // [NG][2][kCols][kPRow]
  off += L::kPB;
  float* red = reinterpret_cast<float*>(smem + off);       // [NG][2][kGW][kCols]
  off += L::kRedB;
  float* col_cq = reinterpret_cast<float*>(smem + off);
  int* col_n = reinterpret_cast<int*>(col_cq + kCols);
  int* col_row = col_n + kCols;
  off += L::kColB;
  int* misc = reinterpret_cast<int*>(smem + off);
  off += L::kMiscB;
  float* rb = reinterpret_cast<float*>(smem + off);
  off += (size_t)L::rb_floats(CL > 0 ? CL : 1) * 4;
  int32_t* lists = reinterpret_cast<int32_t*>(smem + off);
  off += (size_t)L::list_ints(p.list_cap) * 4;
  int32_t* s_pt = reinterpret_cast<int32_t*>(smem + off);

  if (tid == 0) {
    for (int i = 0; i < NG * SG; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  // Matched by the wait before the first remote write of the merge.
  if (CL > 1) cluster_arrive_relaxed();

  // ---- before the dependency wait: step inputs no kernel of the step writes ----
  // The page-table row goes to shared memory by asynchronous copies, so its
  // loads, the queries' and the length's are all in flight together.
  const bool pt_smem = g.MB <= kPtMax;
  if (pt_smem)
    for (int i = tid; i < g.MB; i += kThreads)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(s_pt + i)),
                   "l"(p.page_table + (size_t)b * g.MB + i)
                   : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
  const int Lb = p.seqlens[b];
  const int cap = g.MB * g.P;
  // Queries -> fp16 pre-scaled by a power of two per column (|q|max into
  // [256, 512): exact, and any bf16 magnitude stays inside fp16 range), one
  // warp per column, four dims per lane.
  for (int c = warp; c < kCols; c += NG * kGW) {
    const int j = c / hs, hh = c - (c / hs) * hs;
    const bool real = j < R && hh < hreal;
    uint2 raw = make_uint2(0u, 0u);
    if (real) {
      const int h = kvh * G + h0 + hh;
      raw = *reinterpret_cast<const uint2*>(p.q + ((size_t)(b * R + j) * g.Hq + h) * kD + 4 * lane);
    }
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    const float v0 = __low2float(lo), v1 = __high2float(lo);
    const float v2 = __low2float(hi), v3 = __high2float(hi);
    float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int ebits = (int)((__float_as_uint(amax) >> 23) & 0xFF);
    int sq = (amax > 0.f) ? 135 - ebits : 0;
    sq = sq > 126 ? 126 : (sq < -126 ? -126 : sq);
    const float up = __uint_as_float((uint32_t)(sq + 127) << 23);
    const float down = __uint_as_float((uint32_t)(127 - sq) << 23);
    // 16-byte unit j = lane / 2 of the row sits at qunit(c, j) (a swizzle
    // that spreads the fragment reads below over all banks).
    __half2* dst = reinterpret_cast<__half2*>(qs + c * kD + 8 * qunit(c, lane >> 1) + 4 * (lane & 1));
    dst[0] = __floats2half2_rn(v0 * up, v1 * up);
    dst[1] = __floats2half2_rn(v2 * up, v3 * up);
    if (lane == 0) {
      col_cq[c] = real ? p.k_scale * p.sm_scale * kLog2e * down : 0.f;
      col_n[c] = real ? visible_tokens(Lb, R, j, cap) : 0;
      col_row[c] = real ? j : -1;
    }
  }
  if (tid == 0) misc[1] = 0;   // set when a bounded wait gives up
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  wait_before_list();   // the selections come from an earlier kernel or CTA

  // ---- this CTA's chunks ----------------------------------------------------
  // Candidate chunk c of the row (entry c >> csh, part c & csh) belongs to
  // split c mod splits; entries repeating their predecessor (the selection is
  // ascending) or on an invalid page are dropped.
  if (warp == 0) {
    const int nc = k << csh;
    const int32_t* selrow = p.sel + (size_t)b * k;
    int cnt = 0;
    for (int m0 = 0;; m0 += 32) {
      if (s + (long long)p.splits * m0 >= nc) break;
      const long long c = s + (long long)p.splits * (m0 + lane);
      int page = -1, tok0 = 0;
      if (c < nc) {
        const int e = (int)(c >> csh);
        const int beta = __ldcg(selrow + e);
        const int prev = e > 0 ? __ldcg(selrow + e - 1) : -1;
        if (beta >= 0 && beta < g.MB && beta != prev) {
          const int pg = pt_smem ? s_pt[beta] : p.page_table[(size_t)b * g.MB + beta];
          if (pg >= 0 && pg < g.NP) {
            page = pg;
            tok0 = beta * g.P + (int)(c & csh) * kChunk;
          }
        }
      }
      const unsigned vm = __ballot_sync(0xffffffffu, page >= 0);
      if (page >= 0) {
        const int q = cnt + __popc(vm & ((1u << lane) - 1u));
        if (QSA_GUARD(q < p.list_cap, kChkList)) {
          lists[2 * q] = page;
          lists[2 * q + 1] = tok0;
        }
      }
      cnt += __popc(vm);
    }
    if (lane == 0) misc[0] = min(cnt, p.list_cap);
  }
  __syncthreads();
  const int nch = misc[0];
  after_list();

  // Chunk m of this CTA: candidate chunk s + m * splits of the row.
  auto chunk_of = [&](int m, int& page, int& tok0, int& mask) {
    page = lists[2 * m];
    tok0 = lists[2 * m + 1];
    mask = 1;
  };
  const uint64_t pol = policy_evict_first();
  // Chunk m goes to group m % NG, its stage (m / NG) % SG.
  auto issue = [&](int m) {
    int page, tok0, mask;
    chunk_of(m, page, tok0, mask);
    const int st = (m % NG) * SG + (m / NG) % SG;
    if (!QSA_IN_BOUNDS(m >= 0 && m < p.list_cap && page >= 0 && page < g.NP && tok0 >= 0 &&
                           tok0 < cap && (tok0 & (g.P - 1)) + kChunk <= g.P,
                       kChkChunk))
      return;
    const size_t row0 = ((size_t)page * g.Hkv + kvh) * g.P + (size_t)(tok0 & (g.P - 1));
    uint8_t* dst = stages + (size_t)st * kStage;
    mbar_arrive_expect_tx(&full[st], kStage);
    bulk_g2s(dst, p.k_pool + row0 * kRowB, kKB, &full[st], pol);
    bulk_g2s(dst + kKB, p.v_pool + row0 * kRowB, kKB, &full[st], pol);
    bulk_g2s(dst + 2 * kKB, p.k_sf + row0 * kSfB, kSB, &full[st], pol);
    bulk_g2s(dst + 2 * kKB + kSB, p.v_sf + row0 * kSfB, kSB, &full[st], pol);
  };
  const int nloc = nch > grp ? (nch - grp + NG - 1) / NG : 0;   // this group's chunks
  // Every stage of the CTA is requested now, one lane per chunk.
  if (wg == 0 && lane < SG && lane < nloc) {
    fence_proxy_async_smem();   // after the union's scratch in the stage region
    issue(grp + NG * lane);
  }

  // ---- per-column state and fragments --------------------------------------
  // Per lane column: cq, and the row (low 4 bits, 15 = padding) with the
  // row's visible tokens (upper bits) in one word.
  float cq[NT][2];
  int crn[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int c = nt * 8 + 2 * tig + e;
      cq[nt][e] = col_cq[c];
      crn[nt][e] = (col_n[c] << 4) | (col_row[c] < 0 ? 15 : col_row[c]);
    }
  auto crow_of = [&](int nt, int e) { return crn[nt][e] & 15; };   // 15: padding
  auto cn_of = [&](int nt, int e) { return crn[nt][e] >> 4; };
  // Q^T fragments: column nt*8 + gid, dims [32 tig, 32 tig + 32) = units
  // 4 tig .. 4 tig + 3 of the row.
  uint32_t qf[NT][16];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int c = nt * 8 + gid;
#pragma unroll
    for (int v4 = 0; v4 < 4; ++v4) {
      const uint4 x = *reinterpret_cast<const uint4*>(qs + c * kD + 8 * qunit(c, 4 * tig + v4));
      qf[nt][4 * v4 + 0] = x.x; qf[nt][4 * v4 + 1] = x.y;
      qf[nt][4 * v4 + 2] = x.z; qf[nt][4 * v4 + 3] = x.w;
    }
  }
  float base[NT][2], lsum[NT][2];
  float o[2][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) { base[nt][e] = -INFINITY; lsum[nt][e] = 0.f; }
#pragma unroll
  for (int dt = 0; dt < 2; ++dt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[dt][nt][e] = 0.f;

  // Rows covered by each column tile (over the tile's 8 columns), and the
  // fewest tokens any real column sees: chunks below that need no per-token
  // visibility test.
  int trows[NT];
  int nmin = 0x7FFFFFFF;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    int r = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (crow_of(nt, e) != 15) {
        r |= 1 << crow_of(nt, e);
        nmin = min(nmin, cn_of(nt, e));
      }
    r |= __shfl_xor_sync(0xffffffffu, r, 1);
    r |= __shfl_xor_sync(0xffffffffu, r, 2);
    trows[nt] = r;
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) nmin = min(nmin, __shfl_xor_sync(0xffffffffu, nmin, o));

  // MMA row gid of a 16-token tile <-> token (gid >> 1) + 4 (gid & 1) (and +8);
  // in the P tile that token sits at position gid, which is the order the
  // V^T fragments below pair tokens in (tokens t, t + 4 | t + 8, t + 12).
  const int rA = (gid >> 1) + 4 * (gid & 1);
  const int bar_id = 1 + grp;
  bool dead = false;
  int confirmed = 0;             // issuer: chunks whose copies are known to have landed
  int issued = min(SG, nloc);    // issuer: chunks requested so far

  for (int l = 0; l < nloc; ++l) {
    const int m = grp + NG * l;
    const int st = grp * SG + l % SG;
    const uint8_t* tile = stages + (size_t)st * kStage;
    if (!dead) {
      if (wait_bounded(&full[st], (l / SG) & 1, p.wait_ns)) {
        if (wg == 0 && lane == 0) confirmed = l + 1;
      } else {
        dead = true;
        if (lane == 0) {
          atomicExch(p.status, kStatusWaitTimeout);
          misc[1] = 1;
        }
      }
    }
    int page, tok0, mask;
    chunk_of(m, page, tok0, mask);
    (void)page;
    // Column tiles with a row that selected this chunk (the others' MMAs,
    // logits and P are skipped: their columns get nothing from it).
    bool act[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) act[nt] = (mask & trows[nt]) != 0;

    // ---- S^T = K . Q^T for this warp's 16 tokens ----------------------------
    // With few column tiles the k-steps alternate between two accumulator
    // sets, halving the dependent MMA chain.
    constexpr int KS = NT <= 2 ? 2 : 1;
    float sacc[NT][4], sacc2[KS][NT][4];
#pragma unroll
    for (int u = 0; u < KS; ++u)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc2[u][nt][e] = 0.f;
    {
      const uint8_t* kr = tile + (16 * wg + rA) * kRowB + 16 * tig;
      const uint4 kA = *reinterpret_cast<const uint4*>(kr);
      const uint4 kB = *reinterpret_cast<const uint4*>(kr + 8 * kRowB);
      const uint8_t* sr = tile + 2 * kKB + (16 * wg + rA) * kSfB + 2 * tig;
      const uint32_t sA = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sr));
      const uint32_t sB = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sr + 8 * kSfB));
      const uint32_t scA[2] = {prmt(sA, 0, 0x1010), prmt(sA, 0, 0x3232)};
      const uint32_t scB[2] = {prmt(sB, 0, 0x1010), prmt(sB, 0, 0x3232)};
      const uint32_t wA[4] = {kA.x, kA.y, kA.z, kA.w};
      const uint32_t wB[4] = {kB.x, kB.y, kB.z, kB.w};
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        uint32_t fa[4], fb[4];
        e2m1x8_to_f16x2x4(wA[wd], fa);
        e2m1x8_to_f16x2x4(wB[wd], fb);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int kk = 2 * wd + h;
          uint32_t a[4];
          a[0] = hmul2_u32(fa[2 * h], scA[wd >> 1]);
          a[2] = hmul2_u32(fa[2 * h + 1], scA[wd >> 1]);
          a[1] = hmul2_u32(fb[2 * h], scB[wd >> 1]);
          a[3] = hmul2_u32(fb[2 * h + 1], scB[wd >> 1]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            if (act[nt]) mma_f16_16816(sacc2[kk % KS][nt], a, qf[nt][2 * kk], qf[nt][2 * kk + 1]);
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] = KS == 2 ? sacc2[0][nt][e] + sacc2[KS - 1][nt][e]
                                                        : sacc2[0][nt][e];

    // ---- logits (log2 domain, minus the base), masks ------------------------
    // t = z - base with z = sacc * cq.  A column whose row did not select the
    // chunk gets -inf (cq 0, offset -inf); with no base yet, any visible
    // logit sets one (threshold -inf); tokens past a column's visible length
    // get -inf, tested only in chunks that reach past the shortest row.
    const int tokA = tok0 + 16 * wg + rA, tokB = tokA + 8;
    const bool partial = tok0 + kChunk > nmin;
    bool exceed = false;
    // From here sacc[nt][e] / sacc[nt][2 + e] hold the logits t of the
    // lane's tokens A / B.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (!act[nt]) continue;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool on = ((mask >> crow_of(nt, e)) & 1) != 0;   // padding: bit 15 is 0
        const bool nobase = base[nt][e] == -INFINITY;
        const float c = on ? cq[nt][e] : 0.f;
        const float nb = on ? (nobase ? 0.f : -base[nt][e]) : -INFINITY;
        const float thr = nobase ? -INFINITY : kLazy;
        float za = fmaf(sacc[nt][e], c, nb);
        float zb = fmaf(sacc[nt][2 + e], c, nb);
        if (partial) {
          const int lim = on ? cn_of(nt, e) : 0;
          za = tokA < lim ? za : -INFINITY;
          zb = tokB < lim ? zb : -INFINITY;
        }
        sacc[nt][e] = za;
        sacc[nt][2 + e] = zb;
        exceed |= (za > thr) | (zb > thr);
      }
    }
    __half* pt = ptile + (size_t)((grp * 2 + (l & 1)) * kCols) * kPRow;
    float psum[NT][2];
    auto write_p = [&]() {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (!act[nt]) continue;
        float pa[2], pb[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pa[e] = exp2f(sacc[nt][e]);
          pb[e] = exp2f(sacc[nt][2 + e]);
          psum[nt][e] = pa[e] + pb[e];
        }
        const uint32_t r0 = pack_half2(pa[0], pa[1]);
        const uint32_t r1 = pack_half2(pb[0], pb[1]);
        // lanes 0-7: rows (columns) of positions 0-7, lanes 8-15: positions 8-15
        const int rr = lane & 7, half = (lane >> 3) & 1;
        stsm_x2_trans(smem_u32(pt + (nt * 8 + rr) * kPRow + 16 * wg + 8 * half), r0, r1);
      }
    };
    write_p();
    const bool any = group_sync_or(bar_id, exceed);
    if (any) {
      // Rare: the group moves the base of the columns whose maximum rose.
      float* rd = red + (size_t)((grp * 2 + (l & 1)) * kGW) * kCols;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = act[nt] ? fmaxf(sacc[nt][e], sacc[nt][2 + e]) : -INFINITY;
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
          if (gid == 0) rd[wg * kCols + nt * 8 + 2 * tig + e] = v;
        }
      group_sync(bar_id);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (!act[nt]) continue;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = nt * 8 + 2 * tig + e;
          float cm = fmaxf(fmaxf(rd[c], rd[kCols + c]), fmaxf(rd[2 * kCols + c], rd[3 * kCols + c]));
          // cm is relative to the old base (or absolute when there was none).
          const float thr = base[nt][e] == -INFINITY ? -INFINITY : kLazy;
          if (cm > thr) {
            const float ob = base[nt][e] == -INFINITY ? 0.f : base[nt][e];
            const float nbv = ob + cm;                    // new base, absolute
            const float alpha = base[nt][e] == -INFINITY ? 0.f : exp2f(-cm);
            lsum[nt][e] *= alpha;
#pragma unroll
            for (int dt = 0; dt < 2; ++dt) {
              o[dt][nt][e] *= alpha;
              o[dt][nt][2 + e] *= alpha;
            }
            sacc[nt][e] -= cm;
            sacc[nt][2 + e] -= cm;
            base[nt][e] = nbv;
          }
        }
      }
      write_p();
      group_sync(bar_id);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      if (act[nt])
#pragma unroll
        for (int e = 0; e < 2; ++e) lsum[nt][e] += psum[nt][e];

    // The stage of the group's previous chunk is free: every warp has passed
    // this chunk's barrier, so their reads of it are done.
    if (wg == 0 && lane == 0 && l >= 1 && issued < nloc && issued == l - 1 + SG) {
      if (!dead && misc[1] == 0) {
        fence_proxy_async_smem();
        issue(grp + NG * issued);
        ++issued;
      }
    }

    // ---- O^T += V^T . P^T for this warp's 32 dims ---------------------------
    {
      const uint8_t* vt = tile + kKB;
      const uint8_t* vs = tile + 2 * kKB + kSB;
      const int bo = 16 * wg + 2 * gid;             // the lane's two bytes of a token row
      const int sblk = 2 * wg + (gid >> 2);         // their scale block
      const uint32_t pbase = smem_u32(pt);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int t0 = 16 * ks + tig;
        const uint32_t X = *reinterpret_cast<const uint16_t*>(vt + t0 * kRowB + bo);
        const uint32_t Y = *reinterpret_cast<const uint16_t*>(vt + (t0 + 4) * kRowB + bo);
        const uint32_t X2 = *reinterpret_cast<const uint16_t*>(vt + (t0 + 8) * kRowB + bo);
        const uint32_t Y2 = *reinterpret_cast<const uint16_t*>(vt + (t0 + 12) * kRowB + bo);
        const uint32_t s01 = e4m3x2_to_f16x2((uint32_t)vs[t0 * kSfB + sblk] |
                                             ((uint32_t)vs[(t0 + 4) * kSfB + sblk] << 8));
        const uint32_t s23 = e4m3x2_to_f16x2((uint32_t)vs[(t0 + 8) * kSfB + sblk] |
                                             ((uint32_t)vs[(t0 + 12) * kSfB + sblk] << 8));
        // byte i: low nibble from token t (X), high nibble from token t + 4 (Y)
        const uint32_t LO = (X & 0x0F0Fu) | ((Y << 4) & 0xF0F0u);
        const uint32_t HI = ((X >> 4) & 0x0F0Fu) | (Y & 0xF0F0u);
        const uint32_t LO2 = (X2 & 0x0F0Fu) | ((Y2 << 4) & 0xF0F0u);
        const uint32_t HI2 = ((X2 >> 4) & 0x0F0Fu) | (Y2 & 0xF0F0u);
        uint32_t f0[2], f1[2], f2[2], f3[2];
        e2m1x4_to_f16x2x2(LO, f0[0], f0[1]);
        e2m1x4_to_f16x2x2(HI, f1[0], f1[1]);
        e2m1x4_to_f16x2x2(LO2, f2[0], f2[1]);
        e2m1x4_to_f16x2x2(HI2, f3[0], f3[1]);
        uint32_t a[2][4];
#pragma unroll
        for (int dt = 0; dt < 2; ++dt) {
          a[dt][0] = hmul2_u32(f0[dt], s01);
          a[dt][1] = hmul2_u32(f1[dt], s01);
          a[dt][2] = hmul2_u32(f2[dt], s23);
          a[dt][3] = hmul2_u32(f3[dt], s23);
        }
        // P^T fragments: column nt*8 + gid, positions 16 ks + 2 tig (+8).
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
          if (!act[nt] && !(nt + 1 < NT && act[nt + 1])) continue;
          const int mat = lane >> 3, rr = lane & 7;
          uint32_t b0, b1, b2, b3;
          if (nt + 1 < NT) {
            const int col = (nt + (mat >> 1)) * 8 + rr;
            ldsm_x4(pbase + (uint32_t)((col * kPRow + 16 * ks + 8 * (mat & 1)) * 2), b0, b1, b2,
                    b3);
          } else {
            const int col = nt * 8 + rr;
            ldsm_x2(pbase + (uint32_t)((col * kPRow + 16 * ks + 8 * (mat & 1)) * 2), b0, b1);
            b2 = b3 = 0u;
          }
#pragma unroll
          for (int dt = 0; dt < 2; ++dt) {
            if (act[nt]) mma_f16_16816(o[dt][nt], a[dt], b0, b1);
            if (nt + 1 < NT && act[nt + 1]) mma_f16_16816(o[dt][nt + 1], a[dt], b2, b3);
          }
        }
      }
    }
  }

  // After a wait gave up: stop, and let this group's copies still in flight
  // land before the CTA leaves (the issuer knows which those are).
  if (wg == 0 && lane == 0 && (dead || misc[1] != 0))
    for (int l = confirmed; l < issued; ++l)
      if (!wait_bounded(&full[grp * SG + l % SG], (l / SG) & 1)) break;

  // Row sums over the 8 token lanes of the warp.
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = lsum[nt][e];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      lsum[nt][e] = v;
    }

  // ---- records: (m, l per warp, O) of this group per column ---------------
  // O^T accumulators: o[dt][nt][e] = (dim 32 wg + 4 gid + 2 dt, column
  // nt*8 + 2 tig + e), o[dt][nt][2 + e] the next dim.
  auto write_record = [&](float* rec, int nt, int e) {
    *reinterpret_cast<float4*>(rec + 8 + 32 * wg + 4 * gid) =
        make_float4(o[0][nt][e], o[0][nt][2 + e], o[1][nt][e], o[1][nt][2 + e]);
    if (gid == 0) {
      rec[1 + wg] = lsum[nt][e];
      if (wg == 0) rec[0] = base[nt][e];
    }
  };
  auto store_out = [&](int c, int d4, float4 O, float Lsum, float M) {
    const int j = c / hs, hh = c - (c / hs) * hs;
    if (j >= R || hh >= hreal) return;   // padding column
    const int h = kvh * G + h0 + hh;
    const size_t orow = (size_t)(b * R + j) * g.Hq + h;
    if (!QSA_IN_BOUNDS(b < g.B && h < g.Hq && d4 + 4 <= kD, kChkOut)) return;
    const float sc = Lsum > 0.f ? p.v_scale / Lsum : 0.f;
    __nv_bfloat162 o01 = __floats2bfloat162_rn(O.x * sc, O.y * sc);
    __nv_bfloat162 o23 = __floats2bfloat162_rn(O.z * sc, O.w * sc);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&o01);
    packed.y = *reinterpret_cast<uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(p.out + orow * kD + d4) = packed;
    if (d4 == 0) p.lse[orow] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
  };
  // Merges `nsrc` records per column, record i at rec_at(i) (workspace
  // records are read past L1: other CTAs wrote them).
  auto merge = [&](int nsrc, auto rec_at, int c, int d4, bool global) {
    auto ld = [&](const float* a) { return global ? __ldcg(a) : *a; };
    float M = -INFINITY;
    for (int i = 0; i < nsrc; ++i) M = fmaxf(M, ld(rec_at(i)));
    const float Mb = M == -INFINITY ? 0.f : M;
    float Lsum = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < nsrc; ++i) {
      const float* r = rec_at(i);
      const float w = exp2f(ld(r) - Mb);
      Lsum += (ld(r + 1) + ld(r + 2) + ld(r + 3) + ld(r + 4)) * w;
      const float4 v = global ? __ldcg(reinterpret_cast<const float4*>(r + 8 + d4))
                              : *reinterpret_cast<const float4*>(r + 8 + d4);
      O.x += v.x * w; O.y += v.y * w; O.z += v.z * w; O.w += v.w * w;
    }
    store_out(c, d4, O, Lsum, M);
  };

  if (CL >= 1) {
    // Local (one split) or cluster merge: column c is merged by rank c % CL;
    // record slot [split * NG + group][c / CL] of that rank's receive buffer.
    const int per = (kCols + CL - 1) / CL;
    if (CL > 1) {
      cg::cluster_group cluster = cg::this_cluster();
      cluster_wait_acquire();   // pairs with the arrival at the start
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = nt * 8 + 2 * tig + e;
          float* dst = cluster.map_shared_rank(rb, c % CL) +
                       ((size_t)(s * NG + grp) * per + c / CL) * kRec;
          if (QSA_IN_BOUNDS(s < CL && c < kCols, kChkRecord)) write_record(dst, nt, e);
        }
      cluster_arrive_release();
      cluster_wait_acquire();
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = nt * 8 + 2 * tig + e;
          write_record(rb + ((size_t)grp * per + c) * kRec, nt, e);
        }
      __syncthreads();
    }
    const int nsrc = CL * NG;
    for (int idx = tid; idx < per * (kD / 4); idx += kThreads) {
      const int q = idx / (kD / 4), d4 = (idx % (kD / 4)) * 4;
      const int c = q * CL + s;
      if (c >= kCols) continue;
      merge(nsrc, [&](int i) { return rb + ((size_t)i * per + q) * kRec; }, c, d4, false);
    }
    return;
  }

  // Ticket merge: records to the workspace; the last split of this unit to
  // arrive merges them in split order and resets the ticket.
  const int unit = (b * g.Hkv + kvh) * p.slices + slice;
  if (!QSA_IN_BOUNDS(b < g.B && kvh < g.Hkv && slice < p.slices && s < p.splits, kChkUnit))
    return;
  float* mine = p.partials + ((size_t)(unit * p.splits + s) * NG + grp) * kCols * kRec;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) write_record(mine + (size_t)(nt * 8 + 2 * tig + e) * kRec, nt, e);
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&p.tickets[unit], 1);
    misc[2] = (prev == p.splits - 1);
  }
  __syncthreads();
  if (!misc[2]) return;
  __threadfence();
  const float* parts = p.partials + (size_t)unit * p.splits * NG * kCols * kRec;
  for (int idx = tid; idx < kCols * (kD / 4); idx += kThreads) {
    const int c = idx / (kD / 4), d4 = (idx % (kD / 4)) * 4;
    merge(p.splits * NG, [&](int i) { return parts + ((size_t)i * kCols + c) * kRec; }, c, d4,
          true);
  }
  if (tid == 0) atomicExch(&p.tickets[unit], 0);
}

template <int NT, int NG, int SG>
__global__ void __launch_bounds__(Lay<NT, NG, SG>::kThreads, 1)
attend_kernel(Params p) {
  attend_cta<NT, NG, SG>(
      p, blockIdx.x, blockIdx.y / p.slices, blockIdx.y % p.slices, blockIdx.z,
      [] { pdl_wait(); }, [] { pdl_trigger(); });
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

constexpr size_t kWsHeader = 256;
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Kernel variants: one CTA per SM with 16 stages (147 KB), 16 warps for one
// column tile and 8 warps for wider ones (their fragments take 160 to 240
// registers).
template <int NT_, int NG_, int SG_>
struct Var {
  static constexpr int NT = NT_, NG = NG_, SG = SG_;
  using L = Lay<NT_, NG_, SG_>;
  static constexpr auto kernel = attend_kernel<NT_, NG_, SG_>;
};
// X(NT, NG, SG)
#define QSA_ATT_VARIANTS(X) \
  X(1, 4, 4)                \
  X(2, 2, 8)                \
  X(3, 2, 8)                \
  X(4, 2, 8)

int heads_per_slice(const Geom& g) {
  const int G = g.Hq / g.Hkv;
  int hs = kMaxCols / g.R;
  if (hs > G) hs = G;
  if (hs < 1) hs = 1;
  // Equal slices: the fewest slices, then the narrowest width that keeps it.
  const int slices = (G + hs - 1) / hs;
  return (G + slices - 1) / slices;
}

int ntiles(const Geom& g) { return (g.R * heads_per_slice(g) + 7) / 8; }

int list_cap_for(const Geom& g, int k, int splits) {
  const int cpp = g.P / kChunk;
  return (k * cpp + splits - 1) / splits;
}

template <class V>
size_t smem_for(const Geom& g, int k, int cl, int splits) {
  return V::L::bytes(g.MB, cl, list_cap_for(g, k, splits));
}

template <class V>
cudaLaunchConfig_t make_config(dim3 grid, size_t smem, cudaStream_t stream,
                               cudaLaunchAttribute* attr, bool pdl, int cluster) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(V::L::kThreads);
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

template <class V>
void set_smem_attr(size_t smem, int cl) {
  cudaFuncSetAttribute(V::kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (cl > 8) cudaFuncSetAttribute(V::kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

// Clusters of `cl` CTAs of this variant that can be resident at once (0 when
// none can); sizes above 8 need the non-portable cluster attribute.
template <class V>
int cluster_capacity(int cl, size_t smem) {
  struct Entry { int dev, cl; size_t smem; int n; };
  static std::mutex mu;
  static std::vector<Entry> cache;
  if (cl < 2 || cl > kMaxCl) return 0;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
      if (e.dev == dev && e.cl == cl && e.smem == smem) return e.n;
  }
  set_smem_attr<V>(smem, cl);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_config<V>(dim3(cl, 1, 1), smem, 0, attr, false, cl);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, V::kernel, &cfg) != cudaSuccess) n = 0;
  cudaGetLastError();
  std::lock_guard<std::mutex> lock(mu);
  cache.push_back({dev, cl, smem, n});
  return n;
}

// Largest split count (up to a 16-CTA cluster) that keeps the grid in one
// wave: units * splits CTAs resident at once, every cluster of `splits`
// co-resident, and at least one chunk per warp group.
template <class V>
int plan_splits(const Geom& g, int k, long long units, int max_chunks) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaGetLastError();
  const size_t smem1 = smem_for<V>(g, k, 1, 1);
  set_smem_attr<V>(smem1, 1);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, V::kernel, V::L::kThreads, smem1) !=
      cudaSuccess)
    per_sm = 1;
  cudaGetLastError();
  const long long slots = (long long)sms * (per_sm < 1 ? 1 : per_sm);
  int best = 1;
  for (int sp = 2; sp <= kMaxCl; ++sp) {
    if (units * sp > slots || max_chunks / sp < V::NG) break;
    const int cap = cluster_capacity<V>(sp, smem_for<V>(g, k, sp, sp));
    if (cap * sp >= units * sp && cap >= units) best = sp;
  }
  return best;
}

template <class V>
cudaError_t launch_t(Params prm, dim3 grid, const Geom& g, int k, bool pdl, cudaStream_t stream) {
  int cl = 1;
  if (prm.splits > 1 && prm.splits <= kMaxCl) {
    const size_t smem_cl = smem_for<V>(g, k, prm.splits, prm.splits);
    if (cluster_capacity<V>(prm.splits, smem_cl) > 0) cl = prm.splits;
  }
  prm.cluster = cl;
  const size_t smem = smem_for<V>(g, k, prm.splits == 1 ? 1 : (cl > 1 ? cl : 1), prm.splits);
  set_smem_attr<V>(smem, cl);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_config<V>(grid, smem, stream, attr, pdl, cl);
  return cudaLaunchKernelEx(&cfg, V::kernel, prm);
}

// Runs fn.template operator()<V>() for the variant serving g.
template <class F>
auto with_variant(const Geom& g, F&& fn) -> decltype(fn.template operator()<Var<1, 4, 4>>()) {
  const int nt = ntiles(g);
#define X(NT_, NG_, SG_) \
  if (nt == NT_) return fn.template operator()<Var<NT_, NG_, SG_>>();
  QSA_ATT_VARIANTS(X)
#undef X
  return fn.template operator()<Var<1, 4, 4>>();
}

}  // namespace att

// Whether this kernel serves the geometry: decode rows at head_dim 128.
bool attend_supports(const Geom& g) { return g.D == att::kD && g.R == 1; }

DecodePlan plan_attend(const Geom& g, int k, int num_splits) {
  DecodePlan pl;
  const int G = g.Hq / g.Hkv;
  const int hs = att::heads_per_slice(g);
  const int nt = att::ntiles(g);
  pl.qgroups = (G + hs - 1) / hs;
  pl.cols = nt * 8;
  const long long units = (long long)g.B * g.Hkv * pl.qgroups;
  const int cpp = g.P / att::kChunk;
  const int max_union = min(g.R * k, g.MB);
  const int max_chunks = max(1, max_union * cpp);
  int splits = num_splits;
  if (splits <= 0)
    splits = att::with_variant(g, [&]<class V>() { return att::plan_splits<V>(g, k, units, max_chunks); });
  pl.splits = splits;
  const int ng = att::with_variant(g, [&]<class V>() { return V::NG; });
  size_t ws = att::kWsHeader + att::align256((size_t)units * sizeof(int));
  if (splits > 1) ws += (size_t)units * splits * ng * pl.cols * att::kRec * sizeof(float);
  pl.ws_bytes = ws;
  return pl;
}

cudaError_t launch_attend(const Geom& g, const DecodePlan& plan, const void* q,
                          const uint8_t* k_pool, const uint8_t* k_sf, const uint8_t* v_pool,
                          const uint8_t* v_sf, float k_scale, float v_scale, float sm_scale,
                          const int32_t* page_table, const int32_t* seqlens, const int32_t* sel,
                          int k, void* out, float* lse, void* workspace, bool pdl,
                          cudaStream_t stream) {
  att::Params prm;
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
  prm.tickets = reinterpret_cast<int*>(ws + att::kWsHeader);
  prm.partials = reinterpret_cast<float*>(ws + att::kWsHeader +
                                          att::align256((size_t)units * sizeof(int)));
  prm.splits = plan.splits;
  prm.slices = plan.qgroups;
  prm.hs = att::heads_per_slice(g);
  prm.cluster = 1;
  prm.list_cap = att::list_cap_for(g, k, plan.splits);
  prm.wait_ns = wait_limit_ns();
  dim3 grid(plan.splits, g.Hkv * plan.qgroups, g.B);
  return att::with_variant(g, [&]<class V>() {
    return att::launch_t<V>(prm, grid, g, k, pdl, stream);
  });
}

}  // namespace qsa

QSA_BOUNDS_READER(bounds_word_attend)
