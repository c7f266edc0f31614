// qsa_index_scores.cu -- A1: exact int8 index scores per (query row, KV block).
//
// TensorRT-LLM PR #20937 ("GB300 perf work on
// qwen3_8_flash_next_nvfp4__sm_103__tp1"), What changes / Verify:
// request-tiled index scores; PR #20276 ("Qwen3.8-Flash-Next NVFP4 target"),
// Features table: the QSA index plane is addressed by the same page index as
// the K/V pools.
//
// score(r, beta) = max over visible tokens t of block beta of
//                  sum_h sum_d iq[r,h,d] * ik[page, t, d]
//
// Design (HBM-bound streaming of 64 B per token):
//  * The head sum is taken first: sum_h iq[r,h,:] . ik = (sum_h iq[r,h,:]) . ik.
//    Both sides are exact integer arithmetic, so the result is bit-identical to
//    the per-head sum, and one 64-long int16 x int8 dot product per (row,
//    token) replaces Hq of them.
//  * Request tiling: a CTA serves one request; each warp streams whole blocks
//    (P tokens x 64 B, contiguous in the pool) with 16-byte loads, 4 lanes per
//    token, and scores every one of the request's R rows from the same loads,
//    so verify rows share one read of the keys.
//  * dp2a (int16 pair x int8 pair) accumulates each lane's 16 dims in int32;
//    two xor-shuffles finish the token's dot product and three more the
//    block max.  Invalid pages and invisible blocks are never read.
#include "qsa_common.cuh"

namespace qsa {
namespace {

// Bounds-check codes (reported by bounds-checked builds only).
[[maybe_unused]] constexpr int kChkPage = 0x301;    // index-key page id out of range
[[maybe_unused]] constexpr int kChkScore = 0x302;   // score row or block out of range
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;


__device__ __forceinline__ int4 ld_stream_v4(const int4* p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// RB: compile-time bound on rows per request (R <= RB).  PIPE: a warp owns
// several blocks and loads the next block's keys while scoring the current.
// A CTA none of whose blocks holds a token visible to its rows writes the
// sentinel for all of them and leaves before the head sums (the blocks past
// the shortest contexts of a batch are most of a wide grid).  Returns true
// when the CTA is done.  Rows r0 .. r0 + nrows - 1 of request b.
__device__ __forceinline__ bool only_invisible_blocks(const Geom& g, int P, int b, int r0,
                                                      int nrows, int nmax, int blocks_per_warp,
                                                      int32_t* scores) {
  const int beta0 = blockIdx.x * blocks_per_warp * kWarps;
  if (beta0 * P < nmax) return false;
  const int nb = min(blocks_per_warp * kWarps, g.MB - beta0);
  for (int i = threadIdx.x; i < nrows * nb; i += kThreads) {
    const int j = i / nb, beta = beta0 + i % nb;
    scores[((size_t)b * g.R + r0 + j) * g.MB + beta] = kSentinel;
  }
  return true;
}

template <int P, int RB, bool PIPE>
__global__ void __launch_bounds__(kThreads)
index_scores_kernel(Geom g, const int8_t* __restrict__ iq, const int8_t* __restrict__ ik_pool,
                    const int32_t* __restrict__ page_table, const int32_t* __restrict__ seqlens,
                    int32_t* __restrict__ scores, int blocks_per_warp) {
  __shared__ int32_t wpart[4][RB][kIndexDim];
  __shared__ uint32_t wpack[RB][kIndexDim / 2];

  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int R = g.R;

  pdl_wait();

  const int L = seqlens[b];
  const int cap = g.MB * P;
  const int nmax = visible_tokens(L, R, R - 1, cap);
  if (only_invisible_blocks(g, P, b, 0, R, nmax, blocks_per_warp, scores)) return;

  // Block `it` of this warp: page id and whether it has a visible token.
  auto block_of = [&](int it, int& beta, int& page) -> bool {
    beta = (blockIdx.x * blocks_per_warp + it) * kWarps + warp;
    page = -1;
    if (beta >= g.MB) return false;
    page = page_table[(size_t)b * g.MB + beta];
    return page >= 0 && page < g.NP && beta * P < nmax;
  };
  // Lane (token group lane>>2, part lane&3) loads 16 B of 8 tokens per step.
  auto load_keys = [&](int page, int4 (&kv)[P / 8]) {
    if (!QSA_IN_BOUNDS(page >= 0 && page < g.NP, kChkPage)) return;
    const int4* src = reinterpret_cast<const int4*>(ik_pool + (size_t)page * P * kIndexDim) + lane;
#pragma unroll
    for (int i = 0; i < P / 8; ++i) kv[i] = ld_stream_v4(src + 32 * i);
  };

  // The first block's keys are requested before the query head sums, so the
  // two latencies overlap.
  int beta0, page0;
  bool live0 = block_of(0, beta0, page0);
  int4 kv[P / 8];
  if (live0) load_keys(page0, kv);

  // Head sums of the request's index queries: w[j][d] = sum_h iq[b*R+j][h][d].
  for (int idx = threadIdx.x; idx < 4 * RB * kIndexDim; idx += kThreads) {
    const int hg = idx / (RB * kIndexDim);
    const int j = (idx / kIndexDim) % RB;
    const int d = idx % kIndexDim;
    int s = 0;
    if (j < R) {
      const int8_t* src = iq + ((size_t)(b * R + j) * g.Hq) * kIndexDim + d;
      int h = hg;
      // Batches of eight independent loads keep several L2 requests in flight.
      for (; h + 28 < g.Hq; h += 32) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = src[(size_t)(h + 4 * u) * kIndexDim];
#pragma unroll
        for (int u = 0; u < 8; ++u) s += v[u];
      }
      for (; h < g.Hq; h += 4) s += src[(size_t)h * kIndexDim];
    }
    wpart[hg][j][d] = s;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < RB * (kIndexDim / 2); idx += kThreads) {
    const int j = idx / (kIndexDim / 2), i = idx % (kIndexDim / 2);
    int w0 = 0, w1 = 0;
#pragma unroll
    for (int hg = 0; hg < 4; ++hg) {
      w0 += wpart[hg][j][2 * i];
      w1 += wpart[hg][j][2 * i + 1];
    }
    wpack[j][i] = ((uint32_t)w0 & 0xFFFFu) | ((uint32_t)w1 << 16);
  }
  __syncthreads();
  pdl_trigger();

  // Lane part covers dims [16*part, 16*part+16).
  const int part = lane & 3;
  uint32_t wr[RB][8];
#pragma unroll
  for (int j = 0; j < RB; ++j)
#pragma unroll
    for (int q = 0; q < 8; ++q) wr[j][q] = wpack[j][8 * part + q];

  int nrow[RB];
#pragma unroll
  for (int j = 0; j < RB; ++j) nrow[j] = (j < R) ? visible_tokens(L, R, j, cap) : 0;

  int beta = beta0, page = page0;
  bool live = live0;
  for (int it = 0; it < blocks_per_warp; ++it) {
    if (beta >= g.MB) break;
    // Next block's keys go out before this block is scored.
    int beta_n = g.MB, page_n = -1;
    bool live_n = false;
    [[maybe_unused]] int4 kv_n[PIPE ? P / 8 : 1];
    if constexpr (PIPE) {
      if (it + 1 < blocks_per_warp) {
        live_n = block_of(it + 1, beta_n, page_n);
        if (live_n) load_keys(page_n, kv_n);
      }
    } else if (it + 1 < blocks_per_warp) {
      live_n = block_of(it + 1, beta_n, page_n);
    }
    int32_t* dst = scores + (size_t)b * R * g.MB + beta;
    if (!QSA_IN_BOUNDS(b < g.B && beta >= 0 && beta < g.MB, kChkScore)) break;
    if (!live) {
      if (lane < R) dst[(size_t)lane * g.MB] = kSentinel;
    } else {
      int best[RB];
#pragma unroll
      for (int j = 0; j < RB; ++j) best[j] = kSentinel;
#pragma unroll
      for (int i = 0; i < P / 8; ++i) {
        const int t_abs = beta * P + 8 * i + (lane >> 2);
        const int words[4] = {kv[i].x, kv[i].y, kv[i].z, kv[i].w};
#pragma unroll
        for (int j = 0; j < RB; ++j) {
          if (j < R) {
            int acc = 0;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              acc = __dp2a_lo((int)wr[j][2 * m], words[m], acc);
              acc = __dp2a_hi((int)wr[j][2 * m + 1], words[m], acc);
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (t_abs < nrow[j]) best[j] = max(best[j], acc);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < RB; ++j) {
        if (j < R) {
          int v = best[j];
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 16));
          if (lane == j) dst[(size_t)j * g.MB] = (beta * P < nrow[j]) ? v : kSentinel;
        }
      }
    }
    beta = beta_n;
    page = page_n;
    live = live_n;
    if constexpr (PIPE) {
#pragma unroll
      for (int i = 0; i < P / 8; ++i) kv[i] = kv_n[i];
    } else {
      if (live) load_keys(page, kv);
    }
  }
  (void)page;
}

// ---- verify rows (R >= 2): the dot products on the tensor cores ------------
//
// Per request the head-summed weights w[j][d] (|w| <= 127 * Hq) are split as
// w = 128*a + b with b in [-64, 63] and |a| <= 254: both exact in fp16, as is
// every int8 key.  Per 16 tokens, two mma.sync m16n8k16 (fp16 x fp16 -> fp32)
// give S_a = K . a^T and S_b = K . b^T for all rows at once (the rows are the
// 8 MMA columns); every partial sum stays below 2^24 in magnitude, so both are
// exact integers and 128*S_a + S_b is the exact int32 token score.  Keys
// become fp16 by one byte permute against 0x64 (1024 + (x + 128)) and one
// subtraction of 1152.  Dims are taken in the order each lane holds them
// (lane part tig: dims 16*tig..16*tig+15, k-step kk: 4 of them), the same on
// both operands, so the contraction is unchanged.  Requests with more than 8
// rows (context row groups) take one CTA row per group of 8 rows (grid z).

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Four int8 -> two fp16 pairs (bytes 0,1 and bytes 2,3), exact.
// Head-summed index weights up to this magnitude are exact fp16 integers,
// and then every partial sum of a 64-dim dot product with int8 keys is an
// integer below 2^24 (2047 * 128 * 64), exact in the fp32 accumulators: one
// MMA per product and a float maximum.  Larger weights take the exact split
// w = 128 a + b (two MMAs, integer combination per token).
constexpr int kWholeMax = 2047;
template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};

__device__ __forceinline__ void s8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;                 // x + 128, as unsigned bytes
  const uint32_t bias = 0x64806480u;                  // fp16 pair (1152, 1152)
  lo = hsub2_u32(__byte_perm(u, 0x64646464u, 0x4140), bias);
  hi = hsub2_u32(__byte_perm(u, 0x64646464u, 0x4342), bias);
}

template <int P, bool PIPE>
__global__ void __launch_bounds__(kThreads, (P == 128 && PIPE) ? 1 : 2)
index_scores_mma_kernel(Geom g, const int8_t* __restrict__ iq, const int8_t* __restrict__ ik_pool,
                        const int32_t* __restrict__ page_table,
                        const int32_t* __restrict__ seqlens, int32_t* __restrict__ scores,
                        int blocks_per_warp) {
  constexpr int RB = kMaxRows;                 // the 8 MMA columns hold the rows
  static_assert(RB * 32 == kThreads, "one warp per row of the group for the head sums");
  __shared__ __half wsplit[2][RB][kIndexDim];   // a, b

  const int b = blockIdx.y;
  const int r0 = blockIdx.z * RB;              // first row of this CTA's group
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int R = g.R;

  pdl_wait();

  const int L = seqlens[b];
  const int cap = g.MB * P;
  const int nmax = visible_tokens(L, R, min(R - 1, r0 + RB - 1), cap);
  if (only_invisible_blocks(g, P, b, r0, min(RB, R - r0), nmax, blocks_per_warp, scores))
    return;

  auto block_of = [&](int it, int& beta, int& page) -> bool {
    beta = (blockIdx.x * blocks_per_warp + it) * kWarps + warp;
    page = -1;
    if (beta >= g.MB) return false;
    page = page_table[(size_t)b * g.MB + beta];
    return page >= 0 && page < g.NP && beta * P < nmax;
  };
  // Lane (gid, tig) loads 16 B (dims 16*tig..) of token 8*i + gid per step.
  auto load_keys = [&](int page, int4 (&kv)[P / 8]) {
    if (!QSA_IN_BOUNDS(page >= 0 && page < g.NP, kChkPage)) return;
    const int4* src = reinterpret_cast<const int4*>(ik_pool + (size_t)page * P * kIndexDim) + lane;
#pragma unroll
    for (int i = 0; i < P / 8; ++i) kv[i] = ld_stream_v4(src + 32 * i);
  };

  int beta0, page0;
  bool live0 = block_of(0, beta0, page0);
  int4 kv[P / 8];
  if (live0) load_keys(page0, kv);

  bool split = false;   // some |w| > kWholeMax: the exact two-part products
  // Head sums w[j][d], then the exact split w = 128*a + b.  Thread pair
  // (t >> 1) owns row j = t >> 5 and dims 4*d4..4*d4+3 (d4 = (t >> 1) & 15);
  // the two threads of a pair take alternate heads, 4-byte loads, up to 16
  // of them in flight per thread, then one shuffle adds the pair.
  {
    const int t = threadIdx.x;
    const int j = t >> 5, d4 = (t >> 1) & 15, hs = t & 1;
    int s0 = 0, s1 = 0, s2 = 0, s3 = 0;
    if (r0 + j < R) {
      const int8_t* src = iq + ((size_t)((size_t)b * R + r0 + j) * g.Hq) * kIndexDim + 4 * d4;
      for (int h0 = hs; h0 < g.Hq; h0 += 32) {
        uint32_t v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int h = h0 + 2 * u;
          v[u] = h < g.Hq ? __ldg(reinterpret_cast<const uint32_t*>(src + (size_t)h * kIndexDim))
                          : 0u;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          // byte i sign-extended: prmt selector nibbles (i, 8|i, 8|i, 8|i)
          s0 += (int)prmt(v[u], 0u, 0x8880);
          s1 += (int)prmt(v[u], 0u, 0x9991);
          s2 += (int)prmt(v[u], 0u, 0xAAA2);
          s3 += (int)prmt(v[u], 0u, 0xBBB3);
        }
      }
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
    s3 += __shfl_xor_sync(0xffffffffu, s3, 1);
    const int w4[4] = {s0, s1, s2, s3};
    bool big = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) big |= w4[i] > kWholeMax || w4[i] < -kWholeMax;
    split = __syncthreads_or(big) != 0;
    if (hs == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int w = w4[i];
        const int lo = ((w + 64) & 127) - 64;
        wsplit[0][j][4 * d4 + i] = __int2half_rn(split ? (w - lo) / 128 : w);
        if (split) wsplit[1][j][4 * d4 + i] = __int2half_rn(lo);
      }
    }
  }
  __syncthreads();
  pdl_trigger();

  // B fragments (column gid = row gid): k-step kk, halves 0/1 -> dims
  // 16*tig + 4*kk + {0,1} / {2,3}.
  uint32_t bw[2][4][2];
#pragma unroll
  for (int q = 0; q < 2; ++q)   // (w[1] is unused without the split)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const __half* src = &wsplit[q][gid][16 * tig + 4 * kk];
      bw[q][kk][0] = *reinterpret_cast<const uint32_t*>(src);
      bw[q][kk][1] = *reinterpret_cast<const uint32_t*>(src + 2);
    }
  // This lane's two columns (rows r0 + 2*tig, r0 + 2*tig + 1).
  int ncol[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int j = r0 + 2 * tig + e;
    ncol[e] = (j < R) ? visible_tokens(L, R, j, cap) : 0;
  }

  auto blocks = [&](auto split_tag) {
  constexpr bool SPLIT = decltype(split_tag)::value;
  int beta = beta0, page = page0;
  bool live = live0;
  for (int it = 0; it < blocks_per_warp; ++it) {
    if (beta >= g.MB) break;
    int beta_n = g.MB, page_n = -1;
    bool live_n = false;
    [[maybe_unused]] int4 kv_n[PIPE ? P / 8 : 1];
    if constexpr (PIPE) {
      if (it + 1 < blocks_per_warp) {
        live_n = block_of(it + 1, beta_n, page_n);
        if (live_n) load_keys(page_n, kv_n);
      }
    } else if (it + 1 < blocks_per_warp) {
      live_n = block_of(it + 1, beta_n, page_n);
    }
    int32_t* dst = scores + ((size_t)b * R + r0) * g.MB + beta;
    if (!QSA_IN_BOUNDS(b < g.B && beta >= 0 && beta < g.MB, kChkScore)) break;
    if (!live) {
      if (lane < RB && r0 + lane < R) dst[(size_t)lane * g.MB] = kSentinel;
    } else {
      int best[2] = {kSentinel, kSentinel};
      float bestf[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int mt = 0; mt < P / 16; ++mt) {
        const int4 ka = kv[2 * mt], kb = kv[2 * mt + 1];   // tokens gid and gid + 8
        const uint32_t wa[4] = {(uint32_t)ka.x, (uint32_t)ka.y, (uint32_t)ka.z, (uint32_t)ka.w};
        const uint32_t wb[4] = {(uint32_t)kb.x, (uint32_t)kb.y, (uint32_t)kb.z, (uint32_t)kb.w};
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t a[4];
          s8x4_to_f16x2x2(wa[kk], a[0], a[2]);
          s8x4_to_f16x2x2(wb[kk], a[1], a[3]);
          mma_f16_16816(sa, a, bw[0][kk][0], bw[0][kk][1]);
          if constexpr (SPLIT) mma_f16_16816(sb, a, bw[1][kk][0], bw[1][kk][1]);
        }
        const int tA = beta * P + 16 * mt + gid, tB = tA + 8;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if constexpr (SPLIT) {
            const int vA = __float2int_rn(sa[e]) * 128 + __float2int_rn(sb[e]);
            const int vB = __float2int_rn(sa[2 + e]) * 128 + __float2int_rn(sb[2 + e]);
            if (tA < ncol[e]) best[e] = max(best[e], vA);
            if (tB < ncol[e]) best[e] = max(best[e], vB);
          } else {
            if (tA < ncol[e]) bestf[e] = fmaxf(bestf[e], sa[e]);
            if (tB < ncol[e]) bestf[e] = fmaxf(bestf[e], sa[2 + e]);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        int v;
        if constexpr (SPLIT) {
          v = best[e];
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 16));
        } else {
          float f = bestf[e];
          f = fmaxf(f, __shfl_xor_sync(0xffffffffu, f, 4));
          f = fmaxf(f, __shfl_xor_sync(0xffffffffu, f, 8));
          f = fmaxf(f, __shfl_xor_sync(0xffffffffu, f, 16));
          v = f == -INFINITY ? kSentinel : __float2int_rn(f);
        }
        const int j = 2 * tig + e;
        if (gid == 0 && r0 + j < R) dst[(size_t)j * g.MB] = (beta * P < ncol[e]) ? v : kSentinel;
      }
    }
    beta = beta_n;
    page = page_n;
    live = live_n;
    if constexpr (PIPE) {
#pragma unroll
      for (int i = 0; i < P / 8; ++i) kv[i] = kv_n[i];
    } else {
      if (live) load_keys(page, kv);
    }
  }
  (void)page;
  };
  if (split) blocks(BoolTag<true>{});
  else blocks(BoolTag<false>{});
}

// ---- long row groups (R > 8): 64 rows per CTA ----------------------------
//
// The same exact tensor-core dot products, for eight 8-row groups per CTA: a
// warp converts a block's keys to fp16 A fragments once and runs the MMAs of
// all eight groups from those registers, so the keys are read once per 64
// rows instead of once per 8.  Head sums: thread (row, part) adds the Hq
// 16-byte slices of its row's index queries (all loads in flight at once).
constexpr int kGroupRows = 64;

template <int P>
__global__ void __launch_bounds__(kThreads, P == 128 ? 1 : 2)
index_scores_rows_kernel(Geom g, const int8_t* __restrict__ iq, const int8_t* __restrict__ ik_pool,
                         const int32_t* __restrict__ page_table,
                         const int32_t* __restrict__ seqlens, int32_t* __restrict__ scores,
                         int blocks_per_warp) {
  __shared__ __half wsplit[2][kGroupRows][kIndexDim];   // a, b of w = 128 a + b
  static_assert(kThreads == 4 * kGroupRows, "one thread per (row, 16-dim part)");
  const int b = blockIdx.y;
  const int r0 = blockIdx.z * kGroupRows;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int R = g.R;

  pdl_wait();

  const int L = seqlens[b];
  const int cap = g.MB * P;
  const int nmax = visible_tokens(L, R, min(R - 1, r0 + kGroupRows - 1), cap);
  if (only_invisible_blocks(g, P, b, r0, min(kGroupRows, R - r0), nmax, blocks_per_warp, scores))
    return;

  auto block_of = [&](int it, int& beta, int& page) -> bool {
    beta = (blockIdx.x * blocks_per_warp + it) * kWarps + warp;
    page = -1;
    if (beta >= g.MB) return false;
    page = page_table[(size_t)b * g.MB + beta];
    return page >= 0 && page < g.NP && beta * P < nmax;
  };

  bool split = false;   // some |w| > kWholeMax: the exact two-part products
  {
    const int rr = threadIdx.x >> 2, part = threadIdx.x & 3;
    int acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0;
    if (r0 + rr < R) {
      const int4* src = reinterpret_cast<const int4*>(
                            iq + ((size_t)b * R + r0 + rr) * g.Hq * kIndexDim) + part;
      int h = 0;
      for (; h + 8 <= g.Hq; h += 8) {
        int4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldg(src + (size_t)(h + u) * (kIndexDim / 16));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[4 * q + e] += (int)(int8_t)(w4[q] >> (8 * e));
        }
      }
      for (; h < g.Hq; ++h) {
        const int4 v = __ldg(src + (size_t)h * (kIndexDim / 16));
        const int w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[4 * q + e] += (int)(int8_t)(w4[q] >> (8 * e));
      }
    }
    bool big = false;
#pragma unroll
    for (int i = 0; i < 16; ++i) big |= acc[i] > kWholeMax || acc[i] < -kWholeMax;
    split = __syncthreads_or(big) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int w = acc[i];
      const int lo = ((w + 64) & 127) - 64;
      wsplit[0][rr][16 * part + i] = __int2half_rn(split ? (w - lo) / 128 : w);
      if (split) wsplit[1][rr][16 * part + i] = __int2half_rn(lo);
    }
  }
  __syncthreads();
  pdl_trigger();

  // This lane's columns in every group: rows r0 + 8*grp + 2*tig + e.
  auto blocks = [&](auto split_tag) {
  constexpr bool SPLIT = decltype(split_tag)::value;
  int beta = 0, page = -1;
  for (int it = 0; it < blocks_per_warp; ++it) {
    const bool live = block_of(it, beta, page);
    if (beta >= g.MB) break;
    int32_t* dst = scores + ((size_t)b * R + r0) * g.MB + beta;
    if (!QSA_IN_BOUNDS(b < g.B && beta >= 0 && beta < g.MB, kChkScore)) break;
    if (!live) {
      for (int jr = lane; jr < kGroupRows; jr += 32)
        if (r0 + jr < R) dst[(size_t)jr * g.MB] = kSentinel;
      continue;
    }
    int4 kv[P / 8];
    if (!QSA_IN_BOUNDS(page >= 0 && page < g.NP, kChkPage)) break;
    const int4* src = reinterpret_cast<const int4*>(ik_pool + (size_t)page * P * kIndexDim) + lane;
#pragma unroll
    for (int i = 0; i < P / 8; ++i) kv[i] = ld_stream_v4(src + 32 * i);
    // A fragments of the block, once: [m-tile][k-step][4]
    uint32_t af[P / 16][4][4];
#pragma unroll
    for (int mt = 0; mt < P / 16; ++mt) {
      const int4 ka = kv[2 * mt], kb = kv[2 * mt + 1];   // tokens gid and gid + 8
      const uint32_t wa[4] = {(uint32_t)ka.x, (uint32_t)ka.y, (uint32_t)ka.z, (uint32_t)ka.w};
      const uint32_t wb[4] = {(uint32_t)kb.x, (uint32_t)kb.y, (uint32_t)kb.z, (uint32_t)kb.w};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        s8x4_to_f16x2x2(wa[kk], af[mt][kk][0], af[mt][kk][2]);
        s8x4_to_f16x2x2(wb[kk], af[mt][kk][1], af[mt][kk][3]);
      }
    }
    for (int grp = 0; grp < kGroupRows / 8; ++grp) {
      const int jbase = 8 * grp;
      if (r0 + jbase >= R) break;
      uint32_t bw[2][4][2];
#pragma unroll
      for (int q = 0; q < (SPLIT ? 2 : 1); ++q)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const __half* w = &wsplit[q][jbase + gid][16 * tig + 4 * kk];
          bw[q][kk][0] = *reinterpret_cast<const uint32_t*>(w);
          bw[q][kk][1] = *reinterpret_cast<const uint32_t*>(w + 2);
        }
      int ncol[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = r0 + jbase + 2 * tig + e;
        ncol[e] = (j < R) ? visible_tokens(L, R, j, cap) : 0;
      }
      int best[2] = {kSentinel, kSentinel};
      float bestf[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int mt = 0; mt < P / 16; ++mt) {
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          mma_f16_16816(sa, af[mt][kk], bw[0][kk][0], bw[0][kk][1]);
          if constexpr (SPLIT) mma_f16_16816(sb, af[mt][kk], bw[1][kk][0], bw[1][kk][1]);
        }
        const int tA = beta * P + 16 * mt + gid, tB = tA + 8;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if constexpr (SPLIT) {
            const int vA = __float2int_rn(sa[e]) * 128 + __float2int_rn(sb[e]);
            const int vB = __float2int_rn(sa[2 + e]) * 128 + __float2int_rn(sb[2 + e]);
            if (tA < ncol[e]) best[e] = max(best[e], vA);
            if (tB < ncol[e]) best[e] = max(best[e], vB);
          } else {
            if (tA < ncol[e]) bestf[e] = fmaxf(bestf[e], sa[e]);
            if (tB < ncol[e]) bestf[e] = fmaxf(bestf[e], sa[2 + e]);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        int v;
        if constexpr (SPLIT) {
          v = best[e];
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 16));
        } else {
          float f = bestf[e];
          f = fmaxf(f, __shfl_xor_sync(0xffffffffu, f, 4));
          f = fmaxf(f, __shfl_xor_sync(0xffffffffu, f, 8));
          f = fmaxf(f, __shfl_xor_sync(0xffffffffu, f, 16));
          v = f == -INFINITY ? kSentinel : __float2int_rn(f);
        }
        const int j = jbase + 2 * tig + e;
        if (gid == 0 && r0 + j < R) dst[(size_t)j * g.MB] = (beta * P < ncol[e]) ? v : kSentinel;
      }
    }
  }
  };
  if (split) blocks(BoolTag<true>{});
  else blocks(BoolTag<false>{});
}

// Blocks each warp scores: one, unless the grid would exceed about
// QSA_INDEX_CTAS_PER_SM resident CTAs per SM (at most QSA_INDEX_BPW_MAX).
#ifndef QSA_INDEX_CTAS_PER_SM
#define QSA_INDEX_CTAS_PER_SM 8
#endif
#ifndef QSA_INDEX_BPW_MAX
#define QSA_INDEX_BPW_MAX 4
#endif
int blocks_per_warp_for(const Geom& g) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long warps_needed = (long long)g.B * g.MB;
  const long long warp_slots = (long long)sms * QSA_INDEX_CTAS_PER_SM * kWarps;
  int bpw = (int)((warps_needed + warp_slots - 1) / warp_slots);
  return bpw < 1 ? 1 : (bpw > QSA_INDEX_BPW_MAX ? QSA_INDEX_BPW_MAX : bpw);
}

template <int P, int RB, bool PIPE>
cudaError_t launch_t(const Geom& g, const int8_t* iq, const int8_t* ik_pool,
                     const int32_t* page_table, const int32_t* seqlens, int32_t* scores,
                     bool pdl, cudaStream_t stream) {
  const int bpw = blocks_per_warp_for(g);
  dim3 grid((g.MB + kWarps * bpw - 1) / (kWarps * bpw), g.B);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, index_scores_kernel<P, RB, PIPE>, g, iq, ik_pool, page_table,
                            seqlens, scores, bpw);
}

template <int P, int RB>
cudaError_t launch_rb(const Geom& g, const int8_t* iq, const int8_t* ik_pool,
                      const int32_t* page_table, const int32_t* seqlens, int32_t* scores,
                      bool pdl, cudaStream_t stream) {
  if (blocks_per_warp_for(g) > 1)
    return launch_t<P, RB, true>(g, iq, ik_pool, page_table, seqlens, scores, pdl, stream);
  return launch_t<P, RB, false>(g, iq, ik_pool, page_table, seqlens, scores, pdl, stream);
}

template <int P, bool PIPE>
cudaError_t launch_mma_t(const Geom& g, const int8_t* iq, const int8_t* ik_pool,
                         const int32_t* page_table, const int32_t* seqlens, int32_t* scores,
                         bool pdl, cudaStream_t stream) {
  const int bpw = blocks_per_warp_for(g);
  dim3 grid((g.MB + kWarps * bpw - 1) / (kWarps * bpw), g.B, (g.R + kMaxRows - 1) / kMaxRows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, index_scores_mma_kernel<P, PIPE>, g, iq, ik_pool, page_table,
                            seqlens, scores, bpw);
}

template <int P>
cudaError_t launch_rows(const Geom& g, const int8_t* iq, const int8_t* ik_pool,
                        const int32_t* page_table, const int32_t* seqlens, int32_t* scores,
                        bool pdl, cudaStream_t stream) {
  // Blocks per warp: the grid about fills the SMs at two resident CTAs each
  // (the register cap), so each CTA's head sums serve as many blocks as that
  // allows.
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long groups = (g.R + kGroupRows - 1) / kGroupRows;
  const long long warps_needed = (long long)g.B * g.MB * groups;
  const long long warp_slots = (long long)sms * 2 * kWarps;
  int bpw = (int)((warps_needed + warp_slots - 1) / warp_slots);
  bpw = bpw < 1 ? 1 : (bpw > 8 ? 8 : bpw);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((g.MB + kWarps * bpw - 1) / (kWarps * bpw), g.B, (unsigned)groups);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, index_scores_rows_kernel<P>, g, iq, ik_pool, page_table,
                            seqlens, scores, bpw);
}

template <int P>
cudaError_t launch_p(const Geom& g, const int8_t* iq, const int8_t* ik_pool,
                     const int32_t* page_table, const int32_t* seqlens, int32_t* scores,
                     bool pdl, cudaStream_t stream) {
  // Decode rows: int16 x int8 dp2a.  Two rows and more: the tensor cores,
  // 8 rows per CTA for verify rows, 64 for long row groups.
  if (g.R > kMaxRows) return launch_rows<P>(g, iq, ik_pool, page_table, seqlens, scores, pdl, stream);
  if (g.R >= 2) {
    if (blocks_per_warp_for(g) > 1)
      return launch_mma_t<P, true>(g, iq, ik_pool, page_table, seqlens, scores, pdl, stream);
    return launch_mma_t<P, false>(g, iq, ik_pool, page_table, seqlens, scores, pdl, stream);
  }
  return launch_rb<P, 1>(g, iq, ik_pool, page_table, seqlens, scores, pdl, stream);
}

}  // namespace

cudaError_t launch_index_scores(const Geom& g, const int8_t* iq, const int8_t* ik_pool,
                                const int32_t* page_table, const int32_t* seqlens,
                                int32_t* scores, bool pdl, cudaStream_t stream) {
  if (g.P == 32) return launch_p<32>(g, iq, ik_pool, page_table, seqlens, scores, pdl, stream);
  if (g.P == 64) return launch_p<64>(g, iq, ik_pool, page_table, seqlens, scores, pdl, stream);
  return launch_p<128>(g, iq, ik_pool, page_table, seqlens, scores, pdl, stream);
}

}  // namespace qsa

QSA_BOUNDS_READER(bounds_word_index)
