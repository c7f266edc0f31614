// qsa_select_row.cuh -- canonical top-k selection of one query row by one CTA
// (device function shared by the selection kernel).
//
// TensorRT-LLM PR #20276 ("Qwen3.8-Flash-Next NVFP4 target"), Features table:
// the selection row is a pure function of the scores, the window and k --
// every block strictly above the k-th score, ties to the highest index; and
// Decisions: radix top-k depends on launch order, canonical rows do not.
//
// For a row with nb visible blocks and window start wlo = max(0, nb - W):
//   window = valid blocks among [wlo, nb)                (always kept)
//   cand   = valid blocks among [0, wlo)
//   take   = min(k - |window|, |cand|) candidates ranked by (score desc,
//            block desc)
//   out    = window U taken, ascending, padded with -1
//
// Layout: block i of the row belongs to thread i mod NTHREADS ("round"
// i / NTHREADS), so shared-memory accesses are conflict-free.  The take-th
// largest candidate key is located by radix selection on (key - min key) with
// 11-bit digits starting at the highest bit where candidates differ.  As soon
// as the digit bin that holds it has at most kSelMaxMembers candidates, those
// members are ranked exactly by (key, block) against each other and the
// remaining digits are never visited (one pass for typical score ranges).
// When the last digit is reached instead, the threshold key is exact and ties
// go to the highest block indices by per-(round, warp) ballot counts.  The
// ascending compaction uses the same ballot counts, one barrier.
#pragma once

#include "qsa_common.cuh"

namespace qsa {

constexpr int kSelDigitBits = 11;
constexpr int kSelBins = 1 << kSelDigitBits;
constexpr int kSelMaxMembers = 256;   // boundary-bin members ranked directly
// Bounds-check codes (reported by bounds-checked builds only).
[[maybe_unused]] constexpr int kChkSelMember = 0x401;  // boundary-member list slot past its capacity
[[maybe_unused]] constexpr int kChkSelOut = 0x402;     // selection slot at or past k

// Shared memory a CTA of NTHREADS needs for rows of up to `mb` blocks.
template <int NTHREADS>
__host__ __device__ constexpr size_t select_row_smem(int mb) {
  return (size_t)kSelBins * 4                                      // histogram
         + (size_t)((mb + NTHREADS - 1) / NTHREADS) * (NTHREADS / 32) * 4 * 2  // round counts
         + 64 * 4                                                  // scalars
         + (size_t)kSelMaxMembers * 8                              // boundary members
         + (size_t)mb * 4;                                         // the row
}

__device__ __forceinline__ uint32_t sel_order_key(int s) { return (uint32_t)s ^ 0x80000000u; }

// Selects row `src` (nb visible blocks of which the last W are the window) into
// out[0..k) and returns the count (also written to *nsel by thread 0).
template <int NTHREADS>
__device__ void select_row(const int32_t* __restrict__ src, int nb, int W, int k,
                           int32_t* __restrict__ out, int32_t* __restrict__ nsel,
                           uint8_t* smem) {
  // The 64-int scalar area holds per-warp slots at sc[w], sc[8 + w], ...,
  // sc[32 + w] next to fixed slots from sc[40] on: at most 8 warps.
  static_assert(NTHREADS % 32 == 0 && NTHREADS <= 256, "select_row takes up to 8 warps");
  constexpr int kWarps = NTHREADS / 32;
  constexpr unsigned kFull = 0xffffffffu;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rounds = (nb + NTHREADS - 1) / NTHREADS;
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);
  int* cnt_eq = reinterpret_cast<int*>(smem + kSelBins * 4);
  int* cnt_pick = cnt_eq + rounds * kWarps;
  int* sc = cnt_pick + rounds * kWarps;           // 64 scalars
  uint2* mlist = reinterpret_cast<uint2*>(sc + 64);   // (rel, block) of boundary members
  int32_t* row = reinterpret_cast<int32_t*>(mlist + kSelMaxMembers);
  const int wlo = nb - W > 0 ? nb - W : 0;
  const unsigned lt_mask = (1u << lane) - 1u;

  // Row into shared memory; window and candidate counts and the candidate key
  // range straight from the loaded values.  The first histogram is cleared
  // here too.
  for (int q = tid; q < kSelBins; q += NTHREADS) hist[q] = 0;
  int nwin = 0, ncand = 0;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int i = tid; i < nb; i += NTHREADS) {
    const int s = src[i];
    row[i] = s;
    if (s == kSentinel) continue;
    if (i >= wlo) {
      ++nwin;
    } else {
      ++ncand;
      const uint32_t key = sel_order_key(s);
      kmin = min(kmin, key);
      kmax = max(kmax, key);
    }
  }
  nwin = __reduce_add_sync(kFull, nwin);
  ncand = __reduce_add_sync(kFull, ncand);
  kmin = __reduce_min_sync(kFull, kmin);
  kmax = __reduce_max_sync(kFull, kmax);
  if (lane == 0) {
    sc[warp] = nwin;
    sc[8 + warp] = ncand;
    sc[16 + warp] = (int)kmin;
    sc[24 + warp] = (int)kmax;
  }
  if (tid == 0) sc[50] = 0;   // boundary-member counter
  __syncthreads();
  int tot_win = 0, tot_cand = 0;
  kmin = 0xFFFFFFFFu;
  kmax = 0u;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    tot_win += sc[w];
    tot_cand += sc[8 + w];
    kmin = min(kmin, (uint32_t)sc[16 + w]);
    kmax = max(kmax, (uint32_t)sc[24 + w]);
  }

  const int take = min(k - tot_win, tot_cand);
  const bool none = take <= 0;
  const bool all = !none && take >= tot_cand;
  // Result of the search: candidates whose rel >> shift exceeds prefix are
  // taken; at rel >> shift == prefix, `need` more are taken -- the highest
  // (rel, block) members (ranked, by_rank) or, at shift 0, the highest blocks.
  uint32_t prefix = 0;
  int shift = 0;
  int need = 0;
  bool by_rank = false;
  if (!none && !all) {
    const uint32_t range = kmax - kmin;
    shift = range ? 32 - __clz(range) : 0;
    int remaining = take;
    bool first = true;
    while (shift > 0) {
      const int bits = shift < kSelDigitBits ? shift : kSelDigitBits;
      shift -= bits;
      const int nbins = 1 << bits;
      const uint32_t dmask = (uint32_t)nbins - 1u;
      if (!first) {
        for (int q = tid; q < nbins; q += NTHREADS) hist[q] = 0;
        __syncthreads();
      }
      first = false;
      for (int i = tid; i < wlo; i += NTHREADS) {
        const int s = row[i];
        if (s == kSentinel) continue;
        const uint32_t rel = sel_order_key(s) - kmin;
        const uint32_t high = (shift + bits >= 32) ? 0u : (rel >> (shift + bits));
        if (high == prefix) atomicAdd(&hist[(rel >> shift) & dmask], 1u);
      }
      __syncthreads();
      // Thread t owns bins [t*per, t*per + per); suffix counts from the top.
      constexpr int kPer = (kSelBins + NTHREADS - 1) / NTHREADS;
      int c[kPer];
      int local = 0;
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const int bin = tid * kPer + q;
        c[q] = bin < nbins ? (int)hist[bin] : 0;
        local += c[q];
      }
      // count in higher threads: warp suffix sum + higher warps' totals
      int incl = local;   // inclusive suffix within the warp (lanes >= this)
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(kFull, incl, o);
        if (lane + o < 32) incl += y;
      }
      if (lane == 0) sc[32 + warp] = incl;   // warp total
      __syncthreads();
      int above = incl - local;
#pragma unroll
      for (int w = 0; w < kWarps; ++w)
        if (w > warp) above += sc[32 + w];
#pragma unroll
      for (int q = kPer - 1; q >= 0; --q) {
        if (above < remaining && remaining <= above + c[q]) {
          sc[48] = tid * kPer + q;
          sc[49] = above;
          sc[51] = c[q];
        }
        above += c[q];
      }
      __syncthreads();
      remaining -= sc[49];
      prefix = (prefix << bits) | (uint32_t)sc[48];
      if (shift > 0 && sc[51] <= kSelMaxMembers) {
        by_rank = true;
        break;
      }
    }
    need = remaining;
  }

  if (by_rank) {
    // Boundary members into a list (any order), then each ranks itself.
    for (int i = tid; i < wlo; i += NTHREADS) {
      const int s = row[i];
      if (s == kSentinel) continue;
      const uint32_t rel = sel_order_key(s) - kmin;
      if ((rel >> shift) == prefix) {
        const int slot = atomicAdd(&sc[50], 1);
        if (QSA_IN_BOUNDS(slot < kSelMaxMembers, kChkSelMember))
          mlist[slot] = make_uint2(rel, (uint32_t)i);
      }
    }
    __syncthreads();
    const int m = min(sc[50], kSelMaxMembers);
    for (int rd = 0; rd < rounds; ++rd) {
      const int i = rd * NTHREADS + tid;
      const int s = i < nb ? row[i] : kSentinel;
      bool pick = false;
      if (s != kSentinel) {
        if (i >= wlo) {
          pick = true;
        } else {
          const uint32_t rel = sel_order_key(s) - kmin;
          const uint32_t hi = rel >> shift;
          if (hi > prefix) {
            pick = true;
          } else if (hi == prefix) {
            int rank = 0;   // members above this one in (rel, block) order
            for (int t = 0; t < m; ++t) {
              const uint2 y = mlist[t];
              rank += (y.x > rel || (y.x == rel && (int)y.y > i)) ? 1 : 0;
            }
            pick = rank < need;
          }
        }
      }
      const unsigned pb = __ballot_sync(kFull, pick);
      if (lane == 0) cnt_pick[rd * kWarps + warp] = __popc(pb);
      if (i < nb) row[i] = pick ? 1 : 0;
    }
  } else {
    const uint32_t thr_rel = prefix;   // exact threshold key (shift 0)
    // Tie ranks: equal candidates per (round, warp) first.
    for (int rd = 0; rd < rounds; ++rd) {
      const int i = rd * NTHREADS + tid;
      bool eq = false;
      if (!none && !all && i < wlo) {
        const int s = row[i];
        eq = s != kSentinel && sel_order_key(s) - kmin == thr_rel;
      }
      const unsigned b = __ballot_sync(kFull, eq);
      if (lane == 0) cnt_eq[rd * kWarps + warp] = __popc(b);
    }
    __syncthreads();
    // Picks, from the highest round down: an equal candidate is taken when
    // fewer than `need` equal candidates sit at higher block indices.  The
    // pick flag replaces the score in place.
    int eq_above = 0;   // equal candidates in rounds above the current one
    for (int rd = rounds - 1; rd >= 0; --rd) {
      const int i = rd * NTHREADS + tid;
      const int s = i < nb ? row[i] : kSentinel;
      bool pick = false, eq = false;
      if (s != kSentinel) {
        if (i >= wlo || all) {
          pick = true;
        } else if (!none) {
          const uint32_t rel = sel_order_key(s) - kmin;
          pick = rel > thr_rel;
          eq = rel == thr_rel;
        }
      }
      const unsigned b = __ballot_sync(kFull, eq);
      int in_round = 0, round_tot = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int cw = cnt_eq[rd * kWarps + w];
        round_tot += cw;
        if (w > warp) in_round += cw;
      }
      if (eq) pick = eq_above + in_round + __popc(b & ~lt_mask & ~(1u << lane)) < need;
      eq_above += round_tot;
      const unsigned pb = __ballot_sync(kFull, pick);
      if (lane == 0) cnt_pick[rd * kWarps + warp] = __popc(pb);
      if (i < nb) row[i] = pick ? 1 : 0;
    }
  }
  __syncthreads();
  // Ascending compaction: position = picks at lower indices.
  int below = 0;
  for (int rd = 0; rd < rounds; ++rd) {
    const int i = rd * NTHREADS + tid;
    const bool pick = i < nb && row[i];
    const unsigned pb = __ballot_sync(kFull, pick);
    int in_round = 0, round_tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int cw = cnt_pick[rd * kWarps + w];
      round_tot += cw;
      if (w < warp) in_round += cw;
    }
    const int pos = below + in_round + __popc(pb & lt_mask);
    if (pick && QSA_IN_BOUNDS(pos < k, kChkSelOut)) out[pos] = i;
    below += round_tot;
  }
  const int total = below;
  for (int i = total + tid; i < k; i += NTHREADS) out[i] = -1;
  if (tid == 0 && nsel) *nsel = total;
}

}  // namespace qsa
