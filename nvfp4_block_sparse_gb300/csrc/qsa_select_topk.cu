// qsa_select_topk.cu -- A2: canonical top-k block selection per query row.
//
// TensorRT-LLM PR #20276 ("Qwen3.8-Flash-Next NVFP4 target"), Features table:
// the selection row is a pure function of the scores, the window and k --
// every block strictly above the k-th score, ties to the highest index; and
// Decisions: radix top-k depends on launch order, canonical rows do not.
//
// Per row r (n visible tokens, nb = ceil(n/P) visible blocks):
//   window  = valid blocks among [nb - W, nb)            (always kept)
//   cand    = valid blocks among [0, nb - W)
//   take    = min(k - |window|, |cand|) candidates, ranked by (score desc,
//             block desc)
//   sel[r]  = window U taken, ascending, padded with -1
//
// Design: one CTA per row; the row's scores sit in shared memory and each
// thread owns a contiguous run of blocks.  The take-th largest candidate score
// is found by radix selection on (key - min key) with 11-bit digits, starting
// at the highest bit where the candidates differ (two passes for typical
// score ranges; shared-memory histograms stay uncongested because the digits
// span the actual range).  The selection then takes every candidate above
// that score plus, at that score, the highest block indices -- counted with a
// suffix scan over the threads' runs.  A prefix scan writes the blocks in
// ascending order.  Every step is a deterministic function of the row.
#include "qsa_common.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kDigitBits = 11;
constexpr int kBins = 1 << kDigitBits;

struct Scan {
  int warp_tot[kWarps];
  int out;
};

// Block-wide exclusive prefix sum of `v` in thread order; `total` receives the sum.
__device__ __forceinline__ int block_excl_scan(int v, int& total, Scan& sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sc.warp_tot[warp] = x;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int t = sc.warp_tot[w];
    base += (w < warp) ? t : 0;
    tot += t;
  }
  __syncthreads();
  total = tot;
  return base + x - v;
}

__device__ __forceinline__ uint32_t order_key(int s) { return (uint32_t)s ^ 0x80000000u; }

__global__ void __launch_bounds__(kThreads)
select_topk_kernel(Geom g, const int32_t* __restrict__ scores, const int32_t* __restrict__ seqlens,
                   int k, int W, int32_t* __restrict__ sel, int32_t* __restrict__ nsel) {
  extern __shared__ int32_t s_row[];
  __shared__ uint32_t hist[kBins];
  __shared__ Scan sc;
  __shared__ uint32_t s_minmax[2];
  __shared__ int s_digit, s_above;

  const int r = blockIdx.x;
  const int b = r / g.R, j = r % g.R;
  const int tid = threadIdx.x;

  pdl_wait();
  const int n = visible_tokens(seqlens[b], g.R, j, g.MB * g.P);
  const int nb = (n + g.P - 1) / g.P;
  const int wlo = nb - W > 0 ? nb - W : 0;

  for (int i = tid; i < nb; i += kThreads) s_row[i] = scores[(size_t)r * g.MB + i];
  if (tid == 0) {
    s_minmax[0] = 0xFFFFFFFFu;
    s_minmax[1] = 0u;
  }
  __syncthreads();
  pdl_trigger();

  const int E = (nb + kThreads - 1) / kThreads;
  const int lo = min(nb, tid * E), hi = min(nb, lo + E);

  // Window and candidate counts; candidate key range.
  int nwin = 0, ncand = 0;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int i = lo; i < hi; ++i) {
    const int s = s_row[i];
    if (s == kSentinel) continue;
    if (i >= wlo) {
      ++nwin;
    } else {
      ++ncand;
      const uint32_t key = order_key(s);
      kmin = min(kmin, key);
      kmax = max(kmax, key);
    }
  }
  if (ncand) {
    atomicMin(&s_minmax[0], kmin);
    atomicMax(&s_minmax[1], kmax);
  }
  int tot_win, tot_cand;
  block_excl_scan(nwin, tot_win, sc);
  block_excl_scan(ncand, tot_cand, sc);
  kmin = s_minmax[0];
  kmax = s_minmax[1];

  const int take = min(k - tot_win, tot_cand);
  // Threshold: candidates with rel > thr_rel are taken; at rel == thr_rel the
  // `need` highest block indices are taken.
  uint32_t thr_rel = 0;
  int need = 0;
  const bool none = take <= 0;
  const bool all = !none && take >= tot_cand;
  if (!none && !all) {
    const uint32_t range = kmax - kmin;
    int shift = range ? 32 - __clz(range) : 0;
    uint32_t prefix = 0;
    int remaining = take;
    while (shift > 0) {
      const int bits = shift < kDigitBits ? shift : kDigitBits;
      shift -= bits;
      const uint32_t dmask = (1u << bits) - 1u;
      for (int i = tid; i < (1 << bits); i += kThreads) hist[i] = 0;
      __syncthreads();
      for (int i = lo; i < min(hi, wlo); ++i) {
        const int s = s_row[i];
        if (s == kSentinel) continue;
        const uint32_t rel = order_key(s) - kmin;
        const uint32_t high = (shift + bits >= 32) ? 0u : (rel >> (shift + bits));
        if (high == prefix) atomicAdd(&hist[(rel >> shift) & dmask], 1u);
      }
      __syncthreads();
      // Thread t owns bins [t*8, t*8+8); find the bin holding the remaining-th
      // largest element, scanning from the top bin down.
      constexpr int kPer = kBins / kThreads;
      int local = 0;
      for (int q = 0; q < kPer; ++q) {
        const int bin = tid * kPer + q;
        if (bin < (1 << bits)) local += (int)hist[bin];
      }
      // Suffix sum: count of elements in bins owned by higher threads.
      int tot;
      const int rev = block_excl_scan(local, tot, sc);  // sum over lower threads
      int above = tot - rev - local;                    // sum over higher threads
      for (int q = kPer - 1; q >= 0; --q) {
        const int bin = tid * kPer + q;
        if (bin >= (1 << bits)) continue;
        const int c = (int)hist[bin];
        if (above < remaining && remaining <= above + c) {
          s_digit = bin;
          s_above = above;
        }
        above += c;
      }
      __syncthreads();
      remaining -= s_above;
      prefix = (prefix << bits) | (uint32_t)s_digit;
      __syncthreads();
    }
    thr_rel = prefix;
    need = remaining;
  }

  // Among candidates equal to the threshold, take the `need` highest indices.
  int eq_local = 0;
  if (!none && !all && need > 0)
    for (int i = lo; i < min(hi, wlo); ++i) {
      const int s = s_row[i];
      if (s != kSentinel && order_key(s) - kmin == thr_rel) ++eq_local;
    }
  int eq_tot;
  const int eq_below = block_excl_scan(eq_local, eq_tot, sc);
  int eq_above = eq_tot - eq_below - eq_local;  // equal candidates with higher index

  // Mark (in place: selected blocks keep their index as a flag) and count.
  int cnt = 0;
  for (int i = hi - 1; i >= lo; --i) {
    const int s = s_row[i];
    bool pick = false;
    if (s != kSentinel) {
      if (i >= wlo) {
        pick = true;
      } else if (all) {
        pick = true;
      } else if (!none) {
        const uint32_t rel = order_key(s) - kmin;
        if (rel > thr_rel) {
          pick = true;
        } else if (rel == thr_rel) {
          pick = eq_above < need;
          ++eq_above;
        }
      }
    }
    s_row[i] = pick ? 1 : 0;
    cnt += pick;
  }
  int total;
  int pos = block_excl_scan(cnt, total, sc);
  int32_t* out = sel + (size_t)r * k;
  for (int i = lo; i < hi; ++i)
    if (s_row[i]) out[pos++] = i;
  for (int i = total + tid; i < k; i += kThreads) out[i] = -1;
  if (tid == 0) nsel[r] = total;
}

}  // namespace

cudaError_t launch_select_topk(const Geom& g, const int32_t* scores, const int32_t* seqlens,
                               int k, int window, int32_t* sel, int32_t* nsel, bool pdl,
                               cudaStream_t stream) {
  const size_t smem = (size_t)g.MB * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(select_topk_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.B * g.R);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, select_topk_kernel, g, scores, seqlens, k, window, sel, nsel);
}

}  // namespace qsa
