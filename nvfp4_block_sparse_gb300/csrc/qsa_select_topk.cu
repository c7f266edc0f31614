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
// Design: one CTA per row running select_row (qsa_select_row.cuh): scores in
// shared memory, conflict-free ownership, 11-bit range-adaptive radix
// selection, ballot-ranked ties and compaction; about a dozen barriers per
// row and no serial per-thread runs.  Every step is a deterministic function
// of the row.
#include "qsa_select_row.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
select_topk_kernel(Geom g, const int32_t* __restrict__ scores, const int32_t* __restrict__ seqlens,
                   int k, int W, int32_t* __restrict__ sel, int32_t* __restrict__ nsel) {
  extern __shared__ __align__(16) uint8_t smem_sel[];
  const int r = blockIdx.x;
  const int b = r / g.R, j = r % g.R;
  pdl_wait();
  // Dependents may start their own prologue now: it reads only step inputs,
  // which are complete once this wait has returned.
  pdl_trigger();
  const int n = visible_tokens(seqlens[b], g.R, j, g.MB * g.P);
  const int nb = (n + g.P - 1) / g.P;
  select_row<kThreads>(scores + (size_t)r * g.MB, nb, W, k, sel + (size_t)r * k, nsel + r,
                       smem_sel);
}

}  // namespace

cudaError_t launch_select_topk(const Geom& g, const int32_t* scores, const int32_t* seqlens,
                               int k, int window, int32_t* sel, int32_t* nsel, bool pdl,
                               cudaStream_t stream) {
  const size_t smem = select_row_smem<kThreads>(g.MB);
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
QSA_BOUNDS_READER(bounds_word_select)
