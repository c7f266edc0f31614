/*
 * qsa.h -- C ABI of the GB300 (sm_103a) QSA block-sparse GQA decode / verify
 * library over an NVFP4 paged KV cache.
 *
 * One decode or speculative-verify step is three calls on one stream:
 *
 *   qsa_index_scores   exact int8 index dot products -> one int32 score per
 *                      (query row, KV block)
 *   qsa_select_topk    canonical top-k block selection per query row
 *   qsa_sparse_decode  split-KV GQA attention over the selected NVFP4 pages,
 *                      dequantised in registers, partials merged by log-sum-exp
 *
 * Sources (TensorRT-LLM pull-request pages):
 *   [F]  PR #20276 "Qwen3.8-Flash-Next NVFP4 target", Features table: NVFP4 KV
 *        cache = uint8 e2m1 pages + e4m3 block scales, QSA side planes packed
 *        so that one page index addresses every pool; canonical QSA selection.
 *   [D]  PR #20276, Decisions: canonical selection is a pure function of the
 *        scores, the window and k, identical from launch to launch.
 *   [W]  PR #20937 "GB300 perf work on qwen3_8_flash_next_nvfp4__sm_103__tp1",
 *        What changes: NVFP4 sparse GQA decode as split-K + merge with a lean
 *        one-split variant; verify as request-grouped sparse GQA with a
 *        per-row merge; request-tiled index scores.
 *   [Q]  PR #20937, Per-File QA: invalid-page handling and masking.
 *
 * Conventions shared by every call
 * --------------------------------
 * Geometry (qsa_geom_t, host values): B requests, R = rows_per_req query rows
 * per request (1 for decode, 1 + drafts for verify), T = B*R rows, row r =
 * b*R + j.  Hq query heads, Hkv KV heads, G = Hq/Hkv; query head h reads KV
 * head h / G.  D = head_dim (128, or 256: the geometry of PR #20276,
 * Performance / shared code touched, 24 q / 2 KV heads at head_dim 256),
 * Di = index_dim = 64, P = page_size (64 or 128 tokens at D = 128; 32 or 64
 * at D = 256, 32 being the page size of PR #20276, Known limitations),
 * MB = max_blocks (page-table row stride), NP = num_pages.
 *
 * Visibility: seqlens[b] = L_b counts the request's cached tokens including
 * its R newest rows; row j sees n = clamp(L_b - R + 1 + j, 0, MB*P) tokens
 * (causal among the R rows).  Block beta holds tokens [beta*P, beta*P + P).
 *
 * Page table: page_table[b*MB + beta] is the physical page of block beta of
 * request b; an entry < 0 or >= NP marks an invalid block, which is masked,
 * never dereferenced.
 *
 * Memory: every pointer argument is DEVICE memory owned by the caller; the
 * library never allocates or frees device memory.  Its only global state is
 * the fixed scratch array of qsa_sparse_decode_noalloc (and the diagnostic
 * wait bound of qsa_debug_set_wait_ns).  Calls are asynchronous on `stream`,
 * read no device data on the host, and size their grids from the geometry
 * alone, so a step can be captured in a CUDA graph.
 *
 * Errors: each call validates its arguments on the host and returns a status
 * before launching anything; QSA_ERR_CUDA reports a launch failure.  Bad
 * device data (page ids, seqlens, sel entries) is masked, never trapped.
 */
#ifndef QSA_H_
#define QSA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QSA_OK = 0,
    QSA_ERR_INVALID_ARG = 1,   /* null pointer or inconsistent geometry      */
    QSA_ERR_UNSUPPORTED = 2,   /* shape outside the built kernels, or not sm_103 */
    QSA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed        */
    QSA_ERR_WORKSPACE = 4,     /* workspace missing or too small              */
    QSA_ERR_DEVICE_TIMEOUT = 5 /* a bounded device-side wait gave up (status word) */
} qsa_status_t;

typedef struct {
    int batch;          /* B                                    */
    int rows_per_req;   /* R = 1 + draft rows, 1..8; up to 4096
                           (a context row group) for the index
                           scores, the selection, the prologue
                           and qsa_sparse_prefill             */
    int num_q_heads;    /* Hq, 1..256                           */
    int num_kv_heads;   /* Hkv, divides Hq                      */
    int head_dim;       /* D, 128 or 256                        */
    int index_dim;      /* Di, must be 64                       */
    int page_size;      /* P, 64|128 (D = 128), 32|64 (D = 256) */
    int max_blocks;     /* MB, page-table row stride, >= 1      */
    int num_pages;      /* NP, pages in every pool, >= 1        */
} qsa_geom_t;

/* Human-readable name of a status. Never NULL. */
const char *qsa_status_string(qsa_status_t status);

/*
 * A1 -- index scores ([W] request-tiled index scores; [F] index keys share the
 * page index of the K/V pools).
 *
 *   iq        int8  [T, Hq, Di]   index query of every row and query head
 *   ik_pool   int8  [NP, P, Di]   index key of every cached token
 *   page_table int32 [B, MB]
 *   seqlens   int32 [B]
 *   scores    int32 [T, MB]       output
 *
 * scores[r, beta] = max over the visible tokens t of block beta of
 *                   sum_h sum_d iq[r, h, d] * ik[page, t - beta*P, d],
 * exact in int32 (|value| <= 64*64*127*127 for Hq <= 64; Hq <= 256 keeps it
 * below 2^31), or INT32_MIN when the block's page is invalid or the block has
 * no token visible to row r (all beta >= ceil(n/P) included).
 * Returns QSA_ERR_INVALID_ARG for null pointers or iq / ik_pool not 16-byte
 * aligned; geometry and device checks as for the other calls (rows_per_req up
 * to 4096).
 */
qsa_status_t qsa_index_scores(const qsa_geom_t *geom, const int8_t *iq,
                              const int8_t *ik_pool, const int32_t *page_table,
                              const int32_t *seqlens, int32_t *scores,
                              cudaStream_t stream);

/*
 * A2 -- canonical top-k selection ([F] Features table; [D] Decisions).
 *
 *   scores    int32 [T, MB]  as written by qsa_index_scores (INT32_MIN =
 *                            invalid block)
 *   seqlens   int32 [B]
 *   k         blocks per row, window included, 1..1024
 *   window    always-kept recent blocks, 0..k
 *   sel       int32 [T, k]   output: selected block indices, ascending,
 *                            padded with -1
 *   nsel      int32 [T]      output: number of selected blocks
 *
 * Per row with nb = ceil(n/P) visible blocks: the valid blocks among the last
 * `window` visible ones are always kept; the remaining slots (k minus those)
 * go to the other valid visible blocks ranked by score, higher first, ties to
 * the higher block index -- every block strictly above the k-th score, then
 * the highest-index blocks at the k-th score.  An invalid window block frees
 * its slot.  A pure function of (scores, seqlens, k, window): identical bits
 * on every launch.
 */
qsa_status_t qsa_select_topk(const qsa_geom_t *geom, const int32_t *scores,
                             const int32_t *seqlens, int k, int window,
                             int32_t *sel, int32_t *nsel, cudaStream_t stream);

/*
 * Bytes of device workspace qsa_sparse_decode needs for this geometry and k
 * with the automatic split count (num_splits = 0), or for an explicit
 * num_splits >= 1 with the _ex variant below.  Returns 0 for an invalid
 * geometry.  Host-only; launches nothing.
 */
size_t qsa_sparse_decode_workspace_bytes(const qsa_geom_t *geom, int k);
size_t qsa_sparse_decode_workspace_bytes_ex(const qsa_geom_t *geom, int k,
                                            int num_splits);

/*
 * Zero-fills a workspace (its split-merge tickets and status word must start
 * at zero). Call once after allocating it; every qsa_sparse_decode leaves the
 * tickets at zero again, so a workspace is reusable across steps as long as
 * calls using it do not overlap on the GPU.  Asynchronous on `stream`.
 */
qsa_status_t qsa_workspace_init(void *workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/*
 * A3 -- split-KV sparse GQA over the selected NVFP4 pages ([W] split-K +
 * merge, lean one-split variant, request-grouped verify with a per-row merge;
 * [F] NVFP4 page format; [Q] invalid-page masking).
 *
 *   q         bf16  [T, Hq, D]
 *   k_pool, v_pool  uint8 [NP, Hkv, P, D/2]  two e2m1 codes per byte, low
 *                                            nibble = even element
 *   k_sf, v_sf      uint8 [NP, Hkv, P, D/16] e4m3 scale per 16 elements
 *   k_scale, v_scale  fp32 per-tensor dequant multipliers:
 *                     K = e2m1 * e4m3 * k_scale, V likewise
 *   sm_scale  softmax scale applied to q.K (1/sqrt(D) conventionally)
 *   page_table, seqlens as above
 *   sel       int32 [T, k]   ascending block ids padded with -1 (the output of
 *                            qsa_select_topk)
 *   out       bf16  [T, Hq, D]   output
 *   lse       fp32  [T, Hq]      output, natural-log sum of exp(sm_scale*q.K)
 *   workspace device memory of at least qsa_sparse_decode_workspace_bytes(),
 *             zero-filled once by qsa_workspace_init().
 *
 * For row r and head h, the attended tokens are those of the distinct blocks
 * listed in sel[r, :] whose page is valid, restricted to the row's n visible
 * tokens.  Each (request, KV head) pass reads every page in the union of its
 * rows' selections once and serves all G*R query vectors.  A row with no
 * tokens gets out = 0 and lse = -inf.  Rounding: fp32 accumulation, bf16 RNE
 * output.
 */
qsa_status_t qsa_sparse_decode(const qsa_geom_t *geom, const void *q_bf16,
                               const uint8_t *k_pool, const uint8_t *k_sf,
                               const uint8_t *v_pool, const uint8_t *v_sf,
                               float k_scale, float v_scale, float sm_scale,
                               const int32_t *page_table, const int32_t *seqlens,
                               const int32_t *sel, int k, void *out_bf16,
                               float *lse, void *workspace,
                               size_t workspace_bytes, cudaStream_t stream);

/* As qsa_sparse_decode, with the number of KV splits per (request, KV head)
 * forced to num_splits (>= 1), or chosen automatically when 0.  Results agree
 * across split counts within fp32 rounding. */
qsa_status_t qsa_sparse_decode_ex(const qsa_geom_t *geom, const void *q_bf16,
                                  const uint8_t *k_pool, const uint8_t *k_sf,
                                  const uint8_t *v_pool, const uint8_t *v_sf,
                                  float k_scale, float v_scale, float sm_scale,
                                  const int32_t *page_table,
                                  const int32_t *seqlens, const int32_t *sel,
                                  int k, void *out_bf16, float *lse,
                                  void *workspace, size_t workspace_bytes,
                                  int num_splits, cudaStream_t stream);

/*
 * qsa_select_topk followed by qsa_sparse_decode as one call (same arguments,
 * same sel / nsel / out / lse results, bit for bit).  For decode rows (R = 1)
 * whose selection scratch fits the attention kernel's staging memory (MB up
 * to about 15,000 blocks) it is ONE launch: every attention CTA selects its
 * row from the scores itself and one CTA per row writes sel and nsel, so the
 * selection's separate launch and its round trip through memory leave the
 * step; otherwise it launches the two kernels.  TensorRT-LLM PR #20276
 * ("Qwen3.8-Flash-Next NVFP4 target"), Decisions worth knowing: canonical
 * selection as a separate composition costs a decode step 2-4%; the fast
 * paths produce the same rows from one fused launch, and the composition
 * remains for wide score tables.  `window` as in qsa_select_topk; the
 * workspace and num_splits as in qsa_sparse_decode_ex (0 = the library's
 * choice; size the workspace with qsa_sparse_decode_workspace_bytes_ex).
 */
/* 1 when qsa_select_sparse_decode runs as one launch for this geometry, 0
 * when it launches the selection and the attention kernels (or the geometry
 * is invalid). */
int qsa_select_sparse_decode_fused(const qsa_geom_t *geom);

qsa_status_t qsa_select_sparse_decode(const qsa_geom_t *geom, const int32_t *scores,
                                      int window, const void *q_bf16,
                                      const uint8_t *k_pool, const uint8_t *k_sf,
                                      const uint8_t *v_pool, const uint8_t *v_sf,
                                      float k_scale, float v_scale, float sm_scale,
                                      const int32_t *page_table, const int32_t *seqlens,
                                      int k, int32_t *sel, int32_t *nsel, void *out_bf16,
                                      float *lse, void *workspace, size_t workspace_bytes,
                                      int num_splits, cudaStream_t stream);

/*
 * qsa_sparse_decode for callers that cannot allocate device memory (no
 * counterpart in the method's description: it exists for deployment).  Some
 * callers never get to call cudaMalloc -- an allocator-free runtime, a memory
 * pool that must not grow once serving starts, a plugin that is only handed
 * input and output pointers -- so they have no workspace to pass.  This call
 * takes the same inputs and outputs as qsa_sparse_decode minus the workspace
 * and uses a 4 MiB scratch array built into the library instead; it allocates
 * and frees nothing.
 *
 *  - The array lives on every GPU that loads the library, until the process
 *    exits, and all calls on a GPU share it: calls that overlap on the GPU
 *    (different streams or host threads) race and must be serialised by the
 *    caller.  Its split tickets start at zero and every call leaves them at
 *    zero, so nothing is cleared between calls.
 *  - Every call looks up the array's device address (host-only); the first
 *    call on a device may also load the library's device code, so make it
 *    before capturing any stream into a CUDA graph.
 *  - The KV split count is lowered until the split partials fit the array;
 *    when even one split does not fit (more than about a million
 *    (request, KV head, column group) units), the call returns
 *    QSA_ERR_WORKSPACE without launching.
 *  - A bounded device wait that gives up sets the array's status word, which
 *    stays set until qsa_sparse_decode_noalloc_status() reads it.
 *  - Other arguments are validated as in qsa_sparse_decode.
 */
qsa_status_t qsa_sparse_decode_noalloc(const qsa_geom_t *geom, const void *q_bf16,
                                       const uint8_t *k_pool, const uint8_t *k_sf,
                                       const uint8_t *v_pool, const uint8_t *v_sf,
                                       float k_scale, float v_scale, float sm_scale,
                                       const int32_t *page_table,
                                       const int32_t *seqlens, const int32_t *sel,
                                       int k, void *out_bf16, float *lse,
                                       cudaStream_t stream);

/*
 * Reads and clears the status word of the built-in scratch array of
 * qsa_sparse_decode_noalloc on the current device (synchronising `stream`):
 * *device_code = 0 and QSA_OK when every bounded device wait of the calls
 * since the previous query completed, otherwise the nonzero code and
 * QSA_ERR_DEVICE_TIMEOUT (the outputs of those calls are not valid).
 */
qsa_status_t qsa_sparse_decode_noalloc_status(int *device_code, cudaStream_t stream);

/*
 * Decode prologue: store the step's new tokens into the cache before A1.
 * TensorRT-LLM PR #20937 ("GB300 perf work on
 * qwen3_8_flash_next_nvfp4__sm_103__tp1"), What changes: a decode prologue over
 * the NVFP4 KV cache that also serves verify steps; Walkthrough, changes
 * table: NVFP4 storage in the decode prologue.  [F]: e2m1 pages with e4m3
 * block scales, one page index for every pool.
 *
 *   k_new, v_new  bf16 [T, Hkv, D]    the new rows' keys and values
 *   ik_new        int8 [T, 64]        the new rows' index keys
 *   k_scale,
 *   v_scale       fp32 > 0            per-tensor dequant multipliers (the same
 *                                     values qsa_sparse_decode is given)
 *   page_table, seqlens               as above; seqlens already count the R
 *                                     new rows
 *   k_pool, k_sf, v_pool, v_sf, ik_pool   the cache pools (layouts as in
 *                                     qsa_sparse_decode / qsa_index_scores),
 *                                     written in place
 *
 * Row j of request b is the token at position L_b - R + j: block
 * (L_b - R + j) / P, slot (L_b - R + j) % P of its page; rows whose position
 * is negative, at or past MB*P, or whose page is invalid are skipped.  Each
 * 16-element block of a K or V row is quantised as
 *   sf = e4m3_rne_satfinite((max|x| / 6) / scale)
 *   code_i = e2m1_rne_satfinite(x_i / (e4m3(sf) * scale))
 * (every division and product in IEEE fp32, in that order; all codes 0 when
 * e4m3(sf) * scale is 0; a code rounded to magnitude zero is stored as +0).
 * The index key is copied as is.  Only the written slots change.
 * Returns QSA_ERR_INVALID_ARG for null pointers, non-positive or non-finite
 * scales, k_new / v_new not D/16-byte aligned, ik_new / ik_pool not 4-byte
 * aligned or k_pool / v_pool not D/64-byte aligned; geometry and device
 * checks as for the other calls.
 */
qsa_status_t qsa_store_kv_tokens(const qsa_geom_t *geom, const void *k_new_bf16,
                                 const void *v_new_bf16, const int8_t *ik_new,
                                 float k_scale, float v_scale,
                                 const int32_t *page_table, const int32_t *seqlens,
                                 uint8_t *k_pool, uint8_t *k_sf, uint8_t *v_pool,
                                 uint8_t *v_sf, int8_t *ik_pool, cudaStream_t stream);

/*
 * Speculative rollback of the cache for rejected draft rows.  TensorRT-LLM PR
 * #20937 ("GB300 perf work on qwen3_8_flash_next_nvfp4__sm_103__tp1"), What
 * changes (Rollback and PLE): batched rollback of the QSA index planes; the
 * rollback gather / restore operations; review of their test: rejected rows
 * get their old values back, kept rows stay untouched.
 *
 * A verify step stores its R new rows into the slots at positions
 * L_b - R + j (qsa_store_kv_tokens).  Call qsa_rollback_gather with the
 * step's page_table and seqlens BEFORE that store: it copies what those slots
 * hold now into `saved`.  After the step, qsa_rollback_restore writes the
 * saved bytes back for every row r with rejected[r] != 0 and leaves the other
 * rows' slots as the step left them.  Rows without a slot (negative position,
 * position at or past MB*P, invalid page) are skipped by both calls.
 *
 *   saved     device bytes, qsa_rollback_state_bytes(geom) long, 4-byte
 *             aligned, owned by the caller; row r's part starts at
 *             r * ((D + D/8) * Hkv + 64) and holds, per KV head, the K codes
 *             (D/2 bytes), K scales (D/16), V codes (D/2), V scales (D/16),
 *             then the index key (64)
 *   rejected  int32 [T], nonzero for a rejected row
 *   pools     as in qsa_store_kv_tokens (4-byte aligned here)
 *
 * The caller updates seqlens for the accepted prefix itself.  Returns
 * QSA_ERR_INVALID_ARG for null or misaligned pointers; geometry and device
 * checks as for the other calls.
 */
size_t qsa_rollback_state_bytes(const qsa_geom_t *geom);
qsa_status_t qsa_rollback_gather(const qsa_geom_t *geom, const int32_t *page_table,
                                 const int32_t *seqlens, const uint8_t *k_pool,
                                 const uint8_t *k_sf, const uint8_t *v_pool,
                                 const uint8_t *v_sf, const int8_t *ik_pool, void *saved,
                                 cudaStream_t stream);
qsa_status_t qsa_rollback_restore(const qsa_geom_t *geom, const int32_t *page_table,
                                  const int32_t *seqlens, const int32_t *rejected,
                                  const void *saved, uint8_t *k_pool, uint8_t *k_sf,
                                  uint8_t *v_pool, uint8_t *v_sf, int8_t *ik_pool,
                                  cudaStream_t stream);

/*
 * Context (prefill) row groups: row-tile sparse GQA on the tensor cores.
 * TensorRT-LLM PR #20276 ("Qwen3.8-Flash-Next NVFP4 target"), Performance
 * (what runs on the fast paths): context steps run a row-tile sparse GQA on
 * tcgen05 that reads K/V tiles once per group of rows of one request; Known
 * limitations: context rows read the NVFP4 pages dequantised to bf16 through
 * the row-tile pass.  PR #20937, What changes: the page conversion and the
 * row-tile planning.
 *
 * Same arguments, layouts and result as qsa_sparse_decode (out = softmax
 * attention of every row and head over the tokens of the blocks its row
 * selected that it sees; lse the natural log of the softmax sum, -inf and
 * out = 0 for a row with no such token), for rows_per_req up to 4096: the
 * rows of a request are taken in tiles of floor(128 / G) consecutive rows
 * (the 128 query vectors of one tensor-core tile), each tile reading the
 * union of its rows' selected pages once.  The pages are dequantised on chip
 * to fp16 (e2m1 x e4m3 is exact; the per-tensor scales are applied in fp32),
 * so no converted copy of the cache is written.
 *
 *   workspace   >= qsa_sparse_prefill_workspace_bytes() bytes (its status
 *               word), 256-byte aligned, zero-filled once by
 *               qsa_workspace_init().
 *
 * head_dim 256 (the geometry above, 32-token pages) runs 32-token chunks with
 * 512 tensor-memory columns per tile.
 *
 * Returns QSA_ERR_UNSUPPORTED for more than 128 query heads
 * per KV head, or a tile (floor(128 / G) rows x k selections plus their union)
 * beyond one CTA's shared memory; QSA_ERR_INVALID_ARG for null pointers, k <
 * 1, k_scale or sm_scale not positive and finite, v_scale not finite, pools /
 * scales / q / out not 16-byte aligned; QSA_ERR_WORKSPACE for a
 * missing, short or misaligned workspace.  A bounded device wait that gives
 * up is reported through qsa_workspace_status().
 */
size_t qsa_sparse_prefill_workspace_bytes(const qsa_geom_t *geom, int k);
qsa_status_t qsa_sparse_prefill(const qsa_geom_t *geom, const void *q_bf16,
                                const uint8_t *k_pool, const uint8_t *k_sf,
                                const uint8_t *v_pool, const uint8_t *v_sf, float k_scale,
                                float v_scale, float sm_scale, const int32_t *page_table,
                                const int32_t *seqlens, const int32_t *sel, int k,
                                void *out_bf16, float *lse, void *workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * Diagnostics: sets the bound, in nanoseconds, of the waits of the head_dim
 * 128 sparse decode kernel for its page copies (2 s by default; 0 restores
 * the default).  Process-wide, for tests of the timeout reporting: a bound
 * below 1 us makes each wait one non-blocking probe, which gives up when the
 * copy has not landed yet (the first probe follows the copy's request); the
 * kernel records QSA_ERR_DEVICE_TIMEOUT in its status word, stops issuing
 * copies, lets those in flight land (under the default bound) and finishes;
 * that call's out and lse are not valid.
 */
void qsa_debug_set_wait_ns(unsigned long long ns);

/*
 * Diagnostics: the bounds-checked build (compiled with QSA_DEBUG_BOUNDS)
 * checks, in every kernel, the indices it derives from data before the access
 * (page ids and token offsets of the copies it issues, chunk-list, union and
 * selection slots in shared memory, output rows, workspace units); a failed
 * check records its code in a device word -- the first failure per source
 * file wins -- and skips the access, never trapping.  This call returns the
 * first nonzero code over the library's source files on the current device
 * and clears them all (it synchronises the device): 0 when every check held,
 * -1 in a build without the checks (the normal library) or on a CUDA error.
 * Codes are 0xF0S: F the source file (1 decode-row attention, 2 decode and
 * verify attention, 3 index scores, 4 selection, 5 token store, 6 rollback,
 * 7 row-tile attention), S the check.  Not thread-safe against concurrent
 * calls of the library.
 */
int qsa_debug_bounds_status(void);

/*
 * Reads the workspace's device status word (synchronising `stream`): 0 when
 * every bounded wait since qsa_workspace_init() completed, otherwise a
 * nonzero code and QSA_ERR_DEVICE_TIMEOUT is returned.  Diagnostic only.
 */
qsa_status_t qsa_workspace_status(const void *workspace, int *device_code,
                                  cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H_ */
