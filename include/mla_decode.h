/*
 * mla_decode.h -- C ABI of libmla_decode.so: absorbed multi-head latent
 * attention (MLA) decode on GB300 (sm_103a).
 *
 * The operation (one query token per request, per head):
 *
 *   for request b with context rows K_b = kv_cache[kv_indices[kv_indptr[b] .. kv_indptr[b+1])]
 *   and head h with q = [q_nope[b,h,0:512], q_rope[b,h,0:64]]:
 *       s_t        = sm_scale * (q_nope . c_t + q_rope . k_rope_t)     c_t = row[0:512], k_rope_t = row[512:576]
 *       lse[b,h]   = ln sum_t exp(s_t)
 *       out[b,h,:] = sum_t softmax(s)_t * c_t                            (the latent is also the value)
 *
 * Sources: "实现差距：MLA 与 DeepSeek V3", section 2.4 (MLA Pallas kernel V2,
 * core computation: dual-path score, FA2-style online softmax, kv_c reused as
 * the value) and section 2.1 (the 576-wide row: kv_latent 512 then k_rope 64);
 * "Attention backends", paragraphs "MLA" (one 576-wide vector per token shared
 * by all heads) and "Paged, ragged batches" (page size 1, kv_indptr /
 * kv_indices CSR, a host-side plan() that picks split-KV chunking and balances
 * long and short contexts across SMs); "Attention backends", paragraph
 * "FlashAttention" (Flash-Decoding: keys split across blocks, partial results
 * merged with the same rescaling).
 *
 * Conventions for every entry point:
 *   - All memory is owned by the caller; the library never allocates.
 *   - Device pointers must be 16-byte aligned; tensors are dense row-major.
 *   - bf16 means IEEE bfloat16 (the bits of the upper half of an fp32).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - No function throws or aborts; each returns an mla_status.  Arguments are
 *     checked on the host before any launch; on a bad argument nothing is
 *     launched and nothing is written.
 *   - Supported head counts: 16 and 32 (one CTA per SM) and 48..128 in steps
 *     of 16 (a two-CTA cluster per worker); both work in 64-token tiles.
 *     kv_lora_rank is 512 and qk_rope_head_dim is 64; nothing else is built.
 *   - The natural log is used for every LSE.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, malformed kv_indptr, bad plan */
  MLA_ERR_UNSUPPORTED = 2,   /* head count or dtype the library does not build */
  MLA_ERR_WORKSPACE = 3,     /* plan or workspace buffer too small */
  MLA_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, attribute, device query) */
  MLA_ERR_TIMEOUT = 5,       /* a device-side wait exceeded its limit (~1 s); the kernel returned early */
  MLA_ERR_INDEX_OOB = 6,     /* a kv_indices value was outside [0, num_slots); row 0 was read instead */
  MLA_ERR_PLAN_MISMATCH = 7, /* a plan work item does not lie inside its request's kv_indptr range */
  MLA_ERR_TREE = 8           /* a draft tree names a parent that is not an earlier draft or -1; that draft
                                was verified as a child of the context */
} mla_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* mla_status_string(int status);

/* Library ABI version (currently 1). */
int mla_abi_version(void);

/* mla_decode_plan -- host only, no device work, deterministic.
 *
 * Builds the split-KV work plan for one decode batch ("Attention backends",
 * paragraph "Paged, ragged batches": plan() rebuilt on the CPU per batch,
 * choosing per-request chunking and balancing long and short contexts).
 *
 *   kv_indptr          host int32[batch+1]; kv_indptr[0] == 0, non-decreasing.
 *   batch              number of requests B >= 0.
 *   num_heads          H (see supported head counts above).
 *   num_sms            SMs to plan for; 0 = query the current CUDA device.
 *   plan               host int32 buffer of plan_words words that receives the
 *                      plan, or NULL to only report the sizes.
 *   plan_words_needed  out: words the plan takes (always written when non-NULL).
 *   workspace_bytes    out: device workspace bytes mla_decode_run needs for this
 *                      plan (fp32 partial states plus a 256-byte status header).
 *
 * Rule: tiles of T = 64 tokens; W workers = SMs (H <= 32) or SMs/2; a piece
 * of n tokens costs its whole tiles plus 32 tokens (its epilogue); requests,
 * in order, are poured into workers 0, 1, ... each up to a load budget, so a
 * request is cut only where a worker is full and only at a tile boundary of
 * the request (no cut piece shorter than 64 tokens); the budget starts at the
 * balanced share and grows in steps of 8 tokens until W workers suffice.
 * Requests left whole are written straight to out/lse; cut or empty requests
 * go through the LSE merge.
 *
 * Returns MLA_OK, MLA_ERR_INVALID_ARG (malformed kv_indptr, negative batch),
 * MLA_ERR_UNSUPPORTED (head count), MLA_ERR_WORKSPACE (plan too small; sizes
 * are still reported) or MLA_ERR_CUDA (num_sms == 0 and no device).
 */
int mla_decode_plan(const int32_t* kv_indptr, int32_t batch, int32_t num_heads, int32_t num_sms,
                    int32_t* plan, size_t plan_words, size_t* plan_words_needed,
                    size_t* workspace_bytes);

/* mla_decode_run -- asynchronous on `stream`.
 *
 *   plan_host     host copy of the plan words from mla_decode_plan (read now).
 *   plan_dev      device copy of the same words (read by the kernels).
 *   q_nope        device bf16 [batch, H, 512]: q_nope already multiplied by W_UK.
 *   q_rope        device bf16 [batch, H, 64]: the rotary part of the query.
 *   kv_cache      device bf16 [num_slots, 576]: latent [0,512) then rope key [512,576).
 *   num_slots     rows in kv_cache (1 .. 2^31-1).
 *   kv_indptr     device int32 [batch+1], equal to the host array the plan was built from.
 *   kv_indices    device int32 [kv_indptr[batch]]: slot of every context token.
 *   sm_scale      softmax scale applied to the summed score.
 *   out           device [batch, H, 512], fp32 (out_dtype 0) or bf16 (out_dtype 1).
 *   lse           device fp32 [batch, H] (natural log), or NULL to skip it.
 *   workspace     device buffer of at least the planned workspace_bytes; must be
 *                 zero-filled before its first use (its first 256 bytes hold the
 *                 sticky device status read by mla_check_errors).
 *
 * Launches the decode kernel and, when the plan cut or left empty any request,
 * the merge kernel.  An empty request (kv_indptr[b+1] == kv_indptr[b]) gets
 * out = 0 and lse = -inf.  When no request has a token the decode kernel is
 * not launched (q_nope, q_rope, kv_cache, kv_indptr and kv_indices may then be
 * NULL) and the merge alone writes out and lse; with batch == 0 nothing is
 * launched and only plan_dev and workspace are checked (the other device
 * pointers may be NULL).  Device-side faults are not possible from bad indices: an
 * index outside [0, num_slots) reads row 0 and sets MLA_ERR_INDEX_OOB in the
 * workspace status.  The call does not synchronise; read device-side status
 * with mla_check_errors.  Safe to capture in a CUDA graph (no host sync, no
 * allocation) as long as the plan words stay unchanged.
 */
int mla_decode_run(const int32_t* plan_host, const int32_t* plan_dev,
                   const void* q_nope, const void* q_rope,
                   const void* kv_cache, int64_t num_slots,
                   const int32_t* kv_indptr, const int32_t* kv_indices,
                   float sm_scale, void* out, int32_t out_dtype, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream);

/* mla_decode_attend / mla_decode_merge -- the two launches of mla_decode_run,
 * callable separately (same arguments and checks).  mla_decode_attend runs
 * the decode kernel: requests the plan left whole get their out/lse, cut
 * requests leave fp32 partial states in the workspace.  mla_decode_merge then
 * combines the partials of every cut request (and writes out = 0, lse = -inf
 * for empty requests); it launches nothing when the plan has no such request.
 * mla_decode_run == mla_decode_attend followed by mla_decode_merge. */
int mla_decode_attend(const int32_t* plan_host, const int32_t* plan_dev,
                      const void* q_nope, const void* q_rope,
                      const void* kv_cache, int64_t num_slots,
                      const int32_t* kv_indptr, const int32_t* kv_indices,
                      float sm_scale, void* out, int32_t out_dtype, float* lse,
                      void* workspace, size_t workspace_bytes, void* stream);

int mla_decode_merge(const int32_t* plan_host, const int32_t* plan_dev, void* out,
                     int32_t out_dtype, float* lse, void* workspace, size_t workspace_bytes,
                     void* stream);

/* mla_merge_states -- asynchronous on `stream`.
 *
 * Flash-Decoding merge ("Attention backends", paragraph "FlashAttention"):
 * for request b, partial states i in [merge_indptr[b], merge_indptr[b+1]):
 *   M = max_i s_i;  w_i = exp(s_i - M);  out = sum_i w_i v_i / sum_i w_i;
 *   lse = M + ln sum_i w_i.
 * Partials with s_i = -inf carry no weight; a request with no live partial
 * gets out = 0 and lse = -inf.
 *
 *   v_partial     device fp32 [P, H, 512], each partial already normalised.
 *   s_partial     device fp32 [P, H], the partial LSEs (natural log).
 *   merge_indptr  device int32 [batch+1], non-decreasing, merge_indptr[0] == 0.
 *   out, lse      as for mla_decode_run (lse may be NULL).
 */
int mla_merge_states(const float* v_partial, const float* s_partial, const int32_t* merge_indptr,
                     int32_t batch, int32_t num_heads, void* out, int32_t out_dtype, float* lse,
                     void* stream);

/* mla_decode_run_noalloc -- mla_decode_run without a caller-provided workspace.
 *
 * No counterpart on the pages: this entry point exists for callers that are
 * not allowed to allocate device memory at the point of the call -- code
 * running inside a memory arena owned by another runtime, plugins that only
 * receive tensors they did not allocate, or a decode step that must not call
 * cudaMalloc while it runs.  It takes the same arguments as mla_decode_run
 * except the workspace: the split-KV partial states and the device status go
 * to one static device buffer of MLA_NOALLOC_SCRATCH_BYTES (32 MiB) that is
 * part of the library image, so every GPU that loads the library holds it
 * until the process exits.
 *
 *   - The first call on a device looks the buffer's device address up for
 *     that device (a runtime query, no allocation); make that first call
 *     before any stream capture.  The address is cached per device and per
 *     CUDA context: after cudaDeviceReset (or anything else that replaces
 *     the device's context) the next call looks it up again, so that call,
 *     too, must not be inside a stream capture.
 *   - Plans whose partial states do not fit (256 B + P*H*513*4 bytes larger
 *     than MLA_NOALLOC_SCRATCH_BYTES) are rejected with MLA_ERR_WORKSPACE
 *     and nothing is launched.
 *   - Every call shares the one buffer: calls that overlap on the GPU (on
 *     different streams, or from different threads) race and corrupt each
 *     other's partial states.  Serialise them on one stream.
 *   - The buffer's status word starts at zero (static initialisation) and,
 *     like a caller workspace's, keeps the first device-side error (bad slot
 *     index, timeout, plan mismatch) of any call until
 *     mla_noalloc_check_errors reads and clears it.
 *   - Nothing here calls cudaMalloc, cudaFree or an allocating routine. */
#define MLA_NOALLOC_SCRATCH_BYTES (32u << 20)
int mla_decode_run_noalloc(const int32_t* plan_host, const int32_t* plan_dev,
                           const void* q_nope, const void* q_rope,
                           const void* kv_cache, int64_t num_slots,
                           const int32_t* kv_indptr, const int32_t* kv_indices,
                           float sm_scale, void* out, int32_t out_dtype, float* lse,
                           void* stream);

/* mla_noalloc_check_errors -- the device status of mla_decode_run_noalloc.
 *
 * Synchronises `stream`, then reads the status word of the static buffer on
 * the current device and clears it when it is non-zero (the same contract as
 * mla_check_errors on a caller workspace).  Returns MLA_OK, the first
 * MLA_ERR_* a kernel recorded since the last read, or MLA_ERR_CUDA when the
 * stream or the copy failed.  It allocates nothing: the word is copied into a
 * host int.  Like the entry point it reports on, it has no counterpart on the
 * pages. */
int mla_noalloc_check_errors(void* stream);

/* mla_merge_two_states -- asynchronous on `stream`.
 *
 * Row-wise merge of two attention states over disjoint key sets, for every
 * row r of `rows` (a row is a request-head pair, 512 wide):
 *   m = max(lse_a, lse_b);  w = exp(lse - m);
 *   out = (w_a o_a + w_b o_b) / (w_a + w_b);  lse = m + ln(w_a + w_b)
 * with -inf states weighing nothing (both -inf: out = 0, lse = -inf).  This
 * is the last step of a shared-prefix cascade ("[sglang] EAGLE 트리 검증
 * 어텐션 최적화", section "들어가며": prefix attention shared by every query,
 * suffix attention per query, the two merged by LSE): the prefix pass runs
 * mla_decode_run once over the prefix rows with the G x H query rows of G
 * requests as the heads of one request (each prefix row gathered once), the
 * suffix pass is an ordinary mla_decode_run, both with fp32 out.
 *   o_a, o_b    device fp32 [rows, 512];  lse_a, lse_b  device fp32 [rows].
 *   out         device [rows, 512], fp32 (0) or bf16 (1); may be o_a.
 *   lse         device fp32 [rows] or NULL; may be lse_a. */
int mla_merge_two_states(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b, int64_t rows,
                         void* out, int32_t out_dtype, float* lse, void* stream);

/* mla_decode_run_multi_query -- asynchronous on `stream`.
 *
 * Verification of q_len draft tokens per request in one pass ("[sglang]
 * EAGLE 트리 검증 어텐션 최적화", section "들어가며": every query attends to
 * the shared context and to its ancestor drafts; this is the chain case).
 * Request b's context of L_b rows (kv_indptr / kv_indices) ends with its
 * q_len drafts; query i (0-based) attends to its first L_b - q_len + 1 + i
 * rows.  The q_len x H query rows are read as the heads of one request, so
 * each cache row is gathered once for all of them:
 *   plan        mla_decode_plan(kv_indptr, B, q_len * H, ...).
 *   q_nope      bf16 [B, q_len, H, 512];  q_rope  bf16 [B, q_len, H, 64].
 *   out, lse    [B, q_len, H, 512] (out_dtype as for mla_decode_run), [B, q_len, H].
 * A query row with no row to attend to (L_b < q_len) gets out = 0, lse = -inf.
 * Both decode kernels apply the per-row limit (q_len * H of 16 or 32: one CTA
 * per worker; 48..128: a two-CTA cluster).
 * Errors: MLA_ERR_INVALID_ARG when q_len < 1 or the plan's head count is not a
 * multiple of q_len; otherwise as for mla_decode_run (q_len = 1 is
 * mla_decode_run). */
int mla_decode_run_multi_query(const int32_t* plan_host, const int32_t* plan_dev, int32_t q_len,
                               const void* q_nope, const void* q_rope, const void* kv_cache, int64_t num_slots,
                               const int32_t* kv_indptr, const int32_t* kv_indices, float sm_scale, void* out,
                               int32_t out_dtype, float* lse, void* workspace, size_t workspace_bytes,
                               void* stream);

/* mla_decode_run_tree -- asynchronous on `stream`.
 *
 * Verification of a TREE of W = q_len draft tokens per request in one pass
 * ("[sglang] EAGLE 트리 검증 어텐션 최적화", section "들어가며": with topk > 1
 * the drafts form a tree, and each query token attends to the verified
 * context and to its own ancestor chain among the drafts).  Request b's
 * context of L_b rows ends with its W drafts in generation order; query i
 * sees the first L_b - W rows and, among the last W, the drafts on its path
 * to the root and itself.  Layouts and plan as for mla_decode_run_multi_query
 * (the W x H query rows are the heads of one request, each cache row is
 * gathered once for all of them), plus:
 *   tree_parents  device int32 [B, W]: parents[b][i] = the draft that draft i
 *                 extends (0 <= parent < i), or -1 for a child of the context.
 *                 Read only.  An entry outside [-1, i) records MLA_ERR_TREE
 *                 (mla_check_errors) and draft i is verified as a child of
 *                 the context.
 *   tree_masks    device uint64 [B, W], 8-byte aligned, caller-owned scratch:
 *                 the call writes each draft's ancestor-or-self bits there
 *                 (a small kernel on `stream`) and the decode kernels read
 *                 them; it must stay allocated until the call's work is done.
 * W = 1 is mla_decode_run.  Both decode kernels apply the masks (W * H of 16
 * or 32: one CTA per worker; 48..128: a two-CTA cluster).
 * Errors: MLA_ERR_INVALID_ARG when W < 1, the plan's head count is not a
 * multiple of W, or tree_parents / tree_masks is null or misaligned;
 * MLA_ERR_UNSUPPORTED when W > 64; otherwise as for mla_decode_run. */
int mla_decode_run_tree(const int32_t* plan_host, const int32_t* plan_dev, int32_t q_len,
                        const int32_t* tree_parents, uint64_t* tree_masks, const void* q_nope, const void* q_rope,
                        const void* kv_cache, int64_t num_slots, const int32_t* kv_indptr, const int32_t* kv_indices,
                        float sm_scale, void* out, int32_t out_dtype, float* lse, void* workspace,
                        size_t workspace_bytes, void* stream);

/* mla_decode_step_host -- one decode step from HOST buffers, asynchronous on `stream`.
 *
 * Plans the batch on the host (mla_decode_plan with the current device's SM
 * count) into `plan`, copies the plan words, q_nope, q_rope, kv_indptr and
 * kv_indices into the caller's device `staging` buffer, runs mla_decode_run
 * there, and copies out and lse back into host memory -- seven
 * cudaMemcpyAsync and the decode's launches.  The kernels go on `stream`,
 * the copies in on `copy_in_stream` and the copies out on `copy_out_stream`
 * when those are not NULL (ordered with the kernels through events), else on
 * `stream`.  With page-locked host buffers every copy is asynchronous: keep
 * the host buffers (and `plan`) unchanged until the copies have passed this
 * step.  A serving loop alternates two staging buffers over consecutive
 * steps with one copy-in and one copy-out stream, so one step's copies
 * overlap its neighbours' kernels.
 *
 *   q_nope, q_rope, kv_indptr, kv_indices, out, lse
 *               HOST buffers, same shapes and dtypes as for mla_decode_run.
 *   kv_cache    device, as for mla_decode_run.
 *   plan        host int32 buffer of plan_words (query the size with
 *               mla_decode_plan(..., plan = NULL, ...)).
 *   staging     device buffer of at least mla_step_staging_bytes(batch,
 *               num_heads, nnz, plan words, out_dtype) bytes.
 *   workspace   device, at least the plan's workspace bytes.
 * Errors: those of mla_decode_plan and mla_decode_run; MLA_ERR_WORKSPACE when
 * staging or workspace is too small; MLA_ERR_INVALID_ARG for null pointers or
 * batch < 1.  Nothing is copied or launched on an error found before the
 * first copy. */
size_t mla_step_staging_bytes(int32_t batch, int32_t num_heads, int64_t nnz, size_t plan_words, int32_t out_dtype);
int mla_decode_step_host(const void* q_nope, const void* q_rope, const int32_t* kv_indptr,
                         const int32_t* kv_indices, int32_t batch, int32_t num_heads, const void* kv_cache,
                         int64_t num_slots, float sm_scale, void* out, int32_t out_dtype, float* lse,
                         int32_t* plan, size_t plan_words, void* staging, size_t staging_bytes, void* workspace,
                         size_t workspace_bytes, void* stream, void* copy_in_stream, void* copy_out_stream);

/* mla_absorb_query -- asynchronous on `stream`.
 *
 * The query side of the absorbing path ("MLA and torch.compile: v0.3's two
 * sources", section "MLA: starting from a 439-line commit": q_nope is
 * multiplied by w_kc before attention): for every request b and head h,
 *   q_nope[b, h, :] = q_pre[b, h, 0:128] . w_kc[h]        (fp32 sums, bf16 result)
 * which is the q_nope that mla_decode_run takes.
 *
 *   q_pre     device bf16 [batch, num_heads, nope_dim], nope_dim = 128.
 *   w_kc      device bf16 [num_heads, nope_dim, 512], row-major per head.
 *   q_nope    device bf16 [batch, num_heads, 512] (written).
 *   workspace NULL, or a decode workspace whose status word records a timeout
 *             (read with mla_check_errors).
 * Errors: MLA_ERR_UNSUPPORTED for nope_dim != 128; MLA_ERR_INVALID_ARG for
 * null or non-16-byte-aligned pointers, batch < 0 or num_heads < 1; nothing
 * is launched then.  batch == 0 launches nothing. */
int mla_absorb_query(const void* q_pre, const void* w_kc, void* q_nope, int32_t batch, int32_t num_heads,
                     int32_t nope_dim, void* workspace, void* stream);

/* mla_project_output -- asynchronous on `stream`.
 *
 * The output side of the absorbing path (same section: the attention's
 * latent output is multiplied by w_vc): for every request b and head h,
 *   out[b, h, :] = o_lat[b, h, 0:512] . w_vc[h]            (fp32 sums)
 *
 *   o_lat     device bf16 [batch, num_heads, 512] (mla_decode_run with
 *             out_dtype 1).
 *   w_vc      device bf16 [num_heads, 512, v_dim], row-major per head, v_dim = 128.
 *   out       device [batch, num_heads, v_dim], fp32 (out_dtype 0) or bf16 (1).
 *   workspace as for mla_absorb_query.
 * Errors as for mla_absorb_query (v_dim != 128 or a bad out_dtype give
 * MLA_ERR_UNSUPPORTED). */
int mla_project_output(const void* o_lat, const void* w_vc, void* out, int32_t out_dtype, int32_t batch,
                       int32_t num_heads, int32_t v_dim, void* workspace, void* stream);

/* mla_append_kv -- asynchronous on `stream`.
 *
 * Writes a decode step's new cache rows: rows[b] (576 bf16: the 512-wide
 * latent, then the 64-wide rope key) goes to kv_cache[slots[b]]
 * ("实现差距：MLA 与 DeepSeek V3", section 2.4: the new token's kv_c and k_pe
 * are written to the cache before attention).  Run it before mla_decode_run
 * on the same stream when the new tokens' slots are in kv_indices.
 *
 *   kv_cache   device bf16 [num_slots, 576], written in place.
 *   slots      device int32 [batch], distinct (two rows to one slot: either may win).
 *   rows       device bf16 [batch, 576].
 *   workspace  NULL, or a decode workspace: a slot outside [0, num_slots) is
 *              skipped and recorded there as MLA_ERR_INDEX_OOB (mla_check_errors).
 * Errors: MLA_ERR_INVALID_ARG for null or non-16-byte-aligned pointers,
 * batch < 0 or num_slots < 1; nothing is launched then. */
int mla_append_kv(void* kv_cache, int64_t num_slots, const int32_t* slots, const void* rows, int32_t batch,
                  void* workspace, void* stream);

/* ---- decode with a device-only plan (CUDA-graph replays) -------------------
 * "Attention backends", paragraphs "Paged, ragged batches" and "The
 * interface": for decode the CSR arrays live in buffers sized for the largest
 * captured batch, so a captured graph replays kernels whose inputs change
 * every step; before each replay the runner writes the new plan into those
 * buffers.  mla_decode_run bakes the host plan's merge count and partial
 * layout into its launches; this variant reads everything that changes from
 * the device plan, so one capture serves every plan built for the same
 * (max_batch, num_heads, num_sms). */

/* mla_decode_graph_sizes -- host.  Capacities for plans of up to max_batch
 * requests: *plan_words (int32 words of the device plan buffer) and
 * *workspace_bytes (status header, then room for max_batch + W - 1 partial
 * states, W = the plan's workers).  Any plan mla_decode_plan builds for
 * batch <= max_batch with the same num_heads and num_sms fits.
 * Errors: MLA_ERR_INVALID_ARG for max_batch < 1 or num_sms < 1;
 * MLA_ERR_UNSUPPORTED for an unsupported num_heads. */
int mla_decode_graph_sizes(int32_t max_batch, int32_t num_heads, int32_t num_sms, size_t* plan_words,
                           size_t* workspace_bytes);

/* mla_decode_run_graph -- asynchronous on `stream`; capturable in a CUDA
 * graph and replayable after the buffers' contents change.
 *
 *   plan_dev   device int32 [plan_words]: a plan from mla_decode_plan (same
 *              num_heads and num_sms, batch <= max_batch), copied in before
 *              each launch or replay.  Read only on the device: the kernels
 *              check its header (magic, version, heads, workers, batch, item
 *              count against plan_words) and clamp its ranges; a bad plan
 *              computes nothing and records MLA_ERR_PLAN_MISMATCH.
 *   kv_indptr  device int32 [max_batch + 1]; entries past the plan's batch
 *              repeat its last value.
 *   q_nope, q_rope, out, lse: [max_batch, ...] as for mla_decode_run;
 *              rows of requests past the plan's batch are not written.
 *   workspace  >= the workspace_bytes of mla_decode_graph_sizes, 16-byte
 *              aligned, zero-filled before first use.
 *   other arguments as for mla_decode_run.
 * Launches the decode kernel on the plan's workers and the merge kernel over
 * max_batch possible entries (each block reads the plan's merge count).
 * Errors: MLA_ERR_WORKSPACE when plan_words or workspace_bytes are below the
 * capacities; otherwise as for mla_decode_run, with nothing launched. */
int mla_decode_run_graph(const int32_t* plan_dev, size_t plan_words, int32_t max_batch, int32_t num_heads,
                         int32_t num_sms, const void* q_nope, const void* q_rope, const void* kv_cache,
                         int64_t num_slots, const int32_t* kv_indptr, const int32_t* kv_indices, float sm_scale,
                         void* out, int32_t out_dtype, float* lse, void* workspace, size_t workspace_bytes,
                         void* stream);

/* ---- FP8 latent cache ----------------------------------------------------
 * "MLA and torch.compile: v0.3's two sources", section "MLA: starting from a
 * 439-line commit": an FP8 KV cache is one of the four parts of the 3-7x
 * (the page's FP8 tensors are float8_e4m3fn); "实现差距：MLA 与 DeepSeek V3",
 * section 2.4: new rows are packed into the FP8 cache.  Format taken here:
 * one E4M3 code (OCP "fn" variant: no infinities, largest finite 448) per
 * value, 576 bytes per row (latent 0-511, rope key 512-575), and one float32
 * kv_scale for the whole cache: value = code value x kv_scale. */

/* mla_decode_fp8_workspace_bytes -- host.  Workspace mla_decode_run_fp8 needs
 * for `plan`: the plan's own workspace plus the per-request query images
 * (4 x H x 288 bytes) and per-head factors (H floats).
 * Errors: MLA_ERR_INVALID_ARG for a bad plan or null result pointer. */
int mla_decode_fp8_workspace_bytes(const int32_t* plan_host, size_t* workspace_bytes);

/* mla_decode_run_fp8 -- asynchronous on `stream`.
 *
 * mla_decode_run over an FP8 cache: the same out / lse as the bf16 decode of
 * the cache values (code value x kv_scale), with the bf16 query used as is.
 * Every head count of mla_decode_plan is supported (16 or 32: one CTA per
 * worker; 48..128: a two-CTA cluster; each CTA keeps its own partial score
 * exact and receives its peer's with an error of at most 2^-22 of the largest
 * partial in its 32-token half row).
 *
 *   kv_cache   device uint8 [num_slots, 576] E4M3 codes.
 *   kv_scale   finite, > 0.
 *   workspace  at least mla_decode_fp8_workspace_bytes(plan) bytes, 16-byte
 *              aligned, zero-filled before first use (status word as for
 *              mla_decode_run; the query images are rewritten every call, so
 *              calls sharing a workspace must not overlap on the GPU).
 *   all other arguments as for mla_decode_run.
 * Launches (H 16 / 32) a query-prep kernel (each request's query split into
 * two E4M3 parts after a per-head power-of-two scaling) and the decode kernel
 * as its programmatic dependent, or (H 48..128) the two-CTA kernel, which
 * splits the query itself; then the plan's merge.
 * Errors as for mla_decode_run; nothing is launched on an argument error. */
int mla_decode_run_fp8(const int32_t* plan_host, const int32_t* plan_dev, const void* q_nope, const void* q_rope,
                       const void* kv_cache, int64_t num_slots, float kv_scale, const int32_t* kv_indptr,
                       const int32_t* kv_indices, float sm_scale, void* out, int32_t out_dtype, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream);

/* mla_append_kv_fp8 -- asynchronous on `stream`.
 *
 * mla_append_kv into an FP8 cache: the codes of rows[b] go to slot slots[b],
 * each value divided by kv_scale in float32 (IEEE division) and rounded to
 * the nearest E4M3 value (ties to the even code, magnitudes past 448 to 448).
 *
 *   kv_cache   device uint8 [num_slots, 576], written in place.
 *   rows       device bf16 [batch, 576].
 *   kv_scale   finite, > 0.
 *   slots, workspace as for mla_append_kv.
 * Errors: MLA_ERR_INVALID_ARG for null or non-16-byte-aligned pointers,
 * batch < 0, num_slots < 1 or a bad kv_scale; nothing is launched then. */
int mla_append_kv_fp8(void* kv_cache, int64_t num_slots, const int32_t* slots, const void* rows, int32_t batch,
                      float kv_scale, void* workspace, void* stream);

/* mla_check_errors -- synchronises `stream`, reads the workspace status word,
 * clears it, and returns it (MLA_OK when the kernels found nothing wrong), or
 * MLA_ERR_CUDA if the stream reports a CUDA error. */
int mla_check_errors(void* workspace, void* stream);

/* mla_probe_wait_limit -- asynchronous on `stream`.  A diagnostic of the
 * failure handling, not part of a decode.
 *
 * Every mbarrier wait of the decode and head-product kernels above is bounded:
 * after about 1 s of wall time it gives up, the kernel records MLA_ERR_TIMEOUT in the workspace
 * status word and returns, so a stalled pipeline becomes a status code, not a
 * hung GPU.  This launches one warp whose first thread waits, with that same
 * bounded wait, on a shared-memory barrier that nothing completes: after the
 * limit the status word holds MLA_ERR_TIMEOUT (read and clear it with
 * mla_check_errors) and the context stays usable.  Nothing but the status
 * word is written.
 *
 *   workspace  device, at least 4 bytes, 16-byte aligned (a decode workspace).
 * Errors: MLA_ERR_INVALID_ARG for a null or misaligned workspace; nothing is
 * launched then. */
int mla_probe_wait_limit(void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
