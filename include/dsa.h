/*
 * dsa.h -- C ABI of the DeepSeek Sparse Attention (DSA) forward hot path
 * on NVIDIA GB300 (sm_103a).  Library: libdsa_gb300.so.
 *
 * One decode or prefill step has three stages per query token t:
 *   1. index score  I[t,s] = sum_h w[t,h] * ReLU(q_idx[t,h,:] . k_idx[s,:])
 *      over the keys s that t may see;
 *   2. top-k        the k highest-scoring positions, -1 padded;
 *   3. sparse MLA   softmax attention of q[t] over the selected latent KV
 *      rows (K = the whole row, V = its leading Dv dims), out + lse.
 *
 * Conventions shared by every entry point
 *  - Every tensor pointer is a DEVICE pointer owned by the caller, contiguous
 *    row-major, unless a comment says "host".  The library never allocates or
 *    frees device memory: scratch comes from a caller workspace whose size
 *    the matching *_workspace_size() function returns.
 *  - Work is enqueued on the caller's stream (cudaStream_t passed as
 *    dsa_stream_t; NULL = the legacy default stream).  No entry point
 *    synchronises the host, so results are ready when the stream says so.
 *  - The return value reports errors found on the HOST, before anything is
 *    launched (DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED,
 *    DSA_ERR_WORKSPACE_TOO_SMALL), or a failed launch (DSA_ERR_CUDA).  When
 *    the return is not DSA_OK nothing of that call ran, except for
 *    DSA_ERR_CUDA, where earlier launches of the same call may have run.
 *  - err_flag (optional, device int32, may be NULL) collects errors found on
 *    the DEVICE by OR-ing DSA_DEVERR_* bits into it.  The offending entries
 *    are masked (treated like -1), never read.  The library never clears it.
 *  - Index lists use -1 for "no entry".  A -1 is masked, never clamped into a
 *    read (miles PR #3608 "per-arch DSA sparse attention dispatch", What /
 *    Padding).
 *  - The entry points hold no state between calls and may be captured in a
 *    CUDA graph.
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dsa_stream_t; /* a cudaStream_t */

/* Host-side status codes. */
enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,         /* null pointer, bad size or range   */
  DSA_ERR_UNSUPPORTED = 2,         /* shape / format not supported      */
  DSA_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes below *_workspace_size() */
  DSA_ERR_CUDA = 4                 /* a launch or driver call failed    */
};

/* Device-side error bits OR-ed into *err_flag. */
enum {
  DSA_DEVERR_INDEX_RANGE = 1, /* an index list entry < -1 or >= the pool's rows,
                                 or a key range outside the index-k cache     */
  DSA_DEVERR_TIMEOUT = 2,     /* an internal bounded wait gave up             */
  DSA_DEVERR_FP16_RANGE = 4   /* sparse MLA over an fp8 pool: a dequantised
                                 value or a q element beyond fp16's finite
                                 range (|x| > 65504); that token's output is
                                 not valid                                     */
};

/* Indexer operand types. */
enum { DSA_IDX_BF16 = 0, DSA_IDX_FP8_E4M3 = 1 };

/* KV pool formats (aiter PR #4382 "Paged Sparse Attention Gluon Kernel",
 * section "Supported formats & dtypes"). */
enum {
  DSA_KV_BF16 = 0,        /* data: bf16 [rows, d_nope + d_rope] (576 wide)  */
  DSA_KV_FP8_UNIFORM = 1, /* section "Uniform fp8 pool - 2D": data uint8
                             [rows, D] OCP e4m3, scales fp32 [rows, D/64];
                             x = fp8(byte) * scales[slot, col / 64] for every
                             column, RoPE included                         */
  DSA_KV_FP8_DS_MLA = 2   /* section "Packed fp8 fp8_ds_mla - 3D": data uint8
                             [nb, block, 584]; page = block x 576 data bytes
                             then block x 8 scale bytes; data row = 448 e4m3
                             NoPE bytes + 64 bf16 RoPE; scale row = 7 UE8M0
                             exponents + 1 pad; NoPE x = fp8 * 2^(e - 127)   */
};

/* Limits of the library. */
#define DSA_MAX_TOPK 2048     /* k of dsa_topk / dsa_decode                 */
#define DSA_MAX_INDEX_HEADS 64
#define DSA_MAX_HEADS 128     /* H of dsa_sparse_mla_fwd                    */

/* A latent KV pool.  Slots index rows (bf16, uniform) or tokens
 * (fp8_ds_mla: slot -> page slot / block, row slot % block). */
typedef struct dsa_kv_pool {
  const void *data;     /* device; layout per format above; 16-byte aligned   */
  const float *scales;  /* device; DSA_KV_FP8_UNIFORM only, else NULL          */
  int64_t rows;         /* addressable slots (nb * block for fp8_ds_mla)       */
  int32_t format;       /* DSA_KV_*                                            */
  int32_t block;        /* tokens per page for fp8_ds_mla; 1 otherwise         */
  int32_t d_nope;       /* 512 (bf16) or 448 (fp8 formats)                     */
  int32_t d_rope;       /* 64                                                  */
} dsa_kv_pool;

/* Text for a status code (static storage). */
const char *dsa_status_string(int status);

/* ABI version of this library: 1. */
int dsa_abi_version(void);

/*
 * dsa_index_score -- lightning-indexer scores.
 * The "scores" stage of tokenspeed PR #627 "Add gluon kernel for DSA"
 * (Benchmark results, Decode and Prefill tables); the formula is the DSA
 * indexer's definition:
 *   scores[t*ld_scores + j] = sum_h w[t,h] * ReLU(sq[t,h] * sk[s] *
 *                              (q_idx[t,h,:] . k_idx[s,:])),   s = row_start[t] + j
 * for 0 <= j < row_end[t] - row_start[t].  Entries of a row past its own
 * length are left untouched.  sq, sk are the fp8 per-row scales (all 1 for
 * bf16).
 *   q_idx     [T, H_I, d]  bf16 or e4m3 bytes (idx_dtype)
 *   q_scale   [T, H_I]     fp32, fp8 only (NULL for bf16)
 *   k_idx     [k_rows, d]  same type as q_idx (the index-k cache); k_rows and
 *             T * H_I below 2^31 (else DSA_ERR_UNSUPPORTED)
 *   k_scale   [k_rows]     fp32, fp8 only (NULL for bf16)
 *   w         [T, H_I]     fp32 head weights (any sign)
 *   row_start, row_end [T] int32 key rows [row_start, row_end) of k_idx;
 *             decode: [slot_base, slot_base + seq_len); causal prefill:
 *             [segment start, t + 1)
 *   max_len   host: an upper bound of row_end - row_start over all t
 *   scores    fp32 [T, ld_scores], ld_scores >= max_len
 * Limits: H_I <= 64 and a multiple of 8; d in {64, 128} (bf16) or 128 (fp8).
 * A row range outside [0, k_rows] sets DSA_DEVERR_INDEX_RANGE and that row
 * is skipped.
 */
int dsa_index_score(const void *q_idx, int idx_dtype, const float *q_scale,
                    const void *k_idx, const float *k_scale, int64_t k_rows,
                    const float *w, const int32_t *row_start, const int32_t *row_end,
                    int T, int H_I, int d, int64_t max_len,
                    float *scores, int64_t ld_scores,
                    int32_t *err_flag, dsa_stream_t stream);

/*
 * dsa_index_score_prefill -- dsa_index_score for causal prefill rows.
 * The same arguments, limits, errors and result as dsa_index_score (the
 * "Prefill" table of tokenspeed PR #627 times this stage over causal rows).
 * Rows are taken four at a time (rows 4g .. 4g+3).  Where the group's
 * non-empty rows all start at the same key -- the rows of one segment of a
 * causal prefill, [segment start, t + 1) -- each 128-key tile of the union of
 * their ranges is read and multiplied once for all four rows.  Other groups
 * (a segment boundary inside the group, unrelated ranges) are walked one row
 * at a time.  Any ranges are accepted; grouping pays where consecutive rows
 * share their start.  Shapes without a one-block fast form (bf16 d = 128) and
 * T < 4 run as dsa_index_score does.  Rows of a decode batch, each with its
 * own keys, are better served by dsa_index_score.
 */
int dsa_index_score_prefill(const void *q_idx, int idx_dtype, const float *q_scale,
                            const void *k_idx, const float *k_scale, int64_t k_rows,
                            const float *w, const int32_t *row_start, const int32_t *row_end,
                            int T, int H_I, int d, int64_t max_len,
                            float *scores, int64_t ld_scores,
                            int32_t *err_flag, dsa_stream_t stream);

/*
 * dsa_topk -- per-row top-k with -1 padding.
 * The "TopK" stage of tokenspeed PR #627 (Benchmark results; the selector
 * counts "greater" and "equal" elements against a threshold) with the -1
 * padding of miles PR #3608 (What / Padding).
 * Row t holds row_len[t] valid scores scores[t*ld_scores + 0 .. len-1].
 * Output row t: the min(len, k) positions with the highest scores, then -1
 * up to k.  Ties: the lower position wins, so the selected SET is unique.
 * Order inside a row: positions ascending (deterministic).
 * -0.0 ties +0.0.  Scores must not be NaN (unchecked).
 *   index_base [T] int32 or NULL: added to every selected position
 *              (turns request-local positions into pool slots); -1 stays -1
 *   idx        int32 [T, k];  lens int32 [T] or NULL: min(row_len, k)
 *   max_len    host: an upper bound of row_len
 * Workspace: dsa_topk_workspace_size(T, max_len, k) bytes, 256-byte aligned.
 */
size_t dsa_topk_workspace_size(int T, int64_t max_len, int k);
int dsa_topk(const float *scores, int64_t ld_scores, const int32_t *row_len, int T,
             int64_t max_len, int k, const int32_t *index_base,
             int32_t *idx, int32_t *lens, void *ws, size_t ws_bytes,
             int32_t *err_flag, dsa_stream_t stream);

/*
 * dsa_topk_noalloc -- dsa_topk for callers that cannot allocate device memory.
 * No passage of the DSA pages has a counterpart: this is a service of this
 * library.  Some callers cannot call cudaMalloc or reach an allocator -- for
 * example a plugin whose host framework hands it only its input and output
 * buffers, or code on a latency-critical path where an allocation (which may
 * synchronise the device) is not allowed.  This entry point takes the same
 * arguments as dsa_topk minus the workspace and produces the same result; its
 * scratch memory is a static device array of DSA_TOPK_NOALLOC_SCRATCH_BYTES
 * (4 MiB) that every GPU loading the library holds until the process exits.
 * Limit: the scratch of T rows must fit, i.e. dsa_topk_workspace_size(T,
 * max_len, k) <= 4 MiB (about 80 KiB a row: up to 50 rows of 128K scores);
 * larger calls return DSA_ERR_UNSUPPORTED without launching anything.
 * The first call on a device looks up the array's device address (with that
 * device current), so make that first call before any stream capture.  The
 * address is kept for the life of the process: after cudaDeviceReset the
 * module may be loaded again elsewhere, so do not call this function on a
 * device that was reset.
 * All calls share the array and it keeps the last call's contents; each call
 * clears what must start at zero.  Calls whose work overlaps on the GPU race
 * on the array: serialise them.  The function allocates nothing.
 */
#define DSA_TOPK_NOALLOC_SCRATCH_BYTES (4u << 20)
int dsa_topk_noalloc(const float *scores, int64_t ld_scores, const int32_t *row_len, int T,
                     int64_t max_len, int k, const int32_t *index_base,
                     int32_t *idx, int32_t *lens, int32_t *err_flag, dsa_stream_t stream);

/*
 * dsa_sparse_mla_fwd -- absorbed-MLA attention over selected latent rows.
 * The "sparse attn" stage of tokenspeed PR #627; semantics of miles PR #3608
 * (FlashMLA-style forward: natural-log lse; -1 masked) and the pool formats
 * and two-loop (main + extra list) layout of aiter PR #4382.
 * For each token t and head h:
 *   s_j = softmax_scale * q[t,h,0:D] . K_j   over valid entries j of idx[t,:]
 *         (slots into kv) and of idx_extra[t,:] (slots into kv_extra)
 *   out[t,h,0:Dv] = sum_j softmax(s)_j * K_j[0:Dv],  lse[t,h] = ln sum_j exp(s_j)
 * K_j is the dequantised row, D = d_nope + d_rope of the pool.  A token with
 * no valid entry gets out = 0 and lse = -inf.
 *   q        bf16 [T, H, D]
 *   idx      int32 [T, k] (-1 masked); kv_extra / idx_extra [T, k2] optional
 *            (both NULL with k2 = 0); kv_extra must have kv's D
 *   out      bf16 [T, H, Dv];  lse fp32 [T, H]
 * Limits: D = 576 with Dv = 512 (bf16 pool) or D = 512 with Dv = 448 (fp8
 * pools); 1 <= H <= 128; k + k2 >= 1; q and out 16-byte aligned;
 * softmax_scale positive and finite.  Anything else returns
 * DSA_ERR_INVALID_ARG or DSA_ERR_UNSUPPORTED before any launch.
 * Workspace: dsa_sparse_mla_workspace_size(T, H, Dv, k, k2) bytes.
 */
size_t dsa_sparse_mla_workspace_size(int T, int H, int Dv, int k, int k2);
int dsa_sparse_mla_fwd(const void *q, int T, int H, int D, int Dv, float softmax_scale,
                       const dsa_kv_pool *kv, const int32_t *idx, int k,
                       const dsa_kv_pool *kv_extra, const int32_t *idx_extra, int k2,
                       void *out, float *lse, void *ws, size_t ws_bytes,
                       int32_t *err_flag, dsa_stream_t stream);

/*
 * Attention and step options (dsa_sparse_mla_fwd_ex, dsa_sparse_mla_bwd,
 * dsa_decode_ex, dsa_decode_paged; NULL: none).
 *   sinks     device fp32 [H] or NULL: per-head sink logits.  A sink is one
 *             more logit in every softmax denominator of its head, in the
 *             units of the scores s_j = softmax_scale * q . K_j, with no
 *             value (the "sink folded in" of the Miles sparse-attention
 *             notes):  out = sum_j e^{s_j} K_j[0:Dv] / (sum_j e^{s_j} +
 *             e^{sink}),  lse = ln(sum_j e^{s_j} + e^{sink}).  A token with
 *             no valid entry then gets out = 0 and lse = sink.
 *   lse_log2  nonzero: lse is reported in log2 units (the natural-log lse
 *             divided by ln 2), the form those notes hand to the backward.
 *   rows_per_request  dsa_decode_ex only (0 elsewhere, else
 *             DSA_ERR_INVALID_ARG).  0 or 1: every row is its own request.
 *             2: rows 2r and 2r+1 are two new tokens of one request (a
 *             multi-token decode: speculative verification), so they share
 *             their context start (slot_base[2r] == slot_base[2r+1]) and
 *             their index scores are computed together, each key tile read
 *             once for both rows.  Results are the same bit for bit as
 *             with 0.  Needs an even B, H_I <= 64 and an fp8 indexer with
 *             d_idx = 128 or a bf16 one with d_idx = 64 (else
 *             DSA_ERR_UNSUPPORTED); a pair whose starts differ is reported
 *             (DSA_DEVERR_INDEX_RANGE) and its scores are not computed.
 *             Other values: DSA_ERR_UNSUPPORTED.
 */
typedef struct dsa_attn_opts {
  const float *sinks;
  int32_t lse_log2;
  int32_t rows_per_request;
} dsa_attn_opts;

/* dsa_sparse_mla_fwd with attention options (opts may be NULL). */
int dsa_sparse_mla_fwd_ex(const void *q, int T, int H, int D, int Dv, float softmax_scale,
                          const dsa_kv_pool *kv, const int32_t *idx, int k,
                          const dsa_kv_pool *kv_extra, const int32_t *idx_extra, int k2,
                          void *out, float *lse, void *ws, size_t ws_bytes,
                          int32_t *err_flag, const dsa_attn_opts *opts, dsa_stream_t stream);

/*
 * dsa_sparse_mla_bwd -- backward of dsa_sparse_mla_fwd(_ex) for training
 * (the "fwd + bwd per layer" workload of the Miles pull request #3608):
 * the gradient of its definition given dL/dout, the lse being an auxiliary
 * output that takes no gradient.  With p_j = e^{s_j - lse}:
 *   delta = sum_j p_j (dout . V_j);   dS_j = p_j (dout . V_j - delta)
 *   dq = scale sum_j dS_j K_j;   dK_j = scale sum_h dS_hj q_h, plus
 *   sum_h p_hj dout_h on its V columns;   dsink_h = -e^{sink_h - lse} delta
 * Each selected row's gradient (its K part plus its V part: the row serves as
 * both) is ADDED into dkv at the row's slot, once per selection.
 *   q, kv, idx, k, softmax_scale: as in the forward (bf16 pool, D = 576,
 *            Dv = 512, one list); lse fp32 [T, H] as the forward returned it
 *            with the same opts (sinks folded in; log2 units if lse_log2)
 *   dout     bf16 [T, H, Dv]
 *   dq       fp32 [T, H, D], written
 *   dkv      fp32 [kv->rows, D], accumulated (the caller zeroes it first)
 *   dsinks   fp32 [H], accumulated, or NULL (used with opts->sinks)
 * A SIMT kernel (no tensor cores): correct first, not yet fast.
 */
int dsa_sparse_mla_bwd(const void *q, int T, int H, int D, int Dv, float softmax_scale,
                       const dsa_kv_pool *kv, const int32_t *idx, int k,
                       const float *lse, const void *dout, const dsa_attn_opts *opts,
                       float *dq, float *dkv, float *dsinks,
                       int32_t *err_flag, dsa_stream_t stream);

/*
 * dsa_decode -- one fused decode step: score -> top-k -> sparse MLA for B
 * requests with one query token each (tokenspeed PR #627, Decode table:
 * "scores + TopK + sparse attn = total").
 * Request b sees context positions 0 .. seq_lens[b]-1; position j lives at
 * slot slot_base[b] + j of BOTH the index-k cache and the KV pool kv.
 *   indexer:  q_idx [B, H_I, d_idx], q_scale [B, H_I] (fp8) , k_idx / k_scale
 *             [k_rows, ...], w [B, H_I]   (as dsa_index_score)
 *   top-k:    k <= DSA_MAX_TOPK; max_seq_len (host) >= every seq_lens[b]
 *   attention: q bf16 [B, H, D], kv the pool the top-k indexes; optional
 *             second list kv_swa / idx_swa [B, k_swa] (e.g. a sliding
 *             window held in its own cache) in the same softmax
 *   idx_out   int32 [B, k] or NULL: the selected pool slots, -1 padded
 *   out bf16 [B, H, Dv], lse fp32 [B, H]
 * Workspace: dsa_decode_workspace_size(...) bytes.
 */
size_t dsa_decode_workspace_size(int B, int64_t max_seq_len, int k, int H, int Dv, int k_swa);
int dsa_decode(const void *q_idx, int idx_dtype, const float *q_scale,
               const void *k_idx, const float *k_scale, int64_t k_rows,
               const float *w, int H_I, int d_idx,
               int B, const int32_t *seq_lens, const int32_t *slot_base,
               int64_t max_seq_len, int k,
               const void *q, int H, int D, int Dv, float softmax_scale,
               const dsa_kv_pool *kv,
               const dsa_kv_pool *kv_swa, const int32_t *idx_swa, int k_swa,
               int32_t *idx_out, void *out, float *lse,
               void *ws, size_t ws_bytes, int32_t *err_flag, dsa_stream_t stream);

/* dsa_decode with attention options (opts may be NULL). */
int dsa_decode_ex(const void *q_idx, int idx_dtype, const float *q_scale,
                  const void *k_idx, const float *k_scale, int64_t k_rows,
                  const float *w, int H_I, int d_idx,
                  int B, const int32_t *seq_lens, const int32_t *slot_base,
                  int64_t max_seq_len, int k,
                  const void *q, int H, int D, int Dv, float softmax_scale,
                  const dsa_kv_pool *kv,
                  const dsa_kv_pool *kv_swa, const int32_t *idx_swa, int k_swa,
                  int32_t *idx_out, void *out, float *lse,
                  void *ws, size_t ws_bytes, int32_t *err_flag,
                  const dsa_attn_opts *opts, dsa_stream_t stream);

/*
 * dsa_decode_paged -- dsa_decode on paged caches (the block-table layout of
 * the tokenspeed PR #627 serving stack: pages of page_size slots).  Position
 * j of request b lives at slot
 *     block_table[b * max_pages + j / page_size] * page_size + j % page_size
 * of BOTH the index-k cache (k_idx / k_scale rows) and the KV pool kv; the
 * selection (idx_out) holds those slots.  page_size a multiple of 64;
 * max_pages * page_size >= max_seq_len; block_table int32 [B, max_pages] on
 * the device, entries for positions past seq_lens[b] unused.  A slot outside
 * the pool is reported (DSA_DEVERR_INDEX_RANGE) and masked by the attention;
 * index-k rows outside the cache read as zeros.  Everything else as
 * dsa_decode_ex (opts may be NULL); workspace dsa_decode_workspace_size(...).
 */
int dsa_decode_paged(const void *q_idx, int idx_dtype, const float *q_scale,
                     const void *k_idx, const float *k_scale, int64_t k_rows,
                     const float *w, int H_I, int d_idx,
                     int B, const int32_t *seq_lens,
                     const int32_t *block_table, int max_pages, int page_size,
                     int64_t max_seq_len, int k,
                     const void *q, int H, int D, int Dv, float softmax_scale,
                     const dsa_kv_pool *kv,
                     const dsa_kv_pool *kv_swa, const int32_t *idx_swa, int k_swa,
                     int32_t *idx_out, void *out, float *lse,
                     void *ws, size_t ws_bytes, int32_t *err_flag,
                     const dsa_attn_opts *opts, dsa_stream_t stream);

/*
 * dsa_decode_host -- dsa_decode with the step's inputs and outputs in HOST
 * memory; the model state (index-k cache k_idx / k_scale, the KV pools) stays
 * in device memory.  The same computation and kernels as dsa_decode, with
 * the copies enqueued around them on `stream`: h_q, h_idx_swa, h_seq_lens,
 * h_slot_base, h_q_idx, h_w, h_q_scale into the workspace, then the step,
 * then h_idx_out (optional), h_out and h_lse back.
 * Host pointers (h_*) are read and written by the copies when `stream` gets
 * there: they must stay valid until then, as with cudaMemcpyAsync.  When
 * every given host buffer is page-locked (pinned, so the GPU reaches it at
 * its device-mapped address) and 16-byte aligned, two kernels move the data
 * (one gathers the inputs, one writes the selection back), which avoids the
 * fixed cost of ten copy-engine transfers.  Whenever h_out and h_lse are
 * pinned and 16-byte aligned, the step's last kernel writes them itself at
 * their device-mapped addresses (no copy back for those two).  Otherwise
 * each buffer is copied with cudaMemcpyAsync; pageable memory is accepted
 * and the CUDA runtime then stages those copies itself.  All give the same
 * results bit for bit.
 * Shapes, types and limits are those of dsa_decode.  err_flag, if given, is
 * a device pointer.  No host synchronisation: the outputs are in host memory
 * once `stream` has passed this call (e.g. after cudaStreamSynchronize).
 * Workspace: dsa_decode_host_workspace_size(...) bytes of device memory (the
 * decode workspace plus device copies of the inputs and outputs); calls on
 * the same stream may share it, a call on another stream may not until this
 * one has completed.
 * Returns a status as dsa_decode.
 */
size_t dsa_decode_host_workspace_size(int B, int64_t max_seq_len, int k, int H_I, int d_idx,
                                      int idx_dtype, int H, int D, int Dv, int k_swa);
int dsa_decode_host(const void *h_q_idx, int idx_dtype, const float *h_q_scale,
                    const void *k_idx, const float *k_scale, int64_t k_rows,
                    const float *h_w, int H_I, int d_idx,
                    int B, const int32_t *h_seq_lens, const int32_t *h_slot_base,
                    int64_t max_seq_len, int k,
                    const void *h_q, int H, int D, int Dv, float softmax_scale,
                    const dsa_kv_pool *kv,
                    const dsa_kv_pool *kv_swa, const int32_t *h_idx_swa, int k_swa,
                    int32_t *h_idx_out, void *h_out, float *h_lse,
                    void *ws, size_t ws_bytes, int32_t *err_flag, dsa_stream_t stream);

/*
 * dsa_decode_graph -- the host-buffer decode step (dsa_decode_host) captured
 * once into a CUDA graph and replayed step after step.  No passage of the
 * DSA pages has a counterpart: this is a service of this library for decode
 * loops, where one graph launch replaces the call's ten copies and five
 * kernel launches.
 * dsa_decode_graph_create takes the arguments of dsa_decode_host (no stream:
 * it captures on a stream of its own) and binds every pointer: the graph
 * copies from and to the SAME host buffers, reads the same caches and pools
 * and uses the same workspace at every launch.  Between launches the caller
 * rewrites the inputs in place (h_q, h_q_idx, h_q_scale, h_w, h_seq_lens,
 * h_slot_base, h_idx_swa; the caches and pools on the device) and reads the
 * outputs (h_idx_out, h_out, h_lse) once the launch has completed on its
 * stream.  B, max_seq_len, k and the shapes are fixed at creation; host
 * buffers must be page-locked (pinned); max_seq_len must bound every later
 * seq_lens.  The host checks of dsa_decode_host run once, at creation.
 *   *graph     receives the handle (NULL on error); it owns a CUDA graph,
 *              not device memory
 * dsa_decode_graph_launch enqueues one step on `stream` (a launch on another
 * stream may not overlap one in flight: they share the workspace and the host
 * buffers).  dsa_decode_graph_destroy frees the handle (NULL is accepted);
 * no launch of it may be in flight.
 * Returns a status as dsa_decode; DSA_ERR_CUDA if the capture or the
 * instantiation fails.
 */
typedef struct dsa_decode_graph_s *dsa_decode_graph;
int dsa_decode_graph_create(const void *h_q_idx, int idx_dtype, const float *h_q_scale,
                            const void *k_idx, const float *k_scale, int64_t k_rows,
                            const float *h_w, int H_I, int d_idx,
                            int B, const int32_t *h_seq_lens, const int32_t *h_slot_base,
                            int64_t max_seq_len, int k,
                            const void *h_q, int H, int D, int Dv, float softmax_scale,
                            const dsa_kv_pool *kv,
                            const dsa_kv_pool *kv_swa, const int32_t *h_idx_swa, int k_swa,
                            int32_t *h_idx_out, void *h_out, float *h_lse,
                            void *ws, size_t ws_bytes, int32_t *err_flag,
                            dsa_decode_graph *graph);
int dsa_decode_graph_launch(dsa_decode_graph graph, dsa_stream_t stream);
void dsa_decode_graph_destroy(dsa_decode_graph graph);

/*
 * dsa_selftest_wait_timeout -- a diagnostic of the failure detection: one
 * GPU thread waits, through the same bounded wait every kernel here uses, on
 * a barrier phase that nothing completes.  The wait gives up after its
 * limit (about a second), ORs DSA_DEVERR_TIMEOUT into *err_flag and the
 * kernel returns; the context stays usable.
 *   err_flag  device int32
 *   out       device int64 [3]: 1 if the wait completed (never), the cycles
 *             waited, the limit in cycles
 */
int dsa_selftest_wait_timeout(int32_t *err_flag, long long *out, dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H */
