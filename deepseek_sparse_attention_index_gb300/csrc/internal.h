// Internal launchers shared by the C-ABI layer (dsa_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsa.h"

namespace dsa {

// A row's positions -> pool slots through a block table (paged caches).
struct PageMap {
  const int32_t *table;   // [rows][max_pages], or NULL (not paged)
  int max_pages;
  int page_size;
};

// ------------------------------------------------------------------ top-k
constexpr int kHistBins = 4096;   // first radix level: top 12 bits of the key
constexpr int kListCap = 8192;    // (key, position) entries per row kept for the resolve pass
constexpr int kMinChunk = 2048;   // smallest run of positions one collect CTA covers

struct TopkWs {
  uint32_t *hist;    // [T][kHistBins]        zeroed before the histogram pass
  uint32_t *cnt;     // [T][4]: list entries, -, then one u64 (entries | CTAs done << 32); zeroed before the collect pass
  uint2 *list;       // [T][kListCap]  (key, position): the row's runs, one per collect CTA
  uint2 *tab;        // [T][max_chunks] (run start, run length) by chunk
  int max_chunks;    // ceil(max_len / kMinChunk)
};
size_t topk_ws_layout(int T, int64_t max_len, int k, void *ws, TopkWs *out);  // returns bytes

// Clears hist and cnt (one small kernel, stream-ordered).
cudaError_t topk_clear(const TopkWs &w, int T, cudaStream_t s);
// Histogram pass over a score matrix (the standalone entry point; the fused
// decode builds the histogram in the index-score epilogue instead).
cudaError_t topk_hist(const float *scores, int64_t ld, const int32_t *row_len, int T,
                      int64_t max_len, int k, const TopkWs &w, cudaStream_t s);
cudaError_t topk_select(const float *scores, int64_t ld, const int32_t *row_len, int T,
                        int64_t max_len, int k, const int32_t *index_base, int32_t *idx,
                        int32_t *lens, const TopkWs &w, int32_t *err_flag, cudaStream_t s,
                        const PageMap &pages = PageMap{});

// ------------------------------------------------------------------ index score
struct IndexScoreArgs {
  const void *q_idx;
  int idx_dtype;
  const float *q_scale;
  const void *k_idx;
  const float *k_scale;
  int64_t k_rows;
  const float *w;
  const int32_t *row_start;  // [T] (or NULL when slot_base/seq_lens are used)
  const int32_t *row_end;    // [T]
  const int32_t *slot_base;  // decode form: rows [slot_base[t], slot_base[t]+seq_lens[t])
  const int32_t *seq_lens;
  int T, H_I, d;
  int64_t max_len;
  float *scores;
  int64_t ld_scores;
  uint32_t *hist;            // optional [T][kHistBins]: fused top-k histogram
  int topk_k;                // rows of length <= topk_k skip the histogram
  int inputs_ready;          // the inputs were complete before the previous kernel on the
                             // stream began (fused decode: only the histogram's zeroing
                             // precedes us); else the kernel waits for it first
  int32_t *err_flag;
  // paged caches (decode form, with seq_lens): position j of row t lives at
  // slot block_table[t * max_pages + j / page_size] * page_size + j % page_size
  const int32_t *block_table;  // or NULL
  int max_pages;
  int page_size;               // a multiple of 64
  // 2: rows 2g and 2g + 1 share their keys (a request's two new tokens in a
  // multi-token decode) and are scored together, each key tile read once;
  // 0 or 1: every row on its own
  int rows_per_unit;
};
cudaError_t index_score_launch(const IndexScoreArgs &a, cudaStream_t s);
// The prefill form (row ranges, no histogram): groups of four consecutive
// rows share each key tile where they start at the same key
// (index_score_groups.cu); shapes it does not take go to index_score_launch.
cudaError_t index_score_prefill_launch(const IndexScoreArgs &a, cudaStream_t s);


// ------------------------------------------------------------------ sparse MLA
struct PoolDev {
  const uint8_t *data;
  const float *scales;
  int64_t rows;
  int format;
  int block;
};

struct MlaArgs {
  const void *q;             // bf16 [T, H, D]
  int T, H, D, Dv;
  float softmax_scale;
  PoolDev kv, kv2;
  const int32_t *idx;        // [T, k]
  int k;
  const int32_t *idx2;       // [T, k2] or NULL
  int k2;
  void *out;                 // bf16 [T, H, Dv]
  float *lse;                // [T, H]
  float *part_o;             // workspace partials
  float *part_lse;
  int n_splits;
  int32_t *err_flag;
  int q_ready;               // q was complete before the previous kernel on the stream
                             // began (fused decode): the kernel may load it before pdl_wait
  const float *sinks;        // [H] per-head sink logits (natural-log units) or NULL
  int lse_log2;              // the final lse in log2 units
};
// backward of the sparse attention (bf16 pool, D = 576, Dv = 512, one list)
struct MlaBwdArgs {
  const void *q;             // bf16 [T, H, 576]
  int T, H;
  float softmax_scale;
  PoolDev kv;
  const int32_t *idx;        // [T, k] slots, -1 masked
  int k;
  const float *lse;          // [T, H] from the forward (natural log, or log2 when lse_log2)
  int lse_log2;
  const void *dout;          // bf16 [T, H, 512]
  const float *sinks;        // [H] or NULL
  float *dsinks;             // [H] accumulated, or NULL
  float *dq;                 // [T, H, 576] written
  float *dkv;                // [pool rows, 576] accumulated
  int32_t *err_flag;
};
cudaError_t sparse_mla_bwd_launch(const MlaBwdArgs &a, cudaStream_t s);

int mla_num_splits(int T, int H, int k_total);
size_t mla_ws_bytes(int T, int H, int Dv, int k_total);
void mla_ws_layout(int T, int H, int Dv, int k_total, void *ws, float **part_o, float **part_lse);
cudaError_t sparse_mla_launch(const MlaArgs &a, cudaStream_t s);
// tcgen05 kernels (sparse_mla_tc.cu): the format code of a call they serve
// (bf16 pool, D = 576; uniform or packed fp8 pools, D = 512), or -1 for a call
// the SIMT kernel takes; then the launch for that code.
int sparse_mla_tc_format(const MlaArgs &a);
cudaError_t sparse_mla_tc_launch(const MlaArgs &a, int fmt, cudaStream_t s);

}  // namespace dsa
