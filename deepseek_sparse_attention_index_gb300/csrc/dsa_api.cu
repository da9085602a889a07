// C ABI of the DSA forward hot path (declarations and contracts: include/dsa.h).
// Host side only: argument checks, workspace carving and stream-ordered
// launches of the kernels in index_score.cu, topk.cu and sparse_mla.cu.
#include <stdint.h>
#include <new>
#include <string.h>

#include "common.cuh"
#include "internal.h"

using namespace dsa;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_kv(const dsa_kv_pool *kv, int D) {
  if (!kv || !kv->data || kv->rows < 0) return DSA_ERR_INVALID_ARG;
  if (!aligned16(kv->data)) return DSA_ERR_INVALID_ARG;
  if (kv->d_nope + kv->d_rope != D || kv->d_rope != 64) return DSA_ERR_UNSUPPORTED;
  switch (kv->format) {
    case DSA_KV_BF16:
      if (D != 576) return DSA_ERR_UNSUPPORTED;
      return DSA_OK;
    case DSA_KV_FP8_UNIFORM:
      if (D != 512) return DSA_ERR_UNSUPPORTED;
      if (!kv->scales) return DSA_ERR_INVALID_ARG;
      return DSA_OK;
    case DSA_KV_FP8_DS_MLA:
      if (D != 512 || kv->d_nope != 448) return DSA_ERR_UNSUPPORTED;
      if (kv->block <= 0 || (kv->block & 1)) return DSA_ERR_UNSUPPORTED;
      if (kv->rows % kv->block) return DSA_ERR_INVALID_ARG;
      return DSA_OK;
    default:
      return DSA_ERR_UNSUPPORTED;
  }
}

PoolDev to_dev(const dsa_kv_pool *kv) {
  PoolDev p{};
  if (!kv) return p;
  p.data = static_cast<const uint8_t *>(kv->data);
  p.scales = kv->scales;
  p.rows = kv->rows;
  p.format = kv->format;
  p.block = kv->block > 0 ? kv->block : 1;
  return p;
}

int check_indexer(const void *q_idx, int idx_dtype, const float *q_scale, const void *k_idx,
                  const float *k_scale, int64_t k_rows, const float *w, int T, int H_I, int d) {
  if (T < 0 || k_rows < 0) return DSA_ERR_INVALID_ARG;
  // key rows are tensor-map coordinates (32-bit signed) in the kernel
  if (k_rows > INT32_MAX || (int64_t)T * H_I > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if (T > 0 && (!q_idx || !k_idx || !w)) return DSA_ERR_INVALID_ARG;
  if (H_I < 1 || H_I > DSA_MAX_INDEX_HEADS || (H_I % 8)) return DSA_ERR_UNSUPPORTED;
  if (idx_dtype == DSA_IDX_FP8_E4M3) {
    if (d != 128) return DSA_ERR_UNSUPPORTED;
    if (T > 0 && (!q_scale || !k_scale)) return DSA_ERR_INVALID_ARG;
  } else if (idx_dtype == DSA_IDX_BF16) {
    if (d != 64 && d != 128) return DSA_ERR_UNSUPPORTED;
  } else {
    return DSA_ERR_UNSUPPORTED;
  }
  if (!aligned16(k_idx) || !aligned16(q_idx)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

int check_mla_shape(const void *q, int T, int H, int D, int Dv, float softmax_scale,
                    const dsa_kv_pool *kv, const int32_t *idx, int k, const dsa_kv_pool *kv2,
                    const int32_t *idx2, int k2, const void *out, const float *lse,
                    bool need_idx = true) {
  if (T < 0 || k < 0 || k2 < 0) return DSA_ERR_INVALID_ARG;
  // the softmax keeps its running maximum of the raw products q . K, which
  // is the maximum of the scores only for a positive scale
  if (!(softmax_scale > 0.f) || !(softmax_scale <= 3.4e38f)) return DSA_ERR_INVALID_ARG;
  if (H < 1 || H > DSA_MAX_HEADS) return DSA_ERR_UNSUPPORTED;
  if (!((D == 576 && Dv == 512) || (D == 512 && Dv == 448))) return DSA_ERR_UNSUPPORTED;
  if (k + k2 < 1) return DSA_ERR_INVALID_ARG;
  if (T > 0 && (!q || !out || !lse)) return DSA_ERR_INVALID_ARG;
  if (need_idx && k > 0 && T > 0 && !idx) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
  int st = check_kv(kv, D);
  if (st != DSA_OK) return st;
  if (k2 > 0) {
    if (!idx2) return DSA_ERR_INVALID_ARG;
    st = check_kv(kv2, D);
    if (st != DSA_OK) return st;
  }
  return DSA_OK;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

int64_t scores_ld(int64_t max_len) { return (max_len + 3) & ~int64_t(3); }

struct DecodeLayout {
  float *scores;
  TopkWs topk;
  int32_t *idx;
  float *part_o, *part_lse;
  size_t bytes;
};

DecodeLayout decode_layout(int B, int64_t max_seq_len, int k, int H, int Dv, int k_swa,
                           void *ws) {
  DecodeLayout L{};
  WsCarver c(ws);
  L.scores = c.take<float>((size_t)B * scores_ld(max_seq_len));
  size_t tb = topk_ws_layout(B, max_seq_len, k, nullptr, nullptr);
  char *tp = c.take<char>(tb);
  topk_ws_layout(B, max_seq_len, k, tp, &L.topk);
  L.idx = c.take<int32_t>((size_t)B * k);
  size_t mb = mla_ws_bytes(B, H, Dv, k + k_swa);
  char *mp = c.take<char>(mb);
  if (ws) mla_ws_layout(B, H, Dv, k + k_swa, mp, &L.part_o, &L.part_lse);
  L.bytes = c.bytes();
  return L;
}

// Enqueues one checked fused decode step on s.
int decode_enqueue(const void *q_idx, int idx_dtype, const float *q_scale, const void *k_idx,
                   const float *k_scale, int64_t k_rows, const float *w, int H_I, int d_idx, int B,
                   const int32_t *seq_lens, const int32_t *slot_base, int64_t max_seq_len, int k,
                   const void *q, int H, int D, int Dv, float softmax_scale, const dsa_kv_pool *kv,
                   const dsa_kv_pool *kv_swa, const int32_t *idx_swa, int k_swa, int32_t *idx_out,
                   void *out, float *lse, void *ws, int32_t *err_flag, cudaStream_t s,
                   const dsa_attn_opts *opts = nullptr, const PageMap &pages = PageMap{}) {
  DecodeLayout L = decode_layout(B, max_seq_len, k, H, Dv, k_swa, ws);
  const int64_t ld = scores_ld(max_seq_len);
  int32_t *idx = idx_out ? idx_out : L.idx;

  cudaError_t e = topk_clear(L.topk, B, s);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  IndexScoreArgs ia{};
  ia.q_idx = q_idx; ia.idx_dtype = idx_dtype; ia.q_scale = q_scale;
  ia.k_idx = k_idx; ia.k_scale = k_scale; ia.k_rows = k_rows; ia.w = w;
  ia.slot_base = pages.table ? nullptr : slot_base; ia.seq_lens = seq_lens;
  ia.block_table = pages.table; ia.max_pages = pages.max_pages; ia.page_size = pages.page_size;
  ia.T = B; ia.H_I = H_I; ia.d = d_idx; ia.max_len = max_seq_len;
  ia.scores = L.scores; ia.ld_scores = ld; ia.hist = L.topk.hist; ia.topk_k = k;
  ia.inputs_ready = 1;   // the inputs precede the whole call; only the zeroing precedes us
  ia.err_flag = err_flag;
  ia.rows_per_unit = opts && opts->rows_per_request == 2 && !pages.table ? 2 : 1;
  e = index_score_launch(ia, s);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  e = topk_select(L.scores, ld, seq_lens, B, max_seq_len, k, pages.table ? nullptr : slot_base,
                  idx, nullptr, L.topk, err_flag, s, pages);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  MlaArgs a{};
  a.q = q; a.T = B; a.H = H; a.D = D; a.Dv = Dv; a.softmax_scale = softmax_scale;
  a.q_ready = 1;   // q precedes the whole fused call on the stream
  a.kv = to_dev(kv); a.idx = idx; a.k = k;
  a.kv2 = to_dev(k_swa > 0 ? kv_swa : nullptr); a.idx2 = k_swa > 0 ? idx_swa : nullptr;
  a.k2 = k_swa;
  a.out = out; a.lse = lse; a.err_flag = err_flag;
  a.sinks = opts ? opts->sinks : nullptr;
  a.lse_log2 = opts ? opts->lse_log2 != 0 : 0;
  a.n_splits = mla_num_splits(B, H, k + k_swa);
  a.part_o = L.part_o; a.part_lse = L.part_lse;
  return status_of(sparse_mla_launch(a, s));
}

// Device staging of dsa_decode_host: the decode workspace, then the step's
// inputs and outputs.
struct HostStaging {
  void *dec_ws;
  size_t dec_bytes;
  void *q_idx;
  float *q_scale, *w;
  int32_t *seq_lens, *slot_base;
  void *q;
  int32_t *idx_swa, *idx_out;
  void *out;
  float *lse;
  size_t bytes;
};

size_t idx_elem_bytes(int idx_dtype) { return idx_dtype == DSA_IDX_FP8_E4M3 ? 1 : 2; }

// ------------------------------------------------------------------ host I/O
// The step's host buffers moved by kernels instead of copy-engine transfers:
// with every host buffer pinned (so the GPU reaches it directly through its
// device-mapped address) and 16-byte aligned, one kernel gathers the step's
// inputs into the staging workspace and one writes the outputs back.  Each
// cudaMemcpyAsync costs a few microseconds of fixed copy-engine time; the
// ten of a step added ~60 us to a 155 us step.  Any other buffer keeps the
// copies.
constexpr int kMaxSegs = 8;
struct CopySegs {
  const uint4 *src[kMaxSegs];
  uint4 *dst[kMaxSegs];
  uint32_t n16[kMaxSegs];   // whole 16-byte units of segment i
  uint32_t tail[kMaxSegs];  // then this many bytes (< 16)
  int n;
};

__global__ void __launch_bounds__(256) copy_segments_kernel(const CopySegs c) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (int i = 0; i < c.n; ++i) {
    const uint4 *src = c.src[i];
    uint4 *dst = c.dst[i];
    const uint32_t n = c.n16[i];
    uint32_t j = blockIdx.x * blockDim.x + threadIdx.x;
    // four loads in flight a thread, then their stores
    for (; j + 3 * stride < n; j += 4 * stride) {
      const uint4 a0 = src[j], a1 = src[j + stride], a2 = src[j + 2 * stride],
                  a3 = src[j + 3 * stride];
      dst[j] = a0;
      dst[j + stride] = a1;
      dst[j + 2 * stride] = a2;
      dst[j + 3 * stride] = a3;
    }
    for (; j < n; j += stride) dst[j] = src[j];
    if (blockIdx.x == 0 && threadIdx.x < c.tail[i]) {
      reinterpret_cast<unsigned char *>(dst + n)[threadIdx.x] =
          reinterpret_cast<const unsigned char *>(src + n)[threadIdx.x];
    }
  }
}

// The device address of pinned host memory at p (16-byte aligned), or
// nullptr when p is not pinned host memory or not aligned.
const void *mapped_host(const void *p) {
  if (!p || (reinterpret_cast<uintptr_t>(p) & 15)) return nullptr;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();   // a pageable pointer may set an error on older runtimes: clear it
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
  if ((reinterpret_cast<uintptr_t>(at.devicePointer) & 15) != 0) return nullptr;
  return at.devicePointer;
}

struct SegBuilder {
  CopySegs c{};
  bool ok = true;
  // a host -> device (h2d) or device -> host segment
  void add(const void *host, void *dev, size_t bytes, bool h2d) {
    if (!ok || bytes == 0) return;
    const void *m = mapped_host(host);
    if (!m || c.n == kMaxSegs || bytes / 16 > 0xffffffffu || (reinterpret_cast<uintptr_t>(dev) & 15)) {
      ok = false;
      return;
    }
    c.src[c.n] = static_cast<const uint4 *>(h2d ? m : dev);
    c.dst[c.n] = static_cast<uint4 *>(h2d ? dev : const_cast<void *>(m));
    c.n16[c.n] = (uint32_t)(bytes / 16);
    c.tail[c.n] = (uint32_t)(bytes & 15);
    ++c.n;
  }
  cudaError_t launch(cudaStream_t s) const {
    if (c.n == 0) return cudaSuccess;
    copy_segments_kernel<<<2 * num_sms(), 256, 0, s>>>(c);
    return cudaGetLastError();
  }
};

HostStaging host_staging(int B, int64_t max_seq_len, int k, int H_I, int d_idx, int idx_dtype,
                         int H, int D, int Dv, int k_swa, void *ws) {
  HostStaging S{};
  WsCarver c(ws);
  S.dec_bytes = decode_layout(B, max_seq_len, k, H, Dv, k_swa, nullptr).bytes;
  S.dec_ws = c.take<char>(S.dec_bytes);
  S.q_idx = c.take<char>((size_t)B * H_I * d_idx * idx_elem_bytes(idx_dtype));
  S.q_scale = c.take<float>((size_t)B * H_I);
  S.w = c.take<float>((size_t)B * H_I);
  S.seq_lens = c.take<int32_t>((size_t)B);
  S.slot_base = c.take<int32_t>((size_t)B);
  S.q = c.take<char>((size_t)B * H * D * 2);
  S.idx_swa = c.take<int32_t>((size_t)B * k_swa);
  S.idx_out = c.take<int32_t>((size_t)B * k);
  S.out = c.take<char>((size_t)B * H * Dv * 2);
  S.lse = c.take<float>((size_t)B * H);
  S.bytes = c.bytes();
  return S;
}

// dsa_index_score and dsa_index_score_prefill: the checks and the argument
// block are the same; `groups` picks the kernel
int index_score_entry(const void *q_idx, int idx_dtype, const float *q_scale, const void *k_idx,
                      const float *k_scale, int64_t k_rows, const float *w,
                      const int32_t *row_start, const int32_t *row_end, int T, int H_I, int d,
                      int64_t max_len, float *scores, int64_t ld_scores, int32_t *err_flag,
                      dsa_stream_t stream, bool groups) {
  int st = check_indexer(q_idx, idx_dtype, q_scale, k_idx, k_scale, k_rows, w, T, H_I, d);
  if (st != DSA_OK) return st;
  if (max_len < 0 || ld_scores < max_len) return DSA_ERR_INVALID_ARG;
  if (T > 0 && (!row_start || !row_end || !scores)) return DSA_ERR_INVALID_ARG;
  IndexScoreArgs a{};
  a.q_idx = q_idx; a.idx_dtype = idx_dtype; a.q_scale = q_scale;
  a.k_idx = k_idx; a.k_scale = k_scale; a.k_rows = k_rows; a.w = w;
  a.row_start = row_start; a.row_end = row_end;
  a.T = T; a.H_I = H_I; a.d = d; a.max_len = max_len;
  a.scores = scores; a.ld_scores = ld_scores; a.err_flag = err_flag;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return status_of(groups ? index_score_prefill_launch(a, s) : index_score_launch(a, s));
}

}  // namespace

// A captured host-buffer decode step (dsa_decode_graph_create).
struct dsa_decode_graph_s {
  cudaGraphExec_t exec;
};

extern "C" {

const char *dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported shape or format";
    case DSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case DSA_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

int dsa_abi_version(void) { return 1; }

int dsa_index_score(const void *q_idx, int idx_dtype, const float *q_scale, const void *k_idx,
                    const float *k_scale, int64_t k_rows, const float *w,
                    const int32_t *row_start, const int32_t *row_end, int T, int H_I, int d,
                    int64_t max_len, float *scores, int64_t ld_scores, int32_t *err_flag,
                    dsa_stream_t stream) {
  return index_score_entry(q_idx, idx_dtype, q_scale, k_idx, k_scale, k_rows, w, row_start, row_end,
                           T, H_I, d, max_len, scores, ld_scores, err_flag, stream, false);
}

int dsa_index_score_prefill(const void *q_idx, int idx_dtype, const float *q_scale,
                            const void *k_idx, const float *k_scale, int64_t k_rows,
                            const float *w, const int32_t *row_start, const int32_t *row_end,
                            int T, int H_I, int d, int64_t max_len, float *scores,
                            int64_t ld_scores, int32_t *err_flag, dsa_stream_t stream) {
  return index_score_entry(q_idx, idx_dtype, q_scale, k_idx, k_scale, k_rows, w, row_start, row_end,
                           T, H_I, d, max_len, scores, ld_scores, err_flag, stream, true);
}

size_t dsa_topk_workspace_size(int T, int64_t max_len, int k) {
  if (T <= 0 || k <= 0 || max_len < 0) return 0;
  return topk_ws_layout(T, max_len, k, nullptr, nullptr);
}

int dsa_topk(const float *scores, int64_t ld_scores, const int32_t *row_len, int T,
             int64_t max_len, int k, const int32_t *index_base, int32_t *idx, int32_t *lens,
             void *ws, size_t ws_bytes, int32_t *err_flag, dsa_stream_t stream) {
  if (T < 0 || max_len < 0 || ld_scores < max_len) return DSA_ERR_INVALID_ARG;
  if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!scores || !row_len || !idx) return DSA_ERR_INVALID_ARG;
  const size_t need = dsa_topk_workspace_size(T, max_len, k);
  if (ws_bytes < need || (need && !ws)) return DSA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TopkWs w;
  topk_ws_layout(T, max_len, k, ws, &w);
  cudaError_t e = topk_clear(w, T, s);
  if (e == cudaSuccess) e = topk_hist(scores, ld_scores, row_len, T, max_len, k, w, s);
  if (e == cudaSuccess)
    e = topk_select(scores, ld_scores, row_len, T, max_len, k, index_base, idx, lens, w,
                    err_flag, s);
  return status_of(e);
}

size_t dsa_sparse_mla_workspace_size(int T, int H, int Dv, int k, int k2) {
  if (T <= 0 || H <= 0 || k + k2 <= 0) return 0;
  return mla_ws_bytes(T, H, Dv, k + k2);
}

int dsa_sparse_mla_fwd(const void *q, int T, int H, int D, int Dv, float softmax_scale,
                       const dsa_kv_pool *kv, const int32_t *idx, int k,
                       const dsa_kv_pool *kv_extra, const int32_t *idx_extra, int k2,
                       void *out, float *lse, void *ws, size_t ws_bytes, int32_t *err_flag,
                       dsa_stream_t stream) {
  return dsa_sparse_mla_fwd_ex(q, T, H, D, Dv, softmax_scale, kv, idx, k, kv_extra, idx_extra, k2,
                               out, lse, ws, ws_bytes, err_flag, nullptr, stream);
}

int dsa_sparse_mla_fwd_ex(const void *q, int T, int H, int D, int Dv, float softmax_scale,
                          const dsa_kv_pool *kv, const int32_t *idx, int k,
                          const dsa_kv_pool *kv_extra, const int32_t *idx_extra, int k2,
                          void *out, float *lse, void *ws, size_t ws_bytes, int32_t *err_flag,
                          const dsa_attn_opts *opts, dsa_stream_t stream) {
  if (opts && opts->rows_per_request != 0) return DSA_ERR_INVALID_ARG;
  int st = check_mla_shape(q, T, H, D, Dv, softmax_scale, kv, idx, k, kv_extra, idx_extra, k2, out, lse);
  if (st != DSA_OK) return st;
  if (T == 0) return DSA_OK;
  const size_t need = dsa_sparse_mla_workspace_size(T, H, Dv, k, k2);
  if (ws_bytes < need || (need && !ws)) return DSA_ERR_WORKSPACE_TOO_SMALL;
  MlaArgs a{};
  a.q = q; a.T = T; a.H = H; a.D = D; a.Dv = Dv; a.softmax_scale = softmax_scale;
  a.kv = to_dev(kv); a.idx = idx; a.k = k;
  a.kv2 = to_dev(k2 > 0 ? kv_extra : nullptr); a.idx2 = k2 > 0 ? idx_extra : nullptr; a.k2 = k2;
  a.out = out; a.lse = lse; a.err_flag = err_flag;
  a.sinks = opts ? opts->sinks : nullptr;
  a.lse_log2 = opts ? opts->lse_log2 != 0 : 0;
  a.n_splits = mla_num_splits(T, H, k + k2);
  if (a.n_splits > 1) mla_ws_layout(T, H, Dv, k + k2, ws, &a.part_o, &a.part_lse);
  return status_of(sparse_mla_launch(a, reinterpret_cast<cudaStream_t>(stream)));
}

int dsa_sparse_mla_bwd(const void *q, int T, int H, int D, int Dv, float softmax_scale,
                       const dsa_kv_pool *kv, const int32_t *idx, int k, const float *lse,
                       const void *dout, const dsa_attn_opts *opts, float *dq, float *dkv,
                       float *dsinks, int32_t *err_flag, dsa_stream_t stream) {
  if (opts && opts->rows_per_request != 0) return DSA_ERR_INVALID_ARG;
  if (T < 0 || k < 1) return DSA_ERR_INVALID_ARG;
  if (H < 1 || H > DSA_MAX_HEADS) return DSA_ERR_UNSUPPORTED;
  if (D != 576 || Dv != 512 || !kv || kv->format != DSA_KV_BF16) return DSA_ERR_UNSUPPORTED;
  if (!(softmax_scale > 0.f) || !(softmax_scale <= 3.4e38f)) return DSA_ERR_INVALID_ARG;
  int st = check_kv(kv, D);
  if (st != DSA_OK) return st;
  if (T == 0) return DSA_OK;
  if (!q || !idx || !lse || !dout || !dq || !dkv) return DSA_ERR_INVALID_ARG;
  if (!aligned16(kv->data) || !aligned16(q) || !aligned16(dout)) return DSA_ERR_INVALID_ARG;
  MlaBwdArgs a{};
  a.q = q; a.T = T; a.H = H; a.softmax_scale = softmax_scale;
  a.kv = to_dev(kv); a.idx = idx; a.k = k;
  a.lse = lse; a.lse_log2 = opts ? opts->lse_log2 != 0 : 0;
  a.dout = dout;
  a.sinks = opts ? opts->sinks : nullptr; a.dsinks = dsinks;
  a.dq = dq; a.dkv = dkv; a.err_flag = err_flag;
  return status_of(sparse_mla_bwd_launch(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t dsa_decode_workspace_size(int B, int64_t max_seq_len, int k, int H, int Dv, int k_swa) {
  if (B <= 0 || k <= 0 || H <= 0 || max_seq_len < 0 || k_swa < 0) return 0;
  return decode_layout(B, max_seq_len, k, H, Dv, k_swa, nullptr).bytes;
}

int dsa_decode(const void *q_idx, int idx_dtype, const float *q_scale, const void *k_idx,
               const float *k_scale, int64_t k_rows, const float *w, int H_I, int d_idx, int B,
               const int32_t *seq_lens, const int32_t *slot_base, int64_t max_seq_len, int k,
               const void *q, int H, int D, int Dv, float softmax_scale, const dsa_kv_pool *kv,
               const dsa_kv_pool *kv_swa, const int32_t *idx_swa, int k_swa, int32_t *idx_out,
               void *out, float *lse, void *ws, size_t ws_bytes, int32_t *err_flag,
               dsa_stream_t stream) {
  return dsa_decode_ex(q_idx, idx_dtype, q_scale, k_idx, k_scale, k_rows, w, H_I, d_idx, B,
                       seq_lens, slot_base, max_seq_len, k, q, H, D, Dv, softmax_scale, kv, kv_swa,
                       idx_swa, k_swa, idx_out, out, lse, ws, ws_bytes, err_flag, nullptr, stream);
}

int dsa_decode_ex(const void *q_idx, int idx_dtype, const float *q_scale, const void *k_idx,
                  const float *k_scale, int64_t k_rows, const float *w, int H_I, int d_idx, int B,
                  const int32_t *seq_lens, const int32_t *slot_base, int64_t max_seq_len, int k,
                  const void *q, int H, int D, int Dv, float softmax_scale, const dsa_kv_pool *kv,
                  const dsa_kv_pool *kv_swa, const int32_t *idx_swa, int k_swa, int32_t *idx_out,
                  void *out, float *lse, void *ws, size_t ws_bytes, int32_t *err_flag,
                  const dsa_attn_opts *opts, dsa_stream_t stream) {
  const int rpr = opts ? opts->rows_per_request : 0;
  if (rpr < 0 || rpr > 2) return DSA_ERR_UNSUPPORTED;
  if (B < 0 || max_seq_len < 0) return DSA_ERR_INVALID_ARG;
  if (rpr == 2) {
    // the paired index score: two rows of 64 heads at most, one 128-byte K-block
    if (B % 2 != 0) return DSA_ERR_INVALID_ARG;
    if (H_I > 64 || !((idx_dtype == DSA_IDX_FP8_E4M3 && d_idx == 128) ||
                      (idx_dtype == DSA_IDX_BF16 && d_idx == 64)))
      return DSA_ERR_UNSUPPORTED;
  }
  if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  int st = check_indexer(q_idx, idx_dtype, q_scale, k_idx, k_scale, k_rows, w, B, H_I, d_idx);
  if (st != DSA_OK) return st;
  // idx_out is optional: the selection then lives in the workspace
  st = check_mla_shape(q, B, H, D, Dv, softmax_scale, kv, idx_out, k, kv_swa, idx_swa, k_swa, out, lse,
                       /*need_idx=*/false);
  if (st != DSA_OK) return st;
  if (B == 0) return DSA_OK;
  if (!seq_lens || !slot_base) return DSA_ERR_INVALID_ARG;
  const size_t need = dsa_decode_workspace_size(B, max_seq_len, k, H, Dv, k_swa);
  if (ws_bytes < need || !ws) return DSA_ERR_WORKSPACE_TOO_SMALL;
  return decode_enqueue(q_idx, idx_dtype, q_scale, k_idx, k_scale, k_rows, w, H_I, d_idx, B,
                        seq_lens, slot_base, max_seq_len, k, q, H, D, Dv, softmax_scale, kv, kv_swa,
                        idx_swa, k_swa, idx_out, out, lse, ws, err_flag,
                        reinterpret_cast<cudaStream_t>(stream), opts);
}

int dsa_decode_paged(const void *q_idx, int idx_dtype, const float *q_scale, const void *k_idx,
                     const float *k_scale, int64_t k_rows, const float *w, int H_I, int d_idx,
                     int B, const int32_t *seq_lens, const int32_t *block_table, int max_pages,
                     int page_size, int64_t max_seq_len, int k, const void *q, int H, int D,
                     int Dv, float softmax_scale, const dsa_kv_pool *kv,
                     const dsa_kv_pool *kv_swa, const int32_t *idx_swa, int k_swa,
                     int32_t *idx_out, void *out, float *lse, void *ws, size_t ws_bytes,
                     int32_t *err_flag, const dsa_attn_opts *opts, dsa_stream_t stream) {
  if (opts && opts->rows_per_request != 0) return DSA_ERR_INVALID_ARG;
  if (B < 0 || max_seq_len < 0 || max_pages < 0) return DSA_ERR_INVALID_ARG;
  if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (page_size < 64 || page_size % 64 != 0) return DSA_ERR_UNSUPPORTED;
  if ((int64_t)max_pages * page_size < max_seq_len) return DSA_ERR_INVALID_ARG;
  int st = check_indexer(q_idx, idx_dtype, q_scale, k_idx, k_scale, k_rows, w, B, H_I, d_idx);
  if (st != DSA_OK) return st;
  st = check_mla_shape(q, B, H, D, Dv, softmax_scale, kv, idx_out, k, kv_swa, idx_swa, k_swa, out, lse,
                       /*need_idx=*/false);
  if (st != DSA_OK) return st;
  if (B == 0) return DSA_OK;
  if (!seq_lens || !block_table) return DSA_ERR_INVALID_ARG;
  const size_t need = dsa_decode_workspace_size(B, max_seq_len, k, H, Dv, k_swa);
  if (ws_bytes < need || !ws) return DSA_ERR_WORKSPACE_TOO_SMALL;
  const PageMap pages{block_table, max_pages, page_size};
  return decode_enqueue(q_idx, idx_dtype, q_scale, k_idx, k_scale, k_rows, w, H_I, d_idx, B,
                        seq_lens, nullptr, max_seq_len, k, q, H, D, Dv, softmax_scale, kv, kv_swa,
                        idx_swa, k_swa, idx_out, out, lse, ws, err_flag,
                        reinterpret_cast<cudaStream_t>(stream), opts, pages);
}

size_t dsa_decode_host_workspace_size(int B, int64_t max_seq_len, int k, int H_I, int d_idx,
                                      int idx_dtype, int H, int D, int Dv, int k_swa) {
  if (B < 0 || max_seq_len < 0 || k < 0 || H_I < 0 || d_idx < 0 || H < 0 || D < 0 || Dv < 0 ||
      k_swa < 0)
    return 0;
  return host_staging(B, max_seq_len, k, H_I, d_idx, idx_dtype, H, D, Dv, k_swa, nullptr).bytes;
}

int dsa_decode_host(const void *h_q_idx, int idx_dtype, const float *h_q_scale,
                    const void *k_idx, const float *k_scale, int64_t k_rows, const float *h_w,
                    int H_I, int d_idx, int B, const int32_t *h_seq_lens,
                    const int32_t *h_slot_base, int64_t max_seq_len, int k, const void *h_q,
                    int H, int D, int Dv, float softmax_scale, const dsa_kv_pool *kv,
                    const dsa_kv_pool *kv_swa, const int32_t *h_idx_swa, int k_swa,
                    int32_t *h_idx_out, void *h_out, float *h_lse, void *ws, size_t ws_bytes,
                    int32_t *err_flag, dsa_stream_t stream) {
  if (B < 0 || max_seq_len < 0 || k_swa < 0) return DSA_ERR_INVALID_ARG;
  if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (idx_dtype != DSA_IDX_FP8_E4M3 && idx_dtype != DSA_IDX_BF16) return DSA_ERR_UNSUPPORTED;
  if (B == 0) return DSA_OK;
  if (!h_q_idx || !h_w || !h_seq_lens || !h_slot_base || !h_q || !h_out || !h_lse)
    return DSA_ERR_INVALID_ARG;
  if (idx_dtype == DSA_IDX_FP8_E4M3 && !h_q_scale) return DSA_ERR_INVALID_ARG;
  if (k_swa > 0 && !h_idx_swa) return DSA_ERR_INVALID_ARG;
  if (H_I < 1 || d_idx < 1 || H < 1 || D < 1 || Dv < 1) return DSA_ERR_UNSUPPORTED;
  const size_t need =
      dsa_decode_host_workspace_size(B, max_seq_len, k, H_I, d_idx, idx_dtype, H, D, Dv, k_swa);
  if (!ws || ws_bytes < need) return DSA_ERR_WORKSPACE_TOO_SMALL;
  const HostStaging S =
      host_staging(B, max_seq_len, k, H_I, d_idx, idx_dtype, H, D, Dv, k_swa, ws);
  // the checks of dsa_decode, on the device copies, before anything is enqueued
  int st = check_indexer(S.q_idx, idx_dtype, h_q_scale ? S.q_scale : nullptr, k_idx, k_scale,
                         k_rows, S.w, B, H_I, d_idx);
  if (st != DSA_OK) return st;
  st = check_mla_shape(S.q, B, H, D, Dv, softmax_scale, kv, S.idx_out, k, kv_swa, k_swa > 0 ? S.idx_swa : nullptr,
                       k_swa, S.out, S.lse, /*need_idx=*/false);
  if (st != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t qi_bytes = (size_t)B * H_I * d_idx * idx_elem_bytes(idx_dtype);
  // the inputs, in stream order ahead of the step (a copy on a second stream
  // overlapping the index score was measured slower: the wait for it cost the
  // top-k its early launch), then the step, then the outputs.  Pinned,
  // aligned host buffers are moved by two copy kernels (see SegBuilder),
  // any other by the copy engines.  Pinned, aligned out and lse buffers are
  // written by the step itself through their device addresses (the last
  // kernel's stores cross to host memory), so only the selection is copied
  // back.
  void *d_out = const_cast<void *>(mapped_host(h_out));
  float *d_lse = static_cast<float *>(const_cast<void *>(mapped_host(h_lse)));
  const bool direct_out = d_out && d_lse;
  SegBuilder in, out;
  in.add(h_q, S.q, (size_t)B * H * D * 2, true);
  if (k_swa > 0) in.add(h_idx_swa, S.idx_swa, (size_t)B * k_swa * 4, true);
  in.add(h_seq_lens, S.seq_lens, (size_t)B * 4, true);
  in.add(h_slot_base, S.slot_base, (size_t)B * 4, true);
  in.add(h_q_idx, S.q_idx, qi_bytes, true);
  in.add(h_w, S.w, (size_t)B * H_I * 4, true);
  if (h_q_scale) in.add(h_q_scale, S.q_scale, (size_t)B * H_I * 4, true);
  if (h_idx_out) out.add(h_idx_out, S.idx_out, (size_t)B * k * 4, false);
  if (!direct_out) {
    out.add(h_out, S.out, (size_t)B * H * Dv * 2, false);
    out.add(h_lse, S.lse, (size_t)B * H * 4, false);
  }
  const bool kernels_io = in.ok && out.ok;
  bool ok = kernels_io ? in.launch(s) == cudaSuccess :
            cudaMemcpyAsync(S.q, h_q, (size_t)B * H * D * 2, cudaMemcpyHostToDevice, s) == cudaSuccess &&
            (k_swa == 0 || cudaMemcpyAsync(S.idx_swa, h_idx_swa, (size_t)B * k_swa * 4,
                                           cudaMemcpyHostToDevice, s) == cudaSuccess) &&
            cudaMemcpyAsync(S.seq_lens, h_seq_lens, (size_t)B * 4, cudaMemcpyHostToDevice, s) == cudaSuccess &&
            cudaMemcpyAsync(S.slot_base, h_slot_base, (size_t)B * 4, cudaMemcpyHostToDevice, s) == cudaSuccess &&
            cudaMemcpyAsync(S.q_idx, h_q_idx, qi_bytes, cudaMemcpyHostToDevice, s) == cudaSuccess &&
            cudaMemcpyAsync(S.w, h_w, (size_t)B * H_I * 4, cudaMemcpyHostToDevice, s) == cudaSuccess &&
            (!h_q_scale || cudaMemcpyAsync(S.q_scale, h_q_scale, (size_t)B * H_I * 4,
                                           cudaMemcpyHostToDevice, s) == cudaSuccess);
  if (!ok) return DSA_ERR_CUDA;
  st = decode_enqueue(S.q_idx, idx_dtype, h_q_scale ? S.q_scale : nullptr, k_idx, k_scale,
                      k_rows, S.w, H_I, d_idx, B, S.seq_lens, S.slot_base, max_seq_len, k, S.q,
                      H, D, Dv, softmax_scale, kv, kv_swa, k_swa > 0 ? S.idx_swa : nullptr, k_swa,
                      S.idx_out, direct_out ? d_out : S.out, direct_out ? d_lse : S.lse, S.dec_ws,
                      err_flag, s);
  if (st != DSA_OK) return st;
  if (kernels_io) return status_of(out.launch(s));
  ok = (!h_idx_out || cudaMemcpyAsync(h_idx_out, S.idx_out, (size_t)B * k * 4,
                                      cudaMemcpyDeviceToHost, s) == cudaSuccess) &&
       (direct_out ||
        (cudaMemcpyAsync(h_out, S.out, (size_t)B * H * Dv * 2, cudaMemcpyDeviceToHost, s) == cudaSuccess &&
         cudaMemcpyAsync(h_lse, S.lse, (size_t)B * H * 4, cudaMemcpyDeviceToHost, s) == cudaSuccess));
  return ok ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_decode_graph_create(const void *h_q_idx, int idx_dtype, const float *h_q_scale,
                            const void *k_idx, const float *k_scale, int64_t k_rows,
                            const float *h_w, int H_I, int d_idx, int B,
                            const int32_t *h_seq_lens, const int32_t *h_slot_base,
                            int64_t max_seq_len, int k, const void *h_q, int H, int D, int Dv,
                            float softmax_scale, const dsa_kv_pool *kv, const dsa_kv_pool *kv_swa,
                            const int32_t *h_idx_swa, int k_swa, int32_t *h_idx_out, void *h_out,
                            float *h_lse, void *ws, size_t ws_bytes, int32_t *err_flag,
                            dsa_decode_graph *graph) {
  if (!graph) return DSA_ERR_INVALID_ARG;
  *graph = nullptr;
  if (B < 1) return DSA_ERR_INVALID_ARG;   // an empty step has nothing to capture
  cudaStream_t cs;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return DSA_ERR_CUDA;
  int st = DSA_ERR_CUDA;
  cudaGraph_t g = nullptr;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
    st = dsa_decode_host(h_q_idx, idx_dtype, h_q_scale, k_idx, k_scale, k_rows, h_w, H_I, d_idx, B,
                         h_seq_lens, h_slot_base, max_seq_len, k, h_q, H, D, Dv, softmax_scale, kv,
                         kv_swa, h_idx_swa, k_swa, h_idx_out, h_out, h_lse, ws, ws_bytes, err_flag,
                         reinterpret_cast<dsa_stream_t>(cs));
    // the capture ends whatever happened inside it
    if (cudaStreamEndCapture(cs, &g) != cudaSuccess && st == DSA_OK) st = DSA_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  if (st == DSA_OK && cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) st = DSA_ERR_CUDA;
  if (g) cudaGraphDestroy(g);
  cudaStreamDestroy(cs);
  if (st != DSA_OK) return st;
  dsa_decode_graph h = new (std::nothrow) dsa_decode_graph_s{exec};
  if (!h) {
    cudaGraphExecDestroy(exec);
    return DSA_ERR_CUDA;
  }
  *graph = h;
  return DSA_OK;
}

int dsa_decode_graph_launch(dsa_decode_graph graph, dsa_stream_t stream) {
  if (!graph) return DSA_ERR_INVALID_ARG;
  return status_of(cudaGraphLaunch(graph->exec, reinterpret_cast<cudaStream_t>(stream)));
}

void dsa_decode_graph_destroy(dsa_decode_graph graph) {
  if (!graph) return;
  cudaGraphExecDestroy(graph->exec);
  delete graph;
}

}  // extern "C"
