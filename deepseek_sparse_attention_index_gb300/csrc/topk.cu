// Per-row top-k by radix select, deterministic, -1 padded.
//
// The selector of tokenspeed PR #627 "Add gluon kernel for DSA" (review of
// the top-k kernel: count the elements "greater" than and "equal" to a
// threshold, then reserve output slots) places tied elements with atomics,
// so which of several equal scores survives depends on timing.  Here the
// threshold is found exactly and ties go to the lower position, so the
// selected set is a function of the scores alone:
//
//   1. histogram  -- 4096 bins over the top 12 bits of an order-preserving
//                    uint32 key of each score (fused into the index-score
//                    epilogue in the decode path);
//   2. collect    -- many CTAs per row: find the bin b1 where the count from
//                    the top first reaches k; append positions in bins above
//                    b1 (fewer than k of them) to a per-row list and the
//                    (key, position) pairs of bin b1 to a candidate list;
//   3. resolve    -- one CTA per row: two more radix levels over the
//                    candidates (bits 19..8, then 7..0) give the exact k-th
//                    key K*; a radix select over positions picks the lowest
//                    positions among the elements equal to K*; the k
//                    survivors are sorted by position and written out.
// If a row's candidate list overflows (many near-equal scores), the resolve
// pass reads that row's scores again instead of the list: slower, same
// result.
#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kCollectThreads = 512;
constexpr int kResolveThreads = 1024;
constexpr int kHistThreads = 512;

// Exclusive prefix sum over the block (blockDim.x a multiple of 32, <= 1024).
// Returns this thread's exclusive prefix; *total gets the block sum.
__device__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_sums, uint32_t *total) {
  const unsigned lane = lane_id();
  const unsigned warp = threadIdx.x >> 5;
  const unsigned nwarps = blockDim.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= (unsigned)o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= (unsigned)o) s += y;
    }
    if (lane < nwarps) warp_sums[lane] = s;  // inclusive
  }
  __syncthreads();
  uint32_t before = (warp == 0 ? 0u : warp_sums[warp - 1]) + x - v;
  *total = warp_sums[nwarps - 1];
  __syncthreads();
  return before;
}

// Over a histogram h[0..nbins) in shared memory, find the bin where the
// cumulative count first reaches `need`, walking from the highest bin down
// (descending = true) or from bin 0 up.  *bin_out / *before_out (shared)
// receive that bin and the count strictly before it in walk order.
// nbins must be a multiple of blockDim.x.
__device__ void find_bin(const uint32_t *h, int nbins, uint32_t need, bool descending,
                         uint32_t *warp_sums, int *bin_out, uint32_t *before_out) {
  const int per = nbins / blockDim.x;
  // thread i owns walk positions [i*per, (i+1)*per)
  uint32_t sum = 0;
  for (int j = 0; j < per; ++j) {
    int wpos = threadIdx.x * per + j;
    int b = descending ? nbins - 1 - wpos : wpos;
    sum += h[b];
  }
  uint32_t tot;
  uint32_t cum = block_excl_scan(sum, warp_sums, &tot);
  for (int j = 0; j < per; ++j) {
    int wpos = threadIdx.x * per + j;
    int b = descending ? nbins - 1 - wpos : wpos;
    uint32_t c = h[b];
    if (cum < need && cum + c >= need) {
      *bin_out = b;
      *before_out = cum;
    }
    cum += c;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kHistThreads)
topk_hist_kernel(const float *__restrict__ scores, int64_t ld, const int32_t *__restrict__ row_len,
                 int k, int chunk, uint32_t *__restrict__ hist) {
  __shared__ uint32_t sh[kHistBins];
  const int t = blockIdx.y;
  const int64_t L = max(row_len[t], 0);
  const int64_t lo = (int64_t)blockIdx.x * chunk;
  if (L <= k || lo >= L) return;
  const int64_t hi = min(L, lo + chunk);
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const float *row = scores + (int64_t)t * ld;
  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x)
    atomicAdd(&sh[score_key(row[i]) >> 20], 1u);
  __syncthreads();
  uint32_t *gh = hist + (size_t)t * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
    if (sh[i]) atomicAdd(&gh[i], sh[i]);
}

__global__ void __launch_bounds__(kCollectThreads)
topk_collect_kernel(const float *__restrict__ scores, int64_t ld,
                    const int32_t *__restrict__ row_len, int k, int chunk,
                    const uint32_t *__restrict__ hist, uint32_t *__restrict__ cnt,
                    int32_t *__restrict__ gt_list, uint2 *__restrict__ cand) {
  __shared__ uint32_t sh[kHistBins];
  __shared__ uint32_t warp_sums[32];
  __shared__ int s_bin;
  __shared__ uint32_t s_before;
  const int t = blockIdx.y;
  const int64_t L = max(row_len[t], 0);
  const int64_t lo = (int64_t)blockIdx.x * chunk;
  if (L <= k || lo >= L) return;
  const int64_t hi = min(L, lo + chunk);
  const uint32_t *gh = hist + (size_t)t * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sh[i] = gh[i];
  if (threadIdx.x == 0) { s_bin = 0; s_before = 0; }
  __syncthreads();
  find_bin(sh, kHistBins, (uint32_t)k, true, warp_sums, &s_bin, &s_before);
  const uint32_t b1 = (uint32_t)s_bin;
  const float *row = scores + (int64_t)t * ld;
  const unsigned lane = lane_id();
  const unsigned lt_mask = (1u << lane) - 1u;
  uint32_t *c_gt = cnt + 2 * t;
  uint32_t *c_eq = c_gt + 1;
  int32_t *gl = gt_list + (size_t)t * k;
  uint2 *cl = cand + (size_t)t * kCandCap;
  for (int64_t base = lo; base < hi; base += blockDim.x) {
    const int64_t i = base + threadIdx.x;
    const bool valid = i < hi;
    const uint32_t key = valid ? score_key(row[i]) : 0u;
    const uint32_t bin = key >> 20;
    const bool is_gt = valid && bin > b1;
    const bool is_eq = valid && bin == b1;
    const unsigned mg = __ballot_sync(0xffffffffu, is_gt);
    if (mg) {
      uint32_t off = 0;
      const int leader = __ffs(mg) - 1;
      if ((int)lane == leader) off = atomicAdd(c_gt, (uint32_t)__popc(mg));
      off = __shfl_sync(0xffffffffu, off, leader);
      const uint32_t my = off + __popc(mg & lt_mask);
      if (is_gt && my < (uint32_t)k) gl[my] = (int32_t)i;
    }
    const unsigned me = __ballot_sync(0xffffffffu, is_eq);
    if (me) {
      uint32_t off = 0;
      const int leader = __ffs(me) - 1;
      if ((int)lane == leader) off = atomicAdd(c_eq, (uint32_t)__popc(me));
      off = __shfl_sync(0xffffffffu, off, leader);
      const uint32_t my = off + __popc(me & lt_mask);
      if (is_eq && my < (uint32_t)kCandCap) cl[my] = make_uint2(key, (uint32_t)i);
    }
  }
}

// Source of (key, position) pairs for the resolve passes: the candidate list,
// or -- after an overflow -- the row itself filtered to bin b1.
struct Source {
  const uint2 *cand;
  const float *row;
  int64_t n;        // list length, or the row length when reading the row
  bool from_row;
  uint32_t b1;
  __device__ bool get(int64_t i, uint32_t &key, int32_t &pos) const {
    if (!from_row) {
      uint2 c = cand[i];
      key = c.x;
      pos = (int32_t)c.y;
      return true;
    }
    key = score_key(row[i]);
    pos = (int32_t)i;
    return (key >> 20) == b1;
  }
};

__global__ void __launch_bounds__(kResolveThreads)
topk_resolve_kernel(const float *__restrict__ scores, int64_t ld,
                    const int32_t *__restrict__ row_len, int k,
                    const int32_t *__restrict__ index_base,
                    const uint32_t *__restrict__ hist, const uint32_t *__restrict__ cnt,
                    const int32_t *__restrict__ gt_list, const uint2 *__restrict__ cand,
                    int32_t *__restrict__ idx, int32_t *__restrict__ lens,
                    int32_t *err_flag) {
  __shared__ uint32_t sh[kHistBins];
  __shared__ int32_t sel[DSA_MAX_TOPK];
  __shared__ uint32_t warp_sums[32];
  __shared__ int s_bin;
  __shared__ uint32_t s_before;
  __shared__ uint32_t s_fill;
  const int t = blockIdx.x;
  const int64_t L = max(row_len[t], 0);
  const int32_t base = index_base ? index_base[t] : 0;
  int32_t *out = idx + (size_t)t * k;
  if (L <= k) {
    for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = j < L ? (int32_t)j + base : -1;
    if (lens && threadIdx.x == 0) lens[t] = (int32_t)L;
    return;
  }
  // level 1 again: the bin b1 and the count above it
  const uint32_t *gh = hist + (size_t)t * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sh[i] = gh[i];
  if (threadIdx.x == 0) { s_bin = 0; s_before = 0; }
  __syncthreads();
  find_bin(sh, kHistBins, (uint32_t)k, true, warp_sums, &s_bin, &s_before);
  const uint32_t b1 = (uint32_t)s_bin;
  const uint32_t n_gt = cnt[2 * t];
  const uint32_t n_eq = cnt[2 * t + 1];
  if (n_gt != s_before || n_gt >= (uint32_t)k) {
    // histogram and collect pass disagree: only NaN scores can do this
    if (threadIdx.x == 0) raise_flag(err_flag, DSA_DEVERR_INDEX_RANGE);
    for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = -1;
    if (lens && threadIdx.x == 0) lens[t] = 0;
    return;
  }
  Source src;
  src.cand = cand + (size_t)t * kCandCap;
  src.row = scores + (int64_t)t * ld;
  src.from_row = n_eq > (uint32_t)kCandCap;
  src.n = src.from_row ? L : (int64_t)n_eq;
  src.b1 = b1;
  const uint32_t r1 = (uint32_t)k - n_gt;  // to take from bin b1

  // level 2: bits 19..8
  __syncthreads();
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  for (int64_t i = threadIdx.x; i < src.n; i += blockDim.x) {
    uint32_t key; int32_t pos;
    if (src.get(i, key, pos)) atomicAdd(&sh[(key >> 8) & 0xFFFu], 1u);
  }
  __syncthreads();
  find_bin(sh, kHistBins, r1, true, warp_sums, &s_bin, &s_before);
  const uint32_t b2 = (uint32_t)s_bin;
  const uint32_t r2 = r1 - s_before;

  // level 3: bits 7..0 among keys whose bits 19..8 are b2
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  for (int64_t i = threadIdx.x; i < src.n; i += blockDim.x) {
    uint32_t key; int32_t pos;
    if (src.get(i, key, pos) && ((key >> 8) & 0xFFFu) == b2) atomicAdd(&sh[key & 0xFFu], 1u);
  }
  __syncthreads();
  // 256 bins: use a 256-thread view of find_bin by padding to blockDim bins
  for (int i = 256 + threadIdx.x; i < kResolveThreads; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  // bins 256..1023 are zero; walking descending from 1023 passes them first
  find_bin(sh, kResolveThreads, r2, true, warp_sums, &s_bin, &s_before);
  const uint32_t b3 = (uint32_t)s_bin;
  const uint32_t r3 = r2 - s_before;  // how many elements equal to K* to keep
  const uint32_t m_eq = sh[b3];       // how many elements equal K*
  const uint32_t kstar = (b1 << 20) | (b2 << 8) | b3;

  // positions among the elements equal to K*: keep the r3 lowest
  int32_t pstar = 0x7fffffff;
  if (r3 < m_eq) {
    uint32_t prefix = 0;  // position bits fixed so far
    uint32_t need = r3;
    const int shifts[3] = {20, 10, 0};
    const int widths[3] = {11, 10, 10};
    for (int lvl = 0; lvl < 3; ++lvl) {
      const int sft = shifts[lvl];
      const uint32_t nb = 1u << widths[lvl];
      __syncthreads();
      for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sh[i] = 0;
      __syncthreads();
      for (int64_t i = threadIdx.x; i < src.n; i += blockDim.x) {
        uint32_t key; int32_t pos;
        if (src.get(i, key, pos) && key == kstar) {
          const uint32_t p = (uint32_t)pos;
          const uint32_t hi_bits = lvl == 0 ? 0u : (p >> (sft + widths[lvl]));
          if (hi_bits == prefix) atomicAdd(&sh[(p >> sft) & (nb - 1)], 1u);
        }
      }
      __syncthreads();
      // ascending walk over max(nb, blockDim) bins (extra bins are zero)
      const int nbins = (int)max(nb, (uint32_t)blockDim.x);
      find_bin(sh, nbins, need, false, warp_sums, &s_bin, &s_before);
      need -= s_before;
      prefix = (prefix << widths[lvl]) | (uint32_t)s_bin;
    }
    pstar = (int32_t)prefix;
  }

  // gather the survivors
  if (threadIdx.x == 0) s_fill = n_gt;
  const int32_t *gl = gt_list + (size_t)t * k;
  for (int j = threadIdx.x; j < (int)n_gt; j += blockDim.x) sel[j] = gl[j];
  __syncthreads();
  for (int64_t i = threadIdx.x; i < src.n; i += blockDim.x) {
    uint32_t key; int32_t pos;
    if (src.get(i, key, pos) && (key > kstar || (key == kstar && pos <= pstar))) {
      uint32_t slot = atomicAdd(&s_fill, 1u);
      if (slot < (uint32_t)k) sel[slot] = pos;
    }
  }
  __syncthreads();
  if (s_fill != (uint32_t)k && threadIdx.x == 0) raise_flag(err_flag, DSA_DEVERR_INDEX_RANGE);
  // bitonic sort of sel[0..kp) ascending, kp = next power of two >= k
  int kp = 1;
  while (kp < k) kp <<= 1;
  for (int j = k + threadIdx.x; j < kp; j += blockDim.x) sel[j] = 0x7fffffff;
  __syncthreads();
  for (int size = 2; size <= kp; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (kp >> 1); i += blockDim.x) {
        const int lo_i = 2 * i - (i & (stride - 1));
        const int hi_i = lo_i + stride;
        const bool up = (lo_i & size) == 0;
        const int32_t a = sel[lo_i], b = sel[hi_i];
        if ((a > b) == up) { sel[lo_i] = b; sel[hi_i] = a; }
      }
      __syncthreads();
    }
  }
  for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = sel[j] + base;
  if (lens && threadIdx.x == 0) lens[t] = k;
}

int collect_chunk(int T, int64_t max_len) {
  // enough CTAs to cover the GPU about twice, 2k..16k positions each
  int64_t target = 2LL * num_sms();
  int64_t chunk = 16384;
  while (chunk > 2048 && (int64_t)T * ((max_len + chunk - 1) / chunk) < target) chunk >>= 1;
  return (int)chunk;
}

}  // namespace

size_t topk_ws_layout(int T, int k, void *ws, TopkWs *out) {
  WsCarver c(ws);
  TopkWs w;
  w.hist = c.take<uint32_t>((size_t)T * kHistBins);
  w.cnt = c.take<uint32_t>((size_t)T * 2);
  w.gt_list = c.take<int32_t>((size_t)T * k);
  w.cand = c.take<uint2>((size_t)T * kCandCap);
  if (out) *out = w;
  return c.bytes();
}

cudaError_t topk_clear(const TopkWs &w, int T, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(w.hist, 0, sizeof(uint32_t) * (size_t)T * kHistBins, s);
  if (e != cudaSuccess) return e;
  return cudaMemsetAsync(w.cnt, 0, sizeof(uint32_t) * (size_t)T * 2, s);
}

cudaError_t topk_hist(const float *scores, int64_t ld, const int32_t *row_len, int T,
                      int64_t max_len, int k, const TopkWs &w, cudaStream_t s) {
  if (max_len <= k) return cudaSuccess;
  const int chunk = collect_chunk(T, max_len);
  dim3 grid((unsigned)((max_len + chunk - 1) / chunk), (unsigned)T);
  topk_hist_kernel<<<grid, kHistThreads, 0, s>>>(scores, ld, row_len, k, chunk, w.hist);
  return cudaGetLastError();
}

cudaError_t topk_select(const float *scores, int64_t ld, const int32_t *row_len, int T,
                        int64_t max_len, int k, const int32_t *index_base, int32_t *idx,
                        int32_t *lens, const TopkWs &w, int32_t *err_flag, cudaStream_t s) {
  if (max_len > k) {
    const int chunk = collect_chunk(T, max_len);
    dim3 grid((unsigned)((max_len + chunk - 1) / chunk), (unsigned)T);
    topk_collect_kernel<<<grid, kCollectThreads, 0, s>>>(scores, ld, row_len, k, chunk, w.hist,
                                                          w.cnt, w.gt_list, w.cand);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  topk_resolve_kernel<<<T, kResolveThreads, 0, s>>>(scores, ld, row_len, k, index_base, w.hist,
                                                    w.cnt, w.gt_list, w.cand, idx, lens,
                                                    err_flag);
  return cudaGetLastError();
}

}  // namespace dsa
