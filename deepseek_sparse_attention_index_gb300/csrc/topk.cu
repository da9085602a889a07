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


// Loads this thread's 16 elements of the chunk window starting at `base`:
// element (r, c) is position base + 4 * (r * blockDim.x + threadIdx.x) + c.
// Four float4 loads in flight at once when the row is 16-byte aligned, else
// scalar loads.  Positions at or past `hi` are reported invalid.
struct Elems16 {
  float v[16];
  int64_t p0[4];
};
__device__ __forceinline__ void load16(const float *row, int64_t base, int64_t hi, bool vec,
                                       Elems16 &E) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int64_t p = base + 4 * ((int64_t)r * blockDim.x + threadIdx.x);
    E.p0[r] = p;
    if (vec && p + 3 < hi) {
      const float4 q = __ldcg(reinterpret_cast<const float4 *>(row + p));
      E.v[4 * r] = q.x; E.v[4 * r + 1] = q.y; E.v[4 * r + 2] = q.z; E.v[4 * r + 3] = q.w;
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) E.v[4 * r + c] = (p + c < hi) ? __ldcg(row + p + c) : 0.f;
    }
  }
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
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  for (int64_t base = lo; base < hi; base += 16 * (int64_t)blockDim.x) {
    Elems16 E;
    load16(row, base, hi, vec, E);
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (E.p0[e >> 2] + (e & 3) < hi) atomicAdd(&sh[score_key(E.v[e]) >> 20], 1u);
  }
  __syncthreads();
  uint32_t *gh = hist + (size_t)t * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
    if (sh[i]) atomicAdd(&gh[i], sh[i]);
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

// Resolves row t once its collect pass is complete: two more radix levels
// over the candidates give the exact k-th key, a radix select over positions
// breaks ties toward lower positions, and the k survivors are sorted by
// position.  Run by one whole CTA (blockDim.x a multiple of 32 dividing 512).
struct ResolveSmem {
  uint32_t sh[kHistBins];
  int32_t sel[DSA_MAX_TOPK];
  uint32_t warp_sums[32];
  int s_bin;
  uint32_t s_before;
  uint32_t s_fill;
};

__device__ __noinline__ void resolve_row(int t, ResolveSmem &S, const float *__restrict__ scores, int64_t ld,
                            const int32_t *__restrict__ row_len, int k,
                            const int32_t *__restrict__ index_base,
                            const uint32_t *__restrict__ hist, const uint32_t *__restrict__ cnt,
                            const int32_t *__restrict__ gt_list, const uint2 *__restrict__ cand,
                            int32_t *__restrict__ idx, int32_t *__restrict__ lens,
                            int32_t *err_flag) {
  uint32_t *sh = S.sh;
  int32_t *sel = S.sel;
  uint32_t *warp_sums = S.warp_sums;
  int &s_bin = S.s_bin;
  uint32_t &s_before = S.s_before;
  uint32_t &s_fill = S.s_fill;
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
  const uint32_t n_gt = cnt[4 * t];
  const uint32_t n_eq = cnt[4 * t + 1];
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
  // 256 bins padded with zero bins to a multiple of the block size
  const int nb3 = max(256, (int)blockDim.x);
  for (int i = 256 + threadIdx.x; i < nb3; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  // the zero bins sit above bin 255; walking down from the top passes them first
  find_bin(sh, nb3, r2, true, warp_sums, &s_bin, &s_before);
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

// Collect pass, and the resolve of each row by the last of its CTAs to finish
// (every CTA fences its writes and bumps the row's done counter; the CTA that
// sees the count complete resolves the row -- nobody waits on anybody).
// Each CTA appends its "above the threshold bin" positions and its
// "in the threshold bin" candidates with one atomic per list: per-thread
// counts go through a block scan, thread 0 reserves the CTA's range.
__global__ void __launch_bounds__(kCollectThreads, 2)
topk_collect_kernel(const float *__restrict__ scores, int64_t ld,
                    const int32_t *__restrict__ row_len, int k, int chunk,
                    const int32_t *__restrict__ index_base, const uint32_t *__restrict__ hist,
                    uint32_t *__restrict__ cnt, int32_t *__restrict__ gt_list,
                    uint2 *__restrict__ cand, int32_t *__restrict__ idx,
                    int32_t *__restrict__ lens, int32_t *err_flag) {
  __shared__ ResolveSmem S;
  __shared__ uint32_t s_base_gt, s_base_eq;
  __shared__ int s_last;
  const int t = blockIdx.y;
  const int64_t L = max(row_len[t], 0);
  if (L <= k) {                     // every position is selected: no search
    if (blockIdx.x == 0) {
      const int32_t base = index_base ? index_base[t] : 0;
      int32_t *out = idx + (size_t)t * k;
      for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = j < L ? (int32_t)j + base : -1;
      if (lens && threadIdx.x == 0) lens[t] = (int32_t)L;
    }
    return;
  }
  const int64_t lo = (int64_t)blockIdx.x * chunk;
  if (lo >= L) return;
  const int64_t hi = min(L, lo + chunk);
  const float *row = scores + (int64_t)t * ld;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  Elems16 E;
  load16(row, lo, hi, vec, E);   // first window in flight while the threshold is found
  const uint32_t *gh = hist + (size_t)t * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) S.sh[i] = gh[i];
  if (threadIdx.x == 0) { S.s_bin = 0; S.s_before = 0; }
  __syncthreads();
  find_bin(S.sh, kHistBins, (uint32_t)k, true, S.warp_sums, &S.s_bin, &S.s_before);
  const uint32_t b1 = (uint32_t)S.s_bin;
  uint32_t *c_gt = cnt + 4 * t;
  uint32_t *c_eq = c_gt + 1;
  uint32_t *c_done = c_gt + 2;
  int32_t *gl = gt_list + (size_t)t * k;
  uint2 *cl = cand + (size_t)t * kCandCap;
  for (int64_t base = lo; base < hi; base += 16 * (int64_t)blockDim.x) {
    if (base != lo) load16(row, base, hi, vec, E);
    uint32_t mgt = 0, meq = 0;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const bool valid = E.p0[e >> 2] + (e & 3) < hi;
      const uint32_t bin = score_key(E.v[e]) >> 20;
      mgt |= (valid && bin > b1) ? (1u << e) : 0u;
      meq |= (valid && bin == b1) ? (1u << e) : 0u;
    }
    // counts packed (gt << 16 | eq): a CTA round holds at most 16 * 1024 elements
    uint32_t tot;
    const uint32_t pre = block_excl_scan(((uint32_t)__popc(mgt) << 16) | (uint32_t)__popc(meq),
                                         S.warp_sums, &tot);
    if (threadIdx.x == 0) {
      s_base_gt = (tot >> 16) ? atomicAdd(c_gt, tot >> 16) : 0u;
      s_base_eq = (tot & 0xffffu) ? atomicAdd(c_eq, tot & 0xffffu) : 0u;
    }
    __syncthreads();
    uint32_t og = s_base_gt + (pre >> 16), oe = s_base_eq + (pre & 0xffffu);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int64_t i = E.p0[e >> 2] + (e & 3);
      if ((mgt >> e) & 1u) {
        if (og < (uint32_t)k) gl[og] = (int32_t)i;
        ++og;
      }
      if ((meq >> e) & 1u) {
        if (oe < (uint32_t)kCandCap) cl[oe] = make_uint2(score_key(E.v[e]), (uint32_t)i);
        ++oe;
      }
    }
    __syncthreads();   // s_base_* are reused by the next round
  }
  // publish this CTA's appends; the last CTA of the row resolves it
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t nch = (uint32_t)((L + chunk - 1) / chunk);
    s_last = atomicAdd(c_done, 1u) == nch - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  resolve_row(t, S, scores, ld, row_len, k, index_base, hist, cnt, gt_list, cand, idx, lens,
              err_flag);
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
  w.cnt = c.take<uint32_t>((size_t)T * 4);   // gt, eq, CTAs done, pad
  w.gt_list = c.take<int32_t>((size_t)T * k);
  w.cand = c.take<uint2>((size_t)T * kCandCap);
  if (out) *out = w;
  return c.bytes();
}

cudaError_t topk_clear(const TopkWs &w, int T, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(w.hist, 0, sizeof(uint32_t) * (size_t)T * kHistBins, s);
  if (e != cudaSuccess) return e;
  return cudaMemsetAsync(w.cnt, 0, sizeof(uint32_t) * (size_t)T * 4, s);
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
  const int chunk = collect_chunk(T, max_len);
  const int64_t nch = max_len > k ? (max_len + chunk - 1) / chunk : 1;
  dim3 grid((unsigned)nch, (unsigned)T);
  topk_collect_kernel<<<grid, kCollectThreads, 0, s>>>(scores, ld, row_len, k, chunk, index_base,
                                                        w.hist, w.cnt, w.gt_list, w.cand, idx,
                                                        lens, err_flag);
  return cudaGetLastError();
}

}  // namespace dsa
