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
//   2. collect    -- several CTAs per row, each over one chunk of at most
//                    16384 positions held in registers: find the bin b1 where
//                    the count from the top first reaches k, then append the
//                    (key, position) pair of every element in bin b1 or above
//                    to the row's list as ONE run in ascending position order
//                    (one atomic per CTA reserves it) and record the run's
//                    start and length in the row's chunk table;
//   3. resolve    -- by the row's last CTA to finish: two more radix levels
//                    over the list's bin-b1 entries (bits 19..8, then 7..0)
//                    give the exact k-th key K*; a radix select over
//                    positions picks the lowest positions among the elements
//                    equal to K*; an ordered compaction walks the runs in
//                    chunk order and writes the survivors, which therefore
//                    come out in ascending position order with no sort.
// If a row's list overflows (many near-equal scores), the resolve pass reads
// that row's scores again instead of the list: slower, same result.
//
// Rows of at most eight chunks, when the grid fits on the SMs, take a
// thread-block cluster instead (topk_cluster_kernel): each CTA of a row reads its chunk
// once and keeps only masks, the leader finds the k-th (key, position) among
// the row's bin-b1 entries, gathered in its shared memory over distributed
// shared memory, and each CTA writes its own survivors after those of the
// earlier chunks.  No list, counter or fence in global memory lies on that
// path.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kThreads = 512;               // collect / resolve CTA
constexpr int kPer = 16;                    // positions a thread holds per round
constexpr int kRound = kPer * kThreads;     // 8192 positions per round
constexpr int kRounds = 2;                  // a chunk is one or two rounds
constexpr int kMaxChunk = kRound * kRounds; // 16384
constexpr int kGather = 8;                  // entries per thread per compaction round
constexpr int kBatch = 8;                   // list entries a thread loads at once
constexpr int kListCache = 6144;            // list entries the resolve copies into (dynamic) shared memory
constexpr int kHistThreads = 512;
static_assert(kHistBins == 8 * kThreads, "threshold_bin gives each thread 8 bins");

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
// receive that bin and the count strictly before it in walk order; they are
// left alone when the total stays below `need`.  Warp w owns the walk
// positions [w * seg, (w + 1) * seg), seg = nbins / warps (a multiple of 32);
// consecutive lanes read consecutive bins (no bank conflicts), a scan over
// the warp totals picks the crossing warp, and that warp alone walks its
// segment 32 bins at a time.
template <int nbins, bool descending>
__device__ __forceinline__ void find_bin(const uint32_t *h, uint32_t need, uint32_t *warp_sums,
                                         int *bin_out, uint32_t *before_out) {
  constexpr int nw = kThreads / 32;   // blockDim.x == kThreads
  const int w = threadIdx.x >> 5;
  const unsigned lane = lane_id();
  constexpr int seg = nbins / nw;
  static_assert(seg % 32 == 0, "each warp walks whole 32-bin rows");
  uint32_t s = 0;
#pragma unroll
  for (int j = lane; j < seg; j += 32) {
    const int wpos = w * seg + j;
    s += h[descending ? nbins - 1 - wpos : wpos];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) warp_sums[w] = s;
  __syncthreads();
  if (w == 0) {
    const uint32_t v = lane < (unsigned)nw ? warp_sums[lane] : 0u;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= (unsigned)o) incl += y;
    }
    const uint32_t excl = incl - v;
    const unsigned ball = __ballot_sync(0xffffffffu, excl < need && incl >= need);
    const int cw = ball ? __ffs(ball) - 1 : -1;
    const uint32_t cb = __shfl_sync(0xffffffffu, excl, cw < 0 ? 0 : cw);
    __syncwarp();
    if (lane == 0) {
      warp_sums[0] = (uint32_t)cw;
      warp_sums[1] = cb;
    }
  }
  __syncthreads();
  const int cw = (int)warp_sums[0];
  if (w == cw) {
    uint32_t before = warp_sums[1];
    for (int j0 = 0; j0 < seg; j0 += 32) {
      const int wpos = w * seg + j0 + (int)lane;
      const int b = descending ? nbins - 1 - wpos : wpos;
      const uint32_t c = h[b];
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= (unsigned)o) incl += y;
      }
      const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
      if (before + tot >= need) {
        const unsigned ball = __ballot_sync(0xffffffffu, before + incl >= need);
        if (lane == (unsigned)(__ffs(ball) - 1)) {
          *bin_out = b;
          *before_out = before + incl - c;
        }
        break;
      }
      before += tot;
    }
  }
  __syncthreads();
}

// The first-level threshold straight from a row's histogram in global
// memory: the bin where the count from the top first reaches `need`, and the
// count above it.  Thread i owns bins [4088 - 8i, 4096 - 8i) (descending
// walk positions 8i .. 8i + 7), read with two 16-byte loads that the caller
// issues early (hist_load) and hands to the scan (threshold_bin).
// blockDim.x must be kThreads; the histogram must be 16-byte aligned.
struct HistSlice {
  uint4 lo, hi;
};
__device__ __forceinline__ HistSlice hist_load(const uint32_t *gh) {
  const uint4 *p = reinterpret_cast<const uint4 *>(gh + (kHistBins - 8) - 8 * threadIdx.x);
  return HistSlice{__ldcg(p), __ldcg(p + 1)};
}
__device__ void threshold_bin(const HistSlice &hs, uint32_t need, uint32_t *warp_sums,
                              int *bin_out, uint32_t *before_out) {
  const uint32_t h[8] = {hs.hi.w, hs.hi.z, hs.hi.y, hs.hi.x, hs.lo.w, hs.lo.z, hs.lo.y, hs.lo.x};
  uint32_t sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) sum += h[j];
  uint32_t tot;
  uint32_t cum = block_excl_scan(sum, warp_sums, &tot);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (cum < need && cum + h[j] >= need) {
      *bin_out = kHistBins - 1 - 8 * (int)threadIdx.x - j;
      *before_out = cum;
    }
    cum += h[j];
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
                 int k, int chunk, int nch, uint32_t *__restrict__ hist) {
  __shared__ uint32_t sh[kHistBins];
  // 1-D grid of rows x chunks (a 2-D grid would cap the rows at 65535)
  const int t = (int)(blockIdx.x / (unsigned)nch);
  const int c = (int)(blockIdx.x - (unsigned)t * (unsigned)nch);
  const int64_t L = max(row_len[t], 0);
  const int64_t lo = (int64_t)c * chunk;
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


// Where the resolve pass reads a row's (key, position) pairs: the list in
// shared memory (copied by the first pass when it fits), the list in global
// memory (written by other CTAs, so read through L2), or -- after an
// overflow -- the row itself.
struct Source {
  const uint2 *cache;   // shared copy of the list, or nullptr
  const uint2 *list;
  const float *row;
  int64_t n;            // list length, or the row length when reading the row
  bool from_row;
  __device__ __forceinline__ void get(int64_t i, uint32_t &key, int32_t &pos) const {
    if (cache) {
      const uint2 c = cache[i];
      key = c.x;
      pos = (int32_t)c.y;
    } else if (!from_row) {
      const uint2 c = __ldcg(list + i);
      key = c.x;
      pos = (int32_t)c.y;
    } else {
      key = score_key(__ldcg(row + i));
      pos = (int32_t)i;
    }
  }
};

struct ResolveSmem {
  uint32_t sh[kHistBins];
  uint32_t run_pre[kThreads];    // ordered start of each run of a group of chunks
  uint32_t run_at[kThreads];     // where that run sits in the list
  uint32_t warp_sums[32];
  int s_bin;
  uint32_t s_before;
  PageMap pm;                    // paged caches: the block table (set by the collect kernel)
};

// The exact k-th entry of a row inside its first-level bin b1, once the
// level-2 histogram (bits 19..8 of the bin-b1 keys) is in S.sh: the level-2
// bin, a level-3 pass over bits 7..0, and -- when several entries equal the
// k-th key K* -- a radix select over their positions that keeps the lowest.
// for_each(f) calls f(key, position) for every entry of the source (entries
// of other bins fail the key tests).  r1 is how many entries bin b1
// contributes.  The survivors are then the entries with key > *kstar, or
// key == *kstar at a position <= *pstar.  Run by one whole CTA of kThreads.
template <typename ForEach>
__device__ __forceinline__ void kth_in_bin(ResolveSmem &S, ForEach for_each, uint32_t b1,
                                           uint32_t r1, uint32_t *kstar_out,
                                           int32_t *pstar_out) {
  uint32_t *sh = S.sh;
  find_bin<kHistBins, true>(sh, r1, S.warp_sums, &S.s_bin, &S.s_before);
  const uint32_t b2 = (uint32_t)S.s_bin;
  const uint32_t r2 = r1 - S.s_before;
  const uint32_t hi20 = (b1 << 12) | b2;   // bits 31..8 of K*

  // level 3: bits 7..0 among keys whose bits 31..8 are hi20
  for (int i = threadIdx.x; i < kThreads; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  for_each([&](uint32_t key, int32_t) {
    if ((key >> 8) == hi20) atomicAdd(&sh[key & 0xFFu], 1u);
  });
  __syncthreads();
  // 256 bins padded with zero bins to the block size; walking down from the
  // top passes the zero bins first
  find_bin<kThreads, true>(sh, r2, S.warp_sums, &S.s_bin, &S.s_before);
  const uint32_t b3 = (uint32_t)S.s_bin;
  const uint32_t r3 = r2 - S.s_before;   // how many elements equal to K* to keep
  const uint32_t m_eq = sh[b3];          // how many elements equal K*
  const uint32_t kstar = (hi20 << 8) | b3;

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
      for_each([&](uint32_t key, int32_t pos) {
        if (key == kstar) {
          const uint32_t p = (uint32_t)pos;
          const uint32_t hi_bits = lvl == 0 ? 0u : (p >> (sft + widths[lvl]));
          if (hi_bits == prefix) atomicAdd(&sh[(p >> sft) & (nb - 1)], 1u);
        }
      });
      __syncthreads();
      // ascending walk over max(nb, blockDim) bins (extra bins are zero)
      if (nb == 2048) find_bin<2048, false>(sh, need, S.warp_sums, &S.s_bin, &S.s_before);
      else find_bin<1024, false>(sh, need, S.warp_sums, &S.s_bin, &S.s_before);
      need -= S.s_before;
      prefix = (prefix << widths[lvl]) | (uint32_t)S.s_bin;
    }
    pstar = (int32_t)prefix;
  }
  *kstar_out = kstar;
  *pstar_out = pstar;
}

// Resolves row t once its collect pass is complete.  b1 and n_gt (the count
// above bin b1) come from the caller's threshold_bin, n_list (entries at or
// above bin b1) from the done counter.  Two more radix levels over the
// bin-b1 entries give the exact k-th key K*, a radix select over positions
// breaks ties toward lower positions, and an ordered compaction writes the k
// survivors in ascending position order.  The first pass copies the list
// into `lc` (kListCache entries of dynamic shared memory) when it fits, so
// the later passes read shared memory.  Run by one whole CTA of kThreads.
// The output entry of position pos of row t: its slot through the block
// table (paged caches), else pos + the row's index base.
template <bool PAGED>
__device__ __forceinline__ int32_t slot_of(const PageMap &pm, int t, int32_t pos, int32_t base) {
  if constexpr (!PAGED) {
    return pos + base;
  } else {
    return pm.table[(size_t)t * pm.max_pages + pos / pm.page_size] * pm.page_size +
           pos % pm.page_size;
  }
}

template <bool PAGED>
__device__ __noinline__ void resolve_row(int t, ResolveSmem &S, uint2 *lc, uint32_t b1,
                                         uint32_t n_gt, uint32_t n_list,
                                         const float *__restrict__ scores, int64_t ld, int64_t L,
                                         int k, int chunk, int max_chunks,
                                         const int32_t *__restrict__ index_base,
                                         const uint2 *__restrict__ list,
                                         const uint2 *__restrict__ tab, int32_t *__restrict__ idx,
                                         int32_t *__restrict__ lens, int32_t *err_flag) {
  uint32_t *sh = S.sh;
  const PageMap &pm = S.pm;   // paged caches only
  const int32_t base = index_base ? index_base[t] : 0;
  int32_t *out = idx + (size_t)t * k;
  if (n_gt >= (uint32_t)k || n_list < (uint32_t)k) {
    // histogram and scores disagree (a histogram of other scores, or NaNs)
    if (threadIdx.x == 0) raise_flag(err_flag, DSA_DEVERR_INDEX_RANGE);
    for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = -1;
    if (lens && threadIdx.x == 0) lens[t] = 0;
    return;
  }
  Source src;
  src.cache = nullptr;
  src.list = list + (size_t)t * kListCap;
  src.row = scores + (int64_t)t * ld;
  src.from_row = n_list > (uint32_t)kListCap;
  src.n = src.from_row ? L : (int64_t)n_list;
  const bool to_cache = !src.from_row && n_list <= (uint32_t)kListCache;
  const uint32_t r1 = (uint32_t)k - n_gt;  // to take from bin b1
  const int nch = (int)((L + chunk - 1) / chunk);
  const uint2 *rt = tab + (size_t)t * max_chunks;
  // the first group of the chunk table, loaded now, used by the compaction
  uint2 run0 = make_uint2(0u, 0u);
  if (!src.from_row && (int)threadIdx.x < min(nch, kThreads)) run0 = __ldcg(rt + threadIdx.x);
  // With the list copied and at most kThreads chunks, the copy is made in
  // position order: run c (chunk c) goes to the ordered offsets [pre(c),
  // pre(c + 1)), pre by a block scan in chunk order (so already sorted), and
  // ordered slot o takes the entry at its run's list start plus o - pre(c),
  // its run found by a binary search over pre (an empty run shares its pre
  // with the next run and is never the last one at or before o).
  const bool ordered = to_cache && nch <= kThreads;
  if (ordered) {
    uint32_t tot_runs;
    const uint32_t pre = block_excl_scan(run0.y, S.warp_sums, &tot_runs);
    S.run_at[threadIdx.x] = run0.x;
    S.run_pre[threadIdx.x] = pre;
    __syncthreads();
  }

  // level 2: bits 19..8 of the bin-b1 keys; the same pass copies the list
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  for (int64_t i0 = 0; i0 < src.n; i0 += (int64_t)kBatch * kThreads) {
    uint32_t key[kBatch];
    int32_t pos[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t i = i0 + (int64_t)j * kThreads + threadIdx.x;   // ordered slot, if ordered
      key[j] = 0;
      pos[j] = -1;                       // -1: past the end
      if (i < src.n) {
        if (ordered) {
          int lo = 0, hi = nch;          // the last run c with pre(c) <= i
          while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (S.run_pre[mid] <= (uint32_t)i) lo = mid; else hi = mid;
          }
          src.get(S.run_at[lo] + ((uint32_t)i - S.run_pre[lo]), key[j], pos[j]);
        } else {
          src.get(i, key[j], pos[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t i = i0 + (int64_t)j * kThreads + threadIdx.x;
      if (pos[j] >= 0) {
        if (to_cache) lc[i] = make_uint2(key[j], (uint32_t)pos[j]);
        if ((key[j] >> 20) == b1) atomicAdd(&sh[(key[j] >> 8) & 0xFFFu], 1u);
      }
    }
  }
  __syncthreads();
  if (to_cache) src.cache = lc;
  auto for_each = [&](auto f) {   // every (key, position): the shared copy, else via src
    if (src.cache) {
      const int n = (int)src.n;
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint2 e = src.cache[i];
        f(e.x, (int32_t)e.y);
      }
    } else {
      for (int64_t i = threadIdx.x; i < src.n; i += kThreads) {
        uint32_t key; int32_t pos;
        src.get(i, key, pos);
        f(key, pos);
      }
    }
  };
  uint32_t kstar;
  int32_t pstar;
  kth_in_bin(S, for_each, b1, r1, &kstar, &pstar);

  // ordered compaction of the survivors: key > K*, or key == K* at a
  // position <= pstar.  A thread takes kGather consecutive entries of the
  // ordered sequence per round; a block scan of its survivor count gives
  // where they go.
  uint32_t written = 0;
  if (ordered) {
    // the copy is in position order: one pass, kGather consecutive entries a thread
    const uint32_t n = (uint32_t)src.n;
    for (uint32_t r0 = 0; r0 < n; r0 += (uint32_t)kGather * kThreads) {
      const uint32_t l0 = r0 + (uint32_t)kGather * threadIdx.x;
      uint32_t m = 0;
      int32_t posv[kGather];
#pragma unroll
      for (int j = 0; j < kGather; ++j) {
        posv[j] = 0;
        if (l0 + j < n) {
          const uint2 e = lc[l0 + j];
          posv[j] = (int32_t)e.y;
          if (e.x > kstar || (e.x == kstar && (int32_t)e.y <= pstar)) m |= 1u << j;
        }
      }
      uint32_t tot;
      uint32_t o = written + block_excl_scan((uint32_t)__popc(m), S.warp_sums, &tot);
#pragma unroll
      for (int j = 0; j < kGather; ++j)
        if ((m >> j) & 1u) {
          if (o < (uint32_t)k) out[o] = slot_of<PAGED>(pm, t, posv[j], base);
          ++o;
        }
      written += tot;
    }
  } else if (src.from_row) {
    for (int64_t r0 = 0; r0 < L; r0 += (int64_t)kGather * kThreads) {
      const int64_t p0 = r0 + (int64_t)kGather * threadIdx.x;
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < kGather; ++j) {
        if (p0 + j < L) {
          const uint32_t key = score_key(__ldcg(src.row + p0 + j));
          if (key > kstar || (key == kstar && (int32_t)(p0 + j) <= pstar)) m |= 1u << j;
        }
      }
      uint32_t tot;
      uint32_t o = written + block_excl_scan((uint32_t)__popc(m), S.warp_sums, &tot);
#pragma unroll
      for (int j = 0; j < kGather; ++j)
        if ((m >> j) & 1u) {
          if (o < (uint32_t)k) out[o] = slot_of<PAGED>(pm, t, (int32_t)(p0 + j), base);
          ++o;
        }
      written += tot;
    }
  } else {
    for (int g0 = 0; g0 < nch; g0 += kThreads) {
      // the runs of chunks g0 .. g0 + ng - 1, their ordered starts by a block scan
      const int ng = min(kThreads, nch - g0);
      uint2 run = g0 == 0 ? run0 : make_uint2(0u, 0u);
      if (g0 > 0 && (int)threadIdx.x < ng) run = __ldcg(rt + g0 + threadIdx.x);
      uint32_t n_group;
      const uint32_t pre = block_excl_scan(run.y, S.warp_sums, &n_group);
      S.run_pre[threadIdx.x] = pre;
      S.run_at[threadIdx.x] = run.x;
      __syncthreads();
      for (uint32_t r0 = 0; r0 < n_group; r0 += (uint32_t)kGather * kThreads) {
        const uint32_t l0 = r0 + (uint32_t)kGather * threadIdx.x;
        // list slots of this thread's entries (shared memory only), then all
        // loads at once, then the tests
        uint32_t at[kGather];
        if (l0 < n_group) {
          // the last run starting at or before l0 (runs are non-empty there)
          int lo = 0, hi = ng;
          while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (S.run_pre[mid] <= l0) lo = mid; else hi = mid;
          }
          int c = lo;
#pragma unroll
          for (int j = 0; j < kGather; ++j) {
            const uint32_t l = l0 + j;
            at[j] = 0xffffffffu;
            if (l < n_group) {
              while (c + 1 < ng && S.run_pre[c + 1] <= l) ++c;
              at[j] = S.run_at[c] + (l - S.run_pre[c]);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < kGather; ++j) at[j] = 0xffffffffu;
        }
        uint2 e[kGather];
#pragma unroll
        for (int j = 0; j < kGather; ++j)
          e[j] = at[j] == 0xffffffffu ? make_uint2(0u, 0u)
                 : src.cache    ? src.cache[at[j]]
                                : __ldcg(src.list + at[j]);
        uint32_t m = 0;
        int32_t posv[kGather];
#pragma unroll
        for (int j = 0; j < kGather; ++j) {
          posv[j] = (int32_t)e[j].y;
          if (at[j] != 0xffffffffu && (e[j].x > kstar || (e[j].x == kstar && (int32_t)e[j].y <= pstar)))
            m |= 1u << j;
        }
        uint32_t tot;
        uint32_t o = written + block_excl_scan((uint32_t)__popc(m), S.warp_sums, &tot);
#pragma unroll
        for (int j = 0; j < kGather; ++j)
          if ((m >> j) & 1u) {
            if (o < (uint32_t)k) out[o] = slot_of<PAGED>(pm, t, posv[j], base);
            ++o;
          }
        written += tot;
      }
      __syncthreads();   // run_pre / run_at are rewritten by the next group
    }
  }
  if (threadIdx.x == 0) {
    if (written != (uint32_t)k) raise_flag(err_flag, DSA_DEVERR_INDEX_RANGE);
    if (lens) lens[t] = k;
  }
}

// This thread's positions of NR rounds starting at lo, as score keys:
// position lo + r * kRound + kPer * threadIdx.x + e (round r < NR, e < kPer),
// so the order (r, thread, e) is position order.  Positions at or past hi
// read as 0; callers test p < hi.
template <int NR, typename Pos>
__device__ __forceinline__ void load_round_keys(const float *row, Pos lo, Pos hi, bool vec,
                                                uint32_t (&v)[NR][kPer]) {
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const Pos p = lo + (Pos)(r * kRound) + (Pos)(kPer * threadIdx.x);
    if (vec && p + kPer <= hi) {
      const float4 *q = reinterpret_cast<const float4 *>(row + p);
#pragma unroll
      for (int c = 0; c < kPer / 4; ++c) {
        const float4 f = __ldcg(q + c);
        v[r][4 * c] = __float_as_uint(f.x);
        v[r][4 * c + 1] = __float_as_uint(f.y);
        v[r][4 * c + 2] = __float_as_uint(f.z);
        v[r][4 * c + 3] = __float_as_uint(f.w);
      }
    } else {
#pragma unroll
      for (int e = 0; e < kPer; ++e) v[r][e] = p + e < hi ? __float_as_uint(__ldcg(row + p + e)) : 0u;
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int e = 0; e < kPer; ++e) v[r][e] = score_key(__uint_as_float(v[r][e]));
}

// Collect pass, and the resolve of each row by the last of its CTAs to finish
// (every CTA fences its writes and bumps the row's done counter; the CTA that
// sees the count complete resolves the row -- nobody waits on anybody).
// CTA (x, t) covers positions [x * chunk, (x + 1) * chunk) of row t, chunk <=
// kMaxChunk: thread i holds positions x * chunk + r * kRound + 16 i + e
// (round r < 2, e < 16), so the order (r, i, e) is position order and a
// packed two-round block scan places every entry of the CTA's run.
template <bool PAGED>
__global__ void __launch_bounds__(kThreads, 2)
topk_collect_kernel(const float *__restrict__ scores, int64_t ld,
                    const int32_t *__restrict__ row_len, int k, int chunk, int nch, int max_chunks,
                    const int32_t *__restrict__ index_base, const uint32_t *__restrict__ hist,
                    uint32_t *__restrict__ cnt, uint2 *__restrict__ list,
                    uint2 *__restrict__ tab, int32_t *__restrict__ idx,
                    int32_t *__restrict__ lens, int32_t *err_flag, const PageMap pages) {
  __shared__ ResolveSmem S;
  __shared__ uint32_t s_base;
  __shared__ int s_last;
  __shared__ uint32_t s_total;
  extern __shared__ uint2 list_cache[];   // kListCache entries, used by the resolving CTA
  if (PAGED && threadIdx.x == 0) S.pm = pages;   // read by the resolve, after later barriers
  pdl_wait();      // scores and histogram come from the previous kernel
  pdl_trigger();
  // 1-D grid of rows x chunks (a 2-D grid would cap the rows at 65535)
  const int t = (int)(blockIdx.x / (unsigned)nch);
  const int c = (int)(blockIdx.x - (unsigned)t * (unsigned)nch);
  const int64_t L = max(row_len[t], 0);
  if (L <= k) {                     // every position is selected: no search
    if (c == 0) {
      const int32_t base = index_base ? index_base[t] : 0;
      int32_t *out = idx + (size_t)t * k;
      for (int j = threadIdx.x; j < k; j += blockDim.x)
        out[j] = j < L ? slot_of<PAGED>(pages, t, (int32_t)j, base) : -1;
      if (lens && threadIdx.x == 0) lens[t] = (int32_t)L;
    }
    return;
  }
  const int64_t lo = (int64_t)c * chunk;
  if (lo >= L) return;
  const int64_t hi = min(L, lo + chunk);
  const float *row = scores + (int64_t)t * ld;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;

  // this row's histogram slice first
  const HistSlice hs = hist_load(hist + (size_t)t * kHistBins);
  if (threadIdx.x == 0) { S.s_bin = 0; S.s_before = 0; }
  __syncthreads();
  threshold_bin(hs, (uint32_t)k, S.warp_sums, &S.s_bin, &S.s_before);
  const uint32_t b1 = (uint32_t)S.s_bin;
  const uint32_t n_gt = S.s_before;
  // this thread's scores (after the threshold, whose histogram loads then
  // do not queue behind them)
  uint32_t v[kRounds][kPer];
  load_round_keys<kRounds>(row, lo, hi, vec, v);

  // entries at or above bin b1, counted per round (packed: a round holds at
  // most 8192 of them, so the two 16-bit halves of the scan never carry)
  uint32_t m[kRounds];
  uint32_t packed = 0;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int64_t p = lo + (int64_t)r * kRound + kPer * threadIdx.x;
    m[r] = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if (p + e < hi && (v[r][e] >> 20) >= b1) m[r] |= 1u << e;
    packed += (uint32_t)__popc(m[r]) << (16 * r);
  }
  uint32_t tot;
  const uint32_t pre = block_excl_scan(packed, S.warp_sums, &tot);
  const uint32_t tot0 = tot & 0xffffu;
  const uint32_t n_cta = tot0 + (tot >> 16);
  if (threadIdx.x == 0) {
    s_base = n_cta ? atomicAdd(&cnt[4 * t], n_cta) : 0u;
    tab[(size_t)t * max_chunks + c] = make_uint2(s_base, n_cta);
  }
  __syncthreads();
  uint2 *cl = list + (size_t)t * kListCap;
#pragma unroll
  for (int r = 0; r < kRounds; ++r) {
    const int64_t p = lo + (int64_t)r * kRound + kPer * threadIdx.x;
    uint32_t o = s_base + (r == 0 ? (pre & 0xffffu) : tot0 + (pre >> 16));
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if ((m[r] >> e) & 1u) {
        if (o < (uint32_t)kListCap) cl[o] = make_uint2(v[r][e], (uint32_t)(p + e));
        ++o;
      }
  }

  // publish this CTA's run; the last CTA of the row resolves it
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    // one 64-bit word per row: CTAs done (high half) and entries appended
    // (low half), so the last CTA learns the row's total from its own atomic
    const uint32_t nch = (uint32_t)((L + chunk - 1) / chunk);
    const unsigned long long old = atomicAdd(
        reinterpret_cast<unsigned long long *>(cnt + 4 * t + 2), (1ull << 32) | n_cta);
    s_last = (uint32_t)(old >> 32) == nch - 1;
    s_total = (uint32_t)old + n_cta;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  resolve_row<PAGED>(t, S, list_cache, b1, n_gt, s_total, scores, ld, L, k, chunk, max_chunks,
              index_base, list, tab, idx, lens, err_flag);
}

// Cluster path: a row of at most kMaxCluster chunks is selected by one
// thread-block cluster (CTA rank c covers chunk c: R rounds of kRound
// positions) whose CTAs exchange through distributed shared memory instead
// of a list in global memory:
//   1. every CTA finds b1 from the row's histogram and reads its chunk once;
//      each thread keeps two masks of its positions per round (bin above b1,
//      bin b1) and puts its bin-b1 entries in its CTA's shared memory; the
//      CTA then copies them into the leader's (rank 0) shared memory, into
//      chunk c's region of the candidate buffer, and counts them in the
//      leader's level-2 histogram (bits 19..8) by remote reductions;
//   2. the leader finds the k-th entry (K*, p*) with kth_in_bin over its own
//      shared memory and stores it into every CTA of the row;
//   3. every CTA counts its survivors (key > K*, or key == K* at a position
//      <= p*), stores the count into the CTAs of later chunks, and writes its
//      survivors in position order after those of the earlier chunks.
// When a chunk has more bin-b1 entries than its region holds (many equal or
// near-equal scores), the leader resolves the row alone from its scores (the
// collect kernel's slow path).  Every access to another CTA's shared memory
// lies between two cluster barriers, so no CTA leaves while another may
// still touch its shared memory.
constexpr int kMaxCluster = 8;      // CTAs a row (the portable cluster size)
constexpr int kCandTotal = 8192;    // bin-b1 entries of a row the leader holds (64 KB)
constexpr int kOwnCap = 2048;       // bin-b1 entries of one chunk (the region's size at most)
enum { kModeSplit = 0, kModeDone = 1 };

struct ClusterSmem {
  uint2 own[kOwnCap];               // this chunk's bin-b1 (key, position) entries by slot
  uint32_t n_cand;                  // this chunk's bin-b1 entries (slot counter)
  uint32_t cand_n[kMaxCluster];     // leader: each chunk's bin-b1 entries (stored by its CTA)
  uint32_t surv[kMaxCluster];       // survivors of each earlier chunk (stored by its CTA)
  uint32_t kstar;                   // the leader's decision, stored into every CTA
  int32_t pstar;
  int mode;
};

// Distributed shared memory: the address of this CTA's shared object p in
// the shared memory of cluster CTA `rank`, and stores / reductions there.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, unsigned rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_st(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_st(uint32_t a, uint2 v) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(v.x), "r"(v.y)
               : "memory");
}
__device__ __forceinline__ void cluster_add(uint32_t a, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
// A barrier over every thread of the cluster; shared-memory writes before
// the arrive (local or remote) are visible to every thread after the wait.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Issues this thread's loads of one round starting at p0 (positions p0 +
// kPer * threadIdx.x + e) as raw fp32 bits; positions at or past hl read as 0.
__device__ __forceinline__ void issue_round(const float *row, int p0, int hl, bool vec,
                                            uint32_t (&v)[kPer]) {
  const int p = p0 + kPer * (int)threadIdx.x;
  if (vec && p + kPer <= hl) {
    const float4 *q = reinterpret_cast<const float4 *>(row + p);
#pragma unroll
    for (int c = 0; c < kPer / 4; ++c) {
      const float4 f = __ldcg(q + c);
      v[4 * c] = __float_as_uint(f.x);
      v[4 * c + 1] = __float_as_uint(f.y);
      v[4 * c + 2] = __float_as_uint(f.z);
      v[4 * c + 3] = __float_as_uint(f.w);
    }
  } else {
#pragma unroll
    for (int e = 0; e < kPer; ++e) v[e] = p + e < hl ? __float_as_uint(__ldcg(row + p + e)) : 0u;
  }
}

template <bool PAGED, int R>
__global__ void __launch_bounds__(kThreads, 2)
topk_cluster_kernel(const float *__restrict__ scores, int64_t ld,
                    const int32_t *__restrict__ row_len, int max_len, int k, int nch, int cap,
                    const int32_t *__restrict__ index_base, const uint32_t *__restrict__ hist,
                    int32_t *__restrict__ idx, int32_t *__restrict__ lens, int32_t *err_flag,
                    const PageMap pages) {
  static_assert(R == 1 || R == 2, "one or two rounds a chunk");
  constexpr int kChunk = R * kRound;
  __shared__ ResolveSmem S;
  __shared__ ClusterSmem CS;
  // leader: the row's bin-b1 entries, `cap` per chunk (chunk j at j cap)
  extern __shared__ uint2 cand[];
  if (PAGED && threadIdx.x == 0) S.pm = pages;   // read by the slow path, after later barriers
  // 1-D grid of rows x chunks; the cluster of row t is CTAs [t nch, (t + 1) nch)
  const int t = (int)(blockIdx.x / (unsigned)nch);
  const int c = (int)(blockIdx.x - (unsigned)t * (unsigned)nch);   // the cluster rank
  pdl_wait();      // scores and histogram come from the previous kernel
  pdl_trigger();
  // positions fit 32 bits here: a row has at most kMaxCluster chunks
  const int lo = c * kChunk;
  const float *row = scores + (int64_t)t * ld;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  const int hl = min(max_len, lo + kChunk);   // loads stay inside the row's storage
  // the CTA's first reads at once (each is a long round trip): the row's
  // length, its histogram slice and the first two rounds of its chunk
  const int32_t len = row_len[t];
  const HistSlice hs = hist_load(hist + (size_t)t * kHistBins);
  uint32_t buf[2][kPer];
  issue_round(row, lo, hl, vec, buf[0]);
  if (R > 1) issue_round(row, lo + kRound, hl, vec, buf[1]);
  const int64_t L = max(len, 0);
  int32_t *out = idx + (size_t)t * k;
  const int32_t base = index_base ? index_base[t] : 0;
  if (L <= k) {                     // every position is selected; the whole cluster leaves
    if (c == 0) {
      for (int j = threadIdx.x; j < k; j += blockDim.x)
        out[j] = j < L ? slot_of<PAGED>(pages, t, (int32_t)j, base) : -1;
      if (lens && threadIdx.x == 0) lens[t] = (int32_t)L;
    }
    return;
  }
  const int hi = (int)min(L, (int64_t)(lo + kChunk));   // hi <= lo: the row ends before this chunk

  if (c == 0)   // the level-2 histogram the whole row adds into
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) S.sh[i] = 0;
  if (threadIdx.x == 0) {
    S.s_bin = 0;
    S.s_before = 0;
    CS.n_cand = 0;
  }
  cluster_arrive();   // 0: the leader's histogram is zero (waited for before the first add)
  __syncthreads();
  threshold_bin(hs, (uint32_t)k, S.warp_sums, &S.s_bin, &S.s_before);
  const uint32_t b1 = (uint32_t)S.s_bin;
  const uint32_t n_gt = S.s_before;
  cluster_wait();     // 0
  const uint32_t hist2 = cluster_addr(S.sh, 0);
  const uint32_t region = cluster_addr(cand + (size_t)c * cap, 0);
  // this thread's positions of round r: bin above b1 (bits 0..15 of mk[r])
  // and bin b1 (bits 16..31); the bin-b1 entries of a round get consecutive
  // slots (one shared atomic a warp).  Two rounds are in flight: round r + 2
  // is issued into round r's registers once r is done, and no key outlives
  // its round.
  static_assert(kPer == 16, "a round's two masks share one word");
  uint32_t mk[R];
  uint32_t slot0[R];
  const uint32_t key_lo = b1 << 20;            // keys of bin b1: [key_lo, key_lo + 2^20)
#pragma unroll
  for (int r = 0; r < R; ++r) {
    uint32_t(&v)[kPer] = buf[r & 1];
    const int p = lo + r * kRound + kPer * (int)threadIdx.x;
    const int nv = min(max(hi - p, 0), kPer);   // this thread's positions before hi
    const uint32_t valid = (nv == kPer ? 0xffffu : (1u << nv) - 1u) * 0x10001u;
    uint32_t m = 0;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      v[e] = score_key(__uint_as_float(v[e]));
      const uint32_t d = v[e] - key_lo;
      m |= (d >= (1u << 20) && v[e] > key_lo ? 1u : 0u) << e;   // bin above b1
      m |= (d < (1u << 20) ? 1u : 0u) << (16 + e);             // bin b1
    }
    mk[r] = m & valid;
    const uint32_t nb = (uint32_t)__popc(mk[r] >> 16);
    const unsigned lane = lane_id();
    uint32_t incl = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= (unsigned)o) incl += y;
    }
    uint32_t wbase = 0;
    if (lane == 31 && incl) wbase = atomicAdd(&CS.n_cand, incl);
    uint32_t slot = __shfl_sync(0xffffffffu, wbase, 31) + incl - nb;
    slot0[r] = slot;
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if ((mk[r] >> (16 + e)) & 1u) {
        if (slot < (uint32_t)cap) CS.own[slot] = make_uint2(v[e], (uint32_t)(p + e));
        ++slot;
      }
    if (r + 2 < R) issue_round(row, lo + (r + 2) * kRound, hl, vec, v);
  }
  // the chunk's bin-b1 entries into the leader: its region, and their
  // level-2 bins (one pass, a few entries a thread)
  __syncthreads();
  {
    const uint32_t n = min(CS.n_cand, (uint32_t)cap);
    for (uint32_t i = threadIdx.x; i < n; i += kThreads) {
      const uint2 e = CS.own[i];
      cluster_st(region + 8u * i, e);
      cluster_add(hist2 + 4u * ((e.x >> 8) & 0xFFFu), 1u);
    }
  }
  if (threadIdx.x == 0) cluster_st(cluster_addr(&CS.cand_n[c], 0), CS.n_cand);
  cluster_arrive();   // 1: the row's bin-b1 entries and their histogram are in the leader
  cluster_wait();

  if (c == 0) {
    // ------------------------------------------------ the leader: (K*, p*)
    uint32_t n1 = 0;
    bool ovf = false;
    for (int j = 0; j < nch; ++j) {
      n1 += CS.cand_n[j];
      ovf |= CS.cand_n[j] > (uint32_t)cap;
    }
    int mode = kModeSplit;
    uint32_t kstar = 0;
    int32_t pstar = 0;
    if (n_gt >= (uint32_t)k || n_gt + n1 < (uint32_t)k) {
      // histogram and scores disagree (a histogram of other scores, or NaNs)
      if (threadIdx.x == 0) raise_flag(err_flag, DSA_DEVERR_INDEX_RANGE);
      for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = -1;
      if (lens && threadIdx.x == 0) lens[t] = 0;
      mode = kModeDone;
    } else if (ovf) {
      // more near-equal scores than the regions hold: the row, read again
      resolve_row<PAGED>(t, S, cand, b1, n_gt, (uint32_t)kListCap + 1u, scores, ld, L, k,
                         kChunk, nch, index_base, nullptr, nullptr, idx, lens, err_flag);
      mode = kModeDone;
    } else {
      auto for_each = [&](auto f) {   // every bin-b1 entry of the row
        for (int j = 0; j < nch; ++j) {
          const uint2 *rg = cand + (size_t)j * cap;
          for (uint32_t i = threadIdx.x; i < CS.cand_n[j]; i += kThreads) {
            const uint2 e = rg[i];
            f(e.x, (int32_t)e.y);
          }
        }
      };
      kth_in_bin(S, for_each, b1, (uint32_t)k - n_gt, &kstar, &pstar);
    }
    if ((int)threadIdx.x < nch) {
      const unsigned dst = threadIdx.x;
      cluster_st(cluster_addr(&CS.kstar, dst), kstar);
      cluster_st(cluster_addr(&CS.pstar, dst), (uint32_t)pstar);
      cluster_st(cluster_addr(&CS.mode, dst), (uint32_t)mode);
    }
  }
  cluster_arrive();   // 2: the decision is in every CTA of the row
  cluster_wait();

  // ------------------------------------------------ survivors of this chunk
  // (in split mode no chunk overflowed, so every bin-b1 key is in CS.own)
  const bool split = CS.mode == kModeSplit;
  const uint32_t kstar = CS.kstar;
  const int32_t pstar = CS.pstar;
  uint32_t m[R];
  uint32_t packed = 0;   // round r's survivors in bits 16 r .. 16 r + 15
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int p = lo + r * kRound + kPer * (int)threadIdx.x;
    uint32_t slot = slot0[r];
    m[r] = split ? mk[r] & 0xffffu : 0u;
    uint32_t b = split ? mk[r] >> 16 : 0u;
    while (b) {
      const int e = __ffs(b) - 1;
      b &= b - 1;
      const uint32_t key = CS.own[slot++].x;
      if (key > kstar || (key == kstar && p + e <= pstar)) m[r] |= 1u << e;
    }
    packed += (uint32_t)__popc(m[r]) << (16 * r);   // a round holds at most 8192
  }
  uint32_t tot;
  const uint32_t pre = block_excl_scan(packed, S.warp_sums, &tot);
  const uint32_t n_surv = (tot & 0xffffu) + (tot >> 16);
  if ((int)threadIdx.x > c && (int)threadIdx.x < nch)
    cluster_st(cluster_addr(&CS.surv[c], (unsigned)threadIdx.x), n_surv);
  cluster_arrive();   // 3: every chunk has the survivor counts of the chunks before it
  cluster_wait();
  if (!split) return;
  uint32_t before = 0;
  for (int j = 0; j < c; ++j) before += CS.surv[j];
  uint32_t round_base = before;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int p = lo + r * kRound + kPer * (int)threadIdx.x;
    uint32_t o = round_base + ((pre >> (16 * r)) & 0xffffu);
    round_base += (tot >> (16 * r)) & 0xffffu;
    uint32_t b = m[r];
    while (b) {
      const int e = __ffs(b) - 1;
      b &= b - 1;
      if (o < (uint32_t)k) out[o] = slot_of<PAGED>(pages, t, p + e, base);
      ++o;
    }
  }
  if (c == nch - 1) {
    // the row's survivors number exactly k unless the histogram disagrees
    const uint32_t total = before + n_surv;
    for (uint32_t j = total + threadIdx.x; j < (uint32_t)k; j += blockDim.x) out[j] = -1;
    if (threadIdx.x == 0) {
      if (total != (uint32_t)k) raise_flag(err_flag, DSA_DEVERR_INDEX_RANGE);
      if (lens) lens[t] = k;
    }
  }
}

__global__ void __launch_bounds__(256) zero16_kernel(uint4 *p, size_t n16) {
  pdl_trigger();
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Positions per collect CTA: the smallest power of two in [kMinChunk,
// kMaxChunk] whose grid fits in one wave (two CTAs per SM); kMaxChunk when
// none does.
int collect_chunk(int T, int64_t max_len) {
  const int64_t wave = 2LL * num_sms();
  int64_t chunk = kMinChunk;
  while (chunk < kMaxChunk && (int64_t)T * ((max_len + chunk - 1) / chunk) > wave) chunk <<= 1;
  return (int)chunk;
}

// Rounds a CTA of the cluster path covers: the fewest R in {1, 2} with at
// most kMaxCluster CTAs a row and a grid of at most one CTA an SM (so every
// cluster is resident at once); 0 when neither fits -- long rows or many
// rows, where the collect kernel's wide first pass is faster -- and those
// rows take the collect kernel.
int cluster_rounds(int T, int64_t max_len) {
  for (int R = 1; R <= 2; ++R) {
    const int64_t nch = (max_len + (int64_t)R * kRound - 1) / ((int64_t)R * kRound);
    if (nch <= kMaxCluster && (int64_t)T * nch <= num_sms()) return R;
  }
  return 0;
}

}  // namespace

size_t topk_ws_layout(int T, int64_t max_len, int k, void *ws, TopkWs *out) {
  (void)k;
  WsCarver c(ws);
  TopkWs w;
  w.max_chunks = (int)std::max<int64_t>(1, (max_len + kMinChunk - 1) / kMinChunk);
  w.hist = c.take<uint32_t>((size_t)T * kHistBins);   // hist then cnt, adjacent (one memset clears both)
  w.cnt = c.take<uint32_t>((size_t)T * 4);   // list entries, -, (entries | CTAs done << 32) as u64
  w.list = c.take<uint2>((size_t)T * kListCap);
  w.tab = c.take<uint2>((size_t)T * w.max_chunks);
  if (out) *out = w;
  return c.bytes();
}

cudaError_t topk_clear(const TopkWs &w, int T, cudaStream_t s) {
  // hist and cnt are adjacent in the workspace (topk_ws_layout) and their
  // size is a multiple of 16 bytes: one grid-stride kernel, which the next
  // kernel (launched as its dependent) may overlap
  const char *end = reinterpret_cast<const char *>(w.cnt + (size_t)T * 4);
  const size_t n16 = (size_t)(end - reinterpret_cast<const char *>(w.hist)) / 16;
  const unsigned blocks = (unsigned)std::min<size_t>((n16 + 255) / 256, 4 * (size_t)num_sms());
  zero16_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<uint4 *>(w.hist), n16);
  return cudaGetLastError();
}

cudaError_t topk_hist(const float *scores, int64_t ld, const int32_t *row_len, int T,
                      int64_t max_len, int k, const TopkWs &w, cudaStream_t s) {
  if (max_len <= k) return cudaSuccess;
  const int chunk = collect_chunk(T, max_len);
  const int64_t nch = (max_len + chunk - 1) / chunk;
  if (nch * T >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
  topk_hist_kernel<<<(unsigned)(nch * T), kHistThreads, 0, s>>>(scores, ld, row_len, k, chunk,
                                                                  (int)nch, w.hist);
  return cudaGetLastError();
}

cudaError_t topk_select(const float *scores, int64_t ld, const int32_t *row_len, int T,
                        int64_t max_len, int k, const int32_t *index_base, int32_t *idx,
                        int32_t *lens, const TopkWs &w, int32_t *err_flag, cudaStream_t s,
                        const PageMap &pages) {
  const int R = max_len > k ? cluster_rounds(T, max_len) : 0;
  if (R > 0) {
    const int64_t cn = (max_len + (int64_t)R * kRound - 1) / ((int64_t)R * kRound);
    if (cn * T >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
    const int cap = std::min(kOwnCap, kCandTotal / (int)cn);
    const bool pg = pages.table != nullptr;
    auto kern = R == 1 ? (pg ? topk_cluster_kernel<true, 1> : topk_cluster_kernel<false, 1>)
                       : (pg ? topk_cluster_kernel<true, 2> : topk_cluster_kernel<false, 2>);
    // static + dynamic shared memory pass the default 48 KB: opt in
    const size_t cdyn = sizeof(uint2) * (size_t)cap * (size_t)cn;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(uint2) * kCandTotal));
    if (e != cudaSuccess) return e;
    return launch_pdl_cluster(kern, dim3((unsigned)(cn * T)), dim3(kThreads), cdyn, s,
                              (unsigned)cn, scores, ld, row_len, (int)max_len, k, (int)cn, cap,
                              index_base,
                              (const uint32_t *)w.hist, idx, lens, err_flag, pages);
  }
  const int chunk = collect_chunk(T, max_len);
  const int64_t nch = max_len > k ? (max_len + chunk - 1) / chunk : 1;
  if (nch > w.max_chunks) return cudaErrorInvalidValue;
  if (nch * T >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)(nch * T));
  const size_t dyn = sizeof(uint2) * kListCache;
  auto kern = pages.table ? topk_collect_kernel<true> : topk_collect_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(kThreads), dyn, s, scores, ld, row_len, k, chunk, (int)nch,
                    w.max_chunks, index_base, (const uint32_t *)w.hist, w.cnt, w.list, w.tab, idx,
                    lens, err_flag, pages);
}

}  // namespace dsa
