// Lightning-indexer scores for query rows that share their keys (causal
// prefill: the rows of one segment all start at the segment's first key and
// differ by one key at the end).  The rows are taken four at a time: one
// 128-key tile of the index-k cache is the A operand (M = 128, K = d, loaded
// by TMA) against the B operand of the four rows' head rows (N = 4 x 64),
// so a key tile is read and multiplied once for four query rows.  The score
// definition is that of index_score.cu (the "scores" stage of tokenspeed PR
// #627): I[t,s] = sk[s] sum_h (w[t,h] sq[t,h]) ReLU(q8[t,h,:] . k8[s,:]).
//
// A group of four rows that all start at the same key is "shared": its
// units are the key tiles of the union of the rows' ranges, and each row
// keeps the keys of its own range.  Otherwise (a segment boundary inside the
// group, or rows of different requests) the group is "split": its units are
// each row's own tiles in turn, each unit keeping that one row's scores.
// Every CTA takes an equal share of the units.
//
// Two persistent CTAs per SM, each holding half of TMEM: while one CTA's
// epilogue drains its accumulator the other's MMAs run.  Warp 0 issues the
// TMA loads (four stages of key tiles, the group's q rows, the key scales),
// warp 1 the tcgen05.mma (kind::f8f6f4 or kind::f16) into a 4 N-column
// accumulator of four sub-slots, and eight epilogue warps (two groups, each
// with a warp per TMEM lane quadrant; group e takes rows 2e and 2e+1) drain
// it: per row, the N head columns in chunks of 16, the next chunk's load in
// flight while this one is reduced, weighted by the row's head weights
// (w * sq, in shared memory) after ReLU.  Every wait is bounded.
//
// Measured alternatives, slower on GB300: one CTA per SM holding all of TMEM
// as two accumulator sets (the MMA of the next unit overlapping this unit's
// epilogue), with eight or sixteen epilogue warps; and one epilogue group of
// four warps.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace dsa {

namespace {

constexpr int kGTileKeys = 128;
constexpr int kGRows = 4;                // query rows per group
constexpr int kGEpiThreads = 256;        // two groups of four warps, two rows each
constexpr int kGThreads = 64 + kGEpiThreads;
constexpr int kGCtasPerSm = 2;
constexpr int kGStages = 4;              // key tiles in flight
constexpr int kGScBox = 132;             // fp32 scales per tile load: 128 keys + up to 3 lead-in
constexpr int kGScBytes = 640;           // kGScBox * 4 rounded up to 128
constexpr int kGScSlots = 8;

struct GSmem {
  uint32_t stage0, stage_bytes, q0, q_bytes, wq, sc, bars, total;
};

// N: head rows of one query (H_I rounded up to 16, 32 or 64)
__host__ __device__ inline GSmem gsmem_layout(int N) {
  GSmem L;
  L.stage_bytes = kGTileKeys * 128;
  L.stage0 = 0;
  L.q0 = L.stage0 + L.stage_bytes * kGStages;
  L.q_bytes = kGRows * N * 128;          // a multiple of 1024 for N >= 16
  L.wq = L.q0 + L.q_bytes;             // one query slot: groups change every few hundred tiles
  L.sc = L.wq + kGRows * N * 4;
  L.bars = L.sc + kGScSlots * kGScBytes;
  L.total = L.bars + 640;
  return L;
}

// The key range of query row t: [r0, r0 + len) (len 0 for a bad range,
// which the first CTA reports).
struct GRow {
  int32_t r0, len;
  bool bad;
};
__device__ __forceinline__ GRow grow(const IndexScoreArgs &a, int t) {
  GRow r;
  const int64_t s = a.row_start[t], e = a.row_end[t];
  r.bad = s < 0 || e < s || e > a.k_rows;
  r.r0 = (int32_t)s;
  r.len = r.bad ? 0 : (int32_t)(e - s);
  return r;
}

struct Group {
  int32_t r0, len;                   // shared: the union of the rows' ranges
  bool shared;
  int32_t rs[kGRows], re[kGRows];    // row q keeps the keys [rs, re)
};
__device__ __forceinline__ Group group_of(const IndexScoreArgs &a, int g) {
  Group G;
  int32_t lo = INT32_MAX, hi = INT32_MIN;
#pragma unroll
  for (int q = 0; q < kGRows; ++q) {
    const int t = g * kGRows + q;
    int32_t rs = 0, re = 0;
    if (t < a.T) {
      const GRow r = grow(a, t);
      if (r.len > 0) {
        rs = r.r0;
        re = r.r0 + r.len;
        lo = min(lo, rs);
        hi = max(hi, re);
      }
    }
    G.rs[q] = rs;
    G.re[q] = re;
  }
  G.r0 = lo <= hi ? lo : 0;
  G.len = lo <= hi ? hi - lo : 0;
  G.shared = true;
#pragma unroll
  for (int q = 0; q < kGRows; ++q)
    if (G.re[q] > G.rs[q] && G.rs[q] != G.r0) G.shared = false;
  return G;
}
__device__ __forceinline__ int64_t units_of(const Group &G) {
  if (G.shared) return (G.len + kGTileKeys - 1) / kGTileKeys;
  int64_t n = 0;
#pragma unroll
  for (int q = 0; q < kGRows; ++q) n += (G.re[q] - G.rs[q] + kGTileKeys - 1) / kGTileKeys;
  return n;
}

// A CTA's units in group-major order; next() only while units remain.
struct GIter {
  int g;
  int64_t j, n;
  Group G;
  int32_t y;    // first key slot of the unit's tile
  int qsel;     // split group: the one row the unit scores; shared: -1
  __device__ __forceinline__ void locate() {
    if (G.shared) {
      qsel = -1;
      y = G.r0 + (int32_t)j * kGTileKeys;
      return;
    }
    int64_t jj = j;
#pragma unroll
    for (int q = 0; q < kGRows; ++q) {
      const int64_t nt = (G.re[q] - G.rs[q] + kGTileKeys - 1) / kGTileKeys;
      if (jj >= 0 && jj < nt) {
        qsel = q;
        y = G.rs[q] + (int32_t)jj * kGTileKeys;
      }
      jj -= nt;
    }
  }
  __device__ __forceinline__ void start(const IndexScoreArgs &a, int g0, int64_t j0) {
    g = g0;
    j = j0;
    G = group_of(a, g);
    n = units_of(G);
    locate();
  }
  __device__ __forceinline__ void next(const IndexScoreArgs &a) {
    if (++j == n) {
      j = 0;
      do {
        ++g;
        G = group_of(a, g);
        n = units_of(G);
      } while (n == 0);
    }
    locate();
  }
};

// W consecutive fp32 columns (W = 16 or 32) of this thread's TMEM lane, issued
// without waiting; tmem_wait_regs completes them.
template <int W>
__device__ __forceinline__ void tmem_issue(uint32_t taddr, uint32_t (&r)[W]) {
  if constexpr (W == 32) tc::tmem_ld_x32(taddr, r);
  else tc::tmem_ld_x16(taddr, r);
}
// Waits for this thread's TMEM loads.  The registers pass through empty asm
// statements after the wait, so no use of them is scheduled above it.
template <int W>
__device__ __forceinline__ void tmem_wait_regs(uint32_t (&r)[W]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < W; i += 8)
    asm volatile("" : "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]),
                 "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7]));
}
// p[e % 4] += w[e] * ReLU(d[e]) over W columns (p as two pairs): four
// independent chains, two lanes of each packed fma
template <int W>
__device__ __forceinline__ void relu_dot(const uint32_t (&d)[W], const float *w, float2 (&p)[2]) {
  const float4 *w4 = reinterpret_cast<const float4 *>(w);
#pragma unroll
  for (int i = 0; i < W / 4; ++i) {
    const float4 wv = w4[i];     // the same address in every lane: a broadcast
    const float2 r0 = make_float2(fmaxf(__uint_as_float(d[4 * i + 0]), 0.f),
                                  fmaxf(__uint_as_float(d[4 * i + 1]), 0.f));
    const float2 r1 = make_float2(fmaxf(__uint_as_float(d[4 * i + 2]), 0.f),
                                  fmaxf(__uint_as_float(d[4 * i + 3]), 0.f));
    p[0] = __ffma2_rn(make_float2(wv.x, wv.y), r0, p[0]);
    p[1] = __ffma2_rn(make_float2(wv.z, wv.w), r1, p[1]);
  }
}

// The TMEM accumulator: four sub-slots of N columns.  A unit of a split
// group takes the next sub-slot in turn (its one row's N columns); a unit of
// a shared group takes all four (row q in sub-slot q).  Walked alike by the
// MMA issuer and the epilogue.
struct SubSlots {
  int ptr = 0;          // the next sub-slot of a split unit
  uint32_t par = 0;     // bit s: sub-slot s's phase
  __device__ __forceinline__ uint32_t mask(int qsel) const { return qsel >= 0 ? (1u << ptr) : 0xFu; }
  __device__ __forceinline__ uint32_t parity(int s) const { return (par >> s) & 1u; }
  __device__ __forceinline__ void advance(int qsel) {
    if (qsel >= 0) {
      par ^= 1u << ptr;
      ptr = (ptr + 1) & 3;
    } else {
      par ^= 0xFu;
    }
  }
};

template <bool FP8, int N>
__global__ void __launch_bounds__(kGThreads, kGCtasPerSm)
index_score_groups_kernel(const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap qmap,
                          const __grid_constant__ CUtensorMap smap, IndexScoreArgs a) {
  constexpr int NT = kGRows * N;        // MMA N of a shared unit: the group's head rows
  constexpr uint32_t kTmemCols = NT < 32 ? 32 : NT;
  constexpr int CW = 16;                // TMEM columns per load
  constexpr int kCpr = N / CW;          // loads per row
  extern __shared__ unsigned char smem_raw[];
  const GSmem L = gsmem_layout(N);
  unsigned char *base = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + L.bars);
  uint64_t *full = bars;                 // [kGStages]
  uint64_t *empty = bars + 4;            // [kGStages]
  uint64_t *scfull = bars + 8;           // [kGScSlots]
  uint64_t *scempty = bars + 16;         // [kGScSlots]
  uint64_t *qfull = bars + 24;
  uint64_t *qempty = bars + 25;
  uint64_t *tfull = bars + 26;           // [4] sub-slots
  uint64_t *tempty = bars + 30;          // [4]
  uint64_t *done = bars + 34;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 35);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 36);
  float *wq_s = reinterpret_cast<float *>(base + L.wq);   // [kGRows][N] head weights
  const float *sc_s = reinterpret_cast<const float *>(base + L.sc);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGStages; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kGScSlots; ++i) {
      tc::mbar_init(&scfull[i], 1);
      tc::mbar_init(&scempty[i], 8);       // every epilogue warp reads every tile's scales
    }
    tc::mbar_init(qfull, 1);
    tc::mbar_init(qempty, 1);
    for (int i = 0; i < 4; ++i) {
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], 4);
    }
    tc::mbar_init(done, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();   // the row ranges and inputs may come from the previous kernel

  // ---- this CTA's equal share of the valid (group, key tile) units: every
  // thread sums the units of a run of groups, a block scan gives the total
  // and each run's start, and the run holding this CTA's first unit locates it
  __shared__ int64_t s_warp[kGThreads / 32];
  __shared__ int s_g0;
  __shared__ int64_t s_j0, s_count;
  {
    const int ngroups = (a.T + kGRows - 1) / kGRows;
    const int R = (ngroups + kGThreads - 1) / kGThreads;
    const int glo = min(ngroups, (int)threadIdx.x * R), ghi = min(ngroups, glo + R);
    int64_t mine = 0;
#pragma unroll 2
    for (int g = glo; g < ghi; ++g) mine += units_of(group_of(a, g));
    if (blockIdx.x == 0) {
      // a row range outside the cache is reported once, by the first CTA
      for (int t = glo * kGRows; t < min(a.T, ghi * kGRows); ++t)
        if (grow(a, t).bad) raise_flag(a.err_flag, DSA_DEVERR_INDEX_RANGE);
    }
    int64_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    if (threadIdx.x == 0) s_count = 0;
    __syncthreads();
    int64_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kGThreads / 32; ++w) {
      const int64_t x = s_warp[w];
      if (w < warp) before += x;
      total += x;
    }
    const int64_t pre = before + incl - mine;      // units before this thread's groups
    const int64_t u0 = total * (int64_t)blockIdx.x / gridDim.x;
    const int64_t u1 = total * ((int64_t)blockIdx.x + 1) / gridDim.x;
    if (u0 < u1 && pre <= u0 && u0 < pre + mine) {
      int64_t acc = pre;
      for (int g = glo; g < ghi; ++g) {
        const int64_t n = units_of(group_of(a, g));
        if (u0 < acc + n) {
          s_g0 = g;
          s_j0 = u0 - acc;
          s_count = u1 - u0;
          break;
        }
        acc += n;
      }
    }
    __syncthreads();
  }
  const int64_t count = s_count;
  const int g_first = count > 0 ? s_g0 : 0;
  const int64_t j_first = count > 0 ? s_j0 : 0;
  pdl_trigger();   // the next kernel may be placed as SMs free up; it waits for us

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::prefetch_tmap(&kmap);
      tc::prefetch_tmap(&qmap);
      if (FP8) tc::prefetch_tmap(&smap);
      // a segment's key tiles are read again by each of its groups: they
      // take the normal L2 policy (the score rows are written streaming)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t qphase = 0;
      int cur_g = -1;
      uint32_t issued = 0;         // bit i: stage i has had a load
      uint32_t last_phase = 0;     // bit i: parity of stage i's last load
      bool q_issued = false;
      int ss = 0;                  // scale slot (FP8)
      uint32_t sphase = 0;
      uint32_t s_issued = 0, s_last = 0;
      GIter it;
      if (count > 0) it.start(a, g_first, j_first);
      for (int64_t n = 0; n < count; ++n, (n < count ? it.next(a) : (void)0)) {
        if (it.g != cur_g) {
          if (cur_g >= 0) qphase ^= 1;
          if (!tc::mbar_wait(qempty, qphase ^ 1, abort_flag)) break;
          tc::mbar_arrive_expect_tx(qfull, L.q_bytes);
          // the group's rows, N head rows each, stacked as the NT rows of
          // the B operand (rows past T read as zeros)
          for (int q = 0; q < kGRows; ++q)
            tc::tma_load_2d(&qmap, qfull, base + L.q0 + q * N * 128, 0, (it.g * kGRows + q) * a.H_I);
          q_issued = true;
          cur_g = it.g;
        }
        if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag)) break;
        tc::mbar_arrive_expect_tx(&full[stage], L.stage_bytes);
        tc::tma_load_2d(&kmap, &full[stage], base + L.stage0 + stage * L.stage_bytes, 0, it.y);
        if (FP8) {
          // the 128 key scales, from the nearest 16-byte boundary at or below y,
          // into their own ring (held until the epilogue has read them)
          if (!tc::mbar_wait(&scempty[ss], sphase ^ 1, abort_flag)) break;
          tc::mbar_arrive_expect_tx(&scfull[ss], kGScBox * 4);
          tc::tma_load_1d(&smap, &scfull[ss], base + L.sc + ss * kGScBytes, it.y & ~3);
          s_issued |= 1u << ss;
          s_last = (s_last & ~(1u << ss)) | (sphase << ss);
          if (++ss == kGScSlots) {
            ss = 0;
            sphase ^= 1;
          }
        }
        issued |= 1u << stage;
        last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == kGStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      // every load this thread issued must land before the CTA exits
      for (int i = 0; i < kGStages; ++i)
        if (issued & (1u << i)) tc::mbar_wait_drain(&full[i], (last_phase >> i) & 1u);
      if (q_issued) tc::mbar_wait_drain(qfull, qphase);
      for (int i = 0; i < kGScSlots; ++i)
        if (s_issued & (1u << i)) tc::mbar_wait_drain(&scfull[i], (s_last >> i) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // one row's N head rows, or a shared group's NT
      constexpr uint32_t idesc_one =
          tc::idesc_f32acc(FP8 ? 0u : 1u, FP8 ? 0u : 1u, 0u, 0u, (uint32_t)N, 128u);
      constexpr uint32_t idesc_all =
          tc::idesc_f32acc(FP8 ? 0u : 1u, FP8 ? 0u : 1u, 0u, 0u, (uint32_t)NT, 128u);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t qphase = 0;
      int cur_g = -1;
      SubSlots sub;
      bool any = false;
      GIter it;
      if (count > 0) it.start(a, g_first, j_first);
      for (int64_t n = 0; n < count; ++n, (n < count ? it.next(a) : (void)0)) {
        if (it.g != cur_g) {
          if (cur_g >= 0) {
            tc::mma_commit(qempty);   // the query slot is free once the group's MMAs finish
            qphase ^= 1;
          }
          if (!tc::mbar_wait(qfull, qphase, abort_flag)) break;
          cur_g = it.g;
        }
        const int qsel = it.qsel;
        const uint32_t m = sub.mask(qsel);
        bool got = true;
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2)
          if ((m >> s2) & 1u) got = got && tc::mbar_wait(&tempty[s2], sub.parity(s2) ^ 1, abort_flag);
        if (!got) break;
        if (!tc::mbar_wait(&full[stage], phase, abort_flag)) break;
        tc::fence_after_sync();
        const uint32_t a_addr = tc::smem_u32(base + L.stage0 + stage * L.stage_bytes);
        const uint32_t b_addr = tc::smem_u32(base + L.q0) + (uint32_t)((qsel >= 0 ? qsel : 0) * N * 128);
        const uint32_t idesc = qsel >= 0 ? idesc_one : idesc_all;
        const uint32_t dcol = tmem_base + (uint32_t)(qsel >= 0 ? sub.ptr * N : 0);
        const uint64_t adesc0 = tc::sdesc_sw128(a_addr, 16, 1024);
        const uint64_t bdesc0 = tc::sdesc_sw128(b_addr, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // 32 bytes of K per instruction (K = 32 fp8 or 16 bf16)
          const uint64_t ad = adesc0 + ((kk * 32) >> 4);
          const uint64_t bd = bdesc0 + ((kk * 32) >> 4);
          if constexpr (FP8)
            tc::mma_f8f6f4(dcol, ad, bd, idesc, kk > 0 ? 1u : 0u);
          else
            tc::mma_f16(dcol, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&empty[stage]);
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2)
          if ((m >> s2) & 1u) tc::mma_commit(&tfull[s2]);
        sub.advance(qsel);
        any = true;
        if (++stage == kGStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (any) {
        // all MMAs retired before TMEM is released
        tc::mma_commit(done);
        tc::mbar_wait_drain(done, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Two groups of four warps; in each group one warp per TMEM lane quadrant
    // (32 key rows of the tile).  Group e reduces rows 2e and 2e+1 of a
    // shared unit; a split unit's one row is group 0's.  Both groups walk
    // the same unit sequence and meet at the group-change barriers; a warp
    // whose wait gave up keeps walking, doing no work, so that no warp is
    // left alone at a named barrier.
    const int et = threadIdx.x - 64;         // 0..255
    const int eg = et >> 7;                  // epilogue group
    const int quad = warp & 3;               // TMEM lane quadrant this warp may read
    const int row_in_tile = quad * 32 + lane;
    int cur_g = -1;
    bool dead = false;
    SubSlots sub;
    GIter it;
    if (count > 0) it.start(a, g_first, j_first);
    for (int64_t n = 0; n < count; ++n, (n < count ? it.next(a) : (void)0)) {
      const Group &G = it.G;
      if (it.g != cur_g) {
        // the group's head weights (w * sq) into shared memory, once no
        // thread reads the previous group's any more
        tc::named_bar_sync(1, kGEpiThreads);
        for (int i = et; i < kGRows * N; i += kGEpiThreads) {
          const int q = i / N, h = i - q * N, row = it.g * kGRows + q;
          float wv = 0.f;
          if (h < a.H_I && row < a.T) {
            wv = a.w[(size_t)row * a.H_I + h];
            if (FP8) wv *= a.q_scale[(size_t)row * a.H_I + h];
          }
          wq_s[i] = wv;
        }
        tc::named_bar_sync(1, kGEpiThreads);
        cur_g = it.g;
      }
      if (dead) continue;
      const int qsel = it.qsel;
      // the sub-slots this group reads: its two rows' (shared unit), or the
      // split unit's one (group 0)
      const uint32_t m = qsel < 0 ? (3u << (2 * eg)) : (eg == 0 ? (1u << sub.ptr) : 0u);
      bool got = true;
#pragma unroll
      for (int s2 = 0; s2 < 4; ++s2)
        if ((m >> s2) & 1u) got = got && tc::mbar_wait(&tfull[s2], sub.parity(s2), abort_flag);
      float sk = 1.f;
      if (got && FP8) {
        const int ss = (int)(n % kGScSlots);
        got = tc::mbar_wait(&scfull[ss], (uint32_t)((n / kGScSlots) & 1), abort_flag);
        if (got) {
          sk = sc_s[ss * (kGScBytes / 4) + (it.y & 3) + row_in_tile];
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&scempty[ss]);
        }
      }
      if (!got) {
        dead = true;   // the CTA is winding down: TMEM is not read again
        continue;
      }
      tc::fence_after_sync();
      const int32_t skey = it.y + row_in_tile;   // this lane's key slot
      const uint32_t tlane = tmem_base + ((uint32_t)(quad * 32) << 16);
      // a sub-slot is free once its group's loads of it have completed
      auto release = [&](int s2) {
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&tempty[s2]);
      };
      auto store = [&](int q, float score) {
        if (FP8) score *= sk;
        if (skey >= G.rs[q] && skey < G.re[q])
          __stcs(a.scores + (int64_t)(it.g * kGRows + q) * a.ld_scores + (skey - G.rs[q]), score);
      };
      if (qsel < 0) {
        // shared unit: this group's two rows' N columns as chunks of CW,
        // the next chunk's load in flight while this one is reduced
        constexpr int kMine = 2 * kCpr;
        const uint32_t col0 = tlane + (uint32_t)(eg * 2 * N);
        uint32_t buf[2][CW];
        float2 p[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        tmem_issue<CW>(col0, buf[0]);
        tmem_wait_regs<CW>(buf[0]);
#pragma unroll
        for (int c = 0; c < kMine; ++c) {
          const int qq = c / kCpr, hh = c % kCpr;      // row 2 eg + qq
          if (c + 1 < kMine) tmem_issue<CW>(col0 + (uint32_t)((c + 1) * CW), buf[(c + 1) & 1]);
          if (hh == kCpr - 1) release(2 * eg + qq);
          relu_dot<CW>(buf[c & 1], wq_s + (2 * eg + qq) * N + hh * CW, p);
          if (hh == kCpr - 1) {
            const float score = (p[0].x + p[0].y) + (p[1].x + p[1].y);
            if (eg == 0) store(qq, score);
            else store(2 + qq, score);
            p[0] = p[1] = make_float2(0.f, 0.f);
          }
          if (c + 1 < kMine) tmem_wait_regs<CW>(buf[(c + 1) & 1]);
        }
      } else if (eg == 0) {
        // split unit: one row in one sub-slot
        const int s2 = sub.ptr;
        uint32_t buf[2][CW];
        float2 p[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        tmem_issue<CW>(tlane + (uint32_t)(s2 * N), buf[0]);
        tmem_wait_regs<CW>(buf[0]);
#pragma unroll
        for (int hh = 0; hh < kCpr; ++hh) {
          if (hh + 1 < kCpr) tmem_issue<CW>(tlane + (uint32_t)(s2 * N + (hh + 1) * CW), buf[(hh + 1) & 1]);
          if (hh == kCpr - 1) release(s2);
          relu_dot<CW>(buf[hh & 1], wq_s + qsel * N + hh * CW, p);
          if (hh + 1 < kCpr) tmem_wait_regs<CW>(buf[(hh + 1) & 1]);
        }
        const float score = (p[0].x + p[0].y) + (p[1].x + p[1].y);
#pragma unroll
        for (int q = 0; q < kGRows; ++q)
          if (q == qsel) store(q, score);
      }
      sub.advance(qsel);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) raise_flag(a.err_flag, DSA_DEVERR_TIMEOUT);
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <bool FP8, int N>
cudaError_t launch_groups(const IndexScoreArgs &a, cudaStream_t s) {
  CUtensorMap kmap, qmap;
  const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int eb = FP8 ? 1 : 2;
  const uint32_t box_cols = FP8 ? 128 : 64;  // 128 bytes: the whole of d
  if (!make_tmap_2d(&kmap, a.k_idx, dt, eb, (uint64_t)a.k_rows, (uint64_t)a.d, kGTileKeys, box_cols))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d(&qmap, a.q_idx, dt, eb, (uint64_t)a.T * a.H_I, (uint64_t)a.d, N, box_cols))
    return cudaErrorInvalidValue;
  CUtensorMap smap = kmap;   // unused for bf16
  if (FP8 && !make_tmap_1d(&smap, a.k_scale, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                           (uint64_t)a.k_rows, kGScBox))
    return cudaErrorInvalidValue;
  // at most ceil(T / 4) * 4 * ceil(max_len / 128) valid units (split groups
  // have one unit per row tile); each CTA takes an equal share of the valid
  // ones (computed in the kernel)
  const int64_t tiles_per_row = (a.max_len + kGTileKeys - 1) / kGTileKeys;
  const int64_t total = (int64_t)a.T * tiles_per_row;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((int64_t)kGCtasPerSm * num_sms(), total));
  const GSmem L = gsmem_layout(N);
  const size_t smem = L.total + 1024;
  auto kern = index_score_groups_kernel<FP8, N>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kGThreads), smem, s, kmap, qmap, smap, a);
}

template <bool FP8>
cudaError_t launch_group_heads(const IndexScoreArgs &a, cudaStream_t s) {
  if (a.H_I <= 16) return launch_groups<FP8, 16>(a, s);
  if (a.H_I <= 32) return launch_groups<FP8, 32>(a, s);
  return launch_groups<FP8, 64>(a, s);
}

}  // namespace

cudaError_t index_score_prefill_launch(const IndexScoreArgs &a, cudaStream_t s) {
  // row ranges, no fused histogram, the whole of d in one 128-byte block
  // (fp8 d = 128, bf16 d = 64), at least one full group
  const bool fp8 = a.idx_dtype == DSA_IDX_FP8_E4M3;
  const bool one_block = fp8 ? a.d == 128 : a.d == 64;
  if (a.T < kGRows || a.max_len == 0 || a.slot_base || a.hist || a.block_table || !one_block)
    return index_score_launch(a, s);
  return fp8 ? launch_group_heads<true>(a, s) : launch_group_heads<false>(a, s);
}

}  // namespace dsa
