// Lightning-indexer scores on the 5th-generation tensor cores
// (the "scores" stage of tokenspeed PR #627 "Add gluon kernel for DSA"):
//
//   I[t,s] = sum_h w[t,h] * ReLU(sq[t,h] sk[s] q[t,h,:].k[s,:])
//
// One 128-key tile of the index-k cache is the A operand (M = 128 rows,
// K = d, K-major, 128-byte swizzle, loaded by TMA); the query's H_I head rows
// are the B operand (N = H_I rounded up to 16).  D = A B^T lands in TMEM as
// one key per lane and one head per column, so the epilogue's weighted ReLU
// reduction over heads is thread-local.  The fp8 scales are positive, so
// sq[t,h] folds into the head weight and sk[s] leaves the head sum:
//   I[t,s] = sk[s] * sum_h (w[t,h] sq[t,h]) * ReLU(q8[t,h,:].k8[s,:]).
//
// Persistent warp-specialised CTAs, two per SM (each pipeline's producer,
// MMA issuer and epilogue are single threads of control, so two independent
// pipelines per SM keep more loads in flight than one deeper ring): warp 0
// issues TMA loads into a 4-stage ring (fp8 d = 128 or bf16 d = 64; 2 stages
// for bf16 d = 128) plus a ring of key-scale slots, warp 1 issues
// tcgen05.mma into four TMEM accumulators, warps 2-5 drain the accumulators,
// write the score row and (decode) count each score's 12-bit bin for the
// first radix level of the top-k (topk.cu).
// Multi-token decode: the rows of one request (its new tokens) share their
// keys, so with RQ = 2 a unit is a pair of rows and one key tile: both rows'
// head rows are the B operand (N = 2 x 64), the tile is read and multiplied
// once for the two, and the epilogue reduces each row's 64 columns in turn
// and counts both rows' bins in one shared histogram of 16-bit halves.
// Every wait is bounded (tc::mbar_wait): a stuck CTA raises
// DSA_DEVERR_TIMEOUT and winds down instead of hanging.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace dsa {

namespace {

constexpr int kTileKeys = 128;
// Epilogue groups of four warps (alternate tiles): two, so that one group's
// drain of a tile overlaps the other's.
template <int RQ> struct IdxShape {
  static constexpr int kGroups = 2;
  static constexpr int kEpiThreads = 128 * kGroups;
  static constexpr int kThreads = 64 + kEpiThreads;
};
constexpr int kCtasPerSm = 2;     // two independent pipelines per SM
constexpr int kHistBinsLocal = kHistBins;
constexpr int kAccUnits = 4;      // TMEM accumulators in flight for one-row units (4 x 64 columns)
constexpr int kScBox = 132;       // fp32 scales per tile load: 128 keys + up to 3 lead-in
constexpr int kScBytes = 640;     // kScBox * 4 rounded up to 128 (TMA destinations are 128-byte aligned)
constexpr int kScSlots = 8;       // ring of per-tile scale slots, released by the epilogue

struct IdxSmem {
  // offsets in bytes from the 1024-aligned base
  uint32_t stage0, stage_bytes, q0, q_bytes, hist, sc, wq, bars;
  int stages;
  uint32_t total;
};

// N: the MMA's N (the unit's head rows); qslots: query slots (two for
// one-row units, so the next row's query lands while this row's MMAs run;
// one for row pairs, whose slot is twice the size)
__host__ __device__ inline IdxSmem idx_smem_layout(int N, int kblocks, int qslots) {
  IdxSmem L;
  L.stage_bytes = kTileKeys * 128 * kblocks;
  L.stages = kblocks == 1 ? 4 : 2;
  L.stage0 = 0;
  L.q0 = L.stage0 + L.stage_bytes * L.stages;
  L.q_bytes = N * 128 * kblocks;  // N * 128 is a multiple of 1024 for N >= 8
  L.hist = L.q0 + qslots * L.q_bytes;
  L.sc = L.hist + kHistBinsLocal * 4;   // kScSlots x (the tile's 128 key scales, +4 lead-in)
  L.wq = L.sc + kScSlots * kScBytes;    // [RQ][64] head weights of the current row group
  L.bars = L.wq + 2 * 64 * 4;
  L.total = L.bars + 640;
  return L;
}

struct RowInfo {
  int64_t r0;
  int64_t len;
  bool bad;
};

template <bool PAGED = false>
__device__ __forceinline__ RowInfo row_info(const IndexScoreArgs &a, int t) {
  RowInfo r;
  int64_t s, e;
  if constexpr (PAGED) {
    // positions 0 .. seq_len-1; their slots come from the block table
    const int64_t len = a.seq_lens[t];
    r.bad = len < 0 || len > (int64_t)a.max_pages * a.page_size;
    r.r0 = 0;
    r.len = r.bad ? 0 : len;
    return r;
  }
  if (a.slot_base) {
    s = a.slot_base[t];
    e = s + a.seq_lens[t];
  } else {
    s = a.row_start[t];
    e = a.row_end[t];
  }
  r.bad = s < 0 || e < s || e > a.k_rows;
  r.r0 = s;
  r.len = r.bad ? 0 : e - s;
  return r;
}

__device__ __forceinline__ int64_t tiles_of(const RowInfo &r) {
  return (r.len + kTileKeys - 1) / kTileKeys;
}

// The keys a unit of RQ consecutive rows covers (group g: rows RQ g ..
// RQ g + RQ - 1): their shared start and the longest row.  Rows of a group
// that do not share their start are a caller's error: the group is reported
// and skipped.
template <bool PAGED, int RQ>
__device__ __forceinline__ RowInfo group_info(const IndexScoreArgs &a, int g) {
  RowInfo r = row_info<PAGED>(a, RQ * g);
#pragma unroll
  for (int q = 1; q < RQ; ++q) {
    const RowInfo o = row_info<PAGED>(a, RQ * g + q);
    if (o.bad || (o.len > 0 && r.len > 0 && o.r0 != r.r0)) r.bad = true;
    if (r.len == 0) r.r0 = o.r0;
    r.len = max(r.len, o.len);
  }
  if (r.bad) r.len = 0;
  return r;
}

// Walks a CTA's share of the valid (row group, key tile) units in row-major
// order, skipping groups without keys.  next() may be called only while
// units remain.
template <bool PAGED, int RQ>
struct TileIter {
  int t;   // the group (the row, for RQ = 1)
  int64_t j, ntile;
  RowInfo ri;
  __device__ __forceinline__ void start(const IndexScoreArgs &a, int t0, int64_t j0) {
    t = t0;
    j = j0;
    ri = group_info<PAGED, RQ>(a, t);
    ntile = tiles_of(ri);
  }
  __device__ __forceinline__ void next(const IndexScoreArgs &a) {
    if (++j == ntile) {
      j = 0;
      do {
        ++t;
        ri = group_info<PAGED, RQ>(a, t);
        ntile = tiles_of(ri);
      } while (ntile == 0);
    }
  }
};

// PAGED: the caches are paged (block table, pages of a multiple of 64
// slots): a tile's 128 positions are two runs of 64 slots, each loaded with
// the 64-row maps kmap64 / smap64 from the slot the table gives.
// RQ: rows per unit (2: the rows of a request in a multi-token decode, which
// share their keys); N: the MMA's N, RQ x the padded head count NH.
template <bool FP8, int N, int KB, bool PAGED, int RQ>
__global__ void __launch_bounds__(IdxShape<RQ>::kThreads, kCtasPerSm)
index_score_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap smap,
                      const __grid_constant__ CUtensorMap kmap64,
                      const __grid_constant__ CUtensorMap smap64, IndexScoreArgs a) {
  static_assert(RQ == 1 || (RQ == 2 && N == 128 && !PAGED), "row pairs: 2 x 64 heads, unpaged");
  constexpr int NH = N / RQ;               // head columns of one row
  constexpr int kAcc = kAccUnits / RQ;     // accumulators in flight (half of TMEM)
  constexpr int kQSlots = RQ == 1 ? 2 : 1;
  constexpr int kGroups = IdxShape<RQ>::kGroups;
  constexpr int kEpiThreads = IdxShape<RQ>::kEpiThreads;
  constexpr int kThreads = IdxShape<RQ>::kThreads;
  extern __shared__ unsigned char smem_raw[];
  const IdxSmem L = idx_smem_layout(N, KB, kQSlots);
  unsigned char *base = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + L.bars);
  uint64_t *full = bars;                 // [stages <= 12]
  uint64_t *empty = bars + 12;           // [stages]
  uint64_t *scfull = bars + 24;          // [kScSlots]
  uint64_t *scempty = bars + 40;         // [kScSlots]
  uint64_t *qfull = bars + 56;           // [2]
  uint64_t *qempty = bars + 58;          // [2]
  uint64_t *tfull = bars + 60;           // [kAcc]
  uint64_t *tempty = bars + 68;          // [kAcc]
  uint64_t *done = bars + 76;            // [1]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 77);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 78);
  uint32_t *hist_s = reinterpret_cast<uint32_t *>(base + L.hist);
  const float *sc_s = reinterpret_cast<const float *>(base + L.sc);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = L.stages;
  constexpr uint32_t kTmemCols = (kAcc * N < 32) ? 32 : kAcc * N;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kScSlots; ++i) {
      tc::mbar_init(&scfull[i], 1);
      tc::mbar_init(&scempty[i], 4);
    }
    for (int i = 0; i < kQSlots; ++i) {
      tc::mbar_init(&qfull[i], 1);
      tc::mbar_init(&qempty[i], 1);
    }
    for (int i = 0; i < kAcc; ++i) {
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
  if (warp >= 2) {
    for (int i = threadIdx.x - 64; i < kHistBinsLocal; i += kEpiThreads) hist_s[i] = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // Launched as a dependent of the previous kernel (the fused decode: the
  // histogram's zeroing).  With inputs_ready only the epilogue, which adds
  // into the histogram, waits for it; otherwise every role waits before
  // touching anything, the row ranges included.
  if (!a.inputs_ready) pdl_wait();

  // ---- this CTA's share of the valid tiles.  Rows differ in length (causal
  // prefill: row t has t + 1 keys; ragged decode batches), so the units are
  // split evenly by count: every thread sums the tiles of a run of rows, a
  // block scan gives the total and each run's start, and the run holding
  // this CTA's first unit locates it.
  __shared__ int64_t s_warp[kThreads / 32];
  __shared__ int s_t0;
  __shared__ int64_t s_j0, s_count;
  const int TG = a.T / RQ;   // row groups (the host checks that RQ divides T)
  {
    const int R = (TG + kThreads - 1) / kThreads;
    const int rlo = min(TG, (int)threadIdx.x * R), rhi = min(TG, rlo + R);
    int64_t mine = 0;
#pragma unroll 4
    for (int t = rlo; t < rhi; ++t) {
      const RowInfo r = group_info<PAGED, RQ>(a, t);
      if (r.bad && blockIdx.x == 0) raise_flag(a.err_flag, DSA_DEVERR_INDEX_RANGE);
      mine += tiles_of(r);
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
    for (int w = 0; w < kThreads / 32; ++w) {
      const int64_t x = s_warp[w];
      if (w < warp) before += x;
      total += x;
    }
    const int64_t pre = before + incl - mine;      // units before this thread's rows
    const int64_t u0 = total * (int64_t)blockIdx.x / gridDim.x;
    const int64_t u1 = total * ((int64_t)blockIdx.x + 1) / gridDim.x;
    if (u0 < u1 && pre <= u0 && u0 < pre + mine) {
      int64_t acc = pre;
      for (int t = rlo; t < rhi; ++t) {
        const int64_t n = tiles_of(group_info<PAGED, RQ>(a, t));
        if (u0 < acc + n) {
          s_t0 = t;
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
  const int t_first = count > 0 ? s_t0 : 0;
  const int64_t j_first = count > 0 ? s_j0 : 0;
  if (a.inputs_ready && warp >= 2) pdl_wait();
  pdl_trigger();   // the next kernel may be placed as SMs free up; it waits for us

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::prefetch_tmap(&kmap);
      tc::prefetch_tmap(&qmap);
      // the key tiles and scales are read once: evict them first, so the
      // score rows written by this kernel are still in L2 for the top-k
      const uint64_t stream_policy = tc::l2_policy_evict_first();
      if (FP8) tc::prefetch_tmap(&smap);
      int stage = 0;
      uint32_t phase = 0;
      int qs = 0;
      uint32_t qphase = 0;
      int cur_t = -1;
      uint32_t issued = 0;         // bit i: stage i has had a load
      uint32_t last_phase = 0;     // bit i: parity of stage i's last load
      uint32_t q_issued = 0, q_last = 0;
      int ss = 0;                  // scale slot (FP8)
      uint32_t sphase = 0;
      uint32_t s_issued = 0, s_last = 0;
      bool ok = true;
      TileIter<PAGED, RQ> it;
      if (count > 0) it.start(a, t_first, j_first);
      for (int64_t n = 0; n < count && ok; ++n, (n < count ? it.next(a) : (void)0)) {
        const int t = it.t;
        const int64_t j = it.j;
        const RowInfo &ri = it.ri;
        if (t != cur_t) {
          if (cur_t >= 0) {
            if (++qs == kQSlots) {
              qs = 0;
              qphase ^= 1;
            }
          }
          if (!tc::mbar_wait(&qempty[qs], qphase ^ 1, abort_flag)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(&qfull[qs], L.q_bytes);
          // the group's rows' NH head rows each, stacked (N = RQ x NH)
          for (int kb = 0; kb < KB; ++kb)
            for (int q = 0; q < RQ; ++q)
              tc::tma_load_2d(&qmap, &qfull[qs],
                              base + L.q0 + qs * L.q_bytes + kb * N * 128 + q * NH * 128,
                              kb * (FP8 ? 128 : 64), (t * RQ + q) * a.H_I);
          q_issued |= 1u << qs;
          q_last = (q_last & ~(1u << qs)) | (qphase << qs);
          cur_t = t;
        }
        // paged: the slots of the tile's two runs of 64 positions, read from
        // the block table before the wait, whose time then covers the loads
        int yseg[2] = {0, 0};
        if constexpr (PAGED) {
#pragma unroll
          for (int sg = 0; sg < 2; ++sg) {
            int64_t p = j * kTileKeys + 64 * sg;
            if (p >= ri.len) p = j * kTileKeys;       // a run past the row: reload the first (unused)
            const int32_t pg = __ldg(a.block_table + (size_t)t * a.max_pages + p / a.page_size);
            yseg[sg] = pg * a.page_size + (int)(p % a.page_size);
          }
        }
        if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag)) { ok = false; break; }
        tc::mbar_arrive_expect_tx(&full[stage], L.stage_bytes);
        const int y = (int)(ri.r0 + j * kTileKeys);
        if constexpr (PAGED) {
          for (int kb = 0; kb < KB; ++kb)
            for (int sg = 0; sg < 2; ++sg)
              tc::tma_load_2d_hint(&kmap64, &full[stage],
                                   base + L.stage0 + stage * L.stage_bytes + kb * 16384 + sg * 8192,
                                   kb * (FP8 ? 128 : 64), yseg[sg], stream_policy);
        } else {
          for (int kb = 0; kb < KB; ++kb)
            tc::tma_load_2d_hint(&kmap, &full[stage], base + L.stage0 + stage * L.stage_bytes + kb * 16384,
                                 kb * (FP8 ? 128 : 64), y, stream_policy);
        }
        if (FP8) {
          // the 128 key scales, from the nearest 16-byte boundary at or below y,
          // into their own ring (held until the epilogue has read them)
          if (!tc::mbar_wait(&scempty[ss], sphase ^ 1, abort_flag)) { ok = false; break; }
          if constexpr (PAGED) {
            // the two runs' 64 scales each, at scale 0 and 64 of the slot
            tc::mbar_arrive_expect_tx(&scfull[ss], 2 * 64 * 4);
            for (int sg = 0; sg < 2; ++sg)
              tc::tma_load_2d_hint(&smap64, &scfull[ss], base + L.sc + ss * kScBytes + sg * 256,
                                   yseg[sg], 0, stream_policy);
          } else {
            tc::mbar_arrive_expect_tx(&scfull[ss], kScBox * 4);
            tc::tma_load_2d_hint(&smap, &scfull[ss], base + L.sc + ss * kScBytes, y & ~3, 0,
                                 stream_policy);
          }
          s_issued |= 1u << ss;
          s_last = (s_last & ~(1u << ss)) | (sphase << ss);
          if (++ss == kScSlots) {
            ss = 0;
            sphase ^= 1;
          }
        }
        issued |= 1u << stage;
        last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      // every load this thread issued must land before the CTA exits
      for (int i = 0; i < S; ++i)
        if (issued & (1u << i)) tc::mbar_wait_drain(&full[i], (last_phase >> i) & 1u);
      for (int i = 0; i < kQSlots; ++i)
        if (q_issued & (1u << i)) tc::mbar_wait_drain(&qfull[i], (q_last >> i) & 1u);
      for (int i = 0; i < kScSlots; ++i)
        if (s_issued & (1u << i)) tc::mbar_wait_drain(&scfull[i], (s_last >> i) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc =
          tc::idesc_f32acc(FP8 ? 0u : 1u, FP8 ? 0u : 1u, 0u, 0u, (uint32_t)N, 128u);
      int stage = 0;
      uint32_t phase = 0;
      int qs = 0;
      uint32_t qphase = 0;
      int cur_t = -1;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool any = false;
      TileIter<PAGED, RQ> it;
      if (count > 0) it.start(a, t_first, j_first);
      for (int64_t n = 0; n < count; ++n, (n < count ? it.next(a) : (void)0)) {
        const int t = it.t;
        if (t != cur_t) {
          if (cur_t >= 0) {
            tc::mma_commit(&qempty[qs]);  // the old query slot is free once its MMAs finish
            if (++qs == kQSlots) {
              qs = 0;
              qphase ^= 1;
            }
          }
          if (!tc::mbar_wait(&qfull[qs], qphase, abort_flag)) break;
          cur_t = t;
        }
        if (!tc::mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag)) break;
        if (!tc::mbar_wait(&full[stage], phase, abort_flag)) break;
        tc::fence_after_sync();
        const uint32_t a_addr = tc::smem_u32(base + L.stage0 + stage * L.stage_bytes);
        const uint32_t b_addr = tc::smem_u32(base + L.q0 + qs * L.q_bytes);
        const uint64_t adesc0 = tc::sdesc_sw128(a_addr, 16, 1024);
        const uint64_t bdesc0 = tc::sdesc_sw128(b_addr, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 4 * KB; ++kk) {
          // 32 bytes of K per instruction (K = 32 fp8 or 16 bf16), 4 per 128 B block
          const uint32_t a_off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t b_off = (kk >> 2) * N * 128 + (kk & 3) * 32;
          const uint64_t ad = adesc0 + (a_off >> 4);
          const uint64_t bd = bdesc0 + (b_off >> 4);
          if constexpr (FP8)
            tc::mma_f8f6f4(tmem_base + acc * N, ad, bd, idesc, kk > 0 ? 1u : 0u);
          else
            tc::mma_f16(tmem_base + acc * N, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&empty[stage]);
        tc::mma_commit(&tfull[acc]);
        any = true;
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
        if (++acc == kAcc) {
          acc = 0;
          acc_phase ^= 1;
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
    // Two groups of four warps (each group covers the four TMEM lane
    // quadrants) take alternate tiles.  Both groups walk the same tile
    // sequence, so they meet at the same row-change flushes.  A warp whose
    // wait gave up keeps walking (doing no work) so that no warp is left alone
    // at a named barrier.
    const int et = threadIdx.x - 64;         // 0..255
    const int group = kGroups == 1 ? 0 : (et >> 7);
    const int quad = warp & 3;               // TMEM lane quadrant this warp may read
    const int row_in_tile = quad * 32 + lane;
    int cur_t = -1;
    uint32_t hist_rows = 0;                  // bit q: row q of the group counts its bins
    int64_t rlen[RQ];                        // each row's keys
    int since_flush = 0;                     // row pairs: units counted since the last flush
    bool dead = false;
    float *wq_s = reinterpret_cast<float *>(base + L.wq);   // [RQ][NH] head weights of the group
    // the group's bin counts into the rows' global histograms (every
    // epilogue thread; row pairs count row q in bits 16q .. 16q + 15)
    auto flush = [&](int g) {
      tc::named_bar_sync(1, kEpiThreads);
      for (int i = et; i < kHistBinsLocal; i += kEpiThreads) {
        const uint32_t c = hist_s[i];
        if (!c) continue;
        if (RQ == 1) {
          atomicAdd(&a.hist[(size_t)g * kHistBins + i], c);
        } else {
          if (c & 0xffffu) atomicAdd(&a.hist[(size_t)(RQ * g) * kHistBins + i], c & 0xffffu);
          if (c >> 16) atomicAdd(&a.hist[(size_t)(RQ * g + 1) * kHistBins + i], c >> 16);
        }
        hist_s[i] = 0;
      }
      tc::named_bar_sync(1, kEpiThreads);
    };
    TileIter<PAGED, RQ> it;
    if (count > 0) it.start(a, t_first, j_first);
    // unit n of this CTA (the producer and the issuer walk the same sequence)
    for (int64_t n = 0; n < count; ++n, (n < count ? it.next(a) : (void)0)) {
      const int t = it.t;
      const int64_t j = it.j;
      const RowInfo &ri = it.ri;
      if (t != cur_t) {
        if (hist_rows) flush(cur_t);   // the previous group's bin counts
        hist_rows = 0;
        since_flush = 0;
#pragma unroll
        for (int q = 0; q < RQ; ++q) {
          const RowInfo r = RQ == 1 ? ri : row_info<PAGED>(a, RQ * t + q);
          rlen[q] = (r.bad || ri.bad) ? 0 : r.len;
          if (a.hist != nullptr && rlen[q] > a.topk_k) hist_rows |= 1u << q;
        }
        {
          tc::named_bar_sync(1, kEpiThreads);   // every thread is done with the old weights
          for (int i = et; i < RQ * NH; i += kEpiThreads) {
            const int q = i / NH, h = i - q * NH;
            const size_t row = (size_t)(RQ * t + q);
            float wv = 0.f;
            if (h < a.H_I) {
              wv = a.w[row * a.H_I + h];
              if (FP8) wv *= a.q_scale[row * a.H_I + h];
            }
            wq_s[i] = wv;
          }
          tc::named_bar_sync(1, kEpiThreads);
        }
        cur_t = t;
      }
      if (RQ > 1) {
        // a 16-bit half holds 511 units x 128 keys of one row: flush before
        // it could carry into the other row's half
        if (hist_rows && since_flush == 511) {
          flush(t);
          since_flush = 0;
        }
        ++since_flush;
      }
      const int64_t my_n = n;
      if (dead || (int)(my_n % kGroups) != group) continue;
      const int acc = (int)(my_n % kAcc);
      const uint32_t acc_phase = (uint32_t)((my_n / kAcc) & 1);
      if (!tc::mbar_wait(&tfull[acc], acc_phase, abort_flag)) { dead = true; continue; }
      tc::fence_after_sync();
      const uint32_t tacc = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * N;
      // this key's weighted ReLU head sum of each row of the unit
      float score[RQ];
#pragma unroll
      for (int q = 0; q < RQ; ++q) {
        float d[NH];
        tc::tmem_ld_cols<NH>(tacc + q * NH, d);
        if (q == RQ - 1) {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&tempty[acc]);
        }
        // four independent chains (heads h mod 4), added at the end: a
        // quarter of the dependent FMA latency (padded heads weigh 0)
        const float4 *w4 = reinterpret_cast<const float4 *>(wq_s + q * NH);
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h4 = 0; h4 < NH / 4; ++h4) {
          if (4 * h4 >= a.H_I) break;
          const float4 wv = w4[h4];
          s4[0] = fmaf(wv.x, fmaxf(d[4 * h4], 0.f), s4[0]);
          s4[1] = fmaf(wv.y, fmaxf(d[4 * h4 + 1], 0.f), s4[1]);
          s4[2] = fmaf(wv.z, fmaxf(d[4 * h4 + 2], 0.f), s4[2]);
          s4[3] = fmaf(wv.w, fmaxf(d[4 * h4 + 3], 0.f), s4[3]);
        }
        score[q] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      }
      const int64_t key = j * kTileKeys + row_in_tile;
      float sk = 1.f;
      if (FP8) {
        const int ss = (int)(my_n % kScSlots);
        if (!tc::mbar_wait(&scfull[ss], (uint32_t)((my_n / kScSlots) & 1), abort_flag)) {
          dead = true;
          continue;
        }
        sk = sc_s[ss * (kScBytes / 4) + (PAGED ? 0 : (int)((ri.r0 + j * kTileKeys) & 3)) +
                  row_in_tile];
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&scempty[ss]);
      }
#pragma unroll
      for (int q = 0; q < RQ; ++q) {
        const float sc = FP8 ? score[q] * sk : score[q];
        if (key < rlen[q]) {
          a.scores[(int64_t)(RQ * t + q) * a.ld_scores + key] = sc;
          if ((hist_rows >> q) & 1u) atomicAdd(&hist_s[score_key(sc) >> 20], 1u << (16 * q));
        }
      }
    }
    if (hist_rows) flush(cur_t);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) raise_flag(a.err_flag, DSA_DEVERR_TIMEOUT);
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <bool FP8, int N, int KB, bool PAGED, int RQ>
cudaError_t launch_tc(const IndexScoreArgs &a, cudaStream_t s) {
  constexpr int NH = N / RQ;   // head rows of one query row in the B operand
  CUtensorMap kmap, qmap;
  const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int eb = FP8 ? 1 : 2;
  const uint32_t box_cols = FP8 ? 128 : 64;  // 128 bytes
  if (!make_tmap_2d(&kmap, a.k_idx, dt, eb, (uint64_t)a.k_rows, (uint64_t)a.d, kTileKeys, box_cols))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d(&qmap, a.q_idx, dt, eb, (uint64_t)a.T * a.H_I, (uint64_t)a.d, NH, box_cols))
    return cudaErrorInvalidValue;
  CUtensorMap smap = kmap;   // unused for bf16
  if (FP8 && !make_tmap_1d(&smap, a.k_scale, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                           (uint64_t)a.k_rows, kScBox))
    return cudaErrorInvalidValue;
  // paged: 64-row boxes, one per run of 64 positions (unused otherwise)
  CUtensorMap kmap64 = kmap, smap64 = smap;
  if (PAGED) {
    if (!make_tmap_2d(&kmap64, a.k_idx, dt, eb, (uint64_t)a.k_rows, (uint64_t)a.d, 64, box_cols))
      return cudaErrorInvalidValue;
    if (FP8 && !make_tmap_1d(&smap64, a.k_scale, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                             (uint64_t)a.k_rows, 64))
      return cudaErrorInvalidValue;
  }
  // at most T * ceil(max_len / 128) valid tiles; each CTA takes an equal
  // share of the valid ones (computed in the kernel)
  const int64_t tiles_per_row = (a.max_len + kTileKeys - 1) / kTileKeys;
  const int64_t total = (int64_t)(a.T / RQ) * tiles_per_row;
  const int64_t grid = std::min<int64_t>((int64_t)kCtasPerSm * num_sms(), total);
  const IdxSmem L = idx_smem_layout(N, KB, RQ == 1 ? 2 : 1);
  const size_t smem = L.total + 1024;
  auto kern = index_score_tc_kernel<FP8, N, KB, PAGED, RQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(IdxShape<RQ>::kThreads), smem, s, kmap, qmap,
                    smap, kmap64,
                    smap64, a);
}

template <bool FP8, int KB, bool PAGED>
cudaError_t launch_heads(const IndexScoreArgs &a, cudaStream_t s) {
  if (a.H_I <= 16) return launch_tc<FP8, 16, KB, PAGED, 1>(a, s);
  if (a.H_I <= 32) return launch_tc<FP8, 32, KB, PAGED, 1>(a, s);
  return launch_tc<FP8, 64, KB, PAGED, 1>(a, s);
}

template <bool FP8, int KB>
cudaError_t launch_paging(const IndexScoreArgs &a, cudaStream_t s) {
  if (a.block_table) return launch_heads<FP8, KB, true>(a, s);
  return launch_heads<FP8, KB, false>(a, s);
}

}  // namespace

cudaError_t index_score_launch(const IndexScoreArgs &a, cudaStream_t s) {
  if (a.T == 0 || a.max_len == 0) return cudaSuccess;
  if (a.rows_per_unit == 2) {
    // row pairs (multi-token decode): heads padded to 64, one K-block rows,
    // unpaged; the caller checked these and that T is even
    if (a.block_table || a.H_I > 64 || a.T % 2 != 0) return cudaErrorInvalidValue;
    if (a.idx_dtype == DSA_IDX_FP8_E4M3) return launch_tc<true, 128, 1, false, 2>(a, s);
    if (a.d == 64) return launch_tc<false, 128, 1, false, 2>(a, s);
    return cudaErrorInvalidValue;
  }
  if (a.idx_dtype == DSA_IDX_FP8_E4M3) return launch_paging<true, 1>(a, s);
  if (a.d == 64) return launch_paging<false, 1>(a, s);
  return launch_paging<false, 2>(a, s);
}

}  // namespace dsa
