// Absorbed-MLA sparse attention on the 5th-generation tensor cores, bf16
// latent pool (576 = 512 NoPE + 64 RoPE per row, V = the leading 512).
// (The "sparse attn" stage of tokenspeed PR #627 "Add gluon kernel for DSA";
// semantics of miles PR #3608: natural-log lse, -1 entries masked.)
//
// One CTA handles one (token, piece of its index list, group of <= 64 heads)
// and walks the piece in tiles of 64 gathered rows.  Per tile:
//   S^T[kv, h] = K_tile[kv, :] . Q[h, :]       tcgen05 M = 64 (kv), N = heads,
//                                                K = 576; A = the gathered
//                                                tile (K-major), B = Q
//   softmax over kv per head (online, lazy rescale); P^T to smem as two
//   bf16 terms P_hi + P_lo (P_lo in the tile's RoPE K-block, dead after S),
//   so the PV product carries p to ~2^-17 instead of bf16's 2^-9
//   O^T[dv, h] += V^T[dv, kv] . P^T[kv, h]      tcgen05 M = 128 (dv) x 4,
//                                                K = 64 (kv); A = the SAME
//                                                gathered tile read MN-major,
//                                                B = P^T (MN-major)
// so the rows are read from HBM once and serve as K and as V.  S^T and O^T
// live in TMEM (2 x N + 4 x N columns).  With M = 64 the tensor core puts kv
// row 16q + i in TMEM lane 32q + i, so each of the four math warps owns 16
// rows of S^T and all 32 lanes of one quarter of O^T.
//
// Online softmax with a lazy maximum: a head's reference maximum changes
// only when a tile exceeds it by more than 2^8 (in exp2 units); then O^T and
// the partial sums are rescaled.  Otherwise p <= 256, exact in fp32 and
// representable in bf16.
//
// Warps: 0-3 math (softmax, rescale, epilogue), 4 MMA issue, 5-6 gather
// (one warp per shared-memory stage; cp.async 16-byte copies into the
// 128-byte-swizzled operand layout, zero-filled for masked rows so that a
// -1 entry is never read).
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace dsa {

namespace {

constexpr int kThreads = 224;      // 7 warps (<= 2 per SM sub-partition: no register cap)
constexpr int kTileRows = 64;
constexpr int kKBlocks = 9;        // 576 bf16 = 9 x 128 bytes
constexpr int kKBlockBytes = kTileRows * 128;               // 8 KB
constexpr int kStageBytes = kKBlocks * kKBlockBytes;        // 72 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazy = 8.0f;      // log2 of the largest tolerated p

struct MlaSmem {
  uint32_t q, k, p, red, mref, alpha, flag, bars, total;
};

__host__ __device__ inline MlaSmem mla_smem_layout(int N) {
  MlaSmem L;
  L.q = 0;
  L.k = L.q + kKBlocks * N * 128;
  L.p = L.k + 2 * kStageBytes;
  L.red = L.p + kTileRows * 128;     // [4][64] floats
  L.mref = L.red + 4 * 64 * 4;       // [64]
  L.alpha = L.mref + 64 * 4;         // [64]
  L.flag = L.alpha + 64 * 4;         // int
  L.bars = L.flag + 16;              // 8-byte aligned
  L.total = L.bars + 16 * 8;
  return L;
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// List entry e (of the concatenated main + extra list) of token t: the row
// address, or nullptr when masked.  Flags entries outside [-1, rows).
__device__ __forceinline__ const uint8_t *entry_row(const MlaArgs &a, int t, int e) {
  const PoolDev *pool;
  int64_t slot;
  if (e < a.k) {
    pool = &a.kv;
    slot = a.idx[(size_t)t * a.k + e];
  } else {
    pool = &a.kv2;
    slot = a.idx2[(size_t)t * a.k2 + (e - a.k)];
  }
  if (slot >= 0 && slot < pool->rows) return pool->data + slot * (int64_t)1152;
  return nullptr;
}

// Whether entry e reads a row; an entry other than -1 outside [0, rows) is
// reported through err_flag (and masked like -1).
__device__ __forceinline__ bool entry_valid(const MlaArgs &a, int t, int e) {
  int64_t slot, rows;
  if (e < a.k) {
    slot = a.idx[(size_t)t * a.k + e];
    rows = a.kv.rows;
  } else {
    slot = a.idx2[(size_t)t * a.k2 + (e - a.k)];
    rows = a.kv2.rows;
  }
  const bool ok = slot >= 0 && slot < rows;
  if (!ok && slot != -1) raise_flag(a.err_flag, DSA_DEVERR_INDEX_RANGE);
  return ok;
}

// Reduce N values per lane across the 32 lanes of a warp with op (max or
// add).  Each xor step halves the values a lane keeps (it sends the half it
// drops to its partner), so on return lane l holds, in v[0] (and v[1] for
// N = 64), the result for head(s):  N = 64: 2l, 2l+1;  N = 32: l;  N = 16:
// l >> 1.  Written as a compile-time recursion so every index is constant.
template <int V, int OFF, bool MAX, int N>
__device__ __forceinline__ void reduce_scatter_step(float (&v)[N], unsigned lane) {
  if constexpr (V >= 2) {
    constexpr int half = V / 2;
    const bool upper = (lane & OFF) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = upper ? v[half + i] : v[i];
      const float send = upper ? v[i] : v[half + i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, OFF);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
    if constexpr (OFF > 1) reduce_scatter_step<half, OFF / 2, MAX, N>(v, lane);
  } else {
    const float recv = __shfl_xor_sync(0xffffffffu, v[0], OFF);
    v[0] = MAX ? fmaxf(v[0], recv) : v[0] + recv;
    if constexpr (OFF > 1) reduce_scatter_step<1, OFF / 2, MAX, N>(v, lane);
  }
}

template <int N, bool MAX>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[N]) {
  reduce_scatter_step<N, 16, MAX, N>(v, lane_id());
}

template <int N>
__device__ __forceinline__ int scatter_head(int lane, int which) {
  if (N == 64) return 2 * lane + which;
  if (N == 32) return lane;
  return lane >> 1;
}

template <int N>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_tc_kernel(MlaArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const MlaSmem L = mla_smem_layout(N);
  unsigned char *q_s = smem + L.q;
  unsigned char *k_s = smem + L.k;
  unsigned char *p_s = smem + L.p;
  float *red = reinterpret_cast<float *>(smem + L.red);
  float *mref = reinterpret_cast<float *>(smem + L.mref);
  float *alpha = reinterpret_cast<float *>(smem + L.alpha);
  volatile int *flag = reinterpret_cast<volatile int *>(smem + L.flag);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
  uint64_t *kfull = bars + 0;    // [2]
  uint64_t *kempty = bars + 2;   // [2]
  uint64_t *sfull = bars + 4;    // [2]
  uint64_t *sempty = bars + 6;   // [2]
  uint64_t *pfull = bars + 8;
  uint64_t *pempty = bars + 9;
  uint64_t *done = bars + 10;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 11);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 12);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x;
  const int split = blockIdx.y;
  const int h0 = blockIdx.z * 64;
  const int nh = min(64, a.H - h0);
  const int total = a.k + a.k2;
  const int per = (total + a.n_splits - 1) / a.n_splits;
  const int j0 = min(total, split * per);
  const int je = min(total, j0 + per);
  const int nt = (je - j0 + kTileRows - 1) / kTileRows;
  constexpr uint32_t kTmemCols = 6 * N <= 128 ? 128 : (6 * N <= 256 ? 256 : 512);

  if ((tc::smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need 1 KB alignment
    if (threadIdx.x == 0) raise_flag(a.err_flag, DSA_DEVERR_TIMEOUT);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&kfull[i], 32);
      tc::mbar_init(&kempty[i], 1);
      tc::mbar_init(&sfull[i], 1);
      tc::mbar_init(&sempty[i], 4);
    }
    tc::mbar_init(pfull, 4);
    tc::mbar_init(pempty, 1);
    tc::mbar_init(done, 1);
    *abort_flag = 0;
    *flag = 0;
    tc::fence_barrier_init();
  }
  for (int h = threadIdx.x; h < 64; h += blockDim.x) mref[h] = -INFINITY;
  if (warp == 4) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  // Q of this head group into the K-major 128B-swizzled layout:
  // K-block kb (64 dims) holds N rows of 128 bytes; rows >= nh are zero.
  {
    const uint16_t *qg = static_cast<const uint16_t *>(a.q) + ((size_t)t * a.H + h0) * 576;
    for (int i = threadIdx.x; i < N * 72; i += blockDim.x) {
      const int h = i / 72, c = i % 72;   // c: 16-byte chunk of the 1152-byte row
      const int kb = c >> 3, cc = c & 7;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (h < nh) v = __ldg(reinterpret_cast<const uint4 *>(qg + (size_t)h * 576) + c);
      *reinterpret_cast<uint4 *>(q_s + kb * N * 128 + h * 128 + ((cc ^ (h & 7)) << 4)) = v;
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t s_col0 = 0;         // S^T buffers: columns [0, 2N)
  const uint32_t o_col0 = 2 * N;     // O^T blocks:  columns [2N, 6N)

  if (warp >= 5) {
    // -------------------------------------------------------------- gather
    const int g = warp - 5;            // stage / tile parity this warp serves
    for (int i = g; i < nt; i += 2) {
      const int kcount = i >> 1;
      if (!tc::mbar_wait(&kempty[g], (kcount & 1) ^ 1, abort_flag)) break;
      const uint32_t st = tc::smem_u32(k_s + g * kStageBytes);
      // the 64 row addresses of this tile, two per lane, fetched in parallel
      const int e_lo = j0 + i * kTileRows + lane;
      const uint8_t *row_lo = e_lo < je ? entry_row(a, t, e_lo) : nullptr;
      const uint8_t *row_hi = e_lo + 32 < je ? entry_row(a, t, e_lo + 32) : nullptr;
      for (int r = 0; r < kTileRows; ++r) {
        const uint8_t *row = reinterpret_cast<const uint8_t *>(__shfl_sync(
            0xffffffffu, reinterpret_cast<unsigned long long>(r < 32 ? row_lo : row_hi), r & 31));
        const uint8_t *src = row ? row : a.kv.data;
        const uint32_t nbytes = row ? 16u : 0u;
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          const int c = lane + 32 * q;          // 16-byte chunk of the row, 0..71
          if (c < 72) {
            const int kb = c >> 3, cc = c & 7;
            const uint32_t dst = st + kb * kKBlockBytes + r * 128 + ((cc ^ (r & 7)) << 4);
            cp_async_16(dst, src + (row ? c * 16 : 0), nbytes);
          }
        }
      }
      cp_async_commit();
      cp_async_wait_all();
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&kfull[g]);
    }
    cp_async_wait_all();
  } else if (warp == 4) {
    // -------------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_f32acc(1, 1, 0, 0, N, 64);
      constexpr uint32_t idesc_pv = tc::idesc_f32acc(1, 1, 1, 1, N, 128);
      const uint32_t q_addr = tc::smem_u32(q_s);
      const uint32_t p_addr = tc::smem_u32(p_s);
      bool ok = true;
      auto issue_pv = [&](int i) -> bool {
        const int st = i & 1;
        if (!tc::mbar_wait(pfull, i & 1, abort_flag)) return false;
        tc::fence_after_sync();
        const uint32_t k_addr = tc::smem_u32(k_s + st * kStageBytes);
        // P = P_hi + P_lo, both bf16: O^T += V^T P_hi^T + V^T P_lo^T.  P_lo sits in
        // this stage's RoPE K-block, which S(i) no longer needs.
        const uint32_t plo_addr = k_addr + 8 * kKBlockBytes;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t kr = (kk & 3) * 2048;   // 16 kv rows per instruction
            const uint64_t ad = tc::sdesc_sw128(k_addr + (2 * j) * kKBlockBytes + kr,
                                                kKBlockBytes, 1024);
            const uint64_t bd = tc::sdesc_sw128((kk < 4 ? p_addr : plo_addr) + kr, kKBlockBytes,
                                                1024);
            tc::mma_f16(tmem + o_col0 + j * N, ad, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc::mma_commit(&kempty[st]);
        tc::mma_commit(pempty);
        return true;
      };
      for (int i = 0; i < nt && ok; ++i) {
        const int st = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!tc::mbar_wait(&kfull[st], ph, abort_flag)) { ok = false; break; }
        if (!tc::mbar_wait(&sempty[st], ph ^ 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t k_addr = tc::smem_u32(k_s + st * kStageBytes);
#pragma unroll 1
        for (int kb = 0; kb < kKBlocks; ++kb) {
          const uint64_t ad0 = tc::sdesc_sw128(k_addr + kb * kKBlockBytes, 16, 1024);
          const uint64_t bd0 = tc::sdesc_sw128(q_addr + kb * N * 128, 16, 1024);
#pragma unroll
          for (int ko = 0; ko < 4; ++ko)   // 32 bytes (16 bf16) of K per instruction
            tc::mma_f16(tmem + s_col0 + st * N, ad0 + 2 * ko, bd0 + 2 * ko, idesc_s,
                        (kb > 0 || ko > 0) ? 1u : 0u);
        }
        tc::mma_commit(&sfull[st]);
        if (i >= 1 && !issue_pv(i - 1)) { ok = false; break; }
      }
      if (ok && nt > 0) ok = issue_pv(nt - 1);
      if (nt > 0) {
        tc::mma_commit(done);
        tc::mbar_wait_drain(done, 0);
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- math
    const int quad = warp;                  // TMEM lane quadrant
    const int row = 16 * quad + lane;       // S^T row held by this lane (lane < 16)
    const float c = a.softmax_scale * kLog2e;
    // S^T is processed in column chunks of CW heads to bound live registers:
    // pass A finds the tile maxima, pass B (re-reading TMEM) forms p.
    constexpr int CW = N < 32 ? N : 32;
    constexpr int NC = N / CW;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float lsum[NC];                       // running sum of p for head(s) of this lane
#pragma unroll
    for (int cc = 0; cc < NC; ++cc) lsum[cc] = 0.f;
    bool ok = true;
    for (int i = 0; i < nt; ++i) {
      const int b = i & 1;         // S^T buffer, and the K stage of tile i
      const int b_stage = b;
      const int e = j0 + i * kTileRows + row;
      const bool valid = lane < 16 && e < je && entry_valid(a, t, e);  // load before the wait
      if (!tc::mbar_wait(&sfull[b], (i >> 1) & 1, abort_flag)) { ok = false; break; }
      tc::fence_after_sync();
      // pass A: per-head maxima over this warp's 16 rows
#pragma unroll
      for (int cc = 0; cc < NC; ++cc) {
        float x[CW];
        tc::tmem_ld_cols<CW>(tmem + lane_base + s_col0 + b * N + cc * CW, x);
#pragma unroll
        for (int h = 0; h < CW; ++h) x[h] = valid ? x[h] * c : -INFINITY;
        warp_reduce_scatter<CW, true>(x);
        if (CW == 32 || (lane & 1) == 0) red[quad * 64 + cc * CW + scatter_head<CW>(lane, 0)] = x[0];
      }
      tc::named_bar_sync(1, 128);
      if (warp == 0) {
        int need = 0;
#pragma unroll
        for (int w2 = 0; w2 < 2; ++w2) {
          const int h = 2 * lane + w2;
          if (h < N) {
            const float tm = fmaxf(fmaxf(red[h], red[64 + h]), fmaxf(red[128 + h], red[192 + h]));
            const float m_old = mref[h];
            float al = 1.f;
            if (tm > m_old + kLazy) {
              al = (m_old == -INFINITY) ? 0.f : exp2f(m_old - tm);
              mref[h] = tm;
              need = 1;
            }
            alpha[h] = al;
          }
        }
        need = __any_sync(0xffffffffu, need);
        if (lane == 0) *flag = need;
      }
      tc::named_bar_sync(1, 128);
      const int rescale = *flag;
      // P^T and O^T may be touched only after PV(i-1) retired
      if (i >= 1) {
        if (!tc::mbar_wait(pempty, (i - 1) & 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
      }
      if (rescale && i >= 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) tc::tmem_scale_cols<N>(tmem + lane_base + o_col0 + j * N, alpha);
      }
      // pass B: p = exp2(x - m), P^T row in bf16, tile sums
#pragma unroll
      for (int cc = 0; cc < NC; ++cc) {
        float x[CW];
        tc::tmem_ld_cols<CW>(tmem + lane_base + s_col0 + b * N + cc * CW, x);
        uint32_t pk[CW / 2], pl[CW / 2];
#pragma unroll
        for (int h = 0; h < CW; h += 2) {
          const int hh = cc * CW + h;
          x[h] = valid ? exp2f(x[h] * c - mref[hh]) : 0.f;
          x[h + 1] = valid ? exp2f(x[h + 1] * c - mref[hh + 1]) : 0.f;
          const __nv_bfloat162 hi = __floats2bfloat162_rn(x[h], x[h + 1]);
          const float2 hf = __bfloat1622float2(hi);
          pk[h / 2] = *reinterpret_cast<const uint32_t *>(&hi);
          pl[h / 2] = pack_bf16x2(x[h] - hf.x, x[h + 1] - hf.y);
        }
        if (lane < 16) {
          unsigned char *plo_s = k_s + b_stage * kStageBytes + 8 * kKBlockBytes;
#pragma unroll
          for (int q = 0; q < CW / 8; ++q) {
            const int ch = cc * (CW / 8) + q;      // 16-byte chunk = 8 heads
            const uint32_t off = row * 128 + ((ch ^ (row & 7)) << 4);
            *reinterpret_cast<uint4 *>(p_s + off) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            *reinterpret_cast<uint4 *>(plo_s + off) =
                make_uint4(pl[4 * q], pl[4 * q + 1], pl[4 * q + 2], pl[4 * q + 3]);
          }
        }
        warp_reduce_scatter<CW, false>(x);
        const int h = cc * CW + scatter_head<CW>(lane, 0);
        lsum[cc] = (rescale ? lsum[cc] * alpha[h] : lsum[cc]) + x[0];
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sempty[b]);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(pfull);
    }
    // ---- epilogue: l per head over the four warps, then O^T / l
    tc::named_bar_sync(1, 128);   // everyone is past the last use of red and alpha
#pragma unroll
    for (int cc = 0; cc < NC; ++cc)
      if (CW == 32 || (lane & 1) == 0) red[quad * 64 + cc * CW + scatter_head<CW>(lane, 0)] = lsum[cc];
    tc::named_bar_sync(1, 128);
    if (warp == 0) {
#pragma unroll
      for (int w2 = 0; w2 < 2; ++w2) {
        const int h = 2 * lane + w2;
        if (h < N) alpha[h] = red[h] + red[64 + h] + red[128 + h] + red[192 + h];  // l per head
      }
    }
    tc::named_bar_sync(1, 128);
    if (ok && nt > 0) {
      ok = tc::mbar_wait(pempty, (nt - 1) & 1, abort_flag);
      tc::fence_after_sync();
    }
    const bool have_o = ok && nt > 0;
    const int Dv = a.Dv;
    // 1 / l per head, next to l (mref keeps the maxima for the lse)
    float *inv_l = red;   // red is free again: [64]
    if (warp == 0) {
#pragma unroll
      for (int w2 = 0; w2 < 2; ++w2) {
        const int h = 2 * lane + w2;
        inv_l[h] = (h < N && alpha[h] > 0.f) ? 1.f / alpha[h] : 0.f;
      }
    }
    tc::named_bar_sync(1, 128);
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
      const int dv = 128 * j + 32 * quad + lane;
#pragma unroll 1
      for (int c0 = 0; c0 < N; c0 += 16) {
        float o[16];
        if (have_o) {
          tc::tmem_ld_cols<16>(tmem + lane_base + o_col0 + j * N + c0, o);
        } else {
#pragma unroll
          for (int h = 0; h < 16; ++h) o[h] = 0.f;
        }
        if (dv >= Dv) continue;
#pragma unroll
        for (int hq = 0; hq < 16; ++hq) {
          const int h = c0 + hq;
          if (h < nh) {
            const size_t rec = a.n_splits == 1 ? (size_t)t * a.H + h0 + h
                                               : ((size_t)t * a.n_splits + split) * a.H + h0 + h;
            const float v = o[hq] * inv_l[h];
            if (a.n_splits == 1)
              static_cast<__nv_bfloat16 *>(a.out)[rec * Dv + dv] = __float2bfloat16_rn(v);
            else
              a.part_o[rec * Dv + dv] = v;
          }
        }
      }
    }
    if (warp == 0) {
#pragma unroll
      for (int w2 = 0; w2 < 2; ++w2) {
        const int h = 2 * lane + w2;
        if (h < nh) {
          const float l = alpha[h];
          const float lse = l > 0.f ? (mref[h] + log2f(l)) * kLn2 : -INFINITY;
          if (a.n_splits == 1)
            a.lse[(size_t)t * a.H + h0 + h] = lse;
          else
            a.part_lse[((size_t)t * a.n_splits + split) * a.H + h0 + h] = lse;
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) raise_flag(a.err_flag, DSA_DEVERR_TIMEOUT);
  if (warp == 4) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int N>
cudaError_t launch_n(const MlaArgs &a, cudaStream_t s) {
  const MlaSmem L = mla_smem_layout(N);
  auto kern = sparse_mla_tc_kernel<N>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)a.T, (unsigned)a.n_splits, (unsigned)((a.H + 63) / 64));
  kern<<<grid, kThreads, L.total, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t sparse_mla_tc_bf16_launch(const MlaArgs &a, cudaStream_t s) {
  const int hg = a.H >= 64 ? 64 : a.H;
  if (hg <= 16) return launch_n<16>(a, s);
  if (hg <= 32) return launch_n<32>(a, s);
  return launch_n<64>(a, s);
}

}  // namespace dsa
