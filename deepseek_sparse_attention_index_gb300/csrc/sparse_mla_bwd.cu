// Backward of the absorbed-MLA sparse attention over a bf16 pool (rows of
// 576 = 512 NoPE + 64 RoPE, V = the leading 512) on the 5th-generation tensor
// cores: the other half of the training workload the Miles pull request #3608
// measures ("fwd + bwd per layer"; its TileLang backward adds the row
// gradients into dKV with atomics through the gathered indices).  Given
// dL/dout and the forward's lse (the lse takes no gradient):
//   p_j   = e^{s_j - lse},  s_j = scale q . K_j
//   delta = sum_j p_j (dout . V_j)          (= dout . out)
//   dS_j  = scale p_j (dout . V_j - delta)
//   dq    = sum_j dS_j K_j
//   dK_j  = sum_h dS_hj q_h  (+ sum_h p_hj dout_h on the V columns)
//   dsink = -e^{sink - lse} delta
// Row gradients are added into the pool's gradient at the row's slot (fp32
// reductions, once per selection).
//
// One CTA per (token, group of <= 64 heads) walks the token's list in tiles
// of 32 gathered rows, twice.  Pass 1 sums delta; pass 2 forms dS and the
// gradients.  Pass 1 alternates two tile buffers (the second is the region
// that holds the dS / P operand planes in pass 2), so the next tile's gather
// overlaps the current tile's products.  Per tile (tcgen05, bf16 operands, fp32 accumulators in TMEM):
//   S   = Q  K^T     M = 64 heads, N = 32 rows, K = 576   (pass 1 and 2)
//   dP  = dO V^T     M = 64 heads, N = 32 rows, K = 512   (pass 1 and 2)
//   dQ^T += K^T dS^T M = 128 dims (64 for RoPE), N = 64 heads, K = 32 rows;
//                    accumulated over the whole list
//   dK^T  = Q^T dS + dO^T P   M = 128 dims (64 for RoPE), N = 32 rows,
//                    K = 64 heads; drained per tile into dkv
// K^T, Q^T and dO^T are the same shared-memory tiles read MN-major.  P and
// dS enter the products as two bf16 terms each (hi + lo, ~2^-17 relative):
// dq sums dS over the list, where the terms cancel (they sum to zero without
// a sink), and a single bf16 term would leave ~1e-3 relative error.
//
// TMEM (512 columns): S [0, 32), dP [32, 64) -- the RoPE block of dK^T takes
// [0, 32) once the math warps have read S and dP --, dQ^T [64, 384) (four
// 128-dim blocks of 64 heads, then the 64 RoPE dims), dK^T [384, 512) (four
// 128-dim blocks of 32 rows).
//
// Warps: 0-3 math (softmax terms, dS, dq at the end), 4 the Q / dO loads and
// the S and dQ products, 5 the dP product and dK^T blocks 0-1, 6 dK^T blocks
// 2-3 and RoPE, 7-10 the row gather, 11-14 the per-tile dK drain into dkv.
// The drain reads the RoPE block first, which frees S's columns for the next
// tile, so a tile's reductions overlap the next tile's S, softmax and dQ.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace dsa {

namespace {

constexpr int kR = 32;                 // rows per tile
constexpr int kKB = 9;                 // 64-column K-blocks of a row (576)
constexpr int kKBV = 8;                // K-blocks of V (512)
constexpr int kTileKB = kR * 128;      // one K-block of the tile: 4 KB
constexpr int kHKB = 64 * 128;         // one K-block of Q or dO: 64 head rows, 8 KB
constexpr int kThreads = 15 * 32;
constexpr float kLog2e = 1.4426950408889634f;

// TMEM columns
constexpr uint32_t kColS = 0, kColDP = 32, kColDQ = 64, kColDK = 384, kColDKR = 0;

struct BwdSmem {
  uint32_t q, dout, k, k2, ds_h, ds_t, p_t, lse, slot, bars, total;
};
__host__ __device__ inline BwdSmem bwd_smem_layout() {
  BwdSmem L;
  L.q = 0;                              // bf16 [64 heads][576], 9 swizzled K-blocks
  L.dout = L.q + kKB * kHKB;            // bf16 [64 heads][512], 8 K-blocks
  L.k = L.dout + kKBV * kHKB;           // stage A: bf16 [32 rows][576], 9 K-blocks of 4 KB
  // region 2: pass 1 uses it as a second K stage (B); pass 2 as the dS / P
  // operand planes
  L.k2 = L.k + kKB * kTileKB;
  L.ds_h = L.k2;                        // dS [64 heads][32 rows], hi and lo (128-byte rows)
  L.ds_t = L.ds_h + 2 * kHKB;           // dS^T [32 rows][64 heads], hi and lo
  L.p_t = L.ds_t + 2 * kTileKB;         // P^T  [32 rows][64 heads], hi and lo
  L.lse = L.k2 + kKB * kTileKB;         // fp32 [64] (natural log, padded heads +inf)
  L.slot = L.lse + 64 * 4;              // int [4][32] slots of step g's tile (-1: masked) at g % 4
  L.bars = L.slot + 4 * kR * 4;         // mbarriers (8-byte aligned)
  L.total = L.bars + 16 * 8;
  return L;
}

// Step g (pass 1: g < nt, pass 2 after) uses K stage st and is that stage's
// u-th use: pass 1 alternates stages A and B, pass 2 uses A only.
struct StageUse {
  int st;
  int u;
};
__device__ __forceinline__ StageUse stage_use(int g, int nt) {
  if (g < nt) return StageUse{g & 1, g >> 1};
  return StageUse{0, ((nt + 1) >> 1) + (g - nt)};
}
// 16-bit element (row r, column c) of a 128-byte-swizzled operand buffer
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return (uint32_t)(r * 128 + ((((c >> 3) ^ (r & 7))) << 4) + (c & 7) * 2);
}

__global__ void __launch_bounds__(kThreads, 1)
sparse_mla_bwd_tc_kernel(MlaBwdArgs a, const __grid_constant__ CUtensorMap qmap,
                         const __grid_constant__ CUtensorMap dmap) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const BwdSmem L = bwd_smem_layout();
  unsigned char *q_s = smem + L.q;
  unsigned char *do_s = smem + L.dout;
  unsigned char *k_s = smem + L.k;
  unsigned char *k2_s = smem + L.k2;
  unsigned char *dsh_s = smem + L.ds_h;
  unsigned char *dst_s = smem + L.ds_t;
  unsigned char *pt_s = smem + L.p_t;
  float *lse_s = reinterpret_cast<float *>(smem + L.lse);
  int *slot_s = reinterpret_cast<int *>(smem + L.slot);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
  uint64_t *kfull = bars + 14;    // [2] by K stage: the tile landed (gather lanes)
  uint64_t *kempty = bars + 0;    // [2] by K stage: the tile's readers retired (S / dQ issuer,
                                  //     dP issuer); the second at bars + 1
  uint64_t *sfull = bars + 2;     // S and dP in TMEM (both issuers)
  uint64_t *tfree = bars + 3;     // TMEM [0, 64) free again (math warps; pass 2: drain warps)
  uint64_t *pfull = bars + 4;     // dS / P planes written (math warps)
  uint64_t *dkfull = bars + 5;    // dQ^T and dK^T of the tile retired (three issuers)
  uint64_t *qfull = bars + 6;     // Q and dO landed
  uint64_t *dkfree = bars + 13;   // the drain has read dK^T blocks 0-3 (drain warps)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 7);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // long lists first: token T-1-x (a causal prefill's later tokens select more rows)
  const int t = a.T - 1 - (int)blockIdx.x;
  const int h0 = blockIdx.y * 64;
  const int nh = min(64, a.H - h0);

  if ((tc::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) raise_flag(a.err_flag, DSA_DEVERR_TIMEOUT);
    return;
  }
  if (threadIdx.x == 0) {
    for (int st = 0; st < 2; ++st) {
      tc::mbar_init(&kfull[st], 32 * 4);
      tc::mbar_init(&kempty[st], 2);
    }
    tc::mbar_init(sfull, 2);
    tc::mbar_init(tfree, 4);
    tc::mbar_init(pfull, 4);
    tc::mbar_init(dkfull, 3);
    tc::mbar_init(qfull, 1);
    tc::mbar_init(dkfree, 4);
    for (int b = 9; b < 12; ++b) tc::mbar_init(&bars[b], 1);   // each issuer's final drain
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  // the list's tiles up to its last entry other than -1 (a causal prefill's
  // early tokens end in a long -1 tail: those tiles are skipped)
  int *last_s = reinterpret_cast<int *>(bars + 12);
  if (threadIdx.x == 0) *last_s = -1;
  __syncthreads();
  {
    int last = -1;
    for (int e = threadIdx.x; e < a.k; e += blockDim.x)
      if (__ldg(a.idx + (size_t)t * a.k + e) != -1) last = e;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    if (lane == 0 && last >= 0) atomicMax(last_s, last);
  }
  if (threadIdx.x < 64) {
    const int h = threadIdx.x;
    float l = INFINITY;           // a padded head: p = e^{s - inf} = 0
    if (h < nh) {
      l = a.lse[(size_t)t * a.H + h0 + h];
      if (a.lse_log2) l *= 0.6931471805599453f;   // the forward reported log2 units
    }
    lse_s[h] = l;
  }
  if (warp == 4) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int nt = (*last_s + 1 + kR - 1) / kR;
  const int steps = 2 * nt;       // step g: pass 1 for g < nt, pass 2 after; tile g % nt

  if (warp >= 7 && warp < 11) {
    // ------------------------------------------------------------ gather
    // lane gl < 32 publishes row gl's slot; every lane copies 18 of the
    // tile's 32 x 72 16-byte chunks (row r = c / 72, chunk cc = c % 72 into
    // K-block cc / 8, swizzled)
    const int gl = threadIdx.x - 7 * 32;   // 0..127
    for (int g = 0; g < steps; ++g) {
      const int i = g % nt;
      const StageUse su = stage_use(g, nt);
      if (!tc::mbar_wait(&kempty[su.st], (su.u & 1) ^ 1, abort_flag)) break;
      int *sl = slot_s + (g & 3) * kR;
      if (gl < kR) {
        const int e = i * kR + gl;
        int s = -1;
        if (e < a.k) {
          const int v = a.idx[(size_t)t * a.k + e];
          if (v >= 0 && v < a.kv.rows) s = v;
          else if (v != -1 && g < nt) raise_flag(a.err_flag, DSA_DEVERR_INDEX_RANGE);
        }
        sl[gl] = s;
      }
      tc::named_bar_sync(2, 128);
      const uint32_t kb0 = tc::smem_u32(su.st ? k2_s : k_s);
#pragma unroll 6
      for (int j = 0; j < 18; ++j) {
        const int c = gl + 128 * j;
        const int r = c / 72, cc = c - r * 72;
        const int s = sl[r];
        const uint8_t *src = s >= 0 ? a.kv.data + (int64_t)s * 1152 + cc * 16
                                    : static_cast<const uint8_t *>(a.q);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                         kb0 + (cc >> 3) * kTileKB + r * 128 + (((cc & 7) ^ (r & 7)) << 4)),
                     "l"(src), "r"(s >= 0 ? 16u : 0u)
                     : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&kfull[su.st]);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();
  } else if (warp == 4) {
    // ------------------------------------------------------------ Q, dO; S and dQ^T
    if (lane == 0) {
      tc::prefetch_tmap(&qmap);
      tc::prefetch_tmap(&dmap);
      tc::mbar_arrive_expect_tx(qfull, (kKB + kKBV) * kHKB);
      for (int kb = 0; kb < kKB; ++kb) tc::tma_load_3d(&qmap, qfull, q_s + kb * kHKB, kb * 64, h0, t);
      for (int kb = 0; kb < kKBV; ++kb)
        tc::tma_load_3d(&dmap, qfull, do_s + kb * kHKB, kb * 64, h0, t);
      // S = Q K^T: A = Q (K-major, M = 64), B = the tile (K-major, N = 32)
      constexpr uint32_t idesc_s = tc::idesc_f32acc(1, 1, 0, 0, kR, 64);
      // dQ^T += K^T dS^T: A = K^T (the tile MN-major, M = 128 dims / 64 for
      // RoPE), B = dS [heads][rows] (K-major, N = 64)
      constexpr uint32_t idesc_q = tc::idesc_f32acc(1, 1, 1, 0, 64, 128);
      constexpr uint32_t idesc_qr = tc::idesc_f32acc(1, 1, 1, 0, 64, 64);
      const uint64_t adq = tc::sdesc_sw128(tc::smem_u32(q_s), 16, 1024);
      const uint64_t bds = tc::sdesc_sw128(tc::smem_u32(dsh_s), 16, 1024);
      bool ok = nt == 0 || tc::mbar_wait(qfull, 0, abort_flag);
      for (int g = 0; g < steps && ok; ++g) {
        const StageUse su = stage_use(g, nt);
        if (!tc::mbar_wait(&kfull[su.st], su.u & 1, abort_flag)) break;
        if (g > 0 && !tc::mbar_wait(tfree, (g - 1) & 1, abort_flag)) break;
        tc::fence_after_sync();
        const uint32_t kst = tc::smem_u32(su.st ? k2_s : k_s);
        const uint64_t bdk = tc::sdesc_sw128(kst, 16, 1024);
#pragma unroll 1
        for (int kb = 0; kb < kKB; ++kb)
#pragma unroll
          for (int ko = 0; ko < 4; ++ko)
            tc::mma_f16(tmem + kColS, adq + kb * 512 + 2 * ko, bdk + kb * (kTileKB >> 4) + 2 * ko,
                        idesc_s, (kb > 0 || ko > 0) ? 1u : 0u);
        tc::mma_commit(sfull);
        if (g >= nt) {
          const int g2 = g - nt;
          if (!tc::mbar_wait(pfull, g2 & 1, abort_flag)) break;
          tc::fence_after_sync();
          const uint64_t akt = tc::sdesc_sw128(kst, kTileKB, 1024);
          // dims 0..511: four M = 128 blocks (K-blocks 2j, 2j+1); RoPE: M = 64
#pragma unroll 1
          for (int j = 0; j < 5; ++j) {
#pragma unroll
            for (int pl = 0; pl < 2; ++pl)
#pragma unroll
              for (int kr = 0; kr < 2; ++kr)
                tc::mma_f16(tmem + kColDQ + 64 * j, akt + j * (2 * kTileKB >> 4) + kr * 128,
                            bds + pl * (kHKB >> 4) + 2 * kr, j < 4 ? idesc_q : idesc_qr,
                            (g2 > 0 || pl > 0 || kr > 0) ? 1u : 0u);
          }
          tc::mma_commit(dkfull);
        }
        tc::mma_commit(&kempty[su.st]);
      }
      tc::mma_commit(&bars[9]);
      tc::mbar_wait_drain(&bars[9], 0);
    }
    __syncwarp();
  } else if (warp == 5 || warp == 6) {
    // ------------------------------------------------------------ dP; dK^T
    if (lane == 0) {
      const bool w5 = warp == 5;
      // dP = dO V^T: A = dO (K-major, M = 64), B = the tile's V (K-major, N = 32)
      constexpr uint32_t idesc_p = tc::idesc_f32acc(1, 1, 0, 0, kR, 64);
      // dK^T = Q^T dS + dO^T P: A = Q^T / dO^T (MN-major, M = 128 / 64), B =
      // dS^T / P^T [rows][heads] (K-major, N = 32)
      constexpr uint32_t idesc_k = tc::idesc_f32acc(1, 1, 1, 0, kR, 128);
      constexpr uint32_t idesc_kr = tc::idesc_f32acc(1, 1, 1, 0, kR, 64);
      const uint64_t ado = tc::sdesc_sw128(tc::smem_u32(do_s), 16, 1024);
      const uint64_t aqt = tc::sdesc_sw128(tc::smem_u32(q_s), kHKB, 1024);
      const uint64_t adot = tc::sdesc_sw128(tc::smem_u32(do_s), kHKB, 1024);
      const uint64_t bdst = tc::sdesc_sw128(tc::smem_u32(dst_s), 16, 1024);
      const uint64_t bpt = tc::sdesc_sw128(tc::smem_u32(pt_s), 16, 1024);
      bool ok = nt == 0 || tc::mbar_wait(qfull, 0, abort_flag);
      for (int g = 0; g < steps && ok; ++g) {
        if (w5) {
          const StageUse su = stage_use(g, nt);
          if (!tc::mbar_wait(&kfull[su.st], su.u & 1, abort_flag)) break;
          if (g > 0 && !tc::mbar_wait(tfree, (g - 1) & 1, abort_flag)) break;
          tc::fence_after_sync();
          const uint64_t bdk = tc::sdesc_sw128(tc::smem_u32(su.st ? k2_s : k_s), 16, 1024);
#pragma unroll 1
          for (int kb = 0; kb < kKBV; ++kb)
#pragma unroll
            for (int ko = 0; ko < 4; ++ko)
              tc::mma_f16(tmem + kColDP, ado + kb * 512 + 2 * ko,
                          bdk + kb * (kTileKB >> 4) + 2 * ko, idesc_p, (kb > 0 || ko > 0) ? 1u : 0u);
          tc::mma_commit(sfull);
          tc::mma_commit(&kempty[su.st]);
        }
        if (g < nt) continue;
        const int g2 = g - nt;
        if (!tc::mbar_wait(pfull, g2 & 1, abort_flag)) break;
        // blocks 0-3 of the previous tile drained (the RoPE block: tfree, which S waited for)
        if (g2 > 0 && !tc::mbar_wait(dkfree, (g2 - 1) & 1, abort_flag)) break;
        tc::fence_after_sync();
        // warp 5: blocks 0, 1; warp 6: blocks 2, 3 and the RoPE block
        const int jb = w5 ? 0 : 2, je = w5 ? 2 : 5;
#pragma unroll 1
        for (int j = jb; j < je; ++j) {
          const uint32_t dcol = j < 4 ? kColDK + kR * j : kColDKR;
          const uint32_t id = j < 4 ? idesc_k : idesc_kr;
          // Q^T dS: K = 64 heads in steps of 16 (+2048 B of Q rows = +128)
#pragma unroll
          for (int pl = 0; pl < 2; ++pl)
#pragma unroll
            for (int kh = 0; kh < 4; ++kh)
              tc::mma_f16(dcol, aqt + j * (2 * kHKB >> 4) + kh * 128,
                          bdst + pl * (kTileKB >> 4) + 2 * kh, id, (pl > 0 || kh > 0) ? 1u : 0u);
          if (j < 4) {   // + dO^T P on the V dims
#pragma unroll
            for (int pl = 0; pl < 2; ++pl)
#pragma unroll
              for (int kh = 0; kh < 4; ++kh)
                tc::mma_f16(dcol, adot + j * (2 * kHKB >> 4) + kh * 128,
                            bpt + pl * (kTileKB >> 4) + 2 * kh, id, 1u);
          }
        }
        tc::mma_commit(dkfull);
      }
      tc::mma_commit(&bars[10 + (w5 ? 0 : 1)]);
      tc::mbar_wait_drain(&bars[10 + (w5 ? 0 : 1)], 0);
    }
    __syncwarp();
  } else if (warp >= 11) {
    // ------------------------------------------------------------ dK drain
    // warp w reads TMEM lane quadrant w % 4: dims 128 j + 32 quad + lane of
    // blocks 0-3 (32 rows each), and the RoPE dims 512 + 16 quad + lane % 16
    // (rows 16 (lane / 16) .. +15)
    const int quad = warp & 3;
    const int half = lane >> 4;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    for (int g = nt; g < steps; ++g) {
      if (!tc::mbar_wait(dkfull, (g - nt) & 1, abort_flag)) break;
      tc::fence_after_sync();
      // this tile's slots, before the columns are released: the gather may
      // rewrite the slot table once the next tile is under way
      const int *sl = slot_s + (g & 3) * kR;
      int slots[kR];
#pragma unroll
      for (int r = 0; r < kR; ++r) slots[r] = sl[r];
      float vr[16];
      tc::tmem_ld_16x32bx2_x16<16>(tmem + lane_base + kColDKR, vr);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tfree);     // S of the next tile may be written
      {
        const int d = 512 + 16 * quad + (lane & 15);
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const int sr = half ? slots[16 + r] : slots[r];   // constant indices: registers
          if (sr >= 0) atomicAdd(a.dkv + (size_t)sr * 576 + d, vr[r]);
        }
      }
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        float v[32];
        tc::tmem_ld_cols<32>(tmem + lane_base + kColDK + kR * j, v);
        if (j == 3) {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(dkfree);   // the next tile's dK^T may be written
        }
        const int d = 128 * j + 32 * quad + lane;
#pragma unroll
        for (int r = 0; r < kR; ++r)
          if (slots[r] >= 0) atomicAdd(a.dkv + (size_t)slots[r] * 576 + d, v[r]);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ math
    // lanes l and l+16 of warp q share head hl = 16q + l % 16; lane l < 16
    // holds rows 0..15 of the tile, lane l+16 rows 16..31
    const int quad = warp;
    const int hl = 16 * quad + (lane & 15);
    const int half = lane >> 4;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float c = a.softmax_scale * kLog2e;
    const float lse2 = lse_s[hl] * kLog2e;   // +inf for a padded head
    float dsum = 0.f;                         // this lane's part of delta (pass 1)
    float delta = 0.f;
    bool ok = true;
    for (int g = 0; g < steps && ok; ++g) {
      const bool pass2 = g >= nt;
      if (g == nt) delta = dsum + __shfl_xor_sync(0xffffffffu, dsum, 16);   // pass 2: the head's delta
      if (!tc::mbar_wait(sfull, g & 1, abort_flag)) { ok = false; break; }
      tc::fence_after_sync();
      float s[16], dp[16];
      tc::tmem_ld_16x32bx2_x16<16>(tmem + lane_base + kColS, s);
      tc::tmem_ld_16x32bx2_x16<16>(tmem + lane_base + kColDP, dp);
      const int *sl = slot_s + (g & 3) * kR;
      float p[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const bool valid = sl[16 * half + j] >= 0;
        p[j] = valid ? exp2f(s[j] * c - lse2) : 0.f;   // padded head: exp2(-inf) = 0
      }
      if (!pass2) {
#pragma unroll
        for (int j = 0; j < 16; ++j) dsum = fmaf(p[j], dp[j], dsum);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tfree);
        continue;
      }
      // dS = scale p (dP - delta) and P, each as hi + lo bf16
      uint32_t dsh[8], dsl[8];
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        const float d0 = a.softmax_scale * p[j] * (dp[j] - delta);
        const float d1 = a.softmax_scale * p[j + 1] * (dp[j + 1] - delta);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(d0, d1);
        const float2 hf = __bfloat1622float2(hi);
        dsh[j / 2] = *reinterpret_cast<const uint32_t *>(&hi);
        dsl[j / 2] = pack_bf16x2(d0 - hf.x, d1 - hf.y);
      }
      // the previous tile's dQ^T and dK^T products read these planes: they
      // have retired before the planes are rewritten
      if (g > nt) {
        if (!tc::mbar_wait(dkfull, (g - nt - 1) & 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
      }
      // dS [heads][rows]: this lane's 16 rows are chunks 2 half, 2 half + 1 of row hl
#pragma unroll
      for (int pl = 0; pl < 2; ++pl) {
        const uint32_t *w = pl ? dsl : dsh;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int ch = 2 * half + cc;
          *reinterpret_cast<uint4 *>(dsh_s + pl * kHKB + hl * 128 + ((ch ^ (hl & 7)) << 4)) =
              make_uint4(w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
        }
      }
      // dS^T and P^T [rows][heads]: column hl of rows 16 half + j
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int r = 16 * half + j;
        const uint32_t off = sw_off(r, hl);
        const uint32_t wd = (j & 1) ? (dsh[j / 2] >> 16) : (dsh[j / 2] & 0xffffu);
        const uint32_t wl = (j & 1) ? (dsl[j / 2] >> 16) : (dsl[j / 2] & 0xffffu);
        const float pj = p[j];
        const __nv_bfloat16 ph = __float2bfloat16_rn(pj);
        const __nv_bfloat16 pl2 = __float2bfloat16_rn(pj - __bfloat162float(ph));
        *reinterpret_cast<uint16_t *>(dst_s + off) = (uint16_t)wd;
        *reinterpret_cast<uint16_t *>(dst_s + kTileKB + off) = (uint16_t)wl;
        *reinterpret_cast<__nv_bfloat16 *>(pt_s + off) = ph;
        *reinterpret_cast<__nv_bfloat16 *>(pt_s + kTileKB + off) = pl2;
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(pfull);
    }
    // the last tile's dQ^T products retired (its dkfull) before dq is read
    if (ok && nt > 0 && !tc::mbar_wait(dkfull, (nt - 1) & 1, abort_flag)) ok = false;
    tc::fence_after_sync();
    // ---- dq: dQ^T from TMEM (all dQ products retired: the last dkfull)
    float *dqt = a.dq + (size_t)t * a.H * 576;
    const bool have = ok && nt > 0 && !*abort_flag;
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
      float v[64];
      if (have) {
        tc::tmem_ld_cols<64>(tmem + lane_base + kColDQ + 64 * j, v);
      } else {
#pragma unroll
        for (int h = 0; h < 64; ++h) v[h] = 0.f;
      }
      const int d = 128 * j + 32 * quad + lane;
#pragma unroll
      for (int h = 0; h < 64; ++h)
        if (h < nh) dqt[(size_t)(h0 + h) * 576 + d] = v[h];
    }
    {
      float v[32];
      if (have) {
        tc::tmem_ld_16x32bx2_x32<32>(tmem + lane_base + kColDQ + 256, v);
      } else {
#pragma unroll
        for (int h = 0; h < 32; ++h) v[h] = 0.f;
      }
      const int d = 512 + 16 * quad + (lane & 15);
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        const int hh = 32 * half + h;
        if (hh < nh) dqt[(size_t)(h0 + hh) * 576 + d] = v[h];
      }
    }
    // the sinks' gradients
    if (a.sinks && a.dsinks && half == 0 && hl < nh) {
      const float sk = a.sinks[h0 + hl];
      if (nt == 0) delta = 0.f;
      if (sk != -INFINITY) atomicAdd(&a.dsinks[h0 + hl], -exp2f(sk * kLog2e - lse2) * delta);
    }
  }

  if (warp == 4 && lane == 0) tc::mbar_wait_drain(qfull, 0);
  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) raise_flag(a.err_flag, DSA_DEVERR_TIMEOUT);
  if (warp == 4) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t sparse_mla_bwd_launch(const MlaBwdArgs &a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  CUtensorMap qmap, dmap;
  // q [T][H][576] and dout [T][H][512] bf16 in boxes of 64 columns x 64 heads
  if (!make_tmap_3d(&qmap, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 576, (uint64_t)a.H,
                    (uint64_t)a.T, 64, 64, 1) ||
      !make_tmap_3d(&dmap, a.dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 512, (uint64_t)a.H,
                    (uint64_t)a.T, 64, 64, 1))
    return cudaErrorInvalidValue;
  const BwdSmem L = bwd_smem_layout();
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_bwd_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)a.T, (unsigned)((a.H + 63) / 64));
  sparse_mla_bwd_tc_kernel<<<grid, kThreads, L.total, s>>>(a, qmap, dmap);
  return cudaGetLastError();
}

}  // namespace dsa
