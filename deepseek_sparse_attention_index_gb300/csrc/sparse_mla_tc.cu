// Absorbed-MLA sparse attention on the 5th-generation tensor cores.
//   bf16 pool: rows of 576 = 512 NoPE + 64 RoPE, V = the leading 512; the
//     products run in bf16.
//   fp8 pools (uniform e4m3 with 1 x 64 fp32 scales, or packed fp8_ds_mla
//     pages with UE8M0 exponents and a bf16 RoPE tail): rows of 512 = 448
//     NoPE + 64 RoPE, V = the leading 448.  The gather warps dequantise each
//     row to fp16 in shared memory (an e4m3 value times a power of two is
//     exact in fp16; times an fp32 scale it rounds once, to 2^-11 relative),
//     Q is converted bf16 -> fp16 in shared memory, and the products run in
//     fp16 -- whose 11-bit significand also carries p exactly enough that P
//     needs one term.  The uniform pool's fp32 scales would cost S 2^-11 of
//     relative accuracy if folded into fp16 K (with scores near 20 that moves
//     the lse by ~1e-3), so its K stays the exact fp16 value of the e4m3 byte:
//     each 64-column K-block (one scale group) gets its own TMEM accumulator,
//     and the math warps add the eight products times their fp32 scales.  V
//     (448 columns) is a second plane, the scaled value rounded once to fp16
//     (2^-12 relative in the output).  With that plane a tile holds 32 rows,
//     so that two stages fit beside Q.  A value beyond fp16's range (|x| >
//     65504) raises DSA_DEVERR_FP16_RANGE.
// (The "sparse attn" stage of tokenspeed PR #627 "Add gluon kernel for DSA";
// semantics of miles PR #3608: natural-log lse, -1 entries masked.)
//
// One CTA handles one (token, piece of its index list, group of <= 64 heads)
// and walks the piece in tiles of 64 gathered rows (32 for the uniform pool).
// Per tile:
//   S[h, kv] = Q[h, :] . K_tile[kv, :]          tcgen05 M = 64 (heads, Q
//                                                zero-padded to 64 rows),
//                                                N = 64 (kv), K = 576;
//                                                A = Q, B = the gathered tile
//   softmax over kv per head: with M = 64 the tensor core puts head 16q + i
//   in TMEM lane 32q + i, so lane i < 16 of math warp q owns one head's whole
//   row of 64 scores -- max, exp, sum and the P row are thread-local
//   O^T[dv, h] += V^T[dv, kv] . P^T[kv, h]      tcgen05 M = 128 (dv) x 4,
//                                                N = heads, K = 64 (kv);
//                                                A = the SAME gathered tile
//                                                read MN-major, B = P (K-major)
// so each gathered row is read from HBM once and serves as K and as V.
// P goes in as two bf16 terms P_hi + P_lo (P_lo in the tile's RoPE K-block,
// which S no longer needs), so the PV product carries p to ~2^-17 instead of
// bf16's 2^-9.  S (two buffers) and O^T live in TMEM.
//
// Online softmax with a lazy maximum: a head's reference maximum changes only
// when a tile exceeds it by more than 2^8 (in exp2 units); then O^T (all four
// math warps, one TMEM lane quadrant each) and the sums are rescaled.
// Otherwise p <= 256, exact in fp32 and representable in bf16.
//
// Two gather warps copy each tile's rows with 16-byte cp.async into the
// 128-byte-swizzled operand layout (a masked entry -- -1, out of range, or
// past the list's end -- is zero-filled and never read); Q arrives by TMA.
// Only two 72 KB stages fit beside Q, so each lane first pulls its rows into
// L2 a few tiles ahead: HBM streams ahead of the stages and the copies into
// shared memory see L2 latency.
// (A TMA row gather moves 512 bytes per instruction at a few tens of cycles
// of issue each; one warp of cp.async moves as much per instruction at a
// fraction of that.)
//
// S and PV are issued by four warps.  Small MMAs have a per-instruction
// issue floor (~55 cycles for any N <= 64 from one thread, however many
// accumulators it alternates between), and each further issuing thread adds
// its own stream.  S is split by K-block: warp 4 issues the even K-blocks
// into S_a, warp 10 the odd ones into S_b, and the softmax adds the two.  PV
// is split by dv block: warp 5 issues blocks 0-1, warp 11 blocks 2-3.  The S
// warps run ahead as soon as a tile has landed; the PV warps follow the
// softmax.
//
// Warps: 0-3 math, 4 and 10 S issue, 5 (and the Q load) and 11 PV issue,
// 6-9 gather.
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace dsa {

namespace {

// Warps 0-3 math, 4 and 10 S issue, 5 and 11 PV issue, 6-9 gather: 12
// warps, so at most 168 registers a thread (three warps share an SM
// sub-partition).
constexpr int kQKBlock = 64 * 128;       // one K-block of Q: 64 head rows x 64 16-bit values

enum { kFmtBf16 = 0, kFmtUniform = 1, kFmtPacked = 2 };
// Per pool format: K-blocks of 64 columns per row, stored V width, PV
// K-steps per 128-row block of dv (P_hi + P_lo for bf16, one fp16 term
// otherwise), and the operand type code of the instruction descriptor
// (1 = bf16, 0 = fp16).
template <int FMT> struct FmtTraits {
  // gathered rows per tile: 64, or 32 for the uniform pool, whose two fp16
  // planes per row would otherwise leave room for one stage only
  static constexpr int kRows = FMT == kFmtUniform ? 32 : 64;
  static constexpr int kKBlockBytes = kRows * 128;   // one K-block of a tile: kRows x 64 values
  static constexpr int kKBlocks = FMT == kFmtBf16 ? 9 : 8;
  static constexpr int kDv = FMT == kFmtBf16 ? 512 : 448;
  static constexpr int kPvSteps = FMT == kFmtBf16 ? 8 : kRows / 16;
  static constexpr uint32_t kOpType = FMT == kFmtBf16 ? 1u : 0u;
  // uniform pool: every 64-column K-block is one scale group, so S is the
  // sum over K-blocks g of scale[row, g] * (Q_g . K8_g), where K8 is the
  // e4m3 byte converted to fp16 (exact).  Each K-block's product has its own
  // TMEM accumulator (8 x 32 columns, one buffer) and the math warps apply
  // the fp32 scales as they add them up.  V (the first 448 columns) gets a
  // second plane: the scaled value rounded to fp16 once.
  static constexpr bool kGroupS = FMT == kFmtUniform;
  static constexpr int kVBlocks = kGroupS ? kKBlocks : 0;   // the scaled V plane
  static constexpr int kStages = 2;
  static constexpr int kStageBytes = (kKBlocks + kVBlocks) * kKBlockBytes;   // 72, 64 or 64 KB
  // rows are pulled into L2 this many tiles ahead (256 rows)
  static constexpr int kPrefetchTiles = 256 / kRows;
  // gather warps: four, 16 rows each per tile (bf16: cp.async issue split
  // four ways; fp8: every 16-byte load of a tile in flight at once)
  static constexpr int kGatherWarps = 4;
  static constexpr int kThreads = 32 * (8 + kGatherWarps);
  // register bound: with 12 warps three share an SM sub-partition (16K
  // registers), so at most 168 a thread
  static constexpr int kBoundThreads = 384;
  static constexpr int kQBytes = kKBlocks * 64 * 128;           // Q padded to 64 heads
};
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;      // log2 of the largest tolerated p

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

struct MlaSmem {
  uint32_t q, k, p, alpha, rows, gsc, inv_l, flag, bars, total;
};

template <int FMT>
__host__ __device__ inline MlaSmem mla_smem_layout() {
  using F = FmtTraits<FMT>;
  MlaSmem L;
  L.q = 0;
  L.k = L.q + F::kQBytes;
  L.p = L.k + F::kStages * F::kStageBytes;
  L.alpha = L.p + 64 * 128;          // [2][64] rescale factors, by tile parity
  L.rows = L.alpha + 2 * 64 * 4;     // [2][64] fp8 row descriptors, by tile parity
  L.gsc = L.rows + (FMT == kFmtBf16 ? 0 : 2 * 64 * 16);     // uniform: [2 stages][8 groups][32 rows] scales
  L.inv_l = L.gsc + (FmtTraits<FMT>::kGroupS ? 2 * 8 * 32 * 4 : 0);   // [64] 1 / final sums
  L.flag = L.inv_l + 64 * 4;         // [2][4] ints, by tile parity
  L.bars = L.flag + 32;              // 8-byte aligned
  L.total = L.bars + 32 * 8;
  return L;
}

// Pool slot of list entry e (of the concatenated main + extra list) of token
// t, or -1 when the entry is masked.  An entry other than -1 outside [0,
// rows) is reported through err_flag (when `report`) and masked like -1.
__device__ __forceinline__ int64_t entry_slot(const MlaArgs &a, int t, int e, bool report) {
  const PoolDev *pool;
  int64_t slot;
  if (e < a.k) {
    pool = &a.kv;
    slot = a.idx[(size_t)t * a.k + e];
  } else {
    pool = &a.kv2;
    slot = a.idx2[(size_t)t * a.k2 + (e - a.k)];
  }
  if (slot >= 0 && slot < pool->rows) return slot;
  if (report && slot != -1) raise_flag(a.err_flag, DSA_DEVERR_INDEX_RANGE);
  return -1;
}

// Pool addresses of an fp8 row (slot >= 0): its 512 (uniform) or 576
// (packed: 448 e4m3 + 64 bf16) payload bytes and its scales (8 fp32 |
// 7 UE8M0 bytes + pad).
struct Fp8Row {
  const uint8_t *data;
  const uint8_t *scale;
};
template <int FMT>
__device__ __forceinline__ Fp8Row fp8_row(const PoolDev &p, int64_t slot) {
  if (FMT == kFmtUniform)
    return {p.data + slot * 512, reinterpret_cast<const uint8_t *>(p.scales + slot * 8)};
  const int64_t page = slot / p.block, pos = slot - page * p.block;
  const uint8_t *pg = p.data + page * (int64_t)p.block * 584;
  return {pg + pos * 576, pg + (int64_t)p.block * 576 + pos * 8};
}

// 2^(e - 127) of a UE8M0 byte (e = 255 -> inf, which the range check reports)
__device__ __forceinline__ float ue8m0_scale(uint32_t e) {
  if (e == 0) return __int_as_float(0x00400000);
  if (e == 255) return INFINITY;
  return __int_as_float((int)(e << 23));
}

// Round a pair of fp32 values to an fp16 pair; *bad is set when either is
// not a finite fp16 value.
__device__ __forceinline__ uint32_t to_f16x2(float a, float b, bool &bad) {
  bad |= !(fabsf(a) <= 65504.f) || !(fabsf(b) <= 65504.f);
  const __half2 r = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&r);
}

// 16 e4m3 values (16 bytes, lowest address first) times s -> 16 fp16 in two
// 16-byte words, same order.
__device__ __forceinline__ void deq16_e4m3(const uint4 v, float s, uint4 &o0, uint4 &o1,
                                           bool &bad) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t h[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(
          (__nv_fp8x2_storage_t)((w[i] >> (16 * hh)) & 0xffffu), __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&r));
      h[2 * i + hh] = to_f16x2(f.x * s, f.y * s, bad);
    }
  }
  o0 = make_uint4(h[0], h[1], h[2], h[3]);
  o1 = make_uint4(h[4], h[5], h[6], h[7]);
}

// 16 e4m3 values times 2^k (a UE8M0 scale).  For k in [-15, 7] an fp16
// product is exact and cannot overflow (|e4m3| <= 448; 2^-9 * 2^-15 = 2^-24 is
// fp16's least subnormal), so it runs as packed half2 multiplies; other k
// take the fp32 path with the range check.
__device__ __forceinline__ void deq16_e4m3_pow2(const uint4 v, uint32_t e, uint4 &o0, uint4 &o1,
                                                bool &bad) {
  const int k = (int)e - 127;
  if (k < -15 || k > 7) {
    deq16_e4m3(v, ue8m0_scale(e), o0, o1, bad);
    return;
  }
  const unsigned short sb = k >= -14 ? (unsigned short)((k + 15) << 10) : (unsigned short)0x0200;
  const __half2 s2 = __half2half2(__ushort_as_half(sb));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t h[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(
          (__nv_fp8x2_storage_t)((w[i] >> (16 * hh)) & 0xffffu), __NV_E4M3);
      const __half2 x = __hmul2(*reinterpret_cast<const __half2 *>(&r), s2);
      h[2 * i + hh] = *reinterpret_cast<const uint32_t *>(&x);
    }
  }
  o0 = make_uint4(h[0], h[1], h[2], h[3]);
  o1 = make_uint4(h[4], h[5], h[6], h[7]);
}

// 16 e4m3 values -> their exact fp16 values (kx) and the values times s
// rounded to fp16 (vv), two 16-byte words each, same order.
__device__ __forceinline__ void deq16_e4m3_kx_v(const uint4 v, float s, uint4 (&kx)[2],
                                                uint4 (&vv)[2], bool &bad) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t h[8], r[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const __half2_raw raw = __nv_cvt_fp8x2_to_halfraw2(
          (__nv_fp8x2_storage_t)((w[i] >> (16 * hh)) & 0xffffu), __NV_E4M3);
      h[2 * i + hh] = *reinterpret_cast<const uint32_t *>(&raw);
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&raw));
      r[2 * i + hh] = to_f16x2(f.x * s, f.y * s, bad);
    }
  }
  kx[0] = make_uint4(h[0], h[1], h[2], h[3]);
  kx[1] = make_uint4(h[4], h[5], h[6], h[7]);
  vv[0] = make_uint4(r[0], r[1], r[2], r[3]);
  vv[1] = make_uint4(r[4], r[5], r[6], r[7]);
}

// 8 bf16 values (one 16-byte word) -> 8 fp16, same order.
__device__ __forceinline__ uint4 bf16x8_to_f16(const uint4 v, bool &bad) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    h[i] = to_f16x2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u), bad);
  return make_uint4(h[0], h[1], h[2], h[3]);
}

template <int FMT, int N>   // pool format; heads of the PV product (16, 32 or 64)
__global__ void __launch_bounds__(FmtTraits<FMT>::kBoundThreads, 1)
sparse_mla_tc_kernel(MlaArgs a, const __grid_constant__ CUtensorMap qmap, int per) {
  using F = FmtTraits<FMT>;
  constexpr int kKBlocks = F::kKBlocks;
  constexpr int kStageBytes = F::kStageBytes;
  constexpr int NS = F::kStages;   // tile i uses stage i % NS, phase (i / NS) & 1
  extern __shared__ __align__(1024) unsigned char smem[];
  const MlaSmem L = mla_smem_layout<FMT>();
  unsigned char *q_s = smem + L.q;
  unsigned char *k_s = smem + L.k;
  unsigned char *p_s = smem + L.p;
  float *alpha_s = reinterpret_cast<float *>(smem + L.alpha);
  float *inv_l = reinterpret_cast<float *>(smem + L.inv_l);
  volatile int *flag_s = reinterpret_cast<volatile int *>(smem + L.flag);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
  uint64_t *kfull = bars + 0;    // [2]
  uint64_t *kempty = bars + 2;   // [2]
  uint64_t *sfull = bars + 4;    // [2]
  uint64_t *sempty = bars + 6;   // [2]
  uint64_t *pfull = bars + 8;
  uint64_t *pempty = bars + 9;
  uint64_t *done = bars + 10;     // [2]: S warp, PV warp
  uint64_t *qfull = bars + 12;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 13);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 14);
  uint64_t *qready = bars + 15;   // fp8 pools: Q converted to fp16 by the math warps
  uint64_t *done2 = bars + 16;    // [2]: second S warp, second PV warp
  uint64_t *lastpv = bars + 22;   // [4]: the last tile's PV into dv block j retired

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x;
  const int split = blockIdx.y;
  const int h0 = blockIdx.z * 64;
  const int nh = min(64, a.H - h0);
  const int total = a.k + a.k2;
  const int j0 = min(total, split * per);   // per: a multiple of the tile
  const int je = min(total, j0 + per);
  constexpr int R = F::kRows;          // rows of a tile
  constexpr int RH = R / 2;            // scores of a head a math lane holds
  constexpr int kKBlockBytes = F::kKBlockBytes;
  constexpr int kPrefetchTiles = F::kPrefetchTiles;
  int nt = (je - j0 + R - 1) / R;       // tiles of the piece (trimmed below, one piece a token)
  // TMEM: S_a[2] at columns [0, 128), S_b[2] at [128, 256), O^T blocks at
  // [256, 256 + 4N)
  constexpr uint32_t kSCol = 0, kSbCol = 128, kOCol = 256;
  constexpr uint32_t kTmemCols = 512;

  if ((tc::smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need 1 KB alignment
    if (threadIdx.x == 0) raise_flag(a.err_flag, DSA_DEVERR_TIMEOUT);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&kfull[i], 32 * F::kGatherWarps);
      tc::mbar_init(&kempty[i], 2);       // both PV warps
      tc::mbar_init(&sfull[i], 2);        // both S warps
      tc::mbar_init(&sempty[i], 4);
    }
    tc::mbar_init(pfull, 4);
    tc::mbar_init(pempty, 2);             // both PV warps
    tc::mbar_init(&done[0], 1);
    tc::mbar_init(&done[1], 1);
    tc::mbar_init(&done2[0], 1);
    tc::mbar_init(&done2[1], 1);
    tc::mbar_init(qfull, 1);
    tc::mbar_init(qready, 4);
    for (int j = 0; j < 4; ++j) tc::mbar_init(&lastpv[j], 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 4) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // Q of this head group: 64-column boxes of 64 heads (heads past H lie
  // outside the map and read as zeros).  In the fused decode q precedes the
  // whole call, so it is loaded before waiting for the top-k kernel.
  auto load_q = [&]() {
    tc::prefetch_tmap(&qmap);
    tc::mbar_arrive_expect_tx(qfull, F::kQBytes);
    for (int kb = 0; kb < kKBlocks; ++kb)
      tc::tma_load_3d(&qmap, qfull, q_s + kb * kQKBlock, kb * 64, h0, t);
  };
  if (warp == 5 && lane == 0 && a.q_ready) load_q();
  pdl_wait();      // the index lists come from the previous kernel
  pdl_trigger();
  if (warp == 5 && lane == 0 && !a.q_ready) load_q();
  if (a.n_splits == 1) {
    // one piece a token (prefill): the tiles up to the list's last entry
    // other than -1 -- a causal prefill's early tokens end in a long -1 tail,
    // whose tiles would gather nothing.  (Split decode pieces skip this scan:
    // their lists are full, and the scan's load latency would precede every
    // piece.)
    int *last_s = reinterpret_cast<int *>(bars + 26);
    int last = -1;
    for (int e = j0 + threadIdx.x; e < je; e += blockDim.x) {
      const int32_t v = e < a.k ? __ldg(a.idx + (size_t)t * a.k + e)
                                : __ldg(a.idx2 + (size_t)t * a.k2 + (e - a.k));
      if (v != -1) last = e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    if (threadIdx.x == 0) *last_s = -1;
    __syncthreads();
    if (lane == 0 && last >= 0) atomicMax(last_s, last);
    __syncthreads();
    nt = (*last_s + 1 - j0 + R - 1) / R;
    if (nt < 0) nt = 0;
  }

  if (warp >= 6 && warp < 10 && FMT == kFmtBf16) {
    // -------------------------------------------------------------- gather (bf16)
    const int gw = warp - 6;            // rows [16*gw, 16*gw + 16) of every tile
    // this lane's row of tile i (row 16*gw + lane, lanes < 16), or nullptr
    auto row_of = [&](int i) -> const uint8_t * {
      const int e = j0 + i * R + 16 * gw + lane;
      if (lane >= 16 || e >= je) return nullptr;
      const int64_t slot = entry_slot(a, t, e, false);
      if (slot < 0) return nullptr;
      return (e < a.k ? a.kv.data : a.kv2.data) + slot * (int64_t)1152;
    };
    // each lane pulls its rows into L2 kPrefetchTiles tiles ahead of the copy
    // into shared memory, so the copy meets L2 latency instead of HBM's
    auto prefetch_row = [&](int i) {
      const uint8_t *row = row_of(i);
      if (row) {
#pragma unroll
        for (int c = 0; c < 9; ++c) prefetch_l2(row + 128 * c);
      }
    };
    for (int i = 1; i < min(nt, kPrefetchTiles); ++i) prefetch_row(i);   // tile 0 is copied at once
    const uint8_t *next = nt > 0 ? row_of(0) : nullptr;
    for (int i = 0; i < nt; ++i) {
      const int st = i % NS;
      const uint8_t *my_row = next;
      if (!tc::mbar_wait(&kempty[st], ((i / NS) & 1) ^ 1, abort_flag)) break;
      const uint32_t sbase = tc::smem_u32(k_s + st * kStageBytes);
#pragma unroll
      for (int r0 = 16 * gw; r0 < 16 * gw + 16; r0 += 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {       // row r0 + j: swizzle phase j
          const uint8_t *row = reinterpret_cast<const uint8_t *>(__shfl_sync(
              0xffffffffu, reinterpret_cast<unsigned long long>(my_row), (r0 & 15) + j));
          const uint8_t *src = row ? row : static_cast<const uint8_t *>(a.q);   // not read when masked
          const uint32_t nbytes = row ? 16u : 0u;
          const uint32_t rdst = sbase + (r0 + j) * 128;
#pragma unroll
          for (int q = 0; q < 3; ++q) {
            const int c = lane + 32 * q;          // 16-byte chunk of the row, 0..71
            if (c < 72)
              cp_async_16(rdst + (c >> 3) * kKBlockBytes + (((c & 7) ^ j) << 4),
                          src + (row ? c * 16 : 0), nbytes);
          }
        }
      }
      cp_async_commit();
      if (i + kPrefetchTiles < nt) prefetch_row(i + kPrefetchTiles);
      if (i + 1 < nt) next = row_of(i + 1);   // index loads overlap the copies
      cp_async_wait_all();
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&kfull[st]);
    }
    cp_async_wait_all();
    __syncwarp();
  } else if (warp >= 6 && warp < 10) {
    // -------------------------------------------------------------- gather (fp8)
    // A tile is a flat list of 16-byte chunks, CPR per row (uniform: 32 e4m3
    // chunks; packed: 28 e4m3 NoPE chunks + 8 bf16 RoPE chunks); gather lane
    // gl takes chunks gl + 128 j, issues all its loads, then dequantises them
    // to fp16 and stores them swizzled: chunk cc of a row covers columns
    // [16 cc, 16 cc + 16) (K-block cc / 4, 16-byte slots 2 (cc % 4) and +1),
    // a RoPE chunk the 8 columns 448 + 8 (cc - 28) (K-block 7, slot cc - 28).
    // Lanes 0..R-1 publish the tile's row addresses in shared memory first.
    constexpr int CPR = FMT == kFmtUniform ? 32 : 36;
    constexpr int CPL = R * CPR / 128;             // chunks per lane per tile
    const int gl = threadIdx.x - 192;              // 0..127
    Fp8Row *rtab = reinterpret_cast<Fp8Row *>(smem + L.rows);
    auto row_of = [&](int i) -> Fp8Row {
      Fp8Row r{nullptr, nullptr};
      const int e = j0 + i * R + gl;
      if (gl < R && e < je) {
        const int64_t slot = entry_slot(a, t, e, false);
        if (slot >= 0) r = fp8_row<FMT>(e < a.k ? a.kv : a.kv2, slot);
      }
      return r;
    };
    auto prefetch_row = [&](int i) {
      const Fp8Row r = row_of(i);
      if (r.data) {
        // the 128-byte lines of the row's payload (4 or 5), then its scales
        constexpr uintptr_t kBytes = FMT == kFmtUniform ? 512 : 576;
        const uintptr_t first = reinterpret_cast<uintptr_t>(r.data) >> 7;
        const uintptr_t last = (reinterpret_cast<uintptr_t>(r.data) + kBytes - 1) >> 7;
        for (uintptr_t ln = first; ln <= last; ++ln)
          prefetch_l2(reinterpret_cast<const void *>(ln << 7));
        prefetch_l2(r.scale);
      }
    };
    for (int i = 1; i < min(nt, kPrefetchTiles); ++i) prefetch_row(i);   // tile 0 is loaded at once
    bool bad = false;
    // The row table is double-buffered by tile parity: a lane reads tile i's
    // half only in issue(i), which every lane has left before any lane
    // passes the barrier of issue(i+1).  (Issuing tile i+1's loads before
    // converting tile i, into a second register set, was measured: no gain.)
    uint4 v[CPL];
    uint32_t sc[CPL];                     // fp32 scale bits (uniform) or UE8M0 byte (packed)
    uint32_t has = 0;
    Fp8Row next = nt > 0 ? row_of(0) : Fp8Row{nullptr, nullptr};
    auto issue = [&](int i) {             // publish tile i's rows, then load its chunks
      Fp8Row *rt = rtab + (i & 1) * 64;
      if (gl < R) rt[gl] = next;
      if (i + 1 < nt) next = row_of(i + 1);   // the next index loads overlap these
      tc::named_bar_sync(2, 128);
      has = 0;
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int c = gl + 128 * j;
        const int r = c / CPR, cc = c - r * CPR;
        const Fp8Row R = rt[r];
        v[j] = make_uint4(0u, 0u, 0u, 0u);
        sc[j] = 0u;
        if (R.data) {
          has |= 1u << j;
          if (FMT == kFmtUniform) {
            v[j] = __ldg(reinterpret_cast<const uint4 *>(R.data) + cc);
            sc[j] = __ldg(reinterpret_cast<const uint32_t *>(R.scale) + (cc >> 2));
          } else if (cc < 28) {
            v[j] = __ldg(reinterpret_cast<const uint4 *>(R.data) + cc);
            sc[j] = __ldg(R.scale + (cc >> 2));
          } else {
            v[j] = __ldg(reinterpret_cast<const uint4 *>(R.data + 448) + (cc - 28));
          }
        }
      }
    };
    if (nt > 0) issue(0);
    for (int i = 0; i < nt; ++i) {
      const int st = i % NS;
      if (!tc::mbar_wait(&kempty[st], ((i / NS) & 1) ^ 1, abort_flag)) break;
      unsigned char *stage = k_s + st * kStageBytes;
      const uint32_t chas = has;
      auto chunk = [&](int j) -> const uint4 & { return v[j]; };
      auto scale = [&](int j) -> uint32_t { return sc[j]; };
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int c = gl + 128 * j;
        const int r = c / CPR, cc = c - r * CPR;
        const uint32_t ph = (uint32_t)(r & 7);
        const bool hv = (chas >> j) & 1u;
        if (FMT == kFmtPacked && cc >= 28) {
          const uint4 o = hv ? bf16x8_to_f16(chunk(j), bad) : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4 *>(stage + 7 * kKBlockBytes + r * 128 +
                                     (((uint32_t)(cc - 28) ^ ph) << 4)) = o;
          continue;
        }
        uint4 o[2], ol[2];
        o[0] = o[1] = ol[0] = ol[1] = make_uint4(0u, 0u, 0u, 0u);
        if (hv) {
          if (FMT == kFmtUniform)
            deq16_e4m3_kx_v(chunk(j), __uint_as_float(scale(j)), o, ol, bad);
          else
            deq16_e4m3_pow2(chunk(j), scale(j), o[0], o[1], bad);
        }
        const uint32_t s0 = 2u * (uint32_t)(cc & 3);
        unsigned char *rowp = stage + (cc >> 2) * kKBlockBytes + r * 128;
        *reinterpret_cast<uint4 *>(rowp + ((s0 ^ ph) << 4)) = o[0];
        *reinterpret_cast<uint4 *>(rowp + (((s0 + 1) ^ ph) << 4)) = o[1];
        if (FMT == kFmtUniform) {
          unsigned char *vp = rowp + kKBlocks * kKBlockBytes;   // the scaled V plane
          *reinterpret_cast<uint4 *>(vp + ((s0 ^ ph) << 4)) = ol[0];
          *reinterpret_cast<uint4 *>(vp + (((s0 + 1) ^ ph) << 4)) = ol[1];
          // the row's group scale (0 for a masked row: its S terms are masked anyway)
          if ((cc & 3) == 0)
            reinterpret_cast<float *>(smem + L.gsc)[(st * 8 + (cc >> 2)) * 32 + r] =
                hv ? __uint_as_float(scale(j)) : 0.f;
        }
      }
      if (i + kPrefetchTiles < nt) prefetch_row(i + kPrefetchTiles);
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&kfull[st]);
      if (i + 1 < nt) issue(i + 1);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_flag(a.err_flag, DSA_DEVERR_FP16_RANGE);
    __syncwarp();
  } else if (warp == 4 || warp == 10) {
    // -------------------------------------------------------------- S issue
    // warp 4: the even K-blocks into S_a; warp 10: the odd ones into S_b
    const int sh = warp == 10 ? 1 : 0;
    if (lane == 0) {
      // S = Q K^T: A = Q (K-major, M = 64), B = K tile (K-major, N = 64)
      constexpr uint32_t idesc_s = tc::idesc_f32acc(F::kOpType, F::kOpType, 0, 0, R, 64);
      const uint64_t adq = tc::sdesc_sw128(tc::smem_u32(q_s), 16, 1024);
      bool ok = nt == 0 || tc::mbar_wait(FMT == kFmtBf16 ? qfull : qready, 0, abort_flag);
      for (int i = 0; i < nt && ok; ++i) {
        const int st = i % NS;              // K stage
        const int sb = i & 1;               // S buffer in TMEM
        if (!tc::mbar_wait(&kfull[st], (i / NS) & 1, abort_flag)) break;
        // one S buffer for the per-group accumulators (uniform pool), else two
        if (!tc::mbar_wait(&sempty[F::kGroupS ? 0 : sb],
                           ((F::kGroupS ? i : (i >> 1)) & 1) ^ 1, abort_flag))
          break;
        tc::fence_after_sync();
        // descriptors: the start-address field is the byte address / 16, so
        // a K-block of Q (8192 B) adds 512, one of the tile kKBlockBytes / 16,
        // and 32 bytes of K add 2
        const uint64_t bdk = tc::sdesc_sw128(tc::smem_u32(k_s + st * kStageBytes), 16, 1024);
        const uint32_t dcol = tmem + (sh ? kSbCol : kSCol) + sb * 64;
#pragma unroll
        for (int kb = 0; kb < kKBlocks; ++kb) {
          if ((kb & 1) != sh) continue;
          if constexpr (F::kGroupS) {      // K-block kb into its own accumulator
#pragma unroll
            for (int ko = 0; ko < 4; ++ko)
              tc::mma_f16(tmem + kSCol + kb * R, adq + kb * 512 + 2 * ko,
                          bdk + kb * (kKBlockBytes >> 4) + 2 * ko, idesc_s, ko > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int ko = 0; ko < 4; ++ko)   // 32 bytes (16 values) of K per instruction
              tc::mma_f16(dcol, adq + kb * 512 + 2 * ko, bdk + kb * (kKBlockBytes >> 4) + 2 * ko,
                          idesc_s, (kb > sh || ko > 0) ? 1u : 0u);
          }
        }
        tc::mma_commit(&sfull[F::kGroupS ? 0 : sb]);
      }
      if (nt > 0) {
        // this warp's MMAs retired before TMEM is released
        uint64_t *d = sh ? &done2[0] : &done[0];
        tc::mma_commit(d);
        tc::mbar_wait_drain(d, 0);
      }
    }
    __syncwarp();
  } else if (warp == 5 || warp == 11) {
    // -------------------------------------------------------------- PV issue
    // warp 5: dv blocks 0 and 1; warp 11: blocks 2 and 3
    const int ph = warp == 11 ? 1 : 0;
    if (lane == 0) {
      // O^T += V^T P^T: A = V^T (MN-major, M = 128), B = P (K-major, N heads)
      constexpr uint32_t idesc_pv = tc::idesc_f32acc(F::kOpType, F::kOpType, 1, 0, N, 128);
      const uint32_t p_addr = tc::smem_u32(p_s);
      for (int i = 0; i < nt; ++i) {
        const int st = i % NS;
        if (!tc::mbar_wait(pfull, i & 1, abort_flag)) break;
        tc::fence_after_sync();
        const uint32_t k_addr = tc::smem_u32(k_s + st * kStageBytes);
        // A = V^T: dv block j is K-blocks 2j, 2j+1 (+2 kKBlockBytes / 16 in the
        // descriptor), 16 kv rows = 2048 B (+128); B = P (or P_lo, bf16: the
        // RoPE block), 16 kv = 32 B (+2)
        const uint64_t adv =
            tc::sdesc_sw128(k_addr + (F::kGroupS ? kKBlocks * kKBlockBytes : 0), kKBlockBytes, 1024);
        const uint64_t bdp = tc::sdesc_sw128(p_addr, 16, 1024);
        const uint64_t bdl = tc::sdesc_sw128(k_addr + 8 * kKBlockBytes, 16, 1024);
#pragma unroll
        for (int j = 2 * ph; j < 2 * ph + 2; ++j) {
#pragma unroll
          for (int kk = 0; kk < F::kPvSteps; ++kk) {
            const uint32_t kr = kk & 3;   // 16 kv rows per instruction
            tc::mma_f16(tmem + kOCol + j * N, adv + j * (kKBlockBytes >> 3) + kr * 128,
                        (kk < 4 ? bdp : bdl) + kr * 2, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
          }
          if (i == nt - 1) tc::mma_commit(&lastpv[j]);   // the epilogue of block j may start
        }
        tc::mma_commit(&kempty[st]);
        tc::mma_commit(pempty);
      }
      if (nt > 0) tc::mma_commit(ph ? &done2[1] : &done[1]);   // waited for after the epilogue
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- math
    const int quad = warp;                  // TMEM lane quadrant
    // lanes l and l+16 share head 16q + l % 16: lane l < 16 holds its scores
    // of kv 0..31, lane l+16 those of kv 32..63 (one 16x32bx2 TMEM load)
    const int hl = 16 * quad + (lane & 15);
    const int half = lane >> 4;
    const bool head_lane = half == 0;       // the lane that writes per-head results
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    // The scores stay in the frame of the raw products S = q . K: the
    // reference maximum m is a raw product, p = exp2((S - m) c) with c =
    // softmax_scale log2(e), and the lse is softmax_scale m + ln l.  Rounding
    // S c or m c first would cost the lse several ulps of its magnitude (an
    // fp8 pool with UE8M0 exponents up to 2^7 gives scores near 300).
    const float c = a.softmax_scale * kLog2e;
    float m = -INFINITY;                    // reference maximum (raw products)
    float l = 0.f;                          // running sum of p
    bool ok = true;
    if (FMT != kFmtBf16) {
      // Q (bf16 from the TMA load) -> fp16 in place, elementwise, so the
      // swizzled layout is unchanged
      if (nt > 0 && !tc::mbar_wait(qfull, 0, abort_flag)) ok = false;
      bool bad = false;
      if (ok) {
        uint4 *qw = reinterpret_cast<uint4 *>(q_s);
        for (int i2 = threadIdx.x; i2 < F::kQBytes / 16; i2 += 128)
          qw[i2] = bf16x8_to_f16(qw[i2], bad);
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) raise_flag(a.err_flag, DSA_DEVERR_FP16_RANGE);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(qready);
    }
    for (int i = 0; i < nt && ok; ++i) {
      const int b = i & 1;                  // S buffer of tile i (= its K stage with two stages)
      // validity of the R entries of this tile as a bit mask (1 or 2 loads a lane)
      const int e = j0 + i * R + lane;
      const bool v_lo = e < je && entry_slot(a, t, e, quad == 0) >= 0;
      const bool v_hi = R > 32 && e + 32 < je && entry_slot(a, t, e + 32, quad == 0) >= 0;
      const uint32_t vm_lo = __ballot_sync(0xffffffffu, v_lo);
      const uint32_t vm_hi = __ballot_sync(0xffffffffu, v_hi);
      if (!tc::mbar_wait(&sfull[F::kGroupS ? 0 : b], (F::kGroupS ? i : (i >> 1)) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      float x[RH];                          // this lane's half of its head's R scores
      if constexpr (F::kGroupS) {
        // S = sum over groups g of scale[row, g] * S_g (rows RH half .. + RH - 1)
        const float *gs = reinterpret_cast<const float *>(smem + L.gsc) + (i % NS) * 8 * 32 + RH * half;
#pragma unroll
        for (int j = 0; j < RH; ++j) x[j] = 0.f;
#pragma unroll 1
        for (int g = 0; g < kKBlocks; ++g) {
          float sg[RH];
          tc::tmem_ld_16x32bx2_x16<16>(tmem + lane_base + kSCol + g * R, sg);
#pragma unroll
          for (int j = 0; j < RH; j += 4) {
            const float4 sc4 = *reinterpret_cast<const float4 *>(gs + g * 32 + j);
            x[j] = fmaf(sg[j], sc4.x, x[j]);
            x[j + 1] = fmaf(sg[j + 1], sc4.y, x[j + 1]);
            x[j + 2] = fmaf(sg[j + 2], sc4.z, x[j + 2]);
            x[j + 3] = fmaf(sg[j + 3], sc4.w, x[j + 3]);
          }
        }
      } else {
        float xb[RH];                       // S = S_a + S_b (even and odd K-blocks)
        if constexpr (R == 64) {
          tc::tmem_ld_16x32bx2_x32<32>(tmem + lane_base + kSCol + b * 64, x);
          tc::tmem_ld_16x32bx2_x32<32>(tmem + lane_base + kSbCol + b * 64, xb);
        } else {
          tc::tmem_ld_16x32bx2_x16<16>(tmem + lane_base + kSCol + b * 64, x);
          tc::tmem_ld_16x32bx2_x16<16>(tmem + lane_base + kSbCol + b * 64, xb);
        }
#pragma unroll
        for (int j = 0; j < RH; ++j) x[j] += xb[j];
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sempty[F::kGroupS ? 0 : b]);
      // this lane's entries: kv RH * half + j
      const uint32_t vm = R == 64 ? (half ? vm_hi : vm_lo) : (vm_lo >> (RH * half));
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < RH; ++j) {
        x[j] = ((vm >> j) & 1u) ? x[j] : -INFINITY;
        tmax = fmaxf(tmax, x[j]);
      }
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));   // the head's maximum
      float al = 1.f;
      int need = 0;
      // both lanes of the pair decide alike; nothing valid yet on either
      // side: (-inf) - (-inf) is NaN and the test fails
      if ((tmax - m) * c > kLazy) {
        al = (m == -INFINITY) ? 0.f : exp2f((m - tmax) * c);
        m = tmax;
        need = 1;
      }
      // a rescale of O^T needs every lane of every math warp; the factors and
      // flags are double-buffered by tile parity so that a warp running ahead
      // never overwrites what a slower warp still reads
      float *alpha = alpha_s + b * 64;
      volatile int *flag = flag_s + b * 4;
      need = __any_sync(0xffffffffu, need);
      if (lane == 0) flag[quad] = need;
      if (head_lane) alpha[hl] = al;
      tc::named_bar_sync(1, 128);
      const int rescale = flag[0] | flag[1] | flag[2] | flag[3];
      // p = exp2(x - m), its sum, and this lane's half of the P row (bf16:
      // P_hi + P_lo; fp8 pools: one fp16 term)
      const float msafe = m == -INFINITY ? 0.f : m;   // all masked so far: p = 0
      float ps = 0.f;
      uint32_t phi[RH / 2], plo[4];
#pragma unroll
      for (int j = 0; j < RH; j += 2) {
        const float p0 = exp2f((x[j] - msafe) * c);      // -inf -> 0
        const float p1 = exp2f((x[j + 1] - msafe) * c);
        ps += p0 + p1;
        if (FMT == kFmtBf16) {
          const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
          const float2 hf = __bfloat1622float2(hi);
          phi[j / 2] = *reinterpret_cast<const uint32_t *>(&hi);
          plo[(j / 2) & 3] = pack_bf16x2(p0 - hf.x, p1 - hf.y);
          if ((j & 7) == 6 && hl < N) {
            // P_lo goes straight into this tile's RoPE block (free once S(i)
            // has read it; PV(i-1) never reads it): 8 kv = one 16-byte chunk
            const int ch = 4 * half + (j >> 3);
            *reinterpret_cast<uint4 *>(k_s + (i % NS) * kStageBytes + 8 * kKBlockBytes + hl * 128 +
                                       ((ch ^ (hl & 7)) << 4)) =
                make_uint4(plo[0], plo[1], plo[2], plo[3]);
          }
        } else {
          const __half2 ph = __floats2half2_rn(p0, p1);   // p <= 256: 2^-11 relative
          phi[j / 2] = *reinterpret_cast<const uint32_t *>(&ph);
        }
      }
      ps += __shfl_xor_sync(0xffffffffu, ps, 16);   // the head's sum, alike in both lanes
      l = l * al + ps;
      // P and O^T may be touched only after PV(i-1) retired
      if (i >= 1) {
        if (!tc::mbar_wait(pempty, (i - 1) & 1, abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
      }
      if (rescale && i >= 1) {
#pragma unroll 1
        for (int j = 0; j < 4; ++j) tc::tmem_scale_cols<N>(tmem + lane_base + kOCol + j * N, alpha);
      }
      if (hl < N) {
        // row hl of P (K-major B operand): R kv 16-bit values in a 128-byte
        // swizzled row; this lane's half is chunks CH half .. CH half + CH - 1
        constexpr int CH = RH / 8;          // 16-byte chunks a lane writes
#pragma unroll
        for (int cc = 0; cc < CH; ++cc) {
          const int ch = CH * half + cc;
          const uint32_t off = hl * 128 + ((ch ^ (hl & 7)) << 4);
          *reinterpret_cast<uint4 *>(p_s + off) =
              make_uint4(phi[4 * cc], phi[4 * cc + 1], phi[4 * cc + 2], phi[4 * cc + 3]);
        }
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(pfull);
    }
    // ---- per-head results: 1 / l for the epilogue, and the lse (one piece:
    // with the head's sink folded in, if any; split pieces: the combine folds it)
    if (head_lane) {
      float inv = (l > 0.f) ? 1.f / l : 0.f;
      float lse = l > 0.f ? fmaf(m, a.softmax_scale, logf(l)) : -INFINITY;
      if (a.n_splits == 1 && a.sinks && hl < nh)
        inv = fold_sink(m, a.softmax_scale, l, a.sinks[h0 + hl], &lse);
      inv_l[hl] = inv;
      if (hl < nh) {
        if (a.n_splits == 1)
          a.lse[(size_t)t * a.H + h0 + hl] = lse_report(lse, a.lse_log2);
        else
          a.part_lse[((size_t)t * a.n_splits + split) * a.H + h0 + hl] = lse;
      }
    }
    tc::named_bar_arrive(3, 256);    // inv_l is written: warps 4-7 may start
    tc::named_bar_sync(1, 128);
  }

  // ---- epilogue: O^T / l per head, read from TMEM by warps 0-7 (warp w
  // reaches TMEM lane quadrant w % 4): warps 0-3 take dv blocks 0 and 1,
  // warps 4-7 blocks 2 and 3, each block as soon as the last tile's PV into
  // it has retired.  This CTA's records: [nh heads][kDv] bf16 (one piece) or
  // fp32 partials.
  if (warp < 8) {
    if (warp >= 4) tc::named_bar_sync(3, 256);
    constexpr int kDv = F::kDv;
    const int quad = warp & 3;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const size_t rec0 = a.n_splits == 1 ? (size_t)t * a.H + h0
                                        : ((size_t)t * a.n_splits + split) * a.H + h0;
#pragma unroll 1
    for (int j = 2 * (warp >> 2); j < 2 * (warp >> 2) + 2; ++j) {
      const int dv = 128 * j + 32 * quad + lane;
      if (128 * j + 32 * quad >= kDv) break;   // warp-uniform: the RoPE columns of fp8 rows
      bool have_o = nt > 0 && !*abort_flag;
      if (have_o) {
        have_o = tc::mbar_wait(&lastpv[j], 0, abort_flag);
        tc::fence_after_sync();
      }
      float o[N];
      if (have_o) {
        tc::tmem_ld_cols<N>(tmem + lane_base + kOCol + j * N, o);
      } else {
#pragma unroll
        for (int h = 0; h < N; ++h) o[h] = 0.f;
      }
      if (a.n_splits == 1) {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) + rec0 * kDv + dv;
#pragma unroll
        for (int hq = 0; hq < N; ++hq)
          if (hq < nh) dst[hq * kDv] = __float2bfloat16_rn(o[hq] * inv_l[hq]);
      } else {
        float *dst = a.part_o + rec0 * kDv + dv;
#pragma unroll
        for (int hq = 0; hq < N; ++hq)
          if (hq < nh) dst[hq * kDv] = o[hq] * inv_l[hq];
      }
    }
  }
  if (warp == 5 && lane == 0) {
    // the PV warps' MMAs retired and the Q load landed before TMEM is released
    if (nt > 0) tc::mbar_wait_drain(&done[1], 0);
    tc::mbar_wait_drain(qfull, 0);
  }
  if (warp == 11 && lane == 0 && nt > 0) tc::mbar_wait_drain(&done2[1], 0);

  tc::fence_before_sync();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) raise_flag(a.err_flag, DSA_DEVERR_TIMEOUT);
  if (warp == 4) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int FMT, int N>
cudaError_t launch_n(const MlaArgs &a, cudaStream_t s) {
  using F = FmtTraits<FMT>;
  CUtensorMap qmap;
  // Q [T][H][D] bf16 in boxes of 64 columns x 64 heads
  if (!make_tmap_3d(&qmap, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)F::kKBlocks * 64,
                    (uint64_t)a.H, (uint64_t)a.T, 64, 64, 1))
    return cudaErrorInvalidValue;
  const int total = a.k + a.k2;
  int per = (total + a.n_splits - 1) / a.n_splits;
  per = (per + F::kRows - 1) / F::kRows * F::kRows;
  const MlaSmem L = mla_smem_layout<FMT>();
  auto kern = sparse_mla_tc_kernel<FMT, N>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)a.T, (unsigned)a.n_splits, (unsigned)((a.H + 63) / 64));
  return launch_pdl(kern, grid, dim3(F::kThreads), L.total, s, a, qmap, per);
}

template <int FMT>
cudaError_t launch_fmt(const MlaArgs &a, cudaStream_t s) {
  const int hg = a.H >= 64 ? 64 : a.H;
  if (hg <= 16) return launch_n<FMT, 16>(a, s);
  if (hg <= 32) return launch_n<FMT, 32>(a, s);
  return launch_n<FMT, 64>(a, s);
}

}  // namespace

int sparse_mla_tc_format(const MlaArgs &a) {
  // Q is read by TMA (16-byte aligned base); fp8 rows are read as 16-byte
  // words (16-byte aligned pool data; packed pages of an even token count)
  if ((reinterpret_cast<uintptr_t>(a.q) & 15) != 0) return -1;
  if (a.D == 576 && a.Dv == 512 && a.kv.format == DSA_KV_BF16 &&
      (a.k2 == 0 || a.kv2.format == DSA_KV_BF16))
    return kFmtBf16;
  auto fp8_ok = [](const PoolDev &p) {
    if ((reinterpret_cast<uintptr_t>(p.data) & 15) != 0) return false;
    if (p.format == DSA_KV_FP8_UNIFORM) return p.scales != nullptr;
    return p.format == DSA_KV_FP8_DS_MLA && p.block >= 2 && p.block % 2 == 0;
  };
  if (a.D == 512 && a.Dv == 448 && fp8_ok(a.kv) &&
      (a.k2 == 0 || (a.kv2.format == a.kv.format && fp8_ok(a.kv2))))
    return a.kv.format == DSA_KV_FP8_UNIFORM ? kFmtUniform : kFmtPacked;
  return -1;
}

cudaError_t sparse_mla_tc_launch(const MlaArgs &a, int fmt, cudaStream_t s) {
  if (fmt == kFmtBf16) return launch_fmt<kFmtBf16>(a, s);
  if (fmt == kFmtUniform) return launch_fmt<kFmtUniform>(a, s);
  return launch_fmt<kFmtPacked>(a, s);
}

}  // namespace dsa
