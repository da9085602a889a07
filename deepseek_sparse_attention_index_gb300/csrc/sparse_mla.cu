// Absorbed-MLA sparse attention forward over gathered latent rows
// (the "sparse attn" stage of tokenspeed PR #627 "Add gluon kernel for DSA";
// semantics of miles PR #3608: natural-log lse, -1 entries masked; pool
// formats and the two-loop list of aiter PR #4382).
//
// Split-KV: the concatenated list (idx then idx2) of a token is cut into
// n_splits pieces; each CTA handles one (token, piece, group of <= 64 heads)
// with an online softmax and writes a normalised partial output and its lse;
// a combine kernel merges the pieces (lse = ln sum exp lse_i, out = sum
// exp(lse_i - lse) out_i).  With one piece the CTA writes the result itself.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 8;        // rows gathered per step
constexpr int kHeadsPerCta = 64;
constexpr int kKStride = 580;   // float row stride of the gathered tile (bank spread)
constexpr int kQStride = 584;   // bf16 row stride of q in shared memory
constexpr float kLog2e = 1.4426950408889634f;

// Fetch list entry j (of the concatenated list) for token t: slot and pool.
struct ListRef {
  const PoolDev *pool;
  int64_t slot;
};

__device__ __forceinline__ ListRef list_entry(const MlaArgs &a, int t, int j) {
  ListRef r;
  if (j < a.k) {
    r.pool = &a.kv;
    r.slot = a.idx[(size_t)t * a.k + j];
  } else {
    r.pool = &a.kv2;
    r.slot = a.idx2[(size_t)t * a.k2 + (j - a.k)];
  }
  return r;
}

// Dequantise one latent row into dst[0..D) (fp32).  32 threads (one warp).
__device__ __forceinline__ void load_row(const PoolDev &p, int64_t slot, int D, float *dst) {
  const unsigned lane = lane_id();
  if (p.format == DSA_KV_BF16) {
    const uint32_t *src = reinterpret_cast<const uint32_t *>(p.data + slot * (int64_t)D * 2);
    for (int c = 2 * lane; c < D; c += 64) {
      const uint32_t v = __ldg(src + c / 2);
      dst[c] = __uint_as_float(v << 16);
      dst[c + 1] = __uint_as_float(v & 0xffff0000u);
    }
  } else if (p.format == DSA_KV_FP8_UNIFORM) {
    const uint16_t *src = reinterpret_cast<const uint16_t *>(p.data + slot * (int64_t)D);
    const float *sc = p.scales + slot * (int64_t)(D / 64);
    for (int c = 2 * lane; c < D; c += 64) {
      const float s = __ldg(sc + c / 64);
      const float2 v = e4m3x2_to_float2(__ldg(src + c / 2));
      dst[c] = v.x * s;
      dst[c + 1] = v.y * s;
    }
  } else {  // fp8_ds_mla: 448 NoPE fp8 + 64 RoPE bf16, UE8M0 per 64 NoPE dims
    const int64_t page = slot / p.block, pos = slot % p.block;
    const uint8_t *pg = p.data + page * (int64_t)p.block * 584;
    const uint8_t *row = pg + pos * 576;
    const uint8_t *ex = pg + (int64_t)p.block * 576 + pos * 8;
    const uint16_t *nope = reinterpret_cast<const uint16_t *>(row);
    for (int c = 2 * lane; c < 448; c += 64) {
      const float s = ue8m0_to_float(__ldg(ex + c / 64));
      const float2 v = e4m3x2_to_float2(__ldg(nope + c / 2));
      dst[c] = v.x * s;
      dst[c + 1] = v.y * s;
    }
    const uint32_t *rope = reinterpret_cast<const uint32_t *>(row + 448);
    const uint32_t v = __ldg(rope + lane);
    dst[448 + 2 * lane] = __uint_as_float(v << 16);
    dst[448 + 2 * lane + 1] = __uint_as_float(v & 0xffff0000u);
  }
}

template <int DV>
__global__ void __launch_bounds__(kThreads)
sparse_mla_simt_kernel(MlaArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float *k_s = reinterpret_cast<float *>(smem_raw);                       // [kRows][kKStride]
  float *p_s = k_s + kRows * kKStride;                                      // [64][kRows]
  __nv_bfloat16 *q_s = reinterpret_cast<__nv_bfloat16 *>(p_s + kHeadsPerCta * kRows);  // [64][kQStride]
  __shared__ int s_valid[kRows];

  const int t = blockIdx.x;
  const int split = blockIdx.y;
  const int h0 = blockIdx.z * kHeadsPerCta;
  const int nh = min(kHeadsPerCta, a.H - h0);
  const int D = a.D;
  const int total = a.k + a.k2;
  const int per = (total + a.n_splits - 1) / a.n_splits;
  const int jb = split * per;
  const int je = min(total, jb + per);

  // q for this head group
  {
    const uint16_t *qg = static_cast<const uint16_t *>(a.q) + ((size_t)t * a.H + h0) * D;
    uint16_t *qs = reinterpret_cast<uint16_t *>(q_s);
    for (int i = threadIdx.x; i < kHeadsPerCta * D; i += blockDim.x) {
      const int h = i / D, c = i % D;
      qs[h * kQStride + c] = h < nh ? qg[(size_t)h * D + c] : (uint16_t)0;
    }
  }
  const int hl = threadIdx.x >> 2;     // head within the group
  const int part = threadIdx.x & 3;    // which quarter of the row work
  constexpr int NACC = DV / 16 * 4;    // dv values owned: dv = 16*i + 4*part + e
  float o[NACC];
#pragma unroll
  for (int i = 0; i < NACC; ++i) o[i] = 0.f;
  // m: running maximum of the raw products q . K (the scores before the
  // softmax scale); p = exp2((x - m) sc), lse = softmax_scale m + ln l
  float m = -INFINITY, l = 0.f;
  const float sc = a.softmax_scale * kLog2e;
  __syncthreads();

  for (int j0 = jb; j0 < je; j0 += kRows) {
    // gather: warp w loads row j0 + w
    const int w = threadIdx.x >> 5;
    if (w < kRows) {
      const int j = j0 + w;
      int ok = 0;
      if (j < je) {
        ListRef e = list_entry(a, t, j);
        if (e.slot >= 0 && e.slot < e.pool->rows) {
          ok = 1;
          load_row(*e.pool, e.slot, D, k_s + w * kKStride);
        } else if (e.slot != -1 && lane_id() == 0) {
          raise_flag(a.err_flag, DSA_DEVERR_INDEX_RANGE);
        }
      }
      if (lane_id() == 0) s_valid[w] = ok;
    }
    __syncthreads();
    // scores: thread (hl, part) takes rows 2*part, 2*part+1
    float s2[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = 2 * part + rr;
      float x = 0.f;
      if (s_valid[r]) {
        const float *kr = k_s + r * kKStride;
        const __nv_bfloat162 *qh = reinterpret_cast<const __nv_bfloat162 *>(q_s + hl * kQStride);
        // four partial sums (columns c mod 4), added pairwise at the end
        float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
        for (int c = 0; c < D; c += 4) {
          const float4 kv = *reinterpret_cast<const float4 *>(kr + c);
          const float2 qa = __bfloat1622float2(qh[c / 2]);
          const float2 qb = __bfloat1622float2(qh[c / 2 + 1]);
          x0 = fmaf(qa.x, kv.x, x0);
          x1 = fmaf(qa.y, kv.y, x1);
          x2 = fmaf(qb.x, kv.z, x2);
          x3 = fmaf(qb.y, kv.w, x3);
        }
        x = (x0 + x1) + (x2 + x3);
      } else {
        x = -INFINITY;
      }
      s2[rr] = x;
    }
    // online softmax over the 8 rows for this head (4 lanes share a head)
    float cmax = fmaxf(s2[0], s2[1]);
    cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 1));
    cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 2));
    const float mn = fmaxf(m, cmax);
    float alpha, p0, p1;
    if (mn == -INFINITY) {
      alpha = 1.f; p0 = 0.f; p1 = 0.f;
    } else {
      alpha = exp2f((m - mn) * sc);
      p0 = exp2f((s2[0] - mn) * sc);
      p1 = exp2f((s2[1] - mn) * sc);
    }
    float ps = p0 + p1;
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    l = l * alpha + ps;
    m = mn;
    p_s[hl * kRows + 2 * part] = p0;
    p_s[hl * kRows + 2 * part + 1] = p1;
    __syncthreads();
    float pr[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) pr[r] = p_s[hl * kRows + r];
#pragma unroll
    for (int i = 0; i < DV / 16; ++i) {
      const int dv = 16 * i + 4 * part;
      float4 acc = make_float4(o[4 * i] * alpha, o[4 * i + 1] * alpha, o[4 * i + 2] * alpha,
                               o[4 * i + 3] * alpha);
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        if (pr[r] != 0.f) {
          const float4 v = *reinterpret_cast<const float4 *>(k_s + r * kKStride + dv);
          acc.x = fmaf(pr[r], v.x, acc.x);
          acc.y = fmaf(pr[r], v.y, acc.y);
          acc.z = fmaf(pr[r], v.z, acc.z);
          acc.w = fmaf(pr[r], v.w, acc.w);
        }
      }
      o[4 * i] = acc.x; o[4 * i + 1] = acc.y; o[4 * i + 2] = acc.z; o[4 * i + 3] = acc.w;
    }
    __syncthreads();
  }

  if (hl >= nh) return;
  const int h = h0 + hl;
  float inv = l > 0.f ? 1.f / l : 0.f;
  float lse_v = l > 0.f ? fmaf(m, a.softmax_scale, logf(l)) : -INFINITY;
  if (a.n_splits == 1 && a.sinks) inv = fold_sink(m, a.softmax_scale, l, a.sinks[h], &lse_v);
  if (a.n_splits == 1) {
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + ((size_t)t * a.H + h) * a.Dv;
#pragma unroll
    for (int i = 0; i < DV / 16; ++i) {
      const int dv = 16 * i + 4 * part;
      uint2 pk;
      pk.x = pack_bf16x2(o[4 * i] * inv, o[4 * i + 1] * inv);
      pk.y = pack_bf16x2(o[4 * i + 2] * inv, o[4 * i + 3] * inv);
      *reinterpret_cast<uint2 *>(out + dv) = pk;
    }
    if (part == 0) a.lse[(size_t)t * a.H + h] = lse_report(lse_v, a.lse_log2);
  } else {
    const size_t rec = ((size_t)t * a.n_splits + split) * a.H + h;
    float *po = a.part_o + rec * a.Dv;
#pragma unroll
    for (int i = 0; i < DV / 16; ++i) {
      const int dv = 16 * i + 4 * part;
      *reinterpret_cast<float4 *>(po + dv) =
          make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
    }
    if (part == 0) a.part_lse[rec] = lse_v;
  }
}

// Merge split partials.  A warp per (token, head) record, or, for a call with
// few records (a single-token decode: 64 records), a CTA of eight warps per
// record: a warp per quarter of the columns and half of the splits, the two
// halves then merged through shared memory, so that such a call still has a
// few hundred warps and up to 32 splits wait for one round of L2 latency.
// Lane l holds the float4 columns l + 32 c of its part.  The splits are
// folded in batches whose loads -- lse values and partial columns alike --
// are all issued before any is used, into a running maximum and sum; a call
// with at most one batch of splits (4 a record-warp, 16 a quarter-warp, whose
// lanes hold one column each) waits for one round of L2 latency.
constexpr int kMaxSplits = 256;

constexpr int kCombineWarps = 8;     // warps per 256-thread CTA
constexpr int kFewRecords = 512;     // at most this many records: four warps a record

template <int QPR>   // column parts per record: 1 (a warp a record) or 4 (a CTA a record)
__global__ void __launch_bounds__(32 * kCombineWarps)
mla_combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_lse, int T,
                   int H, int Dv, int n_splits, __nv_bfloat16 *__restrict__ out,
                   float *__restrict__ lse, const float *__restrict__ sinks, int lse_log2) {
  constexpr int CPL = 4 / QPR;                   // float4 columns a lane holds
  constexpr int kCombineBatch = QPR == 4 ? 16 : 4;   // splits whose loads are in flight together
  constexpr int SH = QPR == 4 ? kCombineWarps / QPR : 1;   // split halves (QPR 4: a CTA a record)
  static_assert(QPR == 1 || SH == 2, "a few-record CTA holds four parts x two halves");
  __shared__ float4 x_acc[QPR == 4 ? QPR * 32 : 1];   // the second half's sums, by part and lane
  __shared__ float x_m[QPR], x_t[QPR];
  pdl_wait();      // the partials come from the previous kernel
  const int lane = threadIdx.x & 31;
  int64_t r;                                     // record (t, h)
  int part, half;
  if (QPR == 4) {
    r = blockIdx.x;                              // one CTA a record, warps = parts x halves
    if (r >= (int64_t)T * H) return;             // whole CTA
    part = (threadIdx.x >> 5) & 3;
    half = (threadIdx.x >> 5) >> 2;
  } else {
    const int64_t w = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (w >= (int64_t)T * H) return;
    r = w;
    part = 0;
    half = 0;
  }
  const int64_t t = r / H, h = r - t * H;
  const int nf = Dv >> 2;                        // float4 columns of a record
  const int f0 = 32 * CPL * part + lane;         // this lane's columns: f0 + 32 c
  // this warp's splits: [s0, s1)
  const int hs = (n_splits + SH - 1) / SH;
  const int s0 = min(n_splits, half * hs), s1 = min(n_splits, s0 + hs);
  float mx = -INFINITY, tot = 0.f;
  float4 acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = s0; i0 < s1; i0 += kCombineBatch) {
    float li[kCombineBatch];
    float4 v[kCombineBatch][CPL];
#pragma unroll
    for (int b = 0; b < kCombineBatch; ++b) {
      const int i = i0 + b;
      li[b] = -INFINITY;
#pragma unroll
      for (int c = 0; c < CPL; ++c) v[b][c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < s1) {
        const int64_t rec = (t * n_splits + i) * H + h;
        li[b] = __ldcg(part_lse + rec);
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const int f = f0 + 32 * c;
          if (f < nf) v[b][c] = __ldcg(reinterpret_cast<const float4 *>(part_o + rec * Dv) + f);
        }
      }
    }
    float bm = mx;
#pragma unroll
    for (int b = 0; b < kCombineBatch; ++b) bm = fmaxf(bm, li[b]);
    if (bm == -INFINITY) continue;               // no split with a valid entry yet
    const float sc = mx == -INFINITY ? 0.f : __expf(mx - bm);
    tot *= sc;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      acc[c].x *= sc; acc[c].y *= sc; acc[c].z *= sc; acc[c].w *= sc;
    }
#pragma unroll
    for (int b = 0; b < kCombineBatch; ++b) {
      // a split with no valid entry has lse = -inf and weight 0
      const float wgt = li[b] == -INFINITY ? 0.f : __expf(li[b] - bm);
      tot += wgt;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        acc[c].x = fmaf(wgt, v[b][c].x, acc[c].x);
        acc[c].y = fmaf(wgt, v[b][c].y, acc[c].y);
        acc[c].z = fmaf(wgt, v[b][c].z, acc[c].z);
        acc[c].w = fmaf(wgt, v[b][c].w, acc[c].w);
      }
    }
    mx = bm;
  }
  if (QPR == 4) {
    // the second half hands its (max, sum, columns) to the first
    if (half == 1) {
      x_acc[part * 32 + lane] = acc[0];
      if (lane == 0) {
        x_m[part] = mx;
        x_t[part] = tot;
      }
    }
    __syncthreads();
    if (half == 1) return;
    const float m1 = x_m[part], t1 = x_t[part];
    const float4 a1 = x_acc[part * 32 + lane];
    const float M = fmaxf(mx, m1);
    if (M != -INFINITY) {
      const float sc0 = mx == -INFINITY ? 0.f : __expf(mx - M);
      const float sc1 = m1 == -INFINITY ? 0.f : __expf(m1 - M);
      tot = tot * sc0 + t1 * sc1;
      acc[0].x = fmaf(acc[0].x, sc0, a1.x * sc1);
      acc[0].y = fmaf(acc[0].y, sc0, a1.y * sc1);
      acc[0].z = fmaf(acc[0].z, sc0, a1.z * sc1);
      acc[0].w = fmaf(acc[0].w, sc0, a1.w * sc1);
      mx = M;
    }
  }
  if (sinks) {
    // the head's sink joins the denominator (no value): rescale to a maximum
    // that covers it (all splits empty and no sink: nothing to fold)
    const float sg = sinks[h];
    const float M = fmaxf(mx, sg);
    if (M != -INFINITY) {
      const float sc = mx == -INFINITY ? 0.f : __expf(mx - M);
      tot = tot * sc + __expf(sg - M);
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        acc[c].x *= sc; acc[c].y *= sc; acc[c].z *= sc; acc[c].w *= sc;
      }
      mx = M;
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const int f = f0 + 32 * c;
    if (f < nf) {
      uint2 pk;
      pk.x = pack_bf16x2(acc[c].x * inv, acc[c].y * inv);
      pk.y = pack_bf16x2(acc[c].z * inv, acc[c].w * inv);
      *reinterpret_cast<uint2 *>(out + r * Dv + 4 * f) = pk;
    }
  }
  if (part == 0 && lane == 0) lse[r] = lse_report(tot > 0.f ? mx + logf(tot) : -INFINITY, lse_log2);
}

}  // namespace

int mla_num_splits(int T, int H, int k_total) {
  // one CTA per SM: as many pieces per (token, head group) as fit in one wave,
  // each piece at least one 64-row tile
  const int hgroups = (H + kHeadsPerCta - 1) / kHeadsPerCta;
  const int ctas_per_split = T * hgroups;
  int s = num_sms() / max(ctas_per_split, 1);
  s = min(s, (k_total + 63) / 64);
  s = min(s, kMaxSplits);
  return max(s, 1);
}

size_t mla_ws_bytes(int T, int H, int Dv, int k_total) {
  const int s = mla_num_splits(T, H, k_total);
  if (s <= 1) return 0;
  WsCarver c(nullptr);
  c.take<float>((size_t)T * s * H * Dv);
  c.take<float>((size_t)T * s * H);
  return c.bytes();
}

void mla_ws_layout(int T, int H, int Dv, int k_total, void *ws, float **part_o,
                   float **part_lse) {
  const int s = mla_num_splits(T, H, k_total);
  WsCarver c(ws);
  *part_o = c.take<float>((size_t)T * s * H * Dv);
  *part_lse = c.take<float>((size_t)T * s * H);
}

cudaError_t sparse_mla_launch(const MlaArgs &a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * (kRows * kKStride + kHeadsPerCta * kRows) +
                      sizeof(__nv_bfloat16) * kHeadsPerCta * kQStride;
  dim3 grid((unsigned)a.T, (unsigned)a.n_splits, (unsigned)((a.H + kHeadsPerCta - 1) / kHeadsPerCta));
  cudaError_t e;
  const int fmt = sparse_mla_tc_format(a);
  if (fmt >= 0) {
    e = sparse_mla_tc_launch(a, fmt, s);
  } else if (a.Dv == 512) {
    e = cudaFuncSetAttribute(sparse_mla_simt_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    sparse_mla_simt_kernel<512><<<grid, kThreads, smem, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(sparse_mla_simt_kernel<448>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    sparse_mla_simt_kernel<448><<<grid, kThreads, smem, s>>>(a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || a.n_splits == 1) return e;
  const int64_t recs = (int64_t)a.T * a.H;
  const bool few = recs <= kFewRecords;
  // few records: a CTA of kCombineWarps warps each (see mla_combine_kernel)
  const int64_t warps = recs * (few ? kCombineWarps : 1);
  return launch_pdl(few ? mla_combine_kernel<4> : mla_combine_kernel<1>,
                    dim3((unsigned)((warps + kCombineWarps - 1) / kCombineWarps)),
                    dim3(32 * kCombineWarps), 0, s, (const float *)a.part_o,
                    (const float *)a.part_lse, a.T, a.H, a.Dv, a.n_splits,
                    static_cast<__nv_bfloat16 *>(a.out), a.lse, a.sinks, a.lse_log2);
}

}  // namespace dsa
