// Backward of the absorbed-MLA sparse attention over a bf16 pool (rows of
// 576 = 512 NoPE + 64 RoPE, V = the leading 512): the other half of the
// training workload the Miles pull request #3608 measures ("fwd + bwd per
// layer").  Given dL/dout and the forward's lse (the lse takes no gradient):
//   p_j   = e^{s_j - lse},  s_j = scale q . K_j
//   delta = sum_j p_j (dout . V_j)          (= dout . out)
//   dS_j  = p_j (dout . V_j - delta)
//   dq    = scale sum_j dS_j K_j
//   dK_j  = scale sum_h dS_hj q_h  (+ sum_h p_hj dout_h on the V columns)
//   dsink = -e^{sink - lse} delta
// Row gradients are added into the pool's gradient at the row's slot (fp32
// atomics, once per selection).
//
// One CTA per (token, group of 32 heads), 8 warps of 4 heads; a lane holds
// the columns lane + 32 e of a row.  Pass 1 walks the list for delta, pass 2
// walks it again for dS (recomputing p and dout . V, so the forward's output
// is not needed) and keeps dq in registers; each 16-row tile's row gradients
// are a product over the CTA's heads (dS and p kept per tile in shared
// memory), one global atomic per element.  Written for correctness first: a
// SIMT kernel, with no tensor cores.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kBD = 576, kBDv = 512;
constexpr int kBHeads = 32;            // heads per CTA
constexpr int kBRows = 16;             // rows per tile
constexpr int kBThreads = 256;         // 8 warps x 4 heads
constexpr int kBCol = kBD / 32;        // 18 columns a lane
constexpr int kBColV = kBDv / 32;      // 16 of them in V

struct BwdSmem {
  uint32_t q, dout, rows, ps, dss, delta, lse, slot, total;
};
__host__ __device__ inline BwdSmem bwd_smem_layout() {
  BwdSmem L;
  L.q = 0;                                              // bf16 [32][576]
  L.dout = L.q + kBHeads * kBD * 2;                     // bf16 [32][512]
  L.rows = L.dout + kBHeads * kBDv * 2;                 // bf16 [16][576]
  L.ps = L.rows + kBRows * kBD * 2;                     // fp32 [32][16]: p of (head, row)
  L.dss = L.ps + kBHeads * kBRows * 4;                  // fp32 [32][16]: scale * dS
  L.delta = L.dss + kBHeads * kBRows * 4;               // fp32 [32]
  L.lse = L.delta + kBHeads * 4;                        // fp32 [32]
  L.slot = L.lse + kBHeads * 4;                         // int  [16]
  L.total = L.slot + kBRows * 4;
  return L;
}

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kBThreads, 1) sparse_mla_bwd_kernel(MlaBwdArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const BwdSmem L = bwd_smem_layout();
  __nv_bfloat16 *q_s = reinterpret_cast<__nv_bfloat16 *>(smem + L.q);
  __nv_bfloat16 *do_s = reinterpret_cast<__nv_bfloat16 *>(smem + L.dout);
  __nv_bfloat16 *r_s = reinterpret_cast<__nv_bfloat16 *>(smem + L.rows);
  float *p_s = reinterpret_cast<float *>(smem + L.ps);
  float *ds_s = reinterpret_cast<float *>(smem + L.dss);
  float *delta_s = reinterpret_cast<float *>(smem + L.delta);
  float *lse_s = reinterpret_cast<float *>(smem + L.lse);
  int *slot_s = reinterpret_cast<int *>(smem + L.slot);

  const int t = blockIdx.x;
  const int h0 = blockIdx.y * kBHeads;
  const int nh = min(kBHeads, a.H - h0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
  const __nv_bfloat16 *dout = static_cast<const __nv_bfloat16 *>(a.dout);
  const __nv_bfloat16 *kv = reinterpret_cast<const __nv_bfloat16 *>(a.kv.data);
  const __nv_bfloat16 zero = __float2bfloat16(0.f);

  // the token's q and dout rows of these heads (zeros past H), and their lse
  for (int i = threadIdx.x; i < kBHeads * kBD; i += kBThreads) {
    const int h = i / kBD, d = i - h * kBD;
    q_s[i] = h < nh ? q[((size_t)t * a.H + h0 + h) * kBD + d] : zero;
  }
  for (int i = threadIdx.x; i < kBHeads * kBDv; i += kBThreads) {
    const int h = i / kBDv, d = i - h * kBDv;
    do_s[i] = h < nh ? dout[((size_t)t * a.H + h0 + h) * kBDv + d] : zero;
  }
  if (threadIdx.x < kBHeads) {
    const int h = threadIdx.x;
    float l = h < nh ? a.lse[(size_t)t * a.H + h0 + h] : -INFINITY;
    if (a.lse_log2) l *= 0.6931471805599453f;   // the forward reported log2 units
    lse_s[h] = l;
  }

  // one tile of list entries e0 .. e0+15 into shared memory (masked or
  // out-of-range entries: slot -1, never used)
  auto load_tile = [&](int e0) {
    __syncthreads();
    if (threadIdx.x < kBRows) {
      const int e = e0 + threadIdx.x;
      int s = -1;
      if (e < a.k) {
        const int v = a.idx[(size_t)t * a.k + e];
        if (v >= 0 && v < a.kv.rows) s = v;
        else if (v != -1) raise_flag(a.err_flag, DSA_DEVERR_INDEX_RANGE);
      }
      slot_s[threadIdx.x] = s;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kBRows * kBD / 8; i += kBThreads) {
      const int r = i / (kBD / 8), c = i - r * (kBD / 8);
      const int s = slot_s[r];
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (s >= 0) v = __ldg(reinterpret_cast<const uint4 *>(kv + (size_t)s * kBD) + c);
      reinterpret_cast<uint4 *>(r_s)[i] = v;
    }
    __syncthreads();
  };
  // s (scaled) and dout . V of head h against tile row r, in every lane
  auto scores = [&](int h, int r, float &s, float &dp) {
    const __nv_bfloat16 *qh = q_s + h * kBD, *dh = do_s + h * kBDv, *kr = r_s + r * kBD;
    float acc = 0.f, accv = 0.f;
#pragma unroll
    for (int e = 0; e < kBCol; ++e) {
      const int d = lane + 32 * e;
      const float kd = bf(kr[d]);
      acc = fmaf(bf(qh[d]), kd, acc);
      if (e < kBColV) accv = fmaf(bf(dh[d]), kd, accv);
    }
    s = warp_allsum(acc) * a.softmax_scale;
    dp = warp_allsum(accv);
  };

  // ---- pass 1: delta per head
  float dsum[4] = {0.f, 0.f, 0.f, 0.f};
  for (int e0 = 0; e0 < a.k; e0 += kBRows) {
    load_tile(e0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int h = warp * 4 + i;
      if (h >= nh) continue;
      for (int r = 0; r < kBRows; ++r) {
        if (slot_s[r] < 0) continue;
        float s, dp;
        scores(h, r, s, dp);
        dsum[i] = fmaf(__expf(s - lse_s[h]), dp, dsum[i]);
      }
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) delta_s[warp * 4 + i] = dsum[i];
  }

  // ---- pass 2: dS and dq (registers); each tile's row gradients as a
  // product over the CTA's heads, one atomic add per pool element
  float dq[4][kBCol];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < kBCol; ++e) dq[i][e] = 0.f;
  for (int e0 = 0; e0 < a.k; e0 += kBRows) {
    load_tile(e0);   // its first barrier also publishes delta_s
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int h = warp * 4 + i;
      const float lse_h = lse_s[h], delta_h = delta_s[h];
      for (int r = 0; r < kBRows; ++r) {
        float p = 0.f, ds = 0.f;
        if (h < nh && slot_s[r] >= 0) {
          float s, dp;
          scores(h, r, s, dp);
          p = __expf(s - lse_h);
          ds = p * (dp - delta_h) * a.softmax_scale;   // carries the score scale
          const __nv_bfloat16 *kr = r_s + r * kBD;
#pragma unroll
          for (int e = 0; e < kBCol; ++e) dq[i][e] = fmaf(ds, bf(kr[lane + 32 * e]), dq[i][e]);
        }
        if (lane == 0) {
          p_s[h * kBRows + r] = p;
          ds_s[h * kBRows + r] = ds;
        }
      }
    }
    __syncthreads();
    // row r, column d:  sum_h ds[h][r] q[h][d]  +  (d < Dv) sum_h p[h][r] dout[h][d]
    for (int i = threadIdx.x; i < kBRows * kBD; i += kBThreads) {
      const int r = i / kBD, d = i - r * kBD;
      const int sl = slot_s[r];
      if (sl < 0) continue;
      float g = 0.f;
#pragma unroll 8
      for (int h = 0; h < kBHeads; ++h) {
        g = fmaf(ds_s[h * kBRows + r], bf(q_s[h * kBD + d]), g);
        if (d < kBDv) g = fmaf(p_s[h * kBRows + r], bf(do_s[h * kBDv + d]), g);
      }
      atomicAdd(a.dkv + (size_t)sl * kBD + d, g);
    }
  }

  // ---- dq, and the sinks' gradients
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int h = warp * 4 + i;
    if (h >= nh) continue;
    float *dst = a.dq + ((size_t)t * a.H + h0 + h) * kBD;
#pragma unroll
    for (int e = 0; e < kBCol; ++e) dst[lane + 32 * e] = dq[i][e];
    if (a.sinks && a.dsinks && lane == 0) {
      const float sk = a.sinks[h0 + h];
      if (sk != -INFINITY) atomicAdd(&a.dsinks[h0 + h], -__expf(sk - lse_s[h]) * delta_s[h]);
    }
  }
}

}  // namespace

cudaError_t sparse_mla_bwd_launch(const MlaBwdArgs &a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const BwdSmem L = bwd_smem_layout();
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_bwd_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)a.T, (unsigned)((a.H + kBHeads - 1) / kBHeads));
  sparse_mla_bwd_kernel<<<grid, kBThreads, L.total, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
