// Lightning-indexer scores  I[t,s] = sum_h w[t,h] * ReLU(sq[t,h] sk[s] q[t,h,:].k[s,:])
// (the "scores" stage of tokenspeed PR #627 "Add gluon kernel for DSA").
//
// Since the fp8 scales are positive, sk[s] leaves the ReLU and the head sum
// (ReLU(c x) = c ReLU(x) for c > 0) and sq[t,h] is folded into the query
// once per CTA: score = sk[s] * sum_h w[t,h] * ReLU((sq[t,h] q8[t,h,:]) . k8[s,:]).
//
// The optional fused histogram feeds the first radix level of the top-k
// (topk.cu): the 12-bit bin of each stored score is counted per row.
#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kKeysPerCta = 128;
constexpr int kChunk = 32;  // key dims decoded per step

template <int HMAX>
__global__ void __launch_bounds__(kKeysPerCta)
index_score_simt_kernel(IndexScoreArgs a) {
  extern __shared__ float smem[];
  float *q_s = smem;                 // [HMAX][d], scales folded in
  float *w_s = smem + HMAX * a.d;    // [HMAX]
  const int t = blockIdx.y;
  int64_t r0, r1;
  if (a.slot_base) {
    r0 = a.slot_base[t];
    r1 = r0 + a.seq_lens[t];
  } else {
    r0 = a.row_start[t];
    r1 = a.row_end[t];
  }
  if (r0 < 0 || r1 < r0 || r1 > a.k_rows) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_flag(a.err_flag, DSA_DEVERR_INDEX_RANGE);
    return;
  }
  const int64_t L = r1 - r0;
  const int64_t j0 = (int64_t)blockIdx.x * kKeysPerCta;
  if (j0 >= L) return;
  const int H = a.H_I, d = a.d;
  const bool fp8 = a.idx_dtype == DSA_IDX_FP8_E4M3;
  for (int i = threadIdx.x; i < H * d; i += blockDim.x) {
    const int h = i / d;
    float v;
    if (fp8) {
      v = e4m3_to_float(static_cast<const uint8_t *>(a.q_idx)[(size_t)t * H * d + i]) *
          a.q_scale[(size_t)t * H + h];
    } else {
      v = bf16_bits_to_float(static_cast<const uint16_t *>(a.q_idx)[(size_t)t * H * d + i]);
    }
    q_s[h * d + (i % d)] = v;
  }
  for (int h = threadIdx.x; h < H; h += blockDim.x) w_s[h] = a.w[(size_t)t * H + h];
  __syncthreads();

  const int64_t j = j0 + threadIdx.x;
  const bool valid = j < L;
  float score = 0.f;
  if (valid) {
    const int64_t s = r0 + j;
    float acc[HMAX];
#pragma unroll
    for (int h = 0; h < HMAX; ++h) acc[h] = 0.f;
    for (int c0 = 0; c0 < d; c0 += kChunk) {
      float kf[kChunk];
      if (fp8) {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            static_cast<const uint8_t *>(a.k_idx) + s * d + c0);
#pragma unroll
        for (int v = 0; v < kChunk / 16; ++v) {
          uint4 raw = __ldg(src + v);
          const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float2 lo = e4m3x2_to_float2((uint16_t)(wds[q] & 0xffffu));
            float2 hi = e4m3x2_to_float2((uint16_t)(wds[q] >> 16));
            kf[v * 16 + q * 4 + 0] = lo.x;
            kf[v * 16 + q * 4 + 1] = lo.y;
            kf[v * 16 + q * 4 + 2] = hi.x;
            kf[v * 16 + q * 4 + 3] = hi.y;
          }
        }
      } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            static_cast<const uint16_t *>(a.k_idx) + s * d + c0);
#pragma unroll
        for (int v = 0; v < kChunk / 8; ++v) {
          uint4 raw = __ldg(src + v);
          const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            kf[v * 8 + q * 2 + 0] = __uint_as_float(wds[q] << 16);
            kf[v * 8 + q * 2 + 1] = __uint_as_float(wds[q] & 0xffff0000u);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < HMAX; ++h) {
        if (h < H) {
          const float *qh = q_s + h * d + c0;
          float x = acc[h];
#pragma unroll
          for (int c = 0; c < kChunk; ++c) x = fmaf(qh[c], kf[c], x);
          acc[h] = x;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < HMAX; ++h)
      if (h < H) score = fmaf(w_s[h], fmaxf(acc[h], 0.f), score);
    if (fp8) score *= a.k_scale[s];
    a.scores[(int64_t)t * a.ld_scores + j] = score;
  }
  if (a.hist && L > a.topk_k) {
    // warp-aggregated count of this warp's bins
    const uint32_t bin = score_key(score) >> 20;
    const unsigned act = __ballot_sync(0xffffffffu, valid);
    if (valid) {
      const unsigned peers = __match_any_sync(act, bin);
      if ((int)lane_id() == __ffs(peers) - 1)
        atomicAdd(&a.hist[(size_t)t * kHistBins + bin], (uint32_t)__popc(peers));
    }
  }
}

}  // namespace

cudaError_t index_score_launch(const IndexScoreArgs &a, cudaStream_t s) {
  if (a.T == 0 || a.max_len == 0) return cudaSuccess;
  dim3 grid((unsigned)((a.max_len + kKeysPerCta - 1) / kKeysPerCta), (unsigned)a.T);
  const size_t smem = sizeof(float) * ((size_t)DSA_MAX_INDEX_HEADS * a.d + DSA_MAX_INDEX_HEADS);
  if (a.H_I <= 8) {
    index_score_simt_kernel<8><<<grid, kKeysPerCta, smem, s>>>(a);
  } else if (a.H_I <= 16) {
    index_score_simt_kernel<16><<<grid, kKeysPerCta, smem, s>>>(a);
  } else if (a.H_I <= 32) {
    index_score_simt_kernel<32><<<grid, kKeysPerCta, smem, s>>>(a);
  } else {
    index_score_simt_kernel<64><<<grid, kKeysPerCta, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace dsa
