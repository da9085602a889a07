// Shared device helpers for the DSA kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/dsa.h"

#define DSA_DEVINLINE __device__ __forceinline__

namespace dsa {

// ---------------------------------------------------------------- errors

DSA_DEVINLINE void raise_flag(int32_t *err_flag, int32_t bits) {
  if (err_flag) atomicOr(err_flag, bits);
}

// ---------------------------------------------------------------- numbers

DSA_DEVINLINE float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two OCP e4m3 bytes (low byte first) -> two floats, exact.
DSA_DEVINLINE float2 e4m3x2_to_float2(uint16_t two) {
  __nv_fp8x2_storage_t s = two;
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(s, __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2 *>(&h));
}

DSA_DEVINLINE float e4m3_to_float(uint8_t b) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(b, __NV_E4M3);
  return __half2float(*reinterpret_cast<__half *>(&h));
}

// UE8M0 exponent byte -> 2^(e - 127).  e = 0 gives 2^-127 (an fp32 subnormal);
// e = 255 (NaN in the MX encoding) is not produced by the formats here.
DSA_DEVINLINE float ue8m0_to_float(uint32_t e) {
  return e == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// Order-preserving map fp32 -> uint32: a > b (as floats) iff key(a) > key(b).
// -0.0 is first turned into +0.0 so the two tie.
DSA_DEVINLINE uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u << 1) == 0) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

DSA_DEVINLINE unsigned lane_id() { return threadIdx.x & 31; }

// Programmatic dependent launch.  A kernel launched with launch_pdl may start
// while the previous kernel on the stream is still running; pdl_wait() blocks
// until that kernel has completed and its writes are visible, so everything
// that reads its results comes after pdl_wait().  pdl_trigger() lets this
// kernel's own dependent launch early (it still waits for us to finish).
// Both are no-ops for a kernel launched without the attribute.
DSA_DEVINLINE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
DSA_DEVINLINE void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Pack two floats to a bf16x2 word (round to nearest even), low half = a.
DSA_DEVINLINE uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace dsa

// ---------------------------------------------------------------- host side
namespace dsa {

// Round x up to a multiple of a (a power of two).
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) & ~(a - 1); }

// Carves aligned sub-buffers out of a caller workspace.
struct WsCarver {
  char *base;
  size_t off = 0;
  explicit WsCarver(void *p) : base(static_cast<char *>(p)) {}
  template <typename T>
  T *take(size_t count) {
    off = align_up(off, 256);
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
  size_t bytes() const { return align_up(off, 256); }
};

// A finished softmax over rows: m is the reference maximum in raw products
// q . K (before the softmax scale), l the sum of exp(scale (x - m)) over the
// rows.  A sink logit (natural-log units, -inf: none) joins the denominator.
// Returns the factor that turns the rows' weighted sum (in the frame of m)
// into the output, and sets *lse_nat to the natural log of the whole
// denominator.  No row (l = 0): factor 0, lse = the sink.
__device__ __forceinline__ float fold_sink(float m, float scale, float l, float sink_nat,
                                           float *lse_nat) {
  if (!(l > 0.f)) {
    *lse_nat = sink_nat;
    return 0.f;
  }
  const float r = fmaf(m, scale, logf(l));     // ln of the rows' part
  const float hi = fmaxf(r, sink_nat), lo = fminf(r, sink_nat);
  const float t = hi + log1pf(expf(lo - hi));  // no sink: lo = -inf, t = r
  *lse_nat = t;
  return expf(r - t) / l;
}

// The lse as reported: natural log, or log2 units on request.
__device__ __forceinline__ float lse_report(float lse_nat, int log2_units) {
  return log2_units ? lse_nat * 1.4426950408889634f : lse_nat;
}

// Launch with the programmatic-stream-serialization attribute (see pdl_wait),
// in thread-block clusters of cluster_x CTAs along x (1: no cluster).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t s, unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster_x > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  return launch_pdl_cluster(kern, grid, block, smem, s, 1u, args...);
}

inline int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
  }
  return n;
}

}  // namespace dsa
