// dsa_topk_noalloc: the top-k of dsa_topk with its scratch memory in a
// static device array instead of a caller workspace.
//
// Who needs it: callers that cannot allocate device memory themselves -- for
// example a plugin whose host framework hands it only its input and output
// buffers and no workspace, or code on a latency-critical path where a
// cudaMalloc (which may synchronise the device) is not allowed.  They pass
// inputs and outputs only; the scratch is the array below.
//
// The array is a fixed kTopkNoAllocScratchBytes (4 MiB) in every GPU that
// loads this library, held until the process exits.  All calls share it and
// it keeps the previous call's contents: each call clears the parts that must
// start at zero.  Calls whose kernels overlap on the GPU (two streams, two
// host threads) race on the array and must be serialised by the caller.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr size_t kTopkNoAllocScratchBytes = DSA_TOPK_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_topk_scratch[kTopkNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_topk_scratch on the current device, looked up once per
// device (with that device current).  Returns nullptr on failure.
void *scratch_address(cudaError_t *err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (*err != cudaSuccess || !p) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_topk_noalloc(const float *scores, int64_t ld_scores, const int32_t *row_len,
                                int T, int64_t max_len, int k, const int32_t *index_base,
                                int32_t *idx, int32_t *lens, int32_t *err_flag,
                                dsa_stream_t stream) {
  if (T < 0 || max_len < 0 || ld_scores < max_len) return DSA_ERR_INVALID_ARG;
  if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!scores || !row_len || !idx) return DSA_ERR_INVALID_ARG;
  if (topk_ws_layout(T, max_len, k, nullptr, nullptr) > kTopkNoAllocScratchBytes)
    return DSA_ERR_UNSUPPORTED;  // more rows than the static scratch holds
  cudaError_t e;
  void *scratch = scratch_address(&e);
  if (!scratch) return DSA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TopkWs w;
  topk_ws_layout(T, max_len, k, scratch, &w);
  e = topk_clear(w, T, s);  // the histogram and counters must start at zero
  if (e == cudaSuccess) e = topk_hist(scores, ld_scores, row_len, T, max_len, k, w, s);
  if (e == cudaSuccess)
    e = topk_select(scores, ld_scores, row_len, T, max_len, k, index_base, idx, lens, w,
                    err_flag, s);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
