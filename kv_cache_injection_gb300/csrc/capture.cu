// Context-Window Encoding capture.
//
// InferScale ("Méthodologie", phase 1, "Encodage de la Fenêtre de Contexte")
// encodes each memory fact together with a window of preceding conversation
// turns and keeps only the fact's K (before RoPE) and V.  The engine's prefill
// produces one layer at a time, every token of [window || fact] sequences back
// to back; this kernel keeps the fact tokens' rows and writes them into the
// store's token-major arena, where the fact's K and V rows of each layer sit
// side by side.
#include "common.cuh"
#include "internal.h"

namespace isk {

constexpr int kCaptureThreads = 256;

// One warp per fact token: its K row and V row of `layer`.
__global__ void __launch_bounds__(kCaptureThreads) capture_layer_kernel(const CaptureArgs a) {
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;   // fact token
  const int lane = threadIdx.x & 31;
  if (t >= a.tokens) return;
  // The fact holding t: the last one whose first arena token is <= tok0 + t.
  int lo = 0, hi = a.n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.seg[2 * mid + 1] - a.tok0 <= t) lo = mid; else hi = mid;
  }
  const int64_t src = a.seg[2 * lo] + (t - (a.seg[2 * lo + 1] - a.tok0));
  const uint8_t* ks = a.k + (size_t)src * a.row_bytes;
  const uint8_t* vs = a.v + (size_t)src * a.row_bytes;
  uint8_t* dk = a.kv + ((size_t)(a.tok0 + t) * a.L + a.layer) * 2 * (size_t)a.row_bytes;
  uint8_t* dv = dk + a.row_bytes;
  for (int c = lane; c < a.row_bytes / 16; c += 32) {
    st_v4(dk + (size_t)c * 16, *reinterpret_cast<const uint4*>(ks + (size_t)c * 16));
    st_v4(dv + (size_t)c * 16, *reinterpret_cast<const uint4*>(vs + (size_t)c * 16));
  }
}

cudaError_t launch_capture_layer(const CaptureArgs& a, const LaunchCfg& cfg) {
  if (a.tokens <= 0) return cudaSuccess;
  const int64_t threads = a.tokens * 32;
  const int64_t blocks = (threads + kCaptureThreads - 1) / kCaptureThreads;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  return launch_ex(capture_layer_kernel, dim3((unsigned)blocks), dim3(kCaptureThreads), 0, cfg.stream,
                   cfg.pdl, a);
}

}  // namespace isk
