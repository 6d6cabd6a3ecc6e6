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

// One warp per fact token: its K row and V row of `layer`.  The token's fact
// is found by a 32-way search (each round the lanes probe 32 evenly spaced
// facts and a ballot keeps the last one that starts at or before the token),
// so a capture of n facts costs log32(n) rounds of loads, not log2(n).  Each
// lane then loads up to kCapVecs vectors of the K row and of the V row before
// storing any, so the loads of a row are in flight together.
constexpr int kCapVecs = 4;

__global__ void __launch_bounds__(kCaptureThreads) capture_layer_kernel(const CaptureArgs a) {
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;   // fact token
  const int lane = threadIdx.x & 31;
  if (t >= a.tokens) return;                   // whole warps: t is the same for all lanes
  int lo = 0, hi = a.n;                        // fact lo starts at or before t; facts >= hi start after
  while (hi - lo > 1) {
    const int stride = (hi - lo + 31) >> 5;
    const int idx = lo + lane * stride;
    const bool le = idx < hi && a.seg[2 * idx + 1] - a.tok0 <= t;
    const unsigned m = __ballot_sync(0xffffffffu, le);   // lane 0 probes lo, which qualifies
    lo += (31 - __clz(m)) * stride;
    hi = min(hi, lo + stride);
  }
  const int64_t src = a.seg[2 * lo] + (t - (a.seg[2 * lo + 1] - a.tok0));
  const uint8_t* ks = a.k + (size_t)src * a.row_bytes;
  const uint8_t* vs = a.v + (size_t)src * a.row_bytes;
  uint8_t* dk = a.kv + ((size_t)(a.tok0 + t) * a.L + a.layer) * 2 * (size_t)a.row_bytes;
  uint8_t* dv = dk + a.row_bytes;
  const int nv = a.row_bytes >> 4;
  for (int c0 = lane; c0 < nv; c0 += 32 * kCapVecs) {
    uint4 kx[kCapVecs], vx[kCapVecs];
#pragma unroll
    for (int u = 0; u < kCapVecs; ++u) {
      const int c = c0 + 32 * u;
      if (c < nv) {
        kx[u] = *reinterpret_cast<const uint4*>(ks + (size_t)c * 16);
        vx[u] = *reinterpret_cast<const uint4*>(vs + (size_t)c * 16);
      }
    }
#pragma unroll
    for (int u = 0; u < kCapVecs; ++u) {
      const int c = c0 + 32 * u;
      if (c < nv) {
        st_v4(dk + (size_t)c * 16, kx[u]);
        st_v4(dv + (size_t)c * 16, vx[u]);
      }
    }
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
