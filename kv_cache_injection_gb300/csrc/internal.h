// Host-side launch wrappers shared between the translation units of
// libinjectscale.so.  Each returns the cudaError_t of its launch.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace isk {

struct LaunchCfg {
  cudaStream_t stream;
  int num_sms;
  bool pdl;   // launch with programmatic stream serialisation
};

// cudaLaunchKernelEx with optional programmatic stream serialisation; on the
// first launch of a kernel on a device it also asks for the largest shared
// memory carve-out, so consecutive kernels do not reconfigure L1/shared.
void prefer_max_shared(const void* kern);   // once per (kernel, device)

// Raises a kernel's dynamic shared-memory limit on the current device to at
// least `bytes` (the default stops at 48 KB minus the kernel's static shared
// memory); remembered per kernel and device.
cudaError_t ensure_dynamic_smem(const void* kern, size_t bytes);

template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      bool pdl, Args... args) {
  prefer_max_shared(reinterpret_cast<const void*>(kern));
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kern, args...);
}

cudaError_t launch_emb_norms(const void* emb, int emb_dtype, int E, const int32_t* rows, int n,
                             float* inv_norm, cudaStream_t stream);

// Fused retrieval (cosine similarity, then top-k by the last CTA of each
// query).  `arrive` holds one zeroed counter per query; the kernel leaves it zeroed.
cudaError_t launch_retrieve(const SimArgs& sa, const TopkArgs& ta, int emb_dtype, int max_user_tiles,
                            int64_t max_user_facts, int32_t* arrive, const LaunchCfg& cfg);


cudaError_t launch_plan(const PlanArgs& a, const LaunchCfg& cfg);

// Batched retrieval (tensor cores): tensor maps of the embedding tiles and of
// the packed queries, and the three launches (grouping, contraction, top-k).
size_t operand_map_bytes();
bool make_operand_map(void* map_out, const void* base, int E, int64_t rows, int box_rows);
cudaError_t launch_group(const GroupArgs& ga, const LaunchCfg& cfg);
cudaError_t launch_sim_gemm(const GemmArgs& gg, const void* map_emb, const void* map_q, int Q,
                            int max_user_tiles, const LaunchCfg& cfg);
cudaError_t launch_topk_batched(const TopkArgs& ta, int Q, int32_t max_users, int64_t max_user_facts,
                                const LaunchCfg& cfg);

// Persistent launch: one CTA per SM times the occupancy its shared-memory
// plan allows.  host_src: the arena a.kv is mapped host memory, read with
// plain loads instead of bulk copies.  fp8_cache: the cache is FP8 E4M3
// (a.cache_row_bytes, a.k_inv, a.v_inv set; 16-bit stores only).
cudaError_t launch_inject(const InjectArgs& a, const RopeTurns& turns, int kv_dtype, int style,
                          bool host_src, bool fp8_cache, const LaunchCfg& cfg);

// Context-Window Encoding capture: the fact tokens' rows of one layer into the arena.
cudaError_t launch_capture_layer(const CaptureArgs& a, const LaunchCfg& cfg);

// Whether a row of row_bytes (K or V of one layer) and R requests fit the
// inject kernel's shared-memory plan.
bool inject_shape_ok(int row_bytes, int R);

// Sets the message is_last_error_message() returns on this thread.
void set_last_error_message(const char* msg);


}  // namespace isk
