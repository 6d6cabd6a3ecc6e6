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

cudaError_t launch_emb_norms(const void* emb, int emb_dtype, int E, const int32_t* rows, int n,
                             float* inv_norm, cudaStream_t stream);

cudaError_t launch_similarity(const SimArgs& a, int emb_dtype, int max_user_tiles,
                              const LaunchCfg& cfg);

cudaError_t launch_topk(const TopkArgs& a, const LaunchCfg& cfg);

cudaError_t launch_plan(const PlanArgs& a, const LaunchCfg& cfg);

cudaError_t launch_inject(const InjectArgs& a, const RopeTurns& turns, int kv_dtype, int style,
                          int grid_ctas, const LaunchCfg& cfg);

// Sets the message is_last_error_message() returns on this thread.
void set_last_error_message(const char* msg);

// CTAs per SM the inject kernel reaches for this dtype/style/row shape.
int inject_ctas_per_sm(int kv_dtype, int style, int vecs_per_lane);

}  // namespace isk
