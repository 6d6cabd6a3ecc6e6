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

// Persistent launch: one CTA per SM times the occupancy its shared-memory
// plan allows.
cudaError_t launch_inject(const InjectArgs& a, const RopeTurns& turns, int kv_dtype, int style,
                          const LaunchCfg& cfg);

// Whether a row of row_bytes (K or V of one layer) and R requests fit the
// inject kernel's shared-memory plan.
bool inject_shape_ok(int row_bytes, int R);

// Sets the message is_last_error_message() returns on this thread.
void set_last_error_message(const char* msg);


}  // namespace isk
