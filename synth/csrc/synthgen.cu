// Device implementation of the synthetic K/V generator defined in
// synth/kvgen.py (SplitMix64 words, Irwin-Hall sum of twelve 16-bit
// uniforms, value = (S - 393210) / 65536, rounded to the storage type).
// Input generation only: none of the method's arithmetic lives here.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ inline uint64_t mix_h(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ float irwin_hall(uint64_t base, uint64_t i) {
  int32_t s = 0;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const uint64_t w = mix(base + (3 * i + j + 1) * kGamma);
    s += (int32_t)(w & 0xffff) + (int32_t)((w >> 16) & 0xffff) + (int32_t)((w >> 32) & 0xffff) +
         (int32_t)(w >> 48);
  }
  return (float)(s - 393210) * (1.0f / 65536.0f);   // exact: |s - 393210| < 2^19
}

// dtype: 0 = f32, 1 = bf16, 2 = f16 (same codes as the library's is_dtype_t).
__global__ void fill_kernel(void* out, int dtype, uint64_t base, uint64_t first, uint64_t count) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; t < count; t += stride) {
    const float x = irwin_hall(base, first + t);
    if (dtype == 0) {
      static_cast<float*>(out)[t] = x;
    } else if (dtype == 1) {
      static_cast<__nv_bfloat16*>(out)[t] = __float2bfloat16_rn(x);
    } else {
      static_cast<__half*>(out)[t] = __float2half_rn(x);
    }
  }
}

}  // namespace

extern "C" int synth_fill_kv(void* out, int dtype, uint64_t seed, int stream_id, uint64_t first,
                             uint64_t count, void* cuda_stream) {
  if (!out || dtype < 0 || dtype > 2 || stream_id < 0 || stream_id > 255) return 1;
  if (count == 0) return 0;
  const uint64_t base = mix_h((seed << 8) | (uint64_t)stream_id);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const uint64_t want = (count + 255) / 256;
  const unsigned grid = (unsigned)(want < (uint64_t)sms * 16 ? want : (uint64_t)sms * 16);
  fill_kernel<<<grid, 256, 0, (cudaStream_t)cuda_stream>>>(out, dtype, base, first, count);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
