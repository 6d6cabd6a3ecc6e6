// GPU-resident semantic retrieval: cosine similarity against one user's
// stored embeddings, then an exact top-k by radix select.
//
// InferScale keeps the retrieval index and the KV store both on the GPU so
// retrieved text never crosses PCIe ("Conception de Système Native au GPU"),
// and retrieves a relevant subset of k facts per request ("Problématique").
// The index it names is not described; retrieval here is exact cosine top-k.
#include "block_scan.cuh"
#include "common.cuh"
#include "internal.h"

namespace isk {

template <typename E> struct EmbT;
template <> struct EmbT<__half> { using V = Vec<__half>; };
template <> struct EmbT<float> { using V = Vec<float>; };

// ---------------------------------------------------------------------------
// Inverse norms of newly added embedding rows (one warp per row).
template <typename E>
__global__ void __launch_bounds__(256) emb_norm_kernel(const E* emb, int dim, const int32_t* rows,
                                                       int n, float* inv_norm) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= n) return;
  constexpr int VE = EmbT<E>::V::N;
  const E* row = emb + (size_t)rows[w] * dim;
  float acc = 0.f;
  for (int c = lane * VE; c < dim; c += 32 * VE) {
    float x[VE];
    EmbT<E>::V::unpack(*reinterpret_cast<const uint4*>(row + c), x);
#pragma unroll
    for (int e = 0; e < VE; ++e) acc = fmaf(x[e], x[e], acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) inv_norm[rows[w]] = acc > 0.f ? 1.0f / sqrtf(acc) : 0.f;
}

cudaError_t launch_emb_norms(const void* emb, int emb_dtype, int E, const int32_t* rows, int n,
                             float* inv_norm, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int blocks = (n + 7) / 8;
  if (emb_dtype == IS_F16)
    emb_norm_kernel<__half><<<blocks, 256, 0, stream>>>((const __half*)emb, E, rows, n, inv_norm);
  else
    emb_norm_kernel<float><<<blocks, 256, 0, stream>>>((const float*)emb, E, rows, n, inv_norm);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Similarity: CTA (tile, query) computes the cosine of query q with the up to
// 128 embedding rows of one tile of q's user; a warp per row, fp32
// accumulation.  Rows of one user are numbered 0 .. n_u-1 in fill order (tile
// after tile), which is insertion order.
template <typename E>
__global__ void __launch_bounds__(256) similarity_kernel(const SimArgs a) {
  extern __shared__ float s_q[];                 // [E] query in fp32
  __shared__ float s_red[8];
  const int q = blockIdx.y;
  const int ti = blockIdx.x;
  const int user = a.users[q];
  if (user < 0 || user >= a.max_users) {
    if (ti == 0 && threadIdx.x == 0) latch(a.status, IS_ST_USER_RANGE);
    return;
  }
  const int t0 = a.user_tile_off[user];
  const int ntiles = a.user_tile_off[user + 1] - t0;
  if (ti >= ntiles) return;
  const int tile = a.user_tiles[t0 + ti];
  const int nrows = min(kTile, a.user_nfacts[user] - ti * kTile);
  constexpr int VE = EmbT<E>::V::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  const E* qv = reinterpret_cast<const E*>(a.q_emb) + (size_t)q * a.E;
  float ss = 0.f;
  for (int c = threadIdx.x * VE; c < a.E; c += blockDim.x * VE) {
    float x[VE];
    EmbT<E>::V::unpack(*reinterpret_cast<const uint4*>(qv + c), x);
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      s_q[c + e] = x[e];
      ss = fmaf(x[e], x[e], ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) s_red[warp] = ss;
  __syncthreads();
  float nq = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) nq += s_red[w];
  const float inv_q = nq > 0.f ? 1.0f / sqrtf(nq) : 0.f;

  const E* base = reinterpret_cast<const E*>(a.emb) + (size_t)tile * kTile * a.E;
  float* out = a.scores + (size_t)q * a.score_stride + (size_t)ti * kTile;
  for (int r = warp; r < nrows; r += 8) {
    const E* row = base + (size_t)r * a.E;
    float acc = 0.f;
    for (int c = lane * VE; c < a.E; c += 32 * VE) {
      float x[VE];
      EmbT<E>::V::unpack(*reinterpret_cast<const uint4*>(row + c), x);
#pragma unroll
      for (int e = 0; e < VE; ++e) acc = fmaf(x[e], s_q[c + e], acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) out[r] = acc * inv_q * a.emb_inv_norm[(size_t)tile * kTile + r];
  }
}

cudaError_t launch_similarity(const SimArgs& a, int emb_dtype, int max_user_tiles,
                              const LaunchCfg& cfg) {
  if (max_user_tiles <= 0) return cudaSuccess;
  const dim3 grid(max_user_tiles, a.Q);
  const size_t smem = (size_t)a.E * sizeof(float);
  if (emb_dtype == IS_F16)
    similarity_kernel<__half><<<grid, 256, smem, cfg.stream>>>(a);
  else
    similarity_kernel<float><<<grid, 256, smem, cfg.stream>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Top-k of one query's scores (one CTA per query):
//  1. radix select on order-preserving uint32 keys, 8 bits per pass, finds
//     the k-th largest key `thr` and how many keys equal to it to take;
//  2. keys > thr are all taken; of the keys == thr, the lowest rows (= lowest
//     fact ids) are taken;
//  3. the k picks are sorted by (key desc, row asc) with a bitonic sort;
//  4. ids/scores are written, and the segment plan (prefix of lengths).
constexpr int kTopkThreads = 256;

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkArgs a) {
  __shared__ uint32_t hist[256];
  __shared__ unsigned long long sel[IS_MAX_K];
  __shared__ int32_t scratch[33];
  __shared__ uint32_t s_digit, s_above, s_cnt;

  const int q = blockIdx.x;
  const int tid = threadIdx.x;
  const int user = a.users[q];
  int n = 0;
  if (user >= 0 && user < a.max_users) {
    n = a.user_nfacts[user];
  } else if (tid == 0) {
    latch(a.status, IS_ST_USER_RANGE);
  }
  const int kk = min(a.k, n);
  const float* sc = a.scores + (size_t)q * a.score_stride;

  uint32_t prefix = 0, rem = (uint32_t)kk, eq_total = 0;
  if (kk > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      const uint32_t hmask = pass == 0 ? 0u : (0xffffffffu << (32 - 8 * pass));
      hist[tid] = 0;                             // kTopkThreads == 256 bins
      __syncthreads();
      for (int j = tid; j < n; j += kTopkThreads) {
        const uint32_t key = score_key(sc[j]);
        if ((key & hmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      // Thread t holds the count of digit 255 - t; inclusive scan gives the
      // number of keys whose digit is >= 255 - t.
      const int32_t c = (int32_t)hist[255 - tid];
      int32_t tot;
      const int32_t before = block_exclusive_scan(c, scratch, &tot);
      if (before < (int32_t)rem && before + c >= (int32_t)rem) {
        s_digit = 255u - tid;
        s_above = (uint32_t)before;
        s_cnt = (uint32_t)c;
      }
      __syncthreads();
      prefix |= s_digit << shift;
      rem -= s_above;
      eq_total = s_cnt;                           // after the last pass: keys equal to thr
      __syncthreads();
    }
  }
  const uint32_t thr = prefix;
  const uint32_t n_gt = (uint32_t)kk - rem;

  // Collect.
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  if (kk > 0) {
    if (eq_total == rem) {
      // every key >= thr is taken: order of collection does not matter
      for (int j = tid; j < n; j += kTopkThreads) {
        const uint32_t key = score_key(sc[j]);
        if (key >= thr) {
          const uint32_t pos = atomicAdd(&s_cnt, 1u);
          sel[pos] = ((unsigned long long)key << 32) | (0xffffffffu - (uint32_t)j);
        }
      }
    } else {
      // ties cross the boundary: keys == thr are taken in ascending row order
      uint32_t taken = 0;
      for (int b = 0; b < n; b += kTopkThreads) {
        const int j = b + tid;
        const uint32_t key = j < n ? score_key(sc[j]) : 0u;
        if (j < n && key > thr) {
          const uint32_t pos = atomicAdd(&s_cnt, 1u);
          sel[pos] = ((unsigned long long)key << 32) | (0xffffffffu - (uint32_t)j);
        }
        const int32_t is_eq = (j < n && key == thr) ? 1 : 0;
        int32_t tot;
        const int32_t rank = block_exclusive_scan(is_eq, scratch, &tot);
        if (is_eq && taken + (uint32_t)rank < rem)
          sel[n_gt + taken + rank] = ((unsigned long long)key << 32) | (0xffffffffu - (uint32_t)j);
        taken += (uint32_t)tot;
      }
    }
  }
  __syncthreads();

  // Bitonic sort, descending, over the next power of two >= kk.
  int P = 1;
  while (P < kk) P <<= 1;
  for (int i = kk + tid; i < P; i += kTopkThreads) sel[i] = 0ull;
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P / 2; i += kTopkThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long x = sel[lo], y = sel[hi];
        if ((x < y) == desc) {
          sel[lo] = y;
          sel[hi] = x;
        }
      }
      __syncthreads();
    }
  }

  // Outputs + segment plan.
  const int t0 = (kk > 0) ? a.user_tile_off[user] : 0;
  int32_t carry = 0;
  for (int b = 0; b < a.k; b += kTopkThreads) {
    const int r = b + tid;
    int32_t len = 0;
    if (r < a.k) {
      int64_t id = -1;
      float s = -INFINITY;
      if (r < kk) {
        const unsigned long long v = sel[r];
        const uint32_t j = 0xffffffffu - (uint32_t)(v & 0xffffffffu);
        const int tile = a.user_tiles[t0 + (int)(j / kTile)];
        id = a.tile_fact[(size_t)tile * kTile + (j % kTile)];
        s = key_score((uint32_t)(v >> 32));
        len = a.fact_len[id];
      }
      a.ids_out[(size_t)q * a.k + r] = id;
      a.scores_out[(size_t)q * a.k + r] = s;
    }
    if (a.fact_seg_off) {
      int32_t tot;
      const int32_t ex = block_exclusive_scan(len, scratch, &tot);
      if (r < kk) a.fact_seg_off[(size_t)q * a.seg_stride + r] = carry + ex;
      carry += tot;
    }
  }
  if (a.fact_seg_off && tid == 0) {
    int nn = kk;
    const int32_t start = a.seg_start[q];
    if (start < 0 || (int64_t)start + carry > (int64_t)IS_MAX_POSITION) {
      latch(a.status, IS_ST_POSITION);
      nn = 0;
      carry = 0;
    }
    a.fact_seg_off[(size_t)q * a.seg_stride + nn] = carry;
    a.n_ids_out[q] = nn;
    a.seg_len[q] = carry;
  }
}

cudaError_t launch_topk(const TopkArgs& a, const LaunchCfg& cfg) {
  topk_kernel<<<a.Q, kTopkThreads, 0, cfg.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace isk
