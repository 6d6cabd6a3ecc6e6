// GPU-resident semantic retrieval: cosine similarity against one user's
// stored embeddings, then an exact top-k (topk.cuh).
//
// InferScale keeps the retrieval index and the KV store both on the GPU so
// retrieved text never crosses PCIe ("Conception de Système Native au GPU"),
// and retrieves a relevant subset of k facts per request ("Problématique").
// The index it names is not described; retrieval here is exact cosine top-k.
#include <algorithm>

#include "block_scan.cuh"
#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

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
// Fused retrieval: cosine similarity + exact top-k in one launch.
//
// Grid (tiles * n_sub, Q).  CTA (x, q) scores 128 / n_sub embedding rows of
// one tile of q's user, one warp per row: each lane streams 16-byte chunks of
// the row and of the query together and accumulates q.e and q.q in fp32, so
// the warp needs no shared memory and no barrier.  Rows of one user are
// numbered 0 .. n_u-1 in fill order (tile after tile), which is insertion
// order, hence ascending fact id.  After its rows, each CTA arrives on q's
// counter; the last one (the counter reaches tiles * n_sub) resets the counter
// and runs the top-k of q over the scores, which are then in L2.  Up to
// kRegKeys rows per user, each row's score is also counted into q's cosine
// bins in global memory (ta.hist), so the top-k starts from a finished
// histogram.
//
// Top-k (topk_block): a cosine-bin histogram locates the bin of the k-th
// score, the rows in and above it are the candidates (an exact radix select
// takes over when ties crowd one bin), and the candidates are ordered by
// (score desc, row asc), so ties go to the lower fact id; ids, scores and the
// segment plan (exclusive prefix of the facts' lengths) are written.
template <typename E, bool SMEM_KEYS>
__global__ void __launch_bounds__(kRetThreads, 4) retrieve_kernel(const SimArgs sa, const TopkArgs ta,
                                                               int n_sub, int32_t* arrive) {
  extern __shared__ uint32_t s_keys[];         // [n] keys of the top-k phase (SMEM_KEYS)
  __shared__ TopkShared sh;
  __shared__ int s_last;
  const int q = blockIdx.y;
  const int ti = blockIdx.x / n_sub;
  const int sub = blockIdx.x - ti * n_sub;
  // Pages written later (scores, top-k outputs, plan) and the store's per-user
  // records: warm their translations now, in parallel with the user lookup.
  warm8(sa.scores + (size_t)q * sa.score_stride, ta.ids_out, ta.scores_out, ta.fact_seg_off, ta.fact_src,
        ta.seg_len, sa.user_meta, sa.emb_inv_norm);
  // The query row does not depend on the user lookup: start pulling it into L2.
  if (threadIdx.x * 128 < sa.E * (int)sizeof(E))
    prefetch_l2(reinterpret_cast<const uint8_t*>(sa.q_emb) + ((size_t)q * sa.E * sizeof(E)) + threadIdx.x * 128);
  // The cosine bins the rows below may count into (64 lines of 128 bytes per
  // query, one per CTA in turn) and the start the top-k reads last.
  if (ta.hist && threadIdx.x == 32)
    prefetch_l2(ta.hist + (size_t)q * kCosBins + (blockIdx.x % (kCosBins / 32)) * 32);
  if (ta.seg_start && threadIdx.x == 64 && blockIdx.x == 0) prefetch_l2(ta.seg_start + q);
  const int user = sa.users[q];
  const bool user_ok = user >= 0 && user < sa.max_users;
  const int4 um = user_ok ? sa.user_meta[user] : make_int4(0, 0, 0, -1);
  const int ntiles = um.y;
  if (ntiles == 0) {
    // Unknown user or no facts: CTA x = 0 writes the empty result.
    if (blockIdx.x == 0) {
      if (!user_ok && threadIdx.x == 0) latch(sa.status, IS_ST_USER_RANGE);
      topk_block<SMEM_KEYS>(ta, sh, s_keys, q, um, 0);
    }
    return;
  }
  if (ti >= ntiles) return;
  const int n_u = um.z;
  const int tile = user_tile(sa.user_tiles, um, ti);
  const int rows_per = kTile / n_sub;
  const int r_begin = sub * rows_per;
  const int r_end = min(r_begin + rows_per, n_u - ti * kTile);
  constexpr int VE = EmbT<E>::V::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const E* qv = reinterpret_cast<const E*>(sa.q_emb) + (size_t)q * sa.E;
  const E* base = reinterpret_cast<const E*>(sa.emb) + (size_t)tile * kTile * sa.E;
  float* out = sa.scores + (size_t)q * sa.score_stride + (size_t)ti * kTile;
  uint32_t* bins = topk_uses_hist(ta, n_u) ? ta.hist + (size_t)q * kCosBins : nullptr;
  // The top-k will look up the fact, length and arena token of its candidate
  // rows: warm those lines of this CTA's rows now.
  if (threadIdx.x < 3 && r_begin < r_end) {
    const size_t row0 = (size_t)tile * kTile + r_begin;
    const void* p = threadIdx.x == 0 ? (const void*)(ta.tile_fact + row0)
                  : threadIdx.x == 1 ? (const void*)(ta.tile_len + row0) : (const void*)(ta.tile_tok + row0);
    prefetch_l2(p);
  }
  for (int r = r_begin + warp; r < r_end; r += kRetThreads / 32) {
    const float inv_e = sa.emb_inv_norm[(size_t)tile * kTile + r];
    const E* row = base + (size_t)r * sa.E;
    float dot = 0.f, qq = 0.f;
#pragma unroll 4
    for (int c = lane * VE; c < sa.E; c += 32 * VE) {
      float x[VE], y[VE];
      EmbT<E>::V::unpack(*reinterpret_cast<const uint4*>(row + c), x);
      EmbT<E>::V::unpack(*reinterpret_cast<const uint4*>(qv + c), y);
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        dot = fmaf(x[e], y[e], dot);
        qq = fmaf(y[e], y[e], qq);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      dot += __shfl_xor_sync(0xffffffffu, dot, o);
      qq += __shfl_xor_sync(0xffffffffu, qq, o);
    }
    if (lane == 0) {
      const float score = dot * (qq > 0.f ? 1.0f / sqrtf(qq) : 0.f) * inv_e;
      out[r] = score;
      if (bins) atomicAdd(bins + cos_bin(score), 1u);
    }
  }
  // Arrive; the last CTA of query q runs its top-k.  The arrival releases
  // the CTA's scores and bin counts (ordered before it by the barrier) and,
  // for the last CTA, acquires everyone else's.
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t done = atom_add_acq_rel(reinterpret_cast<uint32_t*>(&arrive[q]), 1u);
    s_last = done == (uint32_t)(ntiles * n_sub - 1);
    if (s_last) arrive[q] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  // The dependent inject grid may launch once every CTA has exited or
  // triggered: here, when the last one starts its top-k.  Its launch latency
  // then hides under the top-k, and its CTAs are placed on SMs the similarity
  // CTAs have left (triggering at kernel start let them land among running
  // similarity CTAs, which measured 6 us slower per Llama-3.1-8B step).
  pdl_trigger();
  topk_block<SMEM_KEYS>(ta, sh, s_keys, q, um, n_u);
}

template <typename E>
static cudaError_t launch_retrieve_t(const SimArgs& sa, const TopkArgs& ta, int n_sub, dim3 grid,
                                     int64_t max_user_facts, int32_t* arrive, const LaunchCfg& cfg) {
  if (max_user_facts <= kSmemKeysMax) {
    const size_t smem = (size_t)std::max<int64_t>(max_user_facts, 1) * sizeof(uint32_t);
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(retrieve_kernel<E, true>), smem);
    if (e != cudaSuccess) return e;
    return launch_ex(retrieve_kernel<E, true>, grid, dim3(kRetThreads), smem, cfg.stream, cfg.pdl, sa,
                     ta, n_sub, arrive);
  }
  return launch_ex(retrieve_kernel<E, false>, grid, dim3(kRetThreads), 0, cfg.stream, cfg.pdl, sa, ta,
                   n_sub, arrive);
}

cudaError_t launch_retrieve(const SimArgs& sa, const TopkArgs& ta, int emb_dtype, int max_user_tiles,
                            int64_t max_user_facts, int32_t* arrive, const LaunchCfg& cfg) {
  // Split tiles into sub-tiles until the grid covers the SMs a few times over.
  const int tiles = std::max(1, max_user_tiles);
  // At most one row per warp: a sub-tile keeps every warp of the CTA busy.
  constexpr int kMaxSub = kTile / (kRetThreads / 32);
  int n_sub = 1;
  while (n_sub < kMaxSub && (int64_t)tiles * sa.Q * n_sub < 4LL * cfg.num_sms) n_sub *= 2;
  const dim3 grid(tiles * n_sub, sa.Q);
  if (emb_dtype == IS_F16)
    return launch_retrieve_t<__half>(sa, ta, n_sub, grid, max_user_facts, arrive, cfg);
  return launch_retrieve_t<float>(sa, ta, n_sub, grid, max_user_facts, arrive, cfg);
}

}  // namespace isk
