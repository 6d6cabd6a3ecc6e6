// Exact top-k of one query's cosine scores by one CTA of kRetThreads threads,
// shared by the per-query retrieval kernel and the batched (tensor-core) path.
#pragma once

#include "block_scan.cuh"
#include "common.cuh"

namespace isk {

constexpr int kRetThreads = 256;
constexpr int64_t kSmemKeysMax = 4096;     // keys staged in shared memory up to this n

// Warp-aggregated slot claim: lanes with `take` get consecutive positions
// from one atomic on *counter per warp.  All 32 lanes must call it.
__device__ __forceinline__ uint32_t warp_claim(bool take, uint32_t* counter, int lane) {
  const unsigned m = __ballot_sync(0xffffffffu, take);
  uint32_t base = 0;
  if (lane == 0 && m) base = atomicAdd(counter, (uint32_t)__popc(m));
  base = __shfl_sync(0xffffffffu, base, 0);
  return base + (uint32_t)__popc(m & ((1u << lane) - 1u));
}

__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t x, int lane, uint32_t* total) {
  uint32_t inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  *total = __shfl_sync(0xffffffffu, inc, 31);
  return inc - x;
}

constexpr int kCandMax = IS_MAX_K;          // candidates sorted exactly (10-bit slot index)
constexpr int kRegPer = 8;                  // scores per thread held in registers (REG mode)
constexpr int kRegKeys = kRegPer * kRetThreads;
static_assert(kCosBins % kRetThreads == 0 && kRetThreads <= kCandMax && kRetThreads <= 1024,
              "bins split evenly over the threads; the rank path holds one candidate per thread");

struct TopkShared {
  uint32_t hist[kCosBins];                  // cosine bins; the radix fallback reuses it as [4][256]
  unsigned long long sel[kCandMax];         // (key << 32) | ((2^20-1 - row) << 10) | slot
  unsigned long long cand[kCandMax];        // (length << 32) | fact id, by slot (by rank on the rank path)
  int64_t rk_tok[kCandMax];                 // rank path: arena token by rank
  int32_t scratch[33];
  int32_t scratch2[kRetThreads / 32];       // second buffer of the one-barrier scans
  uint32_t bstar, above, eq, digit, cnt;
};

// Bin of a cosine in [-1, 1] on a uniform 2048-bin grid (monotone in s).
__device__ __forceinline__ int cos_bin(float s) {
  const int b = (int)((s + 1.0f) * 1024.0f);
  return min(kCosBins - 1, max(0, b));
}

__device__ __forceinline__ unsigned long long sel_entry(uint32_t key, uint32_t row, uint32_t slot) {
  return ((unsigned long long)key << 32) | ((unsigned long long)(0xFFFFFu - row) << 10) | slot;
}

// True when the similarity CTAs of a query over n rows count their scores
// into a.hist and its top-k takes the register path (the two sides must agree:
// the top-k zeroes the bins it read for the next call).
__device__ __forceinline__ bool topk_uses_hist(const TopkArgs& a, int n) {
  return a.hist != nullptr && n >= 1 && n <= kRegKeys;
}

// Records candidate `slot` = row j of the user: its fact id and length.
__device__ __forceinline__ void fetch_cand(const TopkArgs& a, TopkShared& sh, const int4& um, uint32_t j,
                                           uint32_t slot) {
  const int tile = user_tile(a.user_tiles, um, (int)(j / kTile));
  const size_t row = (size_t)tile * kTile + (j % kTile);
  sh.cand[slot] = ((unsigned long long)(uint32_t)a.tile_len[row] << 32) | (uint32_t)a.tile_fact[row];
}

// Writes the segment plan's tail of query q (one thread): the total, the
// fact count and the segment length; `start` is seg_start[q].
__device__ __forceinline__ void plan_tail(const TopkArgs& a, int q, int nn, int32_t total, int32_t start) {
  int32_t* off = a.fact_seg_off + (size_t)q * a.seg_stride;
  if (start < 0 || (int64_t)start + total > (int64_t)IS_MAX_POSITION) {
    latch(a.status, IS_ST_POSITION);
    nn = 0;
    total = 0;
  }
  off[nn] = total;
  a.n_ids_out[q] = nn;
  a.seg_len[q] = total;
  if (a.seg_len_copy) a.seg_len_copy[q] = total;
}

// The top-k of query q by the whole CTA (kRetThreads threads):
//  A. load the n scores (8 loads in flight per thread), stage their
//     order-preserving keys, histogram their cosine bins; or, when the
//     similarity CTAs already counted the bins (topk_uses_hist), load each
//     thread's 8 scores and 8 bins into registers and zero those bins;
//  B. find the bin b* holding the k-th largest score;
//  C. candidates = every row in bins >= b* (k plus the rest of bin b*), with
//     their fact ids and lengths fetched on the way; if more than kCandMax
//     crowd into b* (heavy ties), an exact 4-pass radix select on the keys
//     picks exactly k rows instead (ties to the lower row);
//  D. exact sort of the candidates by (key desc, row asc) and output of the
//     first k, with the segment plan.
template <bool SMEM_KEYS>
__device__ void topk_block(const TopkArgs& a, TopkShared& sh, uint32_t* s_keys, int q, const int4& um,
                           int n) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kk = min(a.k, n);
  const float* sc = a.scores + (size_t)q * a.score_stride;
  const bool reg = topk_uses_hist(a, n);
  auto key_at = [&](int j) -> uint32_t {
    return (SMEM_KEYS && !reg) ? s_keys[j] : score_key(__ldcg(sc + j));
  };
  if (a.block_table) prefetch_row_l2(a.block_table + (size_t)q * a.max_blocks, a.max_blocks, tid, kRetThreads);
  int64_t* ids = a.ids_out + (size_t)q * a.k;
  float* scs = a.scores_out + (size_t)q * a.k;
  // Read now, used at the very end: its latency hides under the selection.
  const int32_t start_q = (a.fact_seg_off && tid == 0) ? a.seg_start[q] : 0;

  // Either path issues its score loads first: with bins counted by the
  // similarity CTAs, all n scores and the thread's bins in one round; without,
  // the first batch of scores before the shared histogram is cleared, so
  // their latency overlaps the clearing and the barrier.
  constexpr int BPT = kCosBins / kRetThreads;
  const int hi = kCosBins - 1 - BPT * tid;     // this thread's bins: hi, hi - 1, .., hi - BPT + 1
  float v[kRegPer];
  uint32_t c[BPT];
  auto load_batch = [&](int b) {
#pragma unroll
    for (int u = 0; u < kRegPer; ++u) {
      const int j = b + u * kRetThreads + tid;
      v[u] = j < n ? __ldcg(sc + j) : 0.f;
    }
  };
  if (reg) {
    // All n scores and this thread's bins in one round of loads; the bins are
    // then zeroed for the next call (this CTA is their only reader).
    // A thread's bins hi - BPT + 1 .. hi are consecutive words, 16-byte
    // aligned in groups of four: two vector loads and stores each.
    static_assert(BPT % 4 == 0, "bins per thread in whole 16-byte groups");
    uint32_t* hg = a.hist + (size_t)q * kCosBins;
    load_batch(0);
#pragma unroll
    for (int i = 0; i < BPT; i += 4) {
      const uint4 w = __ldcg(reinterpret_cast<const uint4*>(hg + hi - i - 3));
      c[i] = w.w;
      c[i + 1] = w.z;
      c[i + 2] = w.y;
      c[i + 3] = w.x;
    }
#pragma unroll
    for (int i = 0; i < BPT; i += 4) __stcg(reinterpret_cast<uint4*>(hg + hi - i - 3), make_uint4(0u, 0u, 0u, 0u));
    if (tid == 0) sh.cnt = 0;
  } else {
    if (kk > 0) load_batch(0);
    for (int i = tid; i < kCosBins; i += kRetThreads) sh.hist[i] = 0;
    if (tid == 0) sh.cnt = 0;
    __syncthreads();
  }
  if (kk > 0 && !reg) {
    for (int b = 0; b < n; b += kRegPer * kRetThreads) {
      if (b > 0) load_batch(b);
#pragma unroll
      for (int u = 0; u < kRegPer; ++u) {
        const int j = b + u * kRetThreads + tid;
        if (j < n) {
          if (SMEM_KEYS) s_keys[j] = score_key(v[u]);
          atomicAdd(&sh.hist[cos_bin(v[u])], 1u);
        }
      }
    }
  }
  for (int r = kk + tid; r < a.k; r += kRetThreads) {
    ids[r] = -1;
    scs[r] = -INFINITY;
  }
  __syncthreads();
  if (kk == 0) {
    if (a.fact_seg_off && tid == 0) plan_tail(a, q, 0, 0, start_q);
    return;
  }

  // B: the bins in descending order, BPT per thread in thread order; a block
  // scan of the per-thread counts finds the thread holding the k-th score.
  {
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      if (!reg) c[i] = sh.hist[hi - i];
      sum += c[i];
    }
    int32_t tot;
    const uint32_t before = (uint32_t)block_exclusive_scan_1bar<kRetThreads / 32>((int32_t)sum, sh.scratch, &tot);
    if (reg) {
      // Rows in the bins above each of this thread's bins: a candidate's
      // first free slot in bin order (the shared histogram is unused here).
      uint32_t run = before;
#pragma unroll
      for (int i = 0; i < BPT; ++i) {
        sh.hist[hi - i] = run;
        run += c[i];
      }
    }
    if (before < (uint32_t)kk && before + sum >= (uint32_t)kk) {
      uint32_t run = before;
#pragma unroll
      for (int i = 0; i < BPT; ++i) {
        if (run < (uint32_t)kk && run + c[i] >= (uint32_t)kk) {
          sh.bstar = hi - i;
          sh.above = run;
          sh.eq = c[i];
        }
        run += c[i];
      }
    }
    __syncthreads();
  }

  uint32_t C;                                   // candidates to sort
  if (sh.above + sh.eq <= (uint32_t)kCandMax) {
    const int bstar = sh.bstar;
    C = sh.above + sh.eq;
    if (reg) {
      // Scores in registers: a candidate takes the next slot of its bin
      // (bins hold their first slot, in descending bin order); the order
      // within a bin does not matter, the ranking below counts.
#pragma unroll
      for (int u = 0; u < kRegPer; ++u) {
        const int j = u * kRetThreads + tid;
        const int b = cos_bin(v[u]);
        if (j < n && b >= bstar) {
          const uint32_t slot = atomicAdd(&sh.hist[b], 1u);
          sh.sel[slot] = sel_entry(score_key(v[u]), (uint32_t)j, slot);
        }
      }
    } else if (SMEM_KEYS) {
      // Keys in shared memory: count this thread's candidates, one block scan
      // gives each thread its first slot, then a second pass writes them.
      uint32_t mine = 0;
      for (int j = tid; j < n; j += kRetThreads) mine += cos_bin(key_score(s_keys[j])) >= bstar ? 1u : 0u;
      int32_t tot;
      uint32_t slot = (uint32_t)block_exclusive_scan_1bar<kRetThreads / 32>((int32_t)mine, sh.scratch2, &tot);
      for (int j = tid; j < n; j += kRetThreads) {
        const uint32_t key = s_keys[j];
        if (cos_bin(key_score(key)) >= bstar) {
          sh.sel[slot] = sel_entry(key, (uint32_t)j, slot);
          ++slot;
        }
      }
    } else {
      for (int b = 0; b < n; b += kRetThreads) {
        const int j = b + tid;
        const uint32_t key = j < n ? key_at(j) : 0u;
        const bool take = j < n && cos_bin(key_score(key)) >= bstar;
        const uint32_t slot = warp_claim(take, &sh.cnt, lane);
        if (take) sh.sel[slot] = sel_entry(key, (uint32_t)j, slot);
      }
    }
  } else {
    // Radix select: 8 bits per pass finds the k-th largest key thr and how
    // many keys equal to it to take.
    uint32_t* h4 = sh.hist;                    // [4][256]
    for (int i = tid; i < 1024; i += kRetThreads) h4[i] = 0;
    __syncthreads();
    uint32_t prefix = 0, rem = (uint32_t)kk;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      const uint32_t hmask = pass == 0 ? 0u : (0xffffffffu << (32 - 8 * pass));
      for (int b = 0; b < n; b += kRetThreads) {
        const int j = b + tid;
        bool in = false;
        uint32_t digit = 256u;
        if (j < n) {
          const uint32_t key = key_at(j);
          in = (key & hmask) == prefix;
          if (in) digit = (key >> shift) & 255u;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, digit);
        if (in && lane == __ffs(peers) - 1) atomicAdd(&h4[pass * 256 + digit], (uint32_t)__popc(peers));
      }
      __syncthreads();
      if (warp == 0) {
        uint32_t c[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = h4[pass * 256 + 255 - 8 * lane - i];
          sum += c[i];
        }
        uint32_t tot;
        const uint32_t before = warp_excl_scan(sum, lane, &tot);
        if (before < rem && before + sum >= rem) {
          uint32_t run = before;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (run < rem && run + c[i] >= rem) {
              sh.digit = 255u - 8u * lane - i;
              sh.above = run;
              sh.eq = c[i];
            }
            run += c[i];
          }
        }
      }
      __syncthreads();
      prefix |= sh.digit << shift;
      rem -= sh.above;
    }
    const uint32_t thr = prefix;
    const uint32_t n_gt = (uint32_t)kk - rem;
    C = (uint32_t)kk;
    uint32_t taken = 0;
    for (int b = 0; b < n; b += kRetThreads) {
      const int j = b + tid;
      const uint32_t key = j < n ? key_at(j) : 0u;
      const bool gt = j < n && key > thr;
      const uint32_t slot = warp_claim(gt, &sh.cnt, lane);
      if (gt) sh.sel[slot] = sel_entry(key, (uint32_t)j, slot);
      // keys == thr in ascending row order, until rem of them are taken
      const int32_t is_eq = (j < n && key == thr) ? 1 : 0;
      int32_t tot;
      const int32_t rank = block_exclusive_scan(is_eq, sh.scratch, &tot);
      if (is_eq && taken + (uint32_t)rank < rem) {
        const uint32_t slot_eq = n_gt + taken + (uint32_t)rank;
        sh.sel[slot_eq] = sel_entry(key, (uint32_t)j, slot_eq);
      }
      taken += (uint32_t)tot;
    }
  }
  __syncthreads();

  if (C <= (uint32_t)kRetThreads) {
    // Rank selection: candidate c's rank is the number of candidates above it
    // (entries are unique), counted by S neighbouring threads over every S-th
    // entry and summed by shuffles; S is the largest power of two up to 8
    // that keeps S threads per candidate.  The fact lookup (by the first of
    // the S) overlaps the ranking.  The top kk are then placed by rank (fact
    // and length in sh.cand, store token in sh.rk_tok, key in the histogram's
    // space), so thread r writes rank r's outputs and one block scan of the
    // lengths gives the segment offsets.
    const uint32_t t = (uint32_t)tid;
    int64_t* rk_tok = sh.rk_tok;
    uint32_t* rk_key = sh.hist;                                       // free by now
    uint32_t S = 1;
    while (S < 8 && C * S * 2 <= (uint32_t)kRetThreads) S <<= 1;
    const uint32_t cidx = t / S, part = t % S;
    const bool have = cidx < C;
    const unsigned long long e = have ? sh.sel[cidx] : 0ull;
    int32_t f = 0, len = 0;
    int64_t tok = 0;
    if (have && part == 0) {
      const uint32_t j = 0xFFFFFu - (uint32_t)((e >> 10) & 0xFFFFFu);
      const int tile = user_tile(a.user_tiles, um, (int)(j / kTile));
      const size_t row = (size_t)tile * kTile + (j % kTile);
      f = a.tile_fact[row];
      len = a.tile_len[row];
      tok = a.tile_tok[row];
    }
    uint32_t rank = 0;
    if (have) {
      // Four independent counts keep four shared-memory reads in flight.
      uint32_t r0 = 0, r1 = 0, r2 = 0, r3 = 0, i = part;
      for (; i + 3 * S < C; i += 4 * S) {
        r0 += sh.sel[i] > e ? 1u : 0u;
        r1 += sh.sel[i + S] > e ? 1u : 0u;
        r2 += sh.sel[i + 2 * S] > e ? 1u : 0u;
        r3 += sh.sel[i + 3 * S] > e ? 1u : 0u;
      }
      for (; i < C; i += S) r0 += sh.sel[i] > e ? 1u : 0u;
      rank = r0 + r1 + r2 + r3;
    }
    for (uint32_t o = 1; o < S; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, (int)o);
    if (have && part == 0 && rank < (uint32_t)kk) {
      sh.cand[rank] = ((unsigned long long)(uint32_t)len << 32) | (uint32_t)f;
      rk_tok[rank] = tok;
      rk_key[rank] = (uint32_t)(e >> 32);
    }
    __syncthreads();
    const unsigned long long cv = t < (uint32_t)kk ? sh.cand[t] : 0ull;
    int32_t total;
    const int32_t off = block_exclusive_scan_1bar<kRetThreads / 32>((int32_t)(cv >> 32), sh.scratch, &total);
    if (t < (uint32_t)kk) {
      ids[t] = (int32_t)(uint32_t)cv;
      scs[t] = key_score(rk_key[t]);
      if (a.fact_seg_off) {
        a.fact_seg_off[(size_t)q * a.seg_stride + t] = off;
        a.fact_src[(size_t)q * a.seg_stride + t] = rk_tok[t];
      }
    }
    if (a.fact_seg_off && t == 0) plan_tail(a, q, kk, total, start_q);
    return;
  }

  // More candidates: fetch their fact ids and lengths, then sort.
  for (uint32_t t = (uint32_t)tid; t < C; t += kRetThreads) {
    const uint32_t j = 0xFFFFFu - (uint32_t)((sh.sel[t] >> 10) & 0xFFFFFu);
    fetch_cand(a, sh, um, j, t);
  }
  // C > 64: bitonic sort in shared memory over the next power of two.
  int P = 1;
  while ((uint32_t)P < C) P <<= 1;
  for (int i = (int)C + tid; i < P; i += kRetThreads) sh.sel[i] = 0ull;
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P / 2; i += kRetThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long x = sh.sel[lo], y = sh.sel[hi];
        if ((x < y) == desc) {
          sh.sel[lo] = y;
          sh.sel[hi] = x;
        }
      }
      __syncthreads();
    }
  }
  int32_t carry = 0;
  for (int b = 0; b < kk; b += kRetThreads) {
    const int r = b + tid;
    int32_t len = 0;
    if (r < kk) {
      const unsigned long long e = sh.sel[r];
      const unsigned long long cv = sh.cand[e & 1023u];
      len = (int32_t)(cv >> 32);
      ids[r] = (int32_t)(uint32_t)cv;
      scs[r] = key_score((uint32_t)(e >> 32));
      if (a.fact_src) a.fact_src[(size_t)q * a.seg_stride + r] = a.fact_tok[(int32_t)(uint32_t)cv];
    }
    if (a.fact_seg_off) {
      int32_t tot;
      const int32_t ex = block_exclusive_scan(len, sh.scratch, &tot);
      if (r < kk) a.fact_seg_off[(size_t)q * a.seg_stride + r] = carry + ex;
      carry += tot;
    }
  }
  if (a.fact_seg_off && tid == 0) plan_tail(a, q, kk, carry, start_q);
}

}  // namespace isk
