// Segment planning and the fused gather + Chunked RoPE + paged scatter-copy.
//
// InferScale ("Méthodologie", phase 2): the retrieved facts are composed into
// one contiguous segment, every stored pre-RoPE key is rotated to its
// serving-time position (Theorem 6: exact) and the composed K/V are
// scatter-copied into vLLM's paged KV cache.  One pass over the data: each
// (token, layer) row pair is read once from the store and written once to the
// cache, the rotation done in registers on the way.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "block_scan.cuh"
#include "common.cuh"
#include "internal.h"

namespace isk {

// ---------------------------------------------------------------------------
// Plan of an explicit fact list: validate ids, prefix sum of their lengths.
// One CTA per request.
__global__ void __launch_bounds__(256) plan_kernel(const PlanArgs a) {
  __shared__ int32_t scratch[33];
  pdl_trigger();
  const int r = blockIdx.x;
  int n = a.n_ids_in[r];
  if (n < 0 || n > a.ids_stride) {
    if (threadIdx.x == 0) latch(a.status, IS_ST_COUNT);
    n = 0;
  }
  const int32_t user = a.users ? a.users[r] : -1;
  int32_t* off = a.fact_seg_off + (size_t)r * a.seg_stride;
  if (a.zero_ctr && r == 0 && threadIdx.x < kPoolCtrs) a.zero_ctr[threadIdx.x * kCtrStride] = 0u;
  if (a.block_table) prefetch_row_l2(a.block_table + (size_t)r * a.max_blocks, a.max_blocks, threadIdx.x, blockDim.x);
  int32_t carry = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    int32_t len = 0;
    if (i < n) {
      const int64_t f = a.ids[(size_t)r * a.ids_stride + i];
      if (f < 0 || f >= a.n_facts) {
        latch(a.status, IS_ST_FACT_RANGE);
      } else if (user >= 0 && a.fact_user[f] != user) {
        latch(a.status, IS_ST_FACT_USER);
      } else {
        len = a.fact_len[f];
        if (a.arena_tokens > 0) {
          const int64_t tok = a.fact_tok[f];
          if (len < 1 || len > a.max_fact_len || tok < 0 || tok > a.arena_tokens - len) {
            latch(a.status, IS_ST_FACT_RANGE);
            len = 0;
          }
        }
        if (a.fact_src) a.fact_src[(size_t)r * a.seg_stride + i] = a.fact_tok[f];
      }
    }
    int32_t tot;
    const int32_t ex = block_exclusive_scan(len, scratch, &tot);
    if (i < n) off[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) {
    const int32_t start = a.seg_start[r];
    if (start < 0 || (int64_t)start + carry > (int64_t)IS_MAX_POSITION) {
      latch(a.status, IS_ST_POSITION);
      n = 0;
      carry = 0;
    }
    off[n] = carry;
    a.n_ids_out[r] = n;
    a.seg_len[r] = carry;
  }
}

// ---------------------------------------------------------------------------
// Gather + Chunked RoPE + paged scatter.
//
// Work item = (segment token t, group of G consecutive layers): per layer the
// K row and the V row, H*D elements each; a token's layers sit back to back in
// the token-major store, so one bulk copy of 2 * G * row_bytes brings the
// group into shared memory.  G is 1 for rows of 2 KiB and more and grows for
// smaller rows so that one copy moves about 4 KiB (per-item costs are per
// copy, not per byte).  Items are numbered t * groups + g over all requests
// back to back and each warp takes one contiguous run.
//
// Each warp runs its own pipeline over a ring of P shared-memory stages: lane
// 0 issues the bulk load of item i + P - 1 while the warp works on item i, so
// the bytes in flight are set by shared memory (P stages per warp), not by
// registers.  On the way out, V leaves shared memory by a bulk store; K is
// read from shared memory, rotated in fp32 and stored with 16-byte vector
// stores.  NeoX pairs (i, i + D/2) lie in vectors v and v ^ half_vecs of the
// row, interleaved pairs inside one vector; either way the frequencies a lane
// needs depend only on its lane index, so it computes VE (or VE/2) sin/cos
// once per position.  Every mbarrier wait is bounded (a.wait_ns, 2 s unless
// the store was told otherwise): on time-out the warp latches IS_ST_TIMEOUT,
// stops issuing, waits up to kWaitBudgetNs for each of its loads in flight to
// land, waits for its bulk stores and returns.
constexpr int kInjectWarpsMax = 8;

struct StageMeta {
  int64_t slot;     // destination slot, -1 = nothing to do
  int32_t p;        // position (rotation angle)
  int16_t l;        // first layer of the group (within this call)
  int16_t nl;       // layers in the group
};

// Chunked RoPE on one 16-byte vector of a key row (VE elements).  x holds the
// vector; for NeoX pairs (i, i + D/2), z holds its partner vector v ^ half_vecs
// and `first` says whether v is the pair's first half (a' = a cos - b sin) or
// second (b' = b cos + a sin); interleaved pairs (2i, 2i + 1) lie inside the
// vector and z is unused.  cs / sn are the lane's cos / sin, one per frequency.
template <typename T, int STYLE>
__device__ __forceinline__ void rotate_vec(const float* x, const float* z, bool first, const float* cs,
                                           const float* sn, float* y) {
  constexpr int VE = Vec<T>::N;
  if (STYLE == 0) {
    if (first) {
#pragma unroll
      for (int e = 0; e < VE; ++e) y[e] = fmaf(x[e], cs[e], -z[e] * sn[e]);
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e) y[e] = fmaf(x[e], cs[e], z[e] * sn[e]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < VE / 2; ++e) {
      const float u = x[2 * e], w = x[2 * e + 1];
      y[2 * e] = fmaf(u, cs[e], -w * sn[e]);
      y[2 * e + 1] = fmaf(w, cs[e], u * sn[e]);
    }
  }
}

// NeoX rotation of one vector with the sines already signed for the lane's
// half of the pair (sx = -sin for the first half, +sin for the second):
// y = x cos + z sx, two lanes per instruction.  Each element is rounded
// exactly as rotate_vec rounds it (-(z sin) is exact), so the two agree bit
// for bit.
template <int VE>
__device__ __forceinline__ void rotate_neox_x2(const float* x, const float* z, const float* cs,
                                               const float* sx, float* y) {
#pragma unroll
  for (int e = 0; e < VE; e += 2) {
    const unsigned long long t = mul2_rn(pk2(z[e], z[e + 1]), pk2(sx[e], sx[e + 1]));
    upk2(fma2_rn(pk2(x[e], x[e + 1]), pk2(cs[e], cs[e + 1]), t), y[e], y[e + 1]);
  }
}

// Rotated key vector v of a row at dk: 16 bytes in the store's type, or 8
// E4M3 bytes (times fp32(1 / k_scale)) for an FP8 cache.
template <typename T, bool F8>
__device__ __forceinline__ void store_key(uint8_t* dk, int v, const float* y, float k_inv) {
  if (F8)
    st_v2(dk + (size_t)v * 8, to_e4m3x8(y, k_inv));
  else
    st_v4(dk + (size_t)v * 16, Vec<T>::pack(y));
}

// x / d for non-negative operands, in 32-bit arithmetic when both fit.
__device__ __forceinline__ int64_t div_nn(int64_t x, int64_t d) {
  return ((x | d) >> 31) == 0 ? (int64_t)((uint32_t)x / (uint32_t)d) : x / d;
}

// Shared-memory ints the request table needs: the prefix (R + 1) and the
// starts (R) for the block-wide scan, or a 66-entry slice per warp when every
// warp scans R <= 32 requests itself.
__host__ __device__ constexpr int prefix_ints(int R, int warps) { return R <= 32 ? warps * 66 : 2 * R + 1; }

// Exclusive prefix of seg_len over the R requests; returns the total token
// count, points *s_off at the prefix (R + 1 entries, the last = total) and
// *s_start at the requests' seg_start (read in the same round, so a token's
// position, and with it its block-table entry, is known before its fact).
// Up to 32 requests, each warp loads and scans them with shuffles into its
// own slice of `region`, so no block-wide barrier sits between the planning
// kernel's outputs and the warp's first copy; more requests are scanned by the
// whole block.  All threads of the block call it.
__device__ __forceinline__ int32_t segment_prefix(const InjectArgs& a, int32_t* region, int32_t* scratch,
                                                  const int32_t** s_off, const int32_t** s_start) {
  if (a.R <= 32) {
    const int lane = threadIdx.x & 31;
    int32_t* mine = region + (threadIdx.x >> 5) * 66;
    const int32_t v = lane < a.R ? a.seg_len[lane] : 0;
    if (lane < a.R) mine[33 + lane] = a.seg_start[lane];
    int32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const int32_t total = __shfl_sync(0xffffffffu, inc, 31);
    if (lane < a.R) mine[lane] = inc - v;
    if (lane == 0) mine[a.R] = total;
    __syncwarp();
    *s_off = mine;
    *s_start = mine + 33;
    return total;
  }
  int32_t total = 0;
  const int per = (a.R + blockDim.x - 1) / blockDim.x;
  const int b = min(a.R, (int)threadIdx.x * per);
  const int e = min(a.R, b + per);
  int32_t sum = 0;
  for (int i = b; i < e; ++i) sum += a.seg_len[i];
  int32_t base = block_exclusive_scan(sum, scratch, &total);
  for (int i = b; i < e; ++i) {
    region[i] = base;
    region[a.R + 1 + i] = a.seg_start[i];
    base += a.seg_len[i];
  }
  if (threadIdx.x == 0) region[a.R] = total;
  __syncthreads();
  *s_off = region;
  *s_start = region + a.R + 1;
  return total;
}

// One warp pulls block-table lines into L1: up to kBtLines 128-byte lines in
// all, split evenly over the requests (at least one each for the first
// kBtLines).  Rows that fit their share are taken whole; longer ones from the
// line of the request's first position on, which costs the warp a dependent
// read of the start first (a delay of its own first item when no dependency
// wait hides it).
constexpr int kBtLines = 128;
__device__ __forceinline__ void prefetch_block_rows(const InjectArgs& a, int lane) {
  if (!a.block_table || a.R <= 0) return;
  const int per = max(1, kBtLines / a.R);
  const int row_lines = (a.max_blocks + 31) >> 5;
  const bool whole = row_lines <= per;
  for (int i = lane; i < kBtLines && i < a.R * per; i += 32) {
    const int r = i / per;
    int line = i % per;
    if (!whole) {
      const int start = a.seg_start[r];
      line += (start >= 0 ? start / a.block_size : 0) / 32;
    }
    if (line < row_lines) prefetch_l1(a.block_table + (size_t)r * a.max_blocks + (size_t)line * 32);
  }
}

// K block of layer l (counted from the call's first layer) in the
// destination: its own tensor, or l layer strides into one cache.
__device__ __forceinline__ uint8_t* layer_base(const InjectArgs& a, int l) {
  return a.per_layer ? a.layer_cache[l] : a.cache + (size_t)l * a.layer_stride;
}

// Warp-uniform walk from a composed-segment token t (all requests back to
// back) to its store token, serving position and destination slot.  Tokens a
// warp visits are consecutive, so the request, fact and block-table entry found
// last time are kept and looked up again only when t leaves them.
//
// Finding the fact of a token is on the critical path of every warp's first
// item, so it is one round of independent loads: the request's fact count and
// the first 128 entries of its plan (segment offset and store token of each
// fact, four per lane); a ballot then picks the last fact whose offset is <=
// the token's.  Longer plans continue with a strided search over the rest.
// The token's block-table entry depends only on its position, so its load is
// issued before the fact lookup and overlaps it.
struct TokenCursor {
  int32_t t = -1, r = -1, j = 0, lo = 0, hi = 0;
  int64_t src0 = 0;     // store token of fact j's first token
  int32_t lb = -1, blk = -1;
  int64_t src = 0;      // store token
  int64_t slot = -1;    // cache slot, -1 if the block table rejects the position
  int32_t p = 0;        // position in the request's sequence

  static constexpr int kPer = 4;    // plan entries per lane in the first round

  __device__ __forceinline__ void find_fact(const InjectArgs& a, int rr, int32_t ts, int lane) {
    const int32_t* off = a.fact_seg_off + (size_t)rr * a.seg_stride;
    const int64_t* fsrc = a.fact_src ? a.fact_src + (size_t)rr * a.seg_stride : nullptr;
    const int n = a.n_ids[rr];
    int32_t o[kPer];
    int64_t sv[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int idx = lane * kPer + e;
      const bool in = idx < a.seg_stride;
      o[e] = in ? off[idx] : 0;
      sv[e] = (in && fsrc) ? fsrc[idx] : 0;
    }
    // Offsets never decrease, so "offset <= ts" holds for a prefix of the
    // facts; its last entry is the fact holding ts (off[0] = 0 <= ts).  A
    // fact the plan left out has length 0: the entry after it has the same
    // offset (or it is the last, whose offset is the segment length > ts), so
    // it is never that last entry.
    int best = -1;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int idx = lane * kPer + e;
      if (idx < n && idx < a.seg_stride && o[e] <= ts) best = idx;
    }
    const unsigned m = __ballot_sync(0xffffffffu, best >= 0);
    const int owner = 31 - __clz(m);
    int jlo = __shfl_sync(0xffffffffu, best, owner);
    constexpr int kFan = 32 * kPer;
    auto pick32 = [&](const int32_t* v, int idx) -> int32_t {
      const int e = idx % kPer;
      int32_t x = v[0];
#pragma unroll
      for (int q = 1; q < kPer; ++q) x = e == q ? v[q] : x;
      return __shfl_sync(0xffffffffu, x, idx / kPer);
    };
    auto pick64 = [&](const int64_t* v, int idx) -> int64_t {
      const int e = idx % kPer;
      int64_t x = v[0];
#pragma unroll
      for (int q = 1; q < kPer; ++q) x = e == q ? v[q] : x;
      return __shfl_sync(0xffffffffu, x, idx / kPer);
    };
    if (jlo == kFan - 1 && n > kFan) {
      // Beyond the first round: strided search over [kFan - 1, n).
      int jhi = n;
      while (jhi - jlo > 1) {
        const int stride = (jhi - jlo + 31) >> 5;
        const int idx = jlo + lane * stride;
        const bool le = idx < jhi && off[idx] <= ts;
        const unsigned mm = __ballot_sync(0xffffffffu, le);
        jlo += (31 - __clz(mm)) * stride;
        jhi = min(jhi, jlo + stride);
      }
      lo = off[jlo];
      hi = off[jlo + 1];
      src0 = fsrc ? fsrc[jlo] : a.fact_tok[a.ids[(size_t)rr * a.ids_stride + jlo]];
    } else {
      lo = pick32(o, jlo);
      const int32_t hnext = pick32(o, min(jlo + 1, kFan - 1));
      hi = jlo + 1 < kFan ? hnext : off[jlo + 1];
      const int64_t s_in = pick64(sv, jlo);
      src0 = fsrc ? s_in : a.fact_tok[a.ids[(size_t)rr * a.ids_stride + jlo]];
    }
    r = rr;
    j = jlo;
  }

  __device__ __forceinline__ void seek(const InjectArgs& a, const int32_t* s_off, const int32_t* s_start,
                                       int32_t tt, int lane) {
    if (tt == t) return;
    t = tt;
    int rlo = 0, rhi = a.R;
    while (rhi - rlo > 1) {
      const int mid = (rlo + rhi) >> 1;
      if (s_off[mid] <= tt) rlo = mid; else rhi = mid;
    }
    const int32_t ts = tt - s_off[rlo];
    const int32_t pn = s_start[rlo] + ts;
    const int32_t lbn = pn / a.block_size;
    if (rlo != r || lbn != lb) {
      blk = lbn < a.max_blocks ? a.block_table[(size_t)rlo * a.max_blocks + lbn] : -1;
      lb = lbn;
    }
    if (rlo != r || ts < lo || ts >= hi) find_fact(a, rlo, ts, lane);
    src = src0 + (ts - lo);
    p = pn;
    slot = -1;
    if (lb >= a.max_blocks) {
      if (lane == 0) latch(a.status, IS_ST_BLOCK_TABLE);
    } else if (blk < 0 || blk >= a.num_blocks) {
      if (lane == 0) latch(a.status, IS_ST_BLOCK_ID);
    } else {
      slot = (int64_t)blk * a.block_size + (p - lb * a.block_size);
    }
  }
};

// A host-buffer call learns that the launch's work is done from a word of
// mapped host memory (a.host_done) rather than from the stream: once a CTA's
// writes are complete it arrives on a.done_ctr, and the last CTA to arrive
// resets the counter and stores a.done_seq into that word.  The calling
// thread polls it and sees the store before the stream reports the grid
// retired.  Every CTA reaches this point exactly once per launch (the kernels
// have no early exit), so the counter is back at zero for the next launch.
__device__ __forceinline__ void signal_host_done(const InjectArgs& a) {
  if (a.host_done == nullptr) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.done_ctr, 1u) == gridDim.x - 1) {
      *a.done_ctr = 0u;
      __threadfence_system();
      *reinterpret_cast<volatile uint32_t*>(a.host_done) = a.done_seq;
    }
  }
}

template <typename T, int STYLE, bool F8>
__global__ void __launch_bounds__(kInjectWarpsMax * 32) inject_kernel(const InjectArgs a,
                                                                      const RopeTurns rt, int P, int G) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int32_t scratch[33];
  constexpr int VE = Vec<T>::N;
  constexpr int NF = STYLE == 0 ? VE : VE / 2;
  static_assert(!F8 || VE == 8, "an FP8 cache takes 16-bit store rows");

  const int nwarps = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t item_bytes = 2u * (uint32_t)G * (uint32_t)a.row_bytes;   // one stage
  int32_t* off_region = reinterpret_cast<int32_t*>(smem);
  const size_t off_bytes = ((size_t)prefix_ints(a.R, kInjectWarpsMax) * 4 + 127) & ~(size_t)127;
  uint8_t* stages = smem + off_bytes + (size_t)warp * P * item_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + off_bytes + (size_t)nwarps * P * item_bytes) +
                   (size_t)warp * P;
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + off_bytes + (size_t)nwarps * P * item_bytes +
                                                 (size_t)nwarps * P * 8) + (size_t)warp * P;

  // While the planning kernel still runs: set up this warp's barriers and warm
  // the pages the first item's lookup reads.
  if (lane == 0) {
    for (int s = 0; s < P; ++s) mbar_init(smem_addr(&bars[s]), 1);
    fence_mbar_init();
  }
  __syncwarp();
  warm8(a.seg_len, a.n_ids, a.fact_seg_off, a.fact_src, a.seg_start, a.block_table, a.slot_mapping, a.ids);
  // What does not depend on the plan is set up before the wait.  Kernel
  // parameters live in the constant bank: reading the remaining ones here
  // (the chunk pool's fields, the FP8 scales, this lane's rotation turns)
  // keeps their first use after the wait from missing there.
  const int groups = (a.n_layers + G - 1) / G;   // items per token
  const int fbase = STYLE == 0 ? (lane % a.half_vecs) * VE : (lane % a.head_vecs) * (VE / 2);
  asm volatile("" ::"r"(a.chunk_items), "l"(a.work_ctr), "l"(a.work_ctr_next), "f"(a.k_inv), "f"(a.v_inv),
               "r"(a.row_bytes), "r"(a.block_size), "r"(a.num_blocks));
  asm volatile("" ::"f"(rt.hi[fbase]), "f"(rt.lo[fbase]), "f"(rt.hi[fbase + NF - 1]), "f"(rt.lo[fbase + NF - 1]));
  // The block table and the starts are the caller's inputs, not the planning
  // kernel's outputs: bring the rows' first lines, from each request's start
  // on, into this SM's L1 now, so position lookups after the wait hit there.
  if (warp == 0) prefetch_block_rows(a, lane);
  pdl_wait();                                   // outputs of the planning kernel

  const int32_t *s_off, *s_start;
  const int32_t total = segment_prefix(a, off_region, scratch, &s_off, &s_start);

  const int64_t n_items = (int64_t)total * groups;
  const int64_t warp_id = (int64_t)blockIdx.x * nwarps + warp;
  const int64_t n_warps = (int64_t)gridDim.x * nwarps;
  // Each warp first takes a fixed, contiguous share of kStaticPct % of an even
  // split; the rest of the items form a pool handed out in chunks of CH to
  // whichever warp asks first.  Warps on SMs that move data faster (the
  // spread is systematic, about +-15 %) take more of the pool, so the launch
  // ends with the work rather than with its slowest warp.  The pool is dealt
  // round-robin over kPoolCtrs counters (chunk c belongs to counter c %
  // kPoolCtrs) and each warp claims from one of them only, so no single
  // address takes every claim and a finished pool costs each warp one failed
  // claim.  A warp claims its next chunk when its current run is down to its
  // last kClaimAhead items, so the claim's latency hides behind them.  The
  // counters of this launch were zeroed by the previous one; this launch
  // zeroes the other set for the next.  Chunks are at most a quarter of the
  // static share; launches with fewer than kMinShare static items per warp
  // split evenly and use no pool.  So do launches into an FP8 cache: their
  // warps end close together without a pool, and a pool's chunks (a position
  // lookup and a claim each, a new token's angles) measured slower there.
  constexpr int kClaimAhead = 2;
  constexpr int kStaticPct = 50;
  constexpr int kMinShare = 4;
  if (blockIdx.x == 0 && threadIdx.x < kPoolCtrs) a.work_ctr_next[threadIdx.x * kCtrStride] = 0u;
  const int home = (int)(warp_id % kPoolCtrs);
  uint32_t* const home_ctr = a.work_ctr + home * kCtrStride;
  int64_t share = div_nn(n_items * kStaticPct / 100, n_warps);
  if (F8 || share < kMinShare) share = div_nn(n_items + n_warps - 1, n_warps);
  const int64_t CH = min((int64_t)a.chunk_items, max((int64_t)1, share >> 2));
  const int64_t pool0 = min(n_items, share * n_warps);   // first pool item
  const int64_t n_chunks = div_nn(n_items - pool0 + CH - 1, CH);
  int64_t next_claim = 0;                        // lane 0: the pool chunk claimed next
  bool claimed = n_chunks == 0;                  // warp-uniform: next_claim is valid (no pool: never claim)
  if (n_chunks == 0) next_claim = 0;             // c = 0 >= n_chunks ends the stream
  const int64_t j0 = warp_id * share;
  int64_t left = max((int64_t)0, min(share, n_items - j0));   // items left in the current run
  bool stream_done = false;
  int32_t nt = (int32_t)div_nn(j0, groups);      // next item: (segment token, layer group)
  int32_t ng = (int32_t)(j0 - (int64_t)nt * groups);

  const uint32_t stage0 = smem_addr(stages);
  const int vpl = a.row_bytes >> 9;             // 16-byte vectors per lane per row
  const int hv = a.half_vecs;

  TokenCursor cur;

  // Warp-uniform: the next item of this warp's stream into (t, l); false
  // once the stream has ended.
  auto next_item = [&](int32_t& t, int32_t& l) -> bool {
    if (left == 0) {
      if (stream_done) return false;
      if (!claimed && lane == 0) next_claim = (int64_t)atomicAdd(home_ctr, 1u) * kPoolCtrs + home;
      claimed = false;
      const int64_t c = __shfl_sync(0xffffffffu, next_claim, 0);
      if (c >= n_chunks) {
        stream_done = true;
        return false;
      }
      const int64_t j = pool0 + c * CH;
      left = min(CH, n_items - j);
      nt = (int32_t)div_nn(j, groups);
      ng = (int32_t)(j - (int64_t)nt * groups);
    }
    t = nt;
    l = ng * G;
    --left;
    if (left <= kClaimAhead && !claimed) {
      if (lane == 0) next_claim = (int64_t)atomicAdd(home_ctr, 1u) * kPoolCtrs + home;
      claimed = true;
    }
    if (++ng == groups) {
      ng = 0;
      ++nt;
    }
    return true;
  };

  // Warp-uniform: resolve item (t, l)'s token and have lane 0 start its bulk
  // load into stage s.  Returns true if a load was issued.
  auto issue = [&](int s, int32_t t, int32_t l) -> bool {
    const int32_t nlay = min(G, a.n_layers - l);
    cur.seek(a, s_off, s_start, t, lane);
    const int64_t tok_slot = cur.slot;
    const int32_t tok_p = cur.p;
    const int64_t tok_src = cur.src;
    if (lane == 0) {
      if (l == 0 && a.slot_mapping) a.slot_mapping[t] = tok_slot;
      meta[s].slot = tok_slot;
      meta[s].p = tok_p;
      meta[s].l = (int16_t)l;
      meta[s].nl = (int16_t)nlay;
      if (tok_slot >= 0) {
        const uint32_t bar = smem_addr(&bars[s]);
        const uint32_t bytes = 2u * (uint32_t)nlay * (uint32_t)a.row_bytes;
        mbar_expect_tx(bar, bytes);
        bulk_load(stage0 + (uint32_t)s * item_bytes,
                  a.kv + ((size_t)tok_src * a.L + a.layer0 + l) * 2 * (size_t)a.row_bytes, bytes, bar);
      }
    }
    return tok_slot >= 0;
  };

  uint32_t phase = 0;        // expected parity of each stage's next completion
  uint32_t pending = 0;      // stages with a bulk load in flight
  int64_t issued = 0;        // items issued; item i sits in stage i % P
  for (int s = 0; s < P; ++s) {
    int32_t t, l;
    if (!next_item(t, l)) break;
    if (issue(s, t, l)) pending |= 1u << s;
    ++issued;
  }
  __syncwarp();

  float cs[NF], sn[NF], sx[NF];
  int32_t cur_p = -1;
  bool aborted = false;
  int s = 0;
  // NeoX with half a head under 32 vectors: vector v = c * 32 + lane is in the
  // first half of its pair exactly when lane & half_vecs is 0, for every c, so
  // each lane signs its sines once per position and rotates two lanes per
  // instruction.
  const bool paired = STYLE == 0 && (VE % 2) == 0 && hv < 32;
  const bool lane_first = (lane & hv) == 0;
  for (int64_t i = 0; i < issued; ++i) {
    const StageMeta m = meta[s];
    if (m.slot >= 0) {
      const uint32_t bar = smem_addr(&bars[s]);
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar, (phase >> s) & 1u, a.wait_ns));
      if (!ok) {
        if (lane == 0) latch(a.status, IS_ST_TIMEOUT);
        aborted = true;
        break;
      }
      phase ^= 1u << s;
      pending &= ~(1u << s);
      if (m.p != cur_p) {
        cur_p = m.p;
        const float pf = (float)m.p;
#pragma unroll
        for (int e = 0; e < NF; ++e) {
          const float fr = angle_turns(pf, rt.hi[fbase + e], rt.lo[fbase + e]);
          sincospif(2.0f * fr, &sn[e], &cs[e]);
          sx[e] = lane_first ? -sn[e] : sn[e];
        }
      }
      for (int gl = 0; gl < m.nl; ++gl) {
        const uint32_t kst = stage0 + (uint32_t)s * item_bytes + (uint32_t)gl * 2u * (uint32_t)a.row_bytes;
        uint8_t* dk = layer_base(a, m.l + gl) + (size_t)m.slot * a.cache_row_bytes;
        uint8_t* dv = dk + (size_t)a.num_blocks * a.block_size * a.cache_row_bytes;
        if (!F8 && lane == 0) bulk_store(dv, kst + a.row_bytes, a.row_bytes);
        for (int c = 0; c < vpl; ++c) {
          const int v = c * 32 + lane;
          float x[VE], z[VE], y[VE];
          Vec<T>::unpack(ld_shared_v4(kst + v * 16), x);
          if (STYLE == 0) Vec<T>::unpack(ld_shared_v4(kst + (v ^ hv) * 16), z);
          if (paired)
            rotate_neox_x2<VE>(x, z, cs, sx, y);
          else
            rotate_vec<T, STYLE>(x, z, (v & hv) == 0, cs, sn, y);
          if (F8) {
            // 8-bit cache: V is converted on the way too (no bulk store).
            float xv[VE];
            Vec<T>::unpack(ld_shared_v4(kst + a.row_bytes + v * 16), xv);
            st_v2(dv + (size_t)v * 8, to_e4m3x8(xv, a.v_inv));
          }
          store_key<T, F8>(dk, v, y, a.k_inv);
        }
      }
    }
    if (lane == 0) bulk_commit();                 // one bulk group per item (maybe empty)
    // Refill the stage of item i - 1 with item i - 1 + P once its V store has
    // finished reading shared memory (all groups but the newest).
    const int sp = s == 0 ? P - 1 : s - 1;
    int32_t t, l;
    if (i > 0 && next_item(t, l)) {
      if (lane == 0) {
        bulk_wait_read<1>();
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (issue(sp, t, l)) pending |= 1u << sp;
      ++issued;
    }
    __syncwarp();
    s = s + 1 == P ? 0 : s + 1;
  }

  if (aborted) {
    // Let loads already in flight land before shared memory goes away.
    for (int q = 0; q < P; ++q)
      if (pending & (1u << q)) {
        const uint32_t bar = smem_addr(&bars[q]);
        __all_sync(0xffffffffu, mbar_wait_bounded(bar, (phase >> q) & 1u, kWaitBudgetNs));
      }
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
  signal_host_done(a);
}

// ---------------------------------------------------------------------------
// The same gather + rotation + scatter for a store kept in host memory mapped
// into the device's address space (InferScale, "Résultats", Scalabilité: the KV store
// offloaded to host DRAM).  The rows come over the CPU-GPU link through
// ordinary 16-byte loads straight into registers: each lane issues the loads
// of up to kHostChunk vectors of the K row and of the V row before using any,
// and dozens of warps per SM keep enough bytes in flight to cover the link's
// latency.  A NeoX partner vector v ^ half_vecs sits in lane lane ^ half_vecs
// (a shuffle) or, when a half head is exactly 32 vectors, in the neighbouring
// register of the same lane.  No waits: nothing here can stall unboundedly.
constexpr int kHostWarps = 8;
constexpr int kHostChunk = 4;

// Plain 16-byte global load: valid for device memory and for mapped host memory.
__device__ __forceinline__ uint4 ld_plain(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

template <typename T, int STYLE, bool F8>
__global__ void __launch_bounds__(kHostWarps * 32) inject_host_kernel(const InjectArgs a,
                                                                      const RopeTurns rt) {
  extern __shared__ __align__(16) int32_t off_region[];   // prefix_ints(R, kHostWarps)
  __shared__ int32_t scratch[33];
  constexpr int VE = Vec<T>::N;
  constexpr int NF = STYLE == 0 ? VE : VE / 2;

  warm8(a.seg_len, a.n_ids, a.fact_seg_off, a.fact_src, a.seg_start, a.block_table, a.slot_mapping, a.ids);
  pdl_wait();                                   // outputs of the planning kernel

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int32_t *s_off, *s_start;
  const int32_t total = segment_prefix(a, off_region, scratch, &s_off, &s_start);
  const int64_t n_items = (int64_t)total * a.n_layers;
  const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t chunk = div_nn(n_items + n_warps - 1, n_warps);
  const int64_t it0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + warp) * chunk;
  const int64_t it_end = min(n_items, it0 + chunk);

  const int vpl = a.row_bytes >> 9;
  const int hv = a.half_vecs;
  const int fbase = STYLE == 0 ? (lane % hv) * VE : (lane % a.head_vecs) * (VE / 2);
  static_assert(!F8 || VE == 8, "an FP8 cache takes 16-bit store rows");
  const size_t plane = (size_t)a.num_blocks * a.block_size * a.cache_row_bytes;
  TokenCursor cur;
  float cs[NF], sn[NF];
  int32_t cur_p = -1;
  int32_t t = (int32_t)div_nn(it0, a.n_layers);
  int32_t l = (int32_t)(it0 - (int64_t)t * a.n_layers) - 1;
  for (int64_t i = it0; i < it_end; ++i) {
    if (++l == a.n_layers) {
      l = 0;
      ++t;
    }
    cur.seek(a, s_off, s_start, t, lane);
    if (l == 0 && lane == 0 && a.slot_mapping) a.slot_mapping[t] = cur.slot;
    if (cur.slot < 0) continue;
    if (cur.p != cur_p) {
      cur_p = cur.p;
      const float pf = (float)cur_p;
#pragma unroll
      for (int e = 0; e < NF; ++e) {
        const float fr = angle_turns(pf, rt.hi[fbase + e], rt.lo[fbase + e]);
        sincospif(2.0f * fr, &sn[e], &cs[e]);
      }
    }
    const uint8_t* src = a.kv + ((size_t)cur.src * a.L + a.layer0 + l) * 2 * (size_t)a.row_bytes;
    uint8_t* dk = layer_base(a, l) + (size_t)cur.slot * a.cache_row_bytes;
    uint8_t* dv = dk + plane;
    for (int c0 = 0; c0 < vpl; c0 += kHostChunk) {
      uint4 kx[kHostChunk], vx[kHostChunk];
#pragma unroll
      for (int c = 0; c < kHostChunk; ++c)
        if (c0 + c < vpl) {
          const size_t o = (size_t)((c0 + c) * 32 + lane) * 16;
          kx[c] = ld_plain(src + o);
          vx[c] = ld_plain(src + a.row_bytes + o);
        }
#pragma unroll
      for (int c = 0; c < kHostChunk; ++c)
        if (c0 + c < vpl) {                     // warp-uniform
          const int v = (c0 + c) * 32 + lane;
          if (F8) {
            float xv[VE];
            Vec<T>::unpack(vx[c], xv);
            st_v2(dv + (size_t)v * 8, to_e4m3x8(xv, a.v_inv));
          } else {
            st_v4(dv + (size_t)v * 16, vx[c]);
          }
          float x[VE], z[VE], y[VE];
          Vec<T>::unpack(kx[c], x);
          if (STYLE == 0) Vec<T>::unpack(hv < 32 ? shfl_xor4(kx[c], hv) : kx[c ^ 1], z);
          rotate_vec<T, STYLE>(x, z, (v & hv) == 0, cs, sn, y);
          store_key<T, F8>(dk, v, y, a.k_inv);
        }
    }
  }
  signal_host_done(a);
}

// ---------------------------------------------------------------------------

cudaError_t launch_plan(const PlanArgs& a, const LaunchCfg& cfg) {
  return launch_ex(plan_kernel, dim3(a.R), dim3(256), 0, cfg.stream, cfg.pdl, a);
}

// Shared memory plan of one inject launch: warps per CTA, stages per warp and
// layers per work item.
struct InjectShape {
  int warps;
  int stages;
  size_t smem;
  int layers_per_item;
};

// Layers per work item: as many as keep one bulk copy within about 4 KiB.
static int layers_per_item(const InjectArgs& a) {
  int g = 1;
  while (g < 8 && 2 * g < std::max(1, a.n_layers) + 1 && 2 * (size_t)(2 * g) * a.row_bytes <= 4096) g *= 2;
  return g;
}

static InjectShape inject_shape(const InjectArgs& a) {
  const int G = layers_per_item(a);
  const size_t item = 2 * (size_t)G * a.row_bytes;
  const size_t off_bytes = ((size_t)prefix_ints(a.R, kInjectWarpsMax) * 4 + 127) & ~(size_t)127;
  const size_t per_stage = item + 8 + sizeof(StageMeta);
  // Two CTAs per SM: the stages get what the request table leaves of ~110 KiB.
  const size_t stage_budget = std::max<size_t>(16 * 1024, std::min<size_t>(96 * 1024, 110 * 1024 - off_bytes));
  const size_t smem_max = 227 * 1024 - 1024;
  for (int w = kInjectWarpsMax; w >= 1; w >>= 1) {
    int p = (int)std::min<size_t>(16, std::max<size_t>(2, stage_budget / (w * item)));
    size_t need = off_bytes + (size_t)w * p * per_stage;
    while (p > 2 && need > smem_max) {
      --p;
      need = off_bytes + (size_t)w * p * per_stage;
    }
    if (need <= smem_max) return {w, p, need, G};
  }
  return {0, 0, 0, 0};
}

// Per device and kernel instance: the dynamic shared memory limit already set
// and the occupancy of the last shape queried.
struct LaunchMemo {
  size_t smem_set = 0;
  size_t occ_smem = 0;
  int occ_warps = 0;
  int occ_blocks = 0;
};
static std::mutex g_launch_mu;

template <typename T, int STYLE, bool F8, bool HOST>
static LaunchMemo& launch_memo(int dev) {
  static LaunchMemo memo[64];
  return memo[dev & 63];
}

// Items per pool chunk: about 32 KiB of K/V.
constexpr size_t kChunkBytes = 32 * 1024;

template <typename T, int STYLE, bool F8>
static cudaError_t launch_inject_t(const InjectArgs& args, const RopeTurns& rt, const LaunchCfg& cfg) {
  const InjectShape sh = inject_shape(args);
  if (sh.warps == 0 || !args.work_ctr || !args.work_ctr_next) return cudaErrorInvalidValue;
  InjectArgs a = args;
  a.chunk_items = (int32_t)std::max<size_t>(1, kChunkBytes / (2 * (size_t)sh.layers_per_item * a.row_bytes));
  auto kern = inject_kernel<T, STYLE, F8>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    LaunchMemo& m = launch_memo<T, STYLE, F8, false>(dev);
    if (sh.smem > m.smem_set) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sh.smem);
      if (e != cudaSuccess) return e;
      m.smem_set = sh.smem;
    }
    if (m.occ_smem != sh.smem || m.occ_warps != sh.warps) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&m.occ_blocks, kern, sh.warps * 32, sh.smem);
      if (e != cudaSuccess) return e;
      m.occ_smem = sh.smem;
      m.occ_warps = sh.warps;
    }
    per_sm = m.occ_blocks;
  }
  return launch_ex(kern, dim3(cfg.num_sms * std::max(1, per_sm)), dim3(sh.warps * 32), sh.smem,
                   cfg.stream, cfg.pdl, a, rt, sh.stages, sh.layers_per_item);
}

template <typename T, int STYLE, bool F8>
static cudaError_t launch_inject_host_t(const InjectArgs& a, const RopeTurns& rt, const LaunchCfg& cfg) {
  auto kern = inject_host_kernel<T, STYLE, F8>;
  const size_t smem = (size_t)prefix_ints(a.R, kHostWarps) * 4;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    LaunchMemo& m = launch_memo<T, STYLE, F8, true>(dev);
    if (m.occ_smem != smem || m.occ_warps != kHostWarps) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&m.occ_blocks, kern, kHostWarps * 32, smem);
      if (e != cudaSuccess) return e;
      m.occ_smem = smem;
      m.occ_warps = kHostWarps;
    }
    per_sm = m.occ_blocks;
  }
  return launch_ex(kern, dim3(cfg.num_sms * std::max(1, per_sm)), dim3(kHostWarps * 32), smem,
                   cfg.stream, cfg.pdl, a, rt);
}

template <typename T, int STYLE, bool F8>
static cudaError_t launch_inject_any(const InjectArgs& a, const RopeTurns& rt, bool host_src,
                                     const LaunchCfg& cfg) {
  return host_src ? launch_inject_host_t<T, STYLE, F8>(a, rt, cfg)
                  : launch_inject_t<T, STYLE, F8>(a, rt, cfg);
}

template <typename T>
static cudaError_t launch_inject_styled(const InjectArgs& a, const RopeTurns& rt, int style, bool host_src,
                                        bool fp8_cache, const LaunchCfg& cfg) {
  if (fp8_cache) {
    if constexpr (Vec<T>::N == 8)
      return style == 0 ? launch_inject_any<T, 0, true>(a, rt, host_src, cfg)
                        : launch_inject_any<T, 1, true>(a, rt, host_src, cfg);
    return cudaErrorInvalidValue;               // an FP8 cache takes 16-bit store rows
  }
  return style == 0 ? launch_inject_any<T, 0, false>(a, rt, host_src, cfg)
                    : launch_inject_any<T, 1, false>(a, rt, host_src, cfg);
}

cudaError_t launch_inject(const InjectArgs& a, const RopeTurns& rt, int kv_dtype, int style,
                          bool host_src, bool fp8_cache, const LaunchCfg& cfg) {
  if (kv_dtype == IS_BF16) return launch_inject_styled<__nv_bfloat16>(a, rt, style, host_src, fp8_cache, cfg);
  if (kv_dtype == IS_F16) return launch_inject_styled<__half>(a, rt, style, host_src, fp8_cache, cfg);
  return launch_inject_styled<float>(a, rt, style, host_src, fp8_cache, cfg);
}

bool inject_shape_ok(int row_bytes, int R) {
  InjectArgs a{};
  a.row_bytes = row_bytes;
  a.R = R;
  return inject_shape(a).warps > 0;
}

}  // namespace isk

// ---------------------------------------------------------------------------
// Allocation-free injection (is_inject_noalloc).
//
// For callers that cannot allocate device memory, the segment plan that
// is_inject keeps in store-owned scratch lives here in one file-scope device
// array of fixed size.  The host never dereferences the array's name: it
// looks up the device address once per device and passes that to the kernels.

namespace {

constexpr int kNaRequests = IS_NOALLOC_MAX_REQUESTS;
constexpr int kNaSegStride = IS_NOALLOC_MAX_FACTS + 1;
constexpr size_t kNaCtrOff = ((size_t)kNaRequests * kNaSegStride + 2 * kNaRequests + 31) & ~(size_t)31;
constexpr size_t kNaWords = kNaCtrOff + 2 * isk::kPoolCtrWords;
constexpr int kNaMaxDevices = 64;

// [0, R*stride): per-request prefix of fact lengths; then n_ids[R]; then
// seg_len[R]; then, from a 128-byte boundary, two sets of the inject kernel's
// chunk counters.  Every call's planning kernel zeroes the first set, which
// that call's inject kernel then claims from; the inject kernel zeroes the
// second set as it would for a following launch, and nothing reads it.  So
// a call depends on no state a previous call left, on the host or the device.
static __device__ __align__(256) int32_t g_noalloc_scratch[kNaWords];

struct NoAllocDevice {
  bool ready = false;
  int32_t* scratch = nullptr;   // device address of g_noalloc_scratch on this device
  int num_sms = 0;
};
NoAllocDevice g_na_dev[kNaMaxDevices];
std::mutex g_na_mu;

is_status_t na_fail(is_status_t st, const char* msg) {
  isk::set_last_error_message(msg);
  if (st == IS_ERR_CUDA) cudaGetLastError();   // a failed launch is reported here, not by a later call
  return st;
}

}  // namespace

extern "C" is_status_t is_inject_noalloc(
    const void* kv_arena, int64_t arena_tokens, const int64_t* fact_tok, const int32_t* fact_len, int64_t n_facts,
    int32_t max_fact_len, int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
    int32_t kv_dtype, int32_t R, const int64_t* fact_ids, const int32_t* n_ids, int32_t ids_stride,
    const int32_t* seg_start, const is_rope_params_t* rope, const int32_t* block_table,
    int32_t max_blocks_per_seq, const is_cache_desc_t* cache, void* kv_cache, int32_t* seg_len_out,
    int64_t* slot_mapping_out, uint32_t* status_out, cudaStream_t stream) {
  using namespace isk;
  if (!kv_arena || !fact_tok || !fact_len || !fact_ids || !n_ids || !seg_start || !rope ||
      !block_table || !cache || !kv_cache || !status_out)
    return na_fail(IS_ERR_INVALID_ARG, "a required pointer is NULL");
  if (R < 1 || R > kNaRequests)
    return na_fail(IS_ERR_UNSUPPORTED, "R must be in [1, IS_NOALLOC_MAX_REQUESTS]");
  if (ids_stride < 1 || ids_stride > IS_NOALLOC_MAX_FACTS)
    return na_fail(IS_ERR_UNSUPPORTED, "ids_stride must be in [1, IS_NOALLOC_MAX_FACTS]");
  if (n_facts < 1 || max_fact_len < 1 || max_blocks_per_seq < 1 || arena_tokens < 1)
    return na_fail(IS_ERR_INVALID_ARG,
                   "arena_tokens, n_facts, max_fact_len, max_blocks_per_seq must be >= 1");
  if ((int64_t)R * ids_stride * max_fact_len >= (int64_t)INT32_MAX)
    return na_fail(IS_ERR_UNSUPPORTED, "R * ids_stride * max_fact_len must stay below 2^31");
  if (kv_dtype != IS_F32 && kv_dtype != IS_BF16 && kv_dtype != IS_F16)
    return na_fail(IS_ERR_INVALID_ARG, "bad kv_dtype");
  if (num_layers < 1 || num_kv_heads < 1 || head_dim < 16 || head_dim > IS_MAX_HEAD_DIM ||
      (head_dim & (head_dim - 1)) != 0)
    return na_fail(IS_ERR_UNSUPPORTED, "head_dim must be a power of two in [16, IS_MAX_HEAD_DIM]");
  const int elt = kv_dtype == IS_F32 ? 4 : 2;
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * elt;
  if (row_bytes % 512 != 0 || !inject_shape_ok((int)row_bytes, R))
    return na_fail(IS_ERR_UNSUPPORTED,
                   "num_kv_heads * head_dim * elt must be a multiple of 512 and at most 32 KiB");
  if (cache->block_size < 1 || cache->num_blocks < 1 || cache->dtype != kv_dtype)
    return na_fail(IS_ERR_INVALID_ARG, "bad cache descriptor");
  if ((((uintptr_t)kv_cache) | ((uintptr_t)kv_arena)) & 15)
    return na_fail(IS_ERR_INVALID_ARG, "kv_cache and kv_arena must be 16-byte aligned");
  double w[kMaxHalfDim];
  if (is_rope_frequencies(rope, head_dim, w) != IS_OK)
    return na_fail(IS_ERR_INVALID_ARG, "bad rope parameters");
  const int ve = 16 / elt;
  const int vecs = rope->style == 0 ? head_dim / 2 / ve : head_dim / ve;
  if (vecs < 1 || vecs > 32)
    return na_fail(IS_ERR_UNSUPPORTED, "head_dim not supported for this dtype and rope style");

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices)
    return na_fail(IS_ERR_CUDA, "cudaGetDevice failed");
  NoAllocDevice& d = g_na_dev[dev];
  {
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (!d.ready) {
      void* ptr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return na_fail(IS_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
      }
      if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return na_fail(IS_ERR_CUDA, "cudaDeviceGetAttribute failed");
      d.scratch = static_cast<int32_t*>(ptr);
      d.ready = true;
    }
  }
  int32_t* seg_off = d.scratch;
  int32_t* na_n_ids = d.scratch + (size_t)kNaRequests * kNaSegStride;
  int32_t* seg_len = seg_len_out ? seg_len_out : na_n_ids + kNaRequests;

  PlanArgs p{};
  p.ids = fact_ids;
  p.ids_stride = ids_stride;
  p.n_ids_in = n_ids;
  p.users = nullptr;
  p.seg_start = seg_start;
  p.fact_len = fact_len;
  p.fact_user = nullptr;
  p.fact_tok = fact_tok;
  p.n_facts = n_facts;
  p.fact_src = nullptr;
  p.block_table = block_table;
  p.max_blocks = max_blocks_per_seq;
  p.n_ids_out = na_n_ids;
  p.fact_seg_off = seg_off;
  p.seg_stride = kNaSegStride;
  p.seg_len = seg_len;
  p.status = status_out;
  p.R = R;
  p.arena_tokens = arena_tokens;
  p.max_fact_len = max_fact_len;
  uint32_t* ctr = reinterpret_cast<uint32_t*>(d.scratch + kNaCtrOff);
  p.zero_ctr = ctr;
  const LaunchCfg cfg{stream, d.num_sms, false};
  if (launch_plan(p, cfg) != cudaSuccess) return na_fail(IS_ERR_CUDA, "plan launch failed");

  InjectArgs a{};
  a.kv = static_cast<const uint8_t*>(kv_arena);
  a.fact_tok = fact_tok;
  a.fact_len = fact_len;
  a.fact_user = nullptr;
  a.n_facts = n_facts;
  a.ids = fact_ids;
  a.ids_stride = ids_stride;
  a.fact_src = nullptr;
  a.n_ids = na_n_ids;
  a.fact_seg_off = seg_off;
  a.seg_stride = kNaSegStride;
  a.seg_len = seg_len;
  a.seg_start = seg_start;
  a.block_table = block_table;
  a.max_blocks = max_blocks_per_seq;
  a.cache = static_cast<uint8_t*>(kv_cache);
  a.block_size = cache->block_size;
  a.num_blocks = cache->num_blocks;
  a.slot_mapping = slot_mapping_out;
  a.status = status_out;
  a.R = R;
  a.L = num_layers;
  a.layer0 = 0;
  a.n_layers = num_layers;
  a.layer_stride = 2LL * cache->num_blocks * cache->block_size * row_bytes;
  a.row_bytes = (int32_t)row_bytes;
  a.cache_row_bytes = (int32_t)row_bytes;
  a.wait_ns = kWaitBudgetNs;
  a.work_ctr = ctr;                              // zeroed by this call's plan kernel
  a.work_ctr_next = ctr + isk::kPoolCtrWords;     // zeroed by the inject kernel, unused
  a.half_vecs = head_dim / 2 / ve;
  a.head_vecs = head_dim / ve;
  RopeTurns rt;
  memset(&rt, 0, sizeof rt);
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < head_dim / 2; ++i) {
    const double turns = w[i] / two_pi;
    rt.hi[i] = (float)turns;
    rt.lo[i] = (float)(turns - (double)rt.hi[i]);
  }
  const LaunchCfg cfg_dep{stream, d.num_sms, true};
  if (launch_inject(a, rt, kv_dtype, rope->style, false, false, cfg_dep) != cudaSuccess)
    return na_fail(IS_ERR_CUDA, "inject launch failed");
  return IS_OK;
}
