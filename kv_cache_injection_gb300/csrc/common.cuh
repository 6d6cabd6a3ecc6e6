// Device helpers and launch-parameter structs shared by the kernels of
// libinjectscale.so (GB300, sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "injectscale.h"

namespace isk {

constexpr int kMaxHalfDim = IS_MAX_HEAD_DIM / 2;
constexpr int kTile = IS_EMB_TILE;

// Rotation frequencies as turns per position (w_i / 2 pi), each split into
// two floats hi + lo so that the angle reduction runs in fp32 (see
// angle_turns).  Passed by value as a kernel parameter (2 KiB).
struct RopeTurns {
  float hi[kMaxHalfDim];
  float lo[kMaxHalfDim];
};

// Everything the gather + Chunked RoPE + paged scatter kernel reads.
struct InjectArgs {
  const uint8_t* kv;            // store arena [max_tokens][L][2][H][D]
  const int64_t* fact_tok;      // first arena token of each fact
  const int32_t* fact_len;
  const int32_t* fact_user;
  int64_t n_facts;
  const int64_t* ids;           // [R][ids_stride]
  int32_t ids_stride;
  const int64_t* fact_src;      // [R][seg_stride] arena token of each planned fact, or null
  const int32_t* n_ids;         // [R] facts per request (after planning)
  const int32_t* fact_seg_off;  // [R][seg_stride]: exclusive prefix of fact lengths
  int32_t seg_stride;
  const int32_t* seg_len;       // [R]
  const int32_t* seg_start;     // [R]
  const int32_t* block_table;   // [R][max_blocks]
  int32_t max_blocks;
  uint8_t* cache;               // [L][2][num_blocks][bs][H][D]
  int32_t block_size;
  int32_t num_blocks;
  int64_t* slot_mapping;        // [sum seg_len] or null
  uint32_t* status;
  int32_t R;
  int32_t L;                    // layers of the store
  int32_t layer0;               // first layer this call injects
  int32_t n_layers;             // layers this call injects
  int64_t layer_stride;         // bytes between consecutive layers of the destination cache
  int32_t row_bytes;            // H * D * elt of the store
  int32_t half_vecs;            // NeoX: 16-byte vectors per half head (D / 2 / VE)
  int32_t head_vecs;            // 16-byte vectors per head (D / VE)
  int32_t cache_row_bytes;      // H * D * elt of the cache (row_bytes, or H * D for FP8)
  float k_inv, v_inv;           // FP8 cache: fp32(1 / k_scale), fp32(1 / v_scale)
  uint64_t wait_ns;             // budget of each pipeline wait (the drain of copies in flight keeps 2 s)
  uint32_t* work_ctr;           // kPoolCtrs counters of pool claims in this launch (zero at its start)
  uint32_t* work_ctr_next;      // the counters of the next launch, zeroed by this one
  int32_t chunk_items;          // items per pool chunk (set by the launcher)
  uint32_t* done_ctr;           // CTAs of this launch that have finished (zero between launches)
  uint32_t* host_done;          // mapped host word the last CTA sets to done_seq, or null
  uint32_t done_seq;
  int32_t per_layer;            // 1: layer l of this call is written to layer_cache[l]
  uint8_t* layer_cache[IS_MAX_LAYERS_PER_CALL];   // per_layer: each layer's own [2][nb][bs][H][D]
};

// One layer of a Context-Window Encoding capture (is_store_capture_layer).
struct CaptureArgs {
  const uint8_t* k;             // engine layer output [src tokens][H][D], keys before RoPE
  const uint8_t* v;             // [src tokens][H][D]
  uint8_t* kv;                  // store arena [max_tokens][L][2][H][D]
  const int64_t* seg;           // [n][2]: first source token of the fact's tokens, first arena token
  int32_t n;                    // facts
  int64_t tok0;                 // arena token of the first fact's first token
  int64_t tokens;               // fact tokens (contiguous in the arena from tok0)
  int32_t L;
  int32_t layer;
  int32_t row_bytes;            // H * D * elt
};

// Segment planning for an explicit fact list (is_inject).
struct PlanArgs {
  const int64_t* ids;
  int32_t ids_stride;
  const int32_t* n_ids_in;      // caller's counts [R]
  const int32_t* users;         // [R] or null
  const int32_t* seg_start;
  const int32_t* fact_len;
  const int32_t* fact_user;
  const int64_t* fact_tok;
  int64_t n_facts;
  int32_t* n_ids_out;           // [R]
  int32_t* fact_seg_off;        // [R][seg_stride]
  int64_t* fact_src;            // [R][seg_stride] arena token of each planned fact, or null
  const int32_t* block_table;   // [R][max_blocks] (prefetched into L2)
  int32_t max_blocks;
  int32_t seg_stride;
  int32_t* seg_len;             // [R]
  uint32_t* status;
  int32_t R;
  // Caller-owned fact tables (is_inject_noalloc) are checked here, since no
  // store checked them when the facts were added: with arena_tokens > 0 a
  // fact whose length lies outside [1, max_fact_len] or whose tokens leave
  // [0, arena_tokens) latches IS_ST_FACT_RANGE and counts as length 0.
  int64_t arena_tokens;
  int32_t max_fact_len;
  // If set, CTA 0 zeroes these kPoolCtrs chunk counters (kCtrStride words
  // apart) for the inject launch that follows this plan in the stream.
  uint32_t* zero_ctr;
};

// The inject kernel's pool of work chunks is claimed through kPoolCtrs
// counters, kCtrStride words (one 128-byte line) apart; a launch uses one set
// of kPoolCtrWords words and zeroes the other for the next launch.
constexpr int kPoolCtrs = 16;
constexpr int kCtrStride = 32;
constexpr int kPoolCtrWords = kPoolCtrs * kCtrStride;
// The store's counter block: two sets of pool counters, then the inject
// kernel's CTA arrival counter of host-buffer calls on a line of its own.
constexpr int kDoneCtrWord = 2 * kPoolCtrWords;
constexpr int kCtrBlockWords = kDoneCtrWord + kCtrStride;

// Uniform bins of the cosine in [-1, 1] used by the top-k's first pass.
constexpr int kCosBins = 2048;

struct SimArgs {
  const void* emb;              // tiles [n_tiles * kTile][E]
  const float* emb_inv_norm;    // [n_tiles * kTile]
  const int4* user_meta;        // [max_users] {tile list offset, tiles, facts, first tile or -1}
  const int32_t* user_tiles;    // tiles of each user, in fill order
  const int32_t* users;         // [Q]
  const void* q_emb;            // [Q][E]
  float* scores;                // [Q][score_stride]
  int64_t score_stride;
  uint32_t* status;
  int32_t Q;
  int32_t E;
  int32_t max_users;
};

struct TopkArgs {
  const float* scores;
  int64_t score_stride;
  const int32_t* users;
  const int4* user_meta;
  const int32_t* user_tiles;
  const int32_t* tile_fact;     // [n_tiles * kTile] fact id per embedding row
  const int32_t* tile_len;      // [n_tiles * kTile] length of that fact
  const int64_t* tile_tok;      // [n_tiles * kTile] arena token of that fact
  const int64_t* fact_tok;
  const int32_t* fact_len;
  const int32_t* seg_start;     // [Q] or null (retrieval only)
  int64_t* ids_out;             // [Q][k]
  float* scores_out;            // [Q][k]
  int32_t* n_ids_out;           // [Q] or null
  int32_t* fact_seg_off;        // [Q][seg_stride] or null
  int64_t* fact_src;            // [Q][seg_stride] or null
  int32_t seg_stride;
  int32_t* seg_len;             // [Q] or null
  int32_t* seg_len_copy;        // [Q] or null: a second destination of seg_len (may be mapped host memory)
  const int32_t* block_table;   // [Q][max_blocks] or null (prefetched into L2)
  int32_t max_blocks;
  uint32_t* hist;               // [Q][kCosBins] cosine-bin counts filled by the similarity CTAs, or null
  uint32_t* status;
  int32_t Q;
  int32_t k;
  int32_t max_users;
};

// Grouping of a retrieval call's queries by user (batched path).
struct GroupArgs {
  const int32_t* users;         // [Q]
  const void* q_emb;            // [Q][E] fp16
  int32_t Q;
  int32_t E;
  const int4* user_meta;
  int32_t max_users;
  __half* qg;                   // [max_queries][E] queries in group order
  float* q_inv;                 // [max_queries] their inverse norms
  int32_t* qperm;               // packed position -> caller's query index
  int4* groups;                 // [max_queries] {user, first position, count, first work item}
  int32_t* counts;              // {groups, work items}
  uint32_t* status;
};

// The tensor-core contraction of the batched path.
struct GemmArgs {
  const int4* groups;
  const int32_t* counts;
  const int32_t* qperm;
  const float* q_inv;
  const int4* user_meta;
  const int32_t* user_tiles;
  const float* emb_inv_norm;
  float* scores;                // [Q][score_stride], indexed by the caller's query
  int64_t score_stride;
  int32_t E;
  uint32_t* status;
  uint64_t wait_ns;             // budget of each pipeline wait (drains keep 2 s)
};

// ------------------------------------------------------------------ device helpers

__device__ __forceinline__ void latch(uint32_t* status, uint32_t bits) { atomicOr(status, bits); }

// Atomic add with acquire-release semantics at GPU scope: the caller's earlier
// writes (and those of its CTA, ordered before by a barrier) are visible to
// whoever observes the new value, and the caller's later reads see what the
// earlier arrivals released.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16-byte streaming load of data that is read once: no L1 allocation,
// evict-first in L2 so it does not push out cache lines attention will read.
__device__ __forceinline__ uint4 ld_once(const void* ptr, uint64_t policy) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(ptr), "l"(policy));
  return r;
}

__device__ __forceinline__ void st_v4(void* ptr, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_v2(void* ptr, const uint2& v) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(ptr), "r"(v.x), "r"(v.y) : "memory");
}

// Eight fp32 values times r into eight FP8 E4M3 bytes (one 8-byte word,
// element 0 in the lowest byte): one fp32 multiply each, then the hardware
// conversion, which rounds to nearest even and saturates to +-448.  With
// r == 1 (the usual unit scale) the multiplies are exact no-ops and skipped.
// Two fp32 values in one 64-bit register, and the Blackwell paired-lane
// multiply and fused multiply-add on them: each lane is rounded to nearest
// exactly as its scalar form (__fmul_rn, fmaf), in one instruction for both.
__device__ __forceinline__ unsigned long long pk2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long mul2_rn(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long fma2_rn(unsigned long long a, unsigned long long b,
                                                      unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint2 to_e4m3x8(const float* x, float r) {
  uint32_t w[4];
  if (r == 1.0f) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = __nv_cvt_float2_to_fp8x2(make_float2(x[2 * e], x[2 * e + 1]), __NV_SATFINITE, __NV_E4M3);
  } else {
    const unsigned long long rr = pk2(r, r);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float a, b;
      upk2(mul2_rn(pk2(x[2 * e], x[2 * e + 1]), rr), a, b);
      w[e] = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    }
  }
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Thread i < 8 prefetches the first line of p_i into L2 (null pointers are
// skipped).  Used at a kernel's start on arrays a later, dependent step will
// read or write: the prefetch fills the address translation and L2 off that
// step's critical path.
__device__ __forceinline__ void warm8(const void* p0, const void* p1, const void* p2, const void* p3,
                                      const void* p4, const void* p5, const void* p6, const void* p7) {
  const int i = threadIdx.x;
  const void* p = i == 0 ? p0 : i == 1 ? p1 : i == 2 ? p2 : i == 3 ? p3
                : i == 4 ? p4 : i == 5 ? p5 : i == 6 ? p6 : i == 7 ? p7 : nullptr;
  if (p) prefetch_l2(p);
}

// Prefetch n int32 entries (one 128-byte line per thread) into L2.
__device__ __forceinline__ void prefetch_row_l2(const int32_t* p, int n, int tid, int nthreads) {
  for (int i = tid * 32; i < n; i += nthreads * 32) prefetch_l2(p + i);
}

// Tile ti of a user: consecutive tiles need no list lookup.
__device__ __forceinline__ int user_tile(const int32_t* user_tiles, const int4& um, int ti) {
  return um.w >= 0 ? um.w + ti : user_tiles[um.x + ti];
}

__device__ __forceinline__ uint4 shfl_xor4(const uint4& v, int mask) {
  uint4 r;
  r.x = __shfl_xor_sync(0xffffffffu, v.x, mask);
  r.y = __shfl_xor_sync(0xffffffffu, v.y, mask);
  r.z = __shfl_xor_sync(0xffffffffu, v.z, mask);
  r.w = __shfl_xor_sync(0xffffffffu, v.w, mask);
  return r;
}

// ---- programmatic dependent launch ------------------------------------------------
// A kernel launched with programmatic stream serialisation may start while the
// previous kernel in the stream still runs; it must call pdl_wait() before
// reading that kernel's outputs.  pdl_trigger() lets the next kernel launch
// once every CTA of this one has been scheduled.
__device__ __forceinline__ void pdl_wait() {
#if defined(__CUDA_ARCH__)
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
__device__ __forceinline__ void pdl_trigger() {
#if defined(__CUDA_ARCH__)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// ---- shared memory, mbarrier and bulk-copy (TMA engine) primitives -------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Default and largest budget of a bounded wait; waits that drain copies
// already in flight before a kernel exits always use it.
constexpr uint64_t kWaitBudgetNs = 2000000000ull;   // 2 s

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for an mbarrier phase: gives up after `budget_ns` of wall time
// (or 2^26 polls) and returns false.  A zero budget looks once, without
// waiting.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t budget_ns) {
  if (budget_ns == 0) return mbar_test_wait(bar, parity);
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 26); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u && global_timer_ns() - t0 > budget_ns) return false;
  }
  return false;
}

// Bulk copy global -> shared, completion counted on an mbarrier (bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bulk copy shared -> global in the calling thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Element access on a 16-byte vector of T.
template <typename T> struct Vec;

template <> struct Vec<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // round to nearest even
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
  }
};

template <> struct Vec<__half> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static uint4 pack(const float* f) {
    return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
  }
};

// Fraction of a turn, in [-1/2, 1/2], of the angle p * w_i = 2 pi p t_i, with
// t_i = hi + lo.  p * hi is split exactly into a rounded product and its
// error term (Dekker's product through a fused multiply-add); the integer part
// of the rounded product is removed exactly, so the result keeps fp32
// precision relative to 1/2 whatever the size of p (p < 2^24).
__device__ __forceinline__ float angle_turns(float p, float hi, float lo) {
  const float prod = p * hi;
  const float err = fmaf(p, hi, -prod);
  const float frac = prod - rintf(prod);
  return frac + fmaf(p, lo, err);
}

// Order-preserving map of fp32 scores onto uint32 keys (larger score, larger key).
__device__ __forceinline__ uint32_t score_key(float s) {
  const uint32_t b = __float_as_uint(s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

}  // namespace isk
