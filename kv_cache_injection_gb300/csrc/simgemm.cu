// Batched retrieval on the 5th-generation tensor cores.
//
// When many queries in one call ask the same user's store, the cosine scores
// are a dense contraction: S = Q_u x E_u^T over the embedding dimension.  The
// queries are grouped by user (up to 64 per group) and packed; each work item
// (group, 128-row embedding tile) is one M=128 x N=64 tile computed by
// tcgen05.mma (kind::f16, fp32 accumulation in tensor memory) from operands
// that TMA brings into shared memory in 128-byte-swizzled K-major chunks of
// 64 elements.  One thread feeds TMA, one issues the MMAs, and all four warps
// read the accumulator back (tcgen05.ld) and scale it by the two inverse norms.
// The per-query top-k then runs one CTA per query.  InferScale retrieves from
// a GPU-resident index ("Conception de Système Native au GPU"); the contraction
// is exact up to fp32 accumulation of fp16 products.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "block_scan.cuh"
#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace isk {

constexpr int kGroupN = 64;                         // queries per group = MMA N
constexpr int kChunkK = 64;                         // fp16 per K chunk = one 128-byte swizzle row
constexpr int kGemmStages = 4;
constexpr uint32_t kATile = 128 * kChunkK * 2;      // 16 KiB
constexpr uint32_t kBTile = kGroupN * kChunkK * 2;  // 8 KiB
constexpr uint32_t kStageBytes = kATile + kBTile;
constexpr uint32_t kTmemCols = 64;
// kind::f16 instruction descriptor: D fp32 (bits 4-5 = 1), A and B fp16
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kGroupN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);

// ---- tcgen05 / TMA primitives -------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row atoms of 1024 bytes
// (stride byte offset), descriptor version 1, layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Bounded mbarrier wait (budget_ns; zero looks once) that also gives up when
// another thread of the CTA has flagged an abort.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              uint64_t budget_ns) {
  if (budget_ns == 0) return mbar_test_wait(bar, parity);
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 26); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u && (*abort_flag || global_timer_ns() - t0 > budget_ns)) return false;
  }
  return false;
}

// ---- query grouping -------------------------------------------------------------

// The call's queries in (user, query index) order, cut into groups of at most
// kGroupN queries of one user, with the (group, tile) work items numbered.
// Grid of ceil(Q / 32) CTAs of 1024 threads, one warp per query: every CTA
// stages the validated user of each of the Q queries in shared memory, and a
// warp finds its query's position in that order by counting the queries that
// precede it (a rank, no sort), then packs the query's fp16 row there and
// computes its inverse norm.  CTA 0 also places each query's user at its
// position and, one thread per position, finds where each user's run starts
// and ends and writes the group table.  The row copies of all warps and the
// user records of all group starts are loaded in parallel, so the grouping
// costs a few load latencies, not a pass over the rows.
constexpr int kGroupThreads = 1024;
constexpr int kGroupWarps = kGroupThreads / 32;
static_assert(kGroupThreads >= IS_MAX_QUERIES, "CTA 0 takes one thread per query position");

__global__ void __launch_bounds__(kGroupThreads) group_kernel(const GroupArgs a) {
  __shared__ uint32_t s_user[IS_MAX_QUERIES];      // validated user of query i; 0xFFFFFFFF = unknown
  __shared__ uint32_t s_sorted[IS_MAX_QUERIES];    // CTA 0: user at each position of the order
  __shared__ int32_t scratch[33];
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Q = a.Q;
  const int q = blockIdx.x * kGroupWarps + warp;
  // The query row does not depend on the order: start pulling it now.
  const __half* src_row = reinterpret_cast<const __half*>(a.q_emb) + (size_t)(q < Q ? q : 0) * a.E;
  if (q < Q && lane * 64 < a.E * 2) prefetch_l2(reinterpret_cast<const uint8_t*>(src_row) + lane * 64);
  for (int i = tid; i < Q; i += kGroupThreads) {
    const int32_t uu = a.users[i];
    const bool ok = uu >= 0 && uu < a.max_users;
    if (ok) {
      if (blockIdx.x == 0) prefetch_l2(a.user_meta + uu);   // CTA 0 reads it after the order
    } else if (blockIdx.x == 0) {
      latch(a.status, IS_ST_USER_RANGE);
    }
    s_user[i] = ok ? (uint32_t)uu : 0xFFFFFFFFu;   // unknown users sort last and form no group
  }
  __syncthreads();
  auto rank_of = [&](int i, uint32_t ui) {          // whole warp; every lane returns the rank
    uint32_t r = 0;
    for (int j = lane; j < Q; j += 32) {
      const uint32_t uj = s_user[j];
      r += (uj < ui || (uj == ui && j < i)) ? 1u : 0u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return (int)r;
  };
  if (q < Q) {
    const int pp = rank_of(q, s_user[q]);
    if (blockIdx.x == 0 && lane == 0) s_sorted[pp] = s_user[q];
    const uint4* src = reinterpret_cast<const uint4*>(src_row);
    uint4* dst = reinterpret_cast<uint4*>(a.qg + (size_t)pp * a.E);
    float ss = 0.f;
    for (int c = lane; c < a.E / 8; c += 32) {
      const uint4 v = src[c];
      dst[c] = v;
      float x[8];
      Vec<__half>::unpack(v, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) {
      a.q_inv[pp] = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
      a.qperm[pp] = q;
    }
  }
  if (blockIdx.x != 0) return;

  // CTA 0: the users of the queries the other CTAs packed, in position order ...
  for (int i = kGroupWarps + warp; i < Q; i += kGroupWarps) {
    const uint32_t ui = s_user[i];
    const int r = rank_of(i, ui);
    if (lane == 0) s_sorted[r] = ui;
  }
  __syncthreads();
  // ... then thread p looks at position p.
  const int p = tid;
  const uint32_t u = p < Q ? s_sorted[p] : 0xFFFFFFFFu;
  int32_t is_start = 0, count = 0, ntiles = 0;
  if (u != 0xFFFFFFFFu) {
    int lo = 0, hi = p;                             // first position of u's run
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_sorted[mid] < u) lo = mid + 1; else hi = mid;
    }
    if ((p - lo) % kGroupN == 0) {
      int end = p, ehi = Q;                         // one past the run's last position
      while (end < ehi) {
        const int mid = (end + ehi) >> 1;
        if (s_sorted[mid] == u) end = mid + 1; else ehi = mid;
      }
      is_start = 1;
      count = min(kGroupN, end - p);
      ntiles = a.user_meta[u].y;
    }
  }
  int32_t n_groups, n_items;
  const int32_t gidx = block_exclusive_scan(is_start, scratch, &n_groups);
  const int32_t item = block_exclusive_scan(ntiles, scratch, &n_items);
  if (is_start) a.groups[gidx] = make_int4((int32_t)u, p, count, item);
  if (tid == 0) {
    a.counts[0] = n_groups;
    a.counts[1] = n_items;
  }
}

// ---- the contraction ---------------------------------------------------------

__global__ void __launch_bounds__(128, 1) sim_gemm_kernel(const __grid_constant__ CUtensorMap tm_emb,
                                                         const __grid_constant__ CUtensorMap tm_q,
                                                         const GemmArgs g) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kGemmStages];
  __shared__ __align__(8) uint64_t bar_empty[kGemmStages];
  __shared__ __align__(8) uint64_t bar_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_tile_full;                        // the MMA thread issued every chunk of this tile
  __shared__ uint32_t s_kc_mma;                      // chunks the MMA thread has consumed so far
  __shared__ int s_tile, s_ti, s_pos, s_cnt, s_rows;

  pdl_wait();                                        // groups of the grouping kernel
  pdl_trigger();
  const int n_items = g.counts[1];
  if ((int)blockIdx.x >= n_items) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_addr(stages);

  if (warp == 0) {
    tmem_alloc(smem_addr(&s_tmem), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(smem_addr(&bar_full[s]), 1);
      mbar_init(smem_addr(&bar_empty[s]), 1);
    }
    mbar_init(smem_addr(&bar_done), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int nk = (g.E + kChunkK - 1) / kChunkK;
  volatile int* abort_flag = &s_abort;
  uint32_t kc_prod = 0, kc_mma = 0, n_done = 0;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    if (threadIdx.x == 0) {
      int lo = 0, hi = g.counts[0];
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (g.groups[mid].w <= it) lo = mid; else hi = mid;
      }
      const int4 gr = g.groups[lo];
      const int ti = it - gr.w;
      const int4 um = g.user_meta[gr.x];
      s_tile = user_tile(g.user_tiles, um, ti);
      s_ti = ti;
      s_pos = gr.y;
      s_cnt = gr.z;
      s_rows = min(128, um.z - ti * 128);
    }
    __syncthreads();
    const int tile = s_tile, ti = s_ti, pos = s_pos, cnt = s_cnt, nrows = s_rows;

    if (warp == 0 && lane == 0) {                    // TMA producer
      for (int kc = 0; kc < nk; ++kc, ++kc_prod) {
        const uint32_t s = kc_prod % kGemmStages, ph = (kc_prod / kGemmStages) & 1u;
        if (!wait_or_abort(smem_addr(&bar_empty[s]), ph ^ 1u, abort_flag, g.wait_ns)) {
          *abort_flag = 1;
          break;
        }
        const uint32_t bar = smem_addr(&bar_full[s]);
        mbar_expect_tx(bar, kStageBytes);
        tma_load_2d(sbase + s * kStageBytes, &tm_emb, kc * kChunkK, tile * 128, bar);
        tma_load_2d(sbase + s * kStageBytes + kATile, &tm_q, kc * kChunkK, pos, bar);
      }
    } else if (warp == 1 && lane == 0) {             // MMA issuer
      const uint32_t kc_mma0 = kc_mma;
      for (int kc = 0; kc < nk; ++kc, ++kc_mma) {
        const uint32_t s = kc_mma % kGemmStages, ph = (kc_mma / kGemmStages) & 1u;
        if (!wait_or_abort(smem_addr(&bar_full[s]), ph, abort_flag, g.wait_ns)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = sbase + s * kStageBytes, b0 = a0 + kATile;
#pragma unroll
        for (int k = 0; k < kChunkK / 16; ++k)
          mma_f16(tmem, sw128_desc(a0 + 32u * k), sw128_desc(b0 + 32u * k), (kc | k) != 0 ? 1u : 0u);
        mma_commit(smem_addr(&bar_empty[s]));
      }
      // Arrives once every MMA issued so far has completed, whether or not
      // the loop ran to the end.
      mma_commit(smem_addr(&bar_done));
      s_tile_full = kc_mma == kc_mma0 + (uint32_t)nk;
      s_kc_mma = kc_mma;
    }
    __syncwarp();
    __syncthreads();

    // Epilogue: warp w reads TMEM lanes 32w .. 32w+31 = tile rows.  The wait
    // for the MMAs drains the tensor core before TMEM is read (or, after an
    // abort, released), so it keeps the full budget and ignores the flag.
    const bool done = __syncthreads_and(mbar_wait_bounded(smem_addr(&bar_done), n_done & 1u, kWaitBudgetNs));
    ++n_done;
    tc_fence_after();
    const bool ok = done && s_tile_full;             // the same in every thread
    uint32_t acc[64];
    if (ok) {
      tmem_ld_32x32b_x64(tmem + ((uint32_t)(32 * warp) << 16), acc);
      tmem_wait_ld();
    }
    const int r = 32 * warp + lane;
    if (ok && r < nrows) {
      const float inv_e = g.emb_inv_norm[(size_t)tile * 128 + r];
      float* out = g.scores + (size_t)ti * 128 + r;
#pragma unroll
      for (int c = 0; c < kGroupN; ++c) {
        if (c < cnt) {
          const int q = g.qperm[pos + c];
          out[(size_t)q * g.score_stride] = __uint_as_float(acc[c]) * g.q_inv[pos + c] * inv_e;
        }
      }
    }
    if (!ok && threadIdx.x == 0) latch(g.status, IS_ST_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (!ok || *abort_flag) break;
  }
  // After an abort the producer may have loads in flight that no MMA
  // consumed (chunks s_kc_mma .. kc_prod - 1): they land before shared
  // memory is released.
  __syncthreads();
  if (warp == 0 && lane == 0) {
    for (uint32_t c = s_kc_mma; c < kc_prod; ++c)
      mbar_wait_bounded(smem_addr(&bar_full[c % kGemmStages]), (c / kGemmStages) & 1u, kWaitBudgetNs);
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---- per-query top-k of the batched path ---------------------------------------

template <bool SMEM_KEYS>
__global__ void __launch_bounds__(kRetThreads) topk_kernel(const TopkArgs ta, int32_t max_users) {
  extern __shared__ uint32_t s_keys[];
  __shared__ TopkShared sh;
  pdl_wait();                                        // scores of the contraction
  pdl_trigger();
  const int q = blockIdx.x;
  const int user = ta.users[q];
  const bool ok = user >= 0 && user < max_users;
  const int4 um = ok ? ta.user_meta[user] : make_int4(0, 0, 0, -1);
  topk_block<SMEM_KEYS>(ta, sh, s_keys, q, um, um.z);
}

// ---- host side ------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

bool make_operand_map(void* map_out, const void* base, int E, int64_t rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || E % 8 != 0 || rows <= 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)E, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)E * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kChunkK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(reinterpret_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

size_t operand_map_bytes() { return sizeof(CUtensorMap); }

cudaError_t launch_group(const GroupArgs& ga, const LaunchCfg& cfg) {
  const int grid = std::max(1, (ga.Q + kGroupWarps - 1) / kGroupWarps);
  return launch_ex(group_kernel, dim3(grid), dim3(kGroupThreads), 0, cfg.stream, cfg.pdl, ga);
}

cudaError_t launch_sim_gemm(const GemmArgs& gg, const void* map_emb, const void* map_q, int Q,
                            int max_user_tiles, const LaunchCfg& cfg) {
  const size_t smem = (size_t)kGemmStages * kStageBytes + 1024;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    const cudaError_t e =
        cudaFuncSetAttribute(sim_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set[dev & 63] = true;
  }
  const int64_t bound = (int64_t)Q * std::max(1, max_user_tiles);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(bound, 2LL * cfg.num_sms));
  const CUtensorMap* me = reinterpret_cast<const CUtensorMap*>(map_emb);
  const CUtensorMap* mq = reinterpret_cast<const CUtensorMap*>(map_q);
  return launch_ex(sim_gemm_kernel, dim3(grid), dim3(128), smem, cfg.stream, cfg.pdl, *me, *mq, gg);
}

cudaError_t launch_topk_batched(const TopkArgs& ta, int Q, int32_t max_users, int64_t max_user_facts,
                                const LaunchCfg& cfg) {
  if (max_user_facts <= kSmemKeysMax) {
    const size_t ks = (size_t)std::max<int64_t>(max_user_facts, 1) * sizeof(uint32_t);
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(topk_kernel<true>), ks);
    if (e != cudaSuccess) return e;
    return launch_ex(topk_kernel<true>, dim3(Q), dim3(kRetThreads), ks, cfg.stream, cfg.pdl, ta, max_users);
  }
  return launch_ex(topk_kernel<false>, dim3(Q), dim3(kRetThreads), 0, cfg.stream, cfg.pdl, ta, max_users);
}

}  // namespace isk
