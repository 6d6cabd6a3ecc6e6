// Segment planning and the fused gather + Chunked RoPE + paged scatter-copy.
//
// InferScale ("Méthodologie", phase 2): the retrieved facts are composed into
// one contiguous segment, every stored pre-RoPE key is rotated to its
// serving-time position (Theorem 6: exact) and the composed K/V are
// scatter-copied into vLLM's paged KV cache.  One pass over the data: each
// (token, layer) row pair is read once from the store and written once to the
// cache, the rotation done in registers on the way.
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
  const int r = blockIdx.x;
  int n = a.n_ids_in[r];
  if (n < 0 || n > a.ids_stride) {
    if (threadIdx.x == 0) latch(a.status, IS_ST_COUNT);
    n = 0;
  }
  const int32_t user = a.users ? a.users[r] : -1;
  int32_t* off = a.fact_seg_off + (size_t)r * a.seg_stride;
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
// Work item = (segment token t, layer l): one K row and one V row of H*D
// elements, contiguous in the token-major store.  Items are numbered t*L + l
// over all requests back to back; each warp takes one contiguous run of
// items, so consecutive items usually share a token and its position, slot
// and rotation angles, which the warp keeps in registers.
//
// Lane mapping: lane handles 16-byte vectors v = lane + 32*m of each row.
// NeoX pairs (i, i + D/2) lie in vectors v and v ^ half_vecs: the partner
// vector comes from lane ^ half_vecs by shuffle (or from the lane's own next
// vector when half_vecs == 32).  Interleaved pairs lie inside one vector.
// Either way the frequencies a lane needs depend only on its lane index, so it
// computes VE (or VE/2) sin/cos once per position.
template <typename T, int VC, int STYLE>
__global__ void __launch_bounds__(256) inject_kernel(const InjectArgs a, const RopeTurns rt) {
  extern __shared__ int32_t s_off[];            // [R + 1] token offset of each request
  __shared__ int32_t scratch[33];
  constexpr int VE = Vec<T>::N;
  constexpr int NF = STYLE == 0 ? VE : VE / 2;

#if defined(__CUDA_ARCH__)
  asm volatile("griddepcontrol.wait;" ::: "memory");   // inputs of the previous kernel
#endif

  // Exclusive prefix of seg_len over requests.
  int32_t total = 0;
  {
    const int per = (a.R + blockDim.x - 1) / blockDim.x;
    const int b = min(a.R, (int)threadIdx.x * per);
    const int e = min(a.R, b + per);
    int32_t sum = 0;
    for (int i = b; i < e; ++i) sum += a.seg_len[i];
    int32_t base = block_exclusive_scan(sum, scratch, &total);
    for (int i = b; i < e; ++i) {
      s_off[i] = base;
      base += a.seg_len[i];
    }
    if (threadIdx.x == 0) s_off[a.R] = total;
    __syncthreads();
  }

  const int lane = threadIdx.x & 31;
  const int64_t n_items = (int64_t)total * a.L;
  const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t chunk = (n_items + n_warps - 1) / n_warps;
  int64_t it = warp_id * chunk;
  const int64_t it_end = min(n_items, it + chunk);
  if (it >= it_end) return;

  const uint64_t pol = policy_evict_first();
  const int vpl = a.row_bytes >> 9;             // vectors per lane per row (row_bytes / 512)
  const int hv = a.half_vecs;
  const int fbase = STYLE == 0 ? (lane % hv) * VE : (lane % a.head_vecs) * (VE / 2);
  const bool lane_first_half = (lane & hv) == 0;  // NeoX, half_vecs < 32

  float cs[NF], sn[NF];
  int32_t cur_t = -1, cur_r = -1, cur_j = 0, seg_lo = 0, seg_hi = 0, cur_p = -1;
  const uint8_t* src = nullptr;
  int64_t slot = -1;

  for (; it < it_end; ++it) {
    const int32_t t = (int32_t)(it / a.L);
    const int32_t l = (int32_t)(it - (int64_t)t * a.L);
    if (t != cur_t) {
      cur_t = t;
      // Request: the last r with s_off[r] <= t (zero-length requests repeat offsets).
      int lo = 0, hi = a.R;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= t) lo = mid; else hi = mid;
      }
      const int r = lo;
      const int32_t ts = t - s_off[r];
      if (r != cur_r || ts < seg_lo || ts >= seg_hi) {
        // Fact: the last j with off[j] <= ts, by a warp-wide search over
        // off[0 .. n] (n + 1 ascending entries, off[n] = segment length).
        const int32_t* off = a.fact_seg_off + (size_t)r * a.seg_stride;
        int jlo = 0, jhi = a.n_ids[r];
        while (jhi - jlo > 1) {
          const int stride = (jhi - jlo + 31) >> 5;
          const int idx = jlo + lane * stride;
          const bool le = idx < jhi && off[idx] <= ts;
          const unsigned m = __ballot_sync(0xffffffffu, le);
          jlo += (31 - __clz(m)) * stride;
          jhi = min(jhi, jlo + stride);
        }
        cur_r = r;
        cur_j = jlo;
        seg_lo = off[jlo];
        seg_hi = off[jlo + 1];
      }
      const int64_t f = a.ids[(size_t)cur_r * a.ids_stride + cur_j];
      const int32_t p = a.seg_start[cur_r] + ts;
      const int32_t lb = p / a.block_size;
      slot = -1;
      if (lb >= a.max_blocks) {
        if (lane == 0) latch(a.status, IS_ST_BLOCK_TABLE);
      } else {
        const int32_t blk = a.block_table[(size_t)cur_r * a.max_blocks + lb];
        if (blk < 0 || blk >= a.num_blocks) {
          if (lane == 0) latch(a.status, IS_ST_BLOCK_ID);
        } else {
          slot = (int64_t)blk * a.block_size + (p - lb * a.block_size);
        }
      }
      src = a.kv + (size_t)(a.fact_tok[f] + (ts - seg_lo)) * a.L * 2 * a.row_bytes;
      if (p != cur_p) {
        cur_p = p;
        const float pf = (float)p;
#pragma unroll
        for (int e = 0; e < NF; ++e) {
          const float fr = angle_turns(pf, rt.hi[fbase + e], rt.lo[fbase + e]);
          sincospif(2.0f * fr, &sn[e], &cs[e]);
        }
      }
    }
    if (l == 0 && lane == 0 && a.slot_mapping) a.slot_mapping[t] = slot;
    if (slot < 0) continue;

    const uint8_t* sk = src + (size_t)l * 2 * a.row_bytes;
    const uint8_t* sv = sk + a.row_bytes;
    uint8_t* dk = a.cache + ((size_t)(2 * l) * a.num_blocks * a.block_size + slot) * a.row_bytes;
    uint8_t* dv = a.cache + ((size_t)(2 * l + 1) * a.num_blocks * a.block_size + slot) * a.row_bytes;

    for (int c = 0; c < vpl; c += VC) {
      uint4 kx[VC], vx[VC];
#pragma unroll
      for (int m = 0; m < VC; ++m) {
        const size_t o = ((size_t)(c + m) * 32 + lane) * 16;
        kx[m] = ld_once(sk + o, pol);
        vx[m] = ld_once(sv + o, pol);
      }
#pragma unroll
      for (int m = 0; m < VC; ++m) st_v4(dv + ((size_t)(c + m) * 32 + lane) * 16, vx[m]);
#pragma unroll
      for (int m = 0; m < VC; ++m) {
        float x[VE], y[VE];
        Vec<T>::unpack(kx[m], x);
        if (STYLE == 0) {
          float z[VE];
          bool first;
          if (hv < 32) {
            Vec<T>::unpack(shfl_xor4(kx[m], hv), z);
            first = lane_first_half;
          } else {                                    // partner is the lane's next/previous vector
            Vec<T>::unpack(kx[m ^ 1], z);
            first = ((c + m) & 1) == 0;
          }
#pragma unroll
          for (int e = 0; e < VE; ++e)
            y[e] = first ? fmaf(x[e], cs[e], -z[e] * sn[e]) : fmaf(x[e], cs[e], z[e] * sn[e]);
        } else {
#pragma unroll
          for (int e = 0; e < VE / 2; ++e) {
            const float u = x[2 * e], w = x[2 * e + 1];
            y[2 * e] = fmaf(u, cs[e], -w * sn[e]);
            y[2 * e + 1] = fmaf(w, cs[e], u * sn[e]);
          }
        }
        st_v4(dk + ((size_t)(c + m) * 32 + lane) * 16, Vec<T>::pack(y));
      }
    }
  }
}

// ---------------------------------------------------------------------------

cudaError_t launch_plan(const PlanArgs& a, const LaunchCfg& cfg) {
  plan_kernel<<<a.R, 256, 0, cfg.stream>>>(a);
  return cudaGetLastError();
}

template <typename T, int VC, int STYLE>
static cudaError_t launch_inject_t(const InjectArgs& a, const RopeTurns& rt, int grid,
                                   const LaunchCfg& cfg) {
  const size_t smem = (size_t)(a.R + 1) * sizeof(int32_t);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(256);
  lc.dynamicSmemBytes = smem;
  lc.stream = cfg.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = cfg.pdl ? 1 : 0;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, inject_kernel<T, VC, STYLE>, a, rt);
}

template <typename T, int STYLE>
static cudaError_t dispatch_vc(const InjectArgs& a, const RopeTurns& rt, int grid,
                               const LaunchCfg& cfg) {
  const int vpl = a.row_bytes >> 9;
  if (vpl % 4 == 0) return launch_inject_t<T, 4, STYLE>(a, rt, grid, cfg);
  if (vpl % 2 == 0) return launch_inject_t<T, 2, STYLE>(a, rt, grid, cfg);
  return launch_inject_t<T, 1, STYLE>(a, rt, grid, cfg);
}

cudaError_t launch_inject(const InjectArgs& a, const RopeTurns& rt, int kv_dtype, int style,
                          int grid, const LaunchCfg& cfg) {
  if (kv_dtype == IS_BF16)
    return style == 0 ? dispatch_vc<__nv_bfloat16, 0>(a, rt, grid, cfg)
                      : dispatch_vc<__nv_bfloat16, 1>(a, rt, grid, cfg);
  if (kv_dtype == IS_F16)
    return style == 0 ? dispatch_vc<__half, 0>(a, rt, grid, cfg)
                      : dispatch_vc<__half, 1>(a, rt, grid, cfg);
  return style == 0 ? dispatch_vc<float, 0>(a, rt, grid, cfg)
                    : dispatch_vc<float, 1>(a, rt, grid, cfg);
}

template <typename T, int STYLE>
static int occupancy_t(int vpl) {
  int n = 0;
  const size_t smem = (size_t)(IS_MAX_REQUESTS + 1) * sizeof(int32_t);
  if (vpl % 4 == 0)
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, inject_kernel<T, 4, STYLE>, 256, smem);
  else if (vpl % 2 == 0)
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, inject_kernel<T, 2, STYLE>, 256, smem);
  else
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, inject_kernel<T, 1, STYLE>, 256, smem);
  return n > 0 ? n : 1;
}

int inject_ctas_per_sm(int kv_dtype, int style, int vpl) {
  if (kv_dtype == IS_BF16)
    return style == 0 ? occupancy_t<__nv_bfloat16, 0>(vpl) : occupancy_t<__nv_bfloat16, 1>(vpl);
  if (kv_dtype == IS_F16)
    return style == 0 ? occupancy_t<__half, 0>(vpl) : occupancy_t<__half, 1>(vpl);
  return style == 0 ? occupancy_t<float, 0>(vpl) : occupancy_t<float, 1>(vpl);
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
constexpr size_t kNaWords = (size_t)kNaRequests * kNaSegStride + 2 * kNaRequests;
constexpr int kNaMaxDevices = 64;

// [0, R*stride): per-request prefix of fact lengths; then n_ids[R]; then seg_len[R].
static __device__ __align__(256) int32_t g_noalloc_scratch[kNaWords];

struct NoAllocDevice {
  bool ready = false;
  int32_t* scratch = nullptr;   // device address of g_noalloc_scratch on this device
  int num_sms = 0;
  int ctas[3][2][3] = {};       // [dtype][style][vpl class], 0 = not yet queried
};
NoAllocDevice g_na_dev[kNaMaxDevices];
std::mutex g_na_mu;

is_status_t na_fail(is_status_t st, const char* msg) {
  isk::set_last_error_message(msg);
  return st;
}

}  // namespace

extern "C" is_status_t is_inject_noalloc(
    const void* kv_arena, const int64_t* fact_tok, const int32_t* fact_len, int64_t n_facts,
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
  if (n_facts < 1 || max_fact_len < 1 || max_blocks_per_seq < 1)
    return na_fail(IS_ERR_INVALID_ARG, "n_facts, max_fact_len, max_blocks_per_seq must be >= 1");
  if ((int64_t)R * ids_stride * max_fact_len >= (int64_t)INT32_MAX)
    return na_fail(IS_ERR_UNSUPPORTED, "R * ids_stride * max_fact_len must stay below 2^31");
  if (kv_dtype != IS_F32 && kv_dtype != IS_BF16 && kv_dtype != IS_F16)
    return na_fail(IS_ERR_INVALID_ARG, "bad kv_dtype");
  if (num_layers < 1 || num_kv_heads < 1 || head_dim < 16 || head_dim > IS_MAX_HEAD_DIM ||
      (head_dim & (head_dim - 1)) != 0)
    return na_fail(IS_ERR_UNSUPPORTED, "head_dim must be a power of two in [16, IS_MAX_HEAD_DIM]");
  const int elt = kv_dtype == IS_F32 ? 4 : 2;
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * elt;
  if (row_bytes % 512 != 0)
    return na_fail(IS_ERR_UNSUPPORTED, "num_kv_heads * head_dim * elt must be a multiple of 512");
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
  const int vpl = (int)(row_bytes >> 9);
  const int vclass = vpl % 4 == 0 ? 0 : (vpl % 2 == 0 ? 1 : 2);
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
    if (d.ctas[kv_dtype][rope->style][vclass] == 0)
      d.ctas[kv_dtype][rope->style][vclass] = inject_ctas_per_sm(kv_dtype, rope->style, vpl);
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
  p.n_facts = n_facts;
  p.n_ids_out = na_n_ids;
  p.fact_seg_off = seg_off;
  p.seg_stride = kNaSegStride;
  p.seg_len = seg_len;
  p.status = status_out;
  p.R = R;
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
  a.row_bytes = (int32_t)row_bytes;
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
  const int grid = d.num_sms * (d.ctas[kv_dtype][rope->style][vclass] > 0
                                    ? d.ctas[kv_dtype][rope->style][vclass] : 1);
  if (launch_inject(a, rt, kv_dtype, rope->style, grid, cfg) != cudaSuccess)
    return na_fail(IS_ERR_CUDA, "inject launch failed");
  return IS_OK;
}
