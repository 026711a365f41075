// route_schedule.cu -- top-k routing and the device-side schedule.
//
// Routing: the router picks the top-k experts per token ("Mixture-of-Kittens:
// Cursor open-sources an MoE training megakernel", key flowchart, Router
// node); weights are the softmax renormalised over the selected experts.
// Schedule: per-expert counts, exclusive prefix sums and the token->slot
// permutation are built on the GPU with no host synchronisation and no token
// dropping (same page, key point 4), so the host never learns the counts.
//
// The schedule is a deterministic counting sort in four launches:
//   1. count : each warp counts the experts of its 256 consecutive
//              assignments (warp match + popcount, no atomics).
//   2. scan  : one CTA per expert turns the per-warp counts into per-warp
//              bases (exclusive scan over warps) and the expert's total.
//   3. final : one CTA scans the totals into offsets / padded offsets and
//              writes the tile list and the padding rows of src_of_row.
//   4. place : each warp re-walks its assignments and places each one at
//              pad_offsets[e] + warp base + rank within the warp.
// Ranks follow the assignment order t*k+j, i.e. ascending token per expert.
#include <float.h>

#include <algorithm>
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__device__ __forceinline__ bool ranks_before(float za, int ia, float zb, int ib) {
  return za > zb || (za == zb && ia < ib);
}

// One warp per token; lane l holds experts l, l+32, ... (EPL per lane).
template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits,
                                                   const float* __restrict__ bias, int64_t N,
                                                   int E, int k, int32_t* __restrict__ ids,
                                                   float* __restrict__ w, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = warp0; t < N; t += nwarps) {
    float v[EPL];
    bool nan = false;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = i * 32 + lane;
      if (e < E) {
        const float z = logits[t * E + e] + (bias ? bias[e] : 0.0f);
        nan |= (z != z);
        v[i] = z;
      } else {
        v[i] = -FLT_MAX;  // never chosen: k <= E real candidates rank first
      }
    }
    if (__any_sync(0xffffffffu, nan) && lane == 0) set_dev_error(err, MOE_DEVERR_NAN_LOGIT);
    uint32_t taken = 0;
    float my_z = 0.0f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
      float bz = 0.0f;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = i * 32 + lane;
        if (e < E && !((taken >> i) & 1u) && (bi == 0x7fffffff || ranks_before(v[i], e, bz, bi))) {
          bz = v[i];
          bi = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float oz = __shfl_xor_sync(0xffffffffu, bz, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (oi != 0x7fffffff && (bi == 0x7fffffff || ranks_before(oz, oi, bz, bi))) {
          bz = oz;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == j) {
        my_z = bz;
        my_id = bi;
      }
    }
    const float zmax = __shfl_sync(0xffffffffu, my_z, 0);
    const float ex = (lane < k) ? expf(my_z - zmax) : 0.0f;
    float denom = 0.0f;
    for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, ex, j);  // ascending j
    if (lane < k) {
      ids[t * k + lane] = my_id;
      w[t * k + lane] = ex / denom;
    }
  }
}

// Kernel 1: per-warp expert counts. warp_counts is expert-major [E][n_warps].
__global__ void __launch_bounds__(256) sched_count_kernel(const int32_t* __restrict__ ids,
                                                          int64_t A, int E, int64_t n_warps,
                                                          int32_t* __restrict__ warp_counts,
                                                          int32_t* err) {
  extern __shared__ int32_t cnt_smem[];  // [8][E]
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * 8 + wib;
  int32_t* cnt = cnt_smem + wib * E;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  if (gw < n_warps) {
    const int64_t base = gw * kSchedSub;
    for (int it = 0; it < kSchedSub / 32; ++it) {
      const int64_t a = base + it * 32 + lane;
      int e = -1;
      if (a < A) {
        e = ids[a];
        if (e < 0 || e >= E) {
          set_dev_error(err, MOE_DEVERR_BAD_EXPERT);
          e = -1;
        }
      }
      const uint32_t same = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(same) - 1) cnt[e] += __popc(same);
      __syncwarp();
    }
    for (int e = lane; e < E; e += 32) warp_counts[static_cast<int64_t>(e) * n_warps + gw] = cnt[e];
  }
}

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int32_t block_exclusive_scan(int32_t v, int32_t* smem32, int32_t* total) {
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int32_t inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) smem32[wib] = inc;
  __syncthreads();
  if (wib == 0) {
    int32_t s = lane < nw ? smem32[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += o;
    }
    if (lane < nw) smem32[lane] = s;  // inclusive warp totals
  }
  __syncthreads();
  const int32_t warp_excl = wib ? smem32[wib - 1] : 0;
  const int32_t tot = smem32[nw - 1];
  __syncthreads();
  if (total) *total = tot;
  return warp_excl + inc - v;
}

// Kernel 2: one CTA per expert; exclusive scan of its per-warp counts.
__global__ void __launch_bounds__(1024) sched_scan_kernel(int32_t* __restrict__ warp_counts,
                                                          int64_t n_warps,
                                                          int32_t* __restrict__ counts) {
  __shared__ int32_t sm[32];
  const int e = blockIdx.x;
  int32_t* col = warp_counts + static_cast<int64_t>(e) * n_warps;
  int32_t carry = 0;
  for (int64_t c0 = 0; c0 < n_warps; c0 += blockDim.x) {
    const int64_t i = c0 + threadIdx.x;
    const int32_t v = i < n_warps ? col[i] : 0;
    int32_t tot;
    const int32_t ex = block_exclusive_scan(v, sm, &tot);
    if (i < n_warps) col[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) counts[e] = carry;
}

// Kernel 3: offsets, padded offsets, tile list, padding rows; optionally the
// SM-pair item list: each expert's segment cut front to back into 256-row
// items, the last one 128 rows when the segment holds an odd number of
// 128-row tiles (ptiles [n][3] = expert, first row, rows; n in *n_ptiles).
__global__ void __launch_bounds__(1024) sched_final_kernel(const int32_t* __restrict__ counts,
                                                           int E, int T,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ pad_offsets,
                                                           int32_t* __restrict__ src_of_row,
                                                           int32_t* __restrict__ tiles,
                                                           int32_t* __restrict__ n_tiles,
                                                           int32_t* __restrict__ ptiles,
                                                           int32_t* __restrict__ n_ptiles) {
  __shared__ int32_t sm[32];
  __shared__ int32_t s_pad[kMaxE + 1];
  __shared__ int32_t s_cnt[kMaxE];
  const int e = threadIdx.x;
  const int32_t c = e < E ? counts[e] : 0;
  const int32_t cp = (c + T - 1) / T * T;
  int32_t tot_c, tot_p, tot_i;
  const int32_t off = block_exclusive_scan(c, sm, &tot_c);
  const int32_t poff = block_exclusive_scan(cp, sm, &tot_p);
  const int32_t n_items = (cp / kTileM + 1) / 2;  // SM-pair items of this segment
  const int32_t ioff = block_exclusive_scan(n_items, sm, &tot_i);
  if (ptiles) {
    for (int32_t j = 0; j < n_items; ++j) {
      ptiles[3 * (ioff + j) + 0] = e;
      ptiles[3 * (ioff + j) + 1] = poff + 2 * kTileM * j;
      ptiles[3 * (ioff + j) + 2] = min(2 * kTileM, cp - 2 * kTileM * j);
    }
    if (e == 0) *n_ptiles = tot_i;
  }
  if (e < E) {
    offsets[e] = off;
    pad_offsets[e] = poff;
    s_pad[e] = poff;
    s_cnt[e] = c;
  }
  if (e == 0) {
    offsets[E] = tot_c;
    pad_offsets[E] = tot_p;
    s_pad[E] = tot_p;
    *n_tiles = tot_p / kTileM;
  }
  __syncthreads();
  const int32_t nt = tot_p / kTileM;
  for (int32_t i = threadIdx.x; i < nt; i += blockDim.x) {
    const int32_t r0 = i * kTileM;
    int lo = 0, hi = E - 1;  // last expert with s_pad[ex] <= r0 (and a non-empty segment)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pad[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    tiles[3 * i + 0] = lo;
    tiles[3 * i + 1] = r0;
    tiles[3 * i + 2] = max(0, min(kTileM, s_pad[lo] + s_cnt[lo] - r0));
  }
  // padding rows of every segment (fewer than T each)
  for (int32_t q = threadIdx.x; q < E * T; q += blockDim.x) {
    const int ex = q / T, r = q % T;
    const int32_t row = s_pad[ex] + s_cnt[ex] + r;
    if (row < s_pad[ex + 1]) src_of_row[row] = -1;
  }
}

// Kernel 4: place every assignment.
__global__ void __launch_bounds__(256) sched_place_kernel(
    const int32_t* __restrict__ ids, int64_t A, int E, int64_t n_warps,
    const int32_t* __restrict__ warp_base, const int32_t* __restrict__ pad_offsets,
    int32_t* __restrict__ slot_of, int32_t* __restrict__ src_of_row) {
  extern __shared__ int32_t run_smem[];  // [8][E]
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * 8 + wib;
  if (gw >= n_warps) return;
  int32_t* run = run_smem + wib * E;
  for (int e = lane; e < E; e += 32)
    run[e] = pad_offsets[e] + warp_base[static_cast<int64_t>(e) * n_warps + gw];
  __syncwarp();
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int64_t base = gw * kSchedSub;
  for (int it = 0; it < kSchedSub / 32; ++it) {
    const int64_t a = base + it * 32 + lane;
    int e = -1;
    if (a < A) {
      e = ids[a];
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    int32_t slot = -1;
    if (e >= 0) slot = run[e] + __popc(same & lt_mask);
    __syncwarp();
    if (e >= 0 && lane == __ffs(same) - 1) run[e] += __popc(same);
    __syncwarp();
    if (a < A) {
      slot_of[a] = slot;
      if (slot >= 0) src_of_row[slot] = static_cast<int32_t>(a);
    }
  }
}

}  // namespace

cudaError_t launch_route_topk(const Layout& L, const float* logits, const float* bias,
                              int32_t* ids, float* w, int32_t* err, cudaStream_t s) {
  if (L.N == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t warps_needed = L.N;
  int blocks = static_cast<int>(std::min<int64_t>((warps_needed + 7) / 8, 152 * 16));
  const int epl = (L.E + 31) / 32;
#define MOE_TOPK_CASE(X)                                                                    \
  if (epl <= X) {                                                                           \
    topk_kernel<X><<<blocks, threads, 0, s>>>(logits, bias, L.N, L.E, L.k, ids, w, err);    \
    note_launch();                                                                          \
    return cudaGetLastError();                                                              \
  }
  MOE_TOPK_CASE(1)
  MOE_TOPK_CASE(2)
  MOE_TOPK_CASE(4)
  MOE_TOPK_CASE(8)
  MOE_TOPK_CASE(16)
  MOE_TOPK_CASE(32)
#undef MOE_TOPK_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_build_schedule_with_scratch(const Layout& L, const int32_t* ids, void* ws,
                                               int32_t* warp_counts, cudaStream_t s) {
  int32_t* err = at<int32_t>(ws, L.err);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* pad = at<int32_t>(ws, L.pad_offsets);
  int32_t* slot_of = at<int32_t>(ws, L.slot_of);
  int32_t* src = at<int32_t>(ws, L.src_of_row);
  int32_t* tiles = at<int32_t>(ws, L.tiles);
  int32_t* n_tiles = at<int32_t>(ws, L.n_tiles);
  const int blocks_w = static_cast<int>((L.n_warps + 7) / 8);
  const size_t smem_w = sizeof(int32_t) * 8 * L.E;
  if (L.n_warps > 0) {
    sched_count_kernel<<<blocks_w, 256, smem_w, s>>>(ids, L.A, L.E, L.n_warps, warp_counts, err);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    sched_scan_kernel<<<L.E, 1024, 0, s>>>(warp_counts, L.n_warps, counts);
    note_launch();
  } else {
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * L.E, s);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sched_final_kernel<<<1, 1024, 0, s>>>(counts, L.E, L.T, offsets, pad, src, tiles, n_tiles,
                                        at<int32_t>(ws, L.ptiles), at<int32_t>(ws, L.n_ptiles));
  note_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess || L.n_warps == 0) return e;
  sched_place_kernel<<<blocks_w, 256, smem_w, s>>>(ids, L.A, L.E, L.n_warps, warp_counts, pad,
                                                   slot_of, src);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_build_schedule(const Layout& L, const int32_t* ids, void* ws, cudaStream_t s) {
  return launch_build_schedule_with_scratch(L, ids, ws, at<int32_t>(ws, L.warp_counts), s);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free schedule build.
//
// Some callers cannot allocate device memory at all (for example a plugin
// whose host application owns the whole device memory pool, or a loop that
// must never call into the allocator), so they cannot provide the scan
// scratch that moe_build_schedule takes from the workspace. This entry point
// keeps that scratch in a library-owned static device array instead; the
// caller only passes the ids and the output tables.
//
// The array is shared by every call on a device and is held until the
// process exits. Nothing in it needs to start at zero: the count kernel writes
// every entry that the scan and place kernels read. Calls whose kernels
// overlap on the GPU (e.g. on two streams) race on the array.
namespace {

constexpr int64_t kNoAllocScratchInts = int64_t(1) << 19;  // 2 MiB of int32
__device__ __align__(256) int32_t g_sched_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
struct ScratchAddr {
  unsigned long long ctx_id;  // unique id of the context the address belongs to (0: none)
  int32_t* ptr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};

// Unique id of the calling thread's current context (driver entry points
// looked up once through the runtime, no libcuda link); 0 if none is current.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_sched_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// the device current and cached per device together with the id of the
// context it was taken in: the first call on a device does the lookup, and so
// does the first call after the device's context was destroyed and created
// again (cudaDeviceReset), where the old address would be stale.
cudaError_t scratch_for_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& c = g_scratch_addr[dev];
  if (ctx == 0 || c.ctx_id != ctx || !c.ptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_sched_scratch);  // also makes the device's context current
    if (e != cudaSuccess) return e;
    c.ptr = static_cast<int32_t*>(p);
    c.ctx_id = current_context_id();
  }
  *out = c.ptr;
  return cudaSuccess;
}

inline bool ok4(const void* p) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3) == 0;
}

}  // namespace

extern "C" moe_status moe_build_schedule_noalloc(const moe_problem* p, const int32_t* topk_ids,
                                                 const moe_schedule* out, int32_t* err_word,
                                                 void* stream) {
  using namespace moe;
  Layout L;
  const moe_status st = make_layout(p, &L);
  if (st != MOE_OK) return st;
  if (L.E * std::max<int64_t>(L.n_warps, 1) > kNoAllocScratchInts) return MOE_ERR_UNSUPPORTED;
  if (!out || !ok4(err_word) || (L.N > 0 && !ok4(topk_ids)) || !ok4(out->counts) ||
      !ok4(out->offsets) || !ok4(out->pad_offsets) || (L.A > 0 && !ok4(out->slot_of)) ||
      !ok4(out->src_of_row) || !ok4(out->tiles) || !ok4(out->n_tiles))
    return MOE_ERR_INVALID_ARG;
  int32_t* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int blocks_w = static_cast<int>((L.n_warps + 7) / 8);
  const size_t smem_w = sizeof(int32_t) * 8 * L.E;
  if (L.n_warps > 0) {
    sched_count_kernel<<<blocks_w, 256, smem_w, s>>>(topk_ids, L.A, L.E, L.n_warps, scratch,
                                                     err_word);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    sched_scan_kernel<<<L.E, 1024, 0, s>>>(scratch, L.n_warps, out->counts);
    note_launch();
  } else if (cudaMemsetAsync(out->counts, 0, sizeof(int32_t) * L.E, s) != cudaSuccess) {
    return MOE_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  sched_final_kernel<<<1, 1024, 0, s>>>(out->counts, L.E, L.T, out->offsets, out->pad_offsets,
                                        out->src_of_row, out->tiles, out->n_tiles, nullptr,
                                        nullptr);
  note_launch();
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  if (L.n_warps == 0) return MOE_OK;
  sched_place_kernel<<<blocks_w, 256, smem_w, s>>>(topk_ids, L.A, L.E, L.n_warps, scratch,
                                                   out->pad_offsets, out->slot_of,
                                                   out->src_of_row);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
