// grouped_gemm_mx.cu -- the expert GEMMs of the MXFP8 layer as block-scaled
// FP8 MMAs on the 5th-generation tensor cores (tcgen05.mma kind::mxf8f6f4,
// E4M3 operands, one E8M0 scale per 32 K values of each row, fp32
// accumulation in TMEM).
//
// The MXFP8 weight format is the one the project summary "Mixture-of-Kittens
// (MoK)" names (core concepts, MXFP8 row: weights pre-quantised by a quantise
// op); the activations are quantised per 1x32 block along each GEMM's K, so
// every product the MMA forms is a product of two MXFP8 numbers.
//
// Structure (one persistent CTA per SM, clusters of two CTAs that share the A
// tile by multicast, as in the bf16 kernels):
//   warp 0      producer: TMA loads of the A (token rows) and B (weight rows)
//               tiles, 128 K values per stage, and 1-D bulk copies of the
//               matching scale chunks (512 bytes per 128 rows);
//   warp 1      MMA issuer: per stage, tcgen05.cp moves the scale chunks into
//               TMEM (32x128b, warpx4: replicated to the four lane quadrants),
//               then four K=32 block-scaled MMAs (M=128, N=256) read them;
//   warps 2..9  epilogue: two warps per TMEM lane quadrant, each takes half
//               of the 256 accumulator columns into registers, releases the
//               accumulator at once (one accumulator fits beside the scale
//               columns), then applies the epilogue and stores from registers.
// Scale chunks of stage s live in TMEM columns 256 + 16 s, so the copy of a
// stage never overwrites scales an MMA of an earlier stage may still read.
// Every wait is bounded (timeout -> MOE_DEVERR_TIMEOUT, drain, free TMEM).
#include <algorithm>
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "tma_map.h"

namespace moe {
namespace {

constexpr int QM = 128, QN = 256, QK = 128;  // tile; K counted in E4M3 values (= bytes)
constexpr int kQStages = 4;
constexpr int kQA = QM * QK;  // 16 KB
constexpr int kQB = QN * QK;  // 32 KB
constexpr int kQSfa = 512, kQSfb = 1024;
constexpr int kQStageUsed = kQA + kQB + kQSfa + kQSfb;
constexpr int kQStageBytes = 51200;  // stages start on 1024-byte boundaries
static_assert(kQStageUsed <= kQStageBytes && kQStageBytes % 1024 == 0, "stage layout");
constexpr int kQSmem = kQStages * kQStageBytes + 1024;
constexpr int kQThreads = 320;
constexpr uint32_t kQTmemCols = 512;
constexpr uint32_t kQSfCol = 256;

enum QMode { Q_GATE_UP = 0, Q_DOWN = 1 };

struct QMaps {
  CUtensorMap a, b0, b1;
};

struct QArgs {
  const int32_t* tiles;    // [n][3] (expert, row0, valid) of the 128-row tiles
  const int32_t* n_tiles;  // device count of those tiles
  int32_t* err;
  int max_mtiles;          // host bound on *n_tiles
  int64_t rows;            // rows of the expert-grouped buffers
  int n_nt;                // N tiles per M tile
  int nkb;                 // K blocks of 128
  int b_rows;              // rows per expert in B's 2-D view
  int E;
  const uint8_t* sfa;      // scale chunks of A [rows, K]
  const uint8_t* sfb0;     // scale chunks of B (gate rows for GATE_UP)
  const uint8_t* sfb1;     // up rows (GATE_UP)
  int64_t a_rblocks;       // rows of A / 128
  int64_t b_rblocks;       // rows of B / 128
  int ld_out;              // output row length (elements)
  int store_gu;            // GATE_UP: also store G and U
  void *out0, *out1, *out2;
};

// ---- PTX used only here --------------------------------------------------

// 1-D bulk copy global -> shared, completion counted on `bar` (16-byte
// aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory descriptor of an unswizzled source: 32 rows of 16 bytes,
// 8-row groups 128 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 32;  // stride between 8-row groups
  d |= static_cast<uint64_t>(1) << 46;         // descriptor version for tcgen05
  return d;
}

// 32 lanes x 128 bits from shared memory into TMEM columns [taddr, taddr + 4),
// replicated into all four lane quadrants.
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Instruction descriptor, kind::mxf8f6f4 with E4M3 A and B (format 0), fp32
// D, E8M0 scales (bit 23), scale byte `id` of each 32-bit scale column for A
// (bits 29-30) and B (bits 4-5).
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, uint32_t id) {
  return (id << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24) | (id << 29);
}

__device__ __forceinline__ void umma_mx(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ bool q_wait_drain(uint64_t* bar, uint32_t parity, int32_t* err) {
  int no_abort = 0;
  return mbar_wait(bar, parity, &no_abort, err);
}

struct QTile {
  int e, row0, nt;
  bool skip;
};

template <int CL>
__device__ __forceinline__ QTile q_decode(const QArgs& a, int64_t t, int crank) {
  QTile ti;
  const int n_ntp = a.n_nt / CL;
  const int mtile = static_cast<int>(t / n_ntp);
  ti.nt = static_cast<int>(t % n_ntp) * CL + crank;
  ti.e = a.tiles[3 * mtile + 0];
  ti.row0 = a.tiles[3 * mtile + 1];
  ti.skip = false;
  if (ti.e < 0 || ti.e >= a.E || ti.row0 < 0 || ti.row0 > a.rows - QM) {
    ti.e = 0;  // corrupt schedule: compute nothing, store nothing
    ti.row0 = 0;
    ti.skip = true;
  }
  return ti;
}

template <int CL>
__device__ __forceinline__ int64_t q_total(const QArgs& a) {
  int n = *a.n_tiles;
  n = n < 0 ? 0 : (n > a.max_mtiles ? a.max_mtiles : n);
  return static_cast<int64_t>(n) * (a.n_nt / CL);
}

__device__ __forceinline__ float q_silu(float g) { return g / (1.0f + expf(-g)); }

// 8 consecutive fp32 values -> one 16-byte bf16 store.
__device__ __forceinline__ void st_bf16x8(void* dst, const float* v) {
  *reinterpret_cast<uint4*>(dst) =
      make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                 pack_bf16x2(v[6], v[7]));
}

template <int MODE, int CL>
__global__ void __launch_bounds__(kQThreads, 1)
    grouped_gemm_mx_kernel(const __grid_constant__ QMaps maps, const QArgs args) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kQStages], empty_bar[kQStages], tfull_bar, tempty_bar, drain_bar;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], CL);  // both CTAs of a pair must have read the stage
    }
    mbar_init(&tfull_bar, 1);
    mbar_init(&tempty_bar, 8);  // one arrive per epilogue warp
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a);
    tma_prefetch_desc(&maps.b0);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_slot, kQTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CL > 1) cluster_sync();  // peers' barriers exist before any multicast
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  volatile int* abortp = &abort_flag;
  const int64_t total = q_total<CL>(args);
  const int crank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int64_t first = blockIdx.x / CL, stride = gridDim.x / CL;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int64_t t = first; t < total && ok; t += stride) {
        const QTile ti = q_decode<CL>(args, t, crank);
        const int nkb = ti.skip ? 0 : args.nkb;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abortp, args.err)) { ok = false; break; }
          uint8_t* sA = smem + stage * kQStageBytes;
          uint8_t* sB = sA + kQA;
          uint8_t* sSa = sB + kQB;
          uint8_t* sSb = sSa + kQSfa;
          uint64_t* bar = &full_bar[stage];
          mbar_arrive_expect_tx(bar, kQStageUsed);
          if constexpr (CL == 1) {
            tma_load_2d(sA, &maps.a, bar, kb * QK, ti.row0);
          } else {
            tma_load_2d_mc(sA + crank * (kQA / 2), &maps.a, bar, kb * QK,
                           ti.row0 + crank * (QM / 2), 0x3);
          }
          bulk_load(sSa, args.sfa + (static_cast<int64_t>(kb) * args.a_rblocks + ti.row0 / 128) * 512,
                    kQSfa, bar);
          if constexpr (MODE == Q_GATE_UP) {
            const int brow = ti.e * args.b_rows + ti.nt * (QN / 2);
            tma_load_2d(sB, &maps.b0, bar, kb * QK, brow);
            tma_load_2d(sB + kQB / 2, &maps.b1, bar, kb * QK, brow);
            const int64_t so = (static_cast<int64_t>(kb) * args.b_rblocks + brow / 128) * 512;
            bulk_load(sSb, args.sfb0 + so, 512, bar);
            bulk_load(sSb + 512, args.sfb1 + so, 512, bar);
          } else {
            const int brow = ti.e * args.b_rows + ti.nt * QN;
            tma_load_2d(sB, &maps.b0, bar, kb * QK, brow);
            bulk_load(sSb, args.sfb0 + (static_cast<int64_t>(kb) * args.b_rblocks + brow / 128) * 512,
                      kQSfb, bar);
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kQStages) { stage = 0; phase ^= 1u; }
        }
      }
      // Every issued copy must land before the CTA may exit.
      for (int s = 0; s < kQStages; ++s)
        if ((issued_mask >> s) & 1u) q_wait_drain(&full_bar[s], (issued_parity >> s) & 1u, args.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t t = first; t < total && ok; t += stride) {
        const QTile ti = q_decode<CL>(args, t, crank);
        const int nkb = ti.skip ? 0 : args.nkb;
        if (!mbar_wait(&tempty_bar, acc_phase ^ 1u, abortp, args.err)) break;
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abortp, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kQStageBytes);
          const uint32_t b_addr = a_addr + kQA;
          const uint32_t sfa_s = b_addr + kQB;
          const uint32_t sfb_s = sfa_s + kQSfa;
          const uint32_t sf_t = tmem_base + kQSfCol + stage * 16;
          tmem_cp_sf(sf_t, sdesc_sf(sfa_s));
          tmem_cp_sf(sf_t + 4, sdesc_sf(sfb_s));
          tmem_cp_sf(sf_t + 8, sdesc_sf(sfb_s + 512));
#pragma unroll
          for (int ks = 0; ks < QK / 32; ++ks) {
            const uint64_t ad = sdesc_sw128(a_addr + ks * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b_addr + ks * 32, 16, 1024);
            umma_mx(tmem_base, ad, bd, idesc_mx(QM, QN, static_cast<uint32_t>(ks)), sf_t,
                    sf_t + 4, (kb > 0 || ks > 0) ? 1u : 0u);
          }
          if constexpr (CL == 1) umma_commit(&empty_bar[stage]);
          else umma_commit_mc(&empty_bar[stage], (1u << CL) - 1);
          if (++stage == kQStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tfull_bar);  // accumulator ready (immediate if no MMA)
        acc_phase ^= 1u;
      }
      umma_commit(&drain_bar);
      q_wait_drain(&drain_bar, 0, args.err);
    }
  } else {
    // ---------------- epilogue warps 2..9 ----------------
    const int quad = warp & 3;        // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;  // which half of the accumulator columns
    uint32_t acc_phase = 0;
    for (int64_t t = first; t < total; t += stride) {
      const QTile ti = q_decode<CL>(args, t, crank);
      if (!mbar_wait(&tfull_bar, acc_phase, abortp, args.err)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
      float v[128];
      {
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          // GATE_UP: G columns [64 half, +64) then U columns [128 + 64 half, +64)
          const int col = MODE == Q_GATE_UP ? (c < 2 ? 64 * half + 32 * c : 128 + 64 * half + 32 * (c - 2))
                                            : 128 * half + 32 * c;
          tmem_ld32(taddr + col, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar);  // the MMAs of the next tile may start
      acc_phase ^= 1u;
      if (ti.skip) {
        if (lane == 0) set_dev_error(args.err, MOE_DEVERR_BAD_EXPERT);
        continue;
      }
      const int64_t row = static_cast<int64_t>(ti.row0) + quad * 32 + lane;
      if constexpr (MODE == Q_GATE_UP) {
        const int64_t o = row * args.ld_out + ti.nt * (QN / 2) + 64 * half;
        __nv_bfloat16* pg = static_cast<__nv_bfloat16*>(args.out0) + o;
        __nv_bfloat16* pu = static_cast<__nv_bfloat16*>(args.out1) + o;
        __nv_bfloat16* pa = static_cast<__nv_bfloat16*>(args.out2) + o;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (args.store_gu) {
            st_bf16x8(pg + 8 * j, v + 8 * j);
            st_bf16x8(pu + 8 * j, v + 64 + 8 * j);
          }
          float act[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) act[i] = q_silu(v[8 * j + i]) * v[64 + 8 * j + i];
          st_bf16x8(pa + 8 * j, act);
        }
      } else {
        __nv_bfloat16* py = static_cast<__nv_bfloat16*>(args.out0) + row * args.ld_out +
                            ti.nt * QN + 128 * half;
#pragma unroll
        for (int j = 0; j < 16; ++j) st_bf16x8(py + 8 * j, v + 8 * j);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kQTmemCols);
  }
  if constexpr (CL > 1) cluster_sync();  // no CTA leaves while its peer may still write to it
}

int q_sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

template <int MODE, int CL>
moe_status q_launch(const QMaps& maps, const QArgs& args, int64_t units, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;
  auto config = [](cudaLaunchConfig_t& cfg, cudaLaunchAttribute* at, int clusters) {
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = CL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(CL * clusters);
    cfg.blockDim = dim3(kQThreads);
    cfg.dynamicSmemBytes = kQSmem;
    cfg.attrs = at;
    cfg.numAttrs = 1;
  };
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_mx_kernel<MODE, CL>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
    if (attr_err != cudaSuccess || CL == 1) return;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    config(cfg, at, 64);
    attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, grouped_gemm_mx_kernel<MODE, CL>, &cfg);
    if (attr_err == cudaSuccess && max_clusters <= 0) attr_err = cudaErrorInvalidConfiguration;
  });
  if (attr_err != cudaSuccess) return MOE_ERR_CUDA;
  if (units <= 0) return MOE_OK;
  if constexpr (CL == 1) {
    const int grid = static_cast<int>(std::min<int64_t>(q_sm_count(), units));
    grouped_gemm_mx_kernel<MODE, 1><<<grid, kQThreads, kQSmem, s>>>(maps, args);
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    config(cfg, at, static_cast<int>(std::min<int64_t>(max_clusters, units)));
    cfg.stream = s;
    if (cudaLaunchKernelEx(&cfg, grouped_gemm_mx_kernel<MODE, CL>, maps, args) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <int MODE>
moe_status q_launch_rows(const QMaps& maps, const QArgs& args, cudaStream_t s) {
  if (args.n_nt % 2 == 0)
    return q_launch<MODE, 2>(maps, args, static_cast<int64_t>(args.max_mtiles) * (args.n_nt / 2), s);
  return q_launch<MODE, 1>(maps, args, static_cast<int64_t>(args.max_mtiles) * args.n_nt, s);
}

bool fp8_map(CUtensorMap* m, const void* base, int64_t k, int64_t rows, int box_rows) {
  return tma_map_2d(m, base, k, rows, box_rows, QK, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1);
}

QArgs q_base(const Layout& L, const void* ws) {
  QArgs a{};
  a.tiles = at<int32_t>(ws, L.tiles);
  a.n_tiles = at<int32_t>(ws, L.n_tiles);
  a.err = const_cast<int32_t*>(at<int32_t>(ws, L.err));
  a.max_mtiles = static_cast<int>(L.R / QM);
  a.rows = L.R;
  a.E = L.E;
  a.a_rblocks = L.R / 128;
  return a;
}

}  // namespace

moe_status gemm_mx_gate_up(const Layout& L, const void* ws, const uint8_t* xq, const uint8_t* xs,
                           const moe_mxfp8_operand& wg, const moe_mxfp8_operand& wu, void* g,
                           void* u, void* act, cudaStream_t s) {
  const int n_nt = L.I / (QN / 2);
  QMaps m{};
  if (!fp8_map(&m.a, xq, L.H, L.R, n_nt % 2 == 0 ? QM / 2 : QM) ||
      !fp8_map(&m.b0, wg.q, L.H, static_cast<int64_t>(L.E) * L.I, QN / 2) ||
      !fp8_map(&m.b1, wu.q, L.H, static_cast<int64_t>(L.E) * L.I, QN / 2))
    return MOE_ERR_CUDA;
  QArgs a = q_base(L, ws);
  a.n_nt = n_nt;
  a.nkb = L.H / QK;
  a.b_rows = L.I;
  a.sfa = xs;
  a.sfb0 = wg.s;
  a.sfb1 = wu.s;
  a.b_rblocks = static_cast<int64_t>(L.E) * L.I / 128;
  a.ld_out = L.I;
  a.store_gu = (g != nullptr && u != nullptr) ? 1 : 0;
  a.out0 = g;
  a.out1 = u;
  a.out2 = act;
  return q_launch_rows<Q_GATE_UP>(m, a, s);
}

moe_status gemm_mx_down(const Layout& L, const void* ws, const uint8_t* aq, const uint8_t* as,
                        const moe_mxfp8_operand& wd, void* ye, cudaStream_t s) {
  const int n_nt = L.H / QN;
  QMaps m{};
  if (!fp8_map(&m.a, aq, L.I, L.R, n_nt % 2 == 0 ? QM / 2 : QM) ||
      !fp8_map(&m.b0, wd.q, L.I, static_cast<int64_t>(L.E) * L.H, QN))
    return MOE_ERR_CUDA;
  m.b1 = m.b0;
  QArgs a = q_base(L, ws);
  a.n_nt = n_nt;
  a.nkb = L.I / QK;
  a.b_rows = L.H;
  a.sfa = as;
  a.sfb0 = wd.s;
  a.sfb1 = wd.s;
  a.b_rblocks = static_cast<int64_t>(L.E) * L.H / 128;
  a.ld_out = L.H;
  a.out0 = ye;
  return q_launch_rows<Q_DOWN>(m, a, s);
}

}  // namespace moe
