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
// Structure (one persistent CTA per SM, each loading its own tiles):
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
//
// Every GEMM is TN (both operands K-major): the backward ones read the
// weights through transposed quantised copies and the weight gradients read
// token-axis quantised, transposed activations, so one operand path serves
//   GATE_UP  G|U = Xe . [Wg[e]; Wu[e]]^T  -> G, U, Act = silu(G) * U (bf16)
//   DOWN     Ye  = Act . Wd[e]^T           -> bf16
//   DACT     dAct = dYe . (Wd[e]^T)^T      -> dG, dU via the SwiGLU backward
//   DXE      dXe = dG . (Wg[e]^T)^T + dU . (Wu[e]^T)^T  (two K phases) -> bf16
//   WGRAD    dW[e] = P_e^T . Q_e (K = the expert's rows) -> fp32, one or two
//            problems per launch (dWg and dWu share Q = Xe).
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
constexpr int kQStageBytes = kQA + kQB;   // operand tiles of a stage (1024-byte multiple)
constexpr int kQSfBytes = kQSfa + kQSfb;   // scale chunks of a stage, in a ring of their own
constexpr int kQStageTx = kQStageBytes + kQSfBytes;  // bytes that complete a stage
// Epilogue staging for TMA stores: per epilogue warp two 32-row x 32-byte buffers.
constexpr int kQOutBuf = 1024;
constexpr int kQOutBytes = 8 * 2 * kQOutBuf;
constexpr int kQSmem = kQStages * (kQStageBytes + kQSfBytes) + kQOutBytes + 1024;
constexpr int kQThreads = 320;
constexpr uint32_t kQTmemCols = 512;
constexpr uint32_t kQSfCol = 256;

enum QMode { Q_GATE_UP = 0, Q_DOWN = 1, Q_DACT = 2, Q_DXE = 3, Q_WGRAD = 4 };

struct QMaps {
  CUtensorMap a0, a1, b0, b1;
  CUtensorMap o0, o1, o2;  // outputs (TMA stores): 32 rows x 32 bytes, no swizzle
  CUtensorMap o3;          // GATE_UP: Act's E4M3 codes (row form, the down GEMM's A)
};

struct QArgs {
  const int32_t* tiles;        // [n][3] (expert, row0, valid) of the 128-row tiles
  const int32_t* n_tiles;      // device count of those tiles
  const int32_t* pad_offsets;  // [E+1] padded segment starts (WGRAD K ranges)
  const int32_t* order;        // [E] experts by descending row count (WGRAD)
  const int32_t* counts;       // [E] rows per expert (WGRAD K = count rounded up to 128)
  int32_t* err;
  int max_mtiles;              // host bound on *n_tiles
  int64_t rows;                // rows of the expert-grouped buffers
  int n_nt;                    // N tiles per M tile (token-row modes)
  int kb1, kb2;                // K blocks of 128 of phase 1 and 2
  int b_rows;                  // GATE_UP / DOWN: rows per expert in B's 2-D view
  int k_exp;                   // DACT / DXE: K per expert in the transposed weights
  int E, w_mt, w_nt, n_probs;  // WGRAD tiling (M, N tiles of dW[e]; problems)
  const uint8_t* sfa0;         // scale chunks of A (phase / problem 0)
  const uint8_t* sfa1;         // ... of the second A (DXE phase 2, WGRAD problem 1)
  const uint8_t* sfb0;         // scale chunks of B (gate rows for GATE_UP)
  const uint8_t* sfb1;         // up rows (GATE_UP), second B (DXE)
  int64_t a_rblocks;           // rows of A / 128
  int64_t b_rblocks;           // rows of B / 128
  int ld_out;                  // output row length (elements)
  int store_gu;                // GATE_UP: also store G and U
  uint8_t* act_sf;             // GATE_UP: Act's scale chunks (row form), with o3; NULL: none
  const void *in0, *in1;       // DACT: the saved G, U
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
  int e, row0, mt, nt, prob, kstart, nkb;
  bool skip;
};

// Tile t of this CTA.
template <int MODE>
__device__ __forceinline__ QTile q_decode(const QArgs& a, int64_t t) {
  QTile ti;
  ti.skip = false;
  if constexpr (MODE == Q_WGRAD) {
    // Largest experts first; within an expert (mt, N tile pair, problem), the
    // problem fastest, so dWg and dWu tiles reading one Xe panel run together.
    const int64_t per_e = static_cast<int64_t>(a.w_mt) * a.w_nt * a.n_probs;
    const int rank = static_cast<int>(t / per_e);
    int64_t r = t % per_e;
    ti.mt = static_cast<int>(r / (a.w_nt * a.n_probs));
    r %= (a.w_nt * a.n_probs);
    ti.nt = static_cast<int>(r / a.n_probs);
    ti.prob = static_cast<int>(r % a.n_probs);
    ti.e = a.order[rank];
    if (ti.e < 0 || ti.e >= a.E) ti.e = 0;
    ti.kstart = a.pad_offsets[ti.e];
    ti.nkb = (a.counts[ti.e] + QK - 1) / QK;  // rows past the count are zero padding
    ti.row0 = 0;
    if (ti.kstart < 0 || ti.kstart % QK != 0 || ti.nkb < 0 ||
        ti.kstart + static_cast<int64_t>(ti.nkb) * QK > a.pad_offsets[ti.e + 1] ||
        ti.kstart + static_cast<int64_t>(ti.nkb) * QK > a.rows) {
      ti.kstart = 0;  // corrupt schedule: compute nothing, store nothing
      ti.nkb = 0;
      ti.skip = true;
    }
  } else {
    const int mtile = static_cast<int>(t / a.n_nt);
    ti.nt = static_cast<int>(t % a.n_nt);
    ti.mt = mtile;
    ti.prob = 0;
    ti.kstart = 0;
    ti.e = a.tiles[3 * mtile + 0];
    ti.row0 = a.tiles[3 * mtile + 1];
    ti.nkb = a.kb1 + a.kb2;
    if (ti.e < 0 || ti.e >= a.E || ti.row0 < 0 || ti.row0 > a.rows - QM) {
      ti.e = 0;
      ti.row0 = 0;
      ti.nkb = 0;
      ti.skip = true;
    }
  }
  return ti;
}

template <int MODE>
__device__ __forceinline__ int64_t q_total(const QArgs& a) {
  if constexpr (MODE == Q_WGRAD) {
    return static_cast<int64_t>(a.n_probs) * a.E * a.w_mt * a.w_nt;
  } else {
    int n = *a.n_tiles;
    n = n < 0 ? 0 : (n > a.max_mtiles ? a.max_mtiles : n);
    return static_cast<int64_t>(n) * a.n_nt;
  }
}

// The copies of one stage: A, B, and the scale chunks of both. Coordinates
// are (K element, row).
template <int MODE>
__device__ __forceinline__ void q_issue_loads(const QMaps& m, const QArgs& a, const QTile& ti,
                                              int kb, uint8_t* sA, uint8_t* sSa, uint64_t* bar) {
  uint8_t* sB = sA + kQA;
  uint8_t* sSb = sSa + kQSfa;
  const CUtensorMap* ma = &m.a0;
  const uint8_t* sfa = a.sfa0;
  int ax, ay;            // A tile origin
  int64_t a_chunk;       // A scale chunk index
  const CUtensorMap* mb = &m.b0;
  const uint8_t* sfb = a.sfb0;
  int bx, by;            // B tile origin
  int64_t b_chunk;
  if constexpr (MODE == Q_WGRAD) {
    if (ti.prob) { ma = &m.a1; sfa = a.sfa1; }
    const int k0 = ti.kstart + kb * QK;
    ax = k0;
    ay = ti.mt * QM;
    a_chunk = static_cast<int64_t>(k0 / QK) * a.a_rblocks + ti.mt;
    bx = k0;
    by = ti.nt * QN;
    b_chunk = static_cast<int64_t>(k0 / QK) * a.b_rblocks + ti.nt * (QN / 128);
  } else if constexpr (MODE == Q_DACT || MODE == Q_DXE) {
    const bool second = (MODE == Q_DXE) && kb >= a.kb1;
    const int kk = second ? kb - a.kb1 : kb;
    if (second) { ma = &m.a1; sfa = a.sfa1; mb = &m.b1; sfb = a.sfb1; }
    ax = kk * QK;
    ay = ti.row0;
    a_chunk = static_cast<int64_t>(kk) * a.a_rblocks + ti.row0 / 128;
    bx = ti.e * a.k_exp + kk * QK;
    by = ti.nt * QN;
    b_chunk = static_cast<int64_t>(bx / QK) * a.b_rblocks + ti.nt * (QN / 128);
  } else {  // GATE_UP, DOWN
    ax = kb * QK;
    ay = ti.row0;
    a_chunk = static_cast<int64_t>(kb) * a.a_rblocks + ti.row0 / 128;
    bx = kb * QK;
    by = MODE == Q_GATE_UP ? ti.e * a.b_rows + ti.nt * (QN / 2) : ti.e * a.b_rows + ti.nt * QN;
    b_chunk = static_cast<int64_t>(kb) * a.b_rblocks + by / 128;
  }
  tma_load_2d(sA, ma, bar, ax, ay);
  bulk_load(sSa, sfa + a_chunk * 512, kQSfa, bar);
  if constexpr (MODE == Q_GATE_UP) {
    // the N tile is 128 gate rows then 128 up rows of the same expert
    tma_load_2d(sB, &m.b0, bar, bx, by);
    tma_load_2d(sB + kQB / 2, &m.b1, bar, bx, by);
    bulk_load(sSb, a.sfb0 + b_chunk * 512, 512, bar);
    bulk_load(sSb + 512, a.sfb1 + b_chunk * 512, 512, bar);
  } else {
    tma_load_2d(sB, mb, bar, bx, by);
    bulk_load(sSb, sfb + b_chunk * 512, kQSfb, bar);
  }
}

// The SwiGLU epilogues use the fast exponential and division intrinsics
// (__expf: at most 2 + floor(1.16 |x|) ulp; __fdividef: 2 ulp): their error is
// far below the bf16 rounding of G, U, Act, dG and dU, and the exact forms
// made the dAct epilogue, not the MMAs, the bound of that GEMM.
__device__ __forceinline__ float q_sigmoid(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }
__device__ __forceinline__ float q_silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// 16 consecutive fp32 values -> 16 bf16 (8 words).
__device__ __forceinline__ void pack16(const float* v, uint32_t (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
}

// One 32-row x 32-byte block of a warp's output (32 bytes of each lane's row)
// through a shared staging buffer to one TMA store at (x, y); two buffers per
// warp let a store overlap the next block.
__device__ __forceinline__ void q_store(const CUtensorMap* om, const uint32_t (&w)[8], int32_t x,
                                        int32_t y, int lane, uint8_t* bufs, uint32_t& n) {
  uint8_t* buf = bufs + (n & 1u) * kQOutBuf;
  if (lane == 0) bulk_wait_read<1>();  // the store that last used this buffer has read it
  __syncwarp();
  const uint32_t a = smem_u32(buf) + lane * 32;
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3])
               : "memory");
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a + 16), "r"(w[4]), "r"(w[5]),
               "r"(w[6]), "r"(w[7])
               : "memory");
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(om, buf, x, y);
    bulk_commit();
  }
  ++n;
}

template <int MODE>
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
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&tfull_bar, 1);
    mbar_init(&tempty_bar, 8);  // one arrive per epilogue warp
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a0);
    tma_prefetch_desc(&maps.b0);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_slot, kQTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  volatile int* abortp = &abort_flag;
  const int64_t total = q_total<MODE>(args);
  const int64_t first = blockIdx.x, stride = gridDim.x;
  uint8_t* sf_ring = smem + kQStages * kQStageBytes;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int64_t t = first; t < total && ok; t += stride) {
        const QTile ti = q_decode<MODE>(args, t);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abortp, args.err)) { ok = false; break; }
          uint64_t* bar = &full_bar[stage];
          mbar_arrive_expect_tx(bar, kQStageTx);
          q_issue_loads<MODE>(maps, args, ti, kb, smem + stage * kQStageBytes,
                              sf_ring + stage * kQSfBytes, bar);
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
        const QTile ti = q_decode<MODE>(args, t);
        if (!mbar_wait(&tempty_bar, acc_phase ^ 1u, abortp, args.err)) break;
        tc_fence_after();
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abortp, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kQStageBytes);
          const uint32_t b_addr = a_addr + kQA;
          const uint32_t sfa_s = smem_u32(sf_ring + stage * kQSfBytes);
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
          umma_commit(&empty_bar[stage]);
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
    uint8_t* out_bufs = sf_ring + kQStages * kQSfBytes + (warp - 2) * 2 * kQOutBuf;
    uint32_t nstore = 0;
    uint32_t acc_phase = 0;
    for (int64_t t = first; t < total; t += stride) {
      const QTile ti = q_decode<MODE>(args, t);
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
      const int32_t y = ti.row0 + quad * 32;  // first output row of this warp (token modes)
      if constexpr (MODE == Q_WGRAD) {
        // fp32 dW[e] rows; an expert without rows has an all-zero gradient
        if (ti.nkb == 0) {
#pragma unroll
          for (int i = 0; i < 128; ++i) v[i] = 0.0f;
        }
        const CUtensorMap* om = ti.prob ? &maps.o1 : &maps.o0;
        const int32_t wy = ti.e * (args.w_mt * QM) + ti.mt * QM + quad * 32;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(v[8 * j + i]);
          q_store(om, w, ti.nt * QN + 128 * half + 8 * j, wy, lane, out_bufs, nstore);
        }
      } else if constexpr (MODE == Q_DACT) {
        // dG, dU from dAct and the saved G, U of the same rows and columns
        const int64_t row = static_cast<int64_t>(y) + lane;
        const int32_t x0 = ti.nt * QN + 128 * half;
        const int64_t o = row * args.ld_out + x0;
        const uint4* pg = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(args.in0) + o);
        const uint4* pu = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(args.in1) + o);
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // fully unrolled: v stays in registers
          uint32_t og[8], ou[8];
#pragma unroll
          for (int hv = 0; hv < 2; ++hv) {
            const uint4 gv = pg[2 * j + hv], uv = pu[2 * j + hv];
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
            const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float dg2[2], du2[2];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const float da = v[16 * j + 8 * hv + 2 * q + h];
                const float g = h ? bf16hi(gw[q]) : bf16lo(gw[q]);
                const float u = h ? bf16hi(uw[q]) : bf16lo(uw[q]);
                const float sg = q_sigmoid(g);
                dg2[h] = da * u * sg * (1.0f + g * (1.0f - sg));
                du2[h] = da * g * sg;
              }
              og[4 * hv + q] = pack_bf16x2(dg2[0], dg2[1]);
              ou[4 * hv + q] = pack_bf16x2(du2[0], du2[1]);
            }
          }
          q_store(&maps.o0, og, x0 + 16 * j, y, lane, out_bufs, nstore);
          q_store(&maps.o1, ou, x0 + 16 * j, y, lane, out_bufs, nstore);
        }
      } else if constexpr (MODE == Q_GATE_UP) {
        const int32_t x0 = ti.nt * (QN / 2) + 64 * half;
        // Act's MXFP8 row form, from its bf16 values: the thread's 64 columns
        // are two 32-value blocks (blocks 4 nt + 2 half + {0, 1} of the row)
        float blk[32];
        uint8_t codes[2] = {0, 0};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t w[8];
          if (args.store_gu) {
            pack16(v + 16 * j, w);
            q_store(&maps.o0, w, x0 + 16 * j, y, lane, out_bufs, nstore);
            pack16(v + 64 + 16 * j, w);
            q_store(&maps.o1, w, x0 + 16 * j, y, lane, out_bufs, nstore);
          }
          float act[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) act[i] = q_silu(v[16 * j + i]) * v[64 + 16 * j + i];
          pack16(act, w);
          q_store(&maps.o2, w, x0 + 16 * j, y, lane, out_bufs, nstore);
          if (args.act_sf) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              blk[16 * (j & 1) + 2 * i] = bf16lo(w[i]);
              blk[16 * (j & 1) + 2 * i + 1] = bf16hi(w[i]);
            }
            if (j & 1) {
              uint32_t cq[8];
              codes[j >> 1] = quant32(blk, cq);
              q_store(&maps.o3, cq, x0 + 32 * (j >> 1), y, lane, out_bufs, nstore);
            }
          }
        }
        if (args.act_sf) {
          const int64_t r = static_cast<int64_t>(y) + lane;
          const int64_t kb = x0 / 32;  // first of the two blocks; kb % 4 == 2 * half
          *reinterpret_cast<uint16_t*>(args.act_sf + sf_mma_index(r, kb, args.rows)) =
              static_cast<uint16_t>(codes[0] | (codes[1] << 8));
        }
      } else {  // DOWN, DXE
        const int32_t x0 = ti.nt * QN + 128 * half;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t w[8];
          pack16(v + 16 * j, w);
          q_store(&maps.o0, w, x0 + 16 * j, y, lane, out_bufs, nstore);
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // stores done before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kQTmemCols);
  }
}

int q_sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

// One persistent CTA per SM, capped by the tiles available.
template <int MODE>
moe_status q_launch(const QMaps& maps, const QArgs& args, int64_t units, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_mx_kernel<MODE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
  });
  if (attr_err != cudaSuccess) return MOE_ERR_CUDA;
  if (units <= 0) return MOE_OK;
  const int grid = static_cast<int>(std::min<int64_t>(q_sm_count(), units));
  grouped_gemm_mx_kernel<MODE><<<grid, kQThreads, kQSmem, s>>>(maps, args);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <int MODE>
moe_status q_launch_rows(const QMaps& maps, const QArgs& args, cudaStream_t s) {
  return q_launch<MODE>(maps, args, static_cast<int64_t>(args.max_mtiles) * args.n_nt, s);
}

bool fp8_map(CUtensorMap* m, const void* base, int64_t k, int64_t rows, int box_rows) {
  return tma_map_2d(m, base, k, rows, box_rows, QK, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1);
}

// Output [rows, cols] for the epilogue's TMA stores: 32 rows x 32 bytes.
bool out_map_bf16(CUtensorMap* m, const void* base, int64_t cols, int64_t rows) {
  return tma_map_2d(m, base, cols, rows, 32, 16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
}
bool out_map_f32(CUtensorMap* m, const void* base, int64_t cols, int64_t rows) {
  return tma_map_2d(m, base, cols, rows, 32, 8, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
}

QArgs q_base(const Layout& L, const void* ws) {
  QArgs a{};
  a.tiles = at<int32_t>(ws, L.tiles);
  a.n_tiles = at<int32_t>(ws, L.n_tiles);
  a.pad_offsets = at<int32_t>(ws, L.pad_offsets);
  a.order = at<int32_t>(ws, L.expert_order);
  a.counts = at<int32_t>(ws, L.counts);
  a.err = const_cast<int32_t*>(at<int32_t>(ws, L.err));
  a.max_mtiles = static_cast<int>(L.R / QM);
  a.rows = L.R;
  a.E = L.E;
  a.a_rblocks = L.R / 128;
  return a;
}

template <int MODE>
moe_status q_launch_wgrad(const QMaps& maps, const QArgs& args, cudaStream_t s) {
  return q_launch<MODE>(maps, args,
                        static_cast<int64_t>(args.n_probs) * args.E * args.w_mt * args.w_nt, s);
}

}  // namespace

moe_status gemm_mx_gate_up(const Layout& L, const void* ws, moe_mxfp8_operand xe,
                           const moe_mxfp8_operand& wg, const moe_mxfp8_operand& wu, void* g,
                           void* u, void* act, const moe_mxfp8_operand* act_q, cudaStream_t s) {
  const int n_nt = L.I / (QN / 2);
  QMaps m{};
  if (!fp8_map(&m.a0, xe.q, L.H, L.R, QM) ||
      !fp8_map(&m.b0, wg.q, L.H, static_cast<int64_t>(L.E) * L.I, QN / 2) ||
      !fp8_map(&m.b1, wu.q, L.H, static_cast<int64_t>(L.E) * L.I, QN / 2))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  QArgs a = q_base(L, ws);
  a.n_nt = n_nt;
  a.kb1 = L.H / QK;
  a.b_rows = L.I;
  a.sfa0 = a.sfa1 = xe.s;
  a.sfb0 = wg.s;
  a.sfb1 = wu.s;
  a.b_rblocks = static_cast<int64_t>(L.E) * L.I / 128;
  a.ld_out = L.I;
  a.store_gu = (g != nullptr && u != nullptr) ? 1 : 0;
  if (!out_map_bf16(&m.o2, act, L.I, L.R)) return MOE_ERR_CUDA;
  if (a.store_gu && (!out_map_bf16(&m.o0, g, L.I, L.R) || !out_map_bf16(&m.o1, u, L.I, L.R)))
    return MOE_ERR_CUDA;
  if (act_q) {  // the epilogue also writes Act's row-form codes and scales
    if (!tma_map_2d(&m.o3, act_q->q, L.I, L.R, 32, 32, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
      return MOE_ERR_CUDA;
    a.act_sf = const_cast<uint8_t*>(act_q->s);
  }
  return q_launch_rows<Q_GATE_UP>(m, a, s);
}

moe_status gemm_mx_down(const Layout& L, const void* ws, moe_mxfp8_operand act,
                        const moe_mxfp8_operand& wd, void* ye, cudaStream_t s) {
  const int n_nt = L.H / QN;
  QMaps m{};
  if (!fp8_map(&m.a0, act.q, L.I, L.R, QM) ||
      !fp8_map(&m.b0, wd.q, L.I, static_cast<int64_t>(L.E) * L.H, QN))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.b1 = m.b0;
  QArgs a = q_base(L, ws);
  a.n_nt = n_nt;
  a.kb1 = L.I / QK;
  a.b_rows = L.H;
  a.sfa0 = a.sfa1 = act.s;
  a.sfb0 = a.sfb1 = wd.s;
  a.b_rblocks = static_cast<int64_t>(L.E) * L.H / 128;
  a.ld_out = L.H;
  if (!out_map_bf16(&m.o0, ye, L.H, L.R)) return MOE_ERR_CUDA;
  return q_launch_rows<Q_DOWN>(m, a, s);
}

moe_status gemm_mx_down_dgrad(const Layout& L, const void* ws, moe_mxfp8_operand dye,
                              const moe_mxfp8_operand& wd_t, const void* g, const void* u,
                              void* dg, void* du, cudaStream_t s) {
  const int n_nt = L.I / QN;
  QMaps m{};
  if (!fp8_map(&m.a0, dye.q, L.H, L.R, QM) ||
      !fp8_map(&m.b0, wd_t.q, static_cast<int64_t>(L.E) * L.H, L.I, QN))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.b1 = m.b0;
  QArgs a = q_base(L, ws);
  a.n_nt = n_nt;
  a.kb1 = L.H / QK;
  a.k_exp = L.H;
  a.sfa0 = a.sfa1 = dye.s;
  a.sfb0 = a.sfb1 = wd_t.s;
  a.b_rblocks = L.I / 128;
  a.ld_out = L.I;
  a.in0 = g;
  a.in1 = u;
  if (!out_map_bf16(&m.o0, dg, L.I, L.R) || !out_map_bf16(&m.o1, du, L.I, L.R))
    return MOE_ERR_CUDA;
  return q_launch_rows<Q_DACT>(m, a, s);
}

moe_status gemm_mx_gate_up_dgrad(const Layout& L, const void* ws, moe_mxfp8_operand dg,
                                 moe_mxfp8_operand du, const moe_mxfp8_operand& wg_t,
                                 const moe_mxfp8_operand& wu_t, void* dxe, cudaStream_t s) {
  const int n_nt = L.H / QN;
  QMaps m{};
  if (!fp8_map(&m.a0, dg.q, L.I, L.R, QM) ||
      !fp8_map(&m.a1, du.q, L.I, L.R, QM) ||
      !fp8_map(&m.b0, wg_t.q, static_cast<int64_t>(L.E) * L.I, L.H, QN) ||
      !fp8_map(&m.b1, wu_t.q, static_cast<int64_t>(L.E) * L.I, L.H, QN))
    return MOE_ERR_CUDA;
  QArgs a = q_base(L, ws);
  a.n_nt = n_nt;
  a.kb1 = L.I / QK;
  a.kb2 = L.I / QK;
  a.k_exp = L.I;
  a.sfa0 = dg.s;
  a.sfa1 = du.s;
  a.sfb0 = wg_t.s;
  a.sfb1 = wu_t.s;
  a.b_rblocks = L.H / 128;
  a.ld_out = L.H;
  if (!out_map_bf16(&m.o0, dxe, L.H, L.R)) return MOE_ERR_CUDA;
  return q_launch_rows<Q_DXE>(m, a, s);
}

moe_status gemm_mx_down_wgrad(const Layout& L, const void* ws, moe_mxfp8_operand dye_t,
                              moe_mxfp8_operand act_t, float* dw_down, cudaStream_t s) {
  const int w_nt = L.I / QN;
  QMaps m{};
  if (!fp8_map(&m.a0, dye_t.q, L.R, L.H, QM) ||
      !fp8_map(&m.b0, act_t.q, L.R, L.I, QN))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.b1 = m.b0;
  QArgs a = q_base(L, ws);
  if (launch_expert_order(L, ws, s) != MOE_OK) return MOE_ERR_CUDA;
  a.w_mt = L.H / QM;
  a.w_nt = w_nt;
  a.n_probs = 1;
  a.sfa0 = a.sfa1 = dye_t.s;
  a.sfb0 = a.sfb1 = act_t.s;
  a.a_rblocks = L.H / 128;
  a.b_rblocks = L.I / 128;
  a.ld_out = L.I;
  if (!out_map_f32(&m.o0, dw_down, L.I, static_cast<int64_t>(L.E) * L.H)) return MOE_ERR_CUDA;
  m.o1 = m.o0;
  return q_launch_wgrad<Q_WGRAD>(m, a, s);
}

moe_status gemm_mx_gate_up_wgrad(const Layout& L, const void* ws, moe_mxfp8_operand dg_t,
                                 moe_mxfp8_operand du_t, moe_mxfp8_operand xe_t, float* dw_gate,
                                 float* dw_up, cudaStream_t s) {
  const int w_nt = L.H / QN;
  QMaps m{};
  if (!fp8_map(&m.a0, dg_t.q, L.R, L.I, QM) ||
      !fp8_map(&m.a1, du_t.q, L.R, L.I, QM) ||
      !fp8_map(&m.b0, xe_t.q, L.R, L.H, QN))
    return MOE_ERR_CUDA;
  m.b1 = m.b0;
  QArgs a = q_base(L, ws);
  if (launch_expert_order(L, ws, s) != MOE_OK) return MOE_ERR_CUDA;
  a.w_mt = L.I / QM;
  a.w_nt = w_nt;
  a.n_probs = 2;
  a.sfa0 = dg_t.s;
  a.sfa1 = du_t.s;
  a.sfb0 = a.sfb1 = xe_t.s;
  a.a_rblocks = L.I / 128;
  a.b_rblocks = L.H / 128;
  a.ld_out = L.H;
  if (!out_map_f32(&m.o0, dw_gate, L.H, static_cast<int64_t>(L.E) * L.I) ||
      !out_map_f32(&m.o1, dw_up, L.H, static_cast<int64_t>(L.E) * L.I))
    return MOE_ERR_CUDA;
  return q_launch_wgrad<Q_WGRAD>(m, a, s);
}

}  // namespace moe
