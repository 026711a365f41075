// grouped_gemm.cu -- the expert FFN GEMMs of the layer on the 5th-generation
// tensor cores (tcgen05, accumulators in TMEM), with their epilogues fused.
//
// The expert FFN is a grouped GEMM with a SwiGLU activation (gate/up, then
// silu * mul, then down) run per minibatch of tokens ("Mixture-of-Kittens:
// Cursor open-sources an MoE training megakernel", key points 3 and 5 and the
// key flowchart node "expert FFN + SwiGLU"). The backward rounds (key point
// 2) need the matching data-gradient and weight-gradient GEMMs.
//
// Persistent kernel templates serve the GEMMs of the layer: the SM-pair
// kernel (tcgen05 cta_group::2, further below) runs the four token-row modes
// and the weight gradients, the fused forward kernel runs dispatch, gate/up
// and down in one launch, and the single-CTA kernel runs the router GEMM. In
// each, every CTA (one per SM) runs three roles that hand work over through
// mbarriers:
//   warp 0      TMA producer: streams 64-wide K slices of the A and B tiles
//               into a ring of shared-memory stages (128-byte swizzle);
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=256,
//               K=16) into one of two TMEM accumulators, and commits each
//               stage back to the producer when the tensor core is done;
//   warps 2..5  epilogue: tcgen05.ld the accumulator (one TMEM lane quadrant
//               per warp, one output row per thread), apply the fused
//               epilogue, store to global memory, release the accumulator.
// The two accumulators let the epilogue of tile i overlap the MMAs of tile
// i+1. Every wait is bounded; a timeout records MOE_DEVERR_TIMEOUT, drains
// the copies and MMAs in flight, frees TMEM and returns.
//
// Modes (rows of the expert-grouped buffer are padded per expert to a
// multiple of 128, and padding rows hold zeros, so every tile is a full
// 128-row tile of one expert):
//   GATE_UP  G|U = Xe . [Wg[e]; Wu[e]]^T   -> G, U, Act = silu(G) * U (bf16)
//   DOWN     Ye  = Act . Wd[e]^T            -> bf16
//   DACT     dAct = dYe . Wd[e]             -> dG, dU via the SwiGLU backward (bf16)
//   DXE      dXe = dG . Wg[e] + dU . Wu[e]  -> bf16 (two K phases)
//   WGRAD    dW[e] = P_e^T . Q_e over the expert's rows (K = tokens) -> fp32,
//            for up to two problems per launch (dWg and dWu share Q = Xe).
#include <algorithm>
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "tma_map.h"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, kStages = 4;
constexpr int kABytes = BM * BK * 2;  // 16 KB
constexpr int kBBytes = BN * BK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
// Epilogue staging for TMA stores: per epilogue warp two 32x32 fp32 blocks.
constexpr int kStageOutBytes = 32 * 32 * 4;
constexpr int kOutBytes = 4 * 2 * kStageOutBytes;
constexpr int kSmemBytes = kStages * kStageBytes + kOutBytes + 1024;  // + alignment slack
constexpr int kGemmThreads = 192;
constexpr uint32_t kTmemCols = 512;  // two 256-column fp32 accumulators

// ROUTER: the dense router GEMM in front of the routing, logits = x . Wr^T
// (M tiles over the N tokens, one N tile of up to 256 experts, fp32 out).
enum Mode { GATE_UP = 0, DOWN = 1, DACT = 2, DXE = 3, WGRAD = 4, ROUTER = 6 };

struct Maps {
  CUtensorMap a0, a1, b0, b1;
  CUtensorMap a0h, a1h;    // SM-pair kernels: A with a 64-row box (128-row items)
  CUtensorMap o0, o1, o2;  // outputs (TMA stores): fp32 32x32 or bf16 64x32 boxes, 128-B swizzle
};

struct Args {
  const int32_t* tiles;        // [n][3] (expert, row0, valid) of the 128-row tiles
  const int32_t* n_tiles;      // device count of those tiles
  const int32_t* ptiles;       // [n][3] (expert, row0, rows 256 or 128) SM-pair items
  const int32_t* n_ptiles;     // device count of those items
  const int32_t* pad_offsets;  // [E+1] padded segment starts (WGRAD K ranges)
  const int32_t* order;        // [E] experts by descending row count (WGRAD)
  const int32_t* counts;       // [E] rows per expert (WGRAD K = count rounded up to 64)
  int32_t* err;
  int max_mtiles;              // host bound on *n_tiles (R / 128)
  int64_t rows;                // rows of the expert-grouped buffers (R)
  int n_nt;                    // N tiles per M tile
  int kb1, kb2;                // K blocks of phase 1 and 2
  int b_rows;                  // rows per expert in B's 2-D view
  int E, w_mt, w_nt, n_probs;  // WGRAD tiling
  int ld_out;                  // output row length (elements)
  const int32_t* src_of_row;   // fused reverse-combine: assignment index of each row (-1: padding)
  int k;                       // fused reverse-combine: experts per token
  int store_gu;                // GATE_UP: also store G and U
  int l2_hint;                 // WGRAD: stores evict-first, panel loads evict-last in L2
  void *out0, *out1, *out2;
  const void *in0, *in1;
  // DACT with the reverse-combine fused in (rc_* set): dYe[row] = w[a] * dY[a / k]
  // and dw[a] = <dY[a / k], Ye[row]> for every row (a = src_of_row[row]),
  // claimed by side warps 8 rows at a time through rc_sync[0]; rc_sync[1 + tile]
  // counts the finished rows of each 128-row tile.
  const uint4* rc_dy;
  const uint4* rc_ye;
  const float* rc_w;
  uint4* rc_dye;
  float* rc_dw;
  int32_t* rc_sync;
  int hv;     // H / 8
  int64_t A;  // assignments
};

template <int MODE>
struct Traits {
  static constexpr bool a_mn = (MODE == WGRAD);
  static constexpr bool b_mn = (MODE == DACT || MODE == DXE || MODE == WGRAD);
};

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, int32_t* err) {
  int no_abort = 0;  // drain waits do not stop at the abort flag
  return mbar_wait(bar, parity, &no_abort, err);
}

struct TileInfo {
  int e, row0, mt, nt, prob, kstart, nkb;
  bool skip;
  bool fold;  // SM-pair item of 128 rows: M=128 pair MMA, 64 rows per CTA
};

// Tile t of this CTA. With CL = 2 (the two CTAs of an SM pair), t numbers
// pair tiles and `crank` (the CTA's rank in the pair) picks the member: in
// WGRAD the members take neighbouring M tiles of one expert, which share the
// B tile of the pair MMA.
template <int MODE, int CL>
__device__ __forceinline__ TileInfo decode_tile(const Args& a, int64_t t, int crank) {
  TileInfo ti;
  ti.fold = false;
  if constexpr (MODE == ROUTER) {
    ti.mt = static_cast<int>(t);
    ti.nt = 0;
    ti.row0 = static_cast<int>(t) * BM;  // rows past N are zero-filled loads, clipped stores
    ti.e = 0;
    ti.prob = 0;
    ti.kstart = 0;
    ti.nkb = a.kb1;
    ti.skip = false;
  } else if constexpr (MODE == WGRAD) {
    // Largest experts first, so the CTAs that stream one expert's long K
    // panels start together and share them through L2; within an expert,
    // (mt, nt, problem) with the problem fastest, so dWg and dWu tiles that
    // read the same Xe panel run side by side.
    const int w_mtp = a.w_mt / CL;
    const int64_t per_e = static_cast<int64_t>(w_mtp) * a.w_nt * a.n_probs;
    const int rank = static_cast<int>(t / per_e);
    int64_t r = t % per_e;
    ti.mt = static_cast<int>(r / (a.w_nt * a.n_probs)) * CL + crank;
    r %= (a.w_nt * a.n_probs);
    ti.nt = static_cast<int>(r / a.n_probs);
    ti.prob = static_cast<int>(r % a.n_probs);
    ti.e = a.order[rank];
    if (ti.e < 0 || ti.e >= a.E) ti.e = 0;
    ti.kstart = a.pad_offsets[ti.e];
    // Rows past the count are zero padding up to the segment end, so K stops
    // at the count rounded up to the k-block.
    ti.nkb = (a.counts[ti.e] + BK - 1) / BK;
    if (ti.kstart + ti.nkb * BK > a.pad_offsets[ti.e + 1]) ti.nkb = -1;
    ti.row0 = 0;
    ti.skip = false;
    if (ti.kstart < 0 || ti.nkb < 0 || ti.kstart + static_cast<int64_t>(ti.nkb) * BK > a.rows) {
      ti.nkb = 0;  // corrupt schedule: compute nothing, store nothing
      ti.skip = true;
    }
  } else {
    const int n_ntp = a.n_nt / CL;
    const int mtile = static_cast<int>(t / n_ntp);
    ti.nt = static_cast<int>(t % n_ntp) * CL + crank;
    ti.mt = mtile;
    ti.e = a.tiles[3 * mtile + 0];
    ti.row0 = a.tiles[3 * mtile + 1];
    ti.prob = 0;
    ti.kstart = 0;
    ti.nkb = a.kb1 + a.kb2;
    ti.skip = false;
    if (ti.e < 0 || ti.e >= a.E || ti.row0 < 0 || ti.row0 > a.rows - BM) {
      ti.e = 0;  // corrupt schedule: compute nothing, store nothing
      ti.row0 = 0;
      ti.nkb = 0;
      ti.skip = true;
    }
  }
  return ti;
}

template <int MODE, int CL>
__device__ __forceinline__ int64_t total_tiles(const Args& a) {
  if constexpr (MODE == ROUTER) {
    return a.max_mtiles;
  } else if constexpr (MODE == WGRAD) {
    return static_cast<int64_t>(a.n_probs) * a.E * (a.w_mt / CL) * a.w_nt;
  } else {
    int n = *a.n_tiles;
    n = n < 0 ? 0 : (n > a.max_mtiles ? a.max_mtiles : n);
    return static_cast<int64_t>(n) * (a.n_nt / CL);
  }
}

// Loads of one k-block for the single-CTA kernel (the router GEMM).
template <int MODE>
__device__ __forceinline__ void issue_loads(const Maps& m, const Args& a, const TileInfo& ti,
                                            int kb, uint8_t* sA, uint8_t* sB, uint64_t* bar) {
  static_assert(MODE == ROUTER, "single-CTA kernel modes");
  tma_load_2d(sA, &m.a0, bar, kb * BK, ti.row0);
  tma_load_2d(sB, &m.b0, bar, kb * BK, 0);  // all E router rows; rows past E read as zeros
}

// silu and the sigmoid with the fast exponential and division intrinsics
// (__expf: at most 2 + floor(1.16 |x|) ulp; __fdividef: 2 ulp), far below the
// bf16 rounding of Act, dG and dU; with the IEEE forms the gate/up epilogue's
// arithmetic cost 3% of that GEMM and the down data-gradient epilogue's 5-7%.
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }
__device__ __forceinline__ float sigmoid(float g) { return __fdividef(1.0f, 1.0f + __expf(-g)); }

// One 32-row x 64-column bf16 block of a warp's output: 64 fp32 values per
// thread (its row) -> bf16 -> shared staging buffer (128-byte swizzle: one
// warp store covers all banks) -> one TMA store. NB staging buffers per warp
// let NB - 1 stores be in flight while the next block is staged.
template <int NB>
__device__ __forceinline__ void store_block_bf16(const CUtensorMap* om, const float (&v)[64],
                                                 int32_t x, int32_t y, int lane,
                                                 uint8_t* stage_out, uint32_t& nstore) {
  uint8_t* buf = stage_out + (nstore % NB) * kStageOutBytes;
  if (lane == 0) bulk_wait_read<NB - 1>();  // the store that last used this buffer has read it
  __syncwarp();
  const uint32_t row = smem_u32(buf) + lane * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t addr = row + ((j ^ (lane & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                 "r"(pack_bf16x2(v[8 * j + 0], v[8 * j + 1])),
                 "r"(pack_bf16x2(v[8 * j + 2], v[8 * j + 3])),
                 "r"(pack_bf16x2(v[8 * j + 4], v[8 * j + 5])),
                 "r"(pack_bf16x2(v[8 * j + 6], v[8 * j + 7]))
                 : "memory");
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(om, buf, x, y);
    bulk_commit();
  }
  ++nstore;
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r0[32], r1[32];
  tmem_ld32(taddr, r0);
  tmem_ld32(taddr + 32, r1);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __uint_as_float(r0[i]);
    v[32 + i] = __uint_as_float(r1[i]);
  }
}

// Epilogues of the token-row modes (bf16 outputs), one warp = 32 tile rows:
//   GATE_UP  G, U and Act = silu(G) * U
//   DOWN/DXE the accumulator rounded to bf16
//   DACT     dG, dU from dAct and the saved G, U of the same rows (stored
//            directly: this epilogue also reads G and U, and interleaving those
//            reads with the stores in 32-column steps measured faster)
// The warp's TMEM lanes hold all BN columns of its 32 rows, except in a
// folded SM-pair item (M=128 over two CTAs, 64 rows each): there TMEM lanes
// 0-63 hold D columns [0, BN/2) of the CTA's 64 rows and lanes 64-127 columns
// [BN/2, BN) of the same rows, both in TMEM columns [0, BN/2).
// GATE_UP D column order: single CTA, 128 G then 128 U columns of the N tile;
// SM pair, per half of the N tile (one CTA's B rows) 64 G then 64 U columns.
template <int MODE, bool PAIR, int NB = 2>
__device__ __forceinline__ void epilogue(const Maps& m, const Args& a, const TileInfo& ti,
                                         uint32_t tmem_acc, int quad, int lane,
                                         uint8_t* stage_out, uint32_t& nstore) {
  const uint32_t taddr = tmem_acc + (static_cast<uint32_t>(quad * 32) << 16);
  const int32_t y = ti.row0 + (ti.fold ? (quad & 1) : quad) * 32;
  const int dc0 = ti.fold ? (quad >> 1) * (BN / 2) : 0;  // first D column held
  const int ncol = ti.fold ? BN / 2 : BN;                // D columns held
  if constexpr (MODE == GATE_UP) {
    const int32_t x0 = ti.nt * (BN / 2);
    for (int c = 0; c < ncol / 2; c += 64) {
      float g[64], u[64];
      const int tg = PAIR ? 2 * c : c, tu = PAIR ? 2 * c + 64 : BN / 2 + c;
      const int32_t xo = x0 + (PAIR ? (dc0 + 2 * c) / 2 : c);
      tmem_ld64(taddr + tg, g);
      tmem_ld64(taddr + tu, u);
      if (a.store_gu) {
        store_block_bf16<NB>(&m.o0, g, xo, y, lane, stage_out, nstore);
        store_block_bf16<NB>(&m.o1, u, xo, y, lane, stage_out, nstore);
      }
#pragma unroll
      for (int i = 0; i < 64; ++i) g[i] = silu(g[i]) * u[i];
      store_block_bf16<NB>(&m.o2, g, xo, y, lane, stage_out, nstore);
    }
  } else if constexpr (MODE == DOWN || MODE == DXE) {
    for (int c = 0; c < ncol; c += 64) {
      float d[64];
      tmem_ld64(taddr + c, d);
      store_block_bf16<NB>(&m.o0, d, ti.nt * BN + dc0 + c, y, lane, stage_out, nstore);
    }
  } else {  // DACT: direct 16-byte stores, G and U read alongside in 32-column steps
    const int64_t row = static_cast<int64_t>(y) + lane;
    const int64_t o = row * a.ld_out + ti.nt * BN + dc0;
    for (int c = 0; c < ncol; c += 32) {
      uint32_t d[32];
      tmem_ld32(taddr + c, d);
      const uint4* pg = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.in0) + o + c);
      const uint4* pu = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.in1) + o + c);
      uint4 gv[4], uv[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        gv[v] = pg[v];
        uv[v] = pu[v];
      }
      tmem_ld_wait();
      uint4* pdg = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out0) + o + c);
      uint4* pdu = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out1) + o + c);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint32_t gw[4] = {gv[v].x, gv[v].y, gv[v].z, gv[v].w};
        const uint32_t uw[4] = {uv[v].x, uv[v].y, uv[v].z, uv[v].w};
        uint32_t og[4], ou[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float dg2[2], du2[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float da = __uint_as_float(d[8 * v + 2 * q + h]);
            const float g = h ? bf16hi(gw[q]) : bf16lo(gw[q]);
            const float u = h ? bf16hi(uw[q]) : bf16lo(uw[q]);
            const float sg = sigmoid(g);
            dg2[h] = da * u * sg * (1.0f + g * (1.0f - sg));
            du2[h] = da * g * sg;
          }
          og[q] = pack_bf16x2(dg2[0], dg2[1]);
          ou[q] = pack_bf16x2(du2[0], du2[1]);
        }
        pdg[v] = make_uint4(og[0], og[1], og[2], og[3]);
        pdu[v] = make_uint4(ou[0], ou[1], ou[2], ou[3]);
      }
    }
  }
}

// fp32 epilogue (WGRAD: dW[e] rows; ROUTER: logits): each warp moves its 32
// rows x the first `ncols` (a multiple of 32) of the 256 columns in 32x32
// blocks: TMEM -> registers -> shared staging buffer (the 128-byte swizzle
// spreads one warp store over all banks) -> one TMA store at (x0 + c, y).
// Two staging buffers per warp let the store of block i overlap block i+1.
template <int NB>
__device__ __forceinline__ void epilogue_f32(const CUtensorMap* om, const TileInfo& ti, int32_t x0,
                                             int32_t y, int ncols, uint32_t tmem_acc, int quad,
                                             int lane, uint8_t* stage_out, uint32_t& nstore,
                                             bool hint = false) {
  const uint64_t pol = hint ? l2_evict_first() : 0ull;
  const uint32_t taddr = tmem_acc + (static_cast<uint32_t>(quad * 32) << 16);
  for (int c = 0; c < ncols; c += 32) {
    uint32_t d[32];
    if (ti.nkb > 0) {
      tmem_ld32(taddr + c, d);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int q = 0; q < 32; ++q) d[q] = 0u;
    }
    uint8_t* buf = stage_out + (nstore % NB) * kStageOutBytes;
    if (lane == 0) bulk_wait_read<NB - 1>();  // the store that last used this buffer has read it
    __syncwarp();
    const uint32_t row = smem_u32(buf) + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t addr = row + ((j ^ (lane & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(d[4 * j]),
                   "r"(d[4 * j + 1]), "r"(d[4 * j + 2]), "r"(d[4 * j + 3])
                   : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (hint) tma_store_2d_hint(om, buf, x0 + c, y, pol);
      else tma_store_2d(om, buf, x0 + c, y);
      bulk_commit();
    }
    ++nstore;
  }
}

template <int NB>
__device__ __forceinline__ void epilogue_wgrad(const Maps& m, const Args& a, const TileInfo& ti,
                                               uint32_t tmem_acc, int quad, int lane,
                                               uint8_t* stage_out, uint32_t& nstore) {
  epilogue_f32<NB>(ti.prob ? &m.o1 : &m.o0, ti, ti.nt * BN, ti.e * (a.w_mt * BM) + ti.mt * BM + quad * 32,
                   BN, tmem_acc, quad, lane, stage_out, nstore, a.l2_hint != 0);
}

// Router logits: row block row0 + quad*32, the first E columns (ld_out = E;
// stores clip the rows past N and the columns past E).
__device__ __forceinline__ void epilogue_router(const Maps& m, const Args& a, const TileInfo& ti,
                                                uint32_t tmem_acc, int quad, int lane,
                                                uint8_t* stage_out, uint32_t& nstore) {
  epilogue_f32<2>(&m.o0, ti, 0, ti.row0 + quad * 32, (a.ld_out + 31) / 32 * 32, tmem_acc, quad, lane,
               stage_out, nstore);
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ Maps maps, const Args args) {
  static_assert(MODE == ROUTER, "single-CTA kernel modes");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 128);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a0);
    tma_prefetch_desc(&maps.b0);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  volatile int* abortp = &abort_flag;
  const int64_t total = total_tiles<MODE, 1>(args);
  const int64_t first = blockIdx.x, stride = gridDim.x;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int64_t t = first; t < total && ok; t += stride) {
        const TileInfo ti = decode_tile<MODE, 1>(args, t, 0);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abortp, args.err)) { ok = false; break; }
          uint8_t* sA = smem + stage * kStageBytes;
          mbar_arrive_expect_tx(&full_bar[stage], kStageBytes);
          issue_loads<MODE>(maps, args, ti, kb, sA, sA + kABytes, &full_bar[stage]);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // Every issued copy must land before the CTA may exit.
      for (int s = 0; s < kStages; ++s)
        if ((issued_mask >> s) & 1u) wait_drain(&full_bar[s], (issued_parity >> s) & 1u, args.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = idesc_bf16(BM, BN, Traits<MODE>::a_mn, Traits<MODE>::b_mn);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t t = first; t < total && ok; t += stride) {
        const TileInfo ti = decode_tile<MODE, 1>(args, t, 0);
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abortp, args.err)) break;
        tc_fence_after();
        const uint32_t dtmem = tmem_base + acc * BN;
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abortp, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            uint64_t ad, bd;
            if constexpr (Traits<MODE>::a_mn) ad = sdesc_sw128(a_addr + ks * 2048, 64 * BK * 2, 1024);
            else ad = sdesc_sw128(a_addr + ks * 32, 16, 1024);
            if constexpr (Traits<MODE>::b_mn) bd = sdesc_sw128(b_addr + ks * 2048, 64 * BK * 2, 1024);
            else bd = sdesc_sw128(b_addr + ks * 32, 16, 1024);
            umma_bf16(dtmem, ad, bd, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(&empty_bar[stage]);  // stage free once read
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tfull_bar[acc]);  // accumulator ready (immediate if no MMA)
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      umma_commit(&drain_bar);
      wait_drain(&drain_bar, 0, args.err);
    }
  } else {
    // ---------------- epilogue warps 2..5 ----------------
    const int quad = warp & 3;  // TMEM lanes this warp may access
    uint8_t* stage_out = smem + kStages * kStageBytes + (warp - 2) * 2 * kStageOutBytes;
    uint32_t nstore = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t t = first; t < total; t += stride) {
      const TileInfo ti = decode_tile<MODE, 1>(args, t, 0);
      if (!mbar_wait(&tfull_bar[acc], acc_phase, abortp, args.err)) break;
      tc_fence_after();
      if (ti.skip) {
        if (lane == 0) set_dev_error(args.err, MOE_DEVERR_BAD_EXPERT);
      } else if constexpr (MODE == ROUTER) {
        epilogue_router(maps, args, ti, tmem_base + acc * BN, quad, lane, stage_out, nstore);
      } else {
        epilogue<MODE, false>(maps, args, ti, tmem_base + acc * BN, quad, lane, stage_out, nstore);
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_all();  // stores done before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// SM-pair variant (tcgen05 cta_group::2), used for the weight gradients.
//
// Two CTAs of a cluster compute one 256 x 256 tile of dW[e] with a single MMA
// stream issued by the even CTA: each CTA stages its own 128 A rows and its
// half (128 columns) of the shared B tile, so a k-block costs each SM 32 KB
// of shared-memory fill instead of 48 KB for the same tensor-core work, and
// six stages fit. D rows land in each CTA's own TMEM and each CTA runs its
// own epilogue. Barriers: the even CTA's full[s] counts both CTAs' bytes (the
// odd CTA's copies signal it across the pair); the MMA commits arrive on both
// CTAs' empty[s] and tfull[a]; the odd CTA's epilogue releases the
// accumulator with a remote arrive on the even CTA's tempty[a].
constexpr int kPairStages = 6;  // the fused forward's ring depth; the GEMM kernel takes S
constexpr int kPairABytes = BM * BK * 2;        // 16 KB: this CTA's 128 A rows
constexpr int kPairBBytes = (BN / 2) * BK * 2;  // 16 KB: this CTA's 128 B columns
constexpr int kPairStageBytes = kPairABytes + kPairBBytes;
constexpr int kPairSmemBytes = kPairStages * kPairStageBytes + kOutBytes + 1024;
// Dynamic shared memory of the SM-pair GEMM kernel with S stages.
// Staging buffers per epilogue warp of the SM-pair GEMM kernel with S stages:
// the shared memory the ring leaves free (2, 4 and 6 at 6, 5 and 4 stages;
// 225 KB in every case) goes to more TMA stores in flight.
constexpr int pair_out_bufs(int S) { return S >= 6 ? 2 : (S == 5 ? 4 : 6); }
constexpr int pair_smem_bytes(int S) {
  return S * kPairStageBytes + 4 * pair_out_bufs(S) * kStageOutBytes + 1024;
}
static_assert(pair_smem_bytes(4) <= 227 * 1024 && pair_smem_bytes(5) <= 227 * 1024 &&
                  pair_smem_bytes(6) <= 227 * 1024,
              "SM-pair ring plus staging within the shared memory of one CTA");

// Pair tiles: WGRAD pairs neighbouring M tiles of one expert (shared B); the
// token-row modes take the schedule's SM-pair items (256 rows of one expert,
// 128 rows per CTA; or an expert's last 128 rows, 64 per CTA, as an M=128
// pair MMA) and split the N tile's B rows/columns between the CTAs.
template <int MODE>
__device__ __forceinline__ TileInfo decode_pair_tile(const Args& a, int64_t t, int crank) {
  if constexpr (MODE == WGRAD) {
    return decode_tile<MODE, 2>(a, t, crank);
  } else {
    const int pm = static_cast<int>(t / a.n_nt);
    TileInfo ti;
    ti.e = a.ptiles[3 * pm + 0];
    const int r0 = a.ptiles[3 * pm + 1], nr = a.ptiles[3 * pm + 2];
    ti.fold = nr == BM;
    ti.row0 = r0 + crank * (ti.fold ? BM / 2 : BM);
    ti.mt = pm;
    ti.nt = static_cast<int>(t % a.n_nt);
    ti.prob = 0;
    ti.kstart = 0;
    ti.nkb = a.kb1 + a.kb2;
    ti.skip = false;
    if (ti.e < 0 || ti.e >= a.E || r0 < 0 || (nr != BM && nr != 2 * BM) || r0 > a.rows - nr) {
      ti.e = 0;  // corrupt schedule: compute nothing, store nothing
      ti.row0 = 0;
      ti.nkb = 0;
      ti.skip = true;
      ti.fold = false;
    }
    return ti;
  }
}

template <int MODE>
__device__ __forceinline__ int64_t total_pair_tiles(const Args& a) {
  if constexpr (MODE == WGRAD) {
    return total_tiles<MODE, 2>(a);
  } else {
    int n = *a.n_ptiles;
    n = n < 0 ? 0 : (n > a.max_mtiles ? a.max_mtiles : n);
    return static_cast<int64_t>(n) * a.n_nt;
  }
}

// Reverse-combine fused into the down-dgrad GEMM: side warps claim 8-row
// chunks of the expert-grouped buffer in row order (the order the GEMM's pair
// items consume them) and publish per-tile row counts; the GEMM producer waits
// for its tile's count before loading dYe. Same arithmetic and summation
// order as reverse_combine_kernel (256 threads per token: thread i covers
// vectors i, i + 256, ...; per-warp shuffle trees; warp sums in order).
constexpr int kRcWarps = 4, kRcRows = 8;

__device__ __forceinline__ void reverse_combine_rows(const Args& a, int lane) {
  int32_t* ticket = a.rc_sync;
  int32_t* done = a.rc_sync + 1;
  int64_t rows = a.pad_offsets[a.E];
  rows = rows < 0 ? 0 : (rows > a.rows ? a.rows : rows);
  const int32_t n_chunks = static_cast<int32_t>(rows / kRcRows);
  while (true) {
    int32_t c = 0;
    if (lane == 0) c = atomicAdd(ticket, 1);
    c = __shfl_sync(0xffffffffu, c, 0);
    if (c >= n_chunks) break;
    for (int r = 0; r < kRcRows; ++r) {
      const int64_t row = static_cast<int64_t>(c) * kRcRows + r;
      const int32_t as = a.src_of_row[row];
      uint4* drow = a.rc_dye + row * a.hv;
      if (as < 0 || as >= a.A) {  // padding row
        for (int v = lane; v < a.hv; v += 32) drow[v] = make_uint4(0u, 0u, 0u, 0u);
        continue;
      }
      const float wj = a.rc_w[as];
      const uint4* gy = a.rc_dy + static_cast<int64_t>(as / a.k) * a.hv;
      const uint4* ey = a.rc_ye + row * a.hv;
      float part[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
      for (int base = 0; base < a.hv; base += 256) {
        uint4 gv[8], ev[8];  // all loads of the step first: 16 in flight per lane
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int v = base + 32 * q + lane;
          if (v < a.hv) {
            gv[q] = __ldg(gy + v);
            ev[q] = __ldg(ey + v);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int v = base + 32 * q + lane;
          if (v < a.hv) {
            float g[8], e8[8], sc[8];
            unpack8(gv[q], g);
#pragma unroll
            for (int i = 0; i < 8; ++i) sc[i] = wj * g[i];
            drow[v] = pack8(sc);
            unpack8(ev[q], e8);
#pragma unroll
            for (int i = 0; i < 8; ++i) part[q] = fmaf(g[i], e8[i], part[q]);
          }
        }
      }
      float tot = 0.0f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float p = part[q];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) p += __shfl_down_sync(0xffffffffu, p, off);
        tot += p;
      }
      if (lane == 0) a.rc_dw[as] = tot;
    }
    __syncwarp();
    if (lane == 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");  // rows seen by the TMA loads
      __threadfence();
      atomicAdd(done + (static_cast<int64_t>(c) * kRcRows) / BM, kRcRows);
    }
  }
}

// Bounded wait until *p >= target (acquire), then order the caller's later
// TMA loads after it.
__device__ __forceinline__ bool wait_count(const int32_t* p, int32_t target, volatile int* abort,
                                           int32_t* err) {
  const long long t0 = clock64();
  while (true) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return true;
    }
    if (*abort) return false;
    if (clock64() - t0 > kWaitBudgetCycles) {
      set_dev_error(err, MOE_DEVERR_TIMEOUT);
      *abort = 1;
      return false;
    }
    __nanosleep(100);
  }
}

// Work items of one CTA pair: a run of k-blocks [kb0, kb1) of tile t on
// accumulator acc, `commit` when it ends the tile.
// The producer, the MMA issuer and the epilogue walk the same items.
//  * Token-row modes: whole tiles in order on alternating accumulators.
//  * WGRAD: the tiles, ordered by expert size (largest first), fall into three
//    regions by K: big tiles (more than kWgChunk k-blocks), mid tiles, and
//    light tiles (at most kWgLight k-blocks). A light tile's MMAs are short
//    and its epilogue (a whole fp32 tile of stores) is long, so it can only
//    hide under another tile's MMAs: when the pair has light tiles, it issues
//    each big tile in chunks of kWgChunk k-blocks and, after each chunk but
//    the last, up to kWgPerSlot light tiles on the other accumulator, at the
//    rate that spreads the pair's light tiles evenly over the chunk
//    boundaries of its big tiles. Mid tiles follow, whole, on alternating
//    accumulators, then any light tiles left. Every tile opens on the
//    accumulator whose last tile committed earlier. Chunks do not change a
//    tile's MMA order, so the results are those of whole tiles.
//    Measured on a GB300 (skewed workload, gate/up weight gradient): 2.72-2.74
//    ms against 2.79-2.80 for big and small tiles taken alternately; two light
//    tiles per boundary, or chunks of 12 or 24 k-blocks, were not faster.
constexpr int kWgChunk = 16, kWgLight = 8, kWgPerSlot = 1;

struct PairItem {
  int64_t t;
  int acc, kb0, kb1;
  bool commit;
};

// WGRAD: this pair's share of the three tile regions (one warp computes it in
// both CTAs of the pair before the roles start).
struct WgSplit {
  int64_t big_end, mid_end;  // tile index bounds of the big and mid regions
  int64_t slots;             // chunk boundaries in this pair's big tiles
  int64_t lights;            // this pair's light tiles
};

// K blocks of the expert at rank r of the size order (the expert as the tile
// decode reads it).
__device__ __forceinline__ int wg_rank_nkb(const Args& a, int r) {
  int e = a.order[r];
  if (e < 0 || e >= a.E) e = 0;
  const int c = a.counts[e];
  return c <= 0 ? 0 : (c + BK - 1) / BK;
}

// The first tile at or after t0 that pair p (of P) takes, and how many of
// [lo, hi) it takes.
__device__ __forceinline__ int64_t first_mine(int64_t t0, int64_t p, int64_t P) {
  return t0 <= p ? p : p + ((t0 - p + P - 1) / P) * P;
}
__device__ __forceinline__ int64_t count_mine(int64_t lo, int64_t hi, int64_t p, int64_t P) {
  const int64_t f = first_mine(lo, p, P);
  return f < hi ? (hi - 1 - f) / P + 1 : 0;
}

__device__ __forceinline__ int warp_min_i32(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}
__device__ __forceinline__ int64_t warp_sum_i64(int64_t v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// The regions are cut at the first rank at or below each K bound, so a rank
// order that is not monotone (a corrupt schedule) still covers every tile once.
__device__ void wg_split(const Args& a, int64_t p, int64_t P, int lane, WgSplit* out) {
  const int64_t per_e = static_cast<int64_t>(a.w_mt / 2) * a.w_nt * a.n_probs;
  int rb = a.E, rl = a.E;
  for (int r = lane; r < a.E; r += 32)
    if (wg_rank_nkb(a, r) <= kWgChunk) { rb = r; break; }
  rb = warp_min_i32(rb);
  for (int r = rb + lane; r < a.E; r += 32)
    if (wg_rank_nkb(a, r) <= kWgLight) { rl = r; break; }
  rl = warp_min_i32(rl);
  int64_t slots = 0, lights = 0;
  for (int r = lane; r < a.E; r += 32) {
    const int64_t n = count_mine(r * per_e, (r + 1) * per_e, p, P);
    if (r < rb) slots += n * max((wg_rank_nkb(a, r) + kWgChunk - 1) / kWgChunk - 1, 0);
    else if (r >= rl) lights += n;
  }
  slots = warp_sum_i64(slots);
  lights = warp_sum_i64(lights);
  if (lane == 0) {
    out->big_end = rb * per_e;
    out->mid_end = rl * per_e;
    out->slots = slots;
    out->lights = lights;
  }
}

template <int MODE>
struct PairPlan {
  int64_t fi, total, stride;
  // WGRAD
  WgSplit sp;
  int64_t lcur, used, lit;  // next light tile, chunk boundaries passed, light tiles issued
  int64_t lt;               // open big tile
  TileInfo lti;             // its decoded tile
  int lkb, lnk, la;         // its next k-block, k-blocks, accumulator
  int last;                 // accumulator of the last committed tile
  int pending;              // light tiles to issue at this chunk boundary
  bool has_l;
  __device__ __forceinline__ PairPlan(int64_t first, int64_t stride_, int64_t total_,
                                      const WgSplit* split = nullptr)
      : fi(first), total(total_), stride(stride_), used(0), lit(0), lt(0), lkb(0), lnk(0), la(0),
        last(1), pending(0), has_l(false) {
    if constexpr (MODE == WGRAD) {
      sp = *split;
      lcur = first_mine(sp.mid_end, first, stride_);
    } else {
      sp = WgSplit{0, 0, 0, 0};
      lcur = total_;
    }
  }

  // A whole tile on the accumulator whose last tile committed earlier.
  __device__ __forceinline__ void whole(PairItem& it, TileInfo& ti, const Args& a, int64_t t,
                                        int acc, int crank) {
    it.t = t;
    ti = decode_pair_tile<MODE>(a, t, crank);
    it.acc = acc;
    it.kb0 = 0;
    it.kb1 = ti.nkb;
    it.commit = true;
    last = acc;
  }

  // The next item and its decoded tile (decoded once per tile).
  __device__ __forceinline__ bool next(PairItem& it, TileInfo& ti, const Args& a, int crank) {
    if constexpr (MODE != WGRAD) {
      if (fi >= total) return false;
      whole(it, ti, a, fi, last ^ 1, crank);
      fi += stride;
      return true;
    } else {
      if (pending > 0) {
        if (lcur < total) {  // a light tile beside the open big tile
          whole(it, ti, a, lcur, la ^ 1, crank);
          lcur += stride;
          ++lit;
          --pending;
          return true;
        }
        pending = 0;
      }
      if (!has_l && fi < sp.big_end) {  // open the next big tile
        lt = fi;
        fi += stride;
        lti = decode_pair_tile<MODE>(a, lt, crank);
        lkb = 0;
        lnk = lti.nkb;
        la = last ^ 1;
        has_l = true;
      }
      if (has_l) {
        ti = lti;
        it.t = lt;
        it.acc = la;
        it.kb0 = lkb;
        it.kb1 = sp.lights > 0 ? min(lkb + kWgChunk, lnk) : lnk;
        if (it.kb1 < it.kb0) it.kb1 = it.kb0;
        it.commit = it.kb1 >= lnk;
        lkb = it.kb1;
        if (it.commit) {
          has_l = false;
          last = la;
        } else if (sp.slots > 0) {
          ++used;
          int64_t target = (used * sp.lights + sp.slots - 1) / sp.slots;
          if (target > sp.lights) target = sp.lights;
          const int64_t owe = target - lit;
          pending = owe <= 0 ? 0 : (owe < kWgPerSlot ? static_cast<int>(owe) : kWgPerSlot);
        }
        return true;
      }
      if (fi < sp.mid_end) {  // a mid tile
        whole(it, ti, a, fi, last ^ 1, crank);
        fi += stride;
        return true;
      }
      if (lcur < total) {  // light tiles left over
        whole(it, ti, a, lcur, last ^ 1, crank);
        lcur += stride;
        return true;
      }
      return false;
    }
  }
};

// Token-row modes: this CTA's A rows of k-block kb (both K phases of DXE).
template <int MODE>
__device__ __forceinline__ void load_a_pair(const Maps& m, const Args& a, const TileInfo& ti,
                                            int kb, uint8_t* sA, uint32_t bar) {
  if constexpr (MODE == DXE) {
    const bool second = kb >= a.kb1;
    const CUtensorMap* ma = second ? (ti.fold ? &m.a1h : &m.a1) : (ti.fold ? &m.a0h : &m.a0);
    tma_load_2d_pair(sA, ma, bar, (second ? kb - a.kb1 : kb) * BK, ti.row0);
  } else {
    tma_load_2d_pair(sA, ti.fold ? &m.a0h : &m.a0, bar, kb * BK, ti.row0);
  }
}

// Token-row modes: this CTA's half of the B tile of N tile nt at k-block kb.
template <int MODE>
__device__ __forceinline__ void load_b_pair(const Maps& m, const Args& a, const TileInfo& ti,
                                            int nt, int kb, uint8_t* sB, uint32_t bar,
                                            int crank) {
  if constexpr (MODE == GATE_UP) {
    // the N tile covers 128 gate and 128 up rows of the weights; each CTA
    // stages 64 gate rows then the 64 up rows of the same I columns
    const int brow = ti.e * a.b_rows + nt * (BN / 2) + crank * (BN / 4);
    tma_load_2d_pair(sB, &m.b0, bar, kb * BK, brow);
    tma_load_2d_pair(sB + (BN / 4) * BK * 2, &m.b1, bar, kb * BK, brow);
  } else if constexpr (MODE == DOWN) {
    tma_load_2d_pair(sB, &m.b0, bar, kb * BK, ti.e * a.b_rows + nt * BN + crank * (BN / 2));
  } else {  // DACT, DXE: B is MN-major, two 64-column chunks per CTA
    const bool second = (MODE == DXE) && kb >= a.kb1;
    const int kk = second ? kb - a.kb1 : kb;
    const CUtensorMap* mb = second ? &m.b1 : &m.b0;
#pragma unroll
    for (int c = 0; c < BN / 128; ++c)
      tma_load_2d_pair(sB + c * (64 * BK * 2), mb, bar, nt * BN + crank * (BN / 2) + c * 64,
                       ti.e * a.b_rows + kk * BK);
  }
}

template <int MODE>
__device__ __forceinline__ void issue_loads_pair(const Maps& m, const Args& a, const TileInfo& ti,
                                                 int kb, uint8_t* sA, uint8_t* sB, uint32_t bar,
                                                 int crank) {
  if constexpr (MODE == WGRAD) {
    const CUtensorMap* ma = ti.prob ? &m.a1 : &m.a0;
    const CUtensorMap* mb = ti.prob ? &m.b1 : &m.b0;
    const int krow = ti.kstart + kb * BK;
    if (a.l2_hint) {
      const uint64_t pol = l2_evict_last();
#pragma unroll
      for (int c = 0; c < BM / 64; ++c)
        tma_load_2d_pair_hint(sA + c * (64 * BK * 2), ma, bar, ti.mt * BM + c * 64, krow, pol);
#pragma unroll
      for (int c = 0; c < BN / 128; ++c)
        tma_load_2d_pair_hint(sB + c * (64 * BK * 2), mb, bar, ti.nt * BN + crank * (BN / 2) + c * 64,
                              krow, pol);
    } else {
#pragma unroll
      for (int c = 0; c < BM / 64; ++c)
        tma_load_2d_pair(sA + c * (64 * BK * 2), ma, bar, ti.mt * BM + c * 64, krow);
#pragma unroll
      for (int c = 0; c < BN / 128; ++c)
        tma_load_2d_pair(sB + c * (64 * BK * 2), mb, bar, ti.nt * BN + crank * (BN / 2) + c * 64,
                         krow);
    }
  } else {
    load_a_pair<MODE>(m, a, ti, kb, sA, bar);
    load_b_pair<MODE>(m, a, ti, ti.nt, kb, sB, bar, crank);
  }
}

// S: stages of the shared-memory ring (4, 5 or 6; the per-shape choice of
// pick_stages below).
template <int MODE, bool RC, int S>
__global__ void __launch_bounds__(kGemmThreads + (RC ? 32 * kRcWarps : 0), 1)
    grouped_gemm_pair_kernel(const __grid_constant__ Maps maps, const Args args) {
  static_assert(!RC || MODE == DACT, "the reverse-combine is fused into DACT only");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[S], empty_bar[S], tfull_bar[2], tempty_bar[2],
      drain_bar;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = static_cast<int>(cluster_ctarank());
  const bool leader = crank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 8);  // one arrive per epilogue warp of both CTAs
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a0);
    tma_prefetch_desc(&maps.b0);
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_slot, kTmemCols);  // one warp of each CTA, collectively
    tmem_relinquish_pair();
  }
  const int64_t first = blockIdx.x / 2, stride = gridDim.x / 2;
  __shared__ WgSplit wsplit;
  if constexpr (MODE == WGRAD) {
    if (warp == 2) wg_split(args, first, stride, lane, &wsplit);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  volatile int* abortp = &abort_flag;
  const int64_t total = total_pair_tiles<MODE>(args);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      PairItem it;
      TileInfo ti;
      for (PairPlan<MODE> plan(first, stride, total, &wsplit); ok && plan.next(it, ti, args, crank);) {
        if constexpr (RC) {  // this CTA's dYe rows come from the side warps
          if (ti.nkb > 0 && !wait_count(args.rc_sync + 1 + ti.row0 / BM, BM, abortp, args.err)) {
            ok = false;
            break;
          }
        }
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abortp, args.err)) { ok = false; break; }
          uint8_t* sA = smem + stage * kPairStageBytes;
          // both CTAs' copies: A (64 rows each in a folded item) and half of B
          if (leader)
            mbar_arrive_expect_tx(&full_bar[stage],
                                  2 * ((ti.fold ? kPairABytes / 2 : kPairABytes) + kPairBBytes));
          issue_loads_pair<MODE>(maps, args, ti, kb, sA, sA + kPairABytes,
                                 cluster_addr(&full_bar[stage], 0), crank);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (leader)  // the even CTA's full barriers count both CTAs' copies
        for (int s = 0; s < S; ++s)
          if ((issued_mask >> s) & 1u) wait_drain(&full_bar[s], (issued_parity >> s) & 1u, args.err);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (even CTA only) ----------------
      constexpr uint32_t idesc256 = idesc_bf16(2 * BM, BN, Traits<MODE>::a_mn, Traits<MODE>::b_mn);
      constexpr uint32_t idesc128 = idesc_bf16(BM, BN, Traits<MODE>::a_mn, Traits<MODE>::b_mn);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t uses0 = 0u, uses1 = 0u;  // tiles committed on each accumulator
      bool ok = true;
      PairItem it;
      TileInfo ti;
      for (PairPlan<MODE> plan(first, stride, total, &wsplit); ok && plan.next(it, ti, args, crank);) {
        const int acc = it.acc;
        if (it.kb0 == 0) {  // a new tile: its accumulator's last tile has been read out
          if (!mbar_wait(&tempty_bar[acc], ((acc ? uses1 : uses0) & 1u) ^ 1u, abortp, args.err))
            break;
          tc_fence_after();
        }
        const uint32_t dtmem = tmem_base + acc * BN;
        const uint32_t idesc = ti.fold ? idesc128 : idesc256;
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abortp, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kPairStageBytes);
          const uint32_t b_addr = a_addr + kPairABytes;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            uint64_t ad, bd;
            if constexpr (Traits<MODE>::a_mn) ad = sdesc_sw128(a_addr + ks * 2048, 64 * BK * 2, 1024);
            else ad = sdesc_sw128(a_addr + ks * 32, 16, 1024);
            if constexpr (Traits<MODE>::b_mn) bd = sdesc_sw128(b_addr + ks * 2048, 64 * BK * 2, 1024);
            else bd = sdesc_sw128(b_addr + ks * 32, 16, 1024);
            umma_bf16_pair(dtmem, ad, bd, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit_pair_mc(&empty_bar[stage], 0x3);  // both CTAs may refill the stage
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (it.commit) {
          umma_commit_pair_mc(&tfull_bar[acc], 0x3);  // both halves of the tile are ready
          if (acc) ++uses1; else ++uses0;
        }
      }
      umma_commit_pair(&drain_bar);
      wait_drain(&drain_bar, 0, args.err);
    }
  } else if (warp >= 6) {
    // ---------------- reverse-combine side warps 6.. (fused DACT only) ----------------
    if constexpr (RC) reverse_combine_rows(args, lane);
  } else {
    // ---------------- epilogue warps 2..5 (both CTAs) ----------------
    const int quad = warp & 3;
    constexpr int NB = pair_out_bufs(S);
    uint8_t* stage_out = smem + S * kPairStageBytes + (warp - 2) * NB * kStageOutBytes;
    uint32_t nstore = 0;
    uint32_t uses0 = 0u, uses1 = 0u;
    PairItem it;
    TileInfo ti;
    for (PairPlan<MODE> plan(first, stride, total, &wsplit); plan.next(it, ti, args, crank);) {
      if (!it.commit) continue;
      const int acc = it.acc;
      if (!mbar_wait(&tfull_bar[acc], (acc ? uses1 : uses0) & 1u, abortp, args.err)) break;
      tc_fence_after();
      if (ti.skip) {
        if (lane == 0) set_dev_error(args.err, MOE_DEVERR_BAD_EXPERT);
      } else if constexpr (MODE == WGRAD) {
        epilogue_wgrad<NB>(maps, args, ti, tmem_base + acc * BN, quad, lane, stage_out, nstore);
      } else {
        epilogue<MODE, true, NB>(maps, args, ti, tmem_base + acc * BN, quad, lane, stage_out,
                                 nstore);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&tempty_bar[acc]);
        else mbar_arrive_cluster(cluster_addr(&tempty_bar[acc], 0));
      }
      if (acc) ++uses1; else ++uses0;
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the even CTA's MMAs into this CTA's TMEM have retired
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
  cluster_sync();  // no CTA leaves while its peer may still signal it
}

// ---------------------------------------------------------------------------
// Wide SM-pair tiles for the token-row modes: each unit of work is one pair
// item and TWO neighbouring N tiles (256 x 512 per pair, 128 x 512 per CTA).
// A k-block's A rows are staged once and feed two pair MMAs (N = 256 each)
// into TMEM columns [0, 256) and [256, 512): per unit of MMA work each SM
// stages 24 KB instead of 32, and the GEMMs are bound by the bytes an SM
// moves through its L2 interface. The whole TMEM is one accumulator, so the
// MMAs of the next unit start after the epilogue has read this one out; the
// producer keeps the ring filled meanwhile. Each 256-column block gets the
// same MMAs in the same order as a narrow tile, so the results are
// bit-identical.
constexpr int kWideStageBytes = kPairABytes + 2 * kPairBBytes;  // 48 KB
constexpr int wide_smem_bytes(int S) { return S * kWideStageBytes + kOutBytes + 1024; }
static_assert(wide_smem_bytes(4) <= 227 * 1024, "wide ring within one CTA's shared memory");

template <int MODE>
__device__ __forceinline__ int64_t total_wide_units(const Args& a) {
  int n = *a.n_ptiles;
  n = n < 0 ? 0 : (n > a.max_mtiles ? a.max_mtiles : n);
  return static_cast<int64_t>(n) * (a.n_nt / 2);
}

// The first (lower) of the unit's two N tiles, as decode_pair_tile gives it.
template <int MODE>
__device__ __forceinline__ TileInfo decode_wide_unit(const Args& a, int64_t u, int crank) {
  const int64_t pm = u / (a.n_nt / 2);
  const int nt = static_cast<int>(u % (a.n_nt / 2)) * 2;
  return decode_pair_tile<MODE>(a, pm * a.n_nt + nt, crank);
}

template <int MODE, int S>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_wide_kernel(const __grid_constant__ Maps maps, const Args args) {
  static_assert(MODE == GATE_UP || MODE == DOWN || MODE == DACT || MODE == DXE,
                "wide tiles serve the token-row modes");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[S], empty_bar[S], tfull_bar, tempty_bar, drain_bar;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = static_cast<int>(cluster_ctarank());
  const bool leader = crank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&tfull_bar, 1);
    mbar_init(&tempty_bar, 8);  // one arrive per epilogue warp of both CTAs
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.a0);
    tma_prefetch_desc(&maps.b0);
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_slot, kTmemCols);  // one warp of each CTA, collectively
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  volatile int* abortp = &abort_flag;
  const int64_t total = total_wide_units<MODE>(args);
  const int64_t first = blockIdx.x / 2, stride = gridDim.x / 2;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int64_t u = first; u < total && ok; u += stride) {
        const TileInfo ti = decode_wide_unit<MODE>(args, u, crank);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abortp, args.err)) { ok = false; break; }
          uint8_t* sA = smem + stage * kWideStageBytes;
          const uint32_t bar = cluster_addr(&full_bar[stage], 0);
          if (leader)
            mbar_arrive_expect_tx(&full_bar[stage],
                                  2 * ((ti.fold ? kPairABytes / 2 : kPairABytes) + 2 * kPairBBytes));
          load_a_pair<MODE>(maps, args, ti, kb, sA, bar);
          load_b_pair<MODE>(maps, args, ti, ti.nt, kb, sA + kPairABytes, bar, crank);
          load_b_pair<MODE>(maps, args, ti, ti.nt + 1, kb, sA + kPairABytes + kPairBBytes, bar,
                            crank);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (leader)  // the even CTA's full barriers count both CTAs' copies
        for (int s = 0; s < S; ++s)
          if ((issued_mask >> s) & 1u) wait_drain(&full_bar[s], (issued_parity >> s) & 1u, args.err);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (even CTA only) ----------------
      constexpr uint32_t idesc256 = idesc_bf16(2 * BM, BN, false, Traits<MODE>::b_mn);
      constexpr uint32_t idesc128 = idesc_bf16(BM, BN, false, Traits<MODE>::b_mn);
      int stage = 0;
      uint32_t phase = 0, uses = 0;
      bool ok = true;
      for (int64_t u = first; u < total && ok; u += stride) {
        const TileInfo ti = decode_wide_unit<MODE>(args, u, crank);
        if (!mbar_wait(&tempty_bar, (uses & 1u) ^ 1u, abortp, args.err)) break;
        tc_fence_after();
        const uint32_t idesc = ti.fold ? idesc128 : idesc256;
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abortp, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kWideStageBytes);
          const uint32_t b_addr = a_addr + kPairABytes;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            const uint64_t ad = sdesc_sw128(a_addr + ks * 32, 16, 1024);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t bh = b_addr + h * kPairBBytes;
              uint64_t bd;
              if constexpr (Traits<MODE>::b_mn) bd = sdesc_sw128(bh + ks * 2048, 64 * BK * 2, 1024);
              else bd = sdesc_sw128(bh + ks * 32, 16, 1024);
              umma_bf16_pair(tmem_base + h * BN, ad, bd, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
            }
          }
          umma_commit_pair_mc(&empty_bar[stage], 0x3);  // both CTAs may refill the stage
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair_mc(&tfull_bar, 0x3);  // both halves of the unit are ready
        ++uses;
      }
      umma_commit_pair(&drain_bar);
      wait_drain(&drain_bar, 0, args.err);
    }
  } else {
    // ---------------- epilogue warps 2..5 (both CTAs) ----------------
    const int quad = warp & 3;
    uint8_t* stage_out = smem + S * kWideStageBytes + (warp - 2) * 2 * kStageOutBytes;
    uint32_t nstore = 0, uses = 0;
    for (int64_t u = first; u < total; u += stride) {
      TileInfo ti = decode_wide_unit<MODE>(args, u, crank);
      if (!mbar_wait(&tfull_bar, uses & 1u, abortp, args.err)) break;
      tc_fence_after();
      if (ti.skip) {
        if (lane == 0) set_dev_error(args.err, MOE_DEVERR_BAD_EXPERT);
      } else {
        epilogue<MODE, true>(maps, args, ti, tmem_base, quad, lane, stage_out, nstore);
        ++ti.nt;
        epilogue<MODE, true>(maps, args, ti, tmem_base + BN, quad, lane, stage_out, nstore);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&tempty_bar);
        else mbar_arrive_cluster(cluster_addr(&tempty_bar, 0));
      }
      ++uses;
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the even CTA's MMAs into this CTA's TMEM have retired
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
  cluster_sync();  // no CTA leaves while its peer may still signal it
}

// ---------------------------------------------------------------------------
// Fused forward: dispatch, gate/up + SwiGLU and down in one persistent launch
// ("Mixture-of-Kittens: Cursor open-sources an MoE training megakernel", key
// point 5 and the key flowchart: a producer pulls a minibatch of token rows,
// local counters wake the expert FFN, which runs gate/up, SwiGLU and down).
//
// On one GPU the pull dispatch is an HBM copy, done by side warps of every
// CTA: they claim 8-row chunks of the expert-grouped buffer in row order
// through a ticket, copy each row's token from x (zero rows for padding) and
// count the finished rows of each 128-row tile. The SM-pair GEMM roles walk
// one list of units: every pair item (256 rows of one expert, or its last 128)
// contributes G gate/up units (one per 128 I columns of gate and up) and D
// down units (one per 256 H columns), the down units of item p placed `lag`
// items after its gate/up units. A gate/up unit's producer waits (bounded)
// until the rows of its tile are dispatched; a down unit's producer waits
// until all G gate/up units of its item have stored Act (each epilogue warp
// counts its stores once they have landed). Every unit depends only on units
// earlier in the list and on the dispatch, which waits on nothing, and the
// grid holds only co-resident CTA pairs, so every wait is satisfied in time.
// The arithmetic of each tile is that of the separate gate/up and down
// launches (same MMAs in the same order, same epilogues), so the results are
// bit-identical to dispatch + gate/up + down.
//
// Ring mode (the context-free forward, which keeps neither Xe nor Act): Xe
// and Act live in a ring of `ring` minibatch slots of 256 rows, item p in
// slot p % ring, instead of in buffers of all R rows, so the forward's
// working set is ring * 256 * (H + I) * 2 bytes whatever N is, and stays in
// L2. The dispatch side warps claim 8-row chunks item by item; before
// copying into item p's slot they wait until the G gate/up units of item
// p - ring are done (so their Xe loads have landed). Before storing item p's
// Act, a gate/up epilogue waits until the D down units of item p - ring have
// started their epilogues (so their Act loads have landed). ring > lag puts
// those down units earlier in the list than the gate/up units that wait for
// them, so every wait is still on earlier work or on the dispatch of earlier
// items.
constexpr int kFfDispWarps = 4;
constexpr int kRingSpare = 4;  // ring slots beyond the lag

struct FusedArgs {
  const uint4* x;            // token rows [N][H/8]
  uint4* xe;                 // expert-grouped rows [R][H/8]
  const int32_t* src_of_row;  // assignment of each row, -1 on padding
  const int32_t* pad_offsets;
  int32_t* ticket;           // dispatch chunk ticket
  int32_t* disp_done;        // [R/128] rows dispatched per 128-row tile
  int32_t* gu_done;          // [R/128] finished gate/up epilogue-warp units per item
  int32_t* dn_done;          // [R/128] ring mode: down epilogue-warp units started per item
  const int32_t* ptiles;     // ring mode: the pair items (expert, row0, rows)
  int64_t A, rows;
  int E, k, hv;
  int G, D, lag;             // units per item (gate/up, down); item lag of the down units
  int ring;                  // slots of the Xe and Act rings (0: buffers of all R rows)
};

// First row of this CTA's part of item p in the ring.
__device__ __forceinline__ int32_t ring_row(const FusedArgs& f, int p, int crank, bool fold) {
  return (p % f.ring) * (2 * BM) + crank * (fold ? BM / 2 : BM);
}

// A bounded wait that every lane of the warp leaves together: lane 0 polls,
// then every lane acquires the counter itself.
__device__ __forceinline__ bool warp_wait_count(const int32_t* p, int32_t target, volatile int* abort,
                                                int32_t* err, int lane) {
  int ok = 1;
  if (lane == 0) ok = wait_count(p, target, abort, err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) {
    asm volatile("{\n\t.reg .b32 v;\n\tld.acquire.gpu.global.b32 v, [%0];\n\t}" ::"l"(p) : "memory");
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  return ok != 0;
}

struct FusedUnit {
  bool valid, down;
  int item, nt;
};

__device__ __forceinline__ FusedUnit fused_unit(const FusedArgs& f, int64_t u, int n_items) {
  const int per = f.G + f.D;
  const int64_t step = u / per;
  const int r = static_cast<int>(u % per);
  FusedUnit x;
  x.down = r >= f.G;
  x.nt = x.down ? r - f.G : r;
  const int64_t item = x.down ? step - f.lag : step;
  x.valid = item >= 0 && item < n_items;
  x.item = x.valid ? static_cast<int>(item) : 0;
  return x;
}

// One row of the dispatch: drow = x[src_of_row[row] / k], or zeros on padding.
__device__ __forceinline__ void copy_token_row(const FusedArgs& f, int64_t row, uint4* drow,
                                               int lane) {
  const int32_t as = f.src_of_row[row];
  if (as < 0 || as >= f.A) {
    for (int v = lane; v < f.hv; v += 32) drow[v] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* srow = f.x + static_cast<int64_t>(as / f.k) * f.hv;
  for (int base = 0; base < f.hv; base += 256) {
    uint4 v8[8];  // all loads of the step first: 8 in flight per lane
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int v = base + 32 * q + lane;
      if (v < f.hv) v8[q] = __ldg(srow + v);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int v = base + 32 * q + lane;
      if (v < f.hv) drow[v] = v8[q];
    }
  }
}

// Dispatch side warps: xe[row] = x[src_of_row[row] / k], padding rows 0.
// They claim chunks from the front as fast as they can: making them wait for
// the gate/up progress (a bounded window of items ahead, so rows are still in
// L2 when read) measured slower, the producers then waiting for rows.
__device__ __forceinline__ void dispatch_rows(const FusedArgs& f, int lane) {
  int64_t rows = f.pad_offsets[f.E];
  rows = rows < 0 ? 0 : (rows > f.rows ? f.rows : rows);
  const int32_t n_chunks = static_cast<int32_t>(rows / kRcRows);
  while (true) {
    int32_t c = 0;
    if (lane == 0) c = atomicAdd(f.ticket, 1);
    c = __shfl_sync(0xffffffffu, c, 0);
    if (c >= n_chunks) break;
    for (int r = 0; r < kRcRows; ++r) {
      const int64_t row = static_cast<int64_t>(c) * kRcRows + r;
      copy_token_row(f, row, f.xe + row * f.hv, lane);
    }
    __syncwarp();
    if (lane == 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");  // rows seen by the TMA loads
      __threadfence();
      atomicAdd(f.disp_done + (static_cast<int64_t>(c) * kRcRows) / BM, kRcRows);
    }
  }
}

// Ring mode: the same copies into the ring, item by item (32 chunks of 8
// rows per slot; a 128-row item fills half of its slot). Rows of a corrupt
// item are not copied: the GEMM roles skip that item.
__device__ __forceinline__ void dispatch_ring(const FusedArgs& f, int n_items, int lane,
                                              volatile int* abort, int32_t* err) {
  constexpr int kChunks = 2 * BM / kRcRows;
  const int64_t n_chunks = static_cast<int64_t>(n_items) * kChunks;
  int freed = -1;  // the last item whose slot this warp has seen free
  while (true) {
    int32_t c = 0;
    if (lane == 0) c = atomicAdd(f.ticket, 1);
    c = __shfl_sync(0xffffffffu, c, 0);
    if (c >= n_chunks) break;
    const int p = c / kChunks, q = c % kChunks;
    const int r0 = f.ptiles[3 * p + 1], nr = f.ptiles[3 * p + 2];
    if ((nr != BM && nr != 2 * BM) || r0 < 0 || r0 > f.rows - nr) continue;
    if (q * kRcRows >= nr) continue;
    if (p >= f.ring && p != freed) {
      if (!warp_wait_count(f.gu_done + (p - f.ring), 8 * f.G, abort, err, lane)) break;
      freed = p;
    }
    uint4* slot = f.xe + (static_cast<int64_t>(p % f.ring) * (2 * BM) + q * kRcRows) * f.hv;
    for (int r = 0; r < kRcRows; ++r)
      copy_token_row(f, static_cast<int64_t>(r0) + q * kRcRows + r, slot + r * f.hv, lane);
    __syncwarp();
    if (lane == 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");  // rows seen by the TMA loads
      __threadfence();
      atomicAdd(f.disp_done + (r0 + q * kRcRows) / BM, kRcRows);
    }
  }
}

__device__ __forceinline__ TileInfo fused_tile(const FusedArgs& f, const Args& gu, const Args& dn,
                                               const FusedUnit& fu, int crank) {
  return fu.down ? decode_pair_tile<DOWN>(dn, static_cast<int64_t>(fu.item) * dn.n_nt + fu.nt, crank)
                 : decode_pair_tile<GATE_UP>(gu, static_cast<int64_t>(fu.item) * gu.n_nt + fu.nt,
                                             crank);
}

__global__ void __launch_bounds__(kGemmThreads + 32 * kFfDispWarps, 1)
    fused_forward_kernel(const __grid_constant__ Maps mgu, const __grid_constant__ Maps mdn,
                         const Args gu, const Args dn, const FusedArgs f) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kPairStages], empty_bar[kPairStages], tfull_bar[2], tempty_bar[2],
      drain_bar;
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = static_cast<int>(cluster_ctarank());
  const bool leader = crank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 8);  // one arrive per epilogue warp of both CTAs
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mgu.a0);
    tma_prefetch_desc(&mgu.b0);
    tma_prefetch_desc(&mdn.a0);
    tma_prefetch_desc(&mdn.b0);
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_slot, kTmemCols);  // one warp of each CTA, collectively
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  volatile int* abortp = &abort_flag;
  int n_items = *gu.n_ptiles;
  n_items = n_items < 0 ? 0 : (n_items > gu.max_mtiles ? gu.max_mtiles : n_items);
  const int64_t total = static_cast<int64_t>(n_items + f.lag) * (f.G + f.D);
  const int64_t first = blockIdx.x / 2, stride = gridDim.x / 2;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int64_t u = first; u < total && ok; u += stride) {
        const FusedUnit fu = fused_unit(f, u, n_items);
        if (!fu.valid) continue;
        TileInfo ti = fused_tile(f, gu, dn, fu, crank);
        if (ti.nkb > 0) {
          const bool ready = fu.down ? wait_count(f.gu_done + fu.item, 8 * f.G, abortp, gu.err)
                                     : wait_count(f.disp_done + ti.row0 / BM, BM, abortp, gu.err);
          if (!ready) break;
        }
        if (f.ring > 0) ti.row0 = ring_row(f, fu.item, crank, ti.fold);  // A rows: the ring slot
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abortp, gu.err)) { ok = false; break; }
          uint8_t* sA = smem + stage * kPairStageBytes;
          if (leader)
            mbar_arrive_expect_tx(&full_bar[stage],
                                  2 * ((ti.fold ? kPairABytes / 2 : kPairABytes) + kPairBBytes));
          if (fu.down)
            issue_loads_pair<DOWN>(mdn, dn, ti, kb, sA, sA + kPairABytes,
                                   cluster_addr(&full_bar[stage], 0), crank);
          else
            issue_loads_pair<GATE_UP>(mgu, gu, ti, kb, sA, sA + kPairABytes,
                                      cluster_addr(&full_bar[stage], 0), crank);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kPairStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (leader)  // the even CTA's full barriers count both CTAs' copies
        for (int s = 0; s < kPairStages; ++s)
          if ((issued_mask >> s) & 1u) wait_drain(&full_bar[s], (issued_parity >> s) & 1u, gu.err);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (even CTA only) ----------------
      constexpr uint32_t idesc256 = idesc_bf16(2 * BM, BN, false, false);
      constexpr uint32_t idesc128 = idesc_bf16(BM, BN, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t uses0 = 0u, uses1 = 0u;
      bool ok = true;
      for (int64_t u = first; u < total && ok; u += stride) {
        const FusedUnit fu = fused_unit(f, u, n_items);
        if (!fu.valid) continue;
        const TileInfo ti = fused_tile(f, gu, dn, fu, crank);
        if (!mbar_wait(&tempty_bar[acc], ((acc ? uses1 : uses0) & 1u) ^ 1u, abortp, gu.err)) break;
        tc_fence_after();
        const uint32_t dtmem = tmem_base + acc * BN;
        const uint32_t idesc = ti.fold ? idesc128 : idesc256;
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abortp, gu.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kPairStageBytes);
          const uint32_t b_addr = a_addr + kPairABytes;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            umma_bf16_pair(dtmem, sdesc_sw128(a_addr + ks * 32, 16, 1024),
                           sdesc_sw128(b_addr + ks * 32, 16, 1024), idesc, (kb > 0 || ks > 0) ? 1u : 0u);
          umma_commit_pair_mc(&empty_bar[stage], 0x3);  // both CTAs may refill the stage
          if (++stage == kPairStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair_mc(&tfull_bar[acc], 0x3);  // both halves of the tile are ready
        if (acc) ++uses1; else ++uses0;
        acc ^= 1;
      }
      umma_commit_pair(&drain_bar);
      wait_drain(&drain_bar, 0, gu.err);
    }
  } else if (warp >= 6) {
    // ---------------- dispatch side warps 6.. ----------------
    if (f.ring > 0) dispatch_ring(f, n_items, lane, abortp, gu.err);
    else dispatch_rows(f, lane);
  } else {
    // ---------------- epilogue warps 2..5 (both CTAs) ----------------
    const int quad = warp & 3;
    uint8_t* stage_out = smem + kPairStages * kPairStageBytes + (warp - 2) * 2 * kStageOutBytes;
    uint32_t nstore = 0;
    int acc = 0;
    uint32_t uses0 = 0u, uses1 = 0u;
    for (int64_t u = first; u < total; u += stride) {
      const FusedUnit fu = fused_unit(f, u, n_items);
      if (!fu.valid) continue;
      TileInfo ti = fused_tile(f, gu, dn, fu, crank);
      if (!mbar_wait(&tfull_bar[acc], (acc ? uses1 : uses0) & 1u, abortp, gu.err)) break;
      tc_fence_after();
      if (f.ring > 0 && fu.down && lane == 0) {  // the tile's MMAs are done: its Act loads have landed
        __threadfence();
        atomicAdd(f.dn_done + fu.item, 1);
      }
      if (ti.skip) {
        if (lane == 0) set_dev_error(gu.err, MOE_DEVERR_BAD_EXPERT);
      } else if (fu.down) {
        epilogue<DOWN, true>(mdn, dn, ti, tmem_base + acc * BN, quad, lane, stage_out, nstore);
      } else {
        if (f.ring > 0) {  // Act goes to the item's ring slot, once the slot's last reader is done
          ti.row0 = ring_row(f, fu.item, crank, ti.fold);
          if (fu.item >= f.ring &&
              !warp_wait_count(f.dn_done + (fu.item - f.ring), 8 * f.D, abortp, gu.err, lane))
            break;
        }
        epilogue<GATE_UP, true>(mgu, gu, ti, tmem_base + acc * BN, quad, lane, stage_out, nstore);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&tempty_bar[acc]);
        else mbar_arrive_cluster(cluster_addr(&tempty_bar[acc], 0));
        if (!fu.down) {  // this warp's Act rows are in global memory: count them
          bulk_wait_all();
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __threadfence();
          atomicAdd(f.gu_done + fu.item, 1);
        }
      }
      if (acc) ++uses1; else ++uses0;
      acc ^= 1;
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the even CTA's MMAs into this CTA's TMEM have retired
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
  cluster_sync();  // no CTA leaves while its peer may still signal it
}

// Experts ranked by row count, descending; equal counts keep ascending
// expert index. One CTA; each thread ranks its experts against all others.
__global__ void __launch_bounds__(1024) expert_order_kernel(const int32_t* __restrict__ counts,
                                                            int E, int32_t* __restrict__ order) {
  __shared__ int32_t cnt[kMaxE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = counts[e];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int32_t c = cnt[e];
    int rank = 0;
    for (int f = 0; f < E; ++f) rank += (cnt[f] > c) || (cnt[f] == c && f < e);
    order[rank] = e;
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launches.

// 2-D view [outer][inner] (inner contiguous) of `elem`-byte elements, box
// box_inner x box_outer, 128-byte swizzle. Returns false on failure.
bool make_map(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int box_outer,
              int box_inner = 64, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              int elem = 2) {
  return tma_map_2d(m, base, inner, outer, box_outer, box_inner, dtype, elem);
}

// bf16 output [rows][cols] for the token-row TMA-store epilogues.
bool make_bf16_out_map(CUtensorMap* m, const void* base, int64_t cols, int64_t rows) {
  return make_map(m, base, cols, rows, 32, 64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2);
}

// fp32 weight-gradient output [rows][cols] for the WGRAD TMA-store epilogue.
bool make_out_map(CUtensorMap* m, const float* base, int64_t cols, int64_t rows) {
  return make_map(m, base, cols, rows, 32, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4);
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

// Launch the single-CTA kernel as a persistent grid: one CTA per SM,
// capped by the tiles available.
template <int MODE>
moe_status launch(const Maps& maps, const Args& args, int64_t units, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return MOE_ERR_CUDA;
  if (units <= 0) return MOE_OK;
  const int grid = static_cast<int>(std::min<int64_t>(sm_count(), units));
  grouped_gemm_kernel<MODE><<<grid, kGemmThreads, kSmemBytes, s>>>(maps, args);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <int MODE, bool RC, int S>
moe_status launch_pair_s(const Maps& maps, const Args& args, int64_t units, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;
  auto config = [](cudaLaunchConfig_t& cfg, cudaLaunchAttribute* at, int clusters) {
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kGemmThreads + (RC ? 32 * kRcWarps : 0));
    cfg.dynamicSmemBytes = pair_smem_bytes(S);
    cfg.attrs = at;
    cfg.numAttrs = 1;
  };
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_pair_kernel<MODE, RC, S>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, pair_smem_bytes(S));
    if (attr_err != cudaSuccess) return;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    config(cfg, at, 64);
    attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, grouped_gemm_pair_kernel<MODE, RC, S>, &cfg);
    if (attr_err == cudaSuccess && max_clusters <= 0) attr_err = cudaErrorInvalidConfiguration;
  });
  if (attr_err != cudaSuccess) return MOE_ERR_CUDA;
  if (units <= 0) return MOE_OK;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  config(cfg, at, static_cast<int>(std::min<int64_t>(max_clusters, units)));
  cfg.stream = s;
  if (cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<MODE, RC, S>, maps, args) != cudaSuccess)
    return MOE_ERR_CUDA;
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// The stage count of the SM-pair GEMM kernel for one GEMM of a problem: the
// caller's moe_problem.pipeline_stages if set, else the library's choice per
// shape, from sweeps of 4, 5 and 6 stages on a GB300 (bench.py
// --sweep-stages, all runs at 2070 MHz; fewer stages leave room for more
// epilogue staging buffers, pair_out_bufs):
//  * weight gradients: 4 stages when the experts average at most 256 tokens
//    (large batch at N = 8192: dWg + dWu 7.48 ms at 4 stages against 7.87 at
//    6 -- the fp32 stores bound them there), else 6 (skewed workload: 2.74
//    at 6 against 2.89 at 5 and 2.99 at 4; uniform routing 2.62 / 2.76 /
//    2.81);
//  * token-row GEMMs: 5 stages when the experts average at least 1024 tokens
//    (skewed and uniform workloads: gate/up 2.27 / 2.13 ms at 5 against
//    2.30 / 2.18 at 6, gate/up dgrad 2.26 / 2.15 against 2.29 / 2.17), else 6
//    (fine-grained forward: gate/up 0.211 at 6 against 0.216 at 5; large
//    batch at N = 8192: 3.22 against 3.34).
int pick_stages(const Layout& L, int mode) {
  if (L.stages == 4 || L.stages == 5 || L.stages == 6) return L.stages;
  if (mode == WGRAD) return L.A <= 256LL * L.E ? 4 : 6;
  return L.A >= 1024LL * L.E ? 5 : 6;
}

// L2 eviction priorities for the weight gradients where their fp32 stores
// bound them (experts of at most 256 tokens on average, the regime that also
// takes 4 ring stages): the stores are marked evict-first and the token-panel
// loads evict-last, so the gradients, written once and never read back, do
// not push out the panels the other tiles of the expert still read. Large
// batch at N = 8192 (256 tokens per expert): dWg + dWu 7.90-7.98 -> 6.37-6.54
// ms, dWd 3.55 -> 3.38-3.39, the step 22.0 -> 20.3-20.5 ms; at 1024 tokens per
// expert (skewed, uniform, large batch at N = 32768) no gain.
int wgrad_l2_hint(const Layout& L) { return L.A <= 256LL * L.E ? 1 : 0; }

template <int MODE, int S>
moe_status launch_wide_s(const Maps& maps, const Args& args, int64_t units, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;
  auto config = [](cudaLaunchConfig_t& cfg, cudaLaunchAttribute* at, int clusters) {
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = wide_smem_bytes(S);
    cfg.attrs = at;
    cfg.numAttrs = 1;
  };
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_wide_kernel<MODE, S>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, wide_smem_bytes(S));
    if (attr_err != cudaSuccess) return;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    config(cfg, at, 64);
    attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, grouped_gemm_wide_kernel<MODE, S>, &cfg);
    if (attr_err == cudaSuccess && max_clusters <= 0) attr_err = cudaErrorInvalidConfiguration;
  });
  if (attr_err != cudaSuccess) return MOE_ERR_CUDA;
  if (units <= 0) return MOE_OK;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  config(cfg, at, static_cast<int>(std::min<int64_t>(max_clusters, units)));
  cfg.stream = s;
  if (cudaLaunchKernelEx(&cfg, grouped_gemm_wide_kernel<MODE, S>, maps, args) != cudaSuccess)
    return MOE_ERR_CUDA;
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Width of the token-row GEMMs' pair tiles in N: the caller's
// moe_problem.tile_n if set, else the library's choice per shape, from
// sweeps on a GB300 (bench.py --sweep-stages, 2070 MHz). The 512-wide tile
// stages each A k-block once for two N tiles, a quarter fewer bytes through
// L2 per flop, but keeps one accumulator, so its epilogue stalls the MMAs.
// With experts of at least 1024 tokens on average it wins for gate/up (skewed
// workload 2.17-2.22 against 2.29-2.32 ms narrow; uniform routing 2.21-2.29
// against 2.23), down (1.14 against 1.17-1.18; uniform 1.12-1.14 against
// 1.13-1.14) and the gate/up data gradient (K = 2 I: 2.09-2.11 against
// 2.25-2.30; uniform 2.05-2.11 against 2.20-2.22). With fewer tokens the
// epilogue weighs more: fine-grained forward (512 per expert) gate/up 0.235
// against 0.215, large batch at N = 8192 (256) even. Never for the down data
// gradient, whose epilogue reads G and U back (+28% and +37%).
bool pick_wide(const Layout& L, int mode, int n_nt) {
  if (n_nt % 2 != 0) return false;
  if (L.tile_n == 256) return false;
  if (L.tile_n == 512) return true;
  return mode != DACT && L.A >= 1024LL * L.E;
}

template <int MODE, bool RC = false>
moe_status launch_pair(const Layout& L, const Maps& maps, const Args& args, int64_t units,
                       cudaStream_t s) {
  switch (pick_stages(L, MODE)) {
    case 4: return launch_pair_s<MODE, RC, 4>(maps, args, units, s);
    case 5: return launch_pair_s<MODE, RC, 5>(maps, args, units, s);
    default: return launch_pair_s<MODE, RC, 6>(maps, args, units, s);
  }
}

// Token-row modes: the SM-pair kernel over the schedule's pair items (at most
// one per 128-row tile).
template <int MODE>
moe_status launch_tokens(const Layout& L, const Maps& maps, const Args& args, cudaStream_t s) {
  if (pick_wide(L, MODE, args.n_nt))
    return launch_wide_s<MODE, 4>(maps, args, static_cast<int64_t>(args.max_mtiles) * (args.n_nt / 2),
                                  s);
  return launch_pair<MODE>(L, maps, args, static_cast<int64_t>(args.max_mtiles) * args.n_nt, s);
}

// A operand maps of the SM-pair token-row kernel: 128-row box (256-row items)
// and 64-row box (128-row items).
bool make_a_maps(CUtensorMap* full, CUtensorMap* half, const void* base, int64_t cols,
                 int64_t rows) {
  return make_map(full, base, cols, rows, BM) && make_map(half, base, cols, rows, BM / 2);
}

Args base_args(const Layout& L, const void* ws) {
  Args a{};
  a.tiles = at<int32_t>(ws, L.tiles);
  a.n_tiles = at<int32_t>(ws, L.n_tiles);
  a.ptiles = at<int32_t>(ws, L.ptiles);
  a.n_ptiles = at<int32_t>(ws, L.n_ptiles);
  a.pad_offsets = at<int32_t>(ws, L.pad_offsets);
  a.order = at<int32_t>(ws, L.expert_order);
  a.counts = at<int32_t>(ws, L.counts);
  a.err = const_cast<int32_t*>(at<int32_t>(ws, L.err));
  a.max_mtiles = static_cast<int>(L.R / BM);
  a.rows = L.R;
  a.E = L.E;
  return a;
}

}  // namespace

moe_status launch_expert_order(const Layout& L, const void* ws, cudaStream_t s) {
  expert_order_kernel<<<1, 1024, 0, s>>>(at<int32_t>(ws, L.counts), L.E,
                                         const_cast<int32_t*>(at<int32_t>(ws, L.expert_order)));
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status gemm_router(const Layout& L, const void* ws, const void* x, const void* w_router,
                       float* logits, cudaStream_t s) {
  if (L.N == 0) return MOE_OK;
  Maps m{};
  if (!make_map(&m.a0, x, L.H, L.N, BM) || !make_map(&m.b0, w_router, L.H, L.E, BN) ||
      !make_out_map(&m.o0, logits, L.E, L.N))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.b1 = m.b0;
  m.o1 = m.o0;
  Args a = base_args(L, ws);
  a.max_mtiles = static_cast<int>((L.N + BM - 1) / BM);
  a.rows = L.N;
  a.n_nt = 1;
  a.kb1 = L.H / BK;
  a.kb2 = 0;
  a.ld_out = L.E;
  return launch<ROUTER>(m, a, a.max_mtiles, s);
}

moe_status gemm_gate_up(const Layout& L, const void* ws, const void* xe, const void* wg,
                        const void* wu, void* g, void* u, void* act, cudaStream_t s) {
  Maps m{};
  if (!make_a_maps(&m.a0, &m.a0h, xe, L.H, L.R) ||
      !make_map(&m.b0, wg, L.H, static_cast<int64_t>(L.E) * L.I, BN / 4) ||
      !make_map(&m.b1, wu, L.H, static_cast<int64_t>(L.E) * L.I, BN / 4))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.a1h = m.a0h;
  const bool store_gu = g != nullptr && u != nullptr;  // G and U are skipped for inference
  if (!make_bf16_out_map(&m.o2, act, L.I, L.R)) return MOE_ERR_CUDA;
  if (store_gu && (!make_bf16_out_map(&m.o0, g, L.I, L.R) || !make_bf16_out_map(&m.o1, u, L.I, L.R)))
    return MOE_ERR_CUDA;
  Args a = base_args(L, ws);
  a.n_nt = L.I / (BN / 2);
  a.kb1 = L.H / BK;
  a.kb2 = 0;
  a.b_rows = L.I;
  a.ld_out = L.I;
  a.out0 = g;
  a.out1 = u;
  a.out2 = act;
  a.store_gu = store_gu ? 1 : 0;
  return launch_tokens<GATE_UP>(L, m, a, s);
}

moe_status gemm_down(const Layout& L, const void* ws, const void* act, const void* wd, void* ye,
                     cudaStream_t s) {
  Maps m{};
  if (!make_a_maps(&m.a0, &m.a0h, act, L.I, L.R) ||
      !make_map(&m.b0, wd, L.I, static_cast<int64_t>(L.E) * L.H, BN / 2))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.a1h = m.a0h;
  m.b1 = m.b0;
  if (!make_bf16_out_map(&m.o0, ye, L.H, L.R)) return MOE_ERR_CUDA;
  Args a = base_args(L, ws);
  a.n_nt = L.H / BN;
  a.kb1 = L.I / BK;
  a.kb2 = 0;
  a.b_rows = L.H;
  a.ld_out = L.H;
  a.out0 = ye;
  return launch_tokens<DOWN>(L, m, a, s);
}

moe_status gemm_down_dgrad(const Layout& L, const void* ws, const void* dye, const void* g,
                           const void* u, const void* wd, void* dg, void* du, cudaStream_t s) {
  return gemm_down_dgrad_rc(L, ws, nullptr, nullptr, nullptr, dye, nullptr, g, u, wd, dg, du, s);
}

moe_status gemm_down_dgrad_rc(const Layout& L, const void* ws, const void* dy, const void* ye,
                              const float* topk_w, const void* dye, float* d_topk_w,
                              const void* g, const void* u, const void* wd, void* dg, void* du,
                              cudaStream_t s) {
  Maps m{};
  if (!make_a_maps(&m.a0, &m.a0h, dye, L.H, L.R) ||
      !make_map(&m.b0, wd, L.I, static_cast<int64_t>(L.E) * L.H, 64))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.a1h = m.a0h;
  m.b1 = m.b0;
  Args a = base_args(L, ws);
  a.n_nt = L.I / BN;
  a.kb1 = L.H / BK;
  a.kb2 = 0;
  a.b_rows = L.H;
  a.ld_out = L.I;
  a.out0 = dg;
  a.out1 = du;
  a.in0 = g;
  a.in1 = u;
  const int64_t units = static_cast<int64_t>(a.max_mtiles) * a.n_nt;
  if (!dy) return launch_tokens<DACT>(L, m, a, s);
  // fused reverse-combine: dYe and dw come from the kernel's side warps
  a.rc_dy = static_cast<const uint4*>(dy);
  a.rc_ye = static_cast<const uint4*>(ye);
  a.rc_w = topk_w;
  a.rc_dye = static_cast<uint4*>(const_cast<void*>(dye));
  a.rc_dw = d_topk_w;
  a.rc_sync = const_cast<int32_t*>(at<int32_t>(ws, L.rc_sync));
  a.src_of_row = at<int32_t>(ws, L.src_of_row);
  a.k = L.k;
  a.hv = L.H / 8;
  a.A = L.A;
  if (cudaMemsetAsync(a.rc_sync, 0, sizeof(int32_t) * (1 + L.R / BM), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  // assignments without a row (rejected expert ids) keep dw = 0, as in the unfused kernel
  if (L.A > 0 && cudaMemsetAsync(d_topk_w, 0, sizeof(float) * L.A, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return launch_pair<DACT, true>(L, m, a, std::max<int64_t>(units, 1), s);
}

moe_status gemm_down_wgrad(const Layout& L, const void* ws, const void* dye, const void* act,
                           float* dw_down, cudaStream_t s) {
  Maps m{};
  if (!make_map(&m.a0, dye, L.H, L.R, 64) || !make_map(&m.b0, act, L.I, L.R, 64))
    return MOE_ERR_CUDA;
  m.a1 = m.a0;
  m.b1 = m.b0;
  if (!make_out_map(&m.o0, dw_down, L.I, static_cast<int64_t>(L.E) * L.H)) return MOE_ERR_CUDA;
  m.o1 = m.o0;
  Args a = base_args(L, ws);
  if (launch_expert_order(L, ws, s) != MOE_OK) return MOE_ERR_CUDA;
  a.w_mt = L.H / BM;
  a.w_nt = L.I / BN;
  a.n_probs = 1;
  a.ld_out = L.I;
  a.out0 = dw_down;
  a.out1 = dw_down;
  a.l2_hint = wgrad_l2_hint(L);
  return launch_pair<WGRAD>(L, m, a, static_cast<int64_t>(L.E) * (a.w_mt / 2) * a.w_nt, s);
}

moe_status gemm_gate_up_dgrad(const Layout& L, const void* ws, const void* dg, const void* du,
                              const void* wg, const void* wu, void* dxe, cudaStream_t s) {
  Maps m{};
  if (!make_a_maps(&m.a0, &m.a0h, dg, L.I, L.R) || !make_a_maps(&m.a1, &m.a1h, du, L.I, L.R) ||
      !make_map(&m.b0, wg, L.H, static_cast<int64_t>(L.E) * L.I, 64) ||
      !make_map(&m.b1, wu, L.H, static_cast<int64_t>(L.E) * L.I, 64))
    return MOE_ERR_CUDA;
  if (!make_bf16_out_map(&m.o0, dxe, L.H, L.R)) return MOE_ERR_CUDA;
  Args a = base_args(L, ws);
  a.n_nt = L.H / BN;
  a.kb1 = L.I / BK;
  a.kb2 = L.I / BK;
  a.b_rows = L.I;
  a.ld_out = L.H;
  a.out0 = dxe;
  return launch_tokens<DXE>(L, m, a, s);
}

moe_status gemm_gate_up_wgrad(const Layout& L, const void* ws, const void* dg, const void* du,
                              const void* xe, float* dw_gate, float* dw_up, cudaStream_t s) {
  Maps m{};
  if (!make_map(&m.a0, dg, L.I, L.R, 64) || !make_map(&m.a1, du, L.I, L.R, 64) ||
      !make_map(&m.b0, xe, L.H, L.R, 64))
    return MOE_ERR_CUDA;
  m.b1 = m.b0;
  if (!make_out_map(&m.o0, dw_gate, L.H, static_cast<int64_t>(L.E) * L.I) ||
      !make_out_map(&m.o1, dw_up, L.H, static_cast<int64_t>(L.E) * L.I))
    return MOE_ERR_CUDA;
  Args a = base_args(L, ws);
  if (launch_expert_order(L, ws, s) != MOE_OK) return MOE_ERR_CUDA;
  a.w_mt = L.I / BM;
  a.w_nt = L.H / BN;
  a.n_probs = 2;
  a.ld_out = L.H;
  a.out0 = dw_gate;
  a.out1 = dw_up;
  a.l2_hint = wgrad_l2_hint(L);
  return launch_pair<WGRAD>(L, m, a, 2LL * L.E * (a.w_mt / 2) * a.w_nt, s);
}

namespace {
void fused_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* att, int clusters) {
  att[0].id = cudaLaunchAttributeClusterDimension;
  att[0].val.clusterDim.x = 2;
  att[0].val.clusterDim.y = 1;
  att[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kGemmThreads + 32 * kFfDispWarps);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cfg.attrs = att;
  cfg.numAttrs = 1;
}

// CTA pairs of the fused forward's grid: the occupancy query's count of
// co-resident clusters (every wait relies on all of them being resident).
// -1 if the query fails.
int fused_clusters() {
  static std::once_flag once;
  static int max_clusters = -1;
  std::call_once(once, [] {
    if (cudaFuncSetAttribute(fused_forward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPairSmemBytes) != cudaSuccess)
      return;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute att[1];
    fused_config(cfg, att, 64);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fused_forward_kernel, &cfg) == cudaSuccess && n > 0)
      max_clusters = n;
  });
  return max_clusters;
}

// The down units of an item follow its gate/up units by about three waves
// of units, so they rarely find its Act unfinished.
int fused_lag(const Layout& L, int clusters) {
  const int units = L.I / (BN / 2) + L.H / BN;
  return std::max(2, (3 * clusters + units - 1) / units);
}
}  // namespace

int fused_ring_slots(const Layout& L) {
  const int clusters = fused_clusters();
  return clusters > 0 ? fused_lag(L, clusters) + kRingSpare : 0;
}

moe_status gemm_fused_forward(const Layout& L, const void* ws, const void* x, const void* wg,
                              const void* wu, const void* wd, void* xe, void* g, void* u,
                              void* act, void* ye, int ring, cudaStream_t s) {
  const int clusters = fused_clusters();
  if (clusters <= 0) return MOE_ERR_CUDA;
  const bool store_gu = g != nullptr && u != nullptr;
  if (ring < 0 || (ring > 0 && (store_gu || ring <= fused_lag(L, clusters))))
    return MOE_ERR_INVALID_ARG;
  // rows of the Xe and Act buffers: all R, or the ring's slots
  const int64_t xrows = ring > 0 ? static_cast<int64_t>(ring) * 2 * BM : L.R;
  Maps mg{}, md{};
  if (!make_a_maps(&mg.a0, &mg.a0h, xe, L.H, xrows) ||
      !make_map(&mg.b0, wg, L.H, static_cast<int64_t>(L.E) * L.I, BN / 4) ||
      !make_map(&mg.b1, wu, L.H, static_cast<int64_t>(L.E) * L.I, BN / 4) ||
      !make_bf16_out_map(&mg.o2, act, L.I, xrows) ||
      !make_a_maps(&md.a0, &md.a0h, act, L.I, xrows) ||
      !make_map(&md.b0, wd, L.I, static_cast<int64_t>(L.E) * L.H, BN / 2) ||
      !make_bf16_out_map(&md.o0, ye, L.H, L.R))
    return MOE_ERR_CUDA;
  if (store_gu && (!make_bf16_out_map(&mg.o0, g, L.I, L.R) || !make_bf16_out_map(&mg.o1, u, L.I, L.R)))
    return MOE_ERR_CUDA;
  mg.a1 = mg.a0;
  mg.a1h = mg.a0h;
  md.a1 = md.a0;
  md.a1h = md.a0h;
  md.b1 = md.b0;
  Args ag = base_args(L, ws);
  ag.n_nt = L.I / (BN / 2);
  ag.kb1 = L.H / BK;
  ag.b_rows = L.I;
  ag.ld_out = L.I;
  ag.store_gu = store_gu ? 1 : 0;
  Args ad = base_args(L, ws);
  ad.n_nt = L.H / BN;
  ad.kb1 = L.I / BK;
  ad.b_rows = L.H;
  ad.ld_out = L.H;
  int32_t* sync = const_cast<int32_t*>(at<int32_t>(ws, L.ff_sync));
  const int64_t n_tiles = L.R / BM;
  FusedArgs f{};
  f.x = static_cast<const uint4*>(x);
  f.xe = static_cast<uint4*>(xe);
  f.src_of_row = at<int32_t>(ws, L.src_of_row);
  f.pad_offsets = at<int32_t>(ws, L.pad_offsets);
  f.ticket = sync;
  f.disp_done = sync + 1;
  f.gu_done = sync + 1 + n_tiles;
  f.dn_done = sync + 1 + 2 * n_tiles;
  f.ptiles = at<int32_t>(ws, L.ptiles);
  f.A = L.A;
  f.rows = L.R;
  f.E = L.E;
  f.k = L.k;
  f.hv = L.H / 8;
  f.G = ag.n_nt;
  f.D = ad.n_nt;
  f.lag = fused_lag(L, clusters);
  f.ring = ring;
  if (cudaMemsetAsync(sync, 0, sizeof(int32_t) * (1 + 3 * n_tiles), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (L.R == 0) return MOE_OK;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute att[1];
  fused_config(cfg, att, clusters);
  cfg.stream = s;
  if (cudaLaunchKernelEx(&cfg, fused_forward_kernel, mg, md, ag, ad, f) != cudaSuccess)
    return MOE_ERR_CUDA;
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
