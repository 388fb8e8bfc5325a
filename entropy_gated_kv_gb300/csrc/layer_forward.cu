// layer_forward.cu — the partial forward of one transformer layer for the recompute set.
//
// EntropyCache, gist.science zh summary §2.2 ("前向传播 / 部分传播"): a partial forward
// recomputes only the recompute set (the masked positions and the last k decoded ones) and
// reads every other position from the K/V cache; a full forward recomputes every position.
// The layer is the LLaMA-style block of the models the pages evaluate (LLaDA-8B, Dream-7B):
// for every recompute row r at position p = idx[r] of a sequence,
//   x = x_src[p]; h = RMSNorm(x) * gamma1
//   q, k, v = h Wq^T, h Wk^T, h Wv^T; q and k rotated by RoPE at position p
//   cache[p] = (k, v)                                    (the K/V refresh, kv_scatter.cu)
//   o = attention of q against the whole cache           (attention.cu)
//   x2 = x + o Wo^T;  y = x2 + (SiLU(h2 Wg^T) * (h2 Wu^T)) Wd^T,  h2 = RMSNorm(x2) * gamma2
//
// Kernels (all read the recompute-set size R from the device, so no host synchronisation):
//   - rmsnorm_kernel: one CTA per row (gathering the rows by idx for the first norm);
//   - gemm_kernel<EPI>: a swap-AB tcgen05 GEMM, out[row, f] = sum_k X[row, k] W[f, k]. M = 128
//     weight rows (output features, A, K-major), N = the block's recompute rows rounded up to
//     32 (B, K-major, at most 256; the instruction descriptor is built on the device from R),
//     K in stages of 64 (one 128-byte swizzle atom per row) through a TMA ring of up to 8
//     stages (as many as fit beside the row blocks' rows: more weight bytes in flight when the
//     rows are few), the row operand in boxes of 128 rows. One
//     thread issues tcgen05.mma into a double-buffered TMEM accumulator (2 x 256 columns), so a
//     tile's epilogue overlaps the next tile's products. Persistent, one CTA per SM; the tiles
//     are (feature tile, live row block) with the feature tile outermost, so that the row
//     blocks of one weight tile run together and share it through L2. The epilogue is fused:
//     RoPE for the q/k tiles (the rotate-half partner feature comes through shared memory), the
//     residual add, or SwiGLU (a tile holds 64 gate rows and the 64 matching up rows of W,
//     loaded as two TMA boxes).
//   - rope_table_kernel: the RoPE angle table, in double precision.
// For few rows the GEMMs stream the weights once (HBM-bound); for a full forward (R = L) they
// are tensor-core bound.
#include <cuda.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "ec_common.cuh"
#include "ec_internal.h"

namespace ec {
namespace {

constexpr int kThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kTileM = 128;     // output features per tile (MMA M)
constexpr int kTileK = 64;      // input features per stage (one 128-byte swizzle atom)
constexpr int kRowBlock = 256;  // recompute rows per tile (MMA N at most)
constexpr int kBoxRows = 128;   // rows per TMA box of the row operand
constexpr int kMaxStages = 8;
constexpr uint32_t kABytes = kTileM * kTileK * 2;      // 16 KB
constexpr uint32_t kBoxBytes = kBoxRows * kTileK * 2;  // 16 KB
constexpr uint32_t kRingBytes = 196 * 1024;            // A and B stages
constexpr int kXPitch = 129;                           // exchange buffer row pitch (floats)
constexpr int kMaxGrid = 256;                          // GEMM CTAs at most (the split-K slab is sized by it)
constexpr uint64_t kWaitLimitNs = 2000000000ull;       // 2 s: far beyond any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kDescHi = sdesc_hi(1024);  // 8 rows of 128 B between core-matrix groups

enum : int { kEpiQkv = 0, kEpiResidual = 1, kEpiSwiglu = 2 };

struct GemmBars {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort;
  int epi_ok;  // the epilogue's shared verdict on its latest wait
};

constexpr uint32_t kXOff = kRingBytes;
constexpr uint32_t kPosOff = kXOff + 32 * kXPitch * 4;  // the tile's row positions (qkv epilogue)
constexpr uint32_t kBarOff = kPosOff + kRowBlock * 4;
constexpr uint32_t kSmemBytes = kBarOff + sizeof(GemmBars) + 1024;  // + slack for 1024-byte alignment

struct GemmArgs {
  int B, L, K;         // sequences, positions per sequence (row stride of X), input features
  int n_ftiles, nrb;   // feature tiles; row blocks per sequence (ceil(L / 256))
  const int32_t* R;    // [B] recompute rows per sequence
  const int32_t* idx;  // [B, L] positions of the rows (RoPE)
  uint16_t* out0;      // qkv: q [B, L, Hq D]; otherwise the output [B, L, n_out]
  uint16_t* out1;      // qkv: k [B, L, Hkv D]
  uint16_t* out2;      // qkv: v [B, L, Hkv D]
  const uint16_t* res;  // residual: [B, L, n_out]
  int n_out;            // output row length (residual, swiglu)
  int q_feats, kv_feats, D;
  const float* rope_cos;  // [L, D/2]
  const float* rope_sin;
  float* slab;    // split-K partials: kMaxGrid x kRowBlock rows of kTileM fp32, in blocks of n_max rows
  int grid;       // the GEMM's grid (the finishing kernel recomputes the plan from it)
  int32_t* dev_err;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// Live row blocks: sequence b has ceil(R[b] / 256) of them. Tiles are (feature tile, live row
// block), the feature tile outermost, so that the row blocks of one weight tile run together.
__device__ __forceinline__ int live_blocks(const GemmArgs& a, int b) {
  const int Rb = min(max(__ldg(a.R + b), 0), a.L);  // R is read-only while the kernel runs
  return (Rb + kRowBlock - 1) / kRowBlock;
}

struct Tile {
  int ft, b, r0, nrows;
};

__device__ __forceinline__ Tile decode_tile(int t, int total_rb, const GemmArgs& a) {
  Tile x;
  x.ft = t / total_rb;
  int j = t - x.ft * total_rb;
  x.b = 0;
  for (;;) {  // the sequence of the j-th live row block
    const int nb = live_blocks(a, x.b);
    if (j < nb) break;
    j -= nb;
    ++x.b;
  }
  x.r0 = j * kRowBlock;
  const int Rb = min(max(__ldg(a.R + x.b), 0), a.L);
  x.nrows = min(kRowBlock, Rb - x.r0);
  return x;
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + ex2_approx(-g * kLog2e)); }

__device__ __forceinline__ uint16_t to_bf16(float v) { return static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu); }

__device__ __forceinline__ float from_bf16(uint16_t u) { return __uint_as_float(static_cast<uint32_t>(u) << 16); }

// Split-K plan, the same in every CTA of the GEMM and of its finishing kernel. A work unit is
// one split of one live tile (kps K stages); CTA c takes the units c, c + grid, ... Each lane
// of the warp prices one split count s = lane + 1 as (rounds of units over the grid) x (K stages
// per unit + 1 for the unit's start-up) and the warp takes the cheapest, the fewer splits on a
// tie: the split evens out the last round when the live tiles are not a multiple of the grid
// (192 SwiGLU tiles on 152 SMs: 3 splits make 576 units, 3.8 rounds, against 1.26 rounds of
// whole tiles that take 2). Split units write fp32 partials to the slab, which holds
// kMaxGrid x 256 rows of 128 features, so the units of a plan are at most that many blocks of
// n_max rows; the finishing kernel sums them and runs the epilogue.
struct SplitPlan {
  int total_rb, live, splits, kps;  // live row blocks, live tiles, splits per tile, K stages per split
  int n_max;                        // rows of the largest row block, rounded up to 32
};

// Whole warp (every lane must call it).
__device__ __forceinline__ SplitPlan split_plan(const GemmArgs& a) {
  SplitPlan sp;
  sp.total_rb = 0;
  int rmax = 0;
  for (int b = 0; b < a.B; ++b) {
    const int Rb = min(max(__ldg(a.R + b), 0), a.L);
    sp.total_rb += (Rb + kRowBlock - 1) / kRowBlock;
    rmax = max(rmax, Rb);
  }
  sp.n_max = min(kRowBlock, (rmax + 31) / 32 * 32);
  sp.live = a.n_ftiles * sp.total_rb;
  const int n_k = a.K / kTileK;
  uint64_t key = ~0ull;
  if (sp.live > 0) {
    const int s = (threadIdx.x & 31) + 1;
    const int kps = (n_k + s - 1) / s;
    const int splits = (n_k + kps - 1) / kps;  // no empty split
    const int units = sp.live * splits;
    const int cap = kMaxGrid * kRowBlock / sp.n_max;
    if (splits == 1 || units <= cap) {
      const int rounds = (units + a.grid - 1) / a.grid;
      key = (static_cast<uint64_t>(rounds) * static_cast<uint64_t>(kps + 1) << 32) |
            (static_cast<uint64_t>(splits) << 16) | static_cast<uint64_t>(kps);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, key, off);
    key = o < key ? o : key;
  }
  sp.splits = sp.live > 0 ? static_cast<int>((key >> 16) & 0xFFFFu) : 1;
  sp.kps = sp.live > 0 ? static_cast<int>(key & 0xFFFFu) : n_k;
  return sp;
}

// A work unit's block of the slab: n_max rows of 128 fp32 features.
__device__ __forceinline__ float* slab_block(const GemmArgs& a, const SplitPlan& sp, int tile_id, int split) {
  return a.slab + static_cast<int64_t>(tile_id * sp.splits + split) * sp.n_max * kTileM;
}

// The fused epilogue of ROWS rows (rows row0 .. row0 + ROWS - 1 of tile x) of one output
// feature per thread: v[c] is the accumulator of row row0 + c. All 128 threads of the epilogue call it; bar() synchronises
// them (the exchange buffer sX carries the RoPE partner or the SwiGLU up value).
// spos (may be null): the positions of these rows, already in shared memory (the qkv epilogue
// reads them instead of idx).
template <int EPI, int ROWS, typename Bar>
__device__ __forceinline__ void epilogue_rows(const GemmArgs& a, const Tile& x, int row0, const float (&v)[ROWS],
                                              float* sX, int f_in, Bar bar, const int* spos = nullptr) {
  static_assert(ROWS <= 32 && ROWS % 8 == 0, "the exchange buffer holds 32 rows");
  constexpr int G = ROWS < 16 ? ROWS : 16;  // rows whose loads are issued before their stores
  const int nvalid = min(ROWS, x.nrows - row0);
  const int64_t rbase = static_cast<int64_t>(x.b) * a.L + x.r0 + row0;
  if constexpr (EPI == kEpiResidual) {
    // the residual loads of G rows are issued before their stores (a store to out0 could
    // otherwise alias the next load, and the rows would take one dependent round trip each)
    const int f = x.ft * kTileM + f_in;
#pragma unroll
    for (int c0 = 0; c0 < ROWS; c0 += G) {
      float rv[G];
#pragma unroll
      for (int c = 0; c < G; ++c)
        rv[c] = c0 + c < nvalid ? from_bf16(__ldg(a.res + (rbase + c0 + c) * a.n_out + f)) : 0.f;
#pragma unroll
      for (int c = 0; c < G; ++c)
        if (c0 + c < nvalid) a.out0[(rbase + c0 + c) * a.n_out + f] = to_bf16(v[c0 + c] + rv[c]);
    }
  } else if constexpr (EPI == kEpiSwiglu) {
    bar();  // the exchange buffer is free
    if (f_in >= 64)
#pragma unroll
      for (int c = 0; c < ROWS; ++c) sX[c * kXPitch + f_in] = v[c];
    bar();
    if (f_in < 64) {
      const int f = x.ft * 64 + f_in;
#pragma unroll
      for (int c = 0; c < ROWS; ++c)
        if (c < nvalid) a.out0[(rbase + c) * a.n_out + f] = to_bf16(silu(v[c]) * sX[c * kXPitch + f_in + 64]);
    }
  } else {  // q / k with RoPE, v as is
    const int f0 = x.ft * kTileM;
    const int part = f0 < a.q_feats ? 0 : (f0 < a.q_feats + a.kv_feats ? 1 : 2);
    uint16_t* dst = part == 0 ? a.out0 : (part == 1 ? a.out1 : a.out2);
    const int feats = part == 0 ? a.q_feats : a.kv_feats;
    const int f = f0 - (part == 0 ? 0 : (part == 1 ? a.q_feats : a.q_feats + a.kv_feats)) + f_in;
    if (part == 2) {
#pragma unroll
      for (int c = 0; c < ROWS; ++c)
        if (c < nvalid) dst[(rbase + c) * feats + f] = to_bf16(v[c]);
    } else {
      const int half = a.D / 2;
      const int j = f_in % a.D;  // feature within its head (a tile holds whole heads)
      const int i = j % half;
      bar();  // the exchange buffer is free
#pragma unroll
      for (int c = 0; c < ROWS; ++c) sX[c * kXPitch + f_in] = v[c];
      bar();
      const int partner = f_in ^ half;  // the rotate-half partner in the same head
#pragma unroll
      for (int c0 = 0; c0 < ROWS; c0 += G) {
        // the positions and angles of G rows are loaded before their stores
        float cs[G], sn[G];
#pragma unroll
        for (int c = 0; c < G; ++c) {
          const int pos = c0 + c >= nvalid ? 0
                          : spos != nullptr ? spos[c0 + c]
                                            : min(max(__ldg(a.idx + rbase + c0 + c), 0), a.L - 1);  // a bad idx is reported by the norm
          cs[c] = __ldg(a.rope_cos + static_cast<int64_t>(pos) * half + i);
          sn[c] = __ldg(a.rope_sin + static_cast<int64_t>(pos) * half + i);
        }
#pragma unroll
        for (int c = 0; c < G; ++c) {
          if (c0 + c < nvalid) {
            const float w = sX[(c0 + c) * kXPitch + partner];
            const float u = v[c0 + c];
            dst[(rbase + c0 + c) * feats + f] = to_bf16(j < half ? u * cs[c] - w * sn[c] : u * cs[c] + w * sn[c]);
          }
        }
      }
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ CUtensorMap tm_a0,
                                                            const __grid_constant__ CUtensorMap tm_a1,
                                                            const __grid_constant__ CUtensorMap tm_a2,
                                                            const __grid_constant__ CUtensorMap tm_x, GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem + kBarOff);
  float* sX = reinterpret_cast<float*>(smem + kXOff);
  int* sPos = reinterpret_cast<int*>(smem + kPosOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_k = a.K / kTileK;
  (void)n_k;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], 128);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_a0);
    if (EPI != kEpiResidual) prefetch_tmap(&tm_a1);
    if (EPI == kEpiQkv) prefetch_tmap(&tm_a2);
    prefetch_tmap(&tm_x);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort;
  pdl_wait();  // the row operand, R and idx come from the previous kernels in the stream
  pdl_launch_dependents();
  const SplitPlan sp = split_plan(a);
  const int n_tiles = sp.live * sp.splits;
  // the ring: as many stages as fit for the launch's largest row block (more weight bytes in
  // flight when the rows are few)
  const uint32_t b_bytes = static_cast<uint32_t>((sp.n_max + kBoxRows - 1) / kBoxRows) * kBoxBytes;
  const int stages = max(2, min(kMaxStages, static_cast<int>(kRingBytes / (kABytes + max(b_bytes, kBoxBytes)))));
  const uint32_t a_off = 0, b_off = static_cast<uint32_t>(stages) * kABytes;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        const Tile x = decode_tile(t / sp.splits, sp.total_rb, a);
        const int k0 = (t % sp.splits) * sp.kps, k1 = min(n_k, k0 + sp.kps);
        const int nbox = (x.nrows + kBoxRows - 1) / kBoxRows;
        const int xrow = x.b * a.L + x.r0;
        for (int kt = k0; kt < k1; ++kt, ++it) {
          const uint32_t s = it % stages, u = it / stages;
          if (!(ok = mbar_wait_bounded(&bars->empty[s], (u & 1u) ^ 1u, abort_flag, a.dev_err, kWaitLimitNs))) break;
          mbar_arrive_expect_tx(&bars->full[s], kABytes + nbox * kBoxBytes);
          uint8_t* as = smem + a_off + s * kABytes;
          if constexpr (EPI == kEpiQkv) {
            const int f0 = x.ft * kTileM;
            if (f0 < a.q_feats) tma_load_2d(as, &tm_a0, &bars->full[s], kt * kTileK, f0);
            else if (f0 < a.q_feats + a.kv_feats) tma_load_2d(as, &tm_a1, &bars->full[s], kt * kTileK, f0 - a.q_feats);
            else tma_load_2d(as, &tm_a2, &bars->full[s], kt * kTileK, f0 - a.q_feats - a.kv_feats);
          } else if constexpr (EPI == kEpiSwiglu) {  // 64 gate rows, then the 64 matching up rows
            tma_load_2d(as, &tm_a0, &bars->full[s], kt * kTileK, x.ft * 64);
            tma_load_2d(as + kABytes / 2, &tm_a1, &bars->full[s], kt * kTileK, x.ft * 64);
          } else {
            tma_load_2d(as, &tm_a0, &bars->full[s], kt * kTileK, x.ft * kTileM);
          }
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_2d(smem + b_off + s * b_bytes + bx * kBoxBytes, &tm_x, &bars->full[s], kt * kTileK,
                        xrow + bx * kBoxRows);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      int n = 0;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        const Tile x = decode_tile(t / sp.splits, sp.total_rb, a);
        const int k0 = (t % sp.splits) * sp.kps, k1 = min(n_k, k0 + sp.kps);
        const int buf = n & 1;
        const uint32_t use = static_cast<uint32_t>(n >> 1);
        ++n;
        const uint32_t N = static_cast<uint32_t>((x.nrows + 31) / 32 * 32);
        const uint32_t idesc = idesc_bf16_f32(128, N, 0);
        if (!(ok = mbar_wait_bounded(&bars->acc_empty[buf], (use & 1u) ^ 1u, abort_flag, a.dev_err, kWaitLimitNs))) break;
        tc_fence_after();
        const uint32_t d_col = tmem + static_cast<uint32_t>(buf * kRowBlock);
        for (int kt = k0; kt < k1; ++kt, ++it) {
          const uint32_t s = it % stages, u = it / stages;
          if (!(ok = mbar_wait_bounded(&bars->full[s], u & 1u, abort_flag, a.dev_err, kWaitLimitNs))) break;
          tc_fence_after();
          const uint32_t a_lo = sdesc_lo(smem_u32(smem + a_off + s * kABytes), 16);
          const uint32_t b_lo = sdesc_lo(smem_u32(smem + b_off + s * b_bytes), 16);
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk)  // 16 elements = 32 bytes = 2 descriptor units
            umma_ss(d_col, a_lo + 2 * kk, b_lo + 2 * kk, kDescHi, idesc, (kt > k0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars->empty[s]);
        }
        if (ok) umma_commit(&bars->acc_full[buf]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;         // 0..127: the TMEM lane = output feature in the tile
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int f_in = 32 * (warp & 3) + lane;  // (tcgen05 warp rule: warp w reads lanes 32 (w % 4) ..)
    int n = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
      const int tile_id = t / sp.splits, split = t % sp.splits;
      const Tile x = decode_tile(tile_id, sp.total_rb, a);
      const int buf = n & 1;
      const uint32_t use = static_cast<uint32_t>(n >> 1);
      ++n;
      const int n_chunks = (x.nrows + 31) / 32;
      // one thread waits and the four warps take its verdict together, so that none of them can
      // be left at a named barrier that the others have abandoned
      named_bar_sync(1, 128);
      if (et == 0) bars->epi_ok = mbar_wait_bounded(&bars->acc_full[buf], use & 1u, abort_flag, a.dev_err, kWaitLimitNs) ? 1 : 0;
      if constexpr (EPI == kEpiQkv) {  // the tile's positions for RoPE, once (the previous tile's reads are done)
        if (sp.splits == 1)
          for (int r = et; r < x.nrows; r += 128)
            sPos[r] = min(max(__ldg(a.idx + static_cast<int64_t>(x.b) * a.L + x.r0 + r), 0), a.L - 1);
      }
      named_bar_sync(1, 128);
      if (!bars->epi_ok) break;
      tc_fence_after();
      for (int ch = 0; ch < n_chunks; ++ch) {
        uint32_t r[32];
        EC_TMEM_LD32(tmem + lane_off + static_cast<uint32_t>(buf * kRowBlock + ch * 32), r);
        tmem_wait_ld();
        if (ch == n_chunks - 1) {  // the accumulator buffer may be overwritten now
          tc_fence_before();
          mbar_arrive(&bars->acc_empty[buf]);
        }
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = __uint_as_float(r[c]);
        if (sp.splits == 1) {
          epilogue_rows<EPI, 32>(a, x, ch * 32, v, sX, f_in, [] { named_bar_sync(1, 128); },
                                 EPI == kEpiQkv ? sPos + ch * 32 : nullptr);
        } else {  // a split's partial: rows of 128 fp32 features, coalesced
          float* blk = slab_block(a, sp, tile_id, split) + static_cast<int64_t>(ch * 32) * kTileM + f_in;
#pragma unroll
          for (int c = 0; c < 32; ++c) blk[c * kTileM] = v[c];
        }
      }
    }
  }

  // ---------------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Sums the split-K partials of each (tile, 8-row group) and runs the fused epilogue; nothing
// when the GEMM ran unsplit. 128 threads, one output feature each. The items are small (8 rows,
// the partials of up to 8 splits in flight at once), so many CTAs share an SM and an item takes
// one round trip per 8 splits.
constexpr int kFinRows = 8;
constexpr int kFinSplits = 8;

template <int EPI>
__global__ void __launch_bounds__(128) gemm_finish_kernel(GemmArgs a) {
  __shared__ float sX[kFinRows * kXPitch];
  pdl_wait();  // the partials come from the GEMM
  pdl_launch_dependents();
  const SplitPlan sp = split_plan(a);
  if (sp.splits == 1) return;
  const int f_in = threadIdx.x;
  const int groups = sp.n_max / kFinRows;  // groups of the largest row block
  const int items = sp.live * groups;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {  // uniform over the CTA
    const int tile_id = it / groups, grp = it - tile_id * groups;
    const Tile x = decode_tile(tile_id, sp.total_rb, a);
    if (grp * kFinRows >= x.nrows) continue;
    float v[kFinRows];
#pragma unroll
    for (int c = 0; c < kFinRows; ++c) v[c] = 0.f;
    for (int s0 = 0; s0 < sp.splits; s0 += kFinSplits) {
      float t[kFinSplits][kFinRows];  // the splits' values in flight at once before any is added
#pragma unroll
      for (int s = 0; s < kFinSplits; ++s) {
        if (s0 + s < sp.splits) {
          const float* blk = slab_block(a, sp, tile_id, s0 + s) + static_cast<int64_t>(grp * kFinRows) * kTileM + f_in;
#pragma unroll
          for (int c = 0; c < kFinRows; ++c) t[s][c] = __ldcg(blk + c * kTileM);
        }
      }
#pragma unroll
      for (int s = 0; s < kFinSplits; ++s)
        if (s0 + s < sp.splits)
#pragma unroll
          for (int c = 0; c < kFinRows; ++c) v[c] += t[s][c];
    }
    epilogue_rows<EPI, kFinRows>(a, x, grp * kFinRows, v, sX, f_in, [] { __syncthreads(); });
  }
}

// One CTA per recompute row (grid-stride over rows): h = RMSNorm(x) * gamma in bf16. With
// GATHER the row is x_src[b, idx[b, r]] and is also copied to xg[b, r] (the residual input);
// without, it is src[b, r]. d % 8 == 0, d <= 8192.
template <bool GATHER>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t* __restrict__ src, const int32_t* __restrict__ idx,
                                                      const int32_t* __restrict__ R, int L, int d,
                                                      const uint16_t* __restrict__ gamma, float eps,
                                                      uint16_t* __restrict__ xg, uint16_t* __restrict__ h,
                                                      int32_t* __restrict__ dev_err) {
  __shared__ float red[8];
  pdl_wait();  // the rows, idx and R may come from the previous kernels in the stream
  pdl_launch_dependents();
  const int b = blockIdx.y, tid = threadIdx.x;
  const int Rb = min(max(__ldcg(R + b), 0), L);
  const int nvec = d / 8;
  for (int r = blockIdx.x; r < Rb; r += gridDim.x) {
    int64_t srow = static_cast<int64_t>(b) * L + r;
    if constexpr (GATHER) {
      const int p = __ldcg(idx + srow);
      if (p < 0 || p >= L) {  // uniform over the CTA
        if (tid == 0) report_error(dev_err, EC_DEVERR_BAD_IDX);
        continue;
      }
      srow = static_cast<int64_t>(b) * L + p;
    }
    const uint4* s = reinterpret_cast<const uint4*>(src + srow * d);
    uint4 v[4];
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = tid + u * 256;
      v[u] = i < nvec ? s[i] : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = bf16lo_to_f32(w[e]), hi = bf16hi_to_f32(w[e]);
        ss = fmaf(lo, lo, fmaf(hi, hi, ss));
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    __syncthreads();  // red is reused by the next row
    const float inv = rsqrtf(tot / static_cast<float>(d) + eps);
    const int64_t orow = (static_cast<int64_t>(b) * L + r) * d;
    const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = tid + u * 256;
      if (i >= nvec) continue;
      const uint4 gv = g4[i];
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        o[e] = pack_bf16x2(bf16lo_to_f32(w[e]) * inv * bf16lo_to_f32(gw[e]), bf16hi_to_f32(w[e]) * inv * bf16hi_to_f32(gw[e]));
      reinterpret_cast<uint4*>(h + orow)[i] = make_uint4(o[0], o[1], o[2], o[3]);
      if constexpr (GATHER) reinterpret_cast<uint4*>(xg + orow)[i] = v[u];
    }
  }
}

// cos / sin of pos * theta^(-2i/D) for pos < L, i < D/2, computed in double precision.
__global__ void rope_table_kernel(int L, int D, double theta, float* __restrict__ cs, float* __restrict__ sn) {
  const int half = D / 2;
  const int64_t n = static_cast<int64_t>(L) * half;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(e / half), i = static_cast<int>(e - static_cast<int64_t>(pos) * half);
    const double ang = static_cast<double>(pos) * pow(theta, -2.0 * i / D);
    double s, c;
    sincos(ang, &s, &c);
    cs[e] = static_cast<float>(c);
    sn[e] = static_cast<float>(s);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A 2D bf16 tensor map over a row-major [rows, cols] matrix, box {64, box_rows}, 128-byte
// swizzle, zero fill outside the matrix.
bool map_2d(EncodeTiledFn enc, CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI>
cudaError_t launch_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& a2, const CUtensorMap& x,
                        const GemmArgs& args, cudaStream_t s) {
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(gemm_kernel<EPI>), kSmemBytes);
  int sms = 0;
  if (e == cudaSuccess) e = current_device_sms(&sms);
  if (e != cudaSuccess) return e;
  GemmArgs g = args;
  g.grid = std::max(1, std::min(sms, kMaxGrid));
  e = launch_pdl(gemm_kernel<EPI>, dim3(g.grid), dim3(kThreads), kSmemBytes, s, a0, a1, a2, x, g);
  if (e != cudaSuccess) return e;
  return launch_pdl(gemm_finish_kernel<EPI>, dim3(8 * g.grid), dim3(128), 0, s, g);
}

}  // namespace

size_t layer_forward_workspace_bytes(const ec_params& p, int32_t d_ff) {
  const size_t rows = static_cast<size_t>(p.B) * p.L;
  const size_t d = static_cast<size_t>(p.Hq) * p.D;
  const size_t kv = static_cast<size_t>(p.Hkv) * p.D;
  size_t off = 0;
  for (size_t n : {d, d, d, kv, kv, d, d, static_cast<size_t>(d_ff)}) off += align_up(rows * n * 2, 256);
  off += align_up(static_cast<size_t>(kMaxGrid) * kRowBlock * kTileM * 4, 256);  // split-K partials
  return off + align_up(attention_workspace_bytes(p), 256);
}

cudaError_t launch_rope_table(int32_t L, int32_t D, float theta, float* cs, float* sn, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(L) * (D / 2);
  const int grid = static_cast<int>(std::min<int64_t>(4096, (n + 255) / 256));
  rope_table_kernel<<<grid, 256, 0, s>>>(L, D, static_cast<double>(theta), cs, sn);
  return cudaGetLastError();
}

cudaError_t launch_layer_forward(const ec_params& p, const ec_layer& w, const int32_t* idx, const int32_t* R,
                                 const void* x_src, void* k_cache, void* v_cache, void* y, void* ws,
                                 int32_t* dev_err, cudaStream_t s, ec_status* status) {
  *status = EC_OK;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) {
    *status = EC_ERR_CUDA;
    return cudaErrorNotSupported;
  }
  const int B = p.B, L = p.L, D = p.D;
  const int d = p.Hq * D, kvf = p.Hkv * D, dff = w.d_ff;
  const int64_t rows = static_cast<int64_t>(B) * L;
  // workspace: xg, h, q, kn, vn, o, x2, a, attention
  char* base = static_cast<char*>(ws);
  size_t off = 0;
  auto take = [&](size_t n) {
    char* ptr = base + off;
    off += align_up(static_cast<size_t>(rows) * n * 2, 256);
    return reinterpret_cast<uint16_t*>(ptr);
  };
  uint16_t* xg = take(d);
  uint16_t* h = take(d);
  uint16_t* q = take(d);
  uint16_t* kn = take(kvf);
  uint16_t* vn = take(kvf);
  uint16_t* o = take(d);
  uint16_t* x2 = take(d);
  uint16_t* act = take(dff);
  float* slab = reinterpret_cast<float*>(base + off);
  off += align_up(static_cast<size_t>(kMaxGrid) * kRowBlock * kTileM * 4, 256);
  void* attn_ws = base + off;

  CUtensorMap m_wq, m_wk, m_wv, m_wo, m_wg, m_wu, m_wd, m_h, m_o, m_act;
  if (!map_2d(enc, &m_wq, w.wq, d, d, kTileM) || !map_2d(enc, &m_wk, w.wk, kvf, d, kTileM) ||
      !map_2d(enc, &m_wv, w.wv, kvf, d, kTileM) || !map_2d(enc, &m_wo, w.wo, d, d, kTileM) ||
      !map_2d(enc, &m_wg, w.wg, dff, d, 64) || !map_2d(enc, &m_wu, w.wu, dff, d, 64) ||
      !map_2d(enc, &m_wd, w.wd, d, dff, kTileM) || !map_2d(enc, &m_h, h, rows, d, kBoxRows) ||
      !map_2d(enc, &m_o, o, rows, d, kBoxRows) || !map_2d(enc, &m_act, act, rows, dff, kBoxRows)) {
    *status = EC_ERR_INVALID_ARG;
    return cudaErrorInvalidValue;
  }
  int sms = 0;
  cudaError_t e = current_device_sms(&sms);
  if (e != cudaSuccess) {
    *status = EC_ERR_CUDA;
    return e;
  }
  const dim3 norm_grid(static_cast<unsigned>(std::min(L, 2 * sms)), static_cast<unsigned>(B));
  const uint16_t* xs = static_cast<const uint16_t*>(x_src);
  const float eps = w.eps;
  GemmArgs ga{};
  ga.B = B;
  ga.L = L;
  ga.nrb = (L + kRowBlock - 1) / kRowBlock;
  ga.R = R;
  ga.idx = idx;
  ga.q_feats = d;
  ga.kv_feats = kvf;
  ga.D = D;
  ga.rope_cos = w.rope_cos;
  ga.rope_sin = w.rope_sin;
  ga.slab = slab;
  ga.dev_err = dev_err;

  // 1. gather the recompute rows and normalise
  e = launch_pdl(rmsnorm_kernel<true>, norm_grid, dim3(256), 0, s, xs, idx, R, L, d,
                 static_cast<const uint16_t*>(w.gamma1), eps, xg, h, dev_err);
  // 2. q, k, v with RoPE
  if (e == cudaSuccess) {
    GemmArgs g = ga;
    g.K = d;
    g.n_ftiles = (d + 2 * kvf) / kTileM;
    g.out0 = q;
    g.out1 = kn;
    g.out2 = vn;
    e = launch_gemm<kEpiQkv>(m_wq, m_wk, m_wv, m_h, g, s);
  }
  // 3. the K/V refresh of the recompute set, 4. attention over the whole cache
  if (e == cudaSuccess) e = launch_kv_scatter(p, k_cache, v_cache, kn, vn, 0, idx, R, nullptr, nullptr, dev_err, s);
  if (e == cudaSuccess) {
    ec_status as = EC_OK;
    e = launch_partial_attention(p, q, k_cache, v_cache, R, 1.0f / sqrtf(static_cast<float>(D)), o, attn_ws, dev_err,
                                 false, s, &as);
    if (as != EC_OK) {
      *status = as;
      return e != cudaSuccess ? e : cudaErrorUnknown;
    }
  }
  // 5. x2 = xg + o Wo^T
  if (e == cudaSuccess) {
    GemmArgs g = ga;
    g.K = d;
    g.n_ftiles = d / kTileM;
    g.out0 = x2;
    g.res = xg;
    g.n_out = d;
    e = launch_gemm<kEpiResidual>(m_wo, m_wo, m_wo, m_o, g, s);
  }
  // 6. h2 = RMSNorm(x2) * gamma2, 7. SwiGLU, 8. y = x2 + act Wd^T
  if (e == cudaSuccess)
    e = launch_pdl(rmsnorm_kernel<false>, norm_grid, dim3(256), 0, s, static_cast<const uint16_t*>(x2), idx, R, L, d,
                   static_cast<const uint16_t*>(w.gamma2), eps, static_cast<uint16_t*>(nullptr), h, dev_err);
  if (e == cudaSuccess) {
    GemmArgs g = ga;
    g.K = d;
    g.n_ftiles = dff / 64;
    g.out0 = act;
    g.n_out = dff;
    e = launch_gemm<kEpiSwiglu>(m_wg, m_wu, m_wu, m_h, g, s);
  }
  if (e == cudaSuccess) {
    GemmArgs g = ga;
    g.K = dff;
    g.n_ftiles = d / kTileM;
    g.out0 = static_cast<uint16_t*>(y);
    g.res = x2;
    g.n_out = d;
    e = launch_gemm<kEpiResidual>(m_wd, m_wd, m_wd, m_act, g, s);
  }
  if (e != cudaSuccess) *status = EC_ERR_CUDA;
  return e;
}

}  // namespace ec
