// ffn.cu -- the blockwise feed-forward block on the sm_103a tensor cores.
//
// ("Large-scale distributed AI model training series: sequence
// parallelism", section 4.2 Blockwise Parallel Transformer: for each query
// block, attention, then the FFN and the residual connection; the FFN is
// the GPT-style pair of linear layers with a 4x up-projection, section 8.)
// For a block of rows x [R][D]:
//   h = gelu(x W1 + b1)      [R][F]   (exact GELU, x Phi(x), Phi the normal CDF)
//   y = x + h W2 + b2        [R][D]
// Only one block's hidden activation h exists at a time (the BPT memory
// saving), in a caller-provided buffer reused block after block.
//
// The backward (same section: the block's activations are recomputed, not
// kept) differentiates the loss sum(dy * y) block by block:
//   a = x W1 + b1, g = gelu'(a), h = gelu(a)     (recomputed)
//   dW2 += h^T dy    da = (dy W2^T) * g    dx = dy + da W1^T    dW1 += x^T da
//
// Every product is one persistent GEMM kernel C = A B^T with A [M][K] and
// B [N][K] bf16 (K-major: the weights are passed output-major), fp32
// accumulation in tensor memory and a fused epilogue:
//   kind 0:  C = bf16(gelu(acc + bias[n]))                 forward layer 1
//   kind 1:  C = bf16(acc + bias[n] + resid[m][n])         forward layer 2, dx
//   kind 2:  C = bf16(gelu'(a)), h^T = bf16(gelu(a))^T     recompute (a = acc + bias)
//   kind 3:  C = bf16(acc * g[m][n]) (and C^T)             da
//   kind 4:  C (fp32) += acc, TMA reduce-add               dW1, dW2
// It runs on CTA pairs (clusters of two CTAs on the two SMs of a TPC,
// tcgen05 cta_group::2): 256 x 256 output tiles, each CTA staging its 128
// rows of A and 128 of the 256 rows of B^T per 64-deep K stage, the even
// CTA issuing the 256x256x16 products.  Per SM a stage then moves 32 KB
// through shared memory for 128x256x64 of product; a single CTA computing
// 128 x 256 would move 48 KB, and the TMA writes plus tensor-core reads of
// that traffic are what bounds a single-CTA tile below the tensor peak.
// Warp roles (256 threads per CTA):
//   warp 0      TMA producer (A and B halves), both CTAs
//   warp 1      tcgen05 issuer (converged warp, one elected lane), even CTA
//   warp 2      tensor-memory allocator (collective over the pair)
//   warps 4-7   epilogue: thread = output row (TMEM lane), 256 columns
// Two accumulators of 256 columns alternate between tiles, so the epilogue
// of one tile overlaps the products of the next.  Every wait is bounded (the
// attention kernels' scheme: abort flag, status word, drain); both CTAs of
// a pair always meet at the cluster barriers around the work.
#include <cmath>

#include "ffn.h"
#include "sm103_pair.cuh"
#include "sm103_ptx.cuh"

namespace ra {

namespace {

constexpr int kGemmThreads = 256;
constexpr int kBM = 128, kBN = 256, kBK = 64;  // rows per CTA, columns per tile, K per stage

struct GemmDev {
  int M, N, K;          // M rows in this launch (ragged tail allowed), N % 256 == 0, K % 64 == 0
  int a_row0, c_row0;   // first row of this launch in the A and C tensor maps
  int c_rows;           // rows of the C tensor (the residual's rows; rows past it are not read)
  int c_end;            // rows [c_row0, c_end) of C belong to this launch: no other row is read or written
  int kind;             // see FfnGemmArgs::kind
  int trans;            // kind 3: also store the transposed output through tm_aux
  int group_rows;       // tile order, see tile_coords
  const float* bias;    // [N] (kinds 0, 1, 2)
  const __nv_bfloat16* resid;  // [c_rows][N]: the residual (kind 1), gelu'(a) (kind 3)
  int* err;
};

// Tile order: groups of G row tiles, row tiles fastest inside a group, so
// that the CTAs resident together share operand tiles in L2 and a group's
// rows of A stay there while its columns go by.
__device__ __forceinline__ void tile_coords(int tile, int n_m, int n_n, int G, int tile_m, int& m0, int& n0) {
  const int per_group = G * n_n;
  const int g = tile / per_group, w = tile % per_group;
  const int rows = min(G, n_m - g * G);
  m0 = (g * G + w % rows) * tile_m;
  n0 = (w / rows) * kBN;
}

// bar.red.and over `nthreads` threads of named barrier `id`: every thread
// gets the conjunction of the predicates.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ void gemm_drain_wait(uint32_t bar, uint32_t parity, int* err) {
  int local = 0;
  mbar_wait(bar, parity, &local, err, kSiteGemmDrain);
}

// 16-byte copy global -> shared that bypasses L1 (cp.async, one group per
// commit); the issuing thread waits for its groups with cp_async_wait_all.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Phi(a), the standard normal distribution function, for the exact GELU
// a Phi(a) and its derivative Phi(a) + a phi(a).  From the complementary
// error function, z = |a| / sqrt 2: Phi(a) = erfc(z) / 2 for a < 0 and
// 1 - erfc(z) / 2 otherwise, with erfc(z) = t exp(-z^2 + c(t)),
// t = 1 / (1 + z / 2), c the degree-9 Chebyshev-fitted polynomial of
// Numerical Recipes in C (2nd ed., section 6.2, erfcc), whose fractional
// error is below 1.2e-7 for every z >= 0.  Unlike (1 + erf(a / sqrt 2)) / 2,
// which cancels in fp32 (to exactly 0 below a = -5.4), the tail a << 0
// keeps its relative accuracy.  z2 = a^2 / 2.
__device__ __forceinline__ float normal_cdf(float a, float z2) {
  const float z = fabsf(a) * 0.70710678118654752f;
  const float t = __fdividef(1.f, fmaf(0.5f, z, 1.f));
  float c = 0.17087277f;
  c = fmaf(c, t, -0.82215223f);
  c = fmaf(c, t, 1.48851587f);
  c = fmaf(c, t, -1.13520398f);
  c = fmaf(c, t, 0.27886807f);
  c = fmaf(c, t, -0.18628806f);
  c = fmaf(c, t, 0.09678418f);
  c = fmaf(c, t, 0.37409196f);
  c = fmaf(c, t, 1.00002368f);
  c = fmaf(c, t, -1.26551223f);
  const float half_erfc = 0.5f * t * __expf(c - z2);
  return a < 0.f ? half_erfc : 1.f - half_erfc;
}

__device__ __forceinline__ float gelu(float x) { return x * normal_cdf(x, 0.5f * x * x); }

// The epilogue of one output tile for the 128 rows this CTA holds (thread =
// row = tensor-memory lane): accumulator columns [t_acc, t_acc + 256) ->
// + bias (bias_s: the tile's 256 columns, staged in shared memory), then
// GELU (kind 0) or + residual (kind 1); or, kind 3 without the transposed
// output, times gelu'(a) -> bf16 into two 64-column staging boxes in turn
// -> TMA stores of 128 x 64.  c_row0 is the
// C row of lane 0; boxes_in_use says whether stores of an earlier tile may
// still be reading the boxes.  release() runs once every accumulator column
// has been read.  Called by the 128 epilogue threads (named barrier 1).
template <class Release>
__device__ __forceinline__ void epilogue_tile(const GemmDev& p, const CUtensorMap* tm_c, uint32_t box0, uint32_t box1,
                                              uint32_t t_acc, const float* bias_s, int row, int c_row0, int n0,
                                              bool boxes_in_use, Release release) {
  const int c_row = c_row0 + row;  // this thread's output row
  const bool has_res = (p.kind == 1 || p.kind == 3) && c_row < p.c_end;
  // a box starts on a 128-row boundary of the launch, whose rows end on one
  // or at the end of C: it lies inside the launch's rows, or all past them
  const bool store = c_row0 < p.c_end;
  const __nv_bfloat16* res_row = has_res ? p.resid + static_cast<size_t>(c_row) * p.N + n0 : nullptr;
  for (int qtr = 0; qtr < 4; ++qtr) {
    const uint32_t box = (qtr & 1) ? box1 : box0;
    if (boxes_in_use || qtr >= 2) {  // the store that used this box two quarters ago has read it
      if (threadIdx.x == 128) bulk_wait_group_read<1>();
      named_bar_sync(1, 128);
    }
#pragma unroll
    for (int h32 = 0; h32 < 2; ++h32) {
      uint32_t r[32];
      const int col0 = qtr * 64 + h32 * 32;  // within the tile
      tmem_ld32(t_acc + col0, r);
      float v[32];
      if (p.kind == 3) {  // no bias: the product is scaled elementwise below
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) + bias_s[col0 + i];
      }
      if (p.kind == 0) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gelu(v[i]);
      } else if (has_res) {  // kind 1: + residual; kind 3: times gelu'(a)
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          const uint4 rv = *reinterpret_cast<const uint4*>(res_row + col0 + 8 * c8);
          const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&rv);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(r2[j]);
            if (p.kind == 1) {
              v[8 * c8 + 2 * j] += f.x;
              v[8 * c8 + 2 * j + 1] += f.y;
            } else {
              v[8 * c8 + 2 * j] *= f.x;
              v[8 * c8 + 2 * j + 1] *= f.y;
            }
          }
        }
      }
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8)
        st_shared_v4(box + sw128_offset(row, h32 * 4 + c8), pack_bf16(v[8 * c8], v[8 * c8 + 1]),
                     pack_bf16(v[8 * c8 + 2], v[8 * c8 + 3]), pack_bf16(v[8 * c8 + 4], v[8 * c8 + 5]),
                     pack_bf16(v[8 * c8 + 6], v[8 * c8 + 7]));
    }
    if (qtr == 3) release();  // every column of this accumulator has been read
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    if (threadIdx.x == 128 && store) {
      tma_store_3d(tm_c, box, n0 + qtr * 64, c_row0, 0);
      bulk_commit_group();
    }
  }
}

// Epilogues with a second, transposed output (the backward's recomputation
// of the first layer, kind 2, and da, kind 3 with tm_aux): per quarter of 64
// columns the normal output is staged in box0 (128-byte swizzle, stored by
// TMA through tm_c) and the transposed output in box1 as two 64 x 64 tiles
// [column][row], 128-byte swizzled, stored through tm_aux (a map over the
// transposed tensor [N][rows], box 64 x 64).  Two neighbouring rows (lanes
// 2j, 2j+1) swap one value so that each writes one 32-bit pair: the even
// lane the pair of column c, the odd lane that of column c+1.  Rows at or
// past c_end go to the transposed output as zeros: they pad the
// weight-gradient GEMMs' K.
//   kind 2: a = acc + bias; normal gelu'(a) = Phi(a) + a phi(a), transposed
//           h = gelu(a) = a Phi(a) (two exponentials per element)
//   kind 3: normal and transposed da = acc * gelu'(a) (gelu'(a) from resid)
template <class Release>
__device__ __forceinline__ void epilogue_tile_trans(const GemmDev& p, const CUtensorMap* tm_c,
                                                    const CUtensorMap* tm_aux, uint32_t box0, uint32_t box1,
                                                    uint32_t t_acc, const float* bias_s, int row, int c_row0, int n0,
                                                    bool boxes_in_use, Release release) {
  const int c_row = c_row0 + row;
  const bool live = c_row < p.c_end;
  const bool store = c_row0 < p.c_end;
  const __nv_bfloat16* res_row = (p.kind == 3 && live) ? p.resid + static_cast<size_t>(c_row) * p.N + n0 : nullptr;
  // this thread's pair of rows in the transposed tile: tile row / 64, byte
  // offset 2 (row % 64) rounded down to the pair, in 16-byte chunk
  // (row % 64) / 8 of the tile's 128-byte rows (swizzled by the tile row)
  const uint32_t tbox = box1 + static_cast<uint32_t>(row >> 6) * 8192u;
  const uint32_t tchunk = static_cast<uint32_t>(row & 63) >> 3, tin = (static_cast<uint32_t>(row & 7) & ~1u) * 2u;
  const bool odd = row & 1;
  for (int qtr = 0; qtr < 4; ++qtr) {
#pragma unroll
    for (int h32 = 0; h32 < 2; ++h32) {
      uint32_t r[32];
      const int col0 = qtr * 64 + h32 * 32;
      tmem_ld32(t_acc + col0, r);
      uint32_t nw[16], tw[16];  // packed bf16 pairs: normal (4 per c8), transposed (4 per c8)
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        float nv[8], tv[8];
        if (p.kind == 2) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float a = __uint_as_float(r[8 * c8 + i]) + bias_s[col0 + 8 * c8 + i];
            const float z2 = 0.5f * a * a;
            const float Phi = normal_cdf(a, z2);
            const float phi = 0.3989422804014327f * __expf(-z2);  // exp(-a^2 / 2) / sqrt(2 pi)
            nv[i] = fmaf(a, phi, Phi);
            tv[i] = a * Phi;
          }
        } else {
          float gr[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (live) {
            const uint4 rv = *reinterpret_cast<const uint4*>(res_row + col0 + 8 * c8);
            const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&rv);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 f = __bfloat1622float2(r2[j]);
              gr[2 * j] = f.x;
              gr[2 * j + 1] = f.y;
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) nv[i] = tv[i] = __uint_as_float(r[8 * c8 + i]) * gr[i];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) nw[4 * c8 + j] = pack_bf16(nv[2 * j], nv[2 * j + 1]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float a0 = live ? tv[2 * j] : 0.f, a1 = live ? tv[2 * j + 1] : 0.f;
          // even lane keeps column c and sends c+1, odd lane the reverse
          const float other = __shfl_xor_sync(0xffffffffu, odd ? a0 : a1, 1);
          tw[4 * c8 + j] = odd ? pack_bf16(other, a1) : pack_bf16(a0, other);
        }
      }
      // the stores of the previous quarter have read both buffers: waited for
      // after the first half's arithmetic, which overlaps them
      if (h32 == 0 && (boxes_in_use || qtr > 0)) {
        if (threadIdx.x == 128) bulk_wait_group_read<0>();
        named_bar_sync(1, 128);
      }
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        st_shared_v4(box0 + sw128_offset(row, h32 * 4 + c8), nw[4 * c8], nw[4 * c8 + 1], nw[4 * c8 + 2], nw[4 * c8 + 3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t c = static_cast<uint32_t>(h32 * 32 + 8 * c8 + 2 * j) + (odd ? 1u : 0u);  // tile row
          const uint32_t addr = tbox + c * 128u + (((tchunk ^ (c & 7u)) << 4) | tin);
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(tw[4 * c8 + j]) : "memory");
        }
      }
    }
    if (qtr == 3) release();
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    if (threadIdx.x == 128 && store) {
      tma_store_3d(tm_c, box0, n0 + qtr * 64, c_row0, 0);
      tma_store_3d(tm_aux, box1, c_row0, n0 + qtr * 64, 0);
      tma_store_3d(tm_aux, box1 + 8192u, c_row0 + 64, n0 + qtr * 64, 0);
      bulk_commit_group();
    }
  }
}

// Kind 4: C (fp32) += acc, by TMA reduce-add of eight 32-column boxes of
// 128 rows (128-byte rows), the two staging buffers in turn; otherwise as
// epilogue_tile.
template <class Release>
__device__ __forceinline__ void epilogue_tile_add(const GemmDev& p, const CUtensorMap* tm_c, uint32_t box0,
                                                  uint32_t box1, uint32_t t_acc, int row, int c_row0, int n0,
                                                  bool boxes_in_use, Release release) {
  const bool store = c_row0 < p.c_end;
  for (int e = 0; e < kBN / 32; ++e) {
    const uint32_t box = (e & 1) ? box1 : box0;
    if (boxes_in_use || e >= 2) {  // the reduction that used this box two steps ago has read it
      if (threadIdx.x == 128) bulk_wait_group_read<1>();
      named_bar_sync(1, 128);
    }
    uint32_t r[32];
    tmem_ld32(t_acc + 32 * e, r);
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
      st_shared_v4(box + sw128_offset(row, ch), r[4 * ch], r[4 * ch + 1], r[4 * ch + 2], r[4 * ch + 3]);
    if (e == kBN / 32 - 1) release();  // every column of this accumulator has been read
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    if (threadIdx.x == 128 && store) {
      tma_reduce_add_3d(tm_c, box, n0 + 32 * e, c_row0, 0);
      bulk_commit_group();
    }
  }
}

constexpr int kPairStages = 6;
constexpr int kPairBRows = kBN / 2;               // rows of B^T each CTA stages
constexpr int kPairATile = kBM * kBK * 2;         // 16 KB
constexpr int kPairBTile = kPairBRows * kBK * 2;  // 16 KB

struct PairSmem {
  alignas(1024) uint8_t a[kPairStages][kPairATile];
  alignas(1024) uint8_t b[kPairStages][kPairBTile];
  alignas(1024) uint8_t c[2][kBM * 64 * 2];
  alignas(16) float bias[2][kBN];          // kinds 0-2: a tile's bias columns, staged one tile ahead
  alignas(8) uint64_t full[kPairStages];   // even CTA: both CTAs' operand bytes of a stage
  alignas(8) uint64_t empty[kPairStages];  // each CTA: its stage may be refilled
  alignas(8) uint64_t acc_full[2];         // each CTA: accumulator ready
  alignas(8) uint64_t acc_empty[2];        // even CTA: both CTAs' epilogues have read the accumulator
  alignas(8) uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// The same GEMM on CTA pairs: 256 x 256 output tiles, one per cluster of
// two CTAs at a time (persistent over tiles), K in stages of 64 through a
// 6-slot ring in each CTA.  Per stage each CTA loads its 128 rows of A and
// its 128 rows of B^T (16 KB each); both loads complete on the even CTA's
// `full` barrier, which expects the 64 KB of the pair.  The even CTA's MMA
// warp issues the four 256x256x16 products of a stage and commits to the
// `empty` barriers of both CTAs (multicast); after a tile it commits to
// both `acc_full` barriers.  Each CTA's epilogue reads its own 128 rows and
// signals the even CTA's `acc_empty` (one arrival per warp, 8 in all).
// Per SM a stage moves 32 KB through shared memory for 128x256x64 of
// product, against 48 KB for the single-CTA 128x256 tile.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    ffn_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_aux,
                         const GemmDev p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the same for both CTAs (same kernel, same layout): skipping the work
  // keeps the collective steps (allocation, cluster barriers) on both sides
  const bool misaligned = (smem_u32(smem_raw) & 1023u) != 0;
  PairSmem& sm = *reinterpret_cast<PairSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const uint32_t leader = rank & ~1u;
  const int pair = static_cast<int>(blockIdx.x >> 1), n_pairs = static_cast<int>(gridDim.x >> 1);
  const int tile_m = 2 * kBM;
  const int n_m = (p.M + tile_m - 1) / tile_m, n_n = p.N / kBN, n_tiles = n_m * n_n, n_k = p.K / kBK;
  const int my_tiles = misaligned ? 0 : (pair < n_tiles ? (n_tiles - 1 - pair) / n_pairs + 1 : 0);
  volatile int* ab = &sm.abort_flag;

  if (threadIdx.x == 0) {
    if (misaligned) atomicCAS(p.err, 0, kSiteGemmMisaligned);
    sm.abort_flag = 0;
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sm.acc_full[a]), 1);
      mbar_init(smem_u32(&sm.acc_empty[a]), 8);
    }
    mbar_init(smem_u32(&sm.drain), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_c);
    if (p.kind == 2 || p.trans) tma_prefetch_desc(&tm_aux);
  }
  if (warp == 2) {  // one warp in each CTA of the pair, collectively
    tmem_alloc_pair(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and tensor memory allocated on both sides
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t total_uses = static_cast<uint32_t>(my_tiles) * n_k;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      uint32_t n = 0;
      const uint32_t full0 = mapa_shared(smem_u32(&sm.full[0]), leader);
      for (int t = 0; t < my_tiles && ok; ++t) {
        int m0, n0;
        tile_coords(pair + t * n_pairs, n_m, n_n, p.group_rows, tile_m, m0, n0);
        for (int ks = 0; ks < n_k && ok; ++ks, ++n) {
          const uint32_t s = n % kPairStages, use = n / kPairStages;
          if (use > 0)
            ok = mbar_wait_cluster(smem_u32(&sm.empty[s]), (use - 1) & 1, ab, p.err, kSiteGemmProducer);
          if (!ok) break;
          if (rank == leader) mbar_arrive_expect_tx(smem_u32(&sm.full[s]), 2 * (kPairATile + kPairBTile));
          const uint32_t fb = full0 + 8u * s;
          tma_load_3d_pair(smem_u32(sm.a[s]), &tm_a, fb, ks * kBK, p.a_row0 + m0 + kBM * static_cast<int>(rank - leader),
                           0);
          tma_load_3d_pair(smem_u32(sm.b[s]), &tm_b, fb, ks * kBK, n0 + kPairBRows * static_cast<int>(rank - leader),
                           0);
        }
      }
      if (!ok && rank == leader) {  // let the copies in flight land before the pair exits
        for (uint32_t i = 0; i < kPairStages && i < n; ++i) {
          const uint32_t last = i + kPairStages * ((n - 1 - i) / kPairStages);
          gemm_drain_wait(smem_u32(&sm.full[i]), (last / kPairStages) & 1, p.err);
        }
      }
    }
  } else if (warp == 1) {
    if (rank == leader) {
      constexpr uint32_t kId = idesc_bf16(2 * kBM, kBN, false, false);
      const uint16_t both = static_cast<uint16_t>(3u << leader);
      bool ok = true;
      uint32_t n = 0;
      for (int t = 0; t < my_tiles && ok; ++t) {
        const uint32_t acc = t & 1;
        if (t >= 2)
          ok = __all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&sm.acc_empty[acc]), ((t >> 1) - 1) & 1, ab,
                                                         p.err, kSiteGemmMma));
        if (!ok) break;
        tc_fence_after();
        for (int ks = 0; ks < n_k && ok; ++ks, ++n) {
          const uint32_t s = n % kPairStages;
          ok = __all_sync(0xffffffffu,
                          mbar_wait_cluster(smem_u32(&sm.full[s]), (n / kPairStages) & 1, ab, p.err, kSiteGemmMma));
          if (!ok) break;
          tc_fence_after();
          const uint32_t aa = smem_u32(sm.a[s]), ba = smem_u32(sm.b[s]);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_pair_warp(tmem + acc * kBN, sdesc_sw128(aa + kk * 32, 16, 1024), sdesc_sw128(ba + kk * 32, 16, 1024),
                           kId, (ks > 0 || kk > 0) ? 1u : 0u);
          if (n + kPairStages < total_uses) umma_commit_pair_mc_warp(smem_u32(&sm.empty[s]), both);
        }
        if (ok) umma_commit_pair_mc_warp(smem_u32(&sm.acc_full[acc]), both);
      }
      if (!ok) {
        umma_commit_pair_mc_warp(smem_u32(&sm.drain), static_cast<uint16_t>(1u << leader));
        gemm_drain_wait(smem_u32(&sm.drain), 0, p.err);
      }
    }
  } else if (warp >= 4) {
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t acc_empty0 = mapa_shared(smem_u32(&sm.acc_empty[0]), leader);
    // kinds 0-2: a tile's 256 bias columns are copied into sm.bias[t & 1] by
    // the first 64 epilogue threads a whole tile ahead, so that the epilogue
    // reads them from shared memory instead of waiting on L2 for each group
    // of columns (the bias pointer is 16-byte aligned, N % 256 == 0)
    const bool stage_bias = p.kind <= 2;
    auto fetch_bias = [&](int tt) {
      if (!stage_bias || tt >= my_tiles || row >= kBN / 4) return;
      int bm0, bn0;
      tile_coords(pair + tt * n_pairs, n_m, n_n, p.group_rows, tile_m, bm0, bn0);
      cp_async_16(smem_u32(&sm.bias[tt & 1][4 * row]), p.bias + bn0 + 4 * row);
      cp_async_commit();
    };
    bool ok = true;
    fetch_bias(0);
    for (int t = 0; t < my_tiles && ok; ++t) {
      int m0, n0;
      tile_coords(pair + t * n_pairs, n_m, n_n, p.group_rows, tile_m, m0, n0);
      const uint32_t acc = t & 1;
      cp_async_wait_all();  // this thread's copies of tile t's columns; the barrier publishes them
      ok = named_bar_and(1, 128, mbar_wait_cluster(smem_u32(&sm.acc_full[acc]), (t >> 1) & 1, ab, p.err,
                                                   kSiteGemmEpilogue));
      if (!ok) break;
      tc_fence_after();
      fetch_bias(t + 1);  // every epilogue thread has finished tile t - 1, the last reader of that buffer
      const float* bias_s = sm.bias[acc];
      auto release = [&] {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8u * acc);
      };
      const int c_row0 = p.c_row0 + m0 + kBM * static_cast<int>(rank - leader);
      if (p.kind == 4)
        epilogue_tile_add(p, &tm_c, smem_u32(sm.c[0]), smem_u32(sm.c[1]), tmem + acc * kBN + lane_off, row, c_row0,
                          n0, t > 0, release);
      else if (p.kind == 2 || (p.kind == 3 && p.trans))
        epilogue_tile_trans(p, &tm_c, &tm_aux, smem_u32(sm.c[0]), smem_u32(sm.c[1]), tmem + acc * kBN + lane_off,
                            bias_s, row, c_row0, n0, t > 0, release);
      else
        epilogue_tile(p, &tm_c, smem_u32(sm.c[0]), smem_u32(sm.c[1]), tmem + acc * kBN + lane_off, bias_s, row,
                      c_row0, n0, t > 0, release);
    }
    cp_async_wait_all();  // no copy into this CTA's memory outlives it (a tile ahead, after an abort)
    if (threadIdx.x == 128) bulk_wait_group<0>();
  }
  tc_fence_before();
  cluster_sync_all();  // no more products, arrivals or reads of the peer's memory
  tc_fence_after();
  if (warp == 2) tmem_dealloc_pair(tmem, 512);
}

// out[c][r] = in[r][c] for bf16 in [rows][cols] (row stride cols) and out
// [cols][ld_out]; columns r in [rows, rows_pad) of out are zero (the K
// padding of the weight-gradient GEMMs).  64 x 64 tiles through shared
// memory, two bf16 per 32-bit access on both sides.  HBM-bound.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const __nv_bfloat16* __restrict__ in,
                                                            __nv_bfloat16* __restrict__ out, int rows, int cols,
                                                            int rows_pad, int ld_out) {
  __shared__ __nv_bfloat16 tile[64][66];
  const int c0 = blockIdx.x * 64, r0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int i = ty; i < 64; i += 8) {
    const int r = r0 + i, c = c0 + 2 * tx;
    __nv_bfloat162 v = __floats2bfloat162_rn(0.f, 0.f);
    if (r < rows && c < cols) v = *reinterpret_cast<const __nv_bfloat162*>(in + static_cast<size_t>(r) * cols + c);
    tile[i][2 * tx] = v.x;
    tile[i][2 * tx + 1] = v.y;
  }
  __syncthreads();
  for (int i = ty; i < 64; i += 8) {
    const int c = c0 + i, r = r0 + 2 * tx;
    if (c < cols && r < rows_pad) {
      __nv_bfloat162 v;
      v.x = tile[2 * tx][i];
      v.y = tile[2 * tx + 1][i];
      *reinterpret_cast<__nv_bfloat162*>(out + static_cast<size_t>(c) * ld_out + r) = v;
    }
  }
}

// out[c] += sum over rows r < rows of x[r][c] (bf16 x, row stride ld, cols
// even): one thread per two columns and a slice of rows per block row,
// partial sums added with fp32 atomics.
__global__ void __launch_bounds__(256) colsum_add_kernel(const __nv_bfloat16* __restrict__ x, int rows, int cols, int ld,
                                                        int rows_per_block, float* __restrict__ out) {
  const int c = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (c >= cols) return;
  const int r0 = blockIdx.y * rows_per_block, r1 = min(rows, r0 + rows_per_block);
  float s0 = 0.f, s1 = 0.f;
  for (int r = r0; r < r1; ++r) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + static_cast<size_t>(r) * ld + c));
    s0 += f.x;
    s1 += f.y;
  }
  atomicAdd(out + c, s0);
  atomicAdd(out + c + 1, s1);
}

}  // namespace

size_t ffn_gemm_smem_bytes() { return sizeof(PairSmem); }

int ffn_pair_max_clusters() {
  const size_t smem = sizeof(PairSmem);
  if (cudaFuncSetAttribute(ffn_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, ffn_gemm_pair_kernel, &cfg) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_ffn_gemm(const FfnGemmArgs& a, cudaStream_t stream) {
  GemmDev p;
  p.M = a.M; p.N = a.N; p.K = a.K;
  p.a_row0 = a.a_row0; p.c_row0 = a.c_row0; p.c_rows = a.c_rows;
  p.c_end = a.c_row0 + a.M < a.c_rows ? a.c_row0 + a.M : a.c_rows;
  p.kind = a.kind; p.bias = a.bias;
  p.trans = a.kind == 3 && a.trans ? 1 : 0;
  p.group_rows = a.group_rows > 0 ? a.group_rows : 1;
  p.resid = static_cast<const __nv_bfloat16*>(a.resid);
  p.err = a.err;
  if (a.pair_clusters <= 0) return cudaErrorInvalidConfiguration;
  // kinds 0-2 stage the bias by 16-byte copies
  if (a.kind <= 2 && (!a.bias || (reinterpret_cast<uintptr_t>(a.bias) & 15u))) return cudaErrorInvalidValue;
  const int n_tiles = ((a.M + 2 * kBM - 1) / (2 * kBM)) * (a.N / kBN);
  const int clusters = n_tiles < a.pair_clusters ? n_tiles : a.pair_clusters;
  const size_t smem = sizeof(PairSmem);
  const cudaError_t e =
      cudaFuncSetAttribute(ffn_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (a.timer) a.timer->mark(kProfFfnGemm, false, stream);
  const bool aux = a.kind == 2 || (a.kind == 3 && a.trans);
  ffn_gemm_pair_kernel<<<2 * clusters, kGemmThreads, smem, stream>>>(a.tm_a, a.tm_b, a.tm_c, aux ? a.tm_aux : a.tm_c,
                                                                      p);
  if (a.timer) a.timer->mark(kProfFfnGemm, true, stream);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const void* in, void* out, int rows, int cols, int rows_pad, int ld_out,
                                  cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((cols + 63) / 64), static_cast<unsigned>((rows_pad + 63) / 64));
  transpose_bf16_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(in),
                                                  static_cast<__nv_bfloat16*>(out), rows, cols, rows_pad, ld_out);
  return cudaGetLastError();
}

cudaError_t launch_colsum_add(const void* x, int rows, int cols, int ld, float* out, cudaStream_t stream) {
  const int rows_per_block = 256;
  const dim3 grid(static_cast<unsigned>((cols / 2 + 255) / 256), static_cast<unsigned>((rows + rows_per_block - 1) /
                                                                                          rows_per_block));
  colsum_add_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), rows, cols, ld, rows_per_block,
                                              out);
  return cudaGetLastError();
}

}  // namespace ra
