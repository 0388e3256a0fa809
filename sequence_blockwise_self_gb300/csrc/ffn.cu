// ffn.cu -- the blockwise feed-forward block on the sm_103a tensor cores.
//
// ("Large-scale distributed AI model training series: sequence
// parallelism", section 4.2 Blockwise Parallel Transformer: for each query
// block, attention, then the FFN and the residual connection; the FFN is
// the GPT-style pair of linear layers with a 4x up-projection, section 8.)
// For a block of rows x [R][D]:
//   h = gelu(x W1 + b1)      [R][F]   (exact GELU, x Phi(x))
//   y = x + h W2 + b2        [R][D]
// Only one block's hidden activation h exists at a time (the BPT memory
// saving), in a caller-provided buffer reused block after block.
//
// Both layers are one persistent GEMM kernel C = A B^T with A [M][K] and
// B [N][K] bf16 (K-major: the weights are passed transposed), fp32
// accumulation in tensor memory and a fused epilogue:
//   kind 0:  C = bf16(gelu(acc + bias[n]))
//   kind 1:  C = bf16(acc + bias[n] + resid[m][n])
// Tiles of 128 x 256 (one tcgen05.mma 128x256x16 per 16 of K, 128 cycles),
// K in stages of 64 through a 4-slot TMA ring.  Warp roles (256 threads):
//   warp 0      TMA producer (A and B tiles)
//   warp 1      tcgen05 issuer (converged warp, one elected lane)
//   warp 2      tensor-memory allocator
//   warps 4-7   epilogue: thread = output row (TMEM lane), 256 columns
// Two accumulators of 256 columns alternate between tiles, so the epilogue
// of one tile overlaps the products of the next.  Every wait is bounded (the
// attention kernels' scheme: abort flag, status word, drain).
#include <cmath>

#include "ffn.h"
#include "sm103_ptx.cuh"

namespace ra {

namespace {

constexpr int kGemmThreads = 256;
constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kATile = kBM * kBK * 2;  // 16 KB
constexpr int kBTile = kBN * kBK * 2;  // 32 KB

struct GemmSmem {
  alignas(1024) uint8_t a[kStages][kATile];
  alignas(1024) uint8_t b[kStages][kBTile];
  alignas(1024) uint8_t c[2][kBM * 64 * 2];  // output staging: two boxes of 128 rows x 64 columns
  alignas(8) uint64_t full[kStages];
  alignas(8) uint64_t empty[kStages];
  alignas(8) uint64_t acc_full[2];
  alignas(8) uint64_t acc_empty[2];
  alignas(8) uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct GemmDev {
  int M, N, K;          // M rows in this launch (ragged tail allowed), N % 256 == 0, K % 64 == 0
  int a_row0, c_row0;   // first row of this launch in the A and C tensor maps
  int c_rows;           // rows of the C tensor (the residual's rows; rows past it are not read)
  int kind;             // 0: gelu(acc + bias), 1: acc + bias + resid
  int group_rows;       // tile order, see tile_coords
  const float* bias;    // [N]
  const __nv_bfloat16* resid;  // [c_rows][N] (kind 1)
  int* err;
};

// Tile order: groups of G row tiles, row tiles fastest inside a group, so
// that the CTAs resident together share operand tiles in L2 and a group's
// rows of A stay there while its columns go by.
__device__ __forceinline__ void tile_coords(int tile, int n_m, int n_n, int G, int& m0, int& n0) {
  const int per_group = G * n_n;
  const int g = tile / per_group, w = tile % per_group;
  const int rows = min(G, n_m - g * G);
  m0 = (g * G + w % rows) * kBM;
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

__device__ __forceinline__ float gelu(float x) { return 0.5f * x * (1.f + erff(x * 0.70710678118654752f)); }

__global__ void __launch_bounds__(kGemmThreads, 1)
    ffn_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_c, const GemmDev p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kSiteGemmMisaligned);
    return;
  }
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_m = (p.M + kBM - 1) / kBM, n_n = p.N / kBN, n_tiles = n_m * n_n, n_k = p.K / kBK;
  // this CTA's tiles: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int my_tiles = blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  volatile int* ab = &sm.abort_flag;

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&sm.acc_full[a]), 1);
      mbar_init(smem_u32(&sm.acc_empty[a]), 128);
    }
    mbar_init(smem_u32(&sm.drain), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_c);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t total_uses = static_cast<uint32_t>(my_tiles) * n_k;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      uint32_t n = 0;
      for (int t = 0; t < my_tiles && ok; ++t) {
        int m0, n0;
        tile_coords(blockIdx.x + t * gridDim.x, n_m, n_n, p.group_rows, m0, n0);
        for (int ks = 0; ks < n_k && ok; ++ks, ++n) {
          const uint32_t s = n % kStages, use = n / kStages;
          if (use > 0) ok = mbar_wait(smem_u32(&sm.empty[s]), (use - 1) & 1, ab, p.err, kSiteGemmProducer);
          if (!ok) break;
          const uint32_t fb = smem_u32(&sm.full[s]);
          mbar_arrive_expect_tx(fb, kATile + kBTile);
          tma_load_3d(smem_u32(sm.a[s]), &tm_a, fb, ks * kBK, p.a_row0 + m0, 0);
          tma_load_3d(smem_u32(sm.b[s]), &tm_b, fb, ks * kBK, n0, 0);
        }
      }
      if (!ok) {  // let the copies in flight land before the CTA exits
        for (uint32_t i = 0; i < kStages && i < n; ++i) {
          const uint32_t last = i + kStages * ((n - 1 - i) / kStages);
          gemm_drain_wait(smem_u32(&sm.full[i]), (last / kStages) & 1, p.err);
        }
      }
    }
  } else if (warp == 1) {
    constexpr uint32_t kId = idesc_bf16(kBM, kBN, false, false);
    bool ok = true;
    uint32_t n = 0;
    for (int t = 0; t < my_tiles && ok; ++t) {
      const uint32_t acc = t & 1;
      if (t >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.acc_empty[acc]), ((t >> 1) - 1) & 1, ab, p.err,
                                               kSiteGemmMma));
      if (!ok) break;
      tc_fence_after();
      for (int ks = 0; ks < n_k && ok; ++ks, ++n) {
        const uint32_t s = n % kStages;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.full[s]), (n / kStages) & 1, ab, p.err, kSiteGemmMma));
        if (!ok) break;
        tc_fence_after();
        const uint32_t aa = smem_u32(sm.a[s]), ba = smem_u32(sm.b[s]);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          umma_ss_warp(tmem + acc * kBN, sdesc_sw128(aa + kk * 32, 16, 1024), sdesc_sw128(ba + kk * 32, 16, 1024), kId,
                       (ks > 0 || kk > 0) ? 1u : 0u);
        // the slot goes back to the producer once these products have read
        // it, if the producer will refill it
        if (n + kStages < total_uses) umma_commit_warp(smem_u32(&sm.empty[s]));
      }
      if (ok) umma_commit_warp(smem_u32(&sm.acc_full[acc]));
    }
    if (!ok) {
      umma_commit_warp(smem_u32(&sm.drain));
      gemm_drain_wait(smem_u32(&sm.drain), 0, p.err);
    }
  } else if (warp >= 4) {
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    bool ok = true;
    for (int t = 0; t < my_tiles && ok; ++t) {
      int m0, n0;
      tile_coords(blockIdx.x + t * gridDim.x, n_m, n_n, p.group_rows, m0, n0);
      const uint32_t acc = t & 1;
      // one decision for the four warps: they meet at named barriers below
      ok = named_bar_and(1, 128, mbar_wait(smem_u32(&sm.acc_full[acc]), (t >> 1) & 1, ab, p.err, kSiteGemmEpilogue));
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_acc = tmem + acc * kBN + lane_off;
      const int c_row = p.c_row0 + m0 + row;  // this thread's output row
      const bool has_res = p.kind == 1 && c_row < p.c_rows;
      const __nv_bfloat16* res_row = has_res ? p.resid + static_cast<size_t>(c_row) * p.N + n0 : nullptr;
      // four quarters of 64 columns, two staging boxes in turn
      for (int qtr = 0; qtr < 4; ++qtr) {
        const uint32_t box = smem_u32(sm.c[qtr & 1]);
        if (t > 0 || qtr >= 2) {  // the store that used this box two quarters ago has read it
          if (threadIdx.x == 128) bulk_wait_group_read<1>();
          named_bar_sync(1, 128);
        }
#pragma unroll
        for (int h32 = 0; h32 < 2; ++h32) {
          uint32_t r[32];
          const int col0 = qtr * 64 + h32 * 32;  // within the tile
          tmem_ld32(t_acc + col0, r);
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) + __ldg(p.bias + n0 + col0 + i);
          if (p.kind == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = gelu(v[i]);
          } else if (has_res) {
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              const uint4 rv = *reinterpret_cast<const uint4*>(res_row + col0 + 8 * c8);
              const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&rv);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float2 f = __bfloat1622float2(r2[j]);
                v[8 * c8 + 2 * j] += f.x;
                v[8 * c8 + 2 * j + 1] += f.y;
              }
            }
          }
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8)
            st_shared_v4(box + sw128_offset(row, h32 * 4 + c8), pack_bf16(v[8 * c8], v[8 * c8 + 1]),
                         pack_bf16(v[8 * c8 + 2], v[8 * c8 + 3]), pack_bf16(v[8 * c8 + 4], v[8 * c8 + 5]),
                         pack_bf16(v[8 * c8 + 6], v[8 * c8 + 7]));
        }
        if (qtr == 3) {  // every column of this accumulator has been read
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.acc_empty[acc]));
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (threadIdx.x == 128) {
          tma_store_3d(&tm_c, box, n0 + qtr * 64, p.c_row0 + m0, 0);
          bulk_commit_group();
        }
      }
    }
    if (threadIdx.x == 128) bulk_wait_group<0>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t ffn_gemm_smem_bytes() { return sizeof(GemmSmem); }

cudaError_t launch_ffn_gemm(const FfnGemmArgs& a, cudaStream_t stream) {
  GemmDev p;
  p.M = a.M; p.N = a.N; p.K = a.K;
  p.a_row0 = a.a_row0; p.c_row0 = a.c_row0; p.c_rows = a.c_rows;
  p.kind = a.kind; p.bias = a.bias;
  p.group_rows = a.group_rows > 0 ? a.group_rows : 1;
  p.resid = static_cast<const __nv_bfloat16*>(a.resid);
  p.err = a.err;
  const int n_sms = a.n_sms;
  const int n_tiles = ((a.M + kBM - 1) / kBM) * (a.N / kBN);
  const int grid = n_tiles < n_sms ? n_tiles : n_sms;
  const size_t smem = sizeof(GemmSmem);
  cudaError_t e = cudaFuncSetAttribute(ffn_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (a.timer) a.timer->mark(kProfFfnGemm, false, stream);
  ffn_gemm_kernel<<<grid, kGemmThreads, smem, stream>>>(a.tm_a, a.tm_b, a.tm_c, p);
  if (a.timer) a.timer->mark(kProfFfnGemm, true, stream);
  return cudaGetLastError();
}

}  // namespace ra
