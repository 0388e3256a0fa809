// ffn.h -- launch interface of the blockwise feed-forward GEMM (ffn.cu).
#pragma once
#include "kernels.h"

namespace ra {

// Device-side error sites of the feed-forward GEMM.
enum FfnErrSite : int {
  kSiteGemmProducer = 0x401,
  kSiteGemmMma = 0x402,
  kSiteGemmEpilogue = 0x404,
  kSiteGemmDrain = 0x405,
  kSiteGemmMisaligned = 0x4FF,
};

// Profiling kind of the feed-forward GEMM (matches the C ABI's list).
constexpr int kProfFfnGemm = 8;

// C = epilogue(A B^T) with A [rows][K] and B [N][K] bf16, K-major, through
// 128B-swizzled tensor maps (boxes of 64 x 128 for A, B and a bf16 C; 32 x
// 128 for an fp32 C), on CTA pairs.
//   kind 0: C = gelu(acc + bias)                      (bf16)
//   kind 1: C = acc + bias + resid                    (bf16)
//   kind 2: C = gelu'(acc + bias), and gelu(acc + bias) transposed through
//           tm_aux                                    (bf16, bf16)
//   kind 3: C = acc * resid   (resid: gelu'(a))       (bf16; with trans, also
//           transposed through tm_aux)
// The transposed outputs go to a [N][rows] tensor through tm_aux (64 x 64
// boxes, 128-byte swizzle), rows at or past the launch's end as zeros.
//   kind 4: C += acc                                  (fp32, TMA reduce-add)
// M rows of C starting at c_row0 are produced from M rows of A starting at
// a_row0; N % 256 == 0, K % 64 == 0; M is a multiple of 128 unless the rows
// end at c_rows.  Only rows [c_row0, min(c_row0 + M, c_rows)) of C and of
// the residual are touched.
struct FfnGemmArgs {
  CUtensorMap tm_a, tm_b, tm_c;
  CUtensorMap tm_aux;  // kinds 2, 3 with trans: the transposed output
  int M = 0, N = 0, K = 0, a_row0 = 0, c_row0 = 0, c_rows = 0, kind = 0;
  int group_rows = 8;  // tile order: row tiles per group (row tiles fastest inside a group)
  const float* bias = nullptr;
  const void* resid = nullptr;  // [c_rows][N] bf16 (kinds 1, 3)
  int trans = 0;                // kind 3: also write the transposed output
  int* err = nullptr;
  int n_sms = 0;
  int pair_clusters = 0;  // clusters of two CTAs resident at once (ffn_pair_max_clusters())
  LaunchTimer* timer = nullptr;
};

cudaError_t launch_ffn_gemm(const FfnGemmArgs& a, cudaStream_t stream);
size_t ffn_gemm_smem_bytes();
// Clusters of two CTAs of the pair kernel that fit on the device at once (0
// if none or the query fails).
int ffn_pair_max_clusters();

// out [cols][ld_out] = transpose of in [rows][cols] (bf16), columns
// [rows, rows_pad) of out zeroed; rows_pad <= ld_out.
cudaError_t launch_transpose_bf16(const void* in, void* out, int rows, int cols, int rows_pad, int ld_out,
                                  cudaStream_t stream);
// out[c] += sum_{r < rows} x[r][c]: x bf16 [rows][ld], cols even; fp32 out.
cudaError_t launch_colsum_add(const void* x, int rows, int cols, int ld, float* out, cudaStream_t stream);

}  // namespace ra
