// ulysses.cu -- the all-to-all layout transforms of Ulysses sequence
// parallelism, on one GPU.
//
// ("Large-scale distributed AI model training series: sequence
// parallelism", section 5 DeepSpeed-Ulysses.)  The input is sharded along
// the sequence: rank r holds tokens [rC, (r+1)C) of every head, C = L/N.
// Before attention an all-to-all gives every rank all L tokens of its H/N
// heads; attention then runs per head group, independently; a second
// all-to-all returns the output to the sequence shards.  With every rank on
// one GPU both all-to-alls are permutations between two layouts of the same
// tensor:
//   sequence shards  [N][B][H][C][d]    (rank r, token rC + i)
//   head shards      [N][B][H/N][L][d]  (rank p holds heads p H/N ..)
// so that element (r, b, h, i) of the first is element
// (h / (H/N), b, h % (H/N), rC + i) of the second.  The kernels copy 16
// bytes per thread (rows of d values: 128 or 256 bytes of bf16, 4 bytes of
// fp32 for lse) and are HBM-bound.
#include "kernels.h"

namespace ra {

namespace {

unsigned blocks_for(long long n) { return static_cast<unsigned>((n + 255) / 256); }

// Row index pairs: sequence-shard row s = ((r*B + b)*H + h)*C + i, head-
// shard row t = ((p*B + b)*Hn + hl)*L + r*C + i with p = h / Hn, hl = h % Hn.
__device__ __forceinline__ long long head_row(long long s, int B, int H, int Hn, int C, int N) {
  const int i = static_cast<int>(s % C);
  long long rest = s / C;
  const int h = static_cast<int>(rest % H);
  rest /= H;
  const int b = static_cast<int>(rest % B);
  const int r = static_cast<int>(rest / B);
  const int p = h / Hn, hl = h % Hn;
  return ((static_cast<long long>(p) * B + b) * Hn + hl) * (static_cast<long long>(C) * N) +
         static_cast<long long>(r) * C + i;
}

// vec16 = 16-byte vectors per row; to_heads: sequence shards -> head shards.
__global__ void __launch_bounds__(256) ulysses_a2a_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                          int vec16, int B, int H, int Hn, int C, int N,
                                                          int to_heads, long long n_vec) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n_vec) return;
  const int c = static_cast<int>(t % vec16);
  const long long s = t / vec16;  // row in the layout this thread walks
  if (to_heads) {
    dst[head_row(s, B, H, Hn, C, N) * vec16 + c] = src[s * vec16 + c];
  } else {
    dst[s * vec16 + c] = src[head_row(s, B, H, Hn, C, N) * vec16 + c];
  }
}

// The same permutation for one fp32 per row (lse): one value per thread.
__global__ void __launch_bounds__(256) ulysses_a2a_rows_kernel(const float* __restrict__ src, float* __restrict__ dst,
                                                               int B, int H, int Hn, int C, int N, int to_heads,
                                                               long long n_rows) {
  const long long s = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (s >= n_rows) return;
  if (to_heads)
    dst[head_row(s, B, H, Hn, C, N)] = src[s];
  else
    dst[s] = src[head_row(s, B, H, Hn, C, N)];
}

}  // namespace

cudaError_t launch_ulysses_a2a(const void* src, void* dst, int row_bytes, int B, int H, int N, int L, bool to_heads,
                               cudaStream_t stream) {
  const int C = L / N, Hn = H / N;
  const long long rows = static_cast<long long>(N) * B * H * C;
  if (row_bytes % 16 == 0) {
    const int vec16 = row_bytes / 16;
    const long long n = rows * vec16;
    ulysses_a2a_kernel<<<blocks_for(n), 256, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                          vec16, B, H, Hn, C, N, to_heads ? 1 : 0, n);
  } else {  // one fp32 per row
    ulysses_a2a_rows_kernel<<<blocks_for(rows), 256, 0, stream>>>(static_cast<const float*>(src),
                                                                  static_cast<float*>(dst), B, H, Hn, C, N,
                                                                  to_heads ? 1 : 0, rows);
  }
  return cudaGetLastError();
}

}  // namespace ra
