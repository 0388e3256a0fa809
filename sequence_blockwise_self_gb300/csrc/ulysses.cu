// ulysses.cu -- the all-to-all layout transforms of Ulysses and USP
// sequence parallelism, on one GPU.
//
// ("Large-scale distributed AI model training series: sequence
// parallelism", section 5 DeepSpeed-Ulysses and section 8.2 USP.)  The
// input is sharded along the sequence over N = U R ranks, rank n = r U + u
// (ring group r, Ulysses rank u) holding C = L/N tokens of every head.  An
// all-to-all within each Ulysses group of U ranks gives every rank all of
// its group's tokens for H/U heads; attention then runs per head group as a
// ring over the R groups (plain Ulysses: R = 1); a second all-to-all returns
// the output to the sequence shards.  With every rank on one GPU both
// all-to-alls are permutations between two layouts of the same tensor:
//   sequence shards  [N][B][H][C][row]      (rank n, its token i)
//   head groups      [U][B][H/U][L][row]    (natural token order)
// Token i of rank (r, u) is sequence position
//   encoder, or R = 1:  n C + i  (contiguous shards)
//   causal, R > 1:      the ring's fold, sub-chunks {r, 2R-1-r} of
//                       c = L/(2R) tokens for group r, each split into U
//                       pieces of c/U: i < c/U -> r c + u c/U + i, else
//                       (2R-1-r) c + u c/U + (i - c/U)
// so that the fused kernel's fold over R chunks is USP's load-balanced
// ring.  The kernels copy 16 bytes per thread (rows of d values: 128 or
// 256 bytes of bf16, 4 bytes of fp32 for lse) and are HBM-bound.
#include <climits>

#include "kernels.h"

namespace ra {

namespace {

unsigned blocks_for(long long n) { return static_cast<unsigned>((n + 255) / 256); }

struct UspMap {
  int B, H, Hn, C, U, R, L, fold;  // Hn = H / U heads per group, C = L / (U R) tokens per rank
};

// Row index pairs: sequence-shard row s = ((n B + b) H + h) C + i, head-
// group row t = ((g B + b) Hn + hl) L + pos with g = h / Hn, hl = h % Hn.
__device__ __forceinline__ long long head_row(long long s, const UspMap& m) {
  const int i = static_cast<int>(s % m.C);
  long long rest = s / m.C;
  const int h = static_cast<int>(rest % m.H);
  rest /= m.H;
  const int b = static_cast<int>(rest % m.B);
  const int n = static_cast<int>(rest / m.B);
  int pos;
  if (!m.fold) {
    pos = n * m.C + i;
  } else {
    const int r = n / m.U, u = n % m.U;
    const int c = m.L / (2 * m.R), piece = c / m.U;
    pos = i < piece ? r * c + u * piece + i : (2 * m.R - 1 - r) * c + u * piece + (i - piece);
  }
  const int g = h / m.Hn, hl = h % m.Hn;
  return ((static_cast<long long>(g) * m.B + b) * m.Hn + hl) * m.L + pos;
}

// kVec = 16-byte vectors per row; to_heads: sequence shards -> head groups.
// Grid: y (and z beyond 65535) = the (n, b, h) slice of C shard rows, x =
// runs of 4 x 256 vectors within it, so the slice's coordinates are
// per-block constants and a thread only splits its vector index into (row,
// vector) by a shift; its four copies are all loaded before any is stored.
// Consecutive threads walk consecutive vectors of both layouts (a shard
// slice's rows are consecutive positions of one head, except across the
// fold's two pieces).
template <int kVec>
__global__ void __launch_bounds__(256) ulysses_a2a_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                          UspMap m, int to_heads, int slices) {
  constexpr int kUnroll = 4;
  const int sl = static_cast<int>(blockIdx.z) * static_cast<int>(gridDim.y) + static_cast<int>(blockIdx.y);
  if (sl >= slices) return;
  const int h = sl % m.H, b = (sl / m.H) % m.B, n = sl / (m.H * m.B);
  const int g = h / m.Hn, hl = h % m.Hn;
  const long long shard0 = static_cast<long long>(sl) * m.C;
  const long long head0 = ((static_cast<long long>(g) * m.B + b) * m.Hn + hl) * m.L;
  const int r = n / m.U, u = n % m.U;
  const int c = m.fold ? m.L / (2 * m.R) : 0, piece = m.fold ? c / m.U : 0;
  const int per_slice = m.C * kVec;
  const int t0 = static_cast<int>(blockIdx.x) * (256 * kUnroll) + static_cast<int>(threadIdx.x);
  uint4 v[kUnroll];
  long long so[kUnroll], ho[kUnroll];
#pragma unroll
  for (int k = 0; k < kUnroll; ++k) {
    const int t = t0 + 256 * k;
    const int i = t / kVec, cc = t % kVec;
    int pos;
    if (!m.fold)
      pos = n * m.C + i;
    else
      pos = i < piece ? r * c + u * piece + i : (2 * m.R - 1 - r) * c + u * piece + (i - piece);
    so[k] = (shard0 + i) * kVec + cc;
    ho[k] = (head0 + pos) * kVec + cc;
    if (t < per_slice) v[k] = src[to_heads ? so[k] : ho[k]];
  }
#pragma unroll
  for (int k = 0; k < kUnroll; ++k)
    if (t0 + 256 * k < per_slice) dst[to_heads ? ho[k] : so[k]] = v[k];
}

// The same permutation for one fp32 per row (lse): one value per thread.
__global__ void __launch_bounds__(256) ulysses_a2a_rows_kernel(const float* __restrict__ src, float* __restrict__ dst,
                                                               UspMap m, int to_heads, long long n_rows) {
  const long long s = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (s >= n_rows) return;
  if (to_heads)
    dst[head_row(s, m)] = src[s];
  else
    dst[s] = src[head_row(s, m)];
}

}  // namespace

cudaError_t launch_ulysses_a2a(const void* src, void* dst, int row_bytes, int B, int H, int U, int R, int L,
                               bool causal, bool to_heads, cudaStream_t stream) {
  UspMap m;
  m.B = B; m.H = H; m.U = U; m.R = R; m.L = L;
  m.Hn = H / U;
  m.C = L / (U * R);
  m.fold = causal && R > 1;
  const long long rows = static_cast<long long>(U) * R * B * H * m.C;
  if (row_bytes == 128 || row_bytes == 256) {  // rows of d = 64 or 128 bf16 values
    const long long slices_ll = static_cast<long long>(U) * R * B * H;
    const long long per_slice_ll = static_cast<long long>(m.C) * (row_bytes / 16);
    if (slices_ll > INT_MAX || per_slice_ll > INT_MAX - 1024) return cudaErrorInvalidValue;
    const int slices = static_cast<int>(slices_ll);
    const int per_slice = static_cast<int>(per_slice_ll);
    const dim3 grid(static_cast<unsigned>((per_slice + 1023) / 1024), static_cast<unsigned>(slices < 65535 ? slices : 65535),
                    static_cast<unsigned>((slices + 65534) / 65535));
    if (row_bytes == 256)
      ulysses_a2a_kernel<16><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), m,
                                                       to_heads ? 1 : 0, slices);
    else
      ulysses_a2a_kernel<8><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), m,
                                                      to_heads ? 1 : 0, slices);
  } else if (row_bytes == 4) {  // one fp32 per row
    ulysses_a2a_rows_kernel<<<blocks_for(rows), 256, 0, stream>>>(static_cast<const float*>(src),
                                                                  static_cast<float*>(dst), m, to_heads ? 1 : 0, rows);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// Token-major [B][L][H][row] <-> head-major [B][H][L][row] (the
// blockwise transformer's FFN rows against the attention kernels' layout),
// 16 bytes per thread, walking the head-major side.
__global__ void __launch_bounds__(256) tokens_heads_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                           int vec16, int H, int L, int to_heads, long long n_vec) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n_vec) return;
  const int c = static_cast<int>(t % vec16);
  const long long hm = t / vec16;  // head-major row ((b H + h) L + l)
  const int l = static_cast<int>(hm % L);
  const long long bh = hm / L;
  const int h = static_cast<int>(bh % H);
  const long long b = bh / H;
  const long long tm = (b * L + l) * H + h;  // token-major row
  if (to_heads)
    dst[hm * vec16 + c] = src[tm * vec16 + c];
  else
    dst[tm * vec16 + c] = src[hm * vec16 + c];
}

cudaError_t launch_tokens_heads(const void* src, void* dst, int row_bytes, int B, int H, int L, bool to_heads,
                                cudaStream_t stream) {
  const int vec16 = row_bytes / 16;
  const long long n = static_cast<long long>(B) * H * L * vec16;
  tokens_heads_kernel<<<blocks_for(n), 256, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                         vec16, H, L, to_heads ? 1 : 0, n);
  return cudaGetLastError();
}

}  // namespace ra
