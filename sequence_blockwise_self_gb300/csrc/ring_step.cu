// ring_step.cu -- the memory-bound kernels of the explicit ring mode.
//
// ("Large-scale distributed AI model training series: sequence
// parallelism", section 2.3 Ring Self-Attention and section 6.2 Ring
// Attention.)  In ring mode every rank keeps its query chunk, computes the
// partial result (o_s, lse_s) of the key/value chunk it holds at each ring
// step (the step mode of the forward kernel, attn_fwd.cu) and merges it into
// its running result with the log-sum-exp rule:
//   lse = log(e^lse_a + e^lse_b),  o = e^(lse_a - lse) o_a + e^(lse_b - lse) o_b.
// The kernels here are that merge and, for running every rank of the ring
// on one GPU, the gather of q, k, v from sequence order into chunk-major
// order and the scatter of the merged result back.  All three move bytes
// and do a few flops per element: HBM-bound, sized for coalesced 16-byte
// accesses.
#include <cmath>

#include "kernels.h"
#include "plan.h"
#include "sm103_ptx.cuh"

namespace ra {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// d/4 threads per row, 32 / (d/4) rows per warp; every lane reads both lse
// values of its row before any lane writes the merged one.
template <int D>
__global__ void __launch_bounds__(256) ring_merge_kernel(float* __restrict__ o, float* __restrict__ lse,
                                                         const float* __restrict__ o_s,
                                                         const float* __restrict__ lse_s,
                                                         __nv_bfloat16* __restrict__ o_out, long long n_rows) {
  constexpr int kPerRow = D / 4;
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = t / kPerRow;
  const int q4 = static_cast<int>(t % kPerRow);
  const bool live = row < n_rows;
  float la = -INFINITY, lb = -INFINITY;
  if (live) {
    la = lse[row];
    lb = lse_s[row];
  }
  __syncwarp();
  if (!live) return;
  float4* pa = reinterpret_cast<float4*>(o + row * D) + q4;
  const float4 b = reinterpret_cast<const float4*>(o_s + row * D)[q4];
  float4 a = *pa;
  float merged;
  if (lb == -INFINITY) {  // the partial sees no key: nothing to add
    merged = la;
  } else if (la == -INFINITY) {
    a = b;
    merged = lb;
  } else {
    const float hi = fmaxf(la, lb);
    // natural-log weights through exp2 on the special-function unit
    const float ea = ex2((la - hi) * kLog2e), eb = ex2((lb - hi) * kLog2e);
    const float inv = 1.f / (ea + eb);
    const float wa = ea * inv, wb = eb * inv;
    merged = hi + log2f(ea + eb) * kLn2;
    a = make_float4(wa * a.x + wb * b.x, wa * a.y + wb * b.y, wa * a.z + wb * b.z, wa * a.w + wb * b.w);
  }
  *pa = a;
  if (o_out) {
    uint2 packed = make_uint2(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w));
    reinterpret_cast<uint2*>(o_out + row * D)[q4] = packed;
  }
  if (q4 == 0) lse[row] = merged;
}

// dst[r][z][i][:] = src[z][pos(r, i)][:], 8 bf16 per thread.
template <int D>
__global__ void __launch_bounds__(256) ring_gather_kernel(const __nv_bfloat16* __restrict__ src,
                                                          __nv_bfloat16* __restrict__ dst, int Z, int L, int N,
                                                          int causal, int sched, long long n_vec) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n_vec) return;
  constexpr int kVec = D / 8;
  const int c8 = static_cast<int>(t % kVec);
  const long long rowg = t / kVec;  // row of dst in [N][Z][C]
  const int C = L / N;
  const int i = static_cast<int>(rowg % C);
  const long long rz = rowg / C;
  const int z = static_cast<int>(rz % Z);
  const int r = static_cast<int>(rz / Z);
  const int pos = chunk_pos(L, N, causal != 0, sched, r, i);
  const uint4 v = reinterpret_cast<const uint4*>(src + (static_cast<size_t>(z) * L + pos) * D)[c8];
  reinterpret_cast<uint4*>(dst + rowg * D)[c8] = v;
}

// o[z][pos(r, i)][:] = bf16(acc[r][z][i][:]), lse likewise; 8 columns per
// thread.
template <int D>
__global__ void __launch_bounds__(256) ring_scatter_kernel(const float* __restrict__ acc,
                                                           const float* __restrict__ lse_acc,
                                                           __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                           int Z, int L, int N, int causal, int sched,
                                                           long long n_vec) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n_vec) return;
  constexpr int kVec = D / 8;
  const int c8 = static_cast<int>(t % kVec);
  const long long rowg = t / kVec;
  const int C = L / N;
  const int i = static_cast<int>(rowg % C);
  const long long rz = rowg / C;
  const int z = static_cast<int>(rz % Z);
  const int r = static_cast<int>(rz / Z);
  const int pos = chunk_pos(L, N, causal != 0, sched, r, i);
  const float4* s = reinterpret_cast<const float4*>(acc + rowg * D) + 2 * c8;
  const float4 a = s[0], b = s[1];
  const size_t out = static_cast<size_t>(z) * L + pos;
  reinterpret_cast<uint4*>(o + out * D)[c8] =
      make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(b.x, b.y), pack_bf16(b.z, b.w));
  if (c8 == 0) lse[out] = lse_acc[rowg];
}

// dst[r][z][i] = src[z][pos(r, i)] for one fp32 per row (lse).
__global__ void __launch_bounds__(256) ring_gather_rows_kernel(const float* __restrict__ src, float* __restrict__ dst,
                                                               int Z, int L, int N, int causal, int sched,
                                                               long long n_rows) {
  const long long rowg = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (rowg >= n_rows) return;
  const int C = L / N;
  const int i = static_cast<int>(rowg % C);
  const long long rz = rowg / C;
  const int z = static_cast<int>(rz % Z);
  const int r = static_cast<int>(rz / Z);
  dst[rowg] = src[static_cast<size_t>(z) * L + chunk_pos(L, N, causal != 0, sched, r, i)];
}

// Gradient back to sequence order: g[z][pos(r, i)][:] = bf16(scale * acc)
// for the fp32 accumulator in chunk order, either plain ([r][z][i][d]) or in
// the backward kernel's tiled dQ layout (per 128-row tile, [d/4][128][4]).
template <int D, bool kTiled>
__global__ void __launch_bounds__(256) ring_scatter_grad_kernel(const float* __restrict__ acc,
                                                                __nv_bfloat16* __restrict__ g, float scale, int Z,
                                                                int L, int N, int causal, int sched,
                                                                long long n_vec) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n_vec) return;
  constexpr int kVec = D / 8;
  const int c8 = static_cast<int>(t % kVec);
  const long long rowg = t / kVec;
  const int C = L / N;
  const int i = static_cast<int>(rowg % C);
  const long long rz = rowg / C;
  const int z = static_cast<int>(rz % Z);
  const int r = static_cast<int>(rz / Z);
  float4 a, b;
  if (kTiled) {  // slice rz of C rows, tile i / 128, column quads 2 c8 and 2 c8 + 1
    const float* base = acc + static_cast<size_t>(rz) * C * D + static_cast<size_t>(i >> 7) * 128 * D +
                        (i & 127) * 4;
    a = *reinterpret_cast<const float4*>(base + (2 * c8) * 512);
    b = *reinterpret_cast<const float4*>(base + (2 * c8 + 1) * 512);
  } else {
    const float4* s = reinterpret_cast<const float4*>(acc + rowg * D) + 2 * c8;
    a = s[0];
    b = s[1];
  }
  const size_t out = static_cast<size_t>(z) * L + chunk_pos(L, N, causal != 0, sched, r, i);
  reinterpret_cast<uint4*>(g + out * D)[c8] =
      make_uint4(pack_bf16(a.x * scale, a.y * scale), pack_bf16(a.z * scale, a.w * scale),
                 pack_bf16(b.x * scale, b.y * scale), pack_bf16(b.z * scale, b.w * scale));
}

unsigned blocks_for(long long n) { return static_cast<unsigned>((n + 255) / 256); }

// dst[i] += src[i], four fp32 per thread (partial gradients arriving from
// another rank: DistFlashAttention's helper blocks)
__global__ void __launch_bounds__(256) add_f32_kernel(float4* __restrict__ dst, const float4* __restrict__ src,
                                                      long long n4) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n4) return;
  float4 a = dst[t];
  const float4 b = src[t];
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
  dst[t] = a;
}

}  // namespace

cudaError_t launch_add_f32(float* dst, const float* src, long long n, cudaStream_t stream) {
  const long long n4 = n / 4;
  add_f32_kernel<<<blocks_for(n4), 256, 0, stream>>>(reinterpret_cast<float4*>(dst),
                                                     reinterpret_cast<const float4*>(src), n4);
  return cudaGetLastError();
}

cudaError_t launch_ring_gather_rows(const float* src, float* dst, int Z, int L, int N, bool causal, int sched,
                                    cudaStream_t stream) {
  const long long n = static_cast<long long>(Z) * L;
  ring_gather_rows_kernel<<<blocks_for(n), 256, 0, stream>>>(src, dst, Z, L, N, causal, sched, n);
  return cudaGetLastError();
}

cudaError_t launch_ring_scatter_grad(const float* acc, void* g, float scale, bool tiled, int Z, int L, int d, int N,
                                     bool causal, int sched, cudaStream_t stream) {
  const long long n = static_cast<long long>(Z) * L * (d / 8);
  auto* out = static_cast<__nv_bfloat16*>(g);
  const unsigned nb = blocks_for(n);
  if (d == 128) {
    if (tiled)
      ring_scatter_grad_kernel<128, true><<<nb, 256, 0, stream>>>(acc, out, scale, Z, L, N, causal, sched, n);
    else
      ring_scatter_grad_kernel<128, false><<<nb, 256, 0, stream>>>(acc, out, scale, Z, L, N, causal, sched, n);
  } else {
    if (tiled)
      ring_scatter_grad_kernel<64, true><<<nb, 256, 0, stream>>>(acc, out, scale, Z, L, N, causal, sched, n);
    else
      ring_scatter_grad_kernel<64, false><<<nb, 256, 0, stream>>>(acc, out, scale, Z, L, N, causal, sched, n);
  }
  return cudaGetLastError();
}

cudaError_t launch_ring_merge(float* o, float* lse, const float* o_s, const float* lse_s, void* o_out,
                              long long n_rows, int d, cudaStream_t stream) {
  const long long n = n_rows * (d / 4);
  auto* out = static_cast<__nv_bfloat16*>(o_out);
  if (d == 128)
    ring_merge_kernel<128><<<blocks_for(n), 256, 0, stream>>>(o, lse, o_s, lse_s, out, n_rows);
  else
    ring_merge_kernel<64><<<blocks_for(n), 256, 0, stream>>>(o, lse, o_s, lse_s, out, n_rows);
  return cudaGetLastError();
}

cudaError_t launch_ring_gather(const void* src, void* dst, int Z, int L, int d, int N, bool causal, int sched,
                               cudaStream_t stream) {
  const long long n = static_cast<long long>(Z) * L * (d / 8);
  auto* s = static_cast<const __nv_bfloat16*>(src);
  auto* t = static_cast<__nv_bfloat16*>(dst);
  if (d == 128)
    ring_gather_kernel<128><<<blocks_for(n), 256, 0, stream>>>(s, t, Z, L, N, causal, sched, n);
  else
    ring_gather_kernel<64><<<blocks_for(n), 256, 0, stream>>>(s, t, Z, L, N, causal, sched, n);
  return cudaGetLastError();
}

cudaError_t launch_ring_scatter(const float* acc, const float* lse_acc, void* o, float* lse, int Z, int L, int d,
                                int N, bool causal, int sched, cudaStream_t stream) {
  const long long n = static_cast<long long>(Z) * L * (d / 8);
  auto* out = static_cast<__nv_bfloat16*>(o);
  if (d == 128)
    ring_scatter_kernel<128><<<blocks_for(n), 256, 0, stream>>>(acc, lse_acc, out, lse, Z, L, N, causal, sched,
                                                               n);
  else
    ring_scatter_kernel<64><<<blocks_for(n), 256, 0, stream>>>(acc, lse_acc, out, lse, Z, L, N, causal, sched,
                                                              n);
  return cudaGetLastError();
}

}  // namespace ra
