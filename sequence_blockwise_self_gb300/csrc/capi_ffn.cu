// capi_ffn.cu -- the C ABI of the blockwise feed-forward block and of the
// blockwise transformer (include/ring_attn.h): tensor maps and launches of
// the CTA-pair GEMM (ffn.cu), the transposes and column sums of the
// backward, and the attention launches per query block.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "../../include/ring_attn.h"
#include "capi_internal.h"
#include "kernels.h"
#include "plan.h"
#include "ffn.h"

namespace ra {
namespace {

std::map<int, int> g_ffn_pair_clusters;  // device -> clusters of two the GEMM can hold at once (0: none)

int ffn_shape(int D, int F, int block_rows) {
  if (D <= 0 || F <= 0 || block_rows <= 0) return RING_ATTN_ERR_SHAPE;
  if (D % 256 || F % 256 || block_rows % 128) return RING_ATTN_ERR_UNSUPPORTED;
  if (D > (1 << 20) || F > (1 << 20)) return RING_ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(block_rows) * F >= (1ll << 40)) return RING_ATTN_ERR_UNSUPPORTED;
  return RING_ATTN_OK;
}

// The blockwise FFN's two GEMM launches over a [rows][D] input, prepared
// once per call (tensor maps, tile order, CTA-pair clusters); ffn_rows then
// runs the block of rb <= block_rows rows starting at row r0, with its
// hidden activation in the workspace (caller holds g_mutex).
struct FfnLaunch {
  FfnGemmArgs g1, g2;
};

int ffn_prepare(int dev, const void* x, const void* w1, const float* b1, const void* w2, const float* b2, void* y,
                int rows, int D, int F, int block_rows, void* workspace, FfnLaunch* out) {
  int n_sms = 0, optin = 0;
  if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (ffn_gemm_smem_bytes() > static_cast<size_t>(optin)) return RING_ATTN_ERR_UNSUPPORTED;
  int* err;
  int rc;
  if ((rc = status_ptr(dev, &err)) != RING_ATTN_OK) return rc;
  // the GEMM runs on CTA pairs: clusters of two that fit at once
  auto it = g_ffn_pair_clusters.find(dev);
  if (it == g_ffn_pair_clusters.end()) it = g_ffn_pair_clusters.emplace(dev, ffn_pair_max_clusters()).first;
  const int pair_clusters = it->second;
  if (pair_clusters <= 0) return RING_ATTN_ERR_UNSUPPORTED;
  const int tile_m = 256, b_box = 128;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // first layer: A = x [rows][D], B = W1 [F][D], C = h [block_rows][F]
  // second layer: A = h, B = W2 [D][F], C = y [rows][D], residual x
  FfnGemmArgs& g1 = out->g1;
  FfnGemmArgs& g2 = out->g2;
  if (!make_map(&g1.tm_a, x, bf, 2, D, rows, 1, 64) || !make_map(&g1.tm_b, w1, bf, 2, D, F, 1, 64, b_box) ||
      !make_map(&g1.tm_c, workspace, bf, 2, F, block_rows, 1, 64) ||
      !make_map(&g2.tm_a, workspace, bf, 2, F, block_rows, 1, 64) ||
      !make_map(&g2.tm_b, w2, bf, 2, F, D, 1, 64, b_box) || !make_map(&g2.tm_c, y, bf, 2, D, rows, 1, 64))
    return RING_ATTN_ERR_CUDA;
  g1.N = F; g1.K = D; g1.c_rows = block_rows; g1.kind = 0; g1.bias = b1;
  g2.N = D; g2.K = F; g2.c_rows = rows; g2.kind = 1; g2.bias = b2; g2.resid = x;
  for (FfnGemmArgs* g : {&g1, &g2}) {
    g->err = err;
    g->n_sms = n_sms;
    g->pair_clusters = pair_clusters;
    g->timer = active_timer();
    // tile order: groups of row tiles whose rows of A take about 16 MiB, so
    // that a group's A stays in L2 while its column tiles go by
    const long long a_tile_bytes = static_cast<long long>(tile_m) * g->K * 2;
    g->group_rows = static_cast<int>(std::max(1ll, (1ll << 24) / a_tile_bytes));
  }
  return RING_ATTN_OK;
}

int ffn_rows(FfnLaunch& f, int r0, int rb, cudaStream_t stream) {
  f.g1.M = rb; f.g1.a_row0 = r0; f.g1.c_row0 = 0;
  f.g2.M = rb; f.g2.a_row0 = 0; f.g2.c_row0 = r0;
  if (launch_ffn_gemm(f.g1, stream) != cudaSuccess || launch_ffn_gemm(f.g2, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  return RING_ATTN_OK;
}

// Parts of the FFN backward workspace (byte offsets, 256-aligned): W1^T
// [D][F] and W2^T [F][D] (bf16), one block's gelu'(a) / da [R][F] (bf16),
// the transposed operands of the weight gradients, h^T / da^T [F][R] and
// dy^T / x^T [D][R] (bf16), and a zero bias [D] (fp32).
struct FfnBwdWorkspace {
  size_t w1t = 0, w2t = 0, g = 0, tbig = 0, tsmall = 0, zero = 0, total = 0;
};

FfnBwdWorkspace ffn_bwd_workspace(int D, int F, int R) {
  auto up = [](size_t x) { return round_up(x, 256); };
  const size_t df = static_cast<size_t>(D) * F * 2, rf = static_cast<size_t>(R) * F * 2,
               rd = static_cast<size_t>(R) * D * 2;
  FfnBwdWorkspace w;
  w.w2t = w.w1t + up(df);
  w.g = w.w2t + up(df);
  w.tbig = w.g + up(rf);
  w.tsmall = w.tbig + up(rf);
  w.zero = w.tsmall + up(rd);
  w.total = w.zero + up(static_cast<size_t>(D) * 4);
  return w;
}

// 2-D (as 3-D) map over a bf16 [rows][cols] tensor with 64 x 64 boxes and a
// 128-byte swizzle: the transposed outputs of the FFN backward's epilogues.
bool make_map_t(CUtensorMap* m, const void* base, int cols, int rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, static_cast<cuuint64_t>(cols) * rows * 2};
  cuuint32_t box[3] = {64u, 64u, 1u};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over a token-major [B][L][H][d] bf16 tensor, box (64, 1, 128, 1),
// 128-byte swizzle: the smem image of a box is that of the 3-D maps' boxes.
bool make_map_tok(CUtensorMap* m, const void* base, int d, int H, int L, int B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(d) * H * 2,
                           static_cast<cuuint64_t>(d) * H * L * 2};
  cuuint32_t box[4] = {64u, 1u, 128u, 1u};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The FFN backward on checked arguments (caller holds g_mutex).
int ffn_bwd_impl(int dev, const void* x, const void* w1, const float* b1, const void* w2, const void* dy,
                        void* dx, float* dw1, float* db1, float* dw2, float* db2, long long M, int D, int F,
                        int block_rows, void* workspace, cudaStream_t stream) {
  int rc;
  const FfnBwdWorkspace w = ffn_bwd_workspace(D, F, block_rows);
  // the gradients are sums over the rows: start from zero
  if (cudaMemsetAsync(dw1, 0, static_cast<size_t>(F) * D * 4, stream) != cudaSuccess ||
      cudaMemsetAsync(dw2, 0, static_cast<size_t>(D) * F * 4, stream) != cudaSuccess ||
      cudaMemsetAsync(db1, 0, static_cast<size_t>(F) * 4, stream) != cudaSuccess ||
      cudaMemsetAsync(db2, 0, static_cast<size_t>(D) * 4, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (M == 0) return RING_ATTN_OK;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void *w1t = ws + w.w1t, *w2t = ws + w.w2t, *g = ws + w.g, *tbig = ws + w.tbig, *tsmall = ws + w.tsmall;
  float* zero = reinterpret_cast<float*>(ws + w.zero);
  const int rows = static_cast<int>(M), R = block_rows;
  int n_sms = 0, optin = 0;
  if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (ffn_gemm_smem_bytes() > static_cast<size_t>(optin)) return RING_ATTN_ERR_UNSUPPORTED;
  int* err;
  if ((rc = status_ptr(dev, &err)) != RING_ATTN_OK) return rc;
  auto it = g_ffn_pair_clusters.find(dev);
  if (it == g_ffn_pair_clusters.end()) it = g_ffn_pair_clusters.emplace(dev, ffn_pair_max_clusters()).first;
  if (it->second <= 0) return RING_ATTN_ERR_UNSUPPORTED;
  LaunchTimer* tmr = active_timer();
  if (cudaMemsetAsync(zero, 0, static_cast<size_t>(D) * 4, stream) != cudaSuccess ||
      launch_transpose_bf16(w1, w1t, F, D, F, F, stream) != cudaSuccess ||   // W1 [F][D] -> W1^T [D][F]
      launch_transpose_bf16(w2, w2t, D, F, D, D, stream) != cudaSuccess)     // W2 [D][F] -> W2^T [F][D]
    return RING_ATTN_ERR_CUDA;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  // per block, in this order:
  //   G1: g = gelu'(x W1^T + b1), h^T = gelu(.)^T     G4: dW2 += dy^T h
  //   G2: da = (dy W2) * g in g's place, and da^T     G3: dx = da W1 + dy
  //   G5: dW1 += da^T x
  // h^T and da^T share one buffer (G4 has read h^T before G2 writes da^T)
  FfnGemmArgs g1, g2, g3, g4, g5;
  if (!make_map(&g1.tm_a, x, bf, 2, D, rows, 1, 64) || !make_map(&g1.tm_b, w1, bf, 2, D, F, 1, 64) ||
      !make_map(&g1.tm_c, g, bf, 2, F, R, 1, 64) || !make_map_t(&g1.tm_aux, tbig, R, F) ||
      !make_map(&g2.tm_a, dy, bf, 2, D, rows, 1, 64) || !make_map(&g2.tm_b, w2t, bf, 2, D, F, 1, 64) ||
      !make_map(&g2.tm_c, g, bf, 2, F, R, 1, 64) || !make_map_t(&g2.tm_aux, tbig, R, F) ||
      !make_map(&g3.tm_a, g, bf, 2, F, R, 1, 64) || !make_map(&g3.tm_b, w1t, bf, 2, F, D, 1, 64) ||
      !make_map(&g3.tm_c, dx, bf, 2, D, rows, 1, 64) ||
      !make_map(&g4.tm_a, tsmall, bf, 2, R, D, 1, 64) || !make_map(&g4.tm_b, tbig, bf, 2, R, F, 1, 64) ||
      !make_map(&g4.tm_c, dw2, f32, 4, F, D, 1, 32) ||
      !make_map(&g5.tm_a, tbig, bf, 2, R, F, 1, 64) || !make_map(&g5.tm_b, tsmall, bf, 2, R, D, 1, 64) ||
      !make_map(&g5.tm_c, dw1, f32, 4, D, F, 1, 32))
    return RING_ATTN_ERR_CUDA;
  g1.N = F; g1.K = D; g1.c_rows = R; g1.kind = 2; g1.bias = b1;
  g2.N = F; g2.K = D; g2.c_rows = R; g2.kind = 3; g2.resid = g; g2.trans = 1;
  g3.N = D; g3.K = F; g3.c_rows = rows; g3.kind = 1; g3.bias = zero; g3.resid = dy;
  g4.M = D; g4.N = F; g4.c_rows = D; g4.kind = 4;
  g5.M = F; g5.N = D; g5.c_rows = F; g5.kind = 4;
  for (FfnGemmArgs* a : {&g1, &g2, &g3, &g4, &g5}) {
    a->err = err;
    a->n_sms = n_sms;
    a->pair_clusters = it->second;
    a->timer = tmr;
  }
  auto group_rows = [](int K) { return static_cast<int>(std::max(1ll, (1ll << 24) / (256ll * K * 2))); };
  g1.group_rows = group_rows(D); g2.group_rows = group_rows(D); g3.group_rows = group_rows(F);
  for (int r0 = 0; r0 < rows; r0 += R) {
    const int rb = std::min(R, rows - r0), kp = (rb + 63) / 64 * 64;
    const uint8_t* dy_blk = static_cast<const uint8_t*>(dy) + static_cast<size_t>(r0) * D * 2;
    const uint8_t* x_blk = static_cast<const uint8_t*>(x) + static_cast<size_t>(r0) * D * 2;
    g1.M = rb; g1.a_row0 = r0; g1.c_row0 = 0;
    g2.M = rb; g2.a_row0 = r0; g2.c_row0 = 0;
    g3.M = rb; g3.a_row0 = 0; g3.c_row0 = r0;
    g4.K = kp; g5.K = kp;
    g4.group_rows = group_rows(kp); g5.group_rows = group_rows(kp);
    if (launch_ffn_gemm(g1, stream) != cudaSuccess ||
        launch_transpose_bf16(dy_blk, tsmall, rb, D, kp, R, stream) != cudaSuccess ||
        launch_ffn_gemm(g4, stream) != cudaSuccess || launch_ffn_gemm(g2, stream) != cudaSuccess ||
        launch_ffn_gemm(g3, stream) != cudaSuccess ||
        launch_transpose_bf16(x_blk, tsmall, rb, D, kp, R, stream) != cudaSuccess ||
        launch_ffn_gemm(g5, stream) != cudaSuccess || launch_colsum_add(g, rb, F, F, db1, stream) != cudaSuccess ||
        launch_colsum_add(dy_blk, rb, D, D, db2, stream) != cudaSuccess)
      return RING_ATTN_ERR_CUDA;
  }
  return RING_ATTN_OK;
}

// Parts of the blockwise transformer's backward workspace (byte offsets,
// 256-aligned): the FFN backward's, the gradient at the attention output
// (token-major), the attention output and that gradient head-major, and the
// fused attention backward's.
struct BptBwdWorkspace {
  size_t ffn = 0, da = 0, o = 0, dO = 0, attn = 0, total = 0;
};

BptBwdWorkspace bpt_bwd_workspace(int B, int Hq, int Hkv, int L, int d, int F, int block_rows) {
  auto up = [](size_t x) { return round_up(x, 256); };
  const size_t act = static_cast<size_t>(B) * L * Hq * d * 2;
  BptBwdWorkspace w;
  w.da = w.ffn + up(ffn_bwd_workspace(Hq * d, F, block_rows).total);
  w.o = w.da + up(act);
  w.dO = w.o + up(act);
  w.attn = w.dO + up(act);
  w.total = w.attn + bwd_workspace(B, Hq, Hkv, L, d).total;
  return w;
}

}  // namespace
}  // namespace ra

using namespace ra;

extern "C" {

size_t ring_attn_ffn_workspace_size(int D, int F, int block_rows) {
  if (ffn_shape(D, F, block_rows) != RING_ATTN_OK) return 0;
  return round_up(static_cast<size_t>(block_rows) * F * 2, 256);
}

int ring_attn_ffn_fwd(const void* x, const void* w1, const float* b1, const void* w2, const float* b2, void* y,
                      long long M, int D, int F, int block_rows, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  int rc = ffn_shape(D, F, block_rows);
  if (rc != RING_ATTN_OK) return rc;
  if (M < 0) return RING_ATTN_ERR_SHAPE;
  if (M >= (1ll << 31)) return RING_ATTN_ERR_UNSUPPORTED;
  if (M == 0) return RING_ATTN_OK;
  if (!x || !w1 || !b1 || !w2 || !b2 || !y) return RING_ATTN_ERR_NULL;
  const void* ptrs[] = {x, w1, b1, w2, b2, y};
  for (const void* p : ptrs)
    if (!aligned16(p)) return RING_ATTN_ERR_UNSUPPORTED;
  const size_t need = ring_attn_ffn_workspace_size(D, F, block_rows);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return RING_ATTN_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  FfnLaunch f;
  if ((rc = ffn_prepare(dev, x, w1, b1, w2, b2, y, static_cast<int>(M), D, F, block_rows, workspace, &f)) !=
      RING_ATTN_OK)
    return rc;
  for (int r0 = 0; r0 < static_cast<int>(M); r0 += block_rows)
    if ((rc = ffn_rows(f, r0, std::min(block_rows, static_cast<int>(M) - r0), stream)) != RING_ATTN_OK) return rc;
  return RING_ATTN_OK;
}

size_t ring_attn_ffn_bwd_workspace_size(int D, int F, int block_rows) {
  if (ffn_shape(D, F, block_rows) != RING_ATTN_OK) return 0;
  return ffn_bwd_workspace(D, F, block_rows).total;
}

int ring_attn_ffn_bwd(const void* x, const void* w1, const float* b1, const void* w2, const void* dy, void* dx,
                      float* dw1, float* db1, float* dw2, float* db2, long long M, int D, int F, int block_rows,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int rc = ffn_shape(D, F, block_rows);
  if (rc != RING_ATTN_OK) return rc;
  if (M < 0) return RING_ATTN_ERR_SHAPE;
  if (M >= (1ll << 31)) return RING_ATTN_ERR_UNSUPPORTED;
  if (!x || !w1 || !b1 || !w2 || !dy || !dx || !dw1 || !db1 || !dw2 || !db2) return RING_ATTN_ERR_NULL;
  const void* ptrs[] = {x, w1, b1, w2, dy, dx, dw1, db1, dw2, db2};
  for (const void* p : ptrs)
    if (!aligned16(p)) return RING_ATTN_ERR_UNSUPPORTED;
  const FfnBwdWorkspace w = ffn_bwd_workspace(D, F, block_rows);
  if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return RING_ATTN_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  return ffn_bwd_impl(dev, x, w1, b1, w2, dy, dx, dw1, db1, dw2, db2, M, D, F, block_rows, workspace, stream);
}

size_t ring_attn_bpt_bwd_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal, int F,
                                        int block_rows) {
  if (check_shape(B, Hq, Hkv, L, d, n_chunks, causal) != RING_ATTN_OK || block_rows <= 0 ||
      block_rows % kQBlockRows || ffn_shape(Hq * d, F, block_rows) != RING_ATTN_OK)
    return 0;
  return bpt_bwd_workspace(B, Hq, Hkv, L, d, F, block_rows).total;
}

int ring_attn_bpt_bwd(const void* q, const void* k, const void* v, const void* a_tok, const float* lse, const void* w1,
                      const float* b1, const void* w2, const void* dy, void* dq, void* dk, void* dv, float* dw1,
                      float* db1, float* dw2, float* db2, int B, int Hq, int Hkv, int L, int d, int n_chunks,
                      int causal, int F, int block_rows, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  int rc = check_shape(B, Hq, Hkv, L, d, n_chunks, causal);
  if (rc != RING_ATTN_OK) return rc;
  if (block_rows <= 0) return RING_ATTN_ERR_SHAPE;
  if (block_rows % kQBlockRows) return RING_ATTN_ERR_UNSUPPORTED;
  const int D = Hq * d;
  if ((rc = ffn_shape(D, F, block_rows)) != RING_ATTN_OK) return rc;
  if (static_cast<long long>(B) * L >= (1ll << 31)) return RING_ATTN_ERR_UNSUPPORTED;
  if (!q || !k || !v || !a_tok || !lse || !w1 || !b1 || !w2 || !dy || !dq || !dk || !dv || !dw1 || !db1 || !dw2 ||
      !db2)
    return RING_ATTN_ERR_NULL;
  const void* ptrs[] = {q, k, v, a_tok, lse, w1, b1, w2, dy, dq, dk, dv, dw1, db1, dw2, db2};
  for (const void* p : ptrs)
    if (!aligned16(p)) return RING_ATTN_ERR_UNSUPPORTED;
  const BptBwdWorkspace w = bpt_bwd_workspace(B, Hq, Hkv, L, d, F, block_rows);
  if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return RING_ATTN_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // FFN: recompute each block's hidden activation; the gradient at the
  // attention output is dy + the FFN's input gradient (its residual path)
  if ((rc = ffn_bwd_impl(dev, a_tok, w1, b1, w2, dy, ws + w.da, dw1, db1, dw2, db2, static_cast<long long>(B) * L,
                         D, F, block_rows, ws + w.ffn, stream)) != RING_ATTN_OK)
    return rc;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  // attention: the fused backward on head-major o and dO
  LaunchTimer* t = active_timer();
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, false, stream);
  if (launch_tokens_heads(a_tok, ws + w.o, d * 2, B, Hq, L, true, stream) != cudaSuccess ||
      launch_tokens_heads(ws + w.da, ws + w.dO, d * 2, B, Hq, L, true, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, true, stream);
  return bwd_impl(dev, q, k, v, ws + w.o, lse, ws + w.dO, dq, dk, dv, B, Hq, Hkv, L, d, n_chunks, causal,
                  ws + w.attn, stream);
}

size_t ring_attn_bpt_workspace_size(int Hq, int d, int F, int block_rows) {
  if (Hq <= 0 || block_rows <= 0 || block_rows % kQBlockRows) return 0;
  return ring_attn_ffn_workspace_size(Hq * d, F, block_rows);
}

int ring_attn_bpt_fwd(const void* q, const void* k, const void* v, void* a_tok, float* lse, const void* w1,
                      const float* b1, const void* w2, const float* b2, void* y, int B, int Hq, int Hkv, int L, int d,
                      int n_chunks, int causal, int F, int block_rows, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  int rc = check_shape(B, Hq, Hkv, L, d, n_chunks, causal);
  if (rc != RING_ATTN_OK) return rc;
  if (block_rows <= 0) return RING_ATTN_ERR_SHAPE;
  if (block_rows % kQBlockRows) return RING_ATTN_ERR_UNSUPPORTED;
  const int D = Hq * d;
  if ((rc = ffn_shape(D, F, block_rows)) != RING_ATTN_OK) return rc;
  if (static_cast<long long>(B) * L >= (1ll << 31)) return RING_ATTN_ERR_UNSUPPORTED;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q || !k || !v || !a_tok || !lse || !w1 || !b1 || !w2 || !b2 || !y) return RING_ATTN_ERR_NULL;
  const void* ptrs[] = {q, k, v, a_tok, lse, w1, b1, w2, b2, y};
  for (const void* p : ptrs)
    if (!aligned16(p)) return RING_ATTN_ERR_UNSUPPORTED;
  const size_t need = ring_attn_bpt_workspace_size(Hq, d, F, block_rows);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return RING_ATTN_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  // attention: the fused forward, one launch per row block, output token-major
  FwdArgs a;
  std::memset(&a, 0, sizeof a);
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map(&a.tm_q, q, bf, 2, d, L, B * Hq, 64) || !make_map(&a.tm_k, k, bf, 2, d, L, B * Hkv, 64) ||
      !make_map(&a.tm_v, v, bf, 2, d, L, B * Hkv, 64) || !make_map_tok(&a.tm_o, a_tok, d, Hq, L, B))
    return RING_ATTN_ERR_CUDA;
  DevicePlan plan;
  if ((rc = get_plan(dev, 0, L, n_chunks, causal != 0, &plan)) != RING_ATTN_OK) return rc;
  int32_t* orders;
  if ((rc = get_block_orders(dev, L, n_chunks, causal, block_rows, &orders)) != RING_ATTN_OK) return rc;
  int* err;
  if ((rc = status_ptr(dev, &err)) != RING_ATTN_OK) return rc;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = L; a.d = d; a.causal = causal != 0;
  a.offsets = plan.offsets(); a.ranges = plan.ranges();
  a.lse = lse; a.err = err; a.timer = active_timer();
  a.o_token_major = 1;
  // feed-forward on the token rows [L][Hq d] of each batch's attention
  // output; one set of tensor maps per batch, so that the stores of a block
  // that ends inside a 128-row box are clipped at that batch's last row
  std::vector<FfnLaunch> f(B);
  const size_t batch_bytes = static_cast<size_t>(L) * D * 2;
  for (int b = 0; b < B; ++b)
    if ((rc = ffn_prepare(dev, static_cast<const uint8_t*>(a_tok) + b * batch_bytes, w1, b1, w2, b2,
                          static_cast<uint8_t*>(y) + b * batch_bytes, L, D, F, block_rows, workspace, &f[b])) !=
        RING_ATTN_OK)
      return rc;
  const int per = block_rows / kQBlockRows;
  for (int r0 = 0; r0 < L; r0 += block_rows) {
    const int u0 = r0 / kQBlockRows;
    a.order = orders + u0;
    a.n_blocks = std::min(per, plan.n_blocks - u0);
    if (launch_fwd(a, stream) != cudaSuccess) return RING_ATTN_ERR_CUDA;
    const int rb = std::min(block_rows, L - r0);
    for (int b = 0; b < B; ++b)
      if ((rc = ffn_rows(f[b], r0, rb, stream)) != RING_ATTN_OK) return rc;
  }
  return RING_ATTN_OK;
}

}  // extern "C"
