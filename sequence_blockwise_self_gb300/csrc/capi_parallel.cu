// capi_parallel.cu -- the C ABI of Ulysses and USP (include/ring_attn.h):
// the sequence-shard <-> head-group all-to-alls (ulysses.cu) around one
// launch of the fused attention kernels.
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

namespace ra {
namespace {

struct UlyssesWorkspace {
  size_t q = 0, k = 0, v = 0, o = 0, lse = 0, dO = 0, dq = 0, dk = 0, dv = 0, bwd = 0, fwd_total = 0, total = 0;
};

// N here is the number of head groups (the Ulysses degree U).
UlyssesWorkspace ulysses_workspace(int B, int Hq, int Hkv, int L, int d, int N) {
  auto up = [](size_t x) { return round_up(x, 256); };
  const size_t nq = static_cast<size_t>(B) * Hq * L * d * 2, nkv = static_cast<size_t>(B) * Hkv * L * d * 2;
  UlyssesWorkspace w;
  w.k = w.q + up(nq);
  w.v = w.k + up(nkv);
  w.o = w.v + up(nkv);
  w.lse = w.o + up(nq);
  w.fwd_total = w.lse + up(static_cast<size_t>(B) * Hq * L * 4);
  w.dO = w.fwd_total;
  w.dq = w.dO + up(nq);
  w.dk = w.dq + up(nq);
  w.dv = w.dk + up(nkv);
  w.bwd = w.dv + up(nkv);
  w.total = w.bwd + bwd_workspace(N * B, Hq / N, Hkv / N, L, d).total;
  return w;
}

// USP over U x R ranks (plain Ulysses: R = 1): every rank of a Ulysses
// group takes H/U of the query heads and of the key/value heads; the ring
// over R groups is the fused kernel's chunking of the head groups' full
// sequences (fold when causal: each of its 2R sub-chunks splits into U
// pieces, one per rank of the group).
int check_usp(int B, int Hq, int Hkv, int L, int d, int U, int R, int causal) {
  if (U <= 0 || R <= 0) return RING_ATTN_ERR_SHAPE;
  int rc = check_shape(B, Hq, Hkv, L, d, 1, causal);
  if (rc != RING_ATTN_OK) return rc;
  if (Hq % U || Hkv % U) return RING_ATTN_ERR_SHAPE;
  const long long N = static_cast<long long>(U) * R;
  if (L % N) return RING_ATTN_ERR_SHAPE;
  if (causal && R > 1 && L % (2 * N)) return RING_ATTN_ERR_SHAPE;
  if (L > 0 && R > 1 && (rc = check_shape(U * B, Hq / U, Hkv / U, L, d, R, causal)) != RING_ATTN_OK) return rc;
  return RING_ATTN_OK;
}

cudaError_t a2a(const void* src, void* dst, int row_bytes, int B, int H, int U, int R, int L, int causal,
                bool to_heads, cudaStream_t stream) {
  return launch_ulysses_a2a(src, dst, row_bytes, B, H, U, R, L, causal != 0, to_heads, stream);
}

}  // namespace
}  // namespace ra

using namespace ra;

extern "C" {

size_t ring_attn_usp_workspace_size(int B, int Hq, int Hkv, int L, int d, int ulysses_degree, int ring_degree,
                                    int causal) {
  if (check_usp(B, Hq, Hkv, L, d, ulysses_degree, ring_degree, causal) != RING_ATTN_OK) return 0;
  return ulysses_workspace(B, Hq, Hkv, L, d, ulysses_degree).total;
}

int ring_attn_usp_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int L,
                      int d, int U, int R, int causal, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_usp(B, Hq, Hkv, L, d, U, R, causal);
  if (rc != RING_ATTN_OK) return rc;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q || !k || !v || !o || !lse) return RING_ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return RING_ATTN_ERR_UNSUPPORTED;
  const UlyssesWorkspace w = ulysses_workspace(B, Hq, Hkv, L, d, U);
  if (!workspace || workspace_bytes < w.fwd_total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return RING_ATTN_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int row = d * 2;
  LaunchTimer* t = active_timer();
  if (t) t->mark(RING_ATTN_KERNEL_ULYSSES_A2A, false, stream);
  if (a2a(q, ws + w.q, row, B, Hq, U, R, L, causal, true, stream) != cudaSuccess ||
      a2a(k, ws + w.k, row, B, Hkv, U, R, L, causal, true, stream) != cudaSuccess ||
      a2a(v, ws + w.v, row, B, Hkv, U, R, L, causal, true, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (t) t->mark(RING_ATTN_KERNEL_ULYSSES_A2A, true, stream);
  // every head group over the whole sequence, the ring over R chunks: one
  // launch, batch U*B
  if ((rc = fwd_impl(dev, ws + w.q, ws + w.k, ws + w.v, ws + w.o, reinterpret_cast<float*>(ws + w.lse), U * B,
                     Hq / U, Hkv / U, L, d, R, causal, stream)) != RING_ATTN_OK)
    return rc;
  if (t) t->mark(RING_ATTN_KERNEL_ULYSSES_A2A, false, stream);
  if (a2a(ws + w.o, o, row, B, Hq, U, R, L, causal, false, stream) != cudaSuccess ||
      a2a(ws + w.lse, lse, 4, B, Hq, U, R, L, causal, false, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (t) t->mark(RING_ATTN_KERNEL_ULYSSES_A2A, true, stream);
  return RING_ATTN_OK;
}

int ring_attn_usp_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                      void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L, int d, int U, int R, int causal,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_usp(B, Hq, Hkv, L, d, U, R, causal);
  if (rc != RING_ATTN_OK) return rc;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return RING_ATTN_ERR_NULL;
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return RING_ATTN_ERR_UNSUPPORTED;
  const UlyssesWorkspace w = ulysses_workspace(B, Hq, Hkv, L, d, U);
  if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return RING_ATTN_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int row = d * 2;
  LaunchTimer* t = active_timer();
  if (t) t->mark(RING_ATTN_KERNEL_ULYSSES_A2A, false, stream);
  if (a2a(q, ws + w.q, row, B, Hq, U, R, L, causal, true, stream) != cudaSuccess ||
      a2a(k, ws + w.k, row, B, Hkv, U, R, L, causal, true, stream) != cudaSuccess ||
      a2a(v, ws + w.v, row, B, Hkv, U, R, L, causal, true, stream) != cudaSuccess ||
      a2a(o, ws + w.o, row, B, Hq, U, R, L, causal, true, stream) != cudaSuccess ||
      a2a(lse, ws + w.lse, 4, B, Hq, U, R, L, causal, true, stream) != cudaSuccess ||
      a2a(dO, ws + w.dO, row, B, Hq, U, R, L, causal, true, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (t) t->mark(RING_ATTN_KERNEL_ULYSSES_A2A, true, stream);
  if ((rc = bwd_impl(dev, ws + w.q, ws + w.k, ws + w.v, ws + w.o, reinterpret_cast<const float*>(ws + w.lse),
                     ws + w.dO, ws + w.dq, ws + w.dk, ws + w.dv, U * B, Hq / U, Hkv / U, L, d, R, causal,
                     ws + w.bwd, stream)) != RING_ATTN_OK)
    return rc;
  if (t) t->mark(RING_ATTN_KERNEL_ULYSSES_A2A, false, stream);
  if (a2a(ws + w.dq, dq, row, B, Hq, U, R, L, causal, false, stream) != cudaSuccess ||
      a2a(ws + w.dk, dk, row, B, Hkv, U, R, L, causal, false, stream) != cudaSuccess ||
      a2a(ws + w.dv, dv, row, B, Hkv, U, R, L, causal, false, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (t) t->mark(RING_ATTN_KERNEL_ULYSSES_A2A, true, stream);
  return RING_ATTN_OK;
}

size_t ring_attn_ulysses_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_ranks, int causal) {
  return ring_attn_usp_workspace_size(B, Hq, Hkv, L, d, n_ranks, 1, causal);
}

int ring_attn_ulysses_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                          int L, int d, int n_ranks, int causal, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  return ring_attn_usp_fwd(q, k, v, o, lse, B, Hq, Hkv, L, d, n_ranks, 1, causal, workspace, workspace_bytes, stream);
}

int ring_attn_ulysses_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L, int d,
                          int n_ranks, int causal, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return ring_attn_usp_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, L, d, n_ranks, 1, causal, workspace,
                           workspace_bytes, stream);
}

}  // extern "C"
