// ring_attn_noalloc.cu -- ring_attn_bwd_noalloc: the backward pass without
// any device allocation, for callers that cannot call cudaMalloc.
//
// Who needs it: code whose device memory is owned entirely by another
// allocator (a framework's caching pool that has reserved the GPU, an
// embedding application with a fixed memory budget), and latency-critical
// callers that cannot afford the implicit device synchronisation cudaMalloc
// and cudaFree may cause.  ring_attn_bwd needs a caller-provided workspace
// and, on the first call for a shape, allocates a small device copy of the
// launch plan; this entry point needs neither.
//
// How: the workspace (per-row statistics and the fp32 accumulators) and
// the launch plan live in one file-scope static __device__ array of
// kNoAllocScratchBytes.  Every GPU that loads the library holds that array
// until the process exits.  Host code cannot pass the array's name to a
// kernel (in host code it names a host-side stand-in, not device memory), so
// the first call on each device, with that device current, looks up its
// device address with cudaGetSymbolAddress and caches it.  That first call
// should therefore happen before any stream capture begins.
//
// All calls share the array and it keeps the previous call's contents: the
// pre-pass kernel rewrites the statistics and zeroes the accumulators, and
// the plan is copied in again on every call.  Two calls whose work overlaps
// on the GPU (different streams, no ordering) race on the array.
#include <cudaTypedefs.h>

#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "../../include/ring_attn.h"
#include "kernels.h"
#include "plan.h"

namespace ra {

int status_word_for_current_device(int** out);  // defined in ring_attn_capi.cu

namespace {

constexpr size_t kNoAllocScratchBytes = RING_ATTN_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
std::map<int, unsigned char*> g_scratch_dev;                           // device -> address of the array
std::map<std::tuple<int, int, int>, std::vector<int32_t>> g_host_plan;  // (L, N, causal) -> flat plan

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Same tensor-map shape the backward kernel expects: [Z][rows][d], box
// (box_cols x box_rows), 128-byte swizzle.
bool map3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int d, int rows, int Z, int box_cols,
           int box_rows) {
  auto fn = encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(Z)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elem, static_cast<cuuint64_t>(d) * rows * elem};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Device address of the static array on the current device (looked up once).
int scratch_address(int dev, unsigned char** out) {
  auto it = g_scratch_dev.find(dev);
  if (it != g_scratch_dev.end()) {
    *out = it->second;
    return RING_ATTN_OK;
  }
  unsigned char* ptr = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch) != cudaSuccess || !ptr)
    return RING_ATTN_ERR_CUDA;
  g_scratch_dev[dev] = ptr;
  *out = ptr;
  return RING_ATTN_OK;
}

const std::vector<int32_t>& host_plan(int L, int N, int causal, int* n_blocks) {
  auto key = std::make_tuple(L, N, causal);
  auto it = g_host_plan.find(key);
  if (it == g_host_plan.end()) {
    Plan p = build_bwd_plan(L, N, causal != 0);
    std::vector<int32_t> flat;
    flat.push_back(p.n_blocks);
    flat.insert(flat.end(), p.order.begin(), p.order.end());
    flat.insert(flat.end(), p.offsets.begin(), p.offsets.end());
    flat.insert(flat.end(), p.ranges.begin(), p.ranges.end());
    it = g_host_plan.emplace(key, std::move(flat)).first;
  }
  *n_blocks = it->second[0];
  return it->second;
}

}  // namespace
}  // namespace ra

using namespace ra;

extern "C" int ring_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                     const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L,
                                     int d, int n_chunks, int causal, cudaStream_t stream) {
  // Argument checks are those of ring_attn_bwd.
  if (B < 0 || Hq <= 0 || Hkv <= 0 || L < 0 || n_chunks <= 0 || Hq % Hkv != 0) return RING_ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return RING_ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq >= 65536 || L > (1 << 30) / 2) return RING_ATTN_ERR_UNSUPPORTED;
  if (L > 0 && !chunking_ok(L, n_chunks, causal != 0)) return RING_ATTN_ERR_SHAPE;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return RING_ATTN_ERR_NULL;
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) & 15u) return RING_ATTN_ERR_UNSUPPORTED;

  // Scratch layout: the backward workspace (see kernels.h), then the plan.
  const BwdWorkspace w = bwd_workspace(B, Hq, Hkv, L, d);
  const size_t Lpad = static_cast<size_t>(w.Lpad);
  const size_t off_plan = w.total;
  if (off_plan > kNoAllocScratchBytes) return RING_ATTN_ERR_WORKSPACE;  // beyond the static array

  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  int dev;
  if (cudaGetDevice(&dev) != cudaSuccess) return RING_ATTN_ERR_CUDA;
  unsigned char* scratch;
  int rc = scratch_address(dev, &scratch);
  if (rc != RING_ATTN_OK) return rc;
  int* err;
  if ((rc = status_word_for_current_device(&err)) != RING_ATTN_OK) return rc;

  int n_blocks = 0;
  const std::vector<int32_t>& flat = host_plan(L, n_chunks, causal != 0, &n_blocks);
  const size_t plan_bytes = (flat.size() - 1) * sizeof(int32_t);
  if (off_plan + plan_bytes > kNoAllocScratchBytes) return RING_ATTN_ERR_WORKSPACE;
  int32_t* dplan = reinterpret_cast<int32_t*>(scratch + off_plan);
  if (cudaMemcpyAsync(dplan, flat.data() + 1, plan_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;

  BwdArgs a;
  std::memset(&a, 0, sizeof a);
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!map3d(&a.tm_q, q, bf, 2, d, L, B * Hq, 64, 128) || !map3d(&a.tm_k, k, bf, 2, d, L, B * Hkv, 64, 128) ||
      !map3d(&a.tm_v, v, bf, 2, d, L, B * Hkv, 64, 128) || !map3d(&a.tm_do, dO, bf, 2, d, L, B * Hq, 64, 128))
    return RING_ATTN_ERR_CUDA;
  if (w.kv_accumulate &&
      (!map3d(&a.tm_dkacc, scratch + w.dk, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, static_cast<int>(Lpad), B * Hkv, 32,
              32) ||
       !map3d(&a.tm_dvacc, scratch + w.dv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, static_cast<int>(Lpad), B * Hkv, 32,
              32)))
    return RING_ATTN_ERR_CUDA;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = L; a.Lpad = static_cast<int>(Lpad); a.d = d; a.causal = causal != 0;
  a.n_blocks = n_blocks;
  a.order = dplan;
  a.offsets = dplan + n_blocks;
  a.ranges = dplan + 2 * n_blocks + 1;
  a.o = o; a.dO = dO; a.lse = lse;
  a.lse2 = reinterpret_cast<float*>(scratch + w.lse2);
  a.Dvec = reinterpret_cast<float*>(scratch + w.dvec);
  a.dq_acc = reinterpret_cast<float*>(scratch + w.dq);
  a.dk_acc = w.kv_accumulate ? reinterpret_cast<float*>(scratch + w.dk) : nullptr;
  a.dv_acc = w.kv_accumulate ? reinterpret_cast<float*>(scratch + w.dv) : nullptr;
  a.dq = dq; a.dk = dk; a.dv = dv; a.err = err; a.timer = nullptr;
  return launch_bwd(a, stream) == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA;
}
