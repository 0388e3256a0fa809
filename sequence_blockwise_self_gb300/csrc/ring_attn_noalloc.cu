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
// device address with cudaGetSymbolAddress and caches it; the first call for
// each (L, n_chunks, causal) builds that plan once in page-locked host
// memory.  Both first calls therefore happen outside stream capture; later
// calls may be captured (the plan copy is then a copy node of the graph).
//
// All calls share the array and it keeps the previous call's contents: the
// pre-pass kernel rewrites the statistics and zeroes the accumulators, and
// the plan is copied in again on every call.  Two calls whose work overlaps
// on the GPU (different streams, no ordering) race on the array.
#include <algorithm>
#include <cstring>
#include <map>
#include <tuple>

#include "../../include/ring_attn.h"
#include "capi_internal.h"
#include "plan.h"

namespace ra {
namespace {

constexpr size_t kNoAllocScratchBytes = RING_ATTN_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// A flattened backward plan (order | offsets | ranges) in page-locked host
// memory, so that its copy to the device is an ordinary asynchronous copy
// (and a copy node under stream capture), never a staged pageable one.
struct HostPlan {
  int n_blocks = 0;
  size_t n_words = 0;
  int32_t* words = nullptr;
};

// Both guarded by the library lock (g_mutex).
std::map<int, unsigned char*> g_scratch_dev;           // device -> address of the array
std::map<std::tuple<int, int, int>, HostPlan> g_plans;  // (L, N, causal) -> flat plan

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

int host_plan(int L, int N, int causal, const HostPlan** out) {
  auto key = std::make_tuple(L, N, causal);
  auto it = g_plans.find(key);
  if (it == g_plans.end()) {
    const Plan p = build_bwd_plan(L, N, causal != 0);
    HostPlan h;
    h.n_blocks = p.n_blocks;
    h.n_words = p.order.size() + p.offsets.size() + p.ranges.size();
    if (cudaMallocHost(&h.words, h.n_words * sizeof(int32_t)) != cudaSuccess) return RING_ATTN_ERR_CUDA;
    int32_t* w = h.words;
    w = std::copy(p.order.begin(), p.order.end(), w);
    w = std::copy(p.offsets.begin(), p.offsets.end(), w);
    std::copy(p.ranges.begin(), p.ranges.end(), w);
    it = g_plans.emplace(key, h).first;
  }
  *out = &it->second;
  return RING_ATTN_OK;
}

}  // namespace
}  // namespace ra

using namespace ra;

extern "C" int ring_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                     const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L,
                                     int d, int n_chunks, int causal, cudaStream_t stream) {
  // The argument checks of ring_attn_bwd.
  int rc = check_shape(B, Hq, Hkv, L, d, n_chunks, causal);
  if (rc != RING_ATTN_OK) return rc;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return RING_ATTN_ERR_NULL;
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return RING_ATTN_ERR_UNSUPPORTED;

  // Scratch layout: the backward workspace (see kernels.h), then the plan.
  const BwdWorkspace w = bwd_workspace(B, Hq, Hkv, L, d);
  const size_t Lpad = static_cast<size_t>(w.Lpad);
  const size_t off_plan = w.total;
  if (off_plan > kNoAllocScratchBytes) return RING_ATTN_ERR_WORKSPACE;  // beyond the static array

  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  unsigned char* scratch;
  if ((rc = scratch_address(dev, &scratch)) != RING_ATTN_OK) return rc;
  int* err;
  if ((rc = status_ptr(dev, &err)) != RING_ATTN_OK) return rc;

  const HostPlan* plan;
  if ((rc = host_plan(L, n_chunks, causal != 0, &plan)) != RING_ATTN_OK) return rc;
  const size_t plan_bytes = plan->n_words * sizeof(int32_t);
  if (off_plan + plan_bytes > kNoAllocScratchBytes) return RING_ATTN_ERR_WORKSPACE;
  int32_t* dplan = reinterpret_cast<int32_t*>(scratch + off_plan);
  if (cudaMemcpyAsync(dplan, plan->words, plan_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;

  BwdArgs a;
  std::memset(&a, 0, sizeof a);
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map(&a.tm_q, q, bf, 2, d, L, B * Hq, 64) || !make_map(&a.tm_k, k, bf, 2, d, L, B * Hkv, 64) ||
      !make_map(&a.tm_v, v, bf, 2, d, L, B * Hkv, 64) || !make_map(&a.tm_do, dO, bf, 2, d, L, B * Hq, 64))
    return RING_ATTN_ERR_CUDA;
  if (w.kv_accumulate &&
      (!make_map(&a.tm_dkacc, scratch + w.dk, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, static_cast<int>(Lpad),
                 B * Hkv, 32, 32) ||
       !make_map(&a.tm_dvacc, scratch + w.dv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, static_cast<int>(Lpad),
                 B * Hkv, 32, 32)))
    return RING_ATTN_ERR_CUDA;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = L; a.Lpad = static_cast<int>(Lpad); a.d = d; a.causal = causal != 0;
  a.n_blocks = plan->n_blocks;
  a.order = dplan;
  a.offsets = dplan + plan->n_blocks;
  a.ranges = dplan + 2 * plan->n_blocks + 1;
  a.o = o; a.dO = dO; a.lse = lse;
  a.lse2 = reinterpret_cast<float*>(scratch + w.lse2);
  a.Dvec = reinterpret_cast<float*>(scratch + w.dvec);
  a.dq_acc = reinterpret_cast<float*>(scratch + w.dq);
  a.dk_acc = w.kv_accumulate ? reinterpret_cast<float*>(scratch + w.dk) : nullptr;
  a.dv_acc = w.kv_accumulate ? reinterpret_cast<float*>(scratch + w.dv) : nullptr;
  a.dq = dq; a.dk = dk; a.dv = dv; a.err = err;
  a.timer = active_timer();  // counted under ring_attn_profile_read like ring_attn_bwd's launches
  return launch_bwd(a, stream) == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA;
}
