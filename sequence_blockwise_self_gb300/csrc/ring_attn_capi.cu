// ring_attn_capi.cu -- the C ABI declared in include/ring_attn.h, attention
// part: argument checks, tensor-map encoding, cached launch plans and the
// launches of the fused kernels and of ring mode; status, self-test and
// profiling.  Ulysses/USP are in capi_parallel.cu, the feed-forward block
// and the blockwise transformer in capi_ffn.cu.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <numeric>
#include <memory>
#include <mutex>
#include <tuple>

#include "../../include/ring_attn.h"
#include "capi_internal.h"
#include "kernels.h"
#include "plan.h"

namespace ra {

std::mutex g_mutex;

namespace {

// Status word the kernels write when a bounded wait gives up (one per
// device: a __device__ variable is instantiated in every device context).
__device__ int g_device_status;

std::map<std::tuple<int, int, int, int, int>, DevicePlan> g_plans;  // (device, kind, L, N, causal)
// ring step plans: (device, L, N, causal, schedule, launch, first worker, end
// worker; a negative end e: the backward plan of workers [first, -e - 1))
std::map<std::tuple<int, int, int, int, int, int, int, int>, DevicePlan> g_step_plans;
// forward work items grouped by row block: (device, L, N, causal, block rows)
std::map<std::tuple<int, int, int, int, int>, int32_t*> g_block_orders;
std::map<int, int*> g_status_ptr;                                   // device -> &g_device_status

// Event pairs around launches while profiling is on.
struct EventTimer : LaunchTimer {
  bool on = false;
  struct Rec { int kind; cudaEvent_t start, stop; };
  std::vector<Rec> recs;
  cudaEvent_t pending[RING_ATTN_N_KERNELS] = {};
  void mark(int kind, bool end, cudaStream_t stream) override {
    if (!end) {
      cudaEvent_t ev;
      if (cudaEventCreate(&ev) != cudaSuccess) return;
      cudaEventRecord(ev, stream);
      pending[kind] = ev;
    } else if (pending[kind]) {
      cudaEvent_t ev;
      if (cudaEventCreate(&ev) != cudaSuccess) return;
      cudaEventRecord(ev, stream);
      recs.push_back({kind, pending[kind], ev});
      pending[kind] = nullptr;
    }
  }
};
EventTimer g_timer;

}  // namespace

LaunchTimer* active_timer() { return g_timer.on ? &g_timer : nullptr; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 3-D map over a [z][L][d] tensor, box (box_cols, box_rows, 1) with a
// 128-byte swizzle; box_cols * element size is 128 bytes, so the shared
// memory image of a box is box_rows rows of 128 bytes.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, int d, int L, int Z,
              int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(Z)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elem_bytes, static_cast<cuuint64_t>(d) * L * elem_bytes};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || L < 0 || n_chunks <= 0) return RING_ATTN_ERR_SHAPE;
  if (Hq % Hkv != 0) return RING_ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return RING_ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq >= 65536) return RING_ATTN_ERR_UNSUPPORTED;
  if (L > 0 && !chunking_ok(L, n_chunks, causal != 0)) return RING_ATTN_ERR_SHAPE;
  if (L > (1 << 30) / 2) return RING_ATTN_ERR_UNSUPPORTED;
  return RING_ATTN_OK;
}

int current_device(int* dev) { return cudaGetDevice(dev) == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int upload_plan(const Plan& p, DevicePlan* out) {
  std::vector<int32_t> flat;
  flat.insert(flat.end(), p.order.begin(), p.order.end());
  flat.insert(flat.end(), p.offsets.begin(), p.offsets.end());
  flat.insert(flat.end(), p.ranges.begin(), p.ranges.end());
  DevicePlan dp;
  dp.n_blocks = p.n_blocks;
  if (cudaMalloc(&dp.dev, flat.size() * sizeof(int32_t)) != cudaSuccess) return RING_ATTN_ERR_CUDA;
  if (cudaMemcpy(dp.dev, flat.data(), flat.size() * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(dp.dev);
    return RING_ATTN_ERR_CUDA;
  }
  *out = dp;
  return RING_ATTN_OK;
}

// Device copy of a plan, built and uploaded on first use of a shape.
int get_plan(int dev, int kind, int L, int N, int causal, DevicePlan* out) {
  auto key = std::make_tuple(dev, kind, L, N, causal);
  auto it = g_plans.find(key);
  if (it != g_plans.end()) {
    *out = it->second;
    return RING_ATTN_OK;
  }
  DevicePlan dp;
  int rc = upload_plan(kind == 0 ? build_fwd_plan(L, N, causal != 0) : build_bwd_plan(L, N, causal != 0), &dp);
  if (rc != RING_ATTN_OK) return rc;
  g_plans[key] = dp;
  *out = dp;
  return RING_ATTN_OK;
}

int status_ptr(int dev, int** out) {
  auto it = g_status_ptr.find(dev);
  if (it != g_status_ptr.end()) {
    *out = it->second;
    return RING_ATTN_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return RING_ATTN_ERR_CUDA;
  g_status_ptr[dev] = static_cast<int*>(p);
  *out = static_cast<int*>(p);
  return RING_ATTN_OK;
}

int get_step_plan(int dev, int L, int N, int causal, int schedule, int step, int rank_lo, int rank_hi,
                  DevicePlan* out) {
  auto key = std::make_tuple(dev, L, N, causal, schedule, step, rank_lo, rank_hi);
  auto it = g_step_plans.find(key);
  if (it != g_step_plans.end()) {
    *out = it->second;
    return RING_ATTN_OK;
  }
  DevicePlan dp;
  // rank_hi < 0: the backward plan of workers [rank_lo, -rank_hi - 1)
  int rc = upload_plan(rank_hi < 0 ? build_bwd_step_plan(L, N, causal != 0, schedule, step, rank_lo, -rank_hi - 1)
                                   : build_step_plan(L, N, causal != 0, schedule, step, rank_lo, rank_hi),
                       &dp);
  if (rc != RING_ATTN_OK) return rc;
  g_step_plans[key] = dp;
  *out = dp;
  return RING_ATTN_OK;
}

// Forward work items (256-row query blocks) grouped by row blocks of R rows
// (R % 256 == 0): the items of row block k, longest first, at [k R/256,
// min((k+1) R/256, n_items)) of a device array.
int get_block_orders(int dev, int L, int N, int causal, int R, int32_t** out) {
  auto key = std::make_tuple(dev, L, N, causal, R);
  auto it = g_block_orders.find(key);
  if (it != g_block_orders.end()) {
    *out = it->second;
    return RING_ATTN_OK;
  }
  const Plan p = build_fwd_plan(L, N, causal != 0);
  const int per = R / kQBlockRows;
  std::vector<int32_t> v(p.n_blocks);
  for (int u0 = 0; u0 < p.n_blocks; u0 += per) {
    const int u1 = std::min(u0 + per, p.n_blocks);
    std::iota(v.begin() + u0, v.begin() + u1, u0);
    std::stable_sort(v.begin() + u0, v.begin() + u1, [&](int a, int b) { return p.work[a] > p.work[b]; });
  }
  int32_t* d = nullptr;
  if (cudaMalloc(&d, v.size() * sizeof(int32_t)) != cudaSuccess) return RING_ATTN_ERR_CUDA;
  if (cudaMemcpy(d, v.data(), v.size() * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(d);
    return RING_ATTN_ERR_CUDA;
  }
  g_block_orders[key] = d;
  *out = d;
  return RING_ATTN_OK;
}

int check_ring_shape(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal, int schedule) {
  // the contiguous schedules are defined for causal attention only
  if (!schedule_ok(schedule, causal != 0)) return RING_ATTN_ERR_UNSUPPORTED;
  // only the fold needs L % 2N == 0; the other chunk maps L % N == 0
  int rc = check_shape(B, Hq, Hkv, L, d, n_chunks, schedule == kSchedFold ? causal : 0);
  if (rc != RING_ATTN_OK) return rc;
  if (L > 0 && !step_chunking_ok(L, n_chunks, causal != 0, schedule)) return RING_ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(n_chunks) * B * Hq >= 65536) return RING_ATTN_ERR_UNSUPPORTED;
  return RING_ATTN_OK;
}

// Launch one ring step for ranks [rank_lo, rank_hi) on chunk buffers: with
// z_rank = 1 the buffers hold every rank's chunk ([N][B][H][C][d]), with
// z_rank = 0 only the chunks of the one rank and its source.
int launch_step(int dev, const void* q, const void* k, const void* v, float* o_s, float* lse_s, int B, int Hq,
                int Hkv, int L, int d, int N, int causal, int schedule, int step, int rank_lo, int rank_hi, int z_rank,
                cudaStream_t stream, int acc_state = 0) {
  const int C = L / N;
  const int zq = (z_rank ? N : 1) * B * Hq, zkv = (z_rank ? N : 1) * B * Hkv;
  FwdArgs a;
  std::memset(&a, 0, sizeof a);
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map(&a.tm_q, q, bf, 2, d, C, zq, 64) || !make_map(&a.tm_k, k, bf, 2, d, C, zkv, 64) ||
      !make_map(&a.tm_v, v, bf, 2, d, C, zkv, 64) ||
      !make_map(&a.tm_o, o_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, C, zq, 32))
    return RING_ATTN_ERR_CUDA;
  DevicePlan plan;
  int rc = get_step_plan(dev, L, N, causal, schedule, step, rank_lo, rank_hi, &plan);
  if (rc != RING_ATTN_OK) return rc;
  int* err;
  if ((rc = status_ptr(dev, &err)) != RING_ATTN_OK) return rc;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = C; a.d = d; a.causal = causal != 0;
  a.n_blocks = plan.n_blocks;
  a.order = plan.order(); a.offsets = plan.offsets(); a.ranges = plan.ranges();
  a.lse = lse_s; a.err = err; a.timer = active_timer();
  a.step_nb = (C + kQBlockRows - 1) / kQBlockRows;
  a.step = step; a.rank_lo = rank_lo; a.n_chunks = N;
  a.sub_len = (causal && schedule == kSchedFold) ? L / (2 * N) : 0;
  a.z_rank = z_rank; a.sched = schedule; a.o32 = o_s; a.acc_state = acc_state;
  return launch_fwd(a, stream) == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA;
}

// Parts of the ring_attn_ring_fwd workspace (byte offsets, 256-aligned):
// q, k, v in chunk order and the running fp32 result.
struct RingWorkspace {
  size_t qc = 0, kc = 0, vc = 0, oacc = 0, lacc = 0, total = 0;
};

RingWorkspace ring_workspace(int B, int Hq, int Hkv, int L, int d) {
  auto up = [](size_t x) { return round_up(x, 256); };
  const size_t nq = static_cast<size_t>(B) * Hq * L, nkv = static_cast<size_t>(B) * Hkv * L;
  RingWorkspace w;
  w.kc = w.qc + up(nq * d * 2);
  w.vc = w.kc + up(nkv * d * 2);
  w.oacc = w.vc + up(nkv * d * 2);
  w.lacc = w.oacc + up(nq * d * 4);
  w.total = w.lacc + up(nq * 4);
  return w;
}


int plan_query(int kind, int L, int n_chunks, int causal, int* n_blocks, int* n_ranges, int32_t* order,
               int32_t* offsets, int32_t* ranges) {
  if (L <= 0 || n_chunks <= 0 || !chunking_ok(L, n_chunks, causal != 0)) return RING_ATTN_ERR_SHAPE;
  Plan p = kind == 0 ? build_fwd_plan(L, n_chunks, causal != 0) : build_bwd_plan(L, n_chunks, causal != 0);
  if (n_blocks) *n_blocks = p.n_blocks;
  if (n_ranges) *n_ranges = static_cast<int>(p.ranges.size() / 2);
  if (order) std::memcpy(order, p.order.data(), p.order.size() * sizeof(int32_t));
  if (offsets) std::memcpy(offsets, p.offsets.data(), p.offsets.size() * sizeof(int32_t));
  if (ranges) std::memcpy(ranges, p.ranges.data(), p.ranges.size() * sizeof(int32_t));
  return RING_ATTN_OK;
}

// The fused forward on checked arguments (caller holds g_mutex).
int fwd_impl(int dev, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int L,
             int d, int n_chunks, int causal, cudaStream_t stream) {
  FwdArgs a;
  std::memset(&a, 0, sizeof a);
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map(&a.tm_q, q, bf, 2, d, L, B * Hq, 64) || !make_map(&a.tm_k, k, bf, 2, d, L, B * Hkv, 64) ||
      !make_map(&a.tm_v, v, bf, 2, d, L, B * Hkv, 64) || !make_map(&a.tm_o, o, bf, 2, d, L, B * Hq, 64))
    return RING_ATTN_ERR_CUDA;
  DevicePlan plan;
  int rc;
  if ((rc = get_plan(dev, 0, L, n_chunks, causal != 0, &plan)) != RING_ATTN_OK) return rc;
  int* err;
  if ((rc = status_ptr(dev, &err)) != RING_ATTN_OK) return rc;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = L; a.d = d; a.causal = causal != 0;
  a.n_blocks = plan.n_blocks;
  a.order = plan.order(); a.offsets = plan.offsets(); a.ranges = plan.ranges();
  a.lse = lse; a.err = err; a.timer = active_timer();
  return launch_fwd(a, stream) == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA;
}

// The fused backward on checked arguments and a workspace of at least
// bwd_workspace(...).total bytes (caller holds g_mutex).
int bwd_impl(int dev, const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
             void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
             void* workspace, cudaStream_t stream) {
  const BwdWorkspace w = bwd_workspace(B, Hq, Hkv, L, d);
  BwdArgs a;
  std::memset(&a, 0, sizeof a);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int Lpad = static_cast<int>(round_up(static_cast<size_t>(L), 128));
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map(&a.tm_q, q, bf, 2, d, L, B * Hq, 64) || !make_map(&a.tm_k, k, bf, 2, d, L, B * Hkv, 64) ||
      !make_map(&a.tm_v, v, bf, 2, d, L, B * Hkv, 64) || !make_map(&a.tm_do, dO, bf, 2, d, L, B * Hq, 64))
    return RING_ATTN_ERR_CUDA;
  if (w.kv_accumulate &&
      (!make_map(&a.tm_dkacc, ws + w.dk, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, Lpad, B * Hkv, 32, 32) ||
       !make_map(&a.tm_dvacc, ws + w.dv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, Lpad, B * Hkv, 32, 32)))
    return RING_ATTN_ERR_CUDA;
  DevicePlan plan;
  int rc;
  if ((rc = get_plan(dev, 1, L, n_chunks, causal != 0, &plan)) != RING_ATTN_OK) return rc;
  int* err;
  if ((rc = status_ptr(dev, &err)) != RING_ATTN_OK) return rc;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = L; a.Lpad = Lpad; a.d = d; a.causal = causal != 0;
  a.n_blocks = plan.n_blocks;
  a.order = plan.order(); a.offsets = plan.offsets(); a.ranges = plan.ranges();
  a.o = o; a.dO = dO; a.lse = lse;
  a.lse2 = reinterpret_cast<float*>(ws + w.lse2);
  a.Dvec = reinterpret_cast<float*>(ws + w.dvec);
  a.dq_acc = reinterpret_cast<float*>(ws + w.dq);
  a.dk_acc = w.kv_accumulate ? reinterpret_cast<float*>(ws + w.dk) : nullptr;
  a.dv_acc = w.kv_accumulate ? reinterpret_cast<float*>(ws + w.dv) : nullptr;
  a.dq = dq; a.dk = dk; a.dv = dv; a.err = err; a.timer = active_timer();
  return launch_bwd(a, stream) == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA;
}

// Ring-mode backward: parts of the workspace (byte offsets, 256-aligned):
// q, k, v, o, dO and lse in chunk order, the statistics (-lse log2 e, -D),
// and the fp32 gradient accumulators (dQ tiled as in the fused backward).
struct RingBwdWorkspace {
  size_t qc = 0, kc = 0, vc = 0, oc = 0, dOc = 0, lsec = 0, lse2 = 0, dvec = 0, dq = 0, dk = 0, dv = 0, total = 0;
};

RingBwdWorkspace ring_bwd_workspace(int B, int Hq, int Hkv, int L, int d) {
  auto up = [](size_t x) { return round_up(x, 256); };
  const size_t nq = static_cast<size_t>(B) * Hq * L, nkv = static_cast<size_t>(B) * Hkv * L;
  RingBwdWorkspace w;
  w.kc = w.qc + up(nq * d * 2);
  w.vc = w.kc + up(nkv * d * 2);
  w.oc = w.vc + up(nkv * d * 2);
  w.dOc = w.oc + up(nq * d * 2);
  w.lsec = w.dOc + up(nq * d * 2);
  w.lse2 = w.lsec + up(nq * 4);
  w.dvec = w.lse2 + up(nq * 4);
  w.dq = w.dvec + up(nq * 4);
  w.dk = w.dq + up(nq * d * 4);
  w.dv = w.dk + up(nkv * d * 4);
  w.total = w.dv + up(nkv * d * 4);
  return w;
}

// Ulysses: parts of the workspace (byte offsets, 256-aligned): head-shard
// copies of q, k, v, o, lse (forward), then dO, dq, dk, dv and the fused
// backward's own workspace for the head-shard problem (backward).
// Device status word of the current device, for the library's other entry
// points (ring_attn_noalloc.cu).
int status_word_for_current_device(int** out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if (current_device(&dev) != RING_ATTN_OK) return RING_ATTN_ERR_CUDA;
  return status_ptr(dev, out);
}

}  // namespace ra

using namespace ra;

extern "C" {

const char* ring_attn_strerror(int status) {
  switch (status) {
    case RING_ATTN_OK: return "ok";
    case RING_ATTN_ERR_NULL: return "a required pointer is NULL";
    case RING_ATTN_ERR_SHAPE: return "invalid shape or chunking";
    case RING_ATTN_ERR_UNSUPPORTED: return "unsupported head dimension, alignment or size";
    case RING_ATTN_ERR_WORKSPACE: return "backward workspace missing or too small";
    case RING_ATTN_ERR_CUDA: return "CUDA runtime or driver call failed";
    case RING_ATTN_ERR_DEVICE_TIMEOUT: return "a kernel aborted a bounded wait";
    default: return "unknown status";
  }
}

int ring_attn_owner_rank(int L, int n_chunks, int causal, int pos) {
  if (L <= 0 || n_chunks <= 0 || !chunking_ok(L, n_chunks, causal != 0)) return RING_ATTN_ERR_SHAPE;
  if (pos < 0 || pos >= L) return RING_ATTN_ERR_SHAPE;
  return owner_rank(L, n_chunks, causal != 0, pos);
}

int ring_attn_fwd_plan(int L, int n_chunks, int causal, int* n_blocks, int* n_ranges, int32_t* block_order,
                       int32_t* range_offsets, int32_t* ranges) {
  return plan_query(0, L, n_chunks, causal, n_blocks, n_ranges, block_order, range_offsets, ranges);
}

int ring_attn_bwd_plan(int L, int n_chunks, int causal, int* n_blocks, int* n_ranges, int32_t* block_order,
                       int32_t* range_offsets, int32_t* ranges) {
  return plan_query(1, L, n_chunks, causal, n_blocks, n_ranges, block_order, range_offsets, ranges);
}

int ring_attn_schedule_launches(int n_chunks, int schedule) {
  if (n_chunks <= 0 || !schedule_ok(schedule, true)) return RING_ATTN_ERR_SHAPE;
  return schedule_launches(n_chunks, schedule);
}

int ring_attn_schedule_pair(int n_chunks, int schedule, int launch, int worker, int* q_chunk, int* kv_chunk) {
  if (n_chunks <= 0 || !schedule_ok(schedule, true)) return RING_ATTN_ERR_SHAPE;
  if (launch < 0 || launch >= schedule_launches(n_chunks, schedule) || worker < 0 || worker >= n_chunks)
    return RING_ATTN_ERR_SHAPE;
  if (!q_chunk || !kv_chunk) return RING_ATTN_ERR_NULL;
  return schedule_pair(n_chunks, schedule, launch, worker, q_chunk, kv_chunk) ? 1 : 0;
}

int ring_attn_step_plan(int L, int n_chunks, int causal, int schedule, int step, int rank, int* n_blocks,
                        int* n_ranges, int32_t* block_order, int32_t* range_offsets, int32_t* ranges) {
  if (L <= 0 || n_chunks <= 0 || !chunking_ok(L, n_chunks, schedule == kSchedFold && causal != 0))
    return RING_ATTN_ERR_SHAPE;
  if (!step_chunking_ok(L, n_chunks, causal != 0, schedule)) return RING_ATTN_ERR_UNSUPPORTED;
  if (step < 0 || step >= schedule_launches(n_chunks, schedule) || rank < 0 || rank >= n_chunks)
    return RING_ATTN_ERR_SHAPE;
  Plan p = build_step_plan(L, n_chunks, causal != 0, schedule, step, rank, rank + 1);
  if (n_blocks) *n_blocks = p.n_blocks;
  if (n_ranges) *n_ranges = static_cast<int>(p.ranges.size() / 2);
  if (block_order) std::memcpy(block_order, p.order.data(), p.order.size() * sizeof(int32_t));
  if (range_offsets) std::memcpy(range_offsets, p.offsets.data(), p.offsets.size() * sizeof(int32_t));
  if (ranges) std::memcpy(ranges, p.ranges.data(), p.ranges.size() * sizeof(int32_t));
  return RING_ATTN_OK;
}

int ring_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int L,
                  int d, int n_chunks, int causal, cudaStream_t stream) {
  int rc = check_shape(B, Hq, Hkv, L, d, n_chunks, causal);
  if (rc != RING_ATTN_OK) return rc;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q || !k || !v || !o || !lse) return RING_ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return RING_ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  return fwd_impl(dev, q, k, v, o, lse, B, Hq, Hkv, L, d, n_chunks, causal, stream);
}

size_t ring_attn_bwd_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal) {
  if (check_shape(B, Hq, Hkv, L, d, n_chunks, causal) != RING_ATTN_OK) return 0;
  return bwd_workspace(B, Hq, Hkv, L, d).total;
}

int ring_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_shape(B, Hq, Hkv, L, d, n_chunks, causal);
  if (rc != RING_ATTN_OK) return rc;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return RING_ATTN_ERR_NULL;
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return RING_ATTN_ERR_UNSUPPORTED;
  const BwdWorkspace w = bwd_workspace(B, Hq, Hkv, L, d);
  if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return RING_ATTN_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  return bwd_impl(dev, q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, L, d, n_chunks, causal, workspace, stream);
}

int ring_attn_device_status(cudaStream_t stream, int* site) {
  if (site) *site = 0;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if (current_device(&dev) != RING_ATTN_OK) return RING_ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return RING_ATTN_ERR_CUDA;
  int* p;
  if (status_ptr(dev, &p) != RING_ATTN_OK) return RING_ATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return RING_ATTN_ERR_CUDA;
  if (v == 0) return RING_ATTN_OK;
  if (site) *site = v;
  const int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return RING_ATTN_ERR_CUDA;
  return RING_ATTN_ERR_DEVICE_TIMEOUT;
}

int ring_attn_selftest_bounded_wait(unsigned timeout_us, cudaStream_t stream) {
  if (timeout_us == 0 || timeout_us > 10000000u) return RING_ATTN_ERR_SHAPE;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if (current_device(&dev) != RING_ATTN_OK) return RING_ATTN_ERR_CUDA;
  int* err;
  if (status_ptr(dev, &err) != RING_ATTN_OK) return RING_ATTN_ERR_CUDA;
  return launch_selftest_wait(err, 1000ull * timeout_us, stream) == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA;
}

int ring_attn_profile_enable(int on) {
  std::lock_guard<std::mutex> lock(g_mutex);
  g_timer.on = on != 0;
  return RING_ATTN_OK;
}

int ring_attn_profile_read(double* ms, long long* launches) {
  std::lock_guard<std::mutex> lock(g_mutex);
  for (int k = 0; k < RING_ATTN_N_KERNELS; ++k) {
    if (ms) ms[k] = 0.0;
    if (launches) launches[k] = 0;
  }
  int rc = RING_ATTN_OK;
  for (auto& r : g_timer.recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      rc = RING_ATTN_ERR_CUDA;
    if (ms) ms[r.kind] += t;
    if (launches) launches[r.kind] += 1;
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_timer.recs.clear();
  return rc;
}

int ring_attn_fwd_step(const void* q_chunk, const void* k_chunk, const void* v_chunk, float* o_s, float* lse_s,
                       int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal, int schedule, int rank, int src,
                       cudaStream_t stream) {
  int rc = check_ring_shape(B, Hq, Hkv, L, d, n_chunks, causal, schedule);
  if (rc != RING_ATTN_OK) return rc;
  if (rank < 0 || rank >= n_chunks || src < 0 || src >= n_chunks) return RING_ATTN_ERR_SHAPE;
  // one block (rank's queries, src's keys): for the contiguous chunk map the
  // schedule only decides who runs it when, so DistFlashAttention's blocks
  // are the plain ring's
  if (schedule == kSchedDfa) schedule = kSchedContig;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q_chunk || !k_chunk || !v_chunk || !o_s || !lse_s) return RING_ATTN_ERR_NULL;
  if (!aligned16(q_chunk) || !aligned16(k_chunk) || !aligned16(v_chunk) || !aligned16(o_s) || !aligned16(lse_s))
    return RING_ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  const int step = ((rank - src) % n_chunks + n_chunks) % n_chunks;
  return launch_step(dev, q_chunk, k_chunk, v_chunk, o_s, lse_s, B, Hq, Hkv, L, d, n_chunks, causal, schedule, step,
                     rank, rank + 1, 0, stream);
}

int ring_attn_fwd_step_accumulate(const void* q_chunk, const void* k_chunk, const void* v_chunk, float* o_run,
                                  float* lse_run, int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                                  int schedule, int rank, int src, cudaStream_t stream) {
  int rc = check_ring_shape(B, Hq, Hkv, L, d, n_chunks, causal, schedule);
  if (rc != RING_ATTN_OK) return rc;
  if (rank < 0 || rank >= n_chunks || src < 0 || src >= n_chunks) return RING_ATTN_ERR_SHAPE;
  if (schedule == kSchedDfa) schedule = kSchedContig;  // the same block
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q_chunk || !k_chunk || !v_chunk || !o_run || !lse_run) return RING_ATTN_ERR_NULL;
  if (!aligned16(q_chunk) || !aligned16(k_chunk) || !aligned16(v_chunk) || !aligned16(o_run) || !aligned16(lse_run))
    return RING_ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  const int step = ((rank - src) % n_chunks + n_chunks) % n_chunks;
  return launch_step(dev, q_chunk, k_chunk, v_chunk, o_run, lse_run, B, Hq, Hkv, L, d, n_chunks, causal, schedule,
                     step, rank, rank + 1, 0, stream, 1);
}

int ring_attn_merge(float* o, float* lse, const float* o_s, const float* lse_s, long long n_rows, int d,
                    void* o_out, cudaStream_t stream) {
  if (n_rows < 0) return RING_ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return RING_ATTN_ERR_UNSUPPORTED;
  if (n_rows == 0) return RING_ATTN_OK;
  if (!o || !lse || !o_s || !lse_s) return RING_ATTN_ERR_NULL;
  if (!aligned16(o) || !aligned16(o_s) || (o_out && !aligned16(o_out))) return RING_ATTN_ERR_UNSUPPORTED;
  LaunchTimer* t = active_timer();
  if (t) t->mark(RING_ATTN_KERNEL_RING_MERGE, false, stream);
  const cudaError_t e = launch_ring_merge(o, lse, o_s, lse_s, o_out, n_rows, d, stream);
  if (t) t->mark(RING_ATTN_KERNEL_RING_MERGE, true, stream);
  return e == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA;
}

size_t ring_attn_ring_fwd_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                                         int schedule) {
  if (check_ring_shape(B, Hq, Hkv, L, d, n_chunks, causal, schedule) != RING_ATTN_OK) return 0;
  return ring_workspace(B, Hq, Hkv, L, d).total;
}

int ring_attn_ring_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                       int L, int d, int n_chunks, int causal, int schedule, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream) {
  int rc = check_ring_shape(B, Hq, Hkv, L, d, n_chunks, causal, schedule);
  if (rc != RING_ATTN_OK) return rc;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q || !k || !v || !o || !lse) return RING_ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return RING_ATTN_ERR_UNSUPPORTED;
  const RingWorkspace w = ring_workspace(B, Hq, Hkv, L, d);
  if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return RING_ATTN_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* qc = ws + w.qc;
  void* kc = ws + w.kc;
  void* vc = ws + w.vc;
  float* oacc = reinterpret_cast<float*>(ws + w.oacc);
  float* lacc = reinterpret_cast<float*>(ws + w.lacc);
  const int N = n_chunks;
  LaunchTimer* t = active_timer();
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, false, stream);
  const bool sc = causal != 0;
  const int st = schedule;
  if (launch_ring_gather(q, qc, B * Hq, L, d, N, sc, st, stream) != cudaSuccess ||
      launch_ring_gather(k, kc, B * Hkv, L, d, N, sc, st, stream) != cudaSuccess ||
      launch_ring_gather(v, vc, B * Hkv, L, d, N, sc, st, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, true, stream);
  // Launch 0 (every worker's own chunk against itself) writes the running
  // result; every later launch continues each block's query chunk from it
  // and overwrites it with the merged result (the step kernel's accumulate
  // mode), so no partial result or separate merge is needed.  A query chunk
  // must appear once per launch: DistFlashAttention's launches run as two,
  // the workers' own chunks (workers t..N-1), then the chunks the idle
  // workers 0..t-1 take over (chunks N-t..N-1, unless t = N - t).
  for (int s = 0; s < schedule_launches(N, schedule); ++s) {
    const int lo = (schedule == kSchedDfa) ? s : 0;
    if ((rc = launch_step(dev, qc, kc, vc, oacc, lacc, B, Hq, Hkv, L, d, N, causal, schedule, s, lo, N, 1, stream,
                          s > 0 ? 1 : 0)) != RING_ATTN_OK)
      return rc;
    if (schedule == kSchedDfa && s > 0 && s < N - s &&
        (rc = launch_step(dev, qc, kc, vc, oacc, lacc, B, Hq, Hkv, L, d, N, causal, schedule, s, 0, s, 1, stream, 1)) !=
            RING_ATTN_OK)
      return rc;
  }
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, false, stream);
  if (launch_ring_scatter(oacc, lacc, o, lse, B * Hq, L, d, N, sc, st, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, true, stream);
  return RING_ATTN_OK;
}

size_t ring_attn_ring_bwd_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                                         int schedule) {
  if (check_ring_shape(B, Hq, Hkv, L, d, n_chunks, causal, schedule) != RING_ATTN_OK) return 0;
  return ring_bwd_workspace(B, Hq, Hkv, L, d).total;
}

int ring_attn_ring_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                       void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                       int schedule, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_ring_shape(B, Hq, Hkv, L, d, n_chunks, causal, schedule);
  if (rc != RING_ATTN_OK) return rc;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return RING_ATTN_ERR_NULL;
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return RING_ATTN_ERR_UNSUPPORTED;
  const RingBwdWorkspace w = ring_bwd_workspace(B, Hq, Hkv, L, d);
  if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return RING_ATTN_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int N = n_chunks, C = L / N;
  const bool sc = causal != 0;
  const int st = schedule;
  LaunchTimer* t = active_timer();
  // every rank's rows in chunk order
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, false, stream);
  if (launch_ring_gather(q, ws + w.qc, B * Hq, L, d, N, sc, st, stream) != cudaSuccess ||
      launch_ring_gather(k, ws + w.kc, B * Hkv, L, d, N, sc, st, stream) != cudaSuccess ||
      launch_ring_gather(v, ws + w.vc, B * Hkv, L, d, N, sc, st, stream) != cudaSuccess ||
      launch_ring_gather(o, ws + w.oc, B * Hq, L, d, N, sc, st, stream) != cudaSuccess ||
      launch_ring_gather(dO, ws + w.dOc, B * Hq, L, d, N, sc, st, stream) != cudaSuccess ||
      launch_ring_gather_rows(lse, reinterpret_cast<float*>(ws + w.lsec), B * Hq, L, N, sc, st, stream) !=
          cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, true, stream);
  BwdArgs a;
  std::memset(&a, 0, sizeof a);
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const int zq = N * B * Hq, zkv = N * B * Hkv;
  if (!make_map(&a.tm_q, ws + w.qc, bf, 2, d, C, zq, 64) || !make_map(&a.tm_k, ws + w.kc, bf, 2, d, C, zkv, 64) ||
      !make_map(&a.tm_v, ws + w.vc, bf, 2, d, C, zkv, 64) || !make_map(&a.tm_do, ws + w.dOc, bf, 2, d, C, zq, 64) ||
      !make_map(&a.tm_dkacc, ws + w.dk, f32, 4, d, C, zkv, 32, 32) ||
      !make_map(&a.tm_dvacc, ws + w.dv, f32, 4, d, C, zkv, 32, 32))
    return RING_ATTN_ERR_CUDA;
  int* err;
  if ((rc = status_ptr(dev, &err)) != RING_ATTN_OK) return rc;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.L = C; a.Lpad = C; a.d = d; a.causal = sc;
  a.o = ws + w.oc; a.dO = ws + w.dOc; a.lse = reinterpret_cast<const float*>(ws + w.lsec);
  a.lse2 = reinterpret_cast<float*>(ws + w.lse2);
  a.Dvec = reinterpret_cast<float*>(ws + w.dvec);
  a.dq_acc = reinterpret_cast<float*>(ws + w.dq);
  a.dk_acc = reinterpret_cast<float*>(ws + w.dk);
  a.dv_acc = reinterpret_cast<float*>(ws + w.dv);
  a.err = err; a.timer = t;
  // statistics of every rank's rows, accumulators zeroed
  if (launch_bwd_pre(a, zq, zkv, stream) != cudaSuccess) return RING_ATTN_ERR_CUDA;
  a.step_nt = C / kTileRows; a.n_chunks = N; a.sched = schedule;
  a.rank_lo = 0; a.z_rank = 1;  // every worker's chunk, chunk-major
  for (int s = 0; s < schedule_launches(N, schedule); ++s) {
    DevicePlan plan;
    if ((rc = get_step_plan(dev, L, N, causal, schedule, s, 0, -N - 1, &plan)) != RING_ATTN_OK) return rc;
    a.n_blocks = plan.n_blocks;
    a.order = plan.order(); a.offsets = plan.offsets(); a.ranges = plan.ranges();
    a.step = s;
    if (launch_bwd(a, stream) != cudaSuccess) return RING_ATTN_ERR_CUDA;
  }
  const float scale = 1.0f / sqrtf(static_cast<float>(d));
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, false, stream);
  if (launch_ring_scatter_grad(a.dq_acc, dq, scale, true, B * Hq, L, d, N, sc, st, stream) != cudaSuccess ||
      launch_ring_scatter_grad(a.dk_acc, dk, scale, false, B * Hkv, L, d, N, sc, st, stream) != cudaSuccess ||
      launch_ring_scatter_grad(a.dv_acc, dv, 1.f, false, B * Hkv, L, d, N, sc, st, stream) != cudaSuccess)
    return RING_ATTN_ERR_CUDA;
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, true, stream);
  return RING_ATTN_OK;
}

// ----------------------------------------------------- one rank's backward
// Workspace of ring_attn_bwd_rank_*: the rank's statistics (-lse log2 e and
// -D, [B*Hq][C] each) and its fp32 dQ accumulator (tiled as in the fused
// backward), 256-byte aligned parts.
struct RankBwdWorkspace {
  size_t lse2 = 0, dvec = 0, dq = 0, total = 0;
};

RankBwdWorkspace rank_bwd_workspace(int B, int Hq, int C, int d) {
  auto up = [](size_t x) { return round_up(x, 256); };
  const size_t rows = static_cast<size_t>(B) * Hq * C;
  RankBwdWorkspace w;
  w.dvec = up(rows * 4);
  w.dq = w.dvec + up(rows * 4);
  w.total = w.dq + up(rows * d * 4);
  return w;
}

size_t ring_attn_bwd_rank_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                                         int schedule) {
  if (check_ring_shape(B, Hq, Hkv, L, d, n_chunks, causal, schedule) != RING_ATTN_OK) return 0;
  return rank_bwd_workspace(B, Hq, L / n_chunks, d).total;
}

namespace {
// Common checks of the ring_attn_bwd_rank_* calls; fills the workspace parts.
int rank_bwd_args(BwdArgs* a, int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal, int schedule,
                  const void* ws, size_t ws_bytes) {
  int rc = check_ring_shape(B, Hq, Hkv, L, d, n_chunks, causal, schedule);
  if (rc != RING_ATTN_OK) return rc;
  const int C = L / n_chunks;
  const RankBwdWorkspace w = rank_bwd_workspace(B, Hq, C, d);
  if (!ws || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return RING_ATTN_ERR_WORKSPACE;
  std::memset(a, 0, sizeof *a);
  uint8_t* p = static_cast<uint8_t*>(const_cast<void*>(ws));
  a->B = B; a->Hq = Hq; a->Hkv = Hkv; a->L = C; a->Lpad = C; a->d = d; a->causal = causal != 0;
  a->lse2 = reinterpret_cast<float*>(p + w.lse2);
  a->Dvec = reinterpret_cast<float*>(p + w.dvec);
  a->dq_acc = reinterpret_cast<float*>(p + w.dq);
  return RING_ATTN_OK;
}
}  // namespace

int ring_attn_bwd_rank_begin(const void* o_chunk, const void* dO_chunk, const float* lse_chunk, int B, int Hq,
                             int Hkv, int L, int d, int n_chunks, int causal, int schedule, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  BwdArgs a;
  int rc = rank_bwd_args(&a, B, Hq, Hkv, L, d, n_chunks, causal, schedule, workspace, workspace_bytes);
  if (rc != RING_ATTN_OK) return rc;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!o_chunk || !dO_chunk || !lse_chunk) return RING_ATTN_ERR_NULL;
  if (!aligned16(o_chunk) || !aligned16(dO_chunk) || !aligned16(lse_chunk)) return RING_ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  a.o = o_chunk; a.dO = dO_chunk; a.lse = lse_chunk; a.timer = active_timer();
  return launch_bwd_pre(a, static_cast<long long>(B) * Hq, 0, stream) == cudaSuccess ? RING_ATTN_OK
                                                                                       : RING_ATTN_ERR_CUDA;
}

int ring_attn_bwd_rank_step(const void* q_chunk, const void* k_chunk, const void* v_chunk, const void* dO_chunk,
                            float* dk_acc, float* dv_acc, int B, int Hq, int Hkv, int L, int d, int n_chunks,
                            int causal, int schedule, int rank, int src, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  BwdArgs a;
  int rc = rank_bwd_args(&a, B, Hq, Hkv, L, d, n_chunks, causal, schedule, workspace, workspace_bytes);
  if (rc != RING_ATTN_OK) return rc;
  if (rank < 0 || rank >= n_chunks || src < 0 || src >= n_chunks) return RING_ATTN_ERR_SHAPE;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!q_chunk || !k_chunk || !v_chunk || !dO_chunk || !dk_acc || !dv_acc) return RING_ATTN_ERR_NULL;
  const void* ptrs[] = {q_chunk, k_chunk, v_chunk, dO_chunk, dk_acc, dv_acc};
  for (const void* p : ptrs)
    if (!aligned16(p)) return RING_ATTN_ERR_UNSUPPORTED;
  if (schedule == kSchedDfa) schedule = kSchedContig;  // one block: DistFlashAttention's is the ring's
  const int N = n_chunks, C = L / N;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (!make_map(&a.tm_q, q_chunk, bf, 2, d, C, B * Hq, 64) || !make_map(&a.tm_k, k_chunk, bf, 2, d, C, B * Hkv, 64) ||
      !make_map(&a.tm_v, v_chunk, bf, 2, d, C, B * Hkv, 64) ||
      !make_map(&a.tm_do, dO_chunk, bf, 2, d, C, B * Hq, 64) ||
      !make_map(&a.tm_dkacc, dk_acc, f32, 4, d, C, B * Hkv, 32, 32) ||
      !make_map(&a.tm_dvacc, dv_acc, f32, 4, d, C, B * Hkv, 32, 32))
    return RING_ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev;
  if ((rc = current_device(&dev)) != RING_ATTN_OK) return rc;
  const int step = ((rank - src) % N + N) % N;
  DevicePlan plan;
  if ((rc = get_step_plan(dev, L, N, causal, schedule, step, rank, -(rank + 1) - 1, &plan)) != RING_ATTN_OK) return rc;
  int* err;
  if ((rc = status_ptr(dev, &err)) != RING_ATTN_OK) return rc;
  a.dk_acc = dk_acc; a.dv_acc = dv_acc;
  a.n_blocks = plan.n_blocks;
  a.order = plan.order(); a.offsets = plan.offsets(); a.ranges = plan.ranges();
  a.err = err; a.timer = active_timer();
  a.step_nt = C / kTileRows; a.n_chunks = N; a.sched = schedule; a.step = step;
  a.rank_lo = rank; a.z_rank = 0;  // buffers hold the block's two chunks only
  return launch_bwd(a, stream) == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA;
}

int ring_attn_bwd_rank_end(void* dq_chunk, int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                           int schedule, const void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  BwdArgs a;
  int rc = rank_bwd_args(&a, B, Hq, Hkv, L, d, n_chunks, causal, schedule, workspace, workspace_bytes);
  if (rc != RING_ATTN_OK) return rc;
  if (B == 0 || L == 0) return RING_ATTN_OK;
  if (!dq_chunk) return RING_ATTN_ERR_NULL;
  if (!aligned16(dq_chunk)) return RING_ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  a.dq = dq_chunk;
  LaunchTimer* t = active_timer();
  if (t) t->mark(RING_ATTN_KERNEL_BWD_POST, false, stream);
  const cudaError_t e = launch_bwd_dq_post(a, static_cast<long long>(B) * Hq, stream);
  if (t) t->mark(RING_ATTN_KERNEL_BWD_POST, true, stream);
  return e == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA;
}

int ring_attn_grad_to_bf16(const float* acc, void* out, long long n_elems, float scale, cudaStream_t stream) {
  if (n_elems < 0 || n_elems % 128 != 0) return RING_ATTN_ERR_SHAPE;
  if (n_elems == 0) return RING_ATTN_OK;
  if (!acc || !out) return RING_ATTN_ERR_NULL;
  if (!aligned16(acc) || !aligned16(out)) return RING_ATTN_ERR_UNSUPPORTED;
  LaunchTimer* t = active_timer();
  if (t) t->mark(RING_ATTN_KERNEL_BWD_POST, false, stream);
  const cudaError_t e = launch_grad_to_bf16(acc, out, scale, n_elems, stream);
  if (t) t->mark(RING_ATTN_KERNEL_BWD_POST, true, stream);
  return e == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA;
}

size_t ring_attn_bwd_rank_dq_offset(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal, int schedule) {
  if (check_ring_shape(B, Hq, Hkv, L, d, n_chunks, causal, schedule) != RING_ATTN_OK) return 0;
  return rank_bwd_workspace(B, Hq, L / n_chunks, d).dq;
}

int ring_attn_add_f32(float* dst, const float* src, long long n_elems, cudaStream_t stream) {
  if (n_elems < 0 || n_elems % 4 != 0) return RING_ATTN_ERR_SHAPE;
  if (n_elems == 0) return RING_ATTN_OK;
  if (!dst || !src) return RING_ATTN_ERR_NULL;
  if (!aligned16(dst) || !aligned16(src)) return RING_ATTN_ERR_UNSUPPORTED;
  LaunchTimer* t = active_timer();
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, false, stream);
  const cudaError_t e = launch_add_f32(dst, src, n_elems, stream);
  if (t) t->mark(RING_ATTN_KERNEL_RING_IO, true, stream);
  return e == cudaSuccess ? RING_ATTN_OK : RING_ATTN_ERR_CUDA;
}

void ring_attn_release(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_plans) {
    cudaSetDevice(std::get<0>(kv.first));
    cudaFree(kv.second.dev);
  }
  for (auto& kv : g_step_plans) {
    cudaSetDevice(std::get<0>(kv.first));
    cudaFree(kv.second.dev);
  }
  for (auto& kv : g_block_orders) {
    cudaSetDevice(std::get<0>(kv.first));
    cudaFree(kv.second);
  }
  cudaSetDevice(cur);
  g_plans.clear();
  g_step_plans.clear();
  g_block_orders.clear();
}

}  // extern "C"
