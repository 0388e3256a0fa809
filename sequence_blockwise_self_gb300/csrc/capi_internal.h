// capi_internal.h -- what the C ABI's translation units (ring_attn_capi.cu,
// capi_parallel.cu, capi_ffn.cu) share: the library lock, tensor-map
// encoding, argument checks, cached device plans, the status word and the
// fused attention launches on checked arguments.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "kernels.h"

namespace ra {

// Serialises the library's host state (plan caches, status words, timer).
extern std::mutex g_mutex;

// Device copy of a launch plan (see plan.h): order | offsets | ranges.
struct DevicePlan {
  int n_blocks = 0;
  int32_t* dev = nullptr;
  const int32_t* order() const { return dev; }
  const int32_t* offsets() const { return dev + n_blocks; }
  const int32_t* ranges() const { return dev + 2 * n_blocks + 1; }
};

// Event timer while profiling is on, else nullptr.
LaunchTimer* active_timer();

// The driver's cuTensorMapEncodeTiled (nullptr if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();

// 3-D map over a [Z][L][d] tensor, box (box_cols, box_rows, 1), 128-byte
// swizzle; box_cols * element size is 128 bytes.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes, int d, int L, int Z,
              int box_cols, int box_rows = 128);

bool aligned16(const void* p);
size_t round_up(size_t x, size_t a);
int current_device(int* dev);

// The fused attention kernels' domain (include/ring_attn.h).
int check_shape(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal);

// Cached device plans: kind 0 forward, 1 backward (plan.h).
int get_plan(int dev, int kind, int L, int N, int causal, DevicePlan* out);
// The forward plan's work items grouped by row blocks of R rows, longest
// first within a block: the items of row block k at [k R/256, ...).
int get_block_orders(int dev, int L, int N, int causal, int R, int32_t** out);
// Address of the device's status word.
int status_ptr(int dev, int** out);

// The fused forward and backward on checked arguments (caller holds
// g_mutex; the backward's workspace of at least bwd_workspace().total).
int fwd_impl(int dev, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int L,
             int d, int n_chunks, int causal, cudaStream_t stream);
int bwd_impl(int dev, const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
             void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
             void* workspace, cudaStream_t stream);

}  // namespace ra
