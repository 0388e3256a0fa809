// kernels.h -- launch interface between the C ABI and the sm_103a kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ra {

// Device-side error sites (recorded when a bounded wait gives up).
enum ErrSite : int {
  kSiteFwdProducer = 0x101,
  kSiteFwdMma = 0x102,
  kSiteFwdSoftmax = 0x103,
  kSiteFwdEpilogue = 0x104,
  kSiteFwdDrain = 0x105,
  kSiteFwdMisaligned = 0x1FF,
  kSiteBwdProducer = 0x201,
  kSiteBwdMma = 0x202,
  kSiteBwdSoftmax = 0x203,
  kSiteBwdEpilogue = 0x204,
  kSiteBwdDrain = 0x205,
  kSiteBwdReducer = 0x206,
  kSiteBwdMisaligned = 0x2FF,
  kSiteSelfTest = 0x301,
};

// Optional hook that brackets each launch with events (measurement only).
struct LaunchTimer {
  virtual void mark(int kind, bool end, cudaStream_t stream) = 0;
};

struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  int B, Hq, Hkv, L, d, causal;
  int n_blocks;             // 256-row query blocks per (b, h)
  const int32_t* order;     // device [n_blocks]
  const int32_t* offsets;   // device [n_blocks + 1]
  const int32_t* ranges;    // device [2 * n_ranges]
  float* lse;               // device [B*Hq*L]
  int* err;                 // device status word
  LaunchTimer* timer;       // nullptr unless profiling
  // ring step mode (step_nb > 0; L is then the chunk length, n_blocks the
  // number of items, tm_o an fp32 map with 32-column boxes, see attn_fwd.cu)
  int step_nb = 0, step = 0, rank_lo = 0, n_chunks = 1, sub_len = 0, z_rank = 0, sched = 0;
  float* o32 = nullptr;
  // ring step that continues from and overwrites the running result in o32
  // and lse (the query chunk's slices) instead of writing a partial result
  int acc_state = 0;
  // not a ring step: o token-major [B][L][Hq][d] through a 4-D tm_o
  // (d, Hq, L, B; box 64 x 1 x 128 x 1)
  int o_token_major = 0;
};

// Backward workspace: byte offsets of its parts (each 256-byte aligned).
//   lse2 [B*Hq][Lpad] fp32, D [B*Hq][Lpad] fp32, dQ accumulator
//   [B*Hq][Lpad][d] fp32, and for grouped-query attention (Hq > Hkv) dK and
//   dV accumulators [B*Hkv][Lpad][d] fp32 (each key tile receives one
//   partial per query head of its group).
struct BwdWorkspace {
  size_t lse2 = 0, dvec = 0, dq = 0, dk = 0, dv = 0, total = 0;
  int Lpad = 0;
  bool kv_accumulate = false;
};

inline BwdWorkspace bwd_workspace(int B, int Hq, int Hkv, int L, int d) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  BwdWorkspace w;
  w.Lpad = (L + 127) / 128 * 128;
  const size_t rows = static_cast<size_t>(B) * Hq * w.Lpad;
  const size_t kv_rows = static_cast<size_t>(B) * Hkv * w.Lpad;
  w.kv_accumulate = Hq > Hkv;
  w.lse2 = 0;
  w.dvec = up(rows * sizeof(float));
  w.dq = w.dvec + up(rows * sizeof(float));
  w.dk = w.dq + up(rows * d * sizeof(float));
  w.dv = w.dk + (w.kv_accumulate ? up(kv_rows * d * sizeof(float)) : 0);
  w.total = w.dv + (w.kv_accumulate ? up(kv_rows * d * sizeof(float)) : 0);
  return w;
}

struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_dkacc, tm_dvacc;
  int B, Hq, Hkv, L, Lpad, d, causal;
  int n_blocks;             // key/value tiles per (b, kv head)
  const int32_t* order;
  const int32_t* offsets;
  const int32_t* ranges;
  const void* o;            // bf16 [B*Hq*L*d]
  const void* dO;           // bf16 [B*Hq*L*d]
  const float* lse;         // fp32 [B*Hq*L]
  float* lse2;              // workspace fp32 [B*Hq*Lpad]: -lse * log2(e), -inf padding
  float* Dvec;              // workspace fp32 [B*Hq*Lpad]: -rowsum(dO * o), 0 padding
  float* dq_acc;            // workspace fp32, B*Hq*Lpad*d, tiled per 128 query rows
  float* dk_acc;            // workspace fp32 [B*Hkv*Lpad*d] (grouped-query attention only, else null)
  float* dv_acc;            // workspace fp32 [B*Hkv*Lpad*d] (grouped-query attention only, else null)
  void* dq;                 // bf16 [B*Hq*L*d]
  void* dk;                 // bf16 [B*Hkv*L*d]
  void* dv;                 // bf16 [B*Hkv*L*d]
  int* err;
  LaunchTimer* timer;       // nullptr unless profiling
  // ring step mode (step_nt > 0: key/value tiles per chunk; n_blocks = n_chunks
  // * step_nt items; L = Lpad = the chunk length; slices chunk-major, see
  // attn_bwd.cu): only the main kernel runs, with dK/dV always reduced into
  // the fp32 accumulators; the driver runs launch_bwd_pre and the conversions
  int step_nt = 0, step = 0, n_chunks = 1, sched = 0;
  // step mode: first worker of the launch, and 1 for chunk-major buffers of
  // every chunk or 0 for buffers holding only the block's two chunks
  int rank_lo = 0, z_rank = 1;
};

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_selftest_wait(int* err, unsigned long long timeout_ns, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);
// The backward's statistics pre-pass alone over q_slices (and kv_slices for
// zeroing the dK/dV accumulators) slices of Lpad rows.
cudaError_t launch_bwd_pre(const BwdArgs& a, long long q_slices, long long kv_slices, cudaStream_t stream);
// dq = bf16(scale * dQ_acc) for q_slices slices of a.L rows (a.Lpad rows
// in the tiled accumulator), scale = 1/sqrt(d).
cudaError_t launch_bwd_dq_post(const BwdArgs& a, long long q_slices, cudaStream_t stream);
// out = bf16(scale * acc) for n_elems fp32 values (a multiple of 128).
cudaError_t launch_grad_to_bf16(const float* acc, void* out, float scale, long long n_elems, cudaStream_t stream);
// dst[0 .. n) += src[0 .. n) in fp32 (n a multiple of 4, 16-byte aligned)
cudaError_t launch_add_f32(float* dst, const float* src, long long n, cudaStream_t stream);

// Ring mode (ring_step.cu): the log-sum-exp merge of n_rows rows (in place
// into o, lse; optional bf16 copy into o_out), and the gather of a [Z][L][d]
// bf16 tensor into chunk order [N][Z][C][d] / the scatter of the fp32 result
// [N][Z][C][d] (+ lse [N][Z][C]) back to sequence order as bf16 (+ lse).
cudaError_t launch_ring_merge(float* o, float* lse, const float* o_s, const float* lse_s, void* o_out,
                              long long n_rows, int d, cudaStream_t stream);
cudaError_t launch_ring_gather(const void* src, void* dst, int Z, int L, int d, int N, bool causal, int sched,
                               cudaStream_t stream);
// Ring-mode backward (ring_step.cu): gather of one fp32 per row (lse) into
// chunk order, and the scatter of an fp32 gradient accumulator in chunk
// order (plain, or the tiled dQ layout) back to sequence order as
// bf16(scale * acc).
cudaError_t launch_ring_gather_rows(const float* src, float* dst, int Z, int L, int N, bool causal, int sched,
                                    cudaStream_t stream);
cudaError_t launch_ring_scatter_grad(const float* acc, void* g, float scale, bool tiled, int Z, int L, int d, int N,
                                     bool causal, int sched, cudaStream_t stream);

// Ulysses / USP (ulysses.cu): the all-to-all between the N = U R sequence
// shards [N][B][H][L/N][row] and the U head groups [U][B][H/U][L][row]
// (to_heads) or back; row_bytes 128 or 256 (d = 64 or 128 values of bf16)
// or 4 (one fp32).  causal with R > 1: the shards follow the ring's fold.
cudaError_t launch_ulysses_a2a(const void* src, void* dst, int row_bytes, int B, int H, int U, int R, int L,
                               bool causal, bool to_heads, cudaStream_t stream);
// Token-major [B][L][H][row] <-> head-major [B][H][L][row]; row_bytes a
// multiple of 16 (ulysses.cu).
cudaError_t launch_tokens_heads(const void* src, void* dst, int row_bytes, int B, int H, int L, bool to_heads,
                                cudaStream_t stream);
cudaError_t launch_ring_scatter(const float* acc, const float* lse_acc, void* o, float* lse, int Z, int L, int d,
                                int N, bool causal, int sched, cudaStream_t stream);

// Dynamic shared memory each kernel needs (bytes), for the C ABI's checks.
size_t fwd_smem_bytes(int d);
size_t bwd_smem_bytes(int d);

}  // namespace ra
