/*
 * ring_attn.h -- C ABI of the GB300 (sm_103a) blockwise Ring Self-Attention
 * library.
 *
 * The operation (web page "Large-scale distributed AI model training series:
 * sequence parallelism", section 2.3 Ring Self-Attention and section 6.2 Ring
 * Attention): self-attention softmax(Q K^T / sqrt(d)) V, computed block by
 * block.  The sequence of length L is cut into n_chunks chunks; the queries of
 * each chunk visit the key/value chunks in ring order, starting with their own
 * chunk and then (r - 1), (r - 2), ... mod n_chunks, and the partial results
 * are merged with a running maximum and log-sum-exp (the online-softmax
 * correction of section 6.2).  With causal = 1 (decoder), position i sees
 * keys j <= i and every rank r owns the folded pair of sub-chunks
 * {r, 2 n_chunks - 1 - r} of length L / (2 n_chunks) (the fold of section 8.2,
 * USP), which gives every rank the same amount of work.  On one GPU the ring
 * is emulated: all ranks' blocks run in one launch, each in its ring order.
 * The result is exact attention; chunking only changes the order of fp32
 * additions.
 *
 * Tensors (all contiguous, row-major, device memory, caller-owned):
 *   q, o, dO, dq : bf16 [B][Hq][L][d]
 *   k, v, dk, dv : bf16 [B][Hkv][L][d]
 *   lse          : fp32 [B][Hq][L], natural log of sum_j exp(q_i.k_j/sqrt(d))
 * Grouped-query attention: query head h uses kv head h / (Hq / Hkv).
 * Scale is fixed at 1/sqrt(d).  Supported: d in {64, 128}; Hq % Hkv == 0;
 * L % n_chunks == 0 (encoder) or L % (2 n_chunks) == 0 (causal); every base
 * pointer 16-byte aligned; B * Hq and B * Hkv below 65536.
 *
 * Errors: argument errors are returned before anything is launched.  Calls
 * are asynchronous on `stream`; a kernel that gives up on a bounded wait
 * records a device status, read (and cleared) by ring_attn_device_status().
 * Thread safety: calls from several host threads are serialised internally.
 */
#ifndef RING_ATTN_H
#define RING_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  RING_ATTN_OK = 0,
  RING_ATTN_ERR_NULL = -1,          /* a required pointer is NULL */
  RING_ATTN_ERR_SHAPE = -2,         /* negative size, Hq % Hkv != 0, bad chunking */
  RING_ATTN_ERR_UNSUPPORTED = -3,   /* d not in {64,128}, misaligned pointer, too many heads */
  RING_ATTN_ERR_WORKSPACE = -4,     /* backward workspace missing or too small */
  RING_ATTN_ERR_CUDA = -5,          /* a CUDA runtime/driver call failed */
  RING_ATTN_ERR_DEVICE_TIMEOUT = -6 /* a kernel gave up on a bounded wait */
};

/*
 * Forward pass.  Writes o (bf16) and lse (fp32).
 * Inputs q, k, v are read only.  n_chunks >= 1 is the ring size N.
 * Returns RING_ATTN_OK or a negative error code.  B == 0 or L == 0 is a
 * no-op returning RING_ATTN_OK.
 */
int ring_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                  int L, int d, int n_chunks, int causal, cudaStream_t stream);

/*
 * Bytes of device workspace ring_attn_bwd needs for this shape (fp32 dq
 * accumulator plus per-row statistics, and fp32 dk/dv accumulators when
 * Hq > Hkv), or 0 for an invalid shape.
 */
size_t ring_attn_bwd_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal);

/*
 * Backward pass of l = sum(dO * o): writes dq, dk, dv (bf16).  o and lse
 * must be the forward outputs for the same q, k, v.  The probabilities are
 * recomputed from lse (no score matrix is stored).  `workspace` is caller
 * owned device memory of at least ring_attn_bwd_workspace_size() bytes,
 * 256-byte aligned; its contents on entry do not matter.
 */
int ring_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Size in bytes of the static device array ring_attn_bwd_noalloc works in
 * (64 MiB per GPU that loads the library, held until the process exits).
 */
#define RING_ATTN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * ring_attn_bwd without any device allocation.  The pages describe no such
 * call; it serves callers that cannot call cudaMalloc: code whose device
 * memory is owned by another allocator (a framework's caching pool, a fixed
 * memory budget) and latency-critical code that cannot accept the device
 * synchronisation cudaMalloc/cudaFree may cause.  Arguments and results are
 * those of ring_attn_bwd minus the workspace: the statistics, the fp32
 * accumulators and the launch plan live in a static device array of
 * RING_ATTN_NOALLOC_SCRATCH_BYTES.  A problem whose workspace
 * (ring_attn_bwd_workspace_size) plus plan does not fit is rejected with
 * RING_ATTN_ERR_WORKSPACE before anything is launched.  The first call on
 * each device looks up the array's device address (cudaGetSymbolAddress),
 * and the first call for each (L, n_chunks, causal) builds its launch plan
 * in page-locked host memory (cudaMallocHost, held until the process
 * exits): make those first calls outside stream capture.  Later calls may
 * be captured into a CUDA graph and replayed; each call (and each replay)
 * copies the plan in and runs the pre-pass, main and conversion kernels on
 * `stream`.  Its launches are counted by ring_attn_profile_read like those
 * of ring_attn_bwd.  All calls share the one array and it keeps the last
 * call's contents (each call rewrites what it needs): calls whose work may
 * overlap on the GPU race and must be ordered by the caller, e.g. by
 * issuing them on one stream.
 */
int ring_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L, int d,
                          int n_chunks, int causal, cudaStream_t stream);

/* ---------------------------------------------------------------------
 * Ring mode: the ring run step by step, the way each rank of a multi-GPU
 * ring runs it ("Large-scale distributed AI model training series: sequence
 * parallelism", section 2.3 Ring Self-Attention: each device keeps its
 * query chunk while the key/value blocks travel round the ring; section 6.2
 * Ring Attention: each step's partial result is merged into the running one
 * with the online-softmax correction).  Rank r holds chunk r of the
 * sequence, in chunk order, C = L / n_chunks rows; `schedule` picks the
 * chunk map and the order of the blocks:
 *   RING_ATTN_SCHEDULE_FOLD (0): rows [rC, (r+1)C) when causal == 0;
 *     sub-chunk r followed by sub-chunk 2N-1-r, each L/(2N) rows, when
 *     causal != 0 (the fold that balances causal work, section 8.2).
 *     N ring steps: at step s rank r holds the keys of rank (r - s) mod N.
 *   RING_ATTN_SCHEDULE_STRIPED (1): positions r, r+N, r+2N, ... (striped
 *     attention, the causal schedule variant the pages compare with the
 *     fold; L % N == 0 suffices); N ring steps.
 *   RING_ATTN_SCHEDULE_CONTIGUOUS (2): causal only, rows [rC, (r+1)C); N
 *     ring steps -- the unbalanced ring (rank r has work only at steps
 *     s <= r) of section 7.2.
 *   RING_ATTN_SCHEDULE_DISTFLASH (3): causal only, rows [rC, (r+1)C);
 *     DistFlashAttention's balanced schedule (section 7.2: a worker that
 *     would wait takes over a later worker's block), N/2 + 1 launches:
 *     at launch t worker w >= t runs block (query chunk w, keys of chunk
 *     w - t) and worker w < t block (N - t + w, w), the block of ring step
 *     N - t, unless t == N - t (then it is idle); see
 *     ring_attn_schedule_pair.
 * Chunks must be whole 128-row tiles -- C, or L/(2N) for the causal fold,
 * a multiple of 128 -- else RING_ATTN_ERR_UNSUPPORTED.  Pointers are device
 * pointers, 16-byte aligned and owned by the caller; calls are asynchronous
 * on `stream`; argument errors return before anything is launched.
 * ------------------------------------------------------------------- */
enum {
  RING_ATTN_SCHEDULE_FOLD = 0,
  RING_ATTN_SCHEDULE_STRIPED = 1,
  RING_ATTN_SCHEDULE_CONTIGUOUS = 2,
  RING_ATTN_SCHEDULE_DISTFLASH = 3
};

/* Host-only: launches of one pass of the schedule (N, or N/2 + 1 for
 * RING_ATTN_SCHEDULE_DISTFLASH), or a negative code. */
int ring_attn_schedule_launches(int n_chunks, int schedule);

/* Host-only: the block worker `worker` runs at launch `launch` of the
 * schedule: *q_chunk (whose queries) and *kv_chunk (whose keys/values).
 * Returns 1 if the worker has a block, 0 if it is idle at that launch, or a
 * negative code. */
int ring_attn_schedule_pair(int n_chunks, int schedule, int launch, int worker, int* q_chunk, int* kv_chunk);

/*
 * One block: the attention of rank `rank`'s query chunk against the
 * key/value chunk of rank `src` (the block rank holds at ring step
 * (rank - src) mod n_chunks), with the causal mask taken on the rows'
 * sequence positions under the schedule's chunk map (the two contiguous
 * schedules share one).
 *   q_chunk           bf16 [B][Hq][C][d]    rank's query rows, chunk order
 *   k_chunk, v_chunk  bf16 [B][Hkv][C][d]   src's key/value rows, chunk order
 *   o_s               fp32 [B][Hq][C][d]    out: the partial result, normalised
 *                                           over src's keys alone
 *   lse_s             fp32 [B][Hq][C]       out: its log-sum-exp (natural log);
 *                                           a row that sees none of src's keys
 *                                           gets lse_s = -inf and o_s = 0
 */
int ring_attn_fwd_step(const void* q_chunk, const void* k_chunk, const void* v_chunk, float* o_s, float* lse_s,
                       int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal, int schedule, int rank, int src,
                       cudaStream_t stream);

/*
 * The same block, accumulated into a running result instead of returned as
 * a partial one: (o_run, lse_run) -- fp32 [B][Hq][C][d] and [B][Hq][C],
 * rank's rows in chunk order -- hold the result of the blocks merged so far
 * and are overwritten with that result merged with this block's (what
 * ring_attn_fwd_step followed by ring_attn_merge gives, without writing the
 * partial result or reading it back).  The kernel continues its online
 * softmax from the running state.  lse_run = -inf (and o_run = 0) is the
 * empty result; rows that see none of src's keys keep theirs.  The order in
 * which a rank's blocks are accumulated changes only the rounding.
 */
int ring_attn_fwd_step_accumulate(const void* q_chunk, const void* k_chunk, const void* v_chunk, float* o_run,
                                  float* lse_run, int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                                  int schedule, int rank, int src, cudaStream_t stream);

/*
 * Merge of two partial results of the same n_rows rows of width d (64 or
 * 128), in place: lse <- log(e^lse + e^lse_s), o <- e^(lse_old - lse) o +
 * e^(lse_s - lse) o_s; a side with lse = -inf contributes nothing.  o, o_s
 * fp32 [n_rows][d], lse, lse_s fp32 [n_rows].  If o_out is not NULL, bf16(o)
 * is written there as well ([n_rows][d]), e.g. after the last step.
 */
int ring_attn_merge(float* o, float* lse, const float* o_s, const float* lse_s, long long n_rows, int d,
                    void* o_out, cudaStream_t stream);

/* Workspace bytes ring_attn_ring_fwd needs for this shape, or 0 if invalid. */
size_t ring_attn_ring_fwd_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                                         int schedule);

/*
 * The whole ring on one GPU, every worker of it, the ring-mode way: q, k, v
 * (sequence order, as for ring_attn_fwd) are gathered into chunk order; at
 * each launch of the schedule one kernel launch runs every worker's block
 * (ring steps: worker r against chunk (r - s) mod n_chunks), each
 * accumulated into the running fp32 result of its query chunk as
 * ring_attn_fwd_step_accumulate does (DistFlashAttention: two kernel
 * launches per schedule launch, the workers' own chunks, then the chunks the
 * idle workers took over); the result is scattered back to sequence order
 * into o (bf16) and lse (fp32), as ring_attn_fwd writes them.  `workspace`
 * (caller-owned device memory of ring_attn_ring_fwd_workspace_size() bytes,
 * 256-byte aligned) holds the gathered chunks and the running result.
 */
int ring_attn_ring_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                       int L, int d, int n_chunks, int causal, int schedule, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* ---------------------------------------------------------------------
 * Ulysses sequence parallelism on one GPU ("Large-scale distributed AI
 * model training series: sequence parallelism", section 5 DeepSpeed-
 * Ulysses): the input is sharded along the sequence, rank r holding tokens
 * [rC, (r+1)C) of every head (C = L / n_ranks); an all-to-all gives every
 * rank all L tokens of H / n_ranks heads, attention runs on each head group
 * independently, and an all-to-all brings the result back to the sequence
 * shards.  Every tensor is passed as the n_ranks shards stacked, rank-major:
 *   q, o, dO, dq  bf16 [n_ranks][B][Hq][C][d]     lse fp32 [n_ranks][B][Hq][C]
 *   k, v, dk, dv  bf16 [n_ranks][B][Hkv][C][d]
 * (rank r's shard is the r-th [B][H][C][d] block).  The head groups must
 * split evenly: Hq, Hkv and L multiples of n_ranks, else
 * RING_ATTN_ERR_SHAPE.  The attention itself is the fused kernel of
 * ring_attn_fwd / ring_attn_bwd on the head shards (batch n_ranks * B),
 * with the whole sequence in view, so the chunk schedule does not apply.
 * `workspace`: caller-owned device memory, 256-byte aligned, of
 * ring_attn_ulysses_workspace_size() bytes (enough for the backward; the
 * forward uses its head-shard part only).
 * ------------------------------------------------------------------- */
size_t ring_attn_ulysses_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_ranks, int causal);

int ring_attn_ulysses_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                          int L, int d, int n_ranks, int causal, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

int ring_attn_ulysses_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L, int d,
                          int n_ranks, int causal, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * USP (same page, section 8.2): Ulysses within groups of U ranks and a ring
 * across R groups, over N = U * R sequence shards; rank n = r * U + u (ring
 * group r, Ulysses rank u) holds L / N tokens of every head, tensors
 * stacked rank-major as for Ulysses ([N][B][H][L/N][d], lse [N][B][Hq][L/N]).
 * The all-to-all within a group gives each rank H/U heads of its group's
 * tokens; attention per head group is a ring over the R groups.  Token i of
 * rank (r, u): encoder, or R == 1, sequence position n L/N + i; causal with
 * R > 1, the ring's fold: group r owns sub-chunks r and 2R-1-r of
 * c = L/(2R) tokens, each split into U pieces of c/U, rank u taking piece u
 * of both (i < c/U: r c + u c/U + i; else (2R-1-r) c + u c/U + i - c/U).
 * Requires Hq % U == 0, Hkv % U == 0, L % N == 0 (causal, R > 1: L % 2N ==
 * 0) and the fused kernels' domain for the head groups.  On one GPU both
 * all-to-alls are permutations (HBM copies) around one launch of the fused
 * kernels with batch U * B, H/U heads and the ring over R chunks.
 * ring_attn_ulysses_* are the case R == 1.
 */
size_t ring_attn_usp_workspace_size(int B, int Hq, int Hkv, int L, int d, int ulysses_degree, int ring_degree,
                                    int causal);

int ring_attn_usp_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int L,
                      int d, int ulysses_degree, int ring_degree, int causal, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

int ring_attn_usp_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                      void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L, int d, int ulysses_degree,
                      int ring_degree, int causal, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes ring_attn_ring_bwd needs for this shape, or 0 if invalid. */
size_t ring_attn_ring_bwd_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                                         int schedule);

/*
 * The backward of ring_attn_ring_fwd, the ring-mode way (the same results
 * as ring_attn_bwd; o and lse from either forward): q, k, v, o, dO, lse are
 * gathered into chunk order; the statistics of every rank's rows are formed
 * once; at each launch of the schedule one kernel launch runs, for every
 * worker, the tiles of its block's key/value chunk against the block's
 * query chunk, adding into that query chunk's fp32 dQ accumulator and
 * into the key/value chunk's fp32 dK, dV accumulators (the gradients that in a
 * multi-GPU ring travel with K and V back to their owner); the gradients
 * are scattered back to sequence order as bf16.  `workspace`: caller-owned
 * device memory of ring_attn_ring_bwd_workspace_size() bytes, 256-byte
 * aligned.
 */
int ring_attn_ring_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                       void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                       int schedule, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------
 * One rank's share of the ring-mode backward, for a ring whose ranks run
 * on different GPUs ("Large-scale distributed AI model training series:
 * sequence parallelism", section 6.2 Ring Attention: the blocks are
 * recomputed in the backward pass; the key/value gradients travel round the
 * ring with their key/value block and end at its owner).  Tensors are the
 * rank's chunks in chunk order, as for ring_attn_fwd_step; C = L/n_chunks.
 *   begin  the rank's statistics from its forward outputs (o_chunk, lse_chunk)
 *          and dO_chunk; zeroes its fp32 dQ accumulator (both in `workspace`,
 *          ring_attn_bwd_rank_workspace_size() bytes, 256-byte aligned)
 *   step   the block (rank's queries, src's keys): adds its dQ contribution
 *          to the workspace's accumulator and its dK, dV contributions to
 *          dk_acc, dv_acc -- fp32 [B][Hkv][C][d], plain row-major, the
 *          accumulators travelling with src's key/value chunk (zeroed by
 *          src before the ring starts; src's own block is the first step)
 *   end    dq_chunk = bf16(dQ / sqrt(d)) [B][Hq][C][d]
 * Once dk_acc, dv_acc are back at their owner, ring_attn_grad_to_bf16 gives
 * dk = bf16(dk_acc / sqrt(d)) and dv = bf16(dv_acc).  The schedule's chunk
 * map decides the causal mask (RING_ATTN_SCHEDULE_DISTFLASH blocks are the
 * contiguous ring's).  Steps of one rank must not overlap on the GPU with
 * each other (they add into the same dQ accumulator) unless ordered by the
 * caller; the workspace must not be shared between ranks.
 * ------------------------------------------------------------------- */
size_t ring_attn_bwd_rank_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                                         int schedule);

int ring_attn_bwd_rank_begin(const void* o_chunk, const void* dO_chunk, const float* lse_chunk, int B, int Hq,
                             int Hkv, int L, int d, int n_chunks, int causal, int schedule, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

int ring_attn_bwd_rank_step(const void* q_chunk, const void* k_chunk, const void* v_chunk, const void* dO_chunk,
                            float* dk_acc, float* dv_acc, int B, int Hq, int Hkv, int L, int d, int n_chunks,
                            int causal, int schedule, int rank, int src, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

int ring_attn_bwd_rank_end(void* dq_chunk, int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                           int schedule, const void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* out = bf16(scale * acc) elementwise for n_elems fp32 values (a multiple
 * of 128); out [n_elems] bf16. */
int ring_attn_grad_to_bf16(const float* acc, void* out, long long n_elems, float scale, cudaStream_t stream);

/* Byte offset, inside a ring_attn_bwd_rank_* workspace of this shape, of
 * the rank's fp32 dQ accumulator: B*Hq*C*d floats in the library's own
 * tiled order, unscaled (0 if the shape is rejected, the offset is never 0
 * otherwise).  With DistFlashAttention's schedule across GPUs (SP series
 * section 7.2: an idle worker computes a block of a later worker's query
 * chunk on its own keys), the helper runs that block through a workspace
 * begun with the owner's o, dO, lse, then sends this accumulator to the
 * owner, who adds it into its own with ring_attn_add_f32 before
 * ring_attn_bwd_rank_end.  Both workspaces have the same shape, hence the
 * same order. */
size_t ring_attn_bwd_rank_dq_offset(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal,
                                    int schedule);

/* dst[i] += src[i] for n_elems fp32 values (a multiple of 4; both 16-byte
 * aligned device pointers; the caller owns both): partial gradients that
 * arrive from another rank.  Errors: SHAPE, NULL, UNSUPPORTED (alignment),
 * CUDA. */
int ring_attn_add_f32(float* dst, const float* src, long long n_elems, cudaStream_t stream);

/* Static description of a status code. */
const char* ring_attn_strerror(int status);

/*
 * Synchronises `stream`, then returns and clears the device status of the
 * current device: RING_ATTN_OK, or RING_ATTN_ERR_DEVICE_TIMEOUT if a kernel
 * aborted a bounded wait since the last call (the site code is written to
 * *site if site is not NULL), or RING_ATTN_ERR_CUDA.
 */
int ring_attn_device_status(cudaStream_t stream, int* site);

/*
 * Failure-detection self-test.  Launches one small kernel whose bounded
 * wait (the same wait the attention kernels use on their mbarriers) can
 * never be satisfied: after timeout_us microseconds it gives up, records the
 * self-test site code (0x301) in the device status word and returns, so the
 * next ring_attn_device_status() reports RING_ATTN_ERR_DEVICE_TIMEOUT and the
 * context stays usable.  timeout_us must be in (0, 10^7].
 */
int ring_attn_selftest_bounded_wait(unsigned timeout_us, cudaStream_t stream);

/* ---------------------------------------------------------------------
 * Blockwise feed-forward (web page "Large-scale distributed AI model
 * training series: sequence parallelism", section 4.2 Blockwise Parallel
 * Transformer: after a query block's attention, the FFN and the residual
 * connection are computed for that block; section 8: the FFN is two linear
 * layers around an up-projection to F = 4 D in the GPT-style model).  For
 * every row x_m of x (a token's hidden state):
 *   y_m = x_m + W2 gelu(W1 x_m + b1) + b2,   gelu(t) = t Phi(t)
 * (the exact GELU, Phi the standard normal CDF, evaluated with relative
 * accuracy in the tail t << 0).
 * The rows are processed in blocks of block_rows rows; only one block's
 * hidden activation (block_rows x F) exists at a time, in the workspace:
 * on return it holds the last block's, bf16 [rows of that block][F].
 *   x, y : bf16 [M][D]     (y may be x: the update is then in place)
 *   w1   : bf16 [F][D]     (W1, output-major: row f holds the weights of
 *                           hidden unit f, the layout of a linear layer's
 *                           weight [out_features][in_features])
 *   b1   : fp32 [F]
 *   w2   : bf16 [D][F]     (W2, output-major)
 *   b2   : fp32 [D]
 * Products accumulate in fp32; the hidden activation is rounded to bf16
 * before the second layer (it is the second GEMM's operand).
 * Supported: D % 256 == 0 and F % 256 == 0 (both >= 256), block_rows a
 * positive multiple of 128, any M >= 0 (M == 0 is a no-op); every pointer
 * 16-byte aligned (RING_ATTN_ERR_UNSUPPORTED otherwise), below 2^31 rows.
 * ------------------------------------------------------------------- */

/* Bytes of workspace ring_attn_ffn_fwd needs (the bf16 hidden block), or 0
 * for an unsupported shape. */
size_t ring_attn_ffn_workspace_size(int D, int F, int block_rows);

/* Forward of the blockwise FFN: two persistent tensor-core GEMM launches per
 * row block (first layer with bias + GELU, second with bias + residual).
 * workspace: device, 256-byte aligned, >= ring_attn_ffn_workspace_size(). */
int ring_attn_ffn_fwd(const void* x, const void* w1, const float* b1, const void* w2, const float* b2, void* y,
                      long long M, int D, int F, int block_rows, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/* Backward of the blockwise FFN: gradients of sum(dy * y) for y as in
 * ring_attn_ffn_fwd (b2 does not enter), block by block with the block's
 * hidden activation recomputed (the BPT section's recomputation):
 *   dx  = dy + (dy W2 * gelu'(a)) W1          bf16 [M][D]
 *   dw1 = sum over rows of da^T x             fp32 [F][D]  (W1's layout)
 *   db1 = sum over rows of da                 fp32 [F]
 *   dw2 = sum over rows of dy^T h             fp32 [D][F]  (W2's layout)
 *   db2 = sum over rows of dy                 fp32 [D]
 * with a = x W1^T + b1, h = gelu(a), da = (dy W2) * gelu'(a).  The four
 * gradient sums are overwritten (started from zero), accumulated in fp32
 * over the blocks.  Per block: five tensor-core GEMM launches (the first
 * layer again with GELU and its derivative, dh * gelu', dx, dw2, dw1), the
 * weight gradients' operands transposed by a copy kernel.  Same domain and
 * errors as ring_attn_ffn_fwd; workspace >= ring_attn_ffn_bwd_workspace_size.
 */
size_t ring_attn_ffn_bwd_workspace_size(int D, int F, int block_rows);

int ring_attn_ffn_bwd(const void* x, const void* w1, const float* b1, const void* w2, const void* dy, void* dx,
                      float* dw1, float* db1, float* dw2, float* db2, long long M, int D, int F, int block_rows,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------
 * Blockwise transformer forward (BPT; same page, section 4.2: the outer
 * loop runs over query blocks, and for each block the attention over every
 * key/value block, with the online-softmax correction, is followed by the
 * feed-forward network and the residual connection of that block).  For
 * each block of block_rows query rows, in order:
 *   a = attention of those rows (all batches and heads; the ring order and
 *       chunk map of ring_attn_fwd), written token-major
 *   y = a + W2 gelu(W1 a + b1) + b2 on the block's token rows, a row being
 *       the Hq * d outputs of one token (hidden size D = Hq * d)
 * so only one block's FFN hidden activation exists at a time.
 *   q, k, v  : as ring_attn_fwd
 *   a_tok, y : bf16 [B][L][Hq * d] (token-major; a_tok keeps the attention
 *              output, the FFN's residual input)
 *   lse      : fp32 [B][Hq][L], as ring_attn_fwd
 *   w1 [F][D], b1 [F], w2 [D][F], b2 [D]: as ring_attn_ffn_fwd
 * Supported: ring_attn_fwd's domain, Hq * d % 256 == 0, F % 256 == 0,
 * block_rows a positive multiple of 256, B * L below 2^31.
 * ------------------------------------------------------------------- */

/* Bytes of workspace ring_attn_bpt_fwd needs (one block's bf16 hidden
 * activation), or 0 for an unsupported shape. */
size_t ring_attn_bpt_workspace_size(int Hq, int d, int F, int block_rows);

/* Per row block: one launch of the fused attention forward (that block's
 * work items), then the two GEMM launches of the FFN per batch. */
int ring_attn_bpt_fwd(const void* q, const void* k, const void* v, void* a_tok, float* lse, const void* w1,
                      const float* b1, const void* w2, const float* b2, void* y, int B, int Hq, int Hkv, int L, int d,
                      int n_chunks, int causal, int F, int block_rows, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/* Backward of the blockwise transformer forward for the loss sum(dy * y):
 * the FFN backward over the token rows, block by block with each block's
 * hidden activation recomputed (ring_attn_ffn_bwd: fp32 dw1 [F][D], db1
 * [F], dw2 [D][F], db2 [D], overwritten), which gives the gradient at the
 * attention output, dy plus the FFN's input gradient; then the fused
 * attention backward (ring_attn_bwd) on the attention output and that
 * gradient, permuted to head-major: dq, dk, dv bf16 as ring_attn_bwd.
 * a_tok and lse are ring_attn_bpt_fwd's outputs; dy bf16 [B][L][Hq * d].
 * Same domain as ring_attn_bpt_fwd; workspace >=
 * ring_attn_bpt_bwd_workspace_size(), 256-byte aligned. */
size_t ring_attn_bpt_bwd_workspace_size(int B, int Hq, int Hkv, int L, int d, int n_chunks, int causal, int F,
                                        int block_rows);

int ring_attn_bpt_bwd(const void* q, const void* k, const void* v, const void* a_tok, const float* lse, const void* w1,
                      const float* b1, const void* w2, const void* dy, void* dq, void* dk, void* dv, float* dw1,
                      float* db1, float* dw2, float* db2, int B, int Hq, int Hkv, int L, int d, int n_chunks,
                      int causal, int F, int block_rows, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/* ---------------------------------------------------------------------
 * Per-kernel timing, for measurement.  While enabled, every kernel launch
 * of the library is bracketed by two CUDA events recorded on the launch
 * stream.  ring_attn_profile_read() waits for those events and returns,
 * per kernel kind, the summed milliseconds and the number of launches since
 * the last read (arrays of RING_ATTN_N_KERNELS entries), then forgets them.
 * ------------------------------------------------------------------- */
enum {
  RING_ATTN_KERNEL_FWD = 0,      /* forward attention kernel */
  RING_ATTN_KERNEL_BWD_PRE = 1,  /* backward pre-pass: D, log2 lse, zero dq accumulator */
  RING_ATTN_KERNEL_BWD_MAIN = 2, /* fused backward kernel */
  RING_ATTN_KERNEL_BWD_POST = 3, /* dq accumulator -> bf16 */
  RING_ATTN_KERNEL_RING_STEP = 4,  /* ring mode: one step of attention (every rank or one) */
  RING_ATTN_KERNEL_RING_MERGE = 5, /* ring mode: log-sum-exp merge */
  RING_ATTN_KERNEL_RING_IO = 6,    /* ring mode: gather into / scatter out of chunk order, partial adds */
  RING_ATTN_KERNEL_ULYSSES_A2A = 7, /* Ulysses: all-to-all between sequence and head shards */
  RING_ATTN_KERNEL_FFN_GEMM = 8,    /* blockwise feed-forward: one of its two GEMMs */
  RING_ATTN_N_KERNELS = 9
};
int ring_attn_profile_enable(int on);
int ring_attn_profile_read(double* ms, long long* launches);

/* Frees cached launch plans (device copies of schedules). Optional. */
void ring_attn_release(void);

/* ---------------------------------------------------------------------
 * Host-only scheduling queries (no GPU needed).  They expose the chunk map
 * and the ring visiting order the kernels follow, at the granularity of the
 * kernels' 128-row tiles.
 * ------------------------------------------------------------------- */

/* Rank (0..n_chunks-1) that owns sequence position pos, or a negative code. */
int ring_attn_owner_rank(int L, int n_chunks, int causal, int pos);

/*
 * Forward plan.  The queries are processed in blocks of two 128-row tiles
 * (256 rows); block u covers rows [256 u, 256 u + 256).  For each block the
 * plan lists the 128-row key/value tiles it visits, in ring order, as
 * half-open ranges [begin, end) of tile indices.
 *   n_blocks, n_ranges : out, sizes (always written if non-NULL)
 *   block_order        : [n_blocks] launch order (longest work first)
 *   range_offsets      : [n_blocks + 1] offsets into ranges
 *   ranges             : [2 * n_ranges] (begin, end) pairs
 * Pass NULL arrays to query sizes only.  Returns RING_ATTN_OK or an error.
 */
int ring_attn_fwd_plan(int L, int n_chunks, int causal, int* n_blocks, int* n_ranges, int32_t* block_order,
                       int32_t* range_offsets, int32_t* ranges);

/*
 * Backward plan: for each 128-row key/value tile t, the 128-row query tiles
 * that see it, in the order the key/value block meets them travelling round
 * the ring (its own rank first, then r + 1, r + 2, ... mod n_chunks).
 * Same array conventions as ring_attn_fwd_plan, with n_blocks = key tiles.
 */
int ring_attn_bwd_plan(int L, int n_chunks, int causal, int* n_blocks, int* n_ranges, int32_t* block_order,
                       int32_t* range_offsets, int32_t* ranges);

/*
 * Ring-mode plan of worker `rank` at launch `step` of the schedule (its
 * block: ring_attn_schedule_pair): for each 256-row block of the block's
 * query chunk (chunk-order rows), the 128-row tiles of its key/value chunk
 * (chunk-order indices, ascending) holding a key some row of the block may
 * see; a block may list none (and an idle worker lists none).  Same array
 * conventions as ring_attn_fwd_plan, with n_blocks = blocks of one chunk.
 * Chunks must be whole 128-row tiles (see ring mode above).
 */
int ring_attn_step_plan(int L, int n_chunks, int causal, int schedule, int step, int rank, int* n_blocks,
                        int* n_ranges, int32_t* block_order, int32_t* range_offsets, int32_t* ranges);

#ifdef __cplusplus
}
#endif

#endif /* RING_ATTN_H */
