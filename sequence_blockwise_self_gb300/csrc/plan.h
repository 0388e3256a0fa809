// plan.h -- host-side chunk scheduler: chunk map, ring visiting order and
// launch order of the attention kernels' work items.
//
// Citations name the web page "Large-scale distributed AI model training
// series: sequence parallelism" and its sections:
//   section 2.3  Ring Self-Attention: L tokens over N devices, L/N each; the
//                key/value blocks move round a ring, N-1 transfers and N
//                block computations per device.
//   section 6.2  Ring Attention: K and V travel together; one ring suffices
//                once the per-step results are merged (online softmax).
//   section 7.2  DistFlashAttention: a causal model leaves the ring with
//                contiguous chunks unbalanced; a worker that would wait
//                takes over blocks of a later worker.
//   section 8.2  USP: splitting the sequence by folding it gives every
//                device about the same work.
#pragma once
#include <cstdint>
#include <vector>

#ifdef __CUDACC__
#define RA_HOST_DEVICE __host__ __device__
#else
#define RA_HOST_DEVICE
#endif

namespace ra {

constexpr int kTileRows = 128;      // rows per query / key-value tile
constexpr int kQBlockRows = 256;    // forward work item: two query tiles

// Rank owning sequence position pos.  Encoder: chunk pos / (L/N).  Causal:
// the folded pair of sub-chunks {r, 2N-1-r}, each of length L/(2N).
inline int owner_rank(int L, int N, bool causal, int pos) {
  if (!causal) return pos / (L / N);
  const int sub = pos / (L / (2 * N));
  return sub < N ? sub : 2 * N - 1 - sub;
}

// True if the chunking is valid for this length.
inline bool chunking_ok(int L, int N, bool causal) {
  if (N < 1 || L < 1) return false;
  const long parts = causal ? 2L * N : N;
  return parts <= L && L % parts == 0;
}

struct Plan {
  int n_blocks = 0;                  // work items per (batch, head)
  std::vector<int32_t> order;        // [n_blocks] launch order, longest first
  std::vector<int32_t> offsets;      // [n_blocks + 1] into ranges
  std::vector<int32_t> ranges;       // (begin, end) tile-index pairs
  std::vector<int64_t> work;         // [n_blocks] tile pairs per item
};

// Forward: item u = query rows [256u, 256u+256).  Lists the key/value tiles
// it visits in the ring order of the rank owning its first row: step s
// brings the block of rank (r - s) mod N; tiles of one step ascending.
Plan build_fwd_plan(int L, int N, bool causal);

// Backward: item t = key/value tile t.  Lists the query tiles that see it in
// the order the block meets them going round the ring: its own rank first,
// then ranks r + 1, r + 2, ... mod N.
Plan build_bwd_plan(int L, int N, bool causal);

// ----------------------------------------------------------- ring step mode
// The ring run explicitly, as each worker of a multi-GPU ring would: worker
// r holds its chunk of C = L/N rows in chunk order, and each launch of the
// schedule gives it one block, a query chunk against a key/value chunk.
// Schedules (the `schedule` argument of the C ABI's ring mode):
//   kSchedFold     encoder: rows [rC, (r+1)C); causal: sub-chunk r, then
//                  sub-chunk 2N-1-r, each L/(2N) rows (section 8.2).  N ring
//                  steps: at step s worker r holds the keys of (r - s) mod N.
//   kSchedStriped  positions r, r+N, r+2N, ...; N ring steps.
//   kSchedContig   causal, rows [rC, (r+1)C); N ring steps (the unbalanced
//                  ring: worker r has work only at steps s <= r).
//   kSchedDfa      causal, rows [rC, (r+1)C); N/2 + 1 launches of
//                  DistFlashAttention's balanced schedule (schedule_pair).
enum : int { kSchedFold = 0, kSchedStriped = 1, kSchedContig = 2, kSchedDfa = 3 };

inline bool schedule_ok(int sched, bool causal) {
  return sched == kSchedFold || sched == kSchedStriped || (causal && (sched == kSchedContig || sched == kSchedDfa));
}

// Launches of one pass over the ring.
inline int schedule_launches(int N, int sched) { return sched == kSchedDfa ? N / 2 + 1 : N; }

// The block of worker w at launch t: its query chunk and key/value chunk.
// Ring schedules: (w, (w - t) mod N).  DistFlashAttention: worker w >= t
// takes (w, w - t); a worker w < t, idle in the plain ring, takes the block
// (N - t + w, w) of ring step N - t, which is then never run on its own;
// when N is even, launch N/2 is its own partner step and its workers
// w < N/2 stay idle (returns false).
RA_HOST_DEVICE inline bool schedule_pair(int N, int sched, int t, int w, int* q_chunk, int* kv_chunk) {
  if (sched != kSchedDfa) {
    *q_chunk = w;
    *kv_chunk = ((w - t) % N + N) % N;
    return true;
  }
  *q_chunk = w;
  *kv_chunk = w;
  if (w >= t) {
    *kv_chunk = w - t;
    return true;
  }
  if (t < N - t) {
    *q_chunk = N - t + w;
    return true;
  }
  return false;
}

// Chunks must be whole 128-row tiles: C (encoder, striped, contiguous) or
// the sub-chunk length (causal fold) a multiple of 128.
inline bool step_chunking_ok(int L, int N, bool causal, int sched) {
  if (!schedule_ok(sched, causal)) return false;
  if (sched != kSchedFold) return N >= 1 && L >= N && L % N == 0 && (L / N) % kTileRows == 0;
  if (!chunking_ok(L, N, causal)) return false;
  return (causal ? L / (2 * N) : L / N) % kTileRows == 0;
}

// Sequence position of row `local` of rank `rank`'s chunk.
RA_HOST_DEVICE inline int chunk_pos(int L, int N, bool causal, int sched, int rank, int local) {
  if (sched == kSchedStriped) return rank + N * local;
  if (!causal || sched != kSchedFold) return rank * (L / N) + local;
  const int c = L / (2 * N);
  return local < c ? rank * c + local : (2 * N - 1 - rank) * c + (local - c);
}

// Launch t for workers [rank_lo, rank_hi): item k is 256-row block k % nb
// of worker w = rank_lo + k / nb's query chunk (nb = ceil(C / 256)), paired
// by schedule_pair; it lists the tiles of the block's key/value chunk
// (chunk-local indices, ascending) that hold a key some query row of the
// block may see.  An item may list none (a causal block entirely before the
// keys, or an idle worker).
Plan build_step_plan(int L, int N, bool causal, int sched, int step, int rank_lo, int rank_hi);

// Backward of launch t for workers [rank_lo, rank_hi): item k is tile k %
// nt (nt = C / 128) of worker w = rank_lo + k / nt's key/value chunk
// (schedule_pair); it lists the tiles of w's query chunk (chunk-local,
// ascending) holding a query that may see a key of that tile.  An item may
// list none.
Plan build_bwd_step_plan(int L, int N, bool causal, int sched, int step, int rank_lo, int rank_hi);

}  // namespace ra
