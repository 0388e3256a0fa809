// attn_bwd.cu -- backward kernels of blockwise Ring Self-Attention, sm_103a.
//
// The backward pass recomputes the attention probabilities from the saved
// log-sum-exp instead of storing them (activation recomputation, as the
// BPT section 4.3 and the Ring Attention section 6.2 of "Large-scale
// distributed AI model training series: sequence parallelism" use).  For
// l = sum(dO * o), with P_ij = exp(s_ij - lse_i):
//   D_i   = sum_c dO_ic o_ic
//   dV_j += sum_i P_ij dO_i
//   dS_ij = P_ij (dO_i . v_j - D_i)
//   dK_j += scale sum_i dS_ij q_i
//   dQ_i += scale sum_j dS_ij k_j
//
// Three launches:
//   bwd_pre   per row: -D_i and -lse_i in log2 units (padded rows get -inf,
//             so their probabilities are 0), and zero the fp32 dQ accumulator.
//   bwd_main  one CTA per (key/value tile, batch, query head).  K_j and V_j
//             stay in shared memory; the CTA loops over the query tiles of
//             its head that see the tile, in the order the key/value block
//             meets them going round the ring.  CTAs launch head by head
//             (longest first within a head), so the CTAs running together
//             add into the dQ rows of one or two heads, which stay in L2.
//             With grouped-query attention the G query heads of a group add
//             their dK/dV partials into fp32 accumulators (TMA reduce-add).
//             Per query tile, five tcgen05 GEMMs:
//               S^T  = K Q^T      (TMEM)      dP^T = V dO^T   (TMEM)
//               dV  += P^T dO     (TMEM)      dK  += dS^T Q   (TMEM)
//               dQ   = dS K       (TMEM, then bulk reduce-add into fp32)
//             P^T (bf16) goes to tensor memory, packed over dP^T columns
//             already read, and feeds dV as the A operand; dS^T (bf16) goes
//             to shared memory (A operand of dK, MN-major A operand of dQ).
//   bwd_post  dq = bf16(scale * dQ_acc); for grouped-query attention also
//             dk = bf16(scale * dK_acc) and dv = bf16(dV_acc).
//
// Warp roles of bwd_main: warp 0 TMA producer, warp 1 tcgen05 issuer
// (converged; one elected lane issues), warp 2 TMEM allocator, warp 3 dQ
// reduce issuer, then the compute warpgroups: two at d = 128 (384
// threads), four at d = 64 (640 threads; see BwdCfg).  All work on the
// same 128 key rows (one thread per row = TMEM lane); of G groups, group h
// takes query columns [h 128/G, (h+1) 128/G) of S^T / dP^T, dQ columns
// [h d/G, (h+1) d/G) in the drain, and in the epilogue dV (d = 128: h = 0;
// d = 64: h = 0, 1 by halves) or dK (the others).
//
// Tensor memory (fp32 columns): S^T [0,128) dP^T [128,256) dV [256,256+d)
// dK [256+d, 256+2d); dQ at [384,448) for d = 64, and over S^T for d = 128
// (S^T has been read by then; the next S^T waits for the dQ drain).  Packed
// P^T of group h occupies the first half of its dP^T columns.
//
// Product order per query tile i: dP^T(i), S^T(i) | dV(i), dK(i) one
// 16-query k-step at a time, each as soon as the compute warps have finished
// that chunk of P^T / dS^T (chunk_ready), so the tensor core runs them
// during the softmax-gradient phase | dQ(i).  dP^T(i+1) then overlaps the
// drain of dQ(i) from tensor memory, and S^T(i+1) (over the drained dQ
// columns) follows it.
//
// Buffers: K, V stationary; Q (with its rows' lse and D) and dO double
// buffered; dS^T single.  The dQ drain of tile i stages fp32 in the Q and
// dO buffers of tile i once dV(i) and dK(i) have finished reading them:
// warpgroup 0's half tile in Q, warpgroup 1's in dO, each in the
// accumulator's own layout.  Warp 3 adds each half into the accumulator
// with one 1-D bulk reduce-add, waits until it has read shared memory and
// then hands the buffer back to the producer (dO first: dP^T(i+2) is the
// first product of tile i+2), so no compute warp ever waits on a bulk copy.  (Vector atomics from
// registers instead of bulk reduce-adds ran slower, with either row layout
// of the accumulator; both paths reduce at the same per-SM rate, ~21 B/clk
// with every SM busy.)
#include <cfloat>

#include "kernels.h"
#include "plan.h"
#include "sm103_ptx.cuh"

namespace ra {

namespace {

// Compute warpgroups per CTA: two of 64 query columns at d = 128, four of
// 32 at d = 64, where registers allow it and the softmax-gradient phase
// rather than the products sets the pace (a 128 x 128 tile is half the
// tensor work of d = 128 for the same per-element work).
template <int D>
struct BwdCfg {
  static constexpr int kWG = D == 64 ? 4 : 2;        // compute warpgroups
  static constexpr int kCols = 128 / kWG;            // query columns per warpgroup
  static constexpr int kChunks = kCols / 16;         // 16-column chunks per warpgroup
  static constexpr int kThreads = 128 + 128 * kWG;   // 4 role warps + the compute warpgroups
  static constexpr int kComputeWarps = 4 * kWG;
};
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdSmem {
  static constexpr int kSub = D / 64;
  static constexpr int kTile = 128 * D * 2;
  alignas(1024) uint8_t k[kTile];
  alignas(1024) uint8_t v[kTile];
  alignas(1024) uint8_t q[2][kTile];
  alignas(1024) uint8_t dO[2][kTile];
  alignas(1024) uint8_t dsT[128 * 128 * 2];
  alignas(16) float lse2[2][128];
  alignas(16) float dvec[2][128];
  alignas(8) uint64_t kv_full;
  alignas(8) uint64_t q_full[2];
  alignas(8) uint64_t q_empty[2];
  alignas(8) uint64_t do_full[2];
  alignas(8) uint64_t do_empty[2];
  alignas(8) uint64_t s_full;
  // P^T and dS^T of query columns [16c, 16c+16) of both halves are in
  // place (one arrival per compute warp)
  alignas(8) uint64_t chunk_ready[4];
  alignas(8) uint64_t dq_full;
  alignas(8) uint64_t dq_free;
  alignas(8) uint64_t qdo_read;    // dV(i), dK(i) done: Q(i), dO(i) free for staging
  // the 8 compute warps staged dQ(i) in slot i % 2; one barrier per slot,
  // so its phases cannot run ahead of the reducer (staging tile i+2 in the
  // slot needs the reducer to have released it after tile i)
  alignas(8) uint64_t stage_full[2];
  alignas(8) uint64_t kv_final;
  alignas(8) uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Offset of element (row i, column col) of the (batch, head) slice z of the
// fp32 dQ accumulator: tiles of 128 query rows, each stored as d/4 column
// quads of [128 rows][4 floats].  The half tile of one compute warpgroup
// (d/2 columns) is then one contiguous block, both here and in its staging
// buffer, and goes into the accumulator as a single bulk reduce-add.
template <int D>
__host__ __device__ __forceinline__ size_t dq_acc_offset(long long z, int Lpad, int i, int col) {
  return static_cast<size_t>(z) * Lpad * D + static_cast<size_t>(i >> 7) * 128 * D + (col >> 2) * 512 +
         (i & 127) * 4 + (col & 3);
}

struct BwdDev {
  int B, Hq, Hkv, L, Lpad, causal;
  int n_blocks;        // key/value tiles per (batch, head)
  int kv_accumulate;   // grouped-query attention: dK/dV partials reduce into fp32
  float scale, scale_log2;
  const int32_t* order;
  const int32_t* offsets;
  const int32_t* ranges;
  const float* lse2;
  const float* dvec;
  float* dq_acc;       // fp32, tiled (dq_acc_offset)
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* err;
  // Ring step mode (step_nt > 0): item k is key/value tile k % step_nt of
  // the block of worker w = k / step_nt at launch `step` of schedule `sched`
  // (schedule_pair: query chunk a, key/value chunk b), against a's query
  // chunk; L = Lpad = the chunk length; slices: q, dO, statistics, dQ at
  // a * B*Hq + (b, h), k, v, dK, dV at b * B*Hkv + (b, kv head); causal keys
  // from the schedule's chunk map.
  int step_nt, step, n_chunks, sched;
  // step mode: the first worker of the launch (item k's worker is rank_lo +
  // k / step_nt), and whether the buffers hold every chunk (z_rank = 1,
  // chunk-major) or only the block's own query and key/value chunks (0)
  int rank_lo, z_rank;
};

// Causal-mask keys of the backward (as in the forward's step mode): a key
// row with key kk is visible to query column qq of a tile whose first row
// has key q0k iff kk <= q0k + qq.
template <bool kStep>
__device__ __forceinline__ int bwd_q_key(const BwdDev& p, int rank, int local) {
  if (!kStep || !p.causal || p.sched == kSchedStriped) return local;
  return chunk_pos(p.L * p.n_chunks, p.n_chunks, true, p.sched, rank, local);
}
template <bool kStep>
__device__ __forceinline__ int bwd_kv_key(const BwdDev& p, int kv_rank, int q_rank, int local) {
  if (!kStep || !p.causal) return local;
  if (p.sched == kSchedStriped) return local + (kv_rank > q_rank ? 1 : 0);
  return chunk_pos(p.L * p.n_chunks, p.n_chunks, true, p.sched, kv_rank, local);
}

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, int* err) {
  int local = 0;
  mbar_wait(bar, parity, &local, err, kSiteBwdDrain);
}

// Visits the query tiles `it` of the CTA's list (ranges of tile indices), in order.
struct QIter {
  const int32_t* rg;
  int nr;
  int ri = 0, it = 0;
  __device__ QIter(const int32_t* rg_, int nr_) : rg(rg_), nr(nr_) { it = nr > 0 ? rg[0] : 0; }
  __device__ bool valid() const { return ri < nr; }
  __device__ void next() {
    if (++it < rg[2 * ri + 1]) return;
    if (++ri < nr) it = rg[2 * ri];
  }
};

template <int D>
__device__ void bwd_producer(BwdSmem<D>& sm, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                             const CUtensorMap* tm_v, const CUtensorMap* tm_do, const BwdDev& p, int kv_z,
                             int q_z, int kv_tile, const int32_t* rg, int nr, volatile int* ab, int* err) {
  using S = BwdSmem<D>;
  const uint32_t kvb = smem_u32(&sm.kv_full);
  mbar_arrive_expect_tx(kvb, 2 * S::kTile);
  for (int sub = 0; sub < S::kSub; ++sub) {
    tma_load_3d(smem_u32(sm.k) + sub * 16384, tm_k, kvb, sub * 64, kv_tile * 128, kv_z);
    tma_load_3d(smem_u32(sm.v) + sub * 16384, tm_v, kvb, sub * 64, kv_tile * 128, kv_z);
  }
  bool ok = true;
  uint32_t nq = 0, ndo = 0;  // Q and dO fills issued
  // dO(i) first: dP^T(i) is the tile's first product, and the dQ reducer
  // hands the dO buffer back first
  for (QIter qi(rg, nr); qi.valid() && ok; qi.next()) {
    const uint32_t i = ndo;
    const uint32_t slot = i & 1;
    if (i >= 2) ok = mbar_wait(smem_u32(&sm.do_empty[slot]), ((i >> 1) - 1) & 1, ab, err, kSiteBwdProducer);
    if (!ok) break;
    const uint32_t db = smem_u32(&sm.do_full[slot]);
    mbar_arrive_expect_tx(db, S::kTile);
    for (int sub = 0; sub < S::kSub; ++sub)
      tma_load_3d(smem_u32(sm.dO[slot]) + sub * 16384, tm_do, db, sub * 64, qi.it * 128, q_z);
    ++ndo;
    if (i >= 2) ok = mbar_wait(smem_u32(&sm.q_empty[slot]), ((i >> 1) - 1) & 1, ab, err, kSiteBwdProducer);
    if (!ok) break;
    const uint32_t qb = smem_u32(&sm.q_full[slot]);
    mbar_arrive_expect_tx(qb, S::kTile + 1024);
    for (int sub = 0; sub < S::kSub; ++sub)
      tma_load_3d(smem_u32(sm.q[slot]) + sub * 16384, tm_q, qb, sub * 64, qi.it * 128, q_z);
    const size_t roff = static_cast<size_t>(q_z) * p.Lpad + qi.it * 128;
    bulk_load_1d(smem_u32(sm.lse2[slot]), p.lse2 + roff, 512, qb);
    bulk_load_1d(smem_u32(sm.dvec[slot]), p.dvec + roff, 512, qb);
    ++nq;
  }
  if (!ok) {
    // Let every copy this thread issued land before the CTA exits.
    wait_drain(kvb, 0, err);
    for (uint32_t s = 0; s < 2 && s < nq; ++s) {
      const uint32_t last = s + 2 * ((nq - 1 - s) / 2);
      wait_drain(smem_u32(&sm.q_full[s]), (last >> 1) & 1, err);
    }
    for (uint32_t s = 0; s < 2 && s < ndo; ++s) {
      const uint32_t last = s + 2 * ((ndo - 1 - s) / 2);
      wait_drain(smem_u32(&sm.do_full[s]), (last >> 1) & 1, err);
    }
  }
}

template <int D>
__device__ void bwd_mma(BwdSmem<D>& sm, uint32_t tmem, uint32_t n_total, volatile int* ab, int* err) {
  constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
  constexpr uint32_t kIdKV = idesc_bf16(128, D, false, true);
  constexpr uint32_t kIdQ = idesc_bf16(128, D, true, true);
  const uint32_t t_s = tmem, t_dp = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 256 + D;
  const uint32_t t_dq = (D == 128) ? tmem : tmem + 384;
  const uint32_t ka = smem_u32(sm.k), va = smem_u32(sm.v), sa = smem_u32(sm.dsT);

  bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.kv_full), 0, ab, err, kSiteBwdMma));
  for (uint32_t i = 0; i < n_total && ok; ++i) {
    const uint32_t slot = i & 1;
    const uint32_t qa = smem_u32(sm.q[slot]), da = smem_u32(sm.dO[slot]);
    // dP^T = V dO^T first: it overwrites the packed P^T of the previous
    // tile, which dV(i-1) read earlier in this thread's issue order, so it
    // waits only for dO(i) and runs while the compute warps drain dQ(i-1).
    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.do_full[slot]), (i >> 1) & 1, ab, err, kSiteBwdMma));
    if (!ok) break;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
      umma_ss_warp(t_dp, sdesc_sw128(va + off, 16, 1024), sdesc_sw128(da + off, 16, 1024), kIdS, kk > 0);
    }
    // S^T = K Q^T (both operands K-major) overwrites dQ(i-1): it waits for
    // Q(i) and for the drain of dQ(i-1) (dq_free).
    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.q_full[slot]), (i >> 1) & 1, ab, err, kSiteBwdMma));
    if (ok && i > 0) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.dq_free), (i - 1) & 1, ab, err, kSiteBwdMma));
    if (!ok) break;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
      umma_ss_warp(t_s, sdesc_sw128(ka + off, 16, 1024), sdesc_sw128(qa + off, 16, 1024), kIdS, kk > 0);
    }
    umma_commit_warp(smem_u32(&sm.s_full));
    // dV += P^T dO and dK += dS^T Q one query k-step (16 queries) at a
    // time, as the compute warps finish each 16-column chunk c of every
    // warpgroup's columns: k-step kChunks h + c of warpgroup h, so the
    // tensor core works while the softmax-gradient phase runs.
    //   dV: A = packed P^T in tensor memory (warpgroup h's chunk c at
    //       column 128 + kCols h + 8 c), B = dO (MN-major)
    //   dK: A = dS^T (K-major), B = Q (MN-major)
    using Cfg = BwdCfg<D>;
    for (int c = 0; c < Cfg::kChunks && ok; ++c) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.chunk_ready[c]), i & 1, ab, err, kSiteBwdMma));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < Cfg::kWG; ++h) {
        const int kk = Cfg::kChunks * h + c;  // 16-query k-step
        // dS^T columns 16 kk.. : 64-column sub-tile kk / 4, bytes 32 (kk % 4)
        const uint32_t ds_off = Cfg::kWG == 2 ? h * 16384 + c * 32 : (kk >> 2) * 16384 + (kk & 3) * 32;
        umma_ts_warp(t_dv, tmem + 128 + Cfg::kCols * h + 8 * c, sdesc_sw128(da + kk * 2048, 16384, 1024), kIdKV,
                     (i > 0 || kk > 0) ? 1u : 0u);
        umma_ss_warp(t_dk, sdesc_sw128(sa + ds_off, 16, 1024), sdesc_sw128(qa + kk * 2048, 16384, 1024), kIdKV,
                     (i > 0 || kk > 0) ? 1u : 0u);
      }
    }
    if (!ok) break;
    umma_commit_warp(smem_u32(&sm.qdo_read));  // Q(i), dO(i) no longer read: free for the dQ staging
    // dQ = dS K : A = dS (MN-major view of dS^T), B = K (MN-major); the
    // last chunk_ready covers every chunk of dS^T.  Over the S^T columns
    // for d = 128 (read by then).
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      umma_ss_warp(t_dq, sdesc_sw128(sa + kk * 2048, 16384, 1024), sdesc_sw128(ka + kk * 2048, 16384, 1024), kIdQ,
                   kk > 0);
    umma_commit_warp(smem_u32(&sm.dq_full));
  }
  if (ok) {
    umma_commit_warp(smem_u32(&sm.kv_final));
  } else {
    umma_commit_warp(smem_u32(&sm.drain));
    wait_drain(smem_u32(&sm.drain), 0, err);
  }
}

// Warp 3, one lane: for each query tile, once the 8 compute warps have
// staged dQ(i), issue the bulk reduce-adds of their halves into the fp32
// accumulator, wait until the copies have read shared memory and return
// the tile's Q and dO buffers to the producer.  Joins the compute warps'
// named barrier before their epilogue, all copies complete.
template <int D>
__device__ void bwd_dq_reducer(BwdSmem<D>& sm, float* dq_acc, int Lpad, int q_z, const int32_t* rg, int nr,
                               volatile int* ab, int* err) {
  bool ok = true;
  uint32_t i = 0;
  for (QIter qi(rg, nr); qi.valid() && ok; qi.next(), ++i) {
    const uint32_t slot = i & 1;
    ok = mbar_wait(smem_u32(&sm.stage_full[slot]), (i >> 1) & 1, ab, err, kSiteBwdReducer);
    if (!ok) break;
    const int q0 = qi.it * 128;
    // warpgroup 1's half tile (staged in the dO buffer), then warpgroup 0's
    // (in the Q buffer), as two groups: dO goes back to the producer (which
    // refills it first, for the tile's first product) as soon as its half
    // has been read
    float* const dst = dq_acc + dq_acc_offset<D>(q_z, Lpad, q0, 0);
    constexpr uint32_t kHalf = 128 * (D / 2) * 4;
    bulk_reduce_add_f32(dst + kHalf / 4, smem_u32(sm.dO[slot]), kHalf);
    bulk_commit_group();
    bulk_reduce_add_f32(dst, smem_u32(sm.q[slot]), kHalf);
    bulk_commit_group();
    bulk_wait_group_read<1>();
    mbar_arrive(smem_u32(&sm.do_empty[slot]));
    bulk_wait_group_read<0>();
    mbar_arrive(smem_u32(&sm.q_empty[slot]));
  }
  bulk_wait_group<0>();
}

template <int D, bool kStep>
__device__ void bwd_compute(BwdSmem<D>& sm, uint32_t tmem, const BwdDev& p, const CUtensorMap* tm_dkacc,
                            const CUtensorMap* tm_dvacc, int kv_z, int q_z, int kv_tile, int q_rank, int kv_rank,
                            const int32_t* rg, int nr, volatile int* ab, int* err) {
  using Cfg = BwdCfg<D>;
  const int wg = ((threadIdx.x >> 5) - 4) >> 2;  // which kCols-column group of the queries
  const int wq = (threadIdx.x >> 5) & 3;         // TMEM lane quadrant
  const int lane = threadIdx.x & 31;
  const int row = wq * 32 + lane;  // key row (S^T lane) and also dQ query row
  const int kv_pos = kv_tile * 128 + row;  // row of the key/value slice
  const int kv_key = bwd_kv_key<kStep>(p, kv_rank, q_rank, kv_pos);
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t t_s = tmem + Cfg::kCols * wg + lane_off;         // this group's S^T columns
  const uint32_t t_dp = tmem + 128 + Cfg::kCols * wg + lane_off;  // this group's dP^T columns
  const uint32_t t_p = t_dp;                               // packed P^T over the first 32 of them
  constexpr int kDqCols = D / Cfg::kWG;  // dQ columns this group drains
  const uint32_t t_dq = ((D == 128) ? tmem : tmem + 384) + kDqCols * wg + lane_off;
  const uint32_t sa = smem_u32(sm.dsT);
  const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
  bool ok = true;
  uint32_t i = 0;
  for (QIter qi(rg, nr); qi.valid() && ok; qi.next(), ++i) {
    const uint32_t slot = i & 1;
    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.q_full[slot]), (i >> 1) & 1, ab, err, kSiteBwdSoftmax));
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full), i & 1, ab, err, kSiteBwdSoftmax));
    if (!ok) break;
    tc_fence_after();
    const int q0 = qi.it * 128;
    // Probabilities are zero where the key is after the query (causal) or
    // past the end; padded query rows have -lse2 = -inf, hence P = 0.
    const int first_valid_q = p.causal ? kv_key - bwd_q_key<kStep>(p, q_rank, q0) : 0;  // local query index
    const bool row_dead = kv_pos >= p.L;
    const bool need_mask = row_dead || first_valid_q > Cfg::kCols * wg;
    const float* nlse2 = sm.lse2[slot];  // -lse * log2(e)
    const float* ndvec = sm.dvec[slot];  // -D

    // 16 query columns: P^T packed into tensor memory, dS^T into shared memory
    auto process = [&](int c, uint32_t (&rs)[16], uint32_t (&rp)[16]) {
      uint32_t pk[8], dk8[8];
#pragma unroll
      for (int x = 0; x < 16; x += 4) {
        const int qq = Cfg::kCols * wg + 16 * c + x;
        const float4 nl = *reinterpret_cast<const float4*>(nlse2 + qq);
        const float4 nd = *reinterpret_cast<const float4*>(ndvec + qq);
        const float2 a0 = __ffma2_rn(make_float2(__uint_as_float(rs[x]), __uint_as_float(rs[x + 1])), c2,
                                     make_float2(nl.x, nl.y));
        const float2 a1 = __ffma2_rn(make_float2(__uint_as_float(rs[x + 2]), __uint_as_float(rs[x + 3])), c2,
                                     make_float2(nl.z, nl.w));
        float2 p0 = make_float2(ex2(a0.x), ex2(a0.y));
        float2 p1 = make_float2(ex2(a1.x), ex2(a1.y));
        if (need_mask) {
          if (row_dead || qq < first_valid_q) p0.x = 0.f;
          if (row_dead || qq + 1 < first_valid_q) p0.y = 0.f;
          if (row_dead || qq + 2 < first_valid_q) p1.x = 0.f;
          if (row_dead || qq + 3 < first_valid_q) p1.y = 0.f;
        }
        const float2 d0 = __fadd2_rn(make_float2(__uint_as_float(rp[x]), __uint_as_float(rp[x + 1])),
                                     make_float2(nd.x, nd.y));
        const float2 d1 = __fadd2_rn(make_float2(__uint_as_float(rp[x + 2]), __uint_as_float(rp[x + 3])),
                                     make_float2(nd.z, nd.w));
        const float2 s0 = __fmul2_rn(p0, d0), s1 = __fmul2_rn(p1, d1);
        pk[x / 2] = pack_bf16(p0.x, p0.y);
        pk[x / 2 + 1] = pack_bf16(p1.x, p1.y);
        dk8[x / 2] = pack_bf16(s0.x, s0.y);
        dk8[x / 2 + 1] = pack_bf16(s1.x, s1.y);
      }
      // packed columns 8c..8c+7 of this group lie in its dP^T columns
      // 0..8 kChunks - 1, all read in the chunks before c's successor (c's
      // own columns, 16c.., are read by the time they are written over)
      tmem_st8_async(t_p + 8 * c, pk);
      const int qb = Cfg::kCols * wg + 16 * c;               // the chunk's first query column
      const uint32_t sub = sa + static_cast<uint32_t>(qb >> 6) * 16384;  // its 64-column sub-tile
      const int ch = (qb & 63) >> 3;  // 16-byte chunk (8 queries) within the sub-tile's 128-byte row
      st_shared_v4(sub + sw128_offset(row, ch), dk8[0], dk8[1], dk8[2], dk8[3]);
      st_shared_v4(sub + sw128_offset(row, ch + 1), dk8[4], dk8[5], dk8[6], dk8[7]);
    };
    // chunk c of this warp's rows is in place -- P^T in tensor memory, dS^T
    // in shared memory, made visible to the tensor core's async proxy -- so
    // the MMA warp may run the chunk's dV and dK k-steps
    auto signal = [&](int c) {
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.chunk_ready[c]));
    };
    {
      uint32_t sA[16], pA[16], sB[16], pB[16];
      tmem_ld16_async(t_s, sA);
      tmem_ld16_async(t_dp, pA);
      tmem_wait_ld(sA);
      reg_fence(pA);
      tmem_ld16_async(t_s + 16, sB);
      tmem_ld16_async(t_dp + 16, pB);
      process(0, sA, pA);
      signal(0);
      tmem_wait_ld(sB);
      reg_fence(pB);
      if constexpr (Cfg::kChunks == 4) {
        tmem_ld16_async(t_s + 32, sA);
        tmem_ld16_async(t_dp + 32, pA);
        process(1, sB, pB);
        signal(1);
        tmem_wait_ld(sA);
        reg_fence(pA);
        tmem_ld16_async(t_s + 48, sB);
        tmem_ld16_async(t_dp + 48, pB);
        process(2, sA, pA);
        signal(2);
        tmem_wait_ld(sB);
        reg_fence(pB);
        process(3, sB, pB);
        signal(3);
      } else {
        process(1, sB, pB);
        signal(1);
      }
    }
    // dQ drain: this thread's dQ row (a query row), this half's columns,
    // leaves tensor memory in one batched load; the columns are released at
    // once, then the row is staged as fp32 in the tile's Q and dO buffers
    // (once dV and dK have read them) for warp 3's reduce-adds into
    // the global accumulator.
    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.dq_full), i & 1, ab, err, kSiteBwdSoftmax));
    if (!ok) break;
    tc_fence_after();
    if constexpr (Cfg::kWG == 2) {
      uint32_t d0[32], d1[32];
      tmem_ld32_async(t_dq, d0);
      if (D == 128) tmem_ld32_async(t_dq + 32, d1);
      tmem_wait_ld(d0);
      if (D == 128) reg_fence(d1);
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.dq_free));
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.qdo_read), i & 1, ab, err, kSiteBwdSoftmax));
      if (!ok) break;
      // staging in the accumulator's own layout: warpgroup wg's half tile in
      // the tile's Q (wg 0) or dO (wg 1) buffer as [d/8 quads][128 rows][4]
      const uint32_t stage = smem_u32(wg == 0 ? sm.q[slot] : sm.dO[slot]) + row * 16;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        st_shared_v4(stage + k * 2048, d0[4 * k], d0[4 * k + 1], d0[4 * k + 2], d0[4 * k + 3]);
      if (D == 128) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          st_shared_v4(stage + (8 + k) * 2048, d1[4 * k], d1[4 * k + 1], d1[4 * k + 2], d1[4 * k + 3]);
      }
    } else {
      // four groups of d/4 dQ columns: group wg's quads of the
      // [d/4 quads][128 rows][4] tile, the first d/8 quads in the Q buffer,
      // the rest in the dO buffer
      uint32_t e[kDqCols];
      if constexpr (kDqCols == 16) {
        tmem_ld16_async(t_dq, e);
      } else {
        tmem_ld32_async(t_dq, e);
      }
      tmem_wait_ld(e);
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.dq_free));
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.qdo_read), i & 1, ab, err, kSiteBwdSoftmax));
      if (!ok) break;
      const int quad0 = (kDqCols / 4) * wg;
      const uint32_t stage = smem_u32(quad0 < D / 8 ? sm.q[slot] : sm.dO[slot]) + (quad0 % (D / 8)) * 2048 + row * 16;
#pragma unroll
      for (int k = 0; k < kDqCols / 4; ++k)
        st_shared_v4(stage + k * 2048, e[4 * k], e[4 * k + 1], e[4 * k + 2], e[4 * k + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.stage_full[slot]));
  }
  // Warp 3's reduce-adds have read every staged half once it joins here;
  // the dK/dV epilogue below reuses the Q and dO buffers across warps.
  named_bar_sync(1, 128 * Cfg::kWG + 32);
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.kv_final), 0, ab, err, kSiteBwdEpilogue));
  if constexpr (Cfg::kWG == 2) {
    if (ok) {
      // Epilogue: warpgroup 0 takes dV, warpgroup 1 takes dK.  Without grouped
      // queries the CTA holds the whole gradient and writes bf16 (dK times
      // scale); with them it adds its fp32 partial into the accumulator
      // through staging boxes in the Q and dO buffers, free once kv_final
      // arrived (every load was consumed by then).
      tc_fence_after();
      const uint32_t t_src = (wg == 0 ? tmem + 256 : tmem + 256 + D) + lane_off;
      if (!p.kv_accumulate) {
        const bool store = kv_pos < p.L;
        const size_t base = (static_cast<size_t>(kv_z) * p.L + (store ? kv_pos : 0)) * D;
        __nv_bfloat16* dst_row = (wg == 0 ? p.dv : p.dk) + base;
        const float s = wg == 0 ? 1.f : p.scale;
  #pragma unroll
        for (int c0 = 0; c0 < D / 32; c0 += 2) {
          uint32_t r0[32], r1[32];
          tmem_ld32_async(t_src + c0 * 32, r0);
          tmem_ld32_async(t_src + c0 * 32 + 32, r1);
          tmem_wait_ld(r0);
          reg_fence(r1);
          if (store) {
            uint4* dst = reinterpret_cast<uint4*>(dst_row + c0 * 32);
  #pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float* f = reinterpret_cast<const float*>(q4 < 4 ? r0 : r1) + (q4 & 3) * 8;
              dst[q4] = make_uint4(pack_bf16(f[0] * s, f[1] * s), pack_bf16(f[2] * s, f[3] * s),
                                   pack_bf16(f[4] * s, f[5] * s), pack_bf16(f[6] * s, f[7] * s));
            }
          }
        }
      } else {
        // warp e = 4 wg + wq stages its 32 rows x d fp32 (d/32 boxes of 4 KB) in
        // half e % 2 of buffer e / 2 of {Q0, Q1, dO0, dO1}
        const int e = 4 * wg + wq;
        uint8_t* buf = e < 4 ? sm.q[e >> 1] : sm.dO[(e - 4) >> 1];
        const uint32_t region = smem_u32(buf) + (e & 1) * (BwdSmem<D>::kTile / 2);
        const CUtensorMap* tm = wg == 0 ? tm_dvacc : tm_dkacc;
  #pragma unroll
        for (int c0 = 0; c0 < D / 32; c0 += 2) {
          uint32_t r0[32], r1[32];
          tmem_ld32_async(t_src + c0 * 32, r0);
          tmem_ld32_async(t_src + c0 * 32 + 32, r1);
          tmem_wait_ld(r0);
          reg_fence(r1);
  #pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            st_shared_v4(region + c0 * 4096 + sw128_offset(lane, c8), r0[c8 * 4], r0[c8 * 4 + 1], r0[c8 * 4 + 2],
                         r0[c8 * 4 + 3]);
            st_shared_v4(region + (c0 + 1) * 4096 + sw128_offset(lane, c8), r1[c8 * 4], r1[c8 * 4 + 1],
                         r1[c8 * 4 + 2], r1[c8 * 4 + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int c0 = 0; c0 < D / 32; ++c0)
            tma_reduce_add_3d(tm, region + c0 * 4096, 32 * c0, kv_tile * 128 + wq * 32, kv_z);
          bulk_commit_group();
          bulk_wait_group<0>();
        }
        __syncwarp();
      }
    }
  } else if (ok) {
    // four groups: groups 0, 1 take dV's columns by halves, groups 2, 3
    // dK's; with grouped queries each warp stages its 32 rows x d/2 fp32
    // (d/64 boxes of 4 KB) in quarter e % 4 of buffer e / 4 of
    // {Q0, Q1, dO0, dO1} and adds it into the accumulator
    tc_fence_after();
    constexpr int kEpCols = D / 2;
    const bool is_dv = wg < 2;
    const int col0 = (wg & 1) * kEpCols;
    const uint32_t t_src = (is_dv ? tmem + 256 : tmem + 256 + D) + col0 + lane_off;
    const int e = 4 * wg + wq;
    uint8_t* buf = (e >> 2) < 2 ? sm.q[e >> 2] : sm.dO[(e >> 2) - 2];
    const uint32_t region = smem_u32(buf) + (e & 3) * (kEpCols / 32) * 4096;
#pragma unroll
    for (int c0 = 0; c0 < kEpCols / 32; ++c0) {
      uint32_t r0[32];
      tmem_ld32_async(t_src + c0 * 32, r0);
      tmem_wait_ld(r0);
      if (!p.kv_accumulate) {
        if (kv_pos < p.L) {
          const float sc = is_dv ? 1.f : p.scale;
          uint4* dst = reinterpret_cast<uint4*>((is_dv ? p.dv : p.dk) + (static_cast<size_t>(kv_z) * p.L + kv_pos) * D +
                                                col0 + 32 * c0);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const float* f = reinterpret_cast<const float*>(r0) + q4 * 8;
            dst[q4] = make_uint4(pack_bf16(f[0] * sc, f[1] * sc), pack_bf16(f[2] * sc, f[3] * sc),
                                 pack_bf16(f[4] * sc, f[5] * sc), pack_bf16(f[6] * sc, f[7] * sc));
          }
        }
      } else {
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          st_shared_v4(region + c0 * 4096 + sw128_offset(lane, c8), r0[c8 * 4], r0[c8 * 4 + 1], r0[c8 * 4 + 2],
                       r0[c8 * 4 + 3]);
      }
    }
    if (p.kv_accumulate) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        for (int c0 = 0; c0 < kEpCols / 32; ++c0)
          tma_reduce_add_3d(is_dv ? tm_dvacc : tm_dkacc, region + c0 * 4096, col0 + 32 * c0, kv_tile * 128 + wq * 32,
                            kv_z);
        bulk_commit_group();
        bulk_wait_group<0>();
      }
      __syncwarp();
    }
  }
}

template <int D, bool kStep>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    ring_attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dkacc,
                         const __grid_constant__ CUtensorMap tm_dvacc, const BwdDev p) {
  using S = BwdSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kSiteBwdMisaligned);
    return;
  }
  S& sm = *reinterpret_cast<S*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // items head-major: all key tiles of query head 0 (longest first), then head 1, ...
  const int qh = blockIdx.x / p.n_blocks;  // b * Hq + h
  const int item = p.order[blockIdx.x % p.n_blocks];
  const int b = qh / p.Hq, h = qh % p.Hq;
  int kv_tile = item, q_rank = 0, kv_rank = 0;
  int q_z = qh, kv_z = b * p.Hkv + h / (p.Hq / p.Hkv);
  if constexpr (kStep) {
    kv_tile = item % p.step_nt;
    schedule_pair(p.n_chunks, p.sched, p.step, p.rank_lo + item / p.step_nt, &q_rank, &kv_rank);
    q_z += q_rank * p.z_rank * p.B * p.Hq;
    kv_z += kv_rank * p.z_rank * p.B * p.Hkv;
  }
  const int32_t* rg = p.ranges + 2 * p.offsets[item];
  const int nr = p.offsets[item + 1] - p.offsets[item];
  if (kStep && nr == 0) return;  // a ring-step tile no query of the rank sees: nothing to add
  volatile int* ab = &sm.abort_flag;

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(smem_u32(&sm.kv_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&sm.q_full[s]), 1);
      mbar_init(smem_u32(&sm.q_empty[s]), 1);  // released by the dQ reduce issuer
      mbar_init(smem_u32(&sm.do_full[s]), 1);
      mbar_init(smem_u32(&sm.do_empty[s]), 1);
    }
    mbar_init(smem_u32(&sm.s_full), 1);
    for (int c = 0; c < 4; ++c) mbar_init(smem_u32(&sm.chunk_ready[c]), BwdCfg<D>::kComputeWarps);
    mbar_init(smem_u32(&sm.dq_full), 1);
    mbar_init(smem_u32(&sm.dq_free), 32 * BwdCfg<D>::kComputeWarps);
    mbar_init(smem_u32(&sm.qdo_read), 1);
    mbar_init(smem_u32(&sm.stage_full[0]), BwdCfg<D>::kComputeWarps);
    mbar_init(smem_u32(&sm.stage_full[1]), BwdCfg<D>::kComputeWarps);
    mbar_init(smem_u32(&sm.kv_final), 1);
    mbar_init(smem_u32(&sm.drain), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    if (p.kv_accumulate) {
      tma_prefetch_desc(&tm_dkacc);
      tma_prefetch_desc(&tm_dvacc);
    }
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  if (warp == 0) {
    if (lane == 0) bwd_producer<D>(sm, &tm_q, &tm_k, &tm_v, &tm_do, p, kv_z, q_z, kv_tile, rg, nr, ab, p.err);
  } else if (warp == 1) {
    // the whole warp runs the issue loop; one elected lane issues
    int nq = 0;
    for (int ri = 0; ri < nr; ++ri) nq += rg[2 * ri + 1] - rg[2 * ri];
    bwd_mma<D>(sm, tmem, static_cast<uint32_t>(nq), ab, p.err);
  } else if (warp == 3) {
    if (lane == 0) bwd_dq_reducer<D>(sm, p.dq_acc, p.Lpad, q_z, rg, nr, ab, p.err);
    __syncwarp();
    named_bar_sync(1, 128 * BwdCfg<D>::kWG + 32);
  } else if (warp >= 4) {
    bwd_compute<D, kStep>(sm, tmem, p, &tm_dkacc, &tm_dvacc, kv_z, q_z, kv_tile, q_rank, kv_rank, rg, nr, ab,
                          p.err);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, 512);
}

// The pre-pass: per row, -D_i = -sum_c dO_ic o_ic and -lse_i log2(e) (0 and
// -inf for padded rows, whose probabilities are then 0); and the fp32 dQ
// accumulator zeroed, with the dK and dV accumulators for rows below
// kv_rows (grouped-query attention; null otherwise).  HBM-bound: a bf16 row
// of o (and of dO) is D/8 16-byte pieces, so a warp covers 32/(D/8) rows at
// once and takes kIter such groups, all loads issued before any use so that
// enough bytes are in flight; the row sums reduce across the row's lanes by
// shuffles.  Each warp then zeroes the accumulator chunks of its rows (the
// accumulators are B*Hq*Lpad*D and B*Hkv*Lpad*D contiguous floats whatever
// their tiling, so the chunks of all rows cover them).
template <int D>
__global__ void __launch_bounds__(256) ring_attn_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                                const __nv_bfloat16* __restrict__ dO,
                                                                const float* __restrict__ lse, float* lse2,
                                                                float* dvec, float* dq_acc, float* dk_acc,
                                                                float* dv_acc, int L, int Lpad, long long n_rows,
                                                                long long kv_rows) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerGroup = 32 / kLanesPerRow;
  constexpr int kIter = 4;
  constexpr int kRowsPerWarp = kRowsPerGroup * kIter;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow, piece = lane % kLanesPerRow;
  const long long r0 = warp_id * kRowsPerWarp;
  if (r0 >= n_rows) return;
  uint4 a[kIter], b[kIter];
#pragma unroll
  for (int it = 0; it < kIter; ++it) {
    const long long r = r0 + it * kRowsPerGroup + sub;
    const long long bh = r / Lpad;
    const int i = static_cast<int>(r % Lpad);
    a[it] = b[it] = make_uint4(0u, 0u, 0u, 0u);
    if (r < n_rows && i < L) {
      const size_t off = (static_cast<size_t>(bh) * L + i) * D + piece * 8;
      a[it] = *reinterpret_cast<const uint4*>(o + off);
      b[it] = *reinterpret_cast<const uint4*>(dO + off);
    }
  }
#pragma unroll
  for (int it = 0; it < kIter; ++it) {
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[it]);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b[it]);
    float acc = 0.f;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float2 fa = __bfloat1622float2(a2[x]), fb = __bfloat1622float2(b2[x]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
#pragma unroll
    for (int s = kLanesPerRow / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    const long long r = r0 + it * kRowsPerGroup + sub;
    if (piece == 0 && r < n_rows) {
      const long long bh = r / Lpad;
      const int i = static_cast<int>(r % Lpad);
      dvec[r] = (i < L) ? -acc : 0.f;
      lse2[r] = (i < L) ? -lse[static_cast<size_t>(bh) * L + i] * kLog2e : -INFINITY;
    }
  }
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  const long long rows_here = min(static_cast<long long>(kRowsPerWarp), n_rows - r0);
  float4* z = reinterpret_cast<float4*>(dq_acc + static_cast<size_t>(r0) * D);
  for (long long x = lane; x < rows_here * (D / 4); x += 32) z[x] = zero;
  if (dk_acc && r0 < kv_rows) {
    const long long kv_here = min(static_cast<long long>(kRowsPerWarp), kv_rows - r0);
    float4* zk = reinterpret_cast<float4*>(dk_acc + static_cast<size_t>(r0) * D);
    float4* zv = reinterpret_cast<float4*>(dv_acc + static_cast<size_t>(r0) * D);
    for (long long x = lane; x < kv_here * (D / 4); x += 32) {
      zk[x] = zero;
      zv[x] = zero;
    }
  }
}

// dst[z][i][:] = bf16(scale * src[z][i][:]) for rows i < L (src has Lpad
// rows per z); 8 elements per thread.
template <int D>
__global__ void __launch_bounds__(256) ring_attn_bwd_post_kernel(const float* __restrict__ dq_acc,
                                                                 __nv_bfloat16* __restrict__ dq, float scale, int L,
                                                                 int Lpad, long long n_out8) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n_out8) return;
  const long long e = t * 8;                      // element index in [B*Hq*L*D)
  const long long row = e / D;                    // (bh, i) flattened over L
  const int col = static_cast<int>(e % D);
  const long long bh = row / L;
  const int i = static_cast<int>(row % L);
  const float4* src = reinterpret_cast<const float4*>(dq_acc + (static_cast<size_t>(bh) * Lpad + i) * D + col);
  const float4 a = src[0], bq = src[1];
  uint4 out = make_uint4(pack_bf16(a.x * scale, a.y * scale), pack_bf16(a.z * scale, a.w * scale),
                         pack_bf16(bq.x * scale, bq.y * scale), pack_bf16(bq.z * scale, bq.w * scale));
  *reinterpret_cast<uint4*>(dq + e) = out;
}

// dq[z][i][:] = bf16(scale * dQ_acc) for rows i < L, reading the tiled
// accumulator: thread t takes query row t % 128 of its tile and 8 columns,
// so a warp reads two contiguous 512-byte runs.
template <int D>
__global__ void __launch_bounds__(256) ring_attn_bwd_dq_post_kernel(const float* __restrict__ dq_acc,
                                                                    __nv_bfloat16* __restrict__ dq, float scale,
                                                                    int L, int Lpad, long long n_threads) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n_threads) return;
  const int r = static_cast<int>(t & 127);
  const long long rest = t >> 7;
  const int k8 = static_cast<int>(rest % (D / 8));  // 8-column group
  const long long zt = rest / (D / 8);               // (z, tile)
  const int tiles = Lpad / 128;
  const long long z = zt / tiles;
  const int i = static_cast<int>(zt % tiles) * 128 + r;
  if (i >= L) return;
  const float* src = dq_acc + dq_acc_offset<D>(z, Lpad, i, 8 * k8);
  const float4 a = *reinterpret_cast<const float4*>(src);
  const float4 bq = *reinterpret_cast<const float4*>(src + 512);
  const uint4 out = make_uint4(pack_bf16(a.x * scale, a.y * scale), pack_bf16(a.z * scale, a.w * scale),
                               pack_bf16(bq.x * scale, bq.y * scale), pack_bf16(bq.z * scale, bq.w * scale));
  *reinterpret_cast<uint4*>(dq + (static_cast<size_t>(z) * L + i) * D + 8 * k8) = out;
}

template <int D>
cudaError_t launch_bwd_pre_d(const BwdArgs& a, long long q_slices, long long kv_slices, cudaStream_t stream) {
  const long long rows = q_slices * a.Lpad;
  constexpr long long kRowsPerWarp = 4 * (32 / (D / 8));  // as in ring_attn_bwd_pre_kernel
  const long long warps = (rows + kRowsPerWarp - 1) / kRowsPerWarp;
  const unsigned pre_blocks = static_cast<unsigned>((warps * 32 + 255) / 256);
  if (a.timer) a.timer->mark(1, false, stream);
  ring_attn_bwd_pre_kernel<D><<<pre_blocks, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dO), a.lse, a.lse2, a.Dvec,
      a.dq_acc, a.dk_acc, a.dv_acc, a.L, a.Lpad, rows, kv_slices * a.Lpad);
  cudaError_t e = cudaGetLastError();
  if (a.timer) a.timer->mark(1, true, stream);
  return e;
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, cudaStream_t stream) {
  cudaError_t e;
  if (!a.step_nt) {
    e = launch_bwd_pre_d<D>(a, static_cast<long long>(a.B) * a.Hq, static_cast<long long>(a.B) * a.Hkv, stream);
    if (e != cudaSuccess) return e;
  }

  BwdDev p;
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.L = a.L; p.Lpad = a.Lpad; p.causal = a.causal;
  p.n_blocks = a.n_blocks;
  p.kv_accumulate = a.dk_acc != nullptr;
  p.scale = 1.0f / sqrtf(static_cast<float>(D));
  p.scale_log2 = p.scale * kLog2e;
  p.order = a.order; p.offsets = a.offsets; p.ranges = a.ranges;
  p.lse2 = a.lse2; p.dvec = a.Dvec; p.dq_acc = a.dq_acc;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.err = a.err;
  p.step_nt = a.step_nt; p.step = a.step; p.n_chunks = a.n_chunks; p.sched = a.sched;
  p.rank_lo = a.rank_lo; p.z_rank = a.z_rank;
  const size_t smem = sizeof(BwdSmem<D>);
  auto kernel = a.step_nt ? ring_attn_bwd_kernel<D, true> : ring_attn_bwd_kernel<D, false>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(a.n_blocks) * a.B * a.Hq);
  const int kind = a.step_nt ? 4 : 2;  // profiling kinds of include/ring_attn.h: ring step / backward main
  if (a.timer) a.timer->mark(kind, false, stream);
  kernel<<<grid, BwdCfg<D>::kThreads, smem, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dkacc, a.tm_dvacc, p);
  e = cudaGetLastError();
  if (a.timer) a.timer->mark(kind, true, stream);
  if (e != cudaSuccess || a.step_nt) return e;  // ring steps: the driver converts the gradients

  const long long nq8 = static_cast<long long>(a.B) * a.Hq * a.Lpad * D / 8;
  if (a.timer) a.timer->mark(3, false, stream);
  ring_attn_bwd_dq_post_kernel<D><<<static_cast<unsigned>((nq8 + 255) / 256), 256, 0, stream>>>(
      a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), p.scale, a.L, a.Lpad, nq8);
  if (p.kv_accumulate) {
    const long long kv8 = static_cast<long long>(a.B) * a.Hkv * a.L * D / 8;
    const unsigned blocks = static_cast<unsigned>((kv8 + 255) / 256);
    ring_attn_bwd_post_kernel<D><<<blocks, 256, 0, stream>>>(a.dk_acc, static_cast<__nv_bfloat16*>(a.dk), p.scale,
                                                             a.L, a.Lpad, kv8);
    ring_attn_bwd_post_kernel<D><<<blocks, 256, 0, stream>>>(a.dv_acc, static_cast<__nv_bfloat16*>(a.dv), 1.f, a.L,
                                                             a.Lpad, kv8);
  }
  e = cudaGetLastError();
  if (a.timer) a.timer->mark(3, true, stream);
  return e;
}

}  // namespace

size_t bwd_smem_bytes(int d) {
  return d == 128 ? sizeof(BwdSmem<128>) : sizeof(BwdSmem<64>);
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_bwd_d<128>(a, stream) : launch_bwd_d<64>(a, stream);
}

cudaError_t launch_bwd_dq_post(const BwdArgs& a, long long q_slices, cudaStream_t stream) {
  const float scale = 1.0f / sqrtf(static_cast<float>(a.d));
  const long long n8 = q_slices * a.Lpad * a.d / 8;
  const unsigned blocks = static_cast<unsigned>((n8 + 255) / 256);
  if (a.d == 128)
    ring_attn_bwd_dq_post_kernel<128><<<blocks, 256, 0, stream>>>(a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), scale,
                                                                   a.L, a.Lpad, n8);
  else
    ring_attn_bwd_dq_post_kernel<64><<<blocks, 256, 0, stream>>>(a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), scale,
                                                                  a.L, a.Lpad, n8);
  return cudaGetLastError();
}

cudaError_t launch_grad_to_bf16(const float* acc, void* out, float scale, long long n_elems, cudaStream_t stream) {
  // [n_elems / 128][128] rows of a plain fp32 accumulator (d = 128 columns a
  // row is only a view: the conversion is elementwise, 8 per thread)
  const long long n8 = n_elems / 8;
  const unsigned blocks = static_cast<unsigned>((n8 + 255) / 256);
  const int rows = static_cast<int>(n_elems / 128);
  ring_attn_bwd_post_kernel<128><<<blocks, 256, 0, stream>>>(acc, static_cast<__nv_bfloat16*>(out), scale, rows, rows,
                                                             n8);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const BwdArgs& a, long long q_slices, long long kv_slices, cudaStream_t stream) {
  return a.d == 128 ? launch_bwd_pre_d<128>(a, q_slices, kv_slices, stream)
                    : launch_bwd_pre_d<64>(a, q_slices, kv_slices, stream);
}

}  // namespace ra
