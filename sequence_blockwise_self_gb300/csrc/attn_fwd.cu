// attn_fwd.cu -- forward kernel of blockwise Ring Self-Attention on sm_103a.
//
// What it computes ("Large-scale distributed AI model training series:
// sequence parallelism", section 2.3 Ring Self-Attention, section 4.2 BPT
// and section 6.2 Ring Attention): for a block of query rows, the two
// products S = Q K^T and O = P V are formed tile by tile over the key/value
// tiles the block may see, visited in ring order (the host plan), and the
// softmax is corrected online with a running maximum and row sum, so the
// partial results of successive ring steps merge into exact attention.
//
// One CTA = one 256-row query block of one (batch, head): two 128-row query
// tiles that share every key/value tile.  Warp roles (384 threads):
//   warp 0      TMA producer: Q once, then K_j, V_j into a ring of slots
//   warp 1      tcgen05 issuer (converged warp, one elected lane issues):
//               S_t = Q_t K_j^T, O_t += P_t V_j
//   warp 2      tensor-memory allocator
//   warps 4-7   softmax of query tile 0 (one thread per row = TMEM lane)
//   warps 8-11  softmax of query tile 1
// Tensor memory (512 columns, fp32), d = 128: S_0 [0,128) S_1 [128,256)
// O_0 [256,384) O_1 [384,512).  P_t (bf16, two per 32-bit column) is
// written over the first 64 columns of S_t once the softmax has the scores
// in registers, and feeds O_t += P_t V as the tensor-memory A operand, so P
// never touches shared memory (whose bandwidth the two SS products nearly
// fill).  The next S_t is issued behind PV_t by the same thread; tcgen05
// MMAs from one thread execute in issue order, so it cannot overwrite P_t
// before PV_t has read it.  Issue order per key/value tile j (as in
// FlashAttention-4 style pipelines):
//   PV_0(j), S_0(j+1), PV_1(j), S_1(j+1)
// and one commit after each S_t(j+1) covers PV_t(j) as well, so when the
// softmax of tile t sees S_t(j+1) the accumulator O_t is quiescent and P_t
// may be overwritten.
//
// d = 64 leaves room for P_t in columns of its own (O_t [256 + 64t, ...),
// P_t [384 + 64t, ...)), so S_t(j+1) no longer has to wait for PV_t(j) to
// read P_t: once P_t(j) is written the issue order is
//   S_t(j+1), PV_t(j)
// and the softmax gets its next scores after one product instead of two;
// it writes P_t(j+1) once PV_t(j) has read P_t(j) (pv_done).  A 128-key
// tile is half the tensor work there for the same softmax work, so the
// softmax's wait for its next scores is what sets the pace.
//
// The running maximum is in log2 units; O and l are rescaled only when the
// maximum grew by more than 8 (a factor 256), which keeps the result exact
// while skipping most rescales.
#include <cfloat>
#include <climits>

#include "kernels.h"
#include "plan.h"
#include "sm103_ptx.cuh"

namespace ra {

namespace {

constexpr int kFwdThreads = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct FwdSmem {
  static constexpr int kSub = D / 64;                // 64-column sub-tiles per row
  static constexpr int kTile = 128 * D * 2;          // bytes of a Q, K or V tile
  static constexpr int kSlots = (D == 128) ? 5 : 10;  // key/value ring slots
  alignas(1024) uint8_t q[2][kTile];
  alignas(1024) uint8_t kv[kSlots][kTile];
  alignas(8) uint64_t q_full;
  alignas(8) uint64_t kv_full[kSlots];
  alignas(8) uint64_t kv_empty[kSlots];
  alignas(8) uint64_t s_full[2];
  alignas(8) uint64_t p_full[2];
  alignas(8) uint64_t pv_done[2];  // d = 64: PV_t has read P_t (and O_t is quiescent)
  alignas(8) uint64_t o_final[2];
  alignas(8) uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Tensor-memory columns.  d = 128: S_0 [0,128) S_1 [128,256) O_0 [256,384)
// O_1 [384,512), P_t over S_t's first 64 columns.  d = 64: S_0, S_1 as
// before, O_0 [256,320) O_1 [320,384) and P_0 [384,448) P_1 [448,512) of
// their own.
template <int D>
struct FwdTmem {
  static constexpr bool kSepP = D == 64;
  __host__ __device__ static constexpr uint32_t s(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t o(int t) { return kSepP ? 256u + 64u * t : 256u + 128u * t; }
  __host__ __device__ static constexpr uint32_t p(int t) { return kSepP ? 384u + 64u * t : 128u * t; }
};

struct FwdDev {
  int B, Hq, Hkv, L, causal;  // L: rows of one (batch, head) slice (step mode: the chunk length C)
  int n_blocks;               // work items per (batch, head) in this launch
  float scale_log2;
  const int32_t* order;
  const int32_t* offsets;
  const int32_t* ranges;
  float* lse;
  int* err;
  // Ring step mode (step_nb > 0): item k = 256-row block k % step_nb of the
  // block of worker w = rank_lo + k / step_nb at launch `step` of schedule
  // `sched` (schedule_pair: query chunk a, key/value chunk b).  Slice z of
  // q is a * z_rank * B*Hq + (b, h), of the output o, lse w * z_rank * B*Hq
  // + (b, h), of k, v b * z_rank * B*Hkv + (b, kv head): z_rank = 1 for
  // chunk-major buffers holding every chunk, 0 for buffers holding one.  The
  // output is the normalised partial result in fp32 (o32 / the fp32 map).
  int step_nb, step, rank_lo, n_chunks, sub_len, z_rank, sched;
  float* o32;
  // Ring step accumulating into the running result (acc_state != 0): o32
  // and lse hold the running fp32 (o, lse) of the block's query chunk (slice
  // q_z), read before the first key tile and overwritten with the merged
  // result; the online softmax simply continues from that state.
  int acc_state;
  // o token-major, [B][L][Hq][d] (tm_o is then 4-D: d, Hq, L, B), for the
  // blockwise transformer whose feed-forward takes token rows of Hq * d
  int o_tok;
};

// Keys of the causal mask: key column i of a tile is visible to a query
// row iff kv_key(tile) + i <= q_key(row).  Rows of the whole sequence use
// their positions.  In ring steps they are the rows' sequence positions:
// with the fold, sub-chunks `rank` and 2N-1-rank of sub_len rows (a tile
// never straddles the two); with contiguous chunks, rank * C + local.  With
// stripes (rank r owns r, r+N, ...), position src + N j <= r + N i  <=>
// j <= i - (src > r), so the keys are the local rows, the key tile's
// shifted by one when its rank is above the query's.
template <bool kStep>
__device__ __forceinline__ int q_key(const FwdDev& p, int rank, int local) {
  if (!kStep || !p.causal || p.sched == kSchedStriped) return local;
  if (p.sched != kSchedFold) return rank * p.L + local;
  return local < p.sub_len ? rank * p.sub_len + local
                           : (2 * p.n_chunks - 1 - rank) * p.sub_len + (local - p.sub_len);
}
template <bool kStep>
__device__ __forceinline__ int kv_key(const FwdDev& p, int kv_rank, int q_rank, int kv0) {
  if (!kStep || !p.causal) return kv0;
  if (p.sched == kSchedStriped) return kv0 + (kv_rank > q_rank ? 1 : 0);
  return q_key<kStep>(p, kv_rank, kv0);
}

// 4-D tiled TMA store (the token-major output map).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

// Wait that ignores the abort flag (used to drain in-flight copies/MMAs
// after an abort), still bounded in time.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, int* err) {
  int local = 0;
  mbar_wait(bar, parity, &local, err, kSiteFwdDrain);
}

template <int D>
__device__ void fwd_producer(FwdSmem<D>& sm, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                             const CUtensorMap* tm_v, int q0, int q_z, int kv_z, const int32_t* rg, int nr,
                             volatile int* ab, int* err) {
  using S = FwdSmem<D>;
  const uint32_t qbar = smem_u32(&sm.q_full);
  mbar_arrive_expect_tx(qbar, 2 * S::kTile);
  for (int t = 0; t < 2; ++t)
    for (int sub = 0; sub < S::kSub; ++sub)
      tma_load_3d(smem_u32(sm.q[t]) + sub * 16384, tm_q, qbar, sub * 64, q0 + 128 * t, q_z);
  uint32_t n = 0;
  bool ok = true;
  for (int ri = 0; ri < nr && ok; ++ri) {
    for (int jt = rg[2 * ri]; jt < rg[2 * ri + 1] && ok; ++jt) {
      for (int sel = 0; sel < 2 && ok; ++sel) {
        const uint32_t slot = n % S::kSlots, use = n / S::kSlots;
        if (use > 0) ok = mbar_wait(smem_u32(&sm.kv_empty[slot]), (use - 1) & 1, ab, err, kSiteFwdProducer);
        if (!ok) break;
        const uint32_t fb = smem_u32(&sm.kv_full[slot]);
        mbar_arrive_expect_tx(fb, S::kTile);
        const CUtensorMap* m = sel ? tm_v : tm_k;
        for (int sub = 0; sub < S::kSub; ++sub)
          tma_load_3d(smem_u32(sm.kv[slot]) + sub * 16384, m, fb, sub * 64, jt * 128, kv_z);
        ++n;
      }
    }
  }
  if (!ok) {
    // Let every copy this thread issued land before the CTA exits.
    wait_drain(qbar, 0, err);
    for (uint32_t i = 0; i < S::kSlots && i < n; ++i) {
      const uint32_t last = i + S::kSlots * ((n - 1 - i) / S::kSlots);
      wait_drain(smem_u32(&sm.kv_full[i]), (last / S::kSlots) & 1, err);
    }
  }
}

template <int D>
__device__ void fwd_mma(FwdSmem<D>& sm, uint32_t tmem, int nkv, bool o_preloaded, volatile int* ab, int* err) {
  using S = FwdSmem<D>;
  using TM = FwdTmem<D>;
  constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
  constexpr uint32_t kIdO = idesc_bf16(128, D, false, true);
  const uint32_t total_uses = 2u * nkv;

  auto issue_s = [&](int t, uint32_t kslot) {
    const uint32_t qa = smem_u32(sm.q[t]), ka = smem_u32(sm.kv[kslot]);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
      umma_ss_warp(tmem + TM::s(t), sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), kIdS,
                   kk > 0);
    }
  };
  auto issue_pv = [&](int t, uint32_t vslot, bool acc) {
    const uint32_t va = smem_u32(sm.kv[vslot]);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)  // A = P_t packed two bf16 per column: 8 columns per 16 keys
      umma_ts_warp(tmem + TM::o(t), tmem + TM::p(t) + 8 * kk, sdesc_sw128(va + kk * 2048, 16384, 1024), kIdO,
                   (acc || kk > 0) ? 1u : 0u);
  };
  // Load n of the producer's sequence (K_0, V_0, K_1, V_1, ...) sits in slot
  // n % kSlots, filled for the (n / kSlots)-th time.
  auto wait_load = [&](uint32_t n) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.kv_full[n % S::kSlots]), (n / S::kSlots) & 1, ab, err,
                                             kSiteFwdMma));
  };
  // Release a slot only if the producer will refill it: every commit is
  // then awaited by someone before the CTA exits.
  auto release = [&](uint32_t n) {
    if (n + S::kSlots < total_uses) umma_commit_warp(smem_u32(&sm.kv_empty[n % S::kSlots]));
  };

  // The loads a tile needs are awaited at the end of the previous tile, while
  // the softmax still runs: an mbarrier wait costs this warp a few hundred
  // cycles beside the softmax warps, which the tensor pipe should not idle
  // through.
  bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.q_full), 0, ab, err, kSiteFwdMma));
  if (ok) ok = wait_load(0);
  if (ok) {
    tc_fence_after();
    issue_s(0, 0);
    umma_commit_warp(smem_u32(&sm.s_full[0]));
    issue_s(1, 0);
    umma_commit_warp(smem_u32(&sm.s_full[1]));
    release(0);
  }
  if (ok) ok = wait_load(1);
  if (ok && nkv > 1) ok = wait_load(2);
  for (int j = 0; j < nkv && ok; ++j) {
    const uint32_t nk = 2u * (j + 1), nv = 2u * j + 1;
    const bool has_next = j + 1 < nkv;
    for (int t = 0; t < 2 && ok; ++t) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.p_full[t]), j & 1, ab, err, kSiteFwdMma));
      if (!ok) break;
      tc_fence_after();
      if constexpr (TM::kSepP) {
        // S_t(j+1) first (the softmax's next scores), then PV_t(j)
        if (has_next) {
          issue_s(t, nk % S::kSlots);
          umma_commit_warp(smem_u32(&sm.s_full[t]));
        }
        issue_pv(t, nv % S::kSlots, j > 0 || o_preloaded);
        umma_commit_warp(smem_u32(has_next ? &sm.pv_done[t] : &sm.o_final[t]));
      } else {
        // PV_t(j), then S_t(j+1) over P_t; the commit covers both
        issue_pv(t, nv % S::kSlots, j > 0 || o_preloaded);
        if (has_next) {
          issue_s(t, nk % S::kSlots);
          umma_commit_warp(smem_u32(&sm.s_full[t]));
        } else {
          umma_commit_warp(smem_u32(&sm.o_final[t]));
        }
      }
    }
    if (!ok) break;
    if (has_next) release(nk);
    release(nv);
    if (j + 2 < nkv) {  // V(j+1), K(j+2)
      const uint32_t a = nv + 2, b = nk + 2;
      ok = __all_sync(0xffffffffu, mbar_wait2(smem_u32(&sm.kv_full[a % S::kSlots]), (a / S::kSlots) & 1,
                                              smem_u32(&sm.kv_full[b % S::kSlots]), (b / S::kSlots) & 1, ab, err,
                                              kSiteFwdMma));
    } else if (j + 1 < nkv) {
      ok = wait_load(nv + 2);
    }
  }
  if (!ok) {
    umma_commit_warp(smem_u32(&sm.drain));
    wait_drain(smem_u32(&sm.drain), 0, err);
  }
}

template <int D, bool kStep>
__device__ void fwd_softmax(FwdSmem<D>& sm, uint32_t tmem, int t, const FwdDev& p, const CUtensorMap* tm_o,
                            int q0, int out_z, int q_rank, int kv_rank, const int32_t* rg, int nr,
                            volatile int* ab, int* err) {
  const int wq = (threadIdx.x >> 5) & 3;  // TMEM lane quadrant of this warp
  const int lane = threadIdx.x & 31;
  const int row = wq * 32 + lane;
  const int qpos = q0 + 128 * t + row;        // row of the slice
  const int qseq = q_key<kStep>(p, q_rank, qpos);  // its key for the causal mask
  using TM = FwdTmem<D>;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t t_s = tmem + TM::s(t) + lane_off;
  const uint32_t t_o = tmem + TM::o(t) + lane_off;
  const uint32_t t_p = tmem + TM::p(t) + lane_off;
  const float c = p.scale_log2;
  float m = -INFINITY, l = 0.f;
  if (kStep && p.acc_state) {
    // Continue from the running result (o_run, lse_run) of this row: the
    // state m = lse_run log2(e), l = 1, O = o_run has exactly that
    // normalised output and log-sum-exp; an empty row (lse_run = -inf)
    // starts from m = -inf, l = 0, O = 0.  O goes to tensor memory before
    // this thread's first p_full arrival, which orders it before PV_t(0).
    const size_t rrow = static_cast<size_t>(out_z) * p.L + qpos;
    const float lrun = qpos < p.L ? p.lse[rrow] : -INFINITY;
    const bool live = lrun != -INFINITY;
    if (live) {
      m = lrun * kLog2e;
      l = 1.f;
    }
    const float4* src = reinterpret_cast<const float4*>(p.o32 + rrow * D);
#pragma unroll
    for (int c0 = 0; c0 < D / 32; ++c0) {
      uint32_t r[32];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const float4 v = live ? src[c0 * 8 + x] : make_float4(0.f, 0.f, 0.f, 0.f);
        r[4 * x] = __float_as_uint(v.x);
        r[4 * x + 1] = __float_as_uint(v.y);
        r[4 * x + 2] = __float_as_uint(v.z);
        r[4 * x + 3] = __float_as_uint(v.w);
      }
      tmem_st32_async(t_o + c0 * 32, r);
    }
    tmem_wait_st();
  }
  bool ok = true;
  int j = 0;
  for (int ri = 0; ri < nr && ok; ++ri) {
    for (int jt = rg[2 * ri]; jt < rg[2 * ri + 1]; ++jt, ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full[t]), j & 1, ab, err, kSiteFwdSoftmax));
      if (!ok) break;
      tc_fence_after();
      // one batched load of the 128 scores of this row, one wait
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld32_async(t_s, r0);
      tmem_ld32_async(t_s + 32, r1);
      tmem_ld32_async(t_s + 64, r2);
      tmem_ld32_async(t_s + 96, r3);
      tmem_wait_ld(r0);
      reg_fence(r1);
      reg_fence(r2);
      reg_fence(r3);
      float s[128];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = __uint_as_float(r0[i]);
        s[32 + i] = __uint_as_float(r1[i]);
        s[64 + i] = __uint_as_float(r2[i]);
        s[96 + i] = __uint_as_float(r3[i]);
      }
      const int kv0 = jt * 128;
      const int kvseq = kv_key<kStep>(p, kv_rank, q_rank, kv0);
      if (kv0 + 128 > p.L || (p.causal && kvseq + 127 > qseq)) {
        const int lim = min(p.L - 1 - kv0, p.causal ? qseq - kvseq : INT_MAX);  // valid columns: i <= lim
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i > lim) s[i] = -INFINITY;
      }
      // four independent max3 chains over s[0..127]: 4 seeds + 15 groups of 8 + 4
      float m0 = s[0], m1 = s[1], m2 = s[2], m3 = s[3];
#pragma unroll
      for (int i = 4; i < 124; i += 8) {
        m0 = max3f(m0, s[i], s[i + 1]);
        m1 = max3f(m1, s[i + 2], s[i + 3]);
        m2 = max3f(m2, s[i + 4], s[i + 5]);
        m3 = max3f(m3, s[i + 6], s[i + 7]);
      }
      m0 = max3f(m0, s[124], s[125]);
      m1 = max3f(m1, s[126], s[127]);
      const float mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
      const float m_new = fmaxf(m, mx * c);
      const bool resc = m_new > m + kRescaleThreshold;
      const float m_old = m;
      if (resc) {
        l *= ex2(m - m_new);
        m = m_new;
      }
      const float ms = (m == -INFINITY) ? 0.f : m;
      const float2 c2 = make_float2(c, c), nm2 = make_float2(-ms, -ms);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      // Rare: the row maximum grew by more than the threshold, so the O_t
      // accumulated so far is rescaled to the new reference (O_t quiescent)
      auto rescale_o = [&] {
        if ((j > 0 || (kStep && p.acc_state)) && __any_sync(0xffffffffu, resc)) {
          const float f = resc ? ex2(m_old - m) : 1.f;
#pragma unroll
          for (int c0 = 0; c0 < D / 32; ++c0) {
            uint32_t r[32];
            tmem_ld32(t_o + c0 * 32, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
            tmem_st32(t_o + c0 * 32, r);
          }
        }
      };
      // P in quarters; each quarter goes to tensor memory (two bf16 per
      // column) as soon as it is packed.  d = 128: over S_t's first 64
      // columns, and O_t is quiescent here (the commit that signalled S_t(j)
      // covers PV_t(j-1)).  d = 64: to P_t's own columns once PV_t(j-1) has
      // read them (which also leaves O_t quiescent), awaited after the first
      // quarter's exponentials.  PV_t(j) is only issued after this thread
      // arrives on p_full.
#pragma unroll
      for (int half = 0; half < 4; ++half) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 32 * half; i < 32 * half + 32; i += 4) {
          const float2 x0 = __ffma2_rn(make_float2(s[i], s[i + 1]), c2, nm2);
          const float2 x1 = __ffma2_rn(make_float2(s[i + 2], s[i + 3]), c2, nm2);
          const float p0 = ex2(x0.x), p1 = ex2(x0.y), p2 = ex2(x1.x), p3 = ex2(x1.y);
          acc0 = __fadd2_rn(acc0, make_float2(p0, p1));
          acc1 = __fadd2_rn(acc1, make_float2(p2, p3));
          pk[(i - 32 * half) / 2] = pack_bf16(p0, p1);
          pk[(i - 32 * half) / 2 + 1] = pack_bf16(p2, p3);
        }
        if (TM::kSepP && half == 0 && j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.pv_done[t]), (j - 1) & 1, ab, err, kSiteFwdSoftmax));
          if (!ok) break;
          tc_fence_after();
        }
        tmem_st16_async(t_p + 16 * half, pk);
      }
      if (!ok) break;
      l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
      rescale_o();
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.p_full[t]));
    }
  }
  // Output staging: a key/value slot that neither of the last two loads (K
  // and V of the last tile, which the other tile's final PV may still read)
  // occupies; every earlier load was consumed before o_final.
  const uint32_t last_v = (2u * static_cast<uint32_t>(j) - 1u) % FwdSmem<D>::kSlots;  // j == tiles visited
  const uint32_t pbase = smem_u32(sm.kv[(last_v + 1 + t) % FwdSmem<D>::kSlots]);
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.o_final[t]), 0, ab, err, kSiteFwdEpilogue));
  if (ok) {
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    if constexpr (kStep) {
      // Ring step: the normalised partial O row in fp32, as 32-column boxes
      // of 128-byte rows: boxes 0 .. d/64-1 in the dead Q_t buffer, the rest
      // in the free key/value slot (Q_t was last read by S_t(last), which
      // o_final covers).
      const uint32_t qbase = smem_u32(sm.q[t]);
#pragma unroll
      for (int c0 = 0; c0 < D / 32; ++c0) {
        uint32_t r[32];
        tmem_ld32(t_o + c0 * 32, r);
        const uint32_t box = (c0 < D / 64 ? qbase + c0 * 16384 : pbase + (c0 - D / 64) * 16384);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          st_shared_v4(box + sw128_offset(row, ch), __float_as_uint(__uint_as_float(r[4 * ch]) * inv),
                       __float_as_uint(__uint_as_float(r[4 * ch + 1]) * inv),
                       __float_as_uint(__uint_as_float(r[4 * ch + 2]) * inv),
                       __float_as_uint(__uint_as_float(r[4 * ch + 3]) * inv));
      }
    } else {
      // Normalised O row -> bf16 -> the staging slot (see above), laid out as
      // the 128-byte-swizzled boxes of the output tensor map.
      auto emit = [&](int c0, const uint32_t (&r)[32]) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int ch = c0 * 4 + q4;
          const float* f = reinterpret_cast<const float*>(r) + q4 * 8;
          st_shared_v4(pbase + (ch >> 3) * 16384 + sw128_offset(row, ch & 7), pack_bf16(f[0] * inv, f[1] * inv),
                       pack_bf16(f[2] * inv, f[3] * inv), pack_bf16(f[4] * inv, f[5] * inv),
                       pack_bf16(f[6] * inv, f[7] * inv));
        }
      };
      {
        uint32_t r0[32], r1[32];
        tmem_ld32_async(t_o, r0);
        tmem_ld32_async(t_o + 32, r1);
        tmem_wait_ld(r0);
        reg_fence(r1);
        emit(0, r0);
        emit(1, r1);
      }
      if (D == 128) {
        uint32_t r2[32], r3[32];
        tmem_ld32_async(t_o + 64, r2);
        tmem_ld32_async(t_o + 96, r3);
        tmem_wait_ld(r2);
        reg_fence(r3);
        emit(2, r2);
        emit(3, r3);
      }
    }
    if (qpos < p.L) p.lse[static_cast<size_t>(out_z) * p.L + qpos] = (m + log2f(l)) * kLn2;
    fence_proxy_async_smem();
  }
  tc_fence_before();
  named_bar_sync(1 + t, 128);
  if (ok && row == 0 && q0 + 128 * t < p.L) {  // no store for a tile wholly past the end
    if constexpr (kStep) {
      for (int c0 = 0; c0 < D / 32; ++c0)
        tma_store_3d(tm_o, c0 < D / 64 ? smem_u32(sm.q[t]) + c0 * 16384 : pbase + (c0 - D / 64) * 16384, 32 * c0,
                     q0 + 128 * t, out_z);
    } else {
      for (int sub = 0; sub < FwdSmem<D>::kSub; ++sub) {
        if (p.o_tok)  // box (64 columns, 1 head, 128 rows, 1 batch): clipped at this batch's L
          tma_store_4d(tm_o, pbase + sub * 16384, sub * 64, out_z % p.Hq, q0 + 128 * t, out_z / p.Hq);
        else
          tma_store_3d(tm_o, pbase + sub * 16384, sub * 64, q0 + 128 * t, out_z);
      }
    }
    bulk_commit_group();
    bulk_wait_group<0>();
  }
}

template <int D, bool kStep>
__global__ void __launch_bounds__(kFwdThreads, 1)
    ring_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                         const FwdDev p) {
  using S = FwdSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kSiteFwdMisaligned);
    return;
  }
  S& sm = *reinterpret_cast<S*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTAs kv group by kv group: within the group of (batch, kv head), the
  // plan's items in its order (longest first), each for the group's G query
  // heads side by side -- the CTAs running together read the keys and values
  // of one kv head (which stay in L2), each tile by G CTAs at about the same
  // time
  const int BH = p.B * p.Hq;
  const int G = p.Hq / p.Hkv;
  const int per_group = p.n_blocks * G;
  const int gz = blockIdx.x / per_group;  // b * Hkv + kv head
  const int rem = blockIdx.x % per_group;
  const int item = p.order[rem / G];
  const int bh = (gz / p.Hkv) * p.Hq + (gz % p.Hkv) * G + rem % G;
  const int b = bh / p.Hq, h = bh % p.Hq;
  int u = item, q_rank = 0, kv_rank = 0;
  int q_z = bh, out_z = bh, kv_z = b * p.Hkv + h / (p.Hq / p.Hkv);
  if constexpr (kStep) {
    const int worker = p.rank_lo + item / p.step_nb;
    u = item % p.step_nb;
    schedule_pair(p.n_chunks, p.sched, p.step, worker, &q_rank, &kv_rank);
    q_z += q_rank * p.z_rank * BH;
    // a partial result goes to the worker's slot; the running result is the
    // query chunk's own
    out_z += (p.acc_state ? q_rank : worker) * p.z_rank * BH;
    kv_z += kv_rank * p.z_rank * (p.B * p.Hkv);
  }
  const int q0 = u * 256;
  const int32_t* rg = p.ranges + 2 * p.offsets[item];
  const int nr = p.offsets[item + 1] - p.offsets[item];
  int nkv = 0;
  for (int ri = 0; ri < nr; ++ri) nkv += rg[2 * ri + 1] - rg[2 * ri];
  volatile int* ab = &sm.abort_flag;

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(smem_u32(&sm.q_full), 1);
    for (int i = 0; i < S::kSlots; ++i) {
      mbar_init(smem_u32(&sm.kv_full[i]), 1);
      mbar_init(smem_u32(&sm.kv_empty[i]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&sm.s_full[t]), 1);
      mbar_init(smem_u32(&sm.p_full[t]), 128);
      mbar_init(smem_u32(&sm.pv_done[t]), 1);
      mbar_init(smem_u32(&sm.o_final[t]), 1);
    }
    mbar_init(smem_u32(&sm.drain), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (kStep && nkv == 0) {
    // A ring-step block that sees none of the source's keys (causal): its
    // partial result is the merge's neutral element, o = 0, lse = -inf (a
    // running result stays as it is).
    if (warp >= 4 && !p.acc_state) {
      const int qpos = q0 + 128 * ((warp - 4) >> 2) + (threadIdx.x & 127);
      if (qpos < p.L) {
        float4* dst = reinterpret_cast<float4*>(p.o32 + (static_cast<size_t>(out_z) * p.L + qpos) * D);
#pragma unroll 4
        for (int x = 0; x < D / 4; ++x) dst[x] = make_float4(0.f, 0.f, 0.f, 0.f);
        p.lse[static_cast<size_t>(out_z) * p.L + qpos] = -INFINITY;
      }
    }
  } else if (warp == 0) {
    if (lane == 0) fwd_producer<D>(sm, &tm_q, &tm_k, &tm_v, q0, q_z, kv_z, rg, nr, ab, p.err);
  } else if (warp == 1) {
    // the whole warp runs the issue loop; one elected lane issues
    fwd_mma<D>(sm, tmem, nkv, kStep && p.acc_state, ab, p.err);
  } else if (warp >= 4) {
    fwd_softmax<D, kStep>(sm, tmem, (warp - 4) >> 2, p, &tm_o, q0, out_z, q_rank, kv_rank, rg, nr, ab, p.err);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, 512);
}

}  // namespace

// Failure-detection self-test: one warp waits on an mbarrier that nothing
// will ever arrive at.  The bounded wait gives up after timeout_ns, raises
// the abort flag and records kSiteSelfTest in the status word, exactly as a
// lost arrival in the attention kernels would; the kernel then returns
// normally, leaving the context usable.
__global__ void ring_attn_selftest_wait_kernel(int* err, unsigned long long timeout_ns) {
  __shared__ alignas(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = mbar_wait(smem_u32(&bar), 0, &abort_flag, err, kSiteSelfTest, timeout_ns);
  if (ok && threadIdx.x == 0) atomicCAS(err, 0, -1);  // cannot happen: nothing arrives
}

cudaError_t launch_selftest_wait(int* err, unsigned long long timeout_ns, cudaStream_t stream) {
  ring_attn_selftest_wait_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
  return cudaGetLastError();
}

size_t fwd_smem_bytes(int d) {
  return d == 128 ? sizeof(FwdSmem<128>) : sizeof(FwdSmem<64>);
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  FwdDev p;
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.L = a.L; p.causal = a.causal;
  p.n_blocks = a.n_blocks;
  p.scale_log2 = kLog2e / sqrtf(static_cast<float>(a.d));
  p.order = a.order; p.offsets = a.offsets; p.ranges = a.ranges;
  p.lse = a.lse; p.err = a.err;
  p.step_nb = a.step_nb; p.step = a.step; p.rank_lo = a.rank_lo; p.n_chunks = a.n_chunks;
  p.sub_len = a.sub_len; p.z_rank = a.z_rank; p.sched = a.sched; p.o32 = a.o32; p.acc_state = a.acc_state;
  p.o_tok = a.o_token_major;
  const size_t smem = fwd_smem_bytes(a.d);
  const dim3 grid(static_cast<unsigned>(a.n_blocks) * a.B * a.Hq);
  cudaError_t e;
  auto kernel = a.step_nb ? (a.d == 128 ? ring_attn_fwd_kernel<128, true> : ring_attn_fwd_kernel<64, true>)
                          : (a.d == 128 ? ring_attn_fwd_kernel<128, false> : ring_attn_fwd_kernel<64, false>);
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int kind = a.step_nb ? 4 : 0;  // profiling kinds of include/ring_attn.h: forward / ring step
  if (a.timer) a.timer->mark(kind, false, stream);
  kernel<<<grid, kFwdThreads, smem, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, p);
  e = cudaGetLastError();
  if (a.timer) a.timer->mark(kind, true, stream);
  return e;
}

}  // namespace ra
