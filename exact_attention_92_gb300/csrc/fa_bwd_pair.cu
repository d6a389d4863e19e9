// dK/dV side of the backward pass for head dim 128 on sm_103a, run by CTA
// pairs ("FlashAttention V2 in depth", section 7.2: key/value tiles in the
// outer loop, dK_j and dV_j accumulated on chip).
//
// Why pairs.  A tcgen05 MMA with both operands in shared memory reads its
// A tile (128 rows x 16) and B tile (N rows x 16) at 128 bytes per clock:
// at N = 128 that is exactly the tensor rate, so the single-CTA kernel's
// S^T and dP^T products have no shared-memory bandwidth to spare for the
// tile copies landing at the same time (measured: an N = 64 product takes
// 48 cycles for 32 cycles of math, an N = 128 one 64).  With
// tcgen05.mma.cta_group::2 two CTAs on neighbouring SMs run one M = 256
// product: each supplies the A rows of its own 128 keys and half of B (the
// hardware splits B by its N dimension), and each gets its own 128 rows of
// the result in its own TMEM.  Per CTA the B reads halve, so the score
// products need 96 bytes per clock and the copies fit beside them.
//
// A unit is a pair of neighbouring 128-key tiles of one key/value head
// (CTA rank r owns key tile 2 tp + r) and walks the query tiles that see the
// first of them.  Per query tile (one step) the products are, with M = 256:
//   S^T = K Q^T     B = Q split by query row:  CTA r holds rows [64 r, 64 r + 64)
//   dP^T = V dO^T   B = dO split the same way
//   dV += P^T dO    B = dO split by head-dim column: CTA r holds columns
//   dK += dS^T Q    B = Q likewise                   [64 r, 64 r + 64)
// so each CTA keeps, per Q (dO) stage, its 64 rows of both 64-column chunks
// (16 KB) and its whole 64-column chunk (16 KB): 32 KB, the size of a full
// tile.  The element-wise work is the single-CTA kernel's (fa_bwd.cu): each
// CTA's eight element-wise warps turn their own TMEM rows of S^T and dP^T
// into P^T and dS^T.
//
// Roles per CTA (384 threads, registers split as in fa_bwd.cu): warp 9 loads
// this CTA's tiles, warps 0-7 do the element-wise work and the dK/dV
// write-out, warp 8 of CTA 0 (the leader) issues every MMA of the pair; warp
// 8 of CTA 1 only takes part in the pair's TMEM allocation.  Synchronisation
// across the pair:
//   * every tile copy of both CTAs completes on the leader's "full"
//     barrier (the leader expects the bytes of both);
//   * the leader's MMA commits arrive on the barrier of the same name in
//     both CTAs ("empty" barriers for the loaders, S^T / dP^T / dK,dV ready
//     for the element-wise warps);
//   * the element-wise warps of both CTAs arrive on the leader's s_free,
//     p_ready and dkv_empty barriers (16 warps each).
// Each CTA's own L and D values for a step sit in a small local ring.
#include <cuda_runtime.h>

#include <atomic>

#include "bwd_elementwise.cuh"
#include "sm103_pair.cuh"
#include "sm103_primitives.cuh"

namespace fa {

using namespace dev;

namespace pr {

constexpr int kD = 128;
constexpr int kChunk = kTileM * 128;        // 128 rows x 64 columns, bf16: 16 KB
constexpr int kHalf = 64 * 128;             // 64 rows x 64 columns: 8 KB
constexpr int kTile = 2 * kChunk;           // a K or V tile: 32 KB
constexpr int kStage = 2 * kHalf + kChunk;  // this CTA's part of a Q or dO tile: 32 KB
constexpr int kQStages = 3;
constexpr int kDoStages = 2;
constexpr int kRvStages = 2;
constexpr int kThreads = 384;
constexpr uint32_t kColDV = 256;
constexpr uint32_t kColDK = 384;
constexpr uint32_t kTmemCols = 512;
constexpr int kOffK = 0;
constexpr int kOffV = kTile;
constexpr int kOffQ = 2 * kTile;
constexpr int kOffDO = kOffQ + kQStages * kStage;
constexpr int kOffRv = kOffDO + kDoStages * kStage;  // kRvStages x (128 L, 128 D) floats
constexpr int kOffBar = kOffRv + kRvStages * 256 * 4;
constexpr int kNumBars = 4 + 2 * kQStages + 2 * kDoStages + 2 * kRvStages + 8 + 2 + 1;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory");
// Within a stage: [rows 64 r.. of chunk 0 | rows 64 r.. of chunk 1 | chunk r].
constexpr int kStageRows = 0;
constexpr int kStageCols = 2 * kHalf;

struct BwdRegs {
  static constexpr int kRegsCtl = 72;
  static constexpr int kRegsMath = 216;
  static_assert(128 * kRegsCtl + 256 * kRegsMath <= 384 * 168, "register split exceeds the launch");
};

struct PairUnit {
  int kvbh;   // key/value head
  int tp;     // key tiles 2 tp (rank 0) and 2 tp + 1 (rank 1)
  int first;  // first query tile that sees key tile 2 tp
  int per;    // query tiles per query head
  int count;  // steps: per x query heads of the group
};

// Pair units, low key tiles first (with the causal mask they are seen by
// the most query rows).
__device__ __forceinline__ PairUnit decode(const BwdParams& p, int u) {
  PairUnit w;
  const int BH = p.B * p.Hkv;
  w.kvbh = u % BH;
  w.tp = u / BH;
  const int first_row = 2 * w.tp * kTileN - p.causal_off;
  w.first = (p.causal && first_row > 0) ? first_row / kTileM : 0;
  w.per = p.num_q_tiles - w.first;
  w.count = w.per * p.group;
  return w;
}
__device__ __forceinline__ int num_pair_units(const BwdParams& p) { return p.B * p.Hkv * ((p.kv_tiles_used + 1) / 2); }

}  // namespace pr

template <bool GQA>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(384, 1)
    fa_bwd_dkdv_pair_kernel(const __grid_constant__ CUtensorMap tm_q64, const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_do64, const __grid_constant__ CUtensorMap tm_do,
                            const BwdParams p) {
  using namespace pr;
  using R = pr::BwdRegs;
  extern __shared__ __align__(1024) uint8_t smem[];
  // Both CTAs take the same path to every cluster barrier below.
  const bool aligned = (smem_u32(smem) & 1023u) == 0u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* k_full = bars;  // leader: K of both CTAs landed
  uint64_t* k_empty = bars + 1;
  uint64_t* v_full = bars + 2;
  uint64_t* v_empty = bars + 3;
  uint64_t* q_full = bars + 4;  // [kQStages]
  uint64_t* q_empty = q_full + kQStages;
  uint64_t* do_full = q_empty + kQStages;  // [kDoStages]
  uint64_t* do_empty = do_full + kDoStages;
  uint64_t* rv_full = do_empty + kDoStages;  // [kRvStages], local
  uint64_t* rv_empty = rv_full + kRvStages;
  uint64_t* s_full = rv_empty + kRvStages;  // [2] S^T of region r (both CTAs)
  uint64_t* dp_full = s_full + 2;           // [2] dP^T of region r (both CTAs)
  uint64_t* s_free = dp_full + 2;           // [2] leader: S^T read by all 16 element-wise warps
  uint64_t* p_ready = s_free + 2;           // [2] leader: P^T, dS^T packed by all 16
  uint64_t* dkv_full = p_ready + 2;         // both CTAs: the unit's dK, dV complete
  uint64_t* dkv_empty = dkv_full + 1;       // leader: ... read out by all 16
  uint64_t* drain = dkv_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  float* sRv = reinterpret_cast<float*>(smem + kOffRv);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cta_rank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    mbar_init(k_empty, 1);
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < kDoStages; ++s) {
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 1);
    }
    for (int s = 0; s < kRvStages; ++s) {
      mbar_init(&rv_full[s], 1);
      mbar_init(&rv_empty[s], 8);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&s_full[r], 1);
      mbar_init(&dp_full[r], 1);
      mbar_init(&s_free[r], 16);
      mbar_init(&p_ready[r], 16);
    }
    mbar_init(dkv_full, 1);
    mbar_init(dkv_empty, 16);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  if (warp == 9 && lane == 0) {
    tma_prefetch_desc(&tm_q64);
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do64);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{p.status, p.timeout_ns};
  if (!aligned && threadIdx.x == 0) atomicCAS(p.status, 0u, (unsigned int)FA_ERR_CUDA);
  const int n_units = aligned ? num_pair_units(p) : 0;
  const int G = (int)gridDim.x >> 1;

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    reg_dealloc<R::kRegsCtl>();
    // Launched while the D preprocess may still run: wait for it before
    // reading D, then let the dQ kernel (which needs nothing from this one)
    // take over SMs as this grid's CTAs finish.
    pdl_wait();
    pdl_trigger();
    const uint32_t k_full_l = at_leader(k_full), v_full_l = at_leader(v_full);
    uint32_t kc = 0, qc = 0;
    uint32_t k_issued = 0, v_issued = 0, q_issued = 0, do_issued = 0;  // copies started (for the drain)
    bool ok = true;
    for (int rnd = 0; ok && rnd * G < n_units; ++rnd) {
      const int u = pair_unit(rnd);
      if (u >= n_units) continue;
      const PairUnit w = decode(p, u);
      const int key0 = (2 * w.tp + (int)rank) * kTileN;
      ok = __all_sync(0xffffffffu, mbar_wait(k_empty, (kc & 1) ^ 1, ctl, kWaitBwdLoad));
      if (!ok) break;
      if (lane == 0) {
        if (leader) mbar_arrive_expect_tx(k_full, 2 * kTile);
        for (int c = 0; c < 2; ++c) tma_load_3d_pair(smem + kOffK + c * kChunk, &tm_k, k_full_l, c * 64, key0, w.kvbh);
      }
      ++k_issued;
      int qh = GQA ? q_head_of(w.kvbh, 0, p.H, p.Hkv) : w.kvbh;
      int qt = w.first;
      for (int ii = 0; ok && ii < w.count; ++ii, ++qc) {
        if constexpr (GQA) {
          if (ii > 0 && ++qt == w.first + w.per) {
            qt = w.first;
            ++qh;
          }
        } else {
          qt = w.first + ii;
        }
        const int row = qt * kTileM;
        const size_t head = (size_t)qh * p.Nq;
        // L and D of the step's 128 query rows, read before the waits below.
        float4 l4, d4;
        {
          float* lp = &l4.x;
          float* dp = &d4.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int qr = row + 4 * lane + e;
            lp[e] = qr < p.Nq ? p.lse[head + qr] : INFINITY;
            dp[e] = qr < p.Nq ? p.dvec[head + qr] : 0.f;
          }
        }
        // This CTA's part of Q_i: rows [64 r, 64 r + 64) of both chunks
        // (B of S^T) and chunk r (B of dK).
        const uint32_t sq = qc % kQStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&q_empty[sq], ((qc / kQStages) & 1) ^ 1, ctl, kWaitBwdLoad));
        if (!ok) break;
        if (lane == 0) {
          uint8_t* st = smem + kOffQ + sq * kStage;
          const uint32_t bar = at_leader(&q_full[sq]);
          if (leader) mbar_arrive_expect_tx(&q_full[sq], 2 * kStage);
          for (int c = 0; c < 2; ++c)
            tma_load_3d_pair(st + kStageRows + c * kHalf, &tm_q64, bar, c * 64, row + 64 * (int)rank, qh);
          tma_load_3d_pair(st + kStageCols, &tm_q, bar, 64 * (int)rank, row, qh);
        }
        ++q_issued;
        const uint32_t sd = qc % kDoStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&do_empty[sd], ((qc / kDoStages) & 1) ^ 1, ctl, kWaitBwdLoad));
        if (!ok) break;
        if (lane == 0) {
          uint8_t* st = smem + kOffDO + sd * kStage;
          const uint32_t bar = at_leader(&do_full[sd]);
          if (leader) mbar_arrive_expect_tx(&do_full[sd], 2 * kStage);
          for (int c = 0; c < 2; ++c)
            tma_load_3d_pair(st + kStageRows + c * kHalf, &tm_do64, bar, c * 64, row + 64 * (int)rank, qh);
          tma_load_3d_pair(st + kStageCols, &tm_do, bar, 64 * (int)rank, row, qh);
        }
        ++do_issued;
        if (ii == 0) {
          // V_j, needed by the first dP^T, after the first step's Q and dO.
          ok = __all_sync(0xffffffffu, mbar_wait(v_empty, (kc & 1) ^ 1, ctl, kWaitBwdLoad));
          if (!ok) break;
          if (lane == 0) {
            if (leader) mbar_arrive_expect_tx(v_full, 2 * kTile);
            for (int c = 0; c < 2; ++c)
              tma_load_3d_pair(smem + kOffV + c * kChunk, &tm_v, v_full_l, c * 64, key0, w.kvbh);
          }
          ++v_issued;
        }
        // The step's L (log2 units; rows past Nq and rows that see no key
        // get +inf so their weights vanish) and D, for this CTA's
        // element-wise warps.
        const uint32_t sr = qc % kRvStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&rv_empty[sr], ((qc / kRvStages) & 1) ^ 1, ctl, kWaitBwdLoad));
        if (!ok) break;
        {
          float* lp = &l4.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) lp[e] = lp[e] == -INFINITY ? INFINITY : lp[e] * 1.4426950408889634f;
          reinterpret_cast<float4*>(sRv + sr * 256)[lane] = l4;
          reinterpret_cast<float4*>(sRv + sr * 256 + 128)[lane] = d4;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rv_full[sr]);
      }
      ++kc;
    }
    if (lane == 0 && leader) {
      // Every copy of the pair has landed before either CTA can exit (the
      // leader's barriers count both CTAs' bytes; the final cluster barrier
      // holds the other CTA until then).
      if (k_issued > 0) mbar_wait(k_full, (k_issued - 1) & 1, ctl, kWaitDrain);
      if (v_issued > 0) mbar_wait(v_full, (v_issued - 1) & 1, ctl, kWaitDrain);
      for (uint32_t pos = q_issued > (uint32_t)kQStages ? q_issued - kQStages : 0u; pos < q_issued; ++pos)
        mbar_wait(&q_full[pos % kQStages], (pos / kQStages) & 1, ctl, kWaitDrain);
      for (uint32_t pos = do_issued > (uint32_t)kDoStages ? do_issued - kDoStages : 0u; pos < do_issued; ++pos)
        mbar_wait(&do_full[pos % kDoStages], (pos / kDoStages) & 1, ctl, kWaitDrain);
    }
    __syncwarp();
  } else if (warp == 8) {
    reg_dealloc<R::kRegsCtl>();
    if (leader) {
      // ------------------------------------------------------ MMA issuer
      // The single-CTA kernel's order (fa_bwd.cu): within step g
      //   dP^T(g), dK(g-1), S^T(g+1), [P^T(g), dS^T(g) ready] dV(g)
      // with pair MMAs.
      constexpr uint32_t id_s = idesc_bf16(256, kTileM, false, false);  // S^T, dP^T
      constexpr uint32_t id_kv = idesc_bf16(256, kD, false, true);      // dV, dK
      constexpr uint32_t hi = sdesc_hi(1024);
      const uint32_t k_lo = sdesc_lo(smem_u32(smem + kOffK), 16);
      const uint32_t v_lo = sdesc_lo(smem_u32(smem + kOffV), 16);
      auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, kWaitBwdMma));
      };
      auto wait_pair = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait_cl(bar, parity, ctl, kWaitBwdMma));
      };
      struct Cur {
        int rnd, ii, un;
        PairUnit w;
        bool valid;
      };
      auto seek = [&](Cur& c, int rnd, int un) {
        c.valid = false;
        for (; rnd * G < n_units; ++rnd) {
          const int u = pair_unit(rnd);
          if (u < n_units) {
            c.rnd = rnd;
            c.ii = 0;
            c.un = un;
            c.w = decode(p, u);
            c.valid = true;
            return;
          }
        }
      };
      auto advance = [&](Cur& c) {
        if (++c.ii >= c.w.count) seek(c, c.rnd + 1, c.un + 1);
      };
      auto q_st = [&](uint32_t g) { return smem_u32(smem + kOffQ + (g % kQStages) * kStage); };
      auto do_st = [&](uint32_t g) { return smem_u32(smem + kOffDO + (g % kDoStages) * kStage); };
      auto issue_s = [&](uint32_t g) {  // S^T(g) = K_j Q_i^T
        const uint32_t q_lo = sdesc_lo(q_st(g) + kStageRows, 16);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma2_ss(tmem + 128u * (g & 1), k_lo + (((kk / 4) * kChunk + (kk % 4) * 32) >> 4),
                  q_lo + (((kk / 4) * kHalf + (kk % 4) * 32) >> 4), hi, id_s, kk > 0 ? 1u : 0u);
        commit2(&s_full[g & 1]);
      };
      auto issue_dp = [&](uint32_t g) {  // dP^T(g) = V_j dO_i^T
        const uint32_t d_lo = sdesc_lo(do_st(g) + kStageRows, 16);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma2_ss(tmem + 128u * (g & 1), v_lo + (((kk / 4) * kChunk + (kk % 4) * 32) >> 4),
                  d_lo + (((kk / 4) * kHalf + (kk % 4) * 32) >> 4), hi, id_s, kk > 0 ? 1u : 0u);
        commit2(&dp_full[g & 1]);
      };
      auto issue_dv = [&](uint32_t g, bool acc) {  // dV += P^T dO_i (B read MN-major)
        const uint32_t b_lo = sdesc_lo(do_st(g) + kStageCols, kChunk);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk)
          mma2_ts(tmem + kColDV, tmem + 128u * (g & 1) + packed_col(kk, false), b_lo + ((kk * 2048) >> 4), hi,
                  id_kv, (acc || kk > 0) ? 1u : 0u);
        commit2(&do_empty[g % kDoStages]);  // dO_i: read by dP^T and dV
      };
      auto issue_dk = [&](uint32_t g, bool acc) {  // dK += dS^T Q_i
        const uint32_t b_lo = sdesc_lo(q_st(g) + kStageCols, kChunk);
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk)
          mma2_ts(tmem + kColDK, tmem + 128u * (g & 1) + packed_col(kk, true), b_lo + ((kk * 2048) >> 4), hi,
                  id_kv, (acc || kk > 0) ? 1u : 0u);
        commit2(&q_empty[g % kQStages]);  // Q_i: read by S^T and dK
      };
      bool ok = true;
      Cur cur, nxt;
      seek(cur, 0, 0);
      if (cur.valid) {
        ok = wait(k_full, 0) && wait(&q_full[0], 0);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          if (cur.w.count == 1) commit2(k_empty);  // K_j: read by S^T only
        }
      }
      nxt = cur;
      if (nxt.valid) advance(nxt);
      uint32_t g = 0;
      bool pend = false, pend_acc = false, pend_last = false;
      for (; ok && cur.valid; ++g) {
        const bool first = cur.ii == 0;
        auto dp_step = [&]() -> bool {
          if (first && !wait(v_full, cur.un & 1)) return false;
          if (!wait(&do_full[g % kDoStages], (g / kDoStages) & 1)) return false;
          if (!wait_pair(&s_free[g & 1], (g >> 1) & 1)) return false;
          tc_fence_after();
          issue_dp(g);
          if (cur.ii + 1 == cur.w.count) commit2(v_empty);  // V_j: read by dP^T only
          return true;
        };
        auto dk_prev = [&]() {
          if (!pend) return;
          issue_dk(g - 1, pend_acc);
          if (pend_last) commit2(dkv_full);
        };
        auto s_next = [&]() -> bool {
          if (!nxt.valid) return true;
          if (nxt.ii == 0 && !wait(k_full, nxt.un & 1)) return false;
          if (!wait(&q_full[(g + 1) % kQStages], ((g + 1) / kQStages) & 1)) return false;
          tc_fence_after();
          issue_s(g + 1);
          if (nxt.ii + 1 == nxt.w.count) commit2(k_empty);
          return true;
        };
        if (first) {
          dk_prev();
          ok = s_next() && dp_step();
        } else {
          ok = dp_step();
          if (ok) {
            dk_prev();
            ok = s_next();
          }
        }
        if (!ok) break;
        ok = wait_pair(&p_ready[g & 1], (g >> 1) & 1);
        if (ok && first && cur.un > 0) ok = wait_pair(dkv_empty, (cur.un - 1) & 1);
        if (!ok) break;
        tc_fence_after();
        issue_dv(g, !first);
        pend = true;
        pend_acc = !first;
        pend_last = cur.ii + 1 == cur.w.count;
        cur = nxt;
        if (nxt.valid) advance(nxt);
      }
      if (ok && pend) {
        issue_dk(g - 1, pend_acc);
        if (pend_last) commit2(dkv_full);
      }
      // Every MMA of the pair completes before either CTA releases TMEM.
      commit2(drain);
      (void)wait(drain, 0);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------ P^T, dS^T and dK/dV output
    reg_alloc<R::kRegsMath>();
    const int gq = warp & 3;   // TMEM lane quarter
    const int hc = warp >> 2;  // query-column half
    const uint32_t lane_off = (uint32_t)(32 * gq) << 16;
    const int r_key = 32 * gq + lane;
    const float sl2 = p.scale_log2;
    const uint32_t s_free_l0 = at_leader(&s_free[0]), s_free_l1 = at_leader(&s_free[1]);
    const uint32_t p_ready_l0 = at_leader(&p_ready[0]), p_ready_l1 = at_leader(&p_ready[1]);
    const uint32_t dkv_empty_l = at_leader(dkv_empty);
    uint32_t uc = 0, qc = 0;
    bool ok = true;
    // dK_j = scale * sum dS^T Q and dV_j = sum P^T dO of this CTA's key
    // tile; this warp writes head-dim columns [64 hc, 64 hc + 64), packed
    // and released from TMEM before the stores.
    auto write_dkdv = [&](int kr, size_t head) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(dkv_full, uc & 1, ctl, kWaitBwdSoftmax))) return false;
      ++uc;
      tc_fence_after();
      const int c0 = 64 * hc;
      uint32_t wv[2][32];
      tmem_read_pack<64>(tmem + lane_off + kColDV + c0, 1.f, wv[0]);
      tmem_read_pack<64>(tmem + lane_off + kColDK + c0, p.scale, wv[1]);
      tc_fence_before();
      arrive_leader_warp(dkv_empty_l);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(which ? p.dk : p.dv) + (head + kr) * kD + c0;
        store_rows<4>(reinterpret_cast<uint8_t*>(dst), (size_t)kD * 2, kr, p.Nk, wv[which], p.store32 != 0);
      }
      return true;
    };
    int pend_kr = -1;
    size_t pend_head = 0;
    for (int rnd = 0; ok && rnd * G < n_units; ++rnd) {
      const int u = pair_unit(rnd);
      if (u >= n_units) continue;
      const PairUnit w = decode(p, u);
      const int kr = (2 * w.tp + (int)rank) * kTileN + r_key;  // key index
      const size_t head = (size_t)w.kvbh * p.Nk;
      int qt = w.first;
      for (int ii = 0; ok && ii < w.count; ++ii, ++qc) {
        if constexpr (GQA) {
          if (ii > 0 && ++qt == w.first + w.per) qt = w.first;
        } else {
          qt = w.first + ii;
        }
        const int q0 = qt * kTileM;
        const uint32_t reg = qc & 1;
        const uint32_t tZ = tmem + lane_off + 128u * reg + 64 * hc;
        const uint32_t sr = qc % kRvStages;
        // P^T = exp2(S^T * scale * log2 e - L) over this warp's 64 query
        // columns; the S^T columns are released as soon as they are read.
        ok = __all_sync(0xffffffffu, mbar_wait(&rv_full[sr], (qc / kRvStages) & 1, ctl, kWaitBwdSoftmax));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&s_full[reg], (qc >> 1) & 1, ctl, kWaitBwdSoftmax));
        if (!ok) break;
        tc_fence_after();
        uint32_t pv[64];
        tmem_ld32(tZ, pv);
        tmem_ld32(tZ + 32, pv + 32);
        tmem_ld_wait<64>(pv);
        tc_fence_before();
        arrive_leader_warp(reg ? s_free_l1 : s_free_l0);
        {
          const float* bl = sRv + sr * 256 + 64 * hc;
          const int qf = q0 + 64 * hc;
          if ((kr >= p.Nk) || (p.causal && kr > qf + p.causal_off))
            p64_colL<true>(pv, bl, sl2, kr - p.causal_off, qf, kr >= p.Nk, p.causal != 0);
          else
            p64_colL<false>(pv, bl, sl2, kr, qf, false, false);
        }
        if (ii == 0 && pend_kr >= 0) {
          ok = write_dkdv(pend_kr, pend_head);
          if (!ok) break;
        }
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = pack_bf16(__uint_as_float(pv[2 * e]), __uint_as_float(pv[2 * e + 1]));
        // dS^T = P^T * (dP^T - D); P^T and dS^T packed over this warp's
        // dP^T columns of the region.
        ok = __all_sync(0xffffffffu, mbar_wait(&dp_full[reg], (qc >> 1) & 1, ctl, kWaitBwdSoftmax));
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t dpv[64];
          tmem_ld32(tZ, dpv);
          tmem_ld32(tZ + 32, dpv + 32);
          tmem_ld_wait<64>(dpv);
          const float* bd = sRv + sr * 256 + 128 + 64 * hc;
          uint32_t dk[32];
#pragma unroll
          for (int e4 = 0; e4 < 16; ++e4) {
            const float4 d4 = reinterpret_cast<const float4*>(bd)[e4];
            const float2 p01 = make_float2(__uint_as_float(pv[4 * e4]), __uint_as_float(pv[4 * e4 + 1]));
            const float2 p23 = make_float2(__uint_as_float(pv[4 * e4 + 2]), __uint_as_float(pv[4 * e4 + 3]));
            const float2 g01 = __fadd2_rn(
                make_float2(__uint_as_float(dpv[4 * e4]), __uint_as_float(dpv[4 * e4 + 1])), make_float2(-d4.x, -d4.y));
            const float2 g23 = __fadd2_rn(
                make_float2(__uint_as_float(dpv[4 * e4 + 2]), __uint_as_float(dpv[4 * e4 + 3])),
                make_float2(-d4.z, -d4.w));
            const float2 ds01 = __fmul2_rn(p01, g01);
            const float2 ds23 = __fmul2_rn(p23, g23);
            dk[2 * e4] = pack_bf16(ds01.x, ds01.y);
            dk[2 * e4 + 1] = pack_bf16(ds23.x, ds23.y);
          }
          tmem_st32(tZ, pk);
          tmem_st32(tZ + 32, dk);
        }
        tmem_st_wait();
        tc_fence_before();
        arrive_leader_warp(reg ? p_ready_l1 : p_ready_l0);
        mbar_arrive_warp(&rv_empty[sr]);  // the step's L and D were read
      }
      if (!ok) break;
      pend_kr = kr;
      pend_head = head;
    }
    if (ok && pend_kr >= 0) write_dkdv(pend_kr, pend_head);
  } else {
    reg_dealloc<R::kRegsCtl>();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the pair's MMAs, copies and remote arrivals are done
  if (warp == 8) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ------------------------------------------------------------------ launch

template <bool GQA>
static cudaError_t launch_pair_t(const CUtensorMap& tq64, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo64, const CUtensorMap& tdo,
                                 const BwdParams& p, int sm_count, cudaStream_t stream) {
  auto* kern = fa_bwd_dkdv_pair_kernel<GQA>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pr::kSmemBytes);
  if (e != cudaSuccess) return e;
  // Pairs resident at once (a pair needs two SMs of one cluster group),
  // asked once per device.
  constexpr int kMaxDevices = 64;
  static std::atomic<int> max_pairs[kMaxDevices];
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int mp = max_pairs[dev].load(std::memory_order_relaxed);
  if (mp == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)(sm_count / 2), 1, 1);
    cfg.blockDim = dim3(pr::kThreads, 1, 1);
    cfg.dynamicSmemBytes = pr::kSmemBytes;
    cfg.stream = stream;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    mp = n;
    max_pairs[dev].store(n, std::memory_order_relaxed);
  }
  const long long units = (long long)p.B * p.Hkv * ((p.kv_tiles_used + 1) / 2);
  const int pairs = (int)(units < mp ? units : mp);
  e = launch_pdl(kern, dim3(2 * pairs), dim3(pr::kThreads), pr::kSmemBytes, stream, tq64, tq, tk, tv, tdo64, tdo, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// dK, dV for head dim 128 by CTA pairs.  tq64 / tdo64: tensor maps of Q and
// dO with 64-row boxes; the others 128-row boxes.
cudaError_t launch_bwd_dkdv_pair(const CUtensorMap& tq64, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo64, const CUtensorMap& tdo,
                                 const BwdParams& p, int sm_count, cudaStream_t stream) {
  return p.Hkv != p.H ? launch_pair_t<true>(tq64, tq, tk, tv, tdo64, tdo, p, sm_count, stream)
                      : launch_pair_t<false>(tq64, tq, tk, tv, tdo64, tdo, p, sm_count, stream);
}

}  // namespace fa
