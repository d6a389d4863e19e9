// Backward pass of exact attention for head dim 256 on sm_103a
// ("FlashAttention V2 in depth", section 7).
//
// At d = 256 the dK and dV accumulators of one 128-key tile would take all
// 512 TMEM columns, leaving none for S^T and dP^T.  The key/value side
// therefore runs as two passes of one kernel over the same units (one
// 128-key tile of a key/value head, the query tiles that see it in steps of
// 64 rows):
//   fa_bwd256_kv_kernel<false>  dV += P^T dO            (S^T = K Q^T)
//   fa_bwd256_kv_kernel<true>   dK += dS^T Q, scaled     (S^T, dP^T = V dO^T)
// which executes S^T twice: 5 products for the 4 of the method (80%).
//   fa_bwd256_dq_kernel         dQ += dS K, scaled, per 128-row query tile,
//                               keys in steps of 64 (S, dP recomputed).
// D = rowsum(dO * O) comes from fa_bwd_preprocess (fa_bwd.cu).
//
// Roles (192 threads): warp 5 loads (TMA; in the key/value kernel the whole
// warp also writes the L and D values of a query step into a small ring),
// warp 4 issues the tcgen05
// products (whole warp, one elected lane), warps 0-3 do the element-wise
// work, one TMEM lane (a key row, or a query row in the dQ kernel) per
// thread and 64 columns per step, and read the accumulator out at the end of
// a unit.  TMEM: two regions of 128 columns (step g uses region g & 1:
// S or S^T in its first 64 columns, dP or dP^T in the next 64; the packed
// bf16 P^T / dS^T / dS go back over columns the same thread has read) and
// the 256-column accumulator from column 256.  The issuer runs, for step g,
// the products that fill region g & 1, then the accumulation of step g - 1
// (once its packed operand is in TMEM), so the tensor core computes step
// g's scores while the element-wise warps work on step g - 1.  The
// accumulator of a unit is read out after the next unit's first element-wise
// step; the next unit's first accumulation waits for that.
//
// Queries and keys may differ in length and take a causal offset, and
// key/value heads may be shared (grouped-query attention), as in fa_bwd.cu.
#include <cuda_runtime.h>

#include "bwd_elementwise.cuh"
#include "sm103_primitives.cuh"

namespace fa {

using namespace dev;

namespace b256 {

constexpr int kD = 256;
constexpr int kStep = 64;                     // query rows (kv kernel) / keys (dq kernel) per step
constexpr int kBig = 128;                     // keys (kv kernel) / queries (dq kernel) per unit
constexpr int kChunkBig = kBig * 128;         // 128 rows x 64 columns, bf16
constexpr int kChunkStep = kStep * 128;       // 64 rows x 64 columns
constexpr int kBigBytes = 4 * kChunkBig;      // 64 KB
constexpr int kStepBytes = 4 * kChunkStep;    // 32 KB
constexpr int kThreads = 192;
constexpr uint32_t kColAcc = 256;
constexpr uint32_t kTmemCols = 512;

// Shared-memory plan of the key/value kernel: K (and V for the dK pass)
// for the whole unit, Q and dO per query step, and the step's L and D
// values in a ring of their own (a tile is released when its last product
// has read it, the values when the element-wise warps have).
template <bool DK>
struct KvCfg {
  static constexpr int kQStages = 2;
  static constexpr int kDoStages = DK ? 1 : 2;
  static constexpr int kRvStages = 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kBigBytes;
  static constexpr int kOffQ = DK ? 2 * kBigBytes : kBigBytes;
  static constexpr int kOffDO = kOffQ + kQStages * kStepBytes;
  static constexpr int kOffRv = kOffDO + kDoStages * kStepBytes;  // kRvStages x (64 L + 64 D) floats
  static constexpr int kOffBar = kOffRv + kRvStages * 2 * kStep * 4;
  static constexpr int kNumBars = 4 + 2 * kQStages + 2 * kDoStages + 2 * kRvStages + 2 + 2 + 2 + 2 + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
  static_assert(kSmemBytes <= 232448, "shared memory");
};

// Shared-memory plan of the dQ kernel: Q and dO for the whole unit, K and V
// per key step.
struct DqCfg {
  static constexpr int kKStages = 2;  // K is read by S (early) and dQ (late)
  static constexpr int kVStages = 1;  // V only by dP
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kBigBytes;
  static constexpr int kOffK = 2 * kBigBytes;
  static constexpr int kOffV = kOffK + kKStages * kStepBytes;
  static constexpr int kOffBar = kOffV + kVStages * kStepBytes;
  static constexpr int kNumBars = 4 + 2 * kKStages + 2 * kVStages + 2 + 2 + 2 + 2 + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
  static_assert(kSmemBytes <= 232448, "shared memory");
};

struct KvUnit {
  int kvbh;   // key/value head
  int t;      // 128-key tile
  int first;  // first 64-row query tile that sees the key tile
  int per;    // query tiles per query head
  int count;  // steps: per x query heads of the group
};

// Key/value units, low key tiles first (with the causal mask they are seen
// by the most query rows).  The host lists only key tiles some row sees.
__device__ __forceinline__ KvUnit decode_kv(const BwdParams& p, int u) {
  KvUnit w;
  const int BH = p.B * p.Hkv;
  w.kvbh = u % BH;
  w.t = u / BH;
  const int first_row = w.t * kBig - p.causal_off;
  w.first = (p.causal && first_row > 0) ? first_row / kStep : 0;
  w.per = (p.Nq + kStep - 1) / kStep - w.first;
  w.count = w.per * p.group;
  return w;
}

struct DqUnit {
  int bh;     // query head
  int t;      // 128-row query tile
  int count;  // 64-key steps
};

// dQ units, high query tiles first; only query tiles that see some key.
__device__ __forceinline__ DqUnit decode_dq(const BwdParams& p, int u) {
  DqUnit w;
  const int BH = p.B * p.H;
  w.bh = u % BH;
  const int nk = (p.Nk + kStep - 1) / kStep;
  w.t = p.causal ? p.num_q_tiles - 1 - u / BH : p.q_tile_first + u / BH;
  if (p.causal) {
    const int last_key = min(p.Nq, (w.t + 1) * kBig) - 1 + p.causal_off;  // >= 0 for these tiles
    w.count = min(nk, last_key / kStep + 1);
  } else {
    w.count = nk;
  }
  return w;
}

// S (or S^T) = A B^T over d = 256: A is a 128-row operand (chunks of
// kChunkBig), B a 64-row one (chunks of kChunkStep), both K-major.  Each
// MMA here is only 32 cycles of tensor work, so the issue cost counts: the
// descriptors are built once and a K-step adds a constant to their low
// halves (the start address field).
__device__ __forceinline__ void issue_scores(uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
  constexpr uint32_t id = idesc_bf16(kBig, kStep, false, false);
  constexpr uint32_t hi = sdesc_hi(1024);
  const uint32_t a_lo = sdesc_lo(a_base, 16);
  const uint32_t b_lo = sdesc_lo(b_base, 16);
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk)
    mma_ss_lh_w(d_tmem, a_lo + (((kk / 4) * kChunkBig + (kk % 4) * 32) >> 4), hi,
                b_lo + (((kk / 4) * kChunkStep + (kk % 4) * 32) >> 4), hi, id, kk > 0 ? 1u : 0u);
}

// acc (+)= X B: X packed bf16 in TMEM (128 rows x 64, 8 columns per 16),
// B a 64-row tile read MN-major (N = 256 = four 64-column blocks).
__device__ __forceinline__ void issue_accumulate(uint32_t acc_tmem, uint32_t x_tmem, uint32_t b_base,
                                                 bool accumulate) {
  constexpr uint32_t id = idesc_bf16(kBig, kD, false, true);
  constexpr uint32_t hi = sdesc_hi(1024);
  const uint32_t b_lo = sdesc_lo(b_base, kChunkStep);
#pragma unroll
  for (int kk = 0; kk < kStep / 16; ++kk)
    mma_ts_lh_w(acc_tmem, x_tmem + kk * 8, b_lo + ((kk * 2048) >> 4), hi, id, (accumulate || kk > 0) ? 1u : 0u);
}

}  // namespace b256

// ------------------------------------------------------------ dK / dV pass

template <bool DK, bool GQA>
__global__ void __launch_bounds__(b256::kThreads, 1)
    fa_bwd256_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                        const BwdParams p) {
  using namespace b256;
  using C = KvCfg<DK>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, (unsigned int)FA_ERR_CUDA);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* k_full = bars;      // K (and V) of the unit
  uint64_t* k_empty = bars + 1;
  uint64_t* v_full = bars + 2;
  uint64_t* v_empty = bars + 3;
  uint64_t* q_full = bars + 4;  // [kQStages]: Q tile
  uint64_t* q_empty = q_full + C::kQStages;
  uint64_t* do_full = q_empty + C::kQStages;  // [kDoStages]: dO tile
  uint64_t* do_empty = do_full + C::kDoStages;
  uint64_t* rv_full = do_empty + C::kDoStages;  // [kRvStages]: L (and D) of a query step
  uint64_t* rv_empty = rv_full + C::kRvStages;
  uint64_t* s_full = rv_empty + C::kRvStages;  // [2]: S^T of region r computed
  uint64_t* dp_full = s_full + 2;              // [2]: dP^T of region r computed (dK pass)
  uint64_t* p_ready = dp_full + 2;             // [2]: packed operand of region r written
  uint64_t* acc_full = p_ready + 2;            // the unit's accumulator complete
  uint64_t* acc_empty = acc_full + 1;          // ... and read out
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  float* sRv = reinterpret_cast<float*>(smem + C::kOffRv);  // stage s: L at 128 s, D at 128 s + 64

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    mbar_init(k_empty, 1);
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    for (int i = 0; i < C::kQStages; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < C::kDoStages; ++i) {
      mbar_init(&do_full[i], 1);
      mbar_init(&do_empty[i], 1);
    }
    for (int i = 0; i < C::kRvStages; ++i) {
      mbar_init(&rv_full[i], 1);
      mbar_init(&rv_empty[i], 4);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&s_full[r], 1);
      mbar_init(&dp_full[r], 1);
      mbar_init(&p_ready[r], 4);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 5 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{p.status, p.timeout_ns};
  auto wait_all = [&](uint64_t* bar, uint32_t parity, uint32_t where) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, where));
  };

  if (warp == 5) {
    // ------------------------------------------------------------ producer
    // Per step: the Q and dO copies first, then the step's L and D values
    // (read from global memory into registers before the copies are
    // issued, stored to the ring after), so the copies never wait behind
    // those reads.
    // Launched while the kernel ahead may still run.  The dV pass follows
    // the D preprocess: it waits for it (it reads no D itself, but the
    // kernels after it rely on D being complete once it has let them
    // launch).  The dK pass follows the dV pass, which it does not read:
    // D was complete before the dV pass let it launch.
    if constexpr (!DK) pdl_wait();
    pdl_trigger();
    uint32_t kc = 0, qc = 0;
    uint32_t q_issued = 0, do_issued = 0, k_issued = 0, v_issued = 0;  // copies started (for the drain)
    bool ok = true;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units_kv; ++rnd) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units_kv) continue;
      const KvUnit w = decode_kv(p, u);
      ok = wait_all(k_empty, (kc & 1) ^ 1, kWaitBwdLoad);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(k_full, kBigBytes);
        for (int c = 0; c < 4; ++c) tma_load_3d(smem + C::kOffK + c * kChunkBig, &tm_k, k_full, c * 64, w.t * kBig, w.kvbh);
      }
      ++k_issued;
      if constexpr (DK) {
        ok = wait_all(v_empty, (kc & 1) ^ 1, kWaitBwdLoad);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(v_full, kBigBytes);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(smem + C::kOffV + c * kChunkBig, &tm_v, v_full, c * 64, w.t * kBig, w.kvbh);
        }
        ++v_issued;
      }
      // Step ii reads query rows [row, row + kStep) of query head qh.
      auto step_pos = [&](int ii, int& qh, int& row) {
        const int grp = ii / w.per;  // query head of the group
        qh = GQA ? q_head_of(w.kvbh, 0, p.H, p.Hkv) + grp : w.kvbh;
        row = (w.first + ii - grp * w.per) * kStep;
      };
      // Q of step ii into ring position pos.
      auto load_q = [&](int ii, uint32_t pos) -> bool {
        int qh, row;
        step_pos(ii, qh, row);
        const uint32_t sq = pos % C::kQStages;
        if (!wait_all(&q_empty[sq], ((pos / C::kQStages) & 1) ^ 1, kWaitBwdLoad)) return false;
        if (lane == 0) {
          mbar_arrive_expect_tx(&q_full[sq], kStepBytes);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(smem + C::kOffQ + sq * kStepBytes + c * kChunkStep, &tm_q, &q_full[sq], c * 64, row, qh);
        }
        ++q_issued;
        return true;
      };
      // dV pass: a Q slot frees when its S^T completes, a dO slot only when
      // its accumulation does, so Q runs a step ahead of dO.
      if (!DK) ok = load_q(0, qc);
      for (int ii = 0; ok && ii < w.count; ++ii, ++qc) {
        int qh, row;
        step_pos(ii, qh, row);
        const size_t head = (size_t)qh * p.Nq;
        // L (log2 units; rows past Nq and rows that see no key get +inf, so
        // their weights vanish) and D of the step.
        float2 l2, d2 = make_float2(0.f, 0.f);
        {
          float* lp = &l2.x;
          float* dp = &d2.x;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int qr = row + 2 * lane + e;
            lp[e] = qr < p.Nq ? p.lse[head + qr] : INFINITY;
            if (DK) dp[e] = qr < p.Nq ? p.dvec[head + qr] : 0.f;
          }
        }
        if (DK || ii + 1 < w.count) ok = load_q(DK ? ii : ii + 1, DK ? qc : qc + 1);
        if (!ok) break;
        const uint32_t sd = qc % C::kDoStages;
        ok = wait_all(&do_empty[sd], ((qc / C::kDoStages) & 1) ^ 1, kWaitBwdLoad);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&do_full[sd], kStepBytes);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(smem + C::kOffDO + sd * kStepBytes + c * kChunkStep, &tm_do, &do_full[sd], c * 64, row, qh);
        }
        ++do_issued;
        // The values, then the arrive that publishes them.
        const uint32_t sr = qc % C::kRvStages;
        ok = wait_all(&rv_empty[sr], ((qc / C::kRvStages) & 1) ^ 1, kWaitBwdLoad);
        if (!ok) break;
        l2.x = l2.x == -INFINITY ? INFINITY : l2.x * 1.4426950408889634f;
        l2.y = l2.y == -INFINITY ? INFINITY : l2.y * 1.4426950408889634f;
        reinterpret_cast<float2*>(sRv + sr * 2 * kStep)[lane] = l2;
        reinterpret_cast<float2*>(sRv + sr * 2 * kStep + kStep)[lane] = d2;
        __syncwarp();
        if (lane == 0) mbar_arrive(&rv_full[sr]);
      }
      ++kc;
    }
    if (lane == 0) {
      // Every copy this warp started lands before the CTA can exit.
      if (k_issued > 0) mbar_wait(k_full, (k_issued - 1) & 1, ctl, kWaitDrain);
      if (v_issued > 0) mbar_wait(v_full, (v_issued - 1) & 1, ctl, kWaitDrain);
      for (uint32_t pos = q_issued > (uint32_t)C::kQStages ? q_issued - C::kQStages : 0u; pos < q_issued; ++pos)
        mbar_wait(&q_full[pos % C::kQStages], (pos / C::kQStages) & 1, ctl, kWaitDrain);
      for (uint32_t pos = do_issued > (uint32_t)C::kDoStages ? do_issued - C::kDoStages : 0u; pos < do_issued; ++pos)
        mbar_wait(&do_full[pos % C::kDoStages], (pos / C::kDoStages) & 1, ctl, kWaitDrain);
    }
    __syncwarp();
  } else if (warp == 4) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t sk = smem_u32(smem + C::kOffK);
    const uint32_t sv = smem_u32(smem + C::kOffV);
    auto q_addr = [&](uint32_t g) { return smem_u32(smem + C::kOffQ + (g % C::kQStages) * kStepBytes); };
    auto do_addr = [&](uint32_t g) { return smem_u32(smem + C::kOffDO + (g % C::kDoStages) * kStepBytes); };
    // The accumulation of step g (pending), its unit's position and whether
    // it opens / closes its unit.
    bool pend = false, pend_first = false, pend_last = false;
    uint32_t pend_un = 0;
    auto accumulate = [&](uint32_t g) -> bool {
      if (!wait_all(&p_ready[g & 1], (g >> 1) & 1, kWaitBwdMma)) return false;
      if (pend_first && pend_un > 0 && !wait_all(acc_empty, (pend_un - 1) & 1, kWaitBwdMma)) return false;
      // dV pass: dO of step g is read by this accumulation only.
      if (!DK && !wait_all(&do_full[g % C::kDoStages], (g / C::kDoStages) & 1, kWaitBwdMma)) return false;
      tc_fence_after();
      const uint32_t region = tmem + 128u * (g & 1);
      if constexpr (DK) {
        // dK += dS^T Q (dS^T packed over the dP^T columns)
        issue_accumulate(tmem + kColAcc, region + 64, q_addr(g), !pend_first);
        mma_commit_w(&q_empty[g % C::kQStages]);
      } else {
        // dV += P^T dO (P^T packed over the S^T columns)
        issue_accumulate(tmem + kColAcc, region, do_addr(g), !pend_first);
        mma_commit_w(&do_empty[g % C::kDoStages]);
      }
      if (pend_last) mma_commit_w(acc_full);
      return true;
    };
    uint32_t g = 0, un = 0;
    bool ok = true;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units_kv; ++rnd, ++un) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units_kv) {
        --un;
        continue;
      }
      const KvUnit w = decode_kv(p, u);
      ok = wait_all(k_full, un & 1, kWaitBwdMma);
      for (int ii = 0; ok && ii < w.count; ++ii, ++g) {
        // Step g: S^T into region g & 1 (its previous contents, step g - 2,
        // were read by an accumulation issued earlier), the accumulation of
        // step g - 1, then (dK pass) dP^T.  With the accumulation ahead of
        // dP^T, the Q tile of step g - 1 (read by S^T and by dK) is released
        // one product earlier, and its slot reloads while dP^T runs.
        ok = wait_all(&q_full[g % C::kQStages], (g / C::kQStages) & 1, kWaitBwdMma);
        if (!ok) break;
        tc_fence_after();
        const uint32_t region = tmem + 128u * (g & 1);
        issue_scores(region, sk, q_addr(g));                      // S^T = K Q^T
        if (!DK) mma_commit_w(&q_empty[g % C::kQStages]);        // dV pass: Q read by S^T only
        mma_commit_w(&s_full[g & 1]);
        if (ii + 1 == w.count) mma_commit_w(k_empty);             // K: read by S^T only
        if (pend) {
          ok = accumulate(g - 1);
          if (!ok) break;
        }
        if constexpr (DK) {
          if (ii == 0) ok = wait_all(v_full, un & 1, kWaitBwdMma);
          if (ok) ok = wait_all(&do_full[g % C::kDoStages], (g / C::kDoStages) & 1, kWaitBwdMma);
          if (!ok) break;
          tc_fence_after();
          issue_scores(region + 64, sv, do_addr(g));  // dP^T = V dO^T
          mma_commit_w(&do_empty[g % C::kDoStages]);  // dO: read by dP^T only
          mma_commit_w(&dp_full[g & 1]);
          if (ii + 1 == w.count) mma_commit_w(v_empty);
        }
        pend = true;
        pend_first = ii == 0;
        pend_last = ii + 1 == w.count;
        pend_un = un;
      }
    }
    if (ok && pend) accumulate(g - 1);
    mma_commit_w(drain);
    (void)wait_all(drain, 0, kWaitDrain);
    __syncwarp();
  } else {
    // ------------------------------------------ element-wise and write-out
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const float sl2 = p.scale_log2;
    uint32_t g = 0, uc = 0;
    bool ok = true;
    // The accumulator of unit (kr, head) -> bf16 rows of dK (scaled) or dV.
    auto write_out = [&](int kr, size_t head) -> bool {
      if (!wait_all(acc_full, uc & 1, kWaitBwdSoftmax)) return false;
      ++uc;
      tc_fence_after();
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(DK ? p.dk : p.dv) + (head + kr) * kD;
      const float sc = DK ? p.scale : 1.f;
#pragma unroll 1
      for (int c = 0; c < kD / 64; ++c) {
        uint32_t wv[32];
        tmem_read_pack<64>(tmem + lane_off + kColAcc + 64 * c, sc, wv);
        if (c + 1 == kD / 64) {
          tc_fence_before();
          mbar_arrive_warp(acc_empty);
        }
        store_rows<4>(reinterpret_cast<uint8_t*>(dst + 64 * c), (size_t)kD * 2, kr, p.Nk, wv, p.store32 != 0);
      }
      return true;
    };
    int pend_kr = -1;
    size_t pend_head = 0;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units_kv; ++rnd) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units_kv) continue;
      const KvUnit w = decode_kv(p, u);
      const int kr = w.t * kBig + 32 * warp + lane;  // key row of this thread
      const size_t head = (size_t)w.kvbh * p.Nk;
      int qt = w.first;
      for (int ii = 0; ok && ii < w.count; ++ii, ++g) {
        if (ii > 0 && ++qt == w.first + w.per) qt = w.first;
        const int q0 = qt * kStep;
        const uint32_t tR = tmem + lane_off + 128u * (g & 1);
        const uint32_t sr = g % C::kRvStages;
        const float* bl = sRv + sr * 2 * kStep;  // L of the step's 64 queries
        const float* bd = bl + kStep;            // D
        ok = wait_all(&rv_full[sr], (g / C::kRvStages) & 1, kWaitBwdSoftmax);
        if (ok) ok = wait_all(&s_full[g & 1], (g >> 1) & 1, kWaitBwdSoftmax);
        if (!ok) break;
        tc_fence_after();
        uint32_t pv[64];
        tmem_ld32(tR, pv);
        tmem_ld32(tR + 32, pv + 32);
        tmem_ld_wait<64>(pv);
        {
          if ((kr >= p.Nk) || (p.causal && kr > q0 + p.causal_off))
            p64_colL<true>(pv, bl, sl2, kr - p.causal_off, q0, kr >= p.Nk, p.causal != 0);
          else
            p64_colL<false>(pv, bl, sl2, kr, q0, false, false);
        }
        uint32_t pk[32];
        if constexpr (DK) {
          // dS^T = P^T * (dP^T - D), packed over this step's dP^T columns.
          ok = wait_all(&dp_full[g & 1], (g >> 1) & 1, kWaitBwdSoftmax);
          if (!ok) break;
          tc_fence_after();
          uint32_t dpv[64];
          tmem_ld32(tR + 64, dpv);
          tmem_ld32(tR + 96, dpv + 32);
          tmem_ld_wait<64>(dpv);
#pragma unroll
          for (int e4 = 0; e4 < 16; ++e4) {
            const float4 d4 = reinterpret_cast<const float4*>(bd)[e4];
            const float2 p01 = make_float2(__uint_as_float(pv[4 * e4]), __uint_as_float(pv[4 * e4 + 1]));
            const float2 p23 = make_float2(__uint_as_float(pv[4 * e4 + 2]), __uint_as_float(pv[4 * e4 + 3]));
            const float2 g01 = __fadd2_rn(make_float2(__uint_as_float(dpv[4 * e4]), __uint_as_float(dpv[4 * e4 + 1])),
                                          make_float2(-d4.x, -d4.y));
            const float2 g23 =
                __fadd2_rn(make_float2(__uint_as_float(dpv[4 * e4 + 2]), __uint_as_float(dpv[4 * e4 + 3])),
                           make_float2(-d4.z, -d4.w));
            const float2 ds01 = __fmul2_rn(p01, g01);
            const float2 ds23 = __fmul2_rn(p23, g23);
            pk[2 * e4] = pack_bf16(ds01.x, ds01.y);
            pk[2 * e4 + 1] = pack_bf16(ds23.x, ds23.y);
          }
          tmem_st32(tR + 64, pk);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) pk[e] = pack_bf16(__uint_as_float(pv[2 * e]), __uint_as_float(pv[2 * e + 1]));
          tmem_st32(tR, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&p_ready[g & 1]);
        mbar_arrive_warp(&rv_empty[sr]);  // L and D of the step were read
        if (ii == 0 && pend_kr >= 0) {
          ok = write_out(pend_kr, pend_head);
          if (!ok) break;
        }
      }
      if (!ok) break;
      pend_kr = kr;
      pend_head = head;
    }
    if (ok && pend_kr >= 0) write_out(pend_kr, pend_head);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------------------------------------------- dQ

__global__ void __launch_bounds__(b256::kThreads, 1)
    fa_bwd256_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                        const BwdParams p) {
  using namespace b256;
  using C = DqCfg;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, (unsigned int)FA_ERR_CUDA);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;  // Q and dO of the unit
  uint64_t* q_empty = bars + 1;
  uint64_t* do_full = bars + 2;
  uint64_t* do_empty = bars + 3;
  uint64_t* k_full = bars + 4;  // [kKStages]
  uint64_t* k_empty = k_full + C::kKStages;
  uint64_t* v_full = k_empty + C::kKStages;  // [kVStages]
  uint64_t* v_empty = v_full + C::kVStages;
  uint64_t* s_full = v_empty + C::kVStages;  // [2]: S of region r computed
  uint64_t* dp_full = s_full + 2;            // [2]: dP of region r computed
  uint64_t* p_ready = dp_full + 2;           // [2]: dS of region r written
  uint64_t* acc_full = p_ready + 2;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(do_full, 1);
    mbar_init(do_empty, 1);
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&s_full[r], 1);
      mbar_init(&dp_full[r], 1);
      mbar_init(&p_ready[r], 4);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 5 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{p.status, p.timeout_ns};
  auto wait_all = [&](uint64_t* bar, uint32_t parity, uint32_t where) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, where));
  };

  if (warp == 5) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t uc = 0, kc = 0;
      uint32_t q_issued = 0, do_issued = 0, k_issued = 0, v_issued = 0;  // copies started (for the drain)
      bool ok = true;
      for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
        const int u = snake_unit(rnd);
        if (u >= p.num_units) continue;
        const DqUnit w = decode_dq(p, u);
        const int kvbh = p.Hkv == p.H ? w.bh : kv_head_of(w.bh, p.H, p.Hkv);
        ok = mbar_wait(q_empty, (uc & 1) ^ 1, ctl, kWaitBwdLoad);
        if (!ok) break;
        mbar_arrive_expect_tx(q_full, kBigBytes);
        for (int c = 0; c < 4; ++c) tma_load_3d(smem + C::kOffQ + c * kChunkBig, &tm_q, q_full, c * 64, w.t * kBig, w.bh);
        ++q_issued;
        ok = mbar_wait(do_empty, (uc & 1) ^ 1, ctl, kWaitBwdLoad);
        if (!ok) break;
        mbar_arrive_expect_tx(do_full, kBigBytes);
        for (int c = 0; c < 4; ++c)
          tma_load_3d(smem + C::kOffDO + c * kChunkBig, &tm_do, do_full, c * 64, w.t * kBig, w.bh);
        ++do_issued;
        for (int jj = 0; ok && jj < w.count; ++jj, ++kc) {
          const int key0 = jj * kStep;
          const uint32_t sk = kc % C::kKStages;
          ok = mbar_wait(&k_empty[sk], ((kc / C::kKStages) & 1) ^ 1, ctl, kWaitBwdLoad);
          if (!ok) break;
          mbar_arrive_expect_tx(&k_full[sk], kStepBytes);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(smem + C::kOffK + sk * kStepBytes + c * kChunkStep, &tm_k, &k_full[sk], c * 64, key0, kvbh);
          ++k_issued;
          const uint32_t sv = kc % C::kVStages;
          ok = mbar_wait(&v_empty[sv], ((kc / C::kVStages) & 1) ^ 1, ctl, kWaitBwdLoad);
          if (!ok) break;
          mbar_arrive_expect_tx(&v_full[sv], kStepBytes);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(smem + C::kOffV + sv * kStepBytes + c * kChunkStep, &tm_v, &v_full[sv], c * 64, key0, kvbh);
          ++v_issued;
        }
        ++uc;
      }
      if (q_issued > 0) mbar_wait(q_full, (q_issued - 1) & 1, ctl, kWaitDrain);
      if (do_issued > 0) mbar_wait(do_full, (do_issued - 1) & 1, ctl, kWaitDrain);
      for (uint32_t pos = k_issued > (uint32_t)C::kKStages ? k_issued - C::kKStages : 0u; pos < k_issued; ++pos)
        mbar_wait(&k_full[pos % C::kKStages], (pos / C::kKStages) & 1, ctl, kWaitDrain);
      for (uint32_t pos = v_issued > (uint32_t)C::kVStages ? v_issued - C::kVStages : 0u; pos < v_issued; ++pos)
        mbar_wait(&v_full[pos % C::kVStages], (pos / C::kVStages) & 1, ctl, kWaitDrain);
    }
    __syncwarp();
  } else if (warp == 4) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t sq = smem_u32(smem + C::kOffQ);
    const uint32_t sdo = smem_u32(smem + C::kOffDO);
    auto k_addr = [&](uint32_t g) { return smem_u32(smem + C::kOffK + (g % C::kKStages) * kStepBytes); };
    auto v_addr = [&](uint32_t g) { return smem_u32(smem + C::kOffV + (g % C::kVStages) * kStepBytes); };
    bool pend = false, pend_first = false, pend_last = false;
    uint32_t pend_un = 0;
    auto accumulate = [&](uint32_t g) -> bool {  // dQ += dS K_g (dS packed over the S columns)
      if (!wait_all(&p_ready[g & 1], (g >> 1) & 1, kWaitBwdMma)) return false;
      if (pend_first && pend_un > 0 && !wait_all(acc_empty, (pend_un - 1) & 1, kWaitBwdMma)) return false;
      tc_fence_after();
      issue_accumulate(tmem + kColAcc, tmem + 128u * (g & 1), k_addr(g), !pend_first);
      mma_commit_w(&k_empty[g % C::kKStages]);
      if (pend_last) mma_commit_w(acc_full);
      return true;
    };
    uint32_t g = 0, un = 0;
    bool ok = true;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd, ++un) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units) {
        --un;
        continue;
      }
      const DqUnit w = decode_dq(p, u);
      ok = wait_all(q_full, un & 1, kWaitBwdMma) && wait_all(do_full, un & 1, kWaitBwdMma);
      for (int jj = 0; ok && jj < w.count; ++jj, ++g) {
        // Step g: S, the accumulation of step g - 1, then dP.  With the
        // accumulation ahead of dP, the K tile of step g - 1 (read by S and
        // by dQ) is released one product earlier, and its slot reloads while
        // dP runs.
        ok = wait_all(&k_full[g % C::kKStages], (g / C::kKStages) & 1, kWaitBwdMma);
        if (!ok) break;
        tc_fence_after();
        const uint32_t region = tmem + 128u * (g & 1);
        issue_scores(region, sq, k_addr(g));  // S = Q K^T
        mma_commit_w(&s_full[g & 1]);
        if (jj + 1 == w.count) mma_commit_w(q_empty);
        if (pend) {
          ok = accumulate(g - 1);
          if (!ok) break;
        }
        ok = wait_all(&v_full[g % C::kVStages], (g / C::kVStages) & 1, kWaitBwdMma);
        if (!ok) break;
        tc_fence_after();
        issue_scores(region + 64, sdo, v_addr(g));  // dP = dO V^T
        mma_commit_w(&v_empty[g % C::kVStages]);    // V: read by dP only
        mma_commit_w(&dp_full[g & 1]);
        if (jj + 1 == w.count) mma_commit_w(do_empty);
        pend = true;
        pend_first = jj == 0;
        pend_last = jj + 1 == w.count;
        pend_un = un;
      }
    }
    if (ok && pend) accumulate(g - 1);
    mma_commit_w(drain);
    (void)wait_all(drain, 0, kWaitDrain);
    __syncwarp();
  } else {
    // ------------------------------------------ element-wise and write-out
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const float sl2 = p.scale_log2;
    uint32_t g = 0, uc = 0;
    bool ok = true;
    auto write_out = [&](int q, size_t head) -> bool {
      if (!wait_all(acc_full, uc & 1, kWaitBwdDq)) return false;
      ++uc;
      tc_fence_after();
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.dq) + (head + q) * kD;
#pragma unroll 1
      for (int c = 0; c < kD / 64; ++c) {
        uint32_t wv[32];
        tmem_read_pack<64>(tmem + lane_off + kColAcc + 64 * c, p.scale, wv);
        if (c + 1 == kD / 64) {
          tc_fence_before();
          mbar_arrive_warp(acc_empty);
        }
        store_rows<4>(reinterpret_cast<uint8_t*>(dst + 64 * c), (size_t)kD * 2, q, p.Nq, wv, p.store32 != 0);
      }
      return true;
    };
    int pend_q = -1;
    size_t pend_head = 0;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units) continue;
      const DqUnit w = decode_dq(p, u);
      const size_t head = (size_t)w.bh * p.Nq;
      const int q = w.t * kBig + 32 * warp + lane;  // query row of this thread
      const int q_lo = w.t * kBig + 32 * warp;      // first query of this warp
      const float Lraw = q < p.Nq ? p.lse[head + q] : INFINITY;
      const float L = Lraw == -INFINITY ? INFINITY : Lraw * 1.4426950408889634f;  // no key seen: weights 0
      const float Dq = q < p.Nq ? p.dvec[head + q] : 0.f;
      for (int jj = 0; ok && jj < w.count; ++jj, ++g) {
        const uint32_t tR = tmem + lane_off + 128u * (g & 1);
        const int k_first = jj * kStep;
        ok = wait_all(&s_full[g & 1], (g >> 1) & 1, kWaitBwdSoftmax);
        if (!ok) break;
        tc_fence_after();
        uint32_t pv[64], dpv[64];
        tmem_ld32(tR, pv);
        tmem_ld32(tR + 32, pv + 32);
        tmem_ld_wait<64>(pv);
        if (k_first + kStep - 1 >= p.Nk || (p.causal && k_first + kStep - 1 > q_lo + p.causal_off))
          p64_rowL<true>(pv, L, sl2, q + p.causal_off, k_first, p.Nk, p.causal != 0);
        else
          p64_rowL<false>(pv, L, sl2, q, k_first, p.Nk, false);
        ok = wait_all(&dp_full[g & 1], (g >> 1) & 1, kWaitBwdSoftmax);
        if (!ok) break;
        tc_fence_after();
        tmem_ld32(tR + 64, dpv);
        tmem_ld32(tR + 96, dpv + 32);
        tmem_ld_wait<64>(dpv);
        uint32_t pk[32];
        const float2 dv2 = make_float2(-Dq, -Dq);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float2 g2 = __fadd2_rn(make_float2(__uint_as_float(dpv[2 * e]), __uint_as_float(dpv[2 * e + 1])), dv2);
          const float2 ds = __fmul2_rn(make_float2(__uint_as_float(pv[2 * e]), __uint_as_float(pv[2 * e + 1])), g2);
          pk[e] = pack_bf16(ds.x, ds.y);
        }
        tmem_st32(tR, pk);  // dS over the S columns this thread has read
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&p_ready[g & 1]);
        if (jj == 0 && pend_q >= 0) {
          ok = write_out(pend_q, pend_head);
          if (!ok) break;
        }
      }
      if (!ok) break;
      pend_q = q;
      pend_head = head;
    }
    if (ok && pend_q >= 0) write_out(pend_q, pend_head);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ launch

template <bool DK, bool GQA>
static cudaError_t launch_kv256_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream) {
  constexpr int smem = b256::KvCfg<DK>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(fa_bwd256_kv_kernel<DK, GQA>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(fa_bwd256_kv_kernel<DK, GQA>, dim3(grid), dim3(b256::kThreads), smem, stream, tq, tk, tv, tdo, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The dV pass (dk_pass = false) or the dK pass over the key tiles some
// query row sees.  Q and dO tensor maps with 64-row boxes, K and V 128-row.
cudaError_t launch_bwd256_kv(bool dk_pass, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream) {
  const bool gqa = p.Hkv != p.H;
  if (dk_pass)
    return gqa ? launch_kv256_t<true, true>(tq, tk, tv, tdo, p, grid, stream)
               : launch_kv256_t<true, false>(tq, tk, tv, tdo, p, grid, stream);
  return gqa ? launch_kv256_t<false, true>(tq, tk, tv, tdo, p, grid, stream)
             : launch_kv256_t<false, false>(tq, tk, tv, tdo, p, grid, stream);
}

// Q and dO tensor maps with 128-row boxes, K and V 64-row.
cudaError_t launch_bwd256_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream) {
  cudaError_t e =
      cudaFuncSetAttribute(fa_bwd256_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, b256::DqCfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  // May start as the dK pass's CTAs finish: it reads only the inputs, L and
  // D, and D was complete before the dV pass let the dK pass launch.
  e = launch_pdl(fa_bwd256_dq_kernel, dim3(grid), dim3(b256::kThreads), b256::DqCfg::kSmemBytes, stream, tq, tk, tv,
                 tdo, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace fa
