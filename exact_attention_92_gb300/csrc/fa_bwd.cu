// Backward pass of exact attention on sm_103a ("FlashAttention V2 in depth",
// section 7).
//
//   fa_bwd_preprocess   D_i = rowsum(dO_i * O_i) (section 7.3), once.
//   fa_bwd_dkdv_kernel  key/value tiles in the outer loop (section 7.2): a
//                       persistent CTA owns one 128-key tile K_j, V_j of one
//                       (batch, head) and walks the query tiles i that can
//                       see it; dK_j and dV_j accumulate in tensor memory.
//   fa_bwd_dq_kernel    query tiles in the outer loop: a CTA owns one
//                       128-query tile Q_i, dO_i and walks the key tiles j it
//                       can see; dQ_i accumulates in tensor memory and is
//                       written once, as bf16.
//
// Both kernels recompute P from the saved logsumexp (section 7.1) and
// dS = P * (dP - D).  Splitting dQ from dK/dV costs the S and dP products a
// second time but removes the fp32 atomic accumulation of dQ over key tiles,
// whose reductions into L2 bound the single-kernel form on this GPU (about
// 24 bytes per clock per SM when every SM reduces).  The products per
// (key tile, query tile) pair are
//   dK/dV kernel (TMEM lanes are keys):
//     S^T = K Q^T,  dP^T = V dO^T,  dV += P^T dO,  dK += dS^T Q
//   dQ kernel (TMEM lanes are queries):
//     S = Q K^T,    dP = dO V^T,    dQ += dS K
// The softmax scale is applied once to dK and dQ when they are written.
//
// Roles (384 threads, three warpgroups, registers split with setmaxnreg as
// in the forward kernel): warp 9 loads (TMA); tcgen05 MMAs are issued by
// warp 8 alone in the dK/dV kernel (one ordered stream of products) and by
// warps 8 and 10 in the dQ kernel (split so that neither's products touch
// the TMEM columns of the other's); an issuing warp walks its schedule as a
// whole warp and an elected lane issues every MMA and commit.  The other
// control warps idle; warps 0-7 do the element-wise work (a TMEM lane per
// thread; warps w and w+4 split the 128 columns of a tile) and write the
// results.
//
// Queries and keys may differ in length (Nq, Nk); with the causal mask query
// row i sees keys j <= i + causal_off.  The dK/dV kernel runs over the key
// tiles some query row sees, the dQ kernel over the query tiles that see
// some key; the host zeroes the gradient rows of the others.  A query row
// that sees no key has L = -inf, which the kernels read as +inf (all of its
// weights are 0).
//
// Head dims 64, 96 and 128; a 96-wide row is staged in the 128-wide layout
// (TMA zero-fills columns 96..127) and the products use K = 96 / N = 96.
//
// Pipelining.  The element-wise warps read a tile of S into registers and
// compute P from it while the tensor core runs other products; they read dP
// when it lands, and P^T / dS^T (dK/dV kernel) or dS (dQ kernel) go back to
// TMEM as bf16 pairs over columns the same warp has already read, where the
// next products take them as the TMEM operand.
#include <cuda_runtime.h>

#include <type_traits>

#include "bwd_elementwise.cuh"
#include "sm103_primitives.cuh"

namespace fa {

using namespace dev;

// Register split shared by both kernels: 168 per thread at launch (three
// warps per SM sub-partition); warpgroup 2 keeps kRegsCtl, the element-wise
// warpgroups get kRegsMath.
struct BwdRegs {
  static constexpr int kRegsAtLaunch = 168;
  static constexpr int kRegsCtl = 72;
  static constexpr int kRegsMath = 216;
  static_assert(128 * kRegsCtl + 256 * kRegsMath <= 384 * kRegsAtLaunch, "register split exceeds the launch");
};

// ---------------------------------------------------------------- dK / dV

// Columns of a D-wide gradient row handled by the element-wise warps with
// hc = 0 (the warps with hc = 1 take the rest): halves of D, or the first 64
// of 96 so that both parts are whole 32-byte units in power-of-two groups.
template <int D>
struct RowSplit {
  static constexpr int kLo = (D == 96) ? 64 : D / 2;
  static constexpr int kHi = D - kLo;
};

template <int D>
struct DkdvCfg {
  static_assert(D == 64 || D == 96 || D == 128, "head dim");
  static constexpr int kChunks = (D + 63) / 64;
  static constexpr int kChunkBytes = kTileM * 128;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kQStages = 3;  // the next step's S^T needs Q early
  static constexpr int kDoStages = 2;
  static constexpr int kThreads = 384;
  // Two 128-column regions, one per step in flight: S^T, then dP^T, then
  // P^T | dS^T packed.
  __host__ __device__ static constexpr uint32_t col_r(uint32_t r) { return 128u * r; }
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + 64 * kChunks;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;
  static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;
  static constexpr int kOffLse = kOffDO + kDoStages * kTileBytes;  // kQStages x 128 floats (log2 units)
  static constexpr int kOffDvec = kOffLse + kQStages * 128 * 4;    // kDoStages x 128 floats
  static constexpr int kOffBar = kOffDvec + kDoStages * 128 * 4;
  static constexpr int kNumBars = 4 + 2 * kQStages + 2 * kDoStages + 11;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
  static_assert(kSmemBytes <= 232448, "shared memory");
};

struct BwdUnit {
  int bh;     // the head: key/value head (dK/dV kernel), query head (dQ kernel)
  int t;      // the tile this CTA owns (key tile / query tile)
  int first;  // first tile of the other operand
  int count;  // steps: tiles of the other operand, times the query heads that
              // share the key/value head in the dK/dV kernel
  int per;    // steps per query head (dK/dV kernel; = count in the dQ kernel)
};

// dK/dV units: with the causal mask, low key tiles see the most query tiles,
// so they come first.
// A dK/dV unit is one key/value tile of one key/value head; its steps walk
// the visible query tiles of every query head that reads that key/value head
// (one head, for plain multi-head attention), so dK and dV sum over them.
__device__ __forceinline__ BwdUnit decode_dkdv(const BwdParams& p, int u) {
  BwdUnit w;
  const int BH = p.B * p.Hkv;
  w.bh = u % BH;
  w.t = u / BH;
  // With the causal mask the first query row that sees key 128 t is
  // 128 t - causal_off; units cover only key tiles some row sees.
  const int first_row = w.t * kTileN - p.causal_off;
  w.first = (p.causal && first_row > 0) ? first_row / kTileM : 0;
  w.per = p.num_q_tiles - w.first;
  w.count = w.per * p.group;
  return w;
}

// dQ units: with the causal mask, high query tiles see the most key tiles.
// Units cover only query tiles [q_tile_first, num_q_tiles), which see keys.
__device__ __forceinline__ BwdUnit decode_dq(const BwdParams& p, int u) {
  BwdUnit w;
  const int BH = p.B * p.H;
  w.bh = u % BH;
  w.t = p.causal ? p.num_q_tiles - 1 - u / BH : p.q_tile_first + u / BH;
  w.first = 0;
  if (p.causal) {
    const int last_key = min(p.Nq, (w.t + 1) * kTileM) - 1 + p.causal_off;  // >= 0 for these tiles
    w.count = min(p.num_k_tiles, last_key / kTileN + 1);
  } else {
    w.count = p.num_k_tiles;
  }
  w.per = w.count;
  return w;
}

// GQA: key/value heads shared by several query heads (the steps of a unit
// then run over (query head, query tile) pairs); the multi-head instance
// keeps the plain per-tile indexing.
template <int D, bool GQA>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using C = DkdvCfg<D>;
  using R = BwdRegs;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, (unsigned int)FA_ERR_CUDA);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  // K_j and V_j of a unit have separate barriers: K is released after the
  // unit's last S^T, two steps before its end, so the next unit's K loads
  // early; V after the last dP^T.
  uint64_t* k_full = bars;
  uint64_t* k_empty = bars + 1;
  uint64_t* v_full = bars + 2;
  uint64_t* v_empty = bars + 3;
  uint64_t* q_full = bars + 4;  // [kQStages]: Q tile and its L values
  uint64_t* q_empty = q_full + C::kQStages;
  uint64_t* do_full = q_empty + C::kQStages;  // [kDoStages]: dO tile and its D values
  uint64_t* do_empty = do_full + C::kDoStages;
  // Per TMEM region r (steps with pos & 1 == r):
  uint64_t* s_full = do_empty + C::kDoStages;  // [2] S^T in region r
  uint64_t* s_free = s_full + 2;               // [2] ... read by all element-wise warps
  uint64_t* dp_full = s_free + 2;              // [2] dP^T in region r
  uint64_t* p_ready = dp_full + 2;             // [2] P^T, dS^T packed in region r
  uint64_t* dkv_full = p_ready + 2;
  uint64_t* dkv_empty = dkv_full + 1;
  uint64_t* drain = dkv_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);
  float* sDv = reinterpret_cast<float*>(smem + C::kOffDvec);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    mbar_init(k_empty, 1);  // the unit's last S^T
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);  // the unit's last dP^T
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);  // dK (issued after the step's S^T)
    }
    for (int s = 0; s < C::kDoStages; ++s) {
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 1);  // dV (issued after the step's dP^T)
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&s_full[r], 1);
      mbar_init(&s_free[r], 8);
      mbar_init(&dp_full[r], 1);
      mbar_init(&p_ready[r], 8);
    }
    mbar_init(dkv_full, 1);
    mbar_init(dkv_empty, 8);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 9 && lane == 0) {
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

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    reg_dealloc<R::kRegsCtl>();
    // Launched while the D preprocess may still run: wait for it before
    // reading D, then let the dQ kernel (which needs nothing from this one)
    // take over SMs as this grid's CTAs finish.
    pdl_wait();
    pdl_trigger();
    uint32_t kc = 0, qc = 0;
    uint32_t k_issued = 0, v_issued = 0, q_issued = 0, do_issued = 0;  // copies started (for the drain)
    bool ok = true;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units_kv; ++rnd) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units_kv) continue;
      const BwdUnit w = decode_dkdv(p, u);
      ok = __all_sync(0xffffffffu, mbar_wait(k_empty, (kc & 1) ^ 1, ctl, kWaitBwdLoad));
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(k_full, C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem + C::kOffK + c * C::kChunkBytes, &tm_k, k_full, c * 64, w.t * kTileN, w.bh);
      }
      ++k_issued;
      // Step ii: query tile first + ii % per of the (ii / per)-th query head
      // that reads this key/value head (with GQA, kept as running counters).
      int qh = GQA ? q_head_of(w.bh, 0, p.H, p.Hkv) : w.bh;
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
        // L_i and D_i of the step, read from global memory before the waits
        // below so that the reads overlap them instead of delaying the copies.
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
        // Q_i with L_i (log2 units; rows past Nq and rows that see no key
        // get +inf so their weights vanish).  The values are written before
        // the arrive that completes the stage together with the copy.
        const uint32_t sq = qc % C::kQStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&q_empty[sq], ((qc / C::kQStages) & 1) ^ 1, ctl, kWaitBwdLoad));
        if (!ok) break;
        {
          float* lp = &l4.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) lp[e] = lp[e] == -INFINITY ? INFINITY : lp[e] * 1.4426950408889634f;
          reinterpret_cast<float4*>(sLse + sq * 128)[lane] = l4;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&q_full[sq], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(smem + C::kOffQ + sq * C::kTileBytes + c * C::kChunkBytes, &tm_q, &q_full[sq], c * 64,
                        row, qh);
        }
        ++q_issued;
        // dO_i with D_i.
        const uint32_t sd = qc % C::kDoStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&do_empty[sd], ((qc / C::kDoStages) & 1) ^ 1, ctl, kWaitBwdLoad));
        if (!ok) break;
        reinterpret_cast<float4*>(sDv + sd * 128)[lane] = d4;
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&do_full[sd], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(smem + C::kOffDO + sd * C::kTileBytes + c * C::kChunkBytes, &tm_do, &do_full[sd],
                        c * 64, row, qh);
        }
        ++do_issued;
        if (ii == 0) {
          // V_j, needed by the first dP^T, after the first step's Q and dO.
          ok = __all_sync(0xffffffffu, mbar_wait(v_empty, (kc & 1) ^ 1, ctl, kWaitBwdLoad));
          if (!ok) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(v_full, C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(smem + C::kOffV + c * C::kChunkBytes, &tm_v, v_full, c * 64, w.t * kTileN, w.bh);
          }
          ++v_issued;
        }
      }
      ++kc;
    }
    if (lane == 0) {
      // Every copy this warp issued has landed before the CTA exits.
      if (k_issued > 0) mbar_wait(k_full, (k_issued - 1) & 1, ctl, kWaitDrain);
      if (v_issued > 0) mbar_wait(v_full, (v_issued - 1) & 1, ctl, kWaitDrain);
      for (uint32_t pos = q_issued > (uint32_t)C::kQStages ? q_issued - C::kQStages : 0u; pos < q_issued; ++pos)
        mbar_wait(&q_full[pos % C::kQStages], (pos / C::kQStages) & 1, ctl, kWaitDrain);
      for (uint32_t pos = do_issued > (uint32_t)C::kDoStages ? do_issued - C::kDoStages : 0u; pos < do_issued; ++pos)
        mbar_wait(&do_full[pos % C::kDoStages], (pos / C::kDoStages) & 1, ctl, kWaitDrain);
    }
    __syncwarp();
  } else if (warp == 8) {
    // ---------------------------------------------------------- MMA issuer
    // One warp issues every product (the warp walks the schedule, an
    // elected lane issues) as one stream of steps over all of this CTA's
    // units.  Step g uses TMEM region g & 1: S^T, then (once S^T has been
    // read) dP^T, then P^T and dS^T packed, which dV and dK read.  Within
    // step g the order is
    //   dP^T(g), dK(g-1), S^T(g+1), [P^T(g), dS^T(g) ready] dV(g)
    // so dP^T, which the element-wise warps wait for next, enters the tensor
    // pipe behind a single product (dV of the step before) rather than
    // behind dV, dK and S^T.  S^T(g+1) goes into the region dK(g-1) has just
    // read (the pipe runs one warp's products in issue order).  At the
    // first step of a unit, V_j is new and may still be loading: dK(g-1) and
    // S^T(g+1) go first.
    reg_dealloc<R::kRegsCtl>();
    constexpr uint32_t id_s = idesc_bf16(kTileM, kTileM, false, false);  // S^T, dP^T
    constexpr uint32_t id_kv = idesc_bf16(kTileM, D, false, true);       // dV, dK
    const uint32_t sk = smem_u32(smem + C::kOffK);
    const uint32_t sv = smem_u32(smem + C::kOffV);
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, kWaitBwdMma));
    };
    // Position in this CTA's stream of steps: unit `rnd` of the snake order
    // (the `un`-th unit this CTA runs), step `ii` of it.
    struct Cur {
      int rnd, ii, un;
      BwdUnit w;
      bool valid;
    };
    auto seek = [&](Cur& c, int rnd, int un) {
      c.valid = false;
      for (; rnd * (int)gridDim.x < p.num_units_kv; ++rnd) {
        const int u = snake_unit(rnd);
        if (u < p.num_units_kv) {
          c.rnd = rnd;
          c.ii = 0;
          c.un = un;
          c.w = decode_dkdv(p, u);
          c.valid = true;
          return;
        }
      }
    };
    auto advance = [&](Cur& c) {
      if (++c.ii >= c.w.count) seek(c, c.rnd + 1, c.un + 1);
    };
    auto q_addr = [&](uint32_t g) { return smem_u32(smem + C::kOffQ + (g % C::kQStages) * C::kTileBytes); };
    auto do_addr = [&](uint32_t g) { return smem_u32(smem + C::kOffDO + (g % C::kDoStages) * C::kTileBytes); };
    auto issue_s = [&](uint32_t g) {  // S^T(g) = K_j Q_i^T
      const uint32_t qa = q_addr(g);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * C::kChunkBytes + (kk % 4) * 32;
        mma_ss_w(tmem + C::col_r(g & 1), sdesc_sw128(sk + off, 16, 1024), sdesc_sw128(qa + off, 16, 1024), id_s,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit_w(&s_full[g & 1]);
    };
    auto issue_dp = [&](uint32_t g) {  // dP^T(g) = V_j dO_i^T
      const uint32_t da = do_addr(g);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * C::kChunkBytes + (kk % 4) * 32;
        mma_ss_w(tmem + C::col_r(g & 1), sdesc_sw128(sv + off, 16, 1024), sdesc_sw128(da + off, 16, 1024), id_s,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit_w(&dp_full[g & 1]);
    };
    auto issue_dv = [&](uint32_t g, bool acc) {  // dV += P^T dO_i (B read MN-major)
      const uint32_t da = do_addr(g);
#pragma unroll
      for (int kk = 0; kk < kTileM / 16; ++kk)
        mma_ts_w(tmem + C::kColDV, tmem + C::col_r(g & 1) + packed_col(kk, false),
                 sdesc_sw128(da + kk * 2048, C::kChunkBytes, 1024), id_kv, (acc || kk > 0) ? 1u : 0u);
      mma_commit_w(&do_empty[g % C::kDoStages]);  // dO_i: read by dP^T and dV
    };
    auto issue_dk = [&](uint32_t g, bool acc) {  // dK += dS^T Q_i
      const uint32_t qa = q_addr(g);
#pragma unroll
      for (int kk = 0; kk < kTileM / 16; ++kk)
        mma_ts_w(tmem + C::kColDK, tmem + C::col_r(g & 1) + packed_col(kk, true),
                 sdesc_sw128(qa + kk * 2048, C::kChunkBytes, 1024), id_kv, (acc || kk > 0) ? 1u : 0u);
      mma_commit_w(&q_empty[g % C::kQStages]);  // Q_i: read by S^T and dK
    };
    bool ok = true;
    Cur cur, nxt;
    seek(cur, 0, 0);
    if (cur.valid) {
      ok = wait(k_full, 0) && wait(&q_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        if (cur.w.count == 1) mma_commit_w(k_empty);  // K_j: read by S^T only
      }
    }
    nxt = cur;
    if (nxt.valid) advance(nxt);
    uint32_t g = 0;
    // dK of step g - 1, issued during step g: pending, accumulate, and
    // whether it closes its unit.
    bool pend = false, pend_acc = false, pend_last = false;
    for (; ok && cur.valid; ++g) {
      const bool first = cur.ii == 0;
      auto dp_step = [&]() -> bool {
        if (first && !wait(v_full, cur.un & 1)) return false;
        if (!wait(&do_full[g % C::kDoStages], (g / C::kDoStages) & 1)) return false;
        if (!wait(&s_free[g & 1], (g >> 1) & 1)) return false;
        tc_fence_after();
        issue_dp(g);
        if (cur.ii + 1 == cur.w.count) mma_commit_w(v_empty);  // V_j: read by dP^T only
        return true;
      };
      auto dk_prev = [&]() {
        if (!pend) return;
        issue_dk(g - 1, pend_acc);
        if (pend_last) mma_commit_w(dkv_full);
      };
      auto s_next = [&]() -> bool {
        if (!nxt.valid) return true;
        if (nxt.ii == 0 && !wait(k_full, nxt.un & 1)) return false;
        if (!wait(&q_full[(g + 1) % C::kQStages], ((g + 1) / C::kQStages) & 1)) return false;
        tc_fence_after();
        issue_s(g + 1);
        if (nxt.ii + 1 == nxt.w.count) mma_commit_w(k_empty);
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
      // dV(g) once P^T(g) and dS^T(g) are in the region; the first step of a
      // unit also needs the previous unit's dV and dK read out of TMEM.
      ok = wait(&p_ready[g & 1], (g >> 1) & 1);
      if (ok && first && cur.un > 0) ok = wait(dkv_empty, (cur.un - 1) & 1);
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
      if (pend_last) mma_commit_w(dkv_full);
    }
    // Every MMA this warp issued completes before TMEM is released.
    mma_commit_w(drain);
    (void)wait(drain, 0);
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------ P^T, dS^T and dK/dV output
    reg_alloc<R::kRegsMath>();
    const int g = warp & 3;    // TMEM lane quarter
    const int hc = warp >> 2;  // query-column half
    const uint32_t lane_off = (uint32_t)(32 * g) << 16;
    const int r_key = 32 * g + lane;  // key row within the tile
    const float sl2 = p.scale_log2;
    uint32_t uc = 0, qc = 0;
    bool ok = true;
    // dK_j = scale * sum dS^T Q and dV_j = sum P^T dO of unit (kr, head);
    // this warp writes head-dim columns [c0, c0 + NC) (RowSplit).  Run after
    // the next unit's first P^T, while its dP^T is computed.  The warp's
    // part of the row of dV and of dK is packed to bf16 and released from
    // TMEM before any store is issued, so that the next unit's accumulation
    // does not wait behind the stores.
    auto write_part = [&](auto nc_tag, int kr, size_t head) {
      constexpr int NC = decltype(nc_tag)::value;
      const int c0 = hc ? RowSplit<D>::kLo : 0;
      uint32_t w[2][NC / 2];
      tmem_read_pack<NC>(tmem + lane_off + C::kColDV + c0, 1.f, w[0]);
      tmem_read_pack<NC>(tmem + lane_off + C::kColDK + c0, p.scale, w[1]);
      tc_fence_before();
      mbar_arrive_warp(dkv_empty);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(which ? p.dk : p.dv) + (head + kr) * D + c0;
        store_rows<NC / 16>(reinterpret_cast<uint8_t*>(dst), (size_t)D * 2, kr, p.Nk, w[which], p.store32 != 0);
      }
    };
    auto write_dkdv = [&](int kr, size_t head) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(dkv_full, uc & 1, ctl, kWaitBwdSoftmax))) return false;
      ++uc;
      tc_fence_after();
      if constexpr (RowSplit<D>::kLo == RowSplit<D>::kHi) {
        write_part(std::integral_constant<int, RowSplit<D>::kLo>{}, kr, head);
      } else {
        if (hc == 0)
          write_part(std::integral_constant<int, RowSplit<D>::kLo>{}, kr, head);
        else
          write_part(std::integral_constant<int, RowSplit<D>::kHi>{}, kr, head);
      }
      return true;
    };
    int pend_kr = -1;  // the unit whose dK / dV are still in TMEM
    size_t pend_head = 0;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units_kv; ++rnd) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units_kv) continue;
      const BwdUnit w = decode_dkdv(p, u);
      const int kr = w.t * kTileN + r_key;  // key index
      const size_t head = (size_t)w.bh * p.Nk;
      int qt = w.first;
      for (int ii = 0; ok && ii < w.count; ++ii, ++qc) {
        if constexpr (GQA) {
          if (ii > 0 && ++qt == w.first + w.per) qt = w.first;  // query tile of step ii
        } else {
          qt = w.first + ii;
        }
        const int q0 = qt * kTileM;
        const uint32_t reg = qc & 1;
        const uint32_t tZ = tmem + lane_off + C::col_r(reg) + 64 * hc;
        const uint32_t sq = qc % C::kQStages;
        const uint32_t sd = qc % C::kDoStages;
        // P^T = exp2(S^T * scale * log2 e - L) over this warp's 64 query
        // columns; the S^T columns are released as soon as they are read.
        ok = __all_sync(0xffffffffu, mbar_wait(&q_full[sq], (qc / C::kQStages) & 1, ctl, kWaitBwdSoftmax));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&s_full[reg], (qc >> 1) & 1, ctl, kWaitBwdSoftmax));
        if (!ok) break;
        tc_fence_after();
        uint32_t pv[64];
        tmem_ld32(tZ, pv);
        tmem_ld32(tZ + 32, pv + 32);
        tmem_ld_wait<64>(pv);
        tc_fence_before();
        mbar_arrive_warp(&s_free[reg]);
        {
          const float* bl = sLse + sq * 128 + 64 * hc;
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
        ok = __all_sync(0xffffffffu, mbar_wait(&do_full[sd], (qc / C::kDoStages) & 1, ctl, kWaitBwdSoftmax));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&dp_full[reg], (qc >> 1) & 1, ctl, kWaitBwdSoftmax));
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t dpv[64];
          tmem_ld32(tZ, dpv);
          tmem_ld32(tZ + 32, dpv + 32);
          tmem_ld_wait<64>(dpv);
          const float* bd = sDv + sd * 128 + 64 * hc;
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
        mbar_arrive_warp(&p_ready[reg]);
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
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// --------------------------------------------------------------------- dQ

template <int D>
struct DqCfg {
  static_assert(D == 64 || D == 96 || D == 128, "head dim");
  static constexpr int kChunks = (D + 63) / 64;
  static constexpr int kChunkBytes = kTileM * 128;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kKStages = 3;  // S two steps ahead needs K early
  static constexpr int kVStages = 2;
  static constexpr int kThreads = 384;
  static constexpr uint32_t kColS0 = 0;    // S of even steps, then their dS packed
  static constexpr uint32_t kColS1 = 128;  // S of odd steps, then their dS packed
  static constexpr uint32_t kColDP = 256;  // dP
  static constexpr uint32_t kColDQ = 384;  // dQ accumulator (D columns)
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kTileBytes;
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
  static constexpr int kNumBars = 4 + 2 * kKStages + 2 * kVStages + 9;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
  static_assert(kSmemBytes <= 232448, "shared memory");
};

template <int D>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdParams p) {
  using C = DqCfg<D>;
  using R = BwdRegs;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, (unsigned int)FA_ERR_CUDA);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  // Q_i (read by S only) and dO_i (read by dP only) have separate barriers,
  // so the next unit's tiles load as soon as the last S / dP was issued.
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* do_full = bars + 2;
  uint64_t* do_empty = bars + 3;
  uint64_t* k_full = bars + 4;  // [kKStages]
  uint64_t* k_empty = k_full + C::kKStages;
  uint64_t* v_full = k_empty + C::kKStages;  // [kVStages]
  uint64_t* v_empty = v_full + C::kVStages;
  uint64_t* s_full = v_empty + C::kVStages;  // [2]: S of even / odd steps in TMEM
  uint64_t* dp_full = s_full + 2;            // dP in TMEM
  uint64_t* dp_free = dp_full + 1;           // dP read by all element-wise warps
  uint64_t* p_ready = dp_free + 1;           // [2] dS packed in S buffer 0 / 1
  uint64_t* dq_full = p_ready + 2;           // the unit's dQ complete
  uint64_t* dq_empty = dq_full + 1;          // ... and read out
  uint64_t* drain = dq_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);  // the unit's last S
    mbar_init(do_full, 1);
    mbar_init(do_empty, 1);  // the unit's last dP
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 8);
    mbar_init(&p_ready[0], 8);
    mbar_init(&p_ready[1], 8);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 8);
    mbar_init(drain, 2);  // both MMA issuers
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 9 && lane == 0) {
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

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    reg_dealloc<R::kRegsCtl>();
    if (lane == 0) {
      uint32_t uc = 0, kc = 0;
      uint32_t q_issued = 0, do_issued = 0, k_issued = 0, v_issued = 0;  // copies started (for the drain)
      bool ok = true;
      for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
        const int u = snake_unit(rnd);
        if (u >= p.num_units) continue;
        const BwdUnit w = decode_dq(p, u);
        const int kvbh = p.Hkv == p.H ? w.bh : kv_head_of(w.bh, p.H, p.Hkv);  // K, V head
        ok = mbar_wait(q_empty, (uc & 1) ^ 1, ctl, kWaitBwdLoad);
        if (!ok) break;
        mbar_arrive_expect_tx(q_full, C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(smem + C::kOffQ + c * C::kChunkBytes, &tm_q, q_full, c * 64, w.t * kTileM, w.bh);
        ++q_issued;
        for (int jj = 0; ok && jj < w.count; ++jj, ++kc) {
          const int key0 = (w.first + jj) * kTileN;
          const uint32_t sk = kc % C::kKStages;
          ok = mbar_wait(&k_empty[sk], ((kc / C::kKStages) & 1) ^ 1, ctl, kWaitBwdLoad);
          if (!ok) break;
          mbar_arrive_expect_tx(&k_full[sk], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(smem + C::kOffK + sk * C::kTileBytes + c * C::kChunkBytes, &tm_k, &k_full[sk], c * 64, key0,
                        kvbh);
          ++k_issued;
          if (jj == 0) {
            // dO_i, needed by the first dP, after the first K.
            ok = mbar_wait(do_empty, (uc & 1) ^ 1, ctl, kWaitBwdLoad);
            if (!ok) break;
            mbar_arrive_expect_tx(do_full, C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(smem + C::kOffDO + c * C::kChunkBytes, &tm_do, do_full, c * 64, w.t * kTileM, w.bh);
            ++do_issued;
          }
          const uint32_t sv = kc % C::kVStages;
          ok = mbar_wait(&v_empty[sv], ((kc / C::kVStages) & 1) ^ 1, ctl, kWaitBwdLoad);
          if (!ok) break;
          mbar_arrive_expect_tx(&v_full[sv], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(smem + C::kOffV + sv * C::kTileBytes + c * C::kChunkBytes, &tm_v, &v_full[sv], c * 64, key0,
                        kvbh);
          ++v_issued;
        }
        ++uc;
      }
      // Every copy this thread issued has landed before the CTA exits.
      if (q_issued > 0) mbar_wait(q_full, (q_issued - 1) & 1, ctl, kWaitDrain);
      if (do_issued > 0) mbar_wait(do_full, (do_issued - 1) & 1, ctl, kWaitDrain);
      for (uint32_t pos = k_issued > (uint32_t)C::kKStages ? k_issued - C::kKStages : 0u; pos < k_issued; ++pos)
        mbar_wait(&k_full[pos % C::kKStages], (pos / C::kKStages) & 1, ctl, kWaitDrain);
      for (uint32_t pos = v_issued > (uint32_t)C::kVStages ? v_issued - C::kVStages : 0u; pos < v_issued; ++pos)
        mbar_wait(&v_full[pos % C::kVStages], (pos / C::kVStages) & 1, ctl, kWaitDrain);
    }
    __syncwarp();
  } else if (warp == 8 || warp == 10) {
    // --------------------------------------------------------- MMA issuers
    // Two warps issue the products, each in its own order, so that one
    // warp's waits overlap the other's issue: warp 8 issues dP, warp 10
    // issues dQ and S (S into a buffer after the dQ that read it, in this
    // warp's order).  No product of one reads or writes TMEM columns the
    // other's products touch; each warp's commits track its own products
    // (the elected lane is the same for every instruction of a warp).
    reg_dealloc<R::kRegsCtl>();
    {
      constexpr uint32_t id_s = idesc_bf16(kTileM, kTileN, false, false);  // S, dP
      constexpr uint32_t id_dq = idesc_bf16(kTileM, D, false, true);       // dQ += dS K
      const uint32_t sq = smem_u32(smem + C::kOffQ);
      const uint32_t sdo = smem_u32(smem + C::kOffDO);
      bool ok = true;
      if (warp == 8) {
        // dP of every step, once the previous dP was read out; dO_i is
        // released after the unit's last dP.
        uint32_t uc = 0, kc = 0, dn = 0;
        for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
          const int u = snake_unit(rnd);
          if (u >= p.num_units) continue;
          const BwdUnit w = decode_dq(p, u);
          ok = __all_sync(0xffffffffu, mbar_wait(do_full, uc & 1, ctl, kWaitBwdMma));
          ++uc;
          for (int jj = 0; ok && jj < w.count; ++jj, ++kc) {
            const uint32_t sv = kc % C::kVStages;
            ok = __all_sync(0xffffffffu, mbar_wait(&v_full[sv], (kc / C::kVStages) & 1, ctl, kWaitBwdMma));
            if (ok && dn > 0) ok = __all_sync(0xffffffffu, mbar_wait(dp_free, (dn - 1) & 1, ctl, kWaitBwdMma));
            if (!ok) break;
            tc_fence_after();
            const uint32_t sv_addr = smem_u32(smem + C::kOffV + sv * C::kTileBytes);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk / 4) * C::kChunkBytes + (kk % 4) * 32;
              mma_ss_w(tmem + C::kColDP, sdesc_sw128(sdo + off, 16, 1024), sdesc_sw128(sv_addr + off, 16, 1024),
                     id_s, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(dp_full);
            mma_commit_w(&v_empty[sv]);
            if (jj + 1 == w.count) mma_commit_w(do_empty);
            ++dn;
          }
        }
      } else {
        // dQ += dS K and S two steps ahead.
        uint32_t uc = 0, kc = 0;
        // S of the step at position `pos` into S buffer (pos & 1).  The
        // buffer last held the dS of step pos - 2, read by a dQ product
        // this warp issued earlier; its S was read before that dS was
        // written.  `last`: the unit's last S, after which Q_i is released.
        auto issue_s = [&](uint32_t pos, bool last) -> bool {
          const uint32_t sk = pos % C::kKStages;
          if (!__all_sync(0xffffffffu, mbar_wait(&k_full[sk], (pos / C::kKStages) & 1, ctl, kWaitBwdMma))) return false;
          tc_fence_after();
          const uint32_t sk_addr = smem_u32(smem + C::kOffK + sk * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * C::kChunkBytes + (kk % 4) * 32;
            mma_ss_w(tmem + ((pos & 1) ? C::kColS1 : C::kColS0), sdesc_sw128(sq + off, 16, 1024),
                   sdesc_sw128(sk_addr + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
          }
          mma_commit_w(&s_full[pos & 1]);
          if (last) mma_commit_w(q_empty);
          return true;
        };
        for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
          const int u = snake_unit(rnd);
          if (u >= p.num_units) continue;
          const BwdUnit w = decode_dq(p, u);
          ok = __all_sync(0xffffffffu, mbar_wait(q_full, uc & 1, ctl, kWaitBwdMma));
          if (!ok) break;
          tc_fence_after();
          ok = issue_s(kc, w.count == 1);
          if (ok && w.count > 1) ok = issue_s(kc + 1, w.count == 2);
          for (int jj = 0; ok && jj < w.count; ++jj, ++kc) {
            ok = __all_sync(0xffffffffu, mbar_wait(&p_ready[kc & 1], (kc >> 1) & 1, ctl, kWaitBwdMma));
            if (!ok) break;
            if (jj == 0 && uc > 0) {
              // The previous unit's dQ has been read out of TMEM.
              ok = __all_sync(0xffffffffu, mbar_wait(dq_empty, (uc - 1) & 1, ctl, kWaitBwdMma));
              if (!ok) break;
            }
            tc_fence_after();
            // dQ += dS K_j: A = dS (bf16 pairs in the step's S buffer), B =
            // K_j read MN-major (N = head dim, K = keys).
            const uint32_t sk = kc % C::kKStages;
            const uint32_t sk_addr = smem_u32(smem + C::kOffK + sk * C::kTileBytes);
            const uint32_t ds_col = (kc & 1) ? C::kColS1 : C::kColS0;
#pragma unroll
            for (int kk = 0; kk < kTileN / 16; ++kk)
              mma_ts_w(tmem + C::kColDQ, tmem + ds_col + packed_col(kk, false),
                     sdesc_sw128(sk_addr + kk * 2048, C::kChunkBytes, 1024), id_dq, (jj > 0 || kk > 0) ? 1u : 0u);
            mma_commit_w(&k_empty[sk]);
            // S two steps ahead, into the buffer this dQ product reads from.
            if (jj + 2 < w.count) {
              ok = issue_s(kc + 2, jj + 3 == w.count);
              if (!ok) break;
            }
          }
          if (!ok) break;
          mma_commit_w(dq_full);
          ++uc;
        }
      }
      mma_commit_w(drain);
      (void)__all_sync(0xffffffffu, mbar_wait(drain, 0, ctl, kWaitDrain));
    }
    __syncwarp();
  } else if (warp < 8) {
    // --------------------------------------------------- P, dS and dQ output
    reg_alloc<R::kRegsMath>();
    const int g = warp & 3;    // TMEM lane quarter: queries [32 g, 32 g + 32)
    const int hc = warp >> 2;  // key-column half
    const uint32_t lane_off = (uint32_t)(32 * g) << 16;
    const float sl2 = p.scale_log2;
    uint32_t uc = 0, kc = 0, dc = 0;
    bool ok = true;
    // dQ_i = scale * sum dS K of a unit: lane = query row q of head `head`,
    // this warp writes head-dim columns [D/2 hc, D/2 hc + D/2).  Run after
    // the next unit's first P, while its dP is computed.
    // This warp's columns [c0, c0 + NC) of the row (RowSplit), read out of
    // TMEM, released, then scaled, packed and stored.  One row per lane
    // here: the dQ stores follow the TMEM release and overlap the next
    // unit's first steps, and the shuffles of store_rows measured slower
    // than the scattered lines they save.
    auto write_part = [&](auto nc_tag, int q, size_t head) {
      constexpr int NC = decltype(nc_tag)::value;
      const int c0 = hc ? RowSplit<D>::kLo : 0;
      uint32_t v[NC];
#pragma unroll
      for (int c = 0; c < NC / 32; ++c) tmem_ld32(tmem + lane_off + C::kColDQ + c0 + 32 * c, v + 32 * c);
      tmem_ld_wait<NC>(v);
      tc_fence_before();
      mbar_arrive_warp(dq_empty);
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.dq) + (head + q) * D + c0;
      const float sc = p.scale;
      uint32_t w[NC / 2];
#pragma unroll
      for (int i = 0; i < NC / 2; ++i)
        w[i] = pack_bf16(__uint_as_float(v[2 * i]) * sc, __uint_as_float(v[2 * i + 1]) * sc);
      if (q < p.Nq) {
        if (p.store32) {
#pragma unroll
          for (int i = 0; i < NC / 16; ++i) st_global_v8(dst + 16 * i, w + 8 * i);
        } else {
#pragma unroll
          for (int i = 0; i < NC / 8; ++i)
            reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    };
    auto write_dq = [&](int q, size_t head) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(dq_full, uc & 1, ctl, kWaitBwdDq))) return false;
      ++uc;
      tc_fence_after();
      if constexpr (RowSplit<D>::kLo == RowSplit<D>::kHi) {
        write_part(std::integral_constant<int, RowSplit<D>::kLo>{}, q, head);
      } else {
        if (hc == 0)
          write_part(std::integral_constant<int, RowSplit<D>::kLo>{}, q, head);
        else
          write_part(std::integral_constant<int, RowSplit<D>::kHi>{}, q, head);
      }
      return true;
    };
    int pend_q = -1;  // the unit whose dQ is still in TMEM
    size_t pend_head = 0;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units) continue;
      const BwdUnit w = decode_dq(p, u);
      const size_t head = (size_t)w.bh * p.Nq;
      const int q = w.t * kTileM + 32 * g + lane;  // query row
      const float Lraw = q < p.Nq ? p.lse[head + q] : INFINITY;
      const float L = Lraw == -INFINITY ? INFINITY : Lraw * 1.4426950408889634f;  // no key seen: weights 0
      const float Dq = q < p.Nq ? p.dvec[head + q] : 0.f;
      const int q_lo = w.t * kTileM + 32 * g;  // first query of this warp
      for (int jj = 0; ok && jj < w.count; ++jj, ++kc) {
        const uint32_t tS = tmem + lane_off + ((kc & 1) ? C::kColS1 : C::kColS0) + 64 * hc;
        const int k_first = (w.first + jj) * kTileN + 64 * hc;
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[kc & 1], (kc >> 1) & 1, ctl, kWaitBwdSoftmax));
        if (!ok) break;
        tc_fence_after();
        uint32_t pv[64];
        tmem_ld32(tS, pv);
        tmem_ld32(tS + 32, pv + 32);
        tmem_ld_wait<64>(pv);
        if (k_first + 63 >= p.Nk || (p.causal && k_first + 63 > q_lo + p.causal_off))
          p64_rowL<true>(pv, L, sl2, q + p.causal_off, k_first, p.Nk, p.causal != 0);
        else
          p64_rowL<false>(pv, L, sl2, q, k_first, p.Nk, false);
        if (jj == 0 && pend_q >= 0) {
          ok = write_dq(pend_q, pend_head);
          if (!ok) break;
        }
        ok = __all_sync(0xffffffffu, mbar_wait(dp_full, dc & 1, ctl, kWaitBwdSoftmax));
        ++dc;
        if (!ok) break;
        tc_fence_after();
        uint32_t dk[32];
        {
          uint32_t dpv[64];
          tmem_ld32(tmem + lane_off + C::kColDP + 64 * hc, dpv);
          tmem_ld32(tmem + lane_off + C::kColDP + 64 * hc + 32, dpv + 32);
          tmem_ld_wait<64>(dpv);
          tc_fence_before();
          mbar_arrive_warp(dp_free);
          const float2 dv2 = make_float2(-Dq, -Dq);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 g2 =
                __fadd2_rn(make_float2(__uint_as_float(dpv[2 * e]), __uint_as_float(dpv[2 * e + 1])), dv2);
            const float2 ds =
                __fmul2_rn(make_float2(__uint_as_float(pv[2 * e]), __uint_as_float(pv[2 * e + 1])), g2);
            dk[e] = pack_bf16(ds.x, ds.y);
          }
        }
        // dS as bf16 pairs over this warp's S columns (already read).
        tmem_st32(tS, dk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&p_ready[kc & 1]);
      }
      if (!ok) break;
      pend_q = q;
      pend_head = head;
    }
    if (ok && pend_q >= 0) write_dq(pend_q, pend_head);
  } else {
    reg_dealloc<R::kRegsCtl>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// D_i = sum_c dO_ic * O_ic.  D/8 lanes per row, 16 bytes of O and of dO
// per lane; a block reads 256 / (D/8) consecutive rows per pass (whole rows,
// 16-byte accesses) and kRowsPerThread passes, whose loads are all issued
// before any is used so that enough bytes are in flight to stream from DRAM.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_preprocess(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dout,
                                                         float* __restrict__ dvec, int rows) {
  // Launched while the kernel before it (the forward, writing O) may still
  // run: its writes are read here.
  pdl_wait();
  constexpr int kVec = (D == 96) ? 3 : 1;     // 16-byte pieces per lane (lanes per row a power of two)
  constexpr int kLanes = D / (8 * kVec);      // lanes per row
  constexpr int kSlots = 256 / kLanes;        // rows per pass
  constexpr int kRowsPerThread = 4;           // passes
  const int part = threadIdx.x % kLanes;
  const int slot = threadIdx.x / kLanes;
  const int base = blockIdx.x * kSlots * kRowsPerThread;
  uint4 a[kRowsPerThread][kVec], b[kRowsPerThread][kVec];
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r) {
    const int row = base + r * kSlots + slot;
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      if (row < rows) {
        a[r][v] = reinterpret_cast<const uint4*>(o + (size_t)row * D)[part * kVec + v];
        b[r][v] = reinterpret_cast<const uint4*>(dout + (size_t)row * D)[part * kVec + v];
      } else {
        a[r][v] = make_uint4(0u, 0u, 0u, 0u);
        b[r][v] = a[r][v];
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r) {
    float acc = 0.f;
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[r][v]);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b[r][v]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(a2[i]);
        const float2 y = __bfloat1622float2(b2[i]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
#pragma unroll
    for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const int row = base + r * kSlots + slot;
    if (row < rows && part == 0) dvec[row] = acc;
  }
}

// A wait on an mbarrier that nothing arrives on: exercises the give-up path.
__global__ void fa_selftest_wait_kernel(unsigned int* status, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const WaitCtl ctl{status, timeout_ns};
  mbar_wait(&bar, 0, ctl, kWaitSelfTest);
}

// ------------------------------------------------------------------ launch

template <int D, bool GQA>
static cudaError_t launch_dkdv_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream) {
  using C = DkdvCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(fa_bwd_dkdv_kernel<D, GQA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(fa_bwd_dkdv_kernel<D, GQA>, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, tq, tk, tv, tdo, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_dq_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream) {
  using C = DqCfg<D>;
  cudaError_t e =
      cudaFuncSetAttribute(fa_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // May start as the dK/dV kernel's CTAs finish: it reads only the inputs,
  // L and D, and D was complete before any dK/dV CTA let it start.
  e = launch_pdl(fa_bwd_dq_kernel<D>, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, tq, tk, tv, tdo, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream) {
  const bool gqa = p.Hkv != p.H;
  switch (d) {
    case 64:
      return gqa ? launch_dkdv_t<64, true>(tq, tk, tv, tdo, p, grid, stream)
                 : launch_dkdv_t<64, false>(tq, tk, tv, tdo, p, grid, stream);
    case 96:
      return gqa ? launch_dkdv_t<96, true>(tq, tk, tv, tdo, p, grid, stream)
                 : launch_dkdv_t<96, false>(tq, tk, tv, tdo, p, grid, stream);
    case 128:
      return gqa ? launch_dkdv_t<128, true>(tq, tk, tv, tdo, p, grid, stream)
                 : launch_dkdv_t<128, false>(tq, tk, tv, tdo, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_dq(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream) {
  switch (d) {
    case 64: return launch_dq_t<64>(tq, tk, tv, tdo, p, grid, stream);
    case 96: return launch_dq_t<96>(tq, tk, tv, tdo, p, grid, stream);
    case 128: return launch_dq_t<128>(tq, tk, tv, tdo, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
static cudaError_t launch_pre_t(const void* o, const void* dout, float* dvec, int rows, cudaStream_t stream) {
  constexpr int kVec = (D == 96) ? 3 : 1;
  const int per_block = (256 / (D / (8 * kVec))) * 4;  // rows per 256-thread block (4 passes)
  const int grid = (rows + per_block - 1) / per_block;
  const cudaError_t e = launch_pdl(fa_bwd_preprocess<D>, dim3(grid), dim3(256), 0, stream,
                                   static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout),
                                   dvec, rows);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess(int d, const void* o, const void* dout, float* dvec, int rows,
                                  cudaStream_t stream) {
  switch (d) {
    case 64: return launch_pre_t<64>(o, dout, dvec, rows, stream);
    case 96: return launch_pre_t<96>(o, dout, dvec, rows, stream);
    case 128: return launch_pre_t<128>(o, dout, dvec, rows, stream);
    case 256: return launch_pre_t<256>(o, dout, dvec, rows, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_selftest_wait(unsigned int* status, unsigned long long timeout_ns, cudaStream_t stream) {
  fa_selftest_wait_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fa
