// Forward pass of exact attention on sm_103a, FlashAttention-2 style
// ("FlashAttention V2 in depth", section 6.1; FlashAttention-2 abstract).
//
// One persistent CTA per SM walks a static list of work units
// (batch*head, 256-row query block, key split).  A unit holds two 128-row
// query tiles Q0, Q1 that stay in shared memory (loaded once, section 2.3)
// and share one stream of 128-key K/V tiles (the inner loop).  Roles:
//   warp 9     TMA producer: Q tiles, then K_j, V_j into a ring of slots.
//              A Q buffer is refilled as soon as the last S product that
//              reads it has completed, so the next unit's Q, K and V arrive
//              while the current unit's last steps run.
//   warp 8     MMA issuer (the whole warp walks the schedule, one elected
//              lane issues): S_t = Q_t K_j^T and O_t += P_t V_j with tcgen05
//              into tensor memory (TMEM).  With grouped-query attention the
//              K, V tiles are those of the query head's key/value head.
//   warps 0-3  softmax of query tile 0, warps 4-7 of tile 1: each thread owns
//              one query row (the "split along Q" of section 4.2), so row max
//              and row sum need no communication.  They also write O and L
//              straight from registers at the end of the unit.
// TMEM (512 columns): S0 | S1 | O0 | O1.  P (bf16) overwrites the first half
// of its own S columns and feeds the PV MMA straight from TMEM.
//
// Online softmax (section 6.1): the running max m and sum l live in registers
// of the row's thread, O~ stays unnormalised in TMEM and is divided by l
// once at the end; L = m + log l is written for the backward pass.  P is
// rounded to bf16 for the PV MMA, and O~ is divided by the sum of those
// rounded weights, so O is an exact weighted mean of the rows of V under the
// weights the MMA used; L takes the sum of the unrounded fp32 weights.  The
// exp(m_old - m_new) correction of O~ is applied only when a row's max grows
// by more than a factor 2^24 over the reference the row's O~ and l are kept
// at; otherwise the old reference stays.  O~ and l always share one
// reference, so the final O~/l is the same; the weights exp(S - m_ref) stay
// <= 2^24, which bf16 P and the fp32 sums and accumulator hold with their
// usual relative precision.  (With peaky rows, logits of standard deviation
// 9, a threshold of 2^8 let most rows correct O~ several times: the GPT-layer
// forward ran 7% slower.)
//
// Causal mask (section 5): key tiles past a query tile's last row are never
// loaded or multiplied; only tiles crossing the diagonal (and the ragged last
// key tile) are masked element by element.  Queries and keys may differ in
// length; row i then sees keys j <= i + causal_off (0: top-left alignment,
// Nk - Nq: bottom-right).  A row that sees no key writes O = 0, L = -inf.
//
// Head dims 64, 96 and 128.  A 96-wide row is staged in the 128-wide layout
// (two 64-column blocks; TMA fills columns 96..127 with zeros) while the
// products use K = 96 (S) and N = 96 (O) exactly.
//
// Units of at most 128 query rows (decoding) would leave tile 1 idle: in
// the dual instantiation both tiles hold the unit's rows, tile t takes the
// key tiles kvb + t, kvb + t + 2, ... of its split, and each writes its own
// fp32 partial result, merged afterwards like the split partials.
#include <cuda_runtime.h>

#include "sm103_primitives.cuh"

namespace fa {

using namespace dev;

template <int D>
struct FwdCfg {
  static_assert(D == 64 || D == 96 || D == 128, "head dim");
  static constexpr int kChunks = (D + 63) / 64;        // 128-byte column blocks per row
  static constexpr int kChunkBytes = kTileM * 128;     // one 128-row x 64-column block
  static constexpr int kTileBytes = kChunks * kChunkBytes;  // one 128-row tile (padded to 64 columns)
  static constexpr int kStages = (D == 64) ? 8 : 4;    // K/V ring slots
  static constexpr int kOCols = kChunks * 64;          // TMEM columns given to one O tile
  // Three warpgroups: 0-1 softmax (one 128-row Q tile each), 2 the MMA
  // issuer (warp 8), the TMA producer (warp 9) and two idle warps.
  static constexpr int kThreads = 384;
  __host__ __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + (uint32_t)kOCols * t; }
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kTileBytes;
  static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
  static constexpr int kNumBars = 2 + 2 + 2 * kStages + 2 + 2 + 2 + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
  static constexpr float kRescaleThreshold = 24.0f;    // log2 units
  // Register split (setmaxnreg).  At 384 threads and one CTA per SM each
  // thread starts with 168 registers (three warps per SM sub-partition share
  // its 16384); warpgroup 2 hands registers back so the softmax warpgroups,
  // which hold a whole 128-column S row, get 216.  The shares must not exceed
  // what the CTA was launched with, or the increase waits forever.
  static constexpr int kRegsAtLaunch = 168;
  static constexpr int kRegsCtl = 72;
  static constexpr int kRegsMath = 216;
  static_assert(128 * kRegsCtl + 256 * kRegsMath <= kThreads * kRegsAtLaunch, "register split exceeds the launch");
  static_assert(kRegsCtl % 8 == 0 && kRegsMath % 8 == 0, "setmaxnreg counts are multiples of 8");
};

struct Unit {
  int bh;
  int q0;     // first query row of the 256-row block
  int kvb;    // first key tile of this split
  int n[2];   // key tiles processed by query tile 0 / 1 (0 = none)
  int split;
};

// Key tile (from kvb) of query tile t's j-th step, and the unit's first
// query row of tile t (both tiles hold the same rows in dual mode).
template <bool DUAL>
__device__ __forceinline__ int step_key_tile(int t, int j) { return DUAL ? 2 * j + t : j; }
template <bool DUAL>
__device__ __forceinline__ int tile_row0(const Unit& w, int t) {
  return DUAL ? w.q0 : w.q0 + kTileM * t;
}

template <bool DUAL>
__device__ __forceinline__ Unit decode_unit(const FwdParams& p, int u) {
  Unit w;
  const int split = u % p.num_splits;
  const int r = u / p.num_splits;
  const int BH = p.B * p.H;
  // Query blocks in decreasing order: with the causal mask the last blocks
  // carry the most key tiles, so they start first (longest job first).
  // Without the mask, head windows (FwdParams::head_window).
  int qb;
  if (p.head_window > 0) {
    const int per_window = p.head_window * p.num_q_blocks;
    const int win = r / per_window;
    const int heads = min(p.head_window, BH - win * p.head_window);
    const int rr = r - win * per_window;
    w.bh = win * p.head_window + rr % heads;
    qb = p.num_q_blocks - 1 - rr / heads;
  } else {
    w.bh = r % BH;
    qb = p.num_q_blocks - 1 - r / BH;
  }
  w.q0 = qb * (kTileM * kQTilesPerCta);
  const int nkv = (p.Nk + kTileN - 1) / kTileN;
  const int lo = split * p.kv_tiles_per_split;
  const int hi = min(nkv, lo + p.kv_tiles_per_split);
  w.kvb = lo;
  w.split = split;
  if constexpr (DUAL) {
    // Both tiles: the rows of tile 0; the keys they see split by parity.
    int h = hi;
    if (p.causal) {
      const int last_key = max_query_pos(w.q0, min(p.Nq, w.q0 + kTileM) - 1, p.q_period) + p.causal_off;
      h = last_key < 0 ? 0 : min(hi, last_key / kTileN + 1);
    }
    const int nk = w.q0 < p.Nq ? max(0, h - lo) : 0;
    w.n[0] = (nk + 1) / 2;
    w.n[1] = nk / 2;
    return w;
  }
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int row0 = w.q0 + kTileM * t;
    if (row0 >= p.Nq) {
      w.n[t] = 0;
    } else {
      int h = hi;
      if (p.causal) {
        // The last key any row of the tile sees; none if it is negative.
        const int last_key = max_query_pos(row0, min(p.Nq, row0 + kTileM) - 1, p.q_period) + p.causal_off;
        h = last_key < 0 ? 0 : min(hi, last_key / kTileN + 1);
      }
      w.n[t] = max(0, h - lo);
    }
  }
  return w;
}

// Key tiles a unit streams through the K/V ring (both tiles' in dual mode).
template <bool DUAL>
__device__ __forceinline__ int unit_key_tiles(const Unit& w) {
  return DUAL ? w.n[0] + w.n[1] : max(w.n[0], w.n[1]);
}

// S = Q K^T: 16-wide K-steps walk 32 bytes inside a 128-byte swizzle row
// (four per 64-column block), then the next 64-column block.  Descriptors
// come as precomputed halves; a K-step only adds to the start address.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tmem_s, uint32_t q_lo, uint32_t k_lo, uint32_t hi) {
  using C = FwdCfg<D>;
  constexpr uint32_t idesc = idesc_bf16(kTileM, kTileN, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk / 4) * C::kChunkBytes + (kk % 4) * 32) >> 4;
    mma_ss_lh_w(tmem_s, q_lo + off, hi, k_lo + off, hi, idesc, kk > 0 ? 1u : 0u);
  }
}

// O += P V: P from TMEM (8 columns per 16 keys), V read MN-major, 16 key rows
// (2048 bytes) per K-step.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_lo, uint32_t hi,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16(kTileM, D, false, true);
#pragma unroll
  for (int kk = 0; kk < kTileN / 16; ++kk)
    mma_ts_lh_w(tmem_o, tmem_p + kk * 8, v_lo + ((kk * 2048) >> 4), hi, idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// DUAL: p.dual (both query tiles on one unit's rows), a separate
// instantiation so the usual path carries none of it.
template <int D, bool DUAL>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // The 128-byte swizzle anchors at 1024-byte boundaries: refuse to run (and
  // report) if the dynamic shared memory base is not aligned.
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, (unsigned int)FA_ERR_CUDA);
    return;
  }
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sKV = smem + C::kOffKV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 2;
  uint64_t* kv_full = bars + 4;
  uint64_t* kv_empty = kv_full + C::kStages;
  uint64_t* s_full = kv_empty + C::kStages;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint64_t* drain = o_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&o_full[i], 1);
    }
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{p.status, p.timeout_ns};
  if (warp == 9) {
    reg_dealloc<C::kRegsCtl>();
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t rc = 0;
      uint32_t qc[2] = {0, 0};
      bool ok = true;
      for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
        const int u = snake_unit(rnd);
        if (u >= p.num_units) continue;
        const Unit w = decode_unit<DUAL>(p, u);
        const int kvbh = p.Hkv == p.H ? w.bh : kv_head_of(w.bh, p.H, p.Hkv);  // K, V head
        for (int t = 0; ok && t < 2; ++t) {
          if (w.n[t] == 0) continue;
          ok = mbar_wait(&q_empty[t], (qc[t] & 1) ^ 1, ctl, kWaitQEmpty);
          if (!ok) break;
          mbar_arrive_expect_tx(&q_full[t], C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(sQ + t * C::kTileBytes + c * C::kChunkBytes, &tm_q, &q_full[t], c * 64,
                        tile_row0<DUAL>(w, t), w.bh);
          ++qc[t];
        }
        const int nk = unit_key_tiles<DUAL>(w);
        for (int j = 0; ok && j < nk; ++j) {
          for (int which = 0; which < 2; ++which) {
            const uint32_t slot = rc % C::kStages;
            ok = mbar_wait(&kv_empty[slot], ((rc / C::kStages) & 1) ^ 1, ctl, kWaitKvEmpty);
            if (!ok) break;
            mbar_arrive_expect_tx(&kv_full[slot], C::kTileBytes);
            const CUtensorMap* m = which ? &tm_v : &tm_k;
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(sKV + slot * C::kTileBytes + c * C::kChunkBytes, m, &kv_full[slot], c * 64,
                          (w.kvb + j) * kTileN, kvbh);
            ++rc;
          }
        }
      }
      // Let every copy this thread started land before the CTA can exit.
      const uint32_t first = rc > (uint32_t)C::kStages ? rc - C::kStages : 0u;
      for (uint32_t pos = first; pos < rc; ++pos)
        mbar_wait(&kv_full[pos % C::kStages], (pos / C::kStages) & 1, ctl, kWaitDrain);
      for (int t = 0; t < 2; ++t)
        if (qc[t] > 0) mbar_wait(&q_full[t], (qc[t] - 1) & 1, ctl, kWaitDrain);
    }
  } else if (warp == 8) {
    reg_dealloc<C::kRegsCtl>();
    // ---------------------------------------------------------- MMA issuer
    // The whole warp walks the schedule (operands stay warp-uniform); one
    // elected lane issues each tcgen05.mma / commit.
    {
      // Descriptor low halves: buffer i of a kind is (i * tile bytes) / 16
      // past the first; V differs from K only in its leading byte offset.
      constexpr uint32_t hi = sdesc_hi(1024);
      constexpr uint32_t kTileStep = C::kTileBytes >> 4;
      const uint32_t q_lo0 = sdesc_lo(smem_u32(sQ), 16);
      const uint32_t k_lo0 = sdesc_lo(smem_u32(sKV), 16);
      const uint32_t v_lo0 = sdesc_lo(smem_u32(sKV), C::kChunkBytes);
      uint32_t rc = 0;
      uint32_t qc[2] = {0, 0}, pc[2] = {0, 0};
      bool ok = true;
      for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
        const int u = snake_unit(rnd);
        if (u >= p.num_units) continue;
        const Unit w = decode_unit<DUAL>(p, u);
        const int nmax = max(w.n[0], w.n[1]);
        if (nmax == 0) continue;
        for (int t = 0; ok && t < 2; ++t) {
          if (w.n[t] == 0) continue;
          ok = __all_sync(0xffffffffu, mbar_wait(&q_full[t], qc[t] & 1, ctl, kWaitQFull));
          ++qc[t];
        }
        if (!ok) break;
        if constexpr (DUAL) {
          // Dual mode: tile t's step j reads key tile 2j + t (K at position
          // rc + 2 (2j + t), V one after it); each K and V has one reader
          // and is released after its product.
          for (int t = 0; ok && t < 2; ++t) {
            if (w.n[t] == 0) continue;
            const uint32_t pos_k = rc + 2 * t;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&kv_full[pos_k % C::kStages], (pos_k / C::kStages) & 1, ctl, kWaitKvFull));
            if (!ok) break;
            tc_fence_after();
            issue_qk<D>(tmem + C::col_s(t), q_lo0 + t * kTileStep, k_lo0 + (pos_k % C::kStages) * kTileStep, hi);
            mma_commit_w(&s_full[t]);
            if (w.n[t] == 1) mma_commit_w(&q_empty[t]);  // Q_t's last product
            mma_commit_w(&kv_empty[pos_k % C::kStages]);
          }
          for (int j = 0; ok && j < nmax; ++j) {
            for (int t = 0; t < 2; ++t) {
              if (j >= w.n[t]) continue;
              const uint32_t pos_v = rc + 2 * (2 * j + t) + 1;
              ok = __all_sync(0xffffffffu,
                              mbar_wait(&kv_full[pos_v % C::kStages], (pos_v / C::kStages) & 1, ctl, kWaitKvFull));
              if (!ok) break;
              ok = __all_sync(0xffffffffu, mbar_wait(&p_full[t], pc[t] & 1, ctl, kWaitPFull));
              ++pc[t];
              if (!ok) break;
              tc_fence_after();
              issue_pv<D>(tmem + C::col_o(t), tmem + C::col_s(t), v_lo0 + (pos_v % C::kStages) * kTileStep, hi, j > 0);
              mma_commit_w(&kv_empty[pos_v % C::kStages]);
              if (j + 1 < w.n[t]) {
                const uint32_t pos_k = rc + 2 * (2 * (j + 1) + t);
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&kv_full[pos_k % C::kStages], (pos_k / C::kStages) & 1, ctl, kWaitKvFull));
                if (!ok) break;
                tc_fence_after();
                issue_qk<D>(tmem + C::col_s(t), q_lo0 + t * kTileStep, k_lo0 + (pos_k % C::kStages) * kTileStep, hi);
                mma_commit_w(&s_full[t]);
                if (j + 2 == w.n[t]) mma_commit_w(&q_empty[t]);  // Q_t's last product
                mma_commit_w(&kv_empty[pos_k % C::kStages]);
              } else {
                mma_commit_w(&o_full[t]);
              }
            }
          }
          rc += 2 * unit_key_tiles<DUAL>(w);
          continue;
        }
        {
          const uint32_t slot_k = rc % C::kStages;
          ok = __all_sync(0xffffffffu, mbar_wait(&kv_full[slot_k], (rc / C::kStages) & 1, ctl, kWaitKvFull));
          if (!ok) break;
          tc_fence_after();
          for (int t = 0; t < 2; ++t) {
            if (w.n[t] == 0) continue;
            issue_qk<D>(tmem + C::col_s(t), q_lo0 + t * kTileStep, k_lo0 + slot_k * kTileStep, hi);
            mma_commit_w(&s_full[t]);
            if (w.n[t] == 1) mma_commit_w(&q_empty[t]);  // Q_t's last product
          }
          mma_commit_w(&kv_empty[slot_k]);
        }
        for (int j = 0; ok && j < nmax; ++j) {
          const uint32_t pos_v = rc + 2 * j + 1;
          const uint32_t pos_k = pos_v + 1;
          const uint32_t slot_v = pos_v % C::kStages;
          const uint32_t slot_k = pos_k % C::kStages;
          ok = __all_sync(0xffffffffu, mbar_wait(&kv_full[slot_v], (pos_v / C::kStages) & 1, ctl, kWaitKvFull));
          if (!ok) break;
          tc_fence_after();
          bool k_ready = false;
          for (int t = 0; t < 2; ++t) {
            if (j >= w.n[t]) continue;
            ok = __all_sync(0xffffffffu, mbar_wait(&p_full[t], pc[t] & 1, ctl, kWaitPFull));
            ++pc[t];
            if (!ok) break;
            tc_fence_after();
            issue_pv<D>(tmem + C::col_o(t), tmem + C::col_s(t), v_lo0 + slot_v * kTileStep, hi, j > 0);
            if (j + 1 < w.n[t]) {
              if (!k_ready) {
                ok = __all_sync(0xffffffffu, mbar_wait(&kv_full[slot_k], (pos_k / C::kStages) & 1, ctl, kWaitKvFull));
                if (!ok) break;
                tc_fence_after();
                k_ready = true;
              }
              issue_qk<D>(tmem + C::col_s(t), q_lo0 + t * kTileStep, k_lo0 + slot_k * kTileStep, hi);
              mma_commit_w(&s_full[t]);
              if (j + 2 == w.n[t]) mma_commit_w(&q_empty[t]);  // Q_t's last product
            } else {
              mma_commit_w(&o_full[t]);
            }
          }
          if (!ok) break;
          mma_commit_w(&kv_empty[slot_v]);
          if (j + 1 < nmax) mma_commit_w(&kv_empty[slot_k]);
        }
        rc += 2 * nmax;
      }
      // Every MMA this warp issued completes before TMEM is released.
      mma_commit_w(drain);
      (void)__all_sync(0xffffffffu, mbar_wait(drain, 0, ctl, kWaitDrain));
    }
    __syncwarp();
  } else if (warp < 8) {
    reg_alloc<C::kRegsMath>();
    // ------------------------------------------------------------- softmax
    const int t = warp >> 2;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_off + C::col_s(t);
    const uint32_t tO = tmem + lane_off + C::col_o(t);
    const int r_in_tile = 32 * (warp & 3) + lane;
    const float sl2 = p.scale_log2;
    uint32_t sc = 0, oc = 0;
    bool ok = true;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units) continue;
      const Unit w = decode_unit<DUAL>(p, u);
      const int row0 = tile_row0<DUAL>(w, t);
      const int row = row0 + r_in_tile;
      // Partial result this tile writes (one per split; two in dual mode).
      const int part = DUAL ? 2 * w.split + t : w.split;
      const bool partial = DUAL || p.num_splits > 1;
      if (w.n[t] == 0) {
        // No row of the tile sees a key (of this split): O = 0, L = -inf
        // (an empty partial when the keys are split).
        if (row < p.Nq) {
          if (partial) {
            const size_t prow = ((size_t)part * p.B * p.H + w.bh) * p.Nq + row;
            float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
            for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            p.lse_part[prow] = -INFINITY;
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.o) + ((size_t)w.bh * p.Nq + row) * (D * 2));
            for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
            p.lse[(size_t)w.bh * p.Nq + row] = -INFINITY;
          }
        }
        continue;
      }
      float m_ref = -INFINITY;  // reference max of this row, log2 units
      float l = 0.f;     // sum of the fp32 weights: L = m + log l
      float l_bf = 0.f;  // sum of the bf16-rounded weights the PV MMA takes: O = O~ / l_bf
      for (int j = 0; j < w.n[t]; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], sc & 1, ctl, kWaitSFull));
        ++sc;
        if (!ok) break;
        tc_fence_after();
        uint32_t s[kTileN];
#pragma unroll
        for (int c = 0; c < kTileN / 32; ++c) tmem_ld32(tS + 32 * c, s + 32 * c);
        tmem_ld_wait<kTileN>(s);
        float x[kTileN];
#pragma unroll
        for (int c = 0; c < kTileN; ++c) x[c] = __uint_as_float(s[c]);
        const int kv0 = (w.kvb + step_key_tile<DUAL>(t, j)) * kTileN;
        const bool need_mask = (kv0 + kTileN > p.Nk) ||
                               (p.causal && (p.q_period > 0 || kv0 + kTileN - 1 > row0 + p.causal_off));
        if (need_mask) {
          const int lim = p.causal ? min(p.Nk - 1, query_pos(row, p.q_period) + p.causal_off) : p.Nk - 1;  // last visible key
#pragma unroll
          for (int c = 0; c < kTileN; ++c)
            if (kv0 + c > lim) x[c] = -INFINITY;
        }
        float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
        for (int c = 4; c + 8 <= kTileN; c += 8) {
          mx0 = fmax3(mx0, x[c], x[c + 1]);
          mx1 = fmax3(mx1, x[c + 2], x[c + 3]);
          mx2 = fmax3(mx2, x[c + 4], x[c + 5]);
          mx3 = fmax3(mx3, x[c + 6], x[c + 7]);
        }
        mx0 = fmax3(mx0, x[kTileN - 4], x[kTileN - 3]);  // the last four columns
        mx1 = fmax3(mx1, x[kTileN - 2], x[kTileN - 1]);
        const float m_tile = fmax3(fmaxf(mx0, mx1), mx2, mx3) * sl2;
        // m_ref stays -inf while the row has seen no key; the first key it
        // sees then takes the rescale path with f = 0 (l and O~ are 0).
        float f = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_ref = m_tile;
        } else if (__any_sync(0xffffffffu, m_tile > m_ref + C::kRescaleThreshold)) {
          const float m_new = fmaxf(m_ref, m_tile);
          f = (m_new == -INFINITY) ? 1.f : ex2_approx(m_ref - m_new);
          l *= f;
          l_bf *= f;
          m_ref = m_new;
          rescale = true;
        }
        const float m_exp = (m_ref == -INFINITY) ? 0.f : m_ref;  // exponent reference (all weights 0 if -inf)
        // P = exp2(S * scale * log2(e) - m_ref), 32 columns at a time, packed
        // to bf16 over the already-read S columns; pairs of columns share the
        // packed fp32x2 FMA and adds.  The rounded weights are summed from
        // the packed pairs (each half converted exactly to fp32).
        const float2 sl2v = make_float2(sl2, sl2);
        const float2 negv = make_float2(-m_exp, -m_exp);
        float2 ls0 = make_float2(0.f, 0.f), ls1 = ls0;
        float lr0 = 0.f, lr1 = 0.f, lr2 = 0.f, lr3 = 0.f;
#pragma unroll
        for (int h = 0; h < kTileN / 32; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 a = __ffma2_rn(make_float2(x[32 * h + e], x[32 * h + e + 1]), sl2v, negv);
            const float p0 = ex2_approx(a.x);
            const float p1 = ex2_approx(a.y);
            const uint32_t pp = pack_bf16(p0, p1);
            if ((e >> 1) & 1) {
              ls1 = __fadd2_rn(ls1, make_float2(p0, p1));
              lr2 = add_bf16_lo(lr2, pp);
              lr3 = add_bf16_hi(lr3, pp);
            } else {
              ls0 = __fadd2_rn(ls0, make_float2(p0, p1));
              lr0 = add_bf16_lo(lr0, pp);
              lr1 = add_bf16_hi(lr1, pp);
            }
            pk[e / 2] = pp;
          }
          tmem_st16(tS + 16 * h, pk);
        }
        l += (ls0.x + ls0.y) + (ls1.x + ls1.y);
        l_bf += (lr0 + lr1) + (lr2 + lr3);
        if (rescale) {
          // O~ <- exp2(m_old - m_new) O~; the previous PV MMA has completed
          // (it was issued before this S tile's MMA) and the next one waits
          // for the arrive below.
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_ld_wait<32>(o);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                          make_float2(f, f));
              o[i] = __float_as_uint(v.x);
              o[i + 1] = __float_as_uint(v.y);
            }
            tmem_st32(tO + 32 * c, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&p_full[t]);
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(&o_full[t], oc & 1, ctl, kWaitOFull));
      ++oc;
      if (!ok) break;
      tc_fence_after();
      // A row that saw no key has l = 0: O = 0, L = -inf.
      const float inv_l = l_bf > 0.f ? 1.0f / l_bf : 0.f;
      const float lse = l > 0.f ? (m_ref + lg2_approx(l)) * 0.69314718055994530942f : -INFINITY;
      if (!partial) {
        // O = O~ / l in bf16, 64 columns (128 bytes of the row) at a time,
        // stored with whole row segments per warp store; rows past N are
        // skipped.
        uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) + ((size_t)w.bh * p.Nq + row) * (D * 2);
        const float2 il = make_float2(inv_l, inv_l);
#pragma unroll 1
        for (int hb = 0; hb < D / 64; ++hb) {
          uint32_t ob[32];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 64 * hb + 32 * c, o);
            tmem_ld_wait<32>(o);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 a = __fmul2_rn(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il);
              ob[16 * c + i] = pack_bf16(a.x, a.y);
            }
          }
          store_rows<4>(orow + 128 * hb, (size_t)D * 2, row, p.Nq, ob, p.store32 != 0);
        }
        if constexpr (D % 64 == 32) {
          // The last 32 columns (64 bytes of the row).
          uint32_t o[32], ob[16];
          tmem_ld32(tO + 64 * (D / 64), o);
          tmem_ld_wait<32>(o);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 a = __fmul2_rn(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il);
            ob[i] = pack_bf16(a.x, a.y);
          }
          store_rows<2>(orow + 128 * (D / 64), (size_t)D * 2, row, p.Nq, ob, p.store32 != 0);
        }
        if (row < p.Nq) p.lse[(size_t)w.bh * p.Nq + row] = lse;
      } else {
        const size_t prow = ((size_t)part * p.B * p.H + w.bh) * p.Nq + row;
        float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_ld_wait<32>(o);
          if (row < p.Nq) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[c * 8 + i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                           __uint_as_float(o[4 * i + 2]) * inv_l,
                                           __uint_as_float(o[4 * i + 3]) * inv_l);
          }
        }
        if (row < p.Nq) p.lse_part[prow] = lse;
      }
    }
    __syncwarp();
  } else {
    reg_dealloc<C::kRegsCtl>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Merge of split-KV partial results: L = log sum_s exp(L_s),
// O = sum_s exp(L_s - L) O_s.  One warp per query row (any head dim of the
// forward kernels, 256 included).
template <int D>
__global__ void __launch_bounds__(256) fa_combine_kernel(const CombineParams p) {
  const int row = blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= p.rows) return;
  constexpr int kPer = D / 32;
  float mx = -INFINITY;
  for (int s = 0; s < p.num_splits; ++s) mx = fmaxf(mx, p.lse_part[(size_t)s * p.rows + row]);
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  float tot = 0.f;
  for (int s = 0; s < p.num_splits; ++s) {
    const float ls = p.lse_part[(size_t)s * p.rows + row];
    const float wgt = (ls == -INFINITY) ? 0.f : exp2f((ls - mx) * 1.4426950408889634f);
    tot += wgt;
    const float* src = p.o_part + ((size_t)s * p.rows + row) * D + lane * kPer;
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = fmaf(wgt, src[i], acc[i]);
  }
  // A row that sees no key in any split: O = 0, L = -inf.
  const float inv = tot > 0.f ? 1.0f / tot : 0.f;
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.o) + (size_t)row * D + lane * kPer;
  if constexpr (kPer == 2) {
    *reinterpret_cast<uint32_t*>(o) = pack_bf16(acc[0] * inv, acc[1] * inv);
  } else if constexpr (kPer == 4) {
    uint2 v;
    v.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    v.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(o) = v;
  } else if constexpr (kPer == 8) {
    uint4 v;
    v.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    v.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    v.z = pack_bf16(acc[4] * inv, acc[5] * inv);
    v.w = pack_bf16(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(o) = v;
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) o[i] = __float2bfloat16_rn(acc[i] * inv);
  }
  if (lane == 0) p.lse[row] = tot > 0.f ? mx + logf(tot) : -INFINITY;
}

// ------------------------------------------------------------------ launch

template <int D, bool DUAL>
static cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdParams& p, int grid, cudaStream_t stream) {
  using C = FwdCfg<D>;
  cudaError_t e =
      cudaFuncSetAttribute(fa_fwd_kernel<D, DUAL>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  fa_fwd_kernel<D, DUAL><<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int grid, cudaStream_t stream) {
  switch (d) {
    case 64: return p.dual ? launch_fwd_t<64, true>(tq, tk, tv, p, grid, stream)
                           : launch_fwd_t<64, false>(tq, tk, tv, p, grid, stream);
    case 96: return p.dual ? launch_fwd_t<96, true>(tq, tk, tv, p, grid, stream)
                           : launch_fwd_t<96, false>(tq, tk, tv, p, grid, stream);
    case 128: return p.dual ? launch_fwd_t<128, true>(tq, tk, tv, p, grid, stream)
                            : launch_fwd_t<128, false>(tq, tk, tv, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine(int d, const CombineParams& p, cudaStream_t stream) {
  const int grid = (p.rows + 7) / 8;
  switch (d) {
    case 64: fa_combine_kernel<64><<<grid, 256, 0, stream>>>(p); break;
    case 96: fa_combine_kernel<96><<<grid, 256, 0, stream>>>(p); break;
    case 128: fa_combine_kernel<128><<<grid, 256, 0, stream>>>(p); break;
    case 256: fa_combine_kernel<256><<<grid, 256, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace fa
