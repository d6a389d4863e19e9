// Forward pass of exact attention for head dim 256 on sm_103a
// ("FlashAttention V2 in depth", section 6.1, with the causal block skip of
// section 5.3).
//
// At d = 256 an O accumulator takes 256 of the 512 TMEM columns, so a CTA
// owns one 128-row query tile (not two as in fa_fwd.cu) and overlaps its
// softmax with the tensor core across key tiles instead: S is double
// buffered, and while the softmax warps turn S_j into P_j, the tensor core
// runs O += P_{j-1} V_{j-1} and S_{j+1} = Q K_{j+1}^T.  Key/value tiles are
// 64 rows (32 KB at d = 256) so that Q (64 KB) and a 5-slot K/V ring fit in
// shared memory (224 KB); a 4-slot ring left too few tile loads in flight
// for the load latency (measured 5-9% slower).  Roles (192 threads):
//   warp 5     TMA producer: Q once per unit, then K_j, V_j alternately.
//   warp 4     MMA issuer (whole warp, one elected lane issues):
//              S_j = Q K_j^T (M128 N64, K = 256) into S buffer j & 1 and
//              O += P_j V_j (M128 N256, K = 64; P from TMEM).
//   warps 0-3  softmax, one query row per thread; they also write O and L.
// TMEM: S0 (64 columns) | S1 (64) | unused | O (256 columns from 256).
//
// The online softmax is the one of fa_fwd.cu: running max and sums in the
// row's thread, O~ unnormalised in TMEM and divided once at the end by the
// sum of the bf16-rounded weights the P V product used, L = m + log l from
// the fp32 weights, and the O~ correction only when a row max grows by more
// than a factor 2^24.  Because the product that reads P_{j-1} may still be running
// when the softmax of step j wants to correct O~, every step first waits for
// the previous step's P V product (one barrier phase per step, so the wait
// is never more than one phase behind).
#include <cuda_runtime.h>

#include "sm103_primitives.cuh"

namespace fa {

using namespace dev;

namespace d256 {

constexpr int kD = 256;
constexpr int kKeys = 64;                              // keys per K/V tile
constexpr int kQChunk = kTileM * 128;                  // 128 rows x 64 columns (bf16)
constexpr int kKVChunk = kKeys * 128;                  // 64 rows x 64 columns
constexpr int kQBytes = 4 * kQChunk;                   // 64 KB
constexpr int kKVBytes = 4 * kKVChunk;                 // 32 KB
constexpr int kStages = 5;                             // K/V ring slots (2.5 steps of lookahead)
constexpr int kThreads = 192;
constexpr uint32_t kColO = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kOffQ = 0;
constexpr int kOffKV = kQBytes;
constexpr int kOffBar = kOffKV + kStages * kKVBytes;
constexpr int kNumBars = 2 + 2 * kStages + 2 + 2 + 1 + 1 + 1 + 1;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
constexpr float kRescaleThreshold = 24.0f;             // log2 units
static_assert(kSmemBytes <= 232448, "shared memory");

struct Unit {
  int bh;
  int row0;   // first query row of the tile
  int kvb;    // first key tile (64 keys) of this split
  int n;      // key tiles processed (0 = none)
  int split;
};

// Units (batch*head, 128-row query tile, key split); query tiles in
// decreasing order (with the causal mask the last ones see the most keys).
__device__ __forceinline__ Unit decode(const FwdParams& p, int u) {
  Unit w;
  w.split = u % p.num_splits;
  const int r = u / p.num_splits;
  const int BH = p.B * p.H;
  int qt;
  if (p.head_window > 0) {  // see FwdParams::head_window
    const int per_window = p.head_window * p.num_q_blocks;
    const int win = r / per_window;
    const int heads = min(p.head_window, BH - win * p.head_window);
    const int rr = r - win * per_window;
    w.bh = win * p.head_window + rr % heads;
    qt = p.num_q_blocks - 1 - rr / heads;
  } else {
    w.bh = r % BH;
    qt = p.num_q_blocks - 1 - r / BH;
  }
  w.row0 = qt * kTileM;
  const int nkv = (p.Nk + kKeys - 1) / kKeys;
  const int lo = w.split * p.kv_tiles_per_split;
  const int hi = min(nkv, lo + p.kv_tiles_per_split);
  w.kvb = lo;
  int h = hi;
  if (p.causal) {
    const int last_key = max_query_pos(w.row0, min(p.Nq, w.row0 + kTileM) - 1, p.q_period) + p.causal_off;
    h = last_key < 0 ? 0 : min(hi, last_key / kKeys + 1);
  }
  w.n = max(0, h - lo);
  return w;
}

}  // namespace d256

__global__ void __launch_bounds__(d256::kThreads, 1)
    fa_fwd256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using namespace d256;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, (unsigned int)FA_ERR_CUDA);
    return;
  }
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sKV = smem + kOffKV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* kv_full = bars + 2;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;  // [2]
  uint64_t* p_full = s_full + 2;          // [2]
  uint64_t* pv_done = p_full + 2;         // one phase per P V product
  uint64_t* o_full = pv_done + 1;         // the unit's last P V product done
  uint64_t* o_empty = o_full + 1;         // O read out by the softmax warps
  uint64_t* drain = o_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
    }
    mbar_init(pv_done, 1);
    mbar_init(o_full, 1);
    mbar_init(o_empty, 4);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{p.status, p.timeout_ns};

  if (warp == 5) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t rc = 0, qc = 0;
      bool ok = true;
      for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
        const int u = snake_unit(rnd);
        if (u >= p.num_units) continue;
        const Unit w = decode(p, u);
        if (w.n == 0) continue;
        const int kvbh = p.Hkv == p.H ? w.bh : kv_head_of(w.bh, p.H, p.Hkv);
        ok = mbar_wait(q_empty, (qc & 1) ^ 1, ctl, kWaitQEmpty);
        if (!ok) break;
        mbar_arrive_expect_tx(q_full, kQBytes);
        for (int c = 0; c < 4; ++c) tma_load_3d(sQ + c * kQChunk, &tm_q, q_full, c * 64, w.row0, w.bh);
        ++qc;
        for (int j = 0; ok && j < w.n; ++j) {
          for (int which = 0; which < 2; ++which) {
            const uint32_t slot = rc % kStages;
            ok = mbar_wait(&kv_empty[slot], ((rc / kStages) & 1) ^ 1, ctl, kWaitKvEmpty);
            if (!ok) break;
            mbar_arrive_expect_tx(&kv_full[slot], kKVBytes);
            const CUtensorMap* m = which ? &tm_v : &tm_k;
            for (int c = 0; c < 4; ++c)
              tma_load_3d(sKV + slot * kKVBytes + c * kKVChunk, m, &kv_full[slot], c * 64, (w.kvb + j) * kKeys,
                          kvbh);
            ++rc;
          }
        }
      }
      // Every copy this thread started lands before the CTA can exit.
      const uint32_t first = rc > (uint32_t)kStages ? rc - kStages : 0u;
      for (uint32_t pos = first; pos < rc; ++pos)
        mbar_wait(&kv_full[pos % kStages], (pos / kStages) & 1, ctl, kWaitDrain);
      if (qc > 0) mbar_wait(q_full, (qc - 1) & 1, ctl, kWaitDrain);
    }
    __syncwarp();
  } else if (warp == 4) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t hi = sdesc_hi(1024);
    constexpr uint32_t id_s = idesc_bf16(kTileM, kKeys, false, false);  // S = Q K^T
    constexpr uint32_t id_o = idesc_bf16(kTileM, kD, false, true);      // O += P V
    const uint32_t q_lo = sdesc_lo(smem_u32(sQ), 16);
    const uint32_t k_lo0 = sdesc_lo(smem_u32(sKV), 16);
    const uint32_t v_lo0 = sdesc_lo(smem_u32(sKV), kKVChunk);  // V read MN-major: 64-column blocks 8 KB apart
    constexpr uint32_t kSlotStep = kKVBytes >> 4;
    auto wait = [&](uint64_t* bar, uint32_t parity, uint32_t where) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, where));
    };
    // S_g = Q K^T of the global step g (buffer g & 1) from ring position pos.
    auto issue_s = [&](uint32_t g, uint32_t pos) {
      const uint32_t k_lo = k_lo0 + (pos % kStages) * kSlotStep;
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t q_off = ((kk / 4) * kQChunk + (kk % 4) * 32) >> 4;
        const uint32_t k_off = ((kk / 4) * kKVChunk + (kk % 4) * 32) >> 4;
        mma_ss_lh_w(tmem + (g & 1) * kKeys, q_lo + q_off, hi, k_lo + k_off, hi, id_s, kk > 0 ? 1u : 0u);
      }
      mma_commit_w(&s_full[g & 1]);
      mma_commit_w(&kv_empty[pos % kStages]);
    };
    uint32_t rc = 0, qc = 0, g = 0, uc = 0;
    bool ok = true;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units) continue;
      const Unit w = decode(p, u);
      if (w.n == 0) continue;
      ok = wait(q_full, qc & 1, kWaitQFull);
      ++qc;
      // S of the unit's first two steps (K_0 at ring position rc, K_1 at rc + 2).
      for (int j = 0; ok && j < 2 && j < w.n; ++j) {
        const uint32_t pos = rc + 2 * j;
        ok = wait(&kv_full[pos % kStages], (pos / kStages) & 1, kWaitKvFull);
        if (!ok) break;
        tc_fence_after();
        issue_s(g + j, pos);
        if (j + 1 == w.n) mma_commit_w(q_empty);  // Q's last product
      }
      for (int j = 0; ok && j < w.n; ++j, ++g) {
        // O += P_j V_j once P_j is in S buffer g & 1 (and, at a unit's first
        // step, the previous unit's O has been read out).
        ok = wait(&p_full[g & 1], (g >> 1) & 1, kWaitPFull);
        if (ok && j == 0 && uc > 0) ok = wait(o_empty, (uc - 1) & 1, kWaitOFull);
        const uint32_t pos_v = rc + 2 * j + 1;
        if (ok) ok = wait(&kv_full[pos_v % kStages], (pos_v / kStages) & 1, kWaitKvFull);
        if (!ok) break;
        tc_fence_after();
        const uint32_t v_lo = v_lo0 + (pos_v % kStages) * kSlotStep;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          mma_ts_lh_w(tmem + kColO, tmem + (g & 1) * kKeys + kk * 8, v_lo + ((kk * 2048) >> 4), hi, id_o,
                      (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit_w(&kv_empty[pos_v % kStages]);
        mma_commit_w(pv_done);
        // S two steps ahead, into the buffer this P V product reads (the
        // tensor core runs one warp's products in issue order).
        if (j + 2 < w.n) {
          const uint32_t pos_k = rc + 2 * (j + 2);
          ok = wait(&kv_full[pos_k % kStages], (pos_k / kStages) & 1, kWaitKvFull);
          if (!ok) break;
          tc_fence_after();
          issue_s(g + 2, pos_k);
          if (j + 3 == w.n) mma_commit_w(q_empty);
        }
      }
      if (!ok) break;
      mma_commit_w(o_full);
      rc += 2 * w.n;
      ++uc;
    }
    mma_commit_w(drain);
    (void)wait(drain, 0, kWaitDrain);
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const uint32_t tO = tmem + lane_off + kColO;
    const float sl2 = p.scale_log2;
    uint32_t g = 0, uc = 0;
    bool ok = true;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units) continue;
      const Unit w = decode(p, u);
      const int row = w.row0 + 32 * warp + lane;
      if (w.n == 0) {
        // No row of the tile sees a key (of this split): O = 0, L = -inf.
        if (row < p.Nq) {
          if (p.num_splits > 1) {
            const size_t prow = ((size_t)w.split * p.B * p.H + w.bh) * p.Nq + row;
            float4* dst = reinterpret_cast<float4*>(p.o_part + prow * kD);
            for (int c = 0; c < kD / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            p.lse_part[prow] = -INFINITY;
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.o) + ((size_t)w.bh * p.Nq + row) * (kD * 2));
            for (int c = 0; c < kD / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
            p.lse[(size_t)w.bh * p.Nq + row] = -INFINITY;
          }
        }
        continue;
      }
      float m_ref = -INFINITY;  // reference max (log2 units); -inf while no key was seen
      float l = 0.f;            // sum of the fp32 weights: L = m + log l
      float l_bf = 0.f;         // sum of the bf16-rounded weights: O = O~ / l_bf
      for (int j = 0; j < w.n; ++j, ++g) {
        const uint32_t tS = tmem + lane_off + (g & 1) * kKeys;
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[g & 1], (g >> 1) & 1, ctl, kWaitSFull));
        if (!ok) break;
        tc_fence_after();
        uint32_t s[kKeys];
        tmem_ld32(tS, s);
        tmem_ld32(tS + 32, s + 32);
        tmem_ld_wait<kKeys>(s);
        float x[kKeys];
#pragma unroll
        for (int c = 0; c < kKeys; ++c) x[c] = __uint_as_float(s[c]);
        const int kv0 = (w.kvb + j) * kKeys;
        if ((kv0 + kKeys > p.Nk) || (p.causal && (p.q_period > 0 || kv0 + kKeys - 1 > w.row0 + p.causal_off))) {
          const int lim = p.causal ? min(p.Nk - 1, query_pos(row, p.q_period) + p.causal_off) : p.Nk - 1;  // last visible key
#pragma unroll
          for (int c = 0; c < kKeys; ++c)
            if (kv0 + c > lim) x[c] = -INFINITY;
        }
        float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
        for (int c = 4; c + 8 <= kKeys; c += 8) {
          mx0 = fmax3(mx0, x[c], x[c + 1]);
          mx1 = fmax3(mx1, x[c + 2], x[c + 3]);
          mx2 = fmax3(mx2, x[c + 4], x[c + 5]);
          mx3 = fmax3(mx3, x[c + 6], x[c + 7]);
        }
        mx0 = fmax3(mx0, x[kKeys - 4], x[kKeys - 3]);  // the last four columns
        mx1 = fmax3(mx1, x[kKeys - 2], x[kKeys - 1]);
        const float m_tile = fmax3(fmaxf(mx0, mx1), mx2, mx3) * sl2;
        float f = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_ref = m_tile;
        } else if (__any_sync(0xffffffffu, m_tile > m_ref + kRescaleThreshold)) {
          const float m_new = fmaxf(m_ref, m_tile);
          f = (m_new == -INFINITY) ? 1.f : ex2_approx(m_ref - m_new);
          l *= f;
          l_bf *= f;
          m_ref = m_new;
          rescale = true;
        }
        const float m_exp = (m_ref == -INFINITY) ? 0.f : m_ref;
        const float2 sl2v = make_float2(sl2, sl2);
        const float2 negv = make_float2(-m_exp, -m_exp);
        float2 ls0 = make_float2(0.f, 0.f), ls1 = ls0;
        float lr0 = 0.f, lr1 = 0.f, lr2 = 0.f, lr3 = 0.f;
        uint32_t pk[kKeys / 2];
#pragma unroll
        for (int e = 0; e < kKeys; e += 2) {
          const float2 a = __ffma2_rn(make_float2(x[e], x[e + 1]), sl2v, negv);
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
        tmem_st32(tS, pk);
        l += (ls0.x + ls0.y) + (ls1.x + ls1.y);
        l_bf += (lr0 + lr1) + (lr2 + lr3);
        // The previous step's P V product (possibly of the previous unit)
        // has completed: O~ may be corrected now.
        if (g > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (g - 1) & 1, ctl, kWaitPFull));
          if (!ok) break;
        }
        if (rescale) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kD / 32; ++c) {
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
        mbar_arrive_warp(&p_full[g & 1]);
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(o_full, uc & 1, ctl, kWaitOFull));
      ++uc;
      if (!ok) break;
      tc_fence_after();
      // A row that saw no key has l = 0: O = 0, L = -inf.
      const float inv_l = l_bf > 0.f ? 1.0f / l_bf : 0.f;
      const float lse = l > 0.f ? (m_ref + lg2_approx(l)) * 0.69314718055994530942f : -INFINITY;
      if (p.num_splits == 1) {
        uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) + ((size_t)w.bh * p.Nq + row) * (kD * 2);
        const float2 il = make_float2(inv_l, inv_l);
#pragma unroll 1
        for (int hb = 0; hb < kD / 64; ++hb) {
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
          if (hb + 1 == kD / 64) {
            // Every column of O~ has been read: the next unit may overwrite it.
            tc_fence_before();
            mbar_arrive_warp(o_empty);
          }
          store_rows<4>(orow + 128 * hb, (size_t)kD * 2, row, p.Nq, ob, p.store32 != 0);
        }
        if (row < p.Nq) p.lse[(size_t)w.bh * p.Nq + row] = lse;
      } else {
        const size_t prow = ((size_t)w.split * p.B * p.H + w.bh) * p.Nq + row;
        float4* dst = reinterpret_cast<float4*>(p.o_part + prow * kD);
#pragma unroll 1
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_ld_wait<32>(o);
          if (c + 1 == kD / 32) {
            tc_fence_before();
            mbar_arrive_warp(o_empty);
          }
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t launch_fwd256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                          int grid, cudaStream_t stream) {
  cudaError_t e =
      cudaFuncSetAttribute(fa_fwd256_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, d256::kSmemBytes);
  if (e != cudaSuccess) return e;
  fa_fwd256_kernel<<<grid, d256::kThreads, d256::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace fa
