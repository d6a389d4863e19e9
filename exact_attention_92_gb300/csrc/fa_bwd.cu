// Backward pass of exact attention on sm_103a ("FlashAttention V2 in depth",
// section 7).
//
//   fa_bwd_preprocess  D_i = rowsum(dO_i * O_i) (section 7.3, a separate
//                      kernel run once) and zeroing of the fp32 dQ
//                      accumulator.
//   fa_bwd_kernel      key/value tiles in the outer loop (section 7.2): a
//                      persistent CTA owns one 128-key tile K_j, V_j of one
//                      (batch, head) and walks the query tiles i that can see
//                      it.  dK_j and dV_j accumulate in tensor memory of that
//                      CTA alone (no atomics); the partial dQ of every step is
//                      added to the fp32 accumulator with atomics.
//   fa_dq_convert      dQ = scale * accumulator, to bf16.
//
// Per step (query tile i of 128 rows), in the transposed orientation so that
// TMEM lanes are keys:
//   S^T  = K_j Q_i^T,   P^T = exp(scale S^T - L_i)   (P recovered from the
//                       saved logsumexp, section 7.1)
//   dP^T = V_j dO_i^T,  dS^T = P^T * (dP^T - D_i)
//   dV_j += P^T dO_i,   dK_j += dS^T Q_i
//   d = 128: dQ_i^T = K_j^T dS^T; the softmax warps write it row-major into
//            the step's Q/dO stage buffer (free once dQ is complete) and the
//            producer adds each 64-row half (32 contiguous KB of the
//            accumulator) with one bulk reduce-add, then refills the stage
//   d = 64:  dQ_i = dS K_j, added with per-thread vector atomics
// The softmax scale is applied once to dK at the end and to dQ in the
// convert kernel.
//
// Roles (320 threads): warp 9 loads (TMA for K, V, Q, dO; plain loads for
// L_i and D_i into shared memory), warp 8 issues tcgen05 MMAs, warps 0-7
// compute P^T and dS^T (a key row per lane, warps w and w+4 split the 128
// query columns), then read their half of dQ out of TMEM, release it and
// stage it for the reduction while the next step's S^T / dP^T run, and
// write dK/dV at the end of a unit.
//
// TMEM (512 columns).  A = [0,128): S^T; P^T (bf16, two per column) goes to
// A[0,32) for queries 0-63 and A[96,128) for queries 64-127, each written
// over S^T columns its own warp has already read.  B = [128,256): dP^T, then
// dS^T in B[0,32) and B[96,128).  dV and dK follow.  At d = 128 the dQ^T
// halves take the free middle columns A[32,96) and B[32,96), so the next
// step's S^T / dP^T wait for them to be read out; at d = 64 dQ has its own
// 64 columns.
#include <cuda_runtime.h>

#include "sm103_primitives.cuh"

namespace fa {

using namespace dev;

template <int D>
struct BwdCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = kTileM * 128;
  static constexpr int kTileBytes = kTileM * D * 2;
  static constexpr int kStages = 2;
  static constexpr int kThreads = 320;
  static constexpr uint32_t kColA = 0;
  static constexpr uint32_t kColB = 128;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
  static constexpr bool kDqT = (D == 128);
  static constexpr uint32_t kColDQ = kDqT ? 32u : 384u;  // d = 128: A+32 and B+32
  static constexpr uint32_t kTmemCols = 512;
  // Shared memory.
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;
  static constexpr int kOffDO = kOffQ + kStages * kTileBytes;
  static constexpr int kOffDS = kOffDO + kStages * kTileBytes;
  static constexpr int kDsBytes = kTileM * kTileN * 2;
  static constexpr int kOffLse = kOffDS + kDsBytes;             // kStages x 128 floats (log2 units)
  static constexpr int kOffDvec = kOffLse + kStages * 128 * 4;  // kStages x 128 floats
  static constexpr int kOffBar = kOffDvec + kStages * 128 * 4;
  static constexpr int kNumBars = 2 + 3 * kStages + 1 + 1 + 1 + 2 + 2 + 1 + 2 * kStages;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
};

// Packed-P^T / dS^T column of the 16 queries [16 kk, 16 kk + 16) in A or B.
__device__ __forceinline__ uint32_t packed_col(int kk) { return kk < 4 ? 8u * kk : 96u + 8u * (kk - 4); }

struct BwdUnit {
  int bh;
  int j;       // key tile
  int i0, nq;  // first query tile and number of query tiles
};

__device__ __forceinline__ BwdUnit decode_bwd(const BwdParams& p, int u) {
  BwdUnit w;
  const int BH = p.B * p.H;
  w.bh = u % BH;
  w.j = u / BH;  // with the causal mask, low key tiles have the most work
  const int nq = p.num_kv_tiles;
  w.i0 = p.causal ? w.j : 0;
  w.nq = nq - w.i0;
  return w;
}

// P^T and dS^T of 32 query columns of one key row: p = exp2(s * sl2 - L),
// ds = p * (dP - D), packed to bf16 pairs.  MASK zeroes the weights the
// causal mask hides (kr > query) and those of a key row past N; it is a
// template argument so the unmasked instance has no branch at all and the
// compiler can interleave its independent chains.
template <bool MASK>
__device__ __forceinline__ void bwd_chunk(const uint32_t* s, const uint32_t* dpv, const float* bl, const float* bd,
                                          float sl2, int kr, int q_first, bool dead, bool causal, uint32_t* pp,
                                          uint32_t* dd) {
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const float4 l4 = reinterpret_cast<const float4*>(bl)[e4];
    const float4 d4 = reinterpret_cast<const float4*>(bd)[e4];
    const float2 a01 = __ffma2_rn(make_float2(__uint_as_float(s[4 * e4]), __uint_as_float(s[4 * e4 + 1])),
                                  make_float2(sl2, sl2), make_float2(-l4.x, -l4.y));
    const float2 a23 = __ffma2_rn(make_float2(__uint_as_float(s[4 * e4 + 2]), __uint_as_float(s[4 * e4 + 3])),
                                  make_float2(sl2, sl2), make_float2(-l4.z, -l4.w));
    float2 p01 = make_float2(ex2_approx(a01.x), ex2_approx(a01.y));
    float2 p23 = make_float2(ex2_approx(a23.x), ex2_approx(a23.y));
    if (MASK) {
      const int col = q_first + 4 * e4;
      p01.x = (dead || (causal && kr > col)) ? 0.f : p01.x;
      p01.y = (dead || (causal && kr > col + 1)) ? 0.f : p01.y;
      p23.x = (dead || (causal && kr > col + 2)) ? 0.f : p23.x;
      p23.y = (dead || (causal && kr > col + 3)) ? 0.f : p23.y;
    }
    const float2 g01 = __fadd2_rn(make_float2(__uint_as_float(dpv[4 * e4]), __uint_as_float(dpv[4 * e4 + 1])),
                                  make_float2(-d4.x, -d4.y));
    const float2 g23 = __fadd2_rn(make_float2(__uint_as_float(dpv[4 * e4 + 2]), __uint_as_float(dpv[4 * e4 + 3])),
                                  make_float2(-d4.z, -d4.w));
    const float2 ds01 = __fmul2_rn(p01, g01);
    const float2 ds23 = __fmul2_rn(p23, g23);
    pp[2 * e4] = pack_bf16(p01.x, p01.y);
    pp[2 * e4 + 1] = pack_bf16(p23.x, p23.y);
    dd[2 * e4] = pack_bf16(ds01.x, ds01.y);
    dd[2 * e4 + 1] = pack_bf16(ds23.x, ds23.y);
  }
}

template <int D>
__global__ void __launch_bounds__(320, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, (unsigned int)FA_ERR_CUDA);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + 1;
  uint64_t* qdo_full = bars + 2;
  uint64_t* qdo_empty = qdo_full + C::kStages;
  uint64_t* stat_full = qdo_empty + C::kStages;  // L_i, D_i of a stage written
  uint64_t* s_full = stat_full + C::kStages;
  uint64_t* p_ready = s_full + 1;
  uint64_t* dq_full = p_ready + 1;
  uint64_t* dq_empty = dq_full + 1;  // [2]: the two dQ^T halves read out (d = 64: [0] only)
  uint64_t* dkv_full = dq_empty + 2;
  uint64_t* dkv_empty = dkv_full + 1;
  uint64_t* drain = dkv_empty + 1;
  // [stage][half]: a dQ^T half written into that stage's buffer (d = 128).
  // One pair per stage: a stage is refilled only after its last use was
  // reduced, so these never run more than one phase ahead of the producer.
  uint64_t* dq_staged = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dq_staged + 2 * C::kStages);
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);
  float* sDv = reinterpret_cast<float*>(smem + C::kOffDvec);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&qdo_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
      mbar_init(&stat_full[s], 32);
    }
    mbar_init(s_full, 1);
    mbar_init(p_ready, 256);
    mbar_init(dq_full, 1);
    // d = 128: one barrier per dQ^T half (the 4 warps reading it); d = 64:
    // all 8 warps release the one dQ tile.
    mbar_init(&dq_empty[0], C::kDqT ? 128 : 256);
    mbar_init(&dq_empty[1], 128);
    mbar_init(dkv_full, 1);
    mbar_init(dkv_empty, 256);
    mbar_init(drain, 1);
    for (int i = 0; i < 2 * C::kStages; ++i) mbar_init(&dq_staged[i], 128);
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
    uint32_t kc = 0, qc = 0;
    // Rows (bh * N + q0) and valid row count of the steps in each stage, for
    // the dQ reduction of d = 128.
    size_t st_row[C::kStages];
    int st_nrow[C::kStages];
    bool ok = true;
    // d = 128: add step `k`'s staged dQ (two 64-row halves in the Q and dO
    // buffers of stage k % kStages) to the accumulator, and wait until the
    // copies have read the buffers.
    auto reduce_step = [&](uint32_t k) -> bool {
      const uint32_t s = k % C::kStages;
      const uint32_t par = (k / C::kStages) & 1;
      bool r = __all_sync(0xffffffffu, mbar_wait(&dq_staged[2 * s], par, ctl, kWaitBwdLoad)) &&
               __all_sync(0xffffffffu, mbar_wait(&dq_staged[2 * s + 1], par, ctl, kWaitBwdLoad));
      if (r && lane == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = min(64, st_nrow[s] - 64 * h);
          if (n > 0)
            bulk_reduce_add_f32(p.dq_acc + (st_row[s] + 64 * h) * D,
                                smem + (h ? C::kOffDO : C::kOffQ) + s * C::kTileBytes, (uint32_t)n * D * 4);
        }
        bulk_commit();
        bulk_wait_read_all();
      }
      __syncwarp();
      return r;
    };
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units) continue;
      const BwdUnit w = decode_bwd(p, u);
      const size_t head = (size_t)w.bh * p.N;
      ok = __all_sync(0xffffffffu, mbar_wait(kv_empty, (kc & 1) ^ 1, ctl, kWaitBwdLoad));
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(smem + C::kOffK + c * C::kChunkBytes, &tm_k, kv_full, c * 64, w.j * kTileN, w.bh);
          tma_load_3d(smem + C::kOffV + c * C::kChunkBytes, &tm_v, kv_full, c * 64, w.j * kTileN, w.bh);
        }
      }
      ++kc;
      for (int ii = 0; ok && ii < w.nq; ++ii) {
        const uint32_t st = qc % C::kStages;
        if constexpr (C::kDqT) {
          // The stage's previous step has finished with Q/dO and its dQ is
          // staged there: reduce it, then refill.
          if (qc >= (uint32_t)C::kStages) ok = reduce_step(qc - C::kStages);
        } else {
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&qdo_empty[st], ((qc / C::kStages) & 1) ^ 1, ctl, kWaitBwdLoad));
        }
        if (!ok) break;
        const int row = (w.i0 + ii) * kTileM;
        st_row[st] = head + row;
        st_nrow[st] = p.N - row;
        if (lane == 0) {
          mbar_arrive_expect_tx(&qdo_full[st], 2 * C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c) {
            tma_load_3d(smem + C::kOffQ + st * C::kTileBytes + c * C::kChunkBytes, &tm_q, &qdo_full[st], c * 64,
                        row, w.bh);
            tma_load_3d(smem + C::kOffDO + st * C::kTileBytes + c * C::kChunkBytes, &tm_do, &qdo_full[st],
                        c * 64, row, w.bh);
          }
        }
        // L_i (log2 units) and D_i of the tile's 128 queries; rows past N get
        // L = +inf so their weights vanish.
        float4 l4, d4;
        float* lp = &l4.x;
        float* dp = &d4.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int qr = row + 4 * lane + e;
          lp[e] = qr < p.N ? p.lse[head + qr] * 1.4426950408889634f : INFINITY;
          dp[e] = qr < p.N ? p.dvec[head + qr] : 0.f;
        }
        reinterpret_cast<float4*>(sLse + st * 128)[lane] = l4;
        reinterpret_cast<float4*>(sDv + st * 128)[lane] = d4;
        mbar_arrive(&stat_full[st]);
        ++qc;
      }
    }
    if constexpr (C::kDqT) {
      // The last steps' dQ.
      const uint32_t first = qc > (uint32_t)C::kStages ? qc - C::kStages : 0u;
      for (uint32_t k = first; ok && k < qc; ++k) ok = reduce_step(k);
    }
    if (lane == 0) {
      bulk_wait_all();  // every reduction has landed
      if (kc > 0) mbar_wait(kv_full, (kc - 1) & 1, ctl, kWaitDrain);
      const uint32_t first = qc > (uint32_t)C::kStages ? qc - C::kStages : 0u;
      for (uint32_t pos = first; pos < qc; ++pos)
        mbar_wait(&qdo_full[pos % C::kStages], (pos / C::kStages) & 1, ctl, kWaitDrain);
    }
    __syncwarp();
  } else if (warp == 8) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(kTileM, kTileM, false, false);  // S^T, dP^T
      constexpr uint32_t id_kv = idesc_bf16(kTileM, D, false, true);       // dV, dK
      constexpr uint32_t id_dq = idesc_bf16(kTileM, 64, true, true);       // dQ^T halves / dQ
      const uint32_t sk = smem_u32(smem + C::kOffK);
      const uint32_t sv = smem_u32(smem + C::kOffV);
      const uint32_t sds = smem_u32(smem + C::kOffDS);
      uint32_t kc = 0, qc = 0, pc = 0, dqc = 0, uc = 0;
      bool ok = true;
      for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
        const int u = snake_unit(rnd);
        if (u >= p.num_units) continue;
        const BwdUnit w = decode_bwd(p, u);
        ok = mbar_wait(kv_full, kc & 1, ctl, kWaitBwdMma);
        ++kc;
        if (!ok) break;
        tc_fence_after();
        for (int ii = 0; ii < w.nq; ++ii) {
          const uint32_t st = qc % C::kStages;
          ok = mbar_wait(&qdo_full[st], (qc / C::kStages) & 1, ctl, kWaitBwdMma);
          if (!ok) break;
          const uint32_t sq = smem_u32(smem + C::kOffQ + st * C::kTileBytes);
          const uint32_t sdo = smem_u32(smem + C::kOffDO + st * C::kTileBytes);
          if (C::kDqT && dqc > 0) {
            // S^T overwrites the columns of the previous dQ^T's first half.
            ok = mbar_wait(&dq_empty[0], (dqc - 1) & 1, ctl, kWaitBwdMma);
            if (!ok) break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * C::kChunkBytes + (kk % 4) * 32;
            mma_ss(tmem + C::kColA, sdesc_sw128(sk + off, 16, 1024), sdesc_sw128(sq + off, 16, 1024), id_s,
                   kk > 0 ? 1u : 0u);
          }
          if (C::kDqT && dqc > 0) {
            ok = mbar_wait(&dq_empty[1], (dqc - 1) & 1, ctl, kWaitBwdMma);
            if (!ok) break;
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * C::kChunkBytes + (kk % 4) * 32;
            mma_ss(tmem + C::kColB, sdesc_sw128(sv + off, 16, 1024), sdesc_sw128(sdo + off, 16, 1024), id_s,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(s_full);
          ok = mbar_wait(p_ready, pc & 1, ctl, kWaitBwdMma);
          ++pc;
          if (!ok) break;
          if (ii == 0 && uc > 0) {
            // dV / dK of the previous unit have been read out.
            ok = mbar_wait(dkv_empty, (uc - 1) & 1, ctl, kWaitBwdMma);
            if (!ok) break;
          }
          if (!C::kDqT && dqc > 0) {
            ok = mbar_wait(&dq_empty[0], (dqc - 1) & 1, ctl, kWaitBwdMma);
            if (!ok) break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk) {
            const uint32_t acc = (ii > 0 || kk > 0) ? 1u : 0u;
            mma_ts(tmem + C::kColDV, tmem + C::kColA + packed_col(kk),
                   sdesc_sw128(sdo + kk * 2048, C::kChunkBytes, 1024), id_kv, acc);
          }
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk) {
            const uint32_t acc = (ii > 0 || kk > 0) ? 1u : 0u;
            mma_ts(tmem + C::kColDK, tmem + C::kColB + packed_col(kk),
                   sdesc_sw128(sq + kk * 2048, C::kChunkBytes, 1024), id_kv, acc);
          }
          if constexpr (C::kDqT) {
            // dQ^T[:, 64h : 64h+64] = K^T dS^T[:, 64h : 64h+64]: A = K^T (K
            // tile read MN-major), B = the 64-query block h of dS^T.
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int kk = 0; kk < kTileN / 16; ++kk)
                mma_ss(tmem + (h ? C::kColB : C::kColA) + C::kColDQ,
                       sdesc_sw128(sk + kk * 2048, C::kChunkBytes, 1024),
                       sdesc_sw128(sds + h * C::kChunkBytes + kk * 2048, C::kChunkBytes, 1024), id_dq,
                       kk > 0 ? 1u : 0u);
          } else {
            // dQ = dS K: A = dS (the dS^T tile read MN-major), B = K.
#pragma unroll
            for (int kk = 0; kk < kTileN / 16; ++kk)
              mma_ss(tmem + C::kColDQ, sdesc_sw128(sds + kk * 2048, C::kChunkBytes, 1024),
                     sdesc_sw128(sk + kk * 2048, C::kChunkBytes, 1024), id_dq, kk > 0 ? 1u : 0u);
          }
          mma_commit(dq_full);
          ++dqc;
          if (!C::kDqT) mma_commit(&qdo_empty[st]);
          ++qc;
        }
        if (!ok) break;
        mma_commit(dkv_full);
        mma_commit(kv_empty);
        ++uc;
      }
      mma_commit(drain);
      mbar_wait(drain, 0, ctl, kWaitDrain);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------ P^T, dS^T, dQ read-out and dK/dV output
    const int g = warp & 3;    // TMEM lane quarter
    const int hc = warp >> 2;  // query-column half
    const uint32_t lane_off = (uint32_t)(32 * g) << 16;
    const int r = 32 * g + lane;  // key row within the tile
    const float sl2 = p.scale_log2;
    uint8_t* sds = smem + C::kOffDS;
    uint32_t sc = 0, uc = 0, qc = 0, dc = 0;
    bool ok = true;
    for (int rnd = 0; ok && rnd * (int)gridDim.x < p.num_units; ++rnd) {
      const int u = snake_unit(rnd);
      if (u >= p.num_units) continue;
      const BwdUnit w = decode_bwd(p, u);
      const int kr = w.j * kTileN + r;  // key index
      const size_t head = (size_t)w.bh * p.N;
      for (int ii = 0; ii < w.nq; ++ii, ++qc) {
        const int q0 = (w.i0 + ii) * kTileM;
        const uint32_t st = qc % C::kStages;
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&stat_full[st], (qc / C::kStages) & 1, ctl, kWaitBwdSoftmax));
        if (!ok) break;
        ok = __all_sync(0xffffffffu, mbar_wait(s_full, sc & 1, ctl, kWaitBwdSoftmax));
        ++sc;
        if (!ok) break;
        tc_fence_after();
        const float* bl = sLse + st * 128;
        const float* bd = sDv + st * 128;
        const bool mask = (kr >= p.N) || (p.causal && kr > q0);
        // Half 0 handles query chunks 0, 1; half 1 handles 3, 2 (in that
        // order), so each packed store lands on S^T / dP^T columns this warp
        // has already read.  Two loads (64 registers) per chunk: a load's
        // registers must not be live across spills before its wait.
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          const int c = hc ? 3 - cc : cc;
          uint32_t s[1][32], dpv[1][32];
          tmem_ld32(tmem + lane_off + C::kColA + 32 * c, s[0]);
          tmem_ld32(tmem + lane_off + C::kColB + 32 * c, dpv[0]);
          tmem_ld_wait<32>(s[0]);
          tmem_ld_wait<32>(dpv[0]);
          uint32_t pp[16], dd[16];
          if (mask)
            bwd_chunk<true>(s[0], dpv[0], bl + 32 * c, bd + 32 * c, sl2, kr, q0 + 32 * c, kr >= p.N, p.causal != 0,
                            pp, dd);
          else
            bwd_chunk<false>(s[0], dpv[0], bl + 32 * c, bd + 32 * c, sl2, kr, q0 + 32 * c, false, false, pp, dd);
          const uint32_t dst = c < 2 ? 16u * c : 96u + 16u * (c - 2);
          tmem_st16(tmem + lane_off + C::kColA + dst, pp);
          tmem_st16(tmem + lane_off + C::kColB + dst, dd);
          // dS^T row r, query columns [32c, 32c+32): 64 bytes of the
          // 128-byte-swizzled [key row][query] tile the dQ MMA reads.
          uint8_t* rowp = sds + (c / 2) * C::kChunkBytes + r * 128;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int unit = (c % 2) * 4 + q4;
            *reinterpret_cast<uint4*>(rowp + ((unit ^ (r & 7)) << 4)) =
                make_uint4(dd[4 * q4], dd[4 * q4 + 1], dd[4 * q4 + 2], dd[4 * q4 + 3]);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive(p_ready);
        // dQ of this step: read this warp's share out of TMEM, release it,
        // then add it to the fp32 accumulator.
        ok = __all_sync(0xffffffffu, mbar_wait(dq_full, dc & 1, ctl, kWaitBwdDq));
        ++dc;
        if (!ok) break;
        tc_fence_after();
        if constexpr (C::kDqT) {
          // Lane = head-dim column dd, 64 query rows of half hc.
          const int dd = 32 * g + lane;
          uint32_t v[64];
          const uint32_t base = tmem + lane_off + (hc ? C::kColB : C::kColA) + C::kColDQ;
          tmem_ld32(base, v);
          tmem_ld32(base + 32, v + 32);
          tmem_ld_wait<64>(v);
          tc_fence_before();
          mbar_arrive(&dq_empty[hc]);
          // Row-major [query][head dim] into the stage's Q (half 0) or dO
          // (half 1) buffer: 32 lanes write one 128-byte run per query.
          float* buf = reinterpret_cast<float*>(smem + (hc ? C::kOffDO : C::kOffQ) + st * C::kTileBytes);
#pragma unroll
          for (int qq = 0; qq < 64; ++qq) buf[qq * D + dd] = __uint_as_float(v[qq]);
          fence_proxy_async_smem();
          mbar_arrive(&dq_staged[2 * st + hc]);
        } else {
          // Lane = query row; head-dim columns [32 hc, 32 hc + 32).
          const int qr = q0 + r;
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + C::kColDQ + 32 * hc, v);
          tmem_ld_wait<32>(v);
          tc_fence_before();
          mbar_arrive(&dq_empty[0]);
          if (qr < p.N) {
            float4* dst = reinterpret_cast<float4*>(p.dq_acc + (head + qr) * D + 32 * hc);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              atomicAdd(dst + c, make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                             __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3])));
          }
        }
      }
      if (!ok) break;
      // dK_j = scale * sum dS^T Q and dV_j = sum P^T dO of this unit; this
      // warp writes head-dim columns [D/2 hc, D/2 hc + D/2).
      ok = __all_sync(0xffffffffu, mbar_wait(dkv_full, uc & 1, ctl, kWaitBwdSoftmax));
      ++uc;
      if (!ok) break;
      tc_fence_after();
      __nv_bfloat16* dvp = reinterpret_cast<__nv_bfloat16*>(p.dv) + (head + kr) * D;
      __nv_bfloat16* dkp = reinterpret_cast<__nv_bfloat16*>(p.dk) + (head + kr) * D;
#pragma unroll 1
      for (int c = hc * (D / 64); c < (hc + 1) * (D / 64); ++c) {
        uint32_t a[32], b[32];
        tmem_ld32(tmem + lane_off + C::kColDV + 32 * c, a);
        tmem_ld32(tmem + lane_off + C::kColDK + 32 * c, b);
        tmem_ld_wait<32>(a);
        tmem_ld_wait<32>(b);
        if (kr < p.N) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 va, vb;
            va.x = pack_bf16(__uint_as_float(a[8 * i + 0]), __uint_as_float(a[8 * i + 1]));
            va.y = pack_bf16(__uint_as_float(a[8 * i + 2]), __uint_as_float(a[8 * i + 3]));
            va.z = pack_bf16(__uint_as_float(a[8 * i + 4]), __uint_as_float(a[8 * i + 5]));
            va.w = pack_bf16(__uint_as_float(a[8 * i + 6]), __uint_as_float(a[8 * i + 7]));
            vb.x = pack_bf16(__uint_as_float(b[8 * i + 0]) * p.scale, __uint_as_float(b[8 * i + 1]) * p.scale);
            vb.y = pack_bf16(__uint_as_float(b[8 * i + 2]) * p.scale, __uint_as_float(b[8 * i + 3]) * p.scale);
            vb.z = pack_bf16(__uint_as_float(b[8 * i + 4]) * p.scale, __uint_as_float(b[8 * i + 5]) * p.scale);
            vb.w = pack_bf16(__uint_as_float(b[8 * i + 6]) * p.scale, __uint_as_float(b[8 * i + 7]) * p.scale);
            reinterpret_cast<uint4*>(dvp)[c * 4 + i] = va;
            reinterpret_cast<uint4*>(dkp)[c * 4 + i] = vb;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(dkv_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// D_i = sum_c dO_ic * O_ic; also zeroes row i of the dQ accumulator.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_preprocess(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dout,
                                                         float* __restrict__ dvec, float* __restrict__ dq_acc,
                                                         int rows) {
  const int row = blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  constexpr int kPer = D / 32;
  const __nv_bfloat16* a = o + (size_t)row * D + lane * kPer;
  const __nv_bfloat16* b = dout + (size_t)row * D + lane * kPer;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc = fmaf(__bfloat162float(a[i]), __bfloat162float(b[i]), acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) dvec[row] = acc;
  float* z = dq_acc + (size_t)row * D + lane * kPer;
#pragma unroll
  for (int i = 0; i < kPer; ++i) z[i] = 0.f;
}

__global__ void __launch_bounds__(256) fa_dq_convert(const float4* __restrict__ acc, uint2* __restrict__ out,
                                                     size_t n4, float scale) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = acc[i];
    uint2 r;
    r.x = pack_bf16(v.x * scale, v.y * scale);
    r.y = pack_bf16(v.z * scale, v.w * scale);
    out[i] = r;
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

template <int D>
static cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream) {
  using C = BwdCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(fa_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  fa_bwd_kernel<D><<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream) {
  return d == 64 ? launch_bwd_t<64>(tq, tk, tv, tdo, p, grid, stream)
                 : launch_bwd_t<128>(tq, tk, tv, tdo, p, grid, stream);
}

cudaError_t launch_bwd_preprocess(int d, const void* o, const void* dout, float* dvec, float* dq_acc, int rows,
                                  cudaStream_t stream) {
  const int grid = (rows + 7) / 8;
  const auto* po = static_cast<const __nv_bfloat16*>(o);
  const auto* pd = static_cast<const __nv_bfloat16*>(dout);
  if (d == 64)
    fa_bwd_preprocess<64><<<grid, 256, 0, stream>>>(po, pd, dvec, dq_acc, rows);
  else
    fa_bwd_preprocess<128><<<grid, 256, 0, stream>>>(po, pd, dvec, dq_acc, rows);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(int d, const float* dq_acc, void* dq, size_t elems, float scale, cudaStream_t stream) {
  (void)d;
  const size_t n4 = elems / 4;
  size_t blocks = (n4 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks == 0) blocks = 1;
  fa_dq_convert<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(dq_acc),
                                                        static_cast<uint2*>(dq), n4, scale);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(unsigned int* status, unsigned long long timeout_ns, cudaStream_t stream) {
  fa_selftest_wait_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fa
