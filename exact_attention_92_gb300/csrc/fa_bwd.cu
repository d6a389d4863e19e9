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
//                      CTA alone (no atomics); the partial dQ_i of every step
//                      is added to the fp32 accumulator with atomics.
//   fa_dq_convert      dQ = scale * accumulator, to bf16.
//
// Per step (query tile i), in the transposed orientation so that TMEM lanes
// are keys:
//   S^T  = K_j Q_i^T,   P^T = exp(scale S^T - L_i)   (P recovered from the
//                       saved logsumexp, section 7.1)
//   dP^T = V_j dO_i^T,  dS^T = P^T * (dP^T - D_i)
//   dV_j += P^T dO_i,   dK_j += dS^T Q_i,   dQ_i += dS K_j
// with the softmax scale applied once to dK at the end and to dQ in the
// convert kernel.
//
// Roles: warp 9 loads (TMA), warp 8 issues tcgen05 MMAs, warps 0-3 compute
// P^T and dS^T (one key row per thread) and write dK/dV at the end of a unit,
// warps 4-7 read dQ_i out of TMEM and add it to the accumulator.
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
  // TMEM columns.  A: S^T then P^T (bf16 in its first 64 columns).
  // B: dP^T then dS^T.  At d = 128 the dQ tile takes the upper halves of A
  // and B (free once P^T and dS^T are written); at d = 64 it has its own.
  static constexpr uint32_t kColA = 0;
  static constexpr uint32_t kColB = 128;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
  static constexpr bool kDqAliased = (D == 128);
  static constexpr uint32_t kColDQ0 = kDqAliased ? 64u : 384u;
  static constexpr uint32_t kColDQ1 = kDqAliased ? 192u : 384u;
  static constexpr uint32_t kTmemCols = 512;
  // Shared memory.
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;
  static constexpr int kOffDO = kOffQ + kStages * kTileBytes;
  static constexpr int kOffDS = kOffDO + kStages * kTileBytes;
  static constexpr int kDsBytes = kTileM * kTileN * 2;
  static constexpr int kOffLse = kOffDS + kDsBytes;      // 2 x 128 floats
  static constexpr int kOffDvec = kOffLse + 2 * 128 * 4;  // 2 x 128 floats
  static constexpr int kOffBar = kOffDvec + 2 * 128 * 4;
  static constexpr int kNumBars = 2 + 2 * kStages + 1 + 1 + 2 + 2 + 1 + 2;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;
};

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

template <int D>
__global__ void __launch_bounds__(320, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // The 128-byte swizzle anchors at 1024-byte boundaries: refuse to run (and
  // report) if the dynamic shared memory base is not aligned.
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, (unsigned int)FA_ERR_CUDA);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + 1;
  uint64_t* qdo_full = bars + 2;
  uint64_t* qdo_empty = qdo_full + C::kStages;
  uint64_t* s_full = qdo_empty + C::kStages;
  uint64_t* p_ready = s_full + 1;
  uint64_t* dq_full = p_ready + 1;
  uint64_t* dq_empty = dq_full + 1;
  uint64_t* dkv_full = dq_empty + 1;
  uint64_t* dkv_empty = dkv_full + 1;
  uint64_t* drain = dkv_empty + 1;
  uint64_t* stat_ready = drain + 1;  // [2]: L_i / D_i of a step staged in smem
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stat_ready + 2);
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
    }
    mbar_init(s_full, 1);
    mbar_init(p_ready, 128);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(dkv_full, 1);
    mbar_init(dkv_empty, 128);
    mbar_init(drain, 1);
    mbar_init(&stat_ready[0], 128);
    mbar_init(&stat_ready[1], 128);
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
    if (lane == 0) {
      uint32_t kc = 0, qc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const BwdUnit w = decode_bwd(p, u);
        ok = mbar_wait(kv_empty, (kc & 1) ^ 1, ctl, kWaitBwdLoad);
        if (!ok) break;
        mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(smem + C::kOffK + c * C::kChunkBytes, &tm_k, kv_full, c * 64, w.j * kTileN, w.bh);
          tma_load_3d(smem + C::kOffV + c * C::kChunkBytes, &tm_v, kv_full, c * 64, w.j * kTileN, w.bh);
        }
        ++kc;
        for (int ii = 0; ok && ii < w.nq; ++ii) {
          const uint32_t st = qc % C::kStages;
          ok = mbar_wait(&qdo_empty[st], ((qc / C::kStages) & 1) ^ 1, ctl, kWaitBwdLoad);
          if (!ok) break;
          mbar_arrive_expect_tx(&qdo_full[st], 2 * C::kTileBytes);
          const int row = (w.i0 + ii) * kTileM;
          for (int c = 0; c < C::kChunks; ++c) {
            tma_load_3d(smem + C::kOffQ + st * C::kTileBytes + c * C::kChunkBytes, &tm_q, &qdo_full[st], c * 64,
                        row, w.bh);
            tma_load_3d(smem + C::kOffDO + st * C::kTileBytes + c * C::kChunkBytes, &tm_do, &qdo_full[st],
                        c * 64, row, w.bh);
          }
          ++qc;
        }
      }
      if (kc > 0) mbar_wait(kv_full, (kc - 1) & 1, ctl, kWaitDrain);
      const uint32_t first = qc > (uint32_t)C::kStages ? qc - C::kStages : 0u;
      for (uint32_t pos = first; pos < qc; ++pos)
        mbar_wait(&qdo_full[pos % C::kStages], (pos / C::kStages) & 1, ctl, kWaitDrain);
    }
    __syncwarp();
  } else if (warp == 8) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(kTileM, kTileM, false, false);   // S^T, dP^T
      constexpr uint32_t id_kv = idesc_bf16(kTileM, D, false, true);        // dV, dK
      constexpr uint32_t id_dq = idesc_bf16(kTileM, 64, true, true);        // dQ (per 64 columns)
      const uint32_t sk = smem_u32(smem + C::kOffK);
      const uint32_t sv = smem_u32(smem + C::kOffV);
      const uint32_t sds = smem_u32(smem + C::kOffDS);
      uint32_t kc = 0, qc = 0, pc = 0, dqc = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
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
          if (C::kDqAliased && dqc > 0) {
            // S^T and dP^T overwrite the columns the previous dQ tile sits in.
            ok = mbar_wait(dq_empty, (dqc - 1) & 1, ctl, kWaitBwdMma);
            if (!ok) break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * C::kChunkBytes + (kk % 4) * 32;
            mma_ss(tmem + C::kColA, sdesc_sw128(sk + off, 16, 1024), sdesc_sw128(sq + off, 16, 1024), id_s,
                   kk > 0 ? 1u : 0u);
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
          if (!C::kDqAliased && dqc > 0) {
            ok = mbar_wait(dq_empty, (dqc - 1) & 1, ctl, kWaitBwdMma);
            if (!ok) break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk) {
            const uint32_t acc = (ii > 0 || kk > 0) ? 1u : 0u;
            mma_ts(tmem + C::kColDV, tmem + C::kColA + kk * 8, sdesc_sw128(sdo + kk * 2048, C::kChunkBytes, 1024),
                   id_kv, acc);
          }
#pragma unroll
          for (int kk = 0; kk < kTileM / 16; ++kk) {
            const uint32_t acc = (ii > 0 || kk > 0) ? 1u : 0u;
            mma_ts(tmem + C::kColDK, tmem + C::kColB + kk * 8, sdesc_sw128(sq + kk * 2048, C::kChunkBytes, 1024),
                   id_kv, acc);
          }
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk) {
            const uint64_t a = sdesc_sw128(sds + kk * 2048, C::kChunkBytes, 1024);
            mma_ss(tmem + C::kColDQ0, a, sdesc_sw128(sk + kk * 2048, C::kChunkBytes, 1024), id_dq,
                   kk > 0 ? 1u : 0u);
            if (D == 128)
              mma_ss(tmem + C::kColDQ1, a, sdesc_sw128(sk + C::kChunkBytes + kk * 2048, C::kChunkBytes, 1024),
                     id_dq, kk > 0 ? 1u : 0u);
          }
          mma_commit(dq_full);
          ++dqc;
          mma_commit(&qdo_empty[st]);
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
  } else if (warp < 4) {
    // -------------------------------------------- P^T, dS^T and dK/dV output
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const int r = 32 * warp + lane;  // key row within the tile
    const float sl2 = p.scale_log2;
    uint8_t* sds = smem + C::kOffDS;
    uint32_t sc = 0, uc = 0, step = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
      const BwdUnit w = decode_bwd(p, u);
      const int kr = w.j * kTileN + r;  // key index
      const size_t head = (size_t)w.bh * p.N;
      for (int ii = 0; ii < w.nq; ++ii, ++step) {
        const int q0 = (w.i0 + ii) * kTileM;
        {
          // L_i (log2 units) and D_i of the tile's 128 queries; rows past N
          // get L = +inf so their weights vanish.
          const int qr = q0 + r;
          float* bl = sLse + (step & 1) * 128;
          float* bd = sDv + (step & 1) * 128;
          bl[r] = qr < p.N ? p.lse[head + qr] * 1.4426950408889634f : INFINITY;
          bd[r] = qr < p.N ? p.dvec[head + qr] : 0.f;
          // Buffer (step & 1) is reused every other step; all 128 threads
          // arrive once per step, so its k-th use completes phase k.
          mbar_arrive(&stat_ready[step & 1]);
          ok = __all_sync(0xffffffffu, mbar_wait(&stat_ready[step & 1], (step >> 1) & 1, ctl, kWaitBwdSoftmax));
          if (!ok) break;
        }
        const float* bl = sLse + (step & 1) * 128;
        const float* bd = sDv + (step & 1) * 128;
        ok = __all_sync(0xffffffffu, mbar_wait(s_full, sc & 1, ctl, kWaitBwdSoftmax));
        ++sc;
        if (!ok) break;
        tc_fence_after();
        const bool mask = (kr >= p.N) || (p.causal && kr > q0);
#pragma unroll 1
        for (int c = 0; c < kTileM / 32; ++c) {
          uint32_t s[32], dp[32];
          tmem_ld32(tmem + lane_off + C::kColA + 32 * c, s);
          tmem_ld32(tmem + lane_off + C::kColB + 32 * c, dp);
          tmem_ld_wait<32>(s);
          tmem_ld_wait<32>(dp);
          uint32_t pp[16], dd[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float pr[2], dr[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int col = 32 * c + e + h;
              float pv = ex2_approx(fmaf(__uint_as_float(s[e + h]), sl2, -bl[col]));
              if (mask && (kr >= p.N || (p.causal && kr > q0 + col))) pv = 0.f;
              pr[h] = pv;
              dr[h] = pv * (__uint_as_float(dp[e + h]) - bd[col]);
            }
            pp[e / 2] = pack_bf16(pr[0], pr[1]);
            dd[e / 2] = pack_bf16(dr[0], dr[1]);
          }
          tmem_st16(tmem + lane_off + C::kColA + 16 * c, pp);
          tmem_st16(tmem + lane_off + C::kColB + 16 * c, dd);
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
      }
      if (!ok) break;
      // dK_j = scale * sum dS^T Q and dV_j = sum P^T dO of this unit.
      ok = __all_sync(0xffffffffu, mbar_wait(dkv_full, uc & 1, ctl, kWaitBwdSoftmax));
      ++uc;
      if (!ok) break;
      tc_fence_after();
      __nv_bfloat16* dvp = reinterpret_cast<__nv_bfloat16*>(p.dv) + (head + kr) * D;
      __nv_bfloat16* dkp = reinterpret_cast<__nv_bfloat16*>(p.dk) + (head + kr) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
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
  } else {
    // ---------------------------------------------- dQ_i out of TMEM, atomics
    const int wq = warp - 4;
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const int r = 32 * wq + lane;  // query row within the tile
    uint32_t dc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
      const BwdUnit w = decode_bwd(p, u);
      const size_t head = (size_t)w.bh * p.N;
      for (int ii = 0; ii < w.nq; ++ii) {
        ok = __all_sync(0xffffffffu, mbar_wait(dq_full, dc & 1, ctl, kWaitBwdDq));
        ++dc;
        if (!ok) break;
        tc_fence_after();
        uint32_t g[D];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          const uint32_t col = (c < 2) ? C::kColDQ0 + 32 * c : C::kColDQ1 + 32 * (c - 2);
          tmem_ld32(tmem + lane_off + col, g + 32 * c);
        }
        tmem_ld_wait<D>(g);
        tc_fence_before();
        mbar_arrive(dq_empty);
        const int qr = (w.i0 + ii) * kTileM + r;
        if (qr < p.N) {
          float4* dst = reinterpret_cast<float4*>(p.dq_acc + (head + qr) * D);
#pragma unroll
          for (int c = 0; c < D / 4; ++c)
            atomicAdd(dst + c, make_float4(__uint_as_float(g[4 * c]), __uint_as_float(g[4 * c + 1]),
                                           __uint_as_float(g[4 * c + 2]), __uint_as_float(g[4 * c + 3])));
        }
      }
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
