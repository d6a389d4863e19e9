// Internal declarations shared by the host API and the kernels.
#pragma once

#include <cstdint>

#include "fa.h"

namespace fa {

// Tile sizes.  A CTA of the forward kernel owns two 128-row query tiles that
// share one stream of 128-row key/value tiles.
constexpr int kTileM = 128;   // query rows per tile (tcgen05 M)
constexpr int kTileN = 128;   // keys per tile
constexpr int kQTilesPerCta = 2;

// Grouped-query attention: H query heads share Hkv key/value heads (H a
// multiple of Hkv), query head h of a batch reading key/value head
// h / (H / Hkv).  Heads are numbered b * H + h (queries) and b * Hkv + hk
// (keys and values).
__host__ __device__ inline int kv_head_of(int bh, int H, int Hkv) {
  return (bh / H) * Hkv + (bh % H) / (H / Hkv);
}
// The j-th query head (j < H / Hkv) that reads key/value head `kvbh`.
__host__ __device__ inline int q_head_of(int kvbh, int j, int H, int Hkv) {
  return (kvbh / Hkv) * H + (kvbh % Hkv) * (H / Hkv) + j;
}

// Codes stored in bits [8,16) of the status word to say which wait gave up.
enum WaitSite : uint32_t {
  kWaitQFull = 1,
  kWaitQEmpty,
  kWaitKvFull,
  kWaitKvEmpty,
  kWaitSFull,
  kWaitPFull,
  kWaitOFull,
  kWaitDrain,
  kWaitSelfTest,
  kWaitBwdLoad,
  kWaitBwdMma,
  kWaitBwdSoftmax,
  kWaitBwdDq,
};

struct FwdParams {
  int B, H, N;
  int Hkv;                     // key/value heads (H for plain multi-head attention)
  int causal;
  float scale_log2;            // scale * log2(e)
  int num_splits;              // 1: write o/lse directly
  int kv_tiles_per_split;
  int num_q_blocks;            // ceil(N / 256)
  int num_units;               // B*H*num_q_blocks*num_splits
  void* o;                     // bf16 [B,H,N,d]            (num_splits == 1)
  float* lse;                  // fp32 [B,H,N]              (num_splits == 1)
  float* o_part;               // fp32 [S,B,H,N,d]          (num_splits > 1)
  float* lse_part;             // fp32 [S,B,H,N]            (num_splits > 1)
  int store32;                 // o is 32-byte aligned: 32-byte stores
  unsigned int* status;
  unsigned long long timeout_ns;
};

struct CombineParams {
  int rows;                    // B*H*N
  int num_splits;
  const float* o_part;
  const float* lse_part;
  void* o;
  float* lse;
};

struct BwdParams {
  int B, H, N;
  int Hkv;                     // key/value heads (H for plain multi-head attention)
  int causal;
  float scale;                 // softmax scale
  float scale_log2;            // scale * log2(e)
  const float* lse;            // fp32 [B,H,N]
  const float* dvec;           // fp32 [B,H,N], D = rowsum(dO * O)
  void* dq;                    // bf16 [B,H,N,d]
  void* dk;                    // bf16 [B,H,N,d]
  void* dv;                    // bf16 [B,H,N,d]
  int store32;                 // dq, dk, dv all 32-byte aligned: 32-byte stores
  int num_tiles;               // ceil(N / 128): key tiles = query tiles
  int num_units;               // B*H*num_tiles (dQ kernel: query heads)
  int num_units_kv;            // B*Hkv*num_tiles (dK/dV kernel: key/value heads)
  int group;                   // H / Hkv: query heads per key/value head
  unsigned int* status;
  unsigned long long timeout_ns;
};

}  // namespace fa
