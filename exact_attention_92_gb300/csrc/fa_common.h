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

// Queries and keys may differ in length (Nq, Nk).  With the causal mask,
// query row i sees key j iff j <= i + causal_off: 0 for top-left alignment,
// Nk - Nq for bottom-right.  A query row that sees no key (i + causal_off <
// 0) gets O = 0 and L = -inf, and zero gradients.
struct FwdParams {
  int B, H;
  int Nq, Nk;                  // query / key rows per head
  int Hkv;                     // key/value heads (H for plain multi-head attention)
  int causal;
  int causal_off;              // query row i sees keys j <= i + causal_off
  float scale_log2;            // scale * log2(e)
  int num_splits;              // 1: write o/lse directly
  int kv_tiles_per_split;
  int num_q_blocks;            // ceil(Nq / 256)
  int num_units;               // B*H*num_q_blocks*num_splits
  void* o;                     // bf16 [B,H,Nq,d]           (num_splits == 1)
  float* lse;                  // fp32 [B,H,Nq]             (num_splits == 1)
  float* o_part;               // fp32 [S,B,H,Nq,d]         (num_splits > 1)
  float* lse_part;             // fp32 [S,B,H,Nq]           (num_splits > 1)
  int store32;                 // o is 32-byte aligned: 32-byte stores
  unsigned int* status;
  unsigned long long timeout_ns;
};

struct CombineParams {
  int rows;                    // B*H*Nq
  int num_splits;
  const float* o_part;
  const float* lse_part;
  void* o;
  float* lse;
};

struct BwdParams {
  int B, H;
  int Nq, Nk;                  // query / key rows per head
  int Hkv;                     // key/value heads (H for plain multi-head attention)
  int causal;
  int causal_off;              // query row i sees keys j <= i + causal_off
  float scale;                 // softmax scale
  float scale_log2;            // scale * log2(e)
  const float* lse;            // fp32 [B,H,Nq]
  const float* dvec;           // fp32 [B,H,Nq], D = rowsum(dO * O)
  void* dq;                    // bf16 [B,H,Nq,d]
  void* dk;                    // bf16 [B,Hkv,Nk,d]
  void* dv;                    // bf16 [B,Hkv,Nk,d]
  int store32;                 // dq, dk, dv all 32-byte aligned: 32-byte stores
  int num_q_tiles;             // ceil(Nq / 128)
  int num_k_tiles;             // ceil(Nk / 128)
  // Tiles that take part: key tiles [0, kv_tiles_used) are seen by some query
  // row, query tiles [q_tile_first, num_q_tiles) see some key.  The host
  // zeroes the gradient rows of the other tiles.
  int kv_tiles_used;
  int q_tile_first;
  int num_units;               // B*H*(num_q_tiles - q_tile_first) (dQ kernel: query heads)
  int num_units_kv;            // B*Hkv*kv_tiles_used (dK/dV kernel: key/value heads)
  int group;                   // H / Hkv: query heads per key/value head
  unsigned int* status;
  unsigned long long timeout_ns;
};

}  // namespace fa
