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
  // 0: row i of a head is query position i.  > 0: the query heads of a
  // key/value group are packed as the rows of one head (the caller's
  // [B, H, Nq, d] seen as [B, Hkv, G*Nq, d]) and row r is query position
  // r % q_period (= Nq) for the causal mask.
  int q_period;
  // > 0: units are listed head window by head window (that many heads at a
  // time, all of their query blocks) instead of query block by query block
  // over all heads, so the K and V read by the CTAs in flight stay in L2.
  // Used without the causal mask, where every unit has the same work.
  int head_window;
  unsigned int* status;
  unsigned long long timeout_ns;
  // 1: every unit has at most 128 query rows (decoding), and both query
  // tiles of a unit hold those rows, tile t taking the key tiles kvb + t,
  // kvb + t + 2, ... of the unit's split; each tile writes its own partial
  // result (partial 2 * split + t of 2 * num_splits, merged afterwards).
  int dual;
};

// Query position of row r (see FwdParams::q_period).
__host__ __device__ inline int query_pos(int r, int q_period) { return q_period > 0 ? r % q_period : r; }

// Largest query position among rows [r0, r1] (r0 <= r1).
__host__ __device__ inline int max_query_pos(int r0, int r1, int q_period) {
  if (q_period <= 0) return r1;
  if (r1 - r0 + 1 >= q_period) return q_period - 1;
  const int a = r0 % q_period, b = r1 % q_period;
  return a <= b ? b : q_period - 1;
}

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
