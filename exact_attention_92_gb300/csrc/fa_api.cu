// Host side of the C ABI declared in include/fa.h: argument validation,
// tensor-map encoding, the split-KV decision, stream-ordered workspace and the
// device status word read by fa_poll_status.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "fa_common.h"

namespace fa {
cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_combine(int d, const CombineParams& p, cudaStream_t stream);
cudaError_t launch_fwd256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                          int grid, cudaStream_t stream);
cudaError_t launch_bwd256_kv(bool dk_pass, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd256_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_dkdv_pair(const CUtensorMap& tq64, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo64, const CUtensorMap& tdo,
                                 const BwdParams& p, int sm_count, cudaStream_t stream);
cudaError_t launch_bwd_dq(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_preprocess(int d, const void* o, const void* dout, float* dvec, int rows,
                                  cudaStream_t stream);
cudaError_t launch_selftest_wait(unsigned int* status, unsigned long long timeout_ns, cudaStream_t stream);
}  // namespace fa

// One status word per device that loads the library.  Kernels record the
// first failing wait here; fa_poll_status reads and clears it.
static __device__ unsigned int g_fa_status_word;

namespace {

using fa::FwdParams;

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::mutex mu;
  bool ready = false;
  int sm_count = 0;
  double l2_bytes = 0.0;
  unsigned int* status = nullptr;  // device address of g_fa_status_word
  cudaMemPool_t pool = nullptr;    // the library's workspace pool on this device
};

DeviceState g_dev[kMaxDevices];
std::atomic<unsigned long long> g_timeout_ns{2000000000ull};

std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// Set-up of the current device: compute capability check, SM count, the
// workspace pool and the address of the status word (cleared).  It is kept once it has succeeded; a
// set-up that failed (for instance inside a stream capture, where the
// clearing memset is not allowed) is tried again by the next call.  A device
// that is not an sm_103 part is refused every time.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  DeviceState& s = g_dev[dev];
  {
    std::lock_guard<std::mutex> g(s.mu);
    if (!s.ready) {
      cudaDeviceProp prop;
      if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FA_ERR_CUDA;
      if (!(prop.major == 10 && prop.minor == 3)) return FA_ERR_UNSUPPORTED;
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_fa_status_word) != cudaSuccess || addr == nullptr) {
        cudaGetLastError();
        return FA_ERR_CUDA;
      }
      if (cudaMemset(addr, 0, sizeof(unsigned int)) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
      }
      // Workspace pool: stream-ordered like the device's default pool, but
      // it keeps freed memory reserved for later calls (no release
      // threshold).  The default pool returns its memory at every
      // synchronisation, so each call after one would map its workspace
      // afresh: 170-200 us for the 67-134 MB of split partials of one
      // 65536-token head.  fa_trim_workspace gives the memory back.
      if (s.pool == nullptr) {
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
          cudaGetLastError();
          return FA_ERR_CUDA;
        }
        cuuint64_t keep = ~(cuuint64_t)0;
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
          cudaGetLastError();
          cudaMemPoolDestroy(pool);
          return FA_ERR_CUDA;
        }
        s.pool = pool;
      }
      s.sm_count = prop.multiProcessorCount;
      s.l2_bytes = (double)prop.l2CacheSize;
      s.status = static_cast<unsigned int*>(addr);
      s.ready = true;
    }
  }
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return FA_ERR_CUDA;
  *out = &s;
  return FA_OK;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Number of key splits with the causal mask (no packed query heads, query
// blocks of q_block rows over key tiles of key_tile keys): units then carry
// unequal work -- the key tiles their last row sees -- and the longest-first
// order balances them, so the count is chosen on an estimate of the
// slowest SM's load in key-tile steps:
//   max(the largest unit split S ways, the average load per SM, plus 2% a
//   split for the extra units) + the split partials' traffic (written by
//   the forward, read by the merge: about half a step per MB at head dim
//   128, measured on B=1 H=1..4 N=16K..64K).
int choose_splits_causal(long long BH, int qblocks, int q_block, int key_tile, int Nq, int nkv, int causal_off,
                         int d, int min_tiles, int sm_count) {
  long long total = 0;
  int max1 = 0;
  for (int qb = 0; qb < qblocks; ++qb) {
    const int last_key = std::min(Nq, (qb + 1) * q_block) - 1 + causal_off;
    const int n = last_key < 0 ? 0 : std::min(nkv, last_key / key_tile + 1);
    total += n;
    max1 = std::max(max1, n);
  }
  const double avg = (double)(total * BH) / sm_count;
  const double rows = (double)BH * Nq;
  int best_s = 1;
  double best = std::max((double)max1, avg);
  // Powers of two only: with 3 splits the unit list's mix of long and short
  // splits broke the longest-first deal (measured 30% slower than 2 or 4).
  for (int s = 2; s <= 16; s *= 2) {
    if (nkv / s < min_tiles) break;
    const double load = std::max((double)((max1 + s - 1) / s), avg * (1.0 + 0.02 * (s - 1)));
    const double cost = load + 0.5e-6 * s * rows * d * 4.0;
    if (cost < best) {
      best = cost;
      best_s = s;
    }
  }
  return best_s;
}

// Number of key splits when each (batch*head) unit has a single query tile
// (decoding steps, or grouped query heads packed into one tile): a step is
// then a chain of one tile's S, softmax and P V, paced by latency rather
// than by the tensor pipe or memory, and each unit pays a fixed start and
// finish (its Q and first K, V from memory, the partial write-out) of about
// three steps (fitted on GQA decoding at head dim 64 and 128 with 8K and
// 32K keys).  So the count minimises waves x (key tiles per split + 3).
// With both query tiles on a unit's rows (dual mode, `chains` = 2) a unit's
// key tiles take half as many steps, and its second partial result one step
// more; dual mode asks for at least 8 key tiles a split (four steps a tile).
// Returns the count, and its estimated cost in *cost (-1: none qualifies).
int choose_splits_single_tile(long long units, int nkv, int min_tiles, int sm_count, int chains,
                              long long* cost_out = nullptr) {
  const int unit_steps = chains == 2 ? 4 : 3;
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= 16; ++s) {
    if (s > 1 && nkv / s < min_tiles) break;
    const int per = (nkv + s - 1) / s;
    if (chains == 2 && per < 8) break;
    const long long u = units * ((nkv + per - 1) / per);  // non-empty splits
    const long long waves = (u + sm_count - 1) / sm_count;
    const long long cost = waves * ((per + chains - 1) / chains + unit_steps);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  if (cost_out) *cost_out = best_cost;
  return best;
}

// Stream-ordered workspace from the device's library pool (returned with
// cudaFreeAsync on the same stream).  For failure-path tests, the
// environment variable FA_TEST_FAIL_ALLOC (any value but "0") makes every
// workspace allocation report failure without allocating.
cudaError_t ws_alloc(cudaMemPool_t pool, void** ptr, size_t bytes, cudaStream_t st) {
  const char* f = std::getenv("FA_TEST_FAIL_ALLOC");
  if (f != nullptr && std::strcmp(f, "0") != 0) return cudaErrorMemoryAllocation;
  return cudaMallocFromPoolAsync(ptr, bytes, pool, st);
}

// Head dims of the library: 64, 96, 128 and 256 (forward and backward).
bool fwd_head_dim(int d) { return d == 64 || d == 96 || d == 128 || d == 256; }
bool bwd_head_dim(int d) { return fwd_head_dim(d); }

int validate(int B, int H, int Nq, int Nk, int d, float scale, bool backward = false) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (!(backward ? bwd_head_dim(d) : fwd_head_dim(d))) return FA_ERR_UNSUPPORTED;
  const long double n = Nq > Nk ? Nq : Nk;
  if ((long double)B * H * n * d >= 9.0e18L) return FA_ERR_INVALID_ARG;
  // Row and unit indices are 32-bit: B*H*Nq rows, (query block, split) units.
  if ((long long)B * H * Nq > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  if ((long long)B * H * ((Nq + 255) / 256) * 64 > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  if ((long long)B * H * ((Nk + 127) / 128) > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Mask offset of the causal code: query row i sees keys j <= i + offset.
int causal_offset(int causal, int Nq, int Nk) { return causal == FA_CAUSAL_BOTTOM_RIGHT ? Nk - Nq : 0; }

// [B*H, N, d] bf16 viewed as a 3-D tensor (d innermost); boxes of 64 x 128 x 1
// with the 128-byte swizzle the MMA descriptors expect.  Rows past N, and the
// columns of the second 64-column box past d = 96, read as zero.
int encode_bhnd(CUtensorMap* m, const void* ptr, int BH, int N, int d, int box_rows = 128) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Number of key splits: only when the (batch*head, query block) units cannot
// fill the GPU.  Picks the split count with the best last-wave occupancy,
// keeping at least 4 key tiles per split.
int choose_splits(long long units, int nkv, int min_tiles, int sm_count) {
  if (units >= 2LL * sm_count) return 1;
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= 16; ++s) {
    if (s > 1 && nkv / s < min_tiles) break;
    const long long u = units * s;
    const long long waves = (u + sm_count - 1) / sm_count;
    const double eff = (double)u / (double)(waves * sm_count) - 0.01 * (s - 1);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

// Size checks shared by the forward call and its plan.
int check_fwd_sizes(int B, int H, int Hkv, int Nq, int Nk, int d, int causal, int num_splits) {
  int e = validate(B, H, Nq, Nk, d, 1.0f);
  if (e) return e;
  if (Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal < FA_CAUSAL_NONE || causal > FA_CAUSAL_BOTTOM_RIGHT) return FA_ERR_INVALID_ARG;
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// The host-side decisions of a forward call (fa_fwd_plan_t), for sizes that
// passed check_fwd_sizes.  FA_ERR_INVALID_ARG when a forced split count
// would make more units than a 32-bit unit index holds.
int plan_fwd(int B, int H, int Hkv, int Nq, int Nk, int d, int causal, int num_splits, int sm_count,
             double l2_bytes, fa_fwd_plan_t* pl) {
  std::memset(pl, 0, sizeof(*pl));
  const int causal_off = causal_offset(causal, Nq, Nk);
  // Grouped query heads with fewer than 128 query rows (decoding, short
  // chunks): the G query heads of a key/value head share one tile as G * Nq
  // rows -- the caller's contiguous [B, H, Nq, d] seen as [B, Hkv, G * Nq, d],
  // so O and L land where they belong -- and K, V are read once per group.
  // Row r of such a tile is query position r % Nq for the causal mask.
  const int G = H / Hkv;
  const bool pack = G > 1 && Nq < 128;
  if (pack) {
    H = Hkv;
    Nq *= G;
  }
  const int BH = B * H;
  // Work units: (batch*head, query block, key split).  A query block is 256
  // rows (two 128-row tiles) with 128-key tiles, or at d = 256 one 128-row
  // tile with 64-key tiles.
  const bool wide = d == 256;
  const int q_block = wide ? 128 : 256;
  const int key_tile = wide ? 64 : 128;
  const int nkv = (Nk + key_tile - 1) / key_tile;
  const int qblocks = (Nq + q_block - 1) / q_block;
  // Units of a single query tile (decoding) leave the second tile of a CTA
  // idle: with enough key tiles both tiles then take the unit's rows and
  // half of its key tiles each (dual mode), their partial results merged,
  // when the step model above prefers that to one tile per unit.
  bool dual = false;
  int S = num_splits;
  if (S == 0) {
    S = choose_splits((long long)BH * qblocks, nkv, wide ? 8 : 4, sm_count);
    if (!wide && Nq <= fa::kTileM) {
      long long c1 = -1, c2 = -1;
      const int s1 = choose_splits_single_tile(BH, nkv, 4, sm_count, 1, &c1);
      const int s2 = choose_splits_single_tile(BH, nkv, 4, sm_count, 2, &c2);
      if (c2 >= 0 && c2 < c1) {
        dual = true;
        S = s2;
      } else if (S > 1 && (pack || causal == FA_CAUSAL_NONE || Nq == 1)) {
        S = s1;
      } else if (S > 1 && causal != FA_CAUSAL_NONE && !pack) {
        S = choose_splits_causal(BH, qblocks, q_block, key_tile, Nq, nkv, causal_off, d, 4, sm_count);
      }
    } else if (S > 1 && causal != FA_CAUSAL_NONE && !pack && !wide) {
      S = choose_splits_causal(BH, qblocks, q_block, key_tile, Nq, nkv, causal_off, d, 4, sm_count);
    }
  }
  if (S > nkv) S = nkv;
  if (S < 1) S = 1;
  const int per_split = (nkv + S - 1) / S;
  S = (nkv + per_split - 1) / per_split;  // no empty split
  if ((long long)BH * qblocks * S > 0x7fffffffLL) return FA_ERR_INVALID_ARG;

  pl->packed_heads = pack ? 1 : 0;
  pl->unit_heads = BH;
  pl->unit_rows = Nq;
  pl->query_block = q_block;
  pl->key_tile = key_tile;
  pl->key_tiles = nkv;
  pl->num_splits = S;
  pl->key_tiles_per_split = per_split;
  pl->dual = dual ? 1 : 0;
  const int parts = dual ? 2 * S : S;  // partial results to merge
  pl->partials = parts > 1 ? parts : 0;
  pl->num_units = BH * qblocks * S;
  pl->grid = pl->num_units < sm_count ? pl->num_units : sm_count;
  // Without the causal mask every unit has the same work, so the units can
  // be listed window by window of heads without losing balance: a window is
  // the fewest heads whose query blocks fill one round of CTAs, and the K, V
  // of the heads in flight then stay in L2.  Only when the K and V of all
  // heads exceed half the L2 (otherwise they stay there anyway).
  const double kv_bytes = 4.0 * (double)B * Hkv * Nk * d;
  if (causal == FA_CAUSAL_NONE && S == 1 && kv_bytes > l2_bytes / 2) {
    const int win = (pl->grid + qblocks - 1) / qblocks;
    pl->head_window = win < BH ? win : 0;
  }
  pl->launches = pl->partials > 0 ? 2 : 1;
  pl->workspace_bytes = pl->partials > 0 ? (uint64_t)parts * BH * Nq * ((uint64_t)d + 1) * sizeof(float) : 0;
  return FA_OK;
}

// Size checks shared by the backward call and its plan.
int check_bwd_sizes(int B, int H, int Hkv, int Nq, int Nk, int d, int causal) {
  int e = validate(B, H, Nq, Nk, d, 1.0f, true);
  if (e) return e;
  if (Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal < FA_CAUSAL_NONE || causal > FA_CAUSAL_BOTTOM_RIGHT) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// The host-side decisions of a backward call (fa_bwd_plan_t), for sizes
// that passed check_bwd_sizes.
void plan_bwd(int B, int H, int Hkv, int Nq, int Nk, int d, int causal, int sm_count, fa_bwd_plan_t* pl) {
  std::memset(pl, 0, sizeof(*pl));
  pl->q_tiles = (Nq + 127) / 128;
  pl->k_tiles = (Nk + 127) / 128;
  // With the causal mask: key tiles past the last key the last query row
  // sees, and query tiles whose rows all see no key (a negative offset),
  // take no part; their gradient rows are zero.
  pl->kv_tiles_used = pl->k_tiles;
  pl->q_tile_first = 0;
  if (causal != FA_CAUSAL_NONE) {
    const int off = causal_offset(causal, Nq, Nk);
    const int last_key = Nq - 1 + off;  // >= 0 for both alignments
    pl->kv_tiles_used = std::min(pl->k_tiles, last_key / 128 + 1);
    if (off < 0) pl->q_tile_first = (-off) / 128;
  }
  pl->dq_units = B * H * (pl->q_tiles - pl->q_tile_first);
  pl->dq_grid = pl->dq_units < sm_count ? pl->dq_units : sm_count;
  pl->kv_cta_pair = d == 128 ? 1 : 0;
  pl->kv_units = B * Hkv * (pl->kv_cta_pair ? (pl->kv_tiles_used + 1) / 2 : pl->kv_tiles_used);
  pl->kv_passes = d == 256 ? 2 : 1;
  pl->launches = 2 + pl->kv_passes;
  const uint64_t row_bytes = (uint64_t)d * 2;
  pl->zeroed_dq_bytes =
      (uint64_t)B * H * std::min((uint64_t)Nq, (uint64_t)pl->q_tile_first * 128) * row_bytes;
  pl->zeroed_dkdv_bytes =
      2ull * B * Hkv * ((uint64_t)Nk - std::min((uint64_t)Nk, (uint64_t)pl->kv_tiles_used * 128)) * row_bytes;
  pl->workspace_bytes = (uint64_t)B * H * Nq * sizeof(float);
}

// ---------------------------------------------------------------- timing

struct TimingRec {
  cudaEvent_t a, b;
  int kernel;
};
std::mutex g_tmu;
bool g_timing = false;
// Launches of each library kernel since the library was loaded (always on).
std::atomic<unsigned long long> g_launches[FA_KERNEL_BWD_DQ + 1];
std::vector<TimingRec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t pool_get() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Runs `launch` (returning cudaError_t); when timing is on, brackets it with
// events on `stream`.
template <typename F>
cudaError_t timed(int kernel, cudaStream_t stream, F&& launch) {
  TimingRec r{nullptr, nullptr, kernel};
  {
    std::lock_guard<std::mutex> g(g_tmu);
    if (g_timing) {
      r.a = pool_get();
      r.b = pool_get();
    }
  }
  if (r.a && r.b) cudaEventRecord(r.a, stream);
  cudaError_t e = launch();
  if (e == cudaSuccess) g_launches[kernel].fetch_add(1, std::memory_order_relaxed);
  if (r.a && r.b) {
    cudaEventRecord(r.b, stream);
    std::lock_guard<std::mutex> g(g_tmu);
    g_recs.push_back(r);
  }
  return e;
}

}  // namespace

namespace fa {
// Accessors for entry points defined in other files of the library.
int internal_device_setup(unsigned int** status, int* sm_count) {
  DeviceState* s = nullptr;
  const int e = device_state(&s);
  if (e) return e;
  *status = s->status;
  *sm_count = s->sm_count;
  return FA_OK;
}
int internal_validate(int B, int H, int N, int d, float scale) { return validate(B, H, N, N, d, scale, true); }
int internal_encode_bhnd(CUtensorMap* m, const void* ptr, int BH, int N, int d, int box_rows) {
  return encode_bhnd(m, ptr, BH, N, d, box_rows);
}
unsigned long long internal_wait_timeout_ns() { return g_timeout_ns.load(); }
// A launch of library kernel `kernel` by another file of the library, counted
// and (while timing is on) bracketed by events like the launches here.
cudaError_t internal_timed_launch(int kernel, cudaStream_t stream, cudaError_t (*launch)(void*), void* ctx) {
  return timed(kernel, stream, [&] { return launch(ctx); });
}
}  // namespace fa

extern "C" {

int fa_timing_enable(int on) {
  std::lock_guard<std::mutex> g(g_tmu);
  for (auto& r : g_recs) {
    cudaEventSynchronize(r.b);
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
  g_timing = on != 0;
  return FA_OK;
}

int fa_launch_count(int kernel, uint64_t* count) {
  if (!count || kernel < 0 || kernel > FA_KERNEL_BWD_DQ) return FA_ERR_INVALID_ARG;
  *count = g_launches[kernel].load(std::memory_order_relaxed);
  return FA_OK;
}

int fa_timing_read(int kernel, int* launches, double* total_ms) {
  if (!launches || !total_ms || kernel < 0 || kernel > FA_KERNEL_BWD_DQ) return FA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(g_tmu);
  int n = 0;
  double ms = 0.0;
  std::vector<TimingRec> keep;
  for (auto& r : g_recs) {
    if (r.kernel != kernel) {
      keep.push_back(r);
      continue;
    }
    if (cudaEventSynchronize(r.b) != cudaSuccess) return FA_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return FA_ERR_CUDA;
    ms += t;
    ++n;
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.swap(keep);
  *launches = n;
  *total_ms = ms;
  return FA_OK;
}

int fa_abi_version(void) { return FA_ABI_VERSION; }

int fa_trim_workspace(void) {
  DeviceState* s = nullptr;
  const int e = device_state(&s);
  if (e) return e;
  return cudaMemPoolTrimTo(s->pool, 0) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null or misaligned pointer, bad size or scale";
    case FA_ERR_UNSUPPORTED:
      return "FA_ERR_UNSUPPORTED: head dim must be 64, 96, 128 or 256 (fa_bwd_noalloc: not 256) on an sm_103 GPU";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA runtime or launch failure";
    case FA_ERR_NO_MEMORY: return "FA_ERR_NO_MEMORY: workspace allocation failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a device-side wait gave up";
    case FA_ERR_SCRATCH_TOO_SMALL:
      return "FA_ERR_SCRATCH_TOO_SMALL: problem needs more than the static scratch of fa_bwd_noalloc";
    default: return "unknown fa_status";
  }
}

uint64_t fa_set_wait_timeout_ns(uint64_t ns) { return g_timeout_ns.exchange(ns); }

int fa_poll_status(void* stream) {
  DeviceState* s = nullptr;
  int e = device_state(&s);
  if (e) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, s->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (word != 0u && cudaMemset(s->status, 0, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
  return (int)(word & 0xffu);
}

int fa_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
  DeviceState* s = nullptr;
  int e = device_state(&s);
  if (e) return e;
  return fa::launch_selftest_wait(s->status, timeout_ns, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

int fa_fwd_plan(int B, int H, int Hkv, int Nq, int Nk, int d, int causal, int num_splits, int sm_count,
                uint64_t l2_bytes, fa_fwd_plan_t* plan) {
  if (plan == nullptr || sm_count < 1) return FA_ERR_INVALID_ARG;
  const int e = check_fwd_sizes(B, H, Hkv, Nq, Nk, d, causal, num_splits);
  if (e) return e;
  fa_fwd_plan_t pl;
  const int e2 = plan_fwd(B, H, Hkv, Nq, Nk, d, causal, num_splits, sm_count, (double)l2_bytes, &pl);
  if (e2 == FA_OK) *plan = pl;
  return e2;
}

int fa_fwd_general(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                   int Nq, int Nk, int d, int causal, float scale, int num_splits, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  int e = check_fwd_sizes(B, H, Hkv, Nq, Nk, d, causal, num_splits);
  if (e) return e;
  DeviceState* s = nullptr;
  e = device_state(&s);
  if (e) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  fa_fwd_plan_t pl;
  e = plan_fwd(B, H, Hkv, Nq, Nk, d, causal, num_splits, s->sm_count, s->l2_bytes, &pl);
  if (e) return e;
  const bool wide = d == 256;
  const int BH = pl.unit_heads;
  const int rows_per_head = pl.unit_rows;

  CUtensorMap tq, tk, tv;
  if (encode_bhnd(&tq, q, BH, rows_per_head, d) || encode_bhnd(&tk, k, B * Hkv, Nk, d, pl.key_tile) ||
      encode_bhnd(&tv, v, B * Hkv, Nk, d, pl.key_tile))
    return FA_ERR_CUDA;

  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.B = B;
  p.H = pl.packed_heads ? Hkv : H;
  p.Hkv = Hkv;
  p.Nq = rows_per_head;
  p.Nk = Nk;
  p.causal = causal != FA_CAUSAL_NONE ? 1 : 0;
  p.causal_off = causal_offset(causal, Nq, Nk);
  p.q_period = pl.packed_heads ? Nq : 0;  // query position of packed row r: r % Nq
  p.scale_log2 = scale * 1.4426950408889634f;
  p.num_splits = pl.num_splits;
  p.kv_tiles_per_split = pl.key_tiles_per_split;
  p.num_q_blocks = (rows_per_head + pl.query_block - 1) / pl.query_block;
  p.num_units = pl.num_units;
  p.o = o;
  p.lse = lse;
  p.store32 = (reinterpret_cast<uintptr_t>(o) & 31) == 0 ? 1 : 0;
  p.head_window = pl.head_window;
  p.status = s->status;
  p.timeout_ns = g_timeout_ns.load();
  p.dual = pl.dual;

  void* ws = nullptr;
  if (pl.partials > 0) {
    if (ws_alloc(s->pool, &ws, pl.workspace_bytes, st) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_NO_MEMORY;
    }
    p.o_part = static_cast<float*>(ws);
    p.lse_part = p.o_part + (size_t)pl.partials * BH * rows_per_head * d;
  }
  cudaError_t ce = timed(FA_KERNEL_FWD, st, [&] {
    return wide ? fa::launch_fwd256(tq, tk, tv, p, pl.grid, st) : fa::launch_fwd(d, tq, tk, tv, p, pl.grid, st);
  });
  if (ce == cudaSuccess && pl.partials > 0) {
    fa::CombineParams c;
    c.rows = BH * rows_per_head;
    c.num_splits = pl.partials;
    c.o_part = p.o_part;
    c.lse_part = p.lse_part;
    c.o = o;
    c.lse = lse;
    ce = timed(FA_KERNEL_COMBINE, st, [&] { return fa::launch_combine(d, c, st); });
  }
  if (ws) cudaFreeAsync(ws, st);
  return ce == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N,
               int d, int causal, float scale, int num_splits, void* stream) {
  return fa_fwd_general(q, k, v, o, lse, B, H, Hkv, N, N, d, causal ? FA_CAUSAL_TOP_LEFT : FA_CAUSAL_NONE, scale,
                        num_splits, stream);
}

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
              int causal, float scale, int num_splits, void* stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, causal, scale, num_splits, stream);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           int causal, float scale, void* stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, causal, scale, 0, stream);
}

int fa_bwd_plan(int B, int H, int Hkv, int Nq, int Nk, int d, int causal, int sm_count, fa_bwd_plan_t* plan) {
  if (plan == nullptr || sm_count < 1) return FA_ERR_INVALID_ARG;
  const int e = check_bwd_sizes(B, H, Hkv, Nq, Nk, d, causal);
  if (e) return e;
  plan_bwd(B, H, Hkv, Nq, Nk, d, causal, sm_count, plan);
  return FA_OK;
}

int fa_bwd_general(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq, int Nk, int d,
                   int causal, float scale, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  int e = check_bwd_sizes(B, H, Hkv, Nq, Nk, d, causal);
  if (e) return e;
  DeviceState* s = nullptr;
  e = device_state(&s);
  if (e) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  fa_bwd_plan_t pl;
  plan_bwd(B, H, Hkv, Nq, Nk, d, causal, s->sm_count, &pl);
  const int BH = B * H;
  const size_t rows = (size_t)BH * Nq;

  // Tensor maps: 128-row boxes; at d = 256 also 64-row ones (the query steps
  // of the key/value kernel, the key steps of the dQ kernel), at d = 128
  // 64-row ones of Q and dO (each CTA's half of a query tile in the CTA-pair
  // dK/dV kernel).
  const bool wide = pl.kv_passes == 2;
  const bool pair = pl.kv_cta_pair != 0;
  CUtensorMap tq, tk, tv, tdo, tq64, tk64, tv64, tdo64;
  if (encode_bhnd(&tq, q, BH, Nq, d) || encode_bhnd(&tk, k, B * Hkv, Nk, d) ||
      encode_bhnd(&tv, v, B * Hkv, Nk, d) || encode_bhnd(&tdo, dout, BH, Nq, d))
    return FA_ERR_CUDA;
  if ((wide || pair) && (encode_bhnd(&tq64, q, BH, Nq, d, 64) || encode_bhnd(&tdo64, dout, BH, Nq, d, 64)))
    return FA_ERR_CUDA;
  if (wide && (encode_bhnd(&tk64, k, B * Hkv, Nk, d, 64) || encode_bhnd(&tv64, v, B * Hkv, Nk, d, 64)))
    return FA_ERR_CUDA;

  fa::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.causal = causal != FA_CAUSAL_NONE ? 1 : 0;
  p.causal_off = causal_offset(causal, Nq, Nk);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.store32 = ((reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) |
                reinterpret_cast<uintptr_t>(dv)) & 31u) == 0 ? 1 : 0;
  p.num_q_tiles = pl.q_tiles;
  p.num_k_tiles = pl.k_tiles;
  p.kv_tiles_used = pl.kv_tiles_used;
  p.q_tile_first = pl.q_tile_first;
  p.num_units = pl.dq_units;
  p.num_units_kv = B * Hkv * pl.kv_tiles_used;  // key tiles; the pair kernel takes two a unit
  p.group = H / Hkv;
  p.status = s->status;
  p.timeout_ns = g_timeout_ns.load();

  // Workspace: D [rows].
  void* ws = nullptr;
  if (ws_alloc(s->pool, &ws, pl.workspace_bytes, st) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_NO_MEMORY;
  }
  float* dvec = static_cast<float*>(ws);
  p.dvec = dvec;

  cudaError_t ce = cudaSuccess;
  const size_t row_bytes = (size_t)d * 2;
  if (p.kv_tiles_used < p.num_k_tiles) {
    const size_t r0 = (size_t)p.kv_tiles_used * 128;
    for (void* g : {dk, dv})
      if (ce == cudaSuccess)
        ce = cudaMemset2DAsync(static_cast<uint8_t*>(g) + r0 * row_bytes, (size_t)Nk * row_bytes, 0,
                               ((size_t)Nk - r0) * row_bytes, (size_t)B * Hkv, st);
  }
  if (ce == cudaSuccess && p.q_tile_first > 0) {
    const size_t r1 = std::min((size_t)Nq, (size_t)p.q_tile_first * 128);
    ce = cudaMemset2DAsync(dq, (size_t)Nq * row_bytes, 0, r1 * row_bytes, (size_t)BH, st);
  }
  const int grid_q = pl.dq_grid;
  const int grid_kv = p.num_units_kv < s->sm_count ? p.num_units_kv : s->sm_count;
  if (ce == cudaSuccess)
    ce = timed(FA_KERNEL_BWD_PRE, st, [&] { return fa::launch_bwd_preprocess(d, o, dout, dvec, (int)rows, st); });
  if (!wide) {
    if (ce == cudaSuccess)
      ce = timed(FA_KERNEL_BWD, st, [&] {
        return pair ? fa::launch_bwd_dkdv_pair(tq64, tq, tk, tv, tdo64, tdo, p, s->sm_count, st)
                    : fa::launch_bwd_dkdv(d, tq, tk, tv, tdo, p, grid_kv, st);
      });
    if (ce == cudaSuccess)
      ce = timed(FA_KERNEL_BWD_DQ, st, [&] { return fa::launch_bwd_dq(d, tq, tk, tv, tdo, p, grid_q, st); });
  } else {
    // Head dim 256: dV pass, dK pass, then dQ.
    for (int pass = 0; pass < pl.kv_passes && ce == cudaSuccess; ++pass)
      ce = timed(FA_KERNEL_BWD, st,
                 [&] { return fa::launch_bwd256_kv(pass == 1, tq64, tk, tv, tdo64, p, grid_kv, st); });
    if (ce == cudaSuccess)
      ce = timed(FA_KERNEL_BWD_DQ, st, [&] { return fa::launch_bwd256_dq(tq, tk64, tv64, tdo, p, grid_q, st); });
  }
  cudaFreeAsync(ws, st);
  return ce == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
               void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d, int causal, float scale,
               void* stream) {
  return fa_bwd_general(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, N, d,
                        causal ? FA_CAUSAL_TOP_LEFT : FA_CAUSAL_NONE, scale, stream);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
           void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, void* stream) {
  return fa_bwd_gqa(q, k, v, o, lse, dout, dq, dk, dv, B, H, H, N, d, causal, scale, stream);
}

}  // extern "C"
