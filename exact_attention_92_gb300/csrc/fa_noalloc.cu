// fa_bwd_noalloc: the backward pass with its workspace in a static device
// array instead of the workspace pool (see include/fa.h for who needs this).
//
// The array below is the only scratch this entry point uses.  Host code may
// not use its name as an address (that is a host-side stand-in): set-up, once
// per device with that device current, asks the runtime for its device
// address and the launches take that pointer.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa_common.h"

static __device__ __align__(256) unsigned char g_fa_bwd_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

namespace fa {
int internal_device_setup(unsigned int** status, int* sm_count);
int internal_validate(int B, int H, int N, int d, float scale);
int internal_encode_bhnd(CUtensorMap* m, const void* ptr, int BH, int N, int d, int box_rows);
unsigned long long internal_wait_timeout_ns();
cudaError_t internal_timed_launch(int kernel, cudaStream_t stream, cudaError_t (*launch)(void*), void* ctx);
cudaError_t launch_bwd_dkdv(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_dkdv_pair(const CUtensorMap& tq64, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo64, const CUtensorMap& tdo,
                                 const BwdParams& p, int sm_count, cudaStream_t stream);
cudaError_t launch_bwd_dq(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_preprocess(int d, const void* o, const void* dout, float* dvec, int rows,
                                  cudaStream_t stream);
}  // namespace fa

namespace {

constexpr int kMaxDevices = 64;

struct ScratchState {
  std::mutex mu;
  unsigned char* ptr = nullptr;  // device address of g_fa_bwd_scratch, once known
};
ScratchState g_scratch[kMaxDevices];

// Device address of the scratch array on the current device.  The lookup is
// kept once it has succeeded; a failed one is tried again by the next call.
int scratch_address(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  ScratchState& s = g_scratch[dev];
  std::lock_guard<std::mutex> g(s.mu);
  if (s.ptr == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_fa_bwd_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    s.ptr = static_cast<unsigned char*>(p);
  }
  *out = s.ptr;
  return FA_OK;
}

// The three launches of the backward pass, each through the library's
// launch counter and per-kernel timing.
struct Launch {
  int d;
  const void* o;
  const void* dout;
  float* dvec;
  int rows;
  const CUtensorMap *tq, *tk, *tv, *tdo, *tq64, *tdo64;
  const fa::BwdParams* p;
  int grid;
  int sm_count;
  cudaStream_t st;
};
cudaError_t run_pre(void* c) {
  const Launch& l = *static_cast<const Launch*>(c);
  return fa::launch_bwd_preprocess(l.d, l.o, l.dout, l.dvec, l.rows, l.st);
}
cudaError_t run_dkdv(void* c) {
  const Launch& l = *static_cast<const Launch*>(c);
  // Head dim 128: the CTA-pair kernel, as in fa_bwd_general.
  if (l.d == 128) return fa::launch_bwd_dkdv_pair(*l.tq64, *l.tq, *l.tk, *l.tv, *l.tdo64, *l.tdo, *l.p, l.sm_count, l.st);
  return fa::launch_bwd_dkdv(l.d, *l.tq, *l.tk, *l.tv, *l.tdo, *l.p, l.grid, l.st);
}
cudaError_t run_dq(void* c) {
  const Launch& l = *static_cast<const Launch*>(c);
  return fa::launch_bwd_dq(l.d, *l.tq, *l.tk, *l.tv, *l.tdo, *l.p, l.grid, l.st);
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                              int causal, float scale, void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  int e = fa::internal_validate(B, H, N, d, scale);
  if (e) return e;
  if (d == 256) return FA_ERR_UNSUPPORTED;  // runs the head-dim 64 / 96 / 128 kernels only
  const size_t rows = (size_t)B * H * N;
  const size_t need = rows * sizeof(float);
  if (need > (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_TOO_SMALL;
  unsigned int* status = nullptr;
  int sm_count = 0;
  e = fa::internal_device_setup(&status, &sm_count);
  if (e) return e;
  unsigned char* scratch = nullptr;
  e = scratch_address(&scratch);
  if (e) return e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = B * H;

  CUtensorMap tq, tk, tv, tdo, tq64, tdo64;
  if (fa::internal_encode_bhnd(&tq, q, BH, N, d, 128) || fa::internal_encode_bhnd(&tk, k, BH, N, d, 128) ||
      fa::internal_encode_bhnd(&tv, v, BH, N, d, 128) || fa::internal_encode_bhnd(&tdo, dout, BH, N, d, 128))
    return FA_ERR_CUDA;
  if (d == 128 && (fa::internal_encode_bhnd(&tq64, q, BH, N, d, 64) || fa::internal_encode_bhnd(&tdo64, dout, BH, N, d, 64)))
    return FA_ERR_CUDA;

  // Scratch layout: D [rows] fp32, every entry written by the preprocess
  // kernel.
  float* dvec = reinterpret_cast<float*>(scratch);

  fa::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.B = B;
  p.H = H;
  p.Hkv = H;
  p.Nq = N;
  p.Nk = N;
  p.causal = causal ? 1 : 0;
  p.causal_off = 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.lse = lse;
  p.dvec = dvec;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.store32 = ((reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) |
                reinterpret_cast<uintptr_t>(dv)) & 31u) == 0 ? 1 : 0;
  p.num_q_tiles = (N + 127) / 128;
  p.num_k_tiles = p.num_q_tiles;
  p.kv_tiles_used = p.num_k_tiles;
  p.q_tile_first = 0;
  p.num_units = BH * p.num_q_tiles;
  p.num_units_kv = p.num_units;
  p.group = 1;
  p.status = status;
  p.timeout_ns = fa::internal_wait_timeout_ns();

  const int grid = p.num_units < sm_count ? p.num_units : sm_count;
  Launch l{d, o, dout, dvec, (int)rows, &tq, &tk, &tv, &tdo, &tq64, &tdo64, &p, grid, sm_count, st};
  cudaError_t ce = fa::internal_timed_launch(FA_KERNEL_BWD_PRE, st, run_pre, &l);
  if (ce == cudaSuccess) ce = fa::internal_timed_launch(FA_KERNEL_BWD, st, run_dkdv, &l);
  if (ce == cudaSuccess) ce = fa::internal_timed_launch(FA_KERNEL_BWD_DQ, st, run_dq, &l);
  return ce == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
