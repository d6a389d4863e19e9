/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library (libfa.so).
 *
 * The library computes exact scaled-dot-product attention the way
 * FlashAttention-2 does ("FlashAttention-2: Faster Attention with Better
 * Parallelism and Work Partitioning", abstract; "FlashAttention V2 in depth",
 * sections 2, 5, 6 and 7): tile by tile with an online softmax, query tiles in
 * the outer (parallel) loop and key/value tiles in the inner loop, an
 * unnormalised accumulator divided once at the end, the row logsumexp kept
 * for the backward pass, fully masked causal tiles skipped, and the matching
 * dQ/dK/dV backward pass with a separate D preprocess.
 *
 * Conventions shared by every entry point:
 *  - Tensors live in device memory of the current CUDA device.  Q, K, V, O,
 *    dO, dQ, dK, dV are bf16, shape [B, H, N, d], contiguous row-major (d is
 *    the fastest index).  LSE is fp32, shape [B, H, N], natural logarithm.
 *  - Pointers must be non-null and 16-byte aligned.
 *  - d must be 64, 96, 128 or 256 (FA_ERR_UNSUPPORTED otherwise; see
 *    fa_bwd_noalloc for its own limit).  B, H, N >= 1.
 *    N need not be a multiple of the tile size.  Queries and keys have the
 *    same length N, except in fa_fwd_general / fa_bwd_general.
 *  - causal != 0 applies the mask of "FlashAttention V2 in depth" section 5.1:
 *    query row i sees key j iff j <= i (top-left aligned).
 *  - scale multiplies Q K^T before the softmax; pass 1/sqrt(d) for the usual
 *    attention.  It must be finite and positive.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; 0 = legacy default
 *    stream) and never synchronise it, except fa_poll_status.  The
 *    backward's kernels are launched with programmatic stream serialization
 *    (each may start while the kernel ahead of it in the stream finishes,
 *    and waits on the device for what it reads); work the caller queues
 *    after a call, if not itself launched with programmatic serialization,
 *    still starts only once all of the call's kernels are done.
 *  - The caller owns every buffer it passes; the library never frees or keeps
 *    them.  Temporary device workspace (the fp32 split-KV partials of the
 *    forward pass, the fp32 D vector of the backward pass) is taken from
 *    the library's own memory pool on the current device with
 *    cudaMallocFromPoolAsync on `stream` and returned with cudaFreeAsync on
 *    the same stream, so it is stream-ordered.  Unlike the device's default
 *    pool, which gives its memory back at every synchronisation, this pool
 *    keeps freed memory reserved for later calls (up to the most workspace
 *    in use at once), so a call made after a synchronisation does not map
 *    its workspace afresh; fa_trim_workspace gives the reserved memory back.
 *  - Return value: FA_OK, or an fa_status code.  Argument errors are detected
 *    on the host before anything is launched.  A workspace allocation that
 *    fails returns FA_ERR_NO_MEMORY before any launch (for tests of that
 *    path, the environment variable FA_TEST_FAIL_ALLOC set to anything but
 *    "0" makes every workspace allocation fail).  A device-side wait that gives
 *    up (see fa_set_wait_timeout_ns) is reported later by fa_poll_status.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_ABI_VERSION 5

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or scale      */
  FA_ERR_UNSUPPORTED = 2, /* head dim not supported, or not an sm_103 GPU   */
  FA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed     */
  FA_ERR_NO_MEMORY = 4,   /* workspace allocation failed                     */
  FA_ERR_TIMEOUT = 5,     /* a device-side wait gave up (fa_poll_status)     */
  FA_ERR_SCRATCH_TOO_SMALL = 6 /* fa_bwd_noalloc: problem exceeds its scratch */
} fa_status;

/*
 * Forward pass.  "FlashAttention V2 in depth", section 6.1 (full forward
 * algorithm) with the causal block skip of section 5.3.
 *   q, k, v : in,  bf16 [B,H,N,d]
 *   o       : out, bf16 [B,H,N,d], O = softmax(scale * Q K^T [+ mask]) V
 *   lse     : out, fp32 [B,H,N],  L_i = m_i + log(l_i) = log sum_j exp(S_ij)
 * Long sequences with few (batch, head) pairs are split along the keys
 * automatically (sequence parallelism, FlashAttention-2 abstract point (2));
 * see fa_fwd_ex.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           int causal, float scale, void* stream);

/*
 * Forward pass with an explicit number of key splits.
 *   num_splits : 0 = automatic, 1 = no split, S > 1 = split the key range of
 *                every query tile into S parts whose partial results (fp32 O
 *                and LSE per part, in workspace) are merged by a second
 *                kernel: L = log sum_s exp(L_s), O = sum_s exp(L_s - L) O_s.
 *                S is clamped to the number of key tiles (128 keys; 64
 *                at d = 256), and lowered so that no split is empty.
 * Other arguments as fa_fwd.
 */
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
              int causal, float scale, int num_splits, void* stream);

/*
 * Forward pass with grouped-query attention (GQA; MQA when Hkv = 1): the H
 * query heads of a batch share Hkv key/value heads, query head h reading
 * key/value head h / (H / Hkv).  The pages list this variant as not
 * evaluated; it is the same computation per query head with K and V taken
 * from that head's key/value head.
 *   q, o    : bf16 [B,H,N,d];  k, v : bf16 [B,Hkv,N,d];  lse : fp32 [B,H,N]
 *   Hkv     : >= 1 and divides H (FA_ERR_INVALID_ARG otherwise)
 * Other arguments as fa_fwd_ex; Hkv = H is fa_fwd_ex.
 */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N,
               int d, int causal, float scale, int num_splits, void* stream);

/*
 * Causal codes of fa_fwd_general / fa_bwd_general.  The pages define the
 * mask for queries and keys of one length N (query row i sees keys j <= i);
 * with Nq query rows and Nk key rows the alignment has to be chosen:
 *   FA_CAUSAL_TOP_LEFT     row i sees keys j <= i
 *   FA_CAUSAL_BOTTOM_RIGHT row i sees keys j <= i + Nk - Nq (the last query
 *                          row sees every key: the newest Nq positions of a
 *                          sequence of Nk, as when decoding)
 * Both equal the pages' mask when Nq = Nk.  A query row that sees no key
 * (bottom-right with Nq > Nk: rows i < Nq - Nk) gets O = 0, L = -inf, and
 * zero gradients; keys no row sees get dK = dV = 0.
 */
#define FA_CAUSAL_NONE 0
#define FA_CAUSAL_TOP_LEFT 1
#define FA_CAUSAL_BOTTOM_RIGHT 2

/*
 * Forward pass with queries and keys of different lengths (and grouped-query
 * attention).  The computation of fa_fwd ("FlashAttention V2 in depth",
 * section 6.1) per query row over the keys it sees; short query blocks over
 * long keys (decoding) are split along the keys as in fa_fwd_ex
 * (FlashAttention-2 abstract, point (2)).  With num_splits = 0 and at most
 * 128 query rows per (batch, key/value head) after grouping, the two query
 * tiles of a CTA may take the even and the odd key tiles of one split; their
 * fp32 partial results then go through the workspace and the merge as for
 * a split.
 *   q, o    : bf16 [B,H,Nq,d];  k, v : bf16 [B,Hkv,Nk,d];  lse : fp32 [B,H,Nq]
 *   Nq, Nk  : >= 1
 *   Hkv     : >= 1 and divides H (FA_ERR_INVALID_ARG otherwise)
 *   causal  : FA_CAUSAL_NONE, FA_CAUSAL_TOP_LEFT or FA_CAUSAL_BOTTOM_RIGHT
 *             (FA_ERR_INVALID_ARG otherwise)
 * Other arguments as fa_fwd_ex.  fa_fwd_gqa is this call with Nq = Nk.
 */
int fa_fwd_general(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                   int Nq, int Nk, int d, int causal, float scale, int num_splits, void* stream);

/*
 * Backward pass.  "FlashAttention V2 in depth", section 7: P recomputed from
 * the saved logsumexp (section 7.1), D_i = rowsum(dO_i * O_i) from a separate
 * preprocess kernel (section 7.3), dK and dV with key/value tiles in the
 * outer loop (section 7.2; a work unit per key tile, at d = 128 a CTA pair
 * per two key tiles; no atomics), and dQ from a second kernel with query
 * tiles in the outer loop (a work unit per query tile, no atomics) instead
 * of the page's fp32 atomic accumulation across key tiles.  Units are dealt
 * to persistent CTAs, at most one per SM.
 *   q, k, v : in,  bf16 [B,H,N,d] (the forward inputs)
 *   o       : in,  bf16 [B,H,N,d] (the forward output)
 *   lse     : in,  fp32 [B,H,N]   (the forward logsumexp)
 *   dout    : in,  bf16 [B,H,N,d] (gradient of the loss w.r.t. O)
 *   dq,dk,dv: out, bf16 [B,H,N,d]
 * Workspace: D, B*H*N*4 bytes from the library's pool on `stream`.  The results
 * are bitwise reproducible from run to run.  At d = 256 the dK and dV
 * accumulators of a key tile do not fit in tensor memory together, so the
 * key/value kernel runs twice (a dV pass and a dK pass, recomputing S^T).
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
           void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, void* stream);

/*
 * Backward pass with grouped-query attention (see fa_fwd_gqa): dK and dV of
 * a key/value head are the sums over the query heads that read it.  A dK/dV
 * CTA owns one key/value tile of one key/value head and walks the visible
 * query tiles of all of those query heads, so the sums stay in tensor memory
 * (no atomics; results bitwise reproducible from run to run).
 *   q, o, dout, dq : bf16 [B,H,N,d];  k, v, dk, dv : bf16 [B,Hkv,N,d]
 *   lse            : fp32 [B,H,N]
 *   Hkv            : >= 1 and divides H (FA_ERR_INVALID_ARG otherwise)
 * Workspace and other arguments as fa_bwd; Hkv = H is fa_bwd.
 */
int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
               void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d, int causal, float scale,
               void* stream);

/*
 * Backward pass with queries and keys of different lengths (see
 * fa_fwd_general for the causal codes), and grouped-query attention.
 *   q, o, dout, dq : bf16 [B,H,Nq,d];  k, v, dk, dv : bf16 [B,Hkv,Nk,d]
 *   lse            : fp32 [B,H,Nq] (from fa_fwd_general with the same causal code)
 * Gradient rows of query tiles that see no key, and of key tiles that no
 * query row sees, are zeroed with cudaMemset2DAsync on `stream`.  Workspace
 * and other arguments as fa_bwd; fa_bwd_gqa is this call with Nq = Nk.
 */
int fa_bwd_general(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq, int Nk, int d,
                   int causal, float scale, void* stream);

/*
 * Launch plans: how fa_fwd_general and fa_bwd_general carry out a call of
 * the given sizes, worked out on the host alone.  No device is touched, so a
 * caller can learn the workspace a call takes, and a test can check the
 * decisions, without a GPU.  The two calls follow exactly this plan, with
 * sm_count and l2_bytes those of the current device.
 *   sizes    : as fa_fwd_general / fa_bwd_general (num_splits for the forward)
 *   sm_count : the device's SM count (>= 1);  l2_bytes : its L2 size in bytes
 *   plan     : out, written on FA_OK only
 * Returns FA_OK; the status the call would return for these sizes (its
 * pointer checks aside); or FA_ERR_INVALID_ARG for a null plan or
 * sm_count < 1.  Both the forward call and its plan refuse, with
 * FA_ERR_INVALID_ARG, a forced split count that would make more than
 * 2^31 - 1 work units (query blocks times splits over all heads).
 */
typedef struct {
  int packed_heads;         /* 1: the H/Hkv query heads of a key/value head
                               share query tiles (H/Hkv > 1 and Nq < 128)  */
  int unit_heads;           /* (batch, head) pairs listed: B*H, or B*Hkv when packed */
  int unit_rows;            /* query rows of each: Nq, or (H/Hkv)*Nq when packed */
  int query_block;          /* query rows per unit: 256 (two 128-row tiles); 128 at d = 256 */
  int key_tile;             /* keys per step: 128; 64 at d = 256 */
  int key_tiles;            /* ceil(Nk / key_tile) */
  int num_splits;           /* key splits S >= 1, none of them empty */
  int key_tiles_per_split;  /* ceil(key_tiles / S) */
  int dual;                 /* 1: both query tiles of a unit hold its rows, one
                               taking the even, the other the odd key tiles of
                               its split (decoding; automatic splits only) */
  int partials;             /* fp32 partial results (O and L) merged by the
                               combine kernel: S, or 2 S when dual; 0 = none */
  int num_units;            /* unit_heads * ceil(unit_rows / query_block) * S */
  int grid;                 /* CTAs of the forward kernel: min(num_units, sm_count) */
  int head_window;          /* 0, or the heads per window when units are listed
                               window by window so that the K, V in flight
                               stay in L2 (no causal mask, S = 1, and the K, V
                               of all heads above half of l2_bytes) */
  int launches;             /* library kernels launched: 1, or 2 with the merge */
  uint64_t workspace_bytes; /* workspace taken: partials * B*H*Nq * (d + 1) * 4 */
} fa_fwd_plan_t;

int fa_fwd_plan(int B, int H, int Hkv, int Nq, int Nk, int d, int causal, int num_splits, int sm_count,
                uint64_t l2_bytes, fa_fwd_plan_t* plan);

typedef struct {
  int q_tiles;                /* ceil(Nq / 128) */
  int k_tiles;                /* ceil(Nk / 128) */
  int q_tile_first;           /* first query tile with a row that sees a key
                                 (> 0 only bottom-right with Nq > Nk) */
  int kv_tiles_used;          /* key tiles that some query row sees */
  int dq_units;               /* units of the dQ kernel: B*H*(q_tiles - q_tile_first) */
  int dq_grid;                /* its CTAs: min(dq_units, sm_count) */
  int kv_units;               /* units of the dK/dV kernel: B*Hkv*kv_tiles_used,
                                 at d = 128 B*Hkv*ceil(kv_tiles_used / 2) CTA pairs */
  int kv_cta_pair;            /* 1 at d = 128: the dK/dV kernel runs on CTA pairs */
  int kv_passes;              /* dK/dV launches: 2 at d = 256 (dV, then dK), else 1 */
  int launches;               /* library kernels launched: D preprocess, kv_passes, dQ */
  uint64_t zeroed_dq_bytes;   /* dQ bytes of the query tiles before q_tile_first,
                                 zeroed with cudaMemset2DAsync */
  uint64_t zeroed_dkdv_bytes; /* dK plus dV bytes of the key rows past
                                 kv_tiles_used * 128, zeroed likewise */
  uint64_t workspace_bytes;   /* workspace taken (D): B*H*Nq*4 */
} fa_bwd_plan_t;

int fa_bwd_plan(int B, int H, int Hkv, int Nq, int Nk, int d, int causal, int sm_count, fa_bwd_plan_t* plan);

/*
 * Backward pass that allocates no device memory.  The paper has no
 * counterpart: this is a library convenience.
 *
 * fa_bwd takes its fp32 workspace (D, B*H*N*4 bytes) from a memory pool
 * on every call.  Some callers cannot allow that: a caller that has handed
 * nearly all device memory to its own pool up front (weights, KV caches,
 * activations) and cannot have a library take memory in the middle of a
 * step, or one whose memory budget is fixed when it starts.  fa_bwd_noalloc
 * runs the same three kernels as fa_bwd, with the workspace in one static
 * device array of FA_BWD_NOALLOC_SCRATCH_BYTES (64 MiB).  The array belongs
 * to the library's module: it is reserved on every device where that module
 * is loaded (at the first use of the library on the device with lazy module
 * loading, the CUDA default; when the context is created with
 * CUDA_MODULE_LOADING=EAGER), and it stays reserved until the process exits.
 *
 *  - Arguments, layouts and ownership as fa_bwd; the caller still passes
 *    (and owns) every input and output.
 *  - Returns FA_ERR_SCRATCH_TOO_SMALL, before any device work, when
 *    B*H*N*4 exceeds FA_BWD_NOALLOC_SCRATCH_BYTES, and FA_ERR_UNSUPPORTED
 *    for d = 256 (it runs the kernels of head dims 64, 96 and 128).
 *  - The first call on a device sets up that device (with it current): it
 *    looks up the array's device address, and the library's status word,
 *    and keeps them (it also creates the library's workspace pool, which
 *    stays empty unless other entry points use it).  Make that first call before any stream capture; a
 *    set-up that fails is not kept, and the next call tries again.
 *  - It calls no cudaMalloc/cudaMallocAsync/cudaMallocFromPoolAsync/cudaFree
 *    and no allocating routine of any other library.
 *  - All calls on a device share the one array, and it keeps the last
 *    call's contents; each call writes all of the part it reads (D) before
 *    reading it.  Two calls whose kernels overlap on the GPU
 *    (different streams, or different host threads) race on the array and
 *    give wrong gradients: serialise them.
 *  - Its launches are counted by fa_launch_count and timed by
 *    fa_timing_enable / fa_timing_read like those of fa_bwd.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (64u << 20)
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                   float scale, void* stream);

/*
 * Synchronise `stream`, then return and clear the device status word of the
 * current device: FA_OK, FA_ERR_TIMEOUT if a kernel's bounded wait gave up
 * since the last poll, or FA_ERR_CUDA if the synchronisation failed.
 */
int fa_poll_status(void* stream);

/*
 * Time limit of every device-side wait (mbarrier waits between the load,
 * MMA and softmax roles).  A wait that exceeds it records FA_ERR_TIMEOUT,
 * and the kernel unwinds: it stops issuing work, waits (bounded) for its
 * own copies and MMAs in flight, frees its tensor memory and returns.
 * Default 2 s.  Returns the previous value.  Applies to later launches.
 */
uint64_t fa_set_wait_timeout_ns(uint64_t ns);

/*
 * Self-test of the give-up path: launches one CTA that waits on an mbarrier
 * nothing ever arrives on, with a time limit of `timeout_ns`.  The kernel
 * records FA_ERR_TIMEOUT and returns; fa_poll_status then reports it.
 */
int fa_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

/*
 * Per-kernel timing for benchmarks.  While enabled, every launch of a library
 * kernel is bracketed by two CUDA events recorded on the launch's stream.
 * Kernel ids: FA_KERNEL_FWD (forward main kernel), FA_KERNEL_COMBINE
 * (split-KV merge), FA_KERNEL_BWD_PRE (D preprocess), FA_KERNEL_BWD
 * (backward dK/dV kernel; at head dim 128 the CTA-pair kernel),
 * FA_KERNEL_BWD_DQ (backward dQ kernel).
 *   fa_timing_enable(on) : 1 starts recording (and drops old records), 0 stops.
 *   fa_timing_read(kernel, launches, total_ms) : waits for the recorded
 *       events of that kernel, returns how many launches were recorded and
 *       their summed device time in milliseconds, and forgets them.
 * Both return FA_OK, FA_ERR_INVALID_ARG (bad id / null out-pointer) or
 * FA_ERR_CUDA.
 */
#define FA_KERNEL_FWD 0
#define FA_KERNEL_COMBINE 1
#define FA_KERNEL_BWD_PRE 2
#define FA_KERNEL_BWD 3
#define FA_KERNEL_BWD_DQ 4
int fa_timing_enable(int on);
int fa_timing_read(int kernel, int* launches, double* total_ms);

/*
 * Launch counter (always on, no events): `*count` receives how many times
 * the kernel with id `kernel` (FA_KERNEL_*) has been launched by this
 * library since it was loaded.  Returns FA_OK or FA_ERR_INVALID_ARG (bad id
 * or null `count`).
 */
int fa_launch_count(int kernel, uint64_t* count);

/*
 * Give back to the device the memory that the library's workspace pool on
 * the current device keeps reserved and no call is using (cudaMemPoolTrimTo
 * to zero).  Workspace of calls still in flight is not touched; later calls
 * take memory from the device again.  Returns FA_OK, FA_ERR_UNSUPPORTED (not
 * an sm_103 device) or FA_ERR_CUDA.
 */
int fa_trim_workspace(void);

/* Human-readable name of an fa_status code (static storage). */
const char* fa_strerror(int status);

/* FA_ABI_VERSION of the loaded library. */
int fa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
