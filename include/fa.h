/*
 * fa.h - C ABI of the GB300 (sm_103a) fused tiled attention library.
 *
 * Exact scaled-dot-product attention, forward and backward, computed tile by
 * tile on the GPU without ever writing an N x N matrix to HBM.
 *
 * Sources for what is computed:
 *  - "ELI5: FlashAttention" (A. Gordic), passages on kernel fusion, tiling of
 *    the N x N scores, the per-row statistics m (maximum) and l (sum of
 *    exponentials) and their exact merge, and recomputation in the backward.
 *  - "Potential algorithmic improvements for backward pass" (FlashAttention
 *    issue 1172): the operand list (Q, K, V, O, log-sum-exp, dO, dV, dK, dQ),
 *    the 5-GEMM backward with fp32 dQ accumulation, the atomic-free 7-GEMM
 *    backward (a dK/dV kernel plus a dQ kernel that walks like the forward),
 *    "implement both and pick what's faster", the 16-byte TMA alignment rule
 *    and the head-dimension specialisation.
 *
 * Definitions (per batch b and head h; rows i, j in [0, N)):
 *   s_ij  = scale * sum_c Q_ic K_jc,  j visible iff (!causal || j <= i)
 *   P_ij  = exp(s_ij - LSE_i),        LSE_i = ln sum_{visible j} exp(s_ij)
 *   O_i   = sum_j P_ij V_j
 *   D_i   = sum_c dO_ic O_ic
 *   dS_ij = P_ij (sum_c dO_ic V_jc - D_i)
 *   dV_j  = sum_i P_ij dO_i,  dQ_i = scale sum_j dS_ij K_j,  dK_j = scale sum_i dS_ij Q_i
 *
 * Layout: every matrix argument is a dense, C-contiguous device array of bf16
 * (raw 16-bit patterns) shaped [B, H, N, d]; LSE is fp32 [B, H, N] holding the
 * NATURAL log-sum-exp of the SCALED scores.  There are no stride arguments.
 *
 * Ownership: the caller allocates and owns every buffer (device memory).  The
 * library allocates nothing per call; it keeps one lazily created 8-byte
 * device error word per device for the bounded-wait watchdog.
 *
 * Synchronisation: calls only enqueue work on `stream` (a cudaStream_t; NULL
 * means the legacy default stream) and return at once.  A returned FA_OK means
 * the launches were accepted; device-side failures are reported by
 * fa_get_device_error.  Calls on distinct streams may run concurrently.
 *
 * Errors: arguments are validated before anything is launched; on any error
 * nothing is launched and no output is touched.
 */
#ifndef TILED_ATTENTION_TMEM_GB300_FA_H_
#define TILED_ATTENTION_TMEM_GB300_FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,    /* null pointer, negative size, non-finite or non-positive scale */
  FA_ERR_UNSUPPORTED = 2,    /* head dimension or variant not built for this library */
  FA_ERR_MISALIGNED = 3,     /* a pointer is not 16-byte aligned (TMA requirement) */
  FA_ERR_WORKSPACE = 4,      /* workspace NULL or smaller than fa_bwd_workspace_size */
  FA_ERR_LAUNCH = 5,         /* the CUDA runtime rejected a launch (see fa_last_cuda_error) */
  FA_ERR_DEVICE_TIMEOUT = 6  /* a bounded in-kernel wait expired; results are invalid */
} fa_status;

typedef enum {
  FA_BWD_AUTO = 0,   /* the variant measured fastest for this shape (see fa_bwd_choose) */
  FA_BWD_5GEMM = 5,  /* one kernel per K/V tile: dK, dV in TMEM, dQ reduced in fp32 */
  FA_BWD_7GEMM = 7   /* dK/dV kernel + dQ kernel walking like the forward; deterministic */
} fa_bwd_variant;

/*
 * Forward.  q, k, v: [B,H,N,d] bf16 (read).  o: [B,H,N,d] bf16 (written).
 * lse: [B,H,N] fp32 (written), natural log.  d must be 64, 96, 128, 192, 256 or
 * 384 (96 runs the 128 kernels on zero-padded tiles; 192 and 384 have their own;
 * at 384 the backward is the 7-GEMM form with lopsided tiles: dV and dK in three
 * column parts per key tile and 32 queries per step, dQ in two column parts).
 * scale: finite and > 0 (typically 1/sqrt(d)).  causal: 0 or 1 (key j is
 * visible to query i iff j <= i).  B*H*N == 0 is a no-op returning FA_OK.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * Split-KV forward: the same results as fa_fwd (up to fp32 rounding of the
 * merge), for shapes with too few query blocks (B*H*ceil(N/rows) below the SM
 * count) to fill the GPU.  Each query block's key tiles are cut into `splits`
 * contiguous parts of equal tile count; each part is a separate work item that
 * writes its normalised fp32 partial output O_s = (sum_j p_ij V_j) / l_s and its
 * log2-domain log-sum-exp L_s, and a second kernel merges the parts exactly:
 *   L = log2 sum_s 2^(L_s),  O = sum_s 2^(L_s - L) O_s,  LSE = L ln 2,
 * the block merge of the running (max, sum) statistics in "ELI5: FlashAttention"
 * (softmax statistics passage) applied to whole parts.  A part with no key
 * visible to a row has L_s = -inf and weight 0.
 * splits: 1..FA_FWD_MAX_SPLITS (1 is fa_fwd, with no workspace and one launch).
 * workspace: device memory of at least fa_fwd_splitkv_workspace_size bytes,
 * 256-byte aligned, owned by the caller and not shared with a concurrent call:
 *   fp32 parts [splits, B, H, N, d] at offset 0, then (256-byte aligned) fp32
 *   log2-domain LSEs [splits, B, H, N].
 * Errors as fa_fwd, plus FA_ERR_INVALID_ARG for splits out of range and
 * FA_ERR_WORKSPACE for a missing, misaligned or short workspace.
 */
#define FA_FWD_MAX_SPLITS 64
size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int splits);
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, float scale, int causal, int splits,
                         void* workspace, size_t workspace_bytes, void* stream);
/*
 * Parts per query block for fa_fwd_splitkv that the library's cost model
 * predicts fastest on the current device (1 = plain fa_fwd); 1 for invalid
 * shapes.  The model weighs the rounds of work items over the SMs against the
 * merge kernel's fp32 traffic.
 */
int fa_fwd_choose_splits(int B, int H, int N, int d, int causal);

/*
 * Bytes of device workspace fa_bwd needs for this shape and variant
 * (FA_BWD_AUTO: the largest over the variants).  0 for invalid shapes.
 *   log2-domain LSE per row:           4*B*H*Npad bytes
 *   D (fp32 row dot products dO.O):    4*B*H*Npad bytes
 *   5-GEMM only, fp32 dQ accumulator:  4*B*H*Npad*Dk bytes (Dk = 64 or 128: the
 *                                      kernel head dim, 128 for d = 96)
 *   query-range split of the dK/dV kernel (shapes with fewer than about two
 *   key tiles per SM; S = fa_bwd_query_parts for this shape and variant, the
 *   larger over both masks):
 *                                      2*4*S*B*H*Npad*Dk bytes of fp32 partial
 *                                      dK and dV (Dk: 64, 128, 256 or 384, the
 *                                      kernel head dim), summed by one extra
 *                                      kernel
 *   key-range split of the 7-GEMM dQ kernel (fewer than about two query tiles
 *   per SM; K = fa_bwd_key_parts for this shape and variant, the larger over
 *   both masks):
 *                                      4*K*B*H*Npad*Dk bytes of fp32 partial
 *                                      dQ, summed by one extra kernel
 *   work-item counters:                256 bytes
 * with Npad = N rounded up to a multiple of 128.  5-GEMM: d <= 128.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d, int variant);

/*
 * Backward.  Reads q, k, v, o, dO ([B,H,N,d] bf16) and lse ([B,H,N] fp32, as
 * written by fa_fwd for the same q, k, v, scale, causal); writes dq, dk, dv
 * ([B,H,N,d] bf16; dq and dk include `scale`).  workspace: device memory of at
 * least fa_bwd_workspace_size(B,H,N,d,variant) bytes, 256-byte aligned, owned
 * by the caller and not shared with a concurrent call.  variant: a
 * fa_bwd_variant value.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, float scale, int causal, int variant,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward that allocates nothing.  The pages have no counterpart to this: it
 * exists for callers that cannot allocate device memory (code inside an
 * allocator or memory-capped host, runtimes that only hand out input and
 * output buffers).  Same arguments and results as fa_bwd, minus the workspace:
 * the row statistics, the fp32 dQ accumulator and the in-kernel error word
 * live in one static device array of FA_NOALLOC_SCRATCH_BYTES (+256) bytes
 * that every GPU loading this library holds until the process exits.
 *   - Scratch needed: 8*B*H*Npad bytes (7-GEMM) or 8*B*H*Npad + 4*B*H*Npad*d
 *     (5-GEMM), Npad = N rounded up to 128.  FA_BWD_AUTO falls back to the
 *     7-GEMM form when only that fits; a shape whose chosen variant does not
 *     fit returns FA_ERR_WORKSPACE without launching anything.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - No cudaMalloc, cudaFree or allocating library routine is called.  Each
 *     call clears the parts that must start at zero (error word, dQ
 *     accumulator) itself.
 *   - All calls share the array: calls that overlap on the GPU (other streams,
 *     other host threads) race and must be serialised by the caller.
 *   - An expired in-kernel wait is recorded in the array's own error word
 *     (the later kernels of the call then skip their work, leaving dq, dk, dv
 *     unwritten).  fa_get_device_error does not see that word: read it with
 *     fa_bwd_noalloc_device_error after the call, before the next call clears it.
 *   - With AUTO, a shape whose 5-GEMM scratch exceeds the array runs the 7-GEMM
 *     form (for example B*H = 64, N = 2048, d = 128 needs 68 MB for 5-GEMM).
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, float scale, int causal, int variant,
                         void* stream);

/*
 * Status of the static array's error word used by fa_bwd_noalloc (the pages
 * have no counterpart: this belongs to the allocation-free entry point above).
 * Synchronises `stream`; returns FA_ERR_DEVICE_TIMEOUT (and clears the word) if a
 * bounded in-kernel wait of an fa_bwd_noalloc call on the current device gave
 * up, FA_ERR_LAUNCH if the CUDA runtime reports an error, else FA_OK.  `site`
 * (may be NULL) receives (kernel id << 8) | wait site.  Allocates nothing; the
 * same first-call and overlap rules as fa_bwd_noalloc apply.
 */
fa_status fa_bwd_noalloc_device_error(void* stream, int* site);

/*
 * Self-test of that error word: launches on `stream` one warp whose bounded
 * wait on a barrier nothing completes gives up after about two seconds and
 * records FA_ERR_DEVICE_TIMEOUT, site (6 << 8) | 1, in the static array's error
 * word (as an expired wait inside an fa_bwd_noalloc kernel would).  Touches no
 * caller memory and allocates nothing.  FA_OK if the launch succeeded.
 */
fa_status fa_bwd_noalloc_watchdog_selftest(void* stream);

/*
 * Query parts per key tile of the dK/dV kernel that fa_bwd uses for this shape
 * and variant (1: no split).  With fewer key tiles than about two per SM (few
 * heads) each key tile's query range is cut into parts that run as separate work
 * items writing fp32 partial dK and dV, added by one extra kernel; the count
 * follows a rule fitted to GB300 measurements of 1 to 8 parts.
 */
int fa_bwd_query_parts(int B, int H, int N, int d, int causal, int variant);

/*
 * Benchmark hook (no counterpart in the method): every later fa_bwd,
 * fa_bwd_workspace_size and fa_bwd_launches call in this process uses `parts`
 * query parts (1..FA_BWD_MAX_QUERY_PARTS; 0 restores the automatic choice).
 * Set it while no fa_bwd call is in flight on any host thread and size the
 * workspace after setting it.  FA_ERR_INVALID_ARG for other values.
 */
#define FA_BWD_MAX_QUERY_PARTS 16
int fa_bwd_force_query_parts(int parts);

/*
 * Key parts per query tile of the 7-GEMM dQ kernel that fa_bwd uses for this
 * shape and variant (1: no split; always 1 for the 5-GEMM form, which has no dQ
 * kernel).  With fewer query tiles than about two per SM (few heads) each query
 * tile's key range is cut into contiguous parts that run as separate work items
 * writing fp32 partial dQ, added in fixed order (and scaled) by one extra
 * kernel; the count follows the query split's rule over the dQ kernel's items.
 */
int fa_bwd_key_parts(int B, int H, int N, int d, int causal, int variant);

/*
 * Benchmark hook like fa_bwd_force_query_parts, for the dQ kernel's key parts
 * (1..FA_BWD_MAX_KEY_PARTS; 0 restores the automatic choice).  Same rules:
 * set it while no fa_bwd call is in flight, size the workspace after setting
 * it; FA_ERR_INVALID_ARG for other values.
 */
#define FA_BWD_MAX_KEY_PARTS 16
int fa_bwd_force_key_parts(int parts);

/* The concrete variant (5 or 7) FA_BWD_AUTO runs for this shape. */
int fa_bwd_choose(int B, int H, int N, int d, int causal);

/*
 * Synchronises `stream`, then returns FA_ERR_DEVICE_TIMEOUT (and clears the
 * device error word of the current device) if any kernel of this library on
 * this device gave up a bounded wait since the last call, FA_ERR_LAUNCH if the
 * CUDA runtime reports an error, else FA_OK.  `site` (may be NULL) receives
 * (kernel id << 8) | wait site of the first expired wait.
 */
fa_status fa_get_device_error(void* stream, int* site);

/*
 * Self-test of the in-kernel watchdog: launches one warp on `stream` that waits
 * on a barrier nothing completes.  After the watchdog limit (4e9 SM cycles,
 * about two seconds) the wait gives up and records FA_ERR_DEVICE_TIMEOUT with
 * site (6 << 8) | 1 in the device error word, which fa_get_device_error then
 * reports and clears; until then, this library's kernels on this device exit
 * without computing.  Touches no caller memory.  Returns FA_OK if the launch
 * succeeded, FA_ERR_LAUNCH otherwise.
 */
fa_status fa_watchdog_selftest(void* stream);

/* The last CUDA runtime error code seen by this library on this thread. */
int fa_last_cuda_error(void);

/* Static description of a status code. */
const char* fa_strerror(fa_status s);

/*
 * Kernel-level timing for benchmarks (no counterpart in the method itself).
 * Between fa_profile_start and fa_profile_stop the library records a pair of
 * CUDA events around every kernel it launches, on that kernel's stream.
 * fa_profile_stop synchronises on those events and fills, per kernel kind
 * (FA_KERNEL_*), the number of launches and their summed device time in
 * milliseconds.  Events are created by the library and reused; recording adds
 * no device work beyond the event markers.  Not thread-safe against
 * concurrent start/stop calls.
 */
enum {
  FA_KERNEL_FWD = 0,      /* fused forward */
  FA_KERNEL_BWD_PRE = 1,  /* D = rowsum(dO o O), log2-domain LSE, dQ accumulator zeroing */
  FA_KERNEL_BWD_KV5 = 2,  /* 5-GEMM main kernel (dK, dV, fp32 dQ reductions) */
  FA_KERNEL_BWD_CONV = 3, /* 5-GEMM dQ fp32 -> bf16 */
  FA_KERNEL_BWD_KV7 = 4,  /* 7-GEMM dK/dV kernel */
  FA_KERNEL_BWD_Q7 = 5,   /* 7-GEMM dQ kernel */
  FA_KERNEL_FWD_MERGE = 6, /* split-KV merge of the forward's parts */
  FA_KERNEL_BWD_KVSUM = 7, /* sum of the dK/dV kernel's query-range parts */
  FA_KERNEL_BWD_QSUM = 8,  /* sum of the dQ kernel's key-range parts */
  FA_KERNEL_KINDS = 9
};
typedef struct {
  int launches[FA_KERNEL_KINDS];
  double ms[FA_KERNEL_KINDS];
} fa_profile;
int fa_profile_start(void);
int fa_profile_stop(fa_profile* out);
const char* fa_kernel_name(int kind);

/*
 * Throughput probe of the exponential unit (for benchmarks; the pages price the
 * exponential by its issue rate per SM per clock, "Potential algorithmic
 * improvements for backward pass", and every exponential of these kernels is one
 * ex2.approx.ftz.f32).  Launches `blocks` CTAs of 256 threads on `stream`; each
 * thread evaluates that instruction `iters` times in each of 8 independent
 * chains and writes one float to sink[blocks * 256] (device memory owned by the
 * caller).  *count (may be NULL) receives the number of evaluations launched;
 * time the launch with events on the same stream.  FA_ERR_INVALID_ARG for a NULL
 * sink or non-positive sizes.
 */
fa_status fa_ex2_probe(float* sink, int blocks, int iters, long long* count, void* stream);

/* Number of kernels one fa_fwd / fa_fwd_splitkv / fa_bwd call launches for this shape. */
int fa_fwd_launches(int B, int H, int N, int d);
int fa_fwd_splitkv_launches(int B, int H, int N, int d, int splits);
int fa_bwd_launches(int B, int H, int N, int d, int variant, int causal);

#ifdef __cplusplus
}
#endif

#endif /* TILED_ATTENTION_TMEM_GB300_FA_H_ */
