/*
 * tsa.h -- C ABI of libtsa.so: truncated-Taylor, fixed-state causal attention
 * on one NVIDIA B300 (sm_103a).
 *
 * The method (source pages, cited by title and section):
 *   "Expanding Attention: A Taylor-Series Route to Linear-Time Transformers
 *    with a Fixed Number of Recurrent States" (wpnews.pro), arXiv 2610.20637v1
 *   abstract; "arXiv Introduces New Linear-Time Transformer Method via Taylor
 *   Series Expansion and Fixed-State Recurrence" (zicq.com), sections
 *   "Technical Mechanism Analysis" and "Engineering Trade-offs and
 *   Performance"; the Hacker News thread on the paper (item 46888355), the
 *   comments on the "+1" normaliser column and on (Q'K)V = Q'(KV).
 *
 * Per head, with T_n(x) = sum_{m<n} x^m/m! (the first n Taylor terms of exp):
 *     out_i = sum_{j<=i} T_n(q_i.k_j) v_j / sum_{j<=i} T_n(q_i.k_j)
 * computed through the symmetric tensor-power features
 *     phi(x) = [phi_0(x) | ... | phi_{n-1}(x)],  phi_m(x)_a = x^a / sqrt(a!)
 * (multi-indices |a| = m in non-decreasing index order, width C(d+m-1, m),
 * so <phi_m(q), phi_m(k)> = (q.k)^m / m!) and the fixed state
 *     S = sum_j phi(k_j) [v_j; 1]^T        (D rows, d_v + 1 columns)
 * whose last column z = sum_j phi(k_j) is the normaliser.
 *
 * Conventions for every call:
 *  - All pointers are DEVICE pointers on the current CUDA device, owned by the
 *    caller; the library never frees them. Calls are asynchronous on the given
 *    stream (a cudaStream_t passed as void*; NULL = legacy default stream).
 *  - A tsa_status reports argument validation and launch errors only; a fault
 *    inside a kernel surfaces at the caller's next synchronisation (or
 *    tsa_sync_status). Nothing is thrown across the ABI. tsa_last_error()
 *    gives a message for the calling thread's last non-OK status.
 *  - Preconditions the library does NOT enforce: q and k rows have unit L2 norm
 *    (the pages make query/key normalisation a prerequisite: it keeps
 *    |q.k| <= 1, where the truncated series is accurate and T_n > 0). A score
 *    temperature is applied by the caller scaling q.
 *  - Pointers must be 16-byte aligned.
 */
#ifndef TSA_H
#define TSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TSA_OK = 0,
  TSA_ERR_INVALID = 1,      /* bad pointer, size, alignment or flag          */
  TSA_ERR_UNSUPPORTED = 2,  /* valid but not built: (d_k, d_v, n_terms, chunk) */
  TSA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed           */
  TSA_ERR_TIMEOUT = 4,      /* a device-side bounded wait gave up             */
  TSA_ERR_DEVICE_CHECK = 5  /* a device-side check of the debug build failed  */
} tsa_status;

typedef enum { TSA_F32 = 0, TSA_BF16 = 1 } tsa_dtype;

typedef struct {
  int B;            /* batch                                                   */
  int H;            /* heads; B*H independent (b,h) heads                     */
  int d_k;          /* query/key width d: 16 or 32                            */
  int d_v;          /* value width: 32, 64 or 128                             */
  int n_terms;      /* n Taylor terms, orders 0..n-1: 1..4 (feature dim <= 1024), or
                       5 at d_k = 16 (4,845 features) with d_v 32 or 64, on the
                       CUDA-core path with each CTA's state slice in global
                       memory */
  tsa_dtype dtype;  /* element type of q, k, v and out (states are always fp32) */
  int chunk;        /* prefill chunk length; 0 = library's choice (see tsa_plan) */
} tsa_config;

/* tsa_prefill flag: continue from the states already in `states` instead of
 * starting from zero. Additivity of the states across chunks (abstract; the
 * "Technical Mechanism Analysis" item 2) makes this exact: prefill(A) then
 * prefill(B, ACCUMULATE) gives the outputs and states of prefill(A||B). */
#define TSA_PREFILL_ACCUMULATE 1u

/* D = sum_{m<n} C(d_k+m-1, m), the feature width ("the m-th state is
 * C(d+m-1, m) wide", abstract). Returns 0 for d_k < 1 or n_terms < 1. */
size_t tsa_feature_dim(int d_k, int n_terms);

/* D_pad = D rounded up to a multiple of 4: rows of the stored state. */
size_t tsa_state_pad_dim(int d_k, int n_terms);

/* Algorithmic state size per head, D * (d_v + 1) fp32 elements (9,945 for
 * d_k=16, d_v=64, n=3: the abstract's figure). 0 if cfg is NULL. */
size_t tsa_state_elems(const tsa_config* cfg);

/* Bytes of the whole `states` buffer: B*H*D_pad*(d_v+1)*4.
 * Layout, per head h = b*H + hh, a contiguous block of D_pad*(d_v+1) floats:
 *   S[a][c] at  h*D_pad*(d_v+1) + a*d_v + c      (a < D_pad, c < d_v)
 *   z[a]    at  h*D_pad*(d_v+1) + D_pad*d_v + a
 * Rows a >= D are padding and stay exactly 0. */
size_t tsa_state_bytes(const tsa_config* cfg);

/* Feature ordering: for row a < D of the state, idx[F*a .. F*a+F-1] are the
 * input indices whose product forms the monomial, F = max(3, n_terms - 1)
 * (-1 = no factor; an order-m row has m indices >= 0, non-decreasing) and
 * weight[a] = 1/sqrt(a!). Host only; idx holds F*D ints, weight D floats. */
tsa_status tsa_feature_index(int d_k, int n_terms, int* idx, float* weight);

/* The feature map phi(x) = [phi_0(x) | ... | phi_{n-1}(x)] of `rows` inputs, in
 * fp32, in the order of tsa_feature_index (so <phi_m(q), phi_m(k)> =
 * (q.k)^m / m!; the m-th block is C(d+m-1, m) wide, abstract). The kernels
 * build these features on chip and never store them; this call exports them,
 * e.g. to check the width of the state by the rank of stacked features.
 *  x   : [rows, d_k] fp32, device;  out : [rows, D] fp32, device (D =
 *        tsa_feature_dim). Asynchronous on the stream. */
tsa_status tsa_feature_map(int d_k, int n_terms, int64_t rows, const float* x, float* out,
                           void* cuda_stream);

/* How tsa_prefill splits the work (host only; num_sms <= 0 asks the current
 * device). The sequence of each head is cut into n_spans spans of
 * chunks_per_span chunks of `chunk` tokens; d_v into n_slices slices of at most
 * slice_width columns. With n_spans > 1 the call launches a span-state pass,
 * an exclusive scan over spans and the output pass (`launches` = 3), and takes
 * scratch_bytes of stream-ordered scratch from the library's pool.
 * path: TSA_PATH_SIMT (fp32 FFMA on the CUDA cores), TSA_PATH_TC (bf16
 * inputs on the tcgen05 tensor cores, fp32 TMEM accumulators) or
 * TSA_PATH_TC_F32 (fp32 inputs on the tensor cores: every operand split into
 * bf16 hi + lo parts and every product taken as three MMAs) or
 * TSA_PATH_SHORT (short segments, e.g. a few tokens appended with
 * TSA_PREFILL_ACCUMULATE: one CTA per head keeps the head's state in shared
 * memory for the whole segment, so the state is read and written once; fp32
 * on the CUDA cores in blocks of chunk = 16 tokens). The library takes
 * TSA_PATH_SHORT where the state fits (d_k = 16 with n <= 3, or d_k = 32 with
 * n <= 2) for N <= 16 with bf16 inputs whose shape the tensor-core append
 * form takes, for N <= 32 otherwise; cfg->chunk = 16 asks for it at any N.
 * ctas_per_sm: CTAs of the output pass resident per SM. On TSA_PATH_TC it is
 * 3 for the append form that bf16 segments of at most 64 tokens take where
 * d_v <= 64 and the state has at most two 128-feature blocks (a short append:
 * the state's bf16 copy in shared memory and its update accumulated apart in
 * 128 TMEM columns, at most 75 KB of shared memory per CTA), 1 otherwise. */
#define TSA_PATH_SIMT 0
#define TSA_PATH_TC 1
#define TSA_PATH_TC_F32 2
#define TSA_PATH_SHORT 3
typedef struct {
  int chunk;
  int slice_width;
  int n_slices;
  int n_spans;
  int chunks_per_span;
  int ctas_per_sm;
  int launches;
  size_t smem_bytes;
  size_t scratch_bytes;
  int path;
  int cluster;      /* CTAs that share one (head, span): 1, or 2 when the bf16
                       head state is too large for one SM's tensor memory and
                       its feature blocks are divided between a CTA pair */
} tsa_plan;

tsa_status tsa_prefill_plan(const tsa_config* cfg, int64_t N, int num_sms, tsa_plan* out);

/* Causal chunked prefill of N tokens for every head.
 *  q, k : [B, H, N, d_k]  dtype, contiguous      (input)
 *  v    : [B, H, N, d_v]  dtype, contiguous      (input)
 *  out  : [B, H, N, d_v]  dtype, contiguous      (output, fully written)
 *  states: tsa_state_bytes(cfg) bytes, fp32, layout above. Output: the state
 *         after the N tokens. With TSA_PREFILL_ACCUMULATE it is also an input
 *         (the state before them) and the outputs attend to it.
 * The library may take stream-ordered scratch from its own memory pool.
 * N = 0 is a no-op (TSA_OK; states untouched unless ACCUMULATE is clear, in
 * which case they are zeroed). Errors: NULL pointers, N < 0, N > 2^31 - 1
 * (token coordinates are 32-bit), misalignment -> TSA_ERR_INVALID;
 * unsupported shapes -> TSA_ERR_UNSUPPORTED. */
tsa_status tsa_prefill(const tsa_config* cfg, int64_t N, const void* q, const void* k,
                       const void* v, void* out, float* states, unsigned flags,
                       void* cuda_stream);

/* tsa_prefill_noalloc -- tsa_prefill for callers that cannot allocate.
 * (A deployment variant: the pages have no counterpart to this call.)
 * Same arguments, layouts, results and errors as tsa_prefill, but the call
 * allocates nothing: no cudaMalloc, cudaMallocAsync, cudaFree or pool. It is
 * for callers that cannot let a library allocate device memory -- a process
 * whose memory budget belongs to its own allocator, a serving loop that must
 * not allocate after start-up, or a GPU without the stream-ordered allocator.
 * Its scratch is one fixed 16 MiB array in device memory that every GPU
 * loading libtsa.so holds until the process exits. Its plan considers only
 * span counts whose span states fit that array: where tsa_prefill's plan
 * (tsa_prefill_plan) needs more scratch, this call splits each head into
 * fewer spans (one span needs none), so every shape tsa_prefill takes runs,
 * with the same results up to the rounding order of the span sums.
 *  - The first call on each device looks up the array's device address (once,
 *    with that device current); make that first call before any stream
 *    capture. The address is kept for the life of the process: after a
 *    cudaDeviceReset of that device it is stale, so do not call this entry
 *    point on a device that has been reset.
 *  - All calls on a device share the one array, and a call leaves its own
 *    contents there. Calls that can overlap on the GPU (different streams with
 *    no ordering between them) race on it: order them on one stream, or use
 *    tsa_prefill. Nothing in the array needs clearing between calls. */
tsa_status tsa_prefill_noalloc(const tsa_config* cfg, int64_t N, const void* q, const void* k,
                               const void* v, void* out, float* states, unsigned flags,
                               void* cuda_stream);

/* The state after N tokens without the outputs: S (+)= sum_j phi(k_j) [v_j; 1]^T
 * for every head (the state sum of a segment; states are additive across
 * segments, abstract: "the states are additive across chunks, so prefill
 * admits a parallel scan"). It is the first step of a prefill whose sequence
 * is split over several devices: each device sums its own segment, the
 * segment sums are exchanged, and each device then runs tsa_prefill on its
 * segment with TSA_PREFILL_ACCUMULATE from the sum of the segments before it.
 *  k : [B, H, N, d_k] dtype;  v : [B, H, N, d_v] dtype  (q is not needed)
 *  states: as for tsa_prefill. Without TSA_PREFILL_ACCUMULATE it receives the
 *          segment's sum; with it, the sum is added to what it holds.
 * Runs the span-state pass of the prefill path and the scan over spans (two
 * launches) with stream-ordered scratch from the library's pool. N = 0, errors
 * and alignment as for tsa_prefill. */
tsa_status tsa_prefill_states(const tsa_config* cfg, int64_t N, const void* k, const void* v,
                              float* states, unsigned flags, void* cuda_stream);

/* One decode token for every head, constant cost in the context length:
 *   S <- S + phi(k)[v; 1]^T;  out = (phi(q)^T S)[:d_v] / (phi(q)^T S)[d_v]
 *  q, k : [B, H, d_k] dtype;  v, out : [B, H, d_v] dtype;
 *  states: as for tsa_prefill, read and updated in place. */
tsa_status tsa_decode_step(const tsa_config* cfg, const void* q, const void* k,
                           const void* v, void* out, float* states, void* cuda_stream);

/* a <- a + b over whole state buffers (the states of consecutive segments add;
 * abstract, "states are additive across chunks"). a and b may not overlap
 * partially; a == b doubles the state. */
tsa_status tsa_state_merge(const tsa_config* cfg, float* a, const float* b,
                           void* cuda_stream);

/* Copy states into the canonical layout [B, H, D, d_v + 1] fp32 row-major
 * (column d_v = z), dropping the padding rows. dst: B*H*D*(d_v+1) floats. */
tsa_status tsa_state_to_canonical(const tsa_config* cfg, const float* states, float* dst,
                                  void* cuda_stream);

/* Synchronise the stream, then report TSA_ERR_CUDA for a pending fault or
 * TSA_ERR_TIMEOUT if a device-side wait gave up since the last check (the
 * tensor-core kernels bound every wait on their mbarriers at 1 s; a CTA whose
 * wait runs out records it here, stops, releases its tensor memory and exits,
 * leaving its outputs incomplete). The flag is per device and is cleared by
 * this call. In the debug build (below) a failed device-side check since the
 * last call is reported first, as TSA_ERR_DEVICE_CHECK. */
tsa_status tsa_sync_status(void* cuda_stream);

/* Testing hooks for the failure path of the bounded waits; not for use in
 * production. Both settings are process-wide and apply to calls made after
 * them.
 *  - tsa_debug_set_wait_limit: the bound, in nanoseconds, of every wait
 *    between the warp roles of the tensor-core kernels (default 1 s; 0
 *    restores the default).
 *  - tsa_debug_withhold_publication(1): the fp32 tensor-core output pass
 *    (TSA_PATH_TC_F32) never publishes the first chunk's completed output
 *    accumulator, so the waits for it run out: each CTA gives up, releases
 *    its tensor memory and exits with its outputs incomplete, and the next
 *    tsa_sync_status returns TSA_ERR_TIMEOUT.
 *    tsa_debug_withhold_publication(2): in the bf16 prefill whose head state
 *    a CTA pair shares (tsa_plan.cluster = 2), rank 0 of each pair never
 *    tells its peer that its first chunk's partial output rows have arrived
 *    in the peer's shared memory; the peer's wait runs out, the peer gives up
 *    and makes rank 0 give up too, both release their tensor memory and
 *    exit, and tsa_sync_status returns TSA_ERR_TIMEOUT.
 *    tsa_debug_withhold_publication(3): the bf16 append form (tsa_plan
 *    ctas_per_sm = 3) never publishes that its output accumulator is
 *    complete; the waits for it run out, each CTA gives up, releases its
 *    tensor memory and exits with its outputs and state incomplete, and
 *    tsa_sync_status returns TSA_ERR_TIMEOUT.
 *    0 turns it off; other values are TSA_ERR_INVALID. */
tsa_status tsa_debug_set_wait_limit(uint64_t ns);
tsa_status tsa_debug_withhold_publication(int what);

/* The debug build (libtsa_debug.so, compiled with -DTSA_DEBUG; same API and
 * kernels) checks on the device, before each access: that TMEM accesses and
 * MMA accumulators stay inside the 512 allocated columns and a warp's TMEM
 * loads and stores inside its own 32-lane quarter; that every MMA operand
 * read from shared memory lies inside the CTA's dynamic shared memory; that
 * tiled TMA copies start at an innermost coordinate that is a multiple of 8
 * elements and stores at no negative coordinate; that bulk copies have
 * 16-byte aligned addresses and sizes and end inside shared memory; and that
 * CTAs map to heads of the launch and state indices to elements of their
 * head's state. A failed check skips that access (a load returns zeros),
 * records what failed and two values (the first failure since the last
 * tsa_sync_status), and the kernel runs on or gives up at its next bounded
 * wait; nothing traps. tsa_sync_status then returns TSA_ERR_DEVICE_CHECK and
 * tsa_last_error names the check, its values, the block and the thread.
 *  - tsa_debug_build: 1 in the debug build, 0 in the release build.
 *  - tsa_debug_check_selftest: queues on the stream one kernel whose TMEM
 *    column check fails on purpose (columns 510..525 of 512; only the check
 *    runs, no TMEM is allocated or touched), so that the next tsa_sync_status
 *    returns TSA_ERR_DEVICE_CHECK. TSA_ERR_UNSUPPORTED in the release build. */
int tsa_debug_build(void);
tsa_status tsa_debug_check_selftest(void* cuda_stream);

const char* tsa_status_string(tsa_status s);
const char* tsa_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* TSA_H */
