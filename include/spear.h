/*
 * spear.h -- C ABI of the GB300 (sm_103a) W4 + input-adaptive error-compensator
 * linear layer.
 *
 * The layer ("SPEAR: A System for Post-Quantization Error-Adaptive Recovery",
 * section 2.1A, Input-Adaptive Error Compensators, "Mechanism") applies to each
 * token x the effective weight
 *
 *     W_q + alpha * B * diag(gamma(A x)) * A,
 *
 * i.e. y = W_q x + alpha * B (gamma(z) (.) z) with z = A x. W_q is a 4-bit
 * weight with bf16 scales and integer zero points per group of 128 input
 * channels or per output channel (section 1 and section 3.1 use 4-bit weights,
 * per-channel being the hard case); A is rank x K, B is N x rank, gamma is the
 * elementwise sigmoid, the constant one (which gives the static low-rank
 * correction W_q + alpha B A that section 1 contrasts with), or the
 * bottleneck MLP that section 2.1A names for gamma. Phase-aware
 * dispatch (section 2.2A) is exposed as two entry points: a fused single-kernel
 * decode path for M <= 32 tokens and a tensor-core prefill path for larger M.
 *
 * Conventions for every call:
 *  - Device pointers are plain CUDA device addresses on the current device;
 *    host pointers are ordinary (preferably pinned) host memory. No call takes
 *    ownership of a caller's buffer.
 *  - bf16 tensors are row-major and contiguous; x, y and every weight buffer
 *    must be 16-byte aligned.
 *  - Argument errors are reported synchronously and leave nothing enqueued.
 *  - Forward calls only enqueue work on `stream` (no allocation, no
 *    synchronisation). Errors detected on the device (a bounded wait that
 *    timed out) are latched in the handle and reported by spear_linear_check.
 *  - A handle is not safe for concurrent forwards (its workspace is shared);
 *    distinct handles are independent.
 */
#ifndef SPEAR_H_
#define SPEAR_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct spear_linear_s* spear_linear_t;

typedef enum {
  SPEAR_OK = 0,
  SPEAR_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, M outside the entry point's range */
  SPEAR_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels implement (see create) */
  SPEAR_ERR_OOM = 3,           /* device allocation failed in create */
  SPEAR_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
  SPEAR_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up (reported by check) */
} spear_status_t;

typedef enum {
  SPEAR_GATE_SIGMOID = 0,      /* gamma(z) = 1 / (1 + exp(-z)), so gamma(z) * z = SiLU(z) */
  SPEAR_GATE_ONE = 1,          /* gamma = 1: static correction W_q + alpha B A */
  SPEAR_GATE_MLP = 2           /* bottleneck MLP ("SPEAR", section 2.1A, "Mechanism"), per token:
                                  gamma(z) = sigmoid(W2 relu(W1 z)), W1 (h x rank), W2 (rank x h);
                                  relu as the hidden activation is this library's reading */
} spear_gate_t;

typedef struct {
  int32_t K;                   /* input features; multiple of 128 */
  int32_t N;                   /* output features; multiple of 8 */
  int32_t group_size;          /* 128, or 0 for one group per output channel (G = K) */
  const uint8_t* qweight;      /* device, uint8 [N][K/2]: byte j of row n holds k = 2j in its
                                  low nibble and k = 2j + 1 in its high nibble, codes 0..15 */
  const void* scales;          /* device, bf16 [N][K/G] */
  const uint8_t* zeros;        /* device, uint8 [N][K/G], values 0..15; NULL means z = 8 */
  int32_t rank;                /* EC rank r: 0 (no compensator) or a multiple of 16, <= 256 */
  const void* A;               /* device, bf16 [rank][K] (ignored when rank == 0) */
  const void* B;               /* device, bf16 [N][rank] (ignored when rank == 0) */
  float alpha;                 /* compensator strength */
  spear_gate_t gate;
  int32_t max_tokens;          /* largest M any forward on this handle will use (>= 1) */
  /* SPEAR_GATE_MLP only (ignored otherwise; zero them for the other gates): */
  int32_t gate_hidden;         /* h, 1 <= h <= 64 */
  const void* gate_w1;         /* device, bf16 [h][rank], 16-byte aligned */
  const void* gate_w2;         /* device, bf16 [rank][h], 16-byte aligned */
} spear_linear_desc_t;

/* Build a handle from user-layout weights ("SPEAR", section 2.1A: the W_q of the
 * effective weight and the compensator's A, B, alpha, gamma).
 * Copies and re-lays-out every weight into handle-owned device memory on
 * `stream`, then synchronises `stream`, so the caller may free or reuse its
 * buffers as soon as this returns. On success *out holds the handle.
 * Errors: INVALID_ARG (null desc/out/pointers, K % 128, N % 8, bad group size,
 * rank not a multiple of 16 or > 256, max_tokens < 1; for SPEAR_GATE_MLP:
 * rank == 0, gate_hidden outside 1..64, null or unaligned gate weights),
 * UNSUPPORTED (shape outside the kernels' limits: N > 16 * 16 * SM count for
 * the decode path, or a decode grid that cannot be resident on the device all
 * at once, which its grid-wide compensator dependency needs), OOM, CUDA. On
 * error *out is left NULL and nothing is leaked.
 * Co-residency: the decode kernel runs at most one CTA per SM and its CTAs
 * wait for each other (bounded). Kernels of other streams or processes that
 * hold SMs while a decode call starts can delay some of its CTAs; if that
 * outlasts the wait limit, the call leaves the compensator out and latches
 * TIMEOUT, which spear_linear_check reports. */
spear_status_t spear_linear_create(const spear_linear_desc_t* desc, cudaStream_t stream,
                                   spear_linear_t* out);

/* Build ONE handle for several linears that read the same input x, such as
 * the q, k and v projections of an attention block or the gate and up
 * projections of an MLP (the paper has no counterpart; this is how serving
 * engines fuse such projections). Each member keeps its own weights, zero
 * points, compensator (A_i, B_i, alpha_i) and result:
 *   y[:, row_i : row_i + N_i] = W_i x + alpha_i B_i (gamma(A_i x) (.) A_i x),
 * row_i = N_0 + ... + N_{i-1}, so y is bf16 [M][N_0 + ... + N_{n-1}] and
 * every forward of the handle computes all members in one call (one launch
 * on the decode path: the stacked projection [A_0; ...; A_{n-1}] x and its
 * gate run once for all members, each output tile then applies its own
 * member's B_i and alpha_i).
 *   descs: n descriptors, 1 <= n <= 8 (n == 1 is spear_linear_create). All
 *   members must have the same K, group_size, rank and gate, N_i a multiple
 *   of 16, and n * rank <= 256; SPEAR_GATE_MLP is not supported here
 *   (UNSUPPORTED). max_tokens of the handle is the largest of the members'.
 * The members' buffers are copied (through temporary device buffers that
 * create frees before returning); errors as for spear_linear_create. */
spear_status_t spear_linear_create_grouped(const spear_linear_desc_t* descs, int32_t n, cudaStream_t stream,
                                           spear_linear_t* out);

/* Decode-phase forward ("SPEAR", section 2.2A: memory-bound, small M; the whole
 * layer, compensator included, runs as one kernel).
 *   x: device bf16 [M][K]; y: device bf16 [M][N] (must not overlap x).
 * 1 <= M <= min(32, max_tokens); M == 0 is a no-op returning OK.
 * y = bf16_RNE(W_q x + alpha B (gamma(Ax) (.) Ax)) with fp32 accumulation. */
spear_status_t spear_linear_forward_decode(spear_linear_t h, const void* x, void* y, int32_t M,
                                           cudaStream_t stream);

/* Prefill-phase forward ("SPEAR", section 2.2A: compute-bound, M > 1): the
 * main contraction runs on tcgen05 tensor cores with in-kernel INT4
 * dequantisation; the compensator's down-projection and gate run in a small
 * pre-kernel and its up-projection is folded into the same accumulator.
 *   x: device bf16 [M][K]; y: device bf16 [M][N]; 1 <= M <= max_tokens
 * (M == 0 is a no-op). Correct for every M; tuned for M >= 256. */
spear_status_t spear_linear_forward_prefill(spear_linear_t h, const void* x, void* y, int32_t M,
                                            cudaStream_t stream);

/* Prefill with the compensator on a concurrent stream ("SPEAR", section 2.2A:
 * in the prefill phase the compensator runs as a separate kernel overlapped
 * with the low-bit GEMM). The same y as spear_linear_forward_prefill, computed
 * as three launches: the compensator pre-kernel (u' = bf16(alpha gamma(Ax) (.)
 * Ax)) on ec_stream, forked from `stream` by an event; the main contraction
 * W x on `stream` into an fp32 buffer of the handle; after an event join, a
 * K-tail launch that adds alpha B u' to it and rounds to bf16 once. Both
 * streams are left joined (ec_stream's work precedes `stream`'s later work),
 * so the call can be captured into one CUDA graph. Requires
 * spear_linear_enable_concurrent_ec on handles with a compensator (a handle
 * without one takes the plain prefill path); ec_stream != stream.
 * Errors: INVALID_ARG, CUDA. */
spear_status_t spear_linear_forward_prefill_concurrent(spear_linear_t h, const void* x, void* y, int32_t M,
                                                       cudaStream_t stream, cudaStream_t ec_stream);

/* Allocates what spear_linear_forward_prefill_concurrent needs: an fp32
 * buffer of max_tokens x N and two events (once; later calls return OK). This
 * is the only allocation outside create. Errors: INVALID_ARG, OOM, CUDA. */
spear_status_t spear_linear_enable_concurrent_ec(spear_linear_t h);

/* Phase dispatch ("SPEAR", section 2.2A): decode path for M <= 32, prefill otherwise. */
spear_status_t spear_linear_forward(spear_linear_t h, const void* x, void* y, int32_t M,
                                    cudaStream_t stream);

/* End-to-end forward on HOST buffers: copies x_host (bf16 [M][K]) to a
 * handle-owned device buffer, runs spear_linear_forward, copies the result
 * into y_host (bf16 [M][N]) and synchronises `stream`. Pinned host memory gives
 * asynchronous copies. 1 <= M <= max_tokens. */
spear_status_t spear_linear_forward_host(spear_linear_t h, const void* x_host, void* y_host,
                                         int32_t M, cudaStream_t stream);

/* End-to-end forward of a batch of calls on HOST buffers with one
 * synchronisation: call i copies x_host[i] (bf16 [Ms[i]][K of hs[i]]) into
 * hs[i]'s staging buffer, runs spear_linear_forward on it and copies the
 * result into y_host[i] (bf16 [Ms[i]][N of hs[i]]); the call returns once
 * every result is in host memory. The forwards run in order on `stream`.
 * The copies run on two copy streams of hs[0], after the work already on
 * `stream`, and overlap the forwards: a call's input copy waits only for the
 * previous forward on the same handle (which has read its staging buffer),
 * its forward for that copy and for the previous result of the handle to be
 * copied out. A handle may appear several times. The copy streams and a
 * handle's four events are made on its first batch and destroyed with it.
 * Every argument is checked before anything is enqueued: INVALID_ARG for a
 * null array or handle, Ms[i] outside 0 .. max_tokens of hs[i], or null
 * buffers with Ms[i] > 0; CUDA if a stream or event cannot be made. Pinned
 * host memory gives asynchronous copies. */
spear_status_t spear_linear_forward_host_batch(const spear_linear_t* hs, const void* const* x_host,
                                               void* const* y_host, const int32_t* Ms, int32_t n,
                                               cudaStream_t stream);

/* Free every device allocation of the handle. cudaFree, which this calls,
 * waits for work already queued on the device, so forwards still in flight
 * finish first; the handle must not be used (or enqueued) afterwards. NULL is
 * accepted. */
spear_status_t spear_linear_destroy(spear_linear_t h);

/* Test surface: write the dequantised weight bf16_RNE((q - z) * s) as bf16
 * [N][K] (device) by unpacking the kernel-side layout of `path`
 * (0 = decode layout, 1 = prefill layout) with the kernels' own unpack code. */
spear_status_t spear_linear_dequantize(spear_linear_t h, int32_t path, void* w_out,
                                       cudaStream_t stream);

/* Synchronise `stream` and report the handle's device status word: OK, or
 * TIMEOUT if a bounded device-side wait gave up since the last check. A
 * TIMEOUT clears the status and resets the handle's workspace so it is usable
 * again. */
spear_status_t spear_linear_check(spear_linear_t h, cudaStream_t stream);

/* Test surface for the bounded waits: wait_ns sets the device-side wait limit
 * (0 restores the default of 100 ms); skip_arrive != 0 makes CTAs skip the
 * arrival another CTA waits for, so that the wait must run out:
 *  - decode: the "compensator projection done" arrival (the kernel then leaves
 *    the compensator out of y and latches TIMEOUT);
 *  - prefill, when the main kernel's stream-K schedule splits a tile over
 *    several CTAs (a handle sized for more than 32 tokens): the "partial tile
 *    stored" flag of the CTAs that run a tile's later K blocks (the tile's
 *    owner then gives up, writes nothing for its tile and latches TIMEOUT).
 * The prefill pre-kernel -> main kernel dependency is a stream (programmatic
 * launch) dependency that the hardware resolves; it has no arrival to skip. */
spear_status_t spear_linear_debug_set(spear_linear_t h, int64_t wait_ns, int32_t skip_arrive);

/* Test surface: the launch plan spear_linear_forward_decode uses for a handle
 * of this shape ("SPEAR", section 2.2A: the decode phase as one fused kernel),
 * computed by the same host code as the launch, with no device work.
 *   N, K: output and input width (as spear_linear_create accepts them);
 *   rank_b, n_members: each member's compensator rank and the member count
 *     (1 for spear_linear_create, 2..8 for a grouped handle with N split
 *     evenly); group_size: 128 or 0 (per output channel);
 *   gate_hidden: the MLP gate's hidden width (16, 32, 48 or 64), else 0;
 *   1 <= M <= 32; sm_count: SMs of the device.
 * info (13 int32 entries, caller-owned): grid, P (16-row tiles per CTA), NW
 * (consumer warps), T (tiles per warp), MT (8-token tiles), KW (warps along
 * K), KC (channels per stage), NS (stages), stage_bytes, smem (dynamic
 * shared memory), n_stages (stages over K), threads, bytes_x (x box bytes).
 * Errors: INVALID_ARG (bad shape or null info), UNSUPPORTED (as create or the
 * launch would report it). */
spear_status_t spear_decode_schedule(int32_t N, int32_t K, int32_t rank_b, int32_t n_members, int32_t group_size,
                                     int32_t gate_hidden, int32_t M, int32_t sm_count, int32_t* info);

/* Test surface: the launch plan spear_linear_forward_prefill uses for a layer
 * of this shape ("SPEAR", section 3.3: the compensator's projection fused
 * ahead of the weight contraction, its output GEMM as the K-tail), computed
 * by the same host code as the launch, with no device work and no GPU.
 *   N, K, rank: the layer (K a multiple of 64, 0 <= rank <= 256);
 *   gate_hidden: the hidden width of SPEAR_GATE_MLP (16, 32, 48 or 64), 0 for
 *     the elementwise gates; M >= 1 tokens;
 *   sm_count: SMs of the device the handle lives on;
 *   with_workspace: nonzero when the handle was created with max_tokens > 32
 *     (it then holds the stream-K partial-tile workspace).
 * info (14 int32 entries, caller-owned): mode (0: the projection runs in
 * the main kernel's prologue or rank = 0; 3: a split-K pre-kernel first),
 * G (main-kernel CTAs), TN (tokens per tile), kpt (units per tile), tail
 * (K-tail units per tile, ceil(rank / 64)), units (tiles x kpt), pro_items
 * (prologue items, one per 128 tokens; 0 in mode 3), pro_d (units each item
 * weighs in the split), NS (pipeline stages), stage_bytes, smem (dynamic
 * shared memory per CTA), pre_ctas (the pre-kernel's CTAs, mode 3),
 * tmem_a (first TMEM column of the dequantised-W slots), max_contrib (the
 * most partial tiles any owner adds).
 * starts (optional, caller-owned, starts_cap >= G + 1 entries): CTA c runs
 * units [starts[c], starts[c + 1]); starts[G] = units.
 * Errors: INVALID_ARG (bad shape, null info, starts_cap too small),
 * UNSUPPORTED (more than 2^31 units). */
spear_status_t spear_prefill_schedule(int32_t N, int32_t K, int32_t rank, int32_t gate_hidden, int32_t M,
                                      int32_t sm_count, int32_t with_workspace, int32_t* info, uint32_t* starts,
                                      int32_t starts_cap);

/* Decode forward that allocates nothing (the paper has no counterpart; this is
 * a deployment convenience). For callers that cannot call cudaMalloc at all,
 * for instance a process whose device memory is entirely reserved up front by
 * another allocator, or a serving loop in which a device allocation (which may
 * synchronise the device) is not allowed: such callers cannot create a handle,
 * so this call takes everything from the caller.
 *   desc: the same descriptor spear_linear_create takes (device pointers to
 *         the user-layout q, scales, zeros, A, B; max_tokens is ignored);
 *         qweight and A 16-byte aligned;
 *   x: device bf16 [M][K], 16-byte aligned; y: device bf16 [M][N];
 *   1 <= M <= 32 (0 is a no-op).
 * Result: y = bf16_RNE(W_q x + alpha B (gamma(Ax) (.) Ax)), fp32 accumulation,
 * as spear_linear_forward_decode computes (summation order differs).
 * SPEAR_GATE_MLP is not supported here (SPEAR_ERR_UNSUPPORTED).
 * Scratch: the compensator projection z lives in one static device array of
 * the library (32,768 bytes, held on every GPU that loads the library until
 * the process exits); it bounds rank <= 256 and M <= 32, and larger values
 * return SPEAR_ERR_INVALID_ARG. The first call on a device looks the array's
 * address up (cudaGetSymbolAddress, with that device current) and caches it;
 * make that first call before any stream capture. Each call enqueues two
 * kernels on `stream` (z = A x into the array, then the output rows), ordered
 * by the stream alone: no wait across blocks, no allocation, no
 * synchronisation. Every z entry a call reads was written by the same call,
 * so nothing needs clearing between calls. All calls share the array, so
 * calls that overlap on the GPU (different streams, or several host threads)
 * race with each other: serialise them. Slower than the handle-based decode
 * path (it reads the unpacked user layout on CUDA cores). */
spear_status_t spear_linear_forward_decode_noalloc(const spear_linear_desc_t* desc, const void* x, void* y,
                                                   int32_t M, cudaStream_t stream);

/* Round-to-nearest 4-bit quantiser (offline; the "RTN" backend of "SPEAR",
 * section 3.1, which the paper does not spell out: the usual asymmetric
 * min/max form). Per group of G input channels (G = 128, or K for
 * group_size 0) of each output row:
 *   lo = min(0, min w), hi = max(0, max w), range = max(hi - lo, 1e-8),
 *   s = bf16_RNE(range / 15), z = clamp(rint(-lo / s), 0, 15),
 *   q = clamp(rint(w / s) + z, 0, 15),
 * all in fp32 with IEEE division and round half to even.
 *   w: device fp32 [N][K], 16-byte aligned; outputs in the layout
 *   spear_linear_desc_t takes: qweight device uint8 [N][K/2] (2-byte
 *   aligned), scales device bf16 [N][K/G], zeros device uint8 [N][K/G].
 * K must be a multiple of 128. Enqueues one kernel on `stream`.
 * Errors: INVALID_ARG (null or misaligned pointers, bad shape or group size),
 * UNSUPPORTED (grid too large), CUDA. */
spear_status_t spear_quantize_rtn(const float* w, int32_t N, int32_t K, int32_t group_size, uint8_t* qweight,
                                  void* scales, uint8_t* zeros, cudaStream_t stream);

/* SLO-constrained, compensator-aware chunk scheduler ("SPEAR", section 2.2C:
 * a latency-aware scheduler driven by precomputed kernel-latency lookup tables
 * picks the largest prefill chunk that meets an inter-token-latency target,
 * adapting to the compensator density). Host only; no device work.
 * The table holds measured times of one whole serving step: ms[i * n_m + j]
 * for density densities[i] (share of layers with a compensator, strictly
 * ascending in [0, 1]) and tokens[j] tokens in the step (strictly ascending,
 * >= 1). Prediction is piecewise linear in the token count (extrapolated
 * linearly past the table's ends) and linear in the density between rows
 * (clamped to the first and last rows). */
typedef struct spear_sched_s* spear_sched_t;

/* Copies the table. Errors: INVALID_ARG (null pointers, empty or unsorted
 * axes, densities outside [0, 1], negative or NaN times), OOM. */
spear_status_t spear_sched_create(const double* densities, int32_t n_d, const int32_t* tokens, int32_t n_m,
                                  const double* ms, spear_sched_t* out);

/* Predicted step time (ms) for M tokens at the given density; -1 for a null
 * handle or M < 0. */
double spear_sched_predict(spear_sched_t s, int32_t M, double density);

/* *chunk_out = the largest candidate chunk c (candidates in any order, >= 0)
 * with predict(n_decode + c, density) <= itl_ms, or 0 if none fits. */
spear_status_t spear_sched_pick_chunk(spear_sched_t s, int32_t n_decode, double density, double itl_ms,
                                      const int32_t* candidates, int32_t n_c, int32_t* chunk_out);

/* Frees the scheduler; NULL is accepted. */
spear_status_t spear_sched_destroy(spear_sched_t s);

/* Human-readable name of a status code (static storage). */
const char* spear_status_string(spear_status_t s);

#ifdef __cplusplus
}
#endif
#endif /* SPEAR_H_ */
