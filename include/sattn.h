/*
 * sattn.h -- C ABI of libsattn.so: quantized exact attention with K smoothing
 * on GB300 (compute capability 10.3, sm_103a).
 *
 * What is computed (the "Experiment Log" page, vortex_exact_attention, entry
 * "Phase 0 Import And Verification": Q/K preparation, K smoothing, INT8
 * quantization, QK traversal, online softmax, FP8 V/P, two-level PV
 * accumulation, final conversion, ragged-tail contract; entry "Phase 1
 * State-Ownership Decision": strict tile order, exact FP8 score bytes,
 * per-tile RO rescaling, two-level PV accumulation, final conversion):
 *
 *   sattn_prepare   K smoothing (K minus its per-channel mean over the
 *                   sequence), INT8 codes of Q and smoothed K with one FP32
 *                   scale per 32-token block, FP8 E4M3 codes of V with one
 *                   FP32 scale per channel.
 *   sattn_forward   attention over the codes: exact integer QK^T, online
 *                   softmax over KV tiles in strictly increasing order, P
 *                   quantised to FP8 E4M3 (p * 448), inner per-tile FP32 PV
 *                   partial plus outer FP32 RO rescaled every tile, final
 *                   reciprocal of the denominator and BF16 output.
 *
 * Arithmetic, stated fully:
 *   mean[c]   FP32 sum over 64-token chunks in ascending token order, chunk
 *             sums added in ascending order, divided by Nkv (IEEE RN).
 *   ks        fl32(k - mean[c]).
 *   INT8      per block of 32 tokens x 128 channels: s = amax / 127,
 *             code = clamp(rint(x / s), -127, 127) (IEEE division, ties to
 *             even); amax = 0 gives s = 0 and codes 0.
 *   FP8 V     s_v[c] = amax_c / 448 over all Nkv tokens;
 *             code = E4M3(v / s_v[c]) round-to-nearest-even, saturating.
 *   score     s2 = float(acc) * ((s_q * s_k) * c0), acc = exact int32 dot
 *             product of the codes, c0 = sm_scale * log2(e) (FP32).
 *   softmax   per KV tile of 256 keys, ascending: m' = max(m, max s2),
 *             alpha = exp2(m - m') (0 while m = -inf),
 *             p8 = E4M3(fl(fl(exp2(fl(s2 - m'))) * 448)), every step rounded
 *             to FP32 in this order (s2 rounded before m' is subtracted) and
 *             exp2 correctly rounded, so each FP8 byte is fixed by the codes
 *             and scales alone;
 *             RO = RO * alpha + sum_j p8_j * v8_j,  d = d * alpha + sum_j p8_j.
 *   output    out[c] = bf16_rne((RO[c] * (1 / d)) * s_v[c]).
 *   mask      key j of query row i is kept when j < Nkv and, if causal,
 *             j <= i + (Nkv - Nq).
 *   GQA       query head h reads KV head h / (Hq / Hkv).
 *
 * Ownership and synchronisation: the caller allocates every buffer (device
 * memory unless stated otherwise) and owns the stream.  Calls only enqueue
 * work and return: on `stream` (a cudaStream_t; NULL is the legacy default
 * stream), and for sattn_prepare and sattn_attention_host also on helper
 * streams of the library that fork from `stream` and join back into it with
 * events, so the caller sees all of a call's work ordered on `stream`.  The
 * helper streams and events are created once per device and kept for the
 * life of the process.  The helper streams are shared by every caller on a
 * device, so two sattn_prepare calls enqueued on unrelated caller streams are
 * ordered behind each other's helper work (each call's Q and V branches wait
 * for the previous call's branches on the same device); callers that need
 * independent streams to stay independent should use sattn_prepare_noalloc or
 * the graph entry points, which keep the serial order on the caller's
 * stream.  Calls never allocate device memory, free or
 * synchronise, except sattn_check_status, which synchronises the stream by
 * design, and sattn_graph_create, which builds a CUDA graph (released by
 * sattn_graph_destroy).  All device pointers must be 16-byte aligned.
 * Buffers of one call must not overlap.
 *
 * Errors: every entry point returns an sattn_status; no exception crosses
 * the ABI.  Argument checks happen before anything is enqueued; a failing
 * call enqueues nothing (except SATTN_ERR_LAUNCH, see below).
 */
#ifndef SATTN_H
#define SATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SATTN_HEAD_DIM 128   /* the only supported head dimension */
#define SATTN_QBLOCK 32      /* tokens per INT8 quantisation block */
#define SATTN_KV_TILE 256    /* keys per KV tile of the forward pass; the tiling is
                                part of the result (P8 is relative to the running
                                max at each tile) */

typedef enum {
    SATTN_OK = 0,
    SATTN_ERR_INVALID = 1,     /* null pointer, D != 128, Hq % Hkv != 0, N < 1,
                                  causal with Nq > Nkv, sizes beyond limits */
    SATTN_ERR_MISALIGNED = 2,  /* a pointer is not 16-byte aligned */
    SATTN_ERR_DEVICE = 3,      /* current device is not compute capability 10.3,
                                  or a CUDA runtime query failed */
    SATTN_ERR_LAUNCH = 4,      /* a kernel launch failed (cudaGetLastError);
                                  earlier kernels of the call may have run */
    SATTN_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out; the
                                  outputs of that call are undefined */
    SATTN_ERR_SCRATCH_LIMIT = 6 /* the shape needs more scratch than the fixed
                                  array of sattn_prepare_noalloc holds */
} sattn_status;

/* Problem shape.  Q is [B][Hq][Nq][D], K and V are [B][Hkv][Nkv][D]. */
typedef struct {
    int32_t B, Hq, Hkv, Nq, Nkv, D;
    int32_t causal;      /* 0 or 1 */
    float sm_scale;      /* softmax scale; <= 0 selects 1 / sqrt(D) */
} sattn_shape;

/* Byte sizes of every buffer for a shape (all multiples of 16). */
typedef struct {
    size_t q, k, v;             /* BF16 inputs */
    size_t q_codes, q_scales;   /* int8 [B][Hq][Nq32][128], FP32 [B][Hq][Nq32/32] */
    size_t k_codes, k_scales;   /* int8 [B][Hkv][Nkv32][128], FP32 [B][Hkv][Nkv32/32] */
    size_t k_mean;              /* FP32 [B][Hkv][128] */
    size_t v_codes, v_scales;   /* E4M3 [B][Hkv][128][Nkv128] (channel-major), FP32 [B][Hkv][128] */
    size_t out;                 /* BF16 [B][Hq][Nq][128] */
    size_t prepare_workspace;   /* scratch of sattn_prepare */
    size_t forward_workspace;   /* scratch of sattn_forward: a 256-byte status block
                                   (status words, then the attention kernel's work-item
                                   counters), then the FP16 copy of the K codes that the
                                   tensor cores read (B * Hkv * Nkv * 256 bytes) */
    size_t arena;               /* one device block holding all of the above,
                                   for sattn_attention_host */
} sattn_sizes;
/* NX = N rounded up to a multiple of X. */

/*
 * sattn_query_sizes -- fill `sizes` for `shape`.  Pure host function.
 * Returns SATTN_OK or SATTN_ERR_INVALID.
 */
int sattn_query_sizes(const sattn_shape *shape, sattn_sizes *sizes);

/*
 * sattn_prepare -- Q/K preparation, K smoothing, INT8 quantisation of Q and
 * K, FP8 preparation of V (page entry "Phase 0 Import And Verification",
 * first three contract stages and "FP8 V").
 *   q, k, v     in:  BF16, [B][Hq][Nq][128] and [B][Hkv][Nkv][128], contiguous
 *   q_codes     out: int8, rows Nq .. Nq32-1 of each head are 0
 *   q_scales    out: FP32, one per 32-token block
 *   k_codes     out: int8 codes of the smoothed K, pad rows 0
 *   k_scales    out: FP32, one per 32-token block
 *   k_mean      out: FP32 per-channel mean of K that was subtracted
 *   v_codes     out: E4M3 bytes, channel-major [B][Hkv][128][Nkv128];
 *               keys Nkv .. Nkv128-1 are 0
 *   v_scales    out: FP32 per channel
 *   workspace   scratch, sizes.prepare_workspace bytes; contents on entry
 *               are ignored
 * Codes and scales are bit-exact functions of the inputs (the arithmetic is
 * fixed above, including the summation order of the mean).
 * Q's quantisation runs on a helper stream of the library (created once per
 * device) concurrently with the K/V kernels on `stream`, and V's beside K's
 * on a second one after the shared K/V statistics; `stream` waits for both
 * before the call's work ends, so everything is ordered on `stream` as the
 * caller sees it (and a CUDA graph capture of the call records the branches).
 */
int sattn_prepare(const sattn_shape *shape, const void *q, const void *k, const void *v,
                  int8_t *q_codes, float *q_scales, int8_t *k_codes, float *k_scales,
                  float *k_mean, uint8_t *v_codes, float *v_scales, void *workspace, void *stream);

/*
 * sattn_forward -- QK traversal, online softmax, FP8 P, two-level PV
 * accumulation, final conversion and ragged tails (page entries "Phase 0
 * Import And Verification" and "Phase 1 State-Ownership Decision").
 *   q_codes, q_scales, k_codes, k_scales, v_codes, v_scales
 *               in: as written by sattn_prepare for the same shape
 *   out         out: BF16 [B][Hq][Nq][128]
 *   workspace   scratch, sizes.forward_workspace bytes: the status block that
 *               sattn_check_status reads, then the FP16 copy of the K codes
 *               (every INT8 code as the same integer in FP16, exact) that the
 *               tensor cores read, since this part has no INT8 tensor-core
 *               product; contents on entry are ignored
 * Two kernels (after a memset of the status block): the K codes are copied to
 * FP16 into the workspace (bound by HBM bandwidth), then a persistent CTA per
 * SM takes the (query tile, head, batch) items, longest first within groups
 * of KV heads that fit in L2, from a counter in the status block as it frees
 * up.  Concurrent calls must use separate workspaces.
 * Exactness: QK^T is computed from the codes with products and sums that are
 * exact integers.  Every FP8 byte of P is the one the arithmetic above defines:
 * the kernel encodes fl(2^x) from the hardware approximation (relative error
 * below 2^-22) scaled by 448 * (1 + 2^-21) and by 448 * (1 - 2^-21); where the
 * two bytes agree they bracket the exact value and that is the byte, and where
 * they differ (about 1.5e-5 of the keys) the byte is recomputed with a
 * correctly rounded 2^x (float-float arithmetic).  alpha uses the hardware
 * approximation of 2^x; PV and the output follow the arithmetic above with
 * the inner PV sum in the tensor core's FP32 order.
 */
int sattn_forward(const sattn_shape *shape, const int8_t *q_codes, const float *q_scales,
                  const int8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                  const float *v_scales, void *out, void *workspace, void *stream);

/*
 * sattn_attention_small -- sattn_prepare followed by sattn_forward in one
 * kernel launch, for one query tile of one head: B = Hq = Hkv = 1, Nq <= 128,
 * Nkv <= 1024 (the small-shape latency path; same page entries as the two
 * calls).  The CTA first runs the preparation with the preparation kernels'
 * own per-thread steps, writing every buffer sattn_prepare writes with the
 * same bytes, then attends exactly as sattn_forward, so `out` equals the
 * two-call result byte for byte.
 *   q, k, v              in: BF16 [1][1][N][128]
 *   q_codes .. v_scales  out: as sattn_prepare (sizes from sattn_query_sizes)
 *   out                  out: BF16 [1][1][Nq][128]
 *   workspace            sizes.forward_workspace bytes, as for sattn_forward
 *                        (no preparation workspace is needed)
 * Returns SATTN_ERR_INVALID for other shapes; other errors as sattn_forward.
 */
int sattn_attention_small(const sattn_shape *shape, const void *q, const void *k, const void *v, int8_t *q_codes,
                          float *q_scales, int8_t *k_codes, float *k_scales, float *k_mean, uint8_t *v_codes,
                          float *v_scales, void *out, void *workspace, void *stream);

/*
 * sattn_prepare_kv -- the K and V part of sattn_prepare (K smoothing, INT8
 * K, FP8 V; same page entry), for sattn_forward_q_bf16, which quantises Q
 * itself.  Arguments as in sattn_prepare without q, q_codes and q_scales;
 * the outputs are byte for byte those of sattn_prepare.
 */
int sattn_prepare_kv(const sattn_shape *shape, const void *k, const void *v, int8_t *k_codes,
                     float *k_scales, float *k_mean, uint8_t *v_codes,
                     float *v_scales, void *workspace, void *stream);

/*
 * sattn_prepare_kv_onepass -- sattn_prepare_kv as one cooperative kernel
 * launch ("Experiment Log" page, "Closed Prior Work" table, row "P2 direct V
 * preparation": V prepared as soon as its per-channel amax is known).  The
 * chunk statistics, the per-head K mean and V scales, and the K and V
 * quantisers run as three phases of one persistent grid, separated by two
 * grid-wide barriers, so the quantisers' second read of K and V follows the
 * statistics' read while K and V are still in L2.  Arguments and outputs as
 * in sattn_prepare_kv, byte for byte.  The launch is cooperative: every CTA
 * is resident, and the barriers' waits are bounded (about one second); a
 * wait that runs out sets a status word in `workspace`, which
 * sattn_check_prepare_status reads (the outputs are then undefined).  Resets
 * its counter with a memset on `stream` first.  Measured slower than
 * sattn_prepare's split launches (c5 0.207 against 0.175 ms): the
 * cooperative grid takes every SM, so sattn_prepare's Q quantiser cannot run
 * beside it.
 */
int sattn_prepare_kv_onepass(const sattn_shape *shape, const void *k, const void *v, int8_t *k_codes,
                             float *k_scales, float *k_mean, uint8_t *v_codes, float *v_scales, void *workspace,
                             void *stream);

/*
 * sattn_check_prepare_status -- synchronise `stream` and read the status word
 * that sattn_prepare_kv_onepass left in `prepare_workspace` (sized for
 * `shape` by sattn_query_sizes).  Returns SATTN_OK, SATTN_ERR_TIMEOUT if a
 * grid barrier's bounded wait ran out, or SATTN_ERR_DEVICE.  Blocks the
 * calling host thread.
 */
int sattn_check_prepare_status(const sattn_shape *shape, const void *prepare_workspace, void *stream);

/*
 * sattn_test_prepare_kv_onepass_withhold -- test hook: sattn_prepare_kv_onepass
 * whose first grid barrier waits for one CTA more than the grid has, so the
 * bounded wait runs out (after about one second), the status word is set and
 * every CTA returns; the context stays usable.
 */
int sattn_test_prepare_kv_onepass_withhold(const sattn_shape *shape, const void *k, const void *v, int8_t *k_codes,
                                           float *k_scales, float *k_mean, uint8_t *v_codes, float *v_scales,
                                           void *workspace, void *stream);

/*
 * sattn_forward_q_bf16 -- sattn_forward with the Q stage of the preparation
 * (the INT8 block quantiser of sattn_prepare) moved into the kernel: each
 * work item's 128 x 128 BF16 Q tile is quantised in shared memory while the
 * previous item computes.  No Q codes or scales reach device memory.
 *   q           in: BF16 [B][Hq][Nq][128], contiguous, 16-byte aligned
 *   k_codes, k_scales, v_codes, v_scales
 *               in: as written by sattn_prepare_kv (or sattn_prepare)
 *   out, workspace
 *               as in sattn_forward
 * The codes and block scales are the ones sattn_prepare would write, so the
 * output equals, byte for byte, sattn_forward's on sattn_prepare's outputs.
 * Errors as sattn_forward.
 */
int sattn_forward_q_bf16(const sattn_shape *shape, const void *q, const int8_t *k_codes,
                         const float *k_scales, const uint8_t *v_codes, const float *v_scales,
                         void *out, void *workspace, void *stream);

/*
 * sattn_test_forward_withhold_v -- test hook for failure detection, not part
 * of the computation (the page has no counterpart).  Same arguments as
 * sattn_forward; the launch loads no V tile, so the MMA thread's wait for V
 * runs out after about one second, the other roles stop at their own bounded
 * waits, every CTA releases its tensor memory and the kernel ends.
 * sattn_check_status then returns SATTN_ERR_TIMEOUT; `out` is undefined.  The
 * CUDA context stays usable: a following sattn_forward computes normally.
 */
int sattn_test_forward_withhold_v(const sattn_shape *shape, const int8_t *q_codes, const float *q_scales,
                                  const int8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                                  const float *v_scales, void *out, void *workspace, void *stream);

/*
 * sattn_test_int8_quantiser -- test hook, not part of the computation: checks
 * the INT8 block quantiser that sattn_prepare and sattn_forward_q_bf16 use
 * (clamp(rint(x / s), -127, 127), s = amax / 127, computed without a
 * division) against the IEEE division, for every positive finite BF16 amax
 * whose bit pattern lies in [amax_lo, amax_hi) (1 <= amax_lo < amax_hi <=
 * 0x7f80) and every BF16 x with |x| <= amax.
 *   result   out: device array of three uint64: mismatching codes, values
 *            that took the division-free tie decision, and the last mismatch
 *            (amax bits << 16 | x bits); valid after the stream synchronises
 */
int sattn_test_int8_quantiser(uint32_t amax_lo, uint32_t amax_hi, unsigned long long *result, void *stream);

/*
 * sattn_test_p8_codes -- test hook, not part of the computation: the FP8 P
 * bytes that sattn_forward writes for n_groups groups of 32 keys, through the
 * forward kernel's own per-block function.  Group i has raw QK accumulators
 * acc[32i .. 32i + 31] (FP32 values; any finite value or -inf, not only the
 * integers the forward produces), block scale product sig[i] and running
 * maximum m[i] (finite).  Byte 32i + k of `out` is
 * E4M3(fl(fl(2^fl(fl(acc * sig) - m)) * 448)) with a correctly rounded 2^x
 * (the P step of the arithmetic above).  Device arrays; acc and out 16-byte
 * aligned; results valid after the stream synchronises.
 */
int sattn_test_p8_codes(int n_groups, const float *acc, const float *sig, const float *m, uint8_t *out,
                        void *stream);

/*
 * sattn_test_exp2 -- test hook, not part of the computation: the correctly
 * rounded FP32 2^x that sattn_forward uses for the rare FP8 P bytes its fast
 * path cannot decide, elementwise over n device floats (x <= 0.5; x <= -40
 * gives 0).  Results valid after the stream synchronises.
 */
int sattn_test_exp2(int n, const float *x, float *out, void *stream);

/*
 * sattn_measure_mma_rate -- measurement hook, not part of the computation:
 * the dense throughput of tcgen05.mma on the current device for the forward's
 * own instruction shapes (M = 128, N = n, a multiple of 16 in [16, 256]):
 * kind 0 = kind::f16 with both operands in shared memory (as QK^T on the FP16
 * carrier), kind 1 = kind::f8f6f4 E4M3 x E4M3 with A in tensor memory (as PV).
 * One CTA per SM issues iters x 4 back-to-back MMAs from one thread.
 *   flop_per_clk_sm  out (host): 2*M*N*K per instruction / SM clock cycles
 *   tflops           out (host): the same over all SMs / wall time (events)
 * Allocates and frees a few bytes of device memory and synchronises the
 * device (a measurement, not a stream operation).  Returns SATTN_OK,
 * SATTN_ERR_INVALID for bad arguments, SATTN_ERR_DEVICE, or SATTN_ERR_LAUNCH
 * if the launch failed or the completion wait ran out.
 */
int sattn_measure_mma_rate(int kind, int n, int iters, double *flop_per_clk_sm, double *tflops);

/*
 * sattn_profile_events -- measurement hook, not part of the computation: while
 * set, every sattn_forward / sattn_forward_q_bf16 call records `before` on its
 * stream just before the attention kernel is launched and `after` just after
 * it (the K carrier conversion that precedes it is outside the pair), so that
 * cudaEventElapsedTime(before, after) is that kernel's own duration.  Both are
 * cudaEvent_t handles owned by the caller (created, with timing, before the
 * call), or both NULL to stop.  Process-wide, not thread-safe: set it from the
 * thread that launches.  Returns SATTN_ERR_INVALID if exactly one is NULL.
 */
int sattn_profile_events(void *before, void *after);

/*
 * sattn_test_host_chunks -- test hook, not part of the computation: the
 * chunk plan sattn_attention_host uses for `shape` on a device with `n_sm`
 * SMs.  Pure host function.
 *   bounds   out: host array of at least 9 int64; chunk c covers the
 *            (batch, KV head) units bounds[c] .. bounds[c + 1] - 1, with units
 *            numbered b * Hkv + kv_head
 *   nchunks  out: the number of chunks (1 to 8)
 */
int sattn_test_host_chunks(const sattn_shape *shape, int n_sm, int64_t *bounds, int *nchunks);

/*
 * sattn_check_status -- synchronise `stream` and read the status word that
 * sattn_forward left in `forward_workspace`.  Returns SATTN_OK, or
 * SATTN_ERR_TIMEOUT if a bounded device wait ran out, or SATTN_ERR_DEVICE if
 * the synchronisation itself failed.  Blocks the calling host thread.
 */
int sattn_check_status(const void *forward_workspace, void *stream);

/*
 * sattn_attention_host -- the whole path from host buffers: copies q, k, v
 * from host memory to the device, runs the preparation and the forward pass,
 * and copies the BF16 output back to host memory.
 *   q_host, k_host, v_host   in:  BF16 host arrays (pinned memory lets the
 *                                 copies overlap the kernels)
 *   out_host                 out: BF16 host array, valid after `stream`
 *                                 has been synchronised
 *   arena                    device scratch of sizes.arena bytes (holds the
 *                            inputs, codes, scales, two preparation
 *                            workspaces, the status block, two FP16 copies
 *                            of the K codes and the output)
 * The (batch, KV head) units are independent problems, so large shapes are
 * cut into up to eight chunks of contiguous units, each with at least two
 * forward work items per SM, sized as a ramp (small first and last chunks,
 * whose copies and kernels nothing else overlaps) when the ends stay that
 * large, else equal.  The host-to-device copies run back to back on
 * one helper stream of the library, each chunk's preparation and forward on
 * `stream` or a second helper stream (alternating, so the end of one chunk's
 * forward overlaps the start of the next), and the copies back on a third.
 * Events hand each chunk from stage to stage.  The helper streams and events
 * are created once per device.  The helpers wait for `stream` at the start,
 * and `stream` waits for the last copy back, so all work is ordered on
 * `stream` as seen by the caller.  The output bytes equal
 * sattn_prepare + sattn_forward on the whole shape.  Every chunk's forward
 * reports into the arena's status block, cleared once per call.
 * Calls on one device serialise their enqueueing (not their execution).
 */
int sattn_attention_host(const sattn_shape *shape, const void *q_host, const void *k_host,
                         const void *v_host, void *out_host, void *arena, size_t arena_bytes,
                         void *stream);

/*
 * sattn_prepare_noalloc -- sattn_prepare without a workspace argument.  The
 * page has no counterpart to this entry point; it exists for callers that
 * cannot hand the library scratch memory: programs whose device memory is
 * owned by an allocator they do not expose, callers that may not call
 * cudaMalloc because it synchronises the whole device, and plain C callers
 * with no device allocator of their own.  The caller still provides every
 * input and output buffer, exactly as for sattn_prepare, and receives the
 * same codes and scales bit for bit.
 *
 * Scratch: a fixed array of SATTN_NOALLOC_SCRATCH_BYTES (8 MiB) in the
 * library's device memory, which every GPU that loads the library holds until
 * the process exits.  The shape must need at most that much:
 * B * Hkv * ceil(Nkv / 64) <= 8192 (for example B4 Hkv8 Nkv8192 needs 4096,
 * B1 Hkv16 Nkv32760 needs 8192); larger shapes return
 * SATTN_ERR_SCRATCH_LIMIT before anything is enqueued.  Nothing in the
 * array needs to start at zero: each call writes every scratch element it
 * reads.  The array keeps the last call's contents.
 *
 * Set-up: the first call on each device (with that device current) looks up
 * the array's device address once (cudaGetSymbolAddress) and caches it; make
 * that first call before any stream capture begins on that device.  The
 * cached address belongs to the device's context at that time: after a
 * cudaDeviceReset (or any teardown of the primary context) the entry point
 * must not be called again in the same process.
 *
 * Concurrency: all calls on one device share the one array, so calls whose
 * kernels may overlap on the GPU (different streams without ordering between
 * them) race on it; order them on one stream or with events.
 * The function never calls cudaMalloc, cudaFree or any allocating routine.
 */
#define SATTN_NOALLOC_SCRATCH_BYTES (8u << 20)
int sattn_prepare_noalloc(const sattn_shape *shape, const void *q, const void *k, const void *v,
                          int8_t *q_codes, float *q_scales, int8_t *k_codes, float *k_scales,
                          float *k_mean, uint8_t *v_codes, float *v_scales,
                          void *stream);

/*
 * sattn_graph_create / sattn_graph_launch / sattn_graph_destroy -- the
 * preparation and the forward pass on fixed buffers, recorded once as a CUDA
 * graph and replayed with one launch per step.  This is the small-shape
 * latency path: at the sizes where the seven launches of a step cost more on
 * the host than the kernels on the GPU, one graph launch replaces them.
 *   create   arguments as sattn_prepare followed by sattn_forward's out and
 *            workspace; the buffers are recorded by address and must stay
 *            allocated until the graph is destroyed.  Each launch reads
 *            whatever q, k, v hold when it runs, and writes every output
 *            sattn_prepare and sattn_forward write.  *graph receives an
 *            opaque handle (NULL on failure).  Capture runs on a private
 *            stream of the call; nothing is executed.
 *   launch   enqueues one replay on `stream`; sattn_check_status on the
 *            forward workspace reads its status after the stream synchronises
 *   destroy  releases the graph (after its last launch has completed)
 * The output of a launch equals sattn_prepare + sattn_forward, byte for byte.
 * Errors as those two calls; launch and destroy return SATTN_ERR_INVALID for a
 * NULL handle.
 */
typedef struct sattn_graph sattn_graph;
int sattn_graph_create(const sattn_shape *shape, const void *q, const void *k, const void *v,
                       int8_t *q_codes, float *q_scales, int8_t *k_codes, float *k_scales,
                       float *k_mean, uint8_t *v_codes, float *v_scales,
                       void *prepare_workspace, void *out, void *forward_workspace, sattn_graph **graph);
int sattn_graph_launch(sattn_graph *graph, void *stream);
int sattn_graph_destroy(sattn_graph *graph);

/* A static, human-readable name for a status code. */
const char *sattn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SATTN_H */
