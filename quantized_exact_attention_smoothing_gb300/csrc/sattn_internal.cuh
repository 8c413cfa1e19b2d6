// sattn_internal.cuh -- shared declarations of the libsattn kernels and launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace sattn {

constexpr int kHeadDim = 128;
constexpr int kQBlock = 32;      // tokens per INT8 quantisation block
constexpr int kMeanChunk = 64;   // tokens per K-mean partial sum
constexpr int kVPad = 128;       // V codes are padded to a multiple of 128 keys
constexpr int kKvTile = 256;     // keys per KV tile of the forward pass (part of the contract)
constexpr int kQTile = 128;      // query rows per CTA of the forward pass

inline int64_t pad_up(int64_t n, int64_t m) { return (n + m - 1) / m * m; }

// Geometry shared by the host code of prepare and forward.
struct Geometry {
    int B, Hq, Hkv, Nq, Nkv, causal;
    float sm_scale;
    int64_t nq32, nk32, nk128;     // padded token counts
    int64_t nbq, nbk;              // INT8 blocks per head
    int64_t nchunks;               // K-mean chunks per KV head
};

// ---- prepare (prepare.cu) ----
// Workspace: [B*Hkv][nchunks][128] FP32 K column sums, then the same for V max |v|.
size_t prepare_workspace_bytes(const Geometry &g);
// The K/V part of launch_prepare with V's quantisation on v_stream: after the
// K/V statistics `fork` is recorded on `stream` and waited by v_stream; `join`
// is recorded on v_stream after V's kernel and waited by `stream` at the end.
cudaError_t launch_prepare_kv_split(const Geometry &g, const void *k, const void *v, int8_t *k_codes,
                                    float *k_scales, float *k_mean, uint8_t *v_codes, float *v_scales,
                                    void *workspace, cudaStream_t stream, cudaStream_t v_stream,
                                    cudaEvent_t fork, cudaEvent_t join);
// The K/V part of launch_prepare as one cooperative launch (statistics,
// finalize, K and V quantisers, separated by grid barriers whose bounded
// waits report through the status word at prepare_status_offset; withhold:
// test hook, the first barrier waits for CTAs that do not exist).
cudaError_t launch_prepare_kv_fused(const Geometry &g, const void *k, const void *v, int8_t *k_codes,
                                    float *k_scales, float *k_mean, uint8_t *v_codes, float *v_scales,
                                    void *workspace, cudaStream_t stream, bool withhold = false);
// Byte offset of the one-pass preparation's status word in the prepare workspace.
size_t prepare_status_offset(const Geometry &g);
// The Q part of launch_prepare alone (INT8 codes and block scales of Q).
cudaError_t launch_prepare_q(const Geometry &g, const void *q, int8_t *q_codes, float *q_scales,
                             cudaStream_t stream);
// Test hook: the INT8 quantiser against IEEE division over BF16 blocks whose
// amax has BF16 bits in [amax_lo, amax_hi) (device result[3], see prepare.cu).
cudaError_t launch_int8_quantiser_sweep(uint32_t amax_lo, uint32_t amax_hi, unsigned long long *result,
                                        cudaStream_t stream);
// q = nullptr skips the Q part (q_codes, q_scales unused).
cudaError_t launch_prepare(const Geometry &g, const void *q, const void *k, const void *v,
                           int8_t *q_codes, float *q_scales, int8_t *k_codes, float *k_scales,
                           float *k_mean, uint8_t *v_codes, float *v_scales, void *workspace,
                           cudaStream_t stream);

// ---- forward (attn_fwd.cu) ----
// Workspace: the 256-byte status block, then the FP16 carrier of the K codes
// ([B][Hkv][Nkv][128], the tensor-core operand of QK^T, written by the forward
// pass itself from the INT8 codes).
constexpr size_t kStatusBytes = 256;
size_t carrier_bytes(const Geometry &g);
size_t forward_workspace_bytes(const Geometry &g);
// Returns 0 on success, 1 if a tensor map could not be encoded, or a CUDA error.
// `status` is the status block, `carrier` the carrier's scratch (both inside
// the forward workspace for the public entry points).
// withhold_v (test hook): no V tile is loaded, so the launch ends through its
// bounded waits and reports a timeout in the status block.  With reset_status false
// the status block is not cleared first (several launches report into one).
// Status block: words 0-1 the status (flag, site of a wait that gave up),
// words 2-3 the item counters of launches in flight at the same time (the
// launch's ticket_slot, 0 or 1, picks one; it is zeroed before each launch).
int launch_forward(const Geometry &g, const int8_t *q_codes, const float *q_scales,
                   const int8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                   const float *v_scales, void *out, void *status, void *carrier, cudaStream_t stream,
                   bool withhold_v = false, bool reset_status = true, int ticket_slot = 0);

// One-time host setup of the forward kernels (tensor-map encoder, register
// check, shared-memory limit), so that launches captured into a CUDA graph
// make no such calls.  Returns 0, 1 without an encoder, or a CUDA error.
int forward_init();

// The forward pass with Q quantised inside the kernel: q is the BF16 Q
// [B, Hq, Nq, 128]; the codes and block scales are those launch_prepare
// writes, and the output is launch_forward's on them, byte for byte.
int launch_forward_q_bf16(const Geometry &g, const void *q, const int8_t *k_codes, const float *k_scales,
                          const uint8_t *v_codes, const float *v_scales, void *out, void *status,
                          void *carrier, cudaStream_t stream);

}  // namespace sattn

namespace sattn {
// Test hooks of the forward's P step (attn_fwd.cu): the FP8 P bytes of groups
// of 32 keys sharing a block scale product and a running maximum, through the
// kernel's own per-block function; and its correctly rounded exp2.
cudaError_t launch_test_p8_codes(int n_groups, const float *acc, const float *sig, const float *m, uint8_t *out,
                                 cudaStream_t stream);
// The preparation's buffers, for the single-launch small-shape path: the
// forward kernel writes them from the BF16 inputs before it attends.
struct SmallPrep {
    const void *q, *k, *v;   // BF16 inputs [1][1][N][128]
    int8_t *q_codes;
    float *q_scales;
    int8_t *k_codes;
    float *k_scales, *k_mean;
    uint8_t *v_codes;
    float *v_scales;
};
// Largest Nkv of the small-shape path (its K-mean chunk sums stay in shared memory).
constexpr int kSmallMaxNkv = 1024;
// prepare + forward in one launch for B = Hq = Hkv = 1, Nq <= 128, Nkv <= kSmallMaxNkv;
// status and carrier as for launch_forward.
int launch_small(const Geometry &g, const SmallPrep &sp, void *out, void *status, void *carrier,
                 cudaStream_t stream);

// tcgen05.mma throughput (mma_rate.cu): kind 0 = kind::f16 with A and B in
// shared memory, kind 1 = kind::f8f6f4 (E4M3) with A in tensor memory; M = 128,
// N = n.  Synchronises the device.  0 on success.
int measure_mma_rate(int kind, int n, int iters, double *flop_per_clk_sm, double *tflops);

// Events recorded around every attention kernel launch (both null: none).
void set_profile_events(cudaEvent_t before, cudaEvent_t after);

cudaError_t launch_test_exp2_rn(int n, const float *x, float *out, cudaStream_t stream);
}  // namespace sattn
