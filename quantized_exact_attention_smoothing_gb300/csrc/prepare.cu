// prepare.cu -- Q/K preparation, K smoothing, INT8 quantisation of Q and K,
// FP8 E4M3 preparation of V ("Experiment Log" page, entry "Phase 0 Import And
// Verification": the first contract stages and "FP8 V").
//
// Four streaming passes, all bound by HBM bandwidth:
//   kv_chunk_stats  per (KV head, 64-token chunk): FP32 column sums of K in
//                   ascending token order, and column max |V|
//   kv_finalize     per KV head: chunk sums added in ascending chunk order,
//                   mean = sum / Nkv; s_v = amax / 448
//   quant_int8      per 32-token block: (K - mean) or Q, amax, s = amax / 127,
//                   codes = clamp(rint(x / s), -127, 127)
//   quant_v         per 128-token tile: E4M3(v / s_v) written channel-major
// Every FP32 operation that decides a code is an IEEE operation in a fixed
// order, so codes and scales are bit-exact functions of the inputs.
#include <cuda_bf16.h>

#include "prep_device.cuh"

namespace sattn {
namespace {


// Block: 16 chunks x 16 channel groups of 8 channels.  Each thread walks its
// chunk's tokens in ascending order, one FP32 add per token and channel.
__global__ void __launch_bounds__(256) kv_chunk_stats_kernel(const uint4 *__restrict__ k,
                                                             const uint4 *__restrict__ v, int Nkv,
                                                             int nchunks, float *__restrict__ ksum,
                                                             float *__restrict__ vmax)
{
    const int bh = blockIdx.y;
    const int g = threadIdx.x & 15;
    const int chunk = blockIdx.x * 16 + (threadIdx.x >> 4);
    if (chunk >= nchunks)
        return;
    float s[8], mx[8];
    prep::chunk_stats8(k, v, Nkv, bh, chunk, g, s, mx);
    const size_t o = (static_cast<size_t>(bh) * nchunks + chunk) * kHeadDim + g * 8;
    reinterpret_cast<float4 *>(ksum + o)[0] = make_float4(s[0], s[1], s[2], s[3]);
    reinterpret_cast<float4 *>(ksum + o)[1] = make_float4(s[4], s[5], s[6], s[7]);
    reinterpret_cast<float4 *>(vmax + o)[0] = make_float4(mx[0], mx[1], mx[2], mx[3]);
    reinterpret_cast<float4 *>(vmax + o)[1] = make_float4(mx[4], mx[5], mx[6], mx[7]);
}

// One thread per (KV head, channel): chunk sums in ascending chunk order.
__global__ void __launch_bounds__(128) kv_finalize_kernel(const float *__restrict__ ksum,
                                                          const float *__restrict__ vmax, int Nkv,
                                                          int nchunks, float *__restrict__ k_mean,
                                                          float *__restrict__ v_scales)
{
    const int bh = blockIdx.x, c = threadIdx.x;
    const float *ks = ksum + static_cast<size_t>(bh) * nchunks * kHeadDim + c;
    const float *vm = vmax + static_cast<size_t>(bh) * nchunks * kHeadDim + c;
    float total = 0.0f, amax = 0.0f;
    int ch = 0;
    for (; ch + 64 <= nchunks; ch += 64) {   // 128 loads in flight, then the ordered sum
        float a[64], b[64];
#pragma unroll
        for (int u = 0; u < 64; ++u) {
            a[u] = ks[static_cast<size_t>(ch + u) * kHeadDim];
            b[u] = vm[static_cast<size_t>(ch + u) * kHeadDim];
        }
#pragma unroll
        for (int u = 0; u < 64; ++u) {
            total = __fadd_rn(total, a[u]);
            amax = fmaxf(amax, b[u]);
        }
    }
    for (; ch < nchunks; ++ch) {
        total = __fadd_rn(total, ks[static_cast<size_t>(ch) * kHeadDim]);
        amax = fmaxf(amax, vm[static_cast<size_t>(ch) * kHeadDim]);
    }
    k_mean[bh * kHeadDim + c] = __fdiv_rn(total, static_cast<float>(Nkv));
    v_scales[bh * kHeadDim + c] = __fdiv_rn(amax, 448.0f);
}

// One CTA per 32-token block of one head; thread = (token, eighth of the
// channels: 16 values), so a thread holds few registers and many CTAs stay
// resident to keep loads in flight.  With kSmooth (K), the per-channel mean
// is subtracted first.
template <bool kSmooth>
__global__ void __launch_bounds__(256) quant_int8_kernel(const uint4 *__restrict__ x, int N,
                                                         int64_t npad, int nblk,
                                                         const float *__restrict__ mean,
                                                         int8_t *__restrict__ codes,
                                                         float *__restrict__ scales)
{
    __shared__ float warp_max[8];
    prep::quant_block<kSmooth>(x, N, npad, nblk, mean, codes, scales, blockIdx.y, blockIdx.x, threadIdx.x,
                               warp_max, [] { __syncthreads(); });
}

// One CTA per 128-token tile of one KV head (prep::quant_v_tile).
__global__ void __launch_bounds__(256) quant_v_kernel(const uint4 *__restrict__ v, int Nkv,
                                                      int64_t nk128,
                                                      const float *__restrict__ v_scales,
                                                      uint8_t *__restrict__ vcodes)
{
    __shared__ __align__(16) uint32_t tile[kVPad * 32];   // [token][32 words]
    __shared__ float sv[kHeadDim], rv[kHeadDim];
    const int bh = blockIdx.y;
    if (threadIdx.x < kHeadDim) {
        const float x = v_scales[bh * kHeadDim + threadIdx.x];
        sv[threadIdx.x] = x;
        rv[threadIdx.x] = x > 0.0f ? __frcp_rn(x) : 0.0f;
    }
    __syncthreads();
    prep::quant_v_tile(v, Nkv, nk128, sv, rv, vcodes, bh, blockIdx.x * kVPad, threadIdx.x, tile,
                       [] { __syncthreads(); });
}

// Test kernel: every BF16 x with |x| <= amax against the INT8 quantiser of
// one block whose amax has BF16 bits blockIdx.x + amax_lo.  result[0] counts
// codes that differ from clamp(rint(fl(x / s))) by IEEE division, result[1]
// the values that took the tie decision, result[2] the last mismatch seen
// (amax bits << 16 | x bits).
__global__ void __launch_bounds__(256) int8_quantiser_sweep_kernel(uint32_t amax_lo, unsigned long long *result)
{
    const uint32_t a = amax_lo + blockIdx.x;
    const float amax = __uint_as_float(a << 16);
    const float s = __fdiv_rn(amax, 127.0f);
    const float rs = __frcp_rn(s);
    unsigned long long bad = 0, near = 0;
    for (uint32_t xb = threadIdx.x; xb < 0x10000u; xb += blockDim.x) {
        if ((xb & 0x7fffu) > a)
            continue;
        const float x = __uint_as_float(xb << 16);
        const float q = __fmul_rn(x, rs);
        near += isfinite(q) && !(fabsf(__fsub_rn(q, __fsub_rn(__fadd_rn(q, kRoundMagic), kRoundMagic))) < kTieMargin);
        if (int8_code(x, s, rs) != int8_code_div(x, s)) {
            ++bad;
            result[2] = (static_cast<unsigned long long>(a) << 16) | xb;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        bad += __shfl_xor_sync(0xffffffffu, bad, o);
        near += __shfl_xor_sync(0xffffffffu, near, o);
    }
    if ((threadIdx.x & 31) == 0) {
        if (bad)
            atomicAdd(result, bad);
        if (near)
            atomicAdd(result + 1, near);
    }
}

}  // namespace

size_t prepare_workspace_bytes(const Geometry &g)
{
    return 2 * static_cast<size_t>(g.B) * g.Hkv * g.nchunks * kHeadDim * sizeof(float);
}

cudaError_t launch_prepare(const Geometry &g, const void *q, const void *k, const void *v,
                           int8_t *q_codes, float *q_scales, int8_t *k_codes, float *k_scales,
                           float *k_mean, uint8_t *v_codes, float *v_scales, void *workspace,
                           cudaStream_t stream)
{
    const int bhk = g.B * g.Hkv, bhq = g.B * g.Hq;
    float *ksum = static_cast<float *>(workspace);
    float *vmax = ksum + static_cast<size_t>(bhk) * g.nchunks * kHeadDim;
    const uint4 *q4 = static_cast<const uint4 *>(q);
    const uint4 *k4 = static_cast<const uint4 *>(k);
    const uint4 *v4 = static_cast<const uint4 *>(v);

    kv_chunk_stats_kernel<<<dim3(static_cast<unsigned>((g.nchunks + 15) / 16), bhk), 256, 0,
                            stream>>>(k4, v4, g.Nkv, static_cast<int>(g.nchunks), ksum, vmax);
    kv_finalize_kernel<<<bhk, kHeadDim, 0, stream>>>(ksum, vmax, g.Nkv, static_cast<int>(g.nchunks),
                                                     k_mean, v_scales);
    quant_int8_kernel<true><<<dim3(static_cast<unsigned>(g.nbk), bhk), 256, 0, stream>>>(
        k4, g.Nkv, g.nk32, static_cast<int>(g.nbk), k_mean, k_codes, k_scales);
    quant_v_kernel<<<dim3(static_cast<unsigned>(g.nk128 / kVPad), bhk), 256, 0, stream>>>(
        v4, g.Nkv, g.nk128, v_scales, v_codes);
    if (q)   // without Q, K and V only (the forward quantises Q itself)
        quant_int8_kernel<false><<<dim3(static_cast<unsigned>(g.nbq), bhq), 256, 0, stream>>>(
            q4, g.Nq, g.nq32, static_cast<int>(g.nbq), nullptr, q_codes, q_scales);
    return cudaGetLastError();
}

cudaError_t launch_prepare_kv_split(const Geometry &g, const void *k, const void *v, int8_t *k_codes,
                                    float *k_scales, float *k_mean, uint8_t *v_codes, float *v_scales,
                                    void *workspace, cudaStream_t stream, cudaStream_t v_stream,
                                    cudaEvent_t fork, cudaEvent_t join)
{
    const int bhk = g.B * g.Hkv;
    float *ksum = static_cast<float *>(workspace);
    float *vmax = ksum + static_cast<size_t>(bhk) * g.nchunks * kHeadDim;
    const uint4 *k4 = static_cast<const uint4 *>(k);
    const uint4 *v4 = static_cast<const uint4 *>(v);
    kv_chunk_stats_kernel<<<dim3(static_cast<unsigned>((g.nchunks + 15) / 16), bhk), 256, 0,
                            stream>>>(k4, v4, g.Nkv, static_cast<int>(g.nchunks), ksum, vmax);
    kv_finalize_kernel<<<bhk, kHeadDim, 0, stream>>>(ksum, vmax, g.Nkv, static_cast<int>(g.nchunks),
                                                     k_mean, v_scales);
    cudaError_t e = cudaEventRecord(fork, stream);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(v_stream, fork, 0);
    if (e != cudaSuccess)
        return e;
    quant_v_kernel<<<dim3(static_cast<unsigned>(g.nk128 / kVPad), bhk), 256, 0, v_stream>>>(
        v4, g.Nkv, g.nk128, v_scales, v_codes);
    if ((e = cudaEventRecord(join, v_stream)) != cudaSuccess)
        return e;
    quant_int8_kernel<true><<<dim3(static_cast<unsigned>(g.nbk), bhk), 256, 0, stream>>>(
        k4, g.Nkv, g.nk32, static_cast<int>(g.nbk), k_mean, k_codes, k_scales);
    if ((e = cudaStreamWaitEvent(stream, join, 0)) != cudaSuccess)
        return e;
    return cudaGetLastError();
}

cudaError_t launch_prepare_q(const Geometry &g, const void *q, int8_t *q_codes, float *q_scales,
                             cudaStream_t stream)
{
    quant_int8_kernel<false><<<dim3(static_cast<unsigned>(g.nbq), static_cast<unsigned>(g.B * g.Hq)), 256, 0,
                               stream>>>(static_cast<const uint4 *>(q), g.Nq, g.nq32, static_cast<int>(g.nbq), nullptr,
                                         q_codes, q_scales);
    return cudaGetLastError();
}

cudaError_t launch_int8_quantiser_sweep(uint32_t amax_lo, uint32_t amax_hi, unsigned long long *result,
                                        cudaStream_t stream)
{
    if (cudaMemsetAsync(result, 0, 3 * sizeof(unsigned long long), stream) != cudaSuccess)
        return cudaGetLastError();
    int8_quantiser_sweep_kernel<<<amax_hi - amax_lo, 256, 0, stream>>>(amax_lo, result);
    return cudaGetLastError();
}

}  // namespace sattn
