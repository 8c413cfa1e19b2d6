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

#include "ptx.cuh"
#include "quant.cuh"
#include "sattn_internal.cuh"

namespace sattn {
namespace {

__device__ __forceinline__ void unpack8(const uint4 &a, float (&f)[8])
{
    f[0] = bf16_lo(a.x); f[1] = bf16_hi(a.x);
    f[2] = bf16_lo(a.y); f[3] = bf16_hi(a.y);
    f[4] = bf16_lo(a.z); f[5] = bf16_hi(a.z);
    f[6] = bf16_lo(a.w); f[7] = bf16_hi(a.w);
}

__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

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
    const int t0 = chunk * kMeanChunk;
    const int t1 = min(Nkv, t0 + kMeanChunk);
    const size_t row0 = static_cast<size_t>(bh) * Nkv + t0;
    const uint4 *kp = k + row0 * 16 + g;
    const uint4 *vp = v + row0 * 16 + g;
    float s[8], mx[8], f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        s[i] = 0.0f;
        mx[i] = 0.0f;
    }
#pragma unroll 16
    for (int t = t0; t < t1; ++t) {
        const uint4 a = ld_stream(kp);
        const uint4 c = ld_stream(vp);
        kp += 16;
        vp += 16;
        unpack8(a, f);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            s[i] = __fadd_rn(s[i], f[i]);
        unpack8(c, f);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            mx[i] = fmaxf(mx[i], fabsf(f[i]));
    }
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

// E4M3(fl(v / s)) (round to nearest even, saturating) without a division in
// the common case: y = fl(v * fl(1/s)) is within 3 ulp (relative 2^-22.4) of
// fl(v / s), so if y * (1 - 2^-21) and y * (1 + 2^-21) round to the same code
// (the conversion is monotonic), fl(v / s) does too.  Otherwise (values near a
// rounding midpoint) the IEEE division decides.  Returns the byte.
__device__ __forceinline__ uint32_t e4m3_code(float v, float s, float rs)
{
    const float y = __fmul_rn(v, rs);
    const uint32_t two = ptx::cvt_e4m3x2(__fmul_rn(y, 1.0f + 0x1p-21f), __fmul_rn(y, 1.0f - 0x1p-21f));
    if ((two & 0xffu) == (two >> 8))
        return two & 0xffu;
    return ptx::cvt_e4m3x2(0.0f, __fdiv_rn(v, s)) & 0xffu;
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
    const int bh = blockIdx.y, blk = blockIdx.x;
    const int r = threadIdx.x >> 3, part = threadIdx.x & 7;
    const int t = blk * kQBlock + r;
    const bool valid = t < N;
    float val[16];
    if (valid) {
        const uint4 *src = x + (static_cast<size_t>(bh) * N + t) * 16 + part * 2;
        const uint4 a = ld_stream(src), b = ld_stream(src + 1);
        float f[8];
        unpack8(a, f);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            val[i] = f[i];
        unpack8(b, f);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            val[8 + i] = f[i];
        if (kSmooth) {
            const float4 *mu = reinterpret_cast<const float4 *>(mean + bh * kHeadDim + part * 16);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float4 m4 = mu[w];
                val[4 * w] = __fsub_rn(val[4 * w], m4.x);
                val[4 * w + 1] = __fsub_rn(val[4 * w + 1], m4.y);
                val[4 * w + 2] = __fsub_rn(val[4 * w + 2], m4.z);
                val[4 * w + 3] = __fsub_rn(val[4 * w + 3], m4.w);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            val[i] = 0.0f;
    }
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        am = fmaxf(am, fabsf(val[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if ((threadIdx.x & 31) == 0)
        warp_max[threadIdx.x >> 5] = am;
    __syncthreads();
    float amax = warp_max[0];
#pragma unroll
    for (int w = 1; w < 8; ++w)
        amax = fmaxf(amax, warp_max[w]);
    const float s = __fdiv_rn(amax, 127.0f);
    const float rs = s > 0.0f ? __frcp_rn(s) : 0.0f;
    uint32_t packed[4];
    if (valid && s > 0.0f) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint32_t lo = __byte_perm(int8_code(val[w * 4], s, rs), int8_code(val[w * 4 + 1], s, rs), 0x0040u);
            const uint32_t hi = __byte_perm(int8_code(val[w * 4 + 2], s, rs), int8_code(val[w * 4 + 3], s, rs), 0x0040u);
            packed[w] = __byte_perm(lo, hi, 0x5410u);
        }
    } else {
#pragma unroll
        for (int w = 0; w < 4; ++w)
            packed[w] = 0u;
    }
    *reinterpret_cast<uint4 *>(codes + (static_cast<size_t>(bh) * npad + t) * kHeadDim + part * 16) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if (threadIdx.x == 0)
        scales[static_cast<size_t>(bh) * nblk + blk] = s;
}

// One CTA per 128-token tile of one KV head.  Phase 1: coalesced 16-byte
// loads of 8 channels of one token, E4M3 codes written token-major into
// shared memory (8 bytes per store).  Phase 2: each thread gathers 16
// consecutive tokens of one channel and writes them channel-major (16-byte
// stores).  Word j of token row t is stored at word j ^ (2 * ((t >> 4) & 7)),
// so the 16-token gathers of one warp hit eight distinct banks.
__global__ void __launch_bounds__(256) quant_v_kernel(const uint4 *__restrict__ v, int Nkv,
                                                      int64_t nk128,
                                                      const float *__restrict__ v_scales,
                                                      uint8_t *__restrict__ vcodes)
{
    __shared__ __align__(16) uint32_t tile[kVPad * 32];   // [token][32 words]
    __shared__ float sv[kHeadDim], rv[kHeadDim];
    const int bh = blockIdx.y;
    const int t0 = blockIdx.x * kVPad;
    if (threadIdx.x < kHeadDim) {
        const float x = v_scales[bh * kHeadDim + threadIdx.x];
        sv[threadIdx.x] = x;
        rv[threadIdx.x] = x > 0.0f ? __frcp_rn(x) : 0.0f;
    }
    __syncthreads();
    const int g = threadIdx.x & 15;                        // this thread's 8 channels, every item
    float s8[8], r8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        s8[i] = sv[g * 8 + i];
        r8[i] = rv[g * 8 + i];
    }
#pragma unroll 2
    for (int it = 0; it < 8; ++it) {
        const int row = (threadIdx.x + it * 256) >> 4;
        const int t = t0 + row;
        uint32_t w0 = 0, w1 = 0;
        if (t < Nkv) {
            float f[8];
            uint32_t cd[8];
            unpack8(ld_stream(v + (static_cast<size_t>(bh) * Nkv + t) * 16 + g), f);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                cd[i] = s8[i] > 0.0f ? e4m3_code(f[i], s8[i], r8[i]) : 0u;
            w0 = __byte_perm(__byte_perm(cd[0], cd[1], 0x0040u), __byte_perm(cd[2], cd[3], 0x0040u), 0x5410u);
            w1 = __byte_perm(__byte_perm(cd[4], cd[5], 0x0040u), __byte_perm(cd[6], cd[7], 0x0040u), 0x5410u);
        }
        const int sw = ((row >> 4) & 7) << 1;
        *reinterpret_cast<uint2 *>(&tile[row * 32 + ((2 * g) ^ sw)]) = make_uint2(w0, w1);
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int idx = threadIdx.x + it * 256;
        const int c = idx >> 3, w = idx & 7;               // channel, 16-token group
        const int word = (c >> 2) ^ (2 * w);
        const uint32_t sel = (c & 3) | ((4 + (c & 3)) << 4);   // byte c % 4 of each of two words
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t *rowp = tile + (16 * w + 4 * q) * 32 + word;
            const uint32_t ab = __byte_perm(rowp[0], rowp[32], sel);
            const uint32_t cdw = __byte_perm(rowp[64], rowp[96], sel);
            o[q] = __byte_perm(ab, cdw, 0x5410u);
        }
        *reinterpret_cast<uint4 *>(vcodes + (static_cast<size_t>(bh) * kHeadDim + c) * nk128 + t0 + w * 16) =
            make_uint4(o[0], o[1], o[2], o[3]);
    }
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
