// prep_device.cuh -- the preparation's per-thread steps as device functions,
// shared by the preparation kernels (prepare.cu) and the single-launch
// small-shape path of the forward (attn_fwd.cu), so both write the same bytes.
// ("Experiment Log" page, entry "Phase 0 Import And Verification": K
// smoothing, INT8 quantisation of Q and K, FP8 V.)
#pragma once
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "quant.cuh"
#include "sattn_internal.cuh"

namespace sattn {
namespace prep {

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

// Column sums of K (FP32, ascending token order) and column max |V| of one
// 64-token chunk, 8 channels (group g: channels 8g .. 8g + 7) of head bh.
__device__ __forceinline__ void chunk_stats8(const uint4 *__restrict__ k, const uint4 *__restrict__ v, int Nkv,
                                             int bh, int chunk, int g, float (&s)[8], float (&mx)[8])
{
    const int t0 = chunk * kMeanChunk;
    const int t1 = min(Nkv, t0 + kMeanChunk);
    const size_t row0 = static_cast<size_t>(bh) * Nkv + t0;
    const uint4 *kp = k + row0 * 16 + g;
    const uint4 *vp = v + row0 * 16 + g;
    float f[8];
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

// INT8 codes and scale of one 32-token block (blk) of head bh: thread tid of
// 256 = (token tid / 8, channels 16 (tid % 8) .. + 15); with kSmooth (K) the
// per-channel mean is subtracted first.  warp_max: 8 floats of shared memory;
// sync(): a barrier over the 256 threads.
template <bool kSmooth, class Sync>
__device__ __forceinline__ void quant_block(const uint4 *__restrict__ x, int N, int64_t npad, int nblk,
                                            const float *__restrict__ mean, int8_t *__restrict__ codes,
                                            float *__restrict__ scales, int bh, int blk, int tid,
                                            float *warp_max, Sync sync)
{
    const int r = tid >> 3, part = tid & 7;
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
    if ((tid & 31) == 0)
        warp_max[tid >> 5] = am;
    sync();
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
    if (tid == 0)
        scales[static_cast<size_t>(bh) * nblk + blk] = s;
}

// E4M3 codes of one 128-token tile (t0 = tile * 128) of KV head bh, written
// channel-major, by thread tid of 256.  sv, rv: the 128 channel scales and
// their reciprocals (shared memory); tile: kVPad * 32 words of shared memory;
// sync(): a barrier over the 256 threads.  Phase 1: coalesced 16-byte loads
// of 8 channels of one token, codes written token-major into shared memory
// (8 bytes per store).  Phase 2: each thread gathers 16 consecutive tokens of
// one channel and writes them channel-major (16-byte stores).  Word j of token
// row t is stored at word j ^ (2 * ((t >> 4) & 7)), so the 16-token gathers of
// one warp hit eight distinct banks.
template <class Sync>
__device__ __forceinline__ void quant_v_tile(const uint4 *__restrict__ v, int Nkv, int64_t nk128,
                                             const float *sv, const float *rv, uint8_t *__restrict__ vcodes,
                                             int bh, int t0, int tid, uint32_t *tile, Sync sync)
{
    const int g = tid & 15;   // this thread's 8 channels, every item
    float s8[8], r8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        s8[i] = sv[g * 8 + i];
        r8[i] = rv[g * 8 + i];
    }
#pragma unroll
    for (int it = 0; it < 8; ++it) {   // all eight loads in flight
        const int row = (tid + it * 256) >> 4;
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
    sync();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int idx = tid + it * 256;
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

}  // namespace prep
}  // namespace sattn
