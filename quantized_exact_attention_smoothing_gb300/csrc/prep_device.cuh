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

// e4m3_code of eight values of one token against their eight channel scales
// s (rs2: the reciprocals in packed pairs; keep: byte mask of the channels
// with s > 0, whose codes are kept, the others 0), four bytes per word, value
// i in byte i % 4 of word i / 4.  The same decision as e4m3_code on packed
// pairs: both brackets of fl(v * fl(1/s)) for two values per instruction, and
// IEEE division for the values of a word whose brackets differ (rare).
__device__ __forceinline__ void e4m3_codes8(const float (&v)[8], const float (&s)[8], const uint64_t (&rs2)[4],
                                            const uint32_t (&keep)[2], uint32_t (&w)[2])
{
    const uint64_t up2 = ptx::f32x2(1.0f + 0x1p-21f, 1.0f + 0x1p-21f);
    const uint64_t dn2 = ptx::f32x2(1.0f - 0x1p-21f, 1.0f - 0x1p-21f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int i = 4 * h + 2 * k;
            const uint64_t y2 = ptx::mul_f32x2(ptx::f32x2(v[i], v[i + 1]), rs2[2 * h + k]);
            const uint64_t a2 = ptx::mul_f32x2(y2, up2), b2 = ptx::mul_f32x2(y2, dn2);
            // value i in the low byte, i + 1 in the high byte
            hi[k] = ptx::cvt_e4m3x2(ptx::f32x2_hi(a2), ptx::f32x2_lo(a2));
            lo[k] = ptx::cvt_e4m3x2(ptx::f32x2_hi(b2), ptx::f32x2_lo(b2));
        }
        uint32_t word = __byte_perm(hi[0], hi[1], 0x5410u);
        const uint32_t other = __byte_perm(lo[0], lo[1], 0x5410u);
        if (word != other) {   // a value of this word is within 2^-21 of an E4M3 rounding boundary
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t d = (word ^ other) >> (8 * u) & 0xffu;
                if (d != 0u && s[4 * h + u] > 0.0f) {
                    const uint32_t code = ptx::cvt_e4m3x2(0.0f, __fdiv_rn(v[4 * h + u], s[4 * h + u])) & 0xffu;
                    word = (word & ~(0xffu << (8 * u))) | (code << (8 * u));
                }
            }
        }
        w[h] = word & keep[h];
    }
}

// int8_code of 16 values (value i -> byte i % 4 of word i / 4) on packed
// pairs: q = fl(x * rs), r = fl(q + 1.5 * 2^23) and the distance of q from
// the integer r - 1.5 * 2^23, for two values per instruction.  A pair with a
// value near a rounding tie (or not finite) takes int8_code_div for both.
// (If the assembler fuses the product into the addition, r can differ from
// the two-step value only when q is within 2^-16 of a half-integer, which the
// tie test sends to the division as well.)
__device__ __forceinline__ void int8_codes16(const float (&val)[16], float s, float rs, uint32_t (&packed)[4])
{
    const uint64_t rs2 = ptx::f32x2(rs, rs), m2 = ptx::f32x2(kRoundMagic, kRoundMagic);
    uint32_t b[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint64_t q2 = ptx::mul_f32x2(ptx::f32x2(val[2 * k], val[2 * k + 1]), rs2);
        const uint64_t r2 = ptx::add_f32x2(q2, m2);
        const uint64_t d2 = ptx::sub_f32x2(q2, ptx::sub_f32x2(r2, m2));
        b[2 * k] = __float_as_uint(ptx::f32x2_lo(r2));
        b[2 * k + 1] = __float_as_uint(ptx::f32x2_hi(r2));
        if (!(fabsf(ptx::f32x2_lo(d2)) < kTieMargin && fabsf(ptx::f32x2_hi(d2)) < kTieMargin)) {
            b[2 * k] = int8_code_div(val[2 * k], s);
            b[2 * k + 1] = int8_code_div(val[2 * k + 1], s);
        }
    }
#pragma unroll
    for (int w = 0; w < 4; ++w)
        packed[w] = __byte_perm(__byte_perm(b[4 * w], b[4 * w + 1], 0x0040u),
                                __byte_perm(b[4 * w + 2], b[4 * w + 3], 0x0040u), 0x5410u);
}

// The 16 values of one thread of a 32-token block (its token's channels
// 16 part .. 16 part + 15, from two 16-byte chunks), with the per-channel mean
// of head bh subtracted first for K (kSmooth).
template <bool kSmooth>
__device__ __forceinline__ void block_values(const uint4 &a, const uint4 &b, const float *__restrict__ mean, int bh,
                                             int part, float (&val)[16])
{
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
}

// INT8 codes and scale of one 32-token block (blk) of head bh from the
// values of thread tid of 256 = (token tid / 8, channels 16 (tid % 8) .. + 15;
// val all 0 for a token past N): amax over the block, s = amax / 127, codes
// and s written.  warp_max: 8 floats of shared memory; sync(): a barrier
// over the 256 threads.
template <class Sync>
__device__ __forceinline__ void quant_block_values(const float (&val)[16], int N, int64_t npad, int nblk,
                                                   int8_t *__restrict__ codes, float *__restrict__ scales, int bh,
                                                   int blk, int tid, float *warp_max, Sync sync)
{
    const int r = tid >> 3, part = tid & 7;
    const int t = blk * kQBlock + r;
    const bool valid = t < N;
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i += 2)
        am = ptx::fmax3(am, fabsf(val[i]), fabsf(val[i + 1]));
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
        int8_codes16(val, s, rs, packed);
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

// INT8 codes and scale of one 32-token block (blk) of head bh, loaded by the
// 256 threads themselves (see block_values, quant_block_values).
template <bool kSmooth, class Sync>
__device__ __forceinline__ void quant_block(const uint4 *__restrict__ x, int N, int64_t npad, int nblk,
                                            const float *__restrict__ mean, int8_t *__restrict__ codes,
                                            float *__restrict__ scales, int bh, int blk, int tid,
                                            float *warp_max, Sync sync)
{
    const int r = tid >> 3, part = tid & 7;
    const int t = blk * kQBlock + r;
    float val[16];
    if (t < N) {
        const uint4 *src = x + (static_cast<size_t>(bh) * N + t) * 16 + part * 2;
        block_values<kSmooth>(ld_stream(src), ld_stream(src + 1), mean, bh, part, val);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            val[i] = 0.0f;
    }
    quant_block_values(val, N, npad, nblk, codes, scales, bh, blk, tid, warp_max, sync);
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
    float s8[8];
    uint64_t rs2[4];
    uint32_t keep[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        s8[i] = sv[g * 8 + i];
        keep[i >> 2] |= (s8[i] > 0.0f ? 0xffu : 0u) << (8 * (i & 3));
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
        rs2[k] = ptx::f32x2(rv[g * 8 + 2 * k], rv[g * 8 + 2 * k + 1]);
    uint4 raw[8];
#pragma unroll
    for (int it = 0; it < 8; ++it) {   // all eight loads in flight
        const int t = t0 + ((tid + it * 256) >> 4);
        raw[it] = t < Nkv ? ld_stream(v + (static_cast<size_t>(bh) * Nkv + t) * 16 + g) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int row = (tid + it * 256) >> 4;
        uint32_t w[2] = {0u, 0u};
        if (t0 + row < Nkv) {
            float f[8];
            unpack8(raw[it], f);
            e4m3_codes8(f, s8, rs2, keep, w);
        }
        const int sw = ((row >> 4) & 7) << 1;
        *reinterpret_cast<uint2 *>(&tile[row * 32 + ((2 * g) ^ sw)]) = make_uint2(w[0], w[1]);
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
