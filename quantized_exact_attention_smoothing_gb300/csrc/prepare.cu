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
#include <algorithm>
#include <mutex>

#include <cuda_bf16.h>

#include "prep_device.cuh"

namespace sattn {
namespace {


// Stages of the statistics pass's copy pipeline, 32 KB each: the 64 tokens of
// one K-mean chunk of K and of V.
constexpr int kStatStages = 3;
constexpr uint32_t kStatStageBytes = 2 * kMeanChunk * kHeadDim * 2;

// FP32 column sums of K (ascending token order) and column max |V| of every
// 64-token chunk, by persistent CTAs: CTA c takes the (KV head, chunk) pairs
// u = c, c + gridDim.x, ... in memory order.  All 256 threads copy the
// chunk's K and V rows (16 KB each, contiguous) into a shared-memory stage
// (cp.async), kStatStages - 1 chunks ahead; then thread j < 128 sums channel j
// of K over the chunk's tokens in ascending order and thread 128 + j takes the
// max |V| of channel j.
__device__ __forceinline__ void chunk_stats_pass(const uint4 *__restrict__ k, const uint4 *__restrict__ v, int Nkv,
                                                 int nchunks, int total, float *__restrict__ ksum,
                                                 float *__restrict__ vmax, uint8_t *stat_smem)
{
    const int tid = threadIdx.x;
    auto copy = [&](int u, int slot) {   // this thread's 8 of the 2048 16-byte pieces of pair u
        const int bh = u / nchunks, t0 = (u - bh * nchunks) * kMeanChunk;
        const uint32_t dst = ptx::smem_u32(stat_smem + slot * kStatStageBytes);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = tid + 256 * (e & 3), tok = j >> 4, piece = j & 15;
            if (t0 + tok < Nkv) {
                const uint4 *src = (e < 4 ? k : v) + (static_cast<size_t>(bh) * Nkv + t0 + tok) * 16 + piece;
                ptx::cp_async16(dst + (e < 4 ? 0u : kStatStageBytes / 2) + 16u * j, src);
            }
        }
    };
    const int step = static_cast<int>(gridDim.x);
#pragma unroll
    for (int s = 0; s < kStatStages - 1; ++s) {
        const int64_t un = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(s) * step;
        if (un < total)
            copy(static_cast<int>(un), s);
        ptx::cp_async_commit();
    }
    const bool is_v = tid >= 128;
    const int c = tid & 127;
    int i = 0;
    for (int u = blockIdx.x; u < total; u += step, ++i) {
        const int64_t un = static_cast<int64_t>(u) + static_cast<int64_t>(kStatStages - 1) * step;
        if (un < total)   // the stage of pair u - step, free since the barrier that ended it
            copy(static_cast<int>(un), (i + kStatStages - 1) % kStatStages);
        ptx::cp_async_commit();
        ptx::cp_async_wait<kStatStages - 1>();
        __syncthreads();   // every thread's pieces of pair u have landed
        const int bh = u / nchunks, chunk = u - bh * nchunks;
        const int n = min(kMeanChunk, Nkv - chunk * kMeanChunk);
        const uint16_t *col = reinterpret_cast<const uint16_t *>(stat_smem + (i % kStatStages) * kStatStageBytes +
                                                                 (is_v ? kStatStageBytes / 2 : 0u)) + c;
        float acc = 0.0f;
        if (!is_v) {
#pragma unroll 16
            for (int t = 0; t < n; ++t)
                acc = __fadd_rn(acc, __uint_as_float(static_cast<uint32_t>(col[t * kHeadDim]) << 16));
            ksum[static_cast<size_t>(u) * kHeadDim + c] = acc;
        } else {
#pragma unroll 16
            for (int t = 0; t < n; ++t)
                acc = fmaxf(acc, fabsf(__uint_as_float(static_cast<uint32_t>(col[t * kHeadDim]) << 16)));
            vmax[static_cast<size_t>(u) * kHeadDim + c] = acc;
        }
        __syncthreads();   // the stage is read: the next pair's copies may overwrite it
    }
    ptx::cp_async_wait<0>();
}

__global__ void __launch_bounds__(256) kv_chunk_stats_kernel(const uint4 *__restrict__ k,
                                                             const uint4 *__restrict__ v, int Nkv,
                                                             int nchunks, int total, float *__restrict__ ksum,
                                                             float *__restrict__ vmax)
{
    extern __shared__ __align__(16) uint8_t stat_smem[];
    chunk_stats_pass(k, v, Nkv, nchunks, total, ksum, vmax, stat_smem);
}

// One CTA per KV head: thread j < 128 adds the chunk sums of channel j of K in
// ascending chunk order (mean = sum / Nkv); thread 128 + j takes the max of
// channel j's chunk maxima of |V| (s_v = amax / 448).  The loads of the next
// 32 chunks are issued before the current 32 are combined, so the chain of
// additions, not the load latency, sets the time.
template <bool kMax>
__device__ __forceinline__ float finalize_column(const float *__restrict__ src, int nchunks)
{
    constexpr int kBatch = 32;
    auto combine = [](float acc, float x) { return kMax ? fmaxf(acc, x) : __fadd_rn(acc, x); };
    float acc = 0.0f;
    const int full = nchunks / kBatch;
    float a[kBatch];
    if (full > 0) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            a[u] = ptx::ld_nc_f32(src + static_cast<size_t>(u) * kHeadDim);
    }
    for (int b = 0; b < full; ++b) {
        float nx[kBatch];
        const int nb = b + 1 < full ? b + 1 : b;   // the last batch reloads itself (never used)
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            nx[u] = ptx::ld_nc_f32(src + static_cast<size_t>(nb * kBatch + u) * kHeadDim);
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            acc = combine(acc, a[u]);
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            a[u] = nx[u];
    }
    for (int ch = full * kBatch; ch < nchunks; ++ch)
        acc = combine(acc, ptx::ld_nc_f32(src + static_cast<size_t>(ch) * kHeadDim));
    return acc;
}

__global__ void __launch_bounds__(256) kv_finalize_kernel(const float *__restrict__ ksum,
                                                          const float *__restrict__ vmax, int Nkv,
                                                          int nchunks, float *__restrict__ k_mean,
                                                          float *__restrict__ v_scales)
{
    const int bh = blockIdx.x, c = threadIdx.x & 127;
    const size_t off = static_cast<size_t>(bh) * nchunks * kHeadDim + c;
    if (threadIdx.x >= 128)
        v_scales[bh * kHeadDim + c] = __fdiv_rn(finalize_column<true>(vmax + off, nchunks), 448.0f);
    else
        k_mean[bh * kHeadDim + c] = __fdiv_rn(finalize_column<false>(ksum + off, nchunks), static_cast<float>(Nkv));
}

// Grid of a persistent kernel on the current device: SMs x CTAs resident per
// SM with `smem` bytes of dynamic shared memory, whose limit is raised first.
// Looked up once per device and kernel (`cache`: one slot per device).
template <class Kernel>
int persistent_grid(Kernel kernel, int smem, int (&cache)[64], cudaError_t *err)
{
    static std::mutex mu;
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess || dev < 0 || dev >= 64) {
        *err = *err != cudaSuccess ? *err : cudaErrorInvalidDevice;
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n_sm = 0, per_sm = 0;
        if ((*err = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (*err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess ||
            (*err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, smem)) != cudaSuccess)
            return 0;
        cache[dev] = std::max(1, n_sm) * std::max(1, per_sm);
    }
    return cache[dev];
}

// The statistics pass: a persistent grid of kv_chunk_stats_kernel (all CTAs
// resident), then kv_finalize_kernel.
cudaError_t launch_kv_stats(const Geometry &g, const uint4 *k4, const uint4 *v4, float *ksum, float *vmax,
                            float *k_mean, float *v_scales, cudaStream_t stream)
{
    static int cache[64];
    const int smem = kStatStages * static_cast<int>(kStatStageBytes);
    cudaError_t e = cudaSuccess;
    const int ctas = persistent_grid(kv_chunk_stats_kernel, smem, cache, &e);
    if (e != cudaSuccess)
        return e;
    const int64_t total = g.nchunks * g.B * g.Hkv;
    kv_chunk_stats_kernel<<<static_cast<int>(std::min<int64_t>(total, ctas)), 256, smem, stream>>>(
        k4, v4, g.Nkv, static_cast<int>(g.nchunks), static_cast<int>(total), ksum, vmax);
    kv_finalize_kernel<<<g.B * g.Hkv, 256, 0, stream>>>(ksum, vmax, g.Nkv, static_cast<int>(g.nchunks), k_mean,
                                                        v_scales);
    return cudaGetLastError();
}

// ---- the K/V preparation as one cooperative launch ----------------------
//
// Statistics, finalize and the K and V quantisers in one persistent kernel,
// phases separated by two grid barriers; the quantisers' second read of K and
// V then follows the statistics' first read directly, walking the heads in
// the reverse order so that the heads read last (still in L2) come first.

constexpr uint64_t kGridBarrierTimeoutNs = 1000000000ull;
constexpr size_t kPrepSyncBytes = 256;   // grid counter and status word, after the statistics

// A barrier over the grid: each CTA arrives once on the counter sync[0]
// (zeroed before the launch) and waits until the counter reaches `target`
// (k * gridDim.x for the k-th barrier).  The launch is cooperative, so every
// CTA is resident and the wait ends; it still gives up after about a second,
// or as soon as another CTA has given up, setting bit 0 of sync[1], and
// returns false.
__device__ __forceinline__ bool grid_barrier(unsigned *sync, unsigned target)
{
    __syncthreads();
    int ok = 1;
    if (threadIdx.x == 0) {
        __threadfence();   // the CTA's writes (ordered by the barrier above) before its arrival
        atomicAdd(sync, 1u);
        const uint64_t t0 = ptx::globaltimer();
        for (unsigned it = 0;; ++it) {
            unsigned c;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(sync) : "memory");
            if (c >= target)
                break;
            if ((it & 63u) == 63u &&
                (*reinterpret_cast<volatile unsigned *>(sync + 1) != 0u || ptx::globaltimer() - t0 > kGridBarrierTimeoutNs)) {
                atomicOr(sync + 1, 1u);
                ok = 0;
                break;
            }
        }
        __threadfence();
    }
    return __syncthreads_and(ok) != 0;
}

// finalize_column for data written earlier in the same launch (loads through L2)
template <bool kMax>
__device__ __forceinline__ float finalize_column_l2(const float *src, int nchunks)
{
    float acc = 0.0f;
    for (int ch = 0; ch < nchunks; ch += 16) {
        float a[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
            a[u] = ch + u < nchunks ? __ldcg(src + static_cast<size_t>(ch + u) * kHeadDim) : 0.0f;
#pragma unroll
        for (int u = 0; u < 16; ++u)
            if (ch + u < nchunks)
                acc = kMax ? fmaxf(acc, a[u]) : __fadd_rn(acc, a[u]);
    }
    return acc;
}

__global__ void __launch_bounds__(256) kv_prep_fused_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                            int Nkv, int nchunks, int bhk, int64_t nk32, int nbk,
                                                            int64_t nk128, float *ksum, float *vmax, float *k_mean,
                                                            float *v_scales, int8_t *__restrict__ k_codes,
                                                            float *__restrict__ k_scales, uint8_t *__restrict__ v_codes,
                                                            unsigned *sync, unsigned withhold)
{
    extern __shared__ __align__(16) uint8_t fsmem[];
    const int tid = threadIdx.x;
    // phase 1: chunk statistics
    chunk_stats_pass(k, v, Nkv, nchunks, bhk * nchunks, ksum, vmax, fsmem);
    // (withhold: test hook, the first barrier waits for CTAs that do not exist)
    if (!grid_barrier(sync, gridDim.x + withhold))
        return;
    // phase 2: per-head mean of K and scale of V
    for (int bh = blockIdx.x; bh < bhk; bh += gridDim.x) {
        const int c = tid & 127;
        const size_t off = static_cast<size_t>(bh) * nchunks * kHeadDim + c;
        if (tid >= 128)
            v_scales[bh * kHeadDim + c] = __fdiv_rn(finalize_column_l2<true>(vmax + off, nchunks), 448.0f);
        else
            k_mean[bh * kHeadDim + c] = __fdiv_rn(finalize_column_l2<false>(ksum + off, nchunks), static_cast<float>(Nkv));
    }
    if (!grid_barrier(sync, 2 * gridDim.x + withhold))
        return;
    // phase 3: the quantisers, heads in reverse order; per head its V tiles, then its K blocks
    uint32_t *tile = reinterpret_cast<uint32_t *>(fsmem);                  // V: [kVPad][32] words
    float *sv = reinterpret_cast<float *>(fsmem + kVPad * 32 * 4);           // V scales of the head
    float *rv = sv + kHeadDim;                                               // and their reciprocals
    float *mean = rv + kHeadDim;                                             // K mean of the head
    float *warp_max = mean + kHeadDim;
    const int nvt = static_cast<int>(nk128 / kVPad);
    const int per_head = nvt + nbk;
    const int64_t total = static_cast<int64_t>(bhk) * per_head;
    auto sync256 = [] { __syncthreads(); };
    int have_v = -1, have_k = -1;   // the head whose scales / mean are in shared memory
    for (int64_t it = blockIdx.x; it < total; it += gridDim.x) {
        const int hi = static_cast<int>(it / per_head), r = static_cast<int>(it - static_cast<int64_t>(hi) * per_head);
        const int bh = bhk - 1 - hi;
        if (r < nvt) {
            if (have_v != bh) {
                if (tid < kHeadDim) {
                    const float x = __ldcg(v_scales + bh * kHeadDim + tid);
                    sv[tid] = x;
                    rv[tid] = x > 0.0f ? __frcp_rn(x) : 0.0f;
                }
                have_v = bh;
            }
            __syncthreads();
            prep::quant_v_tile(v, Nkv, nk128, sv, rv, v_codes, bh, r * kVPad, tid, tile, sync256);
        } else {
            if (have_k != bh) {
                if (tid < kHeadDim)
                    mean[tid] = __ldcg(k_mean + bh * kHeadDim + tid);
                have_k = bh;
            }
            __syncthreads();
            const int blk = r - nvt, row = tid >> 3, part = tid & 7;
            const int t = blk * kQBlock + row;
            float val[16];
            if (t < Nkv) {
                const uint4 *src = k + (static_cast<size_t>(bh) * Nkv + t) * 16 + part * 2;
                prep::block_values<true>(prep::ld_stream(src), prep::ld_stream(src + 1), mean, 0, part, val);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    val[e] = 0.0f;
            }
            prep::quant_block_values(val, Nkv, nk32, nbk, k_codes, k_scales, bh, blk, tid, warp_max, sync256);
        }
        __syncthreads();   // shared memory is reused by the next item
    }
}

// One CTA per 32-token block of one head; thread = (token, eighth of the
// channels: 16 values), so a thread holds few registers and many CTAs stay
// resident to keep loads in flight.  With kSmooth (K), the per-channel mean
// is subtracted first.
template <bool kSmooth>
__global__ void __launch_bounds__(256, 6) quant_int8_kernel(const uint4 *__restrict__ x, int N,
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
__global__ void __launch_bounds__(256, 4) quant_v_kernel(const uint4 *__restrict__ v, int Nkv,
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

size_t prepare_status_offset(const Geometry &g)
{
    return 2 * static_cast<size_t>(g.B) * g.Hkv * g.nchunks * kHeadDim * sizeof(float) + sizeof(unsigned);
}

size_t prepare_workspace_bytes(const Geometry &g)
{
    return 2 * static_cast<size_t>(g.B) * g.Hkv * g.nchunks * kHeadDim * sizeof(float) + kPrepSyncBytes;
}

cudaError_t launch_prepare_kv_fused(const Geometry &g, const void *k, const void *v, int8_t *k_codes,
                                    float *k_scales, float *k_mean, uint8_t *v_codes, float *v_scales,
                                    void *workspace, cudaStream_t stream, bool withhold)
{
    static int cache[64];
    const int smem = kStatStages * static_cast<int>(kStatStageBytes);
    cudaError_t ge = cudaSuccess;
    const int ctas = persistent_grid(kv_prep_fused_kernel, smem, cache, &ge);
    if (ge != cudaSuccess)
        return ge;
    const int bhk = g.B * g.Hkv;
    float *ksum = static_cast<float *>(workspace);
    float *vmax = ksum + static_cast<size_t>(bhk) * g.nchunks * kHeadDim;
    unsigned *sync = reinterpret_cast<unsigned *>(vmax + static_cast<size_t>(bhk) * g.nchunks * kHeadDim);
    cudaError_t e = cudaMemsetAsync(sync, 0, 2 * sizeof(unsigned), stream);
    if (e != cudaSuccess)
        return e;
    const uint4 *k4 = static_cast<const uint4 *>(k);
    const uint4 *v4 = static_cast<const uint4 *>(v);
    int Nkv = g.Nkv, nchunks = static_cast<int>(g.nchunks), nbk = static_cast<int>(g.nbk);
    int64_t nk32 = g.nk32, nk128 = g.nk128;
    unsigned wh = withhold ? 1u : 0u;
    void *args[] = {&k4, &v4, &Nkv, &nchunks, const_cast<int *>(&bhk), &nk32, &nbk, &nk128, &ksum, &vmax,
                    &k_mean, &v_scales, &k_codes, &k_scales, &v_codes, &sync, &wh};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kv_prep_fused_kernel), dim3(ctas), dim3(256),
                                       args, static_cast<size_t>(smem), stream);
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

    const cudaError_t se = launch_kv_stats(g, k4, v4, ksum, vmax, k_mean, v_scales, stream);
    if (se != cudaSuccess)
        return se;
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
    const cudaError_t se = launch_kv_stats(g, k4, v4, ksum, vmax, k_mean, v_scales, stream);
    if (se != cudaSuccess)
        return se;
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
