// mma_rate.cu -- measurement of tcgen05.mma throughput on this device, for the
// forward kernel's roofline: back-to-back MMAs of the forward's own shapes
// (M = 128; kind::f16 with both operands in shared memory, as QK^T;
// kind::f8f6f4 with A in tensor memory, as PV) issued by one thread per SM,
// timed by the SM clock around the issue loop and its completion.  Not part
// of the computation.
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sattn_internal.cuh"

namespace sattn {
namespace {

constexpr uint32_t kRateSmem = 32768 + 65536 + 64;   // A 32 KB, B 64 KB, barrier + TMEM slot

// kind 0: f16, A and B from shared memory; kind 1: E4M3, A from TMEM.  Operands
// hold 1.0 (the values do not change the rate).  cycles: the largest SM-clock
// count over CTAs for iters x 4 MMAs; err: set if the completion wait ran out.
template <int KIND>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int iters, uint32_t N, unsigned long long *cycles,
                                                          unsigned int *err)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = ptx::smem_u32(smem);
    const uint32_t A = sb, B = sb + 32768, BAR = sb + 32768 + 65536, SLOT = BAR + 8;
    for (int i = threadIdx.x; i < (32768 + 65536) / 4; i += blockDim.x)
        reinterpret_cast<uint32_t *>(smem)[i] = KIND == 0 ? 0x3c003c00u : 0x38383838u;
    if (threadIdx.x == 0) {
        ptx::mbar_init(BAR, 1);
        ptx::fence_mbar_init();
    }
    ptx::fence_proxy_async_smem();
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        ptx::tmem_alloc(SLOT, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + 32768 + 65536 + 8);
    if (KIND == 1) {   // A operand: columns [256, 320) of every lane hold E4M3 ones
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            v[i] = 0x38383838u;
        const uint32_t ta = tmem + (static_cast<uint32_t>(warp * 32) << 16) + 256;
        ptx::tmem_st32(ta, v);
        ptx::tmem_st32(ta + 32, v);
        ptx::tmem_wait_st();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (threadIdx.x == 0) {
        const uint32_t idesc = ptx::make_idesc(0, 0, 128, N);
        const unsigned long long t0 = clock64();
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t bd = ptx::sw128_desc(B + s * 32);
                if (KIND == 0)
                    ptx::mma_f16_ss(tmem, ptx::sw128_desc(A + s * 32), bd, idesc, (it | s) != 0);
                else
                    ptx::mma_f8_ts(tmem, tmem + 256 + 8 * s, bd, idesc, (it | s) != 0);
            }
        }
        ptx::mma_commit(BAR);
        const uint64_t g0 = ptx::globaltimer();
        bool done = false;
        while (!(done = ptx::mbar_try_wait(BAR, 0)))
            if (ptx::globaltimer() - g0 > 2000000000ull)
                break;
        if (!done)
            atomicOr(err, 1u);
        atomicMax(cycles, clock64() - t0);
        if (!done) {   // the MMAs have not completed: wait (bounded) before TMEM is freed
            const uint64_t g1 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(BAR, 0) && ptx::globaltimer() - g1 < 2000000000ull) {
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0)
        ptx::tmem_dealloc(tmem, 512);
}

}  // namespace

int measure_mma_rate(int kind, int n, int iters, double *flop_per_clk_sm, double *tflops)
{
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm < 1)
        return 1;
    const size_t smem = 150 * 1024;   // more than half an SM: one CTA per SM
    unsigned long long *cyc = nullptr;
    unsigned int *err = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int rc = 1;
    if (cudaMalloc(&cyc, sizeof(unsigned long long)) != cudaSuccess || cudaMalloc(&err, sizeof(unsigned int)) != cudaSuccess ||
        cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)
        goto done;
    {
        auto launch = [&](int it) {
            if (kind == 0) {
                cudaFuncSetAttribute(mma_rate_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
                mma_rate_kernel<0><<<n_sm, 128, smem>>>(it, static_cast<uint32_t>(n), cyc, err);
            } else {
                cudaFuncSetAttribute(mma_rate_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
                mma_rate_kernel<1><<<n_sm, 128, smem>>>(it, static_cast<uint32_t>(n), cyc, err);
            }
        };
        if (cudaMemset(err, 0, sizeof(unsigned int)) != cudaSuccess)
            goto done;
        launch(16);   // warm-up
        if (cudaMemset(cyc, 0, sizeof(unsigned long long)) != cudaSuccess || cudaEventRecord(e0) != cudaSuccess)
            goto done;
        launch(iters);
        if (cudaEventRecord(e1) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
            cudaGetLastError() != cudaSuccess)
            goto done;
        float ms = 0.0f;
        unsigned long long cy = 0;
        unsigned int er = 0;
        if (cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess ||
            cudaMemcpy(&cy, cyc, sizeof cy, cudaMemcpyDeviceToHost) != cudaSuccess ||
            cudaMemcpy(&er, err, sizeof er, cudaMemcpyDeviceToHost) != cudaSuccess || er != 0 || cy == 0)
            goto done;
        const double k = kind == 0 ? 16.0 : 32.0;   // K per instruction: 32 bytes of each operand row
        const double flop = 2.0 * 128.0 * n * k * 4.0 * iters;   // per SM
        *flop_per_clk_sm = flop / static_cast<double>(cy);
        *tflops = flop * n_sm / (static_cast<double>(ms) * 1e-3) / 1e12;
        rc = 0;
    }
done:
    if (e0)
        cudaEventDestroy(e0);
    if (e1)
        cudaEventDestroy(e1);
    if (cyc)
        cudaFree(cyc);
    if (err)
        cudaFree(err);
    return rc;
}

}  // namespace sattn
