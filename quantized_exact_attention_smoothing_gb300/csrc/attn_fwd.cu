// attn_fwd.cu -- the attention pass over the INT8 / FP8 codes ("Experiment Log"
// page, entry "Phase 0 Import And Verification": QK traversal, online softmax,
// FP8 V/P, two-level PV accumulation, final conversion, ragged tails; entry
// "Phase 1 State-Ownership Decision": strict tile order, exact FP8 score bytes,
// per-tile RO rescaling, two-level PV accumulation, final conversion).
//
// One CTA computes 128 query rows of one (batch, query head) and visits the
// KV tiles of 256 keys in increasing order.  Twelve warps:
//   warps 0-7   two compute warpgroups, thread = query row = TMEM lane; half h
//               owns keys [128h, 128h + 128) of every tile and output channels
//               [64h, 64h + 64): score scaling, masks, running max m (exchanged
//               between the halves), alpha, the FP8 P bytes (written to shared
//               memory), then RO = RO * alpha + PV and d = d * alpha + sum p8
//               for the previous tile, and the final conversion
//   warp 8      TMA producer: K tiles (FP16 carrier of the INT8 codes) and V
//               half-tiles (E4M3, channel-major): one K stage (the next tile
//               loads while PV of the previous one runs) and a ring of four
//               V half-tile slots
//   warp 9      TMEM allocation and the single MMA-issuing thread:
//                 S_j  = Q * K_j^T   tcgen05 kind::f16, A = Q from TMEM, N = 256
//                 PV_j = P_j * V_j   tcgen05 kind::f8f6f4, A = P from shared
//                                    memory, N = 144: V rows plus a row of ones
//                                    whose column gives sum_j p8_j
//   warps 10-11 idle
// Twelve warps launch at 168 registers each; setmaxnreg then gives the compute
// warpgroups 232 (128 scores and 64 RO values per thread) and the
// producer/MMA warpgroup 40.
// Tensor memory (512 columns): S [0,256), PV partial [256,400), Q carrier
// [448,512).  P is double-buffered in shared memory, so the softmax of tile
// j + 1 never waits for PV of tile j.  A tcgen05.mma instruction costs about
// the same time for any N up to 256 on this part, hence the 256-key tiles: QK
// runs at N = 256.
//
// Exactness of QK: INT8 codes are carried as FP16 values (integers of
// magnitude <= 127 are exact in FP16); every product is an integer <= 16129 and
// every partial sum an integer below 2^21, so the FP32 accumulator holds the
// exact int32 dot product.
//
// Every mbarrier wait is bounded: after about a second, or as soon as another
// CTA has reported a failure, the thread records the failure in the status
// word, stops, waits for its own copies and MMAs in flight, and the CTA frees
// its TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>
#include <mutex>
#include <type_traits>

#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "sattn_internal.cuh"

namespace sattn {
namespace {

constexpr int BM = kQTile, BN = kKvTile, HD = kHeadDim;   // 128 rows x 256 keys
constexpr int KSTAGES = 1, VSLOTS = 4;
constexpr uint32_t K_HALF_BYTES = BN * 64 * 2;          // 256 keys x 64 channels, FP16
constexpr uint32_t K_STAGE_BYTES = 2 * K_HALF_BYTES;    // 64 KB
constexpr uint32_t PV_N = 144;                          // V rows + ones row + zero rows
constexpr uint32_t V_SLOT_BYTES = PV_N * 128;           // one 128-key half tile, 18 KB
constexpr uint32_t V_TMA_BYTES = HD * 128;              // 16 KB loaded per half tile
constexpr uint32_t P_HALF_BYTES = BM * 128;             // 128 rows x 128 keys, E4M3
constexpr uint32_t P_BUF_BYTES = 2 * P_HALF_BYTES;      // one tile's P (double-buffered)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;
constexpr uint32_t TM_PV = 256;
constexpr uint32_t TM_Q = 448;
// warp roles: 0-7 compute (two warpgroups), 8 TMA producer, 9 MMA issuer and
// TMEM owner, 10-11 idle
constexpr int WARP_PRODUCER = 8, WARP_MMA = 9;
constexpr int NTHREADS = 12 * 32;
// Registers: launched at 168 per thread (384 x 168 = 64512), then rebalanced
// per warpgroup; the shares add up to exactly the launch total.
constexpr int kLaunchRegs = 168, kRegsCompute = 232, kRegsOther = 40;
static_assert(2 * 128 * kRegsCompute + 128 * kRegsOther == NTHREADS * kLaunchRegs,
              "register split must add up to the launch total");
constexpr uint32_t IDESC_QK = ptx::make_idesc(0, 0, BM, BN);     // F16 x F16 -> F32, N = 256
constexpr uint32_t IDESC_PV = ptx::make_idesc(0, 0, BM, PV_N);   // E4M3 x E4M3 -> F32
constexpr uint64_t TIMEOUT_NS = 1000000000ull;

// shared memory map, offsets from a 1024-byte aligned base
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_V = OFF_K + KSTAGES * K_STAGE_BYTES;
constexpr uint32_t OFF_P = OFF_V + VSLOTS * V_SLOT_BYTES;
constexpr uint32_t OFF_MAXX = OFF_P + 2 * P_BUF_BYTES;      // [tile parity][half][row] row maxima
constexpr uint32_t OFF_BAR = OFF_MAXX + 4 * BM * 4;
enum Bar : int {
    KFULL = 0,
    KEMPTY = KFULL + KSTAGES,
    VFULL = KEMPTY + KSTAGES,
    VEMPTY = VFULL + VSLOTS,
    QFULL = VEMPTY + VSLOTS,
    SFULL = QFULL + 1,
    SFREE = SFULL + 1,
    PFULL = SFREE + 1,       // 2 (per P buffer)
    PDONE = PFULL + 2,       // 2 (per P buffer)
    PVFULL = PDONE + 2,
    PVEMPTY = PVFULL + 1,
    MMADONE = PVEMPTY + 1,
    NBARS = MMADONE + 1
};
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NBARS * 8;
constexpr uint32_t OFF_FLAG = OFF_TMEM_SLOT + 4;
constexpr uint32_t SMEM_BYTES = OFF_FLAG + 4 + 1024;   // + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_V % 1024 == 0 && V_SLOT_BYTES % 1024 == 0 && OFF_P % 1024 == 0,
              "swizzle atoms must be 1024-aligned");

// where a wait gave up (second status word)
enum Site : uint32_t {
    SITE_KE = 1, SITE_VE, SITE_Q, SITE_K, SITE_P, SITE_V, SITE_PVE, SITE_DONE, SITE_S,
    SITE_PV, SITE_DRAIN, SITE_SFREE, SITE_PDONE
};

struct FwdParams {
    const int8_t *q_codes;
    const float *q_scales, *k_scales, *v_scales;
    __nv_bfloat16 *out;
    uint32_t *status;
    int Hq, Hkv, Nq, Nkv, group, n_qtiles, causal;
    int nq32, nbq, nbk;
    float c0;
#ifdef SATTN_DEBUG_DUMP
    // intermediates of query tile 0 of (batch 0, head 0), KV tile 0:
    // [0, 32768) raw S accumulators (128 x 256), [32768, 40960) P8 words
    // (128 x 64), [40960, 40960 + 128 * 144) first PV partial; clock stamps
    // of one CTA from float offset 61440 (16 events x 256 tiles, 64-bit)
    float *dbg;
#endif
};

#ifdef SATTN_DEBUG_DUMP
// Debug builds only: SM clock stamps of one CTA (the first in launch order:
// the last query tile, batch 0, head 0), event `id` of KV tile `j`.
#define SATTN_TRACE(p, t, id, j)                                                                 \
    do {                                                                                         \
        if ((p).dbg && blockIdx.x == 0 && (t).hq == 0 && (t).b == 0 && (j) < 256)               \
            reinterpret_cast<unsigned long long *>((p).dbg + 61440)[(id) * 256 + (j)] = clock64(); \
    } while (0)
#else
#define SATTN_TRACE(p, t, id, j) \
    do {                         \
    } while (0)
#endif

struct Waiter {
    uint32_t *status;

    // Wait for the phase of parity `parity`; false if the wait ran out or the
    // kernel was aborted elsewhere.
    __device__ bool wait(uint32_t bar, uint32_t parity, uint32_t site) const
    {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        const uint64_t t0 = ptx::globaltimer();
        for (uint32_t it = 1;; ++it) {
            if (ptx::mbar_try_wait(bar, parity))
                return true;
            if ((it & 255u) == 0) {
                if (*reinterpret_cast<volatile uint32_t *>(status) != 0)
                    return false;
                if (ptx::globaltimer() - t0 > TIMEOUT_NS) {
                    atomicOr(status, 1u);
                    atomicCAS(status + 1, 0u, site);
                    return false;
                }
            }
        }
    }

    // Wait for copies or MMAs this thread issued; ignores the abort flag, still bounded.
    __device__ void drain(uint32_t bar, uint32_t parity) const
    {
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(bar, parity)) {
            if (ptx::globaltimer() - t0 > TIMEOUT_NS) {
                atomicOr(status, 1u);
                atomicCAS(status + 1, 0u, static_cast<uint32_t>(SITE_DRAIN));
                return;
            }
        }
    }
};

__device__ __forceinline__ uint32_t f16x2_of_i8(uint32_t word, int byte)
{
    const int lo = static_cast<int8_t>((word >> (8 * byte)) & 0xffu);
    const int hi = static_cast<int8_t>((word >> (8 * byte + 8)) & 0xffu);
    const __half2 h = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
    uint32_t u;
    memcpy(&u, &h, sizeof u);
    return u;
}

struct Tile {
    int b, hq, hk, q0, ntiles, mask_from;
};

__device__ __forceinline__ void producer_role(const FwdParams &p, const CUtensorMap *tm_k,
                                              const CUtensorMap *tm_v, uint32_t sb, const Tile &t, int bhk,
                                              const Waiter &wt)
{
    auto bar = [sb](int i) { return sb + OFF_BAR + 8u * i; };
    ptx::prefetch_tensormap(tm_k);
    ptx::prefetch_tensormap(tm_v);
    int issued_k = -1, issued_v = -1;
    bool ok = true;
    for (int j = 0; j < t.ntiles && ok; ++j) {
        const int ks = j % KSTAGES;
        if (!wt.wait(bar(KEMPTY + ks), ((j / KSTAGES) & 1) ^ 1, SITE_KE)) {
            ok = false;
            break;
        }
        const uint32_t kdst = sb + OFF_K + ks * K_STAGE_BYTES;
        ptx::mbar_arrive_expect_tx(bar(KFULL + ks), K_STAGE_BYTES);
        ptx::tma_load_3d(kdst, tm_k, bar(KFULL + ks), 0, j * BN, bhk);
        ptx::tma_load_3d(kdst + K_HALF_BYTES, tm_k, bar(KFULL + ks), 64, j * BN, bhk);
        SATTN_TRACE(p, t, 11, j);
        issued_k = j;
        for (int h = 0; h < 2; ++h) {
            const int u = 2 * j + h, vs = u % VSLOTS;
            if (!wt.wait(bar(VEMPTY + vs), ((u / VSLOTS) & 1) ^ 1, SITE_VE)) {
                ok = false;
                break;
            }
            ptx::mbar_arrive_expect_tx(bar(VFULL + vs), V_TMA_BYTES);
            ptx::tma_load_3d(sb + OFF_V + vs * V_SLOT_BYTES, tm_v, bar(VFULL + vs), j * BN + 128 * h, 0, bhk);
            issued_v = u;
        }
        SATTN_TRACE(p, t, 12, j);
    }
    if (!ok) {
        for (int j = max(0, issued_k - KSTAGES + 1); j <= issued_k; ++j)
            wt.drain(bar(KFULL + j % KSTAGES), (j / KSTAGES) & 1);
        for (int u = max(0, issued_v - VSLOTS + 1); u <= issued_v; ++u)
            wt.drain(bar(VFULL + u % VSLOTS), (u / VSLOTS) & 1);
    }
}

__device__ __forceinline__ void mma_role(const FwdParams &p, uint32_t sb, uint32_t tmem, const Tile &t,
                                         const Waiter &wt)
{
    auto bar = [sb](int i) { return sb + OFF_BAR + 8u * i; };
    if (wt.wait(bar(QFULL), 0, SITE_Q)) {
        ptx::tc_fence_after();
        for (int j = 0; j <= t.ntiles; ++j) {
            if (j < t.ntiles) {                     // S_j = Q K_j^T (256 keys)
                const int ks = j % KSTAGES;
                if (!wt.wait(bar(KFULL + ks), (j / KSTAGES) & 1, SITE_K))
                    break;
                if (j >= 1 && !wt.wait(bar(SFREE), (j - 1) & 1, SITE_SFREE))
                    break;
                ptx::tc_fence_after();
                SATTN_TRACE(p, t, 8, j);
                const uint32_t kb = sb + OFF_K + ks * K_STAGE_BYTES;
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    ptx::mma_f16_ts(tmem + TM_S, tmem + TM_Q + 8 * s,
                                    ptx::sw128_desc(kb + (s >> 2) * K_HALF_BYTES + (s & 3) * 32),
                                    IDESC_QK, s > 0);
                SATTN_TRACE(p, t, 9, j);
                ptx::mma_commit(bar(KEMPTY + ks));
                ptx::mma_commit(bar(SFULL));
                SATTN_TRACE(p, t, 4, j);
            }
            if (j >= 1) {                           // PV_{j-1} = P_{j-1} V_{j-1}
                const int jj = j - 1, pbuf = jj & 1;
                if (!wt.wait(bar(PFULL + pbuf), (jj >> 1) & 1, SITE_P))
                    break;
                if (!wt.wait(bar(PVEMPTY), (jj & 1) ^ 1, SITE_PVE))
                    break;
                bool ok = true;
                for (int h = 0; h < 2 && ok; ++h) {
                    const int u = 2 * jj + h, vs = u % VSLOTS;
                    if (!wt.wait(bar(VFULL + vs), (u / VSLOTS) & 1, SITE_V)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (h == 0)
                        SATTN_TRACE(p, t, 5, jj);
                    const uint32_t vb = sb + OFF_V + vs * V_SLOT_BYTES;
                    const uint32_t pb = sb + OFF_P + pbuf * P_BUF_BYTES + h * P_HALF_BYTES;
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        ptx::mma_f8_ss(tmem + TM_PV, ptx::sw128_desc(pb + s * 32), ptx::sw128_desc(vb + s * 32),
                                       IDESC_PV, (h | s) != 0);
                    ptx::mma_commit(bar(VEMPTY + vs));
                }
                if (!ok)
                    break;
                SATTN_TRACE(p, t, 10, jj);
                ptx::mma_commit(bar(PVFULL));
                ptx::mma_commit(bar(PDONE + pbuf));
            }
        }
    }
    // every MMA of this CTA has finished before the TMEM is released
    ptx::mma_commit(bar(MMADONE));
    wt.drain(bar(MMADONE), 0);
}

// Compute warpgroups.  Half h owns S columns [128h, 128h + 128) of every tile
// and writes the P8 bytes of those keys into shared-memory half h (K-major,
// 128-byte swizzle); the row max is exchanged through shared memory under a
// named barrier, so both halves hold the same running max m and alpha.  Half
// h also owns RO columns [64h, 64h + 64): after writing P_j it folds the
// partial PV_{j-1} into RO with alpha_{j-1} (both halves keep d).
__device__ __forceinline__ void compute_role(const FwdParams &p, uint32_t sb, uint8_t *smem,
                                             uint32_t tmem, int warp, int lane, const Tile &t,
                                             const Waiter &wt)
{
    auto bar = [sb](int i) { return sb + OFF_BAR + 8u * i; };
    const int half = warp >> 2;                               // 0 or 1
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                        // query row in the tile = TMEM lane
    const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int i = t.q0 + r;

    // Q codes 64h .. 64h+63 of row i -> FP16 carrier -> TMEM columns [TM_Q + 32h, TM_Q + 32h + 32)
    {
        uint32_t h[32];
        if (i < p.nq32) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                p.q_codes + (static_cast<size_t>(t.b * p.Hq + t.hq) * p.nq32 + i) * HD + 64 * half);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint4 a = src[w];
                const uint32_t words[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    h[w * 8 + e * 2] = f16x2_of_i8(words[e], 0);
                    h[w * 8 + e * 2 + 1] = f16x2_of_i8(words[e], 2);
                }
            }
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c)
                h[c] = 0u;
        }
        ptx::tmem_st32(taddr + TM_Q + 32 * half, h);
        ptx::tmem_wait_st();
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(bar(QFULL));

    const float sq = (i < p.nq32) ? p.q_scales[static_cast<size_t>(t.b * p.Hq + t.hq) * p.nbq + i / kQBlock]
                                  : 0.0f;
    const int lim = p.causal ? i + (p.Nkv - p.Nq) : 0x7fffffff;   // last kept key of row i
    const float *ksc = p.k_scales + static_cast<size_t>(t.b * p.Hkv + t.hk) * p.nbk;
    float *maxx = reinterpret_cast<float *>(smem + OFF_MAXX);
    uint8_t *prow0 = smem + OFF_P + half * P_HALF_BYTES + r * 128;  // this row's 128 P8 bytes (buffer 0)
    constexpr float kLog2_448 = 8.8073549220576041f;          // log2(448): P is stored as p * 448
    float m = -INFINITY;
    float ro[64];
#pragma unroll
    for (int c = 0; c < 64; ++c)
        ro[c] = 0.0f;
    float d = 0.0f, alpha_prev = 0.0f;

    // RO = RO * alpha + PV partial of tile jj (this half's 64 channels), d likewise
    auto fold_partial = [&](int jj, float alpha) -> bool {
        if (!wt.wait(bar(PVFULL), jj & 1, SITE_PV))
            return false;
        ptx::tc_fence_after();
        if (r == 0 && half == 0)
            SATTN_TRACE(p, t, 6, jj);
#ifdef SATTN_DEBUG_DUMP
        if (p.dbg && jj == 0 && t.q0 == 0 && t.hq == 0 && t.b == 0 && half == 0) {
            for (int c = 0; c < static_cast<int>(PV_N); ++c) {
                uint32_t x;
                ptx::tmem_ld1(taddr + TM_PV + c, x);
                ptx::tmem_wait_ld();
                p.dbg[40960 + r * PV_N + c] = __uint_as_float(x);
            }
        }
#endif
        uint32_t part[2][32], ds;
        ptx::tmem_ld32(taddr + TM_PV + 64 * half, part[0]);
        ptx::tmem_ld32(taddr + TM_PV + 64 * half + 32, part[1]);
        ptx::tmem_ld1(taddr + TM_PV + 128, ds);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(PVEMPTY));                        // the partial buffer may be reused
#pragma unroll
        for (int c = 0; c < 64; ++c)
            ro[c] = fmaf(ro[c], alpha, __uint_as_float(part[c >> 5][c & 31]));
        d = fmaf(d, alpha, __uint_as_float(ds));
        if (r == 0 && half == 0)
            SATTN_TRACE(p, t, 7, jj);
        return true;
    };

    // block scales of this half's four 32-key blocks, one tile ahead
    auto kscale = [&](int j, int c) {
        const int kb = j * (BN / kQBlock) + 4 * half + c;
        return kb < p.nbk ? ksc[kb] : 0.0f;
    };
    float sk[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        sk[c] = kscale(0, c);

    for (int j = 0; j < t.ntiles; ++j) {
        float sig[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            sig[c] = __fmul_rn(__fmul_rn(sq, sk[c]), p.c0);
            sk[c] = kscale(j + 1, c);
        }
        if (!wt.wait(bar(SFULL), j & 1, SITE_S))
            return;
        ptx::tc_fence_after();
        if (r == 0 && half == 0)
            SATTN_TRACE(p, t, 0, j);
        uint32_t s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c)
            ptx::tmem_ld32(taddr + TM_S + static_cast<uint32_t>(128 * half + 32 * c), s[c]);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(SFREE));                          // S may be overwritten now
        if (r == 0 && half == 0)
            SATTN_TRACE(p, t, 1, j);
#ifdef SATTN_DEBUG_DUMP
        if (p.dbg && j == 0 && t.q0 == 0 && t.hq == 0 && t.b == 0)
            for (int k = 0; k < 128; ++k)
                p.dbg[r * BN + 128 * half + k] = __uint_as_float(s[k >> 5][k & 31]);
#endif
        // keys of this half that row i keeps: the first `nvalid` (the mask is a
        // suffix of the half-tile: keys >= Nkv and, if causal, keys > lim)
        const bool masked = j >= t.mask_from;
        int nvalid = 128;
        if (masked) {
            const int lo = j * BN + 128 * half;
            nvalid = max(0, min(128, min(p.Nkv - 1, lim) - lo + 1));
        }
        // max of the raw accumulators per 32-key block: the block scale is
        // positive (or zero), so fl(max(acc) * sig) = max(fl(acc * sig)) exactly
        float tmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float b;
            if (!masked) {
                // eight independent three-input max chains, then a short tree
                float q[8];
#pragma unroll
                for (int a = 0; a < 8; ++a)
                    q[a] = ptx::fmax3(__uint_as_float(s[c][a]), __uint_as_float(s[c][a + 8]),
                                      __uint_as_float(s[c][a + 16]));
#pragma unroll
                for (int a = 0; a < 8; ++a)
                    q[a] = fmaxf(q[a], __uint_as_float(s[c][a + 24]));
                b = fmaxf(ptx::fmax3(q[0], q[1], q[2]), ptx::fmax3(q[3], q[4], q[5]));
                b = ptx::fmax3(b, q[6], q[7]);
            } else {
                float q[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    q[k & 3] = fmaxf(q[k & 3], 32 * c + k < nvalid ? __uint_as_float(s[c][k]) : -INFINITY);
                b = fmaxf(fmaxf(q[0], q[1]), fmaxf(q[2], q[3]));
            }
            tmax = fmaxf(tmax, (b == -INFINITY) ? -INFINITY : __fmul_rn(b, sig[c]));
        }
        // exchange the half-row maxima (double-buffered by tile parity)
        maxx[((j & 1) * 2 + half) * BM + r] = tmax;
        ptx::named_bar_sync(1, 2 * BM);
        tmax = fmaxf(tmax, maxx[((j & 1) * 2 + (half ^ 1)) * BM + r]);
        if (r == 0 && half == 0)
            SATTN_TRACE(p, t, 2, j);

        const float mn = fmaxf(m, tmax);
        const float alpha = (m == -INFINITY) ? 0.0f : ptx::ex2_approx(__fsub_rn(m, mn));
        const float nb = kLog2_448 - mn;                     // exponent offset of p * 448

        // P buffer j % 2 is free once PV_{j-2} has read it
        const int pbuf = j & 1;
        uint8_t *prow = prow0 + pbuf * P_BUF_BYTES;
        if (j >= 2 && !wt.wait(bar(PDONE + pbuf), ((j >> 1) - 1) & 1, SITE_PDONE))
            return;
        // P8 = E4M3(exp2(acc * sig - m') * 448), four keys per 32-bit word,
        // stored 32 keys at a time (16-byte chunk c of the row lands at chunk
        // c ^ (row % 8): the 128-byte swizzle of the K-major operand).  The
        // masked and unmasked forms are separate copies so that the common,
        // unmasked tiles carry no per-key select.
        auto write_p = [&](auto masked_tag) {
            constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[8];
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    float e[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int k = 4 * w + u;
                        float x = fmaf(__uint_as_float(s[c][k]), sig[c], nb);
                        if (kMasked)
                            x = (32 * c + k < nvalid) ? x : -INFINITY;
                        e[u] = ptx::ex2_approx(x);
                    }
                    pk[w] = ptx::cvt_e4m3x4(e[0], e[1], e[2], e[3]);
                }
#ifdef SATTN_DEBUG_DUMP
                if (p.dbg && j == 0 && t.q0 == 0 && t.hq == 0 && t.b == 0)
                    for (int w = 0; w < 8; ++w)
                        p.dbg[32768 + r * 64 + 32 * half + 8 * c + w] = __uint_as_float(pk[w]);
#endif
                *reinterpret_cast<uint4 *>(prow + (((2 * c) ^ (r & 7)) << 4)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4 *>(prow + (((2 * c + 1) ^ (r & 7)) << 4)) =
                    make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
        };
        if (masked)
            write_p(std::true_type{});
        else
            write_p(std::false_type{});
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(bar(PFULL + pbuf));
        if (r == 0 && half == 0)
            SATTN_TRACE(p, t, 3, j);
        if (j >= 1 && !fold_partial(j - 1, alpha_prev))
            return;
        alpha_prev = alpha;
        m = mn;
    }
    if (t.ntiles > 0 && !fold_partial(t.ntiles - 1, alpha_prev))
        return;

    // final conversion: reciprocal of d, per-channel V scale, BF16
    if (i < p.Nq) {
        const float rcp = d > 0.0f ? __frcp_rn(d) : 0.0f;
        const float *sv = p.v_scales + static_cast<size_t>(t.b * p.Hkv + t.hk) * HD + 64 * half;
        uint4 *dst = reinterpret_cast<uint4 *>(p.out + (static_cast<size_t>(t.b * p.Hq + t.hq) * p.Nq + i) * HD +
                                               64 * half);
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            uint32_t u[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = 8 * w + 2 * e;
                const float o0 = __fmul_rn(__fmul_rn(ro[c], rcp), sv[c]);
                const float o1 = __fmul_rn(__fmul_rn(ro[c + 1], rcp), sv[c + 1]);
                const __nv_bfloat162 pr = __floats2bfloat162_rn(o0, o1);
                memcpy(&u[e], &pr, sizeof(uint32_t));
            }
            dst[w] = make_uint4(u[0], u[1], u[2], u[3]);
        }
    }
}

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const FwdParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sb = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    Tile t;
    const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x);   // longest rows first
    t.hq = blockIdx.y;
    t.b = blockIdx.z;
    t.hk = t.hq / p.group;
    t.q0 = qt * BM;
    const int off = p.Nkv - p.Nq;
    int kv_end = p.Nkv;
    if (p.causal)
        kv_end = min(p.Nkv, min(t.q0 + BM, p.Nq) + off);
    t.ntiles = (kv_end + BN - 1) / BN;
    t.mask_from = p.Nkv / BN;                                  // tiles holding keys >= Nkv
    if (p.causal)
        t.mask_from = min(t.mask_from, (t.q0 + off + 1) / BN); // tiles crossing row q0's diagonal
    const Waiter wt{p.status};
    volatile uint32_t *flag = reinterpret_cast<volatile uint32_t *>(smem + OFF_FLAG);

    if (threadIdx.x == 0) {
        *flag = *reinterpret_cast<volatile uint32_t *>(p.status);
        const uint32_t b0 = sb + OFF_BAR;
        for (int s = 0; s < KSTAGES; ++s) {
            ptx::mbar_init(b0 + 8u * (KFULL + s), 1);
            ptx::mbar_init(b0 + 8u * (KEMPTY + s), 1);
        }
        for (int s = 0; s < VSLOTS; ++s) {
            ptx::mbar_init(b0 + 8u * (VFULL + s), 1);
            ptx::mbar_init(b0 + 8u * (VEMPTY + s), 1);
        }
        ptx::mbar_init(b0 + 8u * QFULL, 2 * BM);
        ptx::mbar_init(b0 + 8u * SFULL, 1);
        ptx::mbar_init(b0 + 8u * SFREE, 2 * BM);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(b0 + 8u * (PFULL + s), 2 * BM);
            ptx::mbar_init(b0 + 8u * (PDONE + s), 1);
        }
        ptx::mbar_init(b0 + 8u * PVFULL, 1);
        ptx::mbar_init(b0 + 8u * PVEMPTY, 2 * BM);
        ptx::mbar_init(b0 + 8u * MMADONE, 1);
        ptx::fence_mbar_init();
    }
    // constant rows of every V slot: row 128 holds E4M3 1.0 (0x38), rows 129..143 hold 0
    for (int idx = threadIdx.x; idx < VSLOTS * 16 * 8; idx += NTHREADS) {
        const int st = idx / 128, w = idx % 128, row = 128 + w / 8, ch = w % 8;
        const uint32_t val = (row == 128) ? 0x38383838u : 0u;
        *reinterpret_cast<uint4 *>(smem + OFF_V + st * V_SLOT_BYTES + row * 128 + ch * 16) =
            make_uint4(val, val, val, val);
    }
    ptx::fence_proxy_async_smem();
    if (warp == WARP_MMA) {
        ptx::tmem_alloc(sb + OFF_TMEM_SLOT, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + OFF_TMEM_SLOT);

    if (*flag == 0) {
        if (warp < WARP_PRODUCER) {
            ptx::setmaxnreg_inc<kRegsCompute>();
            compute_role(p, sb, smem, tmem, warp, lane, t, wt);
        } else {
            ptx::setmaxnreg_dec<kRegsOther>();
            if (warp == WARP_PRODUCER) {
                if (lane == 0)
                    producer_role(p, &tm_k, &tm_v, sb, t, t.b * p.Hkv + t.hk, wt);
            } else if (warp == WARP_MMA) {
                if (lane == 0)
                    mma_role(p, sb, tmem, t, wt);
            }
            __syncwarp();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// INT8 K codes -> FP16 carrier [B*Hkv][Nkv][128]; also clears the status words.
__global__ void __launch_bounds__(256) widen_k_kernel(const int8_t *__restrict__ k_codes, int Nkv,
                                                      int64_t nk32, int64_t n8,
                                                      __half *__restrict__ carrier,
                                                      uint32_t *__restrict__ status)
{
    if (blockIdx.x == 0 && threadIdx.x < 2)
        status[threadIdx.x] = 0u;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n8;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = idx >> 4;
        const int g = static_cast<int>(idx & 15);
        const int64_t bh = row / Nkv, tok = row % Nkv;
        const uint2 c = *reinterpret_cast<const uint2 *>(k_codes + (bh * nk32 + tok) * HD + g * 8);
        const uint4 o = make_uint4(f16x2_of_i8(c.x, 0), f16x2_of_i8(c.x, 2), f16x2_of_i8(c.y, 0),
                                   f16x2_of_i8(c.y, 2));
        *reinterpret_cast<uint4 *>(carrier + row * HD + g * 8) = o;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

}  // namespace

#ifdef SATTN_DEBUG_DUMP
static float *g_debug_dump = nullptr;
float *debug_dump_buffer() { return g_debug_dump; }
extern "C" void sattn_debug_set_dump(float *p) { g_debug_dump = p; }
#endif

size_t forward_workspace_bytes(const Geometry &g)
{
    return kStatusBytes + static_cast<size_t>(g.B) * g.Hkv * g.Nkv * HD * sizeof(__half);
}

int launch_forward(const Geometry &g, const int8_t *q_codes, const float *q_scales,
                   const int8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                   const float *v_scales, void *out, void *workspace, cudaStream_t stream)
{
    auto encode = tensor_map_encoder();
    if (!encode)
        return 1;
    uint32_t *status = static_cast<uint32_t *>(workspace);
    __half *carrier = reinterpret_cast<__half *>(static_cast<char *>(workspace) + kStatusBytes);
    const int bhk = g.B * g.Hkv;

    const int64_t n8 = static_cast<int64_t>(bhk) * g.Nkv * (HD / 8);
    const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, 152 * 8);
    widen_k_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(k_codes, g.Nkv, g.nk32, n8,
                                                                       carrier, status);

    CUtensorMap tmk, tmv;
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(g.Nkv),
                                    static_cast<cuuint64_t>(bhk)};
        const cuuint64_t strides[2] = {HD * sizeof(__half), static_cast<cuuint64_t>(g.Nkv) * HD * sizeof(__half)};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BN), 1};   // 256 keys x 64 channels
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tmk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, carrier, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return 1;
    }
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.Nkv), static_cast<cuuint64_t>(HD),
                                    static_cast<cuuint64_t>(bhk)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(g.nk128),
                                       static_cast<cuuint64_t>(g.nk128) * HD};
        const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(HD), 1};   // 128 keys x 128 channels
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tmv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(v_codes), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return 1;
    }

    // The per-warpgroup register split only adds up when the kernel is launched
    // with exactly kLaunchRegs registers per thread; refuse to launch otherwise.
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        cudaFuncAttributes fa;
        attr_err = cudaFuncGetAttributes(&fa, attn_fwd_kernel);
        if (attr_err == cudaSuccess && fa.numRegs != kLaunchRegs)
            attr_err = cudaErrorInvalidConfiguration;
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(SMEM_BYTES));
    });
    if (attr_err != cudaSuccess)
        return static_cast<int>(attr_err);

    FwdParams prm;
    prm.q_codes = q_codes;
    prm.q_scales = q_scales;
    prm.k_scales = k_scales;
    prm.v_scales = v_scales;
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.status = status;
    prm.Hq = g.Hq;
    prm.Hkv = g.Hkv;
    prm.Nq = g.Nq;
    prm.Nkv = g.Nkv;
    prm.group = g.Hq / g.Hkv;
    prm.n_qtiles = static_cast<int>((g.Nq + BM - 1) / BM);
    prm.causal = g.causal;
    prm.nq32 = static_cast<int>(g.nq32);
    prm.nbq = static_cast<int>(g.nbq);
    prm.nbk = static_cast<int>(g.nbk);
    const float sm = g.sm_scale > 0.0f ? g.sm_scale : 1.0f / sqrtf(static_cast<float>(HD));
    prm.c0 = sm * 1.44269504088896340736f;
#ifdef SATTN_DEBUG_DUMP
    prm.dbg = debug_dump_buffer();
#endif

    attn_fwd_kernel<<<dim3(prm.n_qtiles, g.Hq, g.B), NTHREADS, SMEM_BYTES, stream>>>(tmk, tmv, prm);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace sattn
