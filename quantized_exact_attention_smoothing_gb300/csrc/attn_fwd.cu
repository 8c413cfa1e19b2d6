// attn_fwd.cu -- the attention pass over the INT8 / FP8 codes ("Experiment Log"
// page, entry "Phase 0 Import And Verification": QK traversal, online softmax,
// FP8 V/P, two-level PV accumulation, final conversion, ragged tails; entry
// "Phase 1 State-Ownership Decision": strict tile order, exact FP8 score bytes,
// per-tile RO rescaling, two-level PV accumulation, final conversion).
//
// Persistent: one CTA per SM walks work items (128 query rows of one batch and
// query head), the longest of each L2 chunk first, taking each next item from
// a counter shared by the CTAs as it frees up (cta_item); each item visits its
// KV tiles of 256 keys in increasing order.  Twelve warps:
//   warps 0-7   two compute warpgroups, thread = query row = TMEM lane; half h
//               owns keys [128h, 128h + 128) of every tile and output channels
//               [64h, 64h + 64): score scaling, masks, running max m (exchanged
//               between the halves), alpha, the FP8 P bytes (written to TMEM),
//               RO = RO * alpha + PV and d = d * alpha + sum p8 for the
//               previous tile, and the final conversion (each warp's 32 x 64
//               BF16 tile staged in shared memory, then one TMA store)
//   warp 8      K loader (TMA): K half-tiles (FP16 carrier of the INT8 codes,
//               256 keys x 64 channels) into a ring of three slots
//   warp 9      TMEM allocation and the single MMA-issuing thread:
//                 S_j  = Q * K_j^T   tcgen05 kind::f16, A = Q from shared
//                                    memory, N = 256
//                 PV_j = P_j * V_j   tcgen05 kind::f8f6f4, A = P from TMEM,
//                                    N = 144: V rows plus a row of ones whose
//                                    column gives sum_j p8_j
//   warp 10     V and Q loader (TMA): V half-tiles (E4M3, channel-major) into
//               two slots; the next item's INT8 Q tile and V channel scales
//   warp 11     Q converter: the staged INT8 Q tile of the next item -> its
//               FP16 carrier in shared memory, as soon as the current item's
//               last QK has completed (with kFuseQ it also quantises each
//               item's BF16 Q tile itself, staged in the output buffer)
// Twelve warps launch at 168 registers each; setmaxnreg then gives the compute
// warpgroups 232 (128 scores and 64 RO values per thread) and the loader/MMA
// warpgroup 40.
// Tensor memory (512 columns): S [0,256), PV partial [256,400), P8 [448,512)
// (four E4M3 codes per column).  Writing P with tcgen05.st keeps it off the
// shared-memory pipe and needs no async-proxy fence; P_j may be written once
// PV_{j-1} has completed, which in steady state is long before the softmax of
// tile j reaches it.  A tcgen05.mma instruction costs about
// the same time for any N up to 256 on this part, hence the 256-key tiles: QK
// runs at N = 256.  The K ring of half-tile slots lets the next tile's K land
// while the current QK runs; a single full-tile K stage put the whole TMA
// latency of every tile on the critical path.
//
// Exactness of QK: INT8 codes are carried as FP16 values (integers of
// magnitude <= 127 are exact in FP16); every product is an integer <= 16129 and
// every partial sum an integer below 2^21, so the FP32 accumulator holds the
// exact int32 dot product.
//
// Exactness of P: the FP8 byte of a key is E4M3(fl(fl(2^dd) * 448)) with
// dd = fl(fl(acc * sig) - m), s2 and dd rounded exactly as stated (packed FP32
// pairs), and 2^dd from ex2.approx, whose relative error is below 2^-22.7 over
// the range used (measured for every FP32 input; the PTX ISA states 2^-22).
// The byte is taken from y+ = fl(2^dd * 448 * (1 + 2^-21)) and
// y- = fl(2^dd * 448 * (1 - 2^-21)).  With the approximation error, the
// rounding of fl(2^dd) and of both products (2^-24 each), the exact
// fl(fl(2^dd) * 448) lies in [y-, y+] for any approximation error up to
// 2^-22: 2^-21 > 2^-22 + 3 * 2^-24.  Rounding to E4M3 is monotonic, so when
// both give the same byte that is the byte.  Otherwise (within about 2^-21 of
// an E4M3 rounding midpoint, about 1.5e-5 of the keys) the byte is recomputed
// with a correctly rounded exp2, after the tile's P pass (see the compute
// warpgroups).
//
// Every mbarrier wait is bounded: after about a second, or as soon as another
// CTA has reported a failure, the thread records the failure in the status
// word, stops, waits for its own copies and MMAs in flight, and the CTA frees
// its TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>
#include <cstring>
#include <functional>
#include <mutex>
#include <queue>
#include <type_traits>
#include <vector>

#include <cudaTypedefs.h>

#include "prep_device.cuh"
#include "ptx.cuh"
#include "quant.cuh"
#include "sattn_internal.cuh"

namespace sattn {
namespace {

constexpr int BM = kQTile, BN = kKvTile, HD = kHeadDim;   // 128 rows x 256 keys
constexpr int KSLOTS = 3, VSLOTS = 2;                  // K half-tile slots, V half-tile slots
constexpr uint32_t K_HALF_BYTES = BN * 64 * 2;          // 256 keys x 64 channels, FP16
constexpr uint32_t PV_N = 144;                          // V rows + ones row + zero rows
constexpr uint32_t V_SLOT_BYTES = PV_N * 128;           // one 128-key half tile, 18 KB
constexpr uint32_t V_TMA_BYTES = HD * 128;              // 16 KB loaded per half tile
constexpr uint32_t Q_HALF_BYTES = BM * 128;             // 128 rows x 64 channels, FP16
constexpr uint32_t STG_BYTES = BM * HD * 2;             // output tile, BF16
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;
constexpr uint32_t TM_PV = 256;
constexpr uint32_t TM_P = 448;   // P8 of one tile: 256 keys, four per column
// warp roles: 0-7 compute (two warpgroups), 8 K loader, 9 MMA issuer and TMEM
// owner, 10 V and Q loader, 11 Q converter
constexpr int WARP_PRODUCER = 8, WARP_MMA = 9, WARP_VLOAD = 10, WARP_QCONV = 11;
constexpr int NTHREADS = 12 * 32;
// Registers: launched at 168 per thread (384 x 168 = 64512), then rebalanced
// per warpgroup; the shares add up to exactly the launch total.
constexpr int kLaunchRegs = 168, kRegsCompute = 232, kRegsOther = 40;
static_assert(2 * 128 * kRegsCompute + 128 * kRegsOther == NTHREADS * kLaunchRegs,
              "register split must add up to the launch total");
constexpr uint32_t IDESC_QK = ptx::make_idesc(0, 0, BM, BN);     // F16 x F16 -> F32, N = 256
constexpr uint32_t IDESC_PV = ptx::make_idesc(0, 0, BM, PV_N);   // E4M3 x E4M3 -> F32
constexpr uint64_t TIMEOUT_NS = 1000000000ull;
// K and V bytes of the heads whose items run together (see item_tile): well
// inside the 126 MB L2, which also carries the Q tiles and the output.
constexpr int64_t kL2ChunkBytes = 48ll << 20;

// shared memory map, offsets from a 1024-byte aligned base
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_V = OFF_K + KSLOTS * K_HALF_BYTES;
constexpr uint32_t OFF_Q = OFF_V + VSLOTS * V_SLOT_BYTES;   // FP16 carrier of Q, two 64-channel halves (128B swizzle)
constexpr uint32_t OFF_STG = OFF_Q + 2 * Q_HALF_BYTES;      // output staging of the final conversion
constexpr uint32_t OFF_QS = OFF_STG + STG_BYTES;            // INT8 Q tile of the next item (TMA, 128B swizzle)
constexpr uint32_t QS_BYTES = BM * HD;
constexpr uint32_t OFF_MAXX = OFF_QS + QS_BYTES;             // [tile parity][half][row] row maxima
constexpr uint32_t OFF_SV = OFF_MAXX + 4 * BM * 4;          // [item % 3][128] V channel scales
constexpr uint32_t SV_BYTES = HD * 4;
constexpr uint32_t OFF_SQ = OFF_SV + 3 * SV_BYTES;          // [item % 2][4] Q block scales (in-kernel Q quantisation)
constexpr uint32_t OFF_PARK = OFF_SQ + 2 * 4 * 4;         // [half][row] 16 bytes: exponent arguments of an undecided P8 word
constexpr uint32_t OFF_BAR = OFF_PARK + 2 * BM * 16;
constexpr int kItemSlots = 4;   // ring of the CTA's next item indices (see cta_item)
enum Bar : int {
    KFULL = 0,
    KEMPTY = KFULL + KSLOTS,
    VFULL = KEMPTY + KSLOTS,
    VEMPTY = VFULL + VSLOTS,
    QSTAGE = VEMPTY + VSLOTS,   // INT8 Q codes of an item landed in shared memory
    QFULL = QSTAGE + 1,         // its FP16 carrier is in shared memory
    QEMPTY = QFULL + 1,         // the item's last QK has completed: the Q carrier may be replaced
    SFULL = QEMPTY + 1,
    SFREE = SFULL + 1,
    PFULL = SFREE + 1,
    PDONE = PFULL + 1,
    PVFULL = PDONE + 1,
    PVEMPTY = PVFULL + 1,
    MMADONE = PVEMPTY + 1,
    QBF = MMADONE + 1,          // in-kernel Q quantisation: the BF16 Q tile landed in the staging buffer
    QQDONE = QBF + 1,           // its codes and block scales are written; the staging buffer is free
    STGFREE = QQDONE + 1,       // an item's final conversion has left the staging buffer
    ITEMFULL = STGFREE + 1,     // kItemSlots barriers: an item index was written into its ring slot
    NBARS = ITEMFULL + kItemSlots
};
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NBARS * 8;
constexpr uint32_t OFF_FLAG = OFF_TMEM_SLOT + 4;
constexpr uint32_t OFF_ABORT = OFF_FLAG + 4;          // set by a compute warp that gave up
// ring of this CTA's next item indices (see cta_item)
constexpr uint32_t OFF_ITEMS = OFF_ABORT + 4;
constexpr uint32_t SMEM_BYTES = OFF_ITEMS + 4 * kItemSlots + 1024;   // + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_V % 1024 == 0 && V_SLOT_BYTES % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_QS % 1024 == 0,
              "swizzle atoms must be 1024-aligned");

// where a wait gave up (second status word)
enum Site : uint32_t {
    SITE_KE = 1, SITE_VE, SITE_Q, SITE_K, SITE_P, SITE_V, SITE_PVE, SITE_DONE, SITE_S,
    SITE_PV, SITE_DRAIN, SITE_SFREE, SITE_PDONE, SITE_QS, SITE_QE, SITE_QEMPTY, SITE_QBF, SITE_QQ, SITE_STG,
    SITE_ITEM
};

struct FwdParams {
    const int8_t *q_codes;           // prepared INT8 Q [B*Hq][nq32][128] (null with in-kernel Q quantisation)
    const __nv_bfloat16 *q_bf16;     // in-kernel Q quantisation: the BF16 Q [B*Hq][Nq][128]
    const uint4 *k_carrier;          // FP16 carrier of the K codes [B*Hkv][Nkv][128]
    const float *q_scales, *k_scales, *v_scales;
    __nv_bfloat16 *out;
    uint32_t *status;
    int B, Hq, Hkv, Nq, Nkv, group, n_qtiles, n_items, causal;
    int withhold_v;   // test hook: the V loader stages the first Q tile and loads no V
    // item order (see item_tile): B * Hkv units, chunk_units per chunk,
    // chunk_items = chunk_units * group * n_qtiles items per full chunk
    int n_units, chunk_units, chunk_items;
    // reciprocals for exact division (see udiv) by chunk_items, by the items of
    // one query tile in a full chunk and in the last chunk, by Hkv and by group
    unsigned long long m_chunk, m_row, m_row_tail, m_hkv, m_group;
    int nq32, nbq, nbk;
    float c0;
    float zero;   // always +0 (see dd_pair)
    int small;    // the single-launch small-shape path: prepare `sp` first (small_prepare)
    SmallPrep sp;
    uint32_t *ticket;   // the item counter of this launch (one word of the status block, zero at launch)
#ifdef SATTN_DEBUG_DUMP
    // intermediates of query tile 0 of (batch 0, head 0), KV tile 0:
    // [0, 32768) raw S accumulators (128 x 256), [32768, 40960) P8 words
    // (128 x 64), [40960, 40960 + 128 * 144) first PV partial; clock stamps
    // of one CTA from float offset 61440 (16 events x 256 tiles, 64-bit)
    float *dbg;
#endif
};

#ifdef SATTN_DEBUG_DUMP
// Debug dump: KV tile 0 of query tile 0 of (batch 0, head 0) as described in
// FwdParams; the state after KV tile 1 of the same item (running maximum,
// alpha, d after the outer update, [128] each, and RO after it [128][128]);
// d and its reciprocal at the end of the item [128] each.
constexpr int DBG_M1 = 83000, DBG_A1 = 83128, DBG_D1 = 83256, DBG_RO1 = 83384, DBG_DF = 99768, DBG_RCP = 99896;
// Debug builds only: SM clock stamps of one CTA (the first in launch order:
// the last query tile, batch 0, head 0), event `id` of KV tile `j`.
#define SATTN_TRACE(p, t, id, j)                                                                 \
    do {                                                                                         \
        if ((p).dbg && (t).trace && (t).g0 + (j) < 256)                                         \
            reinterpret_cast<unsigned long long *>((p).dbg + 61440)[(id) * 256 + (t).g0 + (j)] =  \
                clock64();                                                                       \
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

struct Tile {
    int b, hq, hk, q0, ntiles, mask_from;
    bool trace;   // debug builds: clock stamps of this CTA's items are recorded
    int g0;       // debug builds: index of the item's first KV tile among the CTA's tiles
};

// floor(x / d) for 0 <= x < 2^31 and 1 <= d < 2^31, with m = floor((2^64 - 1) / d) + 1
// (m = 0 for d = 1): x * m / 2^64 exceeds x / d by less than 2^-33, and the
// fractional part of x / d is at most 1 - 1/d < 1 - 2^-31, so the floor is
// exact.  A multiply-high replaces the reciprocal-based integer division,
// whose reciprocal would queue behind the softmax exponentials.
__device__ __forceinline__ int udiv(int x, int d, unsigned long long m)
{
    return d == 1 ? x : static_cast<int>(__umul64hi(static_cast<unsigned long long>(x), m));
}

// Work item `it` of [0, n_items).  The (batch, KV head) units are cut into
// chunks of chunk_units consecutive units whose K and V fit in L2 together,
// and the chunks are walked in order, so that the CTAs running at the same
// time read the K and V tiles of a few heads, which then come from L2 after
// the first read.  Within a chunk: query tiles in decreasing order (with a
// causal mask the last rows visit the most KV tiles, so the longest items are
// scheduled first), then the chunk's units, then the query heads of a unit's
// GQA group.  Every item has at least one KV tile: a causal mask requires
// Nq <= Nkv, so each row keeps key 0.
__device__ __forceinline__ Tile item_tile(const FwdParams &p, int it)
{
    Tile t;
    const int c = udiv(it, p.chunk_items, p.m_chunk);
    const int r = it - c * p.chunk_items;
    const int u0 = c * p.chunk_units;
    const bool tail = u0 + p.chunk_units > p.n_units;   // the last chunk may hold fewer units
    const int row = (tail ? p.n_units - u0 : p.chunk_units) * p.group;   // items per query tile
    const int qi = udiv(r, row, tail ? p.m_row_tail : p.m_row);
    const int qt = p.n_qtiles - 1 - qi;
    const int rem = r - qi * row;
    const int ul = udiv(rem, p.group, p.m_group);
    const int u = u0 + ul;
    t.b = udiv(u, p.Hkv, p.m_hkv);
    t.hk = u - t.b * p.Hkv;
    t.hq = t.hk * p.group + (rem - ul * p.group);
    t.q0 = qt * BM;
    const int off = p.Nkv - p.Nq;
    int kv_end = p.Nkv;
    if (p.causal)
        kv_end = min(p.Nkv, min(t.q0 + BM, p.Nq) + off);
    t.ntiles = (kv_end + BN - 1) / BN;
    t.mask_from = p.Nkv / BN;                                  // tiles holding keys >= Nkv
    if (p.causal)
        t.mask_from = min(t.mask_from, (t.q0 + off + 1) / BN); // tiles crossing row q0's diagonal
    t.trace = (blockIdx.x == 0);
    t.g0 = 0;
    return t;
}

// Which items a CTA walks.  Items cost in proportion to their KV tiles, and
// a fixed assignment (the stride c, c + grid, ..., or any list made in
// advance from a cost model) leaves CTAs idle while others finish, most where
// a chunk of item_tile's order ends inside a wave.  So the items are handed
// out as the CTAs free up: CTA c starts with item c; its V loader, which runs
// ahead of the other roles, takes item n + 1 from a counter shared by the
// CTAs (item = grid + ticket, in item_tile's order) as it starts loading the
// V tiles of item n, and writes it into a ring of kItemSlots slots in shared
// memory (ITEMFULL per slot).  A CTA thus holds at most one item beyond the
// one it works on, so the CTAs finish within about one short item of each
// other.  Item n + 1 is written once the PV of item n - 1 has freed the V
// slots, so the compute warps and the MMA thread are in item n - 1 or later
// and have read item n - 1; the K loader runs ahead of them, and the Q
// converter has arrived on QFULL of item n - 1 and read item n - 1.  The slot
// rewritten held item n - 3: no slot is rewritten before all have read it, and
// no barrier runs two phases ahead of a reader.  An index past the last item
// is written as -1.

// Item number n (0, 1, ...) of this CTA, or -1 past its last item; false if
// the wait gave up.
__device__ __forceinline__ bool cta_item(uint32_t sb, const Waiter &wt, int n, int &it)
{
    if (n == 0) {
        it = static_cast<int>(blockIdx.x);
        return true;
    }
    const int s = (n - 1) & (kItemSlots - 1);
    if (!wt.wait(sb + OFF_BAR + 8u * (ITEMFULL + s), ((n - 1) / kItemSlots) & 1, SITE_ITEM))
        return false;
    it = static_cast<int>(ptx::ld_shared_u32(sb + OFF_ITEMS + 4u * s));
    return true;
}

// ---------------------------------------------------------------- the P step
//
// 2^x correctly rounded to FP32, for the rare keys whose FP8 byte the bracket
// of the fast path cannot decide.  Written from the Taylor series of e^t with
// t = r ln 2, x = n + r (n the nearest integer, |r| <= 1/2, both exact), in
// "float-float" arithmetic: each quantity is an unevaluated sum of two FP32
// values, products split exactly with a fused multiply-add (Dekker) and sums
// renormalised with the fast two-sum (Dekker; Knuth).  The series is split as
// e^t = A(u) + t B(u) with u = t^2 (even and odd terms), two Horner chains in
// u that run side by side (Estrin's idea: half the dependent steps of one
// chain in t).  Terms above 2^-23 (up to t^6 / 6! in A, t^5 / 5! in B) are
// carried in float-float, the tails (t^8 / 8! to t^12 / 12! and t^7 / 7! to
// t^11 / 11!) in FP32, whose rounding stays below 2^-47; the result is
// within about 2^-44 of 2^r, so its FP32 rounding is the correctly rounded one
// unless 2^x lies that close to a point halfway between two FP32 values.
// The constants are ln 2 and 1/k! split into FP32 high and low parts.
// x <= -40 (and -inf) gives 0, which every FP8 byte of 448 * 2^x agrees with.
__device__ __forceinline__ void fast_two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    e = __fadd_rn(b, __fsub_rn(a, s));
}

// (ph, pl) <- (ch, cl) + (th, tl) * (ph, pl), for |c| > |t * p|
__device__ __forceinline__ void ff_horner_step(float &ph, float &pl, float th, float tl, float ch, float cl)
{
    const float mh = __fmul_rn(ph, th);
    float ml = __fmaf_rn(ph, th, -mh);
    ml = __fmaf_rn(ph, tl, ml);
    ml = __fmaf_rn(pl, th, ml);
    float s, e;
    fast_two_sum(ch, mh, s, e);
    e = __fadd_rn(e, __fadd_rn(ml, cl));
    fast_two_sum(s, e, ph, pl);
}

__device__ __forceinline__ float exp2_rn(float x)
{
    if (!(x > -40.0f))
        return 0.0f;
    const float n = rintf(x);
    const float r = __fsub_rn(x, n);
    const float L1 = 0x1.62e430p-1f, L2 = -0x1.05c610p-29f;   // ln 2 = L1 + L2 + O(2^-54)
    float th = __fmul_rn(r, L1);
    float tl = __fmaf_rn(r, L1, -th);
    tl = __fmaf_rn(r, L2, tl);
    fast_two_sum(th, tl, th, tl);
    // e^t = A(u) + t B(u), u = t^2: two independent Horner chains in u
    float uh = __fmul_rn(th, th);
    float ul = __fmaf_rn(th, th, -uh);
    ul = __fmaf_rn(__fadd_rn(th, th), tl, ul);
    fast_two_sum(uh, ul, uh, ul);
    // FP32 tails (terms below 2^-23): A from u^4 / 8!, B from u^3 / 7!
    float qa = __fmaf_rn(0x1.1eed8ep-29f, uh, 0x1.27e4fcp-22f);   // 1/12!, 1/10!
    qa = __fmaf_rn(qa, uh, 0x1.a01a02p-16f);                      // 1/8!
    float qb = __fmaf_rn(0x1.ae6456p-26f, uh, 0x1.71de3ap-19f);   // 1/11!, 1/9!
    qb = __fmaf_rn(qb, uh, 0x1.a01a02p-13f);                      // 1/7!
    float ah = qa, al = 0.0f, bh = qb, bl = 0.0f;
    ff_horner_step(ah, al, uh, ul, 0x1.6c16c2p-10f, -0x1.27d27ep-35f);   // 1/6!
    ff_horner_step(bh, bl, uh, ul, 0x1.111112p-7f, -0x1.dddddep-32f);    // 1/5!
    ff_horner_step(ah, al, uh, ul, 0x1.555556p-5f, -0x1.555556p-30f);    // 1/4!
    ff_horner_step(bh, bl, uh, ul, 0x1.555556p-3f, -0x1.555556p-28f);    // 1/3!
    ff_horner_step(ah, al, uh, ul, 0.5f, 0.0f);                           // 1/2!
    ff_horner_step(bh, bl, uh, ul, 1.0f, 0.0f);                           // 1/1!
    ff_horner_step(ah, al, uh, ul, 1.0f, 0.0f);                           // 1/0!
    ff_horner_step(bh, bl, th, tl, ah, al);                               // A + t B
    // bh = RN(bh + bl) after the renormalisation; scale by 2^n (exact, n >= -40)
    return __fmul_rn(bh, __int_as_float((static_cast<int>(n) + 127) << 23));
}

// The FP8 byte of one key, every step in the stated order (the slow path).
__device__ __forceinline__ uint32_t p8_exact(float acc, float sig, float mu)
{
    const float dd = __fsub_rn(__fmul_rn(acc, sig), mu);
    return ptx::cvt_e4m3x2(0.0f, __fmul_rn(exp2_rn(dd), 448.0f)) & 0xffu;
}

constexpr float kP8Hi = 448.0f * (1.0f + 0x1p-21f), kP8Lo = 448.0f * (1.0f - 0x1p-21f);   // both exact in FP32

// dd = fl(fl(x * sig) - mu) for two keys in packed FP32 pairs, both roundings
// kept.  The assembler contracts a packed multiply whose only use is a packed
// subtraction into one fused multiply-add (one rounding), .rn or not; the
// product is therefore formed as fl(x * sig + z) with z a zero the compiler
// cannot see (a kernel argument, always +0), which is the same rounded
// product and cannot be fused with the subtraction.
__device__ __forceinline__ uint64_t dd_pair(uint32_t x0, uint32_t x1, uint64_t sg2, uint64_t m2, uint64_t z2)
{
    return ptx::sub_f32x2(ptx::fma_f32x2(ptx::f32x2(__uint_as_float(x0), __uint_as_float(x1)), sg2, z2), m2);
}

// FP8 P bytes of 32 keys (one block of the tile: raw accumulators x as FP32
// bit patterns, -inf for masked keys) with block scale product sig and running
// maximum mu (finite), four bytes per word, key 4w + u in byte u of word w.
// s2 = fl(x * sig), dd = fl(s2 - mu) in packed pairs; the bytes of
// 2^dd * 448 * (1 + 2^-21) (the result) and of 2^dd * 448 * (1 - 2^-21)
// (compared, not kept); keys whose two bytes differ are recomputed with
// p8_exact (rare).
__device__ __forceinline__ void p8_words4(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3, uint64_t sg2,
                                          uint64_t m2, uint64_t z2, uint32_t &hi, uint32_t &lo)
{
    const uint64_t hi2 = ptx::f32x2(kP8Hi, kP8Hi), lo2 = ptx::f32x2(kP8Lo, kP8Lo);
    const uint64_t d01 = dd_pair(x0, x1, sg2, m2, z2), d23 = dd_pair(x2, x3, sg2, m2, z2);
    const uint64_t e01 = ptx::f32x2(ptx::ex2_approx(ptx::f32x2_lo(d01)), ptx::ex2_approx(ptx::f32x2_hi(d01)));
    const uint64_t e23 = ptx::f32x2(ptx::ex2_approx(ptx::f32x2_lo(d23)), ptx::ex2_approx(ptx::f32x2_hi(d23)));
    const uint64_t p01 = ptx::mul_f32x2(e01, hi2), p23 = ptx::mul_f32x2(e23, hi2);
    const uint64_t n01 = ptx::mul_f32x2(e01, lo2), n23 = ptx::mul_f32x2(e23, lo2);
    hi = ptx::cvt_e4m3x4(ptx::f32x2_lo(p01), ptx::f32x2_hi(p01), ptx::f32x2_lo(p23), ptx::f32x2_hi(p23));
    lo = ptx::cvt_e4m3x4(ptx::f32x2_lo(n01), ptx::f32x2_hi(n01), ptx::f32x2_lo(n23), ptx::f32x2_hi(n23));
}

__device__ __forceinline__ void p8_words(const uint32_t (&x)[32], int w, uint64_t sg2, uint64_t m2, uint64_t z2,
                                         uint32_t &hi, uint32_t &lo)
{
    p8_words4(x[4 * w], x[4 * w + 1], x[4 * w + 2], x[4 * w + 3], sg2, m2, z2, hi, lo);
}

// Fast path of one block: the result bytes (upper bracket) in `out`; the
// return value is nonzero if any key's two brackets differ.
__device__ __forceinline__ uint32_t p8_block_fast(const uint32_t (&x)[32], float sig, float mu, float zero,
                                                  uint32_t (&out)[8])
{
    const uint64_t sg2 = ptx::f32x2(sig, sig), m2 = ptx::f32x2(mu, mu), z2 = ptx::f32x2(zero, zero);
    uint32_t diff = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        uint32_t lo;
        p8_words(x, w, sg2, m2, z2, out[w], lo);
        diff |= out[w] ^ lo;
    }
    return diff;
}

// The fast path of one block inside the forward: as p8_block_fast, and for a
// word whose two brackets differ, its four exponent arguments dd are stored
// (predicated, no branch) in the thread's 16-byte slot and bit 8c + w of
// wmask is set.  With one such word in the tile the slot holds it; with more,
// only the last (the caller then recomputes them all from the codes).
__device__ __forceinline__ void p8_block_park(const uint32_t (&x)[32], float sig, float mu, float zero,
                                              uint32_t (&out)[8], uint32_t slot, int c, uint32_t &wmask,
                                              uint32_t force = 0)
{
    const uint64_t sg2 = ptx::f32x2(sig, sig), m2 = ptx::f32x2(mu, mu), z2 = ptx::f32x2(zero, zero);
    const uint64_t hi2 = ptx::f32x2(kP8Hi, kP8Hi), lo2 = ptx::f32x2(kP8Lo, kP8Lo);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint64_t d01 = dd_pair(x[4 * w], x[4 * w + 1], sg2, m2, z2);
        const uint64_t d23 = dd_pair(x[4 * w + 2], x[4 * w + 3], sg2, m2, z2);
        const uint64_t e01 = ptx::f32x2(ptx::ex2_approx(ptx::f32x2_lo(d01)), ptx::ex2_approx(ptx::f32x2_hi(d01)));
        const uint64_t e23 = ptx::f32x2(ptx::ex2_approx(ptx::f32x2_lo(d23)), ptx::ex2_approx(ptx::f32x2_hi(d23)));
        const uint64_t p01 = ptx::mul_f32x2(e01, hi2), p23 = ptx::mul_f32x2(e23, hi2);
        const uint64_t n01 = ptx::mul_f32x2(e01, lo2), n23 = ptx::mul_f32x2(e23, lo2);
        out[w] = ptx::cvt_e4m3x4(ptx::f32x2_lo(p01), ptx::f32x2_hi(p01), ptx::f32x2_lo(p23), ptx::f32x2_hi(p23));
        const uint32_t lo =
            ptx::cvt_e4m3x4(ptx::f32x2_lo(n01), ptx::f32x2_hi(n01), ptx::f32x2_lo(n23), ptx::f32x2_hi(n23));
        // (force: debug builds treat the words whose bit is set as undecided)
        ptx::park_if_differ(out[w], ((force >> (8 * c + w)) & 1u) ? ~out[w] : lo, slot, __float_as_uint(ptx::f32x2_lo(d01)), __float_as_uint(ptx::f32x2_hi(d01)),
                            __float_as_uint(ptx::f32x2_lo(d23)), __float_as_uint(ptx::f32x2_hi(d23)), wmask,
                            1u << (8 * c + w));
    }
}

// Fix-up of one block (rare): the bytes again, with the undecided keys
// recomputed by p8_exact.
__device__ __forceinline__ void p8_block_fix(const uint32_t (&x)[32], float sig, float mu, float zero,
                                             uint32_t (&out)[8])
{
    const uint64_t sg2 = ptx::f32x2(sig, sig), m2 = ptx::f32x2(mu, mu), z2 = ptx::f32x2(zero, zero);
    uint32_t flags = 0;   // bit 4w + u: byte u of word w undecided
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        uint32_t lo;
        p8_words(x, w, sg2, m2, z2, out[w], lo);
        const uint32_t dw = out[w] ^ lo;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            flags |= (((dw >> (8 * u)) & 0xffu) != 0u ? 1u : 0u) << (4 * w + u);
    }
    while (flags != 0u) {
        const int k = __ffs(flags) - 1;
        flags &= flags - 1u;
        uint32_t xk = 0;
#pragma unroll
        for (int e = 0; e < 32; ++e)
            xk = (e == k) ? x[e] : xk;
        const uint32_t code = p8_exact(__uint_as_float(xk), sig, mu);
        const uint32_t sh = 8u * static_cast<uint32_t>(k & 3);
#pragma unroll
        for (int w = 0; w < 8; ++w)
            if ((k >> 2) == w)
                out[w] = (out[w] & ~(0xffu << sh)) | (code << sh);
    }
}

// The raw QK accumulators (exact int32 dot products of the codes) of keys
// key0 .. key0 + 31 for query row r of the item, recomputed by the warp: lane
// l returns key key0 + kl, kl = 2 (l % 16) + l / 16.  K: the 32 FP16 carrier
// rows in global memory (the tile was just read from there; 8 KB, contiguous),
// loaded coalesced, so that lane l holds channels 8 (l % 16) .. + 7 of keys
// 2i + l / 16 (i = 0 .. 15), turned back into their codes; keys from Nkv on
// are not read (their accumulators are not used).  Q: the same eight channels
// of the row, from the FP16 carrier in shared memory while it still holds this
// item (q_smem: KV tiles before the item's last two, whose QK may complete and
// release it during this tile's P); else from the prepared INT8 codes or, with
// in-kernel Q quantisation, quantised again from the BF16 Q with the row's
// block scale sq by the preparation's own quantiser.  Then a transposing
// butterfly over each half-warp sums the sixteen partial products of each key
// (integer sums: any order is exact).
__device__ __forceinline__ int block_accumulators(const FwdParams &p, const Tile &t, int r, int key0, float sq,
                                                  uint32_t sb, bool q_smem, int lane)
{
    const int ch = lane & 15;   // channel chunk: channels 8 ch .. 8 ch + 7
    const uint4 *kb = p.k_carrier + (static_cast<size_t>(t.b * p.Hkv + t.hk) * p.Nkv + key0) * (HD / 8);
    uint32_t q0 = 0, q1 = 0;   // Q codes of the chunk
    if (t.q0 + r < p.Nq) {     // (a pad row's codes are all 0)
        if (q_smem) {
            const uint4 a = ptx::ld_shared_v4(sb + OFF_Q + (ch >> 3) * Q_HALF_BYTES + r * 128 +
                                              ((static_cast<uint32_t>((ch & 7) ^ (r & 7))) << 4));
            q0 = ptx::i8x4_of_f16x2(a.x, a.y);
            q1 = ptx::i8x4_of_f16x2(a.z, a.w);
        } else if (p.q_codes) {
            const uint2 a = __ldg(reinterpret_cast<const uint2 *>(
                p.q_codes + (static_cast<size_t>(t.b * p.Hq + t.hq) * p.nq32 + t.q0 + r) * HD) + ch);
            q0 = a.x, q1 = a.y;
        } else if (sq > 0.0f) {   // (a zero block scale: every code is 0)
            const uint2 c = int8_codes8(__ldg(reinterpret_cast<const uint4 *>(
                                            p.q_bf16 + (static_cast<size_t>(t.b * p.Hq + t.hq) * p.Nq + t.q0 + r) * HD) + ch),
                                        sq, __frcp_rn(sq));
            q0 = c.x, q1 = c.y;
        }
    }
    // the 16 loads in four rounds of four (few registers: this runs beside
    // the tile's live state)
    int part[16];
#pragma unroll
    for (int rd = 0; rd < 4; ++rd) {
        uint4 kv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int ii = 4 * rd + i;
            kv[i] = (key0 + 2 * ii + (lane >> 4) < p.Nkv) ? __ldg(kb + 32 * ii + lane) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            part[4 * rd + i] =
                __dp4a(static_cast<int>(q1), static_cast<int>(ptx::i8x4_of_f16x2(kv[i].z, kv[i].w)),
                       __dp4a(static_cast<int>(q0), static_cast<int>(ptx::i8x4_of_f16x2(kv[i].x, kv[i].y)), 0));
        asm volatile("" ::: "memory");   // keep the next round's loads after these
    }
    // butterfly: at the step over lane bit b, the lane with bit b clear keeps
    // the entries whose index has bit b clear; after four steps lane l holds
    // the half-warp's sum for entry i = l % 16
#pragma unroll
    for (int b = 3; b >= 0; --b) {
        const bool up = (lane >> b) & 1;
#pragma unroll
        for (int i = 0; i < (1 << b); ++i) {
            const int send = up ? part[i] : part[i + (1 << b)];
            const int recv = __shfl_xor_sync(0xffffffffu, send, 1 << b);
            part[i] = (up ? part[i + (1 << b)] : part[i]) + recv;
        }
    }
    return part[0];
}

// The FP8 byte of one key: the bracket of the fast path (the same operations,
// one lane at a time), and p8_exact where the two bytes differ.
__device__ __forceinline__ uint32_t p8_byte(uint32_t x, float sig, float mu)
{
    const float e = ptx::ex2_approx(__fsub_rn(__fmul_rn(__uint_as_float(x), sig), mu));
    const uint32_t hi = ptx::cvt_e4m3x2(0.0f, __fmul_rn(e, kP8Hi)) & 0xffu;
    const uint32_t lo = ptx::cvt_e4m3x2(0.0f, __fmul_rn(e, kP8Lo)) & 0xffu;
    return hi == lo ? hi : p8_exact(__uint_as_float(x), sig, mu);
}

// The forward's rare-of-rare P fix-up: lanes whose bit c of
// `pend` is set have several undecided words and get their block c redone.
// For block c of the row of lane e, the warp recomputes the 32 accumulators
// from the codes (exact, so equal to the tensor core's), each lane the byte of
// one key with p8_byte, and lane e takes the gathered words into its P8 words
// pw (word 8c + w = keys 32c + 4w .. 32c + 4w + 3 of this half).  The block
// scale product of block c is the same for the warp's 32 rows (one Q block).
__device__ __forceinline__ void p8_fix_blocks(const FwdParams &p, const Tile &t, uint32_t pend, int quarter, int half,
                                           int j, int lane, float mu, float sig0, float sig1, float sig2, float sig3,
                                           float sq, uint32_t sb, uint32_t (&pw)[32])
{
#pragma unroll 1
    for (;;) {
        const uint32_t bal = __ballot_sync(0xffffffffu, pend != 0u);
        if (bal == 0u)
            break;
        const int e = __ffs(bal) - 1;
        const int c = __ffs(__shfl_sync(0xffffffffu, pend, e)) - 1;
        if (lane == e)
            pend &= pend - 1u;
        const float mue = __shfl_sync(0xffffffffu, mu, e);
        const float sg = (c == 0) ? sig0 : (c == 1) ? sig1 : (c == 2) ? sig2 : sig3;
        const int re = quarter * 32 + e;
        const int key0 = j * BN + 128 * half + 32 * c;
        const int kl = 2 * (lane & 15) + (lane >> 4);   // this lane's key of the block
        const int lime = p.causal ? t.q0 + re + (p.Nkv - p.Nq) : 0x7fffffff;
        const int acc = block_accumulators(p, t, re, key0, sq, sb, j + 2 < t.ntiles, lane);
        const uint32_t xk = (key0 + kl <= min(p.Nkv - 1, lime)) ? __float_as_uint(static_cast<float>(acc))
                                                                 : 0xff800000u;   // a masked key
        uint32_t v = p8_byte(xk, sg, mue) << (8 * (kl & 3));
        // keys 4w, 4w + 2 sit in lanes 2w, 2w + 1 and keys 4w + 1, 4w + 3 in
        // lanes 2w + 16, 2w + 17: two exchanges assemble word w in lane 2w
        v |= __shfl_xor_sync(0xffffffffu, v, 1);
        v |= __shfl_xor_sync(0xffffffffu, v, 16);
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const uint32_t wd = __shfl_sync(0xffffffffu, v, 2 * w);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                pw[8 * cc + w] = (lane == e && c == cc) ? wd : pw[8 * cc + w];
        }
    }
}

// Both, for one block (the test hook's entry).
__device__ __forceinline__ void p8_block(const uint32_t (&x)[32], float sig, float mu, float zero,
                                         uint32_t (&out)[8])
{
    if (p8_block_fast(x, sig, mu, zero, out) != 0u)
        p8_block_fix(x, sig, mu, zero, out);
}

// K loader.  Half-tile u = 2 * (tile) + h (channels [64h, 64h + 64) of the
// tile's 256 keys) goes to slot u % 3; the ring runs on one tile counter over
// all items of the CTA, so the next tile's halves load while QK of the current
// one runs (each half slot is released as soon as the four MMAs reading it
// complete).
__device__ __forceinline__ void kload_role(const FwdParams &p, const CUtensorMap *tm_k, uint32_t sb,
                                           const Waiter &wt)
{
    auto bar = [sb](int i) { return sb + OFF_BAR + 8u * i; };
    ptx::prefetch_tensormap(tm_k);
    int issued = -1;
    bool ok = true;
    int g = 0, n = 0;   // KV tiles and items of the earlier items
    for (int it = static_cast<int>(blockIdx.x); it >= 0 && ok; ok = ok && cta_item(sb, wt, ++n, it)) {
        Tile t = item_tile(p, it);
        t.g0 = g;
        const int bhk = t.b * p.Hkv + t.hk;
        for (int j = 0; j < t.ntiles && ok; ++j) {
            for (int h = 0; h < 2; ++h) {
                const int u = 2 * (g + j) + h, ks = u % KSLOTS;
                if (!wt.wait(bar(KEMPTY + ks), ((u / KSLOTS) & 1) ^ 1, SITE_KE)) {
                    ok = false;
                    break;
                }
                ptx::mbar_arrive_expect_tx(bar(KFULL + ks), K_HALF_BYTES);
                ptx::tma_load_3d(sb + OFF_K + ks * K_HALF_BYTES, tm_k, bar(KFULL + ks), 64 * h, j * BN, bhk);
                issued = u;
            }
            SATTN_TRACE(p, t, 11, j);
        }
        g += t.ntiles;
    }
    if (!ok)
        for (int u = max(0, issued - KSLOTS + 1); u <= issued; ++u)
            wt.drain(bar(KFULL + u % KSLOTS), (u / KSLOTS) & 1);
}

// V and Q loader.  V half-tiles (128 keys x 128 channels, E4M3) go to the two
// V slots; at the first tile of every item, once that item's Q has left the
// staging buffer (QFULL), the next item's INT8 Q tile (prepared codes only)
// and V channel scales are staged; the next item is taken from the shared
// counter and written into the ring (cta_item) just before.
template <bool kFuseQ>
__device__ __forceinline__ void vload_role(const FwdParams &p, const CUtensorMap *tm_v,
                                           const CUtensorMap *tm_q, uint32_t sb, const Waiter &wt)
{
    auto bar = [sb](int i) { return sb + OFF_BAR + 8u * i; };
    ptx::prefetch_tensormap(tm_v);
    if (!kFuseQ)
        ptx::prefetch_tensormap(tm_q);
    // INT8 Q tile of item `tq` into the staging buffer, and its V channel
    // scales into slot nq % 3 (the final conversion of item nq - 3, the last
    // reader of that slot, ends before QFULL of item nq - 1 is arrived)
    auto load_q = [&](const Tile &tq, int nq) {
        ptx::mbar_arrive_expect_tx(bar(QSTAGE), (kFuseQ ? 0u : QS_BYTES) + SV_BYTES);
        if (!kFuseQ)
            ptx::tma_load_3d(sb + OFF_QS, tm_q, bar(QSTAGE), 0, tq.q0, tq.b * p.Hq + tq.hq);
        ptx::bulk_load(sb + OFF_SV + (nq % 3) * SV_BYTES, p.v_scales + static_cast<size_t>(tq.b * p.Hkv + tq.hk) * HD,
                       SV_BYTES, bar(QSTAGE));
    };
    // the items after the first: grid + a ticket of the launch's counter, -1
    // past the last item (no tickets are taken when every CTA has one item)
    const bool shared = p.n_items > static_cast<int>(gridDim.x);
    auto take = [&]() { return shared ? atomicAdd(p.ticket, 1u) : 0xffffffffu; };
    auto item_of = [&](uint32_t ticket) {
        const long long v = static_cast<long long>(gridDim.x) + ticket;
        return ticket != 0xffffffffu && v < p.n_items ? static_cast<int>(v) : -1;
    };
    auto publish = [&](int k, int v) {   // item k >= 1 of this CTA into its ring slot
        const int sl = (k - 1) & (kItemSlots - 1);
        ptx::st_shared_u32(sb + OFF_ITEMS + 4u * sl, static_cast<uint32_t>(v));
        ptx::mbar_arrive(bar(ITEMFULL + sl));   // (release: the index is visible to the slot's readers)
    };
    if (p.withhold_v) {   // test hook: the MMA thread's wait for V runs out
        publish(1, -1);
        load_q(item_tile(p, static_cast<int>(blockIdx.x)), 0);
        wt.drain(bar(QSTAGE), 0);
        return;
    }
    int issued_v = -1, issued_q = -1;
    bool ok = true;
    int g = 0, n = 0;   // KV tiles and items of this CTA before the current item
    int nx = -1;        // item n + 1, taken at the first V tile of item n
    for (int it = static_cast<int>(blockIdx.x); it >= 0 && ok; ++n, it = nx) {
        Tile t = item_tile(p, it);
        t.g0 = g;
        const int bhk = t.b * p.Hkv + t.hk;
        if (n == 0) {
            load_q(t, 0);
            issued_q = 0;
        }
        for (int j = 0; j < t.ntiles && ok; ++j) {
            for (int h = 0; h < 2; ++h) {
                const int u = 2 * (g + j) + h, vs = u % VSLOTS;
                if (!wt.wait(bar(VEMPTY + vs), ((u / VSLOTS) & 1) ^ 1, SITE_VE)) {
                    ok = false;
                    break;
                }
                ptx::mbar_arrive_expect_tx(bar(VFULL + vs), V_TMA_BYTES);
                ptx::tma_load_3d(sb + OFF_V + vs * V_SLOT_BYTES, tm_v, bar(VFULL + vs), j * BN + 128 * h, 0, bhk);
                issued_v = u;
            }
            if (!ok)
                break;
            SATTN_TRACE(p, t, 12, j);
            if (j == 0) {   // the CTA commits to its next item only now, one item ahead
                nx = item_of(take());
                publish(n + 1, nx);
                if (nx >= 0) {
                    if (!wt.wait(bar(QFULL), n & 1, SITE_QE)) {
                        ok = false;
                        break;
                    }
                    load_q(item_tile(p, nx), n + 1);
                    issued_q = n + 1;
                }
            }
        }
        g += t.ntiles;
    }
    if (!ok) {
        for (int u = max(0, issued_v - VSLOTS + 1); u <= issued_v; ++u)
            wt.drain(bar(VFULL + u % VSLOTS), (u / VSLOTS) & 1);
        if (issued_q >= 0)
            wt.drain(bar(QSTAGE), issued_q & 1);
    }
}

// Single MMA-issuing thread.  Per item: wait for Q in TMEM, then S_j = Q K_j^T
// followed by PV_{j-1}; the last PV of an item is issued before the first QK
// of the next one.
__device__ __forceinline__ void mma_role(const FwdParams &p, uint32_t sb, uint32_t tmem, const Waiter &wt)
{
    auto bar = [sb](int i) { return sb + OFF_BAR + 8u * i; };
    bool ok = true;
    int g = 0, n = 0;
    for (int it = static_cast<int>(blockIdx.x); it >= 0 && ok; ok = ok && cta_item(sb, wt, ++n, it)) {
        Tile t = item_tile(p, it);
        t.g0 = g;
        SATTN_TRACE(p, t, 39, 0);
        if (!wt.wait(bar(QFULL), n & 1, SITE_Q))
            break;
        SATTN_TRACE(p, t, 40, 0);
        ptx::tc_fence_after();
        for (int j = 0; j <= t.ntiles && ok; ++j) {
            if (j < t.ntiles) {                     // S_j = Q K_j^T (256 keys)
                const int gj = g + j;
                if (gj >= 1 && !wt.wait(bar(SFREE), (gj - 1) & 1, SITE_SFREE)) {
                    ok = false;
                    break;
                }
                for (int h = 0; h < 2; ++h) {       // channels [64h, 64h + 64): four K=16 steps
                    const int u = 2 * gj + h, ks = u % KSLOTS;
                    if (!wt.wait(bar(KFULL + ks), (u / KSLOTS) & 1, SITE_K)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (h == 0)
                        SATTN_TRACE(p, t, 8, j);
                    const uint32_t kb = sb + OFF_K + ks * K_HALF_BYTES;
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        ptx::mma_f16_ss(tmem + TM_S, ptx::sw128_desc(sb + OFF_Q + h * Q_HALF_BYTES + s * 32),
                                        ptx::sw128_desc(kb + s * 32), IDESC_QK, (h | s) != 0);
                    ptx::mma_commit(bar(KEMPTY + ks));
                }
                if (!ok)
                    break;
                SATTN_TRACE(p, t, 9, j);
                ptx::mma_commit(bar(SFULL));
                if (j == t.ntiles - 1)
                    ptx::mma_commit(bar(QEMPTY));   // the item's Q carrier is no longer read
                SATTN_TRACE(p, t, 4, j);
            }
            if (j >= 1) {                           // PV_{j-1} = P_{j-1} V_{j-1}
                const int gg = g + j - 1;
                if (!wt.wait(bar(PFULL), gg & 1, SITE_P) ||
                    !wt.wait(bar(PVEMPTY), (gg & 1) ^ 1, SITE_PVE)) {
                    ok = false;
                    break;
                }
                for (int h = 0; h < 2 && ok; ++h) {
                    const int u = 2 * gg + h, vs = u % VSLOTS;
                    if (!wt.wait(bar(VFULL + vs), (u / VSLOTS) & 1, SITE_V)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (h == 0)
                        SATTN_TRACE(p, t, 5, j - 1);
                    const uint32_t vb = sb + OFF_V + vs * V_SLOT_BYTES;
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        ptx::mma_f8_ts(tmem + TM_PV, tmem + TM_P + 32 * h + 8 * s, ptx::sw128_desc(vb + s * 32),
                                       IDESC_PV, (h | s) != 0);
                    ptx::mma_commit(bar(VEMPTY + vs));
                }
                if (!ok)
                    break;
                SATTN_TRACE(p, t, 10, j - 1);
                ptx::mma_commit(bar(PVFULL));
                ptx::mma_commit(bar(PDONE));
            }
        }
        g += t.ntiles;
    }
    // every MMA of this CTA has finished before the TMEM is released
    ptx::mma_commit(bar(MMADONE));
    wt.drain(bar(MMADONE), 0);
}

// In-kernel Q quantisation (the preparation's block quantiser applied to the
// item's BF16 Q tile).  The tile (128 rows x 128 channels, rows >= Nq read as
// zeros) has landed by TMA in the output staging buffer, 256 bytes per row.
// For each 32-row block: amax -> s = fl(amax / 127), rs = fl(1 / s), and the
// INT8 codes go to the INT8 staging buffer in the layout the prepared codes
// arrive in by TMA (16-byte chunk c of row r at chunk c ^ (r % 8)); s goes to
// Q scale slot `slot`.  Thread l reads chunk l % 16 of row 2i + l / 16, so
// each warp instruction reads two whole rows without bank conflicts.
__device__ __forceinline__ void quantize_q_tile(uint32_t sb, int lane, int slot)
{
    const int k = lane & 15, rh = lane >> 4;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
        uint32_t am2 = 0u;   // max |x| of this thread's values, two BF16 lanes
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
            const uint4 a = ptx::ld_shared_v4(sb + OFF_STG + (32 * blk + 2 * i + rh) * 256 + 16 * k);
            am2 = ptx::bf16x2_max(am2, ptx::bf16x2_max(ptx::bf16x2_max(a.x & 0x7fff7fffu, a.y & 0x7fff7fffu),
                                                      ptx::bf16x2_max(a.z & 0x7fff7fffu, a.w & 0x7fff7fffu)));
        }
        float am = fmaxf(bf16_lo(am2), bf16_hi(am2));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        const float s = __fdiv_rn(am, 127.0f);
        const float rs = s > 0.0f ? __frcp_rn(s) : 0.0f;   // s = 0: every value is 0 and so is its code
#pragma unroll 2
        for (int i = 0; i < 16; ++i) {
            const int row = 32 * blk + 2 * i + rh;
            const uint2 c = int8_codes8(ptx::ld_shared_v4(sb + OFF_STG + row * 256 + 16 * k), s, rs);
            ptx::st_shared_v2(sb + OFF_QS + row * 128 + (((k >> 1) ^ (row & 7)) << 4) + 8 * (k & 1), c.x, c.y);
        }
        if (lane == 0)
            ptx::st_shared_f32(sb + OFF_SQ + 16 * slot + 4 * blk, s);
    }
}

// Q converter (one warp): for every item of the CTA, the staged INT8 Q tile
// (16-byte chunk c of row r at chunk c ^ (r % 8)) becomes the FP16 carrier in
// the two 64-channel halves of the Q buffer (same 128-byte swizzle); for items
// after the first it waits until the previous item's last QK has completed.
// Thread l converts rows l, l + 32, l + 64, l + 96, so the 16-byte accesses
// of a warp instruction spread over all banks.
//
// With kFuseQ the INT8 tile is this warp's own.  The first item's tile is
// quantised before the loop (QQDONE phase 0).  Right after the carrier of
// item n is handed over (QFULL), the BF16 Q tile of item n + 1 is staged in
// the output staging buffer and quantised into the INT8 staging buffer and
// the scale slot of its parity (QQDONE phase n + 1), once STGFREE phase n has
// completed: for n = 0 the compute warps have read the first scales, for
// n >= 1 the final conversion of item n - 1 has left the staging buffer.  The
// compute warps wait for QQDONE phase n + 1 before the final conversion of
// item n and only then arrive on STGFREE phase n + 1, so neither barrier runs
// more than one phase ahead of its waiter.
template <bool kFuseQ>
__device__ __forceinline__ void qconv_role(const FwdParams &p, const CUtensorMap *tm_q, uint32_t sb, int lane,
                                           const Waiter &wt)
{
    auto bar = [sb](int i) { return sb + OFF_BAR + 8u * i; };
    // stage and quantise the BF16 Q tile of item `itq`, the CTA's item number nq
    auto quantize_item = [&](int itq, int nq) -> bool {
        if (lane == 0) {
            const Tile tq = item_tile(p, itq);
            ptx::mbar_arrive_expect_tx(bar(QBF), STG_BYTES);
            ptx::tma_load_3d(sb + OFF_STG, tm_q, bar(QBF), 0, tq.q0, tq.b * p.Hq + tq.hq);
        }
        if (!wt.wait(bar(QBF), nq & 1, SITE_QBF)) {
            wt.drain(bar(QBF), nq & 1);   // the copy lands before the CTA may leave
            return false;
        }
        quantize_q_tile(sb, lane, nq & 1);
        __syncwarp();
        if (lane == 0)
            ptx::mbar_arrive(bar(QQDONE));
        return true;
    };
    if (kFuseQ) {
        if (lane == 0)
            ptx::prefetch_tensormap(tm_q);
        if (!quantize_item(static_cast<int>(blockIdx.x), 0))
            return;
    }
    int n = 0;
    for (int it = static_cast<int>(blockIdx.x); it >= 0;) {
        if ((n >= 1 && !wt.wait(bar(QEMPTY), (n - 1) & 1, SITE_QEMPTY)) ||
            !wt.wait(bar(QSTAGE), n & 1, SITE_QS))
            return;
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
            const int r = lane + 32 * i;
            const uint32_t src = sb + OFF_QS + r * HD;
#pragma unroll
            for (int c = 0; c < 8; ++c) {   // codes 16c .. 16c + 15 -> channels of half c / 4
                const uint4 a = ptx::ld_shared_v4(src + ((c ^ (r & 7)) << 4));
                const uint32_t dst = sb + OFF_Q + (c >> 2) * Q_HALF_BYTES + r * 128;
                const int w = 2 * (c & 3);  // FP16 chunk (8 channels) within the half row
                ptx::st_shared_v4(dst + ((w ^ (r & 7)) << 4), ptx::f16x2_of_i8(a.x, 0), ptx::f16x2_of_i8(a.x, 2),
                                  ptx::f16x2_of_i8(a.y, 0), ptx::f16x2_of_i8(a.y, 2));
                ptx::st_shared_v4(dst + (((w + 1) ^ (r & 7)) << 4), ptx::f16x2_of_i8(a.z, 0),
                                  ptx::f16x2_of_i8(a.z, 2), ptx::f16x2_of_i8(a.w, 0), ptx::f16x2_of_i8(a.w, 2));
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(bar(QFULL));
        if (!cta_item(sb, wt, n + 1, it))
            return;
        if (kFuseQ) {
            const int nx = it;
            if (nx >= 0) {
                __syncwarp();   // every lane has read the INT8 tile before it is rewritten
                if (!wt.wait(bar(STGFREE), n & 1, SITE_STG) || !quantize_item(nx, n + 1))
                    return;
            }
        }
        ++n;
    }
}

// Compute warpgroups.  Half h owns S columns [128h, 128h + 128) of every tile
// and writes the P8 bytes of those keys into TMEM columns [TM_P + 32h,
// TM_P + 32h + 32); the row max is exchanged through shared memory under a
// named barrier of the two warps that share those rows, so both halves hold
// the same running max m and alpha.  Half h also owns RO columns [64h, 64h +
// 64): after writing P_j it folds the partial PV_{j-1} into RO with
// alpha_{j-1} (both halves keep d).  The Q block scale of a row comes from
// q_scales, or with kFuseQ from the scale slot the Q converter fills (QQDONE).
template <bool kFuseQ>
__device__ __forceinline__ bool compute_loop(const FwdParams &p, const CUtensorMap *tm_o, uint32_t sb, uint32_t tmem,
                                             int warp, int lane, const Waiter &wt)
{
    auto bar = [sb](int i) { return sb + OFF_BAR + 8u * i; };
    const int half = warp >> 2;                               // 0 or 1
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                        // query row in the tile = TMEM lane
    const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t maxx = sb + OFF_MAXX;                      // [tile parity][half][row] row maxima

    auto qscale = [&](const Tile &tq) {
        const int i = tq.q0 + r;
        const float *a = p.q_scales + static_cast<size_t>(tq.b * p.Hq + tq.hq) * p.nbq + i / kQBlock;
        return i < p.nq32 ? (p.small ? ptx::ld_f32(a) : ptx::ld_nc_f32(a)) : 0.0f;
    };
    // block scales of this half's four 32-key blocks of tile j of an item
    auto kscale = [&](const Tile &tk, int j, int c) {
        const int kb = j * (BN / kQBlock) + 4 * half + c;
        // (the load is pinned here: it is consumed one tile later)
        const float *a = p.k_scales + static_cast<size_t>(tk.b * p.Hkv + tk.hk) * p.nbk + kb;
        return kb < p.nbk ? (p.small ? ptx::ld_f32(a) : ptx::ld_nc_f32(a)) : 0.0f;
    };

    int it = static_cast<int>(blockIdx.x);
    Tile t = item_tile(p, it);
    if (r == 0 && half == 0)
        SATTN_TRACE(p, t, 38, 1);
    float sq;
    if (kFuseQ) {
        if (!wt.wait(bar(QQDONE), 0, SITE_QQ))
            return false;
        sq = ptx::ld_shared_f32(sb + OFF_SQ + 4 * quarter);
        __syncwarp();
        if (lane == 0)   // STGFREE phase 0: the first scales have been read
            ptx::mbar_arrive(bar(STGFREE));
    } else {
        sq = qscale(t);
    }
    float sk[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        sk[c] = kscale(t, 0, c);

    uint64_t ro2[32];   // RO in packed pairs: channels 2i, 2i + 1
    float m, d, alpha_prev;
#ifdef SATTN_DEBUG_DUMP
    float m_tile1 = 0.0f;   // running maximum after KV tile 1 of the dumped item
#endif
    // RO = RO * alpha + PV partial of global tile gg (this half's 64 channels), d likewise
    auto fold_partial = [&](int gg, int jl, const Tile &tt, float alpha) -> bool {
        if (!wt.wait(bar(PVFULL), gg & 1, SITE_PV))
            return false;
        ptx::tc_fence_after();
        if (r == 0 && half == 0)
            SATTN_TRACE(p, tt, 6, jl);
#ifdef SATTN_DEBUG_DUMP
        if (p.dbg && jl == 0 && tt.q0 == 0 && tt.hq == 0 && tt.b == 0 && half == 0) {
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
            if ((c & 1) == 0)   // one packed fused multiply-add per channel pair, each lane rounded once
                ro2[c >> 1] = ptx::fma_f32x2(ro2[c >> 1], ptx::f32x2(alpha, alpha),
                                             ptx::f32x2(__uint_as_float(part[c >> 5][c & 31]),
                                                        __uint_as_float(part[(c + 1) >> 5][(c + 1) & 31])));
        d = fmaf(d, alpha, __uint_as_float(ds));
#ifdef SATTN_DEBUG_DUMP
        if (p.dbg && jl == 1 && tt.q0 == 0 && tt.hq == 0 && tt.b == 0) {   // the state after KV tile 1
            for (int c = 0; c < 64; ++c)
                p.dbg[DBG_RO1 + r * HD + 64 * half + c] = (c & 1) ? ptx::f32x2_hi(ro2[c >> 1]) : ptx::f32x2_lo(ro2[c >> 1]);
            if (half == 0) {
                p.dbg[DBG_M1 + r] = m_tile1;
                p.dbg[DBG_A1 + r] = alpha;
                p.dbg[DBG_D1 + r] = d;
            }
        }
#endif
        if (r == 0 && half == 0)
            SATTN_TRACE(p, tt, 7, jl);
        return true;
    };

    int g = 0, n = 0;   // KV tiles and items of this CTA before the current item
    for (;;) {
        t.g0 = g;
        const int i = t.q0 + r;
        const int lim = p.causal ? i + (p.Nkv - p.Nq) : 0x7fffffff;   // last kept key of row i
        int nx;
        if (!cta_item(sb, wt, n + 1, nx))
            return false;
        const bool has_next = nx >= 0;
        // (the next item's tile is recomputed where needed rather than kept live)
        float sq_next = (!kFuseQ && has_next) ? qscale(item_tile(p, nx)) : 0.0f;
        m = -INFINITY;
        d = 0.0f;
        alpha_prev = 0.0f;
    #pragma unroll
        for (int c = 0; c < 64; ++c)
            ro2[c >> 1] = 0ull;

        if (r == 0 && half == 0)
            SATTN_TRACE(p, t, 39, 1);
        for (int j = 0; j < t.ntiles; ++j) {
            const int gj = g + j;
            float sig[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                sig[c] = __fmul_rn(__fmul_rn(sq, sk[c]), p.c0);
                if (j + 1 < t.ntiles)
                    sk[c] = kscale(t, j + 1, c);
            }
            if (j + 1 == t.ntiles && has_next) {
                const Tile tn = item_tile(p, nx);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    sk[c] = kscale(tn, 0, c);
            }
            if (r == 0 && half == 0 && j == 0)
                SATTN_TRACE(p, t, 40, 1);
            if (r == 0 && half == 0)
                SATTN_TRACE(p, t, 41, j);
            if (!wt.wait(bar(SFULL), gj & 1, SITE_S))
                return false;
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
            // read early, tested before the pair barrier: a partner that gives
            // up after this read arrives on that barrier once, releasing it
            const uint32_t aborted = ptx::ld_shared_u32(sb + OFF_ABORT);
            if (r == 0 && half == 0)
                SATTN_TRACE(p, t, 1, j);
            if ((r & 31) == 0)
                SATTN_TRACE(p, t, 29 + 4 * half + (r >> 5), j);
#ifdef SATTN_DEBUG_DUMP
            if (p.dbg && j == 0 && t.q0 == 0 && t.hq == 0 && t.b == 0)
                for (int k = 0; k < 128; ++k)
                    p.dbg[r * BN + 128 * half + k] = __uint_as_float(s[k >> 5][k & 31]);
#endif
            // keys of this half that row i keeps are the first `nvalid` (the mask
            // is a suffix of the half-tile: keys >= Nkv and, if causal, keys >
            // lim).  Only the last tiles of an item carry masked keys; there the
            // masked scores are set to -inf before both passes, so one copy of
            // each pass serves all tiles.  On such tiles the combined scale is
            // raised to at least FLT_MIN so that -inf * scale stays -inf; a scale
            // below FLT_MIN moves an integer score by less than 1e-31, which no
            // later rounding sees.
            if (j >= t.mask_from) {
                const int lo = j * BN + 128 * half;
                const int nvalid = max(0, min(128, min(p.Nkv - 1, lim) - lo + 1));
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    sig[c] = fmaxf(sig[c], FLT_MIN);
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        s[c][k] = (32 * c + k < nvalid) ? s[c][k] : 0xff800000u;
                }
            }
            // max of the raw accumulators per 32-key block: the block scale is
            // positive (or zero), so fl(max(acc) * sig) = max(fl(acc * sig)) exactly
            float tmax = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                // eight independent three-input max chains, then a short tree
                float q[8];
#pragma unroll
                for (int a = 0; a < 8; ++a)
                    q[a] = ptx::fmax3(__uint_as_float(s[c][a]), __uint_as_float(s[c][a + 8]),
                                      __uint_as_float(s[c][a + 16]));
#pragma unroll
                for (int a = 0; a < 8; ++a)
                    q[a] = fmaxf(q[a], __uint_as_float(s[c][a + 24]));
                float b = fmaxf(ptx::fmax3(q[0], q[1], q[2]), ptx::fmax3(q[3], q[4], q[5]));
                b = ptx::fmax3(b, q[6], q[7]);
                tmax = fmaxf(tmax, __fmul_rn(b, sig[c]));
            }
            // exchange the half-row maxima (double-buffered by tile parity); only
            // warps w and w + 4 share rows, so each such pair has its own barrier
            ptx::st_shared_f32(maxx + 4 * (((gj & 1) * 2 + half) * BM + r), tmax);
            if ((r & 31) == 0)
                SATTN_TRACE(p, t, 21 + 4 * half + (r >> 5), j);
            if (aborted != 0)   // a warp gave up: leave, do not wait for it
                return false;
            ptx::named_bar_sync(1 + quarter, 64);
            tmax = fmaxf(tmax, ptx::ld_shared_f32(maxx + 4 * (((gj & 1) * 2 + (half ^ 1)) * BM + r)));
            if (r == 0 && half == 0)
                SATTN_TRACE(p, t, 2, j);

            const float mn = fmaxf(m, tmax);
            const float alpha = (m == -INFINITY) ? 0.0f : ptx::ex2_approx(__fsub_rn(m, mn));
            // P8 = E4M3(fl(fl(2^fl(fl(acc * sig) - m')) * 448)), four keys per
            // 32-bit word, written in one store into TMEM columns [TM_P + 32h,
            // TM_P + 32h + 32) of this row's lane, where PV reads them as its A
            // operand; the columns are free once the previous PV has completed.  A row with no kept key so far (mn =
            // -inf) has only -inf scores, which any finite maximum maps to 0.
            const float mu = (mn == -INFINITY) ? 0.0f : mn;
            // Rare (about 1.5e-5 of the keys): a key within 2^-21 of an E4M3
            // rounding midpoint.  The loop has no branch on it: a word (four
            // keys) with such a key leaves its four exponent arguments in the
            // thread's slot and its bit in wmask.  The 32 words stay in
            // registers; one vote: if any lane of the warp has such a word, the
            // warp rewrites them there.  A lane with one word recomputes its
            // four bytes from the slot.  A lane with more (rare
            // again) has its blocks redone from the codes (p8_fix_blocks).
            // Then the words go to TMEM in one store.
            const uint32_t slot = sb + OFF_PARK + (half * BM + r) * 16;
            uint32_t wmask = 0;   // bit 8c + w: word w of block c holds an undecided key
            uint32_t force = 0;
#ifdef SATTN_DEBUG_DUMP
            if (p.dbg) {   // test modes: one (1) or two (2) words of each row and tile taken as undecided
                const int mode = static_cast<int>(p.dbg[60012]);
                force = (mode >= 1 ? 1u << ((r + j) & 31) : 0u) | (mode >= 2 ? 1u << ((r + j + 7) & 31) : 0u);
            }
#endif
            uint32_t pw[32];   // P8 words of this half: word 8c + w holds keys 32c + 4w .. 32c + 4w + 3
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[8];
                p8_block_park(s[c], sig[c], mu, p.zero, pk, slot, c, wmask, force);
#pragma unroll
                for (int w = 0; w < 8; ++w)
                    pw[8 * c + w] = pk[w];
            }
            if (__any_sync(0xffffffffu, wmask != 0u)) {
                uint32_t und = 0;   // bit c: block c holds an undecided word
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    und |= ((wmask >> (8 * c)) & 0xffu) ? (1u << c) : 0u;
#ifdef SATTN_DEBUG_DUMP
                const long long fix_t0 = clock64();
                if (p.dbg)
                    atomicAdd(p.dbg + 60000, static_cast<float>(__popc(und)));   // undecided blocks seen
#endif
                const bool one = wmask != 0u && (wmask & (wmask - 1u)) == 0u;
                if (one) {   // the parked word: both brackets per key, the exact path per undecided key
                    const int wi = __ffs(wmask) - 1;
                    const uint4 dq = ptx::ld_shared_v4(slot);
                    const float dd[4] = {__uint_as_float(dq.x), __uint_as_float(dq.y), __uint_as_float(dq.z),
                                         __uint_as_float(dq.w)};
                    uint32_t word = 0, undk = 0;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float e = ptx::ex2_approx(dd[u]);
                        const uint32_t hi = ptx::cvt_e4m3x2(0.0f, __fmul_rn(e, kP8Hi)) & 0xffu;
                        const uint32_t lo = ptx::cvt_e4m3x2(0.0f, __fmul_rn(e, kP8Lo)) & 0xffu;
                        word |= hi << (8 * u);
                        undk |= (hi != lo) ? (1u << u) : 0u;
                    }
#pragma unroll 1
                    while (undk != 0u) {   // one copy of the correctly rounded exp2
                        const int u = __ffs(undk) - 1;
                        undk &= undk - 1u;
                        const float x = (u == 0) ? dd[0] : (u == 1) ? dd[1] : (u == 2) ? dd[2] : dd[3];
                        const uint32_t code = ptx::cvt_e4m3x2(0.0f, __fmul_rn(exp2_rn(x), 448.0f)) & 0xffu;
                        word = (word & ~(0xffu << (8 * u))) | (code << (8 * u));
                    }
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        pw[k] = (wi == k) ? word : pw[k];
                    und = 0u;
                }
                if (__any_sync(0xffffffffu, und != 0u))
                    p8_fix_blocks(p, t, und, quarter, half, j, lane, mu, sig[0], sig[1], sig[2], sig[3], sq, sb, pw);
#ifdef SATTN_DEBUG_DUMP
                if (p.dbg && lane == 0) {   // cycles in the fix-up and its count, per warp
                    atomicAdd(reinterpret_cast<unsigned long long *>(p.dbg + 60002),
                              static_cast<unsigned long long>(clock64() - fix_t0));
                    atomicAdd(reinterpret_cast<unsigned long long *>(p.dbg + 60004), 1ull);
                }
#endif
            }
            // the P8 columns are free once the previous tile's PV has completed
            if (gj >= 1 && !wt.wait(bar(PDONE), (gj - 1) & 1, SITE_PDONE))
                return false;
            ptx::tmem_st32(taddr + TM_P + 32 * half, pw);
#ifdef SATTN_DEBUG_DUMP
            if (p.dbg && j == 0 && t.q0 == 0 && t.hq == 0 && t.b == 0) {   // the bytes as PV will read them
                ptx::tmem_wait_st();
                uint32_t w32[32];
                ptx::tmem_ld32(taddr + TM_P + 32 * half, w32);
                ptx::tmem_wait_ld();
                for (int w = 0; w < 32; ++w)
                    p.dbg[32768 + r * 64 + 32 * half + w] = __uint_as_float(w32[w]);
            }
            if (j == 1)
                m_tile1 = mn;
#endif
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(PFULL));
            if (r == 0 && half == 0)
                SATTN_TRACE(p, t, 3, j);
            if ((r & 31) == 0)
                SATTN_TRACE(p, t, 13 + 4 * half + (r >> 5), j);
            if (j >= 1 && !fold_partial(gj - 1, j - 1, t, alpha_prev))
                return false;
            alpha_prev = alpha;
            m = mn;
        }
        if (!fold_partial(g + t.ntiles - 1, t.ntiles - 1, t, alpha_prev))
            return false;

        if (r == 0 && half == 0)
            SATTN_TRACE(p, t, 39, 2);
        if (kFuseQ && has_next) {   // the next item's Q scales are written and the staging buffer is free
            if (!wt.wait(bar(QQDONE), (n + 1) & 1, SITE_QQ))
                return false;
            sq_next = ptx::ld_shared_f32(sb + OFF_SQ + 16 * ((n + 1) & 1) + 4 * quarter);
        }
        // final conversion: reciprocal of d, per-channel V scale, BF16.  Each
        // warp stages its 32 rows x 64 channels (4 KB of its own, 16-byte chunk
        // c of row l at chunk c ^ (l % 8): the 128-byte swizzle) in shared
        // memory, and one thread stores the tile with TMA (rows >= Nq are
        // clipped by the tensor map).  The previous item's store has long
        // finished reading the staging buffer; the wait only confirms it.
        {
            if (lane == 0)
                ptx::bulk_wait_read();
            __syncwarp();
            const float rcp = d > 0.0f ? __frcp_rn(d) : 0.0f;
#ifdef SATTN_DEBUG_DUMP
            if (p.dbg && t.q0 == 0 && t.hq == 0 && t.b == 0 && half == 0) {
                p.dbg[DBG_DF + r] = d;
                p.dbg[DBG_RCP + r] = rcp;
            }
#endif
            const uint32_t sv4 = sb + OFF_SV + (n % 3) * SV_BYTES + 4 * 64 * half;   // landed with this item's Q
            const uint32_t stage = sb + OFF_STG + (quarter * 2 + half) * 4096;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const uint4 va = ptx::ld_shared_v4(sv4 + 32 * w), vb = ptx::ld_shared_v4(sv4 + 32 * w + 16);
                const float sv[8] = {__uint_as_float(va.x), __uint_as_float(va.y), __uint_as_float(va.z),
                                     __uint_as_float(va.w), __uint_as_float(vb.x), __uint_as_float(vb.y),
                                     __uint_as_float(vb.z), __uint_as_float(vb.w)};
                uint32_t u[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = 8 * w + 2 * e;
                    const float o0 = __fmul_rn(__fmul_rn(ptx::f32x2_lo(ro2[c >> 1]), rcp), sv[2 * e]);
                    const float o1 = __fmul_rn(__fmul_rn(ptx::f32x2_hi(ro2[c >> 1]), rcp), sv[2 * e + 1]);
                    const __nv_bfloat162 pr = __floats2bfloat162_rn(o0, o1);
                    memcpy(&u[e], &pr, sizeof(uint32_t));
                }
                ptx::st_shared_v4(stage + lane * 128 + ((w ^ (lane & 7)) << 4), u[0], u[1], u[2], u[3]);
            }
            ptx::fence_proxy_async_smem();   // the TMA store reads what the threads wrote
            __syncwarp();
            if (lane == 0) {
                ptx::tma_store_3d(tm_o, stage, 64 * half, t.q0 + quarter * 32, t.b * p.Hq + t.hq);
                ptx::bulk_commit();
                if (kFuseQ)   // the Q converter stages the item after next here: the store must have read it
                    ptx::bulk_wait_read();
            }
            __syncwarp();
            if (kFuseQ && lane == 0)   // STGFREE phase n + 1
                ptx::mbar_arrive(bar(STGFREE));
        }
        if (r == 0 && half == 0)
            SATTN_TRACE(p, t, 38, 2);
        g += t.ntiles;
        ++n;
        if (!has_next)
            break;
        it = nx;
        t = item_tile(p, nx);
        sq = sq_next;
    }
    return true;
}

// A compute warp that gave up (a bounded wait ran out, or another role
// reported a failure) marks the CTA as aborting and arrives once on its pair's
// exchange barrier: a partner already waiting there is released, and every
// compute warp checks the mark before that barrier, so none waits for a warp
// that has left.
template <bool kFuseQ>
__device__ __forceinline__ void compute_role(const FwdParams &p, const CUtensorMap *tm_o, uint32_t sb, uint32_t tmem,
                                             int warp, int lane, const Waiter &wt)
{
    const bool ok = compute_loop<kFuseQ>(p, tm_o, sb, tmem, warp, lane, wt);
    if (lane == 0)
        ptx::bulk_wait_all();   // output stores complete before the CTA's shared memory is released
    if (!ok) {
        asm volatile("st.shared.u32 [%0], 1;" ::"r"(sb + OFF_ABORT) : "memory");
        ptx::named_bar_arrive(1 + (warp & 3), 64);
    }
}

// The small-shape preparation for Nkv <= 256, staged: every input is first
// copied into shared memory (bulk copies into the CTA's free buffers, 212 KB
// from OFF_K), so
// the phases that follow read no global memory and run side by side on
// different warps.  Same arithmetic as the preparation kernels, element by
// element: the K column sums of each 64-token chunk in ascending token order,
// chunk sums in ascending chunk order, divided by Nkv; the V column maxima;
// per 32-token block the maximum |x| (of K - mean for K), s = amax / 127 and
// int8_code of every value (pad tokens 0); E4M3 codes v * (1 / s_v) by
// e4m3_code, channel-major, pad keys 0.  Only the assignment of work to
// threads differs, which no result depends on (maxima and elementwise codes).
constexpr int kSmallStagedNkv = 256;
__device__ __forceinline__ bool small_prepare_staged(const FwdParams &p, uint8_t *smem, const Waiter &wt)
{
    const SmallPrep &sp = p.sp;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Nkv = p.Nkv, Nq = p.Nq;
    uint8_t *base = smem + OFF_K;
    const uint4 *k4 = static_cast<const uint4 *>(sp.k), *v4 = static_cast<const uint4 *>(sp.v),
                *q4 = static_cast<const uint4 *>(sp.q);
    uint4 *sk4 = reinterpret_cast<uint4 *>(base), *sv4 = reinterpret_cast<uint4 *>(base + 65536),
          *sq4 = reinterpret_cast<uint4 *>(base + 131072);
    float *ks = reinterpret_cast<float *>(base + 163840);   // [4][128] chunk sums
    float *vm = ks + 4 * HD;                                 // [4][128] chunk maxima
    float *mean = vm + 4 * HD, *svs = mean + HD, *rvs = svs + HD;
    // 1. inputs into shared memory: three bulk copies on one mbarrier
    const uint32_t bar = ptx::smem_u32(base + 196608);
    if (tid == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        const uint32_t kb = static_cast<uint32_t>(Nkv) * 256u, qb = static_cast<uint32_t>(Nq) * 256u;
        ptx::mbar_arrive_expect_tx(bar, 2u * kb + qb);
        ptx::bulk_load(ptx::smem_u32(sk4), k4, kb, bar);
        ptx::bulk_load(ptx::smem_u32(sv4), v4, kb, bar);
        ptx::bulk_load(ptx::smem_u32(sq4), q4, qb, bar);
    }
    if (!wt.wait(bar, 0, SITE_Q) && tid == 0)
        wt.drain(bar, 0);   // the copies land before the CTA may leave
    __syncthreads();
    if (tid == 0)
        ptx::mbar_inval(bar);   // its memory is scratch again from here on
    if (*reinterpret_cast<volatile uint32_t *>(p.status) != 0)
        return false;
    const uint32_t *skw = reinterpret_cast<const uint32_t *>(sk4), *svw = reinterpret_cast<const uint32_t *>(sv4),
                   *sqw = reinterpret_cast<const uint32_t *>(sq4);
    auto kval = [&](int t, int c) {   // BF16 K[t][c] as FP32
        const uint32_t w = skw[t * 64 + (c >> 1)];
        return (c & 1) ? bf16_hi(w) : bf16_lo(w);
    };
    auto vval = [&](int t, int c) {
        const uint32_t w = svw[t * 64 + (c >> 1)];
        return (c & 1) ? bf16_hi(w) : bf16_lo(w);
    };
    auto qval = [&](int t, int c) {
        const uint32_t w = sqw[t * 64 + (c >> 1)];
        return (c & 1) ? bf16_hi(w) : bf16_lo(w);
    };
    // 2. per (chunk, channel): the column sum of K and the column max |V|
    const int nch = (Nkv + kMeanChunk - 1) / kMeanChunk;
    for (int it = tid; it < nch * HD; it += NTHREADS) {
        const int ch = it / HD, c = it % HD;
        const int t1 = min(Nkv, (ch + 1) * kMeanChunk);
        float sum = 0.0f, mx = 0.0f;
        for (int t = ch * kMeanChunk; t < t1; ++t) {
            sum = __fadd_rn(sum, kval(t, c));
            mx = fmaxf(mx, fabsf(vval(t, c)));
        }
        ks[ch * HD + c] = sum;
        vm[ch * HD + c] = mx;
    }
    __syncthreads();
    if (tid < HD) {
        float total = 0.0f, amax = 0.0f;
        for (int ch = 0; ch < nch; ++ch) {
            total = __fadd_rn(total, ks[ch * HD + tid]);
            amax = fmaxf(amax, vm[ch * HD + tid]);
        }
        const float mu = __fdiv_rn(total, static_cast<float>(Nkv));
        const float sc = __fdiv_rn(amax, 448.0f);
        mean[tid] = mu;
        svs[tid] = sc;
        rvs[tid] = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
        sp.k_mean[tid] = mu;
        sp.v_scales[tid] = sc;
    }
    __syncthreads();
    // 3. one warp per 32-token block of K (then of Q): lane l holds channels
    // 4l .. 4l + 3 of the block's 32 tokens
    const int nbk = p.nbk, nbq = p.nbq;
    for (int job = warp; job < nbk + nbq; job += NTHREADS / 32) {
        const bool isk = job < nbk;
        const int blk = isk ? job : job - nbk, N = isk ? Nkv : Nq;
        float am = 0.0f;
        for (int r = 0; r < kQBlock; ++r) {
            const int t = blk * kQBlock + r;
            if (t < N)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = 4 * lane + u;
                    const float x = isk ? __fsub_rn(kval(t, c), mean[c]) : qval(t, c);
                    am = fmaxf(am, fabsf(x));
                }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        const float sc = __fdiv_rn(am, 127.0f);
        const float rs = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
        int8_t *codes = isk ? sp.k_codes : sp.q_codes;
        for (int r = 0; r < kQBlock; ++r) {
            const int t = blk * kQBlock + r;
            uint32_t word = 0;
            if (t < N && sc > 0.0f)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = 4 * lane + u;
                    const float x = isk ? __fsub_rn(kval(t, c), mean[c]) : qval(t, c);
                    word |= int8_code(x, sc, rs) << (8 * u);
                }
            reinterpret_cast<uint32_t *>(codes + static_cast<size_t>(t) * HD)[lane] = word;
            if (isk && t < Nkv) {   // the FP16 carrier of the same four codes
                uint2 *dst = reinterpret_cast<uint2 *>(const_cast<uint4 *>(p.k_carrier) + static_cast<size_t>(t) * 16);
                dst[lane] = make_uint2(ptx::f16x2_of_i8(word, 0), ptx::f16x2_of_i8(word, 2));
            }
        }
        if (lane == 0)
            (isk ? sp.k_scales : sp.q_scales)[blk] = sc;
    }
    // 4. V: per (channel, 16-token group), channel-major
    const int nk128 = (Nkv + kVPad - 1) / kVPad * kVPad;
    for (int it = tid; it < HD * (nk128 / 16); it += NTHREADS) {
        const int c = it % HD, g = it / HD;
        const float sc = svs[c], rc = rvs[c];
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int t = 16 * g + u;
            const uint32_t code = (t < Nkv && sc > 0.0f) ? prep::e4m3_code(vval(t, c), sc, rc) : 0u;
            w[u >> 2] |= code << (8 * (u & 3));
        }
        *reinterpret_cast<uint4 *>(sp.v_codes + static_cast<size_t>(c) * nk128 + 16 * g) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    ptx::fence_proxy_async_global();
    __syncthreads();
    return true;
}

// The single-launch small-shape path (one query tile of one head, Nkv <=
// kSmallMaxNkv): all threads of the CTA run the preparation of the
// preparation kernels, through the same device functions (prep_device.cuh),
// so the buffers hold the same bytes: K column sums per 64-token chunk and
// V column maxima, their ordered totals (mean, V scale), then the INT8 K
// blocks, the FP8 V tiles and the INT8 Q blocks (256 threads, a named
// barrier), then the FP16 carrier of the K codes.  Scratch: the K ring's
// shared memory, which the pipeline fills only afterwards.  The writes are
// ordered before the pipeline's TMA reads by a proxy fence and a CTA barrier.
__device__ __forceinline__ void small_prepare(const FwdParams &p, uint8_t *smem)
{
    const SmallPrep &sp = p.sp;
    const int tid = threadIdx.x;
    const int Nkv = p.Nkv, Nq = p.Nq;
    const int nch = (Nkv + kMeanChunk - 1) / kMeanChunk;   // <= 16
    float *ks = reinterpret_cast<float *>(smem + OFF_K);         // [16][128] chunk sums of K
    float *vm = ks + 16 * HD;                                      // [16][128] chunk maxima of |V|
    float *mean = vm + 16 * HD, *sv = mean + HD, *rv = sv + HD;    // [128] each
    float *warp_max = rv + HD;                                     // [8]
    uint32_t *vtile = reinterpret_cast<uint32_t *>(smem + OFF_K + 24 * 1024);   // [128][32] words
    const uint4 *k4 = static_cast<const uint4 *>(sp.k), *v4 = static_cast<const uint4 *>(sp.v);
    if (tid < 16 * nch) {
        const int chunk = tid >> 4, g = tid & 15;
        float sum[8], mx[8];
        prep::chunk_stats8(k4, v4, Nkv, 0, chunk, g, sum, mx);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            ks[chunk * HD + 8 * g + i] = sum[i];
            vm[chunk * HD + 8 * g + i] = mx[i];
        }
    }
    __syncthreads();
    if (tid < HD) {   // chunk sums in ascending chunk order, as the finalize kernel
        float total = 0.0f, amax = 0.0f;
        for (int ch = 0; ch < nch; ++ch) {
            total = __fadd_rn(total, ks[ch * HD + tid]);
            amax = fmaxf(amax, vm[ch * HD + tid]);
        }
        const float mu = __fdiv_rn(total, static_cast<float>(Nkv));
        const float s = __fdiv_rn(amax, 448.0f);
        mean[tid] = mu;
        sv[tid] = s;
        rv[tid] = s > 0.0f ? __frcp_rn(s) : 0.0f;
        sp.k_mean[tid] = mu;
        sp.v_scales[tid] = s;
    }
    __syncthreads();
    if (tid < 256) {
        auto sync256 = [] { asm volatile("bar.sync 1, 256;" ::: "memory"); };
        const int64_t nk32 = (Nkv + kQBlock - 1) / kQBlock * kQBlock, nq32 = (Nq + kQBlock - 1) / kQBlock * kQBlock;
        const int64_t nk128 = (Nkv + kVPad - 1) / kVPad * kVPad;
        for (int blk = 0; blk < p.nbk; ++blk) {
            prep::quant_block<true>(k4, Nkv, nk32, p.nbk, mean, sp.k_codes, sp.k_scales, 0, blk, tid, warp_max,
                                    sync256);
            sync256();
        }
        for (int t0 = 0; t0 < nk128; t0 += kVPad) {
            prep::quant_v_tile(v4, Nkv, nk128, sv, rv, sp.v_codes, 0, t0, tid, vtile, sync256);
            sync256();
        }
        for (int blk = 0; blk < p.nbq; ++blk) {
            prep::quant_block<false>(static_cast<const uint4 *>(sp.q), Nq, nq32, p.nbq, nullptr, sp.q_codes,
                                     sp.q_scales, 0, blk, tid, warp_max, sync256);
            sync256();
        }
    }
    __syncthreads();
    // the FP16 carrier of the K codes (as k_carrier_kernel)
    uint4 *dst = const_cast<uint4 *>(p.k_carrier);
    const uint4 *src = reinterpret_cast<const uint4 *>(sp.k_codes);
    for (int c = tid; c < Nkv * (HD / 16); c += NTHREADS) {
        const uint4 a = src[c];
        dst[2 * c] = make_uint4(ptx::f16x2_of_i8(a.x, 0), ptx::f16x2_of_i8(a.x, 2), ptx::f16x2_of_i8(a.y, 0),
                                ptx::f16x2_of_i8(a.y, 2));
        dst[2 * c + 1] = make_uint4(ptx::f16x2_of_i8(a.z, 0), ptx::f16x2_of_i8(a.z, 2), ptx::f16x2_of_i8(a.w, 0),
                                    ptx::f16x2_of_i8(a.w, 2));
    }
    ptx::fence_proxy_async_global();
    __syncthreads();
}

// kSmall: the single-launch small-shape path, whose preparation runs first
// (a separate instantiation, so that the other launches carry none of its code)
template <bool kFuseQ, bool kSmall>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sb = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#ifdef SATTN_DEBUG_DUMP
    if (p.dbg && threadIdx.x == 0 && blockIdx.x == 0)
        reinterpret_cast<unsigned long long *>(p.dbg + 61440)[37 * 256 + 0] = clock64();
#endif
    const Waiter wt{p.status};
    volatile uint32_t *flag = reinterpret_cast<volatile uint32_t *>(smem + OFF_FLAG);
    if (kSmall && p.small) {
        if (p.Nkv <= kSmallStagedNkv)
            small_prepare_staged(p, smem, wt);   // a failed copy leaves the status set: the CTA does no more
        else
            small_prepare(p, smem);
    }

    if (threadIdx.x == 0) {
        *flag = *reinterpret_cast<volatile uint32_t *>(p.status);
        *reinterpret_cast<volatile uint32_t *>(smem + OFF_ABORT) = 0u;
        const uint32_t b0 = sb + OFF_BAR;
        for (int s = 0; s < KSLOTS; ++s) {
            ptx::mbar_init(b0 + 8u * (KFULL + s), 1);
            ptx::mbar_init(b0 + 8u * (KEMPTY + s), 1);
        }
        for (int s = 0; s < VSLOTS; ++s) {
            ptx::mbar_init(b0 + 8u * (VFULL + s), 1);
            ptx::mbar_init(b0 + 8u * (VEMPTY + s), 1);
        }
        ptx::mbar_init(b0 + 8u * QSTAGE, 1);
        ptx::mbar_init(b0 + 8u * QFULL, 32);
        ptx::mbar_init(b0 + 8u * QEMPTY, 1);
        ptx::mbar_init(b0 + 8u * SFULL, 1);
        ptx::mbar_init(b0 + 8u * SFREE, 2 * BM);
        ptx::mbar_init(b0 + 8u * PFULL, 2 * BM);
        ptx::mbar_init(b0 + 8u * PDONE, 1);
        ptx::mbar_init(b0 + 8u * PVFULL, 1);
        ptx::mbar_init(b0 + 8u * PVEMPTY, 2 * BM);
        ptx::mbar_init(b0 + 8u * MMADONE, 1);
        ptx::mbar_init(b0 + 8u * QBF, 1);
        ptx::mbar_init(b0 + 8u * QQDONE, 1);
        ptx::mbar_init(b0 + 8u * STGFREE, 8);
        for (int s = 0; s < kItemSlots; ++s)
            ptx::mbar_init(b0 + 8u * (ITEMFULL + s), 1);
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

    if (*flag == 0 && static_cast<int>(blockIdx.x) < p.n_items) {
        if (warp < WARP_PRODUCER) {
            ptx::setmaxnreg_inc<kRegsCompute>();
            compute_role<kFuseQ>(p, &tm_o, sb, tmem, warp, lane, wt);
        } else {
            ptx::setmaxnreg_dec<kRegsOther>();
            if (warp == WARP_PRODUCER) {
                if (lane == 0)
                    kload_role(p, &tm_k, sb, wt);
            } else if (warp == WARP_VLOAD) {
                if (lane == 0)
                    vload_role<kFuseQ>(p, &tm_v, &tm_q, sb, wt);
            } else if (warp == WARP_MMA) {
                if (lane == 0)
                    mma_role(p, sb, tmem, wt);
            } else if (warp == WARP_QCONV) {
                qconv_role<kFuseQ>(p, &tm_q, sb, lane, wt);
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
#ifdef SATTN_DEBUG_DUMP
    if (p.dbg && threadIdx.x == 0 && blockIdx.x == 0)
        reinterpret_cast<unsigned long long *>(p.dbg + 61440)[37 * 256 + 1] = clock64();
#endif
}

// The K codes [B*Hkv][nk32][128] (INT8) -> their FP16 carrier [B*Hkv][Nkv][128],
// the operand of QK^T on the tensor cores (this part has no INT8 tensor-core
// product; integers of magnitude <= 127 are exact in FP16).  Thread = 8 codes
// (an 8-byte load, one 16-byte store, so a warp's store covers 512 contiguous
// bytes), kCarrierUnroll groups per thread; grid y = KV head.  Bound by HBM
// bandwidth: 128 bytes read and 256 written per key.
constexpr int kCarrierUnroll = 8;
__global__ void __launch_bounds__(256) k_carrier_kernel(const uint2 *__restrict__ codes, int Nkv, int64_t nk32,
                                                        uint4 *__restrict__ carrier)
{
    const int64_t bh = blockIdx.y;
    const int64_t n = static_cast<int64_t>(Nkv) * (HD / 8);   // 8-code groups of this head
    const uint2 *src = codes + bh * nk32 * (HD / 8);
    uint4 *dst = carrier + bh * n;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * (256 * kCarrierUnroll) + threadIdx.x;
    uint2 a[kCarrierUnroll];
#pragma unroll
    for (int u = 0; u < kCarrierUnroll; ++u)
        if (c0 + 256 * u < n)
            a[u] = __ldg(src + c0 + 256 * u);
#pragma unroll
    for (int u = 0; u < kCarrierUnroll; ++u) {
        const int64_t c = c0 + 256 * u;
        if (c < n)
            dst[c] = make_uint4(ptx::f16x2_of_i8(a[u].x, 0), ptx::f16x2_of_i8(a[u].x, 2),
                                ptx::f16x2_of_i8(a[u].y, 0), ptx::f16x2_of_i8(a[u].y, 2));
    }
}

// Test kernels of the P step: FP8 bytes of groups of 32 keys through p8_block
// (group i: accumulators acc[32i .. 32i + 31], block scale product sig[i],
// running maximum m[i]), and exp2_rn elementwise.
__global__ void __launch_bounds__(128) test_p8_kernel(int n_groups, const float *__restrict__ acc,
                                                      const float *__restrict__ sig, const float *__restrict__ m,
                                                      uint32_t *__restrict__ out, float zero)
{
    const int gi = blockIdx.x * blockDim.x + threadIdx.x;
    if (gi >= n_groups)
        return;
    uint32_t x[32], w[8];
#pragma unroll
    for (int k = 0; k < 32; ++k)
        x[k] = __float_as_uint(acc[static_cast<size_t>(gi) * 32 + k]);
    p8_block(x, sig[gi], m[gi], zero, w);
#pragma unroll
    for (int k = 0; k < 8; ++k)
        out[static_cast<size_t>(gi) * 8 + k] = w[k];
}

__global__ void __launch_bounds__(256) test_exp2_kernel(int n, const float *__restrict__ x, float *__restrict__ out)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n)
        out[i] = exp2_rn(x[i]);
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

static cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;
void set_profile_events(cudaEvent_t before, cudaEvent_t after)
{
    g_ev_before = before;
    g_ev_after = after;
}

#ifdef SATTN_DEBUG_DUMP
static float *g_debug_dump = nullptr;
float *debug_dump_buffer() { return g_debug_dump; }
extern "C" void sattn_debug_set_dump(float *p) { g_debug_dump = p; }
#endif

size_t carrier_bytes(const Geometry &g)
{
    return static_cast<size_t>(g.B) * g.Hkv * g.Nkv * HD * sizeof(__half);
}

size_t forward_workspace_bytes(const Geometry &g)
{
    return kStatusBytes + carrier_bytes(g);
}

namespace {

// The per-warpgroup register split only adds up when the kernel is launched
// with exactly kLaunchRegs registers per thread; refuse to launch otherwise.
// Also raises the kernel's dynamic shared-memory limit.  Once per process.
template <bool kFuseQ, bool kSmall>
cudaError_t kernel_attributes()
{
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        cudaFuncAttributes fa;
        attr_err = cudaFuncGetAttributes(&fa, attn_fwd_kernel<kFuseQ, kSmall>);
        if (attr_err == cudaSuccess && fa.numRegs != kLaunchRegs)
            attr_err = cudaErrorInvalidConfiguration;
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(attn_fwd_kernel<kFuseQ, kSmall>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
    });
    return attr_err;
}

// The shape fields of the item order (item_tile): the query tiles, the items,
// and the chunks of (batch, KV head) units with the reciprocals of udiv.
// False if the item indices leave udiv's range.
bool plan_items(const Geometry &g, FwdParams &prm)
{
    prm.B = g.B;
    prm.Hq = g.Hq;
    prm.Hkv = g.Hkv;
    prm.Nq = g.Nq;
    prm.Nkv = g.Nkv;
    prm.group = g.Hq / g.Hkv;
    prm.n_qtiles = static_cast<int>((g.Nq + BM - 1) / BM);
    const int64_t n_items = static_cast<int64_t>(prm.n_qtiles) * g.Hq * g.B;
    if (n_items >= (int64_t(1) << 31))
        return false;
    prm.n_items = static_cast<int>(n_items);
    auto recip = [](int d) { return d == 1 ? 0ull : ~0ull / static_cast<unsigned long long>(d) + 1ull; };
    prm.n_units = g.B * g.Hkv;
    {   // the fewest chunks whose units' K carrier (2 bytes) and V codes (1 byte) fit in
        // kL2ChunkBytes, with the units spread evenly over them
        const int64_t unit_bytes = static_cast<int64_t>(g.Nkv) * HD * 3;
        const int64_t cap = std::max<int64_t>(1, std::min<int64_t>(prm.n_units, kL2ChunkBytes / unit_bytes));
        const int64_t n_chunks = (prm.n_units + cap - 1) / cap;
        prm.chunk_units = static_cast<int>((prm.n_units + n_chunks - 1) / n_chunks);
    }
    prm.chunk_items = prm.chunk_units * prm.group * prm.n_qtiles;
    const int tail_units = prm.n_units - (prm.n_units - 1) / prm.chunk_units * prm.chunk_units;
    prm.m_chunk = recip(prm.chunk_items);
    prm.m_row = recip(prm.chunk_units * prm.group);
    prm.m_row_tail = recip(tail_units * prm.group);
    prm.m_hkv = recip(g.Hkv);
    prm.m_group = recip(prm.group);
    prm.causal = g.causal;
    return true;
}

// q: INT8 codes [B, Hq, nq32, 128] with q_scales, or with kFuseQ the BF16 Q
// [B, Hq, Nq, 128] itself (q_scales unused)
template <bool kFuseQ>
int launch_impl(const Geometry &g, const void *q, const float *q_scales, const int8_t *k_codes,
                const float *k_scales, const uint8_t *v_codes, const float *v_scales, void *out,
                void *status_block, void *k_carrier, cudaStream_t stream, bool withhold_v, bool reset_status,
                const SmallPrep *small = nullptr, int ticket_slot = 0)
{
    auto encode = tensor_map_encoder();
    if (!encode)
        return 1;
    uint32_t *status = static_cast<uint32_t *>(status_block);
    const int bhk = g.B * g.Hkv;
    if (reset_status && cudaMemsetAsync(status, 0, 2 * sizeof(uint32_t), stream) != cudaSuccess)
        return static_cast<int>(cudaGetLastError());

    CUtensorMap tmk, tmv, tmo;
    {   // BF16 output, stored per warp as 32 rows x 64 channels (128-byte swizzle); rows >= Nq are clipped
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(g.Nq),
                                    static_cast<cuuint64_t>(g.B) * g.Hq};
        const cuuint64_t strides[2] = {HD * 2, static_cast<cuuint64_t>(g.Nq) * HD * 2};
        const cuuint32_t box[3] = {64, 32, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tmo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return 1;
    }
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(g.Nkv),
                                    static_cast<cuuint64_t>(bhk)};
        const cuuint64_t strides[2] = {HD * sizeof(__half), static_cast<cuuint64_t>(g.Nkv) * HD * sizeof(__half)};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BN), 1};   // 256 keys x 64 channels
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tmk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(k_carrier), dims, strides, box, estr,
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

    CUtensorMap tmq;
    if (kFuseQ) {   // BF16 Q, 128 rows x 128 channels (32 KB, 256-byte rows), rows >= Nq read as zeros
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(g.Nq),
                                    static_cast<cuuint64_t>(g.B) * g.Hq};
        const cuuint64_t strides[2] = {HD * 2, static_cast<cuuint64_t>(g.Nq) * HD * 2};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(HD), static_cast<cuuint32_t>(BM), 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tmq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return 1;
    } else {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(g.nq32),
                                    static_cast<cuuint64_t>(g.B) * g.Hq};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(g.nq32) * HD};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(HD), static_cast<cuuint32_t>(BM), 1};   // 128 rows x 128 codes
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tmq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(q), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return 1;
    }

    cudaError_t attr_err = kernel_attributes<kFuseQ, false>();
    if constexpr (!kFuseQ)
        if (small && attr_err == cudaSuccess)
            attr_err = kernel_attributes<false, true>();
    if (attr_err != cudaSuccess)
        return static_cast<int>(attr_err);

    if (!small) {   // the FP16 carrier of the K codes, read by the attention kernel's K loader
        const int64_t ngroup = static_cast<int64_t>(g.Nkv) * (HD / 8);
        const dim3 grid(static_cast<unsigned>((ngroup + 256 * kCarrierUnroll - 1) / (256 * kCarrierUnroll)),
                        static_cast<unsigned>(bhk));
        k_carrier_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint2 *>(k_codes), g.Nkv, g.nk32,
                                                    static_cast<uint4 *>(k_carrier));
    }

    FwdParams prm;
    prm.q_scales = q_scales;
    prm.k_scales = k_scales;
    prm.v_scales = v_scales;
    prm.out = static_cast<__nv_bfloat16 *>(out);
    prm.status = status;
    prm.withhold_v = withhold_v ? 1 : 0;
    if (!plan_items(g, prm))
        return static_cast<int>(cudaErrorInvalidValue);   // item indices must fit udiv's range
    prm.causal = g.causal;
    prm.nq32 = static_cast<int>(g.nq32);
    prm.nbq = static_cast<int>(g.nbq);
    prm.nbk = static_cast<int>(g.nbk);
    const float sm = g.sm_scale > 0.0f ? g.sm_scale : 1.0f / sqrtf(static_cast<float>(HD));
    prm.q_codes = kFuseQ ? nullptr : static_cast<const int8_t *>(q);
    prm.q_bf16 = kFuseQ ? static_cast<const __nv_bfloat16 *>(q) : nullptr;
    prm.k_carrier = static_cast<const uint4 *>(k_carrier);
    prm.zero = 0.0f;
    prm.small = small ? 1 : 0;
    prm.sp = small ? *small : SmallPrep{};
    prm.c0 = sm * 1.44269504088896340736f;
#ifdef SATTN_DEBUG_DUMP
    prm.dbg = debug_dump_buffer();
#endif

    // persistent: one CTA per SM, each taking items as it frees up (cta_item);
    // the launch's item counter is a word of the status block, zeroed here
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm < 1)
        return static_cast<int>(cudaErrorInvalidDevice);
    const int grid = std::min(prm.n_items, n_sm);
    prm.ticket = status + 2 + (ticket_slot & 1);
    if (prm.n_items > grid && cudaMemsetAsync(prm.ticket, 0, sizeof(uint32_t), stream) != cudaSuccess)
        return static_cast<int>(cudaGetLastError());
    if (g_ev_before && cudaEventRecord(g_ev_before, stream) != cudaSuccess)
        return static_cast<int>(cudaGetLastError());
    bool launched = false;
    if constexpr (!kFuseQ)
        if (small) {
            attn_fwd_kernel<false, true><<<grid, NTHREADS, SMEM_BYTES, stream>>>(tmk, tmv, tmq, tmo, prm);
            launched = true;
        }
    if (!launched)
        attn_fwd_kernel<kFuseQ, false><<<grid, NTHREADS, SMEM_BYTES, stream>>>(tmk, tmv, tmq, tmo, prm);
    const cudaError_t le = cudaGetLastError();
    if (le != cudaSuccess)
        return static_cast<int>(le);
    if (g_ev_after && cudaEventRecord(g_ev_after, stream) != cudaSuccess)
        return static_cast<int>(cudaGetLastError());
    return static_cast<int>(cudaSuccess);
}

}  // namespace

int launch_forward(const Geometry &g, const int8_t *q_codes, const float *q_scales,
                   const int8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                   const float *v_scales, void *out, void *status, void *carrier, cudaStream_t stream,
                   bool withhold_v, bool reset_status, int ticket_slot)
{
    return launch_impl<false>(g, q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, out, status, carrier,
                              stream, withhold_v, reset_status, nullptr, ticket_slot);
}

int forward_init()
{
    if (!tensor_map_encoder())
        return 1;
    const cudaError_t r[3] = {kernel_attributes<false, false>(), kernel_attributes<true, false>(),
                              kernel_attributes<false, true>()};
    for (const cudaError_t e : r)
        if (e != cudaSuccess)
            return static_cast<int>(e);
    return 0;
}

int launch_forward_q_bf16(const Geometry &g, const void *q, const int8_t *k_codes, const float *k_scales,
                          const uint8_t *v_codes, const float *v_scales, void *out, void *status, void *carrier,
                          cudaStream_t stream)
{
    return launch_impl<true>(g, q, nullptr, k_codes, k_scales, v_codes, v_scales, out, status, carrier, stream,
                             false, true);
}

int launch_small(const Geometry &g, const SmallPrep &sp, void *out, void *status, void *carrier, cudaStream_t stream)
{
    return launch_impl<false>(g, sp.q_codes, sp.q_scales, sp.k_codes, sp.k_scales, sp.v_codes, sp.v_scales, out,
                              status, carrier, stream, false, true, &sp);
}

cudaError_t launch_test_p8_codes(int n_groups, const float *acc, const float *sig, const float *m, uint8_t *out,
                                 cudaStream_t stream)
{
    if (n_groups < 1)
        return cudaSuccess;
    test_p8_kernel<<<(n_groups + 127) / 128, 128, 0, stream>>>(n_groups, acc, sig, m,
                                                               reinterpret_cast<uint32_t *>(out), 0.0f);
    return cudaGetLastError();
}

cudaError_t launch_test_exp2_rn(int n, const float *x, float *out, cudaStream_t stream)
{
    if (n < 1)
        return cudaSuccess;
    test_exp2_kernel<<<(n + 255) / 256, 256, 0, stream>>>(n, x, out);
    return cudaGetLastError();
}

}  // namespace sattn
