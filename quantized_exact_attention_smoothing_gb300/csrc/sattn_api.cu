// sattn_api.cu -- the extern "C" boundary of libsattn.so (declared in include/sattn.h):
// argument validation, buffer sizes, and the stream-ordered launches.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/sattn.h"
#include "sattn_internal.cuh"

namespace {

using sattn::Geometry;

constexpr int64_t kMaxElems = int64_t(1) << 40;   // per tensor, keeps every index in int64

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int make_geometry(const sattn_shape *s, Geometry *g)
{
    if (!s || !g)
        return SATTN_ERR_INVALID;
    if (s->D != sattn::kHeadDim || s->B < 1 || s->Hq < 1 || s->Hkv < 1 || s->Hq % s->Hkv != 0 ||
        s->Nq < 1 || s->Nkv < 1 || (s->causal != 0 && s->causal != 1) ||
        (s->causal && s->Nq > s->Nkv))
        return SATTN_ERR_INVALID;
    if (static_cast<int64_t>(s->B) * s->Hq > 65535 || static_cast<int64_t>(s->B) * s->Hkv > 65535)
        return SATTN_ERR_INVALID;   // grid y limit of the launches
    const int64_t nq32 = sattn::pad_up(s->Nq, sattn::kQBlock);
    const int64_t nk128 = sattn::pad_up(s->Nkv, sattn::kVPad);
    if (static_cast<int64_t>(s->B) * s->Hq * nq32 * sattn::kHeadDim > kMaxElems ||
        static_cast<int64_t>(s->B) * s->Hkv * nk128 * sattn::kHeadDim > kMaxElems)
        return SATTN_ERR_INVALID;
    if (s->Nq > (1 << 30) || s->Nkv > (1 << 30))
        return SATTN_ERR_INVALID;
    g->B = s->B;
    g->Hq = s->Hq;
    g->Hkv = s->Hkv;
    g->Nq = s->Nq;
    g->Nkv = s->Nkv;
    g->causal = s->causal;
    g->sm_scale = s->sm_scale;
    g->nq32 = nq32;
    g->nk32 = sattn::pad_up(s->Nkv, sattn::kQBlock);
    g->nk128 = nk128;
    g->nbq = nq32 / sattn::kQBlock;
    g->nbk = g->nk32 / sattn::kQBlock;
    g->nchunks = (s->Nkv + sattn::kMeanChunk - 1) / sattn::kMeanChunk;
    return SATTN_OK;
}

size_t r16(size_t n) { return (n + 15) / 16 * 16; }
size_t r256(size_t n) { return (n + 255) / 256 * 256; }

void fill_sizes(const Geometry &g, sattn_sizes *z)
{
    const size_t bhq = static_cast<size_t>(g.B) * g.Hq, bhk = static_cast<size_t>(g.B) * g.Hkv;
    const size_t D = sattn::kHeadDim;
    z->q = r16(bhq * g.Nq * D * 2);
    z->k = r16(bhk * g.Nkv * D * 2);
    z->v = z->k;
    z->q_codes = r16(bhq * g.nq32 * D);
    z->q_scales = r16(bhq * g.nbq * 4);
    z->k_codes = r16(bhk * g.nk32 * D);
    z->k_scales = r16(bhk * g.nbk * 4);
    z->k_mean = r16(bhk * D * 4);
    z->v_codes = r16(bhk * D * g.nk128);
    z->v_scales = r16(bhk * D * 4);
    z->out = r16(bhq * g.Nq * D * 2);
    z->prepare_workspace = r16(sattn::prepare_workspace_bytes(g));
    z->forward_workspace = r16(sattn::forward_workspace_bytes(g));
    z->arena = r256(z->q) + r256(z->k) + r256(z->v) + r256(z->q_codes) + r256(z->q_scales) +
               r256(z->k_codes) + r256(z->k_scales) + r256(z->k_mean) + r256(z->v_codes) + r256(z->v_scales) +
               r256(z->out) + 2 * r256(z->prepare_workspace) + r256(sattn::kStatusBytes) +
               2 * r256(sattn::carrier_bytes(g));
}

// The current device must be compute capability 10.3; the answer is cached per device.
int check_device()
{
    static int verdict[64];   // 0 unknown, 1 good, 2 bad
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SATTN_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(mu);
    if (verdict[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return SATTN_ERR_DEVICE;
        verdict[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return verdict[dev] == 1 ? SATTN_OK : SATTN_ERR_DEVICE;
}

constexpr int kMaxHostChunks = 8;

// Helper streams and events of the library, created once per device: the
// host-buffer pipeline's three stage streams, and the stream on which the
// preparation quantises Q while the K/V kernels run on the caller's stream.
struct DeviceStreams {
    cudaStream_t h2d = nullptr, compute = nullptr, d2h = nullptr, qprep = nullptr, vprep = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, in[kMaxHostChunks] = {}, done[kMaxHostChunks] = {};
    cudaEvent_t qfork = nullptr, qjoin = nullptr, vfork = nullptr, vjoin = nullptr;
};

struct HelperStreams {
    std::mutex mu;
    DeviceStreams dev[64];
};

HelperStreams &helpers()
{
    static HelperStreams h;
    return h;
}

bool create_streams(DeviceStreams &d)
{
    if (d.h2d)
        return true;
    bool ok = cudaStreamCreateWithFlags(&d.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&d.compute, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&d.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&d.join, cudaEventDisableTiming) == cudaSuccess;
    for (int c = 0; c < kMaxHostChunks && ok; ++c)
        ok = cudaEventCreateWithFlags(&d.in[c], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&d.done[c], cudaEventDisableTiming) == cudaSuccess;
    if (!ok)
        d.h2d = nullptr;   // retried on the next call
    return ok;
}

bool create_qprep_stream(DeviceStreams &d)
{
    if (d.qprep)
        return true;
    const bool ok = cudaStreamCreateWithFlags(&d.qprep, cudaStreamNonBlocking) == cudaSuccess &&
                    cudaStreamCreateWithFlags(&d.vprep, cudaStreamNonBlocking) == cudaSuccess &&
                    cudaEventCreateWithFlags(&d.qfork, cudaEventDisableTiming) == cudaSuccess &&
                    cudaEventCreateWithFlags(&d.qjoin, cudaEventDisableTiming) == cudaSuccess &&
                    cudaEventCreateWithFlags(&d.vfork, cudaEventDisableTiming) == cudaSuccess &&
                    cudaEventCreateWithFlags(&d.vjoin, cudaEventDisableTiming) == cudaSuccess;
    if (!ok)
        d.qprep = nullptr;   // retried on the next call
    return ok;
}

int prepare_impl(const Geometry &g, const void *q, const void *k, const void *v, int8_t *q_codes,
                 float *q_scales, int8_t *k_codes, float *k_scales, float *k_mean, uint8_t *v_codes,
                 float *v_scales, void *workspace, cudaStream_t stream)
{
    // q, q_codes and q_scales are all null for the K/V-only preparation
    const bool with_q = q != nullptr;
    const void *ptrs[] = {k, v, k_codes, k_scales, k_mean, v_codes, v_scales, workspace,
                          with_q ? q : k, with_q ? q_codes : k, with_q ? q_scales : k};
    for (const void *p : ptrs) {
        if (!p)
            return SATTN_ERR_INVALID;
        if (!aligned16(p))
            return SATTN_ERR_MISALIGNED;
    }
    const int dc = check_device();
    if (dc != SATTN_OK)
        return dc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return SATTN_ERR_DEVICE;
    // Q's quantisation depends on nothing the K/V kernels compute: it runs on
    // a helper stream, concurrently with them on `stream`; after the K/V
    // statistics, V's quantisation runs on a second helper stream beside K's.
    // `stream` waits for both at the end (all work stays ordered on `stream`
    // for the caller).
    HelperStreams &h = helpers();
    std::lock_guard<std::mutex> lock(h.mu);
    DeviceStreams &ds = h.dev[dev];
    if (!with_q || !create_qprep_stream(ds))
        return sattn::launch_prepare(g, q, k, v, q_codes, q_scales, k_codes, k_scales, k_mean, v_codes, v_scales,
                                     workspace, stream) == cudaSuccess
                   ? SATTN_OK
                   : SATTN_ERR_LAUNCH;
    if (cudaEventRecord(ds.qfork, stream) != cudaSuccess || cudaStreamWaitEvent(ds.qprep, ds.qfork, 0) != cudaSuccess ||
        sattn::launch_prepare_q(g, q, q_codes, q_scales, ds.qprep) != cudaSuccess ||
        cudaEventRecord(ds.qjoin, ds.qprep) != cudaSuccess ||
        sattn::launch_prepare_kv_split(g, k, v, k_codes, k_scales, k_mean, v_codes, v_scales, workspace, stream,
                                       ds.vprep, ds.vfork, ds.vjoin) != cudaSuccess ||
        cudaStreamWaitEvent(stream, ds.qjoin, 0) != cudaSuccess)
        return SATTN_ERR_LAUNCH;
    return SATTN_OK;
}

// The forward workspace: the status block, then the FP16 carrier of the K codes.
void *carrier_of(void *workspace) { return static_cast<char *>(workspace) + sattn::kStatusBytes; }

// q_bf16 non-null: the forward that quantises Q itself (q_codes, q_scales unused)
int forward_impl(const Geometry &g, const int8_t *q_codes, const float *q_scales,
                 const int8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                 const float *v_scales, void *out, void *workspace, cudaStream_t stream,
                 bool withhold_v = false, const void *q_bf16 = nullptr)
{
    const bool fused = q_bf16 != nullptr;
    const void *ptrs[] = {fused ? q_bf16 : q_codes, fused ? q_bf16 : q_scales, k_codes, k_scales, v_codes,
                          v_scales, out, workspace};
    for (const void *p : ptrs) {
        if (!p)
            return SATTN_ERR_INVALID;
        if (!aligned16(p))
            return SATTN_ERR_MISALIGNED;
    }
    const int dev = check_device();
    if (dev != SATTN_OK)
        return dev;
    const int rc = fused ? sattn::launch_forward_q_bf16(g, q_bf16, k_codes, k_scales, v_codes, v_scales, out,
                                                        workspace, carrier_of(workspace), stream)
                         : sattn::launch_forward(g, q_codes, q_scales, k_codes, k_scales, v_codes, v_scales,
                                                 out, workspace, carrier_of(workspace), stream, withhold_v);
    if (rc == 1)
        return SATTN_ERR_DEVICE;   // no tensor-map encoder in this driver
    return rc == 0 ? SATTN_OK : SATTN_ERR_LAUNCH;
}

// ---------------------------------------------------------------------------
// The host-buffer path, pipelined: the (batch, KV head) units are independent
// problems (their K mean and V scales are their own), so the units are cut
// into contiguous chunks, each a problem of one batch and several KV heads
// whose tensors are contiguous slices of the whole ones.  Three helper
// streams of the library carry the stages: the host-to-device copies run back
// to back on one, the chunks' kernels alternate between the caller's stream
// and a second one (so one chunk's forward tail overlaps the next chunk's
// start), and the copies back run on a third; events hand each chunk from
// stage to stage.  Every chunk's forward reports into the one status block,
// cleared once before the fork; the forwards of the two kernel streams, which
// may run at the same time, take their work items from separate counter words
// of that block (ticket slot = chunk parity).
// ---------------------------------------------------------------------------
struct HostBuffers {
    void *q, *k, *v, *out, *carrier[2], *pws[2], *fws;
    int8_t *q_codes, *k_codes;
    float *q_scales, *k_scales, *k_mean, *v_scales;
    uint8_t *v_codes;
};

// Chunk plan for the pipeline: at most kMaxHostChunks chunks, each of at
// least two work items of the forward per SM (smaller chunks would leave SMs
// idle), sized like a ramp (weights 1, 2, 3, ..., 3, 2, 1): the first chunk's
// copy in and the last chunk's kernels and copy back are the parts of the
// pipeline that nothing overlaps, so those chunks are the small ones.
// bound[c] .. bound[c + 1] are the units of chunk c; returns the chunk count.
int host_chunks(const Geometry &g, int n_sm, int64_t (&bound)[kMaxHostChunks + 1])
{
    const int64_t units = static_cast<int64_t>(g.B) * g.Hkv;
    const int64_t items_per_unit = (g.Nq + sattn::kQTile - 1) / sattn::kQTile * (g.Hq / g.Hkv);
    const int64_t min_units = (2 * static_cast<int64_t>(n_sm) + items_per_unit - 1) / items_per_unit;
    int nc = static_cast<int>(units / min_units < kMaxHostChunks ? units / min_units : kMaxHostChunks);
    if (nc < 1)
        nc = 1;
    for (; nc > 1; --nc) {
        int64_t wsum = 0, w[kMaxHostChunks];
        for (int c = 0; c < nc; ++c)
            wsum += w[c] = (c + 1 < nc - c ? c + 1 : nc - c);
        int64_t acc = 0;
        bool ok = true;
        bound[0] = 0;
        for (int c = 0; c < nc; ++c) {
            acc += w[c];
            bound[c + 1] = (units * acc + wsum / 2) / wsum;
            ok = ok && bound[c + 1] - bound[c] >= min_units;
        }
        if (ok)
            return nc;
        // the ramp leaves an end chunk too small: equal chunks if they fit
        bool eq = true;
        for (int c = 0; c <= nc; ++c)
            bound[c] = units * c / nc;
        for (int c = 0; c < nc; ++c)
            eq = eq && bound[c + 1] - bound[c] >= min_units;
        if (eq)
            return nc;
    }
    bound[0] = 0;
    bound[1] = units;
    return 1;
}

int attention_host_pipelined(const Geometry &g, const sattn_shape &shape, const void *q_host, const void *k_host,
                             const void *v_host, void *out_host, const HostBuffers &hb, cudaStream_t s0)
{
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SATTN_ERR_DEVICE;
    int64_t bound[kMaxHostChunks + 1];
    const int nc = host_chunks(g, n_sm, bound);
    const int grp = g.Hq / g.Hkv;
    const size_t D = sattn::kHeadDim;

    HelperStreams &h = helpers();
    std::lock_guard<std::mutex> lock(h.mu);   // the events are shared by the calls on a device
    DeviceStreams &ds = h.dev[dev];
    if (nc > 1 && !create_streams(ds))
        return SATTN_ERR_DEVICE;
    if (cudaMemsetAsync(hb.fws, 0, 2 * sizeof(uint32_t), s0) != cudaSuccess)
        return SATTN_ERR_LAUNCH;
    // single chunk: every stage on the caller's stream
    cudaStream_t s_in = nc > 1 ? ds.h2d : s0, s_out = nc > 1 ? ds.d2h : s0;
    cudaStream_t s_c[2] = {s0, nc > 1 ? ds.compute : s0};
    if (nc > 1) {
        if (cudaEventRecord(ds.fork, s0) != cudaSuccess || cudaStreamWaitEvent(ds.h2d, ds.fork, 0) != cudaSuccess ||
            cudaStreamWaitEvent(ds.compute, ds.fork, 0) != cudaSuccess ||
            cudaStreamWaitEvent(ds.d2h, ds.fork, 0) != cudaSuccess)
            return SATTN_ERR_LAUNCH;
    }
    auto at = [](const void *base, size_t off) { return static_cast<const char *>(base) + off; };
    auto atw = [](void *base, size_t off) { return static_cast<char *>(base) + off; };
    auto chunk_units = [&](int c, int64_t &u0, int64_t &nu) {
        u0 = bound[c];
        nu = bound[c + 1] - u0;
    };
    // stage 1: host-to-device copies, back to back
    for (int c = 0; c < nc; ++c) {
        int64_t u0, nu;
        chunk_units(c, u0, nu);
        const size_t qo = static_cast<size_t>(u0) * grp * g.Nq * D * 2, ko = static_cast<size_t>(u0) * g.Nkv * D * 2;
        const size_t qb = static_cast<size_t>(nu) * grp * g.Nq * D * 2, kb = static_cast<size_t>(nu) * g.Nkv * D * 2;
        if (cudaMemcpyAsync(atw(hb.q, qo), at(q_host, qo), qb, cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
            cudaMemcpyAsync(atw(hb.k, ko), at(k_host, ko), kb, cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
            cudaMemcpyAsync(atw(hb.v, ko), at(v_host, ko), kb, cudaMemcpyHostToDevice, s_in) != cudaSuccess)
            return SATTN_ERR_LAUNCH;
        if (nc > 1 && cudaEventRecord(ds.in[c], s_in) != cudaSuccess)
            return SATTN_ERR_LAUNCH;
    }
    // stage 2: preparation and forward of each chunk, alternating between two streams
    for (int c = 0; c < nc; ++c) {
        int64_t u0, nu;
        chunk_units(c, u0, nu);
        cudaStream_t st = s_c[c & 1];
        if (nc > 1 && cudaStreamWaitEvent(st, ds.in[c], 0) != cudaSuccess)
            return SATTN_ERR_LAUNCH;
        sattn_shape cs = shape;                 // one batch of nu KV heads
        cs.B = 1;
        cs.Hkv = static_cast<int32_t>(nu);
        cs.Hq = static_cast<int32_t>(nu * grp);
        Geometry gc;
        if (make_geometry(&cs, &gc) != SATTN_OK)
            return SATTN_ERR_INVALID;
        const size_t qh = static_cast<size_t>(u0) * grp, kh = static_cast<size_t>(u0);   // first q / kv head
        void *q = atw(hb.q, qh * g.Nq * D * 2), *k = atw(hb.k, kh * g.Nkv * D * 2), *v = atw(hb.v, kh * g.Nkv * D * 2);
        void *out = atw(hb.out, qh * g.Nq * D * 2);
        int8_t *q_codes = hb.q_codes + qh * g.nq32 * D;
        float *q_scales = hb.q_scales + qh * g.nbq;
        int8_t *k_codes = hb.k_codes + kh * g.nk32 * D;
        float *k_scales = hb.k_scales + kh * g.nbk;
        float *k_mean = hb.k_mean + kh * D;
        uint8_t *v_codes = hb.v_codes + kh * D * g.nk128;
        float *v_scales = hb.v_scales + kh * D;
        if (sattn::launch_prepare(gc, q, k, v, q_codes, q_scales, k_codes, k_scales, k_mean, v_codes, v_scales,
                                  hb.pws[c & 1], st) != cudaSuccess)
            return SATTN_ERR_LAUNCH;
        const int frc = sattn::launch_forward(gc, q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, out,
                                              hb.fws, hb.carrier[c & 1], st, false, false, c & 1);
        if (frc == 1)
            return SATTN_ERR_DEVICE;
        if (frc != 0)
            return SATTN_ERR_LAUNCH;
        if (nc > 1 && cudaEventRecord(ds.done[c], st) != cudaSuccess)
            return SATTN_ERR_LAUNCH;
    }
    // stage 3: device-to-host copies as each chunk's output is complete
    for (int c = 0; c < nc; ++c) {
        int64_t u0, nu;
        chunk_units(c, u0, nu);
        const size_t qo = static_cast<size_t>(u0) * grp * g.Nq * D * 2;
        const size_t qb = static_cast<size_t>(nu) * grp * g.Nq * D * 2;
        if (nc > 1 && cudaStreamWaitEvent(s_out, ds.done[c], 0) != cudaSuccess)
            return SATTN_ERR_LAUNCH;
        if (cudaMemcpyAsync(atw(out_host, qo), at(hb.out, qo), qb, cudaMemcpyDeviceToHost, s_out) != cudaSuccess)
            return SATTN_ERR_LAUNCH;
    }
    // join: the copies back wait for every chunk, so their end is the end of the call
    if (nc > 1 && (cudaEventRecord(ds.join, ds.d2h) != cudaSuccess || cudaStreamWaitEvent(s0, ds.join, 0) != cudaSuccess))
        return SATTN_ERR_LAUNCH;
    return SATTN_OK;
}

}  // namespace

extern "C" {

int sattn_query_sizes(const sattn_shape *shape, sattn_sizes *sizes)
{
    Geometry g;
    const int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    if (!sizes)
        return SATTN_ERR_INVALID;
    fill_sizes(g, sizes);
    return SATTN_OK;
}

int sattn_prepare(const sattn_shape *shape, const void *q, const void *k, const void *v,
                  int8_t *q_codes, float *q_scales, int8_t *k_codes, float *k_scales,
                  float *k_mean, uint8_t *v_codes, float *v_scales, void *workspace, void *stream)
{
    Geometry g;
    const int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    if (!q || !q_codes || !q_scales)
        return SATTN_ERR_INVALID;
    return prepare_impl(g, q, k, v, q_codes, q_scales, k_codes, k_scales, k_mean, v_codes, v_scales, workspace,
                        static_cast<cudaStream_t>(stream));
}

int sattn_forward(const sattn_shape *shape, const int8_t *q_codes, const float *q_scales,
                  const int8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                  const float *v_scales, void *out, void *workspace, void *stream)
{
    Geometry g;
    const int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    return forward_impl(g, q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, out, workspace,
                        static_cast<cudaStream_t>(stream));
}

int sattn_prepare_kv(const sattn_shape *shape, const void *k, const void *v, int8_t *k_codes,
                     float *k_scales, float *k_mean, uint8_t *v_codes, float *v_scales, void *workspace,
                     void *stream)
{
    Geometry g;
    const int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    return prepare_impl(g, nullptr, k, v, nullptr, nullptr, k_codes, k_scales, k_mean, v_codes, v_scales,
                        workspace, static_cast<cudaStream_t>(stream));
}

namespace {
int prepare_kv_onepass_impl(const sattn_shape *shape, const void *k, const void *v, int8_t *k_codes,
                            float *k_scales, float *k_mean, uint8_t *v_codes, float *v_scales, void *workspace,
                            void *stream, bool withhold)
{
    Geometry g;
    const int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    const void *ptrs[] = {k, v, k_codes, k_scales, k_mean, v_codes, v_scales, workspace};
    for (const void *p : ptrs) {
        if (!p)
            return SATTN_ERR_INVALID;
        if (!aligned16(p))
            return SATTN_ERR_MISALIGNED;
    }
    const int dc = check_device();
    if (dc != SATTN_OK)
        return dc;
    return sattn::launch_prepare_kv_fused(g, k, v, k_codes, k_scales, k_mean, v_codes, v_scales, workspace,
                                          static_cast<cudaStream_t>(stream), withhold) == cudaSuccess
               ? SATTN_OK
               : SATTN_ERR_LAUNCH;
}
}  // namespace

int sattn_prepare_kv_onepass(const sattn_shape *shape, const void *k, const void *v, int8_t *k_codes,
                             float *k_scales, float *k_mean, uint8_t *v_codes, float *v_scales, void *workspace,
                             void *stream)
{
    return prepare_kv_onepass_impl(shape, k, v, k_codes, k_scales, k_mean, v_codes, v_scales, workspace, stream,
                                   false);
}

int sattn_test_prepare_kv_onepass_withhold(const sattn_shape *shape, const void *k, const void *v, int8_t *k_codes,
                                           float *k_scales, float *k_mean, uint8_t *v_codes, float *v_scales,
                                           void *workspace, void *stream)
{
    return prepare_kv_onepass_impl(shape, k, v, k_codes, k_scales, k_mean, v_codes, v_scales, workspace, stream,
                                   true);
}

int sattn_check_prepare_status(const sattn_shape *shape, const void *prepare_workspace, void *stream)
{
    Geometry g;
    const int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    if (!prepare_workspace)
        return SATTN_ERR_INVALID;
    if (!aligned16(prepare_workspace))
        return SATTN_ERR_MISALIGNED;
    uint32_t word = 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SATTN_ERR_DEVICE;
    if (cudaMemcpy(&word, static_cast<const char *>(prepare_workspace) + sattn::prepare_status_offset(g),
                   sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SATTN_ERR_DEVICE;
    return word != 0 ? SATTN_ERR_TIMEOUT : SATTN_OK;
}

int sattn_forward_q_bf16(const sattn_shape *shape, const void *q, const int8_t *k_codes, const float *k_scales,
                         const uint8_t *v_codes, const float *v_scales, void *out, void *workspace, void *stream)
{
    Geometry g;
    const int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    return forward_impl(g, nullptr, nullptr, k_codes, k_scales, v_codes, v_scales, out, workspace,
                        static_cast<cudaStream_t>(stream), false, q);
}

int sattn_attention_small(const sattn_shape *shape, const void *q, const void *k, const void *v, int8_t *q_codes,
                          float *q_scales, int8_t *k_codes, float *k_scales, float *k_mean, uint8_t *v_codes,
                          float *v_scales, void *out, void *workspace, void *stream)
{
    Geometry g;
    const int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    if (g.B != 1 || g.Hq != 1 || g.Hkv != 1 || g.Nq > sattn::kQTile || g.Nkv > sattn::kSmallMaxNkv)
        return SATTN_ERR_INVALID;
    const void *ptrs[] = {q, k, v, q_codes, q_scales, k_codes, k_scales, k_mean, v_codes, v_scales, out, workspace};
    for (const void *p : ptrs) {
        if (!p)
            return SATTN_ERR_INVALID;
        if (!aligned16(p))
            return SATTN_ERR_MISALIGNED;
    }
    const int dev = check_device();
    if (dev != SATTN_OK)
        return dev;
    const sattn::SmallPrep sp{q, k, v, q_codes, q_scales, k_codes, k_scales, k_mean, v_codes, v_scales};
    const int lc = sattn::launch_small(g, sp, out, workspace, carrier_of(workspace), static_cast<cudaStream_t>(stream));
    if (lc == 1)
        return SATTN_ERR_DEVICE;   // no tensor-map encoder in this driver
    return lc == 0 ? SATTN_OK : SATTN_ERR_LAUNCH;
}

int sattn_test_forward_withhold_v(const sattn_shape *shape, const int8_t *q_codes, const float *q_scales,
                                  const int8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                                  const float *v_scales, void *out, void *workspace, void *stream)
{
    Geometry g;
    const int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    return forward_impl(g, q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, out, workspace,
                        static_cast<cudaStream_t>(stream), true);
}

int sattn_test_int8_quantiser(uint32_t amax_lo, uint32_t amax_hi, unsigned long long *result, void *stream)
{
    if (!result || amax_lo < 1 || amax_hi > 0x7f80u || amax_lo >= amax_hi)
        return SATTN_ERR_INVALID;
    if (!aligned16(result))
        return SATTN_ERR_MISALIGNED;
    const int dev = check_device();
    if (dev != SATTN_OK)
        return dev;
    return sattn::launch_int8_quantiser_sweep(amax_lo, amax_hi, result, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? SATTN_OK
               : SATTN_ERR_LAUNCH;
}

int sattn_test_p8_codes(int n_groups, const float *acc, const float *sig, const float *m, uint8_t *out,
                        void *stream)
{
    if (n_groups < 0 || (n_groups > 0 && (!acc || !sig || !m || !out)))
        return SATTN_ERR_INVALID;
    if (!aligned16(acc) || !aligned16(out))
        return SATTN_ERR_MISALIGNED;
    const int dev = check_device();
    if (dev != SATTN_OK)
        return dev;
    return sattn::launch_test_p8_codes(n_groups, acc, sig, m, out, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SATTN_OK
               : SATTN_ERR_LAUNCH;
}

int sattn_test_exp2(int n, const float *x, float *out, void *stream)
{
    if (n < 0 || (n > 0 && (!x || !out)))
        return SATTN_ERR_INVALID;
    const int dev = check_device();
    if (dev != SATTN_OK)
        return dev;
    return sattn::launch_test_exp2_rn(n, x, out, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SATTN_OK
               : SATTN_ERR_LAUNCH;
}

int sattn_measure_mma_rate(int kind, int n, int iters, double *flop_per_clk_sm, double *tflops)
{
    if ((kind != 0 && kind != 1) || n < 16 || n > 256 || n % 16 != 0 || iters < 1 || iters > (1 << 20) ||
        !flop_per_clk_sm || !tflops)
        return SATTN_ERR_INVALID;
    const int dev = check_device();
    if (dev != SATTN_OK)
        return dev;
    return sattn::measure_mma_rate(kind, n, iters, flop_per_clk_sm, tflops) == 0 ? SATTN_OK : SATTN_ERR_LAUNCH;
}

int sattn_profile_events(void *before, void *after)
{
    if ((before == nullptr) != (after == nullptr))
        return SATTN_ERR_INVALID;
    sattn::set_profile_events(static_cast<cudaEvent_t>(before), static_cast<cudaEvent_t>(after));
    return SATTN_OK;
}

int sattn_test_host_chunks(const sattn_shape *shape, int n_sm, int64_t *bounds, int *nchunks)
{
    Geometry g;
    const int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    if (!bounds || !nchunks || n_sm < 1)
        return SATTN_ERR_INVALID;
    int64_t b[kMaxHostChunks + 1];
    *nchunks = host_chunks(g, n_sm, b);
    for (int c = 0; c <= *nchunks; ++c)
        bounds[c] = b[c];
    return SATTN_OK;
}

int sattn_check_status(const void *forward_workspace, void *stream)
{
    if (!forward_workspace)
        return SATTN_ERR_INVALID;
    if (!aligned16(forward_workspace))
        return SATTN_ERR_MISALIGNED;
    uint32_t words[2] = {0, 0};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return SATTN_ERR_DEVICE;
    if (cudaMemcpy(words, forward_workspace, sizeof words, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SATTN_ERR_DEVICE;
    return words[0] != 0 ? SATTN_ERR_TIMEOUT : SATTN_OK;
}

int sattn_attention_host(const sattn_shape *shape, const void *q_host, const void *k_host,
                         const void *v_host, void *out_host, void *arena, size_t arena_bytes,
                         void *stream)
{
    Geometry g;
    int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    if (!q_host || !k_host || !v_host || !out_host || !arena)
        return SATTN_ERR_INVALID;
    if (!aligned16(arena))
        return SATTN_ERR_MISALIGNED;
    sattn_sizes z;
    fill_sizes(g, &z);
    if (arena_bytes < z.arena)
        return SATTN_ERR_INVALID;
    rc = check_device();
    if (rc != SATTN_OK)
        return rc;
    char *p = static_cast<char *>(arena);
    auto take = [&p](size_t n) {
        char *r = p;
        p += r256(n);
        return r;
    };
    HostBuffers hb;
    hb.q = take(z.q);
    hb.k = take(z.k);
    hb.v = take(z.v);
    hb.q_codes = reinterpret_cast<int8_t *>(take(z.q_codes));
    hb.q_scales = reinterpret_cast<float *>(take(z.q_scales));
    hb.k_codes = reinterpret_cast<int8_t *>(take(z.k_codes));
    hb.k_scales = reinterpret_cast<float *>(take(z.k_scales));
    hb.k_mean = reinterpret_cast<float *>(take(z.k_mean));
    hb.v_codes = reinterpret_cast<uint8_t *>(take(z.v_codes));
    hb.v_scales = reinterpret_cast<float *>(take(z.v_scales));
    hb.out = take(z.out);
    hb.pws[0] = take(z.prepare_workspace);
    hb.pws[1] = take(z.prepare_workspace);
    hb.fws = take(sattn::kStatusBytes);
    hb.carrier[0] = take(sattn::carrier_bytes(g));
    hb.carrier[1] = take(sattn::carrier_bytes(g));
    return attention_host_pipelined(g, *shape, q_host, k_host, v_host, out_host, hb,
                                    static_cast<cudaStream_t>(stream));
}

struct sattn_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

int sattn_graph_create(const sattn_shape *shape, const void *q, const void *k, const void *v, int8_t *q_codes,
                       float *q_scales, int8_t *k_codes, float *k_scales, float *k_mean, uint8_t *v_codes,
                       float *v_scales, void *prepare_workspace, void *out, void *forward_workspace,
                       sattn_graph **graph)
{
    if (!graph)
        return SATTN_ERR_INVALID;
    *graph = nullptr;
    Geometry g;
    int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    const void *ptrs[] = {q, k, v, q_codes, q_scales, k_codes, k_scales, k_mean, v_codes, v_scales,
                          prepare_workspace, out, forward_workspace};
    for (const void *ptr : ptrs) {
        if (!ptr)
            return SATTN_ERR_INVALID;
        if (!aligned16(ptr))
            return SATTN_ERR_MISALIGNED;
    }
    rc = check_device();
    if (rc != SATTN_OK)
        return rc;
    const int init = sattn::forward_init();   // no one-time setup calls inside the capture
    if (init == 1)
        return SATTN_ERR_DEVICE;
    if (init != 0)
        return SATTN_ERR_LAUNCH;
    {   // nor the creation of the preparation's helper streams
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
            return SATTN_ERR_DEVICE;
        HelperStreams &h = helpers();
        std::lock_guard<std::mutex> lock(h.mu);
        if (!create_qprep_stream(h.dev[dev]))
            return SATTN_ERR_DEVICE;
    }
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess)
        return SATTN_ERR_DEVICE;
    sattn_graph *gr = new sattn_graph;
    rc = SATTN_OK;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        rc = SATTN_ERR_LAUNCH;
    } else {
        rc = prepare_impl(g, q, k, v, q_codes, q_scales, k_codes, k_scales, k_mean, v_codes, v_scales,
                          prepare_workspace, cs);
        if (rc == SATTN_OK)
            rc = forward_impl(g, q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, out, forward_workspace,
                              cs);
        const cudaError_t end = cudaStreamEndCapture(cs, &gr->graph);   // ends the capture in every case
        if (rc == SATTN_OK && end != cudaSuccess)
            rc = SATTN_ERR_LAUNCH;
    }
    if (rc == SATTN_OK && cudaGraphInstantiate(&gr->exec, gr->graph, 0) != cudaSuccess)
        rc = SATTN_ERR_LAUNCH;
    cudaStreamDestroy(cs);
    if (rc != SATTN_OK) {
        sattn_graph_destroy(gr);
        return rc;
    }
    *graph = gr;
    return SATTN_OK;
}

int sattn_graph_launch(sattn_graph *graph, void *stream)
{
    if (!graph || !graph->exec)
        return SATTN_ERR_INVALID;
    return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SATTN_OK
                                                                                          : SATTN_ERR_LAUNCH;
}

int sattn_graph_destroy(sattn_graph *graph)
{
    if (!graph)
        return SATTN_ERR_INVALID;
    if (graph->exec)
        cudaGraphExecDestroy(graph->exec);
    if (graph->graph)
        cudaGraphDestroy(graph->graph);
    delete graph;
    return SATTN_OK;
}

const char *sattn_status_string(int status)
{
    switch (status) {
    case SATTN_OK: return "ok";
    case SATTN_ERR_INVALID: return "invalid argument";
    case SATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case SATTN_ERR_DEVICE: return "unsupported device or CUDA runtime failure";
    case SATTN_ERR_LAUNCH: return "kernel launch failed";
    case SATTN_ERR_TIMEOUT: return "device wait timed out";
    case SATTN_ERR_SCRATCH_LIMIT: return "shape needs more than the fixed no-alloc scratch array";
    default: return "unknown status";
    }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// sattn_prepare_noalloc: the preparation pass with its scratch (per-chunk K
// column sums and V column maxima) in a fixed array of this library's device
// memory instead of a caller-provided workspace.  Declared in sattn.h.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_prepare_scratch[SATTN_NOALLOC_SCRATCH_BYTES];

// Device address of g_prepare_scratch in the current context.  In host code
// the array's name is only a host-side handle; the kernels must be given this
// address.  Looked up on every call (the runtime keeps the module's symbol
// table), so a device reset or a new primary context never leaves a stale
// address behind.
int prepare_scratch_address(void **out)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prepare_scratch) != cudaSuccess || !p)
        return SATTN_ERR_DEVICE;
    *out = p;
    return SATTN_OK;
}

}  // namespace

extern "C" int sattn_prepare_noalloc(const sattn_shape *shape, const void *q, const void *k,
                                     const void *v, int8_t *q_codes, float *q_scales,
                                     int8_t *k_codes, float *k_scales, float *k_mean,
                                     uint8_t *v_codes, float *v_scales, void *stream)
{
    Geometry g;
    int rc = make_geometry(shape, &g);
    if (rc != SATTN_OK)
        return rc;
    const void *ptrs[] = {q, k, v, q_codes, q_scales, k_codes, k_scales, k_mean, v_codes, v_scales};
    for (const void *p : ptrs) {
        if (!p)
            return SATTN_ERR_INVALID;
        if (!aligned16(p))
            return SATTN_ERR_MISALIGNED;
    }
    if (sattn::prepare_workspace_bytes(g) > SATTN_NOALLOC_SCRATCH_BYTES)
        return SATTN_ERR_SCRATCH_LIMIT;
    rc = check_device();
    if (rc != SATTN_OK)
        return rc;
    void *scratch = nullptr;
    rc = prepare_scratch_address(&scratch);
    if (rc != SATTN_OK)
        return rc;
    return sattn::launch_prepare(g, q, k, v, q_codes, q_scales, k_codes, k_scales, k_mean, v_codes, v_scales,
                                 scratch, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SATTN_OK
               : SATTN_ERR_LAUNCH;
}
