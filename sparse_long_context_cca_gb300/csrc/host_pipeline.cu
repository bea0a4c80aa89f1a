// Prefill on host buffers: copy Q, K, V in, pool, run the fused attention,
// copy O (and optionally LSE, Kc, Vc) out.  The (batch, KV head) pairs are
// independent problems (pooling and attention never mix them), so the work is
// cut into slices of consecutive pairs and pipelined over three streams:
//
//   copy-in stream   Q/K/V of slice s  ->  buffer s % NBUF
//   caller's stream  pooling + attention of slice s
//   copy-out stream  O/LSE/Kc/Vc of slice s  ->  host
//
// so that the copies of one slice overlap the kernels of another and the two
// copy directions overlap each other.  A slice of pairs [p0, p1) is one
// contiguous range of rows in every [B, H, N, d] tensor (pair (b, k) owns query
// heads b*Hq + k*r .. + r - 1), so each tensor moves with one copy per slice.
//
// Ordering (events, one set per buffer):
//   copy-in(s)  waits out_done[buf] (slice s - NBUF has left the buffer)
//   kernels(s)  wait  in_done[buf]
//   copy-out(s) waits comp_done[buf]
// The caller's stream finally waits for the last copy-out, so work queued on it
// afterwards sees every output on the host.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "internal.h"

namespace cca {
namespace {

constexpr int NBUF = 3;
constexpr int64_t TARGET_SLICES = 8;
constexpr uint64_t ALIGN = 256;

uint64_t up(uint64_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }

struct Layout {
    int64_t pairs, slice_pairs, n_slices;
    int nbuf;
    uint64_t q, kv, c, lse;  // bytes per pair: Q (r heads), one of K/V, one of Kc/Vc, LSE (r heads)
    uint64_t buf_bytes;      // one buffer: Q, K, V, O, LSE, Kc, Vc of a full slice
};

Layout layout_of(const Shape &s, int dtype) {
    Layout L;
    const uint64_t e = dtype == 0 ? 2 : 4;
    const int r = s.Hq / s.Hkv;
    L.pairs = static_cast<int64_t>(s.B) * s.Hkv;
    L.slice_pairs = (L.pairs + TARGET_SLICES - 1) / TARGET_SLICES;
    L.n_slices = (L.pairs + L.slice_pairs - 1) / L.slice_pairs;
    L.nbuf = static_cast<int>(L.n_slices < NBUF ? L.n_slices : NBUF);
    L.kv = static_cast<uint64_t>(s.N) * s.d * e;
    L.q = L.kv * r;
    L.c = static_cast<uint64_t>(s.N / s.g) * s.d * e;
    L.lse = static_cast<uint64_t>(s.N) * r * 4;
    const uint64_t sp = static_cast<uint64_t>(L.slice_pairs);
    L.buf_bytes = 2 * up(sp * L.q) + 2 * up(sp * L.kv) + up(sp * L.lse) + 2 * up(sp * L.c);
    return L;
}

struct Pipe {
    int device = -1;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t entry = nullptr;
    cudaEvent_t in_done[NBUF] = {}, comp_done[NBUF] = {}, out_done[NBUF] = {};
};

std::mutex g_pipe_mu;
std::vector<Pipe *> g_pipes;  // idle pipes of every device; each call holds one exclusively

cudaError_t create_pipe(int device, Pipe **out) {
    Pipe *p = new Pipe();
    p->device = device;
    cudaError_t e = cudaStreamCreateWithFlags(&p->in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->entry, cudaEventDisableTiming);
    for (int k = 0; k < NBUF && e == cudaSuccess; ++k) {
        e = cudaEventCreateWithFlags(&p->in_done[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->comp_done[k], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->out_done[k], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        // destroy what was made; null handles are skipped
        if (p->in) cudaStreamDestroy(p->in);
        if (p->out) cudaStreamDestroy(p->out);
        if (p->entry) cudaEventDestroy(p->entry);
        for (int k = 0; k < NBUF; ++k) {
            if (p->in_done[k]) cudaEventDestroy(p->in_done[k]);
            if (p->comp_done[k]) cudaEventDestroy(p->comp_done[k]);
            if (p->out_done[k]) cudaEventDestroy(p->out_done[k]);
        }
        delete p;
        return e;
    }
    *out = p;
    return cudaSuccess;
}

// Takes an idle pipe of `device` from the pool, or makes one.  Events and
// streams are only re-used after the previous holder has finished enqueueing:
// a stream wait binds to the event's latest record at the time of the call.
cudaError_t acquire_pipe(int device, Pipe **out) {
    {
        std::lock_guard<std::mutex> lock(g_pipe_mu);
        for (size_t k = 0; k < g_pipes.size(); ++k) {
            if (g_pipes[k]->device == device) {
                *out = g_pipes[k];
                g_pipes.erase(g_pipes.begin() + static_cast<std::ptrdiff_t>(k));
                return cudaSuccess;
            }
        }
    }
    return create_pipe(device, out);
}

void release_pipe(Pipe *p) {
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    g_pipes.push_back(p);
}

cudaError_t copy(void *dst, const void *src, uint64_t bytes, cudaStream_t st) {
    return bytes == 0 ? cudaSuccess : cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, st);
}

cudaError_t enqueue(const Pipe &P, const Layout &L, int dtype, const uint8_t *hQ, const uint8_t *hK,
                    const uint8_t *hV, uint8_t *hO, uint8_t *hLSE, uint8_t *hKc, uint8_t *hVc, const Shape &s,
                    uint8_t *ws, int32_t *status, cudaStream_t stream) {
    const int r = s.Hq / s.Hkv;
    const uint64_t sp = static_cast<uint64_t>(L.slice_pairs);
    cudaError_t e = cudaEventRecord(P.entry, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.in, P.entry, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.entry, 0);
    for (int64_t sl = 0; sl < L.n_slices && e == cudaSuccess; ++sl) {
        const int buf = static_cast<int>(sl % L.nbuf);
        const uint64_t p0 = static_cast<uint64_t>(sl) * sp;
        const uint64_t np = static_cast<uint64_t>(L.pairs) - p0 < sp ? static_cast<uint64_t>(L.pairs) - p0 : sp;
        uint8_t *b = ws + buf * L.buf_bytes;
        uint8_t *dQ = b, *dO = dQ + up(sp * L.q), *dK = dO + up(sp * L.q), *dV = dK + up(sp * L.kv);
        uint8_t *dL = dV + up(sp * L.kv), *dKc = dL + up(sp * L.lse), *dVc = dKc + up(sp * L.c);

        if (sl >= L.nbuf) e = cudaStreamWaitEvent(P.in, P.out_done[buf], 0);
        if (e == cudaSuccess) e = copy(dQ, hQ + p0 * L.q, np * L.q, P.in);
        if (e == cudaSuccess) e = copy(dK, hK + p0 * L.kv, np * L.kv, P.in);
        if (e == cudaSuccess) e = copy(dV, hV + p0 * L.kv, np * L.kv, P.in);
        if (e == cudaSuccess) e = cudaEventRecord(P.in_done[buf], P.in);

        // the slice as its own problem: one batch of np KV heads and np * r query heads
        Shape t = s;
        t.B = 1;
        t.Hkv = static_cast<int>(np);
        t.Hq = static_cast<int>(np) * r;
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, P.in_done[buf], 0);
        if (e == cudaSuccess) e = launch_pool(dtype, dQ, dK, dV, dKc, dVc, t, status, stream);
        if (e == cudaSuccess) {
            if (dtype == 0)
                e = launch_attn_bf16_tc(dQ, dK, dV, dKc, dVc, dO, reinterpret_cast<float *>(dL), t, status, stream);
            else
                e = launch_attn_f32(reinterpret_cast<const float *>(dQ), reinterpret_cast<const float *>(dK),
                                    reinterpret_cast<const float *>(dV), reinterpret_cast<const float *>(dKc),
                                    reinterpret_cast<const float *>(dVc), reinterpret_cast<float *>(dO),
                                    reinterpret_cast<float *>(dL), t, stream);
        }
        if (e == cudaSuccess) e = cudaEventRecord(P.comp_done[buf], stream);

        if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.comp_done[buf], 0);
        if (e == cudaSuccess) e = copy(hO + p0 * L.q, dO, np * L.q, P.out);
        if (e == cudaSuccess && hLSE != nullptr) e = copy(hLSE + p0 * L.lse, dL, np * L.lse, P.out);
        if (e == cudaSuccess && hKc != nullptr) e = copy(hKc + p0 * L.c, dKc, np * L.c, P.out);
        if (e == cudaSuccess && hVc != nullptr) e = copy(hVc + p0 * L.c, dVc, np * L.c, P.out);
        if (e == cudaSuccess) e = cudaEventRecord(P.out_done[buf], P.out);
    }
    // the caller's stream resumes after the last copy-out (the copy-out stream is in order)
    const int last = static_cast<int>((L.n_slices - 1) % L.nbuf);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, P.out_done[last], 0);
    return e;
}

}  // namespace

uint64_t prefill_host_workspace_bytes(const Shape &s, int dtype) {
    const Layout L = layout_of(s, dtype);
    return static_cast<uint64_t>(L.nbuf) * L.buf_bytes;
}

cudaError_t launch_prefill_host(int dtype, const void *hQ, const void *hK, const void *hV, void *hO, float *hLSE,
                                void *hKc, void *hVc, const Shape &s, void *workspace, int32_t *status,
                                cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    Pipe *P = nullptr;
    if ((e = acquire_pipe(dev, &P)) != cudaSuccess) return e;
    const Layout L = layout_of(s, dtype);
    e = enqueue(*P, L, dtype, static_cast<const uint8_t *>(hQ), static_cast<const uint8_t *>(hK),
                static_cast<const uint8_t *>(hV), static_cast<uint8_t *>(hO), reinterpret_cast<uint8_t *>(hLSE),
                static_cast<uint8_t *>(hKc), static_cast<uint8_t *>(hVc), s, static_cast<uint8_t *>(workspace),
                status, stream);
    release_pipe(P);
    return e;
}

}  // namespace cca
