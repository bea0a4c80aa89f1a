// Fused core/local attention in fp32 on CUDA cores ("Core Context Aware
// Transformers for Long Context Language Modeling", Method section, fusion
// equation): query i takes one softmax over the visible core tokens
// (j < lo(i)/g) followed by the raw tokens of its window [lo(i), i].
//
// This path serves fp32 inputs, where tf32 tensor cores would not meet a 1e-4
// output tolerance.  One warp owns one query row; each lane holds d/32
// consecutive elements of q and of the output accumulator, a warp reduction
// forms every logit, and a running (max, sum) spans both segments so the core
// and local parts share a single normalisation.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "visibility.cuh"

namespace cca {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <int D>
struct RowState {
    static constexpr int PL = D / 32;
    float q[PL];
    float o[PL];
    float m = -INFINITY;  // running max, log2 domain
    float l = 0.f;

    __device__ __forceinline__ void step(const float *__restrict__ key, const float *__restrict__ val,
                                         int lane, float scale_log2) {
        float k[PL], v[PL];
#pragma unroll
        for (int e = 0; e < PL; ++e) {
            k[e] = key[lane * PL + e];
            v[e] = val[lane * PL + e];
        }
        float p = 0.f;
#pragma unroll
        for (int e = 0; e < PL; ++e) p = fmaf(q[e], k[e], p);
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) p += __shfl_xor_sync(kFull, p, s);
        const float x = p * scale_log2;
        const float mn = fmaxf(m, x);
        const float corr = exp2f(m - mn);
        const float e_x = exp2f(x - mn);
        l = l * corr + e_x;
#pragma unroll
        for (int e = 0; e < PL; ++e) o[e] = fmaf(e_x, v[e], o[e] * corr);
        m = mn;
    }
};

template <int D>
__global__ void __launch_bounds__(128) attn_f32_kernel(const float *__restrict__ Q, const float *__restrict__ K,
                                                       const float *__restrict__ V,
                                                       const float *__restrict__ Kc,
                                                       const float *__restrict__ Vc, float *__restrict__ O,
                                                       float *__restrict__ LSE, int Hq, int Hkv, int N,
                                                       int g, int w, int window_mode, float scale_log2,
                                                       int64_t total_rows, int q_off, int n_q, int kv_off,
                                                       int n_kv) {
    constexpr int PL = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t u = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (u >= total_rows) return;  // warp-uniform
    // Q, O and LSE hold the rows [q_off, q_off + n_q) of the N-token sequence, K and V the
    // raw tokens from kv_off on; i is the row's index in the sequence.
    const int64_t i = q_off + u % n_q;
    const int64_t bh = u / n_q;
    const int64_t b = bh / Hq, h = bh % Hq;
    const int64_t bk = b * Hkv + h / (Hq / Hkv);
    const int64_t G = N / g;

    RowState<D> st;
#pragma unroll
    for (int e = 0; e < PL; ++e) {
        st.q[e] = Q[u * D + lane * PL + e];
        st.o[e] = 0.f;
    }
    const int64_t n_core = visible_cores(static_cast<int>(i), w, g);
    const int64_t lo = window_start(static_cast<int>(i), w, g, window_mode);  // first raw token of the window
    const float *kc = Kc + bk * G * D;
    const float *vc = Vc + bk * G * D;
    for (int64_t j = 0; j < n_core; ++j) st.step(kc + j * D, vc + j * D, lane, scale_log2);
    const float *kk = K + bk * static_cast<int64_t>(n_kv) * D;
    const float *vv = V + bk * static_cast<int64_t>(n_kv) * D;
    for (int64_t t = lo; t <= i; ++t) st.step(kk + (t - kv_off) * D, vv + (t - kv_off) * D, lane, scale_log2);

    const float inv = 1.f / st.l;
#pragma unroll
    for (int e = 0; e < PL; ++e) O[u * D + lane * PL + e] = st.o[e] * inv;
    if (lane == 0) LSE[u] = (st.m + log2f(st.l)) * 0.6931471805599453f;
}

}  // namespace

cudaError_t launch_attn_f32(const float *Q, const float *K, const float *V, const float *Kc, const float *Vc,
                            float *O, float *LSE, const Shape &s, cudaStream_t stream, const RowRange &rr) {
    const int n_q = rr.n_q < 0 ? s.N : rr.n_q, n_kv = rr.n_kv < 0 ? s.N : rr.n_kv;
    const int64_t rows = static_cast<int64_t>(s.B) * s.Hq * n_q;
    const int warps = 4;
    const unsigned blocks = static_cast<unsigned>((rows + warps - 1) / warps);
    const float scale_log2 = s.scale * 1.4426950408889634f;
    if (s.d == 64) {
        attn_f32_kernel<64><<<blocks, warps * 32, 0, stream>>>(Q, K, V, Kc, Vc, O, LSE, s.Hq, s.Hkv, s.N, s.g,
                                                               s.w, s.window_mode, scale_log2, rows, rr.q_off, n_q,
                                                               rr.kv_off, n_kv);
    } else if (s.d == 128) {
        attn_f32_kernel<128><<<blocks, warps * 32, 0, stream>>>(Q, K, V, Kc, Vc, O, LSE, s.Hq, s.Hkv, s.N,
                                                                s.g, s.w, s.window_mode, scale_log2, rows, rr.q_off,
                                                                n_q, rr.kv_off, n_kv);
    } else {
        return cudaErrorNotSupported;
    }
    return cudaGetLastError();
}

}  // namespace cca
