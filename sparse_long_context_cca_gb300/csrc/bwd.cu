// Backward pass of CCA prefill: gradients of the loss sum(dO * O) with respect
// to Q, K and V, through the fused attention (fusion equation) and through the
// global-aware pooling (pooling equation) of "Core Context Aware Transformers
// for Long Context Language Modeling", Method section.
//
// With P = softmax over the visible set, D_i = dO_i . O_i and
// dS_ix = P_ix (dO_i . v_x - D_i) for every visible key x (core or raw token):
//   dQ_i  = tau * sum_x dS_ix k_x
//   dK_m  = tau * sum_i dS_im q_i,   dV_m  = sum_i P_im dO_i      (raw tokens)
//   dKc_j = tau * sum_i dS_ij q_i,   dVc_j = sum_i P_ij dO_i      (cores)
// and through Kc_j = sum_t a_t k_t, Vc_j = sum_t a_t v_t, a = softmax(s),
// s_t = (tau / r) qsum . k_t with qsum the sum of the r group-last queries:
//   da_t = dKc_j . k_t + dVc_j . v_t,   ds_t = a_t (da_t - sum_u a_u da_u)
//   dk_t += a_t dKc_j + (tau / r) ds_t qsum,   dv_t += a_t dVc_j
//   dq^h_last += (tau / r) sum_t ds_t k_t      for each of the r heads.
// Mean pooling has a_t = 1/g and no score gradient; max pooling passes each
// element's gradient to the row that holds the maximum.  pool_mode 3 has
// a_t = (1/r) sum_h p^h_t with p^h = softmax_t(tau q^h_last . k_t) per head:
//   ds^h_t = p^h_t (da_t - sum_u p^h_u da_u) / r
//   dk_t += a_t dKc_j + tau sum_h ds^h_t q^h_last,   dv_t += a_t dVc_j
//   dq^h_last += tau sum_t ds^h_t k_t.
//
// Four passes on CUDA cores in fp32 (one warp per row; lane l holds d/32
// consecutive elements): per query row (dQ, D), per raw token (dK, dV), per
// core (dKc, dVc into the workspace), per group (pooling backward, added into
// dK, dV and the group-last rows of dQ).  P is recomputed from the forward's LSE.
// bf16 with d = 128 runs the attention part on the tensor cores (bwd_tc.cu); with
// softmax or mean pooling it then computes the cores' gradients first, reduces the
// pooling backward to per-token scalars (a_t, (tau/r) ds_t) and per-group qsum_j, and
// lets the raw tokens' dK/dV kernel add a_t dKc_j + (tau/r) ds_t qsum_j and a_t dVc_j
// to each row as it writes it, instead of a second fp32 pass over dK and dV.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "internal.h"
#include "visibility.cuh"

namespace cca {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float LOG2E = 1.4426950408889634f;


// Lane `lane` owns elements lane*PL .. lane*PL+PL-1 of a d-element row.  Rows start on
// 16-byte boundaries (the entry points require 16-byte aligned tensors and d is 64 or
// 128), so each lane moves its PL elements with one 4-, 8- or 16-byte access and a warp
// covers the row with one coalesced request.
template <typename T, int PL>
__device__ __forceinline__ void load_row(const T *__restrict__ row, int lane, float (&f)[PL]) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value && PL == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(row + lane * 4);
        f[0] = __uint_as_float(v.x << 16);
        f[1] = __uint_as_float(v.x & 0xffff0000u);
        f[2] = __uint_as_float(v.y << 16);
        f[3] = __uint_as_float(v.y & 0xffff0000u);
    } else if constexpr (std::is_same<T, __nv_bfloat16>::value && PL == 2) {
        const uint32_t v = *reinterpret_cast<const uint32_t *>(row + lane * 2);
        f[0] = __uint_as_float(v << 16);
        f[1] = __uint_as_float(v & 0xffff0000u);
    } else if constexpr (std::is_same<T, float>::value && PL == 4) {
        const float4 v = *reinterpret_cast<const float4 *>(row + lane * 4);
        f[0] = v.x;
        f[1] = v.y;
        f[2] = v.z;
        f[3] = v.w;
    } else if constexpr (std::is_same<T, float>::value && PL == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(row + lane * 2);
        f[0] = v.x;
        f[1] = v.y;
    } else {
#pragma unroll
        for (int e = 0; e < PL; ++e) f[e] = static_cast<float>(row[lane * PL + e]);
    }
}

// fp32 row slice of this lane: store, or add to what is there (one vector access each way).
template <int PL>
__device__ __forceinline__ void store_row(float *__restrict__ row, int lane, const float (&f)[PL]) {
    if constexpr (PL == 4) {
        *reinterpret_cast<float4 *>(row + lane * 4) = make_float4(f[0], f[1], f[2], f[3]);
    } else if constexpr (PL == 2) {
        *reinterpret_cast<float2 *>(row + lane * 2) = make_float2(f[0], f[1]);
    } else {
#pragma unroll
        for (int e = 0; e < PL; ++e) row[lane * PL + e] = f[e];
    }
}
template <int PL>
__device__ __forceinline__ void add_row(float *__restrict__ row, int lane, const float (&f)[PL]) {
    float cur[PL];
    load_row<float, PL>(row, lane, cur);
#pragma unroll
    for (int e = 0; e < PL; ++e) cur[e] += f[e];
    store_row<PL>(row, lane, cur);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

template <int PL>
__device__ __forceinline__ float dot(const float (&a)[PL], const float (&b)[PL]) {
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < PL; ++e) s = fmaf(a[e], b[e], s);
    return warp_sum(s);
}

struct BwdArgs {
    int B, Hq, Hkv, N, g, w, window_mode, pool_mode;
    float tau;
};

__device__ __forceinline__ int lo_of(int i, int w) { return window_lo(i, w); }
__device__ __forceinline__ int win_of(const BwdArgs &a, int i) { return window_start(i, a.w, a.g, a.window_mode); }

// Pass 1: one warp per query row -> dQ (fp32, before the pooling term) and D.
template <typename T, int D>
__global__ void __launch_bounds__(128) bwd_dq_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                     const T *__restrict__ V, const T *__restrict__ Kc,
                                                     const T *__restrict__ Vc, const T *__restrict__ O,
                                                     const float *__restrict__ LSE, const T *__restrict__ dO,
                                                     float *__restrict__ dQ, float *__restrict__ Dbuf,
                                                     const BwdArgs a) {
    constexpr int PL = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t u = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (u >= static_cast<int64_t>(a.B) * a.Hq * a.N) return;
    const int i = static_cast<int>(u % a.N);
    const int64_t bh = u / a.N;
    const int64_t bk = (bh / a.Hq) * a.Hkv + (bh % a.Hq) / (a.Hq / a.Hkv);
    const int64_t G = a.N / a.g;
    float q[PL], g_o[PL], o[PL], dq[PL];
    load_row<T, PL>(Q + u * D, lane, q);
    load_row<T, PL>(dO + u * D, lane, g_o);
    load_row<T, PL>(O + u * D, lane, o);
#pragma unroll
    for (int e = 0; e < PL; ++e) dq[e] = 0.f;
    const float Di = dot<PL>(g_o, o);
    const float lse2 = LSE[u] * LOG2E, tau2 = a.tau * LOG2E;
    auto visit = [&](const T *kr, const T *vr) {
        float k[PL], v[PL];
        load_row<T, PL>(kr, lane, k);
        load_row<T, PL>(vr, lane, v);
        const float P = exp2f(dot<PL>(q, k) * tau2 - lse2);
        const float dS = P * (dot<PL>(g_o, v) - Di);
#pragma unroll
        for (int e = 0; e < PL; ++e) dq[e] = fmaf(a.tau * dS, k[e], dq[e]);
    };
    const int nc = lo_of(i, a.w) / a.g;
    for (int j = 0; j < nc; ++j) visit(Kc + (bk * G + j) * D, Vc + (bk * G + j) * D);
    for (int m = win_of(a, i); m <= i; ++m) visit(K + (bk * a.N + m) * D, V + (bk * a.N + m) * D);
    store_row<PL>(dQ + u * D, lane, dq);
    if (lane == 0) Dbuf[u] = Di;
}

// Passes 2 and 3: one warp per key row (raw token or core) -> its dK, dV, summed over
// the query rows [i0, i1] of every query head that reads this KV head.
template <typename T, int D>
__device__ __forceinline__ void key_grad(const T *__restrict__ Q, const T *__restrict__ dO,
                                         const float *__restrict__ LSE, const float *__restrict__ Dbuf,
                                         const float (&k)[D / 32], const float (&v)[D / 32], int64_t b, int64_t kv,
                                         int i0, int i1, const BwdArgs &a, int lane, float (&dk)[D / 32],
                                         float (&dv)[D / 32]) {
    constexpr int PL = D / 32;
    const int r = a.Hq / a.Hkv;
    const float tau2 = a.tau * LOG2E;
    for (int hh = 0; hh < r; ++hh) {
        const int64_t bh = b * a.Hq + kv * r + hh;
        for (int i = i0; i <= i1; ++i) {
            const int64_t u = bh * a.N + i;
            float q[PL], g_o[PL];
            load_row<T, PL>(Q + u * D, lane, q);
            load_row<T, PL>(dO + u * D, lane, g_o);
            const float P = exp2f(dot<PL>(q, k) * tau2 - LSE[u] * LOG2E);
            const float dS = P * (dot<PL>(g_o, v) - Dbuf[u]);
#pragma unroll
            for (int e = 0; e < PL; ++e) {
                dk[e] = fmaf(a.tau * dS, q[e], dk[e]);
                dv[e] = fmaf(P, g_o[e], dv[e]);
            }
        }
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(128) bwd_dkv_raw_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                          const T *__restrict__ V, const float *__restrict__ LSE,
                                                          const T *__restrict__ dO, const float *__restrict__ Dbuf,
                                                          float *__restrict__ dK, float *__restrict__ dV,
                                                          const BwdArgs a) {
    constexpr int PL = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t u = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (u >= static_cast<int64_t>(a.B) * a.Hkv * a.N) return;
    const int m = static_cast<int>(u % a.N);
    const int64_t bk = u / a.N;
    float k[PL], v[PL], dk[PL], dv[PL];
    load_row<T, PL>(K + u * D, lane, k);
    load_row<T, PL>(V + u * D, lane, v);
#pragma unroll
    for (int e = 0; e < PL; ++e) dk[e] = dv[e] = 0.f;
    // rows whose window [win(i), i] holds m: i in [m, i_max], win() being non-decreasing
    const int64_t i_last = a.window_mode ? static_cast<int64_t>(m / a.g + 1) * a.g + a.w - 2
                                         : static_cast<int64_t>(m) + a.w - 1;
    const int i1 = static_cast<int>(i_last < a.N - 1 ? i_last : a.N - 1);
    key_grad<T, D>(Q, dO, LSE, Dbuf, k, v, bk / a.Hkv, bk % a.Hkv, m, i1, a, lane, dk, dv);
    store_row<PL>(dK + u * D, lane, dk);
    store_row<PL>(dV + u * D, lane, dv);
}

template <typename T, int D>
__global__ void __launch_bounds__(128) bwd_dkv_core_kernel(const T *__restrict__ Q, const T *__restrict__ Kc,
                                                           const T *__restrict__ Vc, const float *__restrict__ LSE,
                                                           const T *__restrict__ dO, const float *__restrict__ Dbuf,
                                                           float *__restrict__ dKc, float *__restrict__ dVc,
                                                           const BwdArgs a) {
    constexpr int PL = D / 32;
    const int lane = threadIdx.x & 31;
    const int G = a.N / a.g;
    const int64_t u = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (u >= static_cast<int64_t>(a.B) * a.Hkv * G) return;
    const int j = static_cast<int>(u % G);
    const int64_t bk = u / G;
    float k[PL], v[PL], dk[PL], dv[PL];
    load_row<T, PL>(Kc + u * D, lane, k);
    load_row<T, PL>(Vc + u * D, lane, v);
#pragma unroll
    for (int e = 0; e < PL; ++e) dk[e] = dv[e] = 0.f;
    // core j is visible to row i iff (j+1)*g <= lo(i), i.e. i >= (j+1)*g + w - 1
    const int64_t i0 = static_cast<int64_t>(j + 1) * a.g + a.w - 1;
    if (i0 < a.N) key_grad<T, D>(Q, dO, LSE, Dbuf, k, v, bk / a.Hkv, bk % a.Hkv, static_cast<int>(i0), a.N - 1, a, lane, dk, dv);
#pragma unroll
    for (int e = 0; e < PL; ++e) {
        dKc[u * D + lane * PL + e] = dk[e];
        dVc[u * D + lane * PL + e] = dv[e];
    }
}

// Pass 4: one warp per group -> the pooling backward, added into dK, dV and dQ.
// HM: the pool_mode 3 instantiation (its per-head loop would otherwise cost every
// other mode registers, and this kernel wants all the warps it can get).
template <typename T, int D, bool HM>
__global__ void __launch_bounds__(128) bwd_pool_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                       const T *__restrict__ V, const float *__restrict__ dKc,
                                                       const float *__restrict__ dVc, float *__restrict__ dQ,
                                                       float *__restrict__ dK, float *__restrict__ dV, const BwdArgs a) {
    constexpr int PL = D / 32;
    const int lane = threadIdx.x & 31;
    const int G = a.N / a.g;
    const int64_t u = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (u >= static_cast<int64_t>(a.B) * a.Hkv * G) return;
    const int j = static_cast<int>(u % G);
    const int64_t bk = u / G;
    const int64_t b = bk / a.Hkv, kv = bk % a.Hkv;
    const int r = a.Hq / a.Hkv, g = a.g;
    float dkc[PL], dvc[PL];
#pragma unroll
    for (int e = 0; e < PL; ++e) {
        dkc[e] = dKc[u * D + lane * PL + e];
        dvc[e] = dVc[u * D + lane * PL + e];
    }
    const int64_t row0 = bk * a.N + static_cast<int64_t>(j) * g;  // first token of the group
    if (a.pool_mode == 1) {
        // mean pooling: every token weighs 1/g
        float ak[PL], av[PL];
#pragma unroll
        for (int e = 0; e < PL; ++e) {
            ak[e] = dkc[e] / g;
            av[e] = dvc[e] / g;
        }
#pragma unroll 4
        for (int t = 0; t < g; ++t) {
            add_row<PL>(dK + (row0 + t) * D, lane, ak);
            add_row<PL>(dV + (row0 + t) * D, lane, av);
        }
        return;
    }
    if (a.pool_mode == 2) {
        // max pooling: each element's gradient goes to the first row holding the maximum
        float km[PL], vm[PL];
        int kt[PL], vt[PL];
        for (int t = 0; t < g; ++t) {
            float k[PL], v[PL];
            load_row<T, PL>(K + (row0 + t) * D, lane, k);
            load_row<T, PL>(V + (row0 + t) * D, lane, v);
#pragma unroll
            for (int e = 0; e < PL; ++e) {
                if (t == 0 || k[e] > km[e]) { km[e] = k[e]; kt[e] = t; }
                if (t == 0 || v[e] > vm[e]) { vm[e] = v[e]; vt[e] = t; }
            }
        }
#pragma unroll
        for (int e = 0; e < PL; ++e) {
            dK[(row0 + kt[e]) * D + lane * PL + e] += dkc[e];
            dV[(row0 + vt[e]) * D + lane * PL + e] += dvc[e];
        }
        return;
    }
    if (HM) {
        // per-head softmax weights averaged over the r heads: head by head, its
        // normaliser, sum_u p_u da_u, then its share of every row's gradient
        const int last3 = (j + 1) * g - 1;
        for (int hh = 0; hh < r; ++hh) {
            const int64_t qrow = (b * a.Hq + kv * r + hh) * a.N + last3;
            float qh[PL];
            load_row<T, PL>(Q + qrow * D, lane, qh);
            float mx = -INFINITY, den = 0.f;
#pragma unroll 4
            for (int t = 0; t < g; ++t) {
                float k[PL];
                load_row<T, PL>(K + (row0 + t) * D, lane, k);
                const float s = a.tau * dot<PL>(qh, k);
                const float mn = fmaxf(mx, s);
                den = den * expf(mx - mn) + expf(s - mn);
                mx = mn;
            }
            float sad = 0.f;
#pragma unroll 4
            for (int t = 0; t < g; ++t) {
                float k[PL], v[PL];
                load_row<T, PL>(K + (row0 + t) * D, lane, k);
                load_row<T, PL>(V + (row0 + t) * D, lane, v);
                const float pt = expf(a.tau * dot<PL>(qh, k) - mx) / den;
                sad += pt * (dot<PL>(dkc, k) + dot<PL>(dvc, v));
            }
            float dqh[PL];
#pragma unroll
            for (int e = 0; e < PL; ++e) dqh[e] = 0.f;
#pragma unroll 4
            for (int t = 0; t < g; ++t) {
                float k[PL], v[PL];
                load_row<T, PL>(K + (row0 + t) * D, lane, k);
                load_row<T, PL>(V + (row0 + t) * D, lane, v);
                const float pt = expf(a.tau * dot<PL>(qh, k) - mx) / den;
                const float ds = pt * (dot<PL>(dkc, k) + dot<PL>(dvc, v) - sad) / r;
                float ak[PL], av[PL];
#pragma unroll
                for (int e = 0; e < PL; ++e) {
                    ak[e] = (pt / r) * dkc[e] + a.tau * ds * qh[e];
                    av[e] = (pt / r) * dvc[e];
                    dqh[e] = fmaf(a.tau * ds, k[e], dqh[e]);
                }
                add_row<PL>(dK + (row0 + t) * D, lane, ak);
                add_row<PL>(dV + (row0 + t) * D, lane, av);
            }
            add_row<PL>(dQ + qrow * D, lane, dqh);
        }
        return;
    }
    // softmax pooling scored by the sum of the r group-last queries (1/r folded into c)
    const float c = a.tau / r;
    const int last = (j + 1) * g - 1;
    float qs[PL];
#pragma unroll
    for (int e = 0; e < PL; ++e) qs[e] = 0.f;
    for (int hh = 0; hh < r; ++hh) {
        float f[PL];
        load_row<T, PL>(Q + ((b * a.Hq + kv * r + hh) * a.N + last) * D, lane, f);
#pragma unroll
        for (int e = 0; e < PL; ++e) qs[e] += f[e];
    }
    // pass A: softmax normaliser of the group scores
    float mx = -INFINITY, den = 0.f;
#pragma unroll 4
    for (int t = 0; t < g; ++t) {
        float k[PL];
        load_row<T, PL>(K + (row0 + t) * D, lane, k);
        const float s = c * dot<PL>(qs, k);
        const float mn = fmaxf(mx, s);
        den = den * expf(mx - mn) + expf(s - mn);
        mx = mn;
    }
    // pass B: sum_u a_u da_u
    float sad = 0.f;
#pragma unroll 4
    for (int t = 0; t < g; ++t) {
        float k[PL], v[PL];
        load_row<T, PL>(K + (row0 + t) * D, lane, k);
        load_row<T, PL>(V + (row0 + t) * D, lane, v);
        const float at = expf(c * dot<PL>(qs, k) - mx) / den;
        sad += at * (dot<PL>(dkc, k) + dot<PL>(dvc, v));
    }
    // pass C: per-token gradients and the query-side term
    float dqs[PL];
#pragma unroll
    for (int e = 0; e < PL; ++e) dqs[e] = 0.f;
#pragma unroll 4
    for (int t = 0; t < g; ++t) {
        float k[PL], v[PL];
        load_row<T, PL>(K + (row0 + t) * D, lane, k);
        load_row<T, PL>(V + (row0 + t) * D, lane, v);
        const float at = expf(c * dot<PL>(qs, k) - mx) / den;
        const float ds = at * (dot<PL>(dkc, k) + dot<PL>(dvc, v) - sad);
        float ak[PL], av[PL];
#pragma unroll
        for (int e = 0; e < PL; ++e) {
            ak[e] = at * dkc[e] + c * ds * qs[e];
            av[e] = at * dvc[e];
            dqs[e] = fmaf(c * ds, k[e], dqs[e]);
        }
        add_row<PL>(dK + (row0 + t) * D, lane, ak);
        add_row<PL>(dV + (row0 + t) * D, lane, av);
    }
    for (int hh = 0; hh < r; ++hh) add_row<PL>(dQ + ((b * a.Hq + kv * r + hh) * a.N + last) * D, lane, dqs);
}

// Sums each of the 32 values v[0..31] over the warp in 31 shuffles (a halving butterfly:
// at each step a lane keeps the half of its values whose index bit matches its own lane
// bit and receives the partner's share of it); lane l returns the total of v[l].
__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
    for (int o = 16, n = 16; o > 0; o >>= 1, n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float keep = up ? v[i + n] : v[i];
            const float send = up ? v[i] : v[i + n];
            v[i] = keep + __shfl_xor_sync(kFull, send, o);
        }
    }
    return v[0];
}

// The method's pooling backward, reduced to what the dK/dV kernel needs to fold it into
// the raw tokens' rows (BwdPoolFuse mode 2): per token a_t and (tau/r) ds_t, per group
// qsum_j in fp32; the group-last queries' term (tau/r) sum_t ds_t k_t goes into dQ here.
// One warp per group, keys in chunks of 16: each lane forms its partial dot products for
// the chunk's 16 scores s_t and 16 values da_t = dKc_j . k_t + dVc_j . v_t, one
// transposed reduction finishes all 32, and an online softmax carries the normaliser and
// sum_u exp(s_u) da_u across chunks.  A second pass (reusing the one chunk of a group of
// at most 16 tokens, else recomputing) writes a_t, (tau/r) ds_t and sums the dQ term.
template <typename T, int D>
__global__ void __launch_bounds__(128) bwd_pool_scalars_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                               const T *__restrict__ V, const float *__restrict__ dKc,
                                                               const float *__restrict__ dVc, float *__restrict__ dQ,
                                                               float *__restrict__ pa, float *__restrict__ pcds,
                                                               float *__restrict__ pqs, const BwdArgs a) {
    constexpr int PL = D / 32;
    const int lane = threadIdx.x & 31;
    const int G = a.N / a.g;
    const int64_t u = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (u >= static_cast<int64_t>(a.B) * a.Hkv * G) return;
    const int j = static_cast<int>(u % G);
    const int64_t bk = u / G;
    const int64_t b = bk / a.Hkv, kv = bk % a.Hkv;
    const int r = a.Hq / a.Hkv, g = a.g;
    float dkc[PL], dvc[PL];
    load_row<float, PL>(dKc + u * D, lane, dkc);
    load_row<float, PL>(dVc + u * D, lane, dvc);
    const int64_t row0 = bk * a.N + static_cast<int64_t>(j) * g;  // first token of the group
    const float c = a.tau / r;
    const int last = (j + 1) * g - 1;
    float qs[PL];
#pragma unroll
    for (int e = 0; e < PL; ++e) qs[e] = 0.f;
    for (int hh = 0; hh < r; ++hh) {
        float f[PL];
        load_row<T, PL>(Q + ((b * a.Hq + kv * r + hh) * a.N + last) * D, lane, f);
#pragma unroll
        for (int e = 0; e < PL; ++e) qs[e] += f[e];
    }
    store_row<PL>(pqs + u * D, lane, qs);
    const int nch = (g + 15) / 16;
    const int t16 = lane & 15;
    // this lane's key of chunk ch: its score s and its da (lanes l and l + 16 both get key l)
    auto chunk = [&](int ch, float &sv, float &ev) {
        float val[32];
        // bf16, d = 128: every K and V row of the chunk is requested before any is used
        // (8 bytes per lane and row, 64 registers), so the chunk costs one memory round trip
        uint2 kraw[16], vraw[16];
        if constexpr (std::is_same<T, __nv_bfloat16>::value && PL == 4) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const bool in = ch * 16 + t < g;
                kraw[t] = in ? *reinterpret_cast<const uint2 *>(K + (row0 + ch * 16 + t) * D + lane * 4)
                             : make_uint2(0u, 0u);
                vraw[t] = in ? *reinterpret_cast<const uint2 *>(V + (row0 + ch * 16 + t) * D + lane * 4)
                             : make_uint2(0u, 0u);
            }
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            float k[PL], v[PL];
            if constexpr (std::is_same<T, __nv_bfloat16>::value && PL == 4) {
                k[0] = __uint_as_float(kraw[t].x << 16);
                k[1] = __uint_as_float(kraw[t].x & 0xffff0000u);
                k[2] = __uint_as_float(kraw[t].y << 16);
                k[3] = __uint_as_float(kraw[t].y & 0xffff0000u);
                v[0] = __uint_as_float(vraw[t].x << 16);
                v[1] = __uint_as_float(vraw[t].x & 0xffff0000u);
                v[2] = __uint_as_float(vraw[t].y << 16);
                v[3] = __uint_as_float(vraw[t].y & 0xffff0000u);
            } else if (ch * 16 + t < g) {
                load_row<T, PL>(K + (row0 + ch * 16 + t) * D, lane, k);
                load_row<T, PL>(V + (row0 + ch * 16 + t) * D, lane, v);
            } else {
#pragma unroll
                for (int e = 0; e < PL; ++e) k[e] = v[e] = 0.f;
            }
            float ps = 0.f, pe = 0.f;
#pragma unroll
            for (int e = 0; e < PL; ++e) {
                ps = fmaf(qs[e], k[e], ps);
                pe = fmaf(dkc[e], k[e], fmaf(dvc[e], v[e], pe));
            }
            val[t] = c * ps;
            val[16 + t] = pe;
        }
        const float x = warp_transpose_sum32(val, lane);  // lane t: s of key t; lane 16 + t: its da
        sv = __shfl_sync(kFull, x, t16);
        ev = __shfl_sync(kFull, x, 16 + t16);
    };
    // pass 1: max, normaliser and sum_u exp(s_u - max) da_u, online over the chunks
    float mx = -INFINITY, den = 0.f, num = 0.f, s_keep = 0.f, e_keep = 0.f;
    for (int ch = 0; ch < nch; ++ch) {
        float sv, ev;
        chunk(ch, sv, ev);
        const bool valid = ch * 16 + t16 < g;
        float cm = valid ? sv : -INFINITY;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(kFull, cm, o));
        const float mn = fmaxf(mx, cm);
        const float pk = valid ? expf(sv - mn) : 0.f;
        float ps = pk, pe = pk * ev;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
            ps += __shfl_xor_sync(kFull, ps, o);
            pe += __shfl_xor_sync(kFull, pe, o);
        }
        const float f = expf(mx - mn);
        den = den * f + ps;
        num = num * f + pe;
        mx = mn;
        s_keep = sv;
        e_keep = ev;
    }
    const float sad = num / den;  // sum_u a_u da_u
    // pass 2: the per-token scalars and the query-side term
    float dqs[PL];
#pragma unroll
    for (int e = 0; e < PL; ++e) dqs[e] = 0.f;
    for (int ch = 0; ch < nch; ++ch) {
        float sv = s_keep, ev = e_keep;
        if (nch > 1) chunk(ch, sv, ev);
        const int key = ch * 16 + t16;
        const bool valid = key < g;
        const float at = valid ? expf(sv - mx) / den : 0.f;
        const float cds = c * at * (ev - sad);
        if (lane < 16 && valid) {
            pa[row0 + key] = at;
            pcds[row0 + key] = cds;
        }
        const int nt = min(16, g - ch * 16);
        for (int t = 0; t < nt; ++t) {
            const float w = __shfl_sync(kFull, cds, t);
            float k[PL];
            load_row<T, PL>(K + (row0 + ch * 16 + t) * D, lane, k);
#pragma unroll
            for (int e = 0; e < PL; ++e) dqs[e] = fmaf(w, k[e], dqs[e]);
        }
    }
    for (int hh = 0; hh < r; ++hh) add_row<PL>(dQ + ((b * a.Hq + kv * r + hh) * a.N + last) * D, lane, dqs);
}

// Workspace layout (fp32, every part 256-byte aligned): D [B*Hq*N], dKc and dVc
// [B*Hkv*G*d] each, then for the folded pooling backward a and cds [B*Hkv*N] each and
// qs [B*Hkv*G*d].
struct BwdWorkspace {
    float *Dbuf, *dKc, *dVc, *pa, *pcds, *pqs;
};
inline int64_t round64(int64_t n) { return (n + 63) / 64 * 64; }
inline int64_t bwd_workspace_floats(const Shape &s, float *base, BwdWorkspace *w) {
    const int64_t G = s.N / s.g;
    const int64_t nD = round64(static_cast<int64_t>(s.B) * s.Hq * s.N);
    const int64_t nc = round64(static_cast<int64_t>(s.B) * s.Hkv * G * s.d);
    const int64_t nt = round64(static_cast<int64_t>(s.B) * s.Hkv * s.N);
    if (w != nullptr) {
        w->Dbuf = base;
        w->dKc = w->Dbuf + nD;
        w->dVc = w->dKc + nc;
        w->pa = w->dVc + nc;
        w->pcds = w->pa + nt;
        w->pqs = w->pcds + nt;
    }
    return nD + 3 * nc + 2 * nt;
}

template <typename T, int D>
cudaError_t run(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc, const void *O,
                const float *LSE, const void *dO, float *dQ, float *dK, float *dV, const Shape &s, float *ws,
                int32_t *status, cudaStream_t stream) {
    BwdArgs a{s.B, s.Hq, s.Hkv, s.N, s.g, s.w, s.window_mode, s.pool_mode, s.scale};
    const int64_t G = s.N / s.g;
    BwdWorkspace W;
    bwd_workspace_floats(s, ws, &W);
    float *const Dbuf = W.Dbuf, *const dKc = W.dKc, *const dVc = W.dVc;
    auto blocks = [](int64_t rows) { return static_cast<unsigned>((rows + 3) / 4); };
    const T *q = static_cast<const T *>(Q), *k = static_cast<const T *>(K), *v = static_cast<const T *>(V);
    const T *kc = static_cast<const T *>(Kc), *vc = static_cast<const T *>(Vc);
    const T *o = static_cast<const T *>(O), *dout = static_cast<const T *>(dO);
    if constexpr (std::is_same<T, __nv_bfloat16>::value && D == 128) {
        if (s.pool_mode == 0 || s.pool_mode == 1) {
            // cores first, then the raw tokens with the pooling backward folded into their rows
            cudaError_t e = launch_attn_bwd_tc(Q, K, V, Kc, Vc, O, LSE, dO, dQ, dK, dV, Dbuf, dKc, dVc, s, status, 1,
                                               BwdPoolFuse{0, nullptr, nullptr, nullptr}, stream);
            if (e != cudaSuccess) return e;
            BwdPoolFuse pf{1, nullptr, nullptr, nullptr};
            if (s.pool_mode == 0) {
                bwd_pool_scalars_kernel<T, D><<<blocks(static_cast<int64_t>(s.B) * s.Hkv * G), 128, 0, stream>>>(
                    q, k, v, dKc, dVc, dQ, W.pa, W.pcds, W.pqs, a);
                if ((e = cudaGetLastError()) != cudaSuccess) return e;
                pf = BwdPoolFuse{2, W.pa, W.pcds, W.pqs};
            }
            return launch_attn_bwd_tc(Q, K, V, Kc, Vc, O, LSE, dO, dQ, dK, dV, Dbuf, dKc, dVc, s, status, 2, pf,
                                      stream);
        }
        const cudaError_t e = launch_attn_bwd_tc(Q, K, V, Kc, Vc, O, LSE, dO, dQ, dK, dV, Dbuf, dKc, dVc, s, status,
                                                 0, BwdPoolFuse{0, nullptr, nullptr, nullptr}, stream);
        if (e != cudaSuccess) return e;
    } else {
        bwd_dq_kernel<T, D><<<blocks(static_cast<int64_t>(s.B) * s.Hq * s.N), 128, 0, stream>>>(
            q, k, v, kc, vc, o, LSE, dout, dQ, Dbuf, a);
        bwd_dkv_raw_kernel<T, D><<<blocks(static_cast<int64_t>(s.B) * s.Hkv * s.N), 128, 0, stream>>>(
            q, k, v, LSE, dout, Dbuf, dK, dV, a);
        bwd_dkv_core_kernel<T, D><<<blocks(static_cast<int64_t>(s.B) * s.Hkv * G), 128, 0, stream>>>(
            q, kc, vc, LSE, dout, Dbuf, dKc, dVc, a);
    }
    if (s.pool_mode == 3)
        bwd_pool_kernel<T, D, true><<<blocks(static_cast<int64_t>(s.B) * s.Hkv * G), 128, 0, stream>>>(
            q, k, v, dKc, dVc, dQ, dK, dV, a);
    else
        bwd_pool_kernel<T, D, false><<<blocks(static_cast<int64_t>(s.B) * s.Hkv * G), 128, 0, stream>>>(
            q, k, v, dKc, dVc, dQ, dK, dV, a);
    return cudaGetLastError();
}

}  // namespace

uint64_t prefill_bwd_workspace_bytes(const Shape &s) { return 4ull * bwd_workspace_floats(s, nullptr, nullptr); }

cudaError_t launch_prefill_bwd(int dtype, const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                               const void *O, const float *LSE, const void *dO, float *dQ, float *dK, float *dV,
                               const Shape &s, float *ws, int32_t *status, cudaStream_t stream) {
    if (dtype == 0) {
        if (s.d == 128) return run<__nv_bfloat16, 128>(Q, K, V, Kc, Vc, O, LSE, dO, dQ, dK, dV, s, ws, status, stream);
        if (s.d == 64) return run<__nv_bfloat16, 64>(Q, K, V, Kc, Vc, O, LSE, dO, dQ, dK, dV, s, ws, status, stream);
    } else {
        if (s.d == 128) return run<float, 128>(Q, K, V, Kc, Vc, O, LSE, dO, dQ, dK, dV, s, ws, status, stream);
        if (s.d == 64) return run<float, 64>(Q, K, V, Kc, Vc, O, LSE, dO, dQ, dK, dV, s, ws, status, stream);
    }
    return cudaErrorNotSupported;
}

}  // namespace cca
