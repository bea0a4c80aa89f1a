// Global-aware pooling ("Core Context Aware Transformers for Long Context
// Language Modeling", Method section, pooling equation): every group of g
// tokens becomes one core key and one core value, the softmax-weighted sums of
// the group's keys and values, weighted by softmax(tau * q_last . k_t) where
// q_last is the query of the group's last token (for grouped-query attention,
// the mean of the logits of the query heads sharing the KV head).
//
// Memory-bound: 6*g*d flops per 4*g*d bytes.  One warp owns one group.  Each
// lane holds one 16-byte vector of a row (d=128 bf16: 16 lanes per row, two
// rows per warp-wide load), issues every load of a chunk of rows before any
// arithmetic, reduces the dot products with shuffles, and keeps a running
// (max, sum) so that any g streams through registers in chunks.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace cca {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint4 ld_nc16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <typename T>
struct VecTraits;

template <>
struct VecTraits<__nv_bfloat16> {
    static constexpr int E = 8;
    __device__ static void unpack(const uint4 &v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static uint4 pack(const float (&f)[8]) {
        uint4 v;
        v.x = ptx::pack_bf16x2(f[0], f[1]);
        v.y = ptx::pack_bf16x2(f[2], f[3]);
        v.z = ptx::pack_bf16x2(f[4], f[5]);
        v.w = ptx::pack_bf16x2(f[6], f[7]);
        return v;
    }
};

template <>
struct VecTraits<float> {
    static constexpr int E = 4;
    __device__ static void unpack(const uint4 &v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

// ITERS warp-wide row loads are in flight per chunk (RPI rows each).
template <typename T, int D, int ITERS>
__global__ void __launch_bounds__(256) pool_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                   const T *__restrict__ V, T *__restrict__ Kc,
                                                   T *__restrict__ Vc, int Hq, int Hkv, int N, int g,
                                                   float logit_scale, int64_t n_groups_total) {
    using VT = VecTraits<T>;
    constexpr int E = VT::E;        // elements per 16-byte vector
    constexpr int LPR = D / E;      // lanes per row
    constexpr int RPI = 32 / LPR;   // rows per warp-wide load
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "unsupported head dim");

    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;
    const int cl = lane % LPR;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw >= n_groups_total) return;  // warp-uniform

    const int G = N / g;
    const int64_t j = gw % G;
    const int64_t bk = gw / G;  // b * Hkv + kv
    const int64_t b = bk / Hkv;
    const int64_t kv = bk % Hkv;
    const int r = Hq / Hkv;

    // Sum of the group-last queries of the r query heads; 1/r is in logit_scale.
    float q[E];
#pragma unroll
    for (int e = 0; e < E; ++e) q[e] = 0.f;
    const int64_t last = (j + 1) * g - 1;
    for (int hh = 0; hh < r; ++hh) {
        const T *qp = Q + ((b * Hq + kv * r + hh) * static_cast<int64_t>(N) + last) * D + cl * E;
        float f[E];
        VT::unpack(ld_nc16(qp), f);
#pragma unroll
        for (int e = 0; e < E; ++e) q[e] += f[e];
    }

    const T *Kg = K + (bk * N + j * g) * static_cast<int64_t>(D) + cl * E;
    const T *Vg = V + (bk * N + j * g) * static_cast<int64_t>(D) + cl * E;

    float m = -INFINITY, l = 0.f;
    float ak[E], av[E];
#pragma unroll
    for (int e = 0; e < E; ++e) ak[e] = av[e] = 0.f;

    for (int t0 = 0; t0 < g; t0 += RPI * ITERS) {
        uint4 kr[ITERS], vr[ITERS];
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
            const int t = t0 + it * RPI + sub;
            if (t < g) {
                kr[it] = ld_nc16(Kg + static_cast<int64_t>(t) * D);
                vr[it] = ld_nc16(Vg + static_cast<int64_t>(t) * D);
            } else {
                kr[it] = make_uint4(0, 0, 0, 0);
                vr[it] = make_uint4(0, 0, 0, 0);
            }
        }
        float s[ITERS];
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
            float f[E];
            VT::unpack(kr[it], f);
            float p = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) p = fmaf(q[e], f[e], p);
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) p += __shfl_xor_sync(kFull, p, o);
            const int t = t0 + it * RPI + sub;
            s[it] = (t < g) ? p * logit_scale : -INFINITY;  // log2 domain
        }
        float cm = s[0];
#pragma unroll
        for (int it = 1; it < ITERS; ++it) cm = fmaxf(cm, s[it]);
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(kFull, cm, o));
        const float mn = fmaxf(m, cm);  // finite: row t0 of the chunk is valid
        const float corr = ptx::ex2(m - mn);
        l *= corr;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            ak[e] *= corr;
            av[e] *= corr;
        }
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
            const float p = ptx::ex2(s[it] - mn);
            l += p;
            float fk[E], fv[E];
            VT::unpack(kr[it], fk);
            VT::unpack(vr[it], fv);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ak[e] = fmaf(p, fk[e], ak[e]);
                av[e] = fmaf(p, fv[e], av[e]);
            }
        }
        m = mn;
    }
    // Combine the RPI row-subgroups of the warp.
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) {
        l += __shfl_xor_sync(kFull, l, o);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            ak[e] += __shfl_xor_sync(kFull, ak[e], o);
            av[e] += __shfl_xor_sync(kFull, av[e], o);
        }
    }
    const float inv = 1.f / l;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        ak[e] *= inv;
        av[e] *= inv;
    }
    const int64_t orow = (bk * G + j) * static_cast<int64_t>(D) + cl * E;
    if (RPI >= 2) {
        if (sub == 0) *reinterpret_cast<uint4 *>(Kc + orow) = VT::pack(ak);
        if (sub == 1) *reinterpret_cast<uint4 *>(Vc + orow) = VT::pack(av);
    } else {
        *reinterpret_cast<uint4 *>(Kc + orow) = VT::pack(ak);
        *reinterpret_cast<uint4 *>(Vc + orow) = VT::pack(av);
    }
}

template <typename T, int D>
cudaError_t launch_typed(const void *Q, const void *K, const void *V, void *Kc, void *Vc, const Shape &s,
                         cudaStream_t stream) {
    constexpr int E = VecTraits<T>::E;
    constexpr int RPI = 32 / (D / E);
    constexpr int ITERS = RPI >= 4 ? 4 : 8;  // 16 rows per chunk (8 when one row per load)
    const int64_t total = static_cast<int64_t>(s.B) * s.Hkv * (s.N / s.g);
    const int warps_per_block = 8;
    const int64_t blocks = (total + warps_per_block - 1) / warps_per_block;
    const float log2e = 1.4426950408889634f;
    const float logit_scale = s.scale * log2e / static_cast<float>(s.Hq / s.Hkv);
    pool_kernel<T, D, ITERS><<<static_cast<unsigned>(blocks), warps_per_block * 32, 0, stream>>>(
        static_cast<const T *>(Q), static_cast<const T *>(K), static_cast<const T *>(V),
        static_cast<T *>(Kc), static_cast<T *>(Vc), s.Hq, s.Hkv, s.N, s.g, logit_scale, total);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pool(int dtype, const void *Q, const void *K, const void *V, void *Kc, void *Vc,
                        const Shape &s, cudaStream_t stream) {
    if (dtype == 0) {
        if (s.d == 128) return launch_typed<__nv_bfloat16, 128>(Q, K, V, Kc, Vc, s, stream);
        if (s.d == 64) return launch_typed<__nv_bfloat16, 64>(Q, K, V, Kc, Vc, s, stream);
    } else {
        if (s.d == 128) return launch_typed<float, 128>(Q, K, V, Kc, Vc, s, stream);
        if (s.d == 64) return launch_typed<float, 64>(Q, K, V, Kc, Vc, s, stream);
    }
    return cudaErrorNotSupported;
}

}  // namespace cca
