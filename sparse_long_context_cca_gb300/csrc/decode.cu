// Decoding step of CCA attention: the new token at position `pos` attends, with
// one softmax, to the visible core tokens j < lo(pos)/g and to the raw tokens of
// its window [lo(pos), pos] ("Core Context Aware Transformers for Long Context
// Language Modeling", Method section, fusion equation, evaluated for one query
// row; the write-up's decoding paragraph keeps only cores + window in the KV
// cache).  Plus pooling of a single newly completed group (pooling equation).
//
// Memory-bound: every visible key and value row is read once per KV head and
// used by the r query heads that share it.  The visible list is split across
// CTAs (flash-decoding); each CTA keeps an online-softmax state per query head
// over its slice.  The slices' (max, sum, output) partials are merged either by
// a second kernel, through a caller-provided workspace, or, for long lists with
// enough (b, kv) pairs to fill the GPU, inside a thread-block cluster that holds
// all the slices of one (b, kv), through distributed shared memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "sm100_ptx.cuh"
#include "visibility.cuh"

namespace cca {

// Decode path test hook: 0 automatic, 1 always the split + merge kernels, 2 the
// one-launch cluster merge wherever a cluster of two or more splits fits.
int g_decode_path = 0;

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int DEC_WARPS = 4;
constexpr int MIN_KEYS_PER_SPLIT = 64;
constexpr int MAX_SPLITS = 64;

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
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
        return make_uint4(ptx::pack_bf16x2(f[0], f[1]), ptx::pack_bf16x2(f[2], f[3]), ptx::pack_bf16x2(f[4], f[5]),
                          ptx::pack_bf16x2(f[6], f[7]));
    }
};
template <>
struct Vec<float> {
    static constexpr int E = 4;
    __device__ static void unpack(const uint4 &v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};

__device__ __forceinline__ uint4 ldg16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

struct DecodeArgs {
    int Hq, Hkv, Ncap, g, pos;
    int n_core, lo, L;  // visible cores, first window token, visible keys
    int splits;         // CTAs per (b, kv)
    float scale_log2;
};

// Partials: ws[((b*Hq + h) * MAX_SPLITS + s) * (D + 2) + {0..D-1: o, D: m, D+1: l}]
// CL: the splits of one (b, kv) form a thread-block cluster and merge in it (O, LSE written
// by the cluster's first CTA from the others' shared memory; no workspace, no second kernel).
template <typename T, int D, int R, bool CL>
__global__ void __launch_bounds__(DEC_WARPS * 32, R == 1 ? 4 : 1) decode_split_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                                      const T *__restrict__ V,
                                                                      const T *__restrict__ Kc,
                                                                      const T *__restrict__ Vc, float *__restrict__ ws,
                                                                      T *__restrict__ Oout, float *__restrict__ LSEout,
                                                                      const DecodeArgs a) {
    using VT = Vec<T>;
    constexpr int E = VT::E;
    constexpr int LPR = D / E;     // lanes per key row
    constexpr int RPI = 32 / LPR;  // keys per warp-wide pass
    constexpr int UNROLL = 4;
    __shared__ float sm_m[DEC_WARPS][R], sm_l[DEC_WARPS][R];
    __shared__ float sm_o[DEC_WARPS][R][D];

    // This kernel is launched as a programmatic dependent of whatever ran before it on the
    // stream, so its CTAs may be scheduled while that kernel drains; they wait for its
    // completion first, before they read anything or signal their own dependent.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The merge kernel may be scheduled now: it waits for this grid's completion itself.
    // (With the in-cluster merge there is no merge kernel, and the grid signals nothing: a
    // dependent then starts as this grid completes.)
    if constexpr (!CL) asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / LPR, cl = lane % LPR;
    const int s = blockIdx.x;
    const int bk = blockIdx.y;  // b * Hkv + kv
    const int b = bk / a.Hkv, kv = bk % a.Hkv;
    // this CTA's slice of the visible list, then this warp's part of it
    const int x0 = static_cast<int>(static_cast<int64_t>(a.L) * s / a.splits);
    const int x1 = static_cast<int>(static_cast<int64_t>(a.L) * (s + 1) / a.splits);
    const int wx0 = x0 + (x1 - x0) * warp / DEC_WARPS;
    const int wx1 = x0 + (x1 - x0) * (warp + 1) / DEC_WARPS;

    float q[R][E], o[R][E], m[R], l[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float f[E];
        VT::unpack(ldg16(Q + (static_cast<int64_t>(b) * a.Hq + kv * R + r) * D + cl * E), f);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            q[r][e] = f[e];
            o[r][e] = 0.f;
        }
        m[r] = -INFINITY;
        l[r] = 0.f;
    }
    // list index x < n_core is core x; otherwise window token lo + (x - n_core)
    const T *kc = Kc + static_cast<int64_t>(bk) * (a.Ncap / a.g) * D + cl * E;
    const T *vc = Vc + static_cast<int64_t>(bk) * (a.Ncap / a.g) * D + cl * E;
    const T *kr = K + static_cast<int64_t>(bk) * a.Ncap * D + cl * E;
    const T *vr = V + static_cast<int64_t>(bk) * a.Ncap * D + cl * E;

    // Software-pipelined over batches of RPI * UNROLL keys: the next batch's loads are
    // in flight while the current one is scored (two register sets, used alternately).
    auto load_batch = [&](int xb, uint4 (&kk)[UNROLL], uint4 (&vv)[UNROLL]) {
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int x = xb + u * RPI + sub;
            if (x < wx1) {
                const bool core = x < a.n_core;
                const int64_t row = core ? x : a.lo + (x - a.n_core);
                kk[u] = ldg16((core ? kc : kr) + row * D);
                vv[u] = ldg16((core ? vc : vr) + row * D);
            } else {
                kk[u] = vv[u] = make_uint4(0, 0, 0, 0);
            }
        }
    };
    // One online-softmax update per batch: all logits first, then one max and one
    // rescale per query head, then the batch's exponentials and weighted values.
    auto score_batch = [&](int xb, const uint4 (&kk)[UNROLL], const uint4 (&vv)[UNROLL]) {
        float xl[UNROLL][R];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const bool valid = xb + u * RPI + sub < wx1;
            float kf[E];
            VT::unpack(kk[u], kf);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float dot = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) dot = fmaf(q[r][e], kf[e], dot);
#pragma unroll
                for (int off = LPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(kFull, dot, off);
                xl[u][r] = valid ? dot * a.scale_log2 : -INFINITY;
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float mb = xl[0][r];
#pragma unroll
            for (int u = 1; u < UNROLL; ++u) mb = fmaxf(mb, xl[u][r]);
            const float mn = fmaxf(m[r], mb);
            if (mn == -INFINITY) continue;  // nothing visible yet in this lane group
            const float corr = ptx::ex2(m[r] - mn);  // 0 when m was -inf
            l[r] *= corr;
#pragma unroll
            for (int e = 0; e < E; ++e) o[r][e] *= corr;
            m[r] = mn;
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            float vf[E];
            VT::unpack(vv[u], vf);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                // masked keys (and lane groups that have seen nothing yet) add nothing
                const float p = xl[u][r] == -INFINITY ? 0.f : ptx::ex2(xl[u][r] - m[r]);
                l[r] += p;
#pragma unroll
                for (int e = 0; e < E; ++e) o[r][e] = fmaf(p, vf[e], o[r][e]);
            }
        }
    };
    constexpr int STEP = RPI * UNROLL;
    uint4 k0[UNROLL], v0[UNROLL], k1[UNROLL], v1[UNROLL];
    if (wx0 < wx1) load_batch(wx0, k0, v0);
    for (int xb = wx0; xb < wx1; xb += 2 * STEP) {
        if (xb + STEP < wx1) load_batch(xb + STEP, k1, v1);
        score_batch(xb, k0, v0);
        if (xb + STEP >= wx1) break;
        if (xb + 2 * STEP < wx1) load_batch(xb + 2 * STEP, k0, v0);
        score_batch(xb + STEP, k1, v1);
    }
    // merge the RPI key subgroups of the warp (lanes with the same column chunk)
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
            const float mo = __shfl_xor_sync(kFull, m[r], off);
            const float lo_ = __shfl_xor_sync(kFull, l[r], off);
            const float mn = fmaxf(m[r], mo);
            const float ca = (m[r] == -INFINITY) ? 0.f : ptx::ex2(m[r] - mn);
            const float cb = (mo == -INFINITY) ? 0.f : ptx::ex2(mo - mn);
            l[r] = l[r] * ca + lo_ * cb;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float oo = __shfl_xor_sync(kFull, o[r][e], off);
                o[r][e] = o[r][e] * ca + oo * cb;
            }
            m[r] = mn;
        }
        if (sub == 0) {
#pragma unroll
            for (int e = 0; e < E; ++e) sm_o[warp][r][cl * E + e] = o[r][e];
            if (cl == 0) {
                sm_m[warp][r] = m[r];
                sm_l[warp][r] = l[r];
            }
        }
    }
    __syncthreads();
    // merge the warps and write this split's partial for each query head
    __shared__ float sm_part[CL ? R : 1][CL ? D + 2 : 1];
    for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
        const int r = idx / D, c = idx % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < DEC_WARPS; ++w) mx = fmaxf(mx, sm_m[w][r]);
        float acc = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < DEC_WARPS; ++w) {
            const float f = (sm_m[w][r] == -INFINITY) ? 0.f : ptx::ex2(sm_m[w][r] - mx);
            acc += sm_o[w][r][c] * f;
            lsum += sm_l[w][r] * f;
        }
        float *dst = CL ? &sm_part[r][0]
                        : ws + ((static_cast<int64_t>(b) * a.Hq + kv * R + r) * MAX_SPLITS + s) * (D + 2);
        dst[c] = acc;
        if (c == 0) {
            dst[D] = mx;
            dst[D + 1] = lsum;
        }
    }
    if constexpr (CL) {
        // Every CTA of the cluster has its partial in shared memory after this barrier; the
        // first CTA reads them all (distributed shared memory) and writes O and LSE.  The
        // second barrier keeps the others resident until it has read them.  Every CTA of the
        // cluster reaches both barriers (a CTA with an empty slice has m = -inf, l = 0).
        ptx::cluster_sync();
        if (blockIdx.x == 0) {
            const int splits = a.splits;
            const uint32_t base = ptx::smem_addr(&sm_part[0][0]);
            for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
                const int r = idx / D, c = idx % D;
                const uint32_t row = base + static_cast<uint32_t>(r * (D + 2)) * 4u;
                float mx = -INFINITY;
                for (int q = 0; q < splits; ++q) mx = fmaxf(mx, ptx::ld_dsmem_f32(row + D * 4u, q));
                float acc = 0.f, lsum = 0.f;
                for (int q = 0; q < splits; ++q) {
                    const float mq = ptx::ld_dsmem_f32(row + D * 4u, q);
                    const float f = (mq == -INFINITY) ? 0.f : ptx::ex2(mq - mx);
                    acc = fmaf(ptx::ld_dsmem_f32(row + static_cast<uint32_t>(c) * 4u, q), f, acc);
                    lsum = fmaf(ptx::ld_dsmem_f32(row + (D + 1) * 4u, q), f, lsum);
                }
                const int64_t bh = static_cast<int64_t>(b) * a.Hq + kv * R + r;
                const float val = acc / lsum;
                if constexpr (sizeof(T) == 2) {
                    Oout[bh * D + c] = __float2bfloat16_rn(val);
                } else {
                    Oout[bh * D + c] = val;
                }
                if (c == 0) LSEout[bh] = (mx + __log2f(lsum)) * 0.6931471805599453f;
            }
        }
        ptx::cluster_sync();
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float *__restrict__ ws, T *__restrict__ O,
                                                           float *__restrict__ LSE, int splits) {
    static_assert(D >= MAX_SPLITS, "one thread per split for the weights");
    constexpr int NW = D / 32;
    __shared__ float sh_f[MAX_SPLITS];
    __shared__ float sh_wm[NW], sh_wl[NW];
    // Launched as a programmatic dependent of the split kernel, so its CTAs can start while
    // the split grid drains; this waits until that grid has completed and its partials are
    // visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // A programmatic dependent of this kernel (the next decode step's split kernel, say) may
    // be scheduled from here on, once the split grid has completed; it waits for this grid's
    // completion before it reads anything.  The signal comes after the wait, never before:
    // a merge that signalled first saw its wait return before the split grid had completed.
    asm volatile("griddepcontrol.launch_dependents;");
    const int bh = blockIdx.x;
    const int c = threadIdx.x, lane = c & 31, warp = c >> 5;
    const float *base = ws + static_cast<int64_t>(bh) * MAX_SPLITS * (D + 2);
    // Every load is issued here, at once: column c of each split's partial (they do not
    // depend on the weights) and, in thread s, split s's (max, sum).
    float v[MAX_SPLITS];
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s) v[s] = s < splits ? base[s * (D + 2) + c] : 0.f;
    const float ms = c < splits ? base[c * (D + 2) + D] : -INFINITY;
    const float ls = c < splits ? base[c * (D + 2) + D + 1] : 0.f;
    float mx = ms;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    if (lane == 0) sh_wm[warp] = mx;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < NW; ++w) mx = fmaxf(mx, sh_wm[w]);
    const float f = (ms == -INFINITY) ? 0.f : ptx::ex2(ms - mx);
    if (c < MAX_SPLITS) sh_f[c] = f;
    float lw = ls * f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(kFull, lw, off);
    if (lane == 0) sh_wl[warp] = lw;
    __syncthreads();
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) lsum += sh_wl[w];
    // column c: the splits' values weighed (sh_f is zero past the last split)
    float acc = 0.f;
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s) acc = fmaf(v[s], sh_f[s], acc);
    const float val = acc / lsum;
    if constexpr (sizeof(T) == 2) {
        O[static_cast<int64_t>(bh) * D + c] = __float2bfloat16_rn(val);
    } else {
        O[static_cast<int64_t>(bh) * D + c] = val;
    }
    if (c == 0) LSE[bh] = (mx + __log2f(lsum)) * 0.6931471805599453f;
}

// One warp per (b, kv): pools group j with the supplied group-last queries q[B, Hq, D].
// pool_max: element-wise maximum of the group's rows instead of the weighted sums
// (mean pooling arrives as logit_scale = 0, i.e. equal weights).  headmean (pool_mode
// 3): every query head takes its own softmax over the group and the weights are the
// mean of the r weight vectors; logit_scale is then per head (no 1/r).
constexpr int POOL_GROUP_HM_MAX = 8;

template <typename T, int D>
__global__ void __launch_bounds__(128) pool_group_kernel(const T *__restrict__ q, const T *__restrict__ K,
                                                         const T *__restrict__ V, T *__restrict__ Kc,
                                                         T *__restrict__ Vc, int Hq, int Hkv, int Ncap, int g, int j,
                                                         float logit_scale, int pool_max, int headmean, int n_bk) {
    using VT = Vec<T>;
    constexpr int E = VT::E;
    constexpr int LPR = D / E;
    constexpr int RPI = 32 / LPR;
    const int lane = threadIdx.x & 31;
    const int bk = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (bk >= n_bk) return;
    const int sub = lane / LPR, cl = lane % LPR;
    const int b = bk / Hkv, kv = bk % Hkv, r = Hq / Hkv;
    float qs[E];
#pragma unroll
    for (int e = 0; e < E; ++e) qs[e] = 0.f;
    for (int hh = 0; hh < r; ++hh) {
        float f[E];
        VT::unpack(ldg16(q + (static_cast<int64_t>(b) * Hq + kv * r + hh) * D + cl * E), f);
#pragma unroll
        for (int e = 0; e < E; ++e) qs[e] += f[e];
    }
    const T *kg = K + (static_cast<int64_t>(bk) * Ncap + static_cast<int64_t>(j) * g) * D + cl * E;
    const T *vg = V + (static_cast<int64_t>(bk) * Ncap + static_cast<int64_t>(j) * g) * D + cl * E;
    if (headmean) {
        // Pass 1, head by head: that head's softmax normaliser over the group (max m_h,
        // sum l_h, log2 domain).  Pass 2: weight of row t = (1/r) sum_h 2^(s_h,t - m_h) / l_h.
        __shared__ float2 hml[4][POOL_GROUP_HM_MAX];
        const int wib = threadIdx.x >> 5;
        auto logit = [&](int hh, const float (&kf)[E]) {
            float qf[E];
            VT::unpack(ldg16(q + (static_cast<int64_t>(b) * Hq + kv * r + hh) * D + cl * E), qf);
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) dot = fmaf(qf[e], kf[e], dot);
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(kFull, dot, off);
            return dot * logit_scale;
        };
        for (int hh = 0; hh < r; ++hh) {
            float m = -INFINITY, l = 0.f;
            for (int t0 = 0; t0 < g; t0 += RPI) {
                const int t = t0 + sub;
                float kf[E];
                VT::unpack(t < g ? ldg16(kg + static_cast<int64_t>(t) * D) : make_uint4(0, 0, 0, 0), kf);
                const float xl = logit(hh, kf);
                if (t < g) {
                    const float mn = fmaxf(m, xl);
                    l = l * ptx::ex2(m - mn) + ptx::ex2(xl - mn);
                    m = mn;
                }
            }
#pragma unroll
            for (int off = LPR; off < 32; off <<= 1) {
                const float mo = __shfl_xor_sync(kFull, m, off);
                const float lo_ = __shfl_xor_sync(kFull, l, off);
                const float mn = fmaxf(m, mo);
                const float ca = (m == -INFINITY) ? 0.f : ptx::ex2(m - mn);
                const float cb = (mo == -INFINITY) ? 0.f : ptx::ex2(mo - mn);
                l = l * ca + lo_ * cb;
                m = mn;
            }
            if (lane == 0) hml[wib][hh] = make_float2(m, 1.f / (l * static_cast<float>(r)));
        }
        __syncwarp();
        float ak[E], av[E];
#pragma unroll
        for (int e = 0; e < E; ++e) ak[e] = av[e] = 0.f;
        for (int t0 = 0; t0 < g; t0 += RPI) {
            const int t = t0 + sub;
            float kf[E], vf[E];
            VT::unpack(t < g ? ldg16(kg + static_cast<int64_t>(t) * D) : make_uint4(0, 0, 0, 0), kf);
            VT::unpack(t < g ? ldg16(vg + static_cast<int64_t>(t) * D) : make_uint4(0, 0, 0, 0), vf);
            float wgt = 0.f;
            for (int hh = 0; hh < r; ++hh) {
                const float2 st = hml[wib][hh];
                wgt = fmaf(ptx::ex2(logit(hh, kf) - st.x), st.y, wgt);
            }
            if (t < g) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    ak[e] = fmaf(wgt, kf[e], ak[e]);
                    av[e] = fmaf(wgt, vf[e], av[e]);
                }
            }
        }
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ak[e] += __shfl_xor_sync(kFull, ak[e], off);
                av[e] += __shfl_xor_sync(kFull, av[e], off);
            }
        }
        if (sub == 0) {
            const int64_t orow = (static_cast<int64_t>(bk) * (Ncap / g) + j) * D + cl * E;
            *reinterpret_cast<uint4 *>(Kc + orow) = VT::pack(ak);
            *reinterpret_cast<uint4 *>(Vc + orow) = VT::pack(av);
        }
        return;
    }
    const float init = pool_max ? -INFINITY : 0.f;
    float m = -INFINITY, l = 0.f, ak[E], av[E];
#pragma unroll
    for (int e = 0; e < E; ++e) ak[e] = av[e] = init;
    for (int t0 = 0; t0 < g; t0 += RPI) {
        const int t = t0 + sub;
        float kf[E], vf[E];
        VT::unpack(t < g ? ldg16(kg + static_cast<int64_t>(t) * D) : make_uint4(0, 0, 0, 0), kf);
        VT::unpack(t < g ? ldg16(vg + static_cast<int64_t>(t) * D) : make_uint4(0, 0, 0, 0), vf);
        if (pool_max) {
            if (t < g) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    ak[e] = fmaxf(ak[e], kf[e]);
                    av[e] = fmaxf(av[e], vf[e]);
                }
            }
            continue;
        }
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) dot = fmaf(qs[e], kf[e], dot);
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(kFull, dot, off);
        if (t < g) {
            const float xl = dot * logit_scale;
            const float mn = fmaxf(m, xl);
            const float corr = ptx::ex2(m - mn);
            const float p = ptx::ex2(xl - mn);
            l = l * corr + p;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ak[e] = fmaf(p, kf[e], ak[e] * corr);
                av[e] = fmaf(p, vf[e], av[e] * corr);
            }
            m = mn;
        }
    }
    if (pool_max) {
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ak[e] = fmaxf(ak[e], __shfl_xor_sync(kFull, ak[e], off));
                av[e] = fmaxf(av[e], __shfl_xor_sync(kFull, av[e], off));
            }
        }
    } else {
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
            const float mo = __shfl_xor_sync(kFull, m, off);
            const float lo_ = __shfl_xor_sync(kFull, l, off);
            const float mn = fmaxf(m, mo);
            const float ca = (m == -INFINITY) ? 0.f : ptx::ex2(m - mn);
            const float cb = (mo == -INFINITY) ? 0.f : ptx::ex2(mo - mn);
            l = l * ca + lo_ * cb;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ak[e] = ak[e] * ca + __shfl_xor_sync(kFull, ak[e], off) * cb;
                av[e] = av[e] * ca + __shfl_xor_sync(kFull, av[e], off) * cb;
            }
            m = mn;
        }
        const float inv = 1.f / l;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            ak[e] *= inv;
            av[e] *= inv;
        }
    }
    if (sub == 0) {
        const int64_t orow = (static_cast<int64_t>(bk) * (Ncap / g) + j) * D + cl * E;
        *reinterpret_cast<uint4 *>(Kc + orow) = VT::pack(ak);
        *reinterpret_cast<uint4 *>(Vc + orow) = VT::pack(av);
    }
}

// Slices per (b, kv): enough CTAs for one even wave of `occ` CTAs on every SM (a grid
// of 2 or 3 CTAs on different SMs finishes when the SMs with 3 do), but no slice of
// fewer than MIN_KEYS_PER_SPLIT keys and at most MAX_SPLITS slices.
int decode_splits(int L, int n_bk, int sms, int occ) {
    const int target = occ * sms;
    int sp = (target + n_bk - 1) / n_bk;
    const int by_keys = L / MIN_KEYS_PER_SPLIT;
    if (sp > by_keys) sp = by_keys;
    if (sp > MAX_SPLITS) sp = MAX_SPLITS;
    return sp < 1 ? 1 : sp;
}

// SMs of the current device and resident CTAs per SM of one split-kernel instantiation
// (queried once per device).
template <typename T, int D, int R>
cudaError_t split_occupancy(int &sms, int &occ) {
    struct Info {
        bool ready = false;
        int sms = 0, occ = 0;
        cudaError_t err = cudaSuccess;
    };
    static Info info[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    Info &x = info[dev & 63];
    if (!x.ready) {
        x.err = cudaDeviceGetAttribute(&x.sms, cudaDevAttrMultiProcessorCount, dev);
        if (x.err == cudaSuccess)
            x.err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&x.occ, decode_split_kernel<T, D, R, false>,
                                                                  DEC_WARPS * 32, 0);
        x.ready = true;
    }
    sms = x.sms;
    occ = x.occ < 1 ? 1 : x.occ;
    return x.err;
}

// Largest cluster of split CTAs (one (b, kv) each) that the device schedules for this
// instantiation: 16 with the non-portable size allowed, else 8 (queried once per device;
// 0 when clusters cannot be used).
template <typename T, int D, int R>
int max_split_cluster() {
    struct Info {
        bool ready = false;
        int size = 0;
    };
    static Info info[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    Info &x = info[dev & 63];
    if (!x.ready) {
        x.ready = true;
        auto kern = decode_split_kernel<T, D, R, true>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        for (int size : {16, 8}) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(size, 1);
            cfg.blockDim = dim3(DEC_WARPS * 32);
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = size;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) {
                x.size = size;
                break;
            }
        }
        cudaGetLastError();  // a refused query leaves no error behind
    }
    return x.size;
}

template <typename T, int D, int R>
cudaError_t launch_decode_typed(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc, void *O,
                                float *LSE, const Shape &s, int pos, float *ws, cudaStream_t stream,
                                int *plan_kernels) {
    DecodeArgs a;
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.Ncap = s.N;
    a.g = s.g;
    a.pos = pos;
    a.n_core = visible_cores(pos, s.w, s.g);
    a.lo = window_start(pos, s.w, s.g, s.window_mode);  // first raw token of the window
    a.L = a.n_core + (pos - a.lo + 1);
    int sms = 0, occ = 0;
    cudaError_t oe = split_occupancy<T, D, R>(sms, occ);
    if (oe != cudaSuccess) return oe;
    a.splits = decode_splits(a.L, s.B * s.Hkv, sms, occ);
    a.scale_log2 = s.scale * 1.4426950408889634f;
    const int n_bk = s.B * s.Hkv;
    // Both kernels are programmatic dependent launches: each is scheduled as the grid before
    // it on the stream drains, instead of after it, and orders itself with griddepcontrol.wait
    // (the split kernel on whatever preceded the call, the merge on the split kernel).
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(DEC_WARPS * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // One launch when a cluster per (b, kv) still gives about a full wave of CTAs and every
    // split has at least 256 keys: the splits merge inside their cluster, which saves the
    // merge kernel's hand-off (128K MHA: 28.1 -> 27.3 us per layer).  Otherwise the partials
    // go through the workspace to the merge kernel: with few (b, kv) pairs, which want more
    // splits than a cluster holds, and with short lists, where the 19 splits per (b, kv) of
    // a full wave beat a cluster's 16 (32K MHA: 12.3 against 12.7 us per layer).
    const int csize = g_decode_path == 1 ? 0 : max_split_cluster<T, D, R>();
    const int cl_splits = a.splits < csize ? a.splits : csize;
    const bool fills = 4 * n_bk * cl_splits >= 3 * occ * sms && a.L >= 256 * cl_splits;
    const bool clustered = cl_splits >= 2 && (g_decode_path == 2 || fills);
    if (plan_kernels != nullptr) {  // the plan only: how many kernels the call launches
        *plan_kernels = clustered ? 1 : 2;
        return cudaSuccess;
    }
    if (clustered) {
        a.splits = cl_splits;
        cfg.gridDim = dim3(a.splits, n_bk);
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = a.splits;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, decode_split_kernel<T, D, R, true>, static_cast<const T *>(Q),
                                  static_cast<const T *>(K), static_cast<const T *>(V), static_cast<const T *>(Kc),
                                  static_cast<const T *>(Vc), ws, static_cast<T *>(O), LSE, a);
    }
    cfg.gridDim = dim3(a.splits, n_bk);
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_split_kernel<T, D, R, false>, static_cast<const T *>(Q),
                                       static_cast<const T *>(K), static_cast<const T *>(V),
                                       static_cast<const T *>(Kc), static_cast<const T *>(Vc), ws,
                                       static_cast<T *>(O), LSE, a);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(s.B * s.Hq);
    cfg.blockDim = dim3(D);
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<T, D>, static_cast<const float *>(ws), static_cast<T *>(O),
                              LSE, a.splits);
}

template <typename T, int D>
cudaError_t dispatch_r(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc, void *O,
                       float *LSE, const Shape &s, int pos, float *ws, cudaStream_t stream, int *plan_kernels) {
    switch (s.Hq / s.Hkv) {
        case 1: return launch_decode_typed<T, D, 1>(Q, K, V, Kc, Vc, O, LSE, s, pos, ws, stream, plan_kernels);
        case 2: return launch_decode_typed<T, D, 2>(Q, K, V, Kc, Vc, O, LSE, s, pos, ws, stream, plan_kernels);
        case 4: return launch_decode_typed<T, D, 4>(Q, K, V, Kc, Vc, O, LSE, s, pos, ws, stream, plan_kernels);
        case 8: return launch_decode_typed<T, D, 8>(Q, K, V, Kc, Vc, O, LSE, s, pos, ws, stream, plan_kernels);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

// Scratch of cca_decode_fwd_noalloc: a fixed array in the library's device image.
// Every GPU that loads the library holds it until the process exits.  Host code may
// not use its name as an address (on the host it is only a stand-in); the device
// address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[DECODE_NOALLOC_MAX_BYTES];

// The address belongs to the module loaded into one context: after cudaDeviceReset (or
// any other end of the device's primary context) the next context loads the module
// again, possibly elsewhere.  So the cached address is kept with the context that was
// current when it was looked up, and looked up again when another context is current.
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

static CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    });
    return fn;
}

cudaError_t decode_noalloc_scratch(float **out) {
    static std::mutex mu;
    static void *ptrs[64] = {};
    static CUcontext ctxs[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    CtxGetCurrentFn get_ctx = ctx_get_current();
    if (get_ctx == nullptr) return cudaErrorNotSupported;
    CUcontext ctx = nullptr;  // stays null while no context is current yet
    if (get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorNotSupported;
    std::lock_guard<std::mutex> lock(mu);
    if (ptrs[dev] == nullptr || ctx == nullptr || ctxs[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);  // with `dev` current; binds its context
        if (e != cudaSuccess) return e;
        if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorNotSupported;
        ptrs[dev] = p;
        ctxs[dev] = ctx;
    }
    *out = static_cast<float *>(ptrs[dev]);
    return cudaSuccess;
}

uint64_t decode_workspace_bytes(const Shape &s) {
    return static_cast<uint64_t>(s.B) * s.Hq * MAX_SPLITS * (s.d + 2) * sizeof(float);
}

cudaError_t launch_decode(int dtype, const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                          void *O, float *LSE, const Shape &s, int pos, float *ws, cudaStream_t stream,
                          int *plan_kernels) {
    if (dtype == 0) {
        if (s.d == 128) return dispatch_r<__nv_bfloat16, 128>(Q, K, V, Kc, Vc, O, LSE, s, pos, ws, stream, plan_kernels);
        if (s.d == 64) return dispatch_r<__nv_bfloat16, 64>(Q, K, V, Kc, Vc, O, LSE, s, pos, ws, stream, plan_kernels);
    } else {
        if (s.d == 128) return dispatch_r<float, 128>(Q, K, V, Kc, Vc, O, LSE, s, pos, ws, stream, plan_kernels);
        if (s.d == 64) return dispatch_r<float, 64>(Q, K, V, Kc, Vc, O, LSE, s, pos, ws, stream, plan_kernels);
    }
    return cudaErrorNotSupported;
}

cudaError_t launch_pool_group(int dtype, const void *q, const void *K, const void *V, void *Kc, void *Vc,
                              const Shape &s, int j, cudaStream_t stream) {
    const int n_bk = s.B * s.Hkv;
    const unsigned blocks = static_cast<unsigned>((n_bk + 3) / 4);
    const int hmean = s.pool_mode == 3 ? 1 : 0;
    if (hmean && s.Hq / s.Hkv > POOL_GROUP_HM_MAX) return cudaErrorNotSupported;
    const float ls = s.pool_mode == 1 ? 0.f
                     : s.scale * 1.4426950408889634f / static_cast<float>(hmean ? 1 : s.Hq / s.Hkv);
    const int pmax = s.pool_mode == 2 ? 1 : 0;
    if (dtype == 0) {
        if (s.d == 128)
            pool_group_kernel<__nv_bfloat16, 128><<<blocks, 128, 0, stream>>>(
                static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(K),
                static_cast<const __nv_bfloat16 *>(V), static_cast<__nv_bfloat16 *>(Kc),
                static_cast<__nv_bfloat16 *>(Vc), s.Hq, s.Hkv, s.N, s.g, j, ls, pmax, hmean, n_bk);
        else if (s.d == 64)
            pool_group_kernel<__nv_bfloat16, 64><<<blocks, 128, 0, stream>>>(
                static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(K),
                static_cast<const __nv_bfloat16 *>(V), static_cast<__nv_bfloat16 *>(Kc),
                static_cast<__nv_bfloat16 *>(Vc), s.Hq, s.Hkv, s.N, s.g, j, ls, pmax, hmean, n_bk);
        else
            return cudaErrorNotSupported;
    } else {
        if (s.d == 128)
            pool_group_kernel<float, 128><<<blocks, 128, 0, stream>>>(
                static_cast<const float *>(q), static_cast<const float *>(K), static_cast<const float *>(V),
                static_cast<float *>(Kc), static_cast<float *>(Vc), s.Hq, s.Hkv, s.N, s.g, j, ls, pmax, hmean, n_bk);
        else if (s.d == 64)
            pool_group_kernel<float, 64><<<blocks, 128, 0, stream>>>(
                static_cast<const float *>(q), static_cast<const float *>(K), static_cast<const float *>(V),
                static_cast<float *>(Kc), static_cast<float *>(Vc), s.Hq, s.Hkv, s.N, s.g, j, ls, pmax, hmean, n_bk);
        else
            return cudaErrorNotSupported;
    }
    return cudaGetLastError();
}

}  // namespace cca
