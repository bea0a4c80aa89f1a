// Global-aware pooling ("Core Context Aware Transformers for Long Context
// Language Modeling", Method section, pooling equation): every group of g
// tokens becomes one core key and one core value, the softmax-weighted sums of
// the group's keys and values, weighted by softmax(tau * q_last . k_t) where
// q_last is the query of the group's last token (for grouped-query attention,
// the mean of the logits of the query heads sharing the KV head).
//
// Memory-bound (6*g*d flops per 4*g*d bytes), so the design is about bytes in
// flight.  A persistent grid of one CTA per SM; every warp owns a strided list of
// groups and streams them as "chunks" of up to RS rows (RS*d*e = 4 KB of K and
// 4 KB of V, plus the r group-last query rows with a group's first chunk).
// Each warp feeds its own ring of S shared-memory stages with cp.async.bulk
// copies (one elected lane issues them), so several chunks per warp are in
// flight without holding registers, and the arithmetic on chunk c overlaps the
// copies of chunks c+1 .. c+S-1.  Within a chunk a lane holds one 16-byte
// vector of a row; logits are reduced with shuffles and a running (max, sum)
// carries a group across chunks, so any g works.  Outputs are 16-byte stores.
//
// pool_mode 3 (grouped-query pooling averaged after the softmax): each of the r
// query heads sharing the KV head takes its own softmax over the group and the
// group weights are the mean of the r weight vectors.  Every chunk then carries
// the r query rows.  A group that fits one chunk is done in one pass: head by
// head, the chunk's logits give that head's final (max, sum) and its weights add
// into one weight per row.  A longer group is streamed twice: a first pass over
// its K rows only gathers every head's running (max, sum); the second pass over
// K and V recomputes the logits and sums the weighted rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace cca {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int NW_MAX = 12;                 // warps per CTA (each feeds and consumes its own ring)
constexpr int S_MAX = 8;                   // ring stages per warp
constexpr int HM_MAX = 8;                  // pool_mode 3: query heads per KV head
constexpr uint32_t CHUNK_BYTES = 4096;     // bytes of K (and of V) per chunk
constexpr uint32_t SMEM_BUDGET = 224 * 1024;
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

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

struct PoolArgs {
    int Hq, Hkv, N, g, r;
    int S;                 // ring stages per warp
    uint32_t v_off;        // bytes of one chunk's K rows (V follows them, then the query rows)
    uint32_t stage_bytes;  // K chunk + V chunk + r query rows
    float logit_scale;     // tau * log2(e) / r (0 for mean pooling: equal weights;
                           // tau * log2(e) for pool_mode 3, whose logits are per head)
    int pool_max;          // element-wise max pooling instead of weighted sums
    int headmean;          // pool_mode 3: per-head softmax weights averaged over the r heads
    int npass;             // chunk passes over a group: 2 for pool_mode 3 with more than one chunk
    int64_t n_groups;      // B * Hkv * (N / g)
    int32_t *status;
};

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// HM4: the instantiation for pool_mode 3 with four query heads per KV head and one chunk per
// group, which takes the specialised scoring path below (kept out of the other
// instantiations, whose registers it would otherwise raise).
template <typename T, int D, bool HM4>
__global__ void __launch_bounds__(NW_MAX * 32) pool_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                       const T *__restrict__ V, T *__restrict__ Kc,
                                                       T *__restrict__ Vc, const PoolArgs a) {
    using VT = VecTraits<T>;
    constexpr int E = VT::E;                 // elements per 16-byte vector
    constexpr int LPR = D / E;               // lanes per row
    constexpr int RPI = 32 / LPR;            // rows per warp-wide pass
    constexpr uint32_t ROW_BYTES = D * sizeof(T);
    constexpr int RS = CHUNK_BYTES / ROW_BYTES;  // rows per chunk
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0 && RS % RPI == 0, "unsupported head dim");

    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t bars[NW_MAX][S_MAX];
    __shared__ float2 head_ml[NW_MAX][HM_MAX];  // pool_mode 3: per-head running (max, sum)
    __shared__ int abort_flag;
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int sub = lane / LPR;
    const int cl = lane % LPR;
    if (threadIdx.x == 0) abort_flag = 0;
    if (lane == 0)
        for (int s = 0; s < a.S; ++s) ptx::mbar_init(ptx::smem_addr(&bars[wib][s]), 1);
    ptx::fence_mbar_init();
    __syncthreads();

    const uint32_t ring = ptx::smem_addr(smem_raw) + wib * a.S * a.stage_bytes;
    const int G = a.N / a.g;
    const int nch = (a.g + RS - 1) / RS;  // chunks per group and pass
    const int ncg = nch * a.npass;         // chunks per group
    const int nw = blockDim.x >> 5;
    const int64_t tw = static_cast<int64_t>(gridDim.x) * nw;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * nw + wib;
    const int64_t my_groups = gw < a.n_groups ? (a.n_groups - 1 - gw) / tw + 1 : 0;
    const int64_t n_chunks = my_groups * ncg;

    // Lane 0 brings the warp's chunks into its ring in stream order.  The cursor
    // (stage, chunk of the group, group index j, (b, kv) row bk) advances by counting,
    // so no chunk pays for a 64-bit division.
    int is = 0, ich = 0;
    int64_t ij = gw % G, ibk = gw / G;
    auto issue = [&]() {
        const int ch = ich % nch;                             // chunk within the pass
        const bool with_v = a.npass == 1 || ich >= nch;       // the first of two passes reads K only
        const bool with_q = ch == 0 || a.headmean;            // pool_mode 3 scores every chunk per head
        const int64_t j = ij, bk = ibk;
        const int t0 = ch * RS;
        const int rows = min(RS, a.g - t0);
        const uint32_t stage = ring + static_cast<uint32_t>(is) * a.stage_bytes;
        const uint32_t bar = ptx::smem_addr(&bars[wib][is]);
        const uint32_t kv_bytes = rows * ROW_BYTES;
        ptx::mbar_arrive_expect_tx(bar, (with_v ? 2 : 1) * kv_bytes + (with_q ? a.r * ROW_BYTES : 0));
        const int64_t row0 = bk * a.N + j * a.g + t0;
        ptx::bulk_load(stage, K + row0 * D, kv_bytes, bar);
        if (with_v) ptx::bulk_load(stage + a.v_off, V + row0 * D, kv_bytes, bar);
        if (with_q) {
            const int64_t b = bk / a.Hkv, kv = bk % a.Hkv;
            const int64_t last = (j + 1) * a.g - 1;
            for (int hh = 0; hh < a.r; ++hh)
                ptx::bulk_load(stage + 2 * a.v_off + hh * ROW_BYTES,
                               Q + ((b * a.Hq + kv * a.r + hh) * static_cast<int64_t>(a.N) + last) * D, ROW_BYTES,
                               bar);
        }
        if (++is == a.S) is = 0;
        if (++ich == ncg) {
            ich = 0;
            ij += tw;  // next group of this warp: gid += tw
            if (ij >= G) {
                ibk += ij / G;
                ij %= G;
            }
        }
    };
    if (lane == 0)
        for (int64_t c = 0; c < n_chunks && c < a.S; ++c) issue();
    __syncwarp();

    float q[E], ak[E], av[E];
    float m = -INFINITY, l = 0.f;
    int64_t c = 0;
    int st = 0, ch = 0;   // consumer's stage and chunk-of-group counters (ch < ncg)
    uint32_t ph = 0;      // parity of the stage barrier's current use
    int64_t gid = gw;     // consumer's group
    for (; c < n_chunks; ++c) {
        const uint32_t stage = ring + st * a.stage_bytes;
        volatile int *af = &abort_flag;
        if (!__all_sync(kFull, ptx::wait_bounded(ptx::smem_addr(&bars[wib][st]), ph, af, WAIT_LIMIT_NS)))
            break;
        const int t0 = (ch % nch) * RS;
        const int rows = min(RS, a.g - t0);
        if (ch == 0 && a.headmean) {
#pragma unroll
            for (int e = 0; e < E; ++e) ak[e] = av[e] = 0.f;
        } else if (ch == 0) {
            // new group: sum of the r group-last queries (1/r is in logit_scale)
            const float init = a.pool_max ? -INFINITY : 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                q[e] = 0.f;
                ak[e] = av[e] = init;
            }
            m = -INFINITY;
            l = 0.f;
            for (int hh = 0; hh < a.r; ++hh) {
                float f[E];
                VT::unpack(lds16(stage + 2 * a.v_off + hh * ROW_BYTES + cl * 16), f);
#pragma unroll
                for (int e = 0; e < E; ++e) q[e] += f[e];
            }
        }
        constexpr int PASSES = RS / RPI;
        uint4 kr[PASSES], vr[PASSES];
        float s[PASSES];
        const bool first_pass = a.npass == 1 || ch < nch;  // gathers pool_mode 3's per-head (max, sum)
        const bool last_pass = a.npass == 1 || ch >= nch;  // the chunk's V rows are in the stage
#pragma unroll
        for (int it = 0; it < PASSES; ++it) {
            const int t = it * RPI + sub;
            if (t < rows) {
                kr[it] = lds16(stage + t * ROW_BYTES + cl * 16);
                vr[it] = last_pass ? lds16(stage + a.v_off + t * ROW_BYTES + cl * 16) : make_uint4(0, 0, 0, 0);
            } else {
                kr[it] = vr[it] = make_uint4(0, 0, 0, 0);
            }
        }
        bool scored = false;  // the chunk was taken by a specialised path below
        if constexpr (HM4 && PASSES == 8 && LPR == 16) {
            if (a.headmean && a.npass == 1 && a.r == 4) {
                scored = true;
                // pool_mode 3, four query heads, the whole group in this one chunk: all 32
                // partial dot products (head hh, pass it at index 8 hh + it) first, then one
                // transposed butterfly inside each 16-lane row subgroup (31 -> 30 shuffles
                // for 32 sums), after which lane j of a subgroup holds the scores of head j/4
                // for passes 2 (j%4) and 2 (j%4) + 1 and does that head's softmax for them.
                float val[32];
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    float qh[E];
                    VT::unpack(lds16(stage + 2 * a.v_off + hh * ROW_BYTES + cl * 16), qh);
#pragma unroll
                    for (int it = 0; it < PASSES; ++it) {
                        float f[E];
                        VT::unpack(kr[it], f);
                        float d = qh[0] * f[0];
#pragma unroll
                        for (int e = 1; e < E; ++e) d = fmaf(qh[e], f[e], d);
                        val[hh * PASSES + it] = d;
                    }
                }
#pragma unroll
                for (int o = 8, n = 16; o > 0; o >>= 1, n >>= 1) {
                    const bool up = (lane & o) != 0;
#pragma unroll
                    for (int i = 0; i < n; ++i) {
                        const float keep = up ? val[i + n] : val[i];
                        const float send = up ? val[i] : val[i + n];
                        val[i] = keep + __shfl_xor_sync(kFull, send, o);
                    }
                }
                const int j = lane & 15;
                const int p0 = 2 * (j & 3);  // this lane's passes p0, p0 + 1 of head j / 4
                const float s0 = p0 * RPI + sub < rows ? val[0] * a.logit_scale : -INFINITY;
                const float s1 = (p0 + 1) * RPI + sub < rows ? val[1] * a.logit_scale : -INFINITY;
                // the head's max and sum over its 16 rows: lanes j ^ 1, j ^ 2 and the other subgroup
                float mx = fmaxf(s0, s1);
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));  // finite: row 0 is valid
                const float e0 = ptx::ex2(s0 - mx), e1 = ptx::ex2(s1 - mx);
                float sm = e0 + e1;
                sm += __shfl_xor_sync(kFull, sm, 1);
                sm += __shfl_xor_sync(kFull, sm, 2);
                sm += __shfl_xor_sync(kFull, sm, 16);
                const float inv = 1.f / (sm * 4.f);
                // average over the heads: lanes j ^ 4, j ^ 8 hold the same passes of the others
                float w0 = e0 * inv, w1 = e1 * inv;
                w0 += __shfl_xor_sync(kFull, w0, 4);
                w1 += __shfl_xor_sync(kFull, w1, 4);
                w0 += __shfl_xor_sync(kFull, w0, 8);
                w1 += __shfl_xor_sync(kFull, w1, 8);
                // row weights of this subgroup's passes, from lane it / 2 of the subgroup
                float wgt[PASSES];
#pragma unroll
                for (int it = 0; it < PASSES; ++it)
                    wgt[it] = __shfl_sync(kFull, (it & 1) ? w1 : w0, (lane & 16) + (it >> 1));
#pragma unroll
                for (int it = 0; it < PASSES; ++it) {
                    float fk[E], fv[E];
                    VT::unpack(kr[it], fk);
                    VT::unpack(vr[it], fv);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        ak[e] = fmaf(wgt[it], fk[e], ak[e]);
                        av[e] = fmaf(wgt[it], fv[e], av[e]);
                    }
                }
            }
        }
        if (scored) {
        } else if (a.headmean) {
            // pool_mode 3: weight of row t = (1/r) sum_h 2^(s_h,t - m_h) / l_h
            float wgt[PASSES];
#pragma unroll
            for (int it = 0; it < PASSES; ++it) wgt[it] = 0.f;
#pragma unroll 1
            for (int hh = 0; hh < a.r; ++hh) {
                float qh[E];
                VT::unpack(lds16(stage + 2 * a.v_off + hh * ROW_BYTES + cl * 16), qh);
#pragma unroll
                for (int it = 0; it < PASSES; ++it) {
                    float f[E];
                    VT::unpack(kr[it], f);
                    float p = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) p = fmaf(qh[e], f[e], p);
#pragma unroll
                    for (int o = LPR / 2; o > 0; o >>= 1) p += __shfl_xor_sync(kFull, p, o);
                    s[it] = (it * RPI + sub < rows) ? p * a.logit_scale : -INFINITY;  // log2 domain
                }
                float2 ml = (ch % nch == 0 && first_pass) ? make_float2(-INFINITY, 0.f) : head_ml[wib][hh];
                if (first_pass) {
                    float cm = s[0];
#pragma unroll
                    for (int it = 1; it < PASSES; ++it) cm = fmaxf(cm, s[it]);
#pragma unroll
                    for (int o = LPR; o < 32; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(kFull, cm, o));
                    const float mn = fmaxf(ml.x, cm);  // finite: row t0 of the chunk is valid
                    float cs = 0.f;
#pragma unroll
                    for (int it = 0; it < PASSES; ++it) cs += ptx::ex2(s[it] - mn);
#pragma unroll
                    for (int o = LPR; o < 32; o <<= 1) cs += __shfl_xor_sync(kFull, cs, o);
                    // the reduction ran across row subgroups only: each row counted once
                    ml = make_float2(mn, ml.y * ptx::ex2(ml.x - mn) + cs);
                }
                if (last_pass) {
                    const float wsc = 1.f / (ml.y * static_cast<float>(a.r));
#pragma unroll
                    for (int it = 0; it < PASSES; ++it) wgt[it] = fmaf(ptx::ex2(s[it] - ml.x), wsc, wgt[it]);
                }
                __syncwarp();
                if (lane == 0) head_ml[wib][hh] = ml;
                __syncwarp();
            }
            if (last_pass) {
#pragma unroll
                for (int it = 0; it < PASSES; ++it) {
                    float fk[E], fv[E];
                    VT::unpack(kr[it], fk);
                    VT::unpack(vr[it], fv);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        ak[e] = fmaf(wgt[it], fk[e], ak[e]);
                        av[e] = fmaf(wgt[it], fv[e], av[e]);
                    }
                }
            }
        } else if (a.pool_max) {
            // element-wise maximum of the group's keys and of its values
#pragma unroll
            for (int it = 0; it < PASSES; ++it) {
                if (it * RPI + sub < rows) {
                    float fk[E], fv[E];
                    VT::unpack(kr[it], fk);
                    VT::unpack(vr[it], fv);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        ak[e] = fmaxf(ak[e], fk[e]);
                        av[e] = fmaxf(av[e], fv[e]);
                    }
                }
            }
        } else {
#pragma unroll
        for (int it = 0; it < PASSES; ++it) {
            float f[E];
            VT::unpack(kr[it], f);
            float p = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) p = fmaf(q[e], f[e], p);
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) p += __shfl_xor_sync(kFull, p, o);
            s[it] = (it * RPI + sub < rows) ? p * a.logit_scale : -INFINITY;  // log2 domain
        }
        float cm = s[0];
#pragma unroll
        for (int it = 1; it < PASSES; ++it) cm = fmaxf(cm, s[it]);
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
        for (int it = 0; it < PASSES; ++it) {
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
        // every lane has read the stage: refill it with chunk c + S
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && c + a.S < n_chunks) issue();

        if (ch == ncg - 1) {
            // group done: combine the RPI row-subgroups, normalise, store
            float lt = l, kt[E], vt[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                kt[e] = ak[e];
                vt[e] = av[e];
            }
            if (a.pool_max) {
#pragma unroll
                for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        kt[e] = fmaxf(kt[e], __shfl_xor_sync(kFull, kt[e], o));
                        vt[e] = fmaxf(vt[e], __shfl_xor_sync(kFull, vt[e], o));
                    }
                }
                lt = 1.f;
            } else if (a.headmean) {
#pragma unroll
                for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        kt[e] += __shfl_xor_sync(kFull, kt[e], o);
                        vt[e] += __shfl_xor_sync(kFull, vt[e], o);
                    }
                }
                lt = 1.f;  // the weights are normalised already
            } else {
#pragma unroll
                for (int o = LPR; o < 32; o <<= 1) {
                    lt += __shfl_xor_sync(kFull, lt, o);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        kt[e] += __shfl_xor_sync(kFull, kt[e], o);
                        vt[e] += __shfl_xor_sync(kFull, vt[e], o);
                    }
                }
            }
            const float inv = 1.f / lt;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                kt[e] *= inv;
                vt[e] *= inv;
            }
            const int64_t orow = gid * static_cast<int64_t>(D) + cl * E;  // gid = (b*Hkv + kv)*G + j
            if (RPI >= 2) {
                if (sub == 0) *reinterpret_cast<uint4 *>(Kc + orow) = VT::pack(kt);
                if (sub == 1) *reinterpret_cast<uint4 *>(Vc + orow) = VT::pack(vt);
            } else {
                *reinterpret_cast<uint4 *>(Kc + orow) = VT::pack(kt);
                *reinterpret_cast<uint4 *>(Vc + orow) = VT::pack(vt);
            }
        }
        if (++st == a.S) {
            st = 0;
            ph ^= 1u;
        }
        if (++ch == ncg) {
            ch = 0;
            gid += tw;
        }
    }
    if (c < n_chunks) {
        // gave up: let this warp's copies in flight land before the CTA exits
        volatile int never = 0;
        if (lane == 0) {
            const int64_t end = (c + a.S < n_chunks) ? c + a.S : n_chunks;
            for (int64_t x = c; x < end; ++x)
                ptx::wait_bounded(ptx::smem_addr(&bars[wib][x % a.S]), (x / a.S) & 1, &never, WAIT_LIMIT_NS);
            if (a.status != nullptr) atomicCAS(a.status, 0, static_cast<int32_t>(-4));
        }
        __syncwarp();
    }
}

// Small groups: g = PPG * RPI tokens (PPG row passes per group) with several whole
// groups per chunk: GPC = PASSES / PPG consecutive groups of one (batch, KV head), so
// that no pass of a chunk runs on rows that are not there and no state crosses chunks.
// Every chunk brings its groups' query rows (r per group).  The copies of a chunk are
// issued by several lanes at once.  pool_mode 0, 1 and 2 (pool_mode 3 takes pool_kernel).
// a.n_groups counts chunks here: B * Hkv * ceil(G / GPC).
template <typename T, int D, int PPG>
__global__ void __launch_bounds__(NW_MAX * 32) pool_small_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                             const T *__restrict__ V, T *__restrict__ Kc,
                                                             T *__restrict__ Vc, const PoolArgs a) {
    using VT = VecTraits<T>;
    constexpr int E = VT::E;
    constexpr int LPR = D / E;
    constexpr int RPI = 32 / LPR;
    constexpr uint32_t ROW_BYTES = D * sizeof(T);
    constexpr int RS = CHUNK_BYTES / ROW_BYTES;
    constexpr int PASSES = RS / RPI;
    constexpr int GS = PPG * RPI;      // tokens per group
    constexpr int GPC = PASSES / PPG;  // groups per chunk
    static_assert(PASSES % PPG == 0 && E % 2 == 0, "unsupported small-group shape");

    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t bars[NW_MAX][S_MAX];
    __shared__ int abort_flag;
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int sub = lane / LPR;
    const int cl = lane % LPR;
    if (threadIdx.x == 0) abort_flag = 0;
    if (lane == 0)
        for (int x = 0; x < a.S; ++x) ptx::mbar_init(ptx::smem_addr(&bars[wib][x]), 1);
    ptx::fence_mbar_init();
    __syncthreads();

    const uint32_t ring = ptx::smem_addr(smem_raw) + wib * a.S * a.stage_bytes;
    const int G = a.N / GS;
    const int CPR = (G + GPC - 1) / GPC;  // chunks per (batch, KV head)
    const int nw = blockDim.x >> 5;
    const int64_t tw = static_cast<int64_t>(gridDim.x) * nw;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * nw + wib;
    const int64_t n_chunks = gw < a.n_groups ? (a.n_groups - 1 - gw) / tw + 1 : 0;

    // The whole warp advances the copy cursor (chunk cr of row bk) and issues a chunk:
    // lane 0 arms the barrier, then lane x issues copy x (K, V, then the query rows).
    int is = 0;
    int64_t icr = gw % CPR, ibk = gw / CPR;
    auto issue = [&]() {
        const int j0 = static_cast<int>(icr) * GPC;
        const int ng = min(GPC, G - j0);
        const uint32_t kv_bytes = static_cast<uint32_t>(ng * GS) * ROW_BYTES;
        const uint32_t stage = ring + static_cast<uint32_t>(is) * a.stage_bytes;
        const uint32_t bar = ptx::smem_addr(&bars[wib][is]);
        if (lane == 0) ptx::mbar_arrive_expect_tx(bar, 2 * kv_bytes + static_cast<uint32_t>(ng * a.r) * ROW_BYTES);
        __syncwarp();
        const int64_t bk = ibk;
        const int64_t row0 = bk * a.N + static_cast<int64_t>(j0) * GS;
        const int64_t b = bk / a.Hkv, kv = bk % a.Hkv;
        const int ncopy = 2 + ng * a.r;
        for (int x = lane; x < ncopy; x += 32) {
            if (x == 0) {
                ptx::bulk_load(stage, K + row0 * D, kv_bytes, bar);
            } else if (x == 1) {
                ptx::bulk_load(stage + a.v_off, V + row0 * D, kv_bytes, bar);
            } else {
                const int gi = (x - 2) / a.r, hh = (x - 2) % a.r;
                const int64_t last = static_cast<int64_t>(j0 + gi + 1) * GS - 1;
                ptx::bulk_load(stage + 2 * a.v_off + static_cast<uint32_t>(x - 2) * ROW_BYTES,
                               Q + ((b * a.Hq + kv * a.r + hh) * static_cast<int64_t>(a.N) + last) * D, ROW_BYTES,
                               bar);
            }
        }
        if (++is == a.S) is = 0;
        icr += tw;
        if (icr >= CPR) {
            ibk += icr / CPR;
            icr %= CPR;
        }
    };
    for (int64_t c = 0; c < n_chunks && c < a.S; ++c) issue();

    int64_t c = 0;
    int st = 0;
    uint32_t ph = 0;
    int64_t ccr = gw % CPR, cbk = gw / CPR;  // consumer's chunk
    for (; c < n_chunks; ++c) {
        const uint32_t stage = ring + st * a.stage_bytes;
        volatile int *af = &abort_flag;
        if (!__all_sync(kFull, ptx::wait_bounded(ptx::smem_addr(&bars[wib][st]), ph, af, WAIT_LIMIT_NS)))
            break;
        const int j0 = static_cast<int>(ccr) * GPC;
        const int ng = min(GPC, G - j0);
        const int rows = ng * GS;
        uint4 kr[PASSES], vr[PASSES];
#pragma unroll
        for (int it = 0; it < PASSES; ++it) {
            const int t = it * RPI + sub;
            if (t < rows) {
                kr[it] = lds16(stage + t * ROW_BYTES + cl * 16);
                vr[it] = lds16(stage + a.v_off + t * ROW_BYTES + cl * 16);
            } else {
                kr[it] = vr[it] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int gi = 0; gi < GPC; ++gi) {
            if (gi >= ng) break;  // the same for the whole warp
            float ak[E], av[E];
            if (a.pool_max) {
#pragma unroll
                for (int e = 0; e < E; ++e) ak[e] = av[e] = -INFINITY;
#pragma unroll
                for (int pp = 0; pp < PPG; ++pp) {
                    float fk[E], fv[E];
                    VT::unpack(kr[gi * PPG + pp], fk);
                    VT::unpack(vr[gi * PPG + pp], fv);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        ak[e] = fmaxf(ak[e], fk[e]);
                        av[e] = fmaxf(av[e], fv[e]);
                    }
                }
#pragma unroll
                for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        ak[e] = fmaxf(ak[e], __shfl_xor_sync(kFull, ak[e], o));
                        av[e] = fmaxf(av[e], __shfl_xor_sync(kFull, av[e], o));
                    }
                }
            } else {
                // the sum of the group's r last-token queries (1/r is in logit_scale)
                float q[E];
#pragma unroll
                for (int e = 0; e < E; ++e) q[e] = 0.f;
                for (int hh = 0; hh < a.r; ++hh) {
                    float f[E];
                    VT::unpack(lds16(stage + 2 * a.v_off + static_cast<uint32_t>(gi * a.r + hh) * ROW_BYTES + cl * 16), f);
#pragma unroll
                    for (int e = 0; e < E; ++e) q[e] += f[e];
                }
                float sl[PPG];
#pragma unroll
                for (int pp = 0; pp < PPG; ++pp) {
                    float f[E];
                    VT::unpack(kr[gi * PPG + pp], f);
                    float x = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) x = fmaf(q[e], f[e], x);
#pragma unroll
                    for (int o = LPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
                    sl[pp] = x * a.logit_scale;  // log2 domain; every row of a group is present
                }
                float m = sl[0];
#pragma unroll
                for (int pp = 1; pp < PPG; ++pp) m = fmaxf(m, sl[pp]);
#pragma unroll
                for (int o = LPR; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
                float l = 0.f;
                uint64_t ak2[E / 2], av2[E / 2];
#pragma unroll
                for (int e = 0; e < E / 2; ++e) ak2[e] = av2[e] = 0ull;
#pragma unroll
                for (int pp = 0; pp < PPG; ++pp) {
                    const float w = ptx::ex2(sl[pp] - m);
                    l += w;
                    const uint64_t w2 = ptx::f2(w, w);
                    float fk[E], fv[E];
                    VT::unpack(kr[gi * PPG + pp], fk);
                    VT::unpack(vr[gi * PPG + pp], fv);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) {
                        ak2[e] = ptx::fma2(w2, ptx::f2(fk[2 * e], fk[2 * e + 1]), ak2[e]);
                        av2[e] = ptx::fma2(w2, ptx::f2(fv[2 * e], fv[2 * e + 1]), av2[e]);
                    }
                }
#pragma unroll
                for (int e = 0; e < E / 2; ++e) {
                    ptx::f2_split(ak2[e], ak[2 * e], ak[2 * e + 1]);
                    ptx::f2_split(av2[e], av[2 * e], av[2 * e + 1]);
                }
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
            }
            const int64_t orow = (cbk * G + j0 + gi) * static_cast<int64_t>(D) + cl * E;
            if (RPI >= 2) {
                if (sub == 0) *reinterpret_cast<uint4 *>(Kc + orow) = VT::pack(ak);
                if (sub == 1) *reinterpret_cast<uint4 *>(Vc + orow) = VT::pack(av);
            } else {
                *reinterpret_cast<uint4 *>(Kc + orow) = VT::pack(ak);
                *reinterpret_cast<uint4 *>(Vc + orow) = VT::pack(av);
            }
        }
        // every lane has read the stage: refill it with chunk c + S
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (c + a.S < n_chunks) issue();
        if (++st == a.S) {
            st = 0;
            ph ^= 1u;
        }
        ccr += tw;
        if (ccr >= CPR) {
            cbk += ccr / CPR;
            ccr %= CPR;
        }
    }
    if (c < n_chunks) {
        // gave up: let this warp's copies in flight land before the CTA exits
        volatile int never = 0;
        if (lane == 0) {
            const int64_t end = (c + a.S < n_chunks) ? c + a.S : n_chunks;
            for (int64_t x = c; x < end; ++x)
                ptx::wait_bounded(ptx::smem_addr(&bars[wib][x % a.S]), (x / a.S) & 1, &never, WAIT_LIMIT_NS);
            if (a.status != nullptr) atomicCAS(a.status, 0, static_cast<int32_t>(-4));
        }
        __syncwarp();
    }
}

struct DevInfo {
    bool ready = false;
    int sms = 0;
};

int sm_count() {
    static DevInfo info[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    DevInfo &d = info[dev & 63];
    if (!d.ready) {
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        d.ready = true;
    }
    return d.sms;
}

// Ring geometry shared by both kernels: NW_MAX warps (more warps hide the per-chunk
// arithmetic) and as many stages as the budget allows, at least two per warp, trading
// warps for stages when a stage is large.  Returns the warp count, 0 if a stage does not fit.
int ring_geometry(PoolArgs &a) {
    int nw = NW_MAX;
    a.S = static_cast<int>(SMEM_BUDGET / (nw * a.stage_bytes));
    if (a.S > S_MAX) a.S = S_MAX;
    if (a.S < 2) {
        a.S = 2;
        nw = static_cast<int>(SMEM_BUDGET / (a.S * a.stage_bytes));
        if (nw > NW_MAX) nw = NW_MAX;
    }
    return nw;
}

template <typename T, int D, int PPG>
cudaError_t launch_small(const void *Q, const void *K, const void *V, void *Kc, void *Vc, const Shape &s,
                         int32_t *status, cudaStream_t stream) {
    constexpr uint32_t ROW = D * sizeof(T);
    constexpr int RPI = 32 / (D / VecTraits<T>::E);
    constexpr int GPC = (CHUNK_BYTES / ROW / RPI) / PPG;
    PoolArgs a;
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.N = s.N;
    a.g = s.g;
    a.r = s.Hq / s.Hkv;
    a.v_off = CHUNK_BYTES;
    a.stage_bytes = 2 * CHUNK_BYTES + static_cast<uint32_t>(GPC * a.r) * ROW;
    const int nw = ring_geometry(a);
    if (nw < 1) return cudaErrorNotSupported;
    a.headmean = 0;
    a.npass = 1;
    a.logit_scale = s.pool_mode == 1 ? 0.f : s.scale * 1.4426950408889634f / static_cast<float>(a.r);
    a.pool_max = s.pool_mode == 2 ? 1 : 0;
    const int64_t G = s.N / s.g;
    a.n_groups = static_cast<int64_t>(s.B) * s.Hkv * ((G + GPC - 1) / GPC);  // chunks
    a.status = status;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(pool_small_kernel<T, D, PPG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(SMEM_BUDGET));
    });
    if (attr != cudaSuccess) return attr;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int64_t want = (a.n_groups + nw - 1) / nw;
    const unsigned grid = static_cast<unsigned>(want < sms ? want : sms);
    pool_small_kernel<T, D, PPG><<<grid, nw * 32, nw * a.S * a.stage_bytes, stream>>>(
        static_cast<const T *>(Q), static_cast<const T *>(K), static_cast<const T *>(V), static_cast<T *>(Kc),
        static_cast<T *>(Vc), a);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_typed(const void *Q, const void *K, const void *V, void *Kc, void *Vc, const Shape &s,
                         int32_t *status, cudaStream_t stream) {
    constexpr uint32_t ROW = D * sizeof(T);
    // groups of 1, 2 or 4 row passes take the small-group kernel (not pool_mode 3)
    constexpr int RPI = 32 / (D / VecTraits<T>::E);
    if (s.pool_mode != 3) {
        if (s.g == RPI) return launch_small<T, D, 1>(Q, K, V, Kc, Vc, s, status, stream);
        if (s.g == 2 * RPI) return launch_small<T, D, 2>(Q, K, V, Kc, Vc, s, status, stream);
        if (s.g == 4 * RPI) return launch_small<T, D, 4>(Q, K, V, Kc, Vc, s, status, stream);
    }
    PoolArgs a;
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.N = s.N;
    a.g = s.g;
    a.r = s.Hq / s.Hkv;
    // A chunk carries at most min(g, CHUNK_BYTES / row) rows, so a stage holds just that
    // much K and V plus the r query rows.  NW_MAX warps (more warps hide the per-chunk
    // arithmetic), and as many stages as the budget allows (small groups give small
    // stages, so more of them keep the same bytes in flight); at least two stages per
    // warp, trading warps for stages when a stage is large.
    const uint32_t chunk_rows = static_cast<uint32_t>(s.g) < CHUNK_BYTES / ROW ? static_cast<uint32_t>(s.g)
                                                                               : CHUNK_BYTES / ROW;
    a.v_off = chunk_rows * ROW;
    a.stage_bytes = 2 * a.v_off + static_cast<uint32_t>(a.r) * ROW;
    const int nw = ring_geometry(a);
    if (nw < 1) return cudaErrorNotSupported;  // a stage would not fit (hundreds of query heads per KV head)
    a.headmean = s.pool_mode == 3 ? 1 : 0;
    if (a.headmean && a.r > HM_MAX) return cudaErrorNotSupported;
    a.npass = (a.headmean && static_cast<uint32_t>(s.g) > chunk_rows) ? 2 : 1;
    a.logit_scale = s.pool_mode == 1 ? 0.f
                    : s.scale * 1.4426950408889634f / static_cast<float>(a.headmean ? 1 : a.r);
    a.pool_max = s.pool_mode == 2 ? 1 : 0;
    a.n_groups = static_cast<int64_t>(s.B) * s.Hkv * (s.N / s.g);
    a.status = status;
    const uint32_t smem = nw * a.S * a.stage_bytes;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(pool_kernel<T, D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(SMEM_BUDGET));
        if (attr == cudaSuccess)
            attr = cudaFuncSetAttribute(pool_kernel<T, D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(SMEM_BUDGET));
    });
    if (attr != cudaSuccess) return attr;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int64_t want = (a.n_groups + nw - 1) / nw;
    const unsigned grid = static_cast<unsigned>(want < sms ? want : sms);
    const bool hm4 = a.headmean && a.npass == 1 && a.r == 4;
    if (hm4)
        pool_kernel<T, D, true><<<grid, nw * 32, smem, stream>>>(static_cast<const T *>(Q), static_cast<const T *>(K),
                                                                 static_cast<const T *>(V), static_cast<T *>(Kc),
                                                                 static_cast<T *>(Vc), a);
    else
        pool_kernel<T, D, false><<<grid, nw * 32, smem, stream>>>(static_cast<const T *>(Q),
                                                                  static_cast<const T *>(K),
                                                                  static_cast<const T *>(V), static_cast<T *>(Kc),
                                                                  static_cast<T *>(Vc), a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pool(int dtype, const void *Q, const void *K, const void *V, void *Kc, void *Vc,
                        const Shape &s, int32_t *status, cudaStream_t stream) {
    if (dtype == 0) {
        if (s.d == 128) return launch_typed<__nv_bfloat16, 128>(Q, K, V, Kc, Vc, s, status, stream);
        if (s.d == 64) return launch_typed<__nv_bfloat16, 64>(Q, K, V, Kc, Vc, s, status, stream);
    } else {
        if (s.d == 128) return launch_typed<float, 128>(Q, K, V, Kc, Vc, s, status, stream);
        if (s.d == 64) return launch_typed<float, 64>(Q, K, V, Kc, Vc, s, status, stream);
    }
    return cudaErrorNotSupported;
}

}  // namespace cca
