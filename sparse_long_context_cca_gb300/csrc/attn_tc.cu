// Fused core/local attention, bf16, d = 128, on the sm_103a tensor cores
// ("Core Context Aware Transformers for Long Context Language Modeling",
// Method section, fusion equation
//     Att_i = softmax(Q_i [K^G_{T_i}; K^L_{U_i}]^T / sqrt(d)) [V^G_{T_i}; V^L_{U_i}]).
//
// One CTA owns one tile of 128 query rows of one (batch, query head).  The
// keys it visits form one sequence of 128-key tiles: first the core tokens
// Kc/Vc [0, n_core(last row)), then the raw tokens K/V of the band
// [lo(first row), last row].  A single online-softmax state (row max m, row
// sum l, output accumulator O in tensor memory) runs over the whole sequence,
// so the core and local segments share one normalisation.  Only tiles that
// straddle a visibility edge are masked:
//   core tile:  column c (core y0+c) is visible to row i iff y0 + c < lo(i)/g;
//   local tile: column c (token y0+c) is visible to row i iff lo(i) <= y0+c <= i.
//
// Roles (192 threads):
//   warp 0      TMA producer: Q tile once, then K/V tiles into a ring of NS
//               32 KB shared-memory slots (128-byte swizzle, two 64-column
//               halves per tile);
//   warp 1      MMA issuer (one thread): S = Q K^T into TMEM (fp32), then
//               O += P V with P read from TMEM (bf16);
//   warps 2..5  softmax + epilogue: thread t owns TMEM lane / query row t.
// Tensor memory (512 columns): S0 | S1 | O | P0 | P1, S and P double-buffered
// so that the QK^T of tile j+1 and the PV of tile j-1 overlap the softmax of j.
// Every mbarrier wait is bounded in time; on a time-out the CTA stops, drains
// what it has in flight, frees its tensor memory and reports CCA_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace cca {
namespace {

constexpr int BM = 128;                       // query rows per CTA
constexpr int BN = 128;                       // keys per tile
constexpr int HD = 128;                       // head dimension
constexpr int NS = 5;                         // ring slots
constexpr uint32_t TILE_BYTES = BN * HD * 2;  // one bf16 128x128 tile
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S0 = 0, TM_O = 256, TM_P0 = 384;  // S1 = 128, P1 = 448
constexpr float LAZY_RESCALE_LOG2 = 8.0f;     // keep a stale max while it is within 2^8

constexpr uint32_t IDESC_QK = ptx::idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(BM, HD, 0, 1);  // P (TMEM), V MN-major

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_RING = TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_RING + NS * TILE_BYTES;
// barrier indices
constexpr int B_QFULL = 0;
constexpr int B_FULL = 1;              // NS
constexpr int B_EMPTY = B_FULL + NS;   // NS
constexpr int B_SFULL = B_EMPTY + NS;  // 2
constexpr int B_SFREE = B_SFULL + 2;   // 2
constexpr int B_PFULL = B_SFREE + 2;   // 2
constexpr int B_PVDONE = B_PFULL + 2;  // 2
constexpr int B_DRAIN = B_PVDONE + 2;
constexpr int NUM_BARS = B_DRAIN + 1;
constexpr uint32_t OFF_TMEMPTR = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEMPTR + 4;
constexpr uint32_t SMEM_USED = OFF_ABORT + 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for manual alignment

struct Params {
    int B, Hq, Hkv, N, g, w, n_qtiles;
    float scale_log2;
    __nv_bfloat16 *O;
    float *LSE;
    int32_t *status;
    unsigned long long wait_limit_ns;
    int skip_q_load;  // test hook: never load Q, so the pipeline waits run out
};

struct TileRange {
    int Tc, T, lo0, i0, i1, nc_min, lo1;
};

__device__ __forceinline__ int lo_of(int i, int w) { return i - w + 1 > 0 ? i - w + 1 : 0; }

__device__ __forceinline__ TileRange tile_range(const Params &p, int qt) {
    TileRange r;
    r.i0 = qt * BM;
    r.i1 = min(r.i0 + BM - 1, p.N - 1);
    r.lo0 = lo_of(r.i0, p.w);
    r.lo1 = lo_of(r.i1, p.w);
    const int nc_max = r.lo1 / p.g;
    r.nc_min = r.lo0 / p.g;
    r.Tc = (nc_max + BN - 1) / BN;
    const int Tl = (r.i1 - r.lo0 + 1 + BN - 1) / BN;
    r.T = r.Tc + Tl;
    return r;
}

// Load order shared by the producer and the MMA issuer:
// K0, K1, V0, K2, V1, ..., K(T-1), V(T-2), V(T-1).
__device__ __forceinline__ void decode_load(int u, int T, bool &is_v, int &t) {
    if (u == 0) {
        is_v = false;
        t = 0;
    } else if (u == 2 * T - 1) {
        is_v = true;
        t = T - 1;
    } else if (u & 1) {
        is_v = false;
        t = (u + 1) >> 1;
    } else {
        is_v = true;
        t = (u >> 1) - 1;
    }
}

__device__ __forceinline__ void report_timeout(const Params &p) {
    if (p.status != nullptr) atomicCAS(p.status, 0, static_cast<int32_t>(-4));
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKc,
                        const __grid_constant__ CUtensorMap tmVc, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    auto bar = [&](int idx) -> uint32_t { return base + OFF_BAR + 8u * idx; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + OFF_ABORT);
    uint32_t *tmem_ptr_smem = reinterpret_cast<uint32_t *>(gbase + OFF_TMEMPTR);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Heaviest query tiles first: block x -> (tile rank, batch*head).
    const int BH = p.B * p.Hq;
    const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x / BH);
    const int bh = static_cast<int>(blockIdx.x % BH);
    const int b = bh / p.Hq, h = bh % p.Hq;
    const int kvz = b * p.Hkv + h / (p.Hq / p.Hkv);
    const TileRange tr = tile_range(p, qt);
    const int T = tr.T;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(B_QFULL), 1);
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(bar(B_FULL + s), 1);
            ptx::mbar_init(bar(B_EMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(bar(B_SFULL + s), 1);
            ptx::mbar_init(bar(B_SFREE + s), 128);
            ptx::mbar_init(bar(B_PFULL + s), 128);
            ptx::mbar_init(bar(B_PVDONE + s), 1);
        }
        ptx::mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(base + OFF_TMEMPTR, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_ptr_smem;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tmQ);
            ptx::prefetch_tmap(&tmK);
            ptx::prefetch_tmap(&tmV);
            ptx::prefetch_tmap(&tmKc);
            ptx::prefetch_tmap(&tmVc);
            if (!p.skip_q_load) {
                ptx::mbar_arrive_expect_tx(bar(B_QFULL), TILE_BYTES);
                ptx::tma_load_3d(&tmQ, bar(B_QFULL), base + OFF_Q, 0, tr.i0, bh);
                ptx::tma_load_3d(&tmQ, bar(B_QFULL), base + OFF_Q + HALF_BYTES, 64, tr.i0, bh);
            }
            int issued = 0;
            for (int u = 0; u < 2 * T; ++u) {
                const int slot = u % NS;
                if (!ptx::wait_bounded(bar(B_EMPTY + slot), ((u / NS) & 1) ^ 1, abort_flag, p.wait_limit_ns))
                    break;
                bool is_v;
                int t;
                decode_load(u, T, is_v, t);
                const bool core = t < tr.Tc;
                const void *map = core ? (is_v ? (const void *)&tmVc : (const void *)&tmKc)
                                       : (is_v ? (const void *)&tmV : (const void *)&tmK);
                const int y = core ? t * BN : tr.lo0 + (t - tr.Tc) * BN;
                const uint32_t dst = base + OFF_RING + slot * TILE_BYTES;
                ptx::mbar_arrive_expect_tx(bar(B_FULL + slot), TILE_BYTES);
                ptx::tma_load_3d(map, bar(B_FULL + slot), dst, 0, y, kvz);
                ptx::tma_load_3d(map, bar(B_FULL + slot), dst + HALF_BYTES, 64, y, kvz);
                issued = u + 1;
            }
            if (*abort_flag) {
                // Let the copies already issued land before the CTA exits.
                for (int u = issued - NS > 0 ? issued - NS : 0; u < issued; ++u) {
                    volatile int never = 0;
                    ptx::wait_bounded(bar(B_FULL + u % NS), (u / NS) & 1, &never, p.wait_limit_ns);
                }
                if (!p.skip_q_load) {
                    volatile int never = 0;
                    ptx::wait_bounded(bar(B_QFULL), 0, &never, p.wait_limit_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = ptx::wait_bounded(bar(B_QFULL), 0, abort_flag, p.wait_limit_ns);
            for (int u = 0; ok && u < 2 * T; ++u) {
                const int slot = u % NS;
                if (!ptx::wait_bounded(bar(B_FULL + slot), (u / NS) & 1, abort_flag, p.wait_limit_ns)) break;
                bool is_v;
                int t;
                decode_load(u, T, is_v, t);
                const int sb = t & 1;
                const uint32_t tile = base + OFF_RING + slot * TILE_BYTES;
                if (!is_v) {
                    if (!ptx::wait_bounded(bar(B_SFREE + sb), ((t >> 1) & 1) ^ 1, abort_flag, p.wait_limit_ns))
                        break;
                    ptx::tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t koff = (kk >> 2) * HALF_BYTES + (kk & 3) * 32;
                        const uint64_t ad = ptx::smem_desc_sw128(base + OFF_Q + koff, 16, 1024);
                        const uint64_t bd = ptx::smem_desc_sw128(tile + koff, 16, 1024);
                        ptx::mma_ss(tmem + TM_S0 + sb * BN, ad, bd, IDESC_QK, kk > 0 ? 1u : 0u);
                    }
                    ptx::tc_commit(bar(B_SFULL + sb));
                } else {
                    if (!ptx::wait_bounded(bar(B_PFULL + sb), (t >> 1) & 1, abort_flag, p.wait_limit_ns)) break;
                    ptx::tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        const uint64_t bd = ptx::smem_desc_sw128(tile + kk * 2048, HALF_BYTES, 1024);
                        ptx::mma_ts(tmem + TM_O, tmem + TM_P0 + sb * 64 + kk * 8, bd, IDESC_PV,
                                    (t > 0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::tc_commit(bar(B_PVDONE + sb));
                }
                ptx::tc_commit(bar(B_EMPTY + slot));
            }
            // Whatever was issued must complete before tensor memory is freed.
            ptx::tc_commit(bar(B_DRAIN));
            volatile int never = 0;
            ptx::wait_bounded(bar(B_DRAIN), 0, &never, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const int i = tr.i0 + row;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const int lo_i = lo_of(i, p.w);
        const int nc_i = lo_i / p.g;
        float m = -INFINITY;  // running max of the log2-scaled logits
        float l = 0.f;
        bool ok = true;
        for (int t = 0; t < T && ok; ++t) {
            const int sb = t & 1;
            // Waits are made warp-uniform: the tcgen05.ld/st that follow are warp-collective.
            if (!__all_sync(0xffffffffu, ptx::wait_bounded(bar(B_SFULL + sb), (t >> 1) & 1, abort_flag,
                                                            p.wait_limit_ns))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint32_t s[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tmem + lane_addr + TM_S0 + sb * BN + c * 32, s[c]);
            ptx::tmem_wait_ld(s[0]);
            ptx::reg_touch(s[1]);
            ptx::reg_touch(s[2]);
            ptx::reg_touch(s[3]);
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(B_SFREE + sb));

            // visibility window of this row within the tile: columns [c_lo, c_hi]
            const bool core = t < tr.Tc;
            int c_lo = 0, c_hi = BN - 1;
            bool masked;
            if (core) {
                const int y0 = t * BN;
                masked = y0 + BN > tr.nc_min;
                c_hi = min(nc_i - y0, BN) - 1;
            } else {
                const int y0 = tr.lo0 + (t - tr.Tc) * BN;
                masked = (y0 < tr.lo1) || (y0 + BN - 1 > tr.i0);
                c_lo = max(lo_i - y0, 0);
                c_hi = min(i - y0, BN - 1);
            }
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int col = c * 32 + k;
                    float x = __uint_as_float(s[c][k]);
                    if (masked && (col < c_lo || col > c_hi)) x = -INFINITY;
                    s[c][k] = __float_as_uint(x);
                    mx = fmaxf(mx, x);
                }
            }
            const float m_tile = mx * p.scale_log2;  // -inf stays -inf
            const float m_new = fmaxf(m, m_tile);
            bool rescale = false;
            if (m == -INFINITY) {
                m = m_new;  // nothing accumulated yet for this row
            } else if (m_new > m + LAZY_RESCALE_LOG2) {
                rescale = true;
            }
            if (__any_sync(0xffffffffu, rescale)) {
                // O holds the sum up to tile t-1: wait for that PV, then rescale in place.
                if (!__all_sync(0xffffffffu, ptx::wait_bounded(bar(B_PVDONE + ((t - 1) & 1)), ((t - 1) >> 1) & 1,
                                                                abort_flag, p.wait_limit_ns))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const float f = rescale ? ptx::ex2(m - m_new) : 1.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tmem + lane_addr + TM_O + c * 32, o);
                    ptx::tmem_wait_ld(o);
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
                    ptx::tmem_st32(tmem + lane_addr + TM_O + c * 32, o);
                }
                ptx::tmem_wait_st();
                if (rescale) {
                    l *= f;
                    m = m_new;
                }
            }
            const float mu = (m == -INFINITY) ? 0.f : m;
            // P buffer sb was last read by the PV of tile t-2.
            if (t >= 2 && !__all_sync(0xffffffffu, ptx::wait_bounded(bar(B_PVDONE + sb), ((t - 2) >> 1) & 1,
                                                                      abort_flag, p.wait_limit_ns))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float p0 = ptx::ex2(fmaf(__uint_as_float(s[c][2 * k]), p.scale_log2, -mu));
                    const float p1 = ptx::ex2(fmaf(__uint_as_float(s[c][2 * k + 1]), p.scale_log2, -mu));
                    l += p0 + p1;
                    pk[k] = ptx::pack_bf16x2(p0, p1);
                }
                ptx::tmem_st16(tmem + lane_addr + TM_P0 + sb * 64 + c * 16, pk);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(B_PFULL + sb));
        }
        if (ok && __all_sync(0xffffffffu, ptx::wait_bounded(bar(B_PVDONE + ((T - 1) & 1)), ((T - 1) >> 1) & 1,
                                                             abort_flag, p.wait_limit_ns))) {
            ptx::tc_fence_after();
            const bool valid = i < p.N;
            const float inv = 1.f / l;
            __nv_bfloat16 *orow = p.O + (static_cast<int64_t>(bh) * p.N + i) * HD;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                ptx::tmem_ld32(tmem + lane_addr + TM_O + c * 32, o);
                ptx::tmem_wait_ld(o);
                uint4 v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[k].x = ptx::pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv, __uint_as_float(o[8 * k + 1]) * inv);
                    v[k].y = ptx::pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv);
                    v[k].z = ptx::pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv);
                    v[k].w = ptx::pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv);
                }
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k) dst[k] = v[k];
                }
            }
            if (valid) p.LSE[static_cast<int64_t>(bh) * p.N + i] = (m + __log2f(l)) * 0.6931471805599453f;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) report_timeout(p);
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// [heads, rows, 128] bf16 viewed as a 3-D tensor; box = 64 columns x 128 rows x 1 head.
bool encode_3d(EncodeTiledFn enc, CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t heads) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), rows, heads};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(HD) * 2, rows * HD * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Test hooks (see cca_test_* in cca_api.cu).
unsigned long long g_wait_limit_ns = 1000000000ull;
int g_skip_q_load = 0;

cudaError_t launch_attn_bf16_tc(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                                void *O, float *LSE, const Shape &s, int32_t *dev_status, cudaStream_t stream) {
    EncodeTiledFn enc = get_encoder();
    if (enc == nullptr) return cudaErrorNotSupported;
    const uint64_t G = static_cast<uint64_t>(s.N / s.g);
    CUtensorMap mQ, mK, mV, mKc, mVc;
    const uint64_t qh = static_cast<uint64_t>(s.B) * s.Hq, kh = static_cast<uint64_t>(s.B) * s.Hkv;
    if (!encode_3d(enc, &mQ, Q, s.N, qh) || !encode_3d(enc, &mK, K, s.N, kh) || !encode_3d(enc, &mV, V, s.N, kh) ||
        !encode_3d(enc, &mKc, Kc, G, kh) || !encode_3d(enc, &mVc, Vc, G, kh))
        return cudaErrorInvalidValue;

    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(attn_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(SMEM_BYTES));
    });
    if (attr_err != cudaSuccess) return attr_err;

    Params p;
    p.B = s.B;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.N = s.N;
    p.g = s.g;
    p.w = s.w;
    p.n_qtiles = (s.N + BM - 1) / BM;
    p.scale_log2 = s.scale * 1.4426950408889634f;
    p.O = static_cast<__nv_bfloat16 *>(O);
    p.LSE = LSE;
    p.status = dev_status;
    p.wait_limit_ns = g_wait_limit_ns;
    p.skip_q_load = g_skip_q_load;
    const unsigned grid = static_cast<unsigned>(static_cast<uint64_t>(p.n_qtiles) * s.B * s.Hq);
    attn_bf16_tc_kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(mQ, mK, mV, mKc, mVc, p);
    return cudaGetLastError();
}

}  // namespace cca
