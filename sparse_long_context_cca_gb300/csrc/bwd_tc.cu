// Tensor-core backward of the fused core/local attention (bf16, d = 128): the
// gradient of the fusion equation of "Core Context Aware Transformers for Long
// Context Language Modeling" (Method section), with P recomputed from the
// forward's LSE.  Notation as in bwd.cu: dS = P (dO.v - D), D_i = dO_i . O_i.
//
// Two kernels, both warp-specialised with 320 threads: warp 0 issues the TMA copies,
// warp 1 the tcgen05.mma instructions (one elected lane), warps 2..9 do the
// element-wise work; they hand off through mbarriers, never a CTA-wide barrier
// inside the loop.  For the element-wise work warps w and w + 4 share TMEM lanes
// 32*(w%4)..+31 and split the 128 columns, 64 each.  The fp32 results leave
// through shared memory and tiled TMA stores.
//
//  dq kernel, one 128-row query tile of one (b, h) per CTA, over the same key
//  tiles as the forward (cores, then the band):
//     S = Q K^T, dP = dO V^T (both SS, fp32 in TMEM)  ->  dS (bf16, over S)
//     dQ += dS K  (A = dS in TMEM, B = K tile read MN-major)
//  TMEM: S | dP | dQ.  K/V tiles are double-buffered: the next tile's copy is
//  in flight while this one is processed.
//
//  dkv kernel, one 128-key tile (raw tokens or cores) of one (b, kv) per CTA,
//  over the query tiles of the r query heads that see any of its keys:
//     S^T = K Q^T, dP^T = V dO^T  ->  P^T over S^T, dS^T over dP^T (bf16)
//     dV += P^T dO,  dK += dS^T Q   (A in TMEM, B = Q / dO tiles read MN-major)
//  TMEM: S^T | dP^T | dK | dV.  Q/dO tiles are double-buffered.
//
// The pooling backward (bwd.cu) then adds the paths through the core tokens.
// Every wait is bounded and a time-out sets the CTA's abort flag, which ends every
// other wait at once: the issuer then waits (bounded) for the MMAs it has issued,
// the producer for its copies in flight, TMEM is freed and CCA_ERR_TIMEOUT is
// written to the status word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "sm100_ptx.cuh"
#include "tma_host.h"
#include "visibility.cuh"

namespace cca {

extern unsigned long long g_wait_limit_ns;
extern int g_skip_q_load;

namespace {

constexpr int BT = 128;  // rows per tile (queries or keys)
constexpr int HD = 128;
constexpr uint32_t TILE_BYTES = BT * HD * 2;
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;
constexpr uint32_t IDESC_SS = ptx::idesc_bf16_f32(128, 128, 0, 0);  // K-major A and B
constexpr uint32_t IDESC_TS = ptx::idesc_bf16_f32(128, 128, 0, 1);  // A in TMEM, B MN-major
constexpr float LOG2E = 1.4426950408889634f;
constexpr int32_t STATUS_TIMEOUT = -4;

struct BwdTcParams {
    int B, Hq, Hkv, N, g, w, window_mode, G;
    float tau;
    const float *LSE;
    const __nv_bfloat16 *O, *dO;
    float *Dbuf;  // written by the dq kernel, read by the dkv kernel
    int tile0;    // first key tile of this dkv launch (core tiles come first)
    int core_chunk;  // > 0: core tiles in items of this many query tiles, summed into dKc/dVc
    // pooling backward folded into the raw-token tiles' epilogue (BwdPoolFuse)
    int pool_fuse;
    const float *pool_a, *pool_cds, *pool_qs, *pool_dkc, *pool_dvc;
    int32_t *status;
    unsigned long long wait_limit_ns;
    int skip_loads;  // test hook: issue no copies, so the first wait runs out
};

__device__ __forceinline__ int lo_of(int i, int w) { return window_lo(i, w); }
__device__ __forceinline__ int win_of(const BwdTcParams &p, int i) { return window_start(i, p.w, p.g, p.window_mode); }

__device__ __forceinline__ float bf(uint32_t w, int hi) {
    return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16));
}

__device__ __forceinline__ void load_tile(const void *map, uint32_t bar, uint32_t dst, int y, int z) {
    ptx::tma_load_3d(map, bar, dst, 0, y, z);
    ptx::tma_load_3d(map, bar, dst + HALF_BYTES, 64, y, z);
}

// Writes this thread's 64 fp32 values (columns [64*ch, 64*ch + 64) of TMEM row `row`,
// starting at TMEM column `tcol`) times `scale` into the shared-memory staging of a
// 128 x 128 fp32 tile: four 128-byte-swizzled boxes of 32 columns x 128 rows, 16 KB
// each, as the tiled store expects.  Rows in a group of 8 write different 16-byte
// chunks, so the stores do not collide in banks.
__device__ __forceinline__ void stage_f32_rows(uint32_t tmem_row_addr, int tcol, int ch, int row, float scale,
                                               bool zero, uint32_t stage) {
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {
        const int c = 2 * ch + j;  // 32-column box
        uint32_t v[32];
        if (!zero) {
            ptx::tmem_ld32(tmem_row_addr + tcol + c * 32, v);
            ptx::tmem_wait_ld(v);
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = 0u;
        }
        const uint32_t rbase = stage + c * (BT * 128) + row * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            ptx::st_shared_v4(rbase + ((q ^ (row & 7)) << 4), __uint_as_float(v[4 * q]) * scale,
                              __uint_as_float(v[4 * q + 1]) * scale, __uint_as_float(v[4 * q + 2]) * scale,
                              __uint_as_float(v[4 * q + 3]) * scale);
    }
}
// As stage_f32_rows, adding xs * x + ys * y (x, y: fp32 rows of 128 in global memory;
// y may be nullptr) to every element: the pooling backward's share of a raw token's
// gradient.
__device__ __forceinline__ void stage_f32_rows_plus(uint32_t tmem_row_addr, int tcol, int ch, int row, float scale,
                                                    bool zero, uint32_t stage, const float *x, float xs,
                                                    const float *y, float ys) {
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {
        const int c = 2 * ch + j;  // 32-column box
        uint32_t v[32];
        if (!zero) {
            ptx::tmem_ld32(tmem_row_addr + tcol + c * 32, v);
        } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = 0u;
        }
        float4 xv[8], yv[8];
        const float4 *x4 = reinterpret_cast<const float4 *>(x + c * 32);
        const float4 *y4 = reinterpret_cast<const float4 *>(y + c * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            xv[q] = x4[q];
            yv[q] = y != nullptr ? y4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (!zero) ptx::tmem_wait_ld(v);
        const uint32_t rbase = stage + c * (BT * 128) + row * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            ptx::st_shared_v4(rbase + ((q ^ (row & 7)) << 4),
                              fmaf(ys, yv[q].x, fmaf(xs, xv[q].x, __uint_as_float(v[4 * q]) * scale)),
                              fmaf(ys, yv[q].y, fmaf(xs, xv[q].y, __uint_as_float(v[4 * q + 1]) * scale)),
                              fmaf(ys, yv[q].z, fmaf(xs, xv[q].z, __uint_as_float(v[4 * q + 2]) * scale)),
                              fmaf(ys, yv[q].w, fmaf(xs, xv[q].w, __uint_as_float(v[4 * q + 3]) * scale)));
    }
}

// Thread 0 stores a staged 128 x 128 fp32 tile (four boxes) at rows [y, y + 128) of head z
// (or adds it to what is there); rows past the tensor's end are not written.
__device__ __forceinline__ void store_tile_f32(const CUtensorMap *map, uint32_t stage, int y, int z,
                                               bool add = false) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (add) ptx::tma_reduce_add_3d(map, stage + c * (BT * 128), c * 32, y, z);
        else ptx::tma_store_3d(map, stage + c * (BT * 128), c * 32, y, z);
    }
    ptx::bulk_commit_group();
}

// ---------------------------------------------------------------- dQ
// One 128-row query tile of one (b, h) per CTA, over the forward's key tiles (cores,
// then the band).  Warp-specialised, 320 threads:
//   warp 0      producer: Q and dO once, then K(t) into one of three stages and V(t)
//               into one of two (TMA; K lives longer: S(t) and dQ(t) read it);
//   warp 1      MMA issuer, per tile t:  S(t+1) = Q K(t+1)^T into the other S buffer,
//               then (once the element-wise warps have written dS(t)) dQ += dS(t) K(t),
//               then dP(t+1) = dO V(t+1)^T;
//   warps 2..9  element-wise: P = 2^(S tau log2e - LSE) as soon as S(t) is there (while
//               dP(t) is still being computed), then dS = P (dP - D) as bf16 over S.
//               Warps w and w + 4 share TMEM lanes 32*(w%4)..+31 (the query rows) and
//               split the 128 key columns, 64 each.  Each also computes D = dO . O of its
//               row (the first of the pair stores it for the dK/dV kernel).
// TMEM: S0 | S1 | dP | dQ, 128 columns each.  S is double-buffered so that the tensor
// pipe computes the next tile's S while this tile's dS is formed.
constexpr int DQ_THREADS = 320;
constexpr int DQ_KST = 3, DQ_VST = 2;
constexpr uint32_t DQ_OFF_K = 2 * TILE_BYTES;  // after Q, dO
constexpr uint32_t DQ_OFF_V = DQ_OFF_K + DQ_KST * TILE_BYTES;
constexpr uint32_t DQ_OFF_BAR = DQ_OFF_V + DQ_VST * TILE_BYTES;
constexpr int QB_QD = 0, QB_FULLK = 1, QB_EMPTYK = 4, QB_FULLV = 7, QB_EMPTYV = 9, QB_SFULL = 11, QB_DPFULL = 13,
              QB_PFULL = 14, QB_DONE = 15, QB_DRAIN = 16;
constexpr int DQ_NBARS = 17;
constexpr uint32_t DQ_OFF_TMEM = DQ_OFF_BAR + DQ_NBARS * 8;
constexpr uint32_t DQ_OFF_ABORT = DQ_OFF_TMEM + 4;
constexpr uint32_t DQ_OFF_DPART = DQ_OFF_BAR + 256;                // 2 x 128 partial sums of D
constexpr uint32_t DQ_SMEM = DQ_OFF_DPART + 2 * BT * 4 + 1024;  // + slack for the 1024-byte alignment
static_assert(DQ_OFF_ABORT + 4 <= DQ_OFF_DPART, "control words overlap the D staging");
static_assert(DQ_SMEM <= 232448, "shared memory budget");
static_assert(DQ_KST >= 2, "the fp32 dQ tile is staged over the first two K stages");

__global__ void __launch_bounds__(DQ_THREADS, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmKc, const __grid_constant__ CUtensorMap tmVc,
                     const __grid_constant__ CUtensorMap tmdQ, const BwdTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t r0 = ptx::smem_addr(smem_raw);
    const uint32_t base = (r0 + 1023u) & ~1023u;
    uint8_t *const gb = smem_raw + (base - r0);
    const uint32_t sQ = base, sdO = base + TILE_BYTES;
    auto stage_k = [&](int x) { return base + DQ_OFF_K + static_cast<uint32_t>(x % DQ_KST) * TILE_BYTES; };
    auto stage_v = [&](int x) { return base + DQ_OFF_V + static_cast<uint32_t>(x % DQ_VST) * TILE_BYTES; };
    auto bar = [&](int k) { return base + DQ_OFF_BAR + 8u * k; };
    volatile int *const abort_flag = reinterpret_cast<volatile int *>(gb + DQ_OFF_ABORT);
    const uint64_t lim = p.wait_limit_ns;

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int BH = p.B * p.Hq, n_qt = (p.N + BT - 1) / BT;
    const int qt = n_qt - 1 - static_cast<int>(blockIdx.x / BH);  // heaviest tiles first
    const int bh = static_cast<int>(blockIdx.x % BH);
    const int kvz = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / (p.Hq / p.Hkv);
    const int i0 = qt * BT, i1 = min(i0 + BT - 1, p.N - 1);
    const int lo0 = win_of(p, i0);
    const int Tc = (lo_of(i1, p.w) / p.g + BT - 1) / BT;  // core tiles
    const int T = Tc + (i1 - lo0) / BT + 1;               // + band tiles
    auto tile_y = [&](int x) { return x < Tc ? x * BT : lo0 + (x - Tc) * BT; };

    if (t == 0) {
        // the first use of each descriptor would otherwise wait for its fetch
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmdO);
        ptx::prefetch_tmap(&tmKc);
        ptx::prefetch_tmap(&tmVc);
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        ptx::prefetch_tmap(&tmdQ);
        ptx::mbar_init(bar(QB_QD), 1);
        for (int st = 0; st < DQ_KST; ++st) {
            ptx::mbar_init(bar(QB_FULLK + st), 1);
            ptx::mbar_init(bar(QB_EMPTYK + st), 1);
        }
        for (int st = 0; st < DQ_VST; ++st) {
            ptx::mbar_init(bar(QB_FULLV + st), 1);
            ptx::mbar_init(bar(QB_EMPTYV + st), 1);
        }
        ptx::mbar_init(bar(QB_SFULL), 1);
        ptx::mbar_init(bar(QB_SFULL + 1), 1);
        ptx::mbar_init(bar(QB_DPFULL), 1);
        ptx::mbar_init(bar(QB_PFULL), 8);  // one arrive per element-wise warp
        ptx::mbar_init(bar(QB_DONE), 1);
        ptx::mbar_init(bar(QB_DRAIN), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(base + DQ_OFF_TMEM, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<uint32_t *>(gb + DQ_OFF_TMEM);
    constexpr uint32_t T_DP = 256, T_DQ = 384;  // TMEM columns; S(t) at 128 * (t & 1)

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0 && !p.skip_loads) {
            ptx::mbar_arrive_expect_tx(bar(QB_QD), 2 * TILE_BYTES);
            load_tile(&tmQ, bar(QB_QD), sQ, i0, bh);
            load_tile(&tmdO, bar(QB_QD), sdO, i0, bh);
            int nk = 0, nv = 0;  // tiles whose K / V copies have been issued
            for (int x = 0; x < T; ++x) {
                const bool core = x < Tc;
                // K(x) reuses the stage of K(x - 3) once dQ(x - 3) has read it
                if (x >= DQ_KST &&
                    !ptx::wait_bounded(bar(QB_EMPTYK + x % DQ_KST), (x / DQ_KST - 1) & 1, abort_flag, lim))
                    break;
                ptx::mbar_arrive_expect_tx(bar(QB_FULLK + x % DQ_KST), TILE_BYTES);
                load_tile(core ? (const void *)&tmKc : (const void *)&tmK, bar(QB_FULLK + x % DQ_KST), stage_k(x),
                          tile_y(x), kvz);
                nk = x + 1;
                // V(x) reuses the stage of V(x - 2) once dP(x - 2) has read it
                if (x >= DQ_VST &&
                    !ptx::wait_bounded(bar(QB_EMPTYV + x % DQ_VST), (x / DQ_VST - 1) & 1, abort_flag, lim))
                    break;
                ptx::mbar_arrive_expect_tx(bar(QB_FULLV + x % DQ_VST), TILE_BYTES);
                load_tile(core ? (const void *)&tmVc : (const void *)&tmV, bar(QB_FULLV + x % DQ_VST), stage_v(x),
                          tile_y(x), kvz);
                nv = x + 1;
            }
            if (*abort_flag) {
                // let the copies already issued land before the CTA exits
                volatile int never = 0;
                ptx::wait_bounded(bar(QB_QD), 0, &never, lim);
                for (int x = nk > DQ_KST ? nk - DQ_KST : 0; x < nk; ++x)
                    ptx::wait_bounded(bar(QB_FULLK + x % DQ_KST), (x / DQ_KST) & 1, &never, lim);
                for (int x = nv > DQ_VST ? nv - DQ_VST : 0; x < nv; ++x)
                    ptx::wait_bounded(bar(QB_FULLV + x % DQ_VST), (x / DQ_VST) & 1, &never, lim);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        auto wwait = [&](uint32_t bb, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, ptx::wait_bounded(bb, parity, abort_flag, lim));
        };
        const uint64_t dQd = ptx::smem_desc_sw128(sQ, 16, 1024), ddOd = ptx::smem_desc_sw128(sdO, 16, 1024);
        auto issue_s = [&](int x) {  // S(x) = Q K(x)^T
            ptx::tc_fence_after();
            ptx::mma_ss_k128_warp(tmem + 128u * (x & 1), dQd, ptx::smem_desc_sw128(stage_k(x), 16, 1024), IDESC_SS,
                                  0u);
            ptx::tc_commit_warp(bar(QB_SFULL + (x & 1)));
        };
        auto issue_dp = [&](int x) {  // dP(x) = dO V(x)^T
            ptx::tc_fence_after();
            ptx::mma_ss_k128_warp(tmem + T_DP, ddOd, ptx::smem_desc_sw128(stage_v(x), 16, 1024), IDESC_SS, 0u);
            ptx::tc_commit_warp(bar(QB_DPFULL));
            ptx::tc_commit_warp(bar(QB_EMPTYV + x % DQ_VST));
        };
        bool ok = wwait(bar(QB_QD), 0) && wwait(bar(QB_FULLK), 0);
        if (ok) issue_s(0);
        if (ok && (ok = wwait(bar(QB_FULLV), 0))) issue_dp(0);
        for (int tt = 0; ok && tt < T; ++tt) {
            const int x = tt + 1;
            if (x < T) {
                if (!(ok = wwait(bar(QB_FULLK + x % DQ_KST), (x / DQ_KST) & 1))) break;
                issue_s(x);
            }
            if (!(ok = wwait(bar(QB_PFULL), tt & 1))) break;
            ptx::tc_fence_after();
            ptx::mma_ts_k128_split_warp(tmem + T_DQ, tmem + 128u * (tt & 1),
                                        ptx::smem_desc_sw128(stage_k(tt), HALF_BYTES, 1024), IDESC_TS,
                                        tt > 0 ? 1u : 0u);  // dQ += dS K
            ptx::tc_commit_warp(bar(QB_EMPTYK + tt % DQ_KST));  // K(tt)'s stage is free once this has read it
            if (x < T) {
                if (!(ok = wwait(bar(QB_FULLV + x % DQ_VST), (x / DQ_VST) & 1))) break;
                issue_dp(x);
            }
        }
        ptx::tc_commit_warp(ok ? bar(QB_DONE) : bar(QB_DRAIN));
        if (!ok) {
            // whatever was issued must complete before tensor memory is freed
            volatile int never = 0;
            ptx::wait_bounded(bar(QB_DRAIN), 0, &never, lim);
        }
    } else {
        // ---------------------------------------------------------------- element-wise
        const int ch = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int h0 = ch * 64;  // this warp's 64 key columns of the tile
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        // this thread's row: D = dO . O (the pair's two halves of 64 columns each add their
        // partial sums through shared memory; the first stores D for the dK/dV kernel) and
        // the LSE in log2 units.  O comes from global memory (all eight 16-byte loads in
        // flight at once), dO from the swizzled tile already copied for the MMAs.
        const int i = i0 + row;
        const bool valid = i < p.N;
        const int64_t u = static_cast<int64_t>(bh) * p.N + i;
        uint4 o4[8];
        float lse2 = 0.f;
        if (valid) {
            const uint4 *src = reinterpret_cast<const uint4 *>(p.O + u * HD) + ch * 8;
#pragma unroll
            for (int c = 0; c < 8; ++c) o4[c] = src[c];
            lse2 = p.LSE[u] * LOG2E;
        }
        float Dpart = 0.f;
        if (__all_sync(0xffffffffu, ptx::wait_bounded(bar(QB_QD), 0, abort_flag, lim)) && valid) {
            const uint32_t rbase = sdO + ch * HALF_BYTES + row * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 d = ptx::ld_shared_v4(rbase + ((c ^ (row & 7)) << 4));
                const uint32_t aw[4] = {o4[c].x, o4[c].y, o4[c].z, o4[c].w}, bw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) Dpart += bf(aw[k], 0) * bf(bw[k], 0) + bf(aw[k], 1) * bf(bw[k], 1);
            }
        }
        float *const dpart = reinterpret_cast<float *>(gb + DQ_OFF_DPART);
        dpart[ch * BT + row] = Dpart;
        ptx::named_bar_sync(1, 256);  // the eight element-wise warps, every one of them, always
        const float Di = dpart[row] + dpart[BT + row];
        if (valid && ch == 0) p.Dbuf[u] = Di;
        const int lo_i = win_of(p, i), nc_i = lo_of(i, p.w) / p.g;
        const float c1 = p.tau * LOG2E;
        bool ok = true;
        for (int tt = 0; tt < T; ++tt) {
            if (!__all_sync(0xffffffffu, ptx::wait_bounded(bar(QB_SFULL + (tt & 1)), (tt >> 1) & 1, abort_flag, lim))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t sS = tmem + lane_addr + 128u * (tt & 1) + h0;
            uint32_t pa[32], pb[32];
            ptx::tmem_ld32(sS, pa);
            ptx::tmem_ld32(sS + 32, pb);
            // the row's visible key columns of this tile
            const int y0 = tile_y(tt);
            int c_lo = 0, c_hi = BT - 1;
            if (tt < Tc) {
                c_hi = min(nc_i - y0, BT) - 1;
            } else {
                c_lo = max(lo_i - y0, 0);
                c_hi = min(i - y0, BT - 1);
            }
            if (!valid) c_hi = -1;
            ptx::tmem_wait_ld(pa);
            ptx::reg_touch(pb);
            // P = 2^(S tau log2e - LSE), zero off the visible columns
            if (__all_sync(0xffffffffu, c_lo <= h0 && c_hi >= h0 + 63)) {
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    pa[k] = __float_as_uint(ptx::ex2(fmaf(__uint_as_float(pa[k]), c1, -lse2)));
                    pb[k] = __float_as_uint(ptx::ex2(fmaf(__uint_as_float(pb[k]), c1, -lse2)));
                }
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int ca = h0 + k, cb = h0 + 32 + k;
                    pa[k] = (ca >= c_lo && ca <= c_hi)
                                ? __float_as_uint(ptx::ex2(fmaf(__uint_as_float(pa[k]), c1, -lse2))) : 0u;
                    pb[k] = (cb >= c_lo && cb <= c_hi)
                                ? __float_as_uint(ptx::ex2(fmaf(__uint_as_float(pb[k]), c1, -lse2))) : 0u;
                }
            }
            if (!__all_sync(0xffffffffu, ptx::wait_bounded(bar(QB_DPFULL), tt & 1, abort_flag, lim))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            // dS = P (dP - D), bf16 pairs written over the S columns [h0, h0 + 32), which
            // this warp has already read
            uint32_t dp[32], pk[16];
            ptx::tmem_ld32(tmem + lane_addr + T_DP + h0, dp);
            ptx::tmem_wait_ld(dp);
#pragma unroll
            for (int k = 0; k < 16; ++k)
                pk[k] = ptx::pack_bf16x2(__uint_as_float(pa[2 * k]) * (__uint_as_float(dp[2 * k]) - Di),
                                         __uint_as_float(pa[2 * k + 1]) * (__uint_as_float(dp[2 * k + 1]) - Di));
            ptx::tmem_st16(sS, pk);
            ptx::tmem_ld32(tmem + lane_addr + T_DP + h0 + 32, dp);
            ptx::tmem_wait_ld(dp);
#pragma unroll
            for (int k = 0; k < 16; ++k)
                pk[k] = ptx::pack_bf16x2(__uint_as_float(pb[2 * k]) * (__uint_as_float(dp[2 * k]) - Di),
                                         __uint_as_float(pb[2 * k + 1]) * (__uint_as_float(dp[2 * k + 1]) - Di));
            ptx::tmem_st16(sS + 16, pk);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(QB_PFULL));
        }
        if (ok && !__all_sync(0xffffffffu, ptx::wait_bounded(bar(QB_DONE), 0, abort_flag, lim))) ok = false;
        if (ok) {
            // dQ * tau through shared memory (the first two K stages, idle now) to a tiled store
            ptx::tc_fence_after();
            stage_f32_rows(tmem + lane_addr, T_DQ, ch, row, p.tau, false, base + DQ_OFF_K);
            ptx::fence_proxy_async_smem();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (t == 0 && p.status != nullptr) atomicCAS(p.status, 0, STATUS_TIMEOUT);
    } else if (t == 0) {
        store_tile_f32(&tmdQ, base + DQ_OFF_K, i0, bh);
        ptx::bulk_wait_read();
    }
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- dK, dV
// One 128-key tile (raw tokens or cores) of one (b, kv) per CTA, over the query tiles of
// the r query heads that see it.  Warp-specialised, 320 threads:
//   warp 0      producer: K and V once; per query tile x, Q(x) into one of three stages
//               and dO(x) into one of two (TMA; Q lives longer: S^T(x) and dK(x) read it);
//   warp 1      MMA issuer (whole warp, one elected lane), per query tile x:
//                 dV += P^T dO(x)            once P^T(x) is written,
//                 S^T(x+1) = K Q(x+1)^T      (the S^T buffer is free again),
//                 dK += dS^T Q(x)            once dS^T(x) is written,
//                 dP^T(x+1) = V dO(x+1)^T    (the dP^T buffer is free again);
//   warps 2..9  element-wise, in two phases per tile: P^T = 2^(S^T tau log2e - LSE) as
//               bf16 over S^T (kept in fp32 registers), then dS^T = P^T (dP^T - D) as bf16
//               over dP^T.  Warps w and w + 4 share TMEM lanes 32*(w%4)..+31 (the keys)
//               and split each query tile's 128 columns, 64 each.  They also keep the
//               tile's LSE and D in one shared-memory slot: each of the 256 threads loads
//               one value of the next tile early and writes it between two named barriers.
// The hand-offs are mbarriers.  TMEM: S^T | dP^T | dK | dV; the MMAs of one thread
// complete in issue order, so S^T(x+1) and dP^T(x+1), issued after dV(x) and dK(x),
// never overwrite what those read.
constexpr int DKV_THREADS = 320;
constexpr int BWD_CORE_CHUNK = 64;  // query tiles per core-tile item
constexpr int DKV_QST = 3, DKV_OST = 2;
constexpr uint32_t DKV_OFF_Q = 2 * TILE_BYTES;  // after K, V
constexpr uint32_t DKV_OFF_O = DKV_OFF_Q + DKV_QST * TILE_BYTES;
constexpr uint32_t DKV_OFF_SLOT = DKV_OFF_O + DKV_OST * TILE_BYTES;  // LSE (log2 units) 128 | D 128
constexpr uint32_t DKV_OFF_BAR = DKV_OFF_SLOT + 2 * BT * 4;
constexpr int DB_KV = 0, DB_FULLQ = 1, DB_EMPTYQ = 4, DB_FULLO = 7, DB_EMPTYO = 9, DB_SFULL = 11, DB_DPFULL = 12,
              DB_PFULL = 13, DB_DSFULL = 14, DB_DONE = 15, DB_DRAIN = 16;
constexpr int DKV_NBARS = 17;
constexpr uint32_t DKV_OFF_TMEM = DKV_OFF_BAR + DKV_NBARS * 8;
constexpr uint32_t DKV_OFF_ABORT = DKV_OFF_TMEM + 4;
constexpr uint32_t DKV_SMEM = DKV_OFF_ABORT + 4 + 1024;  // + slack for the 1024-byte alignment
static_assert(DKV_SMEM <= 232448, "shared memory budget");
static_assert(DKV_QST + DKV_OST >= 4, "the fp32 dK and dV tiles are staged over the Q and dO stages");

__global__ void __launch_bounds__(DKV_THREADS, 1)
    bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                      const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmKc, const __grid_constant__ CUtensorMap tmVc,
                      const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                      const __grid_constant__ CUtensorMap tmdKc, const __grid_constant__ CUtensorMap tmdVc,
                      const BwdTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t r0 = ptx::smem_addr(smem_raw);
    const uint32_t base = (r0 + 1023u) & ~1023u;
    uint8_t *const gb = smem_raw + (base - r0);
    const uint32_t sK = base, sV = base + TILE_BYTES;
    auto stage_q = [&](int x) { return base + DKV_OFF_Q + static_cast<uint32_t>(x % DKV_QST) * TILE_BYTES; };
    auto stage_o = [&](int x) { return base + DKV_OFF_O + static_cast<uint32_t>(x % DKV_OST) * TILE_BYTES; };
    auto bar = [&](int k) { return base + DKV_OFF_BAR + 8u * k; };
    volatile int *const abort_flag = reinterpret_cast<volatile int *>(gb + DKV_OFF_ABORT);
    const uint64_t lim = p.wait_limit_ns;

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int BK = p.B * p.Hkv;
    const int n_core_t = (p.G + BT - 1) / BT;
    const int n_qt = (p.N + BT - 1) / BT;
    // core tiles first (they are seen by the most query rows), then raw-token tiles.  With
    // core_chunk > 0 (core tiles only) an item is one core tile over one chunk of query
    // tiles, [c * core_chunk, (c + 1) * core_chunk); items run top chunk first, each chunk
    // head by head, a head's core tiles side by side, so the CTAs that run together stream
    // the same Q/dO tiles.
    int idx, bk, chunk = -1;
    if (p.core_chunk > 0) {
        const int per_chunk = BK * n_core_t;
        const int n_chunks = (n_qt + p.core_chunk - 1) / p.core_chunk;
        chunk = n_chunks - 1 - static_cast<int>(blockIdx.x / per_chunk);
        const int rem = static_cast<int>(blockIdx.x % per_chunk);
        bk = rem / n_core_t;
        idx = rem % n_core_t;
    } else {
        idx = p.tile0 + static_cast<int>(blockIdx.x / BK);
        bk = static_cast<int>(blockIdx.x % BK);
    }
    const bool core = idx < n_core_t;
    const int y0 = core ? idx * BT : (idx - n_core_t) * BT;
    const int n_keys = core ? p.G : p.N;
    const int r = p.Hq / p.Hkv;
    const int b = bk / p.Hkv, kv = bk % p.Hkv;
    // the query rows that see at least one key of the tile
    int r_lo, r_hi;
    if (core) {
        r_lo = (y0 + 1) * p.g + p.w - 1;  // core j is seen from row (j+1)g + w - 1 on
        r_hi = p.N - 1;
    } else {
        const int m_last = min(y0 + BT - 1, p.N - 1);
        const int64_t last = p.window_mode ? static_cast<int64_t>(m_last / p.g + 1) * p.g + p.w - 2
                                           : static_cast<int64_t>(m_last) + p.w - 1;
        r_lo = y0;
        r_hi = static_cast<int>(last < p.N - 1 ? last : p.N - 1);
    }
    int qt_hi = r_hi / BT, qt_lo = r_lo / BT;
    if (chunk >= 0) {
        // this item's part of the range; an item with nothing to do leaves before any setup
        qt_hi = min(qt_hi, (chunk + 1) * p.core_chunk - 1);
        qt_lo = max(qt_lo, chunk * p.core_chunk);
        if (r_lo > r_hi || qt_lo > qt_hi) return;
    }
    const int nq = r_lo <= r_hi ? qt_hi - qt_lo + 1 : 0;
    // (query tile, head) pairs from the last query tile down, heads fastest: every CTA of a
    // KV head (their ranges all end at the last tile, or overlap their neighbours') then
    // reads the same Q/dO tiles at about the same time, so they come from L2
    const int n_it = nq * r;
    auto bh_of = [&](int it) { return b * p.Hq + kv * r + it % r; };
    auto i0_of = [&](int it) { return (qt_hi - it / r) * BT; };

    if (t == 0) {
        // the first use of each descriptor would otherwise wait for its fetch
        ptx::prefetch_tmap(core ? (const void *)&tmKc : (const void *)&tmK);
        ptx::prefetch_tmap(core ? (const void *)&tmVc : (const void *)&tmV);
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmdO);
        ptx::prefetch_tmap(core ? (const void *)&tmdKc : (const void *)&tmdK);
        ptx::prefetch_tmap(core ? (const void *)&tmdVc : (const void *)&tmdV);
        ptx::mbar_init(bar(DB_KV), 1);
        for (int st = 0; st < DKV_QST; ++st) {
            ptx::mbar_init(bar(DB_FULLQ + st), 1);
            ptx::mbar_init(bar(DB_EMPTYQ + st), 1);
        }
        for (int st = 0; st < DKV_OST; ++st) {
            ptx::mbar_init(bar(DB_FULLO + st), 1);
            ptx::mbar_init(bar(DB_EMPTYO + st), 1);
        }
        ptx::mbar_init(bar(DB_SFULL), 1);
        ptx::mbar_init(bar(DB_DPFULL), 1);
        ptx::mbar_init(bar(DB_PFULL), 8);   // one arrive per element-wise warp
        ptx::mbar_init(bar(DB_DSFULL), 8);  // one arrive per element-wise warp
        ptx::mbar_init(bar(DB_DONE), 1);
        ptx::mbar_init(bar(DB_DRAIN), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(base + DKV_OFF_TMEM, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<uint32_t *>(gb + DKV_OFF_TMEM);
    constexpr uint32_t T_DP = 128, T_DK = 256, T_DV = 384;  // TMEM columns; S^T at 0

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0 && !p.skip_loads && n_it > 0) {
            ptx::mbar_arrive_expect_tx(bar(DB_KV), 2 * TILE_BYTES);
            load_tile(core ? (const void *)&tmKc : (const void *)&tmK, bar(DB_KV), sK, y0, bk);
            load_tile(core ? (const void *)&tmVc : (const void *)&tmV, bar(DB_KV), sV, y0, bk);
            int nqd = 0, nod = 0;  // tiles whose Q / dO copies have been issued
            for (int x = 0; x < n_it; ++x) {
                const int bh = bh_of(x), i0 = i0_of(x);
                // Q(x) reuses the stage of Q(x - 3) once dK(x - 3) has read it
                if (x >= DKV_QST &&
                    !ptx::wait_bounded(bar(DB_EMPTYQ + x % DKV_QST), (x / DKV_QST - 1) & 1, abort_flag, lim))
                    break;
                ptx::mbar_arrive_expect_tx(bar(DB_FULLQ + x % DKV_QST), TILE_BYTES);
                load_tile(&tmQ, bar(DB_FULLQ + x % DKV_QST), stage_q(x), i0, bh);
                nqd = x + 1;
                // dO(x) reuses the stage of dO(x - 2) once dV(x - 2) has read it
                if (x >= DKV_OST &&
                    !ptx::wait_bounded(bar(DB_EMPTYO + x % DKV_OST), (x / DKV_OST - 1) & 1, abort_flag, lim))
                    break;
                ptx::mbar_arrive_expect_tx(bar(DB_FULLO + x % DKV_OST), TILE_BYTES);
                load_tile(&tmdO, bar(DB_FULLO + x % DKV_OST), stage_o(x), i0, bh);
                nod = x + 1;
            }
            if (*abort_flag) {
                // let the copies already issued land before the CTA exits
                volatile int never = 0;
                ptx::wait_bounded(bar(DB_KV), 0, &never, lim);
                for (int x = nqd > DKV_QST ? nqd - DKV_QST : 0; x < nqd; ++x)
                    ptx::wait_bounded(bar(DB_FULLQ + x % DKV_QST), (x / DKV_QST) & 1, &never, lim);
                for (int x = nod > DKV_OST ? nod - DKV_OST : 0; x < nod; ++x)
                    ptx::wait_bounded(bar(DB_FULLO + x % DKV_OST), (x / DKV_OST) & 1, &never, lim);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        auto wwait = [&](uint32_t bb, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, ptx::wait_bounded(bb, parity, abort_flag, lim));
        };
        const uint64_t dKk = ptx::smem_desc_sw128(sK, 16, 1024), dVk = ptx::smem_desc_sw128(sV, 16, 1024);
        auto issue_s = [&](int x) {  // S^T(x) = K Q(x)^T
            ptx::tc_fence_after();
            ptx::mma_ss_k128_warp(tmem + 0, dKk, ptx::smem_desc_sw128(stage_q(x), 16, 1024), IDESC_SS, 0u);
            ptx::tc_commit_warp(bar(DB_SFULL));
        };
        auto issue_dp = [&](int x) {  // dP^T(x) = V dO(x)^T
            ptx::tc_fence_after();
            ptx::mma_ss_k128_warp(tmem + T_DP, dVk, ptx::smem_desc_sw128(stage_o(x), 16, 1024), IDESC_SS, 0u);
            ptx::tc_commit_warp(bar(DB_DPFULL));
        };
        bool ok = n_it == 0 || (wwait(bar(DB_KV), 0) && wwait(bar(DB_FULLQ), 0));
        if (ok && n_it > 0) issue_s(0);
        if (ok && n_it > 0 && (ok = wwait(bar(DB_FULLO), 0))) issue_dp(0);
        for (int it = 0; ok && it < n_it; ++it) {
            const int x = it + 1;
            const uint32_t acc = it > 0 ? 1u : 0u;
            if (!(ok = wwait(bar(DB_PFULL), it & 1))) break;
            ptx::tc_fence_after();
            ptx::mma_ts_k128_split_warp(tmem + T_DV, tmem + 0, ptx::smem_desc_sw128(stage_o(it), HALF_BYTES, 1024),
                                        IDESC_TS, acc);  // dV += P^T dO
            ptx::tc_commit_warp(bar(DB_EMPTYO + it % DKV_OST));
            if (x < n_it) {
                if (!(ok = wwait(bar(DB_FULLQ + x % DKV_QST), (x / DKV_QST) & 1))) break;
                issue_s(x);
            }
            if (!(ok = wwait(bar(DB_DSFULL), it & 1))) break;
            ptx::tc_fence_after();
            ptx::mma_ts_k128_split_warp(tmem + T_DK, tmem + T_DP,
                                        ptx::smem_desc_sw128(stage_q(it), HALF_BYTES, 1024), IDESC_TS,
                                        acc);  // dK += dS^T Q
            ptx::tc_commit_warp(bar(DB_EMPTYQ + it % DKV_QST));
            if (x < n_it) {
                if (!(ok = wwait(bar(DB_FULLO + x % DKV_OST), (x / DKV_OST) & 1))) break;
                issue_dp(x);
            }
        }
        ptx::tc_commit_warp(ok ? bar(DB_DONE) : bar(DB_DRAIN));
        if (!ok) {
            // whatever was issued must complete before tensor memory is freed
            volatile int never = 0;
            ptx::wait_bounded(bar(DB_DRAIN), 0, &never, lim);
        }
    } else {
        // ---------------------------------------------------------------- element-wise
        const int ch = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int h0 = ch * 64;  // this warp's 64 query columns of the tile
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const int m = y0 + row;  // this thread's key (core index or token)
        const float c1 = p.tau * LOG2E;
        int64_t key_last = 0;
        if (!core) key_last = p.window_mode ? static_cast<int64_t>(m / p.g + 1) * p.g + p.w - 2 : static_cast<int64_t>(m) + p.w - 1;
        // this thread's value of the LSE/D slot: LSE (log2 units) of query e, or D of query e - 128
        const int e = (warp - 2) * 32 + lane;
        auto slot_value = [&](int x) -> float {
            const int iq = i0_of(x) + (e & (BT - 1));
            if (iq >= p.N) return 0.f;
            const int64_t off = static_cast<int64_t>(bh_of(x)) * p.N + iq;
            return e < BT ? p.LSE[off] * LOG2E : p.Dbuf[off];
        };
        float *const slot_f = reinterpret_cast<float *>(gb + DKV_OFF_SLOT);
        const float4 *const slot4 = reinterpret_cast<const float4 *>(slot_f);
        if (n_it > 0) slot_f[e] = slot_value(0);
        ptx::named_bar_sync(1, 256);
        bool ok = true;
        // the pooling backward's terms for this key's row (raw tiles, folded pooling backward)
        const bool fuse = !core && p.pool_fuse != 0;
        const int mm = m < p.N ? m : p.N - 1;  // rows past N only take part in collective loads
        const int64_t uj = static_cast<int64_t>(bk) * p.G + mm / p.g;
        float am = 0.f, cm = 0.f;
        if (fuse) {
            const int64_t um = static_cast<int64_t>(bk) * p.N + mm;
            am = p.pool_fuse == 1 ? 1.f / p.g : p.pool_a[um];
            cm = p.pool_fuse == 1 ? 0.f : p.pool_cds[um];
        }
        // Every element-wise thread runs every iteration and both named barriers of it, so
        // that a time-out (which skips the work) cannot leave a barrier short of threads.
        for (int it = 0; it < n_it; ++it) {
            const float v_next = it + 1 < n_it ? slot_value(it + 1) : 0.f;
            if (fuse && it == n_it - 1) {
                // bring this row's half of dKc_j, dVc_j (and qsum_j) into L1 for the epilogue
#pragma unroll
                for (int l = 0; l < 2; ++l) {
                    ptx::prefetch_l1(p.pool_dkc + uj * HD + h0 + 32 * l);
                    ptx::prefetch_l1(p.pool_dvc + uj * HD + h0 + 32 * l);
                    if (p.pool_fuse == 2) ptx::prefetch_l1(p.pool_qs + uj * HD + h0 + 32 * l);
                }
            }
            if (ok) ok = __all_sync(0xffffffffu, ptx::wait_bounded(bar(DB_SFULL), it & 1, abort_flag, lim));
            uint32_t pa[32], pb[32];
            if (ok) {
                ptx::tc_fence_after();
                const uint32_t sS = tmem + lane_addr + h0;
                ptx::tmem_ld32(sS, pa);
                ptx::tmem_ld32(sS + 32, pb);
                // this key's visible query columns [q_lo, q_hi] of the tile
                const int i0 = i0_of(it);
                int q_lo, q_hi;
                if (m >= n_keys) {
                    q_lo = 0;
                    q_hi = -1;
                } else if (core) {
                    q_lo = max((m + 1) * p.g + p.w - 1 - i0, 0);
                    q_hi = min(p.N - 1 - i0, BT - 1);
                } else {
                    const int last_i = static_cast<int>(key_last < p.N - 1 ? key_last : p.N - 1);
                    q_lo = max(m - i0, 0);
                    q_hi = min(last_i - i0, BT - 1);
                }
                ptx::tmem_wait_ld(pa);
                ptx::reg_touch(pb);
                // P^T = 2^(S^T tau log2e - LSE), zero off the visible columns (the LSE of four
                // columns per shared-memory load, the same address across the warp)
                if (__all_sync(0xffffffffu, q_lo <= h0 && q_hi >= h0 + 63)) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 la = slot4[h0 / 4 + q], lb = slot4[h0 / 4 + 8 + q];
                        const float lsa[4] = {la.x, la.y, la.z, la.w}, lsb[4] = {lb.x, lb.y, lb.z, lb.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            pa[4 * q + k] = __float_as_uint(ptx::ex2(fmaf(__uint_as_float(pa[4 * q + k]), c1, -lsa[k])));
                            pb[4 * q + k] = __float_as_uint(ptx::ex2(fmaf(__uint_as_float(pb[4 * q + k]), c1, -lsb[k])));
                        }
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 la = slot4[h0 / 4 + q], lb = slot4[h0 / 4 + 8 + q];
                        const float lsa[4] = {la.x, la.y, la.z, la.w}, lsb[4] = {lb.x, lb.y, lb.z, lb.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int ka = 4 * q + k, ca = h0 + ka, cb = h0 + 32 + ka;
                            const float xa = ptx::ex2(fmaf(__uint_as_float(pa[ka]), c1, -lsa[k]));
                            const float xb = ptx::ex2(fmaf(__uint_as_float(pb[ka]), c1, -lsb[k]));
                            pa[ka] = __float_as_uint(ca >= q_lo && ca <= q_hi ? xa : 0.f);
                            pb[ka] = __float_as_uint(cb >= q_lo && cb <= q_hi ? xb : 0.f);
                        }
                    }
                }
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) pk[k] = ptx::pack_bf16x2(__uint_as_float(pa[2 * k]), __uint_as_float(pa[2 * k + 1]));
                ptx::tmem_st16(sS, pk);  // P^T over S^T columns [h0, h0 + 16), already read
#pragma unroll
                for (int k = 0; k < 16; ++k) pk[k] = ptx::pack_bf16x2(__uint_as_float(pb[2 * k]), __uint_as_float(pb[2 * k + 1]));
                ptx::tmem_st16(sS + 16, pk);
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(DB_PFULL));
            }
            if (ok) ok = __all_sync(0xffffffffu, ptx::wait_bounded(bar(DB_DPFULL), it & 1, abort_flag, lim));
            if (ok) {
                ptx::tc_fence_after();
                // dS^T = P^T (dP^T - D), bf16 pairs over dP^T columns [h0, h0 + 32), which this
                // warp has already read
                const uint32_t sD = tmem + lane_addr + T_DP + h0;
                uint32_t dp[32], dd[16];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    ptx::tmem_ld32(sD + 32 * j, dp);
                    ptx::tmem_wait_ld(dp);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 dv = slot4[(BT + h0) / 4 + 8 * j + q];
                        const float Dv[4] = {dv.x, dv.y, dv.z, dv.w};
                        const uint32_t *pp = j ? pb : pa;
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const int c = 4 * q + 2 * k;
                            dd[2 * q + k] = ptx::pack_bf16x2(
                                __uint_as_float(pp[c]) * (__uint_as_float(dp[c]) - Dv[2 * k]),
                                __uint_as_float(pp[c + 1]) * (__uint_as_float(dp[c + 1]) - Dv[2 * k + 1]));
                        }
                    }
                    ptx::tmem_st16(sD + 16 * j, dd);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(DB_DSFULL));
            }
            // the slot moves on to the next tile once every warp is done with this one
            ptx::named_bar_sync(1, 256);
            slot_f[e] = v_next;
            ptx::named_bar_sync(1, 256);
        }
        if (ok && !__all_sync(0xffffffffu, ptx::wait_bounded(bar(DB_DONE), 0, abort_flag, lim))) ok = false;
        if (ok) {
            // dK * tau and dV through shared memory (the Q and dO stages, idle now) to tiled
            // stores; a tile no query row sees stores zeros
            ptx::tc_fence_after();
            if (fuse) {
                // + the pooling backward: a_m dKc_j + (tau/r) ds_m qsum_j and a_m dVc_j, j = m / g
                // (the store drops rows past N)
                const float *qs = p.pool_fuse == 1 ? nullptr : p.pool_qs + uj * HD;
                stage_f32_rows_plus(tmem + lane_addr, T_DK, ch, row, p.tau, n_it == 0, base + DKV_OFF_Q,
                                    p.pool_dkc + uj * HD, am, qs, cm);
                stage_f32_rows_plus(tmem + lane_addr, T_DV, ch, row, 1.f, n_it == 0,
                                    base + DKV_OFF_Q + 2 * TILE_BYTES, p.pool_dvc + uj * HD, am, nullptr, 0.f);
            } else {
                stage_f32_rows(tmem + lane_addr, T_DK, ch, row, p.tau, n_it == 0, base + DKV_OFF_Q);
                stage_f32_rows(tmem + lane_addr, T_DV, ch, row, 1.f, n_it == 0, base + DKV_OFF_Q + 2 * TILE_BYTES);
            }
            ptx::fence_proxy_async_smem();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (t == 0 && p.status != nullptr) atomicCAS(p.status, 0, STATUS_TIMEOUT);
    } else if (t == 0) {
        // a chunked core item adds its share to dKc/dVc (zeroed before the launch)
        store_tile_f32(core ? &tmdKc : &tmdK, base + DKV_OFF_Q, y0, bk, chunk >= 0);
        store_tile_f32(core ? &tmdVc : &tmdV, base + DKV_OFF_Q + 2 * TILE_BYTES, y0, bk, chunk >= 0);
        ptx::bulk_wait_read();
    }
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

struct Attr {
    bool done = false;
    cudaError_t err = cudaSuccess;
};

}  // namespace

cudaError_t launch_attn_bwd_tc(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                               const void *O, const float *LSE, const void *dO, float *dQ, float *dK, float *dV,
                               float *Dbuf, float *dKc, float *dVc, const Shape &s, int32_t *status, int part,
                               const BwdPoolFuse &pf, cudaStream_t stream) {
    EncodeTiledFn enc = get_encoder();
    if (enc == nullptr) return cudaErrorNotSupported;
    static std::mutex mu;
    static Attr attr[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        Attr &a = attr[dev & 63];
        if (!a.done) {
            a.err = cudaFuncSetAttribute(bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM);
            if (a.err == cudaSuccess)
                a.err = cudaFuncSetAttribute(bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             DKV_SMEM);
            a.done = true;
        }
        if (a.err != cudaSuccess) return a.err;
    }
    const uint64_t G = static_cast<uint64_t>(s.N / s.g);
    const uint64_t qh = static_cast<uint64_t>(s.B) * s.Hq, kh = static_cast<uint64_t>(s.B) * s.Hkv;
    CUtensorMap mQ, mdO, mK, mV, mKc, mVc, mdQ, mdK, mdV, mdKc, mdVc;
    if (!encode_3d_bf16_d128(enc, &mQ, Q, s.N, qh) || !encode_3d_bf16_d128(enc, &mdO, dO, s.N, qh) ||
        !encode_3d_bf16_d128(enc, &mK, K, s.N, kh) || !encode_3d_bf16_d128(enc, &mV, V, s.N, kh) ||
        !encode_3d_bf16_d128(enc, &mKc, Kc, G, kh) || !encode_3d_bf16_d128(enc, &mVc, Vc, G, kh) ||
        !encode_3d_f32_d128(enc, &mdQ, dQ, s.N, qh) || !encode_3d_f32_d128(enc, &mdK, dK, s.N, kh) ||
        !encode_3d_f32_d128(enc, &mdV, dV, s.N, kh) || !encode_3d_f32_d128(enc, &mdKc, dKc, G, kh) ||
        !encode_3d_f32_d128(enc, &mdVc, dVc, G, kh))
        return cudaErrorInvalidValue;
    BwdTcParams p;
    p.B = s.B;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.N = s.N;
    p.g = s.g;
    p.w = s.w;
    p.window_mode = s.window_mode;
    p.G = static_cast<int>(G);
    p.tau = s.scale;
    p.LSE = LSE;
    p.O = static_cast<const __nv_bfloat16 *>(O);
    p.dO = static_cast<const __nv_bfloat16 *>(dO);
    p.Dbuf = Dbuf;
    p.tile0 = 0;
    p.core_chunk = 0;
    p.pool_fuse = 0;
    p.pool_a = p.pool_cds = p.pool_qs = nullptr;
    p.pool_dkc = dKc;
    p.pool_dvc = dVc;
    p.status = status;
    p.wait_limit_ns = g_wait_limit_ns;
    p.skip_loads = g_skip_q_load;
    if (part != 2) {
        const unsigned n_qt = static_cast<unsigned>((s.N + BT - 1) / BT);
        bwd_dq_tc_kernel<<<n_qt * static_cast<unsigned>(qh), DQ_THREADS, DQ_SMEM, stream>>>(mQ, mdO, mK, mV, mKc,
                                                                                            mVc, mdQ, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const unsigned n_ct = static_cast<unsigned>((G + BT - 1) / BT), n_rt = static_cast<unsigned>((s.N + BT - 1) / BT);
    unsigned n_kt = n_ct + n_rt;
    unsigned grid = 0;
    if (part == 1) {
        // core tiles in chunks of query tiles, added into zeroed dKc/dVc
        const int n_qt = static_cast<int>((s.N + BT - 1) / BT);
        p.core_chunk = BWD_CORE_CHUNK;
        const unsigned n_chunks = static_cast<unsigned>((n_qt + p.core_chunk - 1) / p.core_chunk);
        const size_t core_bytes = static_cast<size_t>(G) * static_cast<size_t>(kh) * 128 * sizeof(float);
        if (n_ct > 0) {
            if ((e = cudaMemsetAsync(dKc, 0, core_bytes, stream)) != cudaSuccess) return e;
            if ((e = cudaMemsetAsync(dVc, 0, core_bytes, stream)) != cudaSuccess) return e;
        }
        n_kt = n_ct;
        grid = n_chunks * n_ct * static_cast<unsigned>(kh);
    } else if (part == 2) {
        p.tile0 = static_cast<int>(n_ct);
        n_kt = n_rt;
        p.pool_fuse = pf.mode;
        p.pool_a = pf.a;
        p.pool_cds = pf.cds;
        p.pool_qs = pf.qs;
    }
    if (n_kt == 0) return cudaSuccess;
    if (grid == 0) grid = n_kt * static_cast<unsigned>(kh);
    bwd_dkv_tc_kernel<<<grid, DKV_THREADS, DKV_SMEM, stream>>>(
        mQ, mdO, mK, mV, mKc, mVc, mdK, mdV, mdKc, mdVc, p);
    return cudaGetLastError();
}

}  // namespace cca
