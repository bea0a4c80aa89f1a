// Fused core/local attention, bf16, d = 128, on the sm_103a tensor cores
// ("Core Context Aware Transformers for Long Context Language Modeling",
// Method section, fusion equation
//     Att_i = softmax(Q_i [K^G_{T_i}; K^L_{U_i}]^T / sqrt(d)) [V^G_{T_i}; V^L_{U_i}]).
//
// Persistent kernel, one CTA per SM.  A work item is 256 query rows of one
// (batch, query head), split in two 128-row halves A and B that share every
// K/V tile the CTA loads.  The keys form one sequence of 128-key tiles: the
// core tokens Kc/Vc [0, n_core(last row)), then the raw tokens K/V of the band
// [lo(first row), last row].  Each half visits only the tiles it can see (a
// half skips a tile that lies wholly outside its own band or staircase), and
// keeps one online-softmax state (row max m, row sum l, O in tensor memory)
// over its whole sequence, so core and local segments share one normalisation.
// Only tiles that straddle a visibility edge are masked:
//   core tile:  column c (core y0+c) is visible to row i iff y0 + c < lo(i)/g;
//   local tile: column c (token y0+c) is visible to row i iff lo(i) <= y0+c <= i.
//
// Roles (320 threads):
//   warp 0       TMA producer: the two Q tiles of an item, then K(t), V(t) for
//                every tile t into a ring of NS 32 KB slots (128-byte swizzle);
//   warp 1       MMA issuer (the whole warp, one elected lane issues): S_h = Q_h K^T
//                (both operands in shared memory) and O_h += P_h V (P_h in tensor
//                memory, V MN-major);
//   warps 2..5   softmax + epilogue of half A, warps 6..9 the same for half B.
//                A warp may only touch TMEM lanes 32*(warp%4) .. +31, so each
//                group of four consecutive warps covers the 128 lanes once;
//                thread t of the group owns TMEM lane / query row t.
// Tensor memory (512 columns): S_A | S_B | O_A | O_B.  P_h (bf16) overwrites
// the first 64 columns of S_h after the softmax has read S_h.  The issuer
// writes S_h for the next tile only after the PV that read P_h (issue order),
// and a completed S_h therefore also means that every earlier PV of the half
// has completed, which is what lets the softmax rescale O_h in place.
// Work items are ordered heaviest first and dealt round-robin to the CTAs.  A launch may
// cover only the rows [q_off, q_off + n_q) of the sequence (a shard): items then start at
// q_off, rows keep their sequence indices for visibility, and Q/O/LSE rows and K/V tile
// coordinates are taken relative to q_off and kv_off.
// Every mbarrier wait is bounded in time; on a time-out the CTA stops, drains
// what it has in flight, frees its tensor memory and reports CCA_ERR_TIMEOUT.
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
namespace {

constexpr int BM = 128;                       // query rows per half
constexpr int BN = 128;                       // keys per tile
constexpr int HD = 128;                       // head dimension
constexpr int NS = 5;                         // ring slots
constexpr uint32_t TILE_BYTES = BN * HD * 2;  // one bf16 128x128 tile
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;
constexpr int NUM_THREADS = 320;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;    // S_h at h * 128
constexpr uint32_t TM_O = 256;  // O_h at 256 + h * 128
constexpr float LAZY_RESCALE_LOG2 = 16.0f;  // keep a stale max while it is within 2^16

constexpr uint32_t IDESC_QK = ptx::idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(BM, HD, 0, 1);  // P (TMEM), V MN-major

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0;  // Q_A, Q_B
constexpr uint32_t OFF_RING = 2 * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_RING + NS * TILE_BYTES;
constexpr int B_QFULL = 0;
constexpr int B_QFREE = 1;
constexpr int B_FULL = 2;               // NS
constexpr int B_EMPTY = B_FULL + NS;    // NS
constexpr int B_SFULL = B_EMPTY + NS;   // 2 (per half)
constexpr int B_PFULL = B_SFULL + 2;    // 2
constexpr int B_PVDONE = B_PFULL + 2;   // 2
constexpr int B_OFREE = B_PVDONE + 2;   // 2
constexpr int B_DRAIN = B_OFREE + 2;
constexpr int NUM_BARS = B_DRAIN + 1;
constexpr uint32_t OFF_TMEMPTR = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEMPTR + 4;
constexpr uint32_t SMEM_USED = OFF_ABORT + 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for manual alignment
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct Params {
    int B, Hq, Hkv, N, g, w, n_pairs, n_items;
    // Query rows [q_off, q_off + n_q) of the N-token sequence; Q, O and LSE hold those rows,
    // K and V hold the raw tokens from kv_off on.  The whole sequence: 0, N, 0.
    int q_off, n_q, kv_off;
    int window_mode;  // 1: raw window starts at the group boundary g * (lo(i) / g)
    float scale_log2;
    __nv_bfloat16 *O;
    float *LSE;
    int32_t *status;
    unsigned long long wait_limit_ns;
    int skip_q_load;  // test hook: never load Q, so the pipeline waits run out
    int o_align32;    // O is 32-byte aligned: the epilogue may use 32-byte stores
};

__device__ __forceinline__ int lo_of(int i, int w) { return window_lo(i, w); }
// first raw token of row i's window (cores stay j < lo(i)/g in both modes)
__device__ __forceinline__ int win_of(const Params &p, int i) { return window_start(i, p.w, p.g, p.window_mode); }

// The tile sequence of one work item and which half uses which tile.  Per-half
// fields are scalars chosen with selects (no runtime-indexed arrays, which
// would live in local memory).
struct Half {
    int a, b;     // first / last valid row
    bool valid;
    int tc;       // core tiles used: [0, tc)
    int kl, kh;   // local tiles used: [kl, kh)
};

struct Item {
    int bh, kvz;
    Half hA, hB;
    int Tc;   // core tiles loaded (max of the halves' tc)
    int lo0;  // first key of local tile 0
    int T;    // tiles loaded

    __device__ __forceinline__ const Half &half(int h) const { return h ? hB : hA; }
};

__device__ __forceinline__ bool half_uses(const Half &x, int Tc, int t) {
    if (!x.valid) return false;
    if (t < Tc) return t < x.tc;
    const int k = t - Tc;
    return k >= x.kl && k < x.kh;
}
__device__ __forceinline__ int half_first(const Half &x, int Tc) { return x.tc > 0 ? 0 : Tc + x.kl; }
// next used tile after t, or -1
__device__ __forceinline__ int half_next(const Half &x, int Tc, int t) {
    if (t < Tc) return (t + 1 < x.tc) ? t + 1 : Tc + x.kl;
    return (t + 1 < Tc + x.kh) ? t + 1 : -1;
}
__device__ __forceinline__ int half_count(const Half &x) { return x.valid ? x.tc + x.kh - x.kl : 0; }

// Largest step between consecutive tiles of a half: only the step from its last core tile
// to its first local tile can exceed 1.
__device__ __forceinline__ int half_max_step(const Half &x, int Tc) {
    return (x.valid && x.tc > 0) ? Tc + x.kl - (x.tc - 1) : 1;
}

__device__ __forceinline__ Half make_half(const Params &p, int a, int lo0) {
    Half x;
    x.a = a;
    x.valid = a - p.q_off < p.n_q;
    x.b = min(a + BM - 1, p.q_off + p.n_q - 1);
    if (!x.valid) {
        x.tc = x.kl = x.kh = 0;
        return x;
    }
    const int nc = lo_of(x.b, p.w) / p.g;
    x.tc = (nc + BN - 1) / BN;
    x.kl = (win_of(p, a) - lo0) / BN;
    x.kh = (x.b - lo0) / BN + 1;
    return x;
}

__device__ __forceinline__ Item make_item(const Params &p, int k) {
    Item it;
    const int BH = p.B * p.Hq;
    const int pair = p.n_pairs - 1 - k / BH;  // heaviest pairs first
    it.bh = k % BH;
    const int b = it.bh / p.Hq, h = it.bh % p.Hq;
    it.kvz = b * p.Hkv + h / (p.Hq / p.Hkv);
    const int i0 = p.q_off + pair * 2 * BM;  // first row (indices are the sequence's)
    it.lo0 = win_of(p, i0);
    it.hA = make_half(p, i0, it.lo0);
    it.hB = make_half(p, i0 + BM, it.lo0);
    const int last = it.hB.valid ? it.hB.b : it.hA.b;
    it.Tc = max(it.hA.tc, it.hB.tc);
    it.T = it.Tc + (last - it.lo0) / BN + 1;
    return it;
}

// Parity of the FULL barrier of the ring slot holding K for ring index u (u even).
// Only K slots complete a FULL barrier (the tile's V copy completes the same one),
// and with NS odd an even u reaches each slot once every 2*NS indices.
__device__ __forceinline__ uint32_t k_full_parity(uint32_t u) { return (u / (2 * NS)) & 1; }

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

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(B_QFULL), 1);
        ptx::mbar_init(bar(B_QFREE), 1);
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(bar(B_FULL + s), 1);
            ptx::mbar_init(bar(B_EMPTY + s), 1);
        }
        for (int h = 0; h < 2; ++h) {
            ptx::mbar_init(bar(B_SFULL + h), 1);
            ptx::mbar_init(bar(B_PFULL + h), 4);  // one arrive per softmax warp
            ptx::mbar_init(bar(B_PVDONE + h), 1);
            ptx::mbar_init(bar(B_OFREE + h), 4);
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
    const uint64_t lim = p.wait_limit_ns;

    if (warp < 2) {
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------ producer
            ptx::prefetch_tmap(&tmQ);
            ptx::prefetch_tmap(&tmK);
            ptx::prefetch_tmap(&tmV);
            ptx::prefetch_tmap(&tmKc);
            ptx::prefetch_tmap(&tmVc);
            uint32_t u = 0;  // ring loads issued so far
            int n_iter = 0;
            bool ok = true;
            for (int k = blockIdx.x; ok && k < p.n_items; k += gridDim.x, ++n_iter) {
                const Item it = make_item(p, k);
                if (!ptx::wait_bounded(bar(B_QFREE), (n_iter & 1) ^ 1, abort_flag, lim)) break;
                if (!p.skip_q_load) {
                    ptx::mbar_arrive_expect_tx(bar(B_QFULL), 2 * TILE_BYTES);
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t dst = base + OFF_Q + h * TILE_BYTES;
                        const int row0 = (h ? it.hB.a : it.hA.a) - p.q_off;
                        ptx::tma_load_3d(&tmQ, bar(B_QFULL), dst, 0, row0, it.bh);
                        ptx::tma_load_3d(&tmQ, bar(B_QFULL), dst + HALF_BYTES, 64, row0, it.bh);
                    }
                }
                for (int t = 0; ok && t < it.T; ++t, u += 2) {
                    const bool core = t < it.Tc;
                    const int y = core ? t * BN : it.lo0 + (t - it.Tc) * BN - p.kv_off;
                    // K(t) goes to ring slot u % NS, V(t) to the next one; both copies
                    // complete the K slot's FULL barrier (u is even, see k_full_parity)
                    const int ks = u % NS, vs = (u + 1) % NS;
                    if (!ptx::wait_bounded(bar(B_EMPTY + ks), ((u / NS) & 1) ^ 1, abort_flag, lim) ||
                        !ptx::wait_bounded(bar(B_EMPTY + vs), (((u + 1) / NS) & 1) ^ 1, abort_flag, lim)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = bar(B_FULL + ks);
                    const uint32_t kdst = base + OFF_RING + ks * TILE_BYTES;
                    const uint32_t vdst = base + OFF_RING + vs * TILE_BYTES;
                    const void *mk = core ? (const void *)&tmKc : (const void *)&tmK;
                    const void *mv = core ? (const void *)&tmVc : (const void *)&tmV;
                    ptx::mbar_arrive_expect_tx(full, 2 * TILE_BYTES);
                    ptx::tma_load_3d(mk, full, kdst, 0, y, it.kvz);
                    ptx::tma_load_3d(mk, full, kdst + HALF_BYTES, 64, y, it.kvz);
                    ptx::tma_load_3d(mv, full, vdst, 0, y, it.kvz);
                    ptx::tma_load_3d(mv, full, vdst + HALF_BYTES, 64, y, it.kvz);
                }
            }
            if (*abort_flag) {
                // Let the copies already issued land before the CTA exits.
                volatile int never = 0;
                for (uint32_t v = u > 2 * NS ? u - 2 * NS : 0; v < u; v += 2)
                    ptx::wait_bounded(bar(B_FULL + v % NS), k_full_parity(v), &never, lim);
                if (!p.skip_q_load && n_iter > 0)
                    ptx::wait_bounded(bar(B_QFULL), (n_iter - 1) & 1, &never, lim);
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer
            // The whole warp runs the issuer with identical values in every lane; the
            // MMAs and commits are issued by one elected lane.
            auto wwait = [&](uint32_t b, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, ptx::wait_bounded(b, parity, abort_flag, lim));
            };
            uint32_t ubase = 0;
            int n_iter = 0;
            uint32_t kpend = 0;  // pending S issues per ring slot, 2 bits per slot
            uint32_t pf_cnt[2] = {0, 0};
            int n_half[2] = {0, 0};  // items each half has processed
            // Descriptors of step 0 for Q_A, Q_B and for ring slot 0; a slot adds TILE_BYTES/16.
            const uint64_t dq0 = ptx::smem_desc_sw128(base + OFF_Q, 16, 1024);
            const uint64_t dq1 = ptx::smem_desc_sw128(base + OFF_Q + TILE_BYTES, 16, 1024);
            const uint64_t dk0 = ptx::smem_desc_sw128(base + OFF_RING, 16, 1024);
            const uint64_t dv0 = ptx::smem_desc_sw128(base + OFF_RING, HALF_BYTES, 1024);
            bool ok = true;
            for (int k = blockIdx.x; ok && k < p.n_items; k += gridDim.x, ++n_iter) {
                const Item it = make_item(p, k);
                if (!wwait(bar(B_QFULL), n_iter & 1)) break;
                int s_left = half_count(it.hA) + half_count(it.hB);
                // S_h = Q_h K(t)^T into S_h.  The first user of a ring slot waits for the copy.
                auto issue_s = [&](int h, int t) -> bool {
                    const uint32_t uk = ubase + 2 * t;
                    const int slot = uk % NS;
                    uint32_t pend = (kpend >> (2 * slot)) & 3u;
                    if (pend == 0) {
                        // the tile's first S: wait for its K and V copies
                        if (!wwait(bar(B_FULL + slot), k_full_parity(uk))) return false;
                        pend = (half_uses(it.hA, it.Tc, t) ? 1u : 0u) + (half_uses(it.hB, it.Tc, t) ? 1u : 0u);
                    }
                    ptx::tc_fence_after();
                    ptx::mma_ss_k128_warp(tmem + TM_S + h * BN, h ? dq1 : dq0, dk0 + static_cast<uint64_t>(slot) * (TILE_BYTES >> 4),
                                     IDESC_QK, 0u);
                    ptx::tc_commit_warp(bar(B_SFULL + h));
                    --pend;
                    kpend = (kpend & ~(3u << (2 * slot))) | (pend << (2 * slot));
                    if (pend == 0) ptx::tc_commit_warp(bar(B_EMPTY + slot));
                    if (--s_left == 0) ptx::tc_commit_warp(bar(B_QFREE));
                    return true;
                };
                // Prologue: first S of each half, earliest tile first, so that the issuer
                // never waits on a copy that sits behind one it has not consumed yet.
                {
                    const bool b_first = it.hB.valid && half_first(it.hB, it.Tc) < half_first(it.hA, it.Tc);
                    for (int q = 0; ok && q < 2; ++q) {
                        const int h = b_first ? 1 - q : q;
                        const Half &x = it.half(h);
                        if (x.valid) ok = issue_s(h, half_first(x, it.Tc));
                    }
                }
                // The tile loop.  After a half's PV on tile t the issuer starts S on the
                // half's next tile, which first waits for that tile's copies; with a ring of
                // two and a half tiles whose earlier slots only this loop frees, that wait can
                // end only if the next tile is at most t + 2.  With the window aligned to groups
                // of more than 128 tokens, half B's band can start further than that after its
                // last core tile, so items with such a step take the second copy of the loop,
                // which holds the S back (defer[h]) until the loop is two tiles short of it.
                // The copies are separate so that the common loop carries none of that logic.
                if (half_max_step(it.hA, it.Tc) <= 2 && half_max_step(it.hB, it.Tc) <= 2) {
                    bool first_pv[2] = {true, true};
                    for (int t = 0; ok && t < it.T; ++t) {
                        // V(t) has landed: the tile's first S waited for its K and V together
                        const uint32_t uv = ubase + 2 * t + 1;
                        const int vslot = uv % NS;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {  // unrolled: per-half counters stay in registers
                            const Half &x = it.half(h);
                            if (!half_uses(x, it.Tc, t)) continue;
                            if (!wwait(bar(B_PFULL + h), pf_cnt[h] & 1)) {
                                ok = false;
                                break;
                            }
                            ++pf_cnt[h];
                            if (first_pv[h]) {
                                // the epilogue of this half's previous item must have read O_h
                                if (!wwait(bar(B_OFREE + h), (n_half[h] & 1) ^ 1)) {
                                    ok = false;
                                    break;
                                }
                            }
                            ptx::tc_fence_after();
                            ptx::mma_ts_k128_warp(tmem + TM_O + h * HD, tmem + TM_S + h * BN,
                                             dv0 + static_cast<uint64_t>(vslot) * (TILE_BYTES >> 4), IDESC_PV,
                                             first_pv[h] ? 0u : 1u);
                            first_pv[h] = false;
                            const int tn = half_next(x, it.Tc, t);
                            if (tn >= 0) {
                                if (!issue_s(h, tn)) {
                                    ok = false;
                                    break;
                                }
                            } else {
                                ptx::tc_commit_warp(bar(B_PVDONE + h));
                            }
                        }
                        if (!ok) break;
                        ptx::tc_commit_warp(bar(B_EMPTY + vslot));
                    }
                } else {
                    bool first_pv[2] = {true, true};
                    int defer[2] = {-1, -1};
                    for (int t = 0; ok && t < it.T; ++t) {
                        // V(t) has landed: the tile's first S waited for its K and V together
                        const uint32_t uv = ubase + 2 * t + 1;
                        const int vslot = uv % NS;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (defer[h] >= 0 && defer[h] <= t + 2) {
                                if (!issue_s(h, defer[h])) {
                                    ok = false;
                                    break;
                                }
                                defer[h] = -1;
                            }
                        }
                        if (!ok) break;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {  // unrolled: per-half counters stay in registers
                            const Half &x = it.half(h);
                            if (!half_uses(x, it.Tc, t)) continue;
                            if (!wwait(bar(B_PFULL + h), pf_cnt[h] & 1)) {
                                ok = false;
                                break;
                            }
                            ++pf_cnt[h];
                            if (first_pv[h]) {
                                // the epilogue of this half's previous item must have read O_h
                                if (!wwait(bar(B_OFREE + h), (n_half[h] & 1) ^ 1)) {
                                    ok = false;
                                    break;
                                }
                            }
                            ptx::tc_fence_after();
                            ptx::mma_ts_k128_warp(tmem + TM_O + h * HD, tmem + TM_S + h * BN,
                                             dv0 + static_cast<uint64_t>(vslot) * (TILE_BYTES >> 4), IDESC_PV,
                                             first_pv[h] ? 0u : 1u);
                            first_pv[h] = false;
                            const int tn = half_next(x, it.Tc, t);
                            if (tn > t + 2) {
                                defer[h] = tn;
                            } else if (tn >= 0) {
                                if (!issue_s(h, tn)) {
                                    ok = false;
                                    break;
                                }
                            } else {
                                ptx::tc_commit_warp(bar(B_PVDONE + h));
                            }
                        }
                        if (!ok) break;
                        ptx::tc_commit_warp(bar(B_EMPTY + vslot));
                    }
                }
                ubase += 2 * it.T;
                n_half[0] += it.hA.valid ? 1 : 0;
                n_half[1] += it.hB.valid ? 1 : 0;
            }
            // Whatever was issued must complete before tensor memory is freed.
            ptx::tc_commit_warp(bar(B_DRAIN));
            volatile int never = 0;
            ptx::wait_bounded(bar(B_DRAIN), 0, &never, lim);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int h = (warp - 2) >> 2;  // half
        const int quarter = warp & 3;   // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_addr + TM_S + h * BN;
        const uint32_t tO = tmem + lane_addr + TM_O + h * HD;
        uint32_t sf_cnt = 0;
        int n_done = 0;  // items of this half finished
        bool ok = true;
        for (int k = blockIdx.x; ok && k < p.n_items; k += gridDim.x) {
            const Item it = make_item(p, k);
            const Half x = h ? it.hB : it.hA;
            if (!x.valid) continue;
            const int i = x.a + row;
            const int lo_i = win_of(p, i);           // first raw token of this row's window
            const int nc_i = lo_of(i, p.w) / p.g;    // cores visible to this row
            const int nc_first = lo_of(x.a, p.w) / p.g;
            const int lo_last = win_of(p, x.b);
            float m = -INFINITY;  // running max of the log2-scaled logits
            float l = 0.f;
            for (int t = half_first(x, it.Tc); t >= 0; t = half_next(x, it.Tc, t)) {
                if (!__all_sync(0xffffffffu, ptx::wait_bounded(bar(B_SFULL + h), sf_cnt & 1, abort_flag, lim))) {
                    ok = false;
                    break;
                }
                ++sf_cnt;
                ptx::tc_fence_after();
                uint32_t s[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + c * 32, s[c]);
                ptx::tmem_wait_ld(s[0]);
                ptx::reg_touch(s[1]);
                ptx::reg_touch(s[2]);
                ptx::reg_touch(s[3]);

                // visibility window of this row within the tile: columns [c_lo, c_hi]
                int c_lo = 0, c_hi = BN - 1;
                bool masked;
                if (t < it.Tc) {
                    const int y0 = t * BN;
                    masked = y0 + BN > nc_first;
                    c_hi = min(nc_i - y0, BN) - 1;
                } else {
                    const int y0 = it.lo0 + (t - it.Tc) * BN;
                    masked = (y0 < lo_last) || (y0 + BN - 1 > x.a);
                    c_lo = max(lo_i - y0, 0);
                    c_hi = min(i - y0, BN - 1);
                }
                // row max: 3-input max over eight independent partial maxima
                float mp[8];
                if (masked) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int kk = 0; kk < 32; ++kk) {
                            const int col = c * 32 + kk;
                            const float x = __uint_as_float(s[c][kk]);
                            s[c][kk] = __float_as_uint((col < c_lo || col > c_hi) ? -INFINITY : x);
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    mp[q] = fmaxf(__uint_as_float(s[q >> 1][(q & 1) * 16]), __uint_as_float(s[q >> 1][(q & 1) * 16 + 1]));
#pragma unroll
                for (int q = 0; q < 8; ++q) {
#pragma unroll
                    for (int kk = 2; kk < 16; kk += 2)
                        mp[q] = ptx::max3(mp[q], __uint_as_float(s[q >> 1][(q & 1) * 16 + kk]),
                                          __uint_as_float(s[q >> 1][(q & 1) * 16 + kk + 1]));
                }
                const float mx = ptx::max3(ptx::max3(mp[0], mp[1], mp[2]), ptx::max3(mp[3], mp[4], mp[5]),
                                           fmaxf(mp[6], mp[7]));
                const float m_tile = mx * p.scale_log2;  // -inf stays -inf
                const float m_new = fmaxf(m, m_tile);
                bool rescale = false;
                if (m == -INFINITY) {
                    m = m_new;  // nothing accumulated yet for this row
                } else if (m_new > m + LAZY_RESCALE_LOG2) {
                    rescale = true;
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    // S_h complete => every earlier PV of this half is complete: O_h is stable.
                    const float f = rescale ? ptx::ex2(m - m_new) : 1.f;
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        uint32_t o[16];
                        ptx::tmem_ld16(tO + c * 16, o);
                        ptx::tmem_wait_ld16(o);
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk) o[kk] = __float_as_uint(__uint_as_float(o[kk]) * f);
                        ptx::tmem_st16(tO + c * 16, o);
                    }
                    if (rescale) {
                        l *= f;
                        m = m_new;
                    }
                }
                const float mu = (m == -INFINITY) ? 0.f : m;
                // p = 2^(s*scale - mu), two columns per packed FMA; row sum in four packed partials
                const uint64_t sc2 = ptx::f2(p.scale_log2, p.scale_log2);
                const uint64_t nm2 = ptx::f2(-mu, -mu);
                uint64_t lp[2] = {0, 0};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t pk[8];
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const int col = (c & 1) * 16 + 2 * kk;
                        const uint64_t x2 = ptx::fma2(
                            ptx::f2(__uint_as_float(s[c >> 1][col]), __uint_as_float(s[c >> 1][col + 1])), sc2, nm2);
                        float x0, x1;
                        ptx::f2_split(x2, x0, x1);
                        const float p0 = ptx::ex2(x0);
                        const float p1 = ptx::ex2(x1);
                        lp[kk & 1] = ptx::add2(lp[kk & 1], ptx::f2(p0, p1));
                        pk[kk] = ptx::pack_bf16x2(p0, p1);
                    }
                    ptx::tmem_st8(tS + c * 8, pk);  // P_h over the consumed columns of S_h
                }
                {
                    float a0, a1, b0, b1;
                    ptx::f2_split(lp[0], a0, a1);
                    ptx::f2_split(lp[1], b0, b1);
                    l += (a0 + a1) + (b0 + b1);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(B_PFULL + h));
            }
            if (!ok) break;
            // ---- epilogue: O_h / l -> bf16, LSE
            if (!__all_sync(0xffffffffu, ptx::wait_bounded(bar(B_PVDONE + h), n_done & 1, abort_flag, lim))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const int li = i - p.q_off;  // row of O and LSE
            const bool valid = li < p.n_q;
            const float inv = 1.f / l;
            __nv_bfloat16 *orow = p.O + (static_cast<int64_t>(it.bh) * p.n_q + li) * HD;
            uint32_t o[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tO + c * 32, o[c]);
            ptx::tmem_wait_ld(o[0]);
            ptx::reg_touch(o[1]);
            ptx::reg_touch(o[2]);
            ptx::reg_touch(o[3]);
            // O_h is in registers: the issuer may start this half's next item
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(B_OFREE + h));
            // O / l as bf16, one 32-byte sector per store (two 16-byte stores if O is
            // only 16-byte aligned)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t v[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        v[k] = ptx::pack_bf16x2(__uint_as_float(o[c][16 * q + 2 * k]) * inv,
                                                __uint_as_float(o[c][16 * q + 2 * k + 1]) * inv);
                    if (valid) {
                        if (p.o_align32) {
                            ptx::st_global_v8(orow + c * 32 + q * 16, v);
                        } else {
                            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32 + q * 16);
                            dst[0] = make_uint4(v[0], v[1], v[2], v[3]);
                            dst[1] = make_uint4(v[4], v[5], v[6], v[7]);
                        }
                    }
                }
            }
            if (valid) p.LSE[static_cast<int64_t>(it.bh) * p.n_q + li] = (m + __log2f(l)) * 0.6931471805599453f;
            ++n_done;
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
struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    cudaError_t attr_err = cudaSuccess;
};

DeviceInfo &device_info(int dev) {
    static DeviceInfo info[64];
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo &d = info[dev & 63];
    if (!d.ready) {
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        d.attr_err = cudaFuncSetAttribute(attn_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(SMEM_BYTES));
        d.ready = true;
    }
    return d;
}

}  // namespace

// Test hooks (see cca_test_* in cca_api.cu).
unsigned long long g_wait_limit_ns = 1000000000ull;
int g_skip_q_load = 0;

cudaError_t launch_attn_bf16_tc(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                                void *O, float *LSE, const Shape &s, int32_t *dev_status, cudaStream_t stream,
                                const RowRange &rr) {
    EncodeTiledFn enc = get_encoder();
    if (enc == nullptr) return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const DeviceInfo &di = device_info(dev);
    if (di.attr_err != cudaSuccess) return di.attr_err;
    const uint64_t G = static_cast<uint64_t>(s.N / s.g);
    CUtensorMap mQ, mK, mV, mKc, mVc;
    const uint64_t qh = static_cast<uint64_t>(s.B) * s.Hq, kh = static_cast<uint64_t>(s.B) * s.Hkv;
    const int n_q = rr.n_q < 0 ? s.N : rr.n_q, n_kv = rr.n_kv < 0 ? s.N : rr.n_kv;
    if (!encode_3d_bf16_d128(enc, &mQ, Q, n_q, qh) || !encode_3d_bf16_d128(enc, &mK, K, n_kv, kh) ||
        !encode_3d_bf16_d128(enc, &mV, V, n_kv, kh) || !encode_3d_bf16_d128(enc, &mKc, Kc, G, kh) ||
        !encode_3d_bf16_d128(enc, &mVc, Vc, G, kh))
        return cudaErrorInvalidValue;

    Params p;
    p.B = s.B;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.N = s.N;
    p.g = s.g;
    p.w = s.w;
    p.window_mode = s.window_mode;
    p.q_off = rr.q_off;
    p.n_q = n_q;
    p.kv_off = rr.kv_off;
    p.n_pairs = (n_q + 2 * BM - 1) / (2 * BM);
    p.n_items = p.n_pairs * s.B * s.Hq;
    p.scale_log2 = s.scale * 1.4426950408889634f;
    p.O = static_cast<__nv_bfloat16 *>(O);
    p.LSE = LSE;
    p.status = dev_status;
    p.wait_limit_ns = g_wait_limit_ns;
    p.skip_q_load = g_skip_q_load;
    p.o_align32 = (reinterpret_cast<uintptr_t>(O) & 31u) == 0 ? 1 : 0;
    const unsigned grid = static_cast<unsigned>(p.n_items < di.sms ? p.n_items : di.sms);
    attn_bf16_tc_kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(mQ, mK, mV, mKc, mVc, p);
    return cudaGetLastError();
}

}  // namespace cca
