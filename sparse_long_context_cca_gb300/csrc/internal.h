// Internal interface between the C-ABI front end (cca_api.cu) and the kernel
// translation units.  Arguments are already validated when these are called.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace cca {

struct Shape {
    int B, Hq, Hkv, N, d, g, w;
    float scale;  // resolved softmax scale (> 0)
    int window_mode = 0;  // 1: raw window starts at the group boundary g*(lo/g)
    int pool_mode = 0;    // 0 softmax, 1 mean, 2 max
};

// Global-aware pooling. dtype: 0 = bf16, 1 = f32.  `status` (optional device
// int32) receives CCA_ERR_TIMEOUT if a copy wait runs out.
cudaError_t launch_pool(int dtype, const void *Q, const void *K, const void *V, void *Kc, void *Vc,
                        const Shape &s, int32_t *status, cudaStream_t stream);

// The query rows an attention launch computes: rows [q_off, q_off + n_q) of the s.N-token
// sequence, Q/O/LSE holding those rows and K/V the raw tokens [kv_off, kv_off + n_kv).
// Negative counts stand for s.N (the whole sequence).  Kc/Vc always hold all s.N/g cores.
struct RowRange {
    int q_off = 0, n_q = -1, kv_off = 0, n_kv = -1;
};

// fp32 fused attention on CUDA cores (any supported d).
cudaError_t launch_attn_f32(const float *Q, const float *K, const float *V, const float *Kc,
                            const float *Vc, float *O, float *LSE, const Shape &s,
                            cudaStream_t stream, const RowRange &rr = RowRange{});

// bf16 fused attention on the tcgen05 tensor cores (d = 128).
// Returns cudaErrorNotSupported when the tensor-map encoder is unavailable.
cudaError_t launch_attn_bf16_tc(const void *Q, const void *K, const void *V, const void *Kc,
                                const void *Vc, void *O, float *LSE, const Shape &s,
                                int32_t *dev_status, cudaStream_t stream, const RowRange &rr = RowRange{});

// Decode step (row `pos` of the fused attention over the caches) and single-group pooling.
uint64_t decode_workspace_bytes(const Shape &s);
// With plan_kernels set, nothing is launched: *plan_kernels receives the number of kernels
// the call would launch (1: the splits merge inside thread-block clusters; 2: split + merge).
cudaError_t launch_decode(int dtype, const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                          void *O, float *LSE, const Shape &s, int pos, float *ws, cudaStream_t stream,
                          int *plan_kernels = nullptr);
// Fixed scratch of the no-allocation decode entry point (bytes) and its device address
// on the current device (looked up on first use per device).
constexpr uint64_t DECODE_NOALLOC_MAX_BYTES = 4ull << 20;
cudaError_t decode_noalloc_scratch(float **out);
cudaError_t launch_pool_group(int dtype, const void *q, const void *K, const void *V, void *Kc, void *Vc,
                              const Shape &s, int j, cudaStream_t stream);

// Backward pass (fp32 gradients; workspace holds D and the core-token gradients).
uint64_t prefill_bwd_workspace_bytes(const Shape &s);
// bf16 with d = 128 runs the attention part on the tensor cores (launch_attn_bwd_tc).
cudaError_t launch_prefill_bwd(int dtype, const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                               const void *O, const float *LSE, const void *dO, float *dQ, float *dK, float *dV,
                               const Shape &s, float *ws, int32_t *status, cudaStream_t stream);
// The pooling backward's share of a raw token's gradient, added by the dK/dV kernel
// while it writes the token's row: dK_t += a_t dKc_j + cds_t qs_j, dV_t += a_t dVc_j
// (j the token's group).  mode 0: nothing added; 1: mean pooling (a_t = 1/g, cds_t = 0,
// no arrays); 2: a, cds ([B, Hkv, N]) and qs ([B, Hkv, N/g, 128], fp32) as given.
struct BwdPoolFuse {
    int mode;
    const float *a, *cds, *qs;
};
// Tensor-core attention backward (bf16, d = 128).  part 0: dQ (all rows), D = dO.O into
// Dbuf, dK/dV of the raw tokens and dKc/dVc of the cores, no pooling backward; part 1:
// dQ, D and the cores' dKc/dVc only; part 2: the raw tokens' dK/dV only, with the
// pooling backward pf folded in (dKc/dVc already complete).
cudaError_t launch_attn_bwd_tc(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                               const void *O, const float *LSE, const void *dO, float *dQ, float *dK, float *dV,
                               float *Dbuf, float *dKc, float *dVc, const Shape &s, int32_t *status, int part,
                               const BwdPoolFuse &pf, cudaStream_t stream);

// Prefill on host buffers, pipelined over slices of (batch, KV head) pairs (host_pipeline.cu).
uint64_t prefill_host_workspace_bytes(const Shape &s, int dtype);
cudaError_t launch_prefill_host(int dtype, const void *hQ, const void *hK, const void *hV, void *hO, float *hLSE,
                                void *hKc, void *hVc, const Shape &s, void *workspace, int32_t *status,
                                cudaStream_t stream);

}  // namespace cca
