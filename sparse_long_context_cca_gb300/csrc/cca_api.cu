// C ABI front end of libcca.so (declared in include/cca.h): argument checks,
// dtype/shape dispatch and launch.  Every check runs on the host before any
// CUDA call, so a rejected call launches nothing and writes nothing.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/cca.h"
#include "internal.h"
#include "visibility.cuh"

namespace cca {
extern unsigned long long g_wait_limit_ns;
extern int g_skip_q_load;
extern int g_decode_path;
}  // namespace cca

static_assert(cca::DECODE_NOALLOC_MAX_BYTES == CCA_DECODE_NOALLOC_MAX_BYTES, "scratch size mismatch");

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const cca_params_t *p, bool need_w) {
    if (p == nullptr) return CCA_ERR_INVALID_ARG;
    if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->N < 1 || p->d < 1 || p->g < 1) return CCA_ERR_INVALID_ARG;
    if (need_w && p->w < 1) return CCA_ERR_INVALID_ARG;
    if (p->Hq % p->Hkv != 0 || p->N % p->g != 0) return CCA_ERR_INVALID_ARG;
    if (p->dtype != CCA_BF16 && p->dtype != CCA_F32) return CCA_ERR_INVALID_ARG;
    if (!(p->scale == p->scale) || isinf(p->scale)) return CCA_ERR_INVALID_ARG;
    if (p->window_mode < 0 || p->window_mode > 1 || p->pool_mode < 0 || p->pool_mode > 3)
        return CCA_ERR_INVALID_ARG;
    // pool_mode 3 keeps a running (max, sum) per query head of a KV head: at most 8
    if (p->pool_mode == 3 && p->Hq / p->Hkv > 8) return CCA_ERR_UNSUPPORTED;
    // Element counts of the largest tensor must fit the kernels' 64-bit indexing and
    // row counts the 32-bit tensor-map coordinates.
    const double elems = static_cast<double>(p->B) * p->Hq * p->N * p->d;
    if (elems > 9.0e15) return CCA_ERR_INVALID_ARG;
    if (p->d != 64 && p->d != 128) return CCA_ERR_UNSUPPORTED;
    return CCA_OK;
}

cca::Shape to_shape(const cca_params_t *p) {
    cca::Shape s;
    s.B = p->B;
    s.Hq = p->Hq;
    s.Hkv = p->Hkv;
    s.N = p->N;
    s.d = p->d;
    s.g = p->g;
    s.w = p->w;
    s.scale = p->scale > 0.f ? p->scale : 1.0f / sqrtf(static_cast<float>(p->d));
    s.window_mode = p->window_mode;
    s.pool_mode = p->pool_mode;
    return s;
}

// The kernels are built for sm_103a only.
int check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CCA_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return CCA_ERR_CUDA;
    if (major != 10 || minor != 3) return CCA_ERR_UNSUPPORTED;
    return CCA_OK;
}

int from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return CCA_OK;
    if (e == cudaErrorNotSupported) return CCA_ERR_UNSUPPORTED;
    return CCA_ERR_CUDA;
}

}  // namespace

extern "C" {

int cca_pool(const void *Q, const void *K, const void *V, void *Kc, void *Vc, const cca_params_t *params,
             void *stream) {
    int st = check_shape(params, false);
    if (st != CCA_OK) return st;
    const void *ptrs[5] = {Q, K, V, Kc, Vc};
    for (const void *q : ptrs)
        if (q == nullptr || !aligned16(q)) return CCA_ERR_INVALID_ARG;
    if (params->dev_status != nullptr && (reinterpret_cast<uintptr_t>(params->dev_status) & 3u) != 0)
        return CCA_ERR_INVALID_ARG;
    if ((st = check_device()) != CCA_OK) return st;
    return from_cuda(cca::launch_pool(params->dtype, Q, K, V, Kc, Vc, to_shape(params), params->dev_status,
                                      static_cast<cudaStream_t>(stream)));
}

int cca_attn_fwd(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc, void *O, float *LSE,
                 const cca_params_t *params, void *stream) {
    int st = check_shape(params, true);
    if (st != CCA_OK) return st;
    const void *ptrs[7] = {Q, K, V, Kc, Vc, O, LSE};
    for (const void *q : ptrs)
        if (q == nullptr || !aligned16(q)) return CCA_ERR_INVALID_ARG;
    if (params->dev_status != nullptr && (reinterpret_cast<uintptr_t>(params->dev_status) & 3u) != 0)
        return CCA_ERR_INVALID_ARG;
    if (params->dtype == CCA_BF16 && params->d != 128) return CCA_ERR_UNSUPPORTED;
    if ((st = check_device()) != CCA_OK) return st;
    const cca::Shape s = to_shape(params);
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    if (params->dtype == CCA_F32)
        return from_cuda(cca::launch_attn_f32(static_cast<const float *>(Q), static_cast<const float *>(K),
                                              static_cast<const float *>(V), static_cast<const float *>(Kc),
                                              static_cast<const float *>(Vc), static_cast<float *>(O), LSE, s,
                                              strm));
    return from_cuda(cca::launch_attn_bf16_tc(Q, K, V, Kc, Vc, O, LSE, s, params->dev_status, strm));
}

int cca_attn_fwd_rows(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc, void *O,
                      float *LSE, int q_off, int n_q, int kv_off, int n_kv, const cca_params_t *params,
                      void *stream) {
    int st = check_shape(params, true);
    if (st != CCA_OK) return st;
    const void *ptrs[7] = {Q, K, V, Kc, Vc, O, LSE};
    for (const void *q : ptrs)
        if (q == nullptr || !aligned16(q)) return CCA_ERR_INVALID_ARG;
    if (params->dev_status != nullptr && (reinterpret_cast<uintptr_t>(params->dev_status) & 3u) != 0)
        return CCA_ERR_INVALID_ARG;
    // the rows, then the raw tokens they read: every window lies inside [kv_off, kv_off + n_kv)
    const int64_t N = params->N;
    if (n_q < 1 || q_off < 0 || static_cast<int64_t>(q_off) + n_q > N) return CCA_ERR_INVALID_ARG;
    if (kv_off < 0 || n_kv < 1 || static_cast<int64_t>(kv_off) + n_kv > N) return CCA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(kv_off) + n_kv < static_cast<int64_t>(q_off) + n_q) return CCA_ERR_INVALID_ARG;
    if (kv_off > cca::window_start(q_off, params->w, params->g, params->window_mode)) return CCA_ERR_INVALID_ARG;
    if (params->dtype == CCA_BF16 && params->d != 128) return CCA_ERR_UNSUPPORTED;
    if ((st = check_device()) != CCA_OK) return st;
    const cca::Shape s = to_shape(params);
    cca::RowRange rr;
    rr.q_off = q_off;
    rr.n_q = n_q;
    rr.kv_off = kv_off;
    rr.n_kv = n_kv;
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    if (params->dtype == CCA_F32)
        return from_cuda(cca::launch_attn_f32(static_cast<const float *>(Q), static_cast<const float *>(K),
                                              static_cast<const float *>(V), static_cast<const float *>(Kc),
                                              static_cast<const float *>(Vc), static_cast<float *>(O), LSE, s,
                                              strm, rr));
    return from_cuda(cca::launch_attn_bf16_tc(Q, K, V, Kc, Vc, O, LSE, s, params->dev_status, strm, rr));
}

int cca_decode_fwd(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc, void *O, float *LSE,
                   int pos, const cca_params_t *params, void *workspace, uint64_t workspace_bytes, void *stream) {
    int st = check_shape(params, true);
    if (st != CCA_OK) return st;
    const void *ptrs[8] = {Q, K, V, Kc, Vc, O, LSE, workspace};
    for (const void *q : ptrs)
        if (q == nullptr || !aligned16(q)) return CCA_ERR_INVALID_ARG;
    if (pos < 0 || pos >= params->N) return CCA_ERR_INVALID_ARG;
    const int r = params->Hq / params->Hkv;
    if (r != 1 && r != 2 && r != 4 && r != 8) return CCA_ERR_UNSUPPORTED;
    const cca::Shape s = to_shape(params);
    if (workspace_bytes < cca::decode_workspace_bytes(s)) return CCA_ERR_INVALID_ARG;
    if ((st = check_device()) != CCA_OK) return st;
    return from_cuda(cca::launch_decode(params->dtype, Q, K, V, Kc, Vc, O, LSE, s, pos,
                                        static_cast<float *>(workspace), static_cast<cudaStream_t>(stream)));
}

int cca_decode_fwd_noalloc(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc, void *O,
                           float *LSE, int pos, const cca_params_t *params, void *stream) {
    int st = check_shape(params, true);
    if (st != CCA_OK) return st;
    const void *ptrs[7] = {Q, K, V, Kc, Vc, O, LSE};
    for (const void *q : ptrs)
        if (q == nullptr || !aligned16(q)) return CCA_ERR_INVALID_ARG;
    if (pos < 0 || pos >= params->N) return CCA_ERR_INVALID_ARG;
    const int r = params->Hq / params->Hkv;
    if (r != 1 && r != 2 && r != 4 && r != 8) return CCA_ERR_UNSUPPORTED;
    const cca::Shape s = to_shape(params);
    if (cca::decode_workspace_bytes(s) > cca::DECODE_NOALLOC_MAX_BYTES) return CCA_ERR_SCRATCH_LIMIT;
    if ((st = check_device()) != CCA_OK) return st;
    float *scratch = nullptr;
    cudaError_t e = cca::decode_noalloc_scratch(&scratch);
    if (e != cudaSuccess) return CCA_ERR_CUDA;
    return from_cuda(cca::launch_decode(params->dtype, Q, K, V, Kc, Vc, O, LSE, s, pos, scratch,
                                        static_cast<cudaStream_t>(stream)));
}

int cca_prefill_bwd(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc, const void *O,
                    const float *LSE, const void *dO, float *dQ, float *dK, float *dV, const cca_params_t *params,
                    void *workspace, uint64_t workspace_bytes, void *stream) {
    int st = check_shape(params, true);
    if (st != CCA_OK) return st;
    const void *ptrs[12] = {Q, K, V, Kc, Vc, O, LSE, dO, dQ, dK, dV, workspace};
    for (const void *q : ptrs)
        if (q == nullptr || !aligned16(q)) return CCA_ERR_INVALID_ARG;
    const cca::Shape s = to_shape(params);
    if (workspace_bytes < cca::prefill_bwd_workspace_bytes(s)) return CCA_ERR_INVALID_ARG;
    if (params->dev_status != nullptr && (reinterpret_cast<uintptr_t>(params->dev_status) & 3u) != 0)
        return CCA_ERR_INVALID_ARG;
    if ((st = check_device()) != CCA_OK) return st;
    return from_cuda(cca::launch_prefill_bwd(params->dtype, Q, K, V, Kc, Vc, O, LSE, dO, dQ, dK, dV, s,
                                             static_cast<float *>(workspace), params->dev_status,
                                             static_cast<cudaStream_t>(stream)));
}

uint64_t cca_prefill_bwd_workspace_size(const cca_params_t *params) {
    if (check_shape(params, true) != CCA_OK) return 0;
    return cca::prefill_bwd_workspace_bytes(to_shape(params));
}

int cca_decode_kernels(const cca_params_t *params, int pos) {
    int st = check_shape(params, true);
    if (st != CCA_OK) return st;
    if (pos < 0 || pos >= params->N) return CCA_ERR_INVALID_ARG;
    if ((st = check_device()) != CCA_OK) return st;
    int n = 0;
    st = from_cuda(cca::launch_decode(params->dtype, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                      to_shape(params), pos, nullptr, nullptr, &n));
    return st != CCA_OK ? st : n;
}

uint64_t cca_decode_workspace_size(const cca_params_t *params) {
    if (check_shape(params, true) != CCA_OK) return 0;
    return cca::decode_workspace_bytes(to_shape(params));
}

int cca_pool_group(const void *q, const void *K, const void *V, void *Kc, void *Vc, int j, const cca_params_t *params,
                   void *stream) {
    int st = check_shape(params, false);
    if (st != CCA_OK) return st;
    const void *ptrs[5] = {q, K, V, Kc, Vc};
    for (const void *x : ptrs)
        if (x == nullptr || !aligned16(x)) return CCA_ERR_INVALID_ARG;
    if (j < 0 || j >= params->N / params->g) return CCA_ERR_INVALID_ARG;
    if ((st = check_device()) != CCA_OK) return st;
    return from_cuda(cca::launch_pool_group(params->dtype, q, K, V, Kc, Vc, to_shape(params), j,
                                            static_cast<cudaStream_t>(stream)));
}

uint64_t cca_prefill_host_workspace_size(const cca_params_t *params) {
    if (check_shape(params, true) != CCA_OK) return 0;
    return cca::prefill_host_workspace_bytes(to_shape(params), params->dtype);
}

int cca_prefill_host(const void *hQ, const void *hK, const void *hV, void *hO, float *hLSE, void *hKc, void *hVc,
                     const cca_params_t *params, void *workspace, uint64_t workspace_bytes, void *stream) {
    int st = check_shape(params, true);
    if (st != CCA_OK) return st;
    const void *ptrs[5] = {hQ, hK, hV, hO, workspace};
    for (const void *q : ptrs)
        if (q == nullptr) return CCA_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return CCA_ERR_INVALID_ARG;
    if ((hKc == nullptr) != (hVc == nullptr)) return CCA_ERR_INVALID_ARG;
    if (params->dev_status != nullptr && (reinterpret_cast<uintptr_t>(params->dev_status) & 3u) != 0)
        return CCA_ERR_INVALID_ARG;
    if (params->dtype == CCA_BF16 && params->d != 128) return CCA_ERR_UNSUPPORTED;
    const cca::Shape s = to_shape(params);
    if (workspace_bytes < cca::prefill_host_workspace_bytes(s, params->dtype)) return CCA_ERR_INVALID_ARG;
    if ((st = check_device()) != CCA_OK) return st;
    return from_cuda(cca::launch_prefill_host(params->dtype, hQ, hK, hV, hO, hLSE, hKc, hVc, s, workspace,
                                              params->dev_status, static_cast<cudaStream_t>(stream)));
}

const char *cca_status_string(int status) {
    switch (status) {
        case CCA_OK: return "ok";
        case CCA_ERR_INVALID_ARG: return "invalid argument";
        case CCA_ERR_UNSUPPORTED: return "unsupported dtype/head-dim combination or device";
        case CCA_ERR_CUDA: return "CUDA error";
        case CCA_ERR_TIMEOUT: return "device pipeline wait timed out";
        case CCA_ERR_SCRATCH_LIMIT: return "shapes need more scratch than the no-allocation entry point holds";
        default: return "unknown status";
    }
}

int cca_abi_version(void) { return CCA_ABI_VERSION; }

// Test hooks for the bounded-wait path of the bf16 attention kernel: set the
// per-wait time limit, and make later launches skip the Q-tile load so that
// the MMA issuer's first wait runs out.  Not part of the public header.
void cca_test_set_wait_limit_ns(unsigned long long ns) { cca::g_wait_limit_ns = ns; }
void cca_test_skip_q_load(int on) { cca::g_skip_q_load = on ? 1 : 0; }
void cca_test_decode_path(int path) { cca::g_decode_path = (path == 1 || path == 2) ? path : 0; }

}  // extern "C"
