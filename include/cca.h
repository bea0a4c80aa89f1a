/*
 * cca.h - C ABI of libcca.so: prefill forward of Core Context Aware (CCA)
 * attention on an sm_103a GPU.
 *
 * The method ("Core Context Aware Transformers for Long Context Language
 * Modeling", ICML 2025) replaces self-attention over N tokens by two steps:
 *
 *  1. Global-aware pooling (Method section, pooling equation
 *     c_i = softmax(Q_{ig} K'_{I_i}^T / sqrt(d)) X^G_{I_i}): the sequence is cut
 *     into N/g non-overlapping groups of g tokens; each group becomes one core
 *     key and one core value, the softmax-weighted sum of the group's keys and
 *     values, weighted by the logits of the group's last query against the
 *     group's keys.
 *  2. Fused attention (Method section, fusion equation
 *     Att_i = softmax(Q_i [K^G_{T_i}; K^L_{U_i}]^T / sqrt(d)) [V^G_{T_i}; V^L_{U_i}]):
 *     query i takes ONE softmax over the core tokens of the groups that lie
 *     entirely before its local window, followed by the raw tokens of the
 *     window.
 *
 * Index conventions (0-indexed; the pages leave them open):
 *   lo(i)      = max(0, i - w + 1)            first token of i's window
 *   window     = tokens [lo(i), i]           (n_loc = min(w, i + 1) tokens)
 *   core j     visible to i iff (j + 1) * g <= lo(i)   (n_core = lo(i) / g)
 *   group j    = tokens [j*g, (j+1)*g - 1], scored by the query of token (j+1)*g - 1
 *   GQA        query head h reads KV head h / (Hq / Hkv); a KV head's pooling
 *              logit is the mean of the logits of its Hq/Hkv query heads,
 *              taken before the group softmax.
 *   scale      tau = 1/sqrt(d) unless params.scale > 0; the same tau is used by
 *              both steps.  LSE is the natural log-sum-exp of the tau-scaled
 *              logits over the visible set.
 *
 * Layouts (all contiguous, row-major, d innermost; element type = dtype):
 *   Q  [B, Hq,  N,   d]      K, V   [B, Hkv, N,   d]
 *   Kc [B, Hkv, N/g, d]      Vc     [B, Hkv, N/g, d]
 *   O  [B, Hq,  N,   d]      LSE    [B, Hq,  N]  (always fp32)
 *
 * Ownership and execution: the caller allocates and owns every buffer; all
 * pointers except `params` are DEVICE pointers (16-byte aligned).  The library
 * keeps no allocation and no state between calls.  Calls are asynchronous on
 * `stream` (a cudaStream_t, NULL = legacy default stream); results are
 * defined after the stream reaches the call.  Arithmetic: bf16 inputs with
 * fp32 accumulation and fp32 softmax, outputs rounded to nearest even; f32
 * inputs computed in fp32 throughout.
 *
 * Errors: the return value reports host-side checks and the launch.  Nothing
 * is launched and nothing is written when a check fails.  A device-side
 * give-up (a pipeline wait that exceeded its time limit) is reported by
 * writing CCA_ERR_TIMEOUT into *params.dev_status when that pointer is set
 * (a caller-owned device int32 that the caller zeroes); the kernel then
 * returns without hanging and its outputs are unspecified.
 */
#ifndef CCA_H_
#define CCA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CCA_ABI_VERSION 3

enum cca_status {
    CCA_OK = 0,
    CCA_ERR_INVALID_ARG = -1, /* null/misaligned pointer, bad size, N % g != 0, Hq % Hkv != 0 */
    CCA_ERR_UNSUPPORTED = -2, /* dtype/d combination not built, or the device is not sm_103 */
    CCA_ERR_CUDA = -3,        /* a CUDA runtime/driver call or the launch failed */
    CCA_ERR_TIMEOUT = -4,     /* written to dev_status by a kernel that gave up waiting */
    CCA_ERR_SCRATCH_LIMIT = -5 /* cca_decode_fwd_noalloc: shapes exceed its fixed scratch */
};

enum cca_dtype {
    CCA_BF16 = 0, /* bfloat16 storage, fp32 accumulation */
    CCA_F32 = 1   /* float32 storage and arithmetic */
};

typedef struct cca_params {
    int32_t B;          /* batch                                  >= 1 */
    int32_t Hq;         /* query heads                            >= 1, multiple of Hkv */
    int32_t Hkv;        /* key/value heads                        >= 1 */
    int32_t N;          /* tokens per sequence                    >= 1, multiple of g */
    int32_t d;          /* head dimension: 64 or 128 (bf16 attention: 128 only) */
    int32_t g;          /* group size                             >= 1 */
    int32_t w;          /* local window                           >= 1 (w >= N allowed) */
    int32_t dtype;      /* enum cca_dtype */
    float scale;        /* softmax scale; <= 0 selects 1/sqrt(d) */
    int32_t *dev_status;/* optional device int32, see "Errors" above */
    int32_t window_mode;/* 0: raw window [lo(i), i] (the method as read here);
                           1: raw window [g*(lo(i)/g), i], reaching back to the group boundary
                              so that cores + window cover every earlier token */
    int32_t pool_mode;  /* 0: softmax weights of the group-last query (the method; with
                              grouped-query attention the r heads' logits are averaged
                              before the softmax);
                           1: mean pooling; 2: element-wise max pooling (the pages' ablations);
                           3: grouped-query pooling averaged after the softmax: each of the
                              r = Hq/Hkv query heads takes its own softmax over the group,
                              scored by its own group-last query, and the group weights are
                              the mean of the r weight vectors (the OpenReview rebuttal's
                              GQA answer leaves this choice open).  Equals 0 when r = 1.
                              Needs r <= 8 (else CCA_ERR_UNSUPPORTED). */
} cca_params_t;

/*
 * cca_pool - global-aware pooling (pooling equation of the Method section).
 * Reads Q (only the last token of every group is used), K and V; writes
 * Kc[b, kv, j, :] = sum_t a_t K[b, kv, j*g + t, :] and the same for Vc, with
 * a = softmax_t(tau * mean_{h in kv} Q[b, h, (j+1)*g - 1, :] . K[b, kv, j*g + t, :]).
 * Supported: dtype bf16 or f32, d in {64, 128}, any g >= 1.
 */
int cca_pool(const void *Q, const void *K, const void *V, void *Kc, void *Vc,
             const cca_params_t *params, void *stream);

/*
 * cca_attn_fwd - fused core/local attention (fusion equation of the Method
 * section).  For every (b, h, i): one softmax over the logits tau*Q_i.Kc_j for
 * visible cores j < lo(i)/g followed by tau*Q_i.K_m for m in [lo(i), i];
 * O_i = the softmax-weighted sum of the matching Vc_j and V_m rows;
 * LSE_i = log-sum-exp of the same logits.  Kc/Vc are the outputs of cca_pool
 * (or any caller-supplied core tokens of that shape).
 * Supported: bf16 with d = 128 (tensor-core kernel), f32 with d in {64, 128}.
 */
int cca_attn_fwd(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                 void *O, float *LSE, const cca_params_t *params, void *stream);

/*
 * cca_attn_fwd_rows - cca_attn_fwd for the query rows [q_off, q_off + n_q) of a
 * sequence of params->N tokens, reading only the raw tokens [kv_off, kv_off +
 * n_kv).  This is the attention of one shard when a sequence is split across
 * ranks along its length: pooling is group-local, so each rank pools its own
 * whole groups; the ranks then share their core tokens (all N/g of them) and
 * each receives the raw rows its first windows reach back to from the ranks
 * before it.  Rows keep their indices in the whole sequence: visibility, cores
 * and windows are exactly those of cca_attn_fwd over N tokens.
 *   Q, O   [B, Hq, n_q, d]     the rows q_off .. q_off + n_q - 1
 *   LSE    [B, Hq, n_q]        fp32
 *   K, V   [B, Hkv, n_kv, d]   the raw tokens kv_off .. kv_off + n_kv - 1
 *   Kc, Vc [B, Hkv, N/g, d]    core tokens of the whole sequence; rows below
 *                              lo(q_off + n_q - 1)/g must be valid
 * Requirements (else CCA_ERR_INVALID_ARG, nothing launched): n_q >= 1,
 * 0 <= kv_off <= first raw token of row q_off's window (lo(q_off), or its
 * group boundary with window_mode 1), q_off + n_q <= kv_off + n_kv <= N.
 * Everything else (support, alignment, errors) as cca_attn_fwd; with q_off = 0,
 * kv_off = 0 and n_q = n_kv = N it is cca_attn_fwd.
 */
int cca_attn_fwd_rows(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                      void *O, float *LSE, int q_off, int n_q, int kv_off, int n_kv,
                      const cca_params_t *params, void *stream);

/*
 * Decoding (one new token per sequence).  The pages describe a decode step that
 * keeps only the core tokens plus the local window in the KV cache and pools a
 * group once it has filled (news write-up, efficiency and KV-cache paragraphs;
 * OpenReview rebuttal, cache-size answer).  Here a decode step at position
 * `pos` computes exactly row `pos` of cca_attn_fwd over the caches.
 *
 * cca_decode_fwd - for every (b, h): one softmax over the visible cores
 * j < lo(pos)/g followed by the window tokens [lo(pos), pos], lo(pos) =
 * max(0, pos - w + 1).
 *   Q      [B, Hq, d]          query of the token at position pos
 *   K, V   [B, Hkv, Ncap, d]   caches; rows [lo(pos), pos] must be valid
 *   Kc, Vc [B, Hkv, Ncap/g, d] core caches; rows [0, lo(pos)/g) must be valid
 *   O      [B, Hq, d]          output (dtype of Q);  LSE [B, Hq] fp32
 *   params.N = Ncap (cache capacity, a multiple of g); 0 <= pos < Ncap.
 *   workspace: caller-owned device buffer of at least
 *   cca_decode_workspace_size(params) bytes (per-split partial results); it
 *   needs no initialisation and is fully rewritten by every call.
 * The keys are split across CTAs (flash-decoding).  For long visible lists
 * with enough (b, kv) pairs to fill the GPU, the splits of each (b, kv) form a
 * thread-block cluster and merge in it: one kernel, the workspace unused.
 * Otherwise the partial results are merged by a second kernel on the same
 * stream.  The kernels are launched as programmatic dependents: the split
 * kernel of whatever the stream ran before the call, the merge of the split
 * kernel.  Each may be scheduled while the
 * grid before it drains, and waits on the device for that grid's completion
 * before it reads anything, so the stream order is kept.  The merge lets its
 * own programmatic dependents (the next decode step's split kernel, say) be
 * scheduled once the split grid has completed.
 * Supported: bf16 or f32, d in {64, 128}, Hq/Hkv <= 8.
 */
int cca_decode_fwd(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc, void *O,
                   float *LSE, int pos, const cca_params_t *params, void *workspace,
                   uint64_t workspace_bytes, void *stream);

/* Kernels one cca_decode_fwd (or _noalloc) call at `pos` launches on the current
 * device: 1 when the splits of each (b, kv) merge inside a thread-block cluster
 * (long visible lists with enough (b, kv) pairs to fill the GPU), 2 for the
 * split kernel and its merge kernel; a negative status on bad arguments. */
int cca_decode_kernels(const cca_params_t *params, int pos);

/* Bytes of workspace cca_decode_fwd needs for these shapes (0 on bad params). */
uint64_t cca_decode_workspace_size(const cca_params_t *params);

/*
 * cca_decode_fwd_noalloc - cca_decode_fwd for callers that cannot allocate
 * device memory.  The pages have no counterpart: this entry point exists for
 * deployments in which this library may not obtain memory of its own, e.g. a
 * plug-in inside a host framework that owns every device allocation through
 * its own pool, a serving loop whose memory budget is fixed at start-up, or a
 * caller that must avoid cudaMalloc's implicit device-wide synchronisation in
 * its decode loop.  Such a caller can still pass its inputs and outputs, but
 * not a workspace.
 *
 * Same arguments, semantics and support as cca_decode_fwd, minus the
 * workspace: the per-split partial results live in one fixed array of
 * CCA_DECODE_NOALLOC_MAX_BYTES inside the library's device code, which every
 * GPU that loads the library holds until the process exits.  Shapes whose
 * cca_decode_workspace_size() exceeds that maximum are rejected with
 * CCA_ERR_SCRATCH_LIMIT before anything is launched.  The function calls no
 * cudaMalloc/cudaFree and no allocating library routine.
 *
 * The first call on a device (with that device current) looks up the array's
 * device address with cudaGetSymbolAddress; make that first call before any
 * stream capture.  The address is kept together with the CUDA context that was
 * current then; a call made under another context (after cudaDeviceReset, for
 * instance) looks it up again, and is then such a first call.  All calls share the one array: calls whose kernels may
 * overlap on a GPU (different streams without ordering) race on it and give
 * undefined results.  Nothing in it needs to start at zero: every call
 * rewrites each partial it later reads.
 */
#define CCA_DECODE_NOALLOC_MAX_BYTES (4ull << 20)
int cca_decode_fwd_noalloc(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                           void *O, float *LSE, int pos, const cca_params_t *params, void *stream);

/*
 * cca_pool_group - pool one newly completed group j of the caches (the
 * pooling equation for a single group): for every (b, kv),
 *   Kc[b, kv, j] = sum_t a_t K[b, kv, j*g + t],  Vc likewise,
 *   a = softmax_t(tau * mean_{h in kv} q[b, h] . K[b, kv, j*g + t]),
 * where q [B, Hq, d] is the query of the group's last token (j+1)*g - 1, i.e.
 * the token just decoded.  K, V [B, Hkv, Ncap, d]; Kc, Vc [B, Hkv, Ncap/g, d];
 * params.N = Ncap; 0 <= j < Ncap/g.  Same support as cca_pool.
 */
int cca_pool_group(const void *q, const void *K, const void *V, void *Kc, void *Vc, int j,
                   const cca_params_t *params, void *stream);

/*
 * cca_prefill_bwd - backward pass of CCA prefill (pooling + fused attention):
 * gradients of the loss sum(dO * O) with respect to Q, K and V.  The pages
 * fine-tune CCA models ("differentiable fusion", digest page; fine-tuning
 * settings, OpenReview rebuttal); this is the gradient of the two equations.
 *   Q, K, V, Kc, Vc  the forward's inputs and core tokens (dtype of params)
 *   O, LSE           the forward's outputs (cca_attn_fwd)
 *   dO               [B, Hq, N, d] upstream gradient (dtype of params)
 *   dQ               [B, Hq, N, d]  fp32, overwritten
 *   dK, dV           [B, Hkv, N, d] fp32, overwritten (they include the paths
 *                    through the core tokens back into the pooled groups)
 *   workspace        caller-owned device buffer of at least
 *                    cca_prefill_bwd_workspace_size(params) bytes
 * All pooling and window modes are supported, d in {64, 128}, bf16 or f32.
 * Max pooling passes each element's gradient to the first row holding the
 * maximum.  bf16 with d = 128 computes the attention gradients on the tensor
 * cores (bf16 operands, fp32 accumulation, P and dS rounded to bf16 before
 * their products); every other case, and the pooling backward, runs on CUDA
 * cores in fp32 (with softmax or mean pooling at bf16, d = 128, the pooling
 * backward's share of each raw token's row is added as the tensor-core kernel
 * writes that row).  A kernel that gives up waiting writes CCA_ERR_TIMEOUT into
 * *params.dev_status when that pointer is set (4-byte aligned); the gradients
 * are then undefined.
 */
int cca_prefill_bwd(const void *Q, const void *K, const void *V, const void *Kc, const void *Vc,
                    const void *O, const float *LSE, const void *dO, float *dQ, float *dK, float *dV,
                    const cca_params_t *params, void *workspace, uint64_t workspace_bytes, void *stream);

/* Bytes of workspace cca_prefill_bwd needs (0 on bad params). */
uint64_t cca_prefill_bwd_workspace_size(const cca_params_t *params);

/*
 * cca_prefill_host - the whole prefill step (cca_pool, then cca_attn_fwd) on
 * HOST buffers: Q, K, V are copied to the device, pooled and attended, and O
 * (plus LSE, Kc, Vc when asked for) copied back.  The (batch, KV head) pairs
 * are independent problems (the pooling equation and the fusion equation of
 * the digest page, Method section, never mix them), so the call cuts them into
 * about eight slices of consecutive pairs and pipelines the slices over three
 * streams: copies in, kernels on `stream`, copies out.  The copies of one slice
 * overlap the kernels of another.
 *   hQ, hK, hV    host (or any UVA-addressable) [B,Hq,N,d] / [B,Hkv,N,d] inputs
 *   hO            host [B,Hq,N,d] output, dtype of params
 *   hLSE          host [B,Hq,N] fp32 output, or NULL to skip it
 *   hKc, hVc      host [B,Hkv,N/g,d] outputs, or both NULL to skip them
 *   workspace     device buffer, 16-byte aligned, of at least
 *                 cca_prefill_host_workspace_size(params) bytes (three slice buffers)
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister): the
 * copies from and to pageable memory are correct, but the driver stages them
 * and the host may block on each, which removes the overlap.
 * The call returns once everything is enqueued.  Work is ordered after what is
 * already queued on `stream`, and `stream` resumes only after the last copy-out,
 * so synchronising `stream` makes every output valid on the host.  The internal
 * streams and events are kept per device for later calls.  Errors: as
 * cca_attn_fwd, checked before anything is enqueued; a CUDA failure after some
 * slices were enqueued returns CCA_ERR_CUDA with the outputs undefined.
 */
int cca_prefill_host(const void *hQ, const void *hK, const void *hV, void *hO, float *hLSE, void *hKc,
                     void *hVc, const cca_params_t *params, void *workspace, uint64_t workspace_bytes,
                     void *stream);

/* Device bytes of workspace cca_prefill_host needs (0 on bad params). */
uint64_t cca_prefill_host_workspace_size(const cca_params_t *params);

/* Static English text for a status code (never NULL). */
const char *cca_status_string(int status);

/* CCA_ABI_VERSION of the loaded library. */
int cca_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CCA_H_ */
