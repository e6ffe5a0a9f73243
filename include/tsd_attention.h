/*
 * tsd_attention.h -- C ABI of the GB300 (sm_103a) multi-head scaled
 * dot-product attention library (libtsd_attention.so).
 *
 * The operation is eq. (1) of "Attention Is All You Need",
 *     Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V,
 * a query mapped against a set of key/value pairs to a weighted sum of the
 * values ("[논문 리뷰]Attention Is All You Need" (kimjiil.github.io),
 * section 3.2 / 3.2.1), applied per head, and multi-head attention
 *     MultiHead = Concat(head_1..head_h) W^O,
 *     head_i = Attention(X_q W_i^Q, X_kv W_i^K, X_kv W_i^V)
 * (same page, section 3.2.2). Masks set the illegal logits to -inf before
 * the softmax so their weight is exactly 0 (same page, section 3.2.3;
 * "Attention Is All You Need 해부" (sj-techlog), section "mask는 softmax
 * **전**에 더해야 한다").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never frees, retains or allocates device memory on a call. Every call is
 *    asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream) and returns before the GPU work finishes.
 *  - Layouts are row-major and contiguous. bf16 tensors hold IEEE bfloat16
 *    bit patterns (uint16); f32 tensors hold IEEE binary32.
 *  - Host-detected argument errors return before anything is launched.
 *  - kv_lens values are clamped on the device to [0, n_k]. A query row with
 *    no allowed key (kv_len = 0) produces an all-zero output row.
 *  - Kernels never trap or assert. Every wait inside a kernel is bounded;
 *    a kernel that gives up sets a device error word and exits cleanly,
 *    which attn_get_device_status() reports. A kernel whose warp groups
 *    trade registers is not launched when the build gave it fewer registers
 *    per thread than that trade assumes (ATTN_ERR_CUDA,
 *    cudaErrorInvalidConfiguration): it could otherwise wait for registers
 *    that are never released.
 */
#ifndef TSD_ATTENTION_H
#define TSD_ATTENTION_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without pulling in the CUDA headers. */
typedef struct CUstream_st *tsd_stream_t;

typedef enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = 1,        /* an argument is invalid; nothing was launched */
    ATTN_ERR_UNSUPPORTED = 2,    /* valid for eq. (1) but outside what this build runs
                                    (e.g. a head size the bf16 kernel has no variant for) */
    ATTN_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed; see attn_last_cuda_error() */
    ATTN_ERR_DEVICE_TIMEOUT = 4  /* a kernel's bounded wait ran out (attn_get_device_status) */
} attn_status;

/* mask_kind bit flags */
enum {
    ATTN_MASK_NONE = 0,
    ATTN_MASK_CAUSAL = 1,       /* query i sees keys j <= i; requires n_q == n_k
                                   (decoder masked self-attention, section 3.2.3) */
    ATTN_MASK_KEY_PADDING = 2   /* keys j >= kv_lens[b] receive no attention
                                   ("Attention Is All You Need 해부", three-uses table) */
};

/*
 * attn_forward -- scaled dot-product attention, bf16 in/out, fp32 softmax and
 * accumulation, on the tcgen05 tensor cores.
 *
 *   q    [B, h, n_q, d_k]  bf16, device, 16-byte aligned
 *   k    [B, h, n_k, d_k]  bf16, device, 16-byte aligned
 *   v    [B, h, n_k, d_v]  bf16, device, 16-byte aligned
 *   out  [B, h, n_q, d_v]  bf16, device, 16-byte aligned, written in full
 *   d_k == d_v, and d_k in {16, 32, 64, 128, 256}   else ATTN_ERR_UNSUPPORTED
 *     (16, 32 and 256 are the head sizes of Table 3 (A), "[논문 리뷰]Attention
 *     Is All You Need" (kimjiil.github.io), section 6.2; 64 is the base model's)
 *   B, h, n_q, n_k >= 0                      else ATTN_ERR_INVALID
 *     (a zero size launches nothing; n_k = 0 writes all-zero output rows)
 *   mask_kind: OR of ATTN_MASK_* bits; CAUSAL needs n_q == n_k
 *   kv_lens: device int32[B]; required with ATTN_MASK_KEY_PADDING, ignored otherwise
 *   scale: the logit factor; 0 selects 1/sqrt(d_k) (eq. (1))
 * Errors: null/misaligned pointer, bad sizes or flags -> ATTN_ERR_INVALID;
 * a failed launch -> ATTN_ERR_CUDA.
 */
attn_status attn_forward(const void *q, const void *k, const void *v, void *out,
                         int B, int h, int n_q, int n_k, int d_k, int d_v,
                         int mask_kind, const int32_t *kv_lens, float scale,
                         tsd_stream_t stream);

/*
 * encoder_layer_forward -- one Transformer encoder layer, both sub-layers
 * wrapped post-LN as output = LayerNorm(x + Sublayer(x)) ("[논문 리뷰]
 * Attention Is All You Need" (kimjiil.github.io), sections 3.1 and 3.3;
 * LayerNorm(v) = gamma (v - mu) / sqrt(sigma^2 + eps) + beta over one token's
 * d_model features, "Attention Is All You Need 해부" (sj-techlog), section
 * "4. residual connection과 LayerNorm"):
 *   y   = LayerNorm_1(x + MultiHead(x, x))            (mha_forward, self-attention)
 *   out = LayerNorm_2(y + FFN(y)),  FFN(y) = max(0, y W_1 + b_1) W_2 + b_2
 *   x, out   [B, n, d_model] bf16, device; d_model in {256, 512, 1024, 2048}
 *            (else ATTN_ERR_UNSUPPORTED)
 *   w_q, w_k, w_v, w_o: as mha_forward with d_v = d_k (d_model x h*d_k, h*d_k x d_model)
 *   ln1_gamma, ln1_beta, ln2_gamma, ln2_beta: [d_model] bf16
 *   w_1 [d_model, d_ff], b_1 [d_ff], w_2 [d_ff, d_model], b_2 [d_model], bf16;
 *   d_ff a multiple of 8
 *   mask_kind, kv_lens, scale: as mha_forward (self-attention, n_q = n_k = n)
 *   eps: LayerNorm's epsilon (> 0; the pages do not give a value)
 *   workspace: device, 256-byte aligned, >= encoder_layer_workspace_bytes(...)
 *   bytes; scratch (it holds mha_forward's workspace, the attention output,
 *   y, the FFN's hidden layer and y + FFN(y)).
 * Errors: as mha_forward; eps <= 0 -> ATTN_ERR_INVALID. Launches: mha_forward's
 * plus four (LayerNorm, the two FFN GEMMs with their bias / ReLU / residual
 * epilogues, LayerNorm).
 */
size_t encoder_layer_workspace_bytes(int B, int n, int d_model, int h, int d_k, int d_ff);
attn_status encoder_layer_forward(const void *x,
                                  const void *w_q, const void *w_k, const void *w_v,
                                  const void *w_o,
                                  const void *ln1_gamma, const void *ln1_beta,
                                  const void *w_1, const void *b_1,
                                  const void *w_2, const void *b_2,
                                  const void *ln2_gamma, const void *ln2_beta,
                                  void *out,
                                  int B, int n, int d_model, int h, int d_k, int d_ff,
                                  int mask_kind, const int32_t *kv_lens, float scale, float eps,
                                  void *workspace, size_t workspace_bytes, tsd_stream_t stream);

/*
 * attn_decode -- one decoding step against a key/value cache ("Attention Is
 * All You Need 해부" (sj-techlog), section "KV cache는 추론의 같은 계산을
 * 반복하지 않게 한다"; "[논문 리뷰]Attention Is All You Need"
 * (kimjiil.github.io), section 3.7): only the newest tokens' queries are
 * computed; the keys and values of every position so far (theirs included)
 * come from the cache. With L = cache_lens[b] valid rows, query t sits at
 * position L - n_q + t and attends to the keys at positions <= its own (the
 * causal rule aligned to the end of the cache); a query at a negative
 * position sees no key and gets 0.
 *   q        [B, h, n_q, d_k] bf16, device        out [B, h, n_q, d_v] bf16
 *   k_cache  [B, h, n_max, d_k] bf16, device      v_cache [B, h, n_max, d_v]
 *   cache_lens: device int32[B] (clamped to [0, n_max]), or NULL for L = n_max
 *   1 <= n_q <= 8 and n_max <= 131072 (more -> ATTN_ERR_UNSUPPORTED);
 *   d_k == d_v in {64, 128}.
 *   workspace: device, 16-byte aligned, >= attn_decode_workspace_bytes(...)
 *   bytes (per-chunk partial results; scratch, caller-owned).
 *   scale: 0 -> 1/sqrt(d_k). Cache rows at or past L are never used.
 * Errors: as attn_forward; a short workspace -> ATTN_ERR_INVALID. Two
 * launches (per-chunk partials, then the merge), asynchronous on `stream`.
 */
size_t attn_decode_workspace_bytes(int B, int h, int n_q, int n_max, int d_v);
attn_status attn_decode(const void *q, const void *k_cache, const void *v_cache, void *out,
                        int B, int h, int n_q, int n_max, int d_k, int d_v,
                        const int32_t *cache_lens, float scale,
                        void *workspace, size_t workspace_bytes, tsd_stream_t stream);

/*
 * attn_forward_window -- restricted self-attention: query i considers only
 * the keys j with i - window_left <= j <= i + window_right ("[논문 리뷰]
 * Attention Is All You Need" (kimjiil.github.io), section "[4] Why
 * Self-Attention", Table 1, row "Self-Attention (restricted)": O(r n d) work
 * for a neighbourhood of r positions instead of O(n^2 d)). Table 1 sizes the
 * neighbourhood by r only; the bounds here are per side, so a neighbourhood
 * of size r centred on the query is window_left = window_right = (r - 1) / 2
 * and a radius-r window is window_left = window_right = r.
 *   Arguments, layouts, masks and errors as attn_forward, plus:
 *   window_left, window_right: >= 0, or -1 for no bound on that side
 *   (-1, -1 is attn_forward); < -1 -> ATTN_ERR_INVALID. A window needs
 *   n_q == n_k (query i and key i share a position), else ATTN_ERR_INVALID.
 *   The causal bit and key padding combine with the window; a row left with
 *   no key gets output 0. Key tiles outside every row's window are never
 *   loaded.
 */
attn_status attn_forward_window(const void *q, const void *k, const void *v, void *out,
                                int B, int h, int n_q, int n_k, int d_k, int d_v,
                                int mask_kind, const int32_t *kv_lens,
                                int window_left, int window_right,
                                float scale, tsd_stream_t stream);

/*
 * attn_forward_strided -- the same operation as attn_forward on tensors whose
 * (batch, head, row) strides are given in ELEMENTS (the head dimension stays
 * contiguous). This lets a caller read heads straight out of a [B, n, h*d]
 * projection output (head i = column block i, section 3.2.2) and write the
 * merged Concat(head_1..head_h) layout [B, n_q, h*d_v] without a copy.
 * Every stride must be a multiple of 8 elements (16 bytes); rows may not
 * overlap within a head. Other arguments and errors as attn_forward.
 */
attn_status attn_forward_strided(const void *q, int64_t q_sb, int64_t q_sh, int64_t q_sr,
                                 const void *k, int64_t k_sb, int64_t k_sh, int64_t k_sr,
                                 const void *v, int64_t v_sb, int64_t v_sh, int64_t v_sr,
                                 void *out, int64_t o_sb, int64_t o_sh, int64_t o_sr,
                                 int B, int h, int n_q, int n_k, int d_k, int d_v,
                                 int mask_kind, const int32_t *kv_lens, float scale,
                                 tsd_stream_t stream);

/*
 * attn_forward_f32 -- the same operation in fp32 throughout (FFMA, no TF32),
 * for callers that need results within 1e-4 of exact.
 *   q [B,h,n_q,d_k], k [B,h,n_k,d_k], v [B,h,n_k,d_v], out [B,h,n_q,d_v]: f32, device.
 *   1 <= d_k, d_v <= 128. Other arguments and errors as attn_forward.
 */
attn_status attn_forward_f32(const float *q, const float *k, const float *v, float *out,
                             int B, int h, int n_q, int n_k, int d_k, int d_v,
                             int mask_kind, const int32_t *kv_lens, float scale,
                             tsd_stream_t stream);

/*
 * mha_workspace_bytes -- size of the caller-owned device workspace that
 * mha_forward needs for the head-split projections Q, K, V and the merged
 * heads Concat(head_1..head_h) (bf16, each region 256-byte aligned).
 * Returns 0 for invalid sizes.
 */
size_t mha_workspace_bytes(int B, int n_q, int n_k, int h, int d_k, int d_v);

/*
 * mha_forward -- multi-head attention, section 3.2.2 (x.W convention, no
 * biases, as in the pages' formula):
 *   Q = x_q W_Q, K = x_kv W_K, V = x_kv W_V        (tensor-core GEMMs)
 *   head_i = Attention(Q_i, K_i, V_i)              (attn kernel; Q_i = column block i)
 *   out = Concat(head_1..head_h) W_O               (tensor-core GEMM)
 * Short sequences run all three in one or two kernels (mha_forward_launches).
 *
 *   x_q  [B, n_q, d_model] bf16      x_kv [B, n_k, d_model] bf16 (may equal x_q)
 *   w_q  [d_model, h*d_k]  bf16      w_k  [d_model, h*d_k]  bf16
 *   w_v  [d_model, h*d_v]  bf16      w_o  [h*d_v, d_model]  bf16
 *   out  [B, n_q, d_model] bf16
 *   d_k == d_v in {64, 128}; d_model a multiple of 8 (16-byte rows), >= 8.
 *   workspace: device, 256-byte aligned, >= mha_workspace_bytes(...) bytes;
 *   on return its last region holds the merged heads; the Q, K, V regions
 *   are scratch (short sequences -- n_q, n_k <= 128, d_k = d_v = 64, h even,
 *   d_model a multiple of 64 -- are projected and attended in one kernel
 *   and never write them; so is cross-attention, x_kv != x_q, with
 *   n_q <= 128 and 128 < n_k <= 192 source rows, the encoder-decoder
 *   attention of section 3.2.3 at the Transformer-base lengths). With
 *   thread-block clusters in flight, the
 *   merged-heads region is how the CTAs of one batch entry share their
 *   heads: calls running concurrently need distinct workspaces.
 *   mask_kind, kv_lens, scale: as attn_forward (the mask applies to every head).
 * Errors: as attn_forward; a short workspace -> ATTN_ERR_INVALID.
 */
attn_status mha_forward(const void *x_q, const void *x_kv,
                        const void *w_q, const void *w_k, const void *w_v, const void *w_o,
                        void *out,
                        int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                        int mask_kind, const int32_t *kv_lens, float scale,
                        void *workspace, size_t workspace_bytes, tsd_stream_t stream);

/*
 * mha_forward_launches -- how many kernels mha_forward launches for these
 * sizes on the current device (a planning query: no launch, no allocation;
 * it may ask the runtime how many thread-block clusters fit):
 *   1  short sequences, W_O applied in the same kernel (n_q, n_k <= 128, or
 *      cross-attention with n_q <= 128 and n_k <= 192; d_k = d_v = 64, h even,
 *      h/2 <= 8, d_model / (h/2) = 64 or 128, and a cluster of h/2 CTAs fits
 *      on the device);
 *   2  short sequences, then the W_O GEMM;
 *   3  the Q/K/V projection GEMM, the attention kernel, the W_O GEMM;
 *   0  nothing to do (B * n_q == 0);  -1  sizes mha_forward rejects.
 * self_attention: nonzero when x_kv will be passed equal to x_q.
 */
int mha_forward_launches(int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                         int self_attention);

/*
 * mha_concat_heads -- Concat(head_1, ..., head_h), head_i =
 * Attention(X_q W_i^Q, X_kv W_i^K, X_kv W_i^V): multi-head attention up to
 * (not including) the output projection W_O ("[논문 리뷰]Attention Is All You
 * Need" (kimjiil.github.io), section 3.2.2). mha_forward is this followed by
 * mha_project_out.
 *   Arguments and errors as mha_forward, with `concat` in place of w_o/out:
 *   concat: device bf16 [B, n_q, h*d_v] (head i = column block i), 16-byte
 *   aligned. The workspace (mha_workspace_bytes(...) bytes, 256-byte aligned)
 *   is scratch for the Q, K, V projections; short sequences (n_q, n_k <= 128,
 *   d_k = d_v = 64, h even, d_model a multiple of 64) run as one fused kernel
 *   and leave it untouched.
 */
attn_status mha_concat_heads(const void *x_q, const void *x_kv,
                             const void *w_q, const void *w_k, const void *w_v, void *concat,
                             int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                             int mask_kind, const int32_t *kv_lens, float scale,
                             void *workspace, size_t workspace_bytes, tsd_stream_t stream);

/*
 * mha_project_qkv -- the input projections of section 3.2.2, all positions at
 * once, in one launch:
 *   q_out = x_q W_Q  [B, n_q, h*d_k],  k_out = x_kv W_K  [B, n_k, h*d_k],
 *   v_out = x_kv W_V [B, n_k, h*d_v]   (bf16, fp32 accumulation)
 * Head i of each result is its column block i, so the outputs feed
 * attn_forward_strided directly. Shapes, alignment and errors as mha_forward
 * (every pointer device, 16-byte aligned; d_model a multiple of 8).
 */
attn_status mha_project_qkv(const void *x_q, const void *x_kv,
                            const void *w_q, const void *w_k, const void *w_v,
                            void *q_out, void *k_out, void *v_out,
                            int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                            tsd_stream_t stream);

/*
 * mha_project_out -- the output projection of section 3.2.2:
 *   out [B, n_q, d_model] = Concat(head_1..head_h) [B, n_q, h*d_v] . W_O [h*d_v, d_model]
 * (bf16, fp32 accumulation). Errors as mha_forward.
 */
attn_status mha_project_out(const void *concat, const void *w_o, void *out,
                            int B, int n_q, int d_model, int h, int d_v, tsd_stream_t stream);

/*
 * mha_forward_noalloc -- mha_forward for callers that cannot allocate device
 * memory. The pages have no counterpart: this is a deployment variant.
 *
 * Who needs it: a plugin whose host application owns the device-memory budget
 * and forbids allocation inside the plugin; a serving loop whose memory is
 * planned up front and must not call cudaMalloc/cudaFree on the request path
 * (they synchronise the device and stall other streams); a plain C caller
 * with no access to its framework's caching allocator. Such callers cannot
 * provide mha_forward's workspace, so this entry point uses a fixed
 * file-scope device array of TSD_MHA_NOALLOC_SCRATCH_BYTES instead and calls
 * no cudaMalloc, cudaFree or other allocating routine. The caller still
 * passes every input and output.
 *
 *   Arguments, layouts and errors as mha_forward, without the workspace.
 *   mha_workspace_bytes(B, n_q, n_k, h, d_k, d_v) must not exceed
 *   TSD_MHA_NOALLOC_SCRATCH_BYTES, else ATTN_ERR_UNSUPPORTED (before any
 *   CUDA call).
 *
 * The array belongs to the library's device image: every GPU that loads the
 * library holds it until the process exits. The first call on a device, with
 * that device current, looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture. A failed look-up returns ATTN_ERR_CUDA.
 *
 * All calls on a device share the one array, which keeps the last call's
 * contents; calls that overlap on the GPU (other streams or host threads
 * without ordering between them) race on it. No clearing is needed between
 * calls: every byte a call reads from the array is written by that call.
 */
#define TSD_MHA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

attn_status mha_forward_noalloc(const void *x_q, const void *x_kv,
                                const void *w_q, const void *w_k, const void *w_v,
                                const void *w_o, void *out,
                                int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                                int mask_kind, const int32_t *kv_lens, float scale,
                                tsd_stream_t stream);

/*
 * Host-buffer entry points -- attn_forward, attn_forward_window, mha_forward,
 * encoder_layer_forward and attn_decode with the step's inputs and result
 * in HOST memory (the pages' operations unchanged; a deployment variant).
 * Each call copies its host inputs into staging regions at the front of
 * `workspace`, runs the device entry point on the staged copies on
 * `stream`, and copies the result back to the host on `stream`. Weights,
 * LayerNorm parameters and the key/value cache stay DEVICE pointers: they
 * are state that lives on the GPU between steps.
 *
 *   *_host arguments: host memory (pinned -- cudaHostAlloc or
 *   cudaHostRegister -- for the copies to be asynchronous; pageable memory
 *   works and is copied synchronously). Sizes, layouts, masks and errors as
 *   the device entry point; kv_lens / cache_lens are host int32[B] here.
 *   workspace: device, 256-byte aligned, >= the matching
 *   *_host_workspace_bytes(...) (0 for invalid sizes); a workspace serves
 *   one stream at a time and only these calls.
 *
 * Ordering. The input copies run on a copy stream the library creates once
 * per device (non-blocking), after the last computation that read the same
 * workspace's staging region; the computation waits for them. The result
 * copy is on `stream`, so once `stream` has passed the call, the result is
 * in host memory and the host inputs may be reused. A caller that passes
 * two workspaces in turn over consecutive calls overlaps call i+1's input
 * copy with call i's computation and result copy. The first call with a
 * workspace (or after the library's table of 64 workspaces evicted it)
 * orders its copy after everything already on `stream`. Calls are
 * serialised by a library-wide lock while they enqueue (microseconds).
 * Errors: every argument error returns before anything is copied; a failed
 * copy or stream operation returns ATTN_ERR_CUDA.
 */
size_t attn_host_workspace_bytes(int B, int h, int n_q, int n_k, int d_k, int d_v);
attn_status attn_forward_host(const void *q_host, const void *k_host, const void *v_host,
                              void *out_host,
                              int B, int h, int n_q, int n_k, int d_k, int d_v,
                              int mask_kind, const int32_t *kv_lens_host, float scale,
                              void *workspace, size_t workspace_bytes, tsd_stream_t stream);

/* attn_forward_window with host q, k, v, out; the workspace as attn_forward_host's. */
attn_status attn_forward_window_host(const void *q_host, const void *k_host, const void *v_host,
                                     void *out_host,
                                     int B, int h, int n_q, int n_k, int d_k, int d_v,
                                     int mask_kind, const int32_t *kv_lens_host,
                                     int window_left, int window_right, float scale,
                                     void *workspace, size_t workspace_bytes,
                                     tsd_stream_t stream);

size_t mha_host_workspace_bytes(int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v);
/* x_kv_host == x_q_host (with n_q == n_k) is self-attention: x is copied once. */
attn_status mha_forward_host(const void *x_q_host, const void *x_kv_host,
                             const void *w_q, const void *w_k, const void *w_v, const void *w_o,
                             void *out_host,
                             int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                             int mask_kind, const int32_t *kv_lens_host, float scale,
                             void *workspace, size_t workspace_bytes, tsd_stream_t stream);

/*
 * mha_forward_host_async -- mha_forward_host whose result copy runs on a
 * device-to-host stream the library creates once per device, after the
 * computation, instead of on `stream`: consecutive calls (two workspaces in
 * turn) then overlap call i's result copy with call i+1's computation, as a
 * serving loop wants. A call's result is in out_host, and its host inputs
 * may be reused, once `stream` has passed a later attn_host_join(stream).
 * A workspace's next computation waits for the result copy that last read
 * it. Arguments and errors as mha_forward_host.
 */
attn_status mha_forward_host_async(const void *x_q_host, const void *x_kv_host,
                                   const void *w_q, const void *w_k, const void *w_v,
                                   const void *w_o, void *out_host,
                                   int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                                   int mask_kind, const int32_t *kv_lens_host, float scale,
                                   void *workspace, size_t workspace_bytes, tsd_stream_t stream);

/* attn_host_join -- `stream` waits for every result copy the asynchronous
 * host-buffer calls issued so far on the current device (none: a no-op). */
attn_status attn_host_join(tsd_stream_t stream);

size_t encoder_layer_host_workspace_bytes(int B, int n, int d_model, int h, int d_k, int d_ff);
attn_status encoder_layer_forward_host(const void *x_host,
                                       const void *w_q, const void *w_k, const void *w_v,
                                       const void *w_o,
                                       const void *ln1_gamma, const void *ln1_beta,
                                       const void *w_1, const void *b_1,
                                       const void *w_2, const void *b_2,
                                       const void *ln2_gamma, const void *ln2_beta,
                                       void *out_host,
                                       int B, int n, int d_model, int h, int d_k, int d_ff,
                                       int mask_kind, const int32_t *kv_lens_host, float scale,
                                       float eps, void *workspace, size_t workspace_bytes,
                                       tsd_stream_t stream);
/* encoder_layer_forward_host_async -- encoder_layer_forward_host whose
 * result copy runs on the library's device-to-host stream, as
 * mha_forward_host_async: out_host is complete, and may be reused, once
 * `stream` has passed a later attn_host_join(stream). Arguments and errors as
 * encoder_layer_forward_host. */
attn_status encoder_layer_forward_host_async(const void *x_host,
                                             const void *w_q, const void *w_k, const void *w_v,
                                             const void *w_o,
                                             const void *ln1_gamma, const void *ln1_beta,
                                             const void *w_1, const void *b_1,
                                             const void *w_2, const void *b_2,
                                             const void *ln2_gamma, const void *ln2_beta,
                                             void *out_host,
                                             int B, int n, int d_model, int h, int d_k, int d_ff,
                                             int mask_kind, const int32_t *kv_lens_host,
                                             float scale, float eps, void *workspace,
                                             size_t workspace_bytes, tsd_stream_t stream);

size_t attn_decode_host_workspace_bytes(int B, int h, int n_q, int n_max, int d_k, int d_v);
/* q_host [B, h, n_q, d_k] and out_host [B, h, n_q, d_v] on the host; the
 * caches are device memory; cache_lens_host: host int32[B] or NULL. */
attn_status attn_decode_host(const void *q_host, const void *k_cache, const void *v_cache,
                             void *out_host,
                             int B, int h, int n_q, int n_max, int d_k, int d_v,
                             const int32_t *cache_lens_host, float scale,
                             void *workspace, size_t workspace_bytes, tsd_stream_t stream);
/* attn_decode_host_async -- attn_decode_host whose result copy runs on the
 * library's device-to-host stream, as mha_forward_host_async: out_host is
 * complete, and may be reused, once `stream` has passed a later
 * attn_host_join(stream). Arguments and errors as attn_decode_host. */
attn_status attn_decode_host_async(const void *q_host, const void *k_cache,
                                   const void *v_cache, void *out_host,
                                   int B, int h, int n_q, int n_max, int d_k, int d_v,
                                   const int32_t *cache_lens_host, float scale,
                                   void *workspace, size_t workspace_bytes, tsd_stream_t stream);

/*
 * attn_get_device_status -- synchronises `stream`, then reads and clears the
 * device error word the kernels set when a bounded wait runs out.
 * Returns ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT, or ATTN_ERR_CUDA if the
 * synchronisation itself failed.
 */
attn_status attn_get_device_status(tsd_stream_t stream);

/* The last CUDA error code (cudaError_t as int) seen by this library on the
 * calling thread, 0 if none. */
int attn_last_cuda_error(void);

/* A static, human-readable name for a status code. */
const char *attn_status_string(attn_status s);

/*
 * attn_selftest_wait_timeout -- failure-detection self test. Launches one
 * small kernel whose bounded wait is on an mbarrier that nothing ever
 * arrives on, with a limit of `limit_us` microseconds (1..2000000). The
 * kernel records a timeout in the device error word and exits; the caller
 * reads it with attn_get_device_status(), and the context stays usable.
 * No tensor memory or asynchronous copy is involved.
 */
attn_status attn_selftest_wait_timeout(int limit_us, tsd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TSD_ATTENTION_H */
