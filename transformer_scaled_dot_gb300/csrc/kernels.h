// kernels.h -- internal launch interface between the C ABI layer (api.cu)
// and the kernels. Not installed; the public surface is include/tsd_attention.h.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tsd {

constexpr int kMaskCausal = 1;
constexpr int kMaskKeyPadding = 2;

// One attention problem: Q/K/V/O addressed as (batch, head, row, col) with
// element strides; the head dimension is contiguous.
struct AttnProblem {
  int B, h, n_q, n_k, d;
  int mask_kind;
  const int32_t* kv_lens;  // device, may be null without the padding bit
  float scale;             // logit factor (already resolved: never 0)
  uint16_t* out;
  int64_t o_sb, o_sh, o_sr;
  // restricted self-attention: query i sees keys [i - win_left, i + win_right]
  // (n_q == n_k); a negative bound is no bound
  int win_left = -1, win_right = -1;
};

// bf16 tcgen05 attention; tensor maps describe Q, K, V and the output O as
// 4-D (d, rows, heads, batch) bf16 tensors with 128-byte swizzled 64x128 boxes.
cudaError_t launch_attn_bf16(const AttnProblem& p, const CUtensorMap& tm_q,
                             const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const CUtensorMap& tm_o, cudaStream_t stream);

struct AttnF32Problem {
  const float* q;
  const float* k;
  const float* v;
  float* out;
  int B, h, n_q, n_k, d_k, d_v;
  int mask_kind;
  const int32_t* kv_lens;
  float scale;
};
cudaError_t launch_attn_f32(const AttnF32Problem& p, cudaStream_t stream);

// Projection GEMM geometry shared with the host-side tensor maps.
constexpr int kGemmBK = 64;  // K rows per pipeline stage

// Grouped bf16 GEMM C_g[M_g, N_g] = A_g[M_g, K] * B_g[K, N_g] (fp32 accumulate,
// bf16 out). A is K-major (row-major [M, K]); B is N-major (row-major [K, N],
// the x.W weight layout). Up to 3 groups share K and run in one launch.
struct GemmGroup {
  CUtensorMap tm_a;  // 2-D (K, M), box 64 x 128
  CUtensorMap tm_b;  // 2-D (N, K), box 64 x kGemmBK
  CUtensorMap tm_c;  // 2-D (N, M), box 64 x 128 (TMA store of the output tile)
  uint16_t* c;
  int64_t ldc;       // elements
  int M, N;
  int tiles_m, tiles_n, tile_begin;
  // optional epilogue, one of: + bias[col] (bf16 [N]) then max(0, .) (relu
  // set); or + bias[col] + residual_f32[row, col] (row stride ldr) written in
  // fp32 to c_f32 (row stride N) instead of bf16 through tm_c; or (ln_gamma
  // set, one group, N in {128, 256, 512, 1024}) + bias + residual_f32, then
  // LayerNorm over each row's N columns with ln_gamma, ln_beta (bf16 [N])
  // and ln_eps, bf16 through tm_c. N a multiple of 8. Every group of a launch
  // uses the same one.
  const uint16_t* bias;
  const float* residual_f32;
  int64_t ldr;
  int relu;
  float* c_f32;
  const uint16_t* ln_gamma;
  const uint16_t* ln_beta;
  float ln_eps;
};
constexpr int kMaxGemmGroups = 3;
struct GemmProblem {
  GemmGroup g[kMaxGemmGroups];
  int num_groups;
  int K;
  int total_tiles;
};
cudaError_t launch_gemm_bf16(const GemmProblem& p, cudaStream_t stream);

// Raises a kernel's dynamic shared-memory limit once per device and asks
// for the largest shared-memory carveout (else the occupancy query and the
// launch may assume a smaller one, and fewer CTAs share an SM). The
// attributes belong to the device's context, and setting them on every
// launch costs host time comparable to a short kernel. `done` holds one bit
// per device ordinal (ordinals past 63 set them every time).
// A kernel whose warpgroups move registers between them (setmaxnreg) passes
// the per-thread count its split assumes at launch (`split_regs`): were the
// kernel built with fewer, an increase could wait forever for registers no
// one releases, so the launch is refused instead.
template <typename Kernel>
inline cudaError_t set_smem_once(Kernel kernel, int bytes, unsigned long long* done,
                                 int split_regs = 0) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0ull && (__atomic_load_n(done, __ATOMIC_ACQUIRE) & bit) != 0ull) return cudaSuccess;
  if (split_regs > 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < split_regs) return cudaErrorInvalidConfiguration;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && bit != 0ull) __atomic_fetch_or(done, bit, __ATOMIC_RELEASE);
  return e;
}

// Launches `kernel` on `stream` with programmatic stream serialization: it
// may begin (prologue only: barrier set-up, tensor-memory allocation) while
// the kernel ahead of it finishes. The kernels call griddep_wait() before
// their first global-memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Multi-head attention for short sequences in one kernel up to the merged
// heads: the Q/K/V projections of each head pair, their attention, and the
// merged [B, n_q, h*64] output. n_q, n_k <= 128, d_k = d_v = 64, h even,
// d_model a multiple of 64. With `out`, the same launch also applies W_O
// (clusters of h/2 CTAs, h/2 <= 8, d_model / (h/2) = 64 or 128), writing
// `out` [B, n_q, d_model]; the merged buffer is then its scratch.
struct MhaFusedProblem {
  CUtensorMap tm_xq;   // 3-D (d_model, n_q, B), box 64 x 128 x 1
  CUtensorMap tm_xkv;  // 3-D (d_model, n_k, B) (unused when self)
  CUtensorMap tm_xkv_tail;  // the same tensor, box 64 x 64 x 1 (cross-attention past 128 keys)
  CUtensorMap tm_wq, tm_wk, tm_wv;  // 2-D (h*64, d_model), box 64 x 64
  CUtensorMap tm_o;    // 3-D (h*64, n_q, B), box 64 x 128 x 1 (TMA store, and load with out)
  CUtensorMap tm_wo;   // 2-D (d_model, h*64), box 64 x 64 (out only)
  CUtensorMap tm_out;  // 3-D (d_model, n_q, B), box 64 x 128 x 1 (out only)
  int B, h, n_q, n_k, d_model;
  bool self;           // x_kv is x_q (and n_k == n_q)
  bool out;            // apply W_O too
  int mask_kind;
  const int32_t* kv_lens;
  float scale;
};
cudaError_t launch_mha_fused(const MhaFusedProblem& p, cudaStream_t stream);
// Clusters of h/2 output-projecting CTAs that fit on the device at once (0:
// the output projection cannot be fused).
int mha_fused_out_clusters(int h, bool self);
// Cross-attention (x_kv is not x_q) with 128 < n_k <= 192 source rows, n_q <=
// 128, d_k = d_v = 64, h even, d_model a multiple of 64: the same problem
// description and outputs as launch_mha_fused, in one launch (the source's
// rows past 128 projected transposed, then the online softmax over the first
// key tile and that tail).
cudaError_t launch_mha_cross(const MhaFusedProblem& p, cudaStream_t stream);
int mha_cross_out_clusters(int h);

// Per-file device error words (read and cleared; see sm103.cuh).
// One decoding step against a key/value cache: the n_q (<= 8) newest tokens'
// queries, at positions L - n_q .. L - 1 of an L-row cache, each against the
// keys at or before its position. Split over 128-key chunks (partials in a
// workspace of float), then merged per (batch, head).
constexpr int kDecodeMaxQueries = 8;
constexpr int kDecodeMaxChunks = 1024;  // n_max <= 1024 * 128 = 131072
struct DecodeProblem {
  CUtensorMap tm_k, tm_v;      // 3-D (d, n_max, B*h) bf16, box 64 x 128 x 1, 128-byte swizzle
  const void* q;               // [B, h, n_q, d] bf16
  void* out;                   // [B, h, n_q, d] bf16
  const int32_t* cache_lens;   // [B] valid rows, or null (= n_max)
  float* ws_o;                 // [B, h, decode_chunks(n_max), n_q, d]
  float* ws_ml;                // [B, h, decode_chunks(n_max), n_q, 2]
  int B, h, n_q, n_max, d;
  float scale;                 // logit factor (resolved: never 0)
};
int decode_chunks(int n_max);
cudaError_t launch_decode(const DecodeProblem& p, cudaStream_t stream);

// out = LayerNorm(x + r) over rows of d_model (256, 512, 1024 or 2048)
// features: x bf16 (or fp32 when x_f32), r bf16 or null, gamma/beta bf16,
// out bf16 and, when out32 is not null, the same values in fp32 as well.
cudaError_t launch_add_layernorm(const void* x, bool x_f32, const uint16_t* r,
                                 const uint16_t* gamma, const uint16_t* beta, uint16_t* out,
                                 float* out32, int rows, int d_model, float eps,
                                 cudaStream_t stream);

cudaError_t take_device_error_attn(unsigned int* value);
cudaError_t take_device_error_decode(unsigned int* value);
cudaError_t take_device_error_gemm(unsigned int* value);
cudaError_t take_device_error_f32(unsigned int* value);
cudaError_t take_device_error_fused(unsigned int* value);
cudaError_t take_device_error_cross(unsigned int* value);

// Failure-detection self test: a bounded wait on a barrier nobody arrives on.
cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, cudaStream_t stream);

}  // namespace tsd
