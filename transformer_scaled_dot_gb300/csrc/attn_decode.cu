// attn_decode.cu -- one decoding step against a key/value cache: the queries
// of the n_q newest tokens (1..8) against every cached position
// ("Attention Is All You Need 해부" (sj-techlog), section "KV cache는 추론의
// 같은 계산을 반복하지 않게 한다": only the new token's Q is computed, K and V
// come from the cache of positions 0..t-1 plus the new token's own). With L
// valid cache rows the new tokens sit at positions L - n_q .. L - 1 and see
// the keys at or before their own position (the causal rule, aligned to the
// end of the cache).
//
// The step is bound by reading the cache (4 d bytes per key, 2 n_q d
// multiply-adds per key), so it runs on the FMA pipes, split over the keys:
//
//   decode_partial   one CTA per (batch, head, 128-key chunk): the chunk's K
//                    and V by TMA (128-byte swizzle, one box per 64 columns;
//                    32 KB at d = 64, so six CTAs share an SM and their loads
//                    and arithmetic overlap),
//                    a thread per key for the n_q scores (q broadcast from
//                    shared memory), the chunk's max and sum per query in
//                    fp32, P in shared memory, then O_chunk = P V with
//                    threads over (column pair, key group) and a reduction
//                    across the groups; writes m, l (base-2 exponent domain)
//                    and O_chunk (fp32) to the workspace
//   decode_merge     one CTA per (batch, head): m = max_c m_c,
//                    out = sum_c 2^(m_c - m) O_c / sum_c 2^(m_c - m) l_c, bf16
//                    (the O_c loads of a thread issued together, so the merge
//                    costs a few dependent L2 round trips)
//
// Chunks at or past L are neither computed nor read; keys at or past L in
// the last chunk are masked before they can reach a sum (the cache past L
// may hold anything).
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kChunk = 128;    // keys per CTA (one per thread in the score phase)
constexpr int kDecThreads = 128;
constexpr unsigned long long kDrainLimitNs = 100ull * 1000ull * 1000ull;

template <int D, int NQ>
struct DecSmem {
  static constexpr int kAtoms = D / 64;  // 64-column, 128-byte-swizzled boxes
  alignas(1024) uint8_t k[kAtoms][kChunk * 128];
  alignas(1024) uint8_t v[kAtoms][kChunk * 128];
  float p[NQ][kChunk];
  float q[NQ][D];
  float red_max[kDecThreads / 32][NQ];
  float red_sum[kDecThreads / 32][NQ];
  uint64_t full;
  uint32_t abort_flag;
  // the cross-group reduction of O reuses k: (groups x NQ x D) floats
  static_assert((kDecThreads / (D / 2)) * NQ * D * 4 <= kAtoms * kChunk * 128, "reduction fits");
};

struct DecodeArgs {
  const __nv_bfloat16* q;  // [B, h, n_q, D]
  __nv_bfloat16* out;      // [B, h, n_q, D]
  const int32_t* lens;     // [B] or null (= n_max)
  float* ws_o;             // [B, h, chunks, n_q, D]
  float* ws_ml;            // [B, h, chunks, n_q, 2]
  int h, n_q, n_max, chunks;
  float scale_log2;
};

__device__ __forceinline__ int cache_len(const DecodeArgs& a, int b) {
  if (a.lens == nullptr) return a.n_max;
  const int len = a.lens[b];
  return len < 0 ? 0 : (len > a.n_max ? a.n_max : len);
}

__device__ __forceinline__ uint4 ld_shared_v4(const void* p) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(smem_u32(p)));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int D, int NQ>
__global__ void __launch_bounds__(kDecThreads)
    decode_partial_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  using Smem = DecSmem<D, NQ>;
  constexpr int kAtoms = Smem::kAtoms;
  constexpr int kWarps = kDecThreads / 32;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  const int c = static_cast<int>(blockIdx.x), hh = static_cast<int>(blockIdx.y);
  const int b = static_cast<int>(blockIdx.z);
  const int64_t bh = static_cast<int64_t>(b) * a.h + hh;
  if (tid == 0) {
    mbar_init(&sm.full, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncthreads();
  griddep_wait();  // the cache, the queries and the lengths may come from the previous kernel
  // after the wait: the merge starts once every CTA of this grid is past it,
  // so whatever came before this grid is complete when the merge starts
  griddep_launch_dependents();

  const int L = cache_len(a, b);
  const int c0 = c * kChunk;
  if (c0 >= L) return;  // the merge reads only the chunks below L (uniform over the CTA)
  if (tid == 0) {
    mbar_arrive_expect_tx(&sm.full, 2 * kAtoms * kChunk * 128);
    for (int at = 0; at < kAtoms; ++at) {
      tma_load_3d(sm.k[at], &tm_k, &sm.full, at * 64, c0, static_cast<int>(bh));
      tma_load_3d(sm.v[at], &tm_v, &sm.full, at * 64, c0, static_cast<int>(bh));
    }
  }
  // queries -> fp32 in shared memory while the cache chunk is in flight;
  // rows past n_q are zero and masked below
  const __nv_bfloat16* qg = a.q + bh * a.n_q * D;
  for (int i = tid; i < NQ * D; i += kDecThreads) {
    const int t = i / D;
    sm.q[t][i % D] = t < a.n_q ? __bfloat162float(qg[i]) : 0.f;
  }
  const bool ok = __syncthreads_and(mbar_wait(&sm.full, 0, &sm.abort_flag));
  if (!ok) {
    // the copies may still land: keep the shared memory until they have
    volatile uint32_t never = 0;
    if (tid == 0) mbar_wait(&sm.full, 0, &never, kDrainLimitNs);
    return;
  }

  // ---- scores: thread j takes key c0 + j; masked logits are -inf
  const int j = tid;
  const int key = c0 + j;
  float x[NQ];
#pragma unroll
  for (int t = 0; t < NQ; ++t) x[t] = 0.f;
#pragma unroll
  for (int ch = 0; ch < D / 8; ++ch) {  // 16-byte chunk ch of the key row
    const int at = ch >> 3, jj = ch & 7;
    const uint4 w = ld_shared_v4(sm.k[at] + j * 128 + ((jj ^ (j & 7)) << 4));
    const float kf[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                         bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
    for (int t = 0; t < NQ; ++t)
#pragma unroll
      for (int e = 0; e < 8; ++e) x[t] = fmaf(sm.q[t][ch * 8 + e], kf[e], x[t]);
  }
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int pos = L - a.n_q + t;  // this query's position
    x[t] = (t < a.n_q && key <= pos) ? x[t] * a.scale_log2 : -INFINITY;
  }

  // ---- per query: the chunk's max, then p = 2^(x - m) and their sum
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    float m = x[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) sm.red_max[warp][t] = m;
  }
  __syncthreads();
  float mt[NQ];
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    float m = sm.red_max[0][t];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) m = fmaxf(m, sm.red_max[w][t]);
    mt[t] = m;
    const float p = x[t] == -INFINITY ? 0.f : ex2(x[t] - m);
    sm.p[t][j] = p;
    float s = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) sm.red_sum[warp][t] = s;
  }
  __syncthreads();  // P and the sums are complete; K is no longer read

  // ---- O_chunk = P V: thread (column pair pc, key group g); keys at or past
  // L are skipped (their V rows may hold anything)
  constexpr int kPairs = D / 2;
  constexpr int kGroups = kDecThreads / kPairs;
  constexpr int kKeysPerGroup = kChunk / kGroups;
  const int pc = tid % kPairs, g = tid / kPairs;
  const int at = pc >> 5, pw = pc & 31;  // box, and pair within its 128-byte row
  const int nkeys = min(kChunk, L - c0);
  float acc[NQ][2];
#pragma unroll
  for (int t = 0; t < NQ; ++t) acc[t][0] = acc[t][1] = 0.f;
  const int jb = g * kKeysPerGroup;
  const int je = min(jb + kKeysPerGroup, nkeys);
  for (int jj = jb; jj < je; ++jj) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(
        sm.v[at] + jj * 128 + ((((pw >> 2) ^ (jj & 7)) << 4) | ((pw & 3) << 2)));
    const float v0 = bf16_lo(w), v1 = bf16_hi(w);
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
      const float p = sm.p[t][jj];
      acc[t][0] = fmaf(p, v0, acc[t][0]);
      acc[t][1] = fmaf(p, v1, acc[t][1]);
    }
  }
  float* red = reinterpret_cast<float*>(sm.k[0]);  // [kGroups][NQ][D]
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    red[(g * NQ + t) * D + 2 * pc] = acc[t][0];
    red[(g * NQ + t) * D + 2 * pc + 1] = acc[t][1];
  }
  __syncthreads();
  const int64_t slot = (bh * a.chunks + c) * a.n_q;  // (batch, head, chunk) row of the workspace
  for (int i = tid; i < a.n_q * D; i += kDecThreads) {
    const int t = i / D, col = i % D;
    float o = 0.f;
#pragma unroll
    for (int gg = 0; gg < kGroups; ++gg) o += red[(gg * NQ + t) * D + col];
    a.ws_o[(slot + t) * D + col] = o;
  }
  if (tid < a.n_q) {
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) l += sm.red_sum[w][tid];
    float m = -INFINITY;
#pragma unroll
    for (int t = 0; t < NQ; ++t)
      if (t == tid) m = mt[t];
    a.ws_ml[(slot + tid) * 2] = m;
    a.ws_ml[(slot + tid) * 2 + 1] = l;
  }
}

constexpr int kMergeThreads = 256;
constexpr int kMergeBatch = 16;  // chunk partials loaded per thread before they are summed

// shared memory of the merge: the weights [chunks][n_q], 1 / l [n_q] and the
// groups' sums [kMergeThreads / D][n_q][D]
size_t merge_smem_bytes(int chunks, int n_q, int d) {
  return (static_cast<size_t>(chunks) * n_q + n_q + static_cast<size_t>(kMergeThreads / d) * n_q * d) *
         sizeof(float);
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecodeArgs a) {
  // the weights of every (chunk, query) pair go to shared memory first; then
  // kMergeThreads / D groups of D threads (one per column) each sum a share
  // of the chunks, kMergeBatch loads in flight per thread, and the groups'
  // sums are added
  constexpr int kGroups = kMergeThreads / D;
  extern __shared__ float merge_smem[];
  float* w_s = merge_smem;                  // [chunks][n_q]
  float* inv_l_s = w_s + a.chunks * a.n_q;  // [n_q]
  float* part_s = inv_l_s + a.n_q;          // [kGroups][n_q][D]
  const int tid = static_cast<int>(threadIdx.x);
  const int hh = static_cast<int>(blockIdx.x), b = static_cast<int>(blockIdx.y);
  const int64_t bh = static_cast<int64_t>(b) * a.h + hh;
  // the lengths before the wait: the partial grid triggers this launch only
  // after its own dependency wait, so the kernel that wrote them (if any) is
  // complete; the partials themselves are read after the wait
  const int L = cache_len(a, b);
  const int nc = (L + kChunk - 1) / kChunk;       // <= a.chunks
  const int col = tid % D, grp = tid / D;
  const float* o_bh = a.ws_o + bh * a.chunks * a.n_q * D;  // [chunk][query][D]
  griddep_launch_dependents();
  griddep_wait();  // the partials of the previous kernel are complete
  // the first query's first batch of chunk partials is in flight while the
  // weights are computed
  float v0[kMergeBatch];
#pragma unroll
  for (int u = 0; u < kMergeBatch; ++u) {
    const int c = grp + u * kGroups;
    v0[u] = c < nc ? o_bh[c * a.n_q * D + col] : 0.f;
  }
  const float* ml = a.ws_ml + bh * a.chunks * a.n_q * 2;  // [chunk][query][m, l]
  // per query (warp t, lanes over the chunks): m = max_c m_c,
  // w_c = 2^(m_c - m), l = sum_c w_c l_c
  const int warp = tid >> 5, lane = tid & 31;
  for (int t = warp; t < a.n_q; t += kMergeThreads / 32) {
    float m = -INFINITY;
#pragma unroll 4
    for (int c = lane; c < nc; c += 32) m = fmaxf(m, ml[(c * a.n_q + t) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    for (int c = lane; c < nc; c += 32) {
      const float mc = ml[(c * a.n_q + t) * 2];
      // a chunk holding none of this query's keys has m_c = -inf and weight 0
      const float w = mc == -INFINITY ? 0.f : ex2(mc - m);
      l = fmaf(w, ml[(c * a.n_q + t) * 2 + 1], l);
      w_s[c * a.n_q + t] = w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) inv_l_s[t] = l > 0.f ? 1.f / l : 0.f;  // no visible key: output 0
  }
  __syncthreads();
  for (int t = 0; t < a.n_q; ++t) {
    float o = 0.f;
    for (int c0 = grp; c0 < nc; c0 += kMergeBatch * kGroups) {
      float v[kMergeBatch];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const int c = c0 + u * kGroups;
        if (t == 0 && c0 == grp) v[u] = v0[u];
        else v[u] = c < nc ? o_bh[(c * a.n_q + t) * D + col] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const int c = c0 + u * kGroups;
        if (c < nc) o = fmaf(w_s[c * a.n_q + t], v[u], o);
      }
    }
    part_s[(grp * a.n_q + t) * D + col] = o;
  }
  __syncthreads();
  for (int i = tid; i < a.n_q * D; i += kMergeThreads) {
    const int t = i / D, cc = i % D;
    float o = 0.f;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) o += part_s[(g * a.n_q + t) * D + cc];
    a.out[(bh * a.n_q + t) * D + cc] = __float2bfloat16_rn(o * inv_l_s[t]);
  }
}

template <int D, int NQ>
cudaError_t launch_decode_nq(const DecodeProblem& p, cudaStream_t stream) {
  using Smem = DecSmem<D, NQ>;
  const size_t smem_bytes = sizeof(Smem) + 1024;
  auto kernel = decode_partial_kernel<D, NQ>;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(kernel, static_cast<int>(smem_bytes), &configured);
  if (e != cudaSuccess) return e;
  DecodeArgs a;
  a.q = static_cast<const __nv_bfloat16*>(p.q);
  a.out = static_cast<__nv_bfloat16*>(p.out);
  a.lens = p.cache_lens;
  a.h = p.h;
  a.n_q = p.n_q;
  a.n_max = p.n_max;
  a.chunks = decode_chunks(p.n_max);
  a.ws_o = p.ws_o;
  a.ws_ml = p.ws_ml;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  e = launch_pdl(kernel, dim3(a.chunks, p.h, p.B), dim3(kDecThreads), smem_bytes, stream,
                 p.tm_k, p.tm_v, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_merge_kernel<D>, dim3(p.h, p.B), dim3(kMergeThreads),
                    merge_smem_bytes(a.chunks, p.n_q, D), stream, a);
}

template <int D>
cudaError_t launch_decode_d(const DecodeProblem& p, cudaStream_t stream) {
  if (p.n_q <= 1) return launch_decode_nq<D, 1>(p, stream);
  if (p.n_q <= 2) return launch_decode_nq<D, 2>(p, stream);
  if (p.n_q <= 4) return launch_decode_nq<D, 4>(p, stream);
  return launch_decode_nq<D, 8>(p, stream);
}

}  // namespace

int decode_chunks(int n_max) { return (n_max + kChunk - 1) / kChunk; }

cudaError_t launch_decode(const DecodeProblem& p, cudaStream_t stream) {
  if (p.n_q < 1 || p.n_q > kDecodeMaxQueries || p.n_max < 1 || p.B < 1 || p.h < 1 ||
      decode_chunks(p.n_max) > kDecodeMaxChunks)
    return cudaErrorInvalidValue;
  if (p.d == 64) return launch_decode_d<64>(p, stream);
  if (p.d == 128) return launch_decode_d<128>(p, stream);
  return cudaErrorInvalidValue;
}

TSD_DEFINE_ERROR_READER(take_device_error_decode)

}  // namespace tsd
