// attn_f32.cu -- scaled dot-product attention in fp32 throughout (FFMA on the
// CUDA cores; no TF32), for callers that need results within 1e-4 of exact
// ("[논문 리뷰]Attention Is All You Need" (kimjiil.github.io), section 3.2.1,
// eq. (1); masks before the softmax, section 3.2.3).
//
// A CTA of 4 warps owns 32 query rows of one (batch, head); K/V tiles of 32
// keys are staged in shared memory and shared by the warps. Lane j of a warp
// scores key j of the tile; row max and row sum use warp shuffles; each lane
// accumulates the output columns lane, lane+32, ... with the online
// (running max, running sum) softmax in fp32 and expf.
#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 8;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;  // 32
constexpr int kKeys = 32;
constexpr int kMaxD = 128;

__global__ void __launch_bounds__(kWarps * 32) attn_fwd_f32_kernel(const AttnF32Problem p) {
  extern __shared__ float smem[];
  const int dk = p.d_k, dv = p.d_v;
  const int kstride = dk + 1;  // pad: lane j reads row j without bank conflicts
  float* sq = smem;                                  // [32][dk]
  float* sk = sq + kRowsPerCta * dk;                  // [32][dk+1]
  float* sv = sk + kKeys * kstride;                   // [32][dv]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.z, hh = blockIdx.y;
  const int qbase = blockIdx.x * kRowsPerCta;
  const size_t bh = static_cast<size_t>(b) * p.h + hh;
  const float* Q = p.q + bh * p.n_q * dk;
  const float* K = p.k + bh * p.n_k * dk;
  const float* V = p.v + bh * p.n_k * dv;
  float* O = p.out + bh * p.n_q * dv;
  const bool causal = (p.mask_kind & kMaskCausal) != 0;

  int kv_eff = p.n_k;
  if (p.mask_kind & kMaskKeyPadding) {
    const int len = p.kv_lens[b];
    kv_eff = len < 0 ? 0 : (len > p.n_k ? p.n_k : len);
  }
  // keys any row of this CTA may see
  int keys_needed = kv_eff;
  if (causal) keys_needed = min(keys_needed, qbase + kRowsPerCta);

  for (int i = threadIdx.x; i < kRowsPerCta * dk; i += blockDim.x) {
    const int rr = i / dk, c = i - rr * dk;
    const int row = qbase + rr;
    sq[i] = row < p.n_q ? Q[static_cast<size_t>(row) * dk + c] : 0.f;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kMaxD / 32];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxD / 32; ++c) acc[i][c] = 0.f;
  }

  for (int k0 = 0; k0 < keys_needed; k0 += kKeys) {
    __syncthreads();
    for (int i = threadIdx.x; i < kKeys * dk; i += blockDim.x) {
      const int j = i / dk, c = i - j * dk;
      sk[j * kstride + c] = (k0 + j < p.n_k) ? K[static_cast<size_t>(k0 + j) * dk + c] : 0.f;
    }
    for (int i = threadIdx.x; i < kKeys * dv; i += blockDim.x) {
      const int j = i / dv, c = i - j * dv;
      sv[i] = (k0 + j < p.n_k) ? V[static_cast<size_t>(k0 + j) * dv + c] : 0.f;
    }
    __syncthreads();

#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int rr = warp * kRowsPerWarp + i;
      const int row = qbase + rr;
      const int lim = causal ? min(kv_eff, row + 1) : kv_eff;  // keys [0, lim) allowed
      const int key = k0 + lane;
      float s = -INFINITY;
      if (key < lim) {
        float dot = 0.f;
        const float* qr = sq + rr * dk;
        const float* kr = sk + lane * kstride;
        for (int c = 0; c < dk; ++c) dot = fmaf(qr[c], kr[c], dot);
        s = dot * p.scale;
      }
      float tmax = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float m_new = fmaxf(m[i], tmax);
      if (m_new == -INFINITY) continue;  // nothing allowed yet for this row
      const float alpha = expf(m[i] - m_new);  // 0 when m[i] = -inf
      const float pj = (s == -INFINITY) ? 0.f : expf(s - m_new);
      float psum = pj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      l[i] = l[i] * alpha + psum;
      m[i] = m_new;
#pragma unroll
      for (int cc = 0; cc < kMaxD / 32; ++cc) acc[i][cc] *= alpha;
      for (int j = 0; j < kKeys; ++j) {
        const float pb = __shfl_sync(0xffffffffu, pj, j);
        if (pb == 0.f) continue;
        const float* vr = sv + j * dv;
#pragma unroll
        for (int cc = 0; cc < kMaxD / 32; ++cc) {
          const int c = lane + cc * 32;
          if (c < dv) acc[i][cc] = fmaf(pb, vr[c], acc[i][cc]);
        }
      }
    }
  }

#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int row = qbase + warp * kRowsPerWarp + i;
    if (row >= p.n_q) continue;
    const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
#pragma unroll
    for (int cc = 0; cc < kMaxD / 32; ++cc) {
      const int c = lane + cc * 32;
      if (c < dv) O[static_cast<size_t>(row) * dv + c] = acc[i][cc] * inv;
    }
  }
}

}  // namespace

cudaError_t launch_attn_f32(const AttnF32Problem& p, cudaStream_t stream) {
  const size_t smem = sizeof(float) *
                      (static_cast<size_t>(kRowsPerCta) * p.d_k + kKeys * (p.d_k + 1) + kKeys * p.d_v);
  // the limit is raised once, to what the largest head dimensions need
  constexpr int kMaxSmem =
      static_cast<int>(sizeof(float) * (kRowsPerCta * kMaxD + kKeys * (kMaxD + 1) + kKeys * kMaxD));
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(attn_fwd_f32_kernel, kMaxSmem, &configured);
  if (e != cudaSuccess) return e;
  if (smem > static_cast<size_t>(kMaxSmem)) return cudaErrorInvalidValue;
  dim3 grid((p.n_q + kRowsPerCta - 1) / kRowsPerCta, p.h, p.B);
  attn_fwd_f32_kernel<<<grid, kWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Failure-detection self test: one thread waits (bounded) on an mbarrier that
// nothing arrives on; the wait runs out, the device error word is set, and
// the kernel returns.
__global__ void wait_timeout_selftest_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, reinterpret_cast<volatile uint32_t*>(&abort_flag), limit_ns);
}

cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

TSD_DEFINE_ERROR_READER(take_device_error_f32)

}  // namespace tsd
