// layernorm.cu -- the "Add & Norm" of a post-LN sub-layer,
// out = LayerNorm(x + r) = gamma (v - mu) / sqrt(sigma^2 + eps) + beta with
// v = x + r, mu and sigma^2 (population variance) over one token's d_model
// features ("[논문 리뷰]Attention Is All You Need" (kimjiil.github.io),
// section 3.1; "Attention Is All You Need 해부" (sj-techlog), section "4.
// residual connection과 LayerNorm은 깊은 층을 학습 가능하게 한다").
//
// Bound by HBM (it reads 2 and writes 1 row of bf16 per token), so a warp per
// row: each lane holds d_model / 32 features in registers (loaded as 16-byte
// vectors, a warp reading 512 contiguous bytes per step), the mean and then
// the centred variance come from warp shuffles (two passes over registers,
// no cancellation), and the row is written back in the same vectors. The
// input can be fp32 and an fp32 copy of the output can be written too, so a
// residual path need not round to bf16 twice.
#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kLnWarps = 8;

__device__ __forceinline__ void unpack8(uint4 w, float* f) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
  }
}

template <int VPL, bool XF32>  // 8-feature vectors per lane: d_model = 256 VPL; x fp32?
__global__ void __launch_bounds__(kLnWarps * 32)
    add_layernorm_kernel(const void* __restrict__ xv, const uint16_t* __restrict__ r,
                         const uint16_t* __restrict__ gamma, const uint16_t* __restrict__ beta,
                         uint16_t* __restrict__ out, float* __restrict__ out32, int rows,
                         float eps) {
  constexpr int D = 256 * VPL;
  griddep_launch_dependents();
  griddep_wait();  // x and r may come from the previous kernel
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int row = static_cast<int>(blockIdx.x) * kLnWarps + static_cast<int>(threadIdx.x >> 5);
  if (row >= rows) return;
  const size_t base = static_cast<size_t>(row) * D;
  float v[VPL * 8];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int col = (i * 32 + lane) * 8;
    if constexpr (XF32) {
      const float4* xf = reinterpret_cast<const float4*>(static_cast<const float*>(xv) + base + col);
      const float4 a = __ldg(xf), b = __ldg(xf + 1);
      v[i * 8 + 0] = a.x; v[i * 8 + 1] = a.y; v[i * 8 + 2] = a.z; v[i * 8 + 3] = a.w;
      v[i * 8 + 4] = b.x; v[i * 8 + 5] = b.y; v[i * 8 + 6] = b.z; v[i * 8 + 7] = b.w;
    } else {
      unpack8(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(xv) + base + col)),
              v + i * 8);
    }
    if (r != nullptr) {
      float t[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(r + base + col)), t);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[i * 8 + e] += t[e];
    }
  }
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < VPL * 8; ++e) s += v[e];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mu = s * (1.f / D);
  float q = 0.f;
#pragma unroll
  for (int e = 0; e < VPL * 8; ++e) {
    const float c = v[e] - mu;
    q = fmaf(c, c, q);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  const float rstd = rsqrtf(q * (1.f / D) + eps);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int col = (i * 32 + lane) * 8;
    float g[8], b[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(gamma + col)), g);
    unpack8(__ldg(reinterpret_cast<const uint4*>(beta + col)), b);
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = fmaf((v[i * 8 + e] - mu) * rstd, g[e], b[e]);
    st_global_v4(out + base + col, pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                 pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
    if (out32 != nullptr) {
      float4* o32 = reinterpret_cast<float4*>(out32 + base + col);
      o32[0] = make_float4(y[0], y[1], y[2], y[3]);
      o32[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
  }
}

}  // namespace

cudaError_t launch_add_layernorm(const void* x, bool x_f32, const uint16_t* r,
                                 const uint16_t* gamma, const uint16_t* beta, uint16_t* out,
                                 float* out32, int rows, int d_model, float eps,
                                 cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid((rows + kLnWarps - 1) / kLnWarps), block(kLnWarps * 32);
#define TSD_LN_CASE(VPL)                                                                    \
  return x_f32 ? launch_pdl(add_layernorm_kernel<VPL, true>, grid, block, 0, stream, x, r,  \
                            gamma, beta, out, out32, rows, eps)                             \
               : launch_pdl(add_layernorm_kernel<VPL, false>, grid, block, 0, stream, x, r, \
                            gamma, beta, out, out32, rows, eps)
  switch (d_model) {
    case 256: TSD_LN_CASE(1);
    case 512: TSD_LN_CASE(2);
    case 1024: TSD_LN_CASE(4);
    case 2048: TSD_LN_CASE(8);
    default: return cudaErrorInvalidValue;
  }
#undef TSD_LN_CASE
}

}  // namespace tsd
