// gemm_bf16.cu -- the projections of multi-head attention on the sm_103a
// tensor cores: Q = X_q W_Q, K = X_kv W_K, V = X_kv W_V in one grouped
// launch, and Concat(head_1..head_h) W_O ("[논문 리뷰]Attention Is All You
// Need" (kimjiil.github.io), section 3.2.2; weights in the x.W layout,
// [d_model, h*d], no biases).
//
// One CTA computes one 128 x 128 tile of C = A B with fp32 accumulation in
// tensor memory:
//   warp 0     TMA producer: A box (64 K x 128 M, K-major) and two B boxes
//              (64 N x 64 K each, N-major) per 64-deep K block, STAGES deep
//   warp 1     MMA issuer (one thread); owns the 128-column TMEM allocation
//   warps 2-5  epilogue: one thread per output row (TMEM lane), fp32 -> bf16,
//              16-byte stores
// The head split needs no data movement: head i of Q is column block i of
// the [B*n, h*d] result, which the attention kernel reads through strides.
#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 64;
constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr int kTmemCols = 128;

struct GemmSmem {
  alignas(1024) uint8_t a[kStages][kBM * kBK * 2];   // 16 KB: 128 rows x 128 B
  alignas(1024) uint8_t b[kStages][kBK * kBN * 2];   // 16 KB: two 64x64 N-major boxes
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

__global__ void __launch_bounds__(kThreads, 2) gemm_bf16_kernel(const __grid_constant__ GemmProblem p) {
  extern __shared__ uint8_t smem_raw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = warp_id();
  const uint32_t lane = lane_id();

  // tile -> (group, m tile, n tile); m varies fastest
  const int tile = blockIdx.x;
  int g = 0;
  for (int i = 1; i < p.num_groups; ++i)
    if (tile >= p.g[i].tile_begin) g = i;
  const GemmGroup& G = p.g[g];
  const int local = tile - G.tile_begin;
  const int m0 = (local % G.tiles_m) * kBM;
  const int n0 = (local / G.tiles_m) * kBN;
  const int kblocks = (p.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.acc_full, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile uint32_t* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&G.tm_a);
      tma_prefetch_desc(&G.tm_b);
      int issued = 0;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        const int s = kb % kStages;
        const uint32_t ph = static_cast<uint32_t>(kb / kStages) & 1u;
        if (!mbar_wait(&sm.empty[s], ph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sm.full[s], kBM * kBK * 2 + kBK * kBN * 2);
        tma_load_2d(sm.a[s], &G.tm_a, &sm.full[s], kb * kBK, m0);
        tma_load_2d(sm.b[s], &G.tm_b, &sm.full[s], n0, kb * kBK);
        tma_load_2d(sm.b[s] + 8192, &G.tm_b, &sm.full[s], n0 + 64, kb * kBK);
        ++issued;
      }
      if (!ok) {
        volatile uint32_t never = 0;
        for (int i = max(0, issued - kStages); i < issued; ++i)
          mbar_wait(&sm.full[i % kStages], static_cast<uint32_t>(i / kStages) & 1u, &never,
                    100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(kBM, kBN, false, true);
      // descriptors built once, advanced by constant start-address offsets
      const uint64_t da0 = sdesc_sw128(smem_u32(sm.a[0]), 16, 1024);    // K-major A
      const uint64_t db0 = sdesc_sw128(smem_u32(sm.b[0]), 8192, 1024);  // N-major B
      constexpr uint32_t kAStep = (kBM * kBK * 2) >> 4, kBStep = (kBK * kBN * 2) >> 4;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        const int s = kb % kStages;
        if (!mbar_wait(&sm.full[s], static_cast<uint32_t>(kb / kStages) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t da = sdesc_advance(da0, static_cast<uint32_t>(s) * kAStep);
        const uint64_t db = sdesc_advance(db0, static_cast<uint32_t>(s) * kBStep);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // A: K-major, a 16-element K step is 32 bytes inside the swizzle atom;
          // B: N-major, 16 K rows are 2048 bytes (second 64-wide N chunk 8 KB on)
          mma_bf16_ss(tmem, sdesc_advance(da, kk * (32 >> 4)), sdesc_advance(db, kk * (2048 >> 4)),
                      kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&sm.empty[s]);
      }
      mma_commit(&sm.acc_full);
      if (!ok) {
        volatile uint32_t never = 0;
        mbar_wait(&sm.acc_full, 0, &never, 100000000ull);
      }
    }
  } else {
    // epilogue warps 2..5 cover TMEM lane quarters 2, 3, 0, 1
    const int quarter = warp & 3;
    const int r = quarter * 32 + static_cast<int>(lane);
    const int row = m0 + r;
    bool ok = mbar_wait(&sm.acc_full, 0, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (ok && kblocks > 0) {
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
      uint16_t* crow = G.c + static_cast<int64_t>(row) * G.ldc;
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(taddr + c * 32, v);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        if (row < G.M) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const int col = n0 + c * 32 + v4 * 8;
            if (col < G.N)
              st_global_v4(crow + col, w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_gemm_bf16(const GemmProblem& p, cudaStream_t stream) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const size_t smem_bytes = sizeof(GemmSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_bytes));
  if (e != cudaSuccess) return e;
  gemm_bf16_kernel<<<p.total_tiles, kThreads, smem_bytes, stream>>>(p);
  return cudaGetLastError();
}

TSD_DEFINE_ERROR_READER(take_device_error_gemm)

}  // namespace tsd
