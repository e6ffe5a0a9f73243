// gemm_bf16.cu -- the projections of multi-head attention on the sm_103a
// tensor cores: Q = X_q W_Q, K = X_kv W_K, V = X_kv W_V in one grouped
// launch, and Concat(head_1..head_h) W_O ("[논문 리뷰]Attention Is All You
// Need" (kimjiil.github.io), section 3.2.2; weights in the x.W layout,
// [d_model, h*d], no biases).
//
// Persistent kernel: one CTA per SM walks the 128 x 128 output tiles of all
// groups (C = A B, fp32 accumulation in tensor memory):
//   warp 0     TMA producer: per 64-deep K block, one A box (64 K x 128 M,
//              K-major) and two B boxes (64 N x 64 K, N-major), kStages deep,
//              running ahead across tile boundaries
//   warp 1     MMA issuer (one thread), 4 MMAs per K block; owns the TMEM
//              allocation: two 128-column accumulators, so the epilogue of
//              one tile overlaps the main loop of the next
//   warps 2-5  epilogue: one thread per output row (TMEM lane) reads its
//              accumulator row, releases the accumulator, converts to bf16
//              into a 128-byte-swizzled staging tile in shared memory, and
//              one thread writes the tile with two TMA stores. Row-per-thread
//              global stores would leave each warp instruction scattered over
//              32 rows; the TMA store writes whole lines. Two staging tiles
//              alternate, so a store drains while the next tile is staged.
// The head split needs no data movement: head i of Q is column block i of
// the [B*n, h*d] result, which the attention kernel reads through strides.
#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kAccCols = 128;
constexpr int kTmemCols = 2 * kAccCols;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB: one 128-row x 128-byte K atom column
constexpr int kBBytes = kBK * kBN * 2;  // 16 KB: two 64-row (K) x 128-byte N chunks
constexpr int kBChunk = kBK * 128;      // bytes of one 64-wide N chunk
constexpr int kCBytes = kBM * kBN * 2;  // 32 KB: one bf16 output tile (two 64-column boxes)
constexpr uint32_t kEpiBarrier = 1;     // named barrier of the four epilogue warps
constexpr unsigned long long kDrainLimitNs = 100ull * 1000ull * 1000ull;

struct GemmSmem {
  alignas(1024) uint8_t a[kStages][kABytes];
  alignas(1024) uint8_t b[kStages][kBBytes];
  alignas(1024) uint8_t c[2][kCBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drained;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct TileCoord {
  const GemmGroup* g;
  int m0, n0;
};

__device__ __forceinline__ TileCoord tile_coord(const GemmProblem& p, int tile) {
  int gi = 0;
  for (int i = 1; i < p.num_groups; ++i)
    if (tile >= p.g[i].tile_begin) gi = i;
  const GemmGroup& G = p.g[gi];
  const int local = tile - G.tile_begin;
  TileCoord c;
  c.g = &G;
  c.m0 = (local % G.tiles_m) * kBM;  // m fastest: neighbouring CTAs share B
  c.n0 = (local / G.tiles_m) * kBN;
  return c;
}

__global__ void __launch_bounds__(kThreads, 1) gemm_bf16_kernel(const __grid_constant__ GemmProblem p) {
  extern __shared__ uint8_t smem_raw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = warp_id();
  const uint32_t lane = lane_id();
  const int kblocks = (p.K + kBK - 1) / kBK;
  // tiles of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int first = blockIdx.x;
  const int stride = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sm.acc_full[a], 1);
      mbar_init(&sm.acc_empty[a], 128);
    }
    mbar_init(&sm.drained, 1);
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
  // the set-up above may overlap the previous kernel; global memory may not
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int i = 0; i < p.num_groups; ++i) {
        tma_prefetch_desc(&p.g[i].tm_a);
        tma_prefetch_desc(&p.g[i].tm_b);
        tma_prefetch_desc(&p.g[i].tm_c);
      }
      int issued = 0;
      bool ok = true;
      for (int tile = first; ok && tile < p.total_tiles; tile += stride) {
        const TileCoord c = tile_coord(p, tile);
        for (int kb = 0; kb < kblocks; ++kb) {
          const int s = issued % kStages;
          const uint32_t ph = static_cast<uint32_t>(issued / kStages) & 1u;
          if (!mbar_wait(&sm.empty[s], ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.full[s], kABytes + kBBytes);
          const int k0 = kb * kBK;
          tma_load_2d(sm.a[s], &c.g->tm_a, &sm.full[s], k0, c.m0);
          tma_load_2d(sm.b[s], &c.g->tm_b, &sm.full[s], c.n0, k0);
          tma_load_2d(sm.b[s] + kBChunk, &c.g->tm_b, &sm.full[s], c.n0 + 64, k0);
          ++issued;
        }
      }
      if (!ok) {
        volatile uint32_t never = 0;
        for (int i = max(0, issued - kStages); i < issued; ++i)
          mbar_wait(&sm.full[i % kStages], static_cast<uint32_t>(i / kStages) & 1u, &never,
                    kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(kBM, kBN, false, true);
      // descriptors built once, advanced inside the start-address field
      const uint64_t da0 = sdesc_sw128(smem_u32(sm.a[0]), 16, 1024);     // K-major A
      const uint64_t db0 = sdesc_sw128(smem_u32(sm.b[0]), kBChunk, 1024);  // N-major B
      int consumed = 0;
      int it = 0;
      bool ok = true;
      for (int tile = first; ok && tile < p.total_tiles; tile += stride, ++it) {
        const int acc = it & 1;
        // the epilogue has read this accumulator's previous tile
        ok = mbar_wait(&sm.acc_empty[acc], (static_cast<uint32_t>(it >> 1) & 1u) ^ 1u, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * kAccCols;
        for (int kb = 0; kb < kblocks; ++kb) {
          const int s = consumed % kStages;
          ok = mbar_wait(&sm.full[s], static_cast<uint32_t>(consumed / kStages) & 1u, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t da = sdesc_advance(da0, static_cast<uint32_t>(s) * (kABytes >> 4));
          const uint64_t db = sdesc_advance(db0, static_cast<uint32_t>(s) * (kBBytes >> 4));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // A: K-major, 32 bytes per 16-element step inside the atom;
            // B: N-major, 16 K rows = 2048 bytes; the second N chunk is kBChunk on
            mma_bf16_ss(d_tmem, sdesc_advance(da, kk * (32 >> 4)), sdesc_advance(db, kk * (2048 >> 4)),
                        kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&sm.empty[s]);
          ++consumed;
        }
        if (ok) mma_commit(&sm.acc_full[acc]);
      }
      volatile uint32_t never = 0;
      mma_commit(&sm.drained);
      mbar_wait(&sm.drained, 0, &never, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warps 2..5 cover TMEM lane quarters 2, 3, 0, 1
    const int quarter = warp & 3;
    const int r = quarter * 32 + static_cast<int>(lane);
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const bool leader = (warp == 2 && lane == 0);  // issues the tile's TMA stores
    int it = 0;
    for (int tile = first; tile < p.total_tiles; tile += stride, ++it) {
      const int acc = it & 1;
      const TileCoord c = tile_coord(p, tile);
      bool ok = __all_sync(
          0xffffffffu,
          mbar_wait(&sm.acc_full[acc], static_cast<uint32_t>(it >> 1) & 1u, abort_flag));
      // staging tile it&1 was last written out two tiles ago: its store must
      // have finished reading shared memory before it is overwritten
      if (leader) bulk_wait_group_read<1>();
      // one decision for all four warps: none is left waiting at a barrier
      ok = named_bar_and(kEpiBarrier, 128, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t v[kBN];
#pragma unroll
      for (int cc = 0; cc < kBN / 32; ++cc) {
        uint32_t chunk[32];
        tmem_ld32(tmem + lane_base + acc * kAccCols + cc * 32, chunk);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[cc * 32 + i] = chunk[i];
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&sm.acc_empty[acc]);  // the MMA warp may reuse this accumulator

      uint8_t* stage = sm.c[it & 1];
      // 128-byte swizzle of the store's tensor map: the 16-byte chunk j of
      // row r sits at chunk position j ^ (r mod 8) of the row's 128 bytes
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t* e = v + half * 64 + j * 8;
          st_shared_v4(smem_u32(stage + half * 16384 + r * 128 + ((j ^ (r & 7)) << 4)),
                       pack_bf16x2(__uint_as_float(e[0]), __uint_as_float(e[1])),
                       pack_bf16x2(__uint_as_float(e[2]), __uint_as_float(e[3])),
                       pack_bf16x2(__uint_as_float(e[4]), __uint_as_float(e[5])),
                       pack_bf16x2(__uint_as_float(e[6]), __uint_as_float(e[7])));
        }
      }
      fence_proxy_async_smem();  // staged bytes visible to the TMA unit
      named_bar_sync(kEpiBarrier, 128);
      if (leader) {
        // the map clips rows past M and columns past N
        tma_store_2d(&c.g->tm_c, stage, c.n0, c.m0);
        if (c.n0 + 64 < c.g->N) tma_store_2d(&c.g->tm_c, stage + 16384, c.n0 + 64, c.m0);
        bulk_commit_group();
      }
    }
    if (leader) bulk_wait_group<0>();  // stores complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

}  // namespace

cudaError_t launch_gemm_bf16(const GemmProblem& p, cudaStream_t stream) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const size_t smem_bytes = sizeof(GemmSmem) + 1024;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(gemm_bf16_kernel, static_cast<int>(smem_bytes), &configured);
  if (e != cudaSuccess) return e;
  const int grid = p.total_tiles < num_sms() ? p.total_tiles : num_sms();
  return launch_pdl(gemm_bf16_kernel, dim3(grid), dim3(kThreads), smem_bytes, stream, p);
}

TSD_DEFINE_ERROR_READER(take_device_error_gemm)

}  // namespace tsd
