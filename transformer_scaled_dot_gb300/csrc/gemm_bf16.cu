// gemm_bf16.cu -- the projections of multi-head attention on the sm_103a
// tensor cores: Q = X_q W_Q, K = X_kv W_K, V = X_kv W_V in one grouped
// launch, and Concat(head_1..head_h) W_O ("[논문 리뷰]Attention Is All You
// Need" (kimjiil.github.io), section 3.2.2; weights in the x.W layout,
// [d_model, h*d], no biases); and the two linear maps of the position-wise
// feed-forward network (section 3.3), whose bias, ReLU and residual the
// epilogue adds.
//
// Persistent kernel, one CTA per SM walking 128 x BN output tiles (m
// fastest, so CTAs working at the same time share their B (weight) tile in
// L2). The projections are bound by L2 -> SM traffic, not by the tensor
// cores. Per CTA (C = A B, fp32 accumulation in tensor memory):
//   warp 0     TMA producer: per 64-deep K block, the A box (64 K x 128 M,
//              K-major) and the B boxes (64 N each, N-major); kStages deep
//              (as many bytes in flight as shared memory allows: the loads,
//              not the MMAs, set the pace), running ahead across tiles
//   warp 1     MMA issuer (one thread), 4 MMAs per K block, whose completion
//              frees the stage; owns the TMEM allocation: two accumulators,
//              so the epilogue of one tile overlaps the main loop of the next
//   warps 2-5  epilogue: one thread per output row (TMEM lane) reads its
//              accumulator row, releases the accumulator, converts to bf16
//              into a 128-byte-swizzled staging tile in shared memory, and
//              one thread writes the tile with two TMA stores. Row-per-thread
//              global stores would leave each warp instruction scattered over
//              32 rows; the TMA store writes whole lines. The store drains
//              while the next tile's main loop runs.
// The head split needs no data movement: head i of Q is column block i of
// the [B*n, h*d] result, which the attention kernel reads through strides.
//
// LayerNorm epilogue (the feed-forward sub-layer's "Add & Norm", section
// 3.1: out = LayerNorm(y + FFN(y))): a row's N <= 1024 columns are spread
// over a cluster of N / 128 CTAs along N, one 128-row tile per cluster step.
// Each epilogue thread forms its row's v = acc + bias + residual in fp32,
// writes v back over its accumulator, takes the mean and the centred sum of
// squares of its 128 columns, and sends that pair to the other CTAs of the
// cluster (st.async into a double-buffered slot, complete_tx on their
// mbarrier); the cluster's pairs combine exactly (equal counts: the mean of
// the means, and the sums of squares plus 128 times the squared offsets of
// the partial means). It then re-reads v, normalises with gamma and beta,
// and stores its bf16 row segment (256 contiguous bytes) straight to global
// memory: the fp32 sum never goes to memory, and without a staging tile the
// statistics slots fit beside all six stages.
#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = kGemmBK;
constexpr int kStages = 6;
constexpr int kStagesLN = 6;      // LayerNorm epilogue (no staging tile: rows stored directly)
constexpr int kMaxLnCluster = 8;  // N <= 8 x 128
constexpr int kThreads = 192;
constexpr bool kPrefetchL2 = true;  // a share of the first tiles' weights into L2 before the wait
constexpr int kAccCols = 128;
// LayerNorm epilogue: one more 128-column region after the accumulators
// holds the tile's fp32 residual, streamed in while the main loop runs
constexpr int kResCol = 2 * kAccCols;
constexpr int kTmemColsLN = 512;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB: one 128-row x 128-byte K atom column
constexpr int kBChunk = kBK * 128;      // bytes of one 64-wide N chunk
constexpr int kCBytes = kBM * kBN * 2;  // 32 KB: one bf16 output tile (two 64-column boxes)
constexpr int kCStages = 1;             // output staging tiles
constexpr uint32_t kEpiBarrier = 1;     // named barrier of the four epilogue warps
constexpr unsigned long long kDrainLimitNs = 100ull * 1000ull * 1000ull;

template <int ST, bool LN, int BN>
struct GemmSmemT {
  alignas(1024) uint8_t a[ST][kABytes];
  alignas(1024) uint8_t b[ST][kBK * BN * 2];
  alignas(1024) uint8_t c[LN ? 1 : kCStages][LN ? 16 : kCBytes];
  // LayerNorm epilogue: per tile parity, per other CTA of the cluster (in
  // rank order, skipping this one), per row: that CTA's (mean, centred sum
  // of squares) over its 128 columns
  float2 ln_stat[LN ? 2 : 1][LN ? kMaxLnCluster - 1 : 1][LN ? kBM : 1];
  uint64_t ln_full[2];
  uint64_t full[ST];
  uint64_t empty[ST];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drained;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

// acc[i] += the 8 bf16 of w (low half first)
__device__ __forceinline__ void add_bf16x8(float (&acc)[8], uint4 w) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] += __uint_as_float(u[i] << 16);
    acc[2 * i + 1] += __uint_as_float(u[i] & 0xffff0000u);
  }
}

struct TileCoord {
  const GemmGroup* g;
  int m0, n0;
};

// Tile `ct` (over every group's 128 x BN tiles) -> its group and origin.
template <int BN>
__device__ __forceinline__ TileCoord tile_coord(const GemmProblem& p, int ct) {
  int gi = 0;
  for (int i = 1; i < p.num_groups; ++i)
    if (ct >= p.g[i].tile_begin) gi = i;
  const GemmGroup& G = p.g[gi];
  const int local = ct - G.tile_begin;
  TileCoord c;
  c.g = &G;
  c.m0 = (local % G.tiles_m) * kBM;  // m fastest: neighbouring CTAs share B
  c.n0 = (local / G.tiles_m) * BN;
  return c;
}

// Epilogue modes (compile-time, so each instance holds only its own
// registers): plain; + bias then ReLU; + bias + fp32 residual, fp32 output;
// + bias + fp32 residual then LayerNorm over the row, bf16 output.
constexpr int kEpiPlain = 0, kEpiBiasRelu = 1, kEpiBiasResF32 = 2, kEpiResLN = 3;

// Tile width BN = 128, or 256 (plain and bias + ReLU only): the wide tile
// takes 1.5x the operand bytes for 2x the FLOPs of a 128-wide one, and
// runs four stages of 48 KB.
template <int EPI, int BN = 128>
struct GemmStages {
  static constexpr int value = EPI == kEpiResLN ? kStagesLN : (BN == 256 ? 4 : kStages);
};
template <int EPI, int BN = 128>
using GemmSmemFor = GemmSmemT<GemmStages<EPI, BN>::value, EPI == kEpiResLN, BN>;

// CN: CTAs per cluster along N sharing a row tile (LayerNorm epilogue only).
template <int EPI, int CN = 1, int BN = 128>
__global__ void __launch_bounds__(kThreads, 1) gemm_bf16_kernel(const __grid_constant__ GemmProblem p) {
  constexpr bool LN = EPI == kEpiResLN;
  constexpr int kSt = GemmStages<EPI, BN>::value;
  constexpr int CS = CN;  // CTAs per cluster
  constexpr int kBBytesT = kBK * BN * 2;           // one stage's B: BN / 64 chunks of 8 KB
  constexpr int kTmemAlloc = LN ? kTmemColsLN : 2 * BN;  // two BN-column accumulators
  static_assert(!LN || (CN >= 1 && CN <= kMaxLnCluster), "LayerNorm clusters");
  static_assert(LN || CN == 1, "clusters along N only for the LayerNorm epilogue");
  static_assert(BN == 128 || (BN == 256 && (EPI == kEpiPlain || EPI == kEpiBiasRelu)),
                "wide tiles: plain and bias + ReLU epilogues");
  using Smem = GemmSmemFor<EPI, BN>;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = warp_id();
  const uint32_t lane = lane_id();
  const int kblocks = (p.K + kBK - 1) / kBK;
  const int rank = CS > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  // cluster tiles of this CTA's cluster: cluster id, + number of clusters, ...
  const int first = static_cast<int>(blockIdx.x) / CS;
  const int stride = static_cast<int>(gridDim.x) / CS;
  // this CTA's output tile of cluster tile ct (LayerNorm: row tile ct,
  // column block = rank)
  auto coord = [&](int ct) -> TileCoord {
    if constexpr (LN) {
      TileCoord c;
      c.g = &p.g[0];
      c.m0 = ct * kBM;
      c.n0 = rank * kBN;
      return c;
    } else {
      return tile_coord<BN>(p, ct);
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);  // released by the MMA warp's commit
    }
    for (int s = 0; s < 2; ++s) mbar_init(&sm.ln_full[s], 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sm.acc_full[a], 1);
      mbar_init(&sm.acc_empty[a], 128);
    }
    mbar_init(&sm.drained, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemAlloc);
    tmem_relinquish();
  }
  tc_fence_before();
  // barriers of every CTA initialised before any peer writes into them
  if constexpr (CS > 1) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile uint32_t* abort_flag = &sm.abort_flag;
  if (warp == 0 && lane == 0) {
    // descriptors live in the kernel parameters: fetched while the previous
    // kernel finishes
    for (int i = 0; i < p.num_groups; ++i) {
      tma_prefetch_desc(&p.g[i].tm_a);
      tma_prefetch_desc(&p.g[i].tm_b);
      tma_prefetch_desc(&p.g[i].tm_c);
    }
  }
  // Everything up to a role's first global-memory access may overlap the
  // previous kernel: the producer waits for it (griddep_wait) before its
  // first load, the epilogue before its first store.
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      if (kPrefetchL2 && first < p.total_tiles) {
        // While the previous kernel finishes, this CTA prefetches into L2 its
        // share of its first tile's B operand (the weights, from DRAM): the
        // CTAs whose first tiles share a column block split its K blocks by
        // their row-tile index. A, usually the previous kernel's output, is
        // left to the loads after the wait.
        const TileCoord c = coord(first);
        const int tm = c.g->tiles_m > 0 ? c.g->tiles_m : 1;
        for (int kb = c.m0 / kBM; kb < kblocks; kb += tm) {
#pragma unroll
          for (int ch = 0; ch < BN / 64; ++ch)
            tma_prefetch_l2_2d(&c.g->tm_b, c.n0 + 64 * ch, kb * kBK);
        }
      }
      for (int ct = first; ok && ct < p.total_tiles; ct += stride) {
        const TileCoord c = coord(ct);
        for (int kb = 0; kb < kblocks; ++kb) {
          const int s = issued % kSt;
          const uint32_t ph = static_cast<uint32_t>(issued / kSt) & 1u;
          // stage released by the MMAs that read it
          if (!mbar_wait(&sm.empty[s], ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm.full[s], kABytes + kBBytesT);
          if (issued == 0) griddep_wait();
          const int k0 = kb * kBK;
          tma_load_2d(sm.a[s], &c.g->tm_a, &sm.full[s], k0, c.m0);
#pragma unroll
          for (int ch = 0; ch < BN / 64; ++ch)  // 64-column chunks of B, kBChunk apart
            tma_load_2d(sm.b[s] + ch * kBChunk, &c.g->tm_b, &sm.full[s], c.n0 + 64 * ch, k0);
          ++issued;
        }
      }
      // Every stage written has been released: no MMA still reads it when the
      // CTA leaves (and, after an abort, no copy of this CTA is in flight).
      volatile uint32_t never = 0;
      for (int i = max(0, issued - kSt); i < issued; ++i)
        mbar_wait(&sm.empty[i % kSt], static_cast<uint32_t>(i / kSt) & 1u,
                  ok ? abort_flag : &never, kDrainLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(kBM, BN, false, true);
      // descriptors built once, advanced inside the start-address field
      const uint64_t da0 = sdesc_sw128(smem_u32(sm.a[0]), 16, 1024);       // K-major A
      const uint64_t db0 = sdesc_sw128(smem_u32(sm.b[0]), kBChunk, 1024);  // N-major B
      int consumed = 0;
      int it = 0;
      bool ok = true;
      for (int ct = first; ok && ct < p.total_tiles; ct += stride, ++it) {
        const int acc = it & 1;
        // the epilogue has read this accumulator's previous tile
        ok = mbar_wait(&sm.acc_empty[acc], (static_cast<uint32_t>(it >> 1) & 1u) ^ 1u, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          const int s = consumed % kSt;
          ok = mbar_wait(&sm.full[s], static_cast<uint32_t>(consumed / kSt) & 1u, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t da = sdesc_advance(da0, static_cast<uint32_t>(s) * (kABytes >> 4));
          const uint64_t db = sdesc_advance(db0, static_cast<uint32_t>(s) * (kBBytesT >> 4));
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
    // Every thread that touches global memory waits for the previous grid
    // first: the leader before its stores; with an epilogue, every thread
    // (bias and residual may come from earlier kernels, and the fp32 output
    // is stored directly). Kernels release their dependents at entry, so
    // without the wait this grid can run beside a kernel two launches back
    // when the one in between leaves SMs free.
    if (EPI != kEpiPlain || leader) griddep_wait();
    int it = 0;
    for (int ct = first; ct < p.total_tiles; ct += stride, ++it) {
      const int acc = it & 1;
      const TileCoord c = coord(ct);
      // the group's fields once into registers (reads through the pointer
      // into the parameter space would be repeated past every store)
      const uint16_t* const g_bias = c.g->bias;
      const float* const g_res32 = c.g->residual_f32;
      float* const g_c32 = c.g->c_f32;
      const int64_t g_ldr = c.g->ldr;
      const int g_N = c.g->N;
      const int row = c.m0 + r;
      const bool row_ok = row < c.g->M;
      // bias and residual of chunk cc (32 columns) of this thread's row
      auto load_bias = [&](int cc, uint4 (&bw)[4]) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int col = c.n0 + cc * 32 + 8 * k;
          bw[k] = col < g_N ? __ldg(reinterpret_cast<const uint4*>(g_bias + col))
                            : make_uint4(0u, 0u, 0u, 0u);
        }
      };
      auto load_res = [&](int cc, float4 (&rf)[8]) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int col = c.n0 + cc * 32 + 4 * k;
          rf[k] = (col < g_N && row_ok)
                      ? __ldg(reinterpret_cast<const float4*>(g_res32 + row * g_ldr + col))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      };
      // the first chunk's operands (the whole tile's bias with ReLU) are
      // loaded while the main loop runs, later chunks' during the previous
      constexpr bool kBiasAll = EPI == kEpiBiasRelu && BN == 128;  // wide tiles: chunk by chunk
      uint4 bias_all[kBiasAll ? kBN / 8 : 1];
      uint4 bw_next[4];
      float4 rf_next[(EPI == kEpiBiasResF32 || LN) ? 8 : 1];
      if constexpr (kBiasAll) {
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc)
          load_bias(cc, *reinterpret_cast<uint4(*)[4]>(bias_all + 4 * cc));
      }
      if constexpr (EPI == kEpiBiasRelu && !kBiasAll) load_bias(0, bw_next);
      if constexpr (EPI == kEpiBiasResF32) {
        load_bias(0, bw_next);
        load_res(0, *reinterpret_cast<float4(*)[8]>(rf_next));
      }
      if constexpr (LN) {
        // The tile's residual rows -> tensor memory while the MMAs run (this
        // warp's previous reads of the region finished with the last tile):
        // the loads of the next 32 columns are in flight while one chunk is
        // stored, and the epilogue later reads them back at TMEM latency.
        const uint32_t res_addr = tmem + lane_base + kResCol;
        load_res(0, *reinterpret_cast<float4(*)[8]>(rf_next));
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc) {
          float4 rf[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) rf[k] = rf_next[k];
          if (cc + 1 < kBN / 32) load_res(cc + 1, *reinterpret_cast<float4(*)[8]>(rf_next));
          uint32_t w[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            w[4 * k] = __float_as_uint(rf[k].x);
            w[4 * k + 1] = __float_as_uint(rf[k].y);
            w[4 * k + 2] = __float_as_uint(rf[k].z);
            w[4 * k + 3] = __float_as_uint(rf[k].w);
          }
          tmem_st32(res_addr + cc * 32, w);
        }
        tmem_wait_st();
        load_bias(0, bw_next);
      }
      bool ok = __all_sync(
          0xffffffffu,
          mbar_wait(&sm.acc_full[acc], static_cast<uint32_t>(it >> 1) & 1u, abort_flag));
      // this staging tile was last written out kCStages tiles ago: its store
      // must have finished reading shared memory before it is overwritten
      if (leader) bulk_wait_group_read<kCStages - 1>();
      // one decision for all four warps: none is left waiting at a barrier
      ok = named_bar_and<kEpiBarrier>(128, ok);
      if (!ok) break;
      tc_fence_after();
      // 32 columns at a time: TMEM -> registers, the epilogue's additions
      // (their loads issued before the TMEM wait), then bf16 into the
      // swizzled staging tile or fp32 straight to global memory
      uint8_t* stage = sm.c[it % kCStages];
      if constexpr (LN) {
        const uint32_t acc_addr = tmem + lane_base + acc * kAccCols;
        const uint16_t* const g_gamma = c.g->ln_gamma;
        const uint16_t* const g_beta = c.g->ln_beta;
        // (1) v = acc + bias + residual (fp32), written back over the
        // accumulator; the sum of this CTA's 128 columns
        const uint32_t res_addr = tmem + lane_base + kResCol;
        float s1 = 0.f;
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc) {
          uint32_t x[32], rs[32];
          tmem_ld32(acc_addr + cc * 32, x);
          tmem_ld32(res_addr + cc * 32, rs);
          uint4 bw[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) bw[k] = bw_next[k];
          if (cc + 1 < kBN / 32) load_bias(cc + 1, bw_next);  // in flight meanwhile
          float add[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) add[i] = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            add_bf16x8(*reinterpret_cast<float(*)[8]>(add + 8 * k), bw[k]);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float v = __uint_as_float(x[i]) + __uint_as_float(rs[i]) + add[i];
            x[i] = __float_as_uint(v);
            s1 += v;
          }
          tmem_st32(acc_addr + cc * 32, x);
        }
        tmem_wait_st();
        const float mean_l = s1 * (1.f / kBN);
        // (2) the centred sum of squares over the same columns
        float m2 = 0.f;
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc) {
          uint32_t x[32];
          tmem_ld32(acc_addr + cc * 32, x);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float d = __uint_as_float(x[i]) - mean_l;
            m2 = fmaf(d, d, m2);
          }
        }
        // (3) the pair to every other CTA of the cluster: slot (tile
        // parity, this CTA's index among the receiver's others, row)
        const int slot = it & 1;
#pragma unroll
        for (int q = 0; q < CS; ++q) {
          if (q == rank) continue;
          const int idx = rank < q ? rank : rank - 1;
          st_async_f32x2(cluster_map(&sm.ln_stat[slot][idx][r], static_cast<uint32_t>(q)), mean_l,
                         m2, cluster_map(&sm.ln_full[slot], static_cast<uint32_t>(q)));
        }
        if (r == 0) mbar_arrive_expect_tx(&sm.ln_full[slot], (CS - 1) * kBM * 8);
        // gamma and beta of the first chunk while the pairs travel
        uint4 gw[4], btw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          gw[k] = __ldg(reinterpret_cast<const uint4*>(g_gamma + c.n0 + 8 * k));
          btw[k] = __ldg(reinterpret_cast<const uint4*>(g_beta + c.n0 + 8 * k));
        }
        bool okl = __all_sync(0xffffffffu,
                              mbar_wait_cluster(&sm.ln_full[slot], static_cast<uint32_t>(it >> 1) & 1u,
                                                abort_flag));
        // one decision for all four warps before the staging barrier below
        okl = named_bar_and<kEpiBarrier>(128, okl);
        if (!okl) break;
        // (4) the row's mean and variance over all CS x 128 columns
        float mean = mean_l;
#pragma unroll
        for (int q = 0; q < CS - 1; ++q) mean += sm.ln_stat[slot][q][r].x;
        mean *= 1.f / CS;
        float dm = mean_l - mean;
        float M2 = fmaf(static_cast<float>(kBN) * dm, dm, m2);
#pragma unroll
        for (int q = 0; q < CS - 1; ++q) {
          const float2 st = sm.ln_stat[slot][q][r];
          dm = st.x - mean;
          M2 += fmaf(static_cast<float>(kBN) * dm, dm, st.y);
        }
        const float rstd = rsqrtf(M2 * (1.f / (kBN * CS)) + c.g->ln_eps);
        // (5) (v - mean) * rstd * gamma + beta -> bf16 staging tile
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc) {
          uint32_t x[32];
          tmem_ld32(acc_addr + cc * 32, x);
          float g[32], bt[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) g[i] = bt[i] = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            add_bf16x8(*reinterpret_cast<float(*)[8]>(g + 8 * k), gw[k]);
            add_bf16x8(*reinterpret_cast<float(*)[8]>(bt + 8 * k), btw[k]);
          }
          if (cc + 1 < kBN / 32) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              gw[k] = __ldg(reinterpret_cast<const uint4*>(g_gamma + c.n0 + (cc + 1) * 32 + 8 * k));
              btw[k] = __ldg(reinterpret_cast<const uint4*>(g_beta + c.n0 + (cc + 1) * 32 + 8 * k));
            }
          }
          tmem_wait_ld();
          if (cc == kBN / 32 - 1) {
            tc_fence_before();
            mbar_arrive(&sm.acc_empty[acc]);  // the MMA warp may reuse this accumulator
          }
          float y[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = fmaf((__uint_as_float(x[i]) - mean) * rstd, g[i], bt[i]);
          if (row_ok) {
            uint16_t* dst = c.g->c + static_cast<int64_t>(row) * c.g->ldc + c.n0 + cc * 32;
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              const float* e = y + 8 * v4;
              st_global_v4(dst + 8 * v4, pack_bf16x2(e[0], e[1]), pack_bf16x2(e[2], e[3]),
                           pack_bf16x2(e[4], e[5]), pack_bf16x2(e[6], e[7]));
            }
          }
        }
        continue;  // rows stored: no staging tile in this mode
      } else {
#pragma unroll
      for (int cc = 0; cc < BN / 32; ++cc) {
        if (BN > 128 && cc > 0 && cc % 4 == 0) {
          // wide tile: the staged 128-column half goes out, and the staging
          // tile is free again once its store has read it (every warp here)
          fence_proxy_async_smem();
          named_bar_sync<kEpiBarrier>(128);
          if (leader && c.m0 < c.g->M) {
            const int nh = c.n0 + (cc - 4) * 32;
            tma_store_2d(&c.g->tm_c, stage, nh, c.m0);
            if (nh + 64 < c.g->N) tma_store_2d(&c.g->tm_c, stage + 16384, nh + 64, c.m0);
            bulk_commit_group();
            bulk_wait_group_read<0>();
          }
          named_bar_sync<kEpiBarrier>(128);
        }
        const int hc = cc % 4;  // chunk within the staged 128-column half
        uint32_t x[32];
        tmem_ld32(tmem + lane_base + acc * BN + cc * 32, x);
        float add[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) add[i] = 0.f;
        if constexpr (kBiasAll) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            add_bf16x8(*reinterpret_cast<float(*)[8]>(add + 8 * k), bias_all[cc * 4 + k]);
        } else if constexpr (EPI == kEpiBiasRelu) {
          uint4 bw[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) bw[k] = bw_next[k];
          if (cc + 1 < BN / 32) load_bias(cc + 1, bw_next);  // in flight meanwhile
#pragma unroll
          for (int k = 0; k < 4; ++k)
            add_bf16x8(*reinterpret_cast<float(*)[8]>(add + 8 * k), bw[k]);
        }
        if constexpr (EPI == kEpiBiasResF32) {
          uint4 bw[4];
          float4 rf[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) bw[k] = bw_next[k];
#pragma unroll
          for (int k = 0; k < 8; ++k) rf[k] = rf_next[k];
          if (cc + 1 < kBN / 32) {  // the next chunk's, in flight meanwhile
            load_bias(cc + 1, bw_next);
            load_res(cc + 1, *reinterpret_cast<float4(*)[8]>(rf_next));
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            add_bf16x8(*reinterpret_cast<float(*)[8]>(add + 8 * k), bw[k]);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            add[4 * k] += rf[k].x;
            add[4 * k + 1] += rf[k].y;
            add[4 * k + 2] += rf[k].z;
            add[4 * k + 3] += rf[k].w;
          }
        }
        tmem_wait_ld();
        if (cc == BN / 32 - 1) {
          tc_fence_before();
          mbar_arrive(&sm.acc_empty[acc]);  // the MMA warp may reuse this accumulator
        }
        float y[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          y[i] = __uint_as_float(x[i]) + add[i];
          if constexpr (EPI == kEpiBiasRelu) y[i] = fmaxf(y[i], 0.f);
        }
        if constexpr (EPI == kEpiBiasResF32) {
          if (row_ok) {
            float* dst = g_c32 + static_cast<int64_t>(row) * g_N + c.n0 + cc * 32;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (c.n0 + cc * 32 + 4 * k < g_N)
                *reinterpret_cast<float4*>(dst + 4 * k) =
                    make_float4(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]);
          }
        } else {
          // 128-byte swizzle of the store's tensor map: the 16-byte chunk j of
          // row r sits at chunk position j ^ (r mod 8) of the row's 128 bytes
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const int j = (hc & 1) * 4 + v4;
            const float* e = y + 8 * v4;
            st_shared_v4(smem_u32(stage + (hc >> 1) * 16384 + r * 128 + ((j ^ (r & 7)) << 4)),
                         pack_bf16x2(e[0], e[1]), pack_bf16x2(e[2], e[3]),
                         pack_bf16x2(e[4], e[5]), pack_bf16x2(e[6], e[7]));
          }
        }
      }
      }  // LN
      fence_proxy_async_smem();  // staged bytes visible to the TMA unit
      named_bar_sync<kEpiBarrier>(128);
      // a cluster's last row tiles may lie past M: computed on zero rows, not stored
      if (leader && c.m0 < c.g->M && EPI != kEpiBiasResF32) {
        // the map clips rows past M and columns past N (the last 128-column
        // half of a wide tile)
        const int nh = c.n0 + BN - 128;
        tma_store_2d(&c.g->tm_c, stage, nh, c.m0);
        if (nh + 64 < c.g->N) tma_store_2d(&c.g->tm_c, stage + 16384, nh + 64, c.m0);
        bulk_commit_group();
      }
    }
    // the stores have read the staging tile before the CTA's shared memory
    // goes; their global writes complete with the grid
    if (leader) bulk_wait_group_read<0>();
  }

  tc_fence_before();
  // no CTA leaves while a peer may still write into its shared memory
  if constexpr (CS > 1) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemAlloc);
}

int num_sms() {
  static int cached = 0;  // atomic accesses: launches may come from several host threads
  int n = __atomic_load_n(&cached, __ATOMIC_RELAXED);
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    __atomic_store_n(&cached, n, __ATOMIC_RELAXED);
  }
  return n;
}

}  // namespace

static_assert(sizeof(GemmSmemFor<kEpiPlain>) + 1024 <= 227 * 1024, "shared memory per CTA");
static_assert(sizeof(GemmSmemFor<kEpiPlain, 256>) + 1024 <= 227 * 1024, "shared memory per CTA");
static_assert(sizeof(GemmSmemFor<kEpiResLN>) + 1024 <= 227 * 1024, "shared memory per CTA");

// The LayerNorm epilogue: one group, clusters of N / 128 CTAs along N, one
// row tile per cluster step.
template <int CN>
cudaError_t launch_gemm_ln(const GemmProblem& problem, cudaStream_t stream) {
  GemmProblem p = problem;
  p.g[0].tile_begin = 0;
  p.total_tiles = p.g[0].tiles_m;
  if (p.total_tiles <= 0) return cudaSuccess;
  auto kernel = gemm_bf16_kernel<kEpiResLN, CN>;
  const size_t smem_bytes = sizeof(GemmSmemFor<kEpiResLN>) + 1024;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(kernel, static_cast<int>(smem_bytes), &configured);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CN;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  static int cached_clusters = 0;  // atomic accesses, as num_sms()
  int max_clusters = __atomic_load_n(&cached_clusters, __ATOMIC_RELAXED);
  if (max_clusters == 0) {
    cfg.gridDim = dim3(num_sms() / CN * CN);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    max_clusters = n > 0 ? n : 1;
    __atomic_store_n(&cached_clusters, max_clusters, __ATOMIC_RELAXED);
  }
  const int clusters = p.total_tiles < max_clusters ? p.total_tiles : max_clusters;
  cfg.gridDim = dim3(clusters * CN);
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t launch_gemm_bf16(const GemmProblem& problem, cudaStream_t stream) {
  if (problem.g[0].ln_gamma != nullptr) {
    const GemmGroup& g = problem.g[0];
    if (problem.num_groups != 1 || g.bias == nullptr || g.residual_f32 == nullptr ||
        g.ln_beta == nullptr || g.relu || g.c_f32 != nullptr || !(g.ln_eps > 0.f))
      return cudaErrorInvalidValue;
    switch (g.N) {
      case 128: return launch_gemm_ln<1>(problem, stream);
      case 256: return launch_gemm_ln<2>(problem, stream);
      case 512: return launch_gemm_ln<4>(problem, stream);
      case 1024: return launch_gemm_ln<8>(problem, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  GemmProblem p = problem;
  // one epilogue mode per launch (every group's fields must agree)
  const GemmGroup& g0 = p.g[0];
  int epi = kEpiPlain;
  if (g0.c_f32 != nullptr) {
    if (g0.bias == nullptr || g0.residual_f32 == nullptr || g0.relu) return cudaErrorInvalidValue;
    epi = kEpiBiasResF32;
  } else if (g0.bias != nullptr || g0.relu) {
    if (g0.bias == nullptr || !g0.relu || g0.residual_f32 != nullptr) return cudaErrorInvalidValue;
    epi = kEpiBiasRelu;
  }
  for (int i = 1; i < p.num_groups; ++i)
    if (p.g[i].bias != g0.bias || p.g[i].relu != g0.relu || p.g[i].c_f32 != nullptr ||
        p.g[i].residual_f32 != nullptr)
      return cudaErrorInvalidValue;
  for (int i = 0; i < p.num_groups; ++i)
    if (p.g[i].ln_gamma != nullptr) return cudaErrorInvalidValue;
  // 256-column tiles (plain and bias + ReLU, every N a multiple of 256) when
  // their waves cost less: a wide tile moves 1.5x the operand bytes of a
  // 128-column one (the loads set the pace), so wide wins when
  // 1.5 x (its waves) < the narrow tiles' waves over the SMs; and only with
  // three waves or more (measured: the encoder layer's 4096 x 2048 x 512 FFN
  // GEMM, two wide waves, was faster alone but slower inside the layer)
  bool wide = epi == kEpiPlain || epi == kEpiBiasRelu;
  long long wide_tiles = 0, narrow_tiles = 0;
  for (int i = 0; i < p.num_groups; ++i) {
    if (p.g[i].N % 256 != 0) wide = false;
    const long long rows = p.g[i].tiles_m;
    wide_tiles += rows * (p.g[i].N / 256);
    narrow_tiles += rows * ((p.g[i].N + 127) / 128);
  }
  const long long sms = num_sms();
  const long long wide_waves = (wide_tiles + sms - 1) / sms;
  if (wide_waves < 3 || 3 * wide_waves >= 2 * ((narrow_tiles + sms - 1) / sms)) wide = false;
  const int bn = wide ? 256 : 128;
  int t = 0;
  for (int i = 0; i < p.num_groups; ++i) {
    p.g[i].tiles_n = (p.g[i].N + bn - 1) / bn;
    p.g[i].tile_begin = t;
    t += p.g[i].tiles_m * p.g[i].tiles_n;
  }
  p.total_tiles = t;
  if (t <= 0) return cudaSuccess;
  auto kernel = wide ? (epi == kEpiPlain ? gemm_bf16_kernel<kEpiPlain, 1, 256>
                                         : gemm_bf16_kernel<kEpiBiasRelu, 1, 256>)
            : epi == kEpiPlain      ? gemm_bf16_kernel<kEpiPlain>
            : epi == kEpiBiasRelu ? gemm_bf16_kernel<kEpiBiasRelu>
                                    : gemm_bf16_kernel<kEpiBiasResF32>;
  const size_t smem_bytes =
      (wide ? sizeof(GemmSmemFor<kEpiPlain, 256>) : sizeof(GemmSmemFor<kEpiPlain>)) + 1024;
  static unsigned long long configured[5] = {0, 0, 0, 0, 0};
  cudaError_t e = set_smem_once(kernel, static_cast<int>(smem_bytes),
                                &configured[wide ? 3 + epi : epi]);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent: one CTA per SM (the tensor-memory allocation keeps a second
  // CTA off the SM)
  cfg.gridDim = dim3(static_cast<unsigned>(t < sms ? t : sms));
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

TSD_DEFINE_ERROR_READER(take_device_error_gemm)

}  // namespace tsd
