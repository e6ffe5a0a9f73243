// mha_fused.cu -- multi-head attention for short sequences (n_q, n_k <= 128,
// d_k = d_v = 64) in one kernel up to the merged heads: the Q/K/V projections
// of a head pair, their scaled dot-product attention, and the heads written
// side by side ("[논문 리뷰]Attention Is All You Need" (kimjiil.github.io),
// sections 3.2.1-3.2.2: head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V);
// weights in the x.W layout, [d_model, h*d], no biases), and optionally the
// output projection of section 3.2.2 as well (MultiHead = Concat(heads) W_O).
//
// Why fuse: at these sizes the three-kernel path is latency-bound. The
// projection GEMM's operand traffic from L2 is its limit, the attention
// kernel is one short dependency chain per head, and Q/K/V make a round trip
// through memory in between. Here a CTA owns one work item, (batch b, heads
// 2p and 2p+1), so the batch's X tile is loaded once for both heads, and Q,
// K and V never leave the SM.
//
//   warp 0      TMA producer: per 64-wide slice of d_model, X's 128 x 64 tile
//               (and X_kv's, for cross-attention) and the six 64 x 64 weight
//               slices (W_Q, W_K, W_V of both heads), kStages deep
//   warp 1      MMA issuer (one thread): projection MMAs (per head one N=192
//               MMA [Q|K|V] per 16-deep step, or N=64 and N=128 for
//               cross-attention), then per head S = Q K^T and O = P V
//   warps 4..7  head 2p, warps 8..11 head 2p+1, one thread per row (= TMEM
//               lane): (1) the head's projection accumulator row (fp32) ->
//               bf16 rows of 128-byte-swizzled Q, K, V tiles written into the
//               projection ring's memory (now free), Q and K first so the S
//               MMA overlaps V's conversion; (2) the softmax of the
//               single 128 x 128 score tile (masked logits -inf before max and
//               exp2, scale*log2(e) folded); (3) O / l -> bf16 -> swizzled
//               staging -> one TMA store into the merged [B, n_q, h*d] layout
//
// Tensor memory (512 columns): projection accumulators of head e at
// [192e, 192e+192) (Q | K | V); afterwards S_e overwrites Q|K of its own head
// and P_e (bf16) its V part; O_e lives at [384 + 64e, 448 + 64e).
// Rows past n_q / n_k are zero (the tensor maps clip them); they produce
// nothing: keys past n_k are masked, query rows past n_q are not stored.
//
// With the output projection (OUT): the h/2 CTAs of one batch entry form a
// cluster, CTA r owning head pair r and output columns [N r, N r + N),
// N = d_model / (h/2) (64 or 128). Each CTA still stores its two heads into
// the merged buffer; once a store has completed, its head leader signals
// every peer (st.async of a word into the peer's shared memory, complete_tx
// on the peer's mbarrier for this CTA, release at cluster scope). The
// producer of each CTA, having acquired a peer's signals, loads its merged
// tiles back from L2 into the space its own Q/K/V tiles used (6 slots of
// 16 KB), and streams
// the W_O rows of all h heads, columns [N r, N r + N), through the rest of
// the ring (W_O's first chunks already during the attention). The MMA
// warp accumulates out = sum_j head_j W_O[64 j : 64 j + 64, cols] over the
// heads, its own two read straight from the epilogue's staging tiles, into
// TMEM columns [0, N); the head warpgroups store it (bf16) to `out`.
// Moving the merged tiles through L2 rather than distributed shared memory
// is measured, not assumed: on GB300 a CTA receives about 155 GB/s from L2
// by TMA but only about 20 GB/s from the other CTAs of its cluster.
#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kRows = 128;              // query rows and key rows per tile
constexpr int kD = 64;                  // d_k = d_v
constexpr int kTile = kRows * kD * 2;   // 16 KB: a 128 x 64 bf16 tile
constexpr int kWChunk = 64 * kD * 2;    // 8 KB: 64 rows of d_model x 64 columns of one weight
constexpr int kThreads = 384;           // 4 control warps + 2 softmax warpgroups
constexpr uint32_t kLaunchRegs = 65536 / kThreads / 8 * 8;  // 168
constexpr uint32_t kCtrlRegs = 72;
constexpr uint32_t kSoftmaxRegs = (kLaunchRegs * kThreads - kCtrlRegs * 128) / 256 / 8 * 8;
static_assert(kCtrlRegs * 128 + kSoftmaxRegs * 256 <= kLaunchRegs * kThreads, "register split");
constexpr unsigned long long kDrainLimitNs = 100ull * 1000ull * 1000ull;
constexpr bool kPrefetchL2 = true;  // a share of the first wave's operands into L2 before the wait
// output projection (OUT)
constexpr int kSlot = 16384;    // a 128 x 64 merged-heads tile, or 64 rows of W_O x <= 128 columns
constexpr int kOSlots = 6;      // peers' merged tiles, where the Q/K/V tiles were
constexpr int kMaxCluster = 8;  // head pairs per batch entry (portable cluster size)

template <bool SELF>
struct FusedSmem {
  static constexpr int kStages = SELF ? 3 : 2;
  static constexpr int kABytes = SELF ? kTile : 2 * kTile;  // X (and X_kv): 128 rows x 64
  static constexpr int kStageBytes = kABytes + 6 * kWChunk;
  // The projection ring. Once a work item's projections are done, its first
  // 96 KB hold the item's bf16 Q, K, V tiles of both heads (tile 3e + 0/1/2).
  alignas(1024) uint8_t ring[kStages][kStageBytes];
  alignas(1024) uint8_t o[2][kTile];  // epilogue staging, one per head
  uint64_t full[kStages], empty[kStages];
  uint64_t proj_done, qkv_free, tmem_free;
  uint64_t qk_ready[2], v_ready[2], s_full[2], p_full[2], pv_done[2];
  uint64_t drained;
  // output projection (OUT): peer tiles in ring slots [0, kOSlots), W_O
  // chunks in the slots after them
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kWoSlots = (kRingBytes - kOSlots * kSlot) / kSlot;  // self 6, cross 4
  uint64_t o_full[kOSlots], o_empty[kOSlots];
  uint64_t wo_full[kWoSlots], wo_empty[kWoSlots];
  uint64_t o_staged;   // this CTA's two merged tiles are in o[] (256 arrivals)
  uint64_t out_done;   // every out-projection MMA of the item has completed
  // peer slot s's merged tiles are in global memory (item parity): two 4-byte
  // signals (one per head) into o_words
  uint64_t o_ready[2][kMaxCluster - 1];
  uint32_t o_words[2][kMaxCluster - 1][2];
  uint32_t tmem_base;
  uint32_t abort_flag;
  static_assert(kStages * kStageBytes >= 6 * kTile, "Q/K/V tiles fit in the ring");
  static_assert(kOSlots * kSlot == 6 * kTile, "peer tiles take the Q/K/V tiles' place");
  static_assert(kWoSlots >= 2, "W_O ring");
};

struct FusedArgs {
  int h, n_q, n_k, kblocks, num_units, head_pairs;
  int mask_kind;
  const int32_t* kv_lens;
  float scale_log2;
  int n_slice;  // OUT: output columns per CTA (64 or 128)
};

template <bool SELF, bool OUT>
__global__ void __launch_bounds__(kThreads, 1)
    mha_fused_kernel(const __grid_constant__ CUtensorMap tm_xq,
                     const __grid_constant__ CUtensorMap tm_xkv,
                     const __grid_constant__ CUtensorMap tm_wq,
                     const __grid_constant__ CUtensorMap tm_wk,
                     const __grid_constant__ CUtensorMap tm_wv,
                     const __grid_constant__ CUtensorMap tm_o,
                     const __grid_constant__ CUtensorMap tm_wo,
                     const __grid_constant__ CUtensorMap tm_out, const FusedArgs args) {
  using Smem = FusedSmem<SELF>;
  constexpr int kStages = Smem::kStages;
  constexpr int kWoSlots = Smem::kWoSlots;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = warp_id();
  const uint32_t lane = lane_id();
  const int first = static_cast<int>(blockIdx.x);
  const int stride = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.proj_done, 1);
    mbar_init(&sm.qkv_free, 1);
    mbar_init(&sm.tmem_free, 256);  // every softmax thread, after its last TMEM read
    for (int e = 0; e < 2; ++e) {
      mbar_init(&sm.qk_ready[e], 128);
      mbar_init(&sm.v_ready[e], 128);
      mbar_init(&sm.s_full[e], 1);
      mbar_init(&sm.p_full[e], 128);
      mbar_init(&sm.pv_done[e], 1);
    }
    mbar_init(&sm.drained, 1);
    if constexpr (OUT) {
      for (int i = 0; i < kOSlots; ++i) {
        mbar_init(&sm.o_full[i], 1);
        mbar_init(&sm.o_empty[i], 1);
      }
      for (int i = 0; i < kWoSlots; ++i) {
        mbar_init(&sm.wo_full[i], 1);
        mbar_init(&sm.wo_empty[i], 1);
      }
      mbar_init(&sm.o_staged, 256);
      mbar_init(&sm.out_done, 1);
      for (int p = 0; p < 2; ++p)
        for (int i = 0; i < kMaxCluster - 1; ++i) mbar_init(&sm.o_ready[p][i], 1);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  // peers arrive on this CTA's barriers: every CTA of the cluster has
  // initialised its own first
  if constexpr (OUT) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile uint32_t* abort_flag = &sm.abort_flag;
  if (warp == 0 && lane == 0) {
    // descriptors live in the kernel parameters: fetched while the previous
    // kernel finishes
    tma_prefetch_desc(&tm_xq);
    if constexpr (!SELF) tma_prefetch_desc(&tm_xkv);
    tma_prefetch_desc(&tm_wq);
    tma_prefetch_desc(&tm_wk);
    tma_prefetch_desc(&tm_wv);
    tma_prefetch_desc(&tm_o);
    if constexpr (OUT) {
      tma_prefetch_desc(&tm_wo);
      tma_prefetch_desc(&tm_out);
    }
  }
  // Everything up to a role's first global-memory access may overlap the
  // previous kernel: each role waits for it (griddep_wait) just before.
  griddep_launch_dependents();

  if (warp < 4) {
    regs_decrease<kCtrlRegs>();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ producer
      int issued = 0, ui = 0, wo_cnt = 0, o_cnt = 0, armed = -1;
      bool ok = true;
      if (kPrefetchL2 && first < args.num_units) {
        // While the previous kernel finishes, this CTA prefetches into L2 its
        // share of the data the first wave of CTAs reads: 1/C of its batch
        // entry's X rows (the C CTAs of a batch entry split them), and, CTA
        // b of each head pair, one 64-row block of the pair's W_Q, W_K, W_V
        // slices and of its W_O columns; the loads after the wait find them
        // there. A prefetch only reads into L2, the point of coherence.
        const int C = args.head_pairs;
        const int b = first / C;
        const int pair = first % C;
        for (int kb = pair; kb < args.kblocks; kb += C) {
          tma_prefetch_l2_3d(&tm_xq, kb * 64, 0, b);
          if constexpr (!SELF) tma_prefetch_l2_3d(&tm_xkv, kb * 64, 0, b);
        }
        if (b < args.kblocks) {
          for (int e = 0; e < 2; ++e) {
            const int col = (2 * pair + e) * kD;
            tma_prefetch_l2_2d(&tm_wq, col, b * 64);
            tma_prefetch_l2_2d(&tm_wk, col, b * 64);
            tma_prefetch_l2_2d(&tm_wv, col, b * 64);
          }
        }
        if constexpr (OUT) {
          if (b < 2 * C)
            for (int c = 0; c < args.n_slice; c += 64)
              tma_prefetch_l2_2d(&tm_wo, pair * args.n_slice + c, b * kD);
        }
      }
      for (int u = first; ok && u < args.num_units; u += stride, ++ui) {
        const int b = u / args.head_pairs;
        const int pair = u % args.head_pairs;
        const int h0 = 2 * pair;
        // the previous item's tiles in the ring (Q/K/V; with OUT also the
        // peers' merged tiles and W_O) have been consumed
        if (ui > 0) {
          ok = mbar_wait(OUT ? &sm.out_done : &sm.qkv_free, static_cast<uint32_t>(ui - 1) & 1u,
                         abort_flag);
          if (!ok) break;
        }
        if constexpr (OUT) {
          // expect the peers' signals for this item (2 x 4 bytes per peer);
          // they may land before this, the phase completes with both
          for (int s = 0; s < args.head_pairs - 1; ++s)
            mbar_arrive_expect_tx(&sm.o_ready[ui & 1][s], 8);
          armed = ui;
        }
        for (int kb = 0; kb < args.kblocks; ++kb) {
          const int s = issued % kStages;
          ok = mbar_wait(&sm.empty[s], (static_cast<uint32_t>(issued / kStages) & 1u) ^ 1u,
                         abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&sm.full[s], Smem::kStageBytes);
          if (issued == 0) griddep_wait();
          const int k0 = kb * 64;
          uint8_t* st = sm.ring[s];
          tma_load_3d(st, &tm_xq, &sm.full[s], k0, 0, b);
          if constexpr (!SELF) tma_load_3d(st + kTile, &tm_xkv, &sm.full[s], k0, 0, b);
          uint8_t* w = st + Smem::kABytes;
          for (int e = 0; e < 2; ++e) {
            const int col = (h0 + e) * kD;
            tma_load_2d(w + (3 * e + 0) * kWChunk, &tm_wq, &sm.full[s], col, k0);
            tma_load_2d(w + (3 * e + 1) * kWChunk, &tm_wk, &sm.full[s], col, k0);
            tma_load_2d(w + (3 * e + 2) * kWChunk, &tm_wv, &sm.full[s], col, k0);
          }
          ++issued;
        }
        if constexpr (OUT) {
          if (!ok) break;
          const int C = args.head_pairs;
          // chunk j of the output projection: head 2 ((pair + j/2) mod C) + j%2
          // (this CTA's own two heads first)
          auto head_of = [&](int j) { return 2 * ((pair + (j >> 1)) % C) + (j & 1); };
          auto issue_wo = [&](int j) -> bool {  // W_O rows of head j, this CTA's columns
            const int s = wo_cnt % kWoSlots;
            if (!mbar_wait(&sm.wo_empty[s], (static_cast<uint32_t>(wo_cnt / kWoSlots) & 1u) ^ 1u,
                           abort_flag))
              return false;
            uint8_t* dst = sm.ring[0] + (kOSlots + s) * kSlot;
            mbar_arrive_expect_tx(&sm.wo_full[s], static_cast<uint32_t>(args.n_slice) * 128u);
            for (int c = 0; c < args.n_slice; c += 64)
              tma_load_2d(dst + c * 128, &tm_wo, &sm.wo_full[s], pair * args.n_slice + c,
                          head_of(j) * kD);
            ++wo_cnt;
            return true;
          };
          auto issue_o = [&](int j) -> bool {  // a peer's merged tile of head j
            const int s = o_cnt % kOSlots;
            if (!mbar_wait(&sm.o_empty[s], (static_cast<uint32_t>(o_cnt / kOSlots) & 1u) ^ 1u,
                           abort_flag))
              return false;
            mbar_arrive_expect_tx(&sm.o_full[s], kTile);
            tma_load_3d(sm.ring[0] + s * kSlot, &tm_o, &sm.o_full[s], head_of(j) * kD, 0, b);
            ++o_cnt;
            return true;
          };
          const uint32_t ph = static_cast<uint32_t>(ui) & 1u;
          // W_O's first chunks while the attention runs: the projection
          // stages are free once every projection MMA has completed
          ok = mbar_wait(&sm.proj_done, ph, abort_flag);
          int wj = 0;
          for (; ok && wj < args.h && wj < kWoSlots; ++wj) ok = issue_wo(wj);
          // the W_O chunks whose slots the own heads' MMAs free (those need
          // nothing from the peers), then the peers' merged tiles, into the
          // Q/K/V tiles' place once those are consumed, each peer's as soon
          // as it has stored them
          for (; ok && wj < args.h && wj < kWoSlots + 2; ++wj) ok = issue_wo(wj);
          ok = ok && mbar_wait(&sm.qkv_free, ph, abort_flag);
          for (int j = 2; ok && j < args.h; ++j) {
            if ((j & 1) == 0) {
              ok = mbar_wait_cluster(&sm.o_ready[ui & 1][(j >> 1) - 1],
                                     static_cast<uint32_t>(ui >> 1) & 1u, abort_flag);
              fence_proxy_async_global();  // before the TMA reads what the peer's TMA wrote
            }
            ok = ok && issue_o(j);
            while (ok && wj <= j) ok = issue_wo(wj++);
          }
          while (ok && wj < args.h) ok = issue_wo(wj++);
        }
      }
      if (!ok) {
        // wait (bounded) for this thread's copies still in flight
        volatile uint32_t never = 0;
        for (int i = max(0, issued - kStages); i < issued; ++i)
          mbar_wait(&sm.full[i % kStages], static_cast<uint32_t>(i / kStages) & 1u, &never,
                    kDrainLimitNs);
        if constexpr (OUT) {
          for (int i = max(0, wo_cnt - kWoSlots); i < wo_cnt; ++i)
            mbar_wait(&sm.wo_full[i % kWoSlots], static_cast<uint32_t>(i / kWoSlots) & 1u, &never,
                      kDrainLimitNs);
          for (int i = max(0, o_cnt - kOSlots); i < o_cnt; ++i)
            mbar_wait(&sm.o_full[i % kOSlots], static_cast<uint32_t>(i / kOSlots) & 1u, &never,
                      kDrainLimitNs);
        }
      }
      if constexpr (OUT) {
        // the peers' signals this CTA expects have landed before it leaves
        // (at once after a normal run; bounded when a peer gave up)
        volatile uint32_t never = 0;
        if (armed >= 0)
          for (int s = 0; s < args.head_pairs - 1; ++s)
            mbar_wait(&sm.o_ready[armed & 1][s], static_cast<uint32_t>(armed >> 1) & 1u, &never,
                      ok ? kDrainLimitNs : 3 * kWaitLimitNs);
      }
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdescQKV = idesc_bf16(kRows, 3 * kD, false, true);
      constexpr uint32_t kIdescQ = idesc_bf16(kRows, kD, false, true);
      constexpr uint32_t kIdescKV = idesc_bf16(kRows, 2 * kD, false, true);
      constexpr uint32_t kIdescS = idesc_bf16(kRows, kRows, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(kRows, kD, false, true);
      const uint32_t ring0 = smem_u32(sm.ring[0]);
      // X: K-major, rows of 128 bytes; weights: N-major 64-column chunks 8 KB apart
      const uint64_t dx0 = sdesc_sw128(ring0, 16, 1024);
      const uint64_t dw0 = sdesc_sw128(ring0 + Smem::kABytes, kWChunk, 1024);
      // Q/K/V tiles: Q and K K-major (head dimension contiguous); V N-major
      const uint64_t dqk0 = sdesc_sw128(ring0, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(ring0, kTile, 1024);
      constexpr uint32_t kStageStep = Smem::kStageBytes >> 4;
      constexpr uint32_t kTileStep = kTile >> 4;
      constexpr uint32_t kWStep = kWChunk >> 4;
      constexpr uint32_t kIdescOut128 = idesc_bf16(kRows, 128, false, true);
      constexpr uint32_t kIdescOut64 = idesc_bf16(kRows, 64, false, true);
      int consumed = 0, ui = 0, o_used = 0, wo_used = 0;
      bool ok = true;
      for (int u = first; ok && u < args.num_units; u += stride, ++ui) {
        // the previous item's S, P and O (and out) have been read
        if (ui > 0) {
          ok = mbar_wait(&sm.tmem_free, static_cast<uint32_t>(ui - 1) & 1u, abort_flag);
          if (!ok) break;
        }
        tc_fence_after();
        // ---- projections: acc_e = X [W_Q | W_K | W_V] (head e)
        for (int kb = 0; ok && kb < args.kblocks; ++kb) {
          const int s = consumed % kStages;
          ok = mbar_wait(&sm.full[s], static_cast<uint32_t>(consumed / kStages) & 1u, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dx = sdesc_advance(dx0, static_cast<uint32_t>(s) * kStageStep);
          const uint64_t dw = sdesc_advance(dw0, static_cast<uint32_t>(s) * kStageStep);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc_flag = (kb > 0 || kk > 0) ? 1u : 0u;
            const uint32_t aoff = kk * (32 >> 4);     // 16 elements along d_model
            const uint32_t woff = kk * (2048 >> 4);   // 16 rows of the weight slice
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const uint32_t acc = tmem + e * 3 * kD;
              if constexpr (SELF) {
                mma_bf16_ss(acc, sdesc_advance(dx, aoff), sdesc_advance(dw, 3 * e * kWStep + woff),
                            kIdescQKV, acc_flag);
              } else {
                mma_bf16_ss(acc, sdesc_advance(dx, aoff), sdesc_advance(dw, 3 * e * kWStep + woff),
                            kIdescQ, acc_flag);
                mma_bf16_ss(acc + kD, sdesc_advance(dx, kTileStep + aoff),
                            sdesc_advance(dw, (3 * e + 1) * kWStep + woff), kIdescKV, acc_flag);
              }
            }
          }
          mma_commit(&sm.empty[s]);
          ++consumed;
        }
        if (!ok) break;
        mma_commit(&sm.proj_done);
        // ---- S_e = Q_e K_e^T, once head e's Q and K tiles are written
        for (int e = 0; ok && e < 2; ++e) {
          ok = mbar_wait(&sm.qk_ready[e], static_cast<uint32_t>(ui) & 1u, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t a = sdesc_advance(dqk0, (3 * e + 0) * kTileStep);
          const uint64_t bk = sdesc_advance(dqk0, (3 * e + 1) * kTileStep);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_bf16_ss(tmem + e * 3 * kD, sdesc_advance(a, kk * 2), sdesc_advance(bk, kk * 2),
                        kIdescS, kk > 0 ? 1u : 0u);
          mma_commit(&sm.s_full[e]);
        }
        // ---- O_e = P_e V_e, P from tensor memory
        for (int e = 0; ok && e < 2; ++e) {
          ok = mbar_wait(&sm.v_ready[e], static_cast<uint32_t>(ui) & 1u, abort_flag) &&
               mbar_wait(&sm.p_full[e], static_cast<uint32_t>(ui) & 1u, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t bv = sdesc_advance(dv0, (3 * e + 2) * kTileStep);
          const uint32_t p_tmem = tmem + e * 3 * kD + 2 * kD;
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk)
            mma_bf16_ts(tmem + 6 * kD + e * kD, p_tmem + kk * 8, sdesc_advance(bv, kk * (2048 >> 4)),
                        kIdescPV, kk > 0 ? 1u : 0u);
          mma_commit(&sm.pv_done[e]);
        }
        if (!ok) break;
        mma_commit(&sm.qkv_free);  // every MMA reading this item's Q/K/V tiles has completed
        if constexpr (OUT) {
          // ---- out[:, cols] = sum_j head_j W_O[64 j : 64 j + 64, cols], into
          // TMEM columns [0, n_slice) (S_0's, read long ago)
          ok = mbar_wait(&sm.o_staged, static_cast<uint32_t>(ui) & 1u, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t idesc_out = args.n_slice == 128 ? kIdescOut128 : kIdescOut64;
          for (int j = 0; ok && j < args.h; ++j) {
            uint64_t a;
            int os = -1;
            if (j < 2) {  // this CTA's own heads, still in the epilogue's staging tiles
              a = sdesc_sw128(smem_u32(sm.o[j]), 16, 1024);
            } else {
              os = o_used % kOSlots;
              ok = mbar_wait(&sm.o_full[os], static_cast<uint32_t>(o_used / kOSlots) & 1u,
                             abort_flag);
              ++o_used;
              a = sdesc_sw128(ring0 + os * kSlot, 16, 1024);
            }
            const int ws = wo_used % kWoSlots;
            ok = ok && mbar_wait(&sm.wo_full[ws], static_cast<uint32_t>(wo_used / kWoSlots) & 1u,
                                 abort_flag);
            ++wo_used;
            if (!ok) break;
            tc_fence_after();
            // W_O chunk: 64 rows x n_slice columns as 64-column blocks 8 KB apart
            const uint64_t bw = sdesc_sw128(ring0 + (kOSlots + ws) * kSlot, kWChunk, 1024);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_bf16_ss(tmem, sdesc_advance(a, kk * 2), sdesc_advance(bw, kk * (2048 >> 4)),
                          idesc_out, (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&sm.wo_empty[ws]);
            if (os >= 0) mma_commit(&sm.o_empty[os]);
          }
          if (!ok) break;
          mma_commit(&sm.out_done);
        }
      }
      // every issued MMA has completed before tensor memory is released
      volatile uint32_t never = 0;
      mma_commit(&sm.drained);
      mbar_wait(&sm.drained, 0, &never, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------ heads
    regs_increase<kSoftmaxRegs>();
    const int e = (warp - 4) >> 2;      // head of the pair
    const int quarter = warp & 3;       // TMEM lane quarter of this warp
    const int r = quarter * 32 + static_cast<int>(lane);  // row: query (and key) index
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t taddr_acc = tmem + lane_base + e * 3 * kD;  // Q | K | V, then S (Q|K) and P (V)
    const uint32_t taddr_p = taddr_acc + 2 * kD;
    const uint32_t taddr_o = tmem + lane_base + 6 * kD + e * kD;
    const bool leader = (quarter == 0 && lane == 0);  // issues the TMA stores
    const bool causal = (args.mask_kind & kMaskCausal) != 0;
    const float sl2 = args.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    uint8_t* const ring = sm.ring[0];
    bool ok = true;
    griddep_wait();  // the key lengths may come from the previous kernel
    int ui = 0;
    for (int u = first; ok && u < args.num_units; u += stride, ++ui) {
      const int b = u / args.head_pairs;
      const int pair = u % args.head_pairs;
      const int hh = 2 * pair + e;
      int kv_eff = args.n_k;
      if (args.mask_kind & kMaskKeyPadding) {
        const int len = args.kv_lens[b];
        kv_eff = len < 0 ? 0 : (len > args.n_k ? args.n_k : len);
      }
      const uint32_t ph = static_cast<uint32_t>(ui) & 1u;
      // A failed wait is carried to the warpgroup's barrier below, where all
      // four warps stop together (none is left waiting at it).
      bool okw = __all_sync(0xffffffffu, mbar_wait(&sm.proj_done, ph, abort_flag));
      if (okw) {
        // ---- (1) this row of Q, K, V -> bf16 rows of the swizzled tiles;
        // Q and K first, so that S runs while V is converted
        tc_fence_after();
        auto convert = [&](int part) {
          uint8_t* row = ring + (3 * e + part) * kTile + r * 128;
          uint32_t v[64];
          tmem_ld32(taddr_acc + part * kD, *reinterpret_cast<uint32_t(*)[32]>(v));
          tmem_ld32(taddr_acc + part * kD + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 8; ++j) {  // 16-byte chunk j of the 128-byte row
            const uint32_t* x = v + 8 * j;
            st_shared_v4(smem_u32(row + ((j ^ (r & 7)) << 4)),
                         pack_bf16x2(__uint_as_float(x[0]), __uint_as_float(x[1])),
                         pack_bf16x2(__uint_as_float(x[2]), __uint_as_float(x[3])),
                         pack_bf16x2(__uint_as_float(x[4]), __uint_as_float(x[5])),
                         pack_bf16x2(__uint_as_float(x[6]), __uint_as_float(x[7])));
          }
        };
        convert(0);
        convert(1);
        fence_proxy_async_smem();  // the tiles are read by the tensor cores
        tc_fence_before();         // and S overwrites the accumulator just read
        mbar_arrive(&sm.qk_ready[e]);
        convert(2);
        fence_proxy_async_smem();
        tc_fence_before();         // P overwrites V's accumulator columns
        mbar_arrive(&sm.v_ready[e]);
      }
      // ---- (2) softmax of the single score tile
      okw = okw && __all_sync(0xffffffffu, mbar_wait(&sm.s_full[e], ph, abort_flag));
      float l = 0.f;
      if (okw) {
        tc_fence_after();
        float s[kRows];
#pragma unroll
        for (int cc = 0; cc < kRows / 32; ++cc) {
          uint32_t raw[32];
          tmem_ld32(taddr_acc + cc * 32, raw);
#pragma unroll
          for (int x = 0; x < 32; ++x) s[cc * 32 + x] = __uint_as_float(raw[x]);
        }
        tmem_wait_ld();
        const int lim = causal ? min(kv_eff, r + 1) : kv_eff;  // keys [0, lim)
        if (lim < kRows) {
#pragma unroll
          for (int x = 0; x < kRows; ++x)
            if (x >= lim) s[x] = -INFINITY;
        }
        float mx8[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) mx8[x] = fmaxf(s[x], s[x + 8]);
#pragma unroll
        for (int x0 = 16; x0 < kRows; x0 += 16)
#pragma unroll
          for (int x = 0; x < 8; ++x) mx8[x] = fmax3(mx8[x], s[x0 + x], s[x0 + 8 + x]);
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7]));
        const float m = mx == -INFINITY ? 0.f : mx * sl2;
        const uint64_t negm2 = f2_pack(-m, -m);
        uint32_t pk[kRows / 2];
        uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int x = 0; x < kRows / 2; ++x) {
          float x0, x1;
          f2_unpack(ffma2(f2_pack(s[2 * x], s[2 * x + 1]), sl2x2, negm2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          pk[x] = pack_bf16x2(p0, p1);
          acc2[x & 3] = fadd2(acc2[x & 3], f2_pack(p0, p1));
        }
        float r0, r1;
        f2_unpack(fadd2(fadd2(acc2[0], acc2[1]), fadd2(acc2[2], acc2[3])), r0, r1);
        l = r0 + r1;
        // P row -> TMEM lane r, two bf16 per 32-bit column (the MMA's A layout)
        uint32_t half[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) half[x] = pk[x];
        tmem_st32(taddr_p, half);
#pragma unroll
        for (int x = 0; x < 32; ++x) half[x] = pk[32 + x];
        tmem_st32(taddr_p + 32, half);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sm.p_full[e]);
      }
      // ---- (3) epilogue: O / l -> bf16 -> staging -> TMA store
      okw = okw && __all_sync(0xffffffffu, mbar_wait(&sm.pv_done[e], ph, abort_flag));
      if (leader) bulk_wait_group_read<0>();  // the staging tile's previous store has read it
      ok = e == 0 ? named_bar_and<1>(128, okw) : named_bar_and<2>(128, okw);
      if (!ok) break;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int cc = 0; cc < kD / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(taddr_o + cc * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          const int j = cc * 4 + v4;
          const uint32_t* x = o + 8 * v4;
          st_shared_v4(smem_u32(sm.o[e] + r * 128 + ((j ^ (r & 7)) << 4)),
                       pack_bf16x2(__uint_as_float(x[0]) * inv_l, __uint_as_float(x[1]) * inv_l),
                       pack_bf16x2(__uint_as_float(x[2]) * inv_l, __uint_as_float(x[3]) * inv_l),
                       pack_bf16x2(__uint_as_float(x[4]) * inv_l, __uint_as_float(x[5]) * inv_l),
                       pack_bf16x2(__uint_as_float(x[6]) * inv_l, __uint_as_float(x[7]) * inv_l));
        }
      }
      tc_fence_before();
      if constexpr (!OUT) mbar_arrive(&sm.tmem_free);  // this thread's reads of S, P and O are done
      fence_proxy_async_smem();  // staged bytes visible to the TMA unit (and the tensor cores)
      if constexpr (OUT) mbar_arrive(&sm.o_staged);
      if (e == 0) named_bar_sync<1>(128);
      else named_bar_sync<2>(128);
      if (leader) {  // the map clips rows past n_q
        tma_store_3d(&tm_o, sm.o[e], hh * kD, 0, b);
        bulk_commit_group();
        if constexpr (OUT) {
          if (args.head_pairs > 1) {
            // the tile is in global memory: tell every peer of the cluster
            // (CTA rank = head pair: the grid is a whole number of clusters);
            // this CTA is peer slot (pair - q - 1) mod C of CTA q
            bulk_wait_group<0>();
            fence_proxy_async_global();
            const int C = args.head_pairs;
            for (int q = 0; q < C; ++q) {
              if (q == pair) continue;
              const int slot = (pair - q - 1 + C) % C;
              signal_remote(cluster_map(&sm.o_words[ui & 1][slot][e], q),
                            cluster_map(&sm.o_ready[ui & 1][slot], q));
            }
          }
        }
      }
      if constexpr (OUT) {
        // ---- (4) out[:, N pair + 64 e : + 64] (fp32 in TMEM) -> bf16 ->
        // staging -> TMA store
        okw = __all_sync(0xffffffffu, mbar_wait(&sm.out_done, ph, abort_flag));
        if (leader) bulk_wait_group_read<0>();  // the merged tile's store has read the staging tile
        ok = e == 0 ? named_bar_and<1>(128, okw) : named_bar_and<2>(128, okw);
        if (!ok) break;
        tc_fence_after();
        const bool has_cols = e * 64 < args.n_slice;
        if (has_cols) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + e * 64 + cc * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              const int j = cc * 4 + v4;
              const uint32_t* x = o + 8 * v4;
              st_shared_v4(smem_u32(sm.o[e] + r * 128 + ((j ^ (r & 7)) << 4)),
                           pack_bf16x2(__uint_as_float(x[0]), __uint_as_float(x[1])),
                           pack_bf16x2(__uint_as_float(x[2]), __uint_as_float(x[3])),
                           pack_bf16x2(__uint_as_float(x[4]), __uint_as_float(x[5])),
                           pack_bf16x2(__uint_as_float(x[6]), __uint_as_float(x[7])));
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&sm.tmem_free);  // this thread's reads of S, P, O and out are done
        fence_proxy_async_smem();
        if (e == 0) named_bar_sync<1>(128);
        else named_bar_sync<2>(128);
        if (leader && has_cols) {
          tma_store_3d(&tm_out, sm.o[e], pair * args.n_slice + e * 64, 0, b);
          bulk_commit_group();
        }
      }
    }
    // the stores have read the staging tiles before the CTA's shared memory
    // goes; their global writes complete with the grid
    if (leader) bulk_wait_group_read<0>();
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  if constexpr (OUT) {
    // After a normal run every signal a peer sends this CTA has landed (the
    // producer waited for each), so it may leave at once. After a failure a
    // peer might still signal it for a later item: then it stays until every
    // CTA of the cluster has either left or come here too.
    if (__syncthreads_or(*abort_flag != 0u)) cluster_sync();
  }
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

// Clusters of C CTAs of the output-projecting kernel that can be resident
// at once (clusters stay inside one GPC); 0 if none fits. Asked once per C.
template <bool SELF>
int fused_out_max_clusters(int C) {
  static int cache[kMaxCluster + 1] = {};  // 0: not asked yet, -1: none fits
  if (C < 1 || C > kMaxCluster) return 0;
  const int known = __atomic_load_n(&cache[C], __ATOMIC_ACQUIRE);
  if (known != 0) return known > 0 ? known : 0;
  using Smem = FusedSmem<SELF>;
  const size_t smem_bytes = sizeof(Smem) + 1024;
  auto kernel = mha_fused_kernel<SELF, true>;
  static unsigned long long configured = 0;
  if (set_smem_once(kernel, static_cast<int>(smem_bytes), &configured,
                    static_cast<int>(kLaunchRegs)) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms() / C * C);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  __atomic_store_n(&cache[C], n > 0 ? n : -1, __ATOMIC_RELEASE);
  return n > 0 ? n : 0;
}

template <bool SELF, bool OUT>
cudaError_t launch_fused(const MhaFusedProblem& p, cudaStream_t stream) {
  using Smem = FusedSmem<SELF>;
  const size_t smem_bytes = sizeof(Smem) + 1024;  // + alignment slack
  auto kernel = mha_fused_kernel<SELF, OUT>;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(kernel, static_cast<int>(smem_bytes), &configured,
                                static_cast<int>(kLaunchRegs));
  if (e != cudaSuccess) return e;
  FusedArgs a;
  a.h = p.h;
  a.n_q = p.n_q;
  a.n_k = p.n_k;
  a.kblocks = p.d_model / 64;
  a.head_pairs = p.h / 2;
  const long long units = static_cast<long long>(p.B) * a.head_pairs;
  if (units <= 0) return cudaSuccess;
  if (units > 0x7fffffffLL - (1LL << 20)) return cudaErrorInvalidValue;
  a.num_units = static_cast<int>(units);
  a.mask_kind = p.mask_kind;
  a.kv_lens = p.kv_lens;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.n_slice = OUT ? p.d_model / a.head_pairs : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int grid = static_cast<int>(units < num_sms() ? units : num_sms());
  if (OUT) {
    // one cluster per batch entry, CTA rank = head pair; persistent over
    // batch entries when more than the resident clusters
    const int C = a.head_pairs;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    const int max_clusters = fused_out_max_clusters<SELF>(C);
    if (max_clusters <= 0) return cudaErrorInvalidConfiguration;
    grid = (p.B < max_clusters ? p.B : max_clusters) * C;
  }
  cfg.gridDim = dim3(grid);
  return cudaLaunchKernelEx(&cfg, kernel, p.tm_xq, p.tm_xkv, p.tm_wq, p.tm_wk, p.tm_wv, p.tm_o,
                            p.tm_wo, p.tm_out, a);
}

}  // namespace

int mha_fused_out_clusters(int h, bool self) {
  const int C = h / 2;
  if (h % 2 != 0 || C < 1 || C > kMaxCluster) return 0;
  return self ? fused_out_max_clusters<true>(C) : fused_out_max_clusters<false>(C);
}

cudaError_t launch_mha_fused(const MhaFusedProblem& p, cudaStream_t stream) {
  if (p.h % 2 != 0 || p.d_model % 64 != 0 || p.d_model <= 0 || p.n_q < 1 || p.n_q > kRows ||
      p.n_k < 1 || p.n_k > kRows)
    return cudaErrorInvalidValue;
  if (p.out) {
    const int C = p.h / 2;
    if (C > kMaxCluster || p.d_model % C != 0) return cudaErrorInvalidValue;
    const int n_slice = p.d_model / C;
    if (n_slice != 64 && n_slice != 128) return cudaErrorInvalidValue;
    return p.self ? launch_fused<true, true>(p, stream) : launch_fused<false, true>(p, stream);
  }
  return p.self ? launch_fused<true, false>(p, stream) : launch_fused<false, false>(p, stream);
}

TSD_DEFINE_ERROR_READER(take_device_error_fused)

}  // namespace tsd
