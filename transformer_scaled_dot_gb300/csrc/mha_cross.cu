// mha_cross.cu -- encoder-decoder (cross) multi-head attention in one kernel
// when the source is a little longer than one key tile: n_q <= 128 target
// rows, 128 < n_k <= 192 source rows, d_k = d_v = 64. The queries come from
// the decoder's rows, the keys and values from the encoder output
// ("[논문 리뷰]Attention Is All You Need" (kimjiil.github.io), section 3.2.3,
// the encoder-decoder attention row; heads per sections 3.2.1-3.2.2,
// head_i = Attention(X_q W_i^Q, X_kv W_i^K, X_kv W_i^V), weights in the x.W
// layout [d_model, h*64], no biases), up to the merged heads and optionally
// through the output projection (MultiHead = Concat(heads) W_O).
//
// A CTA owns one work item, (batch b, heads 2p and 2p+1), as the fused
// short-sequence kernel does; with the output projection the h/2 CTAs of a
// batch entry form a cluster and exchange their merged heads through L2 (the
// same protocol as in mha_fused.cu). What is new is the source's tail, key
// rows [128, n_k): its K|V projection is taken transposed,
//   T_e = [W_K | W_V]_e^T X_kv[128 : 192]^T    (128 features x 64 keys),
// the weight slice as an MN-major A operand and the 64 tail rows of X_kv as
// the B operand. A 128-row key tile would need 128 more accumulator columns
// per head than the 64 this takes (Q, K|V of the first key tile and the tail
// of both heads fill exactly the 512 tensor-memory columns), and would
// multiply mostly zero rows: at n_k = 160 the tail holds 32 keys. Everything
// is projected in one pass over d_model. A tail accumulator row is one
// feature over the 64 tail keys; written out as rows of 64 keys it is at once
// the MN-major B operand of S = Q K_T^T (N = keys) and the K-major B operand
// of O += P_T V_T (K = keys).
//
//   warp 0      TMA producer
//   warp 1      MMA issuer (one thread): the projections, S and O += P V for
//               the first key tile and the tail, and (OUT) the output
//               projection
//   warps 4..7  head 2p, warps 8..11 head 2p+1, one thread per row (= TMEM
//               lane): the Q, K and V rows and one tail feature row to bf16
//               tiles; the online softmax of its query row over the two key
//               tiles; O / l -> bf16 -> staging -> TMA store
//
// Shared memory: a ring of two 88 KB stages (X_q, X_kv rows [0, 128) and
// [128, 192) of one 64-wide slice of d_model, and the W_Q, W_K, W_V slices
// of both heads); then the K/V tiles in [0, 96) KB (K_e and V_e of the first
// key tile, 16 KB each, and the tail tiles K_T,e and V_T,e, 64 rows x 64 keys,
// 8 KB each), the Q tiles in the epilogue's staging buffers. OUT: the peers'
// merged tiles in [0, 96) KB once the attention MMAs are done; W_O chunks in
// [96, 176) KB, free as soon as the projections are done.
// Tensor memory (512 columns): Q_e at 64e, K|V_e at 128 + 128e, T_e at
// 384 + 64e; then S_e at 128e, P_e (bf16) at 256 + 64e, O_e at 384 + 64e;
// (OUT) the output columns at [0, n_slice).
#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kRows = 128;              // query rows and key rows per tile
constexpr int kD = 64;                  // d_k = d_v
constexpr int kTail = 64;               // tail keys: n_k <= kRows + kTail
constexpr int kTile = kRows * kD * 2;   // 16 KB: a 128 x 64 bf16 tile
constexpr int kTailTile = kTail * kD * 2;  // 8 KB: a 64 x 64 bf16 tile
constexpr int kWChunk = 64 * kD * 2;    // 8 KB: 64 rows of d_model x 64 columns of one weight
constexpr int kThreads = 384;           // 4 control warps + 2 head warpgroups
constexpr uint32_t kLaunchRegs = 65536 / kThreads / 8 * 8;  // 168
constexpr uint32_t kCtrlRegs = 72;
constexpr uint32_t kHeadRegs = (kLaunchRegs * kThreads - kCtrlRegs * 128) / 256 / 8 * 8;
static_assert(kCtrlRegs * 128 + kHeadRegs * 256 <= kLaunchRegs * kThreads, "register split");
constexpr unsigned long long kDrainLimitNs = 100ull * 1000ull * 1000ull;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr bool kPrefetchL2 = true;  // a share of the first wave's operands into L2 before the wait

// one stage: X_q | X_kv rows [0,128) | X_kv rows [128,192) | W_Q0 W_Q1 | W_K0 W_V0 | W_K1 W_V1
constexpr int kXkvOff = kTile;
constexpr int kXtOff = 2 * kTile;
constexpr int kWOff = 2 * kTile + kTailTile;
constexpr int kStage = kWOff + 6 * kWChunk;  // 88 KB
constexpr int kStages = 2;
constexpr int kRingBytes = kStages * kStage;  // 176 KB
__host__ __device__ constexpr int wq_chunk(int e) { return e; }
__host__ __device__ constexpr int wk_chunk(int e) { return 2 + 2 * e; }  // W_V_e follows
// K/V tiles after the projections
__host__ __device__ constexpr int k0_off(int e) { return 2 * e * kTile; }
__host__ __device__ constexpr int v0_off(int e) { return (2 * e + 1) * kTile; }
__host__ __device__ constexpr int kt_off(int e) { return 4 * kTile + 2 * e * kTailTile; }
__host__ __device__ constexpr int vt_off(int e) { return 4 * kTile + (2 * e + 1) * kTailTile; }
constexpr int kTilesEnd = 4 * kTile + 4 * kTailTile;  // 96 KB
// output projection (OUT)
constexpr int kSlot = 16384;  // a merged-heads tile, or 64 rows of W_O x <= 128 columns
constexpr int kOSlots = 6;    // peers' merged tiles, [0, 96) KB
constexpr int kWoSlots = 5;   // W_O chunks, [96, 176) KB
constexpr int kWoBase = kOSlots * kSlot;
constexpr int kMaxCluster = 8;
static_assert(kTilesEnd == kWoBase, "K/V tiles end where the W_O ring starts");
static_assert(kWoBase + kWoSlots * kSlot <= kRingBytes, "W_O ring inside the stages");

__host__ __device__ constexpr uint32_t q_col(int e) { return static_cast<uint32_t>(64 * e); }
__host__ __device__ constexpr uint32_t kv_col(int e) { return static_cast<uint32_t>(128 + 128 * e); }
__host__ __device__ constexpr uint32_t t_col(int e) { return static_cast<uint32_t>(384 + 64 * e); }
__host__ __device__ constexpr uint32_t s_col(int e) { return static_cast<uint32_t>(128 * e); }
__host__ __device__ constexpr uint32_t p_col(int e) { return static_cast<uint32_t>(256 + 64 * e); }
__host__ __device__ constexpr uint32_t o_col(int e) { return static_cast<uint32_t>(384 + 64 * e); }

struct CrossSmem {
  alignas(1024) uint8_t ring[kRingBytes];
  alignas(1024) uint8_t o[2][kTile];  // the Q tiles, then the epilogue's staging, one per head
  uint64_t full[kStages], empty[kStages];
  uint64_t proj_done;  // every projection MMA of the item has completed
  uint64_t conv[2];    // head e's Q, K, V and tail rows turned into tiles (128 arrivals)
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t qkv_free;   // every MMA reading the item's Q/K/V tiles has completed
  uint64_t tmem_free;  // every head thread's reads of the item's tensor memory are done
  uint64_t drained;
  // output projection (OUT)
  uint64_t o_full[kOSlots], o_empty[kOSlots];
  uint64_t wo_full[kWoSlots], wo_empty[kWoSlots];
  uint64_t o_staged;   // this CTA's two merged tiles are in o[] (256 arrivals)
  uint64_t out_done;   // every out-projection MMA of the item has completed
  uint64_t o_ready[2][kMaxCluster - 1];
  uint32_t o_words[2][kMaxCluster - 1][2];
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct CrossArgs {
  int h, n_q, n_k, kblocks, num_units, head_pairs;
  int mask_kind;
  const int32_t* kv_lens;
  float scale_log2;
  int n_slice;  // OUT: output columns per CTA (64 or 128)
};

// Keys [0, kv_eff) of batch entry b are visible (key padding, clamped).
__device__ __forceinline__ int key_limit(const CrossArgs& a, int b) {
  int kv_eff = a.n_k;
  if (a.mask_kind & kMaskKeyPadding) {
    const int len = a.kv_lens[b];
    kv_eff = len < 0 ? 0 : (len > a.n_k ? a.n_k : len);
  }
  return kv_eff;
}
// Key tiles the attention takes (the tail only when keys past 128 are visible).
__device__ __forceinline__ int key_tiles(int kv_eff) { return kv_eff > kRows ? 2 : 1; }

template <bool OUT>
__global__ void __launch_bounds__(kThreads, 1)
    mha_cross_kernel(const __grid_constant__ CUtensorMap tm_xq,
                     const __grid_constant__ CUtensorMap tm_xkv,
                     const __grid_constant__ CUtensorMap tm_xkv_tail,
                     const __grid_constant__ CUtensorMap tm_wq,
                     const __grid_constant__ CUtensorMap tm_wk,
                     const __grid_constant__ CUtensorMap tm_wv,
                     const __grid_constant__ CUtensorMap tm_o,
                     const __grid_constant__ CUtensorMap tm_wo,
                     const __grid_constant__ CUtensorMap tm_out, const CrossArgs args) {
  extern __shared__ uint8_t smem_raw[];
  CrossSmem& sm = *reinterpret_cast<CrossSmem*>(
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
    for (int e = 0; e < 2; ++e) {
      mbar_init(&sm.conv[e], 128);
      mbar_init(&sm.s_full[e], 1);
      mbar_init(&sm.s_free[e], 128);
      mbar_init(&sm.p_full[e], 128);
      mbar_init(&sm.pv_done[e], 1);
    }
    mbar_init(&sm.qkv_free, 1);
    mbar_init(&sm.tmem_free, 256);
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
    tma_prefetch_desc(&tm_xq);
    tma_prefetch_desc(&tm_xkv);
    tma_prefetch_desc(&tm_xkv_tail);
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
        // entry's X_q and X_kv rows (the C CTAs of a batch entry split them),
        // and, CTA b of each head pair, one 64-row block of the pair's W_Q,
        // W_K, W_V slices and of its W_O columns; the loads after the wait
        // find them there. A prefetch only reads into L2, the point of
        // coherence.
        const int C = args.head_pairs;
        const int b = first / C;
        const int pair = first % C;
        for (int kb = pair; kb < args.kblocks; kb += C) {
          tma_prefetch_l2_3d(&tm_xq, kb * 64, 0, b);
          tma_prefetch_l2_3d(&tm_xkv, kb * 64, 0, b);
          tma_prefetch_l2_3d(&tm_xkv_tail, kb * 64, kRows, b);
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
        // the previous item's tiles in the ring (with OUT also the peers'
        // merged tiles and W_O) have been consumed
        if (ui > 0) {
          ok = mbar_wait(OUT ? &sm.out_done : &sm.qkv_free, static_cast<uint32_t>(ui - 1) & 1u,
                         abort_flag);
          if (!ok) break;
        }
        if constexpr (OUT) {
          for (int i = 0; i < args.head_pairs - 1; ++i)
            mbar_arrive_expect_tx(&sm.o_ready[ui & 1][i], 8);
          armed = ui;
        }
        for (int kb = 0; kb < args.kblocks; ++kb) {
          const int s = issued % kStages;
          ok = mbar_wait(&sm.empty[s], (static_cast<uint32_t>(issued / kStages) & 1u) ^ 1u,
                         abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&sm.full[s], kStage);
          if (issued == 0) griddep_wait();
          const int k0 = kb * 64;
          uint8_t* st = sm.ring + s * kStage;
          tma_load_3d(st, &tm_xq, &sm.full[s], k0, 0, b);
          tma_load_3d(st + kXkvOff, &tm_xkv, &sm.full[s], k0, 0, b);
          tma_load_3d(st + kXtOff, &tm_xkv_tail, &sm.full[s], k0, kRows, b);  // rows past n_k: zeros
          uint8_t* w = st + kWOff;
          for (int e = 0; e < 2; ++e) {
            const int col = (h0 + e) * kD;
            tma_load_2d(w + wq_chunk(e) * kWChunk, &tm_wq, &sm.full[s], col, k0);
            tma_load_2d(w + wk_chunk(e) * kWChunk, &tm_wk, &sm.full[s], col, k0);
            tma_load_2d(w + (wk_chunk(e) + 1) * kWChunk, &tm_wv, &sm.full[s], col, k0);
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
            uint8_t* dst = sm.ring + kWoBase + s * kSlot;
            mbar_arrive_expect_tx(&sm.wo_full[s], static_cast<uint32_t>(args.n_slice) * 128u);
            for (int c = 0; c < args.n_slice; c += 64)
              tma_load_2d(dst + c * 128, &tm_wo, &sm.wo_full[s], pair * args.n_slice + c,
                          head_of(j) * kD);
            ++wo_cnt;
            return true;
          };
          const uint32_t ph = static_cast<uint32_t>(ui) & 1u;
          // W_O's first chunks while the attention runs: the stages are free
          // once every projection MMA has completed
          ok = mbar_wait(&sm.proj_done, ph, abort_flag);
          int wj = 0;
          for (; ok && wj < args.h && wj < kWoSlots; ++wj) ok = issue_wo(wj);
          // then the peers' merged tiles, into the K/V tiles' place once those
          // are consumed, each peer's as soon as it has stored them, with the
          // rest of W_O as its slots free up
          ok = ok && mbar_wait(&sm.qkv_free, ph, abort_flag);
          for (int j = 2; ok && j < args.h; ++j) {
            if ((j & 1) == 0) {
              ok = mbar_wait_cluster(&sm.o_ready[ui & 1][(j >> 1) - 1],
                                     static_cast<uint32_t>(ui >> 1) & 1u, abort_flag);
              fence_proxy_async_global();  // before the TMA reads what the peer's TMA wrote
            }
            if (!ok) break;
            const int os = o_cnt % kOSlots;
            ok = mbar_wait(&sm.o_empty[os], (static_cast<uint32_t>(o_cnt / kOSlots) & 1u) ^ 1u,
                           abort_flag);
            if (!ok) break;
            mbar_arrive_expect_tx(&sm.o_full[os], kTile);
            tma_load_3d(sm.ring + os * kSlot, &tm_o, &sm.o_full[os], head_of(j) * kD, 0, b);
            ++o_cnt;
            while (ok && wj <= j + kWoSlots - 2 && wj < args.h) ok = issue_wo(wj++);
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
          for (int i = 0; i < args.head_pairs - 1; ++i)
            mbar_wait(&sm.o_ready[armed & 1][i], static_cast<uint32_t>(armed >> 1) & 1u, &never,
                      ok ? kDrainLimitNs : 3 * kWaitLimitNs);
      }
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdescQ = idesc_bf16(kRows, kD, false, true);
      constexpr uint32_t kIdescKV = idesc_bf16(kRows, 2 * kD, false, true);
      // tail: A = [W_K | W_V]^T (M = 128 features, MN-major), B = X_kv tail (N = 64 keys, K-major)
      constexpr uint32_t kIdescT = idesc_bf16(kRows, kTail, true, false);
      constexpr uint32_t kIdescS = idesc_bf16(kRows, kRows, false, false);
      constexpr uint32_t kIdescST = idesc_bf16(kRows, kTail, false, true);  // B = K_T, MN-major
      constexpr uint32_t kIdescPV = idesc_bf16(kRows, kD, false, true);     // B = V, N-major
      constexpr uint32_t kIdescPVT = idesc_bf16(kRows, kD, false, false);   // B = V_T, K-major
      constexpr uint32_t kIdescOut128 = idesc_bf16(kRows, 128, false, true);
      constexpr uint32_t kIdescOut64 = idesc_bf16(kRows, 64, false, true);
      const uint32_t ring0 = smem_u32(sm.ring);
      // X: K-major, rows of 128 bytes; weights: 64-column chunks 8 KB apart
      const uint64_t dx0 = sdesc_sw128(ring0, 16, 1024);
      const uint64_t dw0 = sdesc_sw128(ring0 + kWOff, kWChunk, 1024);
      constexpr uint32_t kStageStep = kStage >> 4;
      constexpr uint32_t kWStep = kWChunk >> 4;
      int consumed = 0, ui = 0, o_used = 0, wo_used = 0;
      int c[2] = {0, 0};  // S / P tiles per head so far (phase counters)
      bool ok = true;
      griddep_wait();  // the key lengths may come from the previous kernel
      for (int u = first; ok && u < args.num_units; u += stride, ++ui) {
        const int b = u / args.head_pairs;
        const uint32_t ph = static_cast<uint32_t>(ui) & 1u;
        // the previous item's S, P and O (and out) have been read
        if (ui > 0) {
          ok = mbar_wait(&sm.tmem_free, static_cast<uint32_t>(ui - 1) & 1u, abort_flag);
          if (!ok) break;
        }
        tc_fence_after();
        // ---- projections: Q_e = X_q W_Q, [K|V]_e = X_kv[0:128] [W_K | W_V],
        // T_e = [W_K | W_V]^T X_kv[128:192]^T (head e)
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
            const uint32_t aoff = kk * (32 >> 4);    // 16 elements along d_model
            const uint32_t woff = kk * (2048 >> 4);  // 16 rows of the weight slice
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              mma_bf16_ss(tmem + q_col(e), sdesc_advance(dx, aoff),
                          sdesc_advance(dw, wq_chunk(e) * kWStep + woff), kIdescQ, acc_flag);
              const uint64_t wkv = sdesc_advance(dw, wk_chunk(e) * kWStep + woff);
              mma_bf16_ss(tmem + kv_col(e), sdesc_advance(dx, (kXkvOff >> 4) + aoff), wkv,
                          kIdescKV, acc_flag);
              mma_bf16_ss(tmem + t_col(e), wkv, sdesc_advance(dx, (kXtOff >> 4) + aoff), kIdescT,
                          acc_flag);
            }
          }
          mma_commit(&sm.empty[s]);
          ++consumed;
        }
        if (!ok) break;
        mma_commit(&sm.proj_done);
        // ---- attention, once every Q/K/V tile is written and every
        // accumulator under S, P and O has been read
        ok = mbar_wait(&sm.conv[0], ph, abort_flag) && mbar_wait(&sm.conv[1], ph, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const int nkt = key_tiles(key_limit(args, b));
        auto issue_s = [&](int e, int m) {
          const uint64_t a = sdesc_sw128(smem_u32(sm.o[e]), 16, 1024);  // Q tile, K-major
          if (m == 0) {
            const uint64_t bk = sdesc_sw128(ring0 + k0_off(e), 16, 1024);  // K tile, K-major
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_bf16_ss(tmem + s_col(e), sdesc_advance(a, kk * 2), sdesc_advance(bk, kk * 2),
                          kIdescS, kk > 0 ? 1u : 0u);
          } else {
            // K_T: rows = head dimension, 64 keys each (MN-major, N = keys)
            const uint64_t bk = sdesc_sw128(ring0 + kt_off(e), kTailTile, 1024);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_bf16_ss(tmem + s_col(e), sdesc_advance(a, kk * 2),
                          sdesc_advance(bk, kk * (2048 >> 4)), kIdescST, kk > 0 ? 1u : 0u);
          }
          mma_commit(&sm.s_full[e]);
        };
        auto issue_pv = [&](int e, int m) {
          if (m == 0) {
            const uint64_t bv = sdesc_sw128(ring0 + v0_off(e), kTile, 1024);  // V, N-major
#pragma unroll
            for (int kk = 0; kk < kRows / 16; ++kk)
              mma_bf16_ts(tmem + o_col(e), tmem + p_col(e) + kk * 8,
                          sdesc_advance(bv, kk * (2048 >> 4)), kIdescPV, kk > 0 ? 1u : 0u);
          } else {
            // V_T: rows = head dimension, 64 keys each (K-major, K = keys)
            const uint64_t bv = sdesc_sw128(ring0 + vt_off(e), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kTail / 16; ++kk)
              mma_bf16_ts(tmem + o_col(e), tmem + p_col(e) + kk * 8, sdesc_advance(bv, kk * 2),
                          kIdescPVT, 1u);
          }
          mma_commit(&sm.pv_done[e]);
        };
        for (int e = 0; e < 2; ++e) issue_s(e, 0);
        for (int e = 0; ok && e < 2; ++e) {
          ok = mbar_wait(&sm.p_full[e], static_cast<uint32_t>(c[e]) & 1u, abort_flag);
          if (!ok) break;
          tc_fence_after();
          issue_pv(e, 0);
        }
        if (ok && nkt == 2) {
          for (int e = 0; ok && e < 2; ++e) {
            // S_e of the tail overwrites the first key tile's, once it is read
            ok = mbar_wait(&sm.s_free[e], static_cast<uint32_t>(c[e]) & 1u, abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_s(e, 1);
          }
          for (int e = 0; ok && e < 2; ++e) {
            ok = mbar_wait(&sm.p_full[e], static_cast<uint32_t>(c[e] + 1) & 1u, abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_pv(e, 1);
          }
        }
        if (!ok) break;
        c[0] += nkt;
        c[1] += nkt;
        mma_commit(&sm.qkv_free);  // every MMA reading this item's Q/K/V tiles has completed
        if constexpr (OUT) {
          // ---- out[:, cols] = sum_j head_j W_O[64 j : 64 j + 64, cols], into
          // TMEM columns [0, n_slice) (S_0's, read before o_staged)
          ok = mbar_wait(&sm.o_staged, ph, abort_flag);
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
            const uint64_t bw = sdesc_sw128(ring0 + kWoBase + ws * kSlot, kWChunk, 1024);
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
    regs_increase<kHeadRegs>();
    const int e = (warp - 4) >> 2;      // head of the pair
    const int quarter = warp & 3;       // TMEM lane quarter of this warp
    const int r = quarter * 32 + static_cast<int>(lane);  // row: query (and key, feature) index
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t taddr = tmem + lane_base;
    const bool leader = (quarter == 0 && lane == 0);  // issues the TMA stores
    const float sl2 = args.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    uint8_t* const ring = sm.ring;
    int c = 0;  // S / P tiles of this head so far (phase counter)
    bool ok = true;
    griddep_wait();  // the key lengths may come from the previous kernel
    int ui = 0;
    // 64 fp32 accumulator columns from `col` -> one bf16 row of 128 bytes at
    // `row` (row index `ri` within a 128-byte-swizzled tile)
    auto convert = [&](uint32_t col, uint8_t* row, int ri) {
      uint32_t v[64];
      tmem_ld32(taddr + col, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld32(taddr + col + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // 16-byte chunk j of the 128-byte row
        const uint32_t* x = v + 8 * j;
        st_shared_v4(smem_u32(row + ((j ^ (ri & 7)) << 4)),
                     pack_bf16x2(__uint_as_float(x[0]), __uint_as_float(x[1])),
                     pack_bf16x2(__uint_as_float(x[2]), __uint_as_float(x[3])),
                     pack_bf16x2(__uint_as_float(x[4]), __uint_as_float(x[5])),
                     pack_bf16x2(__uint_as_float(x[6]), __uint_as_float(x[7])));
      }
    };
    for (int u = first; ok && u < args.num_units; u += stride, ++ui) {
      const int b = u / args.head_pairs;
      const int pair = u % args.head_pairs;
      const int hh = 2 * pair + e;
      const int kv_eff = key_limit(args, b);
      const int nkt = key_tiles(kv_eff);
      const uint32_t ph = static_cast<uint32_t>(ui) & 1u;
      // A failed wait is carried to the warpgroup's barrier below, where all
      // four warps stop together (none is left waiting at it).
      bool okw = __all_sync(0xffffffffu, mbar_wait(&sm.proj_done, ph, abort_flag));
      // ---- (1) this row of Q, K, V and of the tail -> bf16 tiles, once the
      // previous item's stores from the staging buffer have read it
      if (leader) bulk_wait_group_read<0>();
      okw = e == 0 ? named_bar_and<1>(128, okw) : named_bar_and<2>(128, okw);
      if (okw) {
        tc_fence_after();
        convert(q_col(e), sm.o[e] + r * 128, r);
        convert(kv_col(e), ring + k0_off(e) + r * 128, r);
        convert(kv_col(e) + kD, ring + v0_off(e) + r * 128, r);
        // tail feature r: K_T row r (r < 64), else V_T row r - 64; 64 keys
        const int fr = r & 63;
        convert(t_col(e), ring + (r < 64 ? kt_off(e) : vt_off(e)) + fr * 128, fr);
        fence_proxy_async_smem();  // the tiles are read by the tensor cores
        tc_fence_before();         // and S, P and O overwrite the accumulators just read
        mbar_arrive(&sm.conv[e]);
      }
      // ---- (2) online softmax over the first key tile and the tail
      float m_used = -INFINITY;
      float l = 0.f;
      for (int m = 0; okw && m < nkt; ++m, ++c) {
        okw = __all_sync(0xffffffffu, mbar_wait(&sm.s_full[e], static_cast<uint32_t>(c) & 1u,
                                                abort_flag));
        if (!okw) break;
        tc_fence_after();
        float s[kRows];
#pragma unroll
        for (int cc = 0; cc < kRows / 32; ++cc) {
          uint32_t raw[32];
          tmem_ld32(taddr + s_col(e) + cc * 32, raw);
#pragma unroll
          for (int x = 0; x < 32; ++x) s[cc * 32 + x] = __uint_as_float(raw[x]);
        }
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&sm.s_free[e]);  // the tail's S may overwrite it
        // keys >= lim of this tile are masked (the tail's S has 64 columns:
        // the rest of the row is the first tile's and always masked)
        const int lim = m == 0 ? kv_eff : min(kv_eff - kRows, kTail);
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
        const float m_cand = fmaxf(m_used, mx * sl2);
        const bool raise = m_cand > m_used + kRescaleThreshold;
        float alpha = 1.f;
        if (raise) {
          alpha = ex2(m_used - m_cand);  // 0 on the first tile
          m_used = m_cand;
        }
        const float m_eff = m_used == -INFINITY ? 0.f : m_used;
        const uint64_t negm2 = f2_pack(-m_eff, -m_eff);
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
        const float rowsum = r0 + r1;
        if (m > 0) {
          // P V of the first key tile has finished: O is stable, P is free
          okw = __all_sync(0xffffffffu, mbar_wait(&sm.pv_done[e], static_cast<uint32_t>(c - 1) & 1u,
                                                  abort_flag));
          if (!okw) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
            for (int cc = 0; cc < kD / 32; ++cc) {
              uint32_t o[32];
              tmem_ld32(taddr + o_col(e) + cc * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
              tmem_st32(taddr + o_col(e) + cc * 32, o);
            }
            tmem_wait_st();
          }
        }
        l = l * alpha + rowsum;
        // P row -> TMEM lane r, two bf16 per 32-bit column (the MMA's A layout)
        uint32_t half[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) half[x] = pk[x];
        tmem_st32(taddr + p_col(e), half);
#pragma unroll
        for (int x = 0; x < 32; ++x) half[x] = pk[32 + x];
        tmem_st32(taddr + p_col(e) + 32, half);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sm.p_full[e]);
      }
      // ---- (3) epilogue: O / l -> bf16 -> staging -> TMA store (the Q tile
      // there has been read: its last S MMA completed before the last s_full)
      okw = okw && __all_sync(0xffffffffu, mbar_wait(&sm.pv_done[e], static_cast<uint32_t>(c - 1) & 1u,
                                                     abort_flag));
      ok = e == 0 ? named_bar_and<1>(128, okw) : named_bar_and<2>(128, okw);
      if (!ok) break;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int cc = 0; cc < kD / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(taddr + o_col(e) + cc * 32, o);
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
            tmem_ld32(taddr + e * 64 + cc * 32, o);
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

// Clusters of C CTAs of the output-projecting kernel that can be resident at
// once (clusters stay inside one GPC); 0 if none fits. Asked once per C.
int cross_out_max_clusters(int C) {
  static int cache[kMaxCluster + 1] = {};  // 0: not asked yet, -1: none fits
  if (C < 1 || C > kMaxCluster) return 0;
  const int known = __atomic_load_n(&cache[C], __ATOMIC_ACQUIRE);
  if (known != 0) return known > 0 ? known : 0;
  const size_t smem_bytes = sizeof(CrossSmem) + 1024;
  auto kernel = mha_cross_kernel<true>;
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

template <bool OUT>
cudaError_t launch_cross(const MhaFusedProblem& p, cudaStream_t stream) {
  const size_t smem_bytes = sizeof(CrossSmem) + 1024;  // + alignment slack
  auto kernel = mha_cross_kernel<OUT>;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(kernel, static_cast<int>(smem_bytes), &configured,
                                static_cast<int>(kLaunchRegs));
  if (e != cudaSuccess) return e;
  CrossArgs a;
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
    const int max_clusters = cross_out_max_clusters(C);
    if (max_clusters <= 0) return cudaErrorInvalidConfiguration;
    grid = (p.B < max_clusters ? p.B : max_clusters) * C;
  }
  cfg.gridDim = dim3(grid);
  return cudaLaunchKernelEx(&cfg, kernel, p.tm_xq, p.tm_xkv, p.tm_xkv_tail, p.tm_wq, p.tm_wk,
                            p.tm_wv, p.tm_o, p.tm_wo, p.tm_out, a);
}

}  // namespace

static_assert(sizeof(CrossSmem) + 1024 <= 227 * 1024, "shared memory per CTA");

int mha_cross_out_clusters(int h) {
  const int C = h / 2;
  if (h % 2 != 0 || C < 1 || C > kMaxCluster) return 0;
  return cross_out_max_clusters(C);
}

cudaError_t launch_mha_cross(const MhaFusedProblem& p, cudaStream_t stream) {
  if (p.self || p.h % 2 != 0 || p.d_model % 64 != 0 || p.d_model <= 0 || p.n_q < 1 ||
      p.n_q > kRows || p.n_k <= kRows || p.n_k > kRows + kTail)
    return cudaErrorInvalidValue;
  if (p.out) {
    const int C = p.h / 2;
    if (C > kMaxCluster || p.d_model % C != 0) return cudaErrorInvalidValue;
    const int n_slice = p.d_model / C;
    if (n_slice != 64 && n_slice != 128) return cudaErrorInvalidValue;
    return launch_cross<true>(p, stream);
  }
  return launch_cross<false>(p, stream);
}

TSD_DEFINE_ERROR_READER(take_device_error_cross)

}  // namespace tsd
