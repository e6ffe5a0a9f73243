// mha_cross.cu -- encoder-decoder (cross) multi-head attention in one kernel
// when the source is longer than one key tile: n_q <= 128 target rows,
// 128 < n_k <= 256 source rows, d_k = d_v = 64. The queries come from the
// decoder's rows, the keys and values from the encoder output
// ("[논문 리뷰]Attention Is All You Need" (kimjiil.github.io), section 3.2.3,
// the encoder-decoder attention row; heads per sections 3.2.1-3.2.2,
// head_i = Attention(X_q W_i^Q, X_kv W_i^K, X_kv W_i^V), weights in the x.W
// layout [d_model, h*64], no biases), up to the merged heads and optionally
// through the output projection (MultiHead = Concat(heads) W_O).
//
// A CTA owns one work item, (batch b, heads 2p and 2p+1), as the fused
// short-sequence kernel does; with the output projection the h/2 CTAs of a
// batch entry form a cluster and exchange their merged heads through L2 (the
// same protocol as in mha_fused.cu). What differs is the order of the
// projections. Q of both heads (2 x 64 fp32 columns) and K|V of both heads
// for two 128-row key tiles (4 x 128 columns) would need 640 of the 512
// tensor-memory columns, so:
//   Q pass   Q of both heads into columns [0, 128), its operands streamed
//            through the whole ring (six 32 KB stages); the head warpgroups
//            turn the rows into bf16 Q tiles in the epilogue's staging
//            buffers, which are idle until the epilogue
//   KV pass  K|V of both heads for key rows [0, 128) and [128, 256) (rows past
//            n_k are zero: the tensor map clips them) into all 512 columns,
//            through three 64 KB stages, each loaded as soon as the two Q
//            stages under it have been consumed; the head warpgroups turn
//            them into bf16 K and V tiles in the first 128 KB of the ring
// Each operand crosses from L2 once, with the ring's 192 KB in flight (the
// L2 -> SM rate grows with the bytes in flight: with two 64 KB stages for K|V
// and two 32 KB ones for Q the two passes took 9.6 us, one after the other).
// The attention then takes each head over its one or two key tiles with the
// online softmax (running max and sum in fp32).
//
//   warp 0      TMA producer
//   warp 1      MMA issuer (one thread): the Q pass, the KV pass, S = Q K^T
//               and O += P V per key tile, and (OUT) the output projection
//   warps 4..7  head 2p, warps 8..11 head 2p+1, one thread per row (= TMEM
//               lane): the Q row, then its K/V rows, to bf16 tiles; the
//               softmax of its query row; O / l -> bf16 -> staging -> TMA store
//
// Shared memory (ring, 192 KB):
//   Q pass stage s (32 KB: X_q slice, W_Q slices of both heads) at 32 s KB;
//   KV pass stage p (64 KB: X_kv rows [0,128) and [128,256) of one 64-wide
//   slice of d_model, the W_K, W_V slices of both heads) at 64 p KB, over Q
//   stages 2p and 2p+1; then the K/V tiles, tile (e, m, kv) at
//   16 KB x (4e + 2m + kv), in [0, 128) KB; the Q tiles in o[e]
//   OUT: the peers' merged tiles in [0, 96) KB and W_O chunks in a late ring
//   [96, 160) KB (free once the attention MMAs are done) and an early ring
//   [160, 192) KB for the CTA's own two heads' chunks (free once the KV pass
//   is done)
// Tensor memory (512 columns): Q_e at 64e; then K|V of (head e, key tile m)
// at 128 (2e + m); then S_e at 128e, P_e (bf16) at 256 + 64e, O_e at
// 384 + 64e; (OUT) the output columns at [0, n_slice).
#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kRows = 128;              // query rows and key rows per tile
constexpr int kD = 64;                  // d_k = d_v
constexpr int kTile = kRows * kD * 2;   // 16 KB: a 128 x 64 bf16 tile
constexpr int kWChunk = 64 * kD * 2;    // 8 KB: 64 rows of d_model x 64 columns of one weight
constexpr int kThreads = 384;           // 4 control warps + 2 head warpgroups
constexpr uint32_t kLaunchRegs = 65536 / kThreads / 8 * 8;  // 168
constexpr uint32_t kCtrlRegs = 72;
constexpr uint32_t kHeadRegs = (kLaunchRegs * kThreads - kCtrlRegs * 128) / 256 / 8 * 8;
static_assert(kCtrlRegs * 128 + kHeadRegs * 256 <= kLaunchRegs * kThreads, "register split");
constexpr unsigned long long kDrainLimitNs = 100ull * 1000ull * 1000ull;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

constexpr int kKvStage = 2 * kTile + 4 * kWChunk;  // 64 KB
constexpr int kKvStages = 3;
constexpr int kQStage = kTile + 2 * kWChunk;       // 32 KB
constexpr int kQStages = 6;
constexpr int kRingBytes = kKvStages * kKvStage;   // 192 KB
static_assert(kQStages * kQStage == kRingBytes && 2 * kQStage == kKvStage, "KV stage p over Q stages 2p, 2p+1");
constexpr int kSlot = 16384;     // a merged-heads tile, or 64 rows of W_O x <= 128 columns
constexpr int kOSlots = 6;       // peers' merged tiles, [0, 96) KB
constexpr int kWoLate = 4;       // [96, 160) KB
constexpr int kWoEarly = 2;      // [160, 192) KB
constexpr int kWoLateBase = kOSlots * kSlot;
constexpr int kWoEarlyBase = kWoLateBase + kWoLate * kSlot;
constexpr int kMaxCluster = 8;
static_assert(kWoEarlyBase + kWoEarly * kSlot == kRingBytes, "OUT layout fills the ring");
static_assert(kWoEarlyBase >= 8 * kTile, "early W_O slots clear of the K/V tiles");

__host__ __device__ constexpr uint32_t kv_col(int e, int m) { return static_cast<uint32_t>((2 * e + m) * 128); }
__host__ __device__ constexpr uint32_t q_col(int e) { return static_cast<uint32_t>(64 * e); }
__host__ __device__ constexpr uint32_t s_col(int e) { return static_cast<uint32_t>(128 * e); }
__host__ __device__ constexpr uint32_t p_col(int e) { return static_cast<uint32_t>(256 + 64 * e); }
__host__ __device__ constexpr uint32_t o_col(int e) { return static_cast<uint32_t>(384 + 64 * e); }
__host__ __device__ constexpr int kv_tile(int e, int m, int kv) { return 4 * e + 2 * m + kv; }

struct CrossSmem {
  alignas(1024) uint8_t ring[kRingBytes];
  alignas(1024) uint8_t o[2][kTile];  // epilogue staging, one per head
  uint64_t kv_full[kKvStages], kv_empty[kKvStages];
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t kv_done, q_done;        // KV pass / Q pass MMAs complete
  uint64_t kv_conv[2], q_conv[2];  // head e's accumulator rows turned into tiles
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t qkv_free;   // every MMA reading the item's Q/K/V tiles has completed
  uint64_t tmem_free;  // every head thread's reads of the item's tensor memory are done
  uint64_t drained;
  // output projection (OUT)
  uint64_t o_full[kOSlots], o_empty[kOSlots];
  uint64_t wl_full[kWoLate], wl_empty[kWoLate];
  uint64_t we_full[kWoEarly], we_empty[kWoEarly];
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
// Key tiles the attention takes (the second only when keys past 128 are visible).
__device__ __forceinline__ int key_tiles(int kv_eff) { return kv_eff > kRows ? 2 : 1; }

template <bool OUT>
__global__ void __launch_bounds__(kThreads, 1)
    mha_cross_kernel(const __grid_constant__ CUtensorMap tm_xq,
                     const __grid_constant__ CUtensorMap tm_xkv,
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
    for (int s = 0; s < kKvStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
    }
    mbar_init(&sm.kv_done, 1);
    mbar_init(&sm.q_done, 1);
    for (int e = 0; e < 2; ++e) {
      mbar_init(&sm.kv_conv[e], 128);
      mbar_init(&sm.q_conv[e], 128);
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
      for (int i = 0; i < kWoLate; ++i) {
        mbar_init(&sm.wl_full[i], 1);
        mbar_init(&sm.wl_empty[i], 1);
      }
      for (int i = 0; i < kWoEarly; ++i) {
        mbar_init(&sm.we_full[i], 1);
        mbar_init(&sm.we_empty[i], 1);
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
      int ui = 0, wl_cnt = 0, o_cnt = 0, armed = -1;
      int uq[kQStages] = {0, 0, 0, 0, 0, 0};  // loads issued into each Q stage so far
      int ukv[kKvStages] = {0, 0, 0};         // ... and into each KV stage
      int we_item[kWoEarly] = {-1, -1};  // item whose W_O chunk each early slot was last loaded for
      bool ok = true;
      bool waited = false;
      auto first_load = [&]() {
        if (!waited) {
          griddep_wait();
          waited = true;
        }
      };
      // Q pass k-block kb of head pair h0/2 into Q stage kb % kQStages
      auto load_q = [&](int b, int h0, int kb) -> bool {
        const int st = kb % kQStages;
        if (!mbar_wait(&sm.q_empty[st], (static_cast<uint32_t>(uq[st]) & 1u) ^ 1u, abort_flag))
          return false;
        mbar_arrive_expect_tx(&sm.q_full[st], kQStage);
        first_load();
        const int k0 = kb * 64;
        uint8_t* dst = sm.ring + st * kQStage;
        tma_load_3d(dst, &tm_xq, &sm.q_full[st], k0, 0, b);
        for (int e = 0; e < 2; ++e)
          tma_load_2d(dst + kTile + e * kWChunk, &tm_wq, &sm.q_full[st], (h0 + e) * kD, k0);
        ++uq[st];
        return true;
      };
      // KV pass k-block kb into KV stage (kb + 1) % kKvStages: the stage over
      // the Q stages consumed first (stage 0 lies under the last Q k-blocks)
      auto load_kv = [&](int b, int h0, int kb) -> bool {
        const int st = (kb + 1) % kKvStages;
        if (kb < kKvStages) {
          // first use in this item: the two Q stages under it have been read
          for (int qs = 2 * st; qs < 2 * st + 2; ++qs)
            if (uq[qs] > 0 &&
                !mbar_wait(&sm.q_empty[qs], static_cast<uint32_t>(uq[qs] - 1) & 1u, abort_flag))
              return false;
        }
        if (!mbar_wait(&sm.kv_empty[st], (static_cast<uint32_t>(ukv[st]) & 1u) ^ 1u, abort_flag))
          return false;
        mbar_arrive_expect_tx(&sm.kv_full[st], kKvStage);
        first_load();
        const int k0 = kb * 64;
        uint8_t* dst = sm.ring + st * kKvStage;
        tma_load_3d(dst, &tm_xkv, &sm.kv_full[st], k0, 0, b);
        tma_load_3d(dst + kTile, &tm_xkv, &sm.kv_full[st], k0, kRows, b);  // rows past n_k: zeros
        uint8_t* w = dst + 2 * kTile;
        for (int e = 0; e < 2; ++e) {
          const int col = (h0 + e) * kD;
          tma_load_2d(w + (2 * e) * kWChunk, &tm_wk, &sm.kv_full[st], col, k0);
          tma_load_2d(w + (2 * e + 1) * kWChunk, &tm_wv, &sm.kv_full[st], col, k0);
        }
        ++ukv[st];
        return true;
      };
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
        for (int kb = 0; ok && kb < args.kblocks; ++kb) ok = load_q(b, h0, kb);
        for (int kb = 0; ok && kb < args.kblocks; ++kb) ok = load_kv(b, h0, kb);
        if constexpr (OUT) {
          if (!ok) break;
          const int C = args.head_pairs;
          // chunk j of the output projection: head 2 ((pair + j/2) mod C) + j%2
          auto head_of = [&](int j) { return 2 * ((pair + (j >> 1)) % C) + (j & 1); };
          auto wo_box = [&](uint8_t* dst, uint64_t* bar, int j) {
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(args.n_slice) * 128u);
            for (int c = 0; c < args.n_slice; c += 64)
              tma_load_2d(dst + c * 128, &tm_wo, bar, pair * args.n_slice + c, head_of(j) * kD);
          };
          const uint32_t ph = static_cast<uint32_t>(ui) & 1u;
          // the own heads' W_O chunks once the KV pass has read its stages
          // (the early slots are the upper half of the last one)
          ok = mbar_wait(&sm.kv_done, ph, abort_flag);
          for (int j = 0; ok && j < kWoEarly && j < args.h; ++j) {
            ok = mbar_wait(&sm.we_empty[j], ph ^ 1u, abort_flag);
            if (!ok) break;
            wo_box(sm.ring + kWoEarlyBase + j * kSlot, &sm.we_full[j], j);
            we_item[j] = ui;
          }
          // the peers' merged tiles and the other W_O chunks into the K/V and
          // Q tiles' place, once those are consumed
          ok = ok && mbar_wait(&sm.qkv_free, ph, abort_flag);
          for (int j = kWoEarly; ok && j < args.h; ++j) {
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
            const int ws = wl_cnt % kWoLate;
            ok = mbar_wait(&sm.wl_empty[ws], (static_cast<uint32_t>(wl_cnt / kWoLate) & 1u) ^ 1u,
                           abort_flag);
            if (!ok) break;
            wo_box(sm.ring + kWoLateBase + ws * kSlot, &sm.wl_full[ws], j);
            ++wl_cnt;
          }
        }
      }
      if (!ok) {
        // wait (bounded) for this thread's copies still in flight
        volatile uint32_t never = 0;
        for (int st = 0; st < kKvStages; ++st)
          if (ukv[st] > 0)
            mbar_wait(&sm.kv_full[st], static_cast<uint32_t>(ukv[st] - 1) & 1u, &never,
                      kDrainLimitNs);
        for (int st = 0; st < kQStages; ++st)
          if (uq[st] > 0)
            mbar_wait(&sm.q_full[st], static_cast<uint32_t>(uq[st] - 1) & 1u, &never, kDrainLimitNs);
        if constexpr (OUT) {
          for (int i = max(0, wl_cnt - kWoLate); i < wl_cnt; ++i)
            mbar_wait(&sm.wl_full[i % kWoLate], static_cast<uint32_t>(i / kWoLate) & 1u, &never,
                      kDrainLimitNs);
          for (int i = max(0, o_cnt - kOSlots); i < o_cnt; ++i)
            mbar_wait(&sm.o_full[i % kOSlots], static_cast<uint32_t>(i / kOSlots) & 1u, &never,
                      kDrainLimitNs);
          // the early slots' last loads
          for (int j = 0; j < kWoEarly; ++j)
            if (we_item[j] >= 0)
              mbar_wait(&sm.we_full[j], static_cast<uint32_t>(we_item[j]) & 1u, &never,
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
      constexpr uint32_t kIdescKV = idesc_bf16(kRows, 2 * kD, false, true);
      constexpr uint32_t kIdescQ = idesc_bf16(kRows, kD, false, true);
      constexpr uint32_t kIdescS = idesc_bf16(kRows, kRows, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(kRows, kD, false, true);
      constexpr uint32_t kIdescOut128 = idesc_bf16(kRows, 128, false, true);
      constexpr uint32_t kIdescOut64 = idesc_bf16(kRows, 64, false, true);
      const uint32_t ring0 = smem_u32(sm.ring);
      // X: K-major, rows of 128 bytes; weights: N-major 64-column chunks 8 KB apart
      const uint64_t dkv0 = sdesc_sw128(ring0, 16, 1024);
      const uint64_t dkvw0 = sdesc_sw128(ring0 + 2 * kTile, kWChunk, 1024);
      const uint64_t dq0 = sdesc_sw128(ring0, 16, 1024);
      const uint64_t dqw0 = sdesc_sw128(ring0 + kTile, kWChunk, 1024);
      // Q and K tiles K-major (head dimension contiguous); V tiles N-major
      const uint64_t dt0 = sdesc_sw128(ring0, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(ring0, kTile, 1024);
      constexpr uint32_t kTileStep = kTile >> 4;
      constexpr uint32_t kWStep = kWChunk >> 4;
      int ui = 0, o_used = 0, wl_used = 0;
      int uq[kQStages] = {0, 0, 0, 0, 0, 0};  // each stage's loads consumed so far
      int ukv[kKvStages] = {0, 0, 0};
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
        // ---- Q pass: Q_e = X_q W_Q (head e) into columns [64 e, 64 e + 64)
        for (int kb = 0; ok && kb < args.kblocks; ++kb) {
          const int st = kb % kQStages;
          ok = mbar_wait(&sm.q_full[st], static_cast<uint32_t>(uq[st]) & 1u, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t so = static_cast<uint32_t>(st * kQStage) >> 4;
          const uint64_t dx = sdesc_advance(dq0, so);
          const uint64_t dw = sdesc_advance(dqw0, so);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc_flag = (kb > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
            for (int e = 0; e < 2; ++e)
              mma_bf16_ss(tmem + q_col(e), sdesc_advance(dx, kk * (32 >> 4)),
                          sdesc_advance(dw, e * kWStep + kk * (2048 >> 4)), kIdescQ, acc_flag);
          }
          mma_commit(&sm.q_empty[st]);
          ++uq[st];
        }
        if (!ok) break;
        mma_commit(&sm.q_done);
        // ---- KV pass: KV_{e,m} = X_kv[rows of tile m] [W_K | W_V] (head e),
        // into every column, once both heads have read their Q rows
        ok = mbar_wait(&sm.q_conv[0], ph, abort_flag) && mbar_wait(&sm.q_conv[1], ph, abort_flag);
        if (!ok) break;
        tc_fence_after();
        for (int kb = 0; ok && kb < args.kblocks; ++kb) {
          const int st = (kb + 1) % kKvStages;
          ok = mbar_wait(&sm.kv_full[st], static_cast<uint32_t>(ukv[st]) & 1u, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t so = static_cast<uint32_t>(st * kKvStage) >> 4;
          const uint64_t dx = sdesc_advance(dkv0, so);
          const uint64_t dw = sdesc_advance(dkvw0, so);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc_flag = (kb > 0 || kk > 0) ? 1u : 0u;
            const uint32_t aoff = kk * (32 >> 4);    // 16 elements along d_model
            const uint32_t woff = kk * (2048 >> 4);  // 16 rows of the weight slice
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
              for (int m = 0; m < 2; ++m)
                mma_bf16_ss(tmem + kv_col(e, m), sdesc_advance(dx, m * kTileStep + aoff),
                            sdesc_advance(dw, 2 * e * kWStep + woff), kIdescKV, acc_flag);
          }
          mma_commit(&sm.kv_empty[st]);
          ++ukv[st];
        }
        if (!ok) break;
        mma_commit(&sm.kv_done);
        // ---- attention, once every Q/K/V tile is written and every
        // accumulator under S, P and O has been read
        ok = mbar_wait(&sm.kv_conv[0], ph, abort_flag) && mbar_wait(&sm.kv_conv[1], ph, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const int nkt = key_tiles(key_limit(args, b));
        auto issue_s = [&](int e, int m) {
          const uint64_t a = sdesc_sw128(smem_u32(sm.o[e]), 16, 1024);  // Q tile (K-major)
          const uint64_t bk = sdesc_advance(dt0, static_cast<uint32_t>(kv_tile(e, m, 0)) * kTileStep);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_bf16_ss(tmem + s_col(e), sdesc_advance(a, kk * 2), sdesc_advance(bk, kk * 2),
                        kIdescS, kk > 0 ? 1u : 0u);
          mma_commit(&sm.s_full[e]);
        };
        auto issue_pv = [&](int e, int m) {
          const uint64_t bv = sdesc_advance(dv0, static_cast<uint32_t>(kv_tile(e, m, 1)) * kTileStep);
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk)
            mma_bf16_ts(tmem + o_col(e), tmem + p_col(e) + kk * 8,
                        sdesc_advance(bv, kk * (2048 >> 4)), kIdescPV, (m > 0 || kk > 0) ? 1u : 0u);
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
            // S_e of the second key tile overwrites the first, once it is read
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
            uint64_t a, bw;
            int os = -1;
            if (j < kWoEarly) {  // this CTA's own heads, still in the epilogue's staging tiles
              a = sdesc_sw128(smem_u32(sm.o[j]), 16, 1024);
              ok = mbar_wait(&sm.we_full[j], ph, abort_flag);
              bw = sdesc_sw128(ring0 + kWoEarlyBase + j * kSlot, kWChunk, 1024);
            } else {
              os = o_used % kOSlots;
              ok = mbar_wait(&sm.o_full[os], static_cast<uint32_t>(o_used / kOSlots) & 1u,
                             abort_flag);
              ++o_used;
              a = sdesc_sw128(ring0 + os * kSlot, 16, 1024);
              const int ws = wl_used % kWoLate;
              ok = ok && mbar_wait(&sm.wl_full[ws], static_cast<uint32_t>(wl_used / kWoLate) & 1u,
                                   abort_flag);
              ++wl_used;
              bw = sdesc_sw128(ring0 + kWoLateBase + ws * kSlot, kWChunk, 1024);
            }
            if (!ok) break;
            tc_fence_after();
            // W_O chunk: 64 rows x n_slice columns as 64-column blocks 8 KB apart
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_bf16_ss(tmem, sdesc_advance(a, kk * 2), sdesc_advance(bw, kk * (2048 >> 4)),
                          idesc_out, (j > 0 || kk > 0) ? 1u : 0u);
            if (j < kWoEarly) {
              mma_commit(&sm.we_empty[j]);
            } else {
              mma_commit(&sm.wl_empty[(wl_used - 1) % kWoLate]);
              mma_commit(&sm.o_empty[os]);
            }
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
    const int r = quarter * 32 + static_cast<int>(lane);  // row: query (and key) index in a tile
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
    // accumulator row (64 fp32 columns from `col`) -> bf16 row r of a
    // 128-byte-swizzled tile
    auto convert = [&](uint32_t col, uint8_t* tile) {
      uint8_t* row = tile + r * 128;
      uint32_t v[64];
      tmem_ld32(taddr + col, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld32(taddr + col + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
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
    for (int u = first; ok && u < args.num_units; u += stride, ++ui) {
      const int b = u / args.head_pairs;
      const int pair = u % args.head_pairs;
      const int hh = 2 * pair + e;
      const int kv_eff = key_limit(args, b);
      const int nkt = key_tiles(kv_eff);
      const uint32_t ph = static_cast<uint32_t>(ui) & 1u;
      // A failed wait is carried to the warpgroup's barrier below, where all
      // four warps stop together (none is left waiting at it).
      bool okw = __all_sync(0xffffffffu, mbar_wait(&sm.q_done, ph, abort_flag));
      // ---- (1) this row of Q -> bf16 tile in the staging buffer o[e], once
      // the previous item's stores from it have read it
      if (leader) bulk_wait_group_read<0>();
      okw = e == 0 ? named_bar_and<1>(128, okw) : named_bar_and<2>(128, okw);
      if (okw) {
        tc_fence_after();
        convert(q_col(e), sm.o[e]);
        fence_proxy_async_smem();  // the tile is read by the tensor cores
        tc_fence_before();         // and the KV pass overwrites the accumulator just read
        mbar_arrive(&sm.q_conv[e]);
      }
      // ---- (2) this row of K and V for both key tiles -> bf16 tiles
      okw = okw && __all_sync(0xffffffffu, mbar_wait(&sm.kv_done, ph, abort_flag));
      if (okw) {
        tc_fence_after();
        for (int m = 0; m < 2; ++m) {
          convert(kv_col(e, m), ring + kv_tile(e, m, 0) * kTile);
          convert(kv_col(e, m) + kD, ring + kv_tile(e, m, 1) * kTile);
        }
        fence_proxy_async_smem();
        tc_fence_before();         // S, P and O overwrite the accumulators just read
        mbar_arrive(&sm.kv_conv[e]);
      }
      // ---- (3) online softmax over the key tiles; P goes where head 1's
      // first K|V accumulator was (read once kv_conv[1] has completed)
      okw = okw && __all_sync(0xffffffffu, mbar_wait(&sm.kv_conv[1], ph, abort_flag));
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
        mbar_arrive(&sm.s_free[e]);  // the next key tile's S may overwrite it
        const int lim = kv_eff - m * kRows;  // keys >= lim of this tile are masked
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
          // P V of the previous key tile has finished: O is stable, P is free
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
      // ---- (4) epilogue: O / l -> bf16 -> staging -> TMA store
      okw = okw && __all_sync(0xffffffffu, mbar_wait(&sm.pv_done[e], static_cast<uint32_t>(c - 1) & 1u,
                                                     abort_flag));
      if (leader) bulk_wait_group_read<0>();  // the staging tile's previous store has read it
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
        // ---- (5) out[:, N pair + 64 e : + 64] (fp32 in TMEM) -> bf16 ->
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
  if (set_smem_once(kernel, static_cast<int>(smem_bytes), &configured) != cudaSuccess) return 0;
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
  cudaError_t e = set_smem_once(kernel, static_cast<int>(smem_bytes), &configured);
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
  return cudaLaunchKernelEx(&cfg, kernel, p.tm_xq, p.tm_xkv, p.tm_wq, p.tm_wk, p.tm_wv, p.tm_o,
                            p.tm_wo, p.tm_out, a);
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
      p.n_q > kRows || p.n_k <= kRows || p.n_k > 2 * kRows)
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
