// attn_bf16.cu -- scaled dot-product attention, softmax(Q K^T * scale) V, on
// the sm_103a tensor cores ("[논문 리뷰]Attention Is All You Need"
// (kimjiil.github.io), section 3.2.1, eq. (1)).
//
// Persistent kernel. The work items are (batch, head, query block), a query
// block being NQT tiles of 128 query rows; each pipeline walks its share of
// them (causal: largest blocks first). A CTA holds one pipeline, or two
// ("slots", for single-tile items at d = 64: a CTA that allocates tensor
// memory has its SM to itself, so two pipelines per SM share one CTA, each
// with its own warps, shared memory, barriers and 256 TMEM columns). Per
// pipeline (warp numbers within the slot):
//
//   warp 0      TMA producer: per item the Q tiles (double-buffered where
//               shared memory allows, so the next item's Q loads during this
//               one), then K_0, K_1, V_0, K_2, V_1, ... through two rings;
//               the rings run on across items
//   warps 1-3   MMA issuers (one thread each), S_t = Q_t K_j^T and
//               O_t += P_t V_j into tensor memory. The busier product gets one
//               issuer per query tile: at d = 128 (S: 8 MMAs of N=128 per
//               tile, PV: 8 of N=128) warps 1, 2 issue S for tiles 0, 1 and
//               warp 3 issues PV; at d = 64 (S: 4 MMAs, PV: 8 of N=64, the
//               less efficient shape) warp 1 issues S and warps 2, 3 issue PV
//               for tiles 0, 1. Warp 1 allocates the TMEM of all slots. Several
//               issuing threads keep the tensor pipe fed: each thread's waits
//               and commits (tcgen05.commit tracks only its own MMAs) overlap
//               the others' MMA issue.
//   warps 4..7  softmax for query tile 0; warps 8..11 for query tile 1:
//               one thread per query row (= one TMEM lane), then the epilogue:
//               O / l to bf16 into a 128-byte-swizzled staging tile and one
//               TMA store per 64 columns (a row per thread written straight
//               to global memory would scatter each warp store over 32 rows);
//               the d = 128 paired variant has no shared memory left for the
//               staging tile and stores rows directly
//
// The n_q x n_k weight matrix never leaves the chip: S lives in TMEM, P (bf16)
// in TMEM as the A operand of the PV MMA, one 128x128 tile at a time, with the
// online (running max and running sum) form of the row softmax in fp32.
// Scores become base-2 exponents with the folded factor scale*log2(e); the max
// is subtracted before the exponential, as the pages' reference run does
// ("Attention Is All You Need 해부" (sj-techlog), section "직접 검증").
// Masks: key tiles past the causal diagonal or past kv_len are never loaded
// (but for the first, loaded before kv_len is read, and unused if it is 0);
// inside the boundary tile the masked logits become -inf before the max and
// the exponential, so their weight is exactly 0 (section 3.2.3).
// The running max is only raised when it grows by more than 2^8 (exponents
// stay <= 256, exact in the final division), so the O rescale is rare.
//
// Every barrier phase is counted across items, per role, so each wait names
// the exact phase it needs; no wait can see a barrier two phases ahead of it.
#include <cuda_bf16.h>

#include <type_traits>

#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kRows = 128;                 // query rows per tile (MMA M) and keys per tile
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, int NQT, int SL>
struct AttnShape {
  // per slot: 4 control warps + NQT softmax warpgroups; SL slots per CTA
  static constexpr int kSlotThreads = 128 + 128 * NQT;
  static constexpr int kSlotWarps = kSlotThreads / 32;
  static constexpr int kThreads = SL * kSlotThreads;
  // P (bf16, 64 columns per query tile) gets its own TMEM columns unless S and
  // O of two 128-wide tiles already fill all 512; then it overwrites the first
  // half of its S tile, and S_t(j+1) waits for PV_t(j) to have read it.
  static constexpr bool kPAliasS = (D == 128 && NQT == 2);
  static constexpr int kColsUsed = NQT * kRows + NQT * D + (kPAliasS ? 0 : NQT * 64);
  static constexpr int kTmemCols = kColsUsed <= 256 ? 256 : 512;
  __host__ __device__ static constexpr int s_col(int t) { return t * kRows; }
  __host__ __device__ static constexpr int o_col(int t) { return NQT * kRows + t * D; }
  __host__ __device__ static constexpr int p_col(int t) {
    return kPAliasS ? s_col(t) : NQT * kRows + NQT * D + t * 64;
  }
  static_assert(SL == 1 || kTmemCols <= 256, "slots share the 512 tensor-memory columns");
  // control warps give up registers to the softmax warpgroups (the sum stays
  // within what the CTA was launched with); a single-tile single-slot CTA
  // has registers to spare and needs no split
  static constexpr bool kRegSplit = (NQT == 2) || (SL == 2);
  static constexpr uint32_t kLaunchRegs = 65536 / kThreads / 8 * 8;
  static constexpr uint32_t kCtrlRegs = NQT == 1 ? 56 : (D == 64 ? 72 : 104);
  static constexpr uint32_t kSoftmaxRegs =
      (kLaunchRegs * kSlotThreads - kCtrlRegs * 128) / (128 * NQT) / 8 * 8;
  // one issuer per query tile for S (else for PV), see the role table above
  static constexpr bool kSplitS = (D == 128);
  static constexpr int kSIssuers = kSplitS ? NQT : 1;
  static constexpr int kPVIssuers = kSplitS ? 1 : NQT;
  static_assert(kColsUsed <= 512, "tensor memory budget");
  // setmaxnreg.inc waits for registers released by .dec: the split must fit
  // in what the CTA was launched with, or the increase would never complete
  static_assert(!kRegSplit || kSoftmaxRegs <= 256, "register split");
  static_assert(!kRegSplit ||
                    SL * (kCtrlRegs * 128 + kSoftmaxRegs * 128 * NQT) <= kLaunchRegs * kThreads,
                "register split exceeds the launch allocation");
};

template <int D, int NQT, int NK, int NV, int QB, bool STO>
struct AttnSmem {
  static constexpr int kTileBytes = kRows * D * 2;  // one Q, K, V or O tile
  alignas(1024) uint8_t q[QB][NQT][kTileBytes];
  alignas(1024) uint8_t k[NK][kTileBytes];
  alignas(1024) uint8_t v[NV][kTileBytes];
  alignas(1024) uint8_t o[NQT][STO ? kTileBytes : 16];  // epilogue staging
  uint64_t q_full[QB], q_empty[QB];
  uint64_t k_full[NK], k_empty[NK];
  uint64_t v_full[NV], v_empty[NV];
  uint64_t s_full[NQT];
  uint64_t s_free[NQT];
  uint64_t p_full[NQT];
  uint64_t pv_done[NQT];
  uint64_t s_drained[NQT], pv_drained[NQT];
  uint32_t abort_flag;
};

struct AttnArgs {
  int B, h, n_q, n_k, n_qblocks, num_items;
  int mask_kind;
  const int32_t* kv_lens;
  float scale_log2;
  uint16_t* out;
  int64_t o_sb, o_sh, o_sr;
  int win_left, win_right;  // restricted window (WIN): keys [i - left, i + right]; < 0: no bound
  int tail_start;  // items from here on are single query tiles, two per query block
};

constexpr unsigned long long kDrainLimitNs = 100ull * 1000ull * 1000ull;  // 0.1 s

// One work item: a block of NQT query tiles of one (batch, head).
struct Item {
  int b, hh, q0, kv_eff;
  int nt0, nt1;  // query tile 0 / 1 visits key tiles [lo, nt)
  int lo0, lo1;  // 0 unless a restricted window cuts the keys before the query
  int lo_spec;   // first key tile through the rings (known before the key length)
  int min_load;  // 1 if the key set is not empty by its shape (n_k > 0)
  bool single;   // one query tile of a block (tile 1 of the item is idle)
  __device__ int nt(int t) const { return t == 0 ? nt0 : nt1; }
  __device__ int lo(int t) const { return t == 0 ? lo0 : lo1; }
  __device__ int nt_all() const { return nt0 > nt1 ? nt0 : nt1; }
  // K/V tiles that pass through the rings, from lo_spec: at least one when
  // n_k > 0, so that the first key tile can be loaded before the key length
  // is known (an item whose key set turns out empty releases it unused)
  __device__ int n_load() const {
    const int n = nt_all() - lo_spec;
    return n > min_load ? n : min_load;
  }
};

// First key tile of a query tile whose first row is row0 (restricted window).
template <bool WIN>
__device__ __forceinline__ int window_lo_tile(const AttnArgs& a, int row0) {
  if (!WIN || a.win_left < 0) return 0;
  const int k0 = row0 - a.win_left;
  return k0 > 0 ? k0 / kRows : 0;
}

// Batch, head and first query row of item w (no memory access). TS: the
// instance splits the last partial round of paired items into single tiles.
template <int NQT, bool WIN, bool TS>
__device__ __forceinline__ Item item_coords(const AttnArgs& a, int w) {
  const bool causal = (a.mask_kind & kMaskCausal) != 0;
  const int bh_count = a.B * a.h;
  int bh, qblk;
  if (causal) {  // longest first: every head's last query block, then the one before, ...
    qblk = a.n_qblocks - 1 - w / bh_count;
    bh = w % bh_count;
  } else {       // a head's query blocks together, so its K/V stays in L2
    // past tail_start a query block is two items of one tile each
    const int bw = (!TS || w < a.tail_start) ? w : a.tail_start + ((w - a.tail_start) >> 1);
    bh = bw / a.n_qblocks;
    qblk = bw % a.n_qblocks;
  }
  Item it;
  it.b = bh / a.h;
  it.hh = bh % a.h;
  it.single = TS && !causal && w >= a.tail_start;
  it.q0 = qblk * NQT * kRows + (it.single && ((w - a.tail_start) & 1) ? kRows : 0);
  it.kv_eff = 0;
  it.nt0 = it.nt1 = 0;
  it.lo_spec = window_lo_tile<WIN>(a, it.q0);
  it.lo0 = it.lo_spec;
  it.lo1 = NQT > 1 ? window_lo_tile<WIN>(a, it.q0 + kRows) : it.lo_spec;
  it.min_load = a.n_k > 0 ? 1 : 0;
  return it;
}

// The key range of an item (reads the key length).
template <int NQT, bool WIN, bool TS>
__device__ __forceinline__ Item item_at(const AttnArgs& a, int w) {
  const bool causal = (a.mask_kind & kMaskCausal) != 0;
  Item it = item_coords<NQT, WIN, TS>(a, w);
  int kv_eff = a.n_k;
  if (a.mask_kind & kMaskKeyPadding) {
    const int len = a.kv_lens[it.b];
    kv_eff = len < 0 ? 0 : (len > a.n_k ? a.n_k : len);
  }
  it.kv_eff = kv_eff;
  const int nkt = (kv_eff + kRows - 1) / kRows;
  auto tiles_for = [&](int t) {
    const int row0 = it.q0 + t * kRows;
    int n = nkt;
    if (causal) n = min(n, row0 / kRows + 1);
    if (WIN && a.win_right >= 0) n = min(n, (row0 + kRows + a.win_right + kRows - 1) / kRows);
    if (row0 >= a.n_q) n = 0;
    return n;
  };
  it.nt0 = tiles_for(0);
  it.nt1 = (NQT > 1 && !it.single) ? tiles_for(1) : 0;
  return it;
}

template <int D, int NQT, int NK, int NV, int QB, bool STO, int SL, bool MS, bool WIN, bool TS>
__global__ void __launch_bounds__(AttnShape<D, NQT, SL>::kThreads, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_o, const AttnArgs args) {
  using Smem = AttnSmem<D, NQT, NK, NV, QB, STO>;
  using Shape = AttnShape<D, NQT, SL>;
  constexpr int kKAtoms = D / 64;  // 128-byte swizzle atoms along the head dimension

  // Slots: SL independent pipelines in one CTA (a CTA that allocates tensor
  // memory has an SM to itself, so a second pipeline per SM has to live in
  // the same CTA). Each slot has its own warps, shared memory, barriers and
  // tensor-memory columns, and walks its own items.
  const int slot = SL > 1 ? warp_id() / Shape::kSlotWarps : 0;
  const int warp = warp_id() - slot * Shape::kSlotWarps;  // warp within the slot
  const uint32_t lane = lane_id();
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023))[slot];
  __shared__ uint32_t tmem_all;

  const bool causal = (args.mask_kind & kMaskCausal) != 0;
  // Item i of this slot: round i over all slots of the grid (slot 0 of every
  // CTA before any slot 1, so that no SM holds two items while another is
  // idle), taken in snake order (forward in even rounds, backward in odd
  // ones), so that with causal items sorted longest first every slot's
  // total stays close to the others'.
  const int vcta = slot * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
  const int vgrid = SL * static_cast<int>(gridDim.x);
  auto item_index = [&](int i) { return i * vgrid + ((i & 1) ? vgrid - 1 - vcta : vcta); };

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < QB; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], Shape::kSIssuers);  // one release per S-issuing warp
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], Shape::kSIssuers);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], Shape::kPVIssuers);  // one release per PV-issuing warp
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.s_free[t], kRows);
      mbar_init(&sm.p_full[t], kRows);
      mbar_init(&sm.pv_done[t], 1);
      mbar_init(&sm.s_drained[t], 1);
      mbar_init(&sm.pv_drained[t], 1);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp_id() == 1) {  // one allocation for all slots (the permit is per CTA)
    tmem_alloc(&tmem_all, SL * Shape::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_all + static_cast<uint32_t>(slot * Shape::kTmemCols);
  volatile uint32_t* abort_flag = &sm.abort_flag;
  if (warp == 0 && lane == 0) {
    // descriptors live in the kernel parameters: fetched while the previous
    // kernel finishes
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if constexpr (STO) tma_prefetch_desc(&tm_o);
  }
  // Everything up to a role's first global-memory access may overlap the
  // previous kernel: each role waits for it (griddep_wait) just before.
  griddep_launch_dependents();

  // Descriptors are built once; each MMA only advances the start-address
  // field by a compile-time offset (sdesc_advance keeps the sum inside it).
  constexpr uint32_t kTileStep = Smem::kTileBytes >> 4;
  constexpr uint32_t kIdescS = idesc_bf16(kRows, kRows, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16(kRows, D, false, true);

  if (warp < 4) {
    if constexpr (Shape::kRegSplit) regs_decrease<Shape::kCtrlRegs>();
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        int qn = 0, kn = 0, vn = 0;  // items / tiles issued into each ring
        bool ok = true;
        auto load_k = [&](const Item& it, int j) {
          const int rs = kn % NK;
          if (!mbar_wait(&sm.k_empty[rs], (static_cast<uint32_t>(kn / NK) & 1u) ^ 1u, abort_flag))
            return false;
          mbar_arrive_expect_tx(&sm.k_full[rs], Smem::kTileBytes);
          for (int a = 0; a < kKAtoms; ++a)
            tma_load_4d(sm.k[rs] + a * 16384, &tm_k, &sm.k_full[rs], a * 64, j * kRows, it.hh,
                        it.b);
          ++kn;
          return true;
        };
        auto load_v = [&](const Item& it, int j) {
          const int rs = vn % NV;
          if (!mbar_wait(&sm.v_empty[rs], (static_cast<uint32_t>(vn / NV) & 1u) ^ 1u, abort_flag))
            return false;
          mbar_arrive_expect_tx(&sm.v_full[rs], Smem::kTileBytes);
          for (int a = 0; a < kKAtoms; ++a)
            tma_load_4d(sm.v[rs] + a * 16384, &tm_v, &sm.v_full[rs], a * 64, j * kRows, it.hh,
                        it.b);
          ++vn;
          return true;
        };
        if (NQT == 2 && item_index(0) < args.num_items) {
          // While the previous kernel finishes, the first item's Q tiles and
          // its first key and value tiles (as many as the rings hold, by the
          // item's shape: the key length is read only after the wait) are
          // prefetched into L2; the loads below, issued after the wait, then
          // find them there (measured: causal B=8 h=16 n=1024 600 -> 630
          // TFLOP/s, +0.3-0.6 % on the other paired launches; the
          // single-tile, two-slot launches of short sequences measured
          // slower with it, 8.37 -> 8.69 us, and do without).
          const Item at = item_coords<NQT, WIN, TS>(args, item_index(0));
          for (int t = 0; t < NQT; ++t)
            for (int a = 0; a < kKAtoms; ++a)
              tma_prefetch_l2_4d(&tm_q, a * 64, at.q0 + t * kRows, at.hh, at.b);
          const int last_row = at.q0 + NQT * kRows - 1;
          int nt = (args.n_k + kRows - 1) / kRows;
          if (causal) nt = min(nt, last_row / kRows + 1);
          if (WIN && args.win_right >= 0) nt = min(nt, (last_row + args.win_right) / kRows + 1);
          const int cnt = min(nt - at.lo_spec, NK < NV ? NK : NV);
          for (int jj = 0; jj < cnt; ++jj)
            for (int a = 0; a < kKAtoms; ++a) {
              tma_prefetch_l2_4d(&tm_k, a * 64, (at.lo_spec + jj) * kRows, at.hh, at.b);
              tma_prefetch_l2_4d(&tm_v, a * 64, (at.lo_spec + jj) * kRows, at.hh, at.b);
            }
        }
        for (int i = 0, w = item_index(0); ok && w < args.num_items; w = item_index(++i)) {
          // Q and the first key tile do not depend on the key length: both
          // are on their way before it is read
          const Item at = item_coords<NQT, WIN, TS>(args, w);
          const int qs = qn % QB;
          ok = mbar_wait(&sm.q_empty[qs], (static_cast<uint32_t>(qn / QB) & 1u) ^ 1u, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&sm.q_full[qs], NQT * Smem::kTileBytes);
          if (qn == 0) griddep_wait();
          for (int t = 0; t < NQT; ++t)
            for (int a = 0; a < kKAtoms; ++a)
              tma_load_4d(sm.q[qs][t] + a * 16384, &tm_q, &sm.q_full[qs], a * 64,
                          at.q0 + t * kRows, at.hh, at.b);
          ++qn;
          if (at.min_load > 0) ok = load_k(at, at.lo_spec);
          const int n_load = item_at<NQT, WIN, TS>(args, w).n_load();
          // keys run one tile ahead of values, the order the MMAs consume them
          for (int jj = 0; ok && jj < n_load; ++jj) {
            if (jj + 1 < n_load) ok = load_k(at, at.lo_spec + jj + 1);
            if (ok) ok = load_v(at, at.lo_spec + jj);
          }
        }
        if (!ok) {
          // wait (bounded) for this thread's copies still in flight
          volatile uint32_t never = 0;
          for (int i = max(0, qn - QB); i < qn; ++i)
            mbar_wait(&sm.q_full[i % QB], static_cast<uint32_t>(i / QB) & 1u, &never, kDrainLimitNs);
          for (int i = max(0, kn - NK); i < kn; ++i)
            mbar_wait(&sm.k_full[i % NK], static_cast<uint32_t>(i / NK) & 1u, &never, kDrainLimitNs);
          for (int i = max(0, vn - NV); i < vn; ++i)
            mbar_wait(&sm.v_full[i % NV], static_cast<uint32_t>(i / NV) & 1u, &never, kDrainLimitNs);
        }
      }
    } else if (warp - 1 < Shape::kSIssuers) {
      // ---------------------------------------------------------- S issuer(s)
      // tiles [t_lo, t_hi) of this issuer, in order within each key tile
      const int t_lo = Shape::kSplitS ? warp - 1 : 0;
      const int t_hi = Shape::kSplitS ? warp : NQT;
      if (lane == 0) {
        const uint64_t dq0 = sdesc_sw128(smem_u32(sm.q[0][0]), 16, 1024);  // K-major Q
        const uint64_t dk0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);     // K-major K
        int qc = 0, kc = 0;    // items / key tiles consumed
        int sc0 = 0, sc1 = 0;  // S tiles issued per query tile (phase counters)
        bool ok = true;
        griddep_wait();  // the key lengths may come from the previous kernel
        for (int i = 0, w = item_index(0); ok && w < args.num_items; w = item_index(++i)) {
          const Item it = item_at<NQT, WIN, TS>(args, w);
          const int n_load = it.n_load();
          const int qs = qc % QB;
          ok = mbar_wait(&sm.q_full[qs], static_cast<uint32_t>(qc / QB) & 1u, abort_flag);
          if (!ok) break;
          bool item_issued = false;
          for (int jj = 0; ok && jj < n_load; ++jj) {
            const int j = it.lo_spec + jj;  // key tile
            const int rs = kc % NK;
            // the ring slot holds K_j before this warp releases it, so a release
            // for tiles this issuer skips never counts toward an older use
            ok = mbar_wait(&sm.k_full[rs], static_cast<uint32_t>(kc / NK) & 1u, abort_flag);
            if (!ok) break;
            const uint64_t bk = sdesc_advance(dk0, static_cast<uint32_t>(rs) * kTileStep);
            bool issued = false;
            for (int t = t_lo; ok && t < t_hi; ++t) {
              if (j >= it.nt(t) || j < it.lo(t)) continue;
              int& sc = t == 0 ? sc0 : sc1;
              if (sc > 0) {
                // the previous S_t has been read (or, when P overwrites S,
                // consumed by PV)
                ok = Shape::kPAliasS
                         ? mbar_wait(&sm.pv_done[t], static_cast<uint32_t>(sc - 1) & 1u, abort_flag)
                         : mbar_wait(&sm.s_free[t], static_cast<uint32_t>(sc - 1) & 1u, abort_flag);
                if (!ok) break;
              }
              tc_fence_after();
              // S_t = Q_t K^T : K-major A and B, K = head dimension in steps of 16
              const uint32_t d_tmem = tmem + Shape::s_col(t);
              const uint64_t a =
                  sdesc_advance(dq0, static_cast<uint32_t>(qs * NQT + t) * kTileStep);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = static_cast<uint32_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                mma_bf16_ss(d_tmem, sdesc_advance(a, off), sdesc_advance(bk, off), kIdescS,
                            kk > 0 ? 1u : 0u);
              }
              mma_commit(&sm.s_full[t]);
              ++sc;
              issued = true;
            }
            if (!ok) break;
            if (issued) mma_commit(&sm.k_empty[rs]);
            else mbar_arrive(&sm.k_empty[rs]);
            item_issued = item_issued || issued;
            ++kc;
          }
          if (!ok) break;
          // the Q slot is free once this issuer's S MMAs of the item are done
          if (item_issued) mma_commit(&sm.q_empty[qs]);
          else mbar_arrive(&sm.q_empty[qs]);
          ++qc;
        }
        // every issued MMA has completed before tensor memory is released
        volatile uint32_t never = 0;
        mma_commit(&sm.s_drained[t_lo]);
        mbar_wait(&sm.s_drained[t_lo], 0, &never, kDrainLimitNs);
      }
    } else if (warp - 1 - Shape::kSIssuers < Shape::kPVIssuers) {
      // ---------------------------------------------------------- PV issuer(s)
      const int widx = warp - 1 - Shape::kSIssuers;
      const int t_lo = Shape::kSplitS ? 0 : widx;
      const int t_hi = Shape::kSplitS ? NQT : widx + 1;
      if (lane == 0) {
        const uint64_t dv0 = sdesc_sw128(smem_u32(sm.v[0]), 16384, 1024);  // N-major V
        int vc = 0;            // value tiles consumed
        int pc0 = 0, pc1 = 0;  // PV products issued per query tile (phase counters)
        bool ok = true;
        griddep_wait();
        for (int i = 0, w = item_index(0); ok && w < args.num_items; w = item_index(++i)) {
          const Item it = item_at<NQT, WIN, TS>(args, w);
          const int n_load = it.n_load();
          for (int jj = 0; ok && jj < n_load; ++jj) {
            const int j = it.lo_spec + jj;  // key tile
            const int rs = vc % NV;
            // as for K: the ring slot holds V_j before any release by this warp
            ok = mbar_wait(&sm.v_full[rs], static_cast<uint32_t>(vc / NV) & 1u, abort_flag);
            if (!ok) break;
            const uint64_t bv = sdesc_advance(dv0, static_cast<uint32_t>(rs) * kTileStep);
            bool issued = false;
            for (int t = t_lo; ok && t < t_hi; ++t) {
              if (j >= it.nt(t) || j < it.lo(t)) continue;
              int& pc = t == 0 ? pc0 : pc1;
              ok = mbar_wait(&sm.p_full[t], static_cast<uint32_t>(pc) & 1u, abort_flag);
              if (!ok) break;
              tc_fence_after();
              // O_t (+)= P_t V : P from TMEM (keys = K), V N-major, 16 keys per MMA
              const uint32_t d_tmem = tmem + Shape::o_col(t);
              const uint32_t p_tmem = tmem + Shape::p_col(t);
#pragma unroll
              for (int kk = 0; kk < kRows / 16; ++kk)
                mma_bf16_ts(d_tmem, p_tmem + kk * 8, sdesc_advance(bv, kk * (2048 >> 4)), kIdescPV,
                            (j > it.lo(t) || kk > 0) ? 1u : 0u);
              mma_commit(&sm.pv_done[t]);
              ++pc;
              issued = true;
            }
            if (!ok) break;
            if (issued) mma_commit(&sm.v_empty[rs]);
            else mbar_arrive(&sm.v_empty[rs]);
            ++vc;
          }
        }
        volatile uint32_t never = 0;
        mma_commit(&sm.pv_drained[t_lo]);
        mbar_wait(&sm.pv_drained[t_lo], 0, &never, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    if constexpr (Shape::kRegSplit) regs_increase<Shape::kSoftmaxRegs>();
    const int t = (warp - 4) >> 2;           // query tile of this warpgroup
    const int quarter = warp & 3;             // TMEM lane quarter of this warp
    const int r = quarter * 32 + static_cast<int>(lane);  // row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t taddr_s = tmem + lane_base + Shape::s_col(t);
    const uint32_t taddr_o = tmem + lane_base + Shape::o_col(t);
    const uint32_t taddr_p = tmem + lane_base + Shape::p_col(t);
    const float sl2 = args.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    const bool leader = (quarter == 0 && lane == 0);  // issues the tile's TMA stores
    int c = 0;  // S / P tiles of this query tile so far (phase counter)
    bool ok = true;
    griddep_wait();
    for (int i = 0, w = item_index(0); ok && w < args.num_items; w = item_index(++i)) {
      const Item it = item_at<NQT, WIN, TS>(args, w);
      if (TS && t == 1 && it.single) continue;  // a single-tile item: no rows for tile 1
      const int ntt = it.nt(t);
      const int lot = it.lo(t);                // key tiles [lot, ntt) of this query tile
      const bool has_tiles = ntt > lot;
      const int row = it.q0 + t * kRows + r;  // query index
      // keys [low_row, lim_row) of this row
      int lim_row = causal ? min(it.kv_eff, row + 1) : it.kv_eff;
      int low_row = 0;
      if constexpr (WIN) {
        if (args.win_right >= 0) lim_row = min(lim_row, row + args.win_right + 1);
        if (args.win_left >= 0) low_row = max(0, row - args.win_left);
      }
      float m_used = -INFINITY;
      float l = 0.f;
      for (int j = lot; j < ntt; ++j, ++c) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&sm.s_full[t], static_cast<uint32_t>(c) & 1u, abort_flag));
        if (!ok) break;
        tc_fence_after();
        float s[kRows];
        const int bound = lim_row - j * kRows;   // keys >= bound of this tile are masked
        const int lbound = low_row - j * kRows;  // and (WIN) keys < lbound
        // S row -> registers (masked keys -> -inf) -> row max. With MS there
        // are two copies, and the tiles inside every row's key limit take the
        // one without the masking code: at d = 64 with long rows its mere
        // presence slows the loop by several percent (measured; with the
        // causal mask the single copy measures faster).
        auto load_max = [&](auto masked) -> float {
#pragma unroll
          for (int cc = 0; cc < kRows / 32; ++cc) {
            uint32_t raw[32];
            tmem_ld32(taddr_s + cc * 32, raw);
#pragma unroll
            for (int e = 0; e < 32; ++e) s[cc * 32 + e] = __uint_as_float(raw[e]);
          }
          tmem_wait_ld();
          if constexpr (decltype(masked)::value) {
            if (MS || bound < kRows || (WIN && lbound > 0)) {
#pragma unroll
              for (int e = 0; e < kRows; ++e)
                if (e >= bound || (WIN && e < lbound)) s[e] = -INFINITY;
            }
          }
          // row max: 8 independent chains of 3-input max
          float mx8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(s[e], s[e + 8]);
#pragma unroll
          for (int e0 = 16; e0 < kRows; e0 += 16)
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = fmax3(mx8[e], s[e0 + e], s[e0 + 8 + e]);
          return fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                       fmaxf(mx8[6], mx8[7]));
        };
        const float mx = (MS && __all_sync(0xffffffffu, bound >= kRows && (!WIN || lbound <= 0)))
                             ? load_max(std::false_type{})
                             : load_max(std::true_type{});
        // S_t is free for the next S_t only now, after the row max: the tensor
        // pipe executes MMAs in issue order, and PV_t of the previous tile,
        // issued when its P was stored, should run before the next S_t -- this
        // tile's P store waits for it, while the next S is not needed until
        // this iteration ends.
        tc_fence_before();
        mbar_arrive(&sm.s_free[t]);
        const float m_cand = fmaxf(m_used, mx * sl2);
        const bool raise = m_cand > m_used + kRescaleThreshold;
        float alpha = 1.f;
        if (raise) {
          alpha = ex2(m_used - m_cand);  // 0 on the first tile
          m_used = m_cand;
        }
        const float m_eff = m_used == -INFINITY ? 0.f : m_used;
        const uint64_t negm2 = f2_pack(-m_eff, -m_eff);

        // p = 2^(s*scale*log2e - m): packed FFMA2, two MUFU ex2, packed FADD2
        uint32_t pk[kRows / 2];
        uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int e = 0; e < kRows / 2; ++e) {
          float x0, x1;
          f2_unpack(ffma2(f2_pack(s[2 * e], s[2 * e + 1]), sl2x2, negm2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          pk[e] = pack_bf16x2(p0, p1);
          acc2[e & 3] = fadd2(acc2[e & 3], f2_pack(p0, p1));
        }
        float r0, r1;
        f2_unpack(fadd2(fadd2(acc2[0], acc2[1]), fadd2(acc2[2], acc2[3])), r0, r1);
        const float rowsum = r0 + r1;

        if (j > lot) {
          // PV of the previous tile has finished: O is stable, P is free
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.pv_done[t], static_cast<uint32_t>(c - 1) & 1u,
                                                 abort_flag));
          if (!ok) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t o[32];
              tmem_ld32(taddr_o + cc * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st32(taddr_o + cc * 32, o);
            }
            tmem_wait_st();
          }
        }
        l = l * alpha + rowsum;

        // P row -> TMEM lane r, two bf16 per 32-bit column (the MMA's A layout)
        {
          uint32_t half[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) half[e] = pk[e];
          tmem_st32(taddr_p, half);
#pragma unroll
          for (int e = 0; e < 32; ++e) half[e] = pk[32 + e];
          tmem_st32(taddr_p + 32, half);
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&sm.p_full[t]);
      }
      if (!STO && !ok) break;

      // -------------------------------------------------------- epilogue
      if (ok && has_tiles) {
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.pv_done[t], static_cast<uint32_t>(c - 1) & 1u,
                                               abort_flag));
      }
      if constexpr (STO) {
        // the staging tile's previous store has finished reading it, and the
        // warpgroup's four warps take one decision (none is left at a barrier)
        if (leader) bulk_wait_group_read<0>();
        // one named barrier per (slot, query tile); ids are immediates
        switch (slot * NQT + t) {
          case 0: ok = named_bar_and<1>(kRows, ok); break;
          case 1: ok = named_bar_and<2>(kRows, ok); break;
          case 2: ok = named_bar_and<3>(kRows, ok); break;
          default: ok = named_bar_and<4>(kRows, ok); break;
        }
      }
      if (!ok) break;
      if (has_tiles) tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      uint16_t* dst = args.out + static_cast<int64_t>(it.b) * args.o_sb +
                      static_cast<int64_t>(it.hh) * args.o_sh + static_cast<int64_t>(row) * args.o_sr;
      const bool store = row < args.n_q;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        if (has_tiles) {
          tmem_ld32(taddr_o + cc * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        uint32_t wv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          wv[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
        if constexpr (STO) {
          // 128-byte swizzle of the store's tensor map: 16-byte chunk jj of
          // row r sits at chunk position jj ^ (r mod 8) of the row's 128 bytes
          uint8_t* box = sm.o[t] + (cc >> 1) * 16384 + r * 128;
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const int jj = (cc & 1) * 4 + v4;
            st_shared_v4(smem_u32(box + ((jj ^ (r & 7)) << 4)), wv[4 * v4], wv[4 * v4 + 1],
                         wv[4 * v4 + 2], wv[4 * v4 + 3]);
          }
        } else if (store) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            st_global_v4(dst + cc * 32 + v4 * 8, wv[4 * v4], wv[4 * v4 + 1], wv[4 * v4 + 2],
                         wv[4 * v4 + 3]);
        }
      }
      if constexpr (STO) {
        fence_proxy_async_smem();  // staged bytes visible to the TMA unit
        switch (slot * NQT + t) {
          case 0: named_bar_sync<1>(kRows); break;
          case 1: named_bar_sync<2>(kRows); break;
          case 2: named_bar_sync<3>(kRows); break;
          default: named_bar_sync<4>(kRows); break;
        }
        const int row0 = it.q0 + t * kRows;
        if (leader && row0 < args.n_q) {  // the map clips rows past n_q
#pragma unroll
          for (int bx = 0; bx < D / 64; ++bx)
            tma_store_4d(&tm_o, sm.o[t] + bx * 16384, bx * 64, row0, it.hh, it.b);
          bulk_commit_group();
        }
      }
      // the O reads above complete before this tile's next P store signals PV
      tc_fence_before();
    }
    // the stores have read the staging tiles before the CTA's shared memory
    // goes; their global writes complete with the grid
    if (STO && leader) bulk_wait_group_read<0>();
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp_id() == 1) tmem_dealloc(tmem_all, SL * Shape::kTmemCols);
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

template <int D, int NQT, int NK, int NV, int QB, bool STO, int SL, bool MS = false,
          bool WIN = false, bool TS = false>
cudaError_t launch_variant(const AttnProblem& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, const CUtensorMap& tm_o, cudaStream_t stream) {
  using Smem = AttnSmem<D, NQT, NK, NV, QB, STO>;
  using Shape = AttnShape<D, NQT, SL>;
  const size_t smem_bytes = SL * sizeof(Smem) + 1024;  // + alignment slack
  auto kernel = attn_fwd_bf16_kernel<D, NQT, NK, NV, QB, STO, SL, MS, WIN, TS>;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(kernel, static_cast<int>(smem_bytes), &configured,
                                Shape::kRegSplit ? static_cast<int>(Shape::kLaunchRegs) : 0);
  if (e != cudaSuccess) return e;
  AttnArgs a;
  a.B = p.B;
  a.h = p.h;
  a.n_q = p.n_q;
  a.n_k = p.n_k;
  a.n_qblocks = (p.n_q + NQT * kRows - 1) / (NQT * kRows);
  const long long items = static_cast<long long>(a.n_qblocks) * p.h * p.B;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL - (1LL << 20)) return cudaErrorInvalidValue;  // item indices fit int
  a.num_items = static_cast<int>(items);
  // Quantisation tail: when the last round of paired items over the grid is
  // partial and its blocks, split into single query tiles, still fit in one
  // round, those blocks run as single tiles (about half an item's time each),
  // so the last round ends sooner (measured: B=8 h=16 n=1024 d=64 823 -> 849
  // TFLOP/s; d=128 B=2 n=4096 1100 -> 1142). Non-causal instances only:
  // causal items are already taken longest first, and the causal and window
  // instances measured slower with the split's code compiled in (window
  // n=16384 +-256: 589 -> 545 TFLOP/s, its 4096 items leave no tail worth it).
  a.tail_start = 0x7fffffff;
  if (TS && NQT == 2 && SL == 1 && !(p.mask_kind & kMaskCausal)) {
    const long long G = items < num_sms() ? items : num_sms();
    const long long full = items / G * G;
    const long long tail = items - full;
    if (full > 0 && tail > 0 && 2 * tail <= G) {
      a.tail_start = static_cast<int>(full);
      a.num_items = static_cast<int>(full + 2 * tail);
    }
  }
  a.mask_kind = p.mask_kind;
  a.kv_lens = p.kv_lens;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.out = p.out;
  a.o_sb = p.o_sb;
  a.o_sh = p.o_sh;
  a.o_sr = p.o_sr;
  a.win_left = WIN ? p.win_left : -1;
  a.win_right = WIN ? p.win_right : -1;
  // one CTA per SM (tensor-memory kernels are not co-resident); slot 1 of
  // each CTA takes the items beyond the first grid-full
  const int grid = static_cast<int>(items < num_sms() ? items : num_sms());
  return launch_pdl(kernel, dim3(grid), dim3(Shape::kThreads), smem_bytes, stream, tm_q, tm_k, tm_v,
                    tm_o, a);
}

}  // namespace

cudaError_t launch_attn_bf16(const AttnProblem& p, const CUtensorMap& tm_q,
                             const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const CUtensorMap& tm_o, cudaStream_t stream) {
  // Short query sets use one query tile per work item (at d = 64 two
  // pipelines per CTA, each with one Q buffer so both fit); longer ones pair
  // two query tiles so each K/V tile feeds two MMAs.
  const bool pair = p.n_q > kRows;
  const bool causal = (p.mask_kind & kMaskCausal) != 0;
  // restricted windows run separate instances: the unrestricted loops carry
  // no window code
  if (p.win_left >= 0 || p.win_right >= 0) {
    if (p.n_q != p.n_k) return cudaErrorInvalidValue;
    if (p.d == 64) {
      if (!pair)
        return launch_variant<64, 1, 2, 2, 1, true, 2, false, true>(p, tm_q, tm_k, tm_v, tm_o,
                                                                     stream);
      // one copy of the score load (no unmasked twin): the two window edges
      // put masking in most of a short item's tiles, and the smaller loop
      // measured faster (n = 16384, keys within +-256: 534 -> 588 TFLOP/s)
      return launch_variant<64, 2, 4, 4, 2, true, 1, false, true>(p, tm_q, tm_k, tm_v, tm_o,
                                                                  stream);
    }
    if (p.d == 128) {
      return pair ? launch_variant<128, 2, 2, 2, 1, false, 1, false, true>(p, tm_q, tm_k, tm_v,
                                                                          tm_o, stream)
                  : launch_variant<128, 1, 2, 2, 2, true, 1, false, true>(p, tm_q, tm_k, tm_v,
                                                                         tm_o, stream);
    }
    if (p.d == 256)
      return launch_variant<256, 1, 1, 1, 1, false, 1, false, true>(p, tm_q, tm_k, tm_v, tm_o,
                                                                    stream);
    return cudaErrorInvalidValue;
  }
  if (p.d == 256) {
    // one query tile per item: S (128) + O (256) + P (64) columns of TMEM;
    // one buffer each of Q, K, V (64 KB apiece) and rows stored directly
    return launch_variant<256, 1, 1, 1, 1, false, 1>(p, tm_q, tm_k, tm_v, tm_o, stream);
  }
  if (p.d == 64) {
    if (!pair) return launch_variant<64, 1, 2, 2, 1, true, 2>(p, tm_q, tm_k, tm_v, tm_o, stream);
    if (!causal)
      return launch_variant<64, 2, 4, 4, 2, true, 1, true, false, true>(p, tm_q, tm_k, tm_v, tm_o,
                                                                       stream);
    // causal: the unmasked score-load twin pays once the items are long
    // (measured, TFLOP/s without / with it: n = 1024 601 / 575, 2048 825 /
    // 801, 4096 1060 / 1056, 8192 1146 / 1166, 16384 1195 / 1233)
    return p.n_q >= 8192
               ? launch_variant<64, 2, 4, 4, 2, true, 1, true>(p, tm_q, tm_k, tm_v, tm_o, stream)
               : launch_variant<64, 2, 4, 4, 2, true, 1, false>(p, tm_q, tm_k, tm_v, tm_o, stream);
  }
  if (p.d == 128) {
    if (pair && !causal)
      return launch_variant<128, 2, 2, 2, 1, false, 1, false, false, true>(p, tm_q, tm_k, tm_v,
                                                                          tm_o, stream);
    return pair ? launch_variant<128, 2, 2, 2, 1, false, 1>(p, tm_q, tm_k, tm_v, tm_o, stream)
                : launch_variant<128, 1, 2, 2, 2, true, 1>(p, tm_q, tm_k, tm_v, tm_o, stream);
  }
  return cudaErrorInvalidValue;
}

TSD_DEFINE_ERROR_READER(take_device_error_attn)

}  // namespace tsd
