// attn_bf16.cu -- scaled dot-product attention, softmax(Q K^T * scale) V, on
// the sm_103a tensor cores ("[논문 리뷰]Attention Is All You Need"
// (kimjiil.github.io), section 3.2.1, eq. (1)).
//
// One CTA owns NQT query tiles of 128 rows of one (batch, head) and streams
// that head's key/value tiles (128 keys each) through two shared-memory rings:
//
//   warp 0      TMA producer: Q tiles once, then K_0, K_1, V_0, K_2, V_1, ...
//   warps 1-3   MMA issuers (one thread each), S_t = Q_t K_j^T and
//               O_t += P_t V_j into tensor memory. The busier product gets one
//               issuer per query tile: at d = 128 (S: 8 MMAs of N=128 per
//               tile, PV: 8 of N=128) warps 1, 2 issue S for tiles 0, 1 and
//               warp 3 issues PV; at d = 64 (S: 4 MMAs, PV: 8 of N=64, the
//               less efficient shape) warp 1 issues S and warps 2, 3 issue PV
//               for tiles 0, 1. Warp 1 owns the TMEM allocation.
//   warps 4..7  softmax for query tile 0; warps 8..11 for query tile 1:
//               one thread per query row (= one TMEM lane)
//
// Several issuing threads keep the tensor pipe fed: each thread's barrier
// waits and commits (tcgen05.commit tracks only the issuing thread's MMAs)
// overlap the other threads' MMA issue.
//
// The n_q x n_k weight matrix never leaves the chip: S lives in TMEM, P (bf16)
// in TMEM as the A operand of the PV MMA, one 128x128 tile at a time, with the
// online (running max and running sum) form of the row softmax in fp32.
// Scores become base-2 exponents with the folded factor scale*log2(e); the max
// is subtracted before the exponential, as the pages' reference run does
// ("Attention Is All You Need 해부" (sj-techlog), section "직접 검증").
// Masks: key tiles past the causal diagonal or past kv_len are never loaded;
// inside the boundary tile the masked logits become -inf before the max and
// the exponential, so their weight is exactly 0 (section 3.2.3).
// The running max is only raised when it grows by more than 2^8 (exponents
// stay <= 256, exact in the final division), so the O rescale is rare.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kRows = 128;                 // query rows per tile (MMA M) and keys per tile
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, int NQT>
struct AttnShape {
  static constexpr int kThreads = 128 + 128 * NQT;  // 4 control warps + softmax warpgroups
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
  // register split of the paired variants: control warps give up registers
  // to the softmax warpgroups (sum <= threads x registers at launch)
  static constexpr uint32_t kLaunchRegs = 65536 / kThreads / 8 * 8;
  static constexpr uint32_t kCtrlRegs = D == 64 ? 72 : 88;
  static constexpr uint32_t kSoftmaxRegs =
      (kLaunchRegs * kThreads - kCtrlRegs * 128) / (128 * NQT) / 8 * 8;
  // one issuer per query tile for S (else for PV), see the role table above
  static constexpr bool kSplitS = (D == 128);
  static constexpr int kSIssuers = kSplitS ? NQT : 1;
  static constexpr int kPVIssuers = kSplitS ? 1 : NQT;
  static_assert(kColsUsed <= 512, "tensor memory budget");
  // setmaxnreg.inc waits for registers released by .dec: the split must fit
  // in what the CTA was launched with, or the increase would never complete
  static_assert(kCtrlRegs * 128 + kSoftmaxRegs * 128 * NQT <= kLaunchRegs * kThreads,
                "register split exceeds the launch allocation");
};

template <int D, int NQT, int NK, int NV>
struct AttnSmem {
  static constexpr int kTileBytes = kRows * D * 2;  // one Q, K or V tile
  alignas(1024) uint8_t q[NQT][kTileBytes];
  alignas(1024) uint8_t k[NK][kTileBytes];
  alignas(1024) uint8_t v[NV][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[NK], k_empty[NK];
  uint64_t v_full[NV], v_empty[NV];
  uint64_t s_full[NQT];
  uint64_t s_free[NQT];
  uint64_t p_full[NQT];
  uint64_t pv_done[NQT];
  uint64_t s_drained[NQT], pv_drained[NQT];
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct AttnArgs {
  int n_q, n_k, n_qblocks;
  int mask_kind;
  const int32_t* kv_lens;
  float scale_log2;
  uint16_t* out;
  int64_t o_sb, o_sh, o_sr;
};

constexpr unsigned long long kDrainLimitNs = 100ull * 1000ull * 1000ull;  // 0.1 s

template <int D, int NQT, int NK, int NV>
__global__ void __launch_bounds__(AttnShape<D, NQT>::kThreads, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const AttnArgs args) {
  using Smem = AttnSmem<D, NQT, NK, NV>;
  using Shape = AttnShape<D, NQT>;
  constexpr int kKAtoms = D / 64;  // 128-byte swizzle atoms along the head dimension

  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int warp = warp_id();
  const uint32_t lane = lane_id();
  const int b = blockIdx.z;
  const int hh = blockIdx.y;
  const bool causal = (args.mask_kind & kMaskCausal) != 0;
  // longest causal blocks first (they have the most key tiles)
  const int qblk = causal ? (args.n_qblocks - 1 - static_cast<int>(blockIdx.x))
                          : static_cast<int>(blockIdx.x);
  const int q0 = qblk * NQT * kRows;

  int kv_eff = args.n_k;
  if (args.mask_kind & kMaskKeyPadding) {
    int len = args.kv_lens[b];
    kv_eff = len < 0 ? 0 : (len > args.n_k ? args.n_k : len);
  }
  // key tiles each query tile visits (kept in scalars: a runtime-indexed
  // array would live in local memory)
  const int nkt = (kv_eff + kRows - 1) / kRows;
  auto tiles_for = [&](int t) {
    const int row0 = q0 + t * kRows;
    int n = nkt;
    if (causal) n = min(n, row0 / kRows + 1);
    if (row0 >= args.n_q) n = 0;
    return n;
  };
  const int nt0 = tiles_for(0);
  const int nt1 = NQT > 1 ? tiles_for(1) : 0;
  auto nt = [&](int t) { return t == 0 ? nt0 : nt1; };
  const int nt_all = max(nt0, nt1);

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], Shape::kSIssuers);  // one release per S-issuing warp
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
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(&sm.s_drained[t], 1);
      mbar_init(&sm.pv_drained[t], 1);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, Shape::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile uint32_t* abort_flag = &sm.abort_flag;

  // Descriptors are built once; each MMA only advances the start-address
  // field by a compile-time offset (sdesc_advance keeps the sum inside it).
  constexpr uint32_t kTileStep = Smem::kTileBytes >> 4;
  constexpr uint32_t kIdescS = idesc_bf16(kRows, kRows, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16(kRows, D, false, true);

  if (warp < 4) {
    if constexpr (NQT == 2) regs_decrease<Shape::kCtrlRegs>();
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      if (lane == 0 && nt_all > 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(&sm.q_full, NQT * Smem::kTileBytes);
        for (int t = 0; t < NQT; ++t)
          for (int a = 0; a < kKAtoms; ++a)
            tma_load_4d(sm.q[t] + a * 16384, &tm_q, &sm.q_full, a * 64, q0 + t * kRows, hh, b);

        int kn = 0, vn = 0;  // tiles issued into each ring
        auto load_k = [&]() {
          const int slot = kn % NK;
          if (!mbar_wait(&sm.k_empty[slot], (static_cast<uint32_t>(kn / NK) & 1u) ^ 1u, abort_flag))
            return false;
          mbar_arrive_expect_tx(&sm.k_full[slot], Smem::kTileBytes);
          for (int a = 0; a < kKAtoms; ++a)
            tma_load_4d(sm.k[slot] + a * 16384, &tm_k, &sm.k_full[slot], a * 64, kn * kRows, hh, b);
          ++kn;
          return true;
        };
        auto load_v = [&]() {
          const int slot = vn % NV;
          if (!mbar_wait(&sm.v_empty[slot], (static_cast<uint32_t>(vn / NV) & 1u) ^ 1u, abort_flag))
            return false;
          mbar_arrive_expect_tx(&sm.v_full[slot], Smem::kTileBytes);
          for (int a = 0; a < kKAtoms; ++a)
            tma_load_4d(sm.v[slot] + a * 16384, &tm_v, &sm.v_full[slot], a * 64, vn * kRows, hh, b);
          ++vn;
          return true;
        };
        // keys run one tile ahead of values, the order the MMAs consume them
        bool ok = load_k();
        for (int j = 0; ok && j < nt_all; ++j) {
          if (j + 1 < nt_all) ok = load_k();
          if (ok) ok = load_v();
        }
        if (!ok) {
          // wait (bounded) for this thread's copies still in flight
          volatile uint32_t never = 0;
          mbar_wait(&sm.q_full, 0, &never, kDrainLimitNs);
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
      if (lane == 0 && nt_all > 0) {
        const uint64_t dq0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);  // K-major Q
        const uint64_t dk0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);  // K-major K
        bool ok = mbar_wait(&sm.q_full, 0, abort_flag);
        for (int j = 0; ok && j < nt_all; ++j) {
          const int slot = j % NK;
          // the slot holds K_j before this warp releases it, so a release for
          // tiles this issuer skips never counts toward an older use
          ok = mbar_wait(&sm.k_full[slot], static_cast<uint32_t>(j / NK) & 1u, abort_flag);
          if (!ok) break;
          const uint64_t bk = sdesc_advance(dk0, static_cast<uint32_t>(slot) * kTileStep);
          bool issued = false;
          for (int t = t_lo; ok && t < t_hi; ++t) {
            if (j >= nt(t)) continue;
            if (j > 0) {
              // S_t(j-1) has been read (or, when P overwrites S, consumed by PV)
              ok = Shape::kPAliasS
                       ? mbar_wait(&sm.pv_done[t], static_cast<uint32_t>(j - 1) & 1u, abort_flag)
                       : mbar_wait(&sm.s_free[t], static_cast<uint32_t>(j - 1) & 1u, abort_flag);
              if (!ok) break;
            }
            tc_fence_after();
            // S_t = Q_t K^T : K-major A and B, K = head dimension in steps of 16
            const uint32_t d_tmem = tmem + Shape::s_col(t);
            const uint64_t a = sdesc_advance(dq0, static_cast<uint32_t>(t) * kTileStep);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = static_cast<uint32_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
              mma_bf16_ss(d_tmem, sdesc_advance(a, off), sdesc_advance(bk, off), kIdescS,
                          kk > 0 ? 1u : 0u);
            }
            mma_commit(&sm.s_full[t]);
            issued = true;
          }
          if (!ok) break;
          if (issued) mma_commit(&sm.k_empty[slot]);
          else mbar_arrive(&sm.k_empty[slot]);
        }
        // every issued MMA has completed before tensor memory is released
        volatile uint32_t never = 0;
        mma_commit(&sm.s_drained[t_lo]);
        mbar_wait(&sm.s_drained[t_lo], 0, &never, kDrainLimitNs);
      }
    } else if (warp - 1 - Shape::kSIssuers < Shape::kPVIssuers) {
      // ---------------------------------------------------------- PV issuer(s)
      const int w = warp - 1 - Shape::kSIssuers;
      const int t_lo = Shape::kSplitS ? 0 : w;
      const int t_hi = Shape::kSplitS ? NQT : w + 1;
      if (lane == 0 && nt_all > 0) {
        const uint64_t dv0 = sdesc_sw128(smem_u32(sm.v[0]), 16384, 1024);  // N-major V
        bool ok = true;
        for (int j = 0; ok && j < nt_all; ++j) {
          const int slot = j % NV;
          // as for K: the slot holds V_j before any release by this warp
          ok = mbar_wait(&sm.v_full[slot], static_cast<uint32_t>(j / NV) & 1u, abort_flag);
          if (!ok) break;
          const uint64_t bv = sdesc_advance(dv0, static_cast<uint32_t>(slot) * kTileStep);
          bool issued = false;
          for (int t = t_lo; ok && t < t_hi; ++t) {
            if (j >= nt(t)) continue;
            ok = mbar_wait(&sm.p_full[t], static_cast<uint32_t>(j) & 1u, abort_flag);
            if (!ok) break;
            tc_fence_after();
            // O_t (+)= P_t V : P from TMEM (keys = K), V N-major, 16 keys per MMA
            const uint32_t d_tmem = tmem + Shape::o_col(t);
            const uint32_t p_tmem = tmem + Shape::p_col(t);
#pragma unroll
            for (int kk = 0; kk < kRows / 16; ++kk)
              mma_bf16_ts(d_tmem, p_tmem + kk * 8, sdesc_advance(bv, kk * (2048 >> 4)), kIdescPV,
                          (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&sm.pv_done[t]);
            issued = true;
          }
          if (!ok) break;
          if (issued) mma_commit(&sm.v_empty[slot]);
          else mbar_arrive(&sm.v_empty[slot]);
        }
        volatile uint32_t never = 0;
        mma_commit(&sm.pv_drained[t_lo]);
        mbar_wait(&sm.pv_drained[t_lo], 0, &never, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    if constexpr (NQT == 2) regs_increase<Shape::kSoftmaxRegs>();
    const int t = (warp - 4) >> 2;           // query tile of this warpgroup
    const int quarter = warp & 3;             // TMEM lane quarter of this warp
    const int r = quarter * 32 + static_cast<int>(lane);  // row within the tile
    const int row = q0 + t * kRows + r;       // query index
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t taddr_s = tmem + lane_base + Shape::s_col(t);
    const uint32_t taddr_o = tmem + lane_base + Shape::o_col(t);
    const uint32_t taddr_p = tmem + lane_base + Shape::p_col(t);
    const float sl2 = args.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    const int lim_row = causal ? min(kv_eff, row + 1) : kv_eff;  // keys [0, lim_row) allowed

    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;
    const int ntt = nt(t);
    for (int j = 0; j < ntt; ++j) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&sm.s_full[t], static_cast<uint32_t>(j) & 1u, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float s[kRows];
#pragma unroll
      for (int c = 0; c < kRows / 32; ++c) {
        uint32_t raw[32];
        tmem_ld32(taddr_s + c * 32, raw);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(raw[i]);
      }
      tmem_wait_ld();

      const int bound = lim_row - j * kRows;  // keys c >= bound of this tile are masked
      if (bound < kRows) {
#pragma unroll
        for (int c = 0; c < kRows; ++c)
          if (c >= bound) s[c] = -INFINITY;
      }
      // row max: 8 independent chains of 3-input max
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
      for (int c = 16; c < kRows; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], s[c + i], s[c + 8 + i]);
      const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                             fmaxf(mx8[6], mx8[7]));
      // S_t is free for S_t(j+1) only now, after the row max: the tensor pipe
      // executes MMAs in issue order, and PV_t(j-1), issued when P_t(j-1) was
      // stored, should run before S_t(j+1) -- this tile's next P store waits
      // for it, while the next S is not needed until this iteration ends.
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
      for (int c = 0; c < kRows / 2; ++c) {
        float x0, x1;
        f2_unpack(ffma2(f2_pack(s[2 * c], s[2 * c + 1]), sl2x2, negm2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        pk[c] = pack_bf16x2(p0, p1);
        acc2[c & 3] = fadd2(acc2[c & 3], f2_pack(p0, p1));
      }
      float r0, r1;
      f2_unpack(fadd2(fadd2(acc2[0], acc2[1]), fadd2(acc2[2], acc2[3])), r0, r1);
      const float rowsum = r0 + r1;

      if (j > 0) {
        // PV of the previous tile has finished: O is stable, P is free
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&sm.pv_done[t], static_cast<uint32_t>(j - 1) & 1u, abort_flag));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(taddr_o + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(taddr_o + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      l = l * alpha + rowsum;

      // P row -> TMEM lane r, two bf16 per 32-bit column (the MMA's A layout)
      {
        uint32_t half[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) half[i] = pk[i];
        tmem_st32(taddr_p, half);
#pragma unroll
        for (int i = 0; i < 32; ++i) half[i] = pk[32 + i];
        tmem_st32(taddr_p + 32, half);
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(&sm.p_full[t]);
    }

    // ---------------------------------------------------------- epilogue
    if (ok && ntt > 0) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&sm.pv_done[t], static_cast<uint32_t>(ntt - 1) & 1u, abort_flag));
      tc_fence_after();
    }
    if (ok) {
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      uint16_t* dst = args.out + static_cast<int64_t>(b) * args.o_sb +
                      static_cast<int64_t>(hh) * args.o_sh + static_cast<int64_t>(row) * args.o_sr;
      const bool store = row < args.n_q;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (ntt > 0) {
          tmem_ld32(taddr_o + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        if (store) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            st_global_v4(dst + c * 32 + v4 * 8, w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2],
                         w[4 * v4 + 3]);
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, Shape::kTmemCols);
}

template <int D, int NQT, int NK, int NV>
cudaError_t launch_variant(const AttnProblem& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, cudaStream_t stream) {
  using Smem = AttnSmem<D, NQT, NK, NV>;
  using Shape = AttnShape<D, NQT>;
  const size_t smem_bytes = sizeof(Smem) + 1024;  // + alignment slack
  auto kernel = attn_fwd_bf16_kernel<D, NQT, NK, NV>;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem_once(kernel, static_cast<int>(smem_bytes), &configured);
  if (e != cudaSuccess) return e;
  AttnArgs a;
  a.n_q = p.n_q;
  a.n_k = p.n_k;
  a.n_qblocks = (p.n_q + NQT * kRows - 1) / (NQT * kRows);
  a.mask_kind = p.mask_kind;
  a.kv_lens = p.kv_lens;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.out = p.out;
  a.o_sb = p.o_sb;
  a.o_sh = p.o_sh;
  a.o_sr = p.o_sr;
  dim3 grid(a.n_qblocks, p.h, p.B);
  kernel<<<grid, Shape::kThreads, smem_bytes, stream>>>(tm_q, tm_k, tm_v, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bf16(const AttnProblem& p, const CUtensorMap& tm_q,
                             const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             cudaStream_t stream) {
  // Short query sets use one query tile per CTA; longer ones pair two query
  // tiles so each K/V tile feeds two MMAs.
  const bool pair = p.n_q > kRows;
  if (p.d == 64) {
    return pair ? launch_variant<64, 2, 4, 4>(p, tm_q, tm_k, tm_v, stream)
                : launch_variant<64, 1, 2, 2>(p, tm_q, tm_k, tm_v, stream);
  }
  if (p.d == 128) {
    return pair ? launch_variant<128, 2, 2, 2>(p, tm_q, tm_k, tm_v, stream)
                : launch_variant<128, 1, 2, 2>(p, tm_q, tm_k, tm_v, stream);
  }
  return cudaErrorInvalidValue;
}

TSD_DEFINE_ERROR_READER(take_device_error_attn)

}  // namespace tsd
