// attn_bf16.cu -- scaled dot-product attention, softmax(Q K^T * scale) V, on
// the sm_103a tensor cores ("[논문 리뷰]Attention Is All You Need"
// (kimjiil.github.io), section 3.2.1, eq. (1)).
//
// One CTA owns NQT query tiles of 128 rows of one (batch, head) and streams
// that head's key/value tiles (128 keys each) through a shared-memory ring:
//
//   warp 0      TMA producer: Q tiles once, then K_0, K_1, V_0, K_2, V_1, ...
//   warp 1      MMA issuer (one thread): S_t = Q_t K_j^T into tensor memory,
//               O_t += P_t V_j into tensor memory; owns the TMEM allocation
//   warps 4..7  softmax for query tile 0; warps 8..11 for query tile 1:
//               one thread per query row (= one TMEM lane)
//
// The n_q x n_k weight matrix never leaves the chip: S lives in TMEM, P in
// shared memory, one 128x128 tile at a time, with the online (running max and
// running sum) form of the row softmax in fp32. Scores are turned into
// base-2 exponents with the folded factor scale*log2(e); the max is
// subtracted before the exponential, as the pages' reference run does
// ("Attention Is All You Need 해부" (sj-techlog), section "직접 검증").
// Masks: whole key tiles past the causal diagonal or past kv_len are never
// loaded; inside the boundary tile the masked logits become -inf before the
// max and the exponential, so their weight is exactly 0 (section 3.2.3).
// The running max is only raised when it grows by more than 2^8 (exponents
// stay <= 256, exact in the final division), so the O rescale is rare.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103.cuh"

namespace tsd {

namespace {

constexpr int kRows = 128;   // query rows per tile (MMA M) and keys per tile
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, int NQT, int NSLOT>
struct AttnSmem {
  static constexpr int kTileBytes = kRows * D * 2;        // one Q, K or V tile
  static constexpr int kPBytes = kRows * kRows * 2;       // one P tile
  alignas(1024) uint8_t q[NQT][kTileBytes];
  alignas(1024) uint8_t kv[NSLOT][kTileBytes];
  alignas(1024) uint8_t p[NQT][kPBytes];
  uint64_t q_full;
  uint64_t kv_full[NSLOT];
  uint64_t kv_empty[NSLOT];
  uint64_t s_full[NQT];
  uint64_t s_free[NQT];
  uint64_t p_full[NQT];
  uint64_t pv_done[NQT];
  uint64_t mma_drained;
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

template <int D, int NQT>
struct AttnShape {
  static constexpr int kThreads = 128 + 128 * NQT;      // 4 control warps + softmax warpgroups
  static constexpr int kTmemCols = NQT == 2 ? 512 : 256;
  __host__ __device__ static constexpr int kSCol(int t) { return t * kRows; }
  __host__ __device__ static constexpr int kOCol(int t) { return NQT * kRows + t * D; }
};

template <int D, int NQT, int NSLOT>
__global__ void __launch_bounds__(AttnShape<D, NQT>::kThreads, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const AttnArgs args) {
  using Smem = AttnSmem<D, NQT, NSLOT>;
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
  const int nkt = (kv_eff + kRows - 1) / kRows;
  int nt[NQT];
  int nt_all = 0;
#pragma unroll
  for (int t = 0; t < NQT; ++t) {
    const int row0 = q0 + t * kRows;
    int n = nkt;
    if (causal) n = min(n, row0 / kRows + 1);
    if (row0 >= args.n_q) n = 0;
    nt[t] = n;
    nt_all = max(nt_all, n);
  }

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.s_free[t], kRows);
      mbar_init(&sm.p_full[t], kRows);
      mbar_init(&sm.pv_done[t], 1);
    }
    mbar_init(&sm.mma_drained, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nt_all > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&sm.q_full, NQT * Smem::kTileBytes);
      for (int t = 0; t < NQT; ++t)
        for (int a = 0; a < kKAtoms; ++a)
          tma_load_4d(sm.q[t] + a * 16384, &tm_q, &sm.q_full, a * 64, q0 + t * kRows, hh, b);

      int L = 0;
      bool ok = true;
      auto issue = [&](const CUtensorMap* map, int row0) {
        const int slot = L % NSLOT;
        const uint32_t ph = static_cast<uint32_t>(L / NSLOT) & 1u;
        if (!mbar_wait(&sm.kv_empty[slot], ph ^ 1u, abort_flag)) return false;
        mbar_arrive_expect_tx(&sm.kv_full[slot], Smem::kTileBytes);
        for (int a = 0; a < kKAtoms; ++a)
          tma_load_4d(sm.kv[slot] + a * 16384, map, &sm.kv_full[slot], a * 64, row0, hh, b);
        ++L;
        return true;
      };
      ok = issue(&tm_k, 0);
      for (int j = 0; ok && j < nt_all; ++j) {
        if (j + 1 < nt_all) ok = issue(&tm_k, (j + 1) * kRows);
        if (ok) ok = issue(&tm_v, j * kRows);
      }
      if (!ok) {
        // wait (bounded) for this thread's copies still in flight
        volatile uint32_t never = 0;
        mbar_wait(&sm.q_full, 0, &never, 100000000ull);
        for (int i = max(0, L - NSLOT); i < L; ++i)
          mbar_wait(&sm.kv_full[i % NSLOT], static_cast<uint32_t>(i / NSLOT) & 1u, &never,
                    100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nt_all > 0) {
      constexpr uint32_t kIdescS = idesc_bf16(kRows, kRows, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(kRows, D, false, true);
      const uint32_t q_addr = smem_u32(sm.q[0]);
      const uint32_t kv_addr = smem_u32(sm.kv[0]);
      const uint32_t p_addr = smem_u32(sm.p[0]);
      bool ok = mbar_wait(&sm.q_full, 0, abort_flag);

      // S_t = Q_t K^T : K-major A and B, K = head dimension in steps of 16
      auto issue_s = [&](int t, int slot) {
        const uint32_t d_tmem = tmem + Shape::kSCol(t);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint64_t da =
              sdesc_sw128(q_addr + t * Smem::kTileBytes + off, 16, 1024);
          const uint64_t db =
              sdesc_sw128(kv_addr + slot * Smem::kTileBytes + off, 16, 1024);
          mma_bf16_ss(d_tmem, da, db, kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      // O_t (+)= P_t V : P K-major (keys = K), V N-major (head dim = N)
      auto issue_pv = [&](int t, int slot, bool accumulate) {
        const uint32_t d_tmem = tmem + Shape::kOCol(t);
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk) {
          const uint64_t da = sdesc_sw128(
              p_addr + t * Smem::kPBytes + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          const uint64_t db =
              sdesc_sw128(kv_addr + slot * Smem::kTileBytes + kk * 2048, 16384, 1024);
          mma_bf16_ss(d_tmem, da, db, kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
        }
      };

      int L = 0;
      if (ok) ok = mbar_wait(&sm.kv_full[0], 0, abort_flag);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < NQT; ++t)
          if (nt[t] > 0) {
            issue_s(t, 0);
            mma_commit(&sm.s_full[t]);
          }
        mma_commit(&sm.kv_empty[0]);
        L = 1;
      }
      for (int j = 0; ok && j < nt_all; ++j) {
        const bool have_next = j + 1 < nt_all;
        int slot_k = -1;
        if (have_next) {
          slot_k = L % NSLOT;
          ok = mbar_wait(&sm.kv_full[slot_k], static_cast<uint32_t>(L / NSLOT) & 1u, abort_flag);
          ++L;
        }
        const int slot_v = L % NSLOT;
        if (ok)
          ok = mbar_wait(&sm.kv_full[slot_v], static_cast<uint32_t>(L / NSLOT) & 1u, abort_flag);
        ++L;
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; ok && t < NQT; ++t) {
          if (have_next && j + 1 < nt[t]) {
            ok = mbar_wait(&sm.s_free[t], static_cast<uint32_t>(j) & 1u, abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_s(t, slot_k);
            mma_commit(&sm.s_full[t]);
          }
          if (j < nt[t]) {
            ok = mbar_wait(&sm.p_full[t], static_cast<uint32_t>(j) & 1u, abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, slot_v, j > 0);
            mma_commit(&sm.pv_done[t]);
          }
        }
        if (have_next) mma_commit(&sm.kv_empty[slot_k]);
        mma_commit(&sm.kv_empty[slot_v]);
      }
      // every issued MMA has completed before tensor memory is released
      volatile uint32_t never = 0;
      mma_commit(&sm.mma_drained);
      mbar_wait(&sm.mma_drained, 0, &never, 100000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;           // query tile of this warpgroup
    const int quarter = warp & 3;             // TMEM lane quarter of this warp
    const int r = quarter * 32 + static_cast<int>(lane);  // row within the tile
    const int row = q0 + t * kRows + r;       // query index
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t taddr_s = tmem + lane_base + Shape::kSCol(t);
    const uint32_t taddr_o = tmem + lane_base + Shape::kOCol(t);
    const uint32_t p_row = smem_u32(sm.p[t]) + r * 128;
    const float sl2 = args.scale_log2;
    const int lim_row = causal ? min(kv_eff, row + 1) : kv_eff;  // keys [0, lim_row) allowed

    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;
    const int ntt = nt[t];
    for (int j = 0; j < ntt; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.s_full[t], static_cast<uint32_t>(j) & 1u, abort_flag));
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
      tc_fence_before();
      mbar_arrive(&sm.s_free[t]);

      const int bound = lim_row - j * kRows;  // keys c >= bound of this tile are masked
      if (bound < kRows) {
#pragma unroll
        for (int c = 0; c < kRows; ++c)
          if (c >= bound) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kRows; ++c) mx = fmaxf(mx, s[c]);
      const float m_cand = fmaxf(m_used, mx * sl2);
      const bool raise = m_cand > m_used + kRescaleThreshold;
      float alpha = 1.f;
      if (raise) {
        alpha = ex2(m_used - m_cand);  // 0 on the first tile
        m_used = m_cand;
      }
      const float m_eff = m_used == -INFINITY ? 0.f : m_used;

      uint32_t pk[kRows / 2];
      float rowsum = 0.f;
#pragma unroll
      for (int c = 0; c < kRows / 2; ++c) {
        const float p0 = ex2(fmaf(s[2 * c], sl2, -m_eff));
        const float p1 = ex2(fmaf(s[2 * c + 1], sl2, -m_eff));
        rowsum += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }

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

      // P row -> shared memory in the 128-byte-swizzled K-major layout
#pragma unroll
      for (int c16 = 0; c16 < kRows / 8; ++c16) {
        const int atom = c16 >> 3, cc = c16 & 7;
        const uint32_t addr = p_row + atom * 16384 + ((cc ^ (r & 7)) << 4);
        st_shared_v4(addr, pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
      }
      fence_proxy_async_smem();
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

template <int D, int NQT, int NSLOT>
cudaError_t launch_variant(const AttnProblem& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, cudaStream_t stream) {
  using Smem = AttnSmem<D, NQT, NSLOT>;
  using Shape = AttnShape<D, NQT>;
  const size_t smem_bytes = sizeof(Smem) + 1024;  // + alignment slack
  auto kernel = attn_fwd_bf16_kernel<D, NQT, NSLOT>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes));
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
  // Short query sets use one query tile per CTA (two CTAs share an SM);
  // longer ones pair two query tiles so each K/V tile feeds two MMAs.
  const bool pair = p.n_q > kRows;
  if (p.d == 64) {
    return pair ? launch_variant<64, 2, 6>(p, tm_q, tm_k, tm_v, stream)
                : launch_variant<64, 1, 3>(p, tm_q, tm_k, tm_v, stream);
  }
  if (p.d == 128) {
    return pair ? launch_variant<128, 2, 3>(p, tm_q, tm_k, tm_v, stream)
                : launch_variant<128, 1, 2>(p, tm_q, tm_k, tm_v, stream);
  }
  return cudaErrorInvalidValue;
}

TSD_DEFINE_ERROR_READER(take_device_error_attn)

}  // namespace tsd
