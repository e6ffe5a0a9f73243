// api.cu -- the C ABI (include/tsd_attention.h): argument validation, TMA
// descriptor encoding, and the launch sequence of multi-head attention.
// Every host-detectable error returns before anything is launched.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "host_stage.h"
#include "kernels.h"
#include "tsd_attention.h"

namespace {

thread_local int g_last_cuda_error = 0;

attn_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return ATTN_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library does not link libcuda directly.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder(cudaError_t* err) {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static cudaError_t status = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                              cudaEnableDefault, &q);
    if (status == cudaSuccess && (q != cudaDriverEntryPointSuccess || p == nullptr))
      status = cudaErrorNotSupported;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  *err = status;
  return fn;
}

// Encoded maps are memoised: an encoding costs microseconds of host time,
// about as much as a short attention kernel runs. A map holds nothing but
// its inputs (address, sizes, strides, box), so the key is all of them and
// a hit returns exactly what a fresh encoding would.
struct MapKey {
  const void* base;
  int rank;
  uint64_t dims[4];
  int64_t strides[3];
  uint32_t box[4];
};

constexpr int kMapCacheSlots = 256;  // direct-mapped
struct MapCacheEntry {
  bool used;
  MapKey key;
  CUtensorMap map;
};
std::mutex g_map_cache_mutex;
MapCacheEntry g_map_cache[kMapCacheSlots];

uint32_t map_key_hash(const MapKey& k) {
  const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
  uint32_t h = 2166136261u;  // FNV-1a
  for (size_t i = 0; i < sizeof(MapKey); ++i) h = (h ^ p[i]) * 16777619u;
  return h;
}

cudaError_t encode_bf16_map_uncached(CUtensorMap* map, const void* base, int rank,
                                     const uint64_t* dims, const int64_t* strides_elems,
                                     const uint32_t* box);

// bf16 tensor map, rank 2..4, dims innermost first, strides in elements
// (dims 1..rank-1), 128-byte swizzle, zero fill out of bounds.
cudaError_t encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const int64_t* strides_elems, const uint32_t* box) {
  MapKey key;
  std::memset(&key, 0, sizeof(key));  // padding bytes take part in hash and compare
  key.base = base;
  key.rank = rank;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) key.strides[i] = strides_elems[i];
  MapCacheEntry& slot = g_map_cache[map_key_hash(key) % kMapCacheSlots];
  {
    std::lock_guard<std::mutex> lock(g_map_cache_mutex);
    if (slot.used && std::memcmp(&slot.key, &key, sizeof(key)) == 0) {
      *map = slot.map;
      return cudaSuccess;
    }
  }
  cudaError_t e = encode_bf16_map_uncached(map, base, rank, dims, strides_elems, box);
  if (e == cudaSuccess) {
    std::lock_guard<std::mutex> lock(g_map_cache_mutex);
    slot.used = true;
    slot.key = key;
    slot.map = *map;
  }
  return e;
}

cudaError_t encode_bf16_map_uncached(CUtensorMap* map, const void* base, int rank,
                                     const uint64_t* dims, const int64_t* strides_elems,
                                     const uint32_t* box) {
  cudaError_t err;
  auto enc = tensor_map_encoder(&err);
  if (err != cudaSuccess) return err;
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gstride[i] = static_cast<cuuint64_t>(strides_elems[i]) * 2u;
  auto encode = [&] {
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
               const_cast<void*>(base), gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  CUresult r = encode();
  if (r == CUDA_ERROR_INVALID_CONTEXT) {
    // A host thread whose runtime calls so far needed no device has no
    // current context, and the encoder is a driver call: a no-op runtime
    // call binds the current device's primary context to the thread.
    (void)cudaFree(nullptr);
    r = encode();
  }
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Q/K/V as a 4-D (d, rows, heads, batch) map with 64 x 128 boxes.
cudaError_t encode_head_map(CUtensorMap* map, const void* base, int d, int rows, int h, int B,
                            int64_t sr, int64_t sh, int64_t sb) {
  const uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(rows < 1 ? 1 : rows),
                            static_cast<uint64_t>(h), static_cast<uint64_t>(B)};
  const int64_t strides[3] = {sr, sh, sb};
  const uint32_t box[4] = {64, 128, 1, 1};
  return encode_bf16_map(map, base, 4, dims, strides, box);
}

bool valid_scale(float s) { return std::isfinite(s) && s >= 0.f; }

float resolve_scale(float s, int d_k) {
  return s == 0.f ? static_cast<float>(1.0 / std::sqrt(static_cast<double>(d_k))) : s;
}

// Shared checks of attn_forward / attn_forward_strided / mha_forward.
attn_status check_common(int B, int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                         const int32_t* kv_lens, float scale) {
  if (B < 0 || h < 0 || n_q < 0 || n_k < 0 || d_k <= 0 || d_v <= 0) return ATTN_ERR_INVALID;
  if (h > 65535 || B > 65535) return ATTN_ERR_INVALID;  // grid y / z limits
  if (mask_kind & ~(ATTN_MASK_CAUSAL | ATTN_MASK_KEY_PADDING)) return ATTN_ERR_INVALID;
  if ((mask_kind & ATTN_MASK_CAUSAL) && n_q != n_k) return ATTN_ERR_INVALID;
  if ((mask_kind & ATTN_MASK_KEY_PADDING) &&
      (kv_lens == nullptr || (reinterpret_cast<uintptr_t>(kv_lens) & 3u)))
    return ATTN_ERR_INVALID;
  if (!valid_scale(scale)) return ATTN_ERR_INVALID;
  return ATTN_OK;
}

// Head sizes of the bf16 attention kernels: 64 and 128, and Table 3's other
// rows ("[논문 리뷰]Attention Is All You Need", section 6.2, Table 3 (A)): 16
// and 32 run through the 64-column kernels (the tensor maps zero-fill the
// columns past d on load and clip them on store), 256 through its own.
attn_status check_bf16_head_dims(int d_k, int d_v) {
  if (d_k != d_v) return ATTN_ERR_UNSUPPORTED;
  if (d_k != 16 && d_k != 32 && d_k != 64 && d_k != 128 && d_k != 256) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

attn_status run_attn_bf16(const void* q, int64_t q_sb, int64_t q_sh, int64_t q_sr, const void* k,
                          int64_t k_sb, int64_t k_sh, int64_t k_sr, const void* v, int64_t v_sb,
                          int64_t v_sh, int64_t v_sr, void* out, int64_t o_sb, int64_t o_sh,
                          int64_t o_sr, int B, int h, int n_q, int n_k, int d, int mask_kind,
                          const int32_t* kv_lens, float scale, cudaStream_t stream,
                          int win_left = -1, int win_right = -1) {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  cudaError_t e = encode_head_map(&tm_q, q, d, n_q, h, B, q_sr, q_sh, q_sb);
  if (e == cudaSuccess) e = encode_head_map(&tm_k, k, d, n_k, h, B, k_sr, k_sh, k_sb);
  if (e == cudaSuccess) e = encode_head_map(&tm_v, v, d, n_k, h, B, v_sr, v_sh, v_sb);
  if (e == cudaSuccess) e = encode_head_map(&tm_o, out, d, n_q, h, B, o_sr, o_sh, o_sb);
  if (e != cudaSuccess) return cuda_fail(e);
  tsd::AttnProblem p;
  p.B = B;
  p.h = h;
  p.n_q = n_q;
  p.n_k = n_k;
  p.d = d < 64 ? 64 : d;  // 16 and 32 run through the 64-column kernels
  p.mask_kind = mask_kind;
  p.kv_lens = kv_lens;
  p.scale = resolve_scale(scale, d);
  p.out = static_cast<uint16_t*>(out);
  p.o_sb = o_sb;
  p.o_sh = o_sh;
  p.o_sr = o_sr;
  p.win_left = win_left;
  p.win_right = win_right;
  e = tsd::launch_attn_bf16(p, tm_q, tm_k, tm_v, tm_o, stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

size_t align256(size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); }

struct MhaLayout {
  size_t q_off, k_off, v_off, o_off, total;
};

bool mha_layout(int B, int n_q, int n_k, int h, int d_k, int d_v, MhaLayout* L) {
  if (B < 0 || n_q < 0 || n_k < 0 || h <= 0 || d_k <= 0 || d_v <= 0) return false;
  const size_t q = static_cast<size_t>(B) * n_q * h * d_k * 2;
  const size_t k = static_cast<size_t>(B) * n_k * h * d_k * 2;
  const size_t v = static_cast<size_t>(B) * n_k * h * d_v * 2;
  const size_t o = static_cast<size_t>(B) * n_q * h * d_v * 2;
  L->q_off = 0;
  L->k_off = align256(q);
  L->v_off = L->k_off + align256(k);
  L->o_off = L->v_off + align256(v);
  L->total = L->o_off + align256(o);
  return true;
}

// One GEMM group: C[M, N] = A[M, K] B[K, N], all row-major bf16.
cudaError_t make_gemm_group(tsd::GemmGroup* g, const void* a, const void* b, void* c, int M, int N,
                            int K) {
  const uint64_t adims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  const int64_t astr[1] = {K};
  const uint32_t abox[2] = {64, 128};
  cudaError_t e = encode_bf16_map(&g->tm_a, a, 2, adims, astr, abox);
  if (e != cudaSuccess) return e;
  const uint64_t bdims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K)};
  const int64_t bstr[1] = {N};
  // 64 N columns x the K rows of one pipeline stage
  const uint32_t bbox[2] = {64, static_cast<uint32_t>(tsd::kGemmBK)};
  e = encode_bf16_map(&g->tm_b, b, 2, bdims, bstr, bbox);
  if (e != cudaSuccess) return e;
  const uint64_t cdims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
  const int64_t cstr[1] = {N};
  const uint32_t cbox[2] = {64, 128};  // 64 columns x 128 rows, written by TMA stores
  e = encode_bf16_map(&g->tm_c, c, 2, cdims, cstr, cbox);
  if (e != cudaSuccess) return e;
  g->c = static_cast<uint16_t*>(c);
  g->ldc = N;
  g->M = M;
  g->N = N;
  g->tiles_m = (M + 127) / 128;
  g->tiles_n = (N + 127) / 128;
  return cudaSuccess;
}

void finish_gemm_problem(tsd::GemmProblem* p) {
  int t = 0;
  for (int i = 0; i < p->num_groups; ++i) {
    p->g[i].tile_begin = t;
    t += p->g[i].tiles_m * p->g[i].tiles_n;
  }
  p->total_tiles = t;
}


// Checks shared by the projection entry points.
attn_status check_projection(int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v) {
  if (B < 0 || n_q < 0 || n_k < 0 || h <= 0 || d_k <= 0 || d_v <= 0) return ATTN_ERR_INVALID;
  if (d_model < 8 || (d_model % 8) != 0) return ATTN_ERR_INVALID;
  if ((int64_t(h) * d_k) % 8 != 0 || (int64_t(h) * d_v) % 8 != 0) return ATTN_ERR_INVALID;
  if (int64_t(B) * n_q > INT32_MAX || int64_t(B) * n_k > INT32_MAX) return ATTN_ERR_INVALID;
  if (int64_t(h) * d_k > INT32_MAX || int64_t(h) * d_v > INT32_MAX) return ATTN_ERR_INVALID;
  return ATTN_OK;
}

attn_status launch_qkv(const void* x_q, const void* x_kv, const void* w_q, const void* w_k,
                       const void* w_v, void* Q, void* K, void* V, int B, int n_q, int n_k,
                       int d_model, int h, int d_k, int d_v, cudaStream_t stream) {
  const int Mq = B * n_q, Mk = B * n_k;
  tsd::GemmProblem g;
  std::memset(&g, 0, sizeof(g));
  g.K = d_model;
  g.num_groups = 0;
  cudaError_t e = cudaSuccess;
  if (Mq > 0) e = make_gemm_group(&g.g[g.num_groups++], x_q, w_q, Q, Mq, h * d_k, d_model);
  if (e == cudaSuccess && Mk > 0) {
    e = make_gemm_group(&g.g[g.num_groups++], x_kv, w_k, K, Mk, h * d_k, d_model);
    if (e == cudaSuccess)
      e = make_gemm_group(&g.g[g.num_groups++], x_kv, w_v, V, Mk, h * d_v, d_model);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  if (g.num_groups == 0) return ATTN_OK;
  finish_gemm_problem(&g);
  e = tsd::launch_gemm_bf16(g, stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// Shapes the fused short-sequence kernel takes (projections and attention
// in one launch); others run the projection GEMM and the attention kernel.
bool fused_eligible(int n_q, int n_k, int d_model, int h, int d_k, int d_v) {
  return d_k == 64 && d_v == 64 && n_q >= 1 && n_q <= 128 && n_k >= 1 && n_k <= 128 &&
         h % 2 == 0 && d_model >= 64 && d_model % 64 == 0;
}

// The fused kernel can apply W_O as well: h/2 <= 8 head pairs (one cluster
// per batch entry), d_model / (h/2) output columns per CTA = 64 or 128, and
// such a cluster fits on the device.
bool fused_out_eligible(bool self, int d_model, int h) {
  const int C = h / 2;
  if (C < 1 || C > 8 || d_model % C != 0) return false;
  const int n_slice = d_model / C;
  if (n_slice != 64 && n_slice != 128) return false;
  return tsd::mha_fused_out_clusters(h, self) > 0;
}

// Cross-attention (x_kv is not x_q) whose source is one key tile and a tail
// of up to 64 rows: projections and attention in one launch (mha_cross.cu).
bool cross_eligible(bool self, int n_q, int n_k, int d_model, int h, int d_k, int d_v) {
  return !self && d_k == 64 && d_v == 64 && n_q >= 1 && n_q <= 128 && n_k > 128 &&
         n_k <= 192 && h % 2 == 0 && d_model >= 64 && d_model % 64 == 0;
}
// ... and W_O in the same launch (the clusters of the fused kernel's OUT rule).
bool cross_out_eligible(int d_model, int h) {
  const int C = h / 2;
  if (C < 1 || C > 8 || d_model % C != 0) return false;
  const int n_slice = d_model / C;
  if (n_slice != 64 && n_slice != 128) return false;
  return tsd::mha_cross_out_clusters(h) > 0;
}

// Q/K/V projections + attention of every (batch, head pair) -> the merged
// heads, [B, n_q, h*64], in `concat`; with `w_o` also out = concat W_O in
// the same launch (`concat` is then scratch).
attn_status launch_fused_core(const void* x_q, const void* x_kv, const void* w_q, const void* w_k,
                              const void* w_v, void* concat, int B, int n_q, int n_k, int d_model,
                              int h, int mask_kind, const int32_t* kv_lens, float scale,
                              cudaStream_t stream, const void* w_o = nullptr,
                              void* out = nullptr) {
  tsd::MhaFusedProblem p;
  std::memset(&p, 0, sizeof(p));
  p.self = (x_q == x_kv) && (n_q == n_k);
  p.out = w_o != nullptr;
  const uint32_t xbox[3] = {64, 128, 1};
  const uint64_t xq_dims[3] = {static_cast<uint64_t>(d_model), static_cast<uint64_t>(n_q),
                               static_cast<uint64_t>(B)};
  const int64_t xq_str[2] = {d_model, int64_t(n_q) * d_model};
  cudaError_t e = encode_bf16_map(&p.tm_xq, x_q, 3, xq_dims, xq_str, xbox);
  if (e == cudaSuccess && !p.self) {
    const uint64_t xkv_dims[3] = {static_cast<uint64_t>(d_model), static_cast<uint64_t>(n_k),
                                  static_cast<uint64_t>(B)};
    const int64_t xkv_str[2] = {d_model, int64_t(n_k) * d_model};
    e = encode_bf16_map(&p.tm_xkv, x_kv, 3, xkv_dims, xkv_str, xbox);
    const uint32_t tbox[3] = {64, 64, 1};  // the source's rows past 128, 64 at a time
    if (e == cudaSuccess && n_k > 128)
      e = encode_bf16_map(&p.tm_xkv_tail, x_kv, 3, xkv_dims, xkv_str, tbox);
  } else {
    p.tm_xkv = p.tm_xq;
  }
  const uint64_t w_dims[2] = {static_cast<uint64_t>(h) * 64, static_cast<uint64_t>(d_model)};
  const int64_t w_str[1] = {int64_t(h) * 64};
  const uint32_t wbox[2] = {64, 64};
  if (e == cudaSuccess) e = encode_bf16_map(&p.tm_wq, w_q, 2, w_dims, w_str, wbox);
  if (e == cudaSuccess) e = encode_bf16_map(&p.tm_wk, w_k, 2, w_dims, w_str, wbox);
  if (e == cudaSuccess) e = encode_bf16_map(&p.tm_wv, w_v, 2, w_dims, w_str, wbox);
  const uint64_t o_dims[3] = {static_cast<uint64_t>(h) * 64, static_cast<uint64_t>(n_q),
                              static_cast<uint64_t>(B)};
  const int64_t o_str[2] = {int64_t(h) * 64, int64_t(n_q) * h * 64};
  if (e == cudaSuccess) e = encode_bf16_map(&p.tm_o, concat, 3, o_dims, o_str, xbox);
  if (e == cudaSuccess && p.out) {
    const uint64_t wo_dims[2] = {static_cast<uint64_t>(d_model), static_cast<uint64_t>(h) * 64};
    const int64_t wo_str[1] = {d_model};
    e = encode_bf16_map(&p.tm_wo, w_o, 2, wo_dims, wo_str, wbox);
    if (e == cudaSuccess) e = encode_bf16_map(&p.tm_out, out, 3, xq_dims, xq_str, xbox);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  p.B = B;
  p.h = h;
  p.n_q = n_q;
  p.n_k = n_k;
  p.d_model = d_model;
  p.mask_kind = mask_kind;
  p.kv_lens = kv_lens;
  p.scale = resolve_scale(scale, 64);
  e = (!p.self && n_k > 128) ? tsd::launch_mha_cross(p, stream) : tsd::launch_mha_fused(p, stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// head_i = Attention(X_q W_Q,i, X_kv W_K,i, X_kv W_V,i), written merged,
// [B, n_q, h*d_v]. Short sequences: one fused launch; else the grouped
// projection GEMM into Q, K, V (column block i = head i) and the attention
// kernel reading them through strides.
attn_status concat_heads(const void* x_q, const void* x_kv, const void* w_q, const void* w_k,
                         const void* w_v, void* concat, void* Q, void* K, void* V, int B, int n_q,
                         int n_k, int d_model, int h, int d_k, int d_v, int mask_kind,
                         const int32_t* kv_lens, float scale, cudaStream_t stream) {
  if (fused_eligible(n_q, n_k, d_model, h, d_k, d_v) ||
      cross_eligible(x_q == x_kv && n_q == n_k, n_q, n_k, d_model, h, d_k, d_v))
    return launch_fused_core(x_q, x_kv, w_q, w_k, w_v, concat, B, n_q, n_k, d_model, h,
                             mask_kind, kv_lens, scale, stream);
  const int hdk = h * d_k, hdv = h * d_v;
  attn_status s =
      launch_qkv(x_q, x_kv, w_q, w_k, w_v, Q, K, V, B, n_q, n_k, d_model, h, d_k, d_v, stream);
  if (s != ATTN_OK) return s;
  return run_attn_bf16(Q, int64_t(n_q) * hdk, d_k, hdk, K, int64_t(n_k) * hdk, d_k, hdk, V,
                       int64_t(n_k) * hdv, d_v, hdv, concat, int64_t(n_q) * hdv, d_v, hdv, B, h,
                       n_q, n_k, d_k, mask_kind, kv_lens, scale, stream);
}

attn_status launch_out_proj(const void* concat, const void* w_o, void* out, int B, int n_q,
                            int d_model, int h, int d_v, cudaStream_t stream) {
  const int Mq = B * n_q;
  if (Mq == 0) return ATTN_OK;
  tsd::GemmProblem g;
  std::memset(&g, 0, sizeof(g));
  g.K = h * d_v;
  g.num_groups = 1;
  cudaError_t e = make_gemm_group(&g.g[0], concat, w_o, out, Mq, d_model, h * d_v);
  if (e != cudaSuccess) return cuda_fail(e);
  finish_gemm_problem(&g);
  e = tsd::launch_gemm_bf16(g, stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// Workspace of attn_decode: the chunk partials O (float) then (m, l) pairs.
bool decode_layout(int B, int h, int n_q, int n_max, int d, size_t* o_bytes, size_t* total) {
  if (B < 0 || h < 0 || n_q < 1 || n_q > tsd::kDecodeMaxQueries || n_max < 1 || d < 1)
    return false;
  const uint64_t rows = uint64_t(B) * h * tsd::decode_chunks(n_max) * n_q;
  const uint64_t ob = align256(rows * d * 4), mb = align256(rows * 2 * 4);
  if (ob + mb > (uint64_t(1) << 62)) return false;
  *o_bytes = ob;
  *total = ob + mb;
  return true;
}

// Workspace of encoder_layer_forward: mha_forward's own, then the attention
// output, y = LayerNorm_1(x + attention) in bf16 (the FFN's input) and fp32
// (its residual), the FFN's hidden layer and z = y + FFN(y) in fp32.
struct EncoderLayout {
  size_t mha_bytes, a_off, y_off, y32_off, hid_off, z_off, total;
};

bool encoder_layout(int B, int n, int d_model, int h, int d_k, int d_ff, EncoderLayout* L) {
  if (B < 0 || n < 0 || d_model <= 0 || h <= 0 || d_k <= 0 || d_ff <= 0) return false;
  MhaLayout M;
  if (!mha_layout(B, n, n, h, d_k, d_k, &M)) return false;
  const uint64_t rows = uint64_t(B) * n;
  L->mha_bytes = M.total;
  L->a_off = align256(M.total);
  L->y_off = L->a_off + align256(rows * d_model * 2);
  L->y32_off = L->y_off + align256(rows * d_model * 2);
  L->hid_off = L->y32_off + align256(rows * d_model * 4);
  L->z_off = L->hid_off + align256(rows * uint64_t(d_ff) * 2);
  L->total = L->z_off + align256(rows * d_model * 4);
  return true;
}

// out = x W (+ bias, + residual, ReLU): one GEMM launch with the epilogue;
// out is bf16, or fp32 when out_f32 (then the residual is fp32 too).
attn_status launch_linear(const void* x, const void* w, const void* bias, const void* residual,
                          bool relu, void* out, bool out_f32, int M, int N, int K,
                          cudaStream_t stream) {
  if (M == 0) return ATTN_OK;
  tsd::GemmProblem g;
  std::memset(&g, 0, sizeof(g));
  g.K = K;
  g.num_groups = 1;
  cudaError_t e = make_gemm_group(&g.g[0], x, w, out, M, N, K);
  if (e != cudaSuccess) return cuda_fail(e);
  // the kernel's epilogue modes: + bias, ReLU (bf16 out); + bias + fp32
  // residual (fp32 out)
  if (out_f32 ? (residual == nullptr || relu || bias == nullptr)
              : (residual != nullptr || (bias != nullptr) != relu))
    return ATTN_ERR_INVALID;
  g.g[0].bias = static_cast<const uint16_t*>(bias);
  if (out_f32) {
    g.g[0].residual_f32 = static_cast<const float*>(residual);
    g.g[0].c_f32 = static_cast<float*>(out);
  }
  g.g[0].ldr = N;
  g.g[0].relu = relu ? 1 : 0;
  finish_gemm_problem(&g);
  e = tsd::launch_gemm_bf16(g, stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// out = LayerNorm(x W + bias + residual32) over each row's N columns (N in
// {128, 256, 512, 1024}): one GEMM launch whose epilogue normalises (the
// row's columns spread over a cluster of N / 128 CTAs).
attn_status launch_linear_ln(const void* x, const void* w, const void* bias,
                             const float* residual32, const void* gamma, const void* beta,
                             float eps, void* out, int M, int N, int K, cudaStream_t stream) {
  if (M == 0) return ATTN_OK;
  tsd::GemmProblem g;
  std::memset(&g, 0, sizeof(g));
  g.K = K;
  g.num_groups = 1;
  cudaError_t e = make_gemm_group(&g.g[0], x, w, out, M, N, K);
  if (e != cudaSuccess) return cuda_fail(e);
  g.g[0].bias = static_cast<const uint16_t*>(bias);
  g.g[0].residual_f32 = residual32;
  g.g[0].ldr = N;
  g.g[0].ln_gamma = static_cast<const uint16_t*>(gamma);
  g.g[0].ln_beta = static_cast<const uint16_t*>(beta);
  g.g[0].ln_eps = eps;
  finish_gemm_problem(&g);
  e = tsd::launch_gemm_bf16(g, stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}


// The checks of each entry point, apart from its launches, so that the
// host-buffer entry points can refuse bad arguments before copying anything.
attn_status attn_check(const void* q, const void* k, const void* v, const void* out, int B, int h,
                       int n_q, int n_k, int d_k, int d_v, int mask_kind, const int32_t* kv_lens,
                       float scale) {
  attn_status s = check_common(B, h, n_q, n_k, d_k, d_v, mask_kind, kv_lens, scale);
  if (s != ATTN_OK) return s;
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_ERR_INVALID;
  return check_bf16_head_dims(d_k, d_v);
}

attn_status mha_check(const void* x_q, const void* x_kv, const void* w_q, const void* w_k,
                      const void* w_v, const void* w_o, const void* out, int B, int n_q, int n_k,
                      int d_model, int h, int d_k, int d_v, int mask_kind,
                      const int32_t* kv_lens, float scale, const void* workspace,
                      size_t workspace_bytes) {
  attn_status s = check_common(B, h, n_q, n_k, d_k, d_v, mask_kind, kv_lens, scale);
  if (s != ATTN_OK) return s;
  if (h <= 0 || d_model < 8 || (d_model % 8) != 0) return ATTN_ERR_INVALID;
  const void* ptrs[8] = {x_q, x_kv, w_q, w_k, w_v, w_o, out, workspace};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return ATTN_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_INVALID;
  s = check_bf16_head_dims(d_k, d_v);
  if (s != ATTN_OK) return s;
  MhaLayout L;
  if (!mha_layout(B, n_q, n_k, h, d_k, d_v, &L)) return ATTN_ERR_INVALID;
  if (workspace_bytes < L.total) return ATTN_ERR_INVALID;
  if (int64_t(B) * n_q > INT32_MAX || int64_t(B) * n_k > INT32_MAX) return ATTN_ERR_INVALID;
  return ATTN_OK;
}

attn_status encoder_check(const void* const* ptrs15, int B, int n, int d_model, int h, int d_k,
                          int d_ff, int mask_kind, const int32_t* kv_lens, float scale, float eps,
                          const void* workspace, size_t workspace_bytes) {
  attn_status s = check_common(B, h, n, n, d_k, d_k, mask_kind, kv_lens, scale);
  if (s != ATTN_OK) return s;
  if (!(eps > 0.f) || !std::isfinite(eps)) return ATTN_ERR_INVALID;
  if (d_model != 256 && d_model != 512 && d_model != 1024 && d_model != 2048)
    return ATTN_ERR_UNSUPPORTED;
  if (d_ff < 8 || (d_ff % 8) != 0) return ATTN_ERR_INVALID;
  s = check_bf16_head_dims(d_k, d_k);
  if (s != ATTN_OK) return s;
  for (int i = 0; i < 15; ++i)
    if (ptrs15[i] == nullptr || !aligned16(ptrs15[i])) return ATTN_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_INVALID;
  EncoderLayout L;
  if (!encoder_layout(B, n, d_model, h, d_k, d_ff, &L)) return ATTN_ERR_INVALID;
  if (workspace_bytes < L.total) return ATTN_ERR_INVALID;
  if (int64_t(B) * n > INT32_MAX) return ATTN_ERR_INVALID;
  return ATTN_OK;
}

attn_status decode_check(const void* q, const void* k_cache, const void* v_cache, const void* out,
                         int B, int h, int n_q, int n_max, int d_k, int d_v,
                         const int32_t* cache_lens, float scale, const void* workspace,
                         size_t workspace_bytes) {
  if (B < 0 || h < 0 || n_q < 1 || n_max < 1) return ATTN_ERR_INVALID;
  if (n_q > tsd::kDecodeMaxQueries || tsd::decode_chunks(n_max) > tsd::kDecodeMaxChunks)
    return ATTN_ERR_UNSUPPORTED;
  if (B > 65535 || h > 65535 || int64_t(B) * h > INT32_MAX) return ATTN_ERR_INVALID;
  if (!valid_scale(scale)) return ATTN_ERR_INVALID;
  if (d_k != d_v || (d_k != 64 && d_k != 128)) return ATTN_ERR_UNSUPPORTED;
  const void* ptrs[5] = {q, k_cache, v_cache, out, workspace};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return ATTN_ERR_INVALID;
  if (cache_lens != nullptr && (reinterpret_cast<uintptr_t>(cache_lens) & 3u))
    return ATTN_ERR_INVALID;
  size_t ob = 0, total = 0;
  if (!decode_layout(B, h, n_q, n_max, d_v, &ob, &total)) return ATTN_ERR_INVALID;
  if (workspace_bytes < total) return ATTN_ERR_INVALID;
  return ATTN_OK;
}

// Staging regions of the host-buffer entry points, 256-byte aligned, in
// order; the device entry point's own workspace follows them.
struct StageLayout {
  size_t end = 0;
  bool ok = true;
  size_t add(uint64_t bytes) {
    const size_t off = end;
    if (bytes > (uint64_t(1) << 60) || end > (size_t(1) << 61)) ok = false;
    else end += align256(bytes);
    return off;
  }
};

// Staging layouts of the host-buffer entry points; false for invalid sizes.
bool attn_host_layout(int B, int h, int n_q, int n_k, int d_k, int d_v, size_t* total) {
  if (B < 0 || h < 0 || n_q < 0 || n_k < 0 || d_k <= 0 || d_v <= 0) return false;
  StageLayout S;
  S.add(uint64_t(B) * h * n_q * d_k * 2);
  S.add(uint64_t(B) * h * n_k * d_k * 2);
  S.add(uint64_t(B) * h * n_k * d_v * 2);
  S.add(uint64_t(B) * 4);
  S.add(uint64_t(B) * h * n_q * d_v * 2);
  *total = S.end;
  return S.ok;
}

bool mha_host_layout(int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                     size_t* total) {
  MhaLayout L;
  if (d_model <= 0 || !mha_layout(B, n_q, n_k, h, d_k, d_v, &L)) return false;
  StageLayout S;
  S.add(uint64_t(B) * n_q * d_model * 2);
  S.add(uint64_t(B) * n_k * d_model * 2);
  S.add(uint64_t(B) * 4);
  S.add(uint64_t(B) * n_q * d_model * 2);
  S.add(L.total);
  *total = S.end;
  return S.ok;
}

bool encoder_host_layout(int B, int n, int d_model, int h, int d_k, int d_ff, size_t* total) {
  EncoderLayout L;
  if (!encoder_layout(B, n, d_model, h, d_k, d_ff, &L)) return false;
  StageLayout S;
  S.add(uint64_t(B) * n * d_model * 2);
  S.add(uint64_t(B) * 4);
  S.add(uint64_t(B) * n * d_model * 2);
  S.add(L.total);
  *total = S.end;
  return S.ok;
}

bool decode_host_layout(int B, int h, int n_q, int n_max, int d_k, int d_v, size_t* total) {
  size_t ob = 0, inner = 0;
  if (d_k <= 0 || !decode_layout(B, h, n_q, n_max, d_v, &ob, &inner)) return false;
  StageLayout S;
  S.add(uint64_t(B) * h * n_q * d_k * 2);
  S.add(uint64_t(B) * 4);
  S.add(uint64_t(B) * h * n_q * d_v * 2);
  S.add(inner);
  *total = S.end;
  return S.ok;
}

}  // namespace

extern "C" {

attn_status attn_forward(const void* q, const void* k, const void* v, void* out, int B, int h,
                         int n_q, int n_k, int d_k, int d_v, int mask_kind, const int32_t* kv_lens,
                         float scale, tsd_stream_t stream) {
  attn_status s = attn_check(q, k, v, out, B, h, n_q, n_k, d_k, d_v, mask_kind, kv_lens, scale);
  if (s != ATTN_OK) return s;
  if (B == 0 || h == 0 || n_q == 0) return ATTN_OK;  // nothing to write
  const int64_t d = d_k;
  return run_attn_bf16(q, int64_t(h) * n_q * d, int64_t(n_q) * d, d, k, int64_t(h) * n_k * d,
                       int64_t(n_k) * d, d, v, int64_t(h) * n_k * d, int64_t(n_k) * d, d, out,
                       int64_t(h) * n_q * d, int64_t(n_q) * d, d, B, h, n_q, n_k, d_k, mask_kind,
                       kv_lens, scale, reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_forward_window(const void* q, const void* k, const void* v, void* out, int B,
                                int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                                const int32_t* kv_lens, int window_left, int window_right,
                                float scale, tsd_stream_t stream) {
  attn_status s = check_common(B, h, n_q, n_k, d_k, d_v, mask_kind, kv_lens, scale);
  if (s != ATTN_OK) return s;
  if (window_left < -1 || window_right < -1) return ATTN_ERR_INVALID;
  const bool windowed = window_left >= 0 || window_right >= 0;
  if (windowed && n_q != n_k) return ATTN_ERR_INVALID;
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_ERR_INVALID;
  s = check_bf16_head_dims(d_k, d_v);
  if (s != ATTN_OK) return s;
  if (B == 0 || h == 0 || n_q == 0) return ATTN_OK;  // nothing to write
  const int64_t d = d_k;
  return run_attn_bf16(q, int64_t(h) * n_q * d, int64_t(n_q) * d, d, k, int64_t(h) * n_k * d,
                       int64_t(n_k) * d, d, v, int64_t(h) * n_k * d, int64_t(n_k) * d, d, out,
                       int64_t(h) * n_q * d, int64_t(n_q) * d, d, B, h, n_q, n_k, d_k, mask_kind,
                       kv_lens, scale, reinterpret_cast<cudaStream_t>(stream), window_left,
                       window_right);
}

attn_status attn_forward_strided(const void* q, int64_t q_sb, int64_t q_sh, int64_t q_sr,
                                 const void* k, int64_t k_sb, int64_t k_sh, int64_t k_sr,
                                 const void* v, int64_t v_sb, int64_t v_sh, int64_t v_sr,
                                 void* out, int64_t o_sb, int64_t o_sh, int64_t o_sr, int B,
                                 int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                                 const int32_t* kv_lens, float scale, tsd_stream_t stream) {
  attn_status s = check_common(B, h, n_q, n_k, d_k, d_v, mask_kind, kv_lens, scale);
  if (s != ATTN_OK) return s;
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_ERR_INVALID;
  s = check_bf16_head_dims(d_k, d_v);
  if (s != ATTN_OK) return s;
  const int64_t strides[12] = {q_sb, q_sh, q_sr, k_sb, k_sh, k_sr, v_sb, v_sh, v_sr, o_sb, o_sh, o_sr};
  for (int64_t st : strides)
    if (st <= 0 || (st % 8) != 0 || st > (int64_t(1) << 38)) return ATTN_ERR_INVALID;
  if (q_sr < d_k || k_sr < d_k || v_sr < d_v || o_sr < d_v) return ATTN_ERR_INVALID;
  if (B == 0 || h == 0 || n_q == 0) return ATTN_OK;
  return run_attn_bf16(q, q_sb, q_sh, q_sr, k, k_sb, k_sh, k_sr, v, v_sb, v_sh, v_sr, out, o_sb,
                       o_sh, o_sr, B, h, n_q, n_k, d_k, mask_kind, kv_lens, scale,
                       reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_forward_f32(const float* q, const float* k, const float* v, float* out, int B,
                             int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                             const int32_t* kv_lens, float scale, tsd_stream_t stream) {
  attn_status s = check_common(B, h, n_q, n_k, d_k, d_v, mask_kind, kv_lens, scale);
  if (s != ATTN_OK) return s;
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) & 3u)
    return ATTN_ERR_INVALID;
  if (d_k > 128 || d_v > 128) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || h == 0 || n_q == 0) return ATTN_OK;
  tsd::AttnF32Problem p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.h = h;
  p.n_q = n_q;
  p.n_k = n_k;
  p.d_k = d_k;
  p.d_v = d_v;
  p.mask_kind = mask_kind;
  p.kv_lens = kv_lens;
  p.scale = resolve_scale(scale, d_k);
  cudaError_t e = tsd::launch_attn_f32(p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

size_t mha_workspace_bytes(int B, int n_q, int n_k, int h, int d_k, int d_v) {
  MhaLayout L;
  if (!mha_layout(B, n_q, n_k, h, d_k, d_v, &L)) return 0;
  return L.total;
}

attn_status mha_forward(const void* x_q, const void* x_kv, const void* w_q, const void* w_k,
                        const void* w_v, const void* w_o, void* out, int B, int n_q, int n_k,
                        int d_model, int h, int d_k, int d_v, int mask_kind,
                        const int32_t* kv_lens, float scale, void* workspace,
                        size_t workspace_bytes, tsd_stream_t stream_) {
  attn_status s = mha_check(x_q, x_kv, w_q, w_k, w_v, w_o, out, B, n_q, n_k, d_model, h, d_k, d_v,
                            mask_kind, kv_lens, scale, workspace, workspace_bytes);
  if (s != ATTN_OK) return s;
  MhaLayout L;
  mha_layout(B, n_q, n_k, h, d_k, d_v, &L);
  if (int64_t(B) * n_q == 0) return ATTN_OK;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* Q = ws + L.q_off;
  void* K = ws + L.k_off;
  void* V = ws + L.v_off;
  void* O = ws + L.o_off;
  // Short sequences: projections, attention and W_O in one launch (the
  // merged heads pass through the workspace's last region)
  if (fused_eligible(n_q, n_k, d_model, h, d_k, d_v) &&
      fused_out_eligible(x_q == x_kv && n_q == n_k, d_model, h))
    return launch_fused_core(x_q, x_kv, w_q, w_k, w_v, O, B, n_q, n_k, d_model, h, mask_kind,
                             kv_lens, scale, stream, w_o, out);
  // Cross-attention over one or two source key tiles: the same, in mha_cross.cu
  if (cross_eligible(x_q == x_kv && n_q == n_k, n_q, n_k, d_model, h, d_k, d_v) &&
      cross_out_eligible(d_model, h))
    return launch_fused_core(x_q, x_kv, w_q, w_k, w_v, O, B, n_q, n_k, d_model, h, mask_kind,
                             kv_lens, scale, stream, w_o, out);
  // 1-2. Concat(head_1..head_h) into the workspace's last region
  s = concat_heads(x_q, x_kv, w_q, w_k, w_v, O, Q, K, V, B, n_q, n_k, d_model, h, d_k, d_v,
                   mask_kind, kv_lens, scale, stream);
  if (s != ATTN_OK) return s;
  // 3. out = Concat(head_1..head_h) W_O
  return launch_out_proj(O, w_o, out, B, n_q, d_model, h, d_v, stream);
}

size_t attn_decode_workspace_bytes(int B, int h, int n_q, int n_max, int d_v) {
  size_t ob = 0, total = 0;
  return decode_layout(B, h, n_q, n_max, d_v, &ob, &total) ? total : 0;
}

attn_status attn_decode(const void* q, const void* k_cache, const void* v_cache, void* out, int B,
                        int h, int n_q, int n_max, int d_k, int d_v, const int32_t* cache_lens,
                        float scale, void* workspace, size_t workspace_bytes,
                        tsd_stream_t stream) {
  attn_status s = decode_check(q, k_cache, v_cache, out, B, h, n_q, n_max, d_k, d_v, cache_lens,
                               scale, workspace, workspace_bytes);
  if (s != ATTN_OK) return s;
  size_t ob = 0, total = 0;
  decode_layout(B, h, n_q, n_max, d_v, &ob, &total);
  if (B == 0 || h == 0) return ATTN_OK;
  tsd::DecodeProblem p;
  std::memset(&p, 0, sizeof(p));
  const uint64_t dims[3] = {static_cast<uint64_t>(d_k), static_cast<uint64_t>(n_max),
                            static_cast<uint64_t>(B) * h};
  const int64_t strides[2] = {d_k, int64_t(n_max) * d_k};
  const uint32_t box[3] = {64, 128, 1};
  cudaError_t e = encode_bf16_map(&p.tm_k, k_cache, 3, dims, strides, box);
  if (e == cudaSuccess) e = encode_bf16_map(&p.tm_v, v_cache, 3, dims, strides, box);
  if (e != cudaSuccess) return cuda_fail(e);
  p.q = q;
  p.out = out;
  p.cache_lens = cache_lens;
  p.ws_o = static_cast<float*>(workspace);
  p.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ob);
  p.B = B;
  p.h = h;
  p.n_q = n_q;
  p.n_max = n_max;
  p.d = d_k;
  p.scale = resolve_scale(scale, d_k);
  e = tsd::launch_decode(p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

size_t encoder_layer_workspace_bytes(int B, int n, int d_model, int h, int d_k, int d_ff) {
  EncoderLayout L;
  return encoder_layout(B, n, d_model, h, d_k, d_ff, &L) ? L.total : 0;
}

attn_status encoder_layer_forward(const void* x, const void* w_q, const void* w_k,
                                  const void* w_v, const void* w_o, const void* ln1_gamma,
                                  const void* ln1_beta, const void* w_1, const void* b_1,
                                  const void* w_2, const void* b_2, const void* ln2_gamma,
                                  const void* ln2_beta, void* out, int B, int n, int d_model,
                                  int h, int d_k, int d_ff, int mask_kind,
                                  const int32_t* kv_lens, float scale, float eps,
                                  void* workspace, size_t workspace_bytes,
                                  tsd_stream_t stream_) {
  const void* ptrs[15] = {x, w_q, w_k, w_v, w_o, ln1_gamma, ln1_beta, w_1, b_1, w_2, b_2,
                          ln2_gamma, ln2_beta, out, workspace};
  attn_status s = encoder_check(ptrs, B, n, d_model, h, d_k, d_ff, mask_kind, kv_lens, scale, eps,
                                workspace, workspace_bytes);
  if (s != ATTN_OK) return s;
  EncoderLayout L;
  encoder_layout(B, n, d_model, h, d_k, d_ff, &L);
  const int rows = static_cast<int>(int64_t(B) * n);
  if (rows == 0) return ATTN_OK;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* a = reinterpret_cast<uint16_t*>(ws + L.a_off);
  uint16_t* y = reinterpret_cast<uint16_t*>(ws + L.y_off);
  float* y32 = reinterpret_cast<float*>(ws + L.y32_off);
  uint16_t* hid = reinterpret_cast<uint16_t*>(ws + L.hid_off);
  float* z = reinterpret_cast<float*>(ws + L.z_off);
  // 1. a = MultiHead(x, x)
  s = mha_forward(x, x, w_q, w_k, w_v, w_o, a, B, n, n, d_model, h, d_k, d_k, mask_kind, kv_lens,
                  scale, ws, L.mha_bytes, stream_);
  if (s != ATTN_OK) return s;
  // 2. y = LayerNorm_1(x + a): bf16 for the FFN's GEMM, fp32 for its residual
  cudaError_t e = tsd::launch_add_layernorm(x, false, a,
                                            static_cast<const uint16_t*>(ln1_gamma),
                                            static_cast<const uint16_t*>(ln1_beta), y, y32, rows,
                                            d_model, eps, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  // 3. hid = max(0, y W_1 + b_1)
  s = launch_linear(y, w_1, b_1, nullptr, true, hid, false, rows, d_ff, d_model, stream);
  if (s != ATTN_OK) return s;
  // 4-5. out = LayerNorm_2(y + (hid W_2 + b_2)): in the second GEMM's
  // epilogue when a row's d_model columns fit one cluster (<= 8 x 128)
  if (d_model <= 1024)
    return launch_linear_ln(hid, w_2, b_2, y32, ln2_gamma, ln2_beta, eps, out, rows, d_model, d_ff,
                            stream);
  // 4. z = y + (hid W_2 + b_2), fp32
  s = launch_linear(hid, w_2, b_2, y32, false, z, true, rows, d_model, d_ff, stream);
  if (s != ATTN_OK) return s;
  // 5. out = LayerNorm_2(z)
  e = tsd::launch_add_layernorm(z, true, nullptr, static_cast<const uint16_t*>(ln2_gamma),
                                static_cast<const uint16_t*>(ln2_beta),
                                static_cast<uint16_t*>(out), nullptr, rows, d_model, eps,
                                stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

int mha_forward_launches(int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                         int self_attention) {
  if (B < 0 || n_q < 0 || n_k < 0 || h <= 0 || d_model < 8 || (d_model % 8) != 0 ||
      check_bf16_head_dims(d_k, d_v) != ATTN_OK)
    return -1;
  if (int64_t(B) * n_q == 0) return 0;
  const bool self = self_attention != 0 && n_q == n_k;
  if (cross_eligible(self, n_q, n_k, d_model, h, d_k, d_v))
    return cross_out_eligible(d_model, h) ? 1 : 2;
  if (!fused_eligible(n_q, n_k, d_model, h, d_k, d_v)) return 3;
  return fused_out_eligible(self, d_model, h) ? 1 : 2;
}

attn_status mha_concat_heads(const void* x_q, const void* x_kv, const void* w_q, const void* w_k,
                             const void* w_v, void* concat, int B, int n_q, int n_k, int d_model,
                             int h, int d_k, int d_v, int mask_kind, const int32_t* kv_lens,
                             float scale, void* workspace, size_t workspace_bytes,
                             tsd_stream_t stream_) {
  attn_status s = check_common(B, h, n_q, n_k, d_k, d_v, mask_kind, kv_lens, scale);
  if (s != ATTN_OK) return s;
  if (h <= 0 || d_model < 8 || (d_model % 8) != 0) return ATTN_ERR_INVALID;
  const void* ptrs[7] = {x_q, x_kv, w_q, w_k, w_v, concat, workspace};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return ATTN_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_INVALID;
  s = check_bf16_head_dims(d_k, d_v);
  if (s != ATTN_OK) return s;
  MhaLayout L;
  if (!mha_layout(B, n_q, n_k, h, d_k, d_v, &L)) return ATTN_ERR_INVALID;
  if (workspace_bytes < L.total) return ATTN_ERR_INVALID;
  const int64_t Mq = int64_t(B) * n_q, Mk = int64_t(B) * n_k;
  if (Mq > INT32_MAX || Mk > INT32_MAX) return ATTN_ERR_INVALID;
  if (Mq == 0) return ATTN_OK;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return concat_heads(x_q, x_kv, w_q, w_k, w_v, concat, ws + L.q_off, ws + L.k_off, ws + L.v_off,
                      B, n_q, n_k, d_model, h, d_k, d_v, mask_kind, kv_lens, scale,
                      reinterpret_cast<cudaStream_t>(stream_));
}

attn_status mha_project_qkv(const void* x_q, const void* x_kv, const void* w_q, const void* w_k,
                            const void* w_v, void* q_out, void* k_out, void* v_out, int B, int n_q,
                            int n_k, int d_model, int h, int d_k, int d_v, tsd_stream_t stream) {
  attn_status s = check_projection(B, n_q, n_k, d_model, h, d_k, d_v);
  if (s != ATTN_OK) return s;
  const void* ptrs[8] = {x_q, x_kv, w_q, w_k, w_v, q_out, k_out, v_out};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return ATTN_ERR_INVALID;
  return launch_qkv(x_q, x_kv, w_q, w_k, w_v, q_out, k_out, v_out, B, n_q, n_k, d_model, h, d_k,
                    d_v, reinterpret_cast<cudaStream_t>(stream));
}

attn_status mha_project_out(const void* concat, const void* w_o, void* out, int B, int n_q,
                            int d_model, int h, int d_v, tsd_stream_t stream) {
  attn_status s = check_projection(B, n_q, 0, d_model, h, d_v, d_v);
  if (s != ATTN_OK) return s;
  const void* ptrs[3] = {concat, w_o, out};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return ATTN_ERR_INVALID;
  return launch_out_proj(concat, w_o, out, B, n_q, d_model, h, d_v,
                         reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_get_device_status(tsd_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int a = 0, g = 0, f = 0, m = 0;
  e = tsd::take_device_error_attn(&a);
  if (e == cudaSuccess) e = tsd::take_device_error_gemm(&g);
  if (e == cudaSuccess) e = tsd::take_device_error_f32(&f);
  if (e == cudaSuccess) e = tsd::take_device_error_fused(&m);
  unsigned int cr = 0;
  if (e == cudaSuccess) e = tsd::take_device_error_cross(&cr);
  m |= cr;
  unsigned int dec = 0;
  if (e == cudaSuccess) e = tsd::take_device_error_decode(&dec);
  m |= dec;
  if (e != cudaSuccess) return cuda_fail(e);
  return (a | g | f | m) ? ATTN_ERR_DEVICE_TIMEOUT : ATTN_OK;
}

int attn_last_cuda_error(void) { return g_last_cuda_error; }

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID: return "ATTN_ERR_INVALID";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
  }
  return "ATTN_STATUS_UNKNOWN";
}

attn_status attn_selftest_wait_timeout(int limit_us, tsd_stream_t stream) {
  if (limit_us < 1 || limit_us > 2000000) return ATTN_ERR_INVALID;
  cudaError_t e = tsd::launch_wait_timeout_selftest(static_cast<unsigned long long>(limit_us) * 1000ull,
                                                    reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- host buffers
// The same operations with the step's inputs and result in host memory: the
// inputs are copied into staging regions at the front of the workspace, the
// device entry point runs on them (on `stream`), and the result is copied
// back on `stream` (host_stage.h has the ordering).

size_t attn_host_workspace_bytes(int B, int h, int n_q, int n_k, int d_k, int d_v) {
  size_t t = 0;
  return attn_host_layout(B, h, n_q, n_k, d_k, d_v, &t) ? t : 0;
}

}  // extern "C"

namespace {

// attn_forward_host and attn_forward_window_host (windowed: the window's
// bounds apply, as in attn_forward_window)
attn_status attn_host_call(const void* q_host, const void* k_host, const void* v_host,
                           void* out_host, int B, int h, int n_q, int n_k, int d_k, int d_v,
                           int mask_kind, const int32_t* kv_lens_host, bool windowed,
                           int window_left, int window_right, float scale, void* workspace,
                           size_t workspace_bytes, tsd_stream_t stream) {
  if (!q_host || !k_host || !v_host || !out_host || !workspace) return ATTN_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_INVALID;
  size_t need = 0;
  if (!attn_host_layout(B, h, n_q, n_k, d_k, d_v, &need) || workspace_bytes < need)
    return ATTN_ERR_INVALID;
  if (windowed && (window_left < -1 || window_right < -1 ||
                   ((window_left >= 0 || window_right >= 0) && n_q != n_k)))
    return ATTN_ERR_INVALID;
  StageLayout S;
  const uint64_t qb = uint64_t(B) * h * n_q * d_k * 2, kb = uint64_t(B) * h * n_k * d_k * 2,
                 vb = uint64_t(B) * h * n_k * d_v * 2, ob = uint64_t(B) * h * n_q * d_v * 2;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* q = ws + S.add(qb);
  void* k = ws + S.add(kb);
  void* v = ws + S.add(vb);
  int32_t* lens = reinterpret_cast<int32_t*>(ws + S.add(uint64_t(B) * 4));
  void* out = ws + S.add(ob);
  const bool pad = (mask_kind & ATTN_MASK_KEY_PADDING) != 0 && kv_lens_host != nullptr;
  attn_status s = attn_check(q, k, v, out, B, h, n_q, n_k, d_k, d_v, mask_kind,
                             pad ? lens : nullptr, scale);
  if (s != ATTN_OK) return s;
  if (B == 0 || h == 0 || n_q == 0) return ATTN_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  tsd::HostStage hs(workspace, st);
  hs.copy_in(q, q_host, qb);
  hs.copy_in(k, k_host, kb);
  hs.copy_in(v, v_host, vb);
  if (pad) hs.copy_in(lens, kv_lens_host, size_t(B) * 4);
  if (hs.inputs_ready() != cudaSuccess) return cuda_fail(hs.status());
  s = windowed ? attn_forward_window(q, k, v, out, B, h, n_q, n_k, d_k, d_v, mask_kind,
                                     pad ? lens : nullptr, window_left, window_right, scale,
                                     stream)
               : attn_forward(q, k, v, out, B, h, n_q, n_k, d_k, d_v, mask_kind,
                              pad ? lens : nullptr, scale, stream);
  hs.computed();
  if (s != ATTN_OK) return s;
  return hs.copy_out(out_host, out, ob) == cudaSuccess ? ATTN_OK : cuda_fail(hs.status());
}

}  // namespace

extern "C" {

attn_status attn_forward_host(const void* q_host, const void* k_host, const void* v_host,
                              void* out_host, int B, int h, int n_q, int n_k, int d_k, int d_v,
                              int mask_kind, const int32_t* kv_lens_host, float scale,
                              void* workspace, size_t workspace_bytes, tsd_stream_t stream) {
  return attn_host_call(q_host, k_host, v_host, out_host, B, h, n_q, n_k, d_k, d_v, mask_kind,
                        kv_lens_host, false, -1, -1, scale, workspace, workspace_bytes, stream);
}

attn_status attn_forward_window_host(const void* q_host, const void* k_host, const void* v_host,
                                     void* out_host, int B, int h, int n_q, int n_k, int d_k,
                                     int d_v, int mask_kind, const int32_t* kv_lens_host,
                                     int window_left, int window_right, float scale,
                                     void* workspace, size_t workspace_bytes,
                                     tsd_stream_t stream) {
  return attn_host_call(q_host, k_host, v_host, out_host, B, h, n_q, n_k, d_k, d_v, mask_kind,
                        kv_lens_host, true, window_left, window_right, scale, workspace,
                        workspace_bytes, stream);
}

size_t mha_host_workspace_bytes(int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v) {
  size_t t = 0;
  return mha_host_layout(B, n_q, n_k, d_model, h, d_k, d_v, &t) ? t : 0;
}

}  // extern "C"

namespace {

attn_status mha_host_call(const void* x_q_host, const void* x_kv_host, const void* w_q,
                          const void* w_k, const void* w_v, const void* w_o, void* out_host, int B,
                          int n_q, int n_k, int d_model, int h, int d_k, int d_v, int mask_kind,
                          const int32_t* kv_lens_host, float scale, void* workspace,
                          size_t workspace_bytes, tsd_stream_t stream, bool async) {
  if (!x_q_host || !x_kv_host || !out_host || !workspace) return ATTN_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_INVALID;
  size_t need = 0;
  if (!mha_host_layout(B, n_q, n_k, d_model, h, d_k, d_v, &need) || workspace_bytes < need)
    return ATTN_ERR_INVALID;
  // one host array for both (self-attention) -> one staged copy, so the
  // device entry point sees x_kv == x_q and takes its self-attention path
  const bool self = x_kv_host == x_q_host && n_q == n_k;
  const uint64_t xqb = uint64_t(B) * n_q * d_model * 2, xkb = uint64_t(B) * n_k * d_model * 2;
  StageLayout S;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* x_q = ws + S.add(xqb);
  void* x_kv = ws + S.add(xkb);
  if (self) x_kv = x_q;
  int32_t* lens = reinterpret_cast<int32_t*>(ws + S.add(uint64_t(B) * 4));
  void* out = ws + S.add(xqb);
  const size_t inner_off = S.add(0);
  void* inner = ws + inner_off;
  const size_t inner_bytes = workspace_bytes - inner_off;
  const bool pad = (mask_kind & ATTN_MASK_KEY_PADDING) != 0 && kv_lens_host != nullptr;
  attn_status s = mha_check(x_q, x_kv, w_q, w_k, w_v, w_o, out, B, n_q, n_k, d_model, h, d_k, d_v,
                            mask_kind, pad ? lens : nullptr, scale, inner, inner_bytes);
  if (s != ATTN_OK) return s;
  if (int64_t(B) * n_q == 0) return ATTN_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  tsd::HostStage hs(workspace, st);
  hs.copy_in(x_q, x_q_host, xqb);
  if (!self) hs.copy_in(x_kv, x_kv_host, xkb);
  if (pad) hs.copy_in(lens, kv_lens_host, size_t(B) * 4);
  if (hs.inputs_ready() != cudaSuccess) return cuda_fail(hs.status());
  s = mha_forward(x_q, x_kv, w_q, w_k, w_v, w_o, out, B, n_q, n_k, d_model, h, d_k, d_v, mask_kind,
                  pad ? lens : nullptr, scale, inner, inner_bytes, stream);
  hs.computed();
  if (s != ATTN_OK) return s;
  const cudaError_t e =
      async ? hs.copy_out_async(out_host, out, xqb) : hs.copy_out(out_host, out, xqb);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(hs.status());
}


}  // namespace

extern "C" {

attn_status mha_forward_host(const void* x_q_host, const void* x_kv_host, const void* w_q,
                             const void* w_k, const void* w_v, const void* w_o, void* out_host,
                             int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                             int mask_kind, const int32_t* kv_lens_host, float scale,
                             void* workspace, size_t workspace_bytes, tsd_stream_t stream) {
  return mha_host_call(x_q_host, x_kv_host, w_q, w_k, w_v, w_o, out_host, B, n_q, n_k, d_model, h,
                       d_k, d_v, mask_kind, kv_lens_host, scale, workspace, workspace_bytes, stream,
                       false);
}

attn_status mha_forward_host_async(const void* x_q_host, const void* x_kv_host, const void* w_q,
                                   const void* w_k, const void* w_v, const void* w_o,
                                   void* out_host, int B, int n_q, int n_k, int d_model, int h,
                                   int d_k, int d_v, int mask_kind, const int32_t* kv_lens_host,
                                   float scale, void* workspace, size_t workspace_bytes,
                                   tsd_stream_t stream) {
  return mha_host_call(x_q_host, x_kv_host, w_q, w_k, w_v, w_o, out_host, B, n_q, n_k, d_model, h,
                       d_k, d_v, mask_kind, kv_lens_host, scale, workspace, workspace_bytes, stream,
                       true);
}

attn_status attn_host_join(tsd_stream_t stream) {
  const cudaError_t e = tsd::host_join(reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

size_t encoder_layer_host_workspace_bytes(int B, int n, int d_model, int h, int d_k, int d_ff) {
  size_t t = 0;
  return encoder_host_layout(B, n, d_model, h, d_k, d_ff, &t) ? t : 0;
}

}  // extern "C"

namespace {

attn_status encoder_host_call(const void* x_host, const void* w_q, const void* w_k,
                              const void* w_v, const void* w_o, const void* ln1_gamma,
                              const void* ln1_beta, const void* w_1, const void* b_1,
                              const void* w_2, const void* b_2, const void* ln2_gamma,
                              const void* ln2_beta, void* out_host, int B, int n, int d_model,
                              int h, int d_k, int d_ff, int mask_kind,
                              const int32_t* kv_lens_host, float scale, float eps,
                              void* workspace, size_t workspace_bytes, tsd_stream_t stream,
                              bool async) {
  if (!x_host || !out_host || !workspace) return ATTN_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_INVALID;
  size_t need = 0;
  if (!encoder_host_layout(B, n, d_model, h, d_k, d_ff, &need) || workspace_bytes < need)
    return ATTN_ERR_INVALID;
  const uint64_t xb = uint64_t(B) * n * d_model * 2;
  StageLayout S;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* x = ws + S.add(xb);
  int32_t* lens = reinterpret_cast<int32_t*>(ws + S.add(uint64_t(B) * 4));
  void* out = ws + S.add(xb);
  const size_t inner_off = S.add(0);
  void* inner = ws + inner_off;
  const size_t inner_bytes = workspace_bytes - inner_off;
  const bool pad = (mask_kind & ATTN_MASK_KEY_PADDING) != 0 && kv_lens_host != nullptr;
  const void* ptrs[15] = {x, w_q, w_k, w_v, w_o, ln1_gamma, ln1_beta, w_1, b_1, w_2, b_2,
                          ln2_gamma, ln2_beta, out, inner};
  attn_status s = encoder_check(ptrs, B, n, d_model, h, d_k, d_ff, mask_kind,
                                pad ? lens : nullptr, scale, eps, inner, inner_bytes);
  if (s != ATTN_OK) return s;
  if (int64_t(B) * n == 0) return ATTN_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  tsd::HostStage hs(workspace, st);
  hs.copy_in(x, x_host, xb);
  if (pad) hs.copy_in(lens, kv_lens_host, size_t(B) * 4);
  if (hs.inputs_ready() != cudaSuccess) return cuda_fail(hs.status());
  s = encoder_layer_forward(x, w_q, w_k, w_v, w_o, ln1_gamma, ln1_beta, w_1, b_1, w_2, b_2,
                            ln2_gamma, ln2_beta, out, B, n, d_model, h, d_k, d_ff, mask_kind,
                            pad ? lens : nullptr, scale, eps, inner, inner_bytes, stream);
  hs.computed();
  if (s != ATTN_OK) return s;
  const cudaError_t e = async ? hs.copy_out_async(out_host, out, xb) : hs.copy_out(out_host, out, xb);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(hs.status());
}

}  // namespace

extern "C" {

attn_status encoder_layer_forward_host(const void* x_host, const void* w_q, const void* w_k,
                                       const void* w_v, const void* w_o, const void* ln1_gamma,
                                       const void* ln1_beta, const void* w_1, const void* b_1,
                                       const void* w_2, const void* b_2, const void* ln2_gamma,
                                       const void* ln2_beta, void* out_host, int B, int n,
                                       int d_model, int h, int d_k, int d_ff, int mask_kind,
                                       const int32_t* kv_lens_host, float scale, float eps,
                                       void* workspace, size_t workspace_bytes,
                                       tsd_stream_t stream) {
  return encoder_host_call(x_host, w_q, w_k, w_v, w_o, ln1_gamma, ln1_beta, w_1, b_1, w_2, b_2,
                           ln2_gamma, ln2_beta, out_host, B, n, d_model, h, d_k, d_ff, mask_kind,
                           kv_lens_host, scale, eps, workspace, workspace_bytes, stream, false);
}

attn_status encoder_layer_forward_host_async(
    const void* x_host, const void* w_q, const void* w_k, const void* w_v, const void* w_o,
    const void* ln1_gamma, const void* ln1_beta, const void* w_1, const void* b_1,
    const void* w_2, const void* b_2, const void* ln2_gamma, const void* ln2_beta,
    void* out_host, int B, int n, int d_model, int h, int d_k, int d_ff, int mask_kind,
    const int32_t* kv_lens_host, float scale, float eps, void* workspace,
    size_t workspace_bytes, tsd_stream_t stream) {
  return encoder_host_call(x_host, w_q, w_k, w_v, w_o, ln1_gamma, ln1_beta, w_1, b_1, w_2, b_2,
                           ln2_gamma, ln2_beta, out_host, B, n, d_model, h, d_k, d_ff, mask_kind,
                           kv_lens_host, scale, eps, workspace, workspace_bytes, stream, true);
}

size_t attn_decode_host_workspace_bytes(int B, int h, int n_q, int n_max, int d_k, int d_v) {
  size_t t = 0;
  return decode_host_layout(B, h, n_q, n_max, d_k, d_v, &t) ? t : 0;
}

}  // extern "C"

namespace {

attn_status decode_host_call(const void* q_host, const void* k_cache, const void* v_cache,
                             void* out_host, int B, int h, int n_q, int n_max, int d_k, int d_v,
                             const int32_t* cache_lens_host, float scale, void* workspace,
                             size_t workspace_bytes, tsd_stream_t stream, bool async) {
  if (!q_host || !out_host || !workspace) return ATTN_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_INVALID;
  size_t need = 0;
  if (!decode_host_layout(B, h, n_q, n_max, d_k, d_v, &need)) {
    // the device entry point's own code for these sizes (query and cache
    // limits are ATTN_ERR_UNSUPPORTED there)
    const attn_status s = decode_check(workspace, k_cache, v_cache, workspace, B, h, n_q, n_max,
                                       d_k, d_v, nullptr, scale, workspace, 0);
    return s != ATTN_OK ? s : ATTN_ERR_INVALID;
  }
  if (workspace_bytes < need) return ATTN_ERR_INVALID;
  const uint64_t qb = uint64_t(B) * h * n_q * d_k * 2, ob = uint64_t(B) * h * n_q * d_v * 2;
  StageLayout S;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* q = ws + S.add(qb);
  int32_t* lens = reinterpret_cast<int32_t*>(ws + S.add(uint64_t(B) * 4));
  void* out = ws + S.add(ob);
  const size_t inner_off = S.add(0);
  void* inner = ws + inner_off;
  const size_t inner_bytes = workspace_bytes - inner_off;
  const bool has_lens = cache_lens_host != nullptr;
  attn_status s = decode_check(q, k_cache, v_cache, out, B, h, n_q, n_max, d_k, d_v,
                               has_lens ? lens : nullptr, scale, inner, inner_bytes);
  if (s != ATTN_OK) return s;
  if (B == 0 || h == 0) return ATTN_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  tsd::HostStage hs(workspace, st);
  hs.copy_in(q, q_host, qb);
  if (has_lens) hs.copy_in(lens, cache_lens_host, size_t(B) * 4);
  if (hs.inputs_ready() != cudaSuccess) return cuda_fail(hs.status());
  s = attn_decode(q, k_cache, v_cache, out, B, h, n_q, n_max, d_k, d_v, has_lens ? lens : nullptr,
                  scale, inner, inner_bytes, stream);
  hs.computed();
  if (s != ATTN_OK) return s;
  const cudaError_t e = async ? hs.copy_out_async(out_host, out, ob) : hs.copy_out(out_host, out, ob);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(hs.status());
}

}  // namespace

extern "C" {

attn_status attn_decode_host(const void* q_host, const void* k_cache, const void* v_cache,
                             void* out_host, int B, int h, int n_q, int n_max, int d_k, int d_v,
                             const int32_t* cache_lens_host, float scale, void* workspace,
                             size_t workspace_bytes, tsd_stream_t stream) {
  return decode_host_call(q_host, k_cache, v_cache, out_host, B, h, n_q, n_max, d_k, d_v,
                          cache_lens_host, scale, workspace, workspace_bytes, stream, false);
}

attn_status attn_decode_host_async(const void* q_host, const void* k_cache, const void* v_cache,
                                   void* out_host, int B, int h, int n_q, int n_max, int d_k,
                                   int d_v, const int32_t* cache_lens_host, float scale,
                                   void* workspace, size_t workspace_bytes, tsd_stream_t stream) {
  return decode_host_call(q_host, k_cache, v_cache, out_host, B, h, n_q, n_max, d_k, d_v,
                          cache_lens_host, scale, workspace, workspace_bytes, stream, true);
}

}  // extern "C"
