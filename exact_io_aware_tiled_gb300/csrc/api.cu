// api.cu -- host side of the C ABI declared in include/fa.h.
//
// Validates arguments, lays out the caller's workspace, encodes the TMA
// tensor maps (cuTensorMapEncodeTiled, fetched through the runtime's
// driver-entry-point query so the library needs no -lcuda), and enqueues the
// kernels on the caller's stream.  It never allocates, frees or synchronises
// device memory (fa_check_status excepted) and keeps no mutable global state.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
  size_t status = 0, rlist = 0, rcnt = 0, clist = 0, ccnt = 0, lse2 = 0, dvec = 0, dqacc = 0, sched = 0, total = 0;
  bool sparse = false;
  int nb = 0, nq = 0, npad = 0;
};

Layout layout(const fa_params* p, bool bwd) {
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  L.nq = (p->N + kTile - 1) / kTile;
  L.npad = L.nq * kTile;
  L.status = take(256);
  if (p->block_mask != nullptr) {
    L.sparse = true;
    L.nb = L.nq;
    L.rlist = take((size_t)L.nb * L.nb * sizeof(int16_t));
    L.rcnt = take((size_t)L.nb * sizeof(int32_t));
    L.clist = take((size_t)L.nb * L.nb * sizeof(int16_t));
    L.ccnt = take((size_t)L.nb * sizeof(int32_t));
  }
  if (bwd) {
    const size_t rows = (size_t)p->B * p->H * L.npad;
    L.lse2 = take(rows * sizeof(float));
    L.dvec = take(rows * sizeof(float));
    if (p->dtype != FA_DT_F32) L.dqacc = take((size_t)p->B * p->H * p->N * p->d * sizeof(float));
    L.sched = take(sizeof(int));
  }
  L.total = off;
  return L;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

int elem_bytes(int dt) { return dt == FA_DT_F32 ? 4 : 2; }

int hkv_of(const fa_params* p) { return p->H_kv == 0 ? p->H : p->H_kv; }

bool kv_strides_given(const fa_params* p) { return p->kv_stride_b || p->kv_stride_h || p->kv_stride_n; }

// Shape / dtype / stride / alignment checks shared by fa_fwd and fa_bwd.
fa_status check_params(const fa_params* p) {
  if (p == nullptr) return FA_ERR_INVALID_ARG;
  if (p->B < 1 || p->H < 1 || p->N < 1 || p->d < 1) return FA_ERR_INVALID_ARG;
  if (p->dtype != FA_DT_F32 && p->dtype != FA_DT_F16 && p->dtype != FA_DT_BF16) return FA_ERR_INVALID_ARG;
  // d = 64 on every path; d = 128 on the 16-bit tensor-core forward
  if (p->d != 64 && !(p->d == 128 && p->dtype != FA_DT_F32)) return FA_ERR_UNSUPPORTED;
  if (p->stride_n < p->d || p->stride_h < 1 || p->stride_b < 1) return FA_ERR_INVALID_ARG;
  if (!(p->dropout_p >= 0.f && p->dropout_p < 1.f)) return FA_ERR_INVALID_ARG;
  if ((long long)p->B * p->H * p->N >= (1ll << 32)) return FA_ERR_UNSUPPORTED;
  if (p->block_mask != nullptr && p->block_size != kTile) return FA_ERR_UNSUPPORTED;
  if (p->block_mask != nullptr && (p->N + kTile - 1) / kTile > 32767) return FA_ERR_UNSUPPORTED;
  const int64_t unit = 16 / elem_bytes(p->dtype);   // elements per 16 bytes
  if (p->stride_n % unit || p->stride_h % unit || p->stride_b % unit) return FA_ERR_MISALIGNED;
  if (p->o_f32 != nullptr && !aligned16(p->o_f32)) return FA_ERR_MISALIGNED;
  const int hkv = hkv_of(p);
  if (hkv < 1 || p->H % hkv != 0) return FA_ERR_INVALID_ARG;
  if (kv_strides_given(p)) {
    if (p->kv_stride_n < p->d || p->kv_stride_h < 1 || p->kv_stride_b < 1) return FA_ERR_INVALID_ARG;
    if (p->kv_stride_n % unit || p->kv_stride_h % unit || p->kv_stride_b % unit) return FA_ERR_MISALIGNED;
  } else if (hkv != p->H) {
    return FA_ERR_INVALID_ARG;   // K/V with fewer heads need their own strides
  }
  if (p->window < 0) return FA_ERR_INVALID_ARG;
  if (p->window > 0 && !p->causal) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Singleton dimensions carry whatever stride the caller had; normalise them
// so every stride handed to TMA is a valid, representable byte stride.
Strides normalised(Strides s, const fa_params* p, int heads) {
  if (heads == 1) s.h = (int64_t)p->N * s.n;
  if (p->B == 1) s.b = (int64_t)heads * s.h;
  return s;
}

// Strides of Q, O, dO, dQ ([B,H,N,d]).
Strides strides_of(const fa_params* p) { return normalised({p->stride_b, p->stride_h, p->stride_n}, p, p->H); }

// Strides of K, V, dK, dV ([B,H_kv,N,d]).
Strides kv_strides_of(const fa_params* p) {
  if (!kv_strides_given(p)) return strides_of(p);
  return normalised({p->kv_stride_b, p->kv_stride_h, p->kv_stride_n}, p, hkv_of(p));
}

float scale_of(const fa_params* p) {
  return (p->scale > 0.f && std::isfinite(p->scale)) ? p->scale : 1.f / std::sqrt((float)p->d);
}

DropoutArgs dropout_of(const fa_params* p) {
  DropoutArgs d{};
  d.k0 = (uint32_t)(p->seed & 0xFFFFFFFFu);
  d.k1 = (uint32_t)(p->seed >> 32);
  // Philox4x32 key schedule (Salmon et al., SC'11): the key is bumped by the
  // Weyl constants before every round after the first.  It depends on the
  // seed only, so it is computed once here and the kernels read each round's
  // key as a constant.
  for (int r = 0; r < 10; ++r) {
    d.rk0[r] = d.k0 + (uint32_t)r * 0x9E3779B9u;
    d.rk1[r] = d.k1 + (uint32_t)r * 0xBB67AE85u;
  }
  d.off_lo = (uint32_t)(p->offset & 0xFFFFFFFFu);
  d.off_hi = (uint32_t)(p->offset >> 32);
  const double t = std::floor((double)p->dropout_p * 65536.0 + 0.5);
  d.threshold = (uint32_t)t;
  d.rp = 1.f / (1.f - p->dropout_p);
  d.enabled = p->dropout_p > 0.f ? 1 : 0;
  return d;
}

// 4-D map over a [B,heads,N,cols] tensor: dims (cols, N, heads, B), box (box_c, box_r, 1, 1), 128-byte swizzle.
fa_status make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int cols, int box_c,
                   const fa_params* p, int heads, Strides s, int box_r = kTile) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return FA_ERR_CUDA;
  cuuint64_t dims[4] = {(cuuint64_t)cols, (cuuint64_t)p->N, (cuuint64_t)heads, (cuuint64_t)p->B};
  cuuint64_t strides[3] = {(cuuint64_t)(s.n * esize), (cuuint64_t)(s.h * esize), (cuuint64_t)(s.b * esize)};
  cuuint32_t box[4] = {(cuuint32_t)box_c, (cuuint32_t)box_r, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

fa_status map16(CUtensorMap* m, const void* base, const fa_params* p, int heads, Strides s, int rows = kTile) {
  const CUtensorMapDataType dt =
      p->dtype == FA_DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return make_map(m, base, dt, 2, p->d, 64, p, heads, s, rows);   // 64-column (128-byte) boxes
}

MaskArgs mask_of(const fa_params* p, const Layout& L, uint8_t* ws) {
  MaskArgs m{};
  m.causal = p->causal ? 1 : 0;
  m.window = p->window;
  m.seqlens_k = p->seqlens_k;
  if (L.sparse) {
    m.row_list = reinterpret_cast<const int16_t*>(ws + L.rlist);
    m.row_cnt = reinterpret_cast<const int32_t*>(ws + L.rcnt);
    m.col_list = reinterpret_cast<const int16_t*>(ws + L.clist);
    m.col_cnt = reinterpret_cast<const int32_t*>(ws + L.ccnt);
    m.nb = L.nb;
  }
  return m;
}

fa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

fa_status prepare_common(const fa_params* p, const Layout& L, uint8_t* ws, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(ws + L.status, 0, sizeof(int), st);
  if (e == cudaSuccess && L.sparse)
    e = launch_block_lists(p->block_mask, L.nb, reinterpret_cast<int16_t*>(ws + L.rlist),
                           reinterpret_cast<int32_t*>(ws + L.rcnt), reinterpret_cast<int16_t*>(ws + L.clist),
                           reinterpret_cast<int32_t*>(ws + L.ccnt), st);
  return cuda_status(e);
}

// Records the caller's optional profiling events around the main kernel.
struct ProfScope {
  cudaEvent_t a, b;
  cudaStream_t s;
  ProfScope(const fa_params* p, cudaStream_t st)
      : a((cudaEvent_t)p->prof_start), b((cudaEvent_t)p->prof_stop), s(st) {
    if (a && b) cudaEventRecord(a, s);
  }
  ~ProfScope() {
    if (a && b) cudaEventRecord(b, s);
  }
};

// ---- FP8 forward -------------------------------------------------------------
struct Fp8Layout {
  size_t q8 = 0, k8 = 0, v8t = 0, sq = 0, sk = 0, sv = 0, amax = 0, total = 0;
  int nt = 0, npad = 0;
};

Fp8Layout fp8_layout(const fa_params* p) {
  Fp8Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  const int hkv = hkv_of(p);
  L.nt = (p->N + kTile - 1) / kTile;
  L.npad = L.nt * kTile;
  const size_t rq = (size_t)p->B * p->H, rk = (size_t)p->B * hkv;
  L.q8 = take(rq * p->N * p->d);
  L.k8 = take(rk * p->N * p->d);
  L.v8t = take(rk * p->d * L.npad);
  L.sq = take(rq * L.nt * sizeof(float));
  L.sk = take(rk * L.nt * sizeof(float));
  L.sv = take(rk * L.nt * sizeof(float));
  L.amax = take(4 * sizeof(float));
  L.total = off;
  return L;
}

// What the FP8 path supports on top of check_params.
fa_status check_fp8(const fa_params* p, const fa_fp8_params* f) {
  fa_status s = check_params(p);
  if (s != FA_OK) return s;
  if (f == nullptr) return FA_ERR_INVALID_ARG;
  if (p->dtype == FA_DT_F32 || (p->d != 64 && p->d != 128) || p->dropout_p > 0.f) return FA_ERR_UNSUPPORTED;
  if (f->per_tensor != 0 && f->per_tensor != 1) return FA_ERR_INVALID_ARG;
  if (f->signs != nullptr && !aligned16(f->signs)) return FA_ERR_MISALIGNED;
  return FA_OK;
}

// 4-D byte map: dims (d0, d1, d2, d3), byte strides of dims 1-3, box (b0, b1, 1, 1).
fa_status map_u8(CUtensorMap* m, const void* base, const cuuint64_t (&dims)[4], const cuuint64_t (&strides)[3],
                 cuuint32_t b0, cuuint32_t b1, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return FA_ERR_CUDA;
  cuuint32_t box[4] = {b0, b1, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

size_t fa_fwd_workspace_size(const fa_params* p) {
  if (p == nullptr || p->N < 1) return 256;
  return layout(p, false).total;
}

size_t fa_bwd_workspace_size(const fa_params* p) {
  if (p == nullptr || p->N < 1 || p->B < 1 || p->H < 1) return 256;
  return layout(p, true).total;
}

fa_status fa_fwd(const fa_params* p, const void* q, const void* k, const void* v, void* o, float* lse, void* ws,
                 size_t ws_bytes, void* stream) {
  fa_status s = check_params(p);
  if (s != FA_OK) return s;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_MISALIGNED;
  const Layout L = layout(p, false);
  if (ws == nullptr || ws_bytes < L.total || !aligned16(ws)) return FA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const Strides sd = strides_of(p), skv = kv_strides_of(p);
  const int hkv = hkv_of(p);

  FwdArgs a{};
  a.B = p->B; a.H = p->H; a.N = p->N;
  a.group = p->H / hkv;
  a.nq = L.nq;
  a.npairs = (L.nq + 1) / 2;
  a.scale_log2 = scale_of(p) * 1.4426950408889634f;
  a.mask = mask_of(p, L, w);
  a.drop = dropout_of(p);
  a.fwd_kernel = p->fwd_kernel;
  a.lse = lse;
  a.o_f32 = p->o_f32;
  a.status = reinterpret_cast<int*>(w + L.status);

  if ((s = prepare_common(p, L, w, st)) != FA_OK) return s;
  if (p->dtype == FA_DT_F32) {
    if (p->o_f32 != nullptr) return FA_ERR_UNSUPPORTED;   // O is already float32
    ProfScope prof(p, st);
    return cuda_status(
        launch_fwd_simt((const float*)q, (const float*)k, (const float*)v, (float*)o, sd, skv, a, st));
  }
  CUtensorMap mq, mk, mv, mo;
  if ((s = map16(&mq, q, p, p->H, sd)) != FA_OK || (s = map16(&mk, k, p, hkv, skv)) != FA_OK ||
      (s = map16(&mv, v, p, hkv, skv)) != FA_OK || (s = map16(&mo, o, p, p->H, sd)) != FA_OK)
    return s;
  ProfScope prof(p, st);
  return cuda_status(launch_fwd_tc(p->dtype, p->d, mq, mk, mv, mo, a, st));
}

fa_status fa_bwd(const fa_params* p, const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream) {
  fa_status s = check_params(p);
  if (s != FA_OK) return s;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  const Layout L = layout(p, true);
  if (ws == nullptr || ws_bytes < L.total || !aligned16(ws)) return FA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const Strides sd = strides_of(p), skv = kv_strides_of(p);
  const int hkv = hkv_of(p);

  BwdArgs a{};
  a.B = p->B; a.H = p->H; a.N = p->N;
  a.group = p->H / hkv;
  a.H_kv = hkv;
  a.nq = L.nq;
  a.npad = L.npad;
  a.scale = scale_of(p);
  a.scale_log2 = a.scale * 1.4426950408889634f;
  a.mask = mask_of(p, L, w);
  a.drop = dropout_of(p);
  a.lse2 = reinterpret_cast<const float*>(w + L.lse2);
  a.dvec = reinterpret_cast<const float*>(w + L.dvec);
  a.status = reinterpret_cast<int*>(w + L.status);

  if ((s = prepare_common(p, L, w, st)) != FA_OK) return s;
  float* dqacc = p->dtype == FA_DT_F32 ? nullptr : reinterpret_cast<float*>(w + L.dqacc);
  a.sched = reinterpret_cast<int*>(w + L.sched);
  // The bf16 backward kernels fold tau into dS (dS' = (tau dP - tau D) o P
  // with one packed FMA against -tau D), so their dQ, dK products come out
  // scaled; the fp16 and fp32 kernels read D itself.
  const float dscale = p->dtype == FA_DT_BF16 ? -a.scale : 1.f;
  cudaError_t e = launch_bwd_prep(p->dtype, o, dout, sd, lse, p->B, p->H, p->N, L.npad, p->d,
                                  reinterpret_cast<float*>(w + L.lse2), reinterpret_cast<float*>(w + L.dvec), dqacc,
                                  a.sched, dscale, st);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if (p->dtype == FA_DT_F32) {
    ProfScope prof(p, st);
    return cuda_status(launch_bwd_simt((const float*)q, (const float*)k, (const float*)v, (const float*)dout,
                                       (float*)dq, (float*)dk, (float*)dv, sd, skv, a, st));
  }
  // d = 64: 128-row query steps; d = 128: 64-row query steps (Q, dO and the
  // float32 dQ accumulator are moved in 64-row boxes)
  CUtensorMap mq, mk, mv, mdo, macc;
  const int qrows = p->d == 128 ? 64 : kTile;
  Strides acc_st{(int64_t)p->H * p->N * p->d, (int64_t)p->N * p->d, p->d};
  if ((s = map16(&mq, q, p, p->H, sd, qrows)) != FA_OK || (s = map16(&mk, k, p, hkv, skv)) != FA_OK ||
      (s = map16(&mv, v, p, hkv, skv)) != FA_OK || (s = map16(&mdo, dout, p, p->H, sd, qrows)) != FA_OK ||
      (s = make_map(&macc, dqacc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p->d, 32, p, p->H, acc_st, qrows)) != FA_OK)
    return s;
  a.dk = dk;
  a.dv = dv;
  a.kst = skv;
  // 32-byte row pieces (16 columns of 16 bits) can go out as single 32-byte stores
  a.dkv_v8 = ((reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 31u) == 0 &&
             skv.n % 16 == 0 && skv.h % 16 == 0 && skv.b % 16 == 0;
  {
    ProfScope prof(p, st);
    e = p->d == 128 ? launch_bwd_tc128(p->dtype, mq, mk, mv, mdo, macc, a, st)
                    : launch_bwd_tc(p->dtype, mq, mk, mv, mdo, macc, a, st);
    if (e != cudaSuccess) return FA_ERR_CUDA;
  }
  return cuda_status(launch_dq_convert(p->dtype, dqacc, dq, sd, p->B, p->H, p->N, p->d, st));
}

fa_status fa_check_status(const void* ws, void* stream) {
  if (ws == nullptr) return FA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  return v == 0 ? FA_OK : (fa_status)v;
}

fa_status fa_dropout_mask(const fa_params* p, int32_t b, int32_t h, int32_t row0, int32_t nrows, uint8_t* out,
                          void* stream) {
  if (p == nullptr || out == nullptr) return FA_ERR_INVALID_ARG;
  if (p->B < 1 || p->H < 1 || p->N < 1) return FA_ERR_INVALID_ARG;
  if (!(p->dropout_p >= 0.f && p->dropout_p < 1.f)) return FA_ERR_INVALID_ARG;
  if (b < 0 || b >= p->B || h < 0 || h >= p->H || row0 < 0 || nrows < 0 || row0 + (int64_t)nrows > p->N)
    return FA_ERR_INVALID_ARG;
  if ((long long)p->B * p->H * p->N >= (1ll << 32)) return FA_ERR_UNSUPPORTED;
  return cuda_status(launch_dropout_mask(dropout_of(p), p->H, p->N, b, h, row0, nrows, out,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

fa_status fa_selftest_wait_timeout(void* ws, int32_t* out, uint64_t* out_ns, void* stream) {
  if (ws == nullptr || out == nullptr || out_ns == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned16(ws) || (reinterpret_cast<uintptr_t>(out_ns) & 7u) != 0) return FA_ERR_MISALIGNED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int), st);
  if (e == cudaSuccess)
    e = launch_wait_selftest(static_cast<int*>(ws), reinterpret_cast<int*>(out),
                             reinterpret_cast<unsigned long long*>(out_ns), st);
  return cuda_status(e);
}

fa_status fa_fp8_buffer_layout(const fa_params* p, fa_fp8_layout* out) {
  if (p == nullptr || out == nullptr || p->B < 1 || p->H < 1 || p->N < 1 || p->d < 1) return FA_ERR_INVALID_ARG;
  const int hkv = hkv_of(p);
  if (hkv < 1 || p->H % hkv != 0) return FA_ERR_INVALID_ARG;
  const Fp8Layout L = fp8_layout(p);
  out->q8 = L.q8; out->k8 = L.k8; out->v8t = L.v8t;
  out->sq = L.sq; out->sk = L.sk; out->sv = L.sv; out->amax = L.amax;
  out->total = L.total;
  return FA_OK;
}

fa_status fa_fp8_quantize(const fa_params* p, const fa_fp8_params* f, const void* q, const void* k, const void* v,
                          void* buf, size_t buf_bytes, void* stream) {
  fa_status s = check_fp8(p, f);
  if (s != FA_OK) return s;
  if (!q || !k || !v) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return FA_ERR_MISALIGNED;
  const Fp8Layout L = fp8_layout(p);
  if (buf == nullptr || buf_bytes < L.total || !aligned16(buf)) return FA_ERR_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(buf);
  const int hkv = hkv_of(p);
  Fp8QuantArgs a{};
  a.src[0] = q; a.src[1] = k; a.src[2] = v;
  a.st[0] = strides_of(p); a.st[1] = a.st[2] = kv_strides_of(p);
  a.heads[0] = p->H; a.heads[1] = a.heads[2] = hkv;
  a.dst[0] = w + L.q8; a.dst[1] = w + L.k8; a.dst[2] = w + L.v8t;
  a.scale[0] = reinterpret_cast<float*>(w + L.sq);
  a.scale[1] = reinterpret_cast<float*>(w + L.sk);
  a.scale[2] = reinterpret_cast<float*>(w + L.sv);
  a.amax = reinterpret_cast<float*>(w + L.amax);
  a.signs = f->signs;
  a.B = p->B; a.N = p->N; a.nt = L.nt; a.npad = L.npad;
  a.d = p->d;
  return cuda_status(launch_fp8_quantize(p->dtype, a, f->per_tensor, reinterpret_cast<cudaStream_t>(stream)));
}

fa_status fa_fwd_fp8(const fa_params* p, const fa_fp8_params* f, const void* buf, size_t buf_bytes, void* o,
                     float* lse, void* ws, size_t ws_bytes, void* stream) {
  fa_status s = check_fp8(p, f);
  if (s != FA_OK) return s;
  if (!o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(lse)) return FA_ERR_MISALIGNED;
  const Fp8Layout Q = fp8_layout(p);
  if (buf == nullptr || buf_bytes < Q.total || !aligned16(buf)) return FA_ERR_WORKSPACE;
  const Layout L = layout(p, false);
  if (ws == nullptr || ws_bytes < L.total || !aligned16(ws)) return FA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const uint8_t* qb = static_cast<const uint8_t*>(buf);
  const int hkv = hkv_of(p);

  FwdArgs a{};
  a.B = p->B; a.H = p->H; a.N = p->N;
  a.group = p->H / hkv;
  a.nq = L.nq;
  a.npairs = (L.nq + 1) / 2;
  a.scale_log2 = scale_of(p) * 1.4426950408889634f;
  a.mask = mask_of(p, L, w);
  a.drop = dropout_of(p);
  a.lse = lse;
  a.o_f32 = p->o_f32;
  a.status = reinterpret_cast<int*>(w + L.status);
  a.f8.sq = reinterpret_cast<const float*>(qb + Q.sq);
  a.f8.sk = reinterpret_cast<const float*>(qb + Q.sk);
  a.f8.sv = reinterpret_cast<const float*>(qb + Q.sv);
  a.f8.signs = f->signs;
  a.f8.nt = Q.nt;
  a.f8.o_bf16 = p->dtype == FA_DT_BF16 ? 1 : 0;

  const cuuint64_t N = (cuuint64_t)p->N, npad = (cuuint64_t)Q.npad, H = (cuuint64_t)p->H, Hk = (cuuint64_t)hkv;
  const cuuint64_t d = (cuuint64_t)p->d;
  // Q8 / K8 rows are d bytes: 64-byte swizzle for d = 64, 128-byte for d = 128
  const CUtensorMapSwizzle swqk = p->d == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap mq, mk, mv, mo;
  if ((s = map_u8(&mq, qb + Q.q8, {d, N, H, (cuuint64_t)p->B}, {d, d * N, d * N * H}, (cuuint32_t)d, kTile, swqk)) !=
          FA_OK ||
      (s = map_u8(&mk, qb + Q.k8, {d, N, Hk, (cuuint64_t)p->B}, {d, d * N, d * N * Hk}, (cuuint32_t)d, kTile, swqk)) !=
          FA_OK ||
      (s = map_u8(&mv, qb + Q.v8t, {npad, d, Hk, (cuuint64_t)p->B}, {npad, d * npad, d * npad * Hk}, kTile,
                  (cuuint32_t)d, CU_TENSOR_MAP_SWIZZLE_128B)) != FA_OK ||
      (s = map16(&mo, o, p, p->H, strides_of(p))) != FA_OK)
    return s;
  if ((s = prepare_common(p, L, w, st)) != FA_OK) return s;
  ProfScope prof(p, st);
  return cuda_status(launch_fwd_fp8(p->d, mq, mk, mv, mo, a, st));
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

int32_t fa_version(void) { return 103; }

}  // extern "C"
