// fa_internal.h -- definitions shared by the host library and the kernels.
#pragma once
#include <cstdint>
#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// A bounded device-side wait gives up after this many nanoseconds.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

constexpr int kTile = 128;       // query rows (and key rows) per tile

struct Strides { int64_t b, h, n; };

struct DropoutArgs {
  uint32_t k0, k1;         // Philox key = (lo32(seed), hi32(seed))
  uint32_t rk0[10], rk1[10];  // the key of each of the ten rounds: k + r * (Weyl constant), mod 2^32
  uint32_t off_lo, off_hi; // counter words 2, 3
  uint32_t threshold;      // keep iff 16-bit slice >= threshold
  float rp;                // 1 / (1 - p)
  int enabled;
};

struct MaskArgs {
  int causal;
  int window;                 // sliding window w (causal only), 0 = none
  const int32_t* seqlens_k;   // device [B] or nullptr
  const int16_t* row_list;    // [nb][nb]: kept kv tiles of each q tile, ascending
  const int32_t* row_cnt;     // [nb]
  const int16_t* col_list;    // [nb][nb]: q tiles that keep each kv tile, ascending
  const int32_t* col_cnt;     // [nb]
  int nb;                     // tiles per side (0 when dense)
};

// FP8 forward: per-tile scales of the quantised operands and the rotation.
struct Fp8Args {
  const float* sq;            // [B*H][nt]: dequantisation scale of each 128-row Q tile
  const float* sk;            // [B*H_kv][nt]
  const float* sv;            // [B*H_kv][nt]
  const int8_t* signs;        // [d] signs of the rotation, or nullptr (no rotation)
  int nt;                     // tiles per head, ceil(N / 128)
  int o_bf16;                 // O is stored as bfloat16 (else float16)
};

struct FwdArgs {
  int B, H, N;
  int group;                  // query heads per K/V head (H / H_kv)
  int nq;                     // ceil(N / 128)
  int npairs;                 // ceil(nq / 2)
  float scale_log2;           // tau * log2(e)
  MaskArgs mask;
  DropoutArgs drop;
  float* lse;                 // [B,H,N]
  float* o_f32;               // optional [B,H,N,64]
  int* status;
  Fp8Args f8;                 // FP8 forward only
  int fwd_kernel;             // head dim 64: 0 = library's choice, 1 = one query tile per CTA, 2 = two
};

// Quantiser of the FP8 forward: Q, K and V rows (optionally rotated) to E4M3
// with one scale per 128-row tile (or per tensor).
struct Fp8QuantArgs {
  const void* src[3];         // Q [B,H,N,d], K and V [B,H_kv,N,d], 16-bit
  Strides st[3];              // element strides of each source
  int heads[3];               // H, H_kv, H_kv
  uint8_t* dst[3];            // Q8 [B,H,N,d], K8 [B,H_kv,N,d], V8^T [B,H_kv,d,npad]
  float* scale[3];            // [B*heads][nt]
  float* amax;                // [3] per-tensor maxima (scratch of the per-tensor mode)
  const int8_t* signs;        // [d] or nullptr
  int B, N, nt, npad;
  int d;                      // head dimension, 64 or 128
};

struct BwdArgs {
  int B, H, N;
  int group;                  // query heads per K/V head (H / H_kv)
  int H_kv;
  int nq;                     // ceil(N / 128)
  int npad;                   // nq * 128
  float scale;                // tau
  float scale_log2;           // tau * log2(e)
  MaskArgs mask;
  DropoutArgs drop;
  const float* lse2;          // [B*H][npad]: LSE*log2(e), +inf for rows without keys / padding
  const float* dvec;          // [B*H][npad]: D = rowsum(dO o O) (bf16: -tau * D), 0 on padding
  void* dk;                   // [B,H_kv,N,64] outputs, element strides kst
  void* dv;
  Strides kst;
  int dkv_v8;                 // dk, dv and kst allow 32-byte stores
  int* sched;                 // work-item counter of the persistent kernel (zeroed by the prepass)
  int* status;
};

// ---------------------------------------------------------------------------
// Launchers (defined in the .cu files; all enqueue on `stream`).
// ---------------------------------------------------------------------------
// d: head dimension, 64 or 128
cudaError_t launch_fwd_tc(int dtype, int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& o, const FwdArgs& a, cudaStream_t s);
// Head dimension 64: one query tile per CTA, two CTAs per SM.
cudaError_t launch_fwd_tc1(int dtype, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& o, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_tc(int dtype, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& dout, const CUtensorMap& dqacc, const BwdArgs& a, cudaStream_t s);
// Head dimension 128 (Q, dO and the dQ accumulator maps have 64-row boxes).
cudaError_t launch_bwd_tc128(int dtype, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const CUtensorMap& dout, const CUtensorMap& dqacc, const BwdArgs& a, cudaStream_t s);

// st: strides of Q, O, dO, dQ ([B,H,N,d]); kst: strides of K, V, dK, dV ([B,H_kv,N,d]).
cudaError_t launch_fwd_simt(const float* q, const float* k, const float* v, float* o, Strides st,
                            Strides kst, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_simt(const float* q, const float* k, const float* v, const float* dout,
                            float* dq, float* dk, float* dv, Strides st, Strides kst, const BwdArgs& a,
                            cudaStream_t s);

// D = rowsum(dO o O) and the padded LSE*log2e / D arrays; the same pass clears dqacc if given.
// dvec = dscale * D (the bf16 backward kernels fold -tau into it, see fa_bwd).
cudaError_t launch_bwd_prep(int dtype, const void* o, const void* dout, Strides st, const float* lse,
                            int B, int H, int N, int npad, int d, float* lse2, float* dvec, float* dqacc,
                            int* sched, float dscale, cudaStream_t s);
// dq = dqacc (already scaled) cast to dtype with strides.
cudaError_t launch_dq_convert(int dtype, const float* dqacc, void* dq, Strides st, int B, int H, int N, int d,
                              cudaStream_t s);
// Row / column block lists of a dense [nb][nb] uint8 block mask.
cudaError_t launch_block_lists(const uint8_t* mask, int nb, int16_t* row_list, int32_t* row_cnt,
                               int16_t* col_list, int32_t* col_cnt, cudaStream_t s);
cudaError_t launch_dropout_mask(const DropoutArgs& d, int H, int N, int b, int h, int row0, int nrows,
                                uint8_t* out, cudaStream_t s);
// FP8 forward: quantise Q, K, V (per_tensor selects one scale per tensor),
// then the attention forward on the quantised operands (head dimension d = 64 or 128).
cudaError_t launch_fp8_quantize(int dtype, const Fp8QuantArgs& a, int per_tensor, cudaStream_t s);
cudaError_t launch_fwd_fp8(int d, const CUtensorMap& q8, const CUtensorMap& k8, const CUtensorMap& v8t,
                           const CUtensorMap& o, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_wait_selftest(int* status, int* out, unsigned long long* out_ns, cudaStream_t s);

}  // namespace fa
