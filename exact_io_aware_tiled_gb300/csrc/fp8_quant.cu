// fp8_quant.cu -- quantiser of the FP8 forward (sm_103a).
//
// Method (living-dl-book, "Atencao Eficiente em Escala", section 10;
// marketmaker.cc, "FA3: Mecanica da tremonha", item 3): Q, K and V are
// quantised to FP8 one block (tile) at a time with one scale factor per
// block, after a random Hadamard-style rotation of every row that spreads
// an outlying coordinate over all coordinates.
//
// Readings fixed here (the pages leave them open):
//   * the format is E4M3 (largest finite 448), rounded to nearest even and
//     saturated;
//   * the rotation is M = diag(s) H_D / sqrt(D) with s the caller's random
//     signs (D = 64 or 128);
//     Q, K and V rows are all rotated (the scores are unchanged because M is
//     orthogonal; the forward rotates O back);
//   * a block is 128 rows x D of one head; its scale is amax / 448 and its
//     codes are E4M3(x * (448 / amax)); an all-zero block has scale 0;
//   * the per-tensor variant (the pages' baseline) uses the amax of the
//     whole tensor for every block.
// The codes are integers decided by float32 arithmetic, so the order is
// fixed: sign flip, butterflies (stage h = 1, 2, ..., D/2), multiply by the
// float32 value of 1/sqrt(D) (1/8 exactly for D = 64),
// amax, inv = 448 / amax (correctly rounded), x * inv, E4M3 rounding.
//
// One CTA of 128 threads per block; thread r owns row r.  The block's rows
// are loaded and stored cooperatively (consecutive threads move consecutive
// 16-byte chunks) through shared memory, whose 16-byte chunks are XOR-
// swizzled with the row so that the per-row accesses are free of bank
// conflicts.  Q and K codes are written row-major ([B, heads, N, D] bytes);
// V codes are written transposed ([B, H_kv, D, npad] bytes, keys
// contiguous, zero past N) so that the P V product reads both of its
// operands K-major.
#include "fp8.cuh"

namespace fa {
namespace {

constexpr float kE4M3Max = 448.f;
enum QuantMode { kPerBlock = 0, kAmaxOnly = 1, kPerTensor = 2 };

// 16-byte chunk position of code chunk k of row q in the staging tile (rows
// of D bytes): XOR-swizzled so that a warp's per-row accesses spread over
// all banks
template <int D> __device__ __forceinline__ int swz_code(int k, int q) {
  return D == 64 ? ((k ^ (q >> 1)) & 3) : ((k ^ q) & 7);
}

// float32 value of 1 / sqrt(D): 1/8 exactly, or the rounded 1/sqrt(128)
template <int D> __device__ __forceinline__ float inv_sqrt_d() {
  return D == 64 ? 0.125f : __int_as_float(0x3db504f3);
}

template <typename T, int D, int kMode>
__global__ void __launch_bounds__(128) fp8_quant_kernel(const Fp8QuantArgs a) {
  constexpr int RB = D * 2;          // bytes of a 16-bit row
  constexpr int CH = RB / 16;        // its 16-byte chunks
  __shared__ float red[4];
  // the block's 16-bit rows (128 x RB bytes), later its codes: Q / K rows
  // (128 x D bytes) or the transposed V codes (D x 128 bytes)
  __shared__ __align__(128) uint8_t tile[kTile * RB];

  // tensor x and block (b, head, tile) of this CTA
  int blk = (int)blockIdx.x;
  int x = 0;
  const int n0 = a.B * a.heads[0] * a.nt, n1 = a.B * a.heads[1] * a.nt;
  if (blk >= n0) {
    blk -= n0;
    x = 1;
    if (blk >= n1) {
      blk -= n1;
      x = 2;
    }
  }
  const int t = blk % a.nt;
  const int bh = blk / a.nt;
  const int heads = a.heads[x];
  const int b = bh / heads, h = bh % heads;
  const int r = (int)threadIdx.x;
  const int n = t * kTile + r;
  const Strides st = a.st[x];

  // cooperative load: chunk k (16 bytes) of row q goes to q * RB + (k ^ (q & 7)) * 16
  const T* base = static_cast<const T*>(a.src[x]) + b * st.b + h * st.h;
  const int rows = min(kTile, a.N - t * kTile);
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int idx = r + i * kTile, q = idx / CH, k = idx % CH;
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (q < rows) u = *reinterpret_cast<const uint4*>(base + (int64_t)(t * kTile + q) * st.n + k * 8);
    *reinterpret_cast<uint4*>(tile + q * RB + ((k ^ (q & 7)) << 4)) = u;
  }
  __syncthreads();
  float v[D];
#pragma unroll
  for (int j = 0; j < CH; ++j) {
    const uint4 u = *reinterpret_cast<const uint4*>(tile + r * RB + ((j ^ (r & 7)) << 4));
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[8 * j + 2 * e] = Cvt<T>::lo(w4[e]);
      v[8 * j + 2 * e + 1] = Cvt<T>::hi(w4[e]);
    }
  }
  if (a.signs != nullptr) {
    const uint4* sp = reinterpret_cast<const uint4*>(a.signs);
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      const uint4 u = sp[j];
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int8_t sg = (int8_t)((w4[c >> 2] >> ((c & 3) * 8)) & 0xFFu);
        if (sg < 0) v[16 * j + c] = -v[16 * j + c];
      }
    }
    fwht_rows<D>(v);
    scale_rows<D>(v, inv_sqrt_d<D>());
  }

  // block amax
  float am = 0.f;
#pragma unroll
  for (int c = 0; c < D; ++c) am = fmaxf(am, fabsf(v[c]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  if ((r & 31) == 0) red[r >> 5] = am;
  __syncthreads();
  am = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  // (the barrier above also ends every thread's reads of the 16-bit tile)

  float* sc = a.scale[x] + (size_t)bh * a.nt + t;
  if constexpr (kMode == kAmaxOnly) {
    if (r == 0) *sc = am;
    return;
  }
  if constexpr (kMode == kPerTensor) am = a.amax[x];
  if (r == 0) *sc = __fdiv_rn(am, kE4M3Max);
  const float inv = am > 0.f ? __fdiv_rn(kE4M3Max, am) : 0.f;
  scale_rows<D>(v, inv);
  uint32_t w[D / 4];
#pragma unroll
  for (int j = 0; j < D / 4; ++j) w[j] = e4m3x4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);

  if (x < 2) {
    // codes of row r (D bytes, D / 16 chunks) to swizzled chunk positions,
    // then cooperative stores
    constexpr int CC = D / 16;
#pragma unroll
    for (int j = 0; j < CC; ++j)
      *reinterpret_cast<uint4*>(tile + r * D + (swz_code<D>(j, r) << 4)) =
          make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    __syncthreads();
    uint8_t* dst = a.dst[x] + ((size_t)bh * a.N + (size_t)t * kTile) * D;
#pragma unroll
    for (int i = 0; i < CC; ++i) {
      const int idx = r + i * kTile, q = idx / CC, k = idx % CC;
      if (q < rows)
        *reinterpret_cast<uint4*>(dst + q * D + k * 16) =
            *reinterpret_cast<const uint4*>(tile + q * D + (swz_code<D>(k, q) << 4));
    }
  } else {
    // transpose through shared memory: vt[c][r] = code c of row r.  Keys past
    // N get the code 0 (the rotated zero row can hold -0, code 0x80).
    if (n >= a.N) {
#pragma unroll
      for (int j = 0; j < D / 4; ++j) w[j] = 0u;
    }
#pragma unroll
    for (int c = 0; c < D; ++c) tile[c * kTile + r] = (uint8_t)((w[c >> 2] >> ((c & 3) * 8)) & 0xFFu);
    __syncthreads();
    // D rows of 128 bytes: thread r writes D bytes of row r * D / 128
    const int c = (r * D) / kTile, off = (r * D) % kTile;
    const uint4* src = reinterpret_cast<const uint4*>(tile + c * kTile + off);
    uint4* dst = reinterpret_cast<uint4*>(a.dst[2] + ((size_t)bh * D + c) * a.npad + t * kTile + off);
#pragma unroll
    for (int j = 0; j < D / 16; ++j) dst[j] = src[j];
  }
}

// Per-tensor mode: the largest block amax of each tensor (left in the scale
// slots by the kAmaxOnly pass).
__global__ void __launch_bounds__(256) fp8_amax_reduce_kernel(const Fp8QuantArgs a) {
  __shared__ float red[8];
  const int x = (int)blockIdx.x;
  const int n = a.B * a.heads[x] * a.nt;
  float m = 0.f;
  for (int i = (int)threadIdx.x; i < n; i += 256) m = fmaxf(m, a.scale[x][i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
    a.amax[x] = fmaxf(m, red[0]);
  }
}

template <typename T, int D>
cudaError_t launch_t(const Fp8QuantArgs& a, int per_tensor, cudaStream_t s) {
  const long long nblk = (long long)a.B * (a.heads[0] + a.heads[1] + a.heads[2]) * a.nt;
  if (nblk <= 0) return cudaSuccess;
  if (nblk >= (1ll << 31)) return cudaErrorInvalidValue;
  if (!per_tensor) {
    fp8_quant_kernel<T, D, kPerBlock><<<(unsigned)nblk, 128, 0, s>>>(a);
    return cudaGetLastError();
  }
  fp8_quant_kernel<T, D, kAmaxOnly><<<(unsigned)nblk, 128, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fp8_amax_reduce_kernel<<<3, 256, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fp8_quant_kernel<T, D, kPerTensor><<<(unsigned)nblk, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_quantize(int dtype, const Fp8QuantArgs& a, int per_tensor, cudaStream_t s) {
  if (a.d == 128)
    return dtype == FA_DT_BF16 ? launch_t<__nv_bfloat16, 128>(a, per_tensor, s) : launch_t<__half, 128>(a, per_tensor, s);
  return dtype == FA_DT_BF16 ? launch_t<__nv_bfloat16, 64>(a, per_tensor, s) : launch_t<__half, 64>(a, per_tensor, s);
}

}  // namespace fa
