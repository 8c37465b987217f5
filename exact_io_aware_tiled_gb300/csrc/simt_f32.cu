// simt_f32.cu -- float32 attention forward / backward on CUDA cores.
//
// The float32 path must agree with the float64 definition to ~1e-5, which
// tensor-core float32 formats (tf32, 10-bit mantissa) cannot reach, so these
// kernels use plain FFMA.  They implement the same method as the tensor-core
// kernels: forward = Q-outer tiles with the online-softmax recurrence
// (lynx-cortex, "El algoritmo Flash (forward)"); backward = recomputation of
// P from the saved logsumexp, D = rowsum(dO o O) (tonho.wtf, "como
// funciona"), with the same masks, block lists and Philox dropout mapping.
// Head dimension 64; one thread per query row (forward, dQ) or key row
// (dK, dV); K/V or Q/dO sub-tiles of 32 rows staged in shared memory.
// Grouped-query heads read K/V head h / g, and a dK/dV block sums over the g
// query heads of its K/V head; the sliding window bounds both tile lists and
// masks inside the boundary tiles.
#include "common.cuh"

namespace fa {
namespace {

constexpr int kRows = 128;   // rows per block
constexpr int kSub = 32;     // staged rows per sub-tile
constexpr int kD = 64;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ int kv_limit_tiles(int Lk) { return (Lk + kTile - 1) / kTile; }

// Number of 128-row tiles on the other side visible from tile `t`, and the
// tile at position s of that list.
struct TileList {
  int n;
  int first;
  const int16_t* list;
  __device__ __forceinline__ int at(int s) const { return list ? (int)list[s] : first + s; }
};

__device__ __forceinline__ TileList fwd_list(const MaskArgs& m, int qt, int Lk) {
  TileList tl{0, 0, nullptr};
  int lim = kv_limit_tiles(Lk);
  if (m.causal) lim = min(lim, qt + 1);
  const int lo = m.window > 0 ? max(0, qt * kTile - m.window + 1) / kTile : 0;
  if (m.row_list) {
    const int16_t* list = m.row_list + (size_t)qt * m.nb;
    const int cnt = m.row_cnt[qt];
    int s0 = 0;
    while (s0 < cnt && list[s0] < lo) ++s0;
    int n = s0;
    while (n < cnt && list[n] < lim) ++n;
    tl.list = list + s0;
    tl.n = n - s0;
  } else {
    tl.first = lo;
    tl.n = max(0, lim - lo);
  }
  return tl;
}

__device__ __forceinline__ TileList bwd_list(const MaskArgs& m, int jt, int nq, int Lk) {
  TileList tl{0, 0, nullptr};
  if (jt * kTile >= Lk) return tl;
  int qlast = nq - 1;   // key j is seen by queries j .. j + w - 1 under a window
  if (m.window > 0) qlast = min(qlast, (jt * kTile + kTile - 1 + m.window - 1) / kTile);
  if (m.col_list) {
    const int16_t* list = m.col_list + (size_t)jt * m.nb;
    const int cnt = m.col_cnt[jt];
    int s0 = 0;
    if (m.causal) while (s0 < cnt && list[s0] < jt) ++s0;
    int e = s0;
    while (e < cnt && list[e] <= qlast) ++e;
    tl.list = list + s0;
    tl.n = e - s0;
  } else {
    tl.first = m.causal ? jt : 0;
    tl.n = max(0, qlast - tl.first + 1);
  }
  return tl;
}

__global__ void __launch_bounds__(kRows)
fwd_simt_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                float* __restrict__ o, Strides st, Strides kst, const FwdArgs a) {
  __shared__ float Ks[kSub][kD];
  __shared__ float Vs[kSub][kD];
  const int qt = blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / a.H, h = bh % a.H;
  const int r = threadIdx.x;
  const int i = qt * kRows + r;
  int Lk = a.N;
  if (a.mask.seqlens_k) Lk = max(0, min(a.N, a.mask.seqlens_k[b]));
  const size_t base = (size_t)b * st.b + (size_t)h * st.h;
  const size_t kbase = (size_t)b * kst.b + (size_t)(h / a.group) * kst.h;
  float qr[kD], acc[kD];
#pragma unroll
  for (int c = 0; c < kD; ++c) {
    qr[c] = i < a.N ? q[base + (size_t)i * st.n + c] : 0.f;
    acc[c] = 0.f;
  }
  const int jmax = a.mask.causal ? min(Lk - 1, i) : Lk - 1;
  const int jmin = a.mask.window > 0 ? i - a.mask.window + 1 : 0;
  const float sl2 = a.scale_log2;
  const uint32_t row_g = (uint32_t)bh * (uint32_t)a.N + (uint32_t)i;
  float m = -INFINITY, l = 0.f;
  const TileList tl = fwd_list(a.mask, qt, Lk);
  for (int s = 0; s < tl.n; ++s) {
    const int kvt = tl.at(s);
    for (int sub = 0; sub < kTile / kSub; ++sub) {
      const int j0 = kvt * kTile + sub * kSub;
      __syncthreads();
      for (int e = r; e < kSub * kD; e += kRows) {
        const int jj = j0 + e / kD, c = e % kD;
        Ks[e / kD][c] = jj < a.N ? k[kbase + (size_t)jj * kst.n + c] : 0.f;
        Vs[e / kD][c] = jj < a.N ? v[kbase + (size_t)jj * kst.n + c] : 0.f;
      }
      __syncthreads();
      float sc[kSub];
      float mx = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < kSub; ++jj) {
        float d = 0.f;
#pragma unroll
        for (int c = 0; c < kD; ++c) d = fmaf(qr[c], Ks[jj][c], d);
        sc[jj] = (j0 + jj <= jmax && j0 + jj >= jmin) ? d * sl2 : -INFINITY;
        mx = fmaxf(mx, sc[jj]);
      }
      const float mn = fmaxf(m, mx);
      const float mref = mn == -INFINITY ? 0.f : mn;
      const float alpha = m == -INFINITY ? 0.f : ex2(m - mref);
      l *= alpha;
#pragma unroll
      for (int c = 0; c < kD; ++c) acc[c] *= alpha;
      uint32_t keep = ~0u;
      if (a.drop.enabled) {
        keep = 0;
#pragma unroll
        for (int g = 0; g < kSub / 8; ++g)
          keep |= dropout_keep8((uint32_t)((j0 >> 3) + g), row_g, a.drop) << (8 * g);
      }
#pragma unroll
      for (int jj = 0; jj < kSub; ++jj) {
        const float p = ex2(sc[jj] - mref);
        l += p;
        const float pt = ((keep >> jj) & 1u) ? p * (a.drop.enabled ? a.drop.rp : 1.f) : 0.f;
#pragma unroll
        for (int c = 0; c < kD; ++c) acc[c] = fmaf(pt, Vs[jj][c], acc[c]);
      }
      m = mn;
    }
  }
  if (i < a.N) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < kD; ++c) o[base + (size_t)i * st.n + c] = acc[c] * inv;
    a.lse[(size_t)bh * a.N + i] = l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
  }
}

// dK, dV: one thread per key row.
__global__ void __launch_bounds__(kRows)
bwd_dkdv_simt_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                     const float* __restrict__ dout, float* __restrict__ dk, float* __restrict__ dv, Strides st,
                     Strides kst, const BwdArgs a) {
  extern __shared__ float dyn_smem[];
  auto KVs = reinterpret_cast<float (*)[kRows][kD + 1]>(dyn_smem);   // [2][kRows][kD + 1]
  __shared__ float Qs[kSub][kD];
  __shared__ float Ds[kSub][kD];
  __shared__ float Ls[kSub], Dv[kSub];
  const int jt = blockIdx.x;
  const int bk = blockIdx.y;                  // (b, K/V head)
  const int b = bk / a.H_kv, hk = bk % a.H_kv;
  const int r = threadIdx.x;
  const int j = jt * kRows + r;
  int Lk = a.N;
  if (a.mask.seqlens_k) Lk = max(0, min(a.N, a.mask.seqlens_k[b]));
  const size_t kbase = (size_t)b * kst.b + (size_t)hk * kst.h;
  for (int c = 0; c < kD; ++c) {
    KVs[0][r][c] = j < a.N ? k[kbase + (size_t)j * kst.n + c] : 0.f;
    KVs[1][r][c] = j < a.N ? v[kbase + (size_t)j * kst.n + c] : 0.f;
  }
  float gk[kD], gv[kD];
#pragma unroll
  for (int c = 0; c < kD; ++c) { gk[c] = 0.f; gv[c] = 0.f; }
  const bool key_ok = j < Lk;
  const TileList tl = bwd_list(a.mask, jt, a.nq, Lk);
  const float rp = a.drop.enabled ? a.drop.rp : 1.f;
  for (int s = 0; s < tl.n * a.group; ++s) {
    const int qti = tl.at(s % tl.n);
    const int h = hk * a.group + s / tl.n;     // query head of this step
    const int bh = b * a.H + h;
    const size_t base = (size_t)b * st.b + (size_t)h * st.h;
    for (int sub = 0; sub < kTile / kSub; ++sub) {
      const int i0 = qti * kTile + sub * kSub;
      __syncthreads();
      for (int e = r; e < kSub * kD; e += kRows) {
        const int ii = i0 + e / kD, c = e % kD;
        Qs[e / kD][c] = ii < a.N ? q[base + (size_t)ii * st.n + c] : 0.f;
        Ds[e / kD][c] = ii < a.N ? dout[base + (size_t)ii * st.n + c] : 0.f;
      }
      if (r < kSub) {
        Ls[r] = a.lse2[(size_t)bh * a.npad + i0 + r];
        Dv[r] = a.dvec[(size_t)bh * a.npad + i0 + r];
      }
      __syncthreads();
      if (!key_ok) continue;
      for (int ii = 0; ii < kSub; ++ii) {
        const int i = i0 + ii;
        if (a.mask.causal && j > i) continue;
        if (a.mask.window > 0 && i >= j + a.mask.window) continue;
        float sdot = 0.f, ddot = 0.f;
#pragma unroll
        for (int c = 0; c < kD; ++c) {
          sdot = fmaf(Qs[ii][c], KVs[0][r][c], sdot);
          ddot = fmaf(Ds[ii][c], KVs[1][r][c], ddot);
        }
        const float p = ex2(fmaf(sdot, a.scale_log2, -Ls[ii]));
        bool kept = true;
        if (a.drop.enabled)
          kept = (dropout_keep8((uint32_t)j >> 3, (uint32_t)bh * (uint32_t)a.N + (uint32_t)i, a.drop) >> (j & 7)) & 1u;
        const float pt = kept ? p * rp : 0.f;
        const float ds = p * ((kept ? ddot * rp : 0.f) - Dv[ii]);
#pragma unroll
        for (int c = 0; c < kD; ++c) {
          gv[c] = fmaf(pt, Ds[ii][c], gv[c]);
          gk[c] = fmaf(ds, Qs[ii][c], gk[c]);
        }
      }
    }
  }
  if (j < a.N) {
#pragma unroll
    for (int c = 0; c < kD; ++c) {
      dk[kbase + (size_t)j * kst.n + c] = gk[c] * a.scale;
      dv[kbase + (size_t)j * kst.n + c] = gv[c];
    }
  }
}

// dQ: one thread per query row.
__global__ void __launch_bounds__(kRows)
bwd_dq_simt_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                   const float* __restrict__ dout, float* __restrict__ dq, Strides st, Strides kst,
                   const BwdArgs a) {
  extern __shared__ float dyn_smem[];
  auto QDs = reinterpret_cast<float (*)[kRows][kD + 1]>(dyn_smem);   // [2][kRows][kD + 1]
  __shared__ float Ks[kSub][kD];
  __shared__ float Vs[kSub][kD];
  const int qt = blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / a.H, h = bh % a.H;
  const int r = threadIdx.x;
  const int i = qt * kRows + r;
  int Lk = a.N;
  if (a.mask.seqlens_k) Lk = max(0, min(a.N, a.mask.seqlens_k[b]));
  const size_t base = (size_t)b * st.b + (size_t)h * st.h;
  for (int c = 0; c < kD; ++c) {
    QDs[0][r][c] = i < a.N ? q[base + (size_t)i * st.n + c] : 0.f;
    QDs[1][r][c] = i < a.N ? dout[base + (size_t)i * st.n + c] : 0.f;
  }
  float g[kD];
#pragma unroll
  for (int c = 0; c < kD; ++c) g[c] = 0.f;
  const size_t kbase = (size_t)b * kst.b + (size_t)(h / a.group) * kst.h;
  const float lse2 = a.lse2[(size_t)bh * a.npad + i];
  const float Di = a.dvec[(size_t)bh * a.npad + i];
  const int jmax = a.mask.causal ? min(Lk - 1, i) : Lk - 1;
  const int jmin = a.mask.window > 0 ? i - a.mask.window + 1 : 0;
  const float rp = a.drop.enabled ? a.drop.rp : 1.f;
  const uint32_t row_g = (uint32_t)bh * (uint32_t)a.N + (uint32_t)i;
  const TileList tl = fwd_list(a.mask, qt, Lk);
  for (int s = 0; s < tl.n; ++s) {
    const int kvt = tl.at(s);
    for (int sub = 0; sub < kTile / kSub; ++sub) {
      const int j0 = kvt * kTile + sub * kSub;
      __syncthreads();
      for (int e = r; e < kSub * kD; e += kRows) {
        const int jj = j0 + e / kD, c = e % kD;
        Ks[e / kD][c] = jj < a.N ? k[kbase + (size_t)jj * kst.n + c] : 0.f;
        Vs[e / kD][c] = jj < a.N ? v[kbase + (size_t)jj * kst.n + c] : 0.f;
      }
      __syncthreads();
      uint32_t keep = ~0u;
      if (a.drop.enabled) {
        keep = 0;
#pragma unroll
        for (int gg = 0; gg < kSub / 8; ++gg)
          keep |= dropout_keep8((uint32_t)((j0 >> 3) + gg), row_g, a.drop) << (8 * gg);
      }
      for (int jj = 0; jj < kSub; ++jj) {
        if (j0 + jj > jmax || j0 + jj < jmin) continue;
        float sdot = 0.f, ddot = 0.f;
#pragma unroll
        for (int c = 0; c < kD; ++c) {
          sdot = fmaf(QDs[0][r][c], Ks[jj][c], sdot);
          ddot = fmaf(QDs[1][r][c], Vs[jj][c], ddot);
        }
        const float p = ex2(fmaf(sdot, a.scale_log2, -lse2));
        const bool kept = (keep >> jj) & 1u;
        const float ds = p * ((kept ? ddot * rp : 0.f) - Di);
#pragma unroll
        for (int c = 0; c < kD; ++c) g[c] = fmaf(ds, Ks[jj][c], g[c]);
      }
    }
  }
  if (i < a.N) {
#pragma unroll
    for (int c = 0; c < kD; ++c) dq[base + (size_t)i * st.n + c] = g[c] * a.scale;
  }
}

}  // namespace

cudaError_t launch_fwd_simt(const float* q, const float* k, const float* v, float* o, Strides st,
                            Strides kst, const FwdArgs& a, cudaStream_t s) {
  dim3 grid(a.nq, a.B * a.H);
  fwd_simt_kernel<<<grid, kRows, 0, s>>>(q, k, v, o, st, kst, a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const float* q, const float* k, const float* v, const float* dout, float* dq,
                            float* dk, float* dv, Strides st, Strides kst, const BwdArgs& a, cudaStream_t s) {
  dim3 grid(a.nq, a.B * a.H), kgrid(a.nq, a.B * a.H_kv);
  constexpr int dyn = 2 * kRows * (kD + 1) * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_dq_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  bwd_dkdv_simt_kernel<<<kgrid, kRows, dyn, s>>>(q, k, v, dout, dk, dv, st, kst, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_dq_simt_kernel<<<grid, kRows, dyn, s>>>(q, k, v, dout, dq, st, kst, a);
  return cudaGetLastError();
}

}  // namespace fa
