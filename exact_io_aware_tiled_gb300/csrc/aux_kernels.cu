// aux_kernels.cu -- small HBM-bound kernels around the attention kernels.
//
//   * bwd_prep: D_i = dO_i . O_i (tonho.wtf, "como funciona": the softmax
//     gradient's row term is a length-d dot product instead of a length-N
//     reduction), the logsumexp rescaled to log2 units, both written to
//     128-row-padded arrays the backward kernel bulk-copies per tile;
//   * dq_convert: float32 dQ accumulator -> storage dtype;
//   * block_lists: row / column index lists of a block-sparse mask
//     (agihunt.info, block-sparse paragraph: only nonzero blocks are visited);
//   * dropout_mask: the keep-mask of the Philox mapping, for tests;
//   * wait_selftest: the bounded-wait path of the attention kernels, run on
//     mbarriers that nothing ever arrives at.
#include "common.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Eight threads per query row, each loading 8 consecutive columns (16 B for
// 16-bit inputs) of O and dO; a 3-step shuffle reduces the row.
template <typename T> struct Vec8;
template <> struct Vec8<float> {
  static __device__ __forceinline__ float dot(const float* a, const float* b) {
    const float4 a0 = *reinterpret_cast<const float4*>(a), a1 = *reinterpret_cast<const float4*>(a + 4);
    const float4 b0 = *reinterpret_cast<const float4*>(b), b1 = *reinterpret_cast<const float4*>(b + 4);
    return a0.x * b0.x + a0.y * b0.y + a0.z * b0.z + a0.w * b0.w + a1.x * b1.x + a1.y * b1.y + a1.z * b1.z +
           a1.w * b1.w;
  }
};
template <typename T> struct Vec8 {
  static __device__ __forceinline__ float dot(const T* a, const T* b) {
    const uint4 ua = *reinterpret_cast<const uint4*>(a), ub = *reinterpret_cast<const uint4*>(b);
    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
    float s = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t)
      s += Cvt<T>::lo(wa[t]) * Cvt<T>::lo(wb[t]) + Cvt<T>::hi(wa[t]) * Cvt<T>::hi(wb[t]);
    return s;
  }
};

// Head dimension d (64 or 128): thread `part` of a row takes columns
// part*8 + 64m.  It also clears the float32 dQ accumulator row (when there is
// one): the same threads write the row's d zeros, 32 bytes per 8 columns, so
// the clearing rides on this pass instead of a separate memset.
template <typename T>
__global__ void bwd_prep_kernel(const T* __restrict__ o, const T* __restrict__ dout, Strides st,
                                const float* __restrict__ lse, int B, int H, int N, int npad, int dh,
                                float* __restrict__ lse2, float* __restrict__ dvec, float* __restrict__ dqacc,
                                int* __restrict__ sched, float dscale) {
  if (sched != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *sched = 0;   // backward work counter
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 3;
  const int part = threadIdx.x & 7;
  const long long total = (long long)B * H * npad;
  const bool live = row < total;
  const int bh = live ? (int)(row / npad) : 0;
  const int i = live ? (int)(row % npad) : N;
  float d = 0.f;
  if (live && i < N) {
    const int b = bh / H, h = bh % H;
    const size_t off = (size_t)b * st.b + (size_t)h * st.h + (size_t)i * st.n;
    for (int c = part * 8; c < dh; c += 64) {
      d += Vec8<T>::dot(o + off + c, dout + off + c);
      if (dqacc != nullptr) {
        float4* z = reinterpret_cast<float4*>(dqacc + ((size_t)bh * N + i) * dh + c);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  d += __shfl_xor_sync(0xffffffffu, d, 1);
  d += __shfl_xor_sync(0xffffffffu, d, 2);
  d += __shfl_xor_sync(0xffffffffu, d, 4);
  if (live && part == 0) {
    float l2 = INFINITY;
    if (i < N) {
      const float v = lse[(size_t)bh * N + i];
      l2 = (v == -INFINITY) ? INFINITY : v * kLog2e;
    }
    lse2[row] = l2;
    dvec[row] = i < N ? d * dscale : 0.f;
  }
}

template <typename T>
__global__ void dq_convert_kernel(const float* __restrict__ acc, T* __restrict__ dq, Strides st, int H, int N,
                                  int dh, long long nrows) {
  // 8 consecutive elements per thread; rows of dh (64 or 128) columns
  const long long e = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (e >= nrows * dh) return;
  const long long row = e / dh;
  const int c = (int)(e % dh);
  const int bh = (int)(row / N), i = (int)(row % N);
  const int b = bh / H, h = bh % H;
  const float4 x0 = *reinterpret_cast<const float4*>(acc + e);
  const float4 x1 = *reinterpret_cast<const float4*>(acc + e + 4);
  uint4 w;
  w.x = Cvt<T>::pack(x0.x, x0.y);
  w.y = Cvt<T>::pack(x0.z, x0.w);
  w.z = Cvt<T>::pack(x1.x, x1.y);
  w.w = Cvt<T>::pack(x1.z, x1.w);
  *reinterpret_cast<uint4*>(dq + (size_t)b * st.b + (size_t)h * st.h + (size_t)i * st.n + c) = w;
}

// blockIdx.y == 0: row lists (kept kv tiles of q tile blockIdx.x);
// blockIdx.y == 1: column lists (q tiles keeping kv tile blockIdx.x).
__global__ void block_lists_kernel(const uint8_t* __restrict__ mask, int nb, int16_t* __restrict__ row_list,
                                   int32_t* __restrict__ row_cnt, int16_t* __restrict__ col_list,
                                   int32_t* __restrict__ col_cnt) {
  const int t = blockIdx.x;
  const bool rows = blockIdx.y == 0;
  int16_t* out = (rows ? row_list : col_list) + (size_t)t * nb;
  __shared__ int base;
  if (threadIdx.x == 0) base = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  for (int s0 = 0; s0 < nb; s0 += blockDim.x) {
    const int s = s0 + threadIdx.x;
    const bool keep = s < nb && (rows ? mask[(size_t)t * nb + s] : mask[(size_t)s * nb + t]) != 0;
    // ordered compaction: warp ballot, then warps in order
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    __shared__ int wcount[32];
    if (lane == 0) wcount[threadIdx.x >> 5] = __popc(bal);
    __syncthreads();
    int before = base;
    for (int w = 0; w < (int)(threadIdx.x >> 5); ++w) before += wcount[w];
    if (keep) out[before + __popc(bal & ((1u << lane) - 1u))] = (int16_t)s;
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += wcount[w];
      base += tot;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) (rows ? row_cnt : col_cnt)[t] = base;
}

__global__ void dropout_mask_kernel(DropoutArgs d, int H, int N, int b, int h, int row0, int nrows,
                                    uint8_t* __restrict__ out) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;   // one 8-key group
  const int groups = (N + 7) / 8;
  if (e >= (long long)nrows * groups) return;
  const int r = (int)(e / groups), g = (int)(e % groups);
  const uint32_t row_g = (uint32_t)(b * H + h) * (uint32_t)N + (uint32_t)(row0 + r);
  const uint32_t bits = dropout_keep8((uint32_t)g, row_g, d);
  for (int t = 0; t < 8; ++t) {
    const int j = g * 8 + t;
    if (j < N) out[(size_t)r * N + j] = (uint8_t)((bits >> t) & 1u);
  }
}

}  // namespace

cudaError_t launch_bwd_prep(int dtype, const void* o, const void* dout, Strides st, const float* lse, int B, int H,
                            int N, int npad, int d, float* lse2, float* dvec, float* dqacc, int* sched,
                            float dscale, cudaStream_t s) {
  const long long rows = (long long)B * H * npad;
  const int threads = 256;
  const long long blocks = (rows * 8 + threads - 1) / threads;
  if (dtype == FA_DT_BF16)
    bwd_prep_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, s>>>(
        (const __nv_bfloat16*)o, (const __nv_bfloat16*)dout, st, lse, B, H, N, npad, d, lse2, dvec, dqacc, sched,
        dscale);
  else if (dtype == FA_DT_F16)
    bwd_prep_kernel<__half><<<(unsigned)blocks, threads, 0, s>>>((const __half*)o, (const __half*)dout, st, lse, B,
                                                                 H, N, npad, d, lse2, dvec, dqacc, sched, dscale);
  else
    bwd_prep_kernel<float><<<(unsigned)blocks, threads, 0, s>>>((const float*)o, (const float*)dout, st, lse, B, H,
                                                                N, npad, d, lse2, dvec, dqacc, sched, dscale);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(int dtype, const float* dqacc, void* dq, Strides st, int B, int H, int N, int d,
                              cudaStream_t s) {
  const long long nrows = (long long)B * H * N;
  const long long threads_total = nrows * d / 8;
  const int threads = 256;
  const unsigned blocks = (unsigned)((threads_total + threads - 1) / threads);
  if (blocks == 0) return cudaSuccess;
  if (dtype == FA_DT_BF16)
    dq_convert_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>(dqacc, (__nv_bfloat16*)dq, st, H, N, d, nrows);
  else
    dq_convert_kernel<__half><<<blocks, threads, 0, s>>>(dqacc, (__half*)dq, st, H, N, d, nrows);
  return cudaGetLastError();
}

cudaError_t launch_block_lists(const uint8_t* mask, int nb, int16_t* row_list, int32_t* row_cnt, int16_t* col_list,
                               int32_t* col_cnt, cudaStream_t s) {
  dim3 grid(nb, 2);
  block_lists_kernel<<<grid, 256, 0, s>>>(mask, nb, row_list, row_cnt, col_list, col_cnt);
  return cudaGetLastError();
}

cudaError_t launch_dropout_mask(const DropoutArgs& d, int H, int N, int b, int h, int row0, int nrows, uint8_t* out,
                                cudaStream_t s) {
  const long long groups = (long long)nrows * ((N + 7) / 8);
  if (groups == 0) return cudaSuccess;
  const int threads = 256;
  dropout_mask_kernel<<<(unsigned)((groups + threads - 1) / threads), threads, 0, s>>>(d, H, N, b, h, row0, nrows,
                                                                                         out);
  return cudaGetLastError();
}

// Two warps each wait, with the same bounded wait the attention kernels
// use, on an mbarrier that nothing arrives at: warp 0 polling (as in the
// backward kernels), warp 1 sleeping between tries (as in the forward
// kernels).  Warp 1 starts its wait half the limit later than warp 0.  Warp 0's wait runs out first, records
// FA_ERR_TIMEOUT in the status word and raises the CTA abort flag; warp 1's
// wait then returns on the flag, about half the limit after it started,
// instead of running its own limit out.  out[w] = 1 if warp w's wait
// returned false; out_ns = how long warp 1's wait lasted.
__global__ void wait_selftest_kernel(int* status, int* out, unsigned long long* out_ns) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int w = threadIdx.x >> 5;
  // warp 0 polls (the backward's waits), warp 1 sleeps between tries (the
  // forward's): both give up, warp 1 on the abort flag warp 0 raises
  WaitCtl ctl{status, &abort_flag, w == 1 ? kWaitSleepNs : 0u};
  if ((threadIdx.x & 31) == 0) {
    if (w == 1) {   // a bounded delay of half the wait limit
      const uint64_t d0 = globaltimer_ns();
      while (globaltimer_ns() - d0 < kWaitTimeoutNs / 2) __nanosleep(1000);
    }
    const uint64_t t0 = globaltimer_ns();
    const bool ok = mbar_wait(&bars[w], 0, ctl);
    out[w] = ok ? 0 : 1;
    if (w == 1) *out_ns = globaltimer_ns() - t0;
  }
}

cudaError_t launch_wait_selftest(int* status, int* out, unsigned long long* out_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 64, 0, s>>>(status, out, out_ns);
  return cudaGetLastError();
}

}  // namespace fa
