// bwd_tc.cu -- backward attention kernel for 16-bit inputs on sm_103a.
//
// Method (the pages): the backward pass stores nothing N x N; it rebuilds
// the score and probability tiles on chip from Q, K and the saved softmax
// statistics, replays the dropout mask from the RNG state, and uses
// D_i = dO_i . O_i (tonho.wtf, "como funciona"; agihunt.info, backward
// paragraph; marketmaker.cc, "Passo para tras").  Per (key tile j, query
// tile i) pair it forms
//     P^T = exp(tau K Q_i^T - LSE_i)           (masked, dropout replayed)
//     dP^T = Z o (V dO_i^T) / (1 - p)
//     dS^T = P^T o (dP^T - D_i)
//     dV += P~^T dO_i,  dK += dS^T Q_i,  dQ_i += dS K      (tau applied at the end)
//
// GB300 mapping (ours): one CTA per (b, h, 128-key tile), looping over the
// query tiles that see it (causal / sparse lists).
//   * warp 8: TMA loads of K, V once and of Q_i, dO_i (+ LSE_i, D_i rows) into
//     a two-stage ring;
//   * warp 9: tcgen05 MMAs; S^T and dP^T go to tensor memory, dK and dV
//     accumulate in tensor memory for the whole loop, dQ_i goes to tensor
//     memory per step;
//   * warps 0-3: one thread per key row: P^T, dS^T in registers, written as
//     16-bit swizzled tiles to shared memory (they feed dV, dK as K-major A
//     operands and dQ as an MN-major A operand);
//   * warps 4-7: one thread per query row: read dQ_i from tensor memory,
//     scale by tau, stage in shared memory, TMA reduce-add into a float32
//     accumulator in global memory.
// Tensor memory: S^T 0-127 | dP^T 128-255 | dK 256-319 | dV 320-383 | dQ 384-447.
#include "common.cuh"

namespace fa {
namespace {

constexpr int kThreads = 320;
constexpr int NSB = 2;   // Q / dO stages

struct BwdSmem {
  static constexpr int kK = 0;
  static constexpr int kV = 16384;
  static constexpr int kQ = 32768;              // NSB x 16 KB
  static constexpr int kDO = kQ + NSB * 16384;  // NSB x 16 KB
  static constexpr int kPT = kDO + NSB * 16384; // 32 KB: P~^T [2 chunks][128 keys][64 q]
  static constexpr int kDS = kPT + 32768;       // 32 KB: dS^T, same layout
  static constexpr int kDQ = kDS + 32768;       // 32 KB: float32 dQ staging [2][128][32]
  static constexpr int kLD = kDQ + 32768;       // NSB x (LSE2[128] + D[128]) floats
  static constexpr int kBar = kLD + NSB * 1024;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kDyn = kBytes + 1024;
};

struct BBars {
  uint64_t kv_full;
  uint64_t q_full[NSB], q_empty[NSB];
  uint64_t st_full, ds_full, pds_free, dq_full, dq_free, dkv_full, mma_done;
  uint32_t tmem_base;
  int abort;
};

struct QList {
  int n;
  int i0;                 // first query tile (dense)
  const int16_t* list;    // sparse list or nullptr
  __device__ __forceinline__ int qt(int t) const { return list ? (int)list[t] : i0 + t; }
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
              const __grid_constant__ CUtensorMap tmDQ, const BwdArgs a) {
  using L = BwdSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BBars* bars = reinterpret_cast<BBars*>(smem + L::kBar);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (b, h, key tile jt); for causal the longest lists first
  const int BH = a.B * a.H;
  const int jt = (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / a.H, h = bh % a.H;
  int Lk = a.N;
  if (a.mask.seqlens_k != nullptr) Lk = max(0, min(a.N, a.mask.seqlens_k[b]));
  QList ql;
  ql.list = nullptr;
  ql.i0 = a.mask.causal ? jt : 0;
  ql.n = 0;
  if (jt * kTile < Lk) {
    if (a.mask.col_list != nullptr) {
      ql.list = a.mask.col_list + (size_t)jt * a.mask.nb;
      const int cnt = a.mask.col_cnt[jt];
      int s0 = 0;
      if (a.mask.causal) while (s0 < cnt && ql.list[s0] < jt) ++s0;
      ql.list += s0;
      ql.n = cnt - s0;
    } else {
      ql.n = a.nq - ql.i0;
    }
  }
  const int n = ql.n;
  WaitCtl ctl{a.status, &bars->abort};

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < NSB; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    mbar_init(&bars->st_full, 1);
    mbar_init(&bars->ds_full, 128);
    mbar_init(&bars->pds_free, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 128);
    mbar_init(&bars->dkv_full, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const size_t ld_row0 = (size_t)bh * a.npad;

  if (warp == 8) {
    // ===================== TMA producer =====================
    if (lane == 0 && n > 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmDO);
      mbar_expect_tx(&bars->kv_full, 32768);
      tma_load_4d(smem + L::kK, &tmK, &bars->kv_full, 0, jt * kTile, h, b);
      tma_load_4d(smem + L::kV, &tmV, &bars->kv_full, 0, jt * kTile, h, b);
      int issued = 0;
      for (int t = 0; t < n; ++t) {
        const int st = t % NSB;
        const uint32_t ph = (uint32_t)(t / NSB) & 1u;
        if (!mbar_wait(&bars->q_empty[st], ph ^ 1u, ctl)) break;
        const int qi = ql.qt(t);
        mbar_expect_tx(&bars->q_full[st], 32768 + 1024);
        tma_load_4d(smem + L::kQ + st * 16384, &tmQ, &bars->q_full[st], 0, qi * kTile, h, b);
        tma_load_4d(smem + L::kDO + st * 16384, &tmDO, &bars->q_full[st], 0, qi * kTile, h, b);
        bulk_load(smem + L::kLD + st * 1024, a.lse2 + ld_row0 + (size_t)qi * kTile, 512, &bars->q_full[st]);
        bulk_load(smem + L::kLD + st * 1024 + 512, a.dvec + ld_row0 + (size_t)qi * kTile, 512, &bars->q_full[st]);
        ++issued;
      }
      for (int t = max(0, issued - NSB); t < issued; ++t)
        mbar_wait(&bars->q_full[t % NSB], (uint32_t)(t / NSB) & 1u, ctl);
      mbar_wait(&bars->kv_full, 0, ctl);
    }
  } else if (warp == 9) {
    // ===================== MMA issuer =====================
    if (lane == 0 && n > 0) {
      constexpr int ab = Cvt<T>::kAB;
      constexpr uint32_t idST = idesc_f16(128, 128, ab, 0, 0);   // S^T, dP^T
      constexpr uint32_t idKV = idesc_f16(128, 64, ab, 0, 1);    // dV, dK (A K-major, B MN-major)
      constexpr uint32_t idQ = idesc_f16(128, 64, ab, 1, 1);     // dQ (A MN-major, B MN-major)
      const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
      const uint32_t sQ = smem_u32(smem + L::kQ), sDO = smem_u32(smem + L::kDO);
      const uint32_t sPT = smem_u32(smem + L::kPT), sDS = smem_u32(smem + L::kDS);
      const uint32_t tST = tmem, tDP = tmem + 128, tDK = tmem + 256, tDV = tmem + 320, tDQ = tmem + 384;
      bool ok = mbar_wait(&bars->kv_full, 0, ctl) && mbar_wait(&bars->q_full[0], 0, ctl);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tST, sdesc_sw128(sK + k * 32, 16, 1024), sdesc_sw128(sQ + k * 32, 16, 1024), idST, k > 0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tDP, sdesc_sw128(sV + k * 32, 16, 1024), sdesc_sw128(sDO + k * 32, 16, 1024), idST, k > 0);
        mma_commit(&bars->st_full);
      }
      for (int t = 0; t < n && ok; ++t) {
        const int st = t % NSB;
        if (!(ok = mbar_wait(&bars->ds_full, (uint32_t)t & 1u, ctl))) break;
        tc_fence_after();
        if (t + 1 < n) {
          const int st1 = (t + 1) % NSB;
          if (!(ok = mbar_wait(&bars->q_full[st1], (uint32_t)((t + 1) / NSB) & 1u, ctl))) break;
          tc_fence_after();
          const uint32_t q1 = sQ + st1 * 16384, d1 = sDO + st1 * 16384;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tST, sdesc_sw128(sK + k * 32, 16, 1024), sdesc_sw128(q1 + k * 32, 16, 1024), idST, k > 0);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tDP, sdesc_sw128(sV + k * 32, 16, 1024), sdesc_sw128(d1 + k * 32, 16, 1024), idST, k > 0);
          mma_commit(&bars->st_full);
        }
        const uint32_t qb = sQ + st * 16384, db = sDO + st * 16384;
        // dV += P~^T dO_i ; dK += dS^T Q_i   (K-dim = 128 queries, 8 steps of 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t aoff = (k >> 2) * 16384 + (k & 3) * 32;
          mma_ss(tDV, sdesc_sw128(sPT + aoff, 16, 1024), sdesc_sw128(db + k * 2048, 16384, 1024), idKV,
                 (t > 0 || k > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t aoff = (k >> 2) * 16384 + (k & 3) * 32;
          mma_ss(tDK, sdesc_sw128(sDS + aoff, 16, 1024), sdesc_sw128(qb + k * 2048, 16384, 1024), idKV,
                 (t > 0 || k > 0) ? 1u : 0u);
        }
        // dQ_i = dS K  (M = 128 queries, K-dim = 128 keys)
        if (t > 0 && !(ok = mbar_wait(&bars->dq_free, (uint32_t)(t - 1) & 1u, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss(tDQ, sdesc_sw128(sDS + k * 2048, 16384, 1024), sdesc_sw128(sK + k * 2048, 16384, 1024), idQ,
                 k > 0 ? 1u : 0u);
        mma_commit(&bars->dq_full);
        mma_commit(&bars->pds_free);
        mma_commit(&bars->q_empty[st]);
      }
      mma_commit(&bars->dkv_full);
      mma_commit(&bars->mma_done);
      mbar_wait(&bars->mma_done, 0, ctl);
    }
  } else if (warp < 4) {
    // ===================== P^T / dS^T (one thread per key) =====================
    const int r = warp * 32 + lane;
    const int j = jt * kTile + r;                     // global key
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tST = tmem + lane_off, tDP = tST + 128;
    const bool key_ok = j < Lk;
    const float sl2 = a.scale_log2;
    const uint32_t bh_rows = (uint32_t)bh * (uint32_t)a.N;
    bool ok = true;
    for (int t = 0; t < n && ok; ++t) {
      const int st = t % NSB;
      const int qi = ql.qt(t);
      if (!(ok = warp_wait(&bars->st_full, (uint32_t)t & 1u, ctl) &&
                 warp_wait(&bars->q_full[st], (uint32_t)(t / NSB) & 1u, ctl))) break;
      tc_fence_after();
      if (t > 0 && !(ok = warp_wait(&bars->pds_free, (uint32_t)(t - 1) & 1u, ctl))) break;
      const float* lse2 = reinterpret_cast<const float*>(smem + L::kLD + st * 1024);
      const float* dvec = lse2 + 128;
      uint8_t* pt = smem + L::kPT;
      uint8_t* ds = smem + L::kDS;
      // last query (relative to the tile) that this key is hidden from under causal: q < j
      const int qlo = a.mask.causal ? (j - qi * kTile) : -1;   // columns c < qlo... masked when c < qlo
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t sv[32], dv[32];
        tmem_ld32(tST + cc * 32, sv);
        tmem_ld32(tDP + cc * 32, dv);
        tmem_wait_ld();
        uint32_t keep = ~0u;
        if (a.drop.enabled) {
          keep = 0;
#pragma unroll 4
          for (int c = 0; c < 32; ++c) {
            const uint32_t q = (uint32_t)(qi * kTile + cc * 32 + c);
            const uint32_t bits = dropout_keep8((uint32_t)j >> 3, bh_rows + q, a.drop);
            keep |= ((bits >> (j & 7)) & 1u) << c;
          }
        }
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float p[2], d[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int cq = cc * 32 + c + e;
            float pv = ex2(fmaf(__uint_as_float(sv[c + e]), sl2, -lse2[cq]));
            if (!key_ok || cq < qlo) pv = 0.f;
            const bool kept = (keep >> (c + e)) & 1u;
            const float dpv = kept ? __uint_as_float(dv[c + e]) * a.drop.rp : 0.f;
            p[e] = kept ? pv * a.drop.rp : 0.f;
            d[e] = pv * (dpv - dvec[cq]);
          }
          pw[c >> 1] = Cvt<T>::pack(p[0], p[1]);
          dw[c >> 1] = Cvt<T>::pack(d[0], d[1]);
        }
        // columns cc*32 .. +31 -> chunk cc/2, 16-byte pieces (cc&1)*4 .. +3
        const uint32_t base = (cc >> 1) * 16384 + r * 128;
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
          const uint32_t piece = (cc & 1) * 4 + pc;
          const uint32_t off = base + (((piece ^ (uint32_t)r) & 7u) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                       :: "r"(smem_u32(pt + off)), "r"(pw[pc * 4]), "r"(pw[pc * 4 + 1]), "r"(pw[pc * 4 + 2]),
                          "r"(pw[pc * 4 + 3]) : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                       :: "r"(smem_u32(ds + off)), "r"(dw[pc * 4]), "r"(dw[pc * 4 + 1]), "r"(dw[pc * 4 + 2]),
                          "r"(dw[pc * 4 + 3]) : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->ds_full);
    }
    // ---- epilogue: dK (x tau), dV -> 16 bit -> shared -> TMA store
    named_bar_sync(1, 128);
    if (!bars->abort) {
      uint32_t kraw[2][32], vraw[2][32];
      bool have = false;
      if (n > 0 && warp_wait(&bars->dkv_full, 0, ctl)) {
        tc_fence_after();
        tmem_ld32(tmem + lane_off + 256, kraw[0]);
        tmem_ld32(tmem + lane_off + 288, kraw[1]);
        tmem_ld32(tmem + lane_off + 320, vraw[0]);
        tmem_ld32(tmem + lane_off + 352, vraw[1]);
        tmem_wait_ld();
        have = true;
      }
      uint8_t* kb = smem + L::kPT;          // P^T / dS^T are dead after dkv_full
      uint8_t* vb = smem + L::kPT + 16384;
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {
        uint32_t wk[4], wv[4];
#pragma unroll
        for (int t2 = 0; t2 < 4; ++t2) {
          const int c = pc * 8 + 2 * t2;
          const float k0 = have ? __uint_as_float(kraw[c >> 5][c & 31]) * a.scale : 0.f;
          const float k1 = have ? __uint_as_float(kraw[(c + 1) >> 5][(c + 1) & 31]) * a.scale : 0.f;
          const float v0 = have ? __uint_as_float(vraw[c >> 5][c & 31]) : 0.f;
          const float v1 = have ? __uint_as_float(vraw[(c + 1) >> 5][(c + 1) & 31]) : 0.f;
          wk[t2] = Cvt<T>::pack(k0, k1);
          wv[t2] = Cvt<T>::pack(v0, v1);
        }
        const uint32_t off = r * 128 + (((pc ^ r) & 7) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     :: "r"(smem_u32(kb + off)), "r"(wk[0]), "r"(wk[1]), "r"(wk[2]), "r"(wk[3]) : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     :: "r"(smem_u32(vb + off)), "r"(wv[0]), "r"(wv[1]), "r"(wv[2]), "r"(wv[3]) : "memory");
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (r == 0) {
        tma_store_4d(&tmDK, kb, 0, jt * kTile, h, b);
        tma_store_4d(&tmDV, vb, 0, jt * kTile, h, b);
        bulk_commit();
        bulk_wait0();
      }
    }
  } else {
    // ===================== dQ: one thread per query row =====================
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t tDQ = tmem + ((uint32_t)(quarter * 32) << 16) + 384;
    float* stg = reinterpret_cast<float*>(smem + L::kDQ);
    bool ok = true;
    for (int t = 0; t < n && ok; ++t) {
      const int qi = ql.qt(t);
      if (!(ok = warp_wait(&bars->dq_full, (uint32_t)t & 1u, ctl))) break;
      tc_fence_after();
      uint32_t g[2][32];
      tmem_ld32(tDQ, g[0]);
      tmem_ld32(tDQ + 32, g[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->dq_free);
      // the previous reduce must have finished reading the staging buffer
      if (r == 0) bulk_wait_read0();
      named_bar_sync(2, 128);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int pc = 0; pc < 8; ++pc) {
          const uint32_t off = hf * 16384 + r * 128 + (((pc ^ r) & 7) << 4);
          const float* gv = reinterpret_cast<const float*>(&g[hf][pc * 4]);
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};"
                       :: "r"(smem_u32(reinterpret_cast<uint8_t*>(stg) + off)),
                          "f"(gv[0] * a.scale), "f"(gv[1] * a.scale), "f"(gv[2] * a.scale), "f"(gv[3] * a.scale)
                       : "memory");
        }
      fence_proxy_async_smem();
      named_bar_sync(2, 128);
      if (r == 0) {
        tma_reduce_add_4d(&tmDQ, stg, 0, qi * kTile, h, b);
        tma_reduce_add_4d(&tmDQ, reinterpret_cast<uint8_t*>(stg) + 16384, 32, qi * kTile, h, b);
        bulk_commit();
      }
    }
    if (r == 0) bulk_wait0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <typename T>
cudaError_t launch_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                     const CUtensorMap& dk, const CUtensorMap& dv, const CUtensorMap& dqacc, const BwdArgs& a,
                     cudaStream_t s) {
  auto kern = bwd_tc_kernel<T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdSmem::kDyn);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(a.nq * a.B * a.H);
  if (grid == 0) return cudaSuccess;
  kern<<<grid, kThreads, BwdSmem::kDyn, s>>>(q, k, v, dout, dk, dv, dqacc, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc(int dtype, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& dout, const CUtensorMap& dk, const CUtensorMap& dv,
                          const CUtensorMap& dqacc, const BwdArgs& a, cudaStream_t s) {
  if (dtype == FA_DT_BF16) return launch_t<__nv_bfloat16>(q, k, v, dout, dk, dv, dqacc, a, s);
  return launch_t<__half>(q, k, v, dout, dk, dv, dqacc, a, s);
}

}  // namespace fa
