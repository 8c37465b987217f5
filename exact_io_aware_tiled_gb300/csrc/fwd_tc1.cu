// fwd_tc1.cu -- forward attention kernel for 16-bit inputs at head dimension 64,
// one query tile per CTA, two CTAs per SM.
//
// Method (the pages): Q-outer tiling with the online-softmax recurrence and
// deferred normalisation (lynx-cortex "FlashAttention como una optimizacion
// de roofline", section "El algoritmo Flash (forward)"; marketmaker.cc,
// "O algoritmo de atencao do Flash"), causal / padded / sparse tiles skipped
// (marketmaker.cc, "O mascaramento causal"; agihunt.info, block-sparse
// paragraph), mask and dropout applied to the score tile on chip
// (agihunt.info, fused-kernel paragraph).  Only O and the per-row
// logsumexp leave the chip.  Grouped-query attention: query head h reads K/V
// head h / g (living-dl-book, "Atencao eficiente", section 6); sliding window
// as in the two-tile kernel (lynx-cortex, "Problemas de practica").
//
// GB300 mapping (ours).  A CTA with one 128-row query tile spends about 2 us
// filling its pipeline (Q load from HBM, first K/V tiles, first S) and about
// 1.5 us draining it (last P V product, O out) around its steps; at short
// causal rows that is comparable to the steps themselves.  This kernel keeps
// a CTA small -- 112 KB of shared memory, 256 tensor-memory columns, 256
// threads at 128 registers -- so that two CTAs share an SM and one CTA's
// fill and drain run under the other's steps:
//   * warp 4 (one thread) streams K/V with TMA into a ring of NS stages;
//   * warp 5 issues S = Q K^T as soon as the softmax has copied the previous
//     S into registers; warp 6 issues O += P V (P from tensor memory).  Each
//     product is a latency chain (consecutive MMAs into one accumulator
//     complete ~126 cycles apart), so the two chains are issued by separate
//     warps;
//   * warps 0-3 run the softmax, one thread per query row (= TMEM lane); the
//     same register-resident row code as the two-tile kernel: conditional
//     2^8 rescale, O normalised by the sum of the rounded P the MMA consumed;
//   * epilogue: O / l -> 16 bit -> shared memory (the dead Q tile, 128-B
//     swizzle) -> TMA store, which clips rows >= N; logsumexp with plain stores.
// Tensor memory: S 128 columns | P 64 | O 64 (256 of the SM's 512).
#include "common.cuh"

namespace fa {
namespace {

constexpr int kThreads1 = 256;   // warps 0-3 softmax, 4 TMA, 5 S MMAs, 6 PV MMAs, 7 idle
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

struct Fwd1Cfg {
  static constexpr int kTB = 128 * 64 * 2;               // one [128][64] 16-bit tile
  static constexpr int NS = 3;                           // K/V stages
  static constexpr int kQ = 0;
  static constexpr int kK = kTB;
  static constexpr int kV = kK + NS * kTB;
  static constexpr int kBar = kV + NS * kTB;
  static constexpr int kBytes = kBar + 256;
};
// Two CTAs of this size fit the SM's 228 KB (each also holds 1 KB the system
// reserves).  The dynamic shared memory must start 1024-byte aligned (the
// 128-byte swizzle atoms); the kernel checks that and refuses otherwise.

struct Bars1 {
  uint64_t q_full, s_full, s_free, p_full, pv_done;
  uint64_t done[2];
  uint64_t k_full[Fwd1Cfg::NS], v_full[Fwd1Cfg::NS], k_empty[Fwd1Cfg::NS], v_empty[Fwd1Cfg::NS];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars1) <= 256, "barrier block overflows its shared-memory slot");

// The kv tiles query tile qt visits, in ascending order (causal: j <= qt;
// padding: j < ceil(Lk / 128); window: from the first tile the window
// reaches; block-sparse: the tile's row list).
struct Tile1 {
  int qt, n, lo;
  const int16_t* list;
  template <bool kWin>
  __device__ __forceinline__ int kv(int s) const { return list ? (int)list[s] : (kWin ? lo + s : s); }
};

__device__ __forceinline__ Tile1 make_tile1(const FwdArgs& a, int qt, int Lk) {
  Tile1 t;
  t.qt = qt;
  t.list = nullptr;
  t.n = 0;
  t.lo = 0;
  int lim = (Lk + kTile - 1) / kTile;
  if (a.mask.causal) lim = min(lim, qt + 1);
  if (a.mask.window > 0) t.lo = max(0, qt * kTile - a.mask.window + 1) / kTile;
  if (a.mask.row_list != nullptr) {
    const int16_t* list = a.mask.row_list + (size_t)qt * a.mask.nb;
    const int cnt = a.mask.row_cnt[qt];
    int s0 = 0;
    while (s0 < cnt && list[s0] < t.lo) ++s0;
    int n = s0;
    while (n < cnt && list[n] < lim) ++n;
    t.list = list + s0;
    t.n = n - s0;
  } else {
    t.n = max(0, lim - t.lo);
  }
  return t;
}

__device__ __forceinline__ bool warp_wait1(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

template <typename T, bool kDrop, bool kWin>
__global__ void __launch_bounds__(kThreads1, 2)
fwd_tc1_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
               const FwdArgs a) {
  using C = Fwd1Cfg;
  constexpr int NS = C::NS;
  constexpr int TB = C::kTB;
  constexpr uint32_t kColP = 128, kColO = 192;
  extern __shared__ __align__(1024) uint8_t smem[];
  // The 128-byte swizzle needs 1024-byte aligned tiles: refuse (every thread
  // alike, before any barrier or allocation) if the runtime placed the
  // dynamic shared memory otherwise.
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicExch(a.status, (int)FA_ERR_CUDA);
    return;
  }
  Bars1* bars = reinterpret_cast<Bars1*>(smem + C::kBar);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (b, h, query tile); heaviest tiles launch first
  const int BH = a.B * a.H;
  const int qt = a.nq - 1 - (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / a.H, h = bh % a.H;
  const int hk = h / a.group;
  int Lk = a.N;
  if (a.mask.seqlens_k != nullptr) Lk = max(0, min(a.N, a.mask.seqlens_k[b]));
  const Tile1 tile = make_tile1(a, qt, Lk);
  const int n = tile.n;

  // The role threads mostly wait on the softmax warps: they sleep while they
  // wait, leaving the issue slots to the softmax.
  WaitCtl ctl{a.status, &bars->abort, kWaitSleepNs};

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 128);
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->pv_done, 1);
    for (int i = 0; i < 2; ++i) mbar_init(&bars->done[i], 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Tensor memory: warp 5 allocates it, and only the warps that use it (the
  // softmax warps 0-3 and the MMA issuers 5 and 6: 192 threads) meet on named
  // barrier 2 to read its address.  The TMA producer does not wait for the
  // allocation, so its first loads (Q, then K(0), from HBM / L2 with a latency
  // of about a microsecond) overlap it.
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, 256);
    tmem_relinquish();
  }
  uint32_t tmem = 0;
  auto tmem_ready = [&]() {
    if constexpr (!kDrop) {
      tc_fence_before();
      named_bar_sync(2, 192);
      tc_fence_after();
      tmem = bars->tmem_base;
    }
  };
  if constexpr (kDrop) {
    // With dropout (Philox-bound steps) the early start measured slower
    // (2-3 % at BERT-large sizes): every warp waits for the allocation.
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tmem = bars->tmem_base;
  }
  constexpr int ab = Cvt<T>::kAB;
  // Register split of the 256 x 128 launch budget (two CTAs per SM): the
  // softmax warpgroup holds a whole 128-column score row per thread; the
  // TMA / MMA warps (and the idle warp 7) need few.
  // 4 x 32 x 208 + 4 x 32 x 48 = 32768 = 256 x 128.

  if (warp >= 4) {
    regs_dec<48>();
    if (warp == 4) {
      // ===================== TMA producer =====================
      if (lane == 0 && n > 0) {
        mbar_expect_tx(&bars->q_full, TB);
        tma_load_4d(smem + C::kQ, &tmQ, &bars->q_full, 0, qt * kTile, h, b);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        bool ok = true;
        for (int s = 0; s < n && ok; ++s) {
          const int st = s % NS;
          const uint32_t ph = (uint32_t)(s / NS) & 1u;
          const int kv = tile.kv<kWin>(s);
          // a stage's first use needs no wait
          if (s >= NS &&
              !(ok = mbar_wait(&bars->k_empty[st], ph ^ 1u, ctl) && mbar_wait(&bars->v_empty[st], ph ^ 1u, ctl)))
            break;
          mbar_expect_tx(&bars->k_full[st], TB);
          tma_load_4d(smem + C::kK + st * TB, &tmK, &bars->k_full[st], 0, kv * kTile, hk, b);
          mbar_expect_tx(&bars->v_full[st], TB);
          tma_load_4d(smem + C::kV + st * TB, &tmV, &bars->v_full[st], 0, kv * kTile, hk, b);
        }
        // Before leaving, make sure no load is still writing shared memory.
        for (int j = max(0, n - NS); j < n; ++j) {
          mbar_wait(&bars->k_full[j % NS], (uint32_t)(j / NS) & 1u, ctl);
          mbar_wait(&bars->v_full[j % NS], (uint32_t)(j / NS) & 1u, ctl);
        }
        mbar_wait(&bars->q_full, 0, ctl);
      }
    } else if (warp == 5) {
      // ===================== S issuer =====================
      tmem_ready();
      if (lane == 0 && n > 0) {
        constexpr uint32_t idS = idesc_f16(128, 128, ab, 0, 0);
        const uint64_t qd = sdesc_sw128(smem_u32(smem + C::kQ), 16, 1024);
        const uint64_t kd0 = sdesc_sw128(smem_u32(smem + C::kK), 16, 1024);
        bool ok = mbar_wait(&bars->q_full, 0, ctl);
        for (int s = 0; s < n && ok; ++s) {
          const int st = s % NS;
          // S(s) overwrites S(s-1) once the softmax has read it
          if (s > 0 && !(ok = mbar_wait(&bars->s_free, (uint32_t)(s - 1) & 1u, ctl))) break;
          if (!(ok = mbar_wait(&bars->k_full[st], (uint32_t)(s / NS) & 1u, ctl))) break;
          tc_fence_after();
          const uint64_t kd = kd0 + (uint64_t)((st * TB) >> 4);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem, qd + (uint64_t)((k * 32) >> 4), kd + (uint64_t)((k * 32) >> 4), idS, k > 0 ? 1u : 0u);
          mma_commit(&bars->s_full);
          mma_commit(&bars->k_empty[st]);
        }
        mma_commit(&bars->done[0]);
        mbar_wait(&bars->done[0], 0, ctl);
      }
    } else if (warp == 6) {
      // ===================== PV issuer =====================
      tmem_ready();
      if (lane == 0 && n > 0) {
        constexpr uint32_t idPV = idesc_f16(128, 64, ab, 0, 1);
        const uint64_t vd0 = sdesc_sw128(smem_u32(smem + C::kV), 16384, 1024);
        const uint32_t tP = tmem + kColP, tO = tmem + kColO;
        bool ok = true;
        for (int s = 0; s < n && ok; ++s) {
          const int st = s % NS;
          if (!(ok = mbar_wait(&bars->p_full, (uint32_t)s & 1u, ctl) &&
                     mbar_wait(&bars->v_full[st], (uint32_t)(s / NS) & 1u, ctl)))
            break;
          tc_fence_after();
          const uint64_t vd = vd0 + (uint64_t)((st * TB) >> 4);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tO, tP + k * 8, vd + (uint64_t)(k * (2048 >> 4)), idPV, (s > 0 || k > 0) ? 1u : 0u);
          mma_commit(&bars->pv_done);
          mma_commit(&bars->v_empty[st]);
        }
        mma_commit(&bars->done[1]);
        mbar_wait(&bars->done[1], 0, ctl);
      }
    }
  } else {
    regs_inc<208>();
    tmem_ready();
    // ===================== softmax warps =====================
    const int r = warp * 32 + lane;             // row within the tile = TMEM lane
    const int i = qt * kTile + r;               // global query row
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off, tP = tS + kColP, tO = tS + kColO;
    const float sl2 = a.scale_log2;
    const int jmax = a.mask.causal ? min(Lk - 1, i) : (Lk - 1);
    const int jmin = kWin ? i - a.mask.window + 1 : 0;   // first key of the sliding window
    const uint32_t row_g = (uint32_t)(b * a.H + h) * (uint32_t)a.N + (uint32_t)i;

    float m_run = -INFINITY;
    float l_true = 0.f, l_rnd = 0.f;
    bool ok = true;
    for (int s = 0; s < n; ++s) {
      const int kv = tile.kv<kWin>(s);
      if (!(ok = warp_wait1(&bars->s_full, (uint32_t)s & 1u, ctl))) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, sr[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) reg_fence32(sr[cc]);
      tc_fence_before();
      mbar_arrive(&bars->s_free);               // S(s+1) may now overwrite the S columns

      // mask (only boundary tiles) and row max of the raw scores
      const int jl = jmax - kv * kTile;
      const int jlo = jmin - kv * kTile;
      if (jl < kTile - 1 || (kWin && jlo > 0)) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > jl || (kWin && c < jlo)) sr[c >> 5][c & 31] = __float_as_uint(-INFINITY);
      }
      // row max: 8 independent chains of 3-input max, then a short tree
      float m8[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) m8[t] = __uint_as_float(sr[0][t]);
#pragma unroll
      for (int c = 8; c < 128; c += 16) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int c0 = c + t, c1 = c + 8 + t;
          m8[t] = (c1 < 128) ? max3f(m8[t], __uint_as_float(sr[c0 >> 5][c0 & 31]), __uint_as_float(sr[c1 >> 5][c1 & 31]))
                             : fmaxf(m8[t], __uint_as_float(sr[c0 >> 5][c0 & 31]));
        }
      }
      float mx = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      mx *= sl2;
      // running reference max: moved only when the tile max exceeds it by 2^8
      float m_new = m_run;
      if (mx > m_run + kRescaleThreshold) m_new = mx;
      const bool rescale = (m_new != m_run) && (m_run != -INFINITY) && (s > 0);
      const float alpha = (m_new != m_run && m_run != -INFINITY) ? ex2(m_run - m_new) : 1.f;
      m_run = m_new;
      l_true *= alpha;
      l_rnd *= alpha;
      const float mref = (m_run == -INFINITY) ? 0.f : m_run;
      const float nmref = -mref;

      uint32_t keep[4] = {~0u, ~0u, ~0u, ~0u};
      if constexpr (kDrop) {
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          const uint32_t bits = dropout_keep8((uint32_t)(kv * 16 + g), row_g, a.drop);
          keep[g >> 2] = (g & 3) == 0 ? bits : (keep[g >> 2] | (bits << ((g & 3) * 8)));
        }
      }
      // P = exp2(S * tau*log2e - m), packed to 16 bits, one pair of keys per
      // call.  l_true sums the unrounded P (for the logsumexp); l_rnd sums
      // exactly the 16-bit values the PV MMA consumes before dropout zeroes
      // some of them (P, or P/(1-p) with dropout), so O / l_rnd is a
      // consistently rounded convex combination of V rows.
      const float pscale = kDrop ? a.drop.rp : 1.f;
      float lt[4] = {0.f, 0.f, 0.f, 0.f}, lr[4] = {0.f, 0.f, 0.f, 0.f};
      auto p_pair = [&](int c) -> uint32_t {
        const int ch = (c >> 1) & 1;
        float x0, x1;
        fma2(x0, x1, __uint_as_float(sr[c >> 5][c & 31]), __uint_as_float(sr[(c + 1) >> 5][(c + 1) & 31]), sl2,
             sl2, nmref, nmref);
        const float p0 = ex2(x0), p1 = ex2(x1);
        add2(lt[2 * ch], lt[2 * ch + 1], p0, p1);
        uint32_t u = kDrop ? Cvt<T>::pack(p0 * pscale, p1 * pscale) : Cvt<T>::pack(p0, p1);
        Cvt<T>::acc2(lr[2 * ch], lr[2 * ch + 1], u);
        if constexpr (kDrop) {
          const uint32_t kb = keep[c >> 5] >> (c & 31);
          u &= ((kb & 1u) ? 0x0000FFFFu : 0u) | ((kb & 2u) ? 0xFFFF0000u : 0u);
        }
        return u;
      };
      // PV(s-1) must be done before the P columns are reused and O is
      // rescaled.  Its chain of eight dependent MMAs (about 1,000 cycles) was
      // issued at the end of the previous step.  Without dropout the wait
      // comes after this step's exponentials (the whole packed row is held in
      // registers), which keeps it off the softmax's path.  With dropout the
      // Philox words leave no room for that: the wait comes first and P goes
      // out per half of 64 keys.
      if constexpr (kDrop) {
        if (s > 0 && !(ok = warp_wait1(&bars->pv_done, (uint32_t)(s - 1) & 1u, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[32];
#pragma unroll
          for (int c2 = 0; c2 < 64; c2 += 2) pk[c2 >> 1] = p_pair(hf * 64 + c2);
          tmem_st32(tP + hf * 32, pk);
        }
      } else {
        uint32_t pk[2][32];
#pragma unroll
        for (int c2 = 0; c2 < 128; c2 += 2) pk[c2 >> 6][(c2 >> 1) & 31] = p_pair(c2);
        if (s > 0 && !(ok = warp_wait1(&bars->pv_done, (uint32_t)(s - 1) & 1u, ctl))) break;
        tc_fence_after();
        tmem_st32(tP, pk[0]);
        tmem_st32(tP + 32, pk[1]);
      }
      l_true += (lt[0] + lt[1]) + (lt[2] + lt[3]);
      l_rnd += ((lr[0] + lr[1]) + (lr[2] + lr[3])) / pscale;
      // tcgen05.ld / st are warp-collective: the warp rescales together when
      // any of its rows needs it (alpha is exactly 1 for the other rows)
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t o[32];
          tmem_ld32(tO + hf * 32, o);
          tmem_wait_ld();
          reg_fence32(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st32(tO + hf * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }

    // ---- epilogue: O / l -> 16 bit -> shared (the Q tile, dead once O is
    //      final) -> TMA store; logsumexp
    if (!named_bar_or(1, 128, !ok || bars->abort)) {
      const bool have = n > 0 && warp_wait1(&bars->pv_done, (uint32_t)(n - 1) & 1u, ctl);
      if (have) tc_fence_after();
      const float inv = l_rnd > 0.f ? 1.f / l_rnd : 0.f;
      const bool row_ok = i < a.N;
      const size_t row = (size_t)(b * a.H + h) * a.N + i;
      uint8_t* ob = smem + C::kQ;
      float o[64];
      if (have) {
        uint32_t raw[2][32];
        tmem_ld32(tO, raw[0]);
        tmem_ld32(tO + 32, raw[1]);
        tmem_wait_ld();
        reg_fence32(raw[0]);
        reg_fence32(raw[1]);
#pragma unroll
        for (int c = 0; c < 64; ++c) o[c] = __uint_as_float(raw[c >> 5][c & 31]) * inv;
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) o[c] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) w[t] = Cvt<T>::pack(o[j * 8 + 2 * t], o[j * 8 + 2 * t + 1]);
        const uint32_t off = r * 128 + (((j ^ r) & 7) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     :: "r"(smem_u32(ob + off)), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
      }
      if (row_ok && a.o_f32 != nullptr) {
        float4* dst = reinterpret_cast<float4*>(a.o_f32 + row * 64);
#pragma unroll
        for (int c = 0; c < 16; ++c) dst[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (r == 0) {
        tma_store_4d(&tmO, ob, 0, qt * kTile, h, b);
        bulk_commit();
        bulk_wait_read0();
      }
      if (row_ok) a.lse[row] = l_true > 0.f ? (m_run + lg2(l_true)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <typename T, bool kDrop, bool kWin>
cudaError_t launch_t1(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                      const FwdArgs& a, cudaStream_t s) {
  auto kern = fwd_tc1_kernel<T, kDrop, kWin>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Fwd1Cfg::kBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(a.nq * a.B * a.H);
  if (grid == 0) return cudaSuccess;
  kern<<<grid, kThreads1, Fwd1Cfg::kBytes, s>>>(q, k, v, o, a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_d1(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                      const FwdArgs& a, cudaStream_t s) {
  const int sel = (a.drop.enabled ? 1 : 0) | (a.mask.window > 0 ? 2 : 0);
  switch (sel) {
    case 0: return launch_t1<T, false, false>(q, k, v, o, a, s);
    case 1: return launch_t1<T, true, false>(q, k, v, o, a, s);
    case 2: return launch_t1<T, false, true>(q, k, v, o, a, s);
    default: return launch_t1<T, true, true>(q, k, v, o, a, s);
  }
}

}  // namespace

cudaError_t launch_fwd_tc1(int dtype, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& o, const FwdArgs& a, cudaStream_t s) {
  if (dtype == FA_DT_BF16) return launch_d1<__nv_bfloat16>(q, k, v, o, a, s);
  return launch_d1<__half>(q, k, v, o, a, s);
}

}  // namespace fa
