// fwd_tc.cu -- forward attention kernel for 16-bit inputs on sm_103a.
//
// Method (the pages): Q-outer tiling with the online-softmax recurrence and
// deferred normalisation (lynx-cortex "FlashAttention como una optimizacion
// de roofline", section "El algoritmo Flash (forward)"; marketmaker.cc,
// "O algoritmo de atencao do Flash"), causal / padded / sparse tiles skipped
// (marketmaker.cc, "O mascaramento causal"; agihunt.info, block-sparse
// paragraph), mask and dropout applied to the score tile on chip
// (agihunt.info, fused-kernel paragraph).  Only O and the per-row
// logsumexp leave the chip.
//
// Grouped-query attention (living-dl-book, "Atencao eficiente", section 6):
// query head h reads K/V head h / g.  Sliding window (lynx-cortex, "Problemas
// de practica"): a query tile reads only the K/V tiles its rows' windows
// reach, and the window's lower edge is masked like the causal upper edge.
//
// GB300 mapping (ours, not the pages'):
//   * one CTA = two 128-row query tiles ("slots") of one (b, h) head;
//   * warp 8 (one thread) streams K/V tiles with TMA into a ring of NS
//     stages; a stage is shared by both slots when both need the same KV tile
//     at the same step;
//   * tcgen05 MMAs are issued by three warps: consecutive MMAs that
//     accumulate into the same tensor-memory tile complete about 126 cycles
//     apart whatever their N (measured on GB300), so each product is a
//     latency chain and independent chains are issued from separate warps:
//       warp 9  issues S_x = Q_x K^T for both slots, as soon as the softmax
//               has copied the previous S_x into registers;
//       warp 10 / 11 issue O_x += P_x V for slot 0 / 1 (P_x from tensor
//               memory);
//   * warps 0-3 / 4-7 run the softmax of slot 0 / 1, one thread per query
//     row (= tensor-memory lane).  The next S is computed while the
//     softmax of this one runs; the P store and the O rescale wait for the
//     previous PV MMA, which normally finished during the row max;
//   * O is rescaled only when the running row max grows by more than 2^8
//     (the final O / l and the logsumexp use the same reference max, so the
//     result is unchanged); O is normalised by the sum of the rounded P that
//     the MMA actually consumed;
//   * epilogue: O / l -> 16 bit -> shared memory (128-B swizzle) -> TMA store,
//     which clips rows >= N; the logsumexp goes out with plain stores.
// Tensor memory per slot: S 128 columns | P 64 | O 64  (512 in total).
#include "common.cuh"
#include "fwd_plan.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// Shared memory for head dimension D: the two query tiles, then rings of NS
// K and NS V tiles.  A 128-row tile is D / 64 boxes of [128 rows][128 bytes]
// (128-byte swizzle), 16 KB each.
template <int D>
struct FwdCfg {
  static constexpr int kTB = 128 * D * 2;                // one tile
  static constexpr int NS = D == 64 ? 5 : 2;             // K/V stages
  static constexpr int kQ = 0;                           // 2 tiles
  static constexpr int kK = 2 * kTB;                     // NS tiles
  static constexpr int kV = kK + NS * kTB;               // NS tiles
  static constexpr int kBar = kV + NS * kTB;
  static constexpr int kBytes = kBar + 512;
  static constexpr int kDyn = kBytes + 1024;             // + alignment slack
};
static_assert(FwdCfg<64>::kDyn <= 232448 && FwdCfg<128>::kDyn <= 232448, "shared memory over the per-block limit");

template <int NS>
struct Bars {
  uint64_t q_full;
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t done[3];
  uint64_t k_full[NS], v_full[NS], k_empty[NS], v_empty[NS];
  uint32_t tmem_base;
  int abort;
};

template <typename T, int D, bool kDrop, bool kWin>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
              const FwdArgs a) {
  using C = FwdCfg<D>;
  constexpr int NS = C::NS;
  constexpr int TB = C::kTB;
  constexpr int NC = D / 64;                  // 64-column boxes per tile
  // Tensor memory per slot (256 columns): S 128 | P 64 | O 64 for D = 64.
  // For D = 128, O takes 128 columns and P (16 bit, packed two per column)
  // overwrites the first 64 columns of S once the softmax has read S; the
  // next S of the slot then waits for the PV MMA that reads P.
  constexpr uint32_t kColP = D == 64 ? 128 : 0, kColO = D == 64 ? 192 : 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars<NS>* bars = reinterpret_cast<Bars<NS>*>(smem + C::kBar);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (b, h, pair of query tiles); heaviest pairs launch first
  const int BH = a.B * a.H;
  const int pair = a.npairs - 1 - (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / a.H, h = bh % a.H;
  const int hk = h / a.group;            // K/V head shared by this query head's group
  int Lk = a.N;
  if (a.mask.seqlens_k != nullptr) Lk = max(0, min(a.N, a.mask.seqlens_k[b]));
  Slot sl[2];
  sl[0] = make_slot(a, 2 * pair, Lk);
  sl[1] = make_slot(a, 2 * pair + 1, Lk);
  const int smax = max(sl[0].n, sl[1].n);

  // The role threads mostly wait on the softmax warps: they sleep while they
  // wait, leaving the issue slots to the softmax.
  WaitCtl ctl{a.status, &bars->abort, kWaitSleepNs};

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->s_free[x], 128);
      mbar_init(&bars->p_full[x], 128);
      mbar_init(&bars->pv_done[x], 1);
    }
    for (int i = 0; i < 3; ++i) mbar_init(&bars->done[i], 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_empty[s], 2);
    }
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
  constexpr int ab = Cvt<T>::kAB;
  // Register split of the 384 x 168 launch budget: the softmax warpgroups
  // hold a whole 128-column score row per thread; the four TMA / MMA warps
  // need few registers.  8 x 32 x 224 + 4 x 32 x 56 = 64512 = 384 x 168.

  if (warp >= 8) {
   regs_dec<56>();
   if (warp == 8) {
    // ===================== TMA producer =====================
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const uint32_t qbytes = (sl[0].n > 0 ? (uint32_t)TB : 0u) + (sl[1].n > 0 ? (uint32_t)TB : 0u);
      if (qbytes > 0) {
        mbar_expect_tx(&bars->q_full, qbytes);
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (sl[x].n > 0)
#pragma unroll
            for (int c = 0; c < NC; ++c)
              tma_load_4d(smem + C::kQ + x * TB + c * 16384, &tmQ, &bars->q_full, c * 64, sl[x].qt * kTile, h, b);
      }
      int ld = 0;
      bool ok = true;
      for (int s = 0; s < smax && ok; ++s) {
        const StepPlan p = plan_step<NS, kWin>(sl, s, ld);
#pragma unroll
        for (int l = 0; l < 2; ++l) {
          if (l >= p.nl) break;
          const int st = p.st[l];
          if (!(ok = mbar_wait(&bars->k_empty[st], p.ph[l] ^ 1u, ctl) &&
                     mbar_wait(&bars->v_empty[st], p.ph[l] ^ 1u, ctl)))
            break;
          mbar_expect_tx(&bars->k_full[st], TB);
#pragma unroll
          for (int c = 0; c < NC; ++c)
            tma_load_4d(smem + C::kK + st * TB + c * 16384, &tmK, &bars->k_full[st], c * 64, p.kv[l] * kTile, hk, b);
          mbar_expect_tx(&bars->v_full[st], TB);
#pragma unroll
          for (int c = 0; c < NC; ++c)
            tma_load_4d(smem + C::kV + st * TB + c * 16384, &tmV, &bars->v_full[st], c * 64, p.kv[l] * kTile, hk, b);
        }
      }
      // Before leaving, make sure no load is still writing shared memory.
      for (int j = max(0, ld - NS); j < ld; ++j) {
        mbar_wait(&bars->k_full[j % NS], (uint32_t)(j / NS) & 1u, ctl);
        mbar_wait(&bars->v_full[j % NS], (uint32_t)(j / NS) & 1u, ctl);
      }
      if (qbytes > 0) mbar_wait(&bars->q_full, 0, ctl);
    }
  } else if (warp == 9) {
    // ===================== S issuer (both slots) =====================
    if (lane == 0 && smax > 0) {
      constexpr uint32_t idS = idesc_f16(128, 128, ab, 0, 0);
      const uint64_t qd[2] = {sdesc_sw128(smem_u32(smem + C::kQ), 16, 1024),
                              sdesc_sw128(smem_u32(smem + C::kQ + TB), 16, 1024)};
      const uint64_t kd0 = sdesc_sw128(smem_u32(smem + C::kK), 16, 1024);
      bool ok = mbar_wait(&bars->q_full, 0, ctl);
      int ld = 0;
      for (int s = 0; s < smax && ok; ++s) {
        const StepPlan p = plan_step<NS, kWin>(sl, s, ld);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!ok || s >= sl[x].n) continue;
          const int l = p.use[x];
          // S_x(s) overwrites S_x(s-1) (D = 64: once the softmax has read it)
          // or P_x(s-1) (D = 128: once PV_x(s-1) has read it)
          if (s > 0 && !(ok = mbar_wait(D == 64 ? &bars->s_free[x] : &bars->pv_done[x], (uint32_t)(s - 1) & 1u, ctl)))
            break;
          if (!(ok = mbar_wait(&bars->k_full[p.stage(l)], p.parity(l), ctl))) break;
          tc_fence_after();
          const uint64_t kd = kd0 + (uint64_t)((p.stage(l) * TB) >> 4);
          const uint32_t tS = tmem + x * 256;
          // K-dim = D in steps of 16: box k / 4, 32 bytes per step within it
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t o = (uint64_t)(((k >> 2) * 16384 + (k & 3) * 32) >> 4);
            mma_ss(tS, qd[x] + o, kd + o, idS, k > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[x]);
        }
#pragma unroll
        for (int l = 0; l < 2; ++l)
          if (ok && l < p.nl) mma_commit(&bars->k_empty[p.st[l]]);
      }
      mma_commit(&bars->done[0]);
      mbar_wait(&bars->done[0], 0, ctl);
    }
  } else if (warp >= 10) {
    // ===================== PV issuer of slot x =====================
    const int x = warp - 10;
    if (lane == 0 && smax > 0) {
      constexpr uint32_t idPV = idesc_f16(128, D, ab, 0, 1);
      const uint64_t vd0 = sdesc_sw128(smem_u32(smem + C::kV), 16384, 1024);
      const uint32_t tP = tmem + x * 256 + kColP, tO = tmem + x * 256 + kColO;
      const int n = x ? sl[1].n : sl[0].n;
      int ld = 0;
      bool ok = true;
      for (int s = 0; s < smax && ok; ++s) {
        const StepPlan p = plan_step<NS, kWin>(sl, s, ld);
        const int mine = p.load_of(x);
        if (s < n) {
          const int st = p.stage(mine);
          if (!(ok = mbar_wait(&bars->p_full[x], (uint32_t)s & 1u, ctl) &&
                     mbar_wait(&bars->v_full[st], p.parity(mine), ctl)))
            break;
          tc_fence_after();
          const uint64_t vd = vd0 + (uint64_t)((st * TB) >> 4);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tO, tP + k * 8, vd + (uint64_t)(k * (2048 >> 4)), idPV, (s > 0 || k > 0) ? 1u : 0u);
          mma_commit(&bars->pv_done[x]);
        }
        // one arrival per slot on every loaded stage: after our MMAs for a
        // stage we read, right away (once it is loaded) for one we did not
#pragma unroll
        for (int l = 0; l < 2; ++l) {
          if (!ok || l >= p.nl) continue;
          if (s < n && l == mine) {
            mma_commit(&bars->v_empty[p.st[l]]);
          } else {
            if (!(ok = mbar_wait(&bars->v_full[p.st[l]], p.ph[l], ctl))) continue;
            mbar_arrive(&bars->v_empty[p.st[l]]);
          }
        }
      }
      mma_commit(&bars->done[1 + x]);
      mbar_wait(&bars->done[1 + x], 0, ctl);
    }
   }
  } else {
    regs_inc<224>();
    // ===================== softmax warps =====================
    const int x = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;          // row within the tile = TMEM lane
    const Slot S = x ? sl[1] : sl[0];
    const int i = S.qt * kTile + r;             // global query row
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + x * 256 + lane_off, tP = tS + kColP, tO = tS + kColO;
    const float sl2 = a.scale_log2;
    const int jmax = a.mask.causal ? min(Lk - 1, i) : (Lk - 1);
    const int jmin = kWin ? i - a.mask.window + 1 : 0;   // first key of the sliding window
    const uint32_t row_g = (uint32_t)(b * a.H + h) * (uint32_t)a.N + (uint32_t)i;

    float m_run = -INFINITY;
    float l_true = 0.f, l_rnd = 0.f;
    bool ok = true;
    for (int s = 0; s < S.n; ++s) {
      const int kv = S.kv<kWin>(s);
      if (!(ok = warp_wait(&bars->s_full[x], (uint32_t)s & 1u, ctl))) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, sr[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) reg_fence32(sr[cc]);
      tc_fence_before();
      if constexpr (D == 64) mbar_arrive(&bars->s_free[x]);   // S_x(s+1) may now overwrite the S columns

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
      // pair accumulators (packed f32x2 adds): two chains each for l_true, l_rnd
      float lt[4] = {0.f, 0.f, 0.f, 0.f}, lr[4] = {0.f, 0.f, 0.f, 0.f};
      auto p_pair = [&](int c) -> uint32_t {
        const int ch = (c >> 1) & 1;       // which of the two accumulator chains
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
      // PV(s-1) must be done before O is rescaled and the P columns reused.
      // At D = 64 without dropout the exponentials go into registers first
      // and the wait comes only before P is stored, after them (the chain of
      // eight dependent PV MMAs, issued at the end of the previous step, then
      // stays off the softmax's path).  At D = 128 P lies over S, so PV(s-1)
      // is done before S(s) exists; with dropout the Philox words leave no
      // registers for a whole packed row.
      if constexpr (D == 64 && !kDrop) {
        uint32_t pk[2][32];
#pragma unroll
        for (int c2 = 0; c2 < 128; c2 += 2) pk[c2 >> 6][(c2 >> 1) & 31] = p_pair(c2);
        if (s > 0 && !(ok = warp_wait(&bars->pv_done[x], (uint32_t)(s - 1) & 1u, ctl))) break;
        tc_fence_after();
        tmem_st32(tP, pk[0]);
        tmem_st32(tP + 32, pk[1]);
      } else {
        if (s > 0 && !(ok = warp_wait(&bars->pv_done[x], (uint32_t)(s - 1) & 1u, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[32];
#pragma unroll
          for (int c2 = 0; c2 < 64; c2 += 2) pk[c2 >> 1] = p_pair(hf * 64 + c2);
          tmem_st32(tP + hf * 32, pk);
        }
      }
      l_true += (lt[0] + lt[1]) + (lt[2] + lt[3]);
      l_rnd += ((lr[0] + lr[1]) + (lr[2] + lr[3])) / pscale;
      // tcgen05.ld / st are warp-collective: the warp rescales together when
      // any of its rows needs it (alpha is exactly 1 for the other rows)
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int hf = 0; hf < D / 32; ++hf) {
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
      mbar_arrive(&bars->p_full[x]);
    }

    // ---- epilogue: O / l -> 16 bit -> shared -> TMA store; logsumexp
    if (!named_bar_or(1 + x, 128, !ok || bars->abort)) {
      // the last PV of the slot (warp-uniform: warp_wait agrees across the warp)
      const bool have = S.n > 0 && warp_wait(&bars->pv_done[x], (uint32_t)(S.n - 1) & 1u, ctl);
      if (have) tc_fence_after();
      const float inv = l_rnd > 0.f ? 1.f / l_rnd : 0.f;
      const bool row_ok = i < a.N && S.qt < a.nq;
      const size_t row = (size_t)(b * a.H + h) * a.N + i;
      uint8_t* ob = smem + C::kQ + x * TB;      // Q_x is dead once O_x is final
      // 64 columns at a time: tensor memory -> O / l -> 16 bit -> swizzled box hh
#pragma unroll 1
      for (int hh = 0; hh < NC; ++hh) {
        float o[64];
        if (have) {
          uint32_t raw[2][32];
          tmem_ld32(tO + hh * 64, raw[0]);
          tmem_ld32(tO + hh * 64 + 32, raw[1]);
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
          const uint32_t off = hh * 16384 + r * 128 + (((j ^ r) & 7) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                       :: "r"(smem_u32(ob + off)), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
        }
        if (row_ok && a.o_f32 != nullptr) {
          float4* dst = reinterpret_cast<float4*>(a.o_f32 + row * D + hh * 64);
#pragma unroll
          for (int c = 0; c < 16; ++c) dst[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + x, 128);
      if (r == 0 && S.qt < a.nq) {
#pragma unroll
        for (int hh = 0; hh < NC; ++hh) tma_store_4d(&tmO, ob + hh * 16384, hh * 64, S.qt * kTile, h, b);
        bulk_commit();
        bulk_wait_read0();
      }
      if (row_ok) a.lse[row] = l_true > 0.f ? (m_run + lg2(l_true)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <typename T, int D, bool kDrop, bool kWin>
cudaError_t launch_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                     const FwdArgs& a, cudaStream_t s) {
  auto kern = fwd_tc_kernel<T, D, kDrop, kWin>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<D>::kDyn);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(a.npairs * a.B * a.H);
  if (grid == 0) return cudaSuccess;
  kern<<<grid, kThreads, FwdCfg<D>::kDyn, s>>>(q, k, v, o, a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_d(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                     const FwdArgs& a, cudaStream_t s) {
  const int sel = (a.drop.enabled ? 1 : 0) | (a.mask.window > 0 ? 2 : 0);
  switch (sel) {
    case 0: return launch_t<T, D, false, false>(q, k, v, o, a, s);
    case 1: return launch_t<T, D, true, false>(q, k, v, o, a, s);
    case 2: return launch_t<T, D, false, true>(q, k, v, o, a, s);
    default: return launch_t<T, D, true, true>(q, k, v, o, a, s);
  }
}

}  // namespace

// Head dimension 64 has two forward kernels.  The one-tile kernel
// (fwd_tc1.cu: one query tile per CTA, two CTAs per SM) overlaps each CTA's
// pipeline fill and drain with the other CTA's steps, and its finer grid
// fills the SMs better; it wins wherever rows are short or the grid is small.
// This two-tile kernel shares every K/V tile between its two query tiles,
// halving the L2 -> shared-memory traffic, which long rows make the limit:
// it is used when the query tiles average at least 64 key tiles (dense or
// causal, no window, no block mask) and there are at least four waves of
// work (same-box measurements: N = 1,024 ... 32,768 causal with B*H down to
// 1, the one-tile kernel 2-21 % faster; N = 23,400 with 12 heads, 5 % slower).
bool use_two_tile_d64(const FwdArgs& a) {
  if (a.fwd_kernel == 1 || a.fwd_kernel == 2) return a.fwd_kernel == 2;
  if (a.mask.window > 0 || a.mask.row_list != nullptr) return false;
  const int avg_tiles = a.mask.causal ? (a.nq + 1) / 2 : a.nq;
  if (avg_tiles < 64) return false;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  return (long long)a.npairs * a.B * a.H >= 4ll * sms;
}

cudaError_t launch_fwd_tc(int dtype, int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& o, const FwdArgs& a, cudaStream_t s) {
  if (d == 64 && !use_two_tile_d64(a)) return launch_fwd_tc1(dtype, q, k, v, o, a, s);
  if (dtype == FA_DT_BF16)
    return d == 128 ? launch_d<__nv_bfloat16, 128>(q, k, v, o, a, s) : launch_d<__nv_bfloat16, 64>(q, k, v, o, a, s);
  return d == 128 ? launch_d<__half, 128>(q, k, v, o, a, s) : launch_d<__half, 64>(q, k, v, o, a, s);
}

}  // namespace fa
