// fwd_fp8.cu -- FP8 (E4M3) attention forward on sm_103a, head dimension 64 or 128.
//
// Method: the Q-outer online-softmax forward of fwd_tc.cu (lynx-cortex, "El
// algoritmo Flash (forward)"; marketmaker.cc, "O algoritmo de atencao do
// Flash"; causal / padded / sparse tiles skipped) run on operands that
// fp8_quant.cu quantised block by block after the random rotation
// (living-dl-book, "Atencao Eficiente em Escala", section 10;
// marketmaker.cc, "FA3: Mecanica da tremonha", item 3).  Both products run
// on the tensor cores in E4M3 (tcgen05.mma kind::f8f6f4):
//
//   S   = Q8 K8^T                  M = 128, N = 128, K = D    (D / 32 MMAs of K 32)
//   O' += A V8 (A = P8, V8^T)      M = 128, N = D,   K = 128  (4 MMAs of K 32)
//
// Scales: the scores of query tile i and key tile t are
// tau * sq_i * sk_t * (Q8 K8^T), folded into the softmax's exponent
// multiplier per step.  The probabilities of key tile t are rounded to E4M3
// as A = E4M3(exp(S - m) * 256 * sv_t / SV), SV the largest V scale of the
// head, so that one float32 accumulator serves every key tile whatever its
// V scale; m is the running row max, moved (and O rescaled) whenever it
// grows, so exp(S - m) <= 1 and A <= 256 < 448.  The row sum l uses the
// unrounded probabilities.  At the end O' = (SV / 256) acc / l is rotated
// back, O = (O' H_D) o s / sqrt(D), and stored in the input's 16-bit type.
//
// GB300 mapping: as fwd_tc.cu -- one CTA holds two 128-row query tiles of
// one head; warp 8 streams K8 / V8^T tiles (D x 128 bytes each) with TMA into a ring;
// warp 9 issues S for both slots; warps 10 / 11 issue the P V products; warps
// 0-3 / 4-7 are the softmax of slot 0 / 1, one thread per row.  The E4M3
// probabilities go to shared memory (128-byte swizzle, K-major), not to
// tensor memory, so both operands of the second product come from shared
// memory.  Tensor memory per slot: S 128 columns | O D.  Q8 / K8 rows are
// D bytes: 64-byte swizzle for D = 64, 128-byte swizzle for D = 128.
#include "common.cuh"
#include "fp8.cuh"
#include "fwd_plan.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kPScale = 256.f;

template <int D>
struct Fp8Cfg {
  static constexpr int kQT = kTile * D;        // Q8 / K8 tile: 128 rows x D bytes
  static constexpr int kVT = D * kTile;        // V8^T tile: D rows x 128 bytes (128-byte swizzle)
  static constexpr int kPT = kTile * kTile;    // P8 tile: 128 rows x 128 bytes; also a staging box of O
  static constexpr int NS = D == 64 ? 6 : 4;   // K/V stages
  static constexpr int kQ = 0;                 // 2 Q tiles
  static constexpr int kK = 2 * kQT;           // NS K tiles
  static constexpr int kV = kK + NS * kQT;     // NS V tiles
  static constexpr int kP = kV + NS * kVT;     // 2 P tiles
  static constexpr int kRed = kP + 2 * kPT;    // 8 floats: per-warp maxima of the V scales
  static constexpr int kBar = kRed + 64;
  static constexpr int kBytes = kBar + 512;
  static constexpr int kDyn = kBytes + 1024;   // + alignment slack
};
static_assert(Fp8Cfg<64>::kDyn <= 232448 && Fp8Cfg<128>::kDyn <= 232448, "shared memory over the per-block limit");
static_assert(Fp8Cfg<128>::kK % 1024 == 0 && Fp8Cfg<128>::kV % 1024 == 0 && Fp8Cfg<128>::kP % 1024 == 0 &&
              Fp8Cfg<64>::kK % 1024 == 0 && Fp8Cfg<64>::kV % 1024 == 0 && Fp8Cfg<64>::kP % 1024 == 0,
              "tiles are 1024-B aligned");

template <int NS>
struct Fp8Bars {
  uint64_t q_full;
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t done[3];
  uint64_t k_full[NS], v_full[NS], k_empty[NS], v_empty[NS];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Fp8Bars<6>) <= 512, "barrier block overflows its shared-memory slot");

// Shared-memory descriptor of a Q8 / K8 tile (rows of D bytes, K-major).
template <int D>
__device__ __forceinline__ uint64_t qk_desc(uint32_t saddr) {
  return D == 64 ? sdesc_sw64(saddr, 512) : sdesc_sw128(saddr, 16, 1024);
}

template <int D, bool kWin>
__global__ void __launch_bounds__(kThreads, 1)
fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
               const FwdArgs a) {
  using C = Fp8Cfg<D>;
  constexpr int NS = C::NS;
  constexpr uint32_t kColO = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Fp8Bars<NS>* bars = reinterpret_cast<Fp8Bars<NS>*>(smem + C::kBar);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (b, h, pair of query tiles); heaviest pairs launch first
  const int BH = a.B * a.H;
  const int pair = a.npairs - 1 - (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / a.H, h = bh % a.H;
  const int hk = h / a.group;
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

  if (warp >= 8) {
   regs_dec<56>();
   if (warp == 8) {
    // ===================== TMA producer =====================
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const uint32_t qbytes = (sl[0].n > 0 ? (uint32_t)C::kQT : 0u) + (sl[1].n > 0 ? (uint32_t)C::kQT : 0u);
      if (qbytes > 0) {
        mbar_expect_tx(&bars->q_full, qbytes);
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (sl[x].n > 0) tma_load_4d(smem + C::kQ + x * C::kQT, &tmQ, &bars->q_full, 0, sl[x].qt * kTile, h, b);
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
          mbar_expect_tx(&bars->k_full[st], C::kQT);
          tma_load_4d(smem + C::kK + st * C::kQT, &tmK, &bars->k_full[st], 0, p.kv[l] * kTile, hk, b);
          mbar_expect_tx(&bars->v_full[st], C::kVT);
          tma_load_4d(smem + C::kV + st * C::kVT, &tmV, &bars->v_full[st], p.kv[l] * kTile, 0, hk, b);
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
      constexpr uint32_t idS = idesc_e4m3(128, 128);
      const uint64_t qd[2] = {qk_desc<D>(smem_u32(smem + C::kQ)), qk_desc<D>(smem_u32(smem + C::kQ + C::kQT))};
      const uint64_t kd0 = qk_desc<D>(smem_u32(smem + C::kK));
      bool ok = mbar_wait(&bars->q_full, 0, ctl);
      int ld = 0;
      for (int s = 0; s < smax && ok; ++s) {
        const StepPlan p = plan_step<NS, kWin>(sl, s, ld);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!ok || s >= sl[x].n) continue;
          const int l = p.use[x];
          // S_x(s) overwrites S_x(s-1) once the softmax has read it
          if (s > 0 && !(ok = mbar_wait(&bars->s_free[x], (uint32_t)(s - 1) & 1u, ctl))) break;
          if (!(ok = mbar_wait(&bars->k_full[p.stage(l)], p.parity(l), ctl))) break;
          tc_fence_after();
          const uint64_t kd = kd0 + (uint64_t)((p.stage(l) * C::kQT) >> 4);
          const uint32_t tS = tmem + x * 256;
          // K-dim = D bytes in steps of 32 within the D-byte rows
#pragma unroll
          for (int k = 0; k < D / 32; ++k) mma_ss_e4m3(tS, qd[x] + 2 * k, kd + 2 * k, idS, k > 0 ? 1u : 0u);
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
    // ===================== P V issuer of slot x =====================
    const int x = warp - 10;
    if (lane == 0 && smax > 0) {
      constexpr uint32_t idPV = idesc_e4m3(128, D);
      const uint64_t pd = sdesc_sw128(smem_u32(smem + C::kP + x * C::kPT), 16, 1024);
      const uint64_t vd0 = sdesc_sw128(smem_u32(smem + C::kV), 16, 1024);
      const uint32_t tO = tmem + x * 256 + kColO;
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
          const uint64_t vd = vd0 + (uint64_t)((st * C::kVT) >> 4);
          // K-dim = 128 keys in four steps of 32 bytes within the 128-byte rows
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_ss_e4m3(tO, pd + 2 * k, vd + 2 * k, idPV, (s > 0 || k > 0) ? 1u : 0u);
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
    const uint32_t tS = tmem + x * 256 + lane_off, tO = tS + kColO;
    const int jmax = a.mask.causal ? min(Lk - 1, i) : (Lk - 1);
    const int jmin = kWin ? i - a.mask.window + 1 : 0;
    const int nt = a.f8.nt;
    const float* skp = a.f8.sk + (size_t)(b * (a.H / a.group) + hk) * nt;
    const float* svp = a.f8.sv + (size_t)(b * (a.H / a.group) + hk) * nt;
    const float sq = S.qt < a.nq ? a.f8.sq[(size_t)bh * nt + S.qt] : 0.f;
    const float sl2q = a.scale_log2 * sq;

    // SV: the largest V scale of the head, over the 256 softmax threads
    float* red = reinterpret_cast<float*>(smem + C::kRed);
    {
      float m = 0.f;
      for (int t = (int)threadIdx.x; t < nt; t += 256) m = fmaxf(m, svp[t]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) red[warp] = m;
      named_bar_sync(3, 256);
    }
    float SV = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) SV = fmaxf(SV, red[w]);
    const float inv_sv = SV > 0.f ? kPScale / SV : 0.f;
    uint8_t* pt = smem + C::kP + x * C::kPT;
    const uint32_t prow = smem_u32(pt + r * 128);

    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int s = 0; s < S.n; ++s) {
      const int kv = S.kv<kWin>(s);
      const float sl2 = fmaxf(sl2q * skp[kv], 1.17549435e-38f);   // > 0, so -inf * sl2 = -inf
      const float ct = svp[kv] * inv_sv;                            // 256 sv_t / SV
      if (!(ok = warp_wait(&bars->s_full[x], (uint32_t)s & 1u, ctl))) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, sr[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) reg_fence32(sr[cc]);
      tc_fence_before();
      mbar_arrive(&bars->s_free[x]);   // S_x(s+1) may now overwrite the S columns

      const int jl = jmax - kv * kTile;
      const int jlo = jmin - kv * kTile;
      if (jl < kTile - 1 || (kWin && jlo > 0)) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > jl || (kWin && c < jlo)) sr[c >> 5][c & 31] = __float_as_uint(-INFINITY);
      }
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
      const float mx = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * sl2;
      // exact running max: exp(S - m) <= 1, so the E4M3 probabilities stay <= 256
      const float m_new = fmaxf(m_run, mx);
      const bool rescale = (m_new > m_run) && (m_run != -INFINITY);
      const float alpha = rescale ? ex2(m_run - m_new) : 1.f;
      m_run = m_new;
      l_run *= alpha;
      const float nmref = (m_run == -INFINITY) ? 0.f : -m_run;

      // The E4M3 codes of the whole row go into registers first; PV(s-1)
      // must be done before the P tile is rewritten and O rescaled, and the
      // wait for it comes only then, after this step's exponentials (its
      // chain of dependent MMAs, issued at the end of the previous step, stays
      // off the softmax's path).
      float lt[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t w[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {             // 16 keys (one 16-byte chunk) at a time
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int c = j * 16 + q4 * 4;
          float x0, x1, x2, x3;
          fma2(x0, x1, __uint_as_float(sr[c >> 5][c & 31]), __uint_as_float(sr[(c + 1) >> 5][(c + 1) & 31]), sl2,
               sl2, nmref, nmref);
          fma2(x2, x3, __uint_as_float(sr[(c + 2) >> 5][(c + 2) & 31]),
               __uint_as_float(sr[(c + 3) >> 5][(c + 3) & 31]), sl2, sl2, nmref, nmref);
          float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
          add2(lt[(q4 & 1) * 2], lt[(q4 & 1) * 2 + 1], p0, p1);
          add2(lt[(q4 & 1) * 2], lt[(q4 & 1) * 2 + 1], p2, p3);
          mul2(p0, p1, p0, p1, ct, ct);
          mul2(p2, p3, p2, p3, ct, ct);
          w[j][q4] = e4m3x4(p0, p1, p2, p3);
        }
      }
      if (s > 0 && !(ok = warp_wait(&bars->pv_done[x], (uint32_t)(s - 1) & 1u, ctl))) break;
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     :: "r"(prow + (((uint32_t)(j ^ r) & 7u) << 4)), "r"(w[j][0]), "r"(w[j][1]), "r"(w[j][2]),
                        "r"(w[j][3]) : "memory");
      l_run += (lt[0] + lt[1]) + (lt[2] + lt[3]);
      fence_proxy_async_smem();   // the P tile is read by the tensor core (async proxy)
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
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(&bars->p_full[x]);
    }

    // ---- epilogue: O' (SV / 256) / l -> rotate back -> 16 bit -> shared -> TMA store; logsumexp
    if (!named_bar_or(1 + x, 128, !ok || bars->abort)) {
      const bool have = S.n > 0 && warp_wait(&bars->pv_done[x], (uint32_t)(S.n - 1) & 1u, ctl);
      if (have) tc_fence_after();
      const float post = l_run > 0.f ? (SV / kPScale) / l_run : 0.f;
      const bool row_ok = i < a.N && S.qt < a.nq;
      const size_t row = (size_t)(b * a.H + h) * a.N + i;
      float o[D];
      if (have) {
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          uint32_t raw[2][32];
          tmem_ld32(tO + hf * 64, raw[0]);
          tmem_ld32(tO + hf * 64 + 32, raw[1]);
          tmem_wait_ld();
          reg_fence32(raw[0]);
          reg_fence32(raw[1]);
#pragma unroll
          for (int c = 0; c < 64; ++c) o[hf * 64 + c] = __uint_as_float(raw[c >> 5][c & 31]) * post;
        }
      } else {
#pragma unroll
        for (int c = 0; c < D; ++c) o[c] = 0.f;
      }
      if (a.f8.signs != nullptr) {
        // O = O' M^T = (O' H) o s / sqrt(D)
        fwht_rows<D>(o);
        const float sc = D == 64 ? 0.125f : __int_as_float(0x3db504f3);
        const uint4* sp = reinterpret_cast<const uint4*>(a.f8.signs);
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          const uint4 u = sp[j];
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int8_t sg = (int8_t)((w4[c >> 2] >> ((c & 3) * 8)) & 0xFFu);
            o[16 * j + c] *= (sg < 0 ? -sc : sc);
          }
        }
      }
      // 64-column boxes of O staged in the slot's P tile (free once its last
      // P V product is done) and, for D = 128, its Q tile (free once its last S is)
      uint8_t* obox[2] = {pt, smem + C::kQ + x * C::kQT};
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t w[4];
          const int c0 = hh * 64 + j * 8;
          if (a.f8.o_bf16) {
#pragma unroll
            for (int t = 0; t < 4; ++t) w[t] = Cvt<__nv_bfloat16>::pack(o[c0 + 2 * t], o[c0 + 2 * t + 1]);
          } else {
#pragma unroll
            for (int t = 0; t < 4; ++t) w[t] = Cvt<__half>::pack(o[c0 + 2 * t], o[c0 + 2 * t + 1]);
          }
          const uint32_t off = r * 128 + (((j ^ r) & 7) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                       :: "r"(smem_u32(obox[hh] + off)), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
        }
      }
      if (row_ok && a.o_f32 != nullptr) {
        float4* dst = reinterpret_cast<float4*>(a.o_f32 + row * D);
#pragma unroll
        for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + x, 128);
      if (r == 0 && S.qt < a.nq) {
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) tma_store_4d(&tmO, obox[hh], hh * 64, S.qt * kTile, h, b);
        bulk_commit();
        bulk_wait_read0();
      }
      if (row_ok) a.lse[row] = l_run > 0.f ? (m_run + lg2(l_run)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kWin>
cudaError_t launch_w(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                     const FwdArgs& a, cudaStream_t s) {
  auto kern = fwd_fp8_kernel<D, kWin>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Fp8Cfg<D>::kDyn);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(a.npairs * a.B * a.H);
  if (grid == 0) return cudaSuccess;
  kern<<<grid, kThreads, Fp8Cfg<D>::kDyn, s>>>(q, k, v, o, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp8(int d, const CUtensorMap& q8, const CUtensorMap& k8, const CUtensorMap& v8t,
                           const CUtensorMap& o, const FwdArgs& a, cudaStream_t s) {
  if (d == 128)
    return a.mask.window > 0 ? launch_w<128, true>(q8, k8, v8t, o, a, s) : launch_w<128, false>(q8, k8, v8t, o, a, s);
  return a.mask.window > 0 ? launch_w<64, true>(q8, k8, v8t, o, a, s) : launch_w<64, false>(q8, k8, v8t, o, a, s);
}

}  // namespace fa
