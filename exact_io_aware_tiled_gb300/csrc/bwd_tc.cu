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
// Grouped-query attention (living-dl-book, "Atencao eficiente", section 6):
// dK and dV of a K/V head shared by g query heads sum over those heads.  The
// sliding window (lynx-cortex, "Problemas de practica") limits the query
// tiles that see a key tile and masks the window's far edge.
//
// GB300 mapping (ours): a persistent kernel, one CTA per SM.  The work items
// are (b, K/V head, 128-key tile) in head-major order; each CTA takes the
// next one from a global counter as it goes (its producer thread fetches it
// and hands it to the other roles through a two-slot shared-memory mailbox),
// so CTAs that drew short items take more, and the CTAs working at one time
// cover a few adjacent heads, whose Q / dO tiles and dQ accumulator rows
// stay in L2.  Per item the CTA
// loops over the query tiles that see the key tile, for each query head of
// the group, so dK and dV accumulate over the group in tensor memory.  The
// steps of consecutive items form one global sequence: every ring and
// barrier phase runs on the global step index, K is double-buffered so the
// next item's K load overlaps the current item (V, needed later in a step,
// has one buffer, reloaded as soon as the last dP^T of an item has read it),
// and an item's dK, dV leave tensor memory while the next item starts.
//   * warp 16: TMA loads of K, V per item and of Q_i, dO_i (+ LSE_i, D_i
//     rows) per step into a three-stage ring (the Q / dO loads are latency-
//     bound: with two stages a step often waited for its tiles), and, three
//     steps behind, the two TMA reduce-adds of each staged dQ_i into the
//     float32 accumulator;
//   * three MMA-issuing warps (one thread each): consecutive MMAs into the
//     same accumulator complete about 126 cycles apart whatever their N, so
//     each product is a latency chain, and independent chains are issued
//     from separate warps so that they overlap:
//       warp 17: S^T(i) = K Q_i^T and dP^T(i) = V dO_i^T, each as soon as
//                the softmax warps have read the previous one;
//       warp 18: dV += P~^T dO_i (A from tensor memory) and
//                dK += dS^T Q_i (A from the shared dS^T tile);
//       warp 19: dQ_i = dS K (A = the same tile read MN-major);
//   * warps 0-15: four warpgroups, each owning 32 of the 128 query columns
//     of every key row (= tensor-memory lane):
//       part 1: P from S^T, P~^T (16 bit) into tensor memory for dV;
//       part 2: dS from dP^T, dS^T (16 bit) into a swizzled shared tile
//               that both dK and dQ read (bf16: tau dS, so that dK and dQ
//               come out scaled);
//       drain:  16 of the 64 columns of dQ_i from tensor memory (x tau for
//               fp16) -> shared staging (in the following step);
//       item end: 16 of the 64 columns of dK (x tau for fp16) and dV from
//               tensor memory straight to global memory (with dropout:
//               dK or dV, 16 key rows a warp, as whole 128-byte rows).
// Tensor memory (512 columns):
//   S^T 0-127 | dP^T 128-255 | dK 256-319 | dV 320-383 | dQ 384-447 |
//   P~^T (16 bit, queries 32w..32w+31 packed at 448+16w .. +16) 448-511.
// Registers: 96 a thread (640 threads, one CTA per SM).
#include <algorithm>
#include <type_traits>

#include "bwd_items.cuh"

namespace fa {
namespace {

constexpr int kThreads = 640;
constexpr int kCompute = 512;   // threads of warps 0-15
constexpr int NSB = 3;   // Q / dO stages
constexpr int NSTG = 1;  // float32 dQ staging buffers
constexpr int kLag = 3;  // dQ reduce-adds trail the loads by this many steps

struct BwdSmem {
  static constexpr int kK = 0;                      // 2 x 16 KB (double-buffered per item)
  static constexpr int kV = 32768;                  // 16 KB
  static constexpr int kQ = 49152;                  // NSB x 16 KB
  static constexpr int kDO = kQ + NSB * 16384;      // NSB x 16 KB
  static constexpr int kDS = kDO + NSB * 16384;     // 32 KB: dS^T [2 chunks][128 keys][64 q]
  static constexpr int kDQ = kDS + 32768;           // NSTG x 32 KB: float32 dQ staging [buf][half][128][32]
  static constexpr int kLD = kDQ + NSTG * 32768;    // NSB x (LSE2[128] + D[128]) floats
  static constexpr int kInfo = kLD + NSB * 1024;    // (query tile, query head, batch) of the last kLag+1 steps
  static constexpr int kItem = kInfo + 64;          // the two published work items
  static constexpr int kBar = kItem + 64;
  static constexpr int kBytes = kBar + 320;
  static constexpr int kDyn = kBytes + 1024;
};

struct BBars {
  uint64_t item_full[2], item_empty[2];   // the work-item hand-off from warp 16 to the other roles
  uint64_t k_full[2], k_empty[2], v_full, v_empty;
  uint64_t q_full[NSB], q_empty[NSB];
  uint64_t s_full, p_full, dp_full, ds_full, dq_full, dq_free, dkv_full, pt_free;
  uint64_t dsm_free;
  uint64_t done[3];
  uint64_t stg_full[NSTG], stg_free[NSTG];
  uint32_t tmem_base;
  int abort;
};

static_assert(sizeof(BBars) <= 320, "barrier block overflows its shared-memory slot");
static_assert(BwdSmem::kDyn <= 232448, "shared memory over the per-block limit");

constexpr uint32_t kColST = 0, kColDP = 128, kColDK = 256, kColDV = 320, kColDQ = 384, kColPT = 448;

template <typename T, bool kDrop, bool kWin>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmDQ, const BwdArgs a) {
  using L = BwdSmem;
  // bf16: tau is folded into dS (the D rows hold -tau * D, and part 2 forms
  // (tau dP - tau D) o P with one packed FMA), so dQ and dK leave the tensor
  // core already scaled.  At the usual tau = 2^-3 that is exact.  Not for
  // fp16, whose smaller range would push small dS values into subnormals.
  constexpr bool kFold = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BBars* bars = reinterpret_cast<BBars*>(smem + L::kBar);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total = a.nq * a.B * a.H_kv;
  WaitCtl ctl{a.status, &bars->abort};

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->item_full[s], 1);
      mbar_init(&bars->item_empty[s], 3 + kCompute);   // warps 17-19 and the compute threads
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 2);    // S^T warp and dQ warp read K
    }
    for (int s = 0; s < NSB; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, kCompute);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->ds_full, kCompute);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, kCompute);
    mbar_init(&bars->dkv_full, 1);
    mbar_init(&bars->v_full, 1);
    mbar_init(&bars->v_empty, 1);        // dP^T warp reads V
    mbar_init(&bars->pt_free, 1);
    mbar_init(&bars->dsm_free, 2);     // dK and dQ both read the shared dS^T tile
    for (int i = 0; i < 3; ++i) mbar_init(&bars->done[i], 1);
    for (int i = 0; i < NSTG; ++i) {
      mbar_init(&bars->stg_full[i], kCompute);
      mbar_init(&bars->stg_free[i], 1);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 17) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= 16) {
    constexpr int ab = Cvt<T>::kAB;
    constexpr uint32_t idST = idesc_f16(128, 128, ab, 0, 0);   // S^T, dP^T (both operands K-major)
    constexpr uint32_t idKV = idesc_f16(128, 64, ab, 0, 1);    // dV, dK (A K-major or in tensor memory, B MN-major)
    constexpr uint32_t idQ = idesc_f16(128, 64, ab, 1, 1);     // dQ (A MN-major, B MN-major)
    const uint32_t sQ = smem_u32(smem + L::kQ), sDO = smem_u32(smem + L::kDO);
    const uint32_t sDS = smem_u32(smem + L::kDS);
    volatile int* item_u = reinterpret_cast<volatile int*>(smem + L::kItem);
    // the next work item from warp 16's mailbox (-1: no more, or a wait gave up)
    int kc = 0;
    auto fetch = [&]() -> int {
      const int slot = kc & 1;
      if (!mbar_wait(&bars->item_full[slot], (uint32_t)(kc >> 1) & 1u, ctl)) return -1;
      const int v = item_u[slot];
      mbar_arrive(&bars->item_empty[slot]);
      ++kc;
      return v;
    };
    if (warp == 16) {
      // ===================== TMA producer + dQ reduce =====================
      // The loads of step g and the reduce of the staged dQ of step g - kLag
      // run interleaved in one thread.  The reduce of step r can only be
      // staged after the load of step r + 1, and the load of step g needs,
      // through the compute chain, the reduce of step g - 5; so this order
      // never waits on itself.
      if (lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmDO);
        prefetch_tmap(&tmDQ);
        int4* info = reinterpret_cast<int4*>(smem + L::kInfo);
        int g = 0, nkv = 0;
        bool ok = true;
        auto reduce = [&](int r) -> bool {
          const int bi = r % NSTG;
          if (!mbar_wait(&bars->stg_full[bi], (uint32_t)(r / NSTG) & 1u, ctl)) return false;
          const uint8_t* sb = smem + L::kDQ + bi * 32768;
          const int4 inf = info[r & 3];
          tma_reduce_add_4d(&tmDQ, sb, 0, inf.x * kTile, inf.y, inf.z);
          tma_reduce_add_4d(&tmDQ, sb + 16384, 32, inf.x * kTile, inf.y, inf.z);
          bulk_commit();
          bulk_wait_read0();
          mbar_arrive(&bars->stg_free[bi]);
          return true;
        };
        // the next item from the global counter, handed to the other roles
        // through the two-slot mailbox (-1: none left; -2: a wait gave up)
        int kf = 0;
        auto publish = [&]() -> int {
          const int slot = kf & 1;
          if (!mbar_wait(&bars->item_empty[slot], ((uint32_t)(kf >> 1) & 1u) ^ 1u, ctl)) return -2;
          int v = atomicAdd(a.sched, 1);
          if (v >= total) v = -1;
          item_u[slot] = v;
          mbar_arrive(&bars->item_full[slot]);
          ++kf;
          return v;
        };
        // reduces run in step order; rd is the next one owed
        int rd = 0;
        auto reduce_to = [&](int last) -> bool {
          for (; rd <= last; ++rd)
            if (!reduce(rd)) return false;
          return true;
        };
        int u;
        while (ok) {
          // Without dropout the reduce owed here goes before the next item is
          // claimed, so the producer claims it and issues its first loads only
          // once the compute threads have drained dQ of the current item's
          // third-last step.  That later claim was measured faster for short
          // items (a reduce done first only when already possible was not);
          // with dropout's longer steps it was slower.
          if constexpr (!kDrop) {
            if (!(ok = reduce_to(g - kLag))) break;
          }
          u = publish();
          if (u < 0) {
            ok = u == -1;
            break;
          }
          const Item it = make_item(a, u);
          if (it.steps == 0) {
            // An empty item loads nothing, so the reduce that normally follows
            // a load is not reached; do the reduces the compute threads need to
            // finish their current item (through step g - 3), or a run of empty
            // items would fill the mailbox while they wait for one.
            ok = reduce_to(g - 3);
            continue;
          }
          const int kb = nkv & 1;
          if (!(ok = mbar_wait(&bars->k_empty[kb], ((uint32_t)(nkv >> 1) & 1u) ^ 1u, ctl))) break;
          mbar_expect_tx(&bars->k_full[kb], 16384);
          tma_load_4d(smem + L::kK + kb * 16384, &tmK, &bars->k_full[kb], 0, it.jt * kTile, it.hk, it.b);
          const int vi = nkv;
          ++nkv;
          int qu = 0, hq = it.h0;
          for (int t = 0; t < it.steps && ok; ++t, ++g) {
            const int st = g % NSB;
            if (!(ok = mbar_wait(&bars->q_empty[st], ((uint32_t)(g / NSB) & 1u) ^ 1u, ctl))) break;
            const int qi = it.qt(qu);
            const size_t ld_row = ((size_t)it.b * a.H + hq) * a.npad + (size_t)qi * kTile;
            mbar_expect_tx(&bars->q_full[st], 32768 + 1024);
            tma_load_4d(smem + L::kQ + st * 16384, &tmQ, &bars->q_full[st], 0, qi * kTile, hq, it.b);
            tma_load_4d(smem + L::kDO + st * 16384, &tmDO, &bars->q_full[st], 0, qi * kTile, hq, it.b);
            bulk_load(smem + L::kLD + st * 1024, a.lse2 + ld_row, 512, &bars->q_full[st]);
            bulk_load(smem + L::kLD + st * 1024 + 512, a.dvec + ld_row, 512, &bars->q_full[st]);
            info[g & 3] = make_int4(qi, hq, it.b, 0);
            if (t == 0) {
              // V has one buffer: it is reloaded once the previous item's last dP^T is done
              if (!(ok = mbar_wait(&bars->v_empty, ((uint32_t)vi & 1u) ^ 1u, ctl))) break;
              mbar_expect_tx(&bars->v_full, 16384);
              tma_load_4d(smem + L::kV, &tmV, &bars->v_full, 0, it.jt * kTile, it.hk, it.b);
            }
            if (++qu == it.n) { qu = 0; ++hq; }
            if (!(ok = reduce_to(g - kLag))) break;
          }
        }
        // the reduces still owed, then no copy may still be in flight
        if (ok) ok = reduce_to(g - 1);
        for (int t = max(0, g - NSB); t < g; ++t) mbar_wait(&bars->q_full[t % NSB], (uint32_t)(t / NSB) & 1u, ctl);
        for (int t = max(0, nkv - 2); t < nkv; ++t) mbar_wait(&bars->k_full[t & 1], (uint32_t)(t >> 1) & 1u, ctl);
        if (nkv > 0) mbar_wait(&bars->v_full, (uint32_t)(nkv - 1) & 1u, ctl);
        bulk_wait_read0();
      }
    } else if (warp == 17) {
      // ===================== S^T / dP^T issuer =====================
      if (lane == 0) {
        int g = 0, nkv = 0;
        bool ok = true;
        int u;
        while (ok && (u = fetch()) >= 0) {
          const Item it = make_item(a, u);
          if (it.steps == 0) continue;
          const int kb = nkv & 1;
          if (!(ok = mbar_wait(&bars->k_full[kb], (uint32_t)(nkv >> 1) & 1u, ctl))) break;
          const int vi = nkv;
          ++nkv;
          const uint32_t sK = smem_u32(smem + L::kK + kb * 16384), sV = smem_u32(smem + L::kV);
          for (int t = 0; t < it.steps && ok; ++t, ++g) {
            const int st = g % NSB;
            // S^T(g) = K Q_g^T once part 1 of step g-1 has read S^T(g-1)
            if (g > 0 && !(ok = mbar_wait(&bars->p_full, (uint32_t)(g - 1) & 1u, ctl))) break;
            if (!(ok = mbar_wait(&bars->q_full[st], (uint32_t)(g / NSB) & 1u, ctl))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(tmem + kColST, sdesc_sw128(sK + k * 32, 16, 1024), sdesc_sw128(sQ + st * 16384 + k * 32, 16, 1024),
                     idST, k > 0 ? 1u : 0u);
            mma_commit(&bars->s_full);
            // dP^T(g) = V dO_g^T once part 2 of step g-1 has read dP^T(g-1)
            if (g > 0 && !(ok = mbar_wait(&bars->ds_full, (uint32_t)(g - 1) & 1u, ctl))) break;
            if (t == 0 && !(ok = mbar_wait(&bars->v_full, (uint32_t)vi & 1u, ctl))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(tmem + kColDP, sdesc_sw128(sV + k * 32, 16, 1024), sdesc_sw128(sDO + st * 16384 + k * 32, 16, 1024),
                     idST, k > 0 ? 1u : 0u);
            mma_commit(&bars->dp_full);
          }
          mma_commit(&bars->k_empty[kb]);    // this item's S^T are done with K
          mma_commit(&bars->v_empty);        // and its dP^T with V
        }
        mma_commit(&bars->done[0]);
        mbar_wait(&bars->done[0], 0, ctl);
      }
    } else if (warp == 18) {
      // ===================== dV / dK issuer =====================
      // The first dV / dK of an item restart the accumulators; they follow
      // p_full / ds_full of that step, which the compute warps arrive at only
      // after reading the previous item's dK and dV out of tensor memory.
      if (lane == 0) {
        int g = 0;
        bool ok = true;
        int u;
        while (ok && (u = fetch()) >= 0) {
          const Item it = make_item(a, u);
          if (it.steps == 0) continue;
          for (int t = 0; t < it.steps && ok; ++t, ++g) {
            const int st = g % NSB;
            const uint32_t qb = sQ + st * 16384, db = sDO + st * 16384;
            // dV += P~^T dO_g  (A = P~^T in tensor memory; K-dim = 128 queries, 8 steps of 16)
            if (!(ok = mbar_wait(&bars->p_full, (uint32_t)g & 1u, ctl) &&
                       mbar_wait(&bars->q_full[st], (uint32_t)(g / NSB) & 1u, ctl))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ts(tmem + kColDV, tmem + kColPT + k * 8, sdesc_sw128(db + k * 2048, 16384, 1024), idKV,
                     (t > 0 || k > 0) ? 1u : 0u);
            mma_commit(&bars->pt_free);
            // dK += dS^T Q_g  (A = dS^T from the shared tile, K-major: chunk k / 4, 32 bytes per 16 queries)
            if (!(ok = mbar_wait(&bars->ds_full, (uint32_t)g & 1u, ctl))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ss(tmem + kColDK, sdesc_sw128(sDS + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                     sdesc_sw128(qb + k * 2048, 16384, 1024), idKV, (t > 0 || k > 0) ? 1u : 0u);
            mma_commit(&bars->dsm_free);
            mma_commit(&bars->q_empty[st]);
          }
          mma_commit(&bars->dkv_full);       // this item's dK, dV are final
        }
        mma_commit(&bars->done[1]);
        mbar_wait(&bars->done[1], 0, ctl);
      }
    } else {
      // ===================== dQ issuer (warp 19) =====================
      if (lane == 0) {
        int g = 0, nkv = 0;
        bool ok = true;
        int u;
        while (ok && (u = fetch()) >= 0) {
          const Item it = make_item(a, u);
          if (it.steps == 0) continue;
          const int kb = nkv & 1;
          ++nkv;
          const uint32_t sK = smem_u32(smem + L::kK + kb * 16384);
          for (int t = 0; t < it.steps && ok; ++t, ++g) {
            // dQ_g = dS K  (M = 128 queries from the MN-major view of dS^T, K-dim = 128 keys)
            if (!(ok = mbar_wait(&bars->ds_full, (uint32_t)g & 1u, ctl))) break;
            if (g > 0 && !(ok = mbar_wait(&bars->dq_free, (uint32_t)(g - 1) & 1u, ctl))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ss(tmem + kColDQ, sdesc_sw128(sDS + k * 2048, 16384, 1024),
                     sdesc_sw128(sK + k * 2048, 16384, 1024), idQ, k > 0 ? 1u : 0u);
            mma_commit(&bars->dq_full);
            mma_commit(&bars->dsm_free);
          }
          mma_commit(&bars->k_empty[kb]);    // this item's dQ MMAs are done with K
        }
        mma_commit(&bars->done[2]);
        mbar_wait(&bars->done[2], 0, ctl);
      }
    }
  } else {
    // ===================== softmax-gradient warpgroups =====================
    const int wg = warp >> 2;                 // query columns 32 wg .. 32 wg + 31
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;        // key row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tl = tmem + lane_off;
    const float sl2 = a.scale_log2;
    const int c0 = wg * 32;                   // first query column of this warpgroup
    // 16-byte pieces (w & 1) * 4 .. + 4 of a 128-byte swizzled row belong to this warpgroup
    const int pc_base = (wg & 1) * 4;
    bool ok = true;

    // dQ_t: 16 of its 64 columns, tensor memory -> x tau (fp16; bf16 is
    // already scaled) -> staging buffer t % NSTG
    // (warp 16 reduces it)
    auto drain_dq = [&](int t) -> bool {
      if (!warp_wait(&bars->dq_full, (uint32_t)t & 1u, ctl)) return false;
      tc_fence_after();
      uint32_t g[16];
      tmem_ld16(tl + kColDQ + wg * 16, g);
      tmem_wait_ld();
      reg_fence16(g);
      tc_fence_before();
      mbar_arrive(&bars->dq_free);
      const int bi = t % NSTG;
      if (t >= NSTG && !warp_wait(&bars->stg_free[bi], (uint32_t)((t - NSTG) / NSTG) & 1u, ctl)) return false;
      uint8_t* sb = smem + L::kDQ + bi * 32768 + (wg >> 1) * 16384 + r * 128;
      if constexpr (!kFold) {
#pragma unroll
        for (int e = 0; e < 16; ++e) g[e] = __float_as_uint(__uint_as_float(g[e]) * a.scale);
      }
#pragma unroll
      for (int pc4 = 0; pc4 < 4; ++pc4) {
        const uint32_t off = ((((pc_base + pc4) ^ r) & 7) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                     :: "r"(smem_u32(sb + off)), "r"(g[pc4 * 4]), "r"(g[pc4 * 4 + 1]), "r"(g[pc4 * 4 + 2]),
                        "r"(g[pc4 * 4 + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->stg_full[bi]);
      return true;
    };


    // dK (x tau for fp16) and dV of an item: 16 of the 64 columns of this thread's key
    // row, straight from registers to global memory (32 bytes each).
    auto store_dkv = [&](const Item& it, const uint32_t (&kraw)[16], const uint32_t (&vraw)[16], bool have) {
      const int j = it.jt * kTile + r;
      if (j >= a.N) return;
      const size_t off = (size_t)it.b * a.kst.b + (size_t)it.hk * a.kst.h + (size_t)j * a.kst.n + wg * 16;
      uint32_t wk[8], wv[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float ks = kFold ? 1.f : a.scale;   // bf16: dK is already scaled
        wk[c] = Cvt<T>::pack(have ? __uint_as_float(kraw[2 * c]) * ks : 0.f,
                             have ? __uint_as_float(kraw[2 * c + 1]) * ks : 0.f);
        wv[c] = Cvt<T>::pack(have ? __uint_as_float(vraw[2 * c]) : 0.f, have ? __uint_as_float(vraw[2 * c + 1]) : 0.f);
      }
      if (a.dkv_v8) {
        // one 32-byte store per tensor: whole sectors in one instruction
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                     :: "l"(static_cast<T*>(a.dk) + off), "r"(wk[0]), "r"(wk[1]), "r"(wk[2]), "r"(wk[3]),
                        "r"(wk[4]), "r"(wk[5]), "r"(wk[6]), "r"(wk[7]) : "memory");
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                     :: "l"(static_cast<T*>(a.dv) + off), "r"(wv[0]), "r"(wv[1]), "r"(wv[2]), "r"(wv[3]),
                        "r"(wv[4]), "r"(wv[5]), "r"(wv[6]), "r"(wv[7]) : "memory");
        return;
      }
      uint4* dk = reinterpret_cast<uint4*>(static_cast<T*>(a.dk) + off);
      uint4* dv = reinterpret_cast<uint4*>(static_cast<T*>(a.dv) + off);
      dk[0] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
      dk[1] = make_uint4(wk[4], wk[5], wk[6], wk[7]);
      dv[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      dv[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
    };

    // With dropout, the item end instead has warpgroups 0-1 write dK (x tau
    // for fp16) and 2-3 write dV, each warp 16 key rows of its lane quarter
    // (wg & 1 picks which 16).  The 16x256b tensor-memory shape gives each
    // lane two of every eight columns of two rows; a transpose within each
    // group of four lanes then gives every lane 32 consecutive bytes, so one
    // warp store covers eight whole 128-byte rows instead of a 32-byte piece
    // of 32 rows.  That is faster only when the Philox work fills the compute
    // warps' issue slots (measured); without dropout the 64 shuffles and
    // selects a warp adds cost more than the store transactions they save.
    const bool kv_is_v = wg >= 2;
    const uint32_t kv_taddr = tmem + ((uint32_t)(quarter * 32 + (wg & 1) * 16) << 16) + (kv_is_v ? kColDV : kColDK);
    const int kv_row = quarter * 32 + (wg & 1) * 16 + (lane >> 2);   // rows kv_row and kv_row + 8
    auto store_dkv_rows = [&](const Item& it, const uint32_t (&raw)[32], bool have) {
      uint32_t w[2][8];     // [row][word]
      if (have) {
        const float ks = (!kv_is_v && !kFold) ? a.scale : 1.f;   // bf16: dK is already scaled
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            w[h][k] = Cvt<T>::pack(__uint_as_float(raw[4 * k + 2 * h]) * ks, __uint_as_float(raw[4 * k + 2 * h + 1]) * ks);
          // w[h][k] belongs at byte 16k + 4 (lane & 3) of its row.  As a 4 x 4
          // matrix of word pairs (w[2c], w[2c+1]) over the group's lanes, it is
          // transposed in two exchanges (lane ^ 2, then lane ^ 1), each swapping
          // the pairs whose column bit differs from the lane's bit.
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int lo = (e >> 1) * 2 + (e & 1), hi = lo + 4;   // pair columns 0/1 against 2/3
            const bool b1 = lane & 2;
            const uint32_t got = __shfl_xor_sync(0xffffffffu, b1 ? w[h][lo] : w[h][hi], 2);
            if (b1) w[h][lo] = got; else w[h][hi] = got;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int lo = (e >> 1) * 4 + (e & 1), hi = lo + 2;   // pair columns 0/2 against 1/3
            const bool b0 = lane & 1;
            const uint32_t got = __shfl_xor_sync(0xffffffffu, b0 ? w[h][lo] : w[h][hi], 1);
            if (b0) w[h][lo] = got; else w[h][hi] = got;
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int k = 0; k < 8; ++k) w[h][k] = 0u;
      }
      // lane q of its group now holds, in pair c, row bytes 32q + 4c (word 0)
      // and 32q + 16 + 4c (word 1)
      T* base = static_cast<T*>(kv_is_v ? a.dv : a.dk);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = it.jt * kTile + kv_row + 8 * h;
        if (j >= a.N) continue;
        T* p = base + (size_t)it.b * a.kst.b + (size_t)it.hk * a.kst.h + (size_t)j * a.kst.n + (lane & 3) * 16;
        if (a.dkv_v8) {
          asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                       :: "l"(p), "r"(w[h][0]), "r"(w[h][2]), "r"(w[h][4]), "r"(w[h][6]), "r"(w[h][1]), "r"(w[h][3]),
                          "r"(w[h][5]), "r"(w[h][7]) : "memory");
        } else {
          uint4* q = reinterpret_cast<uint4*>(p);
          q[0] = make_uint4(w[h][0], w[h][2], w[h][4], w[h][6]);
          q[1] = make_uint4(w[h][1], w[h][3], w[h][5], w[h][7]);
        }
      }
    };

    // the next work item from warp 16's mailbox (-1: none left, or a wait gave up)
    volatile int* item_u = reinterpret_cast<volatile int*>(smem + L::kItem);
    int kc = 0;
    auto fetch = [&]() -> int {
      const int slot = kc & 1;
      if (!warp_wait(&bars->item_full[slot], (uint32_t)(kc >> 1) & 1u, ctl)) return -1;
      const int v = item_u[slot];
      mbar_arrive(&bars->item_empty[slot]);
      ++kc;
      return v;
    };
    int t = 0;        // global step
    int nit = 0;      // items with steps (dkv_full phases)
    int u;
    while (ok && (u = fetch()) >= 0) {
      const Item it = make_item(a, u);
      if (it.steps == 0) {            // no query tile sees this key tile: dK = dV = 0
        if constexpr (kDrop) {
          const uint32_t zero[32] = {};
          store_dkv_rows(it, zero, false);
        } else {
          const uint32_t zero[16] = {};
          store_dkv(it, zero, zero, false);
        }
        continue;
      }
      const int j = it.jt * kTile + r;          // global key
      const bool key_ok = j < it.Lk;
      // qu: tile position within the current query head qh of the item;
      // t: the global step (across items), which every ring and phase follows
      int qu = 0, qh = it.h0;
      for (int tt = 0; tt < it.steps && ok; ++tt, ++t, qu = (qu + 1 == it.n) ? 0 : qu + 1, qh += (qu == 0) ? 1 : 0) {
      const int st = t % NSB;
      const int qi = it.qt(qu);
      const uint32_t bh_rows = ((uint32_t)it.b * (uint32_t)a.H + (uint32_t)qh) * (uint32_t)a.N;
        // LSE*log2e and D of this warpgroup's 32 query columns, in shared memory
        const uint32_t s_lse = smem_u32(smem + L::kLD + st * 1024) + c0 * 4;
        const uint32_t s_d = s_lse + 512;
        // query column c of the tile is hidden from this key under causal iff
        // c < qlo, and outside its sliding window iff c >= qhe
        const int qlo = a.mask.causal ? (j - qi * kTile) : -1;
        const int qhe = kWin ? (j + a.mask.window - qi * kTile) : kTile;
        const bool any_mask = !key_ok || qlo > c0 || (kWin && qhe < c0 + 32);

        // ---- part 1: P from S^T, in two halves of 16 query columns; the
        //      tensor-memory load of the second half overlaps the first's math
        if (!(ok = warp_wait(&bars->s_full, (uint32_t)t & 1u, ctl) &&
                   warp_wait(&bars->q_full[st], (uint32_t)(t / NSB) & 1u, ctl))) break;
        tc_fence_after();
        uint32_t sv[2][16];
        tmem_ld16(tl + kColST + c0, sv[0]);
        uint32_t keep = ~0u;
        if constexpr (kDrop) {
          // One Philox call covers 8 consecutive keys of one query row, and the
          // 8 lanes 8m..8m+7 hold 8 consecutive keys (j & 7 == lane & 7).  So
          // lane t of each group evaluates the calls of queries t, t+8, t+16,
          // t+24 (4 instead of 32), packs their 8-key keep bytes into one word,
          // and the group exchanges the words.
          const int t8 = lane & 7;
          uint32_t mine = 0;
  #pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t q = (uint32_t)(qi * kTile + c0 + t8 + 8 * m);
            mine |= dropout_keep8((uint32_t)j >> 3, bh_rows + q, a.drop) << (8 * m);
          }
          uint32_t kb = 0;
  #pragma unroll
          for (int src = 0; src < 8; ++src) {
            const uint32_t w = __shfl_sync(0xffffffffu, mine, (lane & ~7) | src);
  #pragma unroll
            for (int m = 0; m < 4; ++m) kb |= ((w >> (8 * m + t8)) & 1u) << (src + 8 * m);
          }
          keep = kb;
        }
        uint32_t pp[16];      // undropped P, 16 bit, kept for part 2
        uint32_t pt[16];      // P~ = Z o P / (1 - p), 16 bit, operand of dV
  #pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          tmem_wait_ld();
          reg_fence16(sv[hf]);
          if (hf == 0) tmem_ld16(tl + kColST + c0 + 16, sv[1]);
  #pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int cc = hf * 16 + q4 * 4;    // column within this warpgroup's 32
            const float4 l4 = lds128(s_lse + cc * 4);
            float x[4];
            fma2(x[0], x[1], __uint_as_float(sv[hf][q4 * 4]), __uint_as_float(sv[hf][q4 * 4 + 1]), sl2, sl2, -l4.x, -l4.y);
            fma2(x[2], x[3], __uint_as_float(sv[hf][q4 * 4 + 2]), __uint_as_float(sv[hf][q4 * 4 + 3]), sl2, sl2, -l4.z, -l4.w);
            float p[4];
  #pragma unroll
            for (int e = 0; e < 4; ++e) p[e] = ex2(x[e]);
            if (any_mask) {
  #pragma unroll
              for (int e = 0; e < 4; ++e)
                if (!key_ok || c0 + cc + e < qlo || (kWin && c0 + cc + e >= qhe)) p[e] = 0.f;
            }
            const uint32_t w0 = Cvt<T>::pack(p[0], p[1]), w1 = Cvt<T>::pack(p[2], p[3]);
            pp[cc / 2] = w0;
            pp[cc / 2 + 1] = w1;
            if constexpr (kDrop) {
              const uint32_t kb = keep >> cc;
              const float rp = a.drop.rp;
              pt[cc / 2] = Cvt<T>::pack((kb & 1u) ? p[0] * rp : 0.f, (kb & 2u) ? p[1] * rp : 0.f);
              pt[cc / 2 + 1] = Cvt<T>::pack((kb & 4u) ? p[2] * rp : 0.f, (kb & 8u) ? p[3] * rp : 0.f);
            } else {
              pt[cc / 2] = w0;
              pt[cc / 2 + 1] = w1;
            }
          }
        }
        // dV of the previous step must have read P~^T
        if (t > 0 && !(ok = warp_wait(&bars->pt_free, (uint32_t)(t - 1) & 1u, ctl))) break;
        tmem_st16(tl + kColPT + wg * 16, pt);
        // dP^T(t) is usually complete by now: start its first load before the store is waited on
        if (!(ok = warp_wait(&bars->dp_full, (uint32_t)t & 1u, ctl))) break;
        tc_fence_after();
        uint32_t dv[2][16];
        tmem_ld16(tl + kColDP + c0, dv[0]);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full);

        // ---- part 2: dS from dP^T, in the same two halves
        // dS^T also goes to the shared tile, once dQ of the previous step has read it
        if (t >= 1 && !(ok = warp_wait(&bars->dsm_free, (uint32_t)(t - 1) & 1u, ctl))) break;
        uint8_t* dsb = smem + L::kDS + (wg >> 1) * 16384 + r * 128;
  #pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          tmem_wait_ld();
          reg_fence16(dv[hf]);
          if (hf == 0) tmem_ld16(tl + kColDP + c0 + 16, dv[1]);
          uint32_t dsw[8];
  #pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int cc = hf * 16 + q4 * 4;
            const float4 d4 = lds128(s_d + cc * 4);
            float g[4] = {__uint_as_float(dv[hf][q4 * 4]), __uint_as_float(dv[hf][q4 * 4 + 1]),
                          __uint_as_float(dv[hf][q4 * 4 + 2]), __uint_as_float(dv[hf][q4 * 4 + 3])};
            if constexpr (kDrop) {
              const uint32_t kb = keep >> cc;
              const float rp = a.drop.rp;
  #pragma unroll
              for (int e = 0; e < 4; ++e) g[e] = ((kb >> e) & 1u) ? g[e] * rp : 0.f;
            }
            const uint32_t w0 = pp[cc / 2], w1 = pp[cc / 2 + 1];
            float y[4];
            if constexpr (kFold) {      // d4 holds -tau * D
              fma2(y[0], y[1], g[0], g[1], a.scale, a.scale, d4.x, d4.y);
              fma2(y[2], y[3], g[2], g[3], a.scale, a.scale, d4.z, d4.w);
            } else {
              sub2(y[0], y[1], g[0], g[1], d4.x, d4.y);
              sub2(y[2], y[3], g[2], g[3], d4.z, d4.w);
            }
            mul2(y[0], y[1], y[0], y[1], Cvt<T>::lo(w0), Cvt<T>::hi(w0));
            mul2(y[2], y[3], y[2], y[3], Cvt<T>::lo(w1), Cvt<T>::hi(w1));
            dsw[q4 * 2] = Cvt<T>::pack(y[0], y[1]);
            dsw[q4 * 2 + 1] = Cvt<T>::pack(y[2], y[3]);
          }
  #pragma unroll
          for (int pc2 = 0; pc2 < 2; ++pc2) {
            const uint32_t off = ((((pc_base + hf * 2 + pc2) ^ r) & 7) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         :: "r"(smem_u32(dsb + off)), "r"(dsw[pc2 * 4]), "r"(dsw[pc2 * 4 + 1]), "r"(dsw[pc2 * 4 + 2]),
                            "r"(dsw[pc2 * 4 + 3]) : "memory");
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->ds_full);

        // ---- drain dQ of the previous step
        if (t > 0 && !(ok = drain_dq(t - 1))) break;
      }
      if (!ok) break;
      // ---- item end: dK, dV out of tensor memory.  The next item's first
      //      dV / dK (which restart the accumulators) follow this thread's
      //      next p_full / ds_full arrivals, hence these loads.
      if (!(ok = warp_wait(&bars->dkv_full, (uint32_t)nit & 1u, ctl))) break;
      ++nit;
      tc_fence_after();
      if constexpr (kDrop) {
        uint32_t raw[32];
        tmem_ld16x256b_x8(kv_taddr, raw);
        tmem_wait_ld();
        reg_fence32(raw);
        tc_fence_before();
        store_dkv_rows(it, raw, true);
      } else {
        uint32_t kraw[16], vraw[16];
        tmem_ld16(tl + kColDK + wg * 16, kraw);
        tmem_ld16(tl + kColDV + wg * 16, vraw);
        tmem_wait_ld();
        reg_fence16(kraw);
        reg_fence16(vraw);
        tc_fence_before();
        store_dkv(it, kraw, vraw, true);
      }
    }
    if (ok && t > 0) ok = drain_dq(t - 1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 17) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <typename T, bool kDrop, bool kWin>
cudaError_t launch_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                     const CUtensorMap& dqacc, const BwdArgs& a, cudaStream_t s) {
  auto kern = bwd_tc_kernel<T, kDrop, kWin>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdSmem::kDyn);
  if (e != cudaSuccess) return e;
  const long long total = (long long)a.nq * a.B * a.H_kv;
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const unsigned grid = (unsigned)std::min<long long>(total, (long long)std::max(sms, 1));
  kern<<<grid, kThreads, BwdSmem::kDyn, s>>>(q, k, v, dout, dqacc, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc(int dtype, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& dout, const CUtensorMap& dqacc, const BwdArgs& a, cudaStream_t s) {
  const int sel = (a.drop.enabled ? 1 : 0) | (a.mask.window > 0 ? 2 : 0);
  if (dtype == FA_DT_BF16) {
    using B = __nv_bfloat16;
    switch (sel) {
      case 0: return launch_t<B, false, false>(q, k, v, dout, dqacc, a, s);
      case 1: return launch_t<B, true, false>(q, k, v, dout, dqacc, a, s);
      case 2: return launch_t<B, false, true>(q, k, v, dout, dqacc, a, s);
      default: return launch_t<B, true, true>(q, k, v, dout, dqacc, a, s);
    }
  }
  switch (sel) {
    case 0: return launch_t<__half, false, false>(q, k, v, dout, dqacc, a, s);
    case 1: return launch_t<__half, true, false>(q, k, v, dout, dqacc, a, s);
    case 2: return launch_t<__half, false, true>(q, k, v, dout, dqacc, a, s);
    default: return launch_t<__half, true, true>(q, k, v, dout, dqacc, a, s);
  }
}

}  // namespace fa
