// bwd_tc128.cu -- backward attention kernel for head dimension 128, 16-bit
// inputs, on sm_103a.
//
// Method: as in bwd_tc.cu (the pages: the backward pass rebuilds the score
// and probability tiles on chip from Q, K and the saved softmax statistics,
// replays the dropout mask and uses D_i = dO_i . O_i -- tonho.wtf, "como
// funciona"; agihunt.info, backward paragraph; marketmaker.cc, "Passo para
// tras").  The pages single out d = 128 as the case where the on-chip tile
// budget gets tight and the tiles must shrink (marketmaker.cc, "O que isso
// custou"; lynx-cortex, "Lo que Flash forward no hace").  Here the key tile
// stays at 128 rows and a step covers 64 query rows instead of 128, which is
// what lets the products fit the 512 tensor-memory columns:
//
//   S^T 0-63 | dP^T 64-127 | dK 128-255 | dV 256-383 | dQ^T 384-447 |
//   P~^T (16 bit, queries 16w..16w+15 packed at 448+8w .. +8) 448-479.
//
// Per (128-key tile, 64-query step) it forms
//     S^T  = K Q^T          M=128 keys, N=64 queries, K=128   (both K-major)
//     dP^T = V dO^T         same shape
//     dV  += P~^T dO        M=128, N=128 (d), K=64 queries  (A in tensor memory)
//     dK  += dS^T Q         M=128, N=128, K=64              (A = shared dS^T tile)
//     dQ^T = K^T dS^T       M=128 (d), N=64 queries, K=128 keys (A, B MN-major)
// dQ is produced transposed (head dims on the tensor-memory lanes) so that
// its M is 128 too; the drain writes it back row-major into the float32
// staging tile that the TMA reduce-adds into the accumulator.
//
// Work distribution, roles and barriers are those of bwd_tc.cu: a
// persistent kernel, one CTA per SM, dynamic (b, K/V head, key tile) items
// taken from a global counter and handed through a two-slot mailbox; the
// steps of an item are the 64-row halves of every 128-row query tile that
// sees the key tile, for each query head of the group.  K and V (32 KB each
// here) have one buffer each; Q, dO and their LSE / D rows a three-stage
// ring.  Warps 0-15 are four warpgroups of 16 query columns each.
#include <algorithm>
#include <type_traits>

#include "bwd_items.cuh"

namespace fa {
namespace {

constexpr int kThreads = 640;
constexpr int kCompute = 512;   // threads of warps 0-15
constexpr int kQS = 64;         // query rows per step
constexpr int NQ = 3;           // Q / dO stages
constexpr int kLag = 3;         // dQ reduce-adds trail the loads by this many steps

struct Smem128 {
  static constexpr int kK = 0;                      // 32 KB: K [2 boxes][128 keys][64 d]
  static constexpr int kV = 32768;                  // 32 KB
  static constexpr int kQ = 65536;                  // NQ x 16 KB: Q [2 boxes][64 q][64 d]
  static constexpr int kDO = kQ + NQ * 16384;       // NQ x 16 KB
  static constexpr int kDS = kDO + NQ * 16384;      // 16 KB: dS^T [128 keys][64 q]
  static constexpr int kDQ = kDS + 16384;           // 32 KB: float32 dQ staging [4 boxes][64 q][32 d]
  static constexpr int kLD = kDQ + 32768;           // NQ x (LSE2[64] + D[64]) floats
  static constexpr int kInfo = kLD + NQ * 512;      // (first query row, query head, batch) of the last kLag+1 steps
  static constexpr int kItem = kInfo + 64;          // the two published work items
  static constexpr int kBar = kItem + 64;
  static constexpr int kBytes = kBar + 320;
  static constexpr int kDyn = kBytes + 1024;
};

struct Bars128 {
  uint64_t item_full[2], item_empty[2];
  uint64_t kv_full, kv_empty;
  uint64_t q_full[NQ], q_empty[NQ];
  uint64_t s_full, p_full, dp_full, ds_full, dq_full, dq_free, dkv_full, pt_free;
  uint64_t dsm_free;
  uint64_t done[3];
  uint64_t stg_full, stg_free;
  uint32_t tmem_base;
  int abort;
};

static_assert(sizeof(Bars128) <= 320, "barrier block overflows its shared-memory slot");
static_assert(Smem128::kDyn <= 232448, "shared memory over the per-block limit");

constexpr uint32_t kColST = 0, kColDP = 64, kColDK = 128, kColDV = 256, kColDQ = 384, kColPT = 448;

// Step decode shared by every role: the item's steps are (query head, 128-row
// tile, 64-row half) in that order.
struct StepPos {
  int qu = 0, hq = 0, hf = 0;
  __device__ __forceinline__ void next(const Item& it) {
    if (++hf == 2) {
      hf = 0;
      if (++qu == it.n) { qu = 0; ++hq; }
    }
  }
};

template <typename T, bool kDrop, bool kWin>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                 const __grid_constant__ CUtensorMap tmDQ, const BwdArgs a) {
  using L = Smem128;
  // bf16: tau is folded into dS (the D rows hold -tau * D, and part 2 forms
  // (tau dP - tau D) o P with one packed FMA), so dQ and dK leave the tensor
  // core already scaled.  Not for fp16, whose smaller range would push small
  // dS values into subnormals.
  constexpr bool kFold = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars128* bars = reinterpret_cast<Bars128*>(smem + L::kBar);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total = a.nq * a.B * a.H_kv;
  WaitCtl ctl{a.status, &bars->abort};

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->item_full[s], 1);
      mbar_init(&bars->item_empty[s], 3 + kCompute);   // warps 17-19 and the compute threads
    }
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 2);      // S^T / dP^T warp and dQ warp read K, V
    for (int s = 0; s < NQ; ++s) {
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
    mbar_init(&bars->pt_free, 1);
    mbar_init(&bars->dsm_free, 2);     // dK and dQ^T both read the shared dS^T tile
    for (int i = 0; i < 3; ++i) mbar_init(&bars->done[i], 1);
    mbar_init(&bars->stg_full, kCompute);
    mbar_init(&bars->stg_free, 1);
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
    constexpr uint32_t idST = idesc_f16(128, 64, ab, 0, 0);    // S^T, dP^T (both operands K-major)
    constexpr uint32_t idKV = idesc_f16(128, 128, ab, 0, 1);   // dV, dK (A K-major or in tensor memory, B MN-major)
    constexpr uint32_t idQ = idesc_f16(128, 64, ab, 1, 1);     // dQ^T (A = K^T MN-major, B = dS^T MN-major)
    const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
    const uint32_t sQ = smem_u32(smem + L::kQ), sDO = smem_u32(smem + L::kDO);
    const uint32_t sDS = smem_u32(smem + L::kDS);
    volatile int* item_u = reinterpret_cast<volatile int*>(smem + L::kItem);
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
      if (lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmDO);
        prefetch_tmap(&tmDQ);
        int4* info = reinterpret_cast<int4*>(smem + L::kInfo);
        int g = 0, nkv = 0;
        bool ok = true;
        // the staged dQ of step r: four 32-column boxes; a half tile that
        // starts at or past N (the second half of a ragged last tile) has
        // nothing to add
        auto reduce = [&](int r) -> bool {
          if (!mbar_wait(&bars->stg_full, (uint32_t)r & 1u, ctl)) return false;
          const uint8_t* sb = smem + L::kDQ;
          const int4 inf = info[r & 3];
          if (inf.x < a.N) {
#pragma unroll
            for (int c = 0; c < 4; ++c) tma_reduce_add_4d(&tmDQ, sb + c * 8192, c * 32, inf.x, inf.y, inf.z);
            bulk_commit();
            bulk_wait_read0();
          }
          mbar_arrive(&bars->stg_free);
          return true;
        };
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
          // third-last step (measured faster at head dimension 64).
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
            // no load follows, so do the reduces the compute threads need to
            // finish their current item (a run of empty items would
            // otherwise fill the mailbox while they wait for one)
            ok = reduce_to(g - 3);
            continue;
          }
          // K, V: one buffer each, free once the previous item's S^T, dP^T
          // and dQ^T MMAs are done
          if (!(ok = mbar_wait(&bars->kv_empty, ((uint32_t)nkv & 1u) ^ 1u, ctl))) break;
          mbar_expect_tx(&bars->kv_full, 65536);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            tma_load_4d(smem + L::kK + c * 16384, &tmK, &bars->kv_full, c * 64, it.jt * kTile, it.hk, it.b);
            tma_load_4d(smem + L::kV + c * 16384, &tmV, &bars->kv_full, c * 64, it.jt * kTile, it.hk, it.b);
          }
          ++nkv;
          StepPos sp;
          sp.hq = it.h0;
          const int nsteps = 2 * it.steps;
          for (int t = 0; t < nsteps && ok; ++t, ++g, sp.next(it)) {
            const int st = g % NQ;
            if (!(ok = mbar_wait(&bars->q_empty[st], ((uint32_t)(g / NQ) & 1u) ^ 1u, ctl))) break;
            const int q0 = it.qt(sp.qu) * kTile + sp.hf * kQS;
            const size_t ld_row = ((size_t)it.b * a.H + sp.hq) * a.npad + (size_t)q0;
            mbar_expect_tx(&bars->q_full[st], 32768 + 512);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              tma_load_4d(smem + L::kQ + st * 16384 + c * 8192, &tmQ, &bars->q_full[st], c * 64, q0, sp.hq, it.b);
              tma_load_4d(smem + L::kDO + st * 16384 + c * 8192, &tmDO, &bars->q_full[st], c * 64, q0, sp.hq, it.b);
            }
            bulk_load(smem + L::kLD + st * 512, a.lse2 + ld_row, 256, &bars->q_full[st]);
            bulk_load(smem + L::kLD + st * 512 + 256, a.dvec + ld_row, 256, &bars->q_full[st]);
            info[g & 3] = make_int4(q0, sp.hq, it.b, 0);
            if (!(ok = reduce_to(g - kLag))) break;
          }
        }
        if (ok) ok = reduce_to(g - 1);
        for (int t = max(0, g - NQ); t < g; ++t) mbar_wait(&bars->q_full[t % NQ], (uint32_t)(t / NQ) & 1u, ctl);
        if (nkv > 0) mbar_wait(&bars->kv_full, (uint32_t)(nkv - 1) & 1u, ctl);
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
          if (!(ok = mbar_wait(&bars->kv_full, (uint32_t)nkv & 1u, ctl))) break;
          ++nkv;
          const int nsteps = 2 * it.steps;
          for (int t = 0; t < nsteps && ok; ++t, ++g) {
            const int st = g % NQ;
            // S^T(g) = K Q_g^T once part 1 of step g-1 has read S^T(g-1)
            if (g > 0 && !(ok = mbar_wait(&bars->p_full, (uint32_t)(g - 1) & 1u, ctl))) break;
            if (!(ok = mbar_wait(&bars->q_full[st], (uint32_t)(g / NQ) & 1u, ctl))) break;
            tc_fence_after();
            // K-dim = 128 head dims in steps of 16: box k / 4, 32 bytes per step within it
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ss(tmem + kColST, sdesc_sw128(sK + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                     sdesc_sw128(sQ + st * 16384 + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024), idST, k > 0 ? 1u : 0u);
            mma_commit(&bars->s_full);
            // dP^T(g) = V dO_g^T once part 2 of step g-1 has read dP^T(g-1)
            if (g > 0 && !(ok = mbar_wait(&bars->ds_full, (uint32_t)(g - 1) & 1u, ctl))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ss(tmem + kColDP, sdesc_sw128(sV + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                     sdesc_sw128(sDO + st * 16384 + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024), idST, k > 0 ? 1u : 0u);
            mma_commit(&bars->dp_full);
          }
          mma_commit(&bars->kv_empty);    // this item's S^T and dP^T are done with K, V
        }
        mma_commit(&bars->done[0]);
        mbar_wait(&bars->done[0], 0, ctl);
      }
    } else if (warp == 18) {
      // ===================== dV / dK issuer =====================
      if (lane == 0) {
        int g = 0;
        bool ok = true;
        int u;
        while (ok && (u = fetch()) >= 0) {
          const Item it = make_item(a, u);
          if (it.steps == 0) continue;
          const int nsteps = 2 * it.steps;
          for (int t = 0; t < nsteps && ok; ++t, ++g) {
            const int st = g % NQ;
            const uint32_t qb = sQ + st * 16384, db = sDO + st * 16384;
            // dV += P~^T dO_g: A = P~^T in tensor memory, B = dO MN-major
            // (two 64-column boxes 8 KB apart); K-dim = 64 queries, 4 steps of 16
            if (!(ok = mbar_wait(&bars->p_full, (uint32_t)g & 1u, ctl) &&
                       mbar_wait(&bars->q_full[st], (uint32_t)(g / NQ) & 1u, ctl))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ts(tmem + kColDV, tmem + kColPT + k * 8, sdesc_sw128(db + k * 2048, 8192, 1024), idKV,
                     (t > 0 || k > 0) ? 1u : 0u);
            mma_commit(&bars->pt_free);
            // dK += dS^T Q_g: A = dS^T K-major (32 bytes per 16 queries), B = Q MN-major
            if (!(ok = mbar_wait(&bars->ds_full, (uint32_t)g & 1u, ctl))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(tmem + kColDK, sdesc_sw128(sDS + k * 32, 16, 1024), sdesc_sw128(qb + k * 2048, 8192, 1024), idKV,
                     (t > 0 || k > 0) ? 1u : 0u);
            mma_commit(&bars->dsm_free);
            mma_commit(&bars->q_empty[st]);
          }
          mma_commit(&bars->dkv_full);
        }
        mma_commit(&bars->done[1]);
        mbar_wait(&bars->done[1], 0, ctl);
      }
    } else {
      // ===================== dQ^T issuer (warp 19) =====================
      if (lane == 0) {
        int g = 0;
        bool ok = true;
        int u;
        while (ok && (u = fetch()) >= 0) {
          const Item it = make_item(a, u);
          if (it.steps == 0) continue;
          const int nsteps = 2 * it.steps;
          for (int t = 0; t < nsteps && ok; ++t, ++g) {
            // dQ^T_g = K^T dS^T: A = K read MN-major (M = 128 head dims in two
            // 64-wide boxes 16 KB apart), B = dS^T MN-major (N = 64 queries);
            // K-dim = 128 keys, 8 steps of 16 rows (2 KB)
            if (!(ok = mbar_wait(&bars->ds_full, (uint32_t)g & 1u, ctl))) break;
            if (g > 0 && !(ok = mbar_wait(&bars->dq_free, (uint32_t)(g - 1) & 1u, ctl))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ss(tmem + kColDQ, sdesc_sw128(sK + k * 2048, 16384, 1024), sdesc_sw128(sDS + k * 2048, 8192, 1024),
                     idQ, k > 0 ? 1u : 0u);
            mma_commit(&bars->dq_full);
            mma_commit(&bars->dsm_free);
          }
          mma_commit(&bars->kv_empty);    // this item's dQ^T MMAs are done with K
        }
        mma_commit(&bars->done[2]);
        mbar_wait(&bars->done[2], 0, ctl);
      }
    }
  } else {
    // ===================== softmax-gradient warpgroups =====================
    const int wg = warp >> 2;                 // query columns 16 wg .. 16 wg + 15 of the step
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;        // key row (S^T, dP^T, dK, dV) or head dim (dQ^T) = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tl = tmem + lane_off;
    const float sl2 = a.scale_log2;
    const int c0 = wg * 16;                   // first query column of this warpgroup
    bool ok = true;

    // dQ_t: head dim r of this warpgroup's 16 queries, tensor memory -> x tau (fp16; bf16 is already scaled)
    // -> float32 staging box r / 32 (rows = queries, 32 floats = 128 bytes
    // with the 128-byte swizzle); warp 16 reduces it
    auto drain_dq = [&](int t) -> bool {
      if (!warp_wait(&bars->dq_full, (uint32_t)t & 1u, ctl)) return false;
      tc_fence_after();
      uint32_t g[16];
      tmem_ld16(tl + kColDQ + c0, g);
      tmem_wait_ld();
      reg_fence16(g);
      tc_fence_before();
      mbar_arrive(&bars->dq_free);
      if (t >= 1 && !warp_wait(&bars->stg_free, (uint32_t)(t - 1) & 1u, ctl)) return false;
      uint8_t* sb = smem + L::kDQ + quarter * 8192;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int q = c0 + c;
        const uint32_t off = q * 128 + ((((lane >> 2) ^ q) & 7) << 4) + (lane & 3) * 4;
        const float v = kFold ? __uint_as_float(g[c]) : __uint_as_float(g[c]) * a.scale;
        asm volatile("st.shared.f32 [%0], %1;" :: "r"(smem_u32(sb + off)), "f"(v) : "memory");
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->stg_full);
      return true;
    };

    // dK (x tau for fp16) and dV of an item: columns 32 wg .. 32 wg + 31 of this
    // thread's key row, in two halves of 16, straight to global memory
    auto store_dkv = [&](const Item& it, int half, const uint32_t (&kraw)[16], const uint32_t (&vraw)[16],
                         bool have) {
      const int j = it.jt * kTile + r;
      if (j >= a.N) return;
      const size_t off =
          (size_t)it.b * a.kst.b + (size_t)it.hk * a.kst.h + (size_t)j * a.kst.n + wg * 32 + half * 16;
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
        const uint32_t zero[16] = {};
        store_dkv(it, 0, zero, zero, false);
        store_dkv(it, 1, zero, zero, false);
        continue;
      }
      const int j = it.jt * kTile + r;          // global key
      const bool key_ok = j < it.Lk;
      StepPos sp;
      sp.hq = it.h0;
      const int nsteps = 2 * it.steps;
      for (int tt = 0; tt < nsteps && ok; ++tt, ++t, sp.next(it)) {
        const int st = t % NQ;
        const int q0 = it.qt(sp.qu) * kTile + sp.hf * kQS;   // first query row of the step
        const uint32_t bh_rows = ((uint32_t)it.b * (uint32_t)a.H + (uint32_t)sp.hq) * (uint32_t)a.N;
        const uint32_t s_lse = smem_u32(smem + L::kLD + st * 512) + c0 * 4;
        const uint32_t s_d = s_lse + 256;
        // query column c of the step is hidden from this key under causal iff
        // c < qlo, and outside its sliding window iff c >= qhe
        const int qlo = a.mask.causal ? (j - q0) : -1;
        const int qhe = kWin ? (j + a.mask.window - q0) : kQS;
        const bool any_mask = !key_ok || qlo > c0 || (kWin && qhe < c0 + 16);

        // ---- part 1: P from S^T (16 query columns)
        if (!(ok = warp_wait(&bars->s_full, (uint32_t)t & 1u, ctl) &&
                   warp_wait(&bars->q_full[st], (uint32_t)(t / NQ) & 1u, ctl))) break;
        tc_fence_after();
        uint32_t sv[16];
        tmem_ld16(tl + kColST + c0, sv);
        uint32_t keep = ~0u;
        if constexpr (kDrop) {
          // One Philox call covers 8 consecutive keys of one query row; the 8
          // lanes 8m..8m+7 hold 8 consecutive keys (j & 7 == lane & 7), so
          // lane t of each group evaluates queries t and t+8 and the group
          // exchanges the 8-key keep bytes.
          const int t8 = lane & 7;
          uint32_t mine = 0;
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const uint32_t q = (uint32_t)(q0 + c0 + t8 + 8 * m);
            mine |= dropout_keep8((uint32_t)j >> 3, bh_rows + q, a.drop) << (8 * m);
          }
          uint32_t kb = 0;
#pragma unroll
          for (int src = 0; src < 8; ++src) {
            const uint32_t w = __shfl_sync(0xffffffffu, mine, (lane & ~7) | src);
#pragma unroll
            for (int m = 0; m < 2; ++m) kb |= ((w >> (8 * m + t8)) & 1u) << (src + 8 * m);
          }
          keep = kb;
        }
        tmem_wait_ld();
        reg_fence16(sv);
        uint32_t pp[8];       // undropped P, 16 bit, kept for part 2
        uint32_t pt[8];       // P~ = Z o P / (1 - p), 16 bit, operand of dV
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int cc = q4 * 4;
          const float4 l4 = lds128(s_lse + cc * 4);
          float x[4];
          fma2(x[0], x[1], __uint_as_float(sv[cc]), __uint_as_float(sv[cc + 1]), sl2, sl2, -l4.x, -l4.y);
          fma2(x[2], x[3], __uint_as_float(sv[cc + 2]), __uint_as_float(sv[cc + 3]), sl2, sl2, -l4.z, -l4.w);
          float p[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) p[e] = ex2(x[e]);
          if (any_mask) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (!key_ok || c0 + cc + e < qlo || (kWin && c0 + cc + e >= qhe)) p[e] = 0.f;
          }
          const uint32_t w0 = Cvt<T>::pack(p[0], p[1]), w1 = Cvt<T>::pack(p[2], p[3]);
          pp[q4 * 2] = w0;
          pp[q4 * 2 + 1] = w1;
          if constexpr (kDrop) {
            const uint32_t kb = keep >> cc;
            const float rp = a.drop.rp;
            pt[q4 * 2] = Cvt<T>::pack((kb & 1u) ? p[0] * rp : 0.f, (kb & 2u) ? p[1] * rp : 0.f);
            pt[q4 * 2 + 1] = Cvt<T>::pack((kb & 4u) ? p[2] * rp : 0.f, (kb & 8u) ? p[3] * rp : 0.f);
          } else {
            pt[q4 * 2] = w0;
            pt[q4 * 2 + 1] = w1;
          }
        }
        // dV of the previous step must have read P~^T
        if (t > 0 && !(ok = warp_wait(&bars->pt_free, (uint32_t)(t - 1) & 1u, ctl))) break;
        tmem_st8(tl + kColPT + wg * 8, pt);
        if (!(ok = warp_wait(&bars->dp_full, (uint32_t)t & 1u, ctl))) break;
        tc_fence_after();
        uint32_t dv[16];
        tmem_ld16(tl + kColDP + c0, dv);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full);

        // ---- part 2: dS from dP^T; dS^T (16 bit) into the shared tile once
        //      dK and dQ^T of the previous step have read it
        if (t >= 1 && !(ok = warp_wait(&bars->dsm_free, (uint32_t)(t - 1) & 1u, ctl))) break;
        tmem_wait_ld();
        reg_fence16(dv);
        uint32_t dsw[8];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int cc = q4 * 4;
          const float4 d4 = lds128(s_d + cc * 4);
          float g[4] = {__uint_as_float(dv[cc]), __uint_as_float(dv[cc + 1]), __uint_as_float(dv[cc + 2]),
                        __uint_as_float(dv[cc + 3])};
          if constexpr (kDrop) {
            const uint32_t kb = keep >> cc;
            const float rp = a.drop.rp;
#pragma unroll
            for (int e = 0; e < 4; ++e) g[e] = ((kb >> e) & 1u) ? g[e] * rp : 0.f;
          }
          const uint32_t w0 = pp[q4 * 2], w1 = pp[q4 * 2 + 1];
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
        // this warpgroup's 16 queries are the 16-byte pieces 2 wg, 2 wg + 1 of the key's 128-byte row
        uint8_t* dsb = smem + L::kDS + r * 128;
#pragma unroll
        for (int pc2 = 0; pc2 < 2; ++pc2) {
          const uint32_t off = ((((2 * wg + pc2) ^ r) & 7) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                       :: "r"(smem_u32(dsb + off)), "r"(dsw[pc2 * 4]), "r"(dsw[pc2 * 4 + 1]), "r"(dsw[pc2 * 4 + 2]),
                          "r"(dsw[pc2 * 4 + 3]) : "memory");
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->ds_full);

        // ---- drain dQ of the previous step
        if (t > 0 && !(ok = drain_dq(t - 1))) break;
      }
      if (!ok) break;
      // ---- item end: dK, dV out of tensor memory (the next item's first dV /
      //      dK follow this thread's next p_full / ds_full arrivals)
      if (!(ok = warp_wait(&bars->dkv_full, (uint32_t)nit & 1u, ctl))) break;
      ++nit;
      tc_fence_after();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t kraw[16], vraw[16];
        tmem_ld16(tl + kColDK + wg * 32 + half * 16, kraw);
        tmem_ld16(tl + kColDV + wg * 32 + half * 16, vraw);
        tmem_wait_ld();
        reg_fence16(kraw);
        reg_fence16(vraw);
        store_dkv(it, half, kraw, vraw, true);
      }
      tc_fence_before();
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
  auto kern = bwd_tc128_kernel<T, kDrop, kWin>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem128::kDyn);
  if (e != cudaSuccess) return e;
  const long long total = (long long)a.nq * a.B * a.H_kv;
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const unsigned grid = (unsigned)std::min<long long>(total, (long long)std::max(sms, 1));
  kern<<<grid, kThreads, Smem128::kDyn, s>>>(q, k, v, dout, dqacc, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc128(int dtype, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
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
