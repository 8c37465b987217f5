// fwd_plan.cuh -- the forward kernels' tile schedule (shared by the 16-bit
// and FP8 forward kernels).
//
// A CTA holds two 128-row query tiles ("slots") of one head.  Each slot
// visits the K/V tiles its rows can see (marketmaker.cc, "O mascaramento
// causal": future tiles are skipped; agihunt.info, block-sparse paragraph:
// only kept blocks are visited; lynx-cortex, "Problemas de practica": a
// sliding window starts at the first tile its rows reach), in ascending
// order.  The TMA producer, the MMA issuers and the softmax warps all walk
// the same step plan, so they agree on ring stages and barrier phases.
#pragma once
#include "common.cuh"

namespace fa {
namespace {

struct Slot {
  int qt;                 // query tile index
  int n;                  // kv steps
  int lo;                 // first kv tile (dense)
  const int16_t* list;    // sparse kv list or nullptr
  // kv tile of step s (lo is nonzero only under a sliding window)
  template <bool kWin>
  __device__ __forceinline__ int kv(int s) const { return list ? (int)list[s] : (kWin ? lo + s : s); }
};

__device__ __forceinline__ Slot make_slot(const FwdArgs& a, int qt, int Lk) {
  Slot sl;
  sl.qt = qt;
  sl.list = nullptr;
  sl.n = 0;
  sl.lo = 0;
  if (qt >= a.nq) return sl;
  int lim = (Lk + kTile - 1) / kTile;
  if (a.mask.causal) lim = min(lim, qt + 1);
  // sliding window: the tile's first query sees keys from qt*128 - w + 1 on
  if (a.mask.window > 0) sl.lo = max(0, qt * kTile - a.mask.window + 1) / kTile;
  if (a.mask.row_list != nullptr) {
    const int16_t* list = a.mask.row_list + (size_t)qt * a.mask.nb;
    const int cnt = a.mask.row_cnt[qt];
    int s0 = 0;
    while (s0 < cnt && list[s0] < sl.lo) ++s0;
    int n = s0;
    while (n < cnt && list[n] < lim) ++n;
    sl.list = list + s0;
    sl.n = n - s0;
  } else {
    sl.n = max(0, lim - sl.lo);
  }
  return sl;
}

// The K/V tiles loaded at one step: one stage when both slots need the same
// tile (or only one slot has a step), two otherwise.  Every role walks the
// same sequence, so all agree on stage indices and phases.
struct StepPlan {
  int nl;                 // loads at this step (0..2)
  int st[2];              // stage of each load
  uint32_t ph[2];         // phase parity of each load
  int kv[2];              // kv tile of each load
  int use[2];             // load index used by slot x, or -1
  // Accessors by select rather than by indexing with a run-time value, so
  // the plan stays in registers (an indexed array would live in local memory
  // and cost the single-thread issuers a memory round trip per access).
  __device__ __forceinline__ int stage(int l) const { return l ? st[1] : st[0]; }
  __device__ __forceinline__ uint32_t parity(int l) const { return l ? ph[1] : ph[0]; }
  __device__ __forceinline__ int load_of(int x) const { return x ? use[1] : use[0]; }
};

template <int NS, bool kWin>
__device__ __forceinline__ StepPlan plan_step(const Slot (&sl)[2], int s, int& ld) {
  StepPlan p;
  p.nl = 0;
  p.use[0] = p.use[1] = -1;
  const int kvA = s < sl[0].n ? sl[0].kv<kWin>(s) : -1;
  const int kvB = s < sl[1].n ? sl[1].kv<kWin>(s) : -1;
  if (kvA >= 0) {
    p.st[0] = ld % NS; p.ph[0] = (uint32_t)(ld / NS) & 1u; p.kv[0] = kvA; ++ld;
    p.use[0] = 0; p.nl = 1;
  }
  if (kvB >= 0) {
    if (kvB == kvA) {
      p.use[1] = 0;
    } else {
      p.st[p.nl] = ld % NS; p.ph[p.nl] = (uint32_t)(ld / NS) & 1u; p.kv[p.nl] = kvB; ++ld;
      p.use[1] = p.nl; ++p.nl;
    }
  }
  return p;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

}  // namespace
}  // namespace fa
