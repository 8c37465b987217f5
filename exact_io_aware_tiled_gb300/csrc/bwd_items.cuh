// bwd_items.cuh -- the work items of the backward kernels (head dims 64 and
// 128): which query tiles see a 128-key tile of one K/V head, under the
// causal, padding, block-sparse and sliding-window masks.
#pragma once
#include "common.cuh"

namespace fa {
namespace {

// One work item: key tile jt of K/V head hk of batch b, and its steps:
// every query tile that sees the key tile, for each of the g query heads
// that share the K/V head (head-major: step t is tile t % n of query head
// h0 + t / n; the loops track both with counters).
struct Item {
  int b, hk, jt, Lk;
  int n;                  // query tiles per query head
  int i0;                 // first query tile (dense)
  int h0;                 // first query head of the group
  const int16_t* list;    // sparse list or nullptr
  int steps;              // n * g
  __device__ __forceinline__ int qt(int u) const { return list ? (int)list[u] : i0 + u; }
};

__device__ __forceinline__ Item make_item(const BwdArgs& a, int u) {
  Item it;
  const int bk = u / a.nq;
  it.jt = u - bk * a.nq;
  it.b = bk / a.H_kv;
  it.hk = bk - it.b * a.H_kv;
  it.Lk = a.N;
  if (a.mask.seqlens_k != nullptr) it.Lk = max(0, min(a.N, a.mask.seqlens_k[it.b]));
  it.list = nullptr;
  it.i0 = a.mask.causal ? it.jt : 0;
  it.h0 = it.hk * a.group;
  it.n = 0;
  // last query tile that sees this key tile: under a sliding window of w keys,
  // key j is seen by queries j .. j + w - 1
  int qlast = a.nq - 1;
  if (a.mask.window > 0) qlast = min(qlast, (it.jt * kTile + kTile - 1 + a.mask.window - 1) / kTile);
  if (it.jt * kTile < it.Lk) {
    if (a.mask.col_list != nullptr) {
      const int16_t* list = a.mask.col_list + (size_t)it.jt * a.mask.nb;
      const int cnt = a.mask.col_cnt[it.jt];
      int s0 = 0;
      if (a.mask.causal) while (s0 < cnt && list[s0] < it.jt) ++s0;
      int e = s0;
      while (e < cnt && list[e] <= qlast) ++e;
      it.list = list + s0;
      it.n = e - s0;
    } else {
      it.n = max(0, qlast - it.i0 + 1);
    }
  }
  it.steps = it.n * a.group;
  return it;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

}  // namespace
}  // namespace fa
