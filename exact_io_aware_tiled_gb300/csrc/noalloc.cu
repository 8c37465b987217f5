// noalloc.cu -- fa_bwd_noalloc: the backward pass without a caller workspace.
//
// Why it exists: fa_bwd needs device scratch memory (a float32 dQ
// accumulator, the padded LSE / D rows and a status word) that the caller
// passes in as `ws`.  Some callers cannot allocate device memory at the point
// where they run the backward pass -- for example code that runs inside a
// memory pool it does not own, a framework hook that forbids allocation, or a
// plain C program that links this library without any allocator of its own.
// For them this entry point takes its scratch from a fixed array that lives
// in the library's own device image, so it allocates nothing itself.
//
// How: the array below is a file-scope static __device__ object of
// kNoAllocScratchBytes bytes.  The CUDA runtime reserves it on every device
// that loads this library's device code and keeps it there until the process
// exits.  Host code only knows a host-side stand-in for its name, so before
// the first use on a device we ask the runtime for its device address
// (cudaGetSymbolAddress, with that device current) and cache the address per
// device.  The cached address is then handed to the unchanged fa_bwd path as
// its workspace.
//
// Contract (stated in include/fa.h as well):
//   * problems whose workspace would exceed kNoAllocScratchBytes are refused
//     with FA_ERR_WORKSPACE and nothing is enqueued;
//   * the first call on a device does the address look-up; make that first
//     call before capturing a stream into a CUDA graph;
//   * every call on a device shares the one array and leaves its contents
//     behind: fa_bwd clears what must start at zero (status word, dQ
//     accumulator) on the stream before using it, but two calls whose work
//     overlaps on the GPU (different streams, no ordering between them) race
//     on the array and produce garbage.  Serialise them;
//   * no cudaMalloc, cudaFree or other allocating call is made.
#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;   // 64 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (cached).
fa_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_bwd_noalloc(const fa_params* p, const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv, void* stream) {
  if (p == nullptr) return FA_ERR_INVALID_ARG;
  const size_t need = fa_bwd_workspace_size(p);
  if (need > fa::kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  void* ws = nullptr;
  const fa_status s = fa::scratch_address(&ws);
  if (s != FA_OK) return s;
  return fa_bwd(p, q, k, v, o, dout, lse, dq, dk, dv, ws, fa::kNoAllocScratchBytes, stream);
}

}  // extern "C"
