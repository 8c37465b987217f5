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
// exits.  Host code only knows a host-side stand-in for its name, so every
// call asks the runtime for its device address on the current device
// (cudaGetSymbolAddress).  The address is not cached: a device reset or a
// re-created primary context reloads the module, and the array may then sit
// elsewhere.  The address is handed to the unchanged fa_bwd path as its
// workspace.
//
// Contract (stated in include/fa.h as well):
//   * problems whose workspace would exceed kNoAllocScratchBytes are refused
//     with FA_ERR_WORKSPACE and nothing is enqueued;
//   * the first call on a device loads the module's device image and looks
//     up the address; make that first call before capturing a stream into a
//     CUDA graph;
//   * every call on a device shares the one array and leaves its contents
//     behind: fa_bwd clears what must start at zero (status word, dQ
//     accumulator) on the stream before using it, but two calls whose work
//     overlaps on the GPU (different streams, no ordering between them) race
//     on the array and produce garbage.  Serialise them;
//   * the status word (a bounded device wait that gave up) sits at the start
//     of the array; fa_noalloc_check_status reads it;
//   * no cudaMalloc, cudaFree or other allocating call is made.
#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;   // 64 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device.
fa_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
  *out = p;
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

fa_status fa_noalloc_check_status(void* stream) {
  void* ws = nullptr;
  const fa_status s = fa::scratch_address(&ws);
  if (s != FA_OK) return s;
  return fa_check_status(ws, stream);
}

fa_status fa_noalloc_scratch(void** addr, size_t* bytes) {
  if (addr == nullptr || bytes == nullptr) return FA_ERR_INVALID_ARG;
  const fa_status s = fa::scratch_address(addr);
  if (s != FA_OK) return s;
  *bytes = fa::kNoAllocScratchBytes;
  return FA_OK;
}

}  // extern "C"
