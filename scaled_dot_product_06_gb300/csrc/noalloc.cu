// sdpa_bwd_noalloc: the backward pass without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// backward pass: a host framework that hands every byte of the GPU to its own
// pool and forbids allocations from outside it, or a latency-critical loop
// where cudaMalloc's implicit device synchronisation and unbounded latency are
// not acceptable. For them this entry point keeps the backward scratch (the
// per-row statistics D = rowsum(dO * O) and -LSE*log2e that the backward
// kernels share) in a fixed,
// file-scope device array that exists for as long as the library is loaded,
// on every GPU that loads it. It calls no cudaMalloc, cudaFree or other
// allocating routine. It runs the deterministic backward
// (SDPA_BWD_DETERMINISTIC), whose scratch is only those statistics, so its
// results are bitwise those of sdpa_bwd_phases with that flag.
//
// Limits and sharing:
// * The array holds kNoAllocScratchBytes (16 MiB). A problem whose scratch
//   (sdpa_bwd_workspace_size_ex with deterministic = 1) is larger is
//   rejected with SDPA_ERR_WORKSPACE.
// * Every call on a device uses the same array and leaves its contents behind;
//   the preprocess kernel of each call overwrites the statistics before the other kernels
//   read it, so nothing carries over.
//   Calls whose kernels overlap on the GPU (for example on two streams at
//   once) race on the array and give wrong gradients: serialise them.
// * Host code cannot use the array's name as a device address. The first call
//   on each device looks the address up with cudaGetSymbolAddress while that
//   device is current and caches it; make that first call before any stream
//   capture begins.
#include <mutex>

#include "../../include/sdpa.h"
#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t{16} << 20;

// The scratch itself. Only device code may name it directly.
static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device (looked up once).
sdpa_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    sdpa::set_last_error("sdpa_bwd_noalloc: cudaGetDevice failed");
    return SDPA_ERR_CUDA;
  }
  if (dev >= kMaxDevices) {
    sdpa::set_last_error("sdpa_bwd_noalloc: device index exceeds the 64-device scratch cache");
    return SDPA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || ptr == nullptr) {
      sdpa::set_last_error("sdpa_bwd_noalloc: cudaGetSymbolAddress of the static scratch failed");
      return SDPA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return SDPA_OK;
}

}  // namespace

extern "C" {

sdpa_status_t sdpa_bwd_noalloc(int64_t b, int64_t h, int64_t s_q, int64_t s_kv, int64_t d_qk,
                               int64_t d_v, float scale, int is_causal, float dropout_p,
                               uint64_t seed, uint64_t offset, sdpa_dtype_t dtype, const void* q,
                               const void* k, const void* v, const float* bias, const void* o,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               float* dbias, void* stream) {
  // Validate everything but the workspace without touching CUDA: sdpa_bwd
  // checks sizes, pointers and alignment first and, given no workspace,
  // answers SDPA_ERR_WORKSPACE only when all of them are fine (an empty
  // problem returns SDPA_OK there and launches nothing).
  constexpr int kPhases = SDPA_BWD_ALL | SDPA_BWD_DETERMINISTIC;
  const sdpa_status_t pre =
      sdpa_bwd_phases(kPhases, b, h, s_q, s_kv, d_qk, d_v, scale, is_causal, dropout_p, seed, offset,
                      dtype, q, k, v, bias, o, dout, lse, dq, dk, dv, dbias, nullptr, 0, stream);
  if (pre != SDPA_ERR_WORKSPACE) return pre;
  if (sdpa_bwd_workspace_size_ex(b, h, h, s_q, s_kv, d_qk, d_v, 1) > kNoAllocScratchBytes) {
    sdpa::set_last_error(
        "sdpa_bwd_noalloc: the problem needs more backward scratch than the 16 MiB static array "
        "holds; use sdpa_bwd with a caller-allocated workspace");
    return SDPA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  if (sdpa_status_t s = scratch_address(&scratch)) return s;
  return sdpa_bwd_phases(kPhases, b, h, s_q, s_kv, d_qk, d_v, scale, is_causal, dropout_p, seed,
                         offset, dtype, q, k, v, bias, o, dout, lse, dq, dk, dv, dbias, scratch,
                         kNoAllocScratchBytes, stream);
}

}  // extern "C"
