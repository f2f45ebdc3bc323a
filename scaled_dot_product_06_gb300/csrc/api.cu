// C ABI of libsdpa.so: argument validation, TMA descriptor encoding and kernel
// launches. Mirrors the parameter set of PyTorch cudnn MHA.cpp
// run_cudnn_SDP_fprop / run_cudnn_SDP_bprop (sizes, scale by value, causal
// flag, dropout probability with seed and offset, optional bias, fp32 softmax
// statistics) with plain pointers and a status return instead of exceptions,
// the way oneDNN's sdpa micro.cpp reports failures through status codes.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/sdpa.h"
#include "common.cuh"

namespace {

using namespace sdpa;

// One error word per device, in this library's static device memory.
__device__ uint32_t g_sdpa_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
uint32_t* g_err_ptr[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

thread_local char g_last_error[256] = "";

// Test hook (sdpa_debug_fault): the fault the next forward launches inject and
// the wall-clock limit of their device waits (0 = the default two seconds).
std::atomic<int> g_debug_fault{0};
std::atomic<uint64_t> g_debug_wait_ns{0};

sdpa_status_t fail(sdpa_status_t s, const char* what, cudaError_t e = cudaSuccess) {
  if (e != cudaSuccess)
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, cudaGetErrorString(e));
  else
    snprintf(g_last_error, sizeof(g_last_error), "%s", what);
  return s;
}

sdpa_status_t cuda_status(cudaError_t e, const char* what) {
  return e == cudaSuccess ? SDPA_OK : fail(SDPA_ERR_CUDA, what, e);
}

// Device-side error word of the current device (looked up once per device).
sdpa_status_t error_word_ptr(uint32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(SDPA_ERR_CUDA, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_err_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_sdpa_error_word);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "cudaGetSymbolAddress(error word)", e);
    g_err_ptr[dev] = static_cast<uint32_t*>(ptr);
  }
  *out = g_err_ptr[dev];
  return SDPA_OK;
}

sdpa_status_t encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        fn == nullptr || q != cudaDriverEntryPointSuccess)
      return fail(SDPA_ERR_CUDA, "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = g_encode;
  return SDPA_OK;
}

// Maps encoded by this host thread's recent calls. A training or serving
// loop passes the same tensors step after step, and a lookup costs far less
// host time than an encode; a map depends on nothing but these fields.
struct MapKey {
  const void* ptr;
  int64_t inner, rows, outer;
  uint32_t box_rows;
  int type, elem_bytes, swizzle;
  bool same(const MapKey& o) const {
    return ptr == o.ptr && inner == o.inner && rows == o.rows && outer == o.outer &&
           box_rows == o.box_rows && type == o.type && elem_bytes == o.elem_bytes && swizzle == o.swizzle;
  }
};
struct MapSlot {
  CUtensorMap map;
  MapKey key;
  bool used;
};
constexpr int kMapSlots = 32;
thread_local MapSlot g_maps[kMapSlots];
thread_local int g_map_next = 0;

sdpa_status_t encode_map(CUtensorMap* m, CUtensorMapDataType type, int elem_bytes, const void* ptr,
                         int64_t inner, int64_t rows, int64_t outer, uint32_t box_rows, bool swizzle);

// 3-D map over a [outer][rows][inner] tensor, box {64, box_rows, 1}.
sdpa_status_t make_map(CUtensorMap* m, CUtensorMapDataType type, int elem_bytes, const void* ptr,
                       int64_t inner, int64_t rows, int64_t outer, uint32_t box_rows, bool swizzle) {
  const MapKey key{ptr, inner, rows, outer, box_rows, static_cast<int>(type), elem_bytes, swizzle ? 1 : 0};
  for (int i = 0; i < kMapSlots; ++i) {
    if (g_maps[i].used && g_maps[i].key.same(key)) {
      *m = g_maps[i].map;
      return SDPA_OK;
    }
  }
  if (sdpa_status_t s = encode_map(m, type, elem_bytes, ptr, inner, rows, outer, box_rows, swizzle))
    return s;
  MapSlot& slot = g_maps[g_map_next];
  g_map_next = (g_map_next + 1) % kMapSlots;
  slot.map = *m;
  slot.key = key;
  slot.used = true;
  return SDPA_OK;
}

sdpa_status_t encode_map(CUtensorMap* m, CUtensorMapDataType type, int elem_bytes, const void* ptr,
                         int64_t inner, int64_t rows, int64_t outer, uint32_t box_rows, bool swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  if (sdpa_status_t s = encoder(&enc)) return s;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner * elem_bytes),
                           static_cast<cuuint64_t>(inner * rows * elem_bytes)};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, type, 3, const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed (CUresult %d)",
             static_cast<int>(r));
    return SDPA_ERR_CUDA;
  }
  return SDPA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Map over the fp32 bias [h][s_q][s_kv] for the backward kernels' bias
// tiles, box {box_keys, box_rows, 1 head}: the dQ kernel's {32, 128} with
// the 128-byte swizzle, the dK/dV kernel's {128, query tile rows} plain
// row-major; out-of-range elements read as zero. Needs s_kv % 4 == 0 (row
// strides are multiples of 16 bytes) and a 16-byte-aligned base.
sdpa_status_t encode_bias_map(CUtensorMap* m, const float* bias, int64_t h, int64_t s_q, int64_t s_kv,
                              uint32_t box_keys, uint32_t box_rows, bool swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  if (sdpa_status_t s = encoder(&enc)) return s;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(s_kv), static_cast<cuuint64_t>(s_q), static_cast<cuuint64_t>(h)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(s_kv * 4), static_cast<cuuint64_t>(s_kv * s_q * 4)};
  cuuint32_t box[3] = {box_keys, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(bias), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled (bias) failed (CUresult %d)",
             static_cast<int>(r));
    return SDPA_ERR_CUDA;
  }
  return SDPA_OK;
}

bool head_sizes_ok(int64_t d_qk, int64_t d_v) {
  return (d_qk == 64 && d_v == 64) || (d_qk == 128 && d_v == 128) || (d_qk == 192 && d_v == 128);
}

// Sequence lengths (and packed totals) below 2^29 keep every sum of a row or
// key index with a window offset inside an int on the device.
constexpr int64_t kMaxSeq = (int64_t{1} << 29) - 256;

// A scale whose product with log2(e) is finite (the kernels work in the
// exp2 domain); any sign, zero included.
bool scale_ok(float scale) { return std::isfinite(scale) && std::isfinite(scale * kLog2e); }

// Checks shared by fwd and bwd that need no pointer. Sets *empty for a
// zero-sized problem.
sdpa_status_t check_sizes(int64_t b, int64_t h, int64_t s_q, int64_t s_kv, int64_t d_qk, int64_t d_v,
                          float dropout_p, int dtype, bool* empty) {
  if (b < 0 || h < 0 || s_q < 0 || s_kv < 0 || d_qk < 0 || d_v < 0) return SDPA_ERR_INVALID_ARG;
  if (!(dropout_p >= 0.0f && dropout_p < 1.0f)) return SDPA_ERR_INVALID_ARG;
  if (dtype != SDPA_BF16 && dtype != SDPA_FP16) return SDPA_ERR_UNSUPPORTED;
  if (!head_sizes_ok(d_qk, d_v)) return SDPA_ERR_UNSUPPORTED;
  // b and h bounded one by one before their product, which could overflow
  if (b > (int64_t{1} << 24) || h > (int64_t{1} << 24)) return SDPA_ERR_UNSUPPORTED;
  if (s_q > kMaxSeq || s_kv > kMaxSeq || b * h > (int64_t{1} << 24)) return SDPA_ERR_UNSUPPORTED;
  if (dropout_p > 0.0f && (s_kv % 4) != 0) return SDPA_ERR_UNSUPPORTED;
  *empty = (b == 0 || h == 0 || s_q == 0 || s_kv == 0);
  return SDPA_OK;
}

// h_kv K/V heads serve h query heads: 1 <= h_kv <= h and h_kv divides h (any
// h_kv >= 1 when there are no query heads).
bool kv_heads_ok(int64_t h, int64_t h_kv) {
  if (h_kv < 1 || h_kv > (int64_t{1} << 24)) return h == 0 && h_kv == 0;
  return h == 0 || (h_kv <= h && h % h_kv == 0);
}

uint32_t drop_threshold(float p) {
  return static_cast<uint32_t>(std::floor(static_cast<double>(p) * 4294967296.0));
}

}  // namespace

namespace sdpa {
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

cudaError_t prepare_kernel(const void* kern, int smem, int regs) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> ready;  // (kernel, device) pairs prepared
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& r : ready)
    if (r.first == kern && r.second == dev) return cudaSuccess;
  if (regs > 0) {
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != regs) {
      set_last_error("kernel compiled with an unexpected register count");
      return cudaErrorInvalidConfiguration;
    }
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ready.emplace_back(kern, dev);
  return cudaSuccess;
}
}  // namespace sdpa

namespace {

// Visible keys: key j visible to query i iff i + off - left <= j <= i + off + right,
// off = s_kv - s_q when bottom_right, else 0; a negative size is unbounded.
struct Mask {
  int64_t left, right;
  int bottom_right;
  const float* alibi = nullptr;  // ALiBi slopes (device), slope of (b, h) at b * alibi_stride + h
  int64_t alibi_stride = 0;
  const uint32_t* keep_bits = nullptr;  // dropout keep bits drawn beforehand (device)
  uint32_t* keep_out = nullptr;         // forward: record of the keep bits it draws (device)
};
Mask causal_mask(int is_causal) { return Mask{-1, is_causal ? 0 : -1, 0}; }

// A window size of s_q + s_kv or more admits every key on that side: it is
// stored as unbounded, which keeps the device arithmetic in range.
// general = 0 for the plain kernels' cases (top-left, causal or unmasked).
// ALiBi is aligned top-left under a top-left mask (any window size given),
// bottom-right otherwise.
template <typename P>
void set_window(const Mask& mk, int64_t s_q, int64_t s_kv, P* p) {
  auto norm = [&](int64_t w) { return (w < 0 || w >= s_q + s_kv) ? -1 : static_cast<int>(w); };
  p->win_left = norm(mk.left);
  p->win_right = norm(mk.right);
  p->win_br = mk.bottom_right ? 1 : 0;
  p->win_general = (p->win_left >= 0 || p->win_right > 0 || p->win_br) ? 1 : 0;
  p->alibi = mk.alibi;
  p->alibi_stride = static_cast<int>(mk.alibi_stride);
  const bool masked = mk.left >= 0 || mk.right >= 0;
  p->alibi_br = (masked && !mk.bottom_right) ? 0 : 1;
}

// ALiBi slopes: 4-byte aligned; the stride between batch rows 0 (one row for
// all) or at least h, and small enough for an int index.
sdpa_status_t check_alibi(const Mask& mk, int64_t b, int64_t h) {
  if ((reinterpret_cast<uintptr_t>(mk.keep_bits) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(mk.keep_out) & 3u) != 0)
    return SDPA_ERR_MISALIGNED;
  if (mk.alibi == nullptr) return SDPA_OK;
  if ((reinterpret_cast<uintptr_t>(mk.alibi) & 3u) != 0) return SDPA_ERR_MISALIGNED;
  if (mk.alibi_stride < 0 || (mk.alibi_stride > 0 && mk.alibi_stride < h) ||
      (b - 1) * mk.alibi_stride + h > (int64_t{1} << 30))
    return fail(SDPA_ERR_INVALID_ARG, "alibi_stride");
  return SDPA_OK;
}

// A high-priority side stream and two events per (host thread, device), made
// on first use and kept: the full backward runs the dK/dV kernel there,
// concurrently with the dQ kernel on the caller's stream (both need only the
// preprocess output), so that dQ's CTAs fill the SMs dK/dV's last wave leaves
// idle (dK/dV's CTAs are preferred while any is pending). Per thread, so that
// concurrent callers never share an event. Returns false if they cannot be
// made; the kernels then run one after the other on the caller's stream.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
bool side_stream(SideStream* out) {
  thread_local SideStream cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  SideStream& c = cache[dev];
  if (c.stream == nullptr) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return false;
    SideStream n;
    if (cudaStreamCreateWithPriority(&n.stream, cudaStreamNonBlocking, greatest) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming) != cudaSuccess) {
      cudaStreamDestroy(n.stream);
      return false;
    }
    c = n;
  }
  *out = c;
  return true;
}

// Grouped K/V heads whose key tiles make few CTAs split each group's query
// heads over several CTAs per key tile (BwdParams::kv_split): the largest
// divisor of the group size not above ceil(8 * 152 / CTAs), about eight CTAs
// per SM of a GB300; 1 without groups. Batch mode only.
int64_t dkdv_splits(int64_t b, int64_t h, int64_t h_kv, int64_t s_kv) {
  if (h_kv <= 0 || h <= h_kv || b <= 0 || s_kv <= 0) return 1;
  const int64_t grp = h / h_kv;
  const int64_t ctas = ((s_kv + 127) / 128) * b * h_kv;
  const int64_t want = (8 * 152 + ctas - 1) / ctas;
  int64_t best = 1;
  for (int64_t d = 1; d <= grp; ++d)
    if (grp % d == 0 && d <= want) best = d;
  return best;
}

// Workspace of a split dK/dV past the row statistics: one counter per key
// tile (rounded up to 256 bytes), then the fp32 partial rows.
size_t split_counter_bytes(int64_t b, int64_t h_kv, int64_t s_kv) {
  const size_t tiles = static_cast<size_t>((s_kv + 127) / 128) * b * h_kv;
  return (tiles * sizeof(int) + 255) & ~size_t(255);
}
size_t split_bytes(int64_t b, int64_t h, int64_t h_kv, int64_t s_kv, int64_t d_qk, int64_t d_v) {
  const int64_t ns = dkdv_splits(b, h, h_kv, s_kv);
  if (ns <= 1) return 0;
  const size_t tiles = static_cast<size_t>((s_kv + 127) / 128) * b * h_kv;
  return split_counter_bytes(b, h_kv, s_kv) + tiles * ns * 128 * (d_qk + d_v) * sizeof(float);
}

// Packed-sequence arguments of the varlen entry points; seqstart_q null means
// batch mode (rows of (b, h) contiguous, s_q / s_kv of them).
struct Packing {
  const int32_t* seqstart_q = nullptr;
  const int32_t* seqstart_k = nullptr;
  int64_t total_q = 0, total_k = 0;
};

// Rows and z extent of the 3-D tensor maps ([z][rows][d]) and the statistics
// rows per z: batch mode z = (b, h) with s_q / s_kv rows; packed z = head with
// the packed totals.
struct Rows {
  int64_t q, k, zq, zk, stat_pad;
};
Rows rows_of(const Packing& pk, int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv) {
  if (pk.seqstart_q == nullptr) return Rows{s_q, s_kv, b * h, b * h_kv, stat_pad(static_cast<int>(s_q))};
  return Rows{pk.total_q, pk.total_k, h, h_kv, packed_stat_pad(pk.total_q, b)};
}

// Checks of the packed-sequence arguments (none in batch mode): totals in
// range, both seqstart arrays present and 4-byte aligned, no bias (bias and
// dBias are per padded batch entry on the pages, not defined for packed
// rows). Sets *empty when either total is zero.
sdpa_status_t check_packing(const Packing& pk, int64_t b, const float* bias, bool* empty) {
  if (pk.seqstart_q == nullptr && pk.seqstart_k == nullptr) return SDPA_OK;
  if (pk.total_q < 0 || pk.total_k < 0) return SDPA_ERR_INVALID_ARG;
  if (pk.total_q > kMaxSeq || pk.total_k > kMaxSeq || b > (int64_t{1} << 24) ||
      packed_stat_pad(pk.total_q, b) > (int64_t{1} << 31) - 1)
    return SDPA_ERR_UNSUPPORTED;
  if (bias != nullptr) return fail(SDPA_ERR_UNSUPPORTED, "bias with packed sequences");
  if (pk.total_q == 0 || pk.total_k == 0) *empty = true;
  if (*empty) return SDPA_OK;
  if (pk.seqstart_q == nullptr || pk.seqstart_k == nullptr) return SDPA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(pk.seqstart_q) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(pk.seqstart_k) & 3u) != 0)
    return SDPA_ERR_MISALIGNED;
  return SDPA_OK;
}

// Bytes of the row statistics (-LSE log2e and D per query row, rows padded
// to 128 per (b, h)), rounded up to 256: the whole workspace of the
// deterministic backward.
size_t stats_bytes(int64_t b, int64_t h, int64_t s_q) {
  const size_t prows = static_cast<size_t>(b) * h * static_cast<size_t>(sdpa::stat_pad(static_cast<int>(s_q)));
  return (prows * 2 * sizeof(float) + 255) & ~size_t(255);
}

// Bytes of the fused backward's fp32 dQ accumulator: d_qk floats per query
// row, rows padded to 128 per (b, h) (a multiple of 256 bytes).
size_t dq_acc_bytes(int64_t b, int64_t h, int64_t s_q, int64_t d_qk) {
  return static_cast<size_t>(b) * h * static_cast<size_t>((s_q + 127) / 128) * 128 * d_qk * sizeof(float);
}

// The fused backward (one key/value-stationary kernel that also accumulates
// dQ) serves d_qk <= 128 unless the caller asks for the deterministic
// backward; tensor memory has no room for its dQ tile beside dK at d_qk = 192.
// (Packed calls also need a workspace with room for the accumulator; see
// bwd_impl.)
bool use_fused(int phases, int64_t d_qk) {
  return (phases & SDPA_BWD_DETERMINISTIC) == 0 && d_qk <= 128;
}

// Bytes of the packed statistics: per head, each sequence's rows in a block
// of its own (packed_stat_pad), two floats a row, rounded up to 256.
size_t packed_stats_bytes(int64_t b, int64_t h, int64_t total_q) {
  const size_t prows = static_cast<size_t>(h) * static_cast<size_t>(packed_stat_pad(total_q, b));
  return (prows * 2 * sizeof(float) + 255) & ~size_t(255);
}

sdpa_status_t fwd_impl(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv, int64_t d_qk,
                       int64_t d_v, float scale, const Mask& mask, float dropout_p, uint64_t seed,
                       uint64_t offset, sdpa_dtype_t dtype, const void* q, const void* k,
                       const void* v, const float* bias, void* o, float* lse, void* stream,
                       const Packing& pk) {
  bool empty = false;
  if (sdpa_status_t s = check_sizes(b, h, s_q, s_kv, d_qk, d_v, dropout_p, dtype, &empty)) return s;
  if (!scale_ok(scale)) return fail(SDPA_ERR_INVALID_ARG, "scale must be finite");
  if (!kv_heads_ok(h, h_kv)) return fail(SDPA_ERR_INVALID_ARG, "h_kv must divide h");
  if (sdpa_status_t s = check_packing(pk, b, bias, &empty)) return s;
  if (sdpa_status_t s = check_alibi(mask, b, h)) return s;
  if (dropout_p > 0.0f && mask.keep_out != nullptr) {  // a record of the keep bits drawn
    if (mask.keep_bits != nullptr)
      return fail(SDPA_ERR_INVALID_ARG, "keep_bits and keep_bits_out together");
    if (s_kv % 32 != 0) return fail(SDPA_ERR_UNSUPPORTED, "keep_bits_out needs s_kv % 32 == 0");
  }
  if (empty) return SDPA_OK;
  if (!q || !k || !v || !o || !lse) return SDPA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (bias && !aligned16(bias)))
    return SDPA_ERR_MISALIGNED;

  const bool bf16 = dtype == SDPA_BF16;
  const CUtensorMapDataType tt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const Rows rw = rows_of(pk, b, h, h_kv, s_q, s_kv);
  CUtensorMap mq, mk, mv;
  if (sdpa_status_t s = make_map(&mq, tt, 2, q, d_qk, rw.q, rw.zq, 128, true)) return s;
  if (sdpa_status_t s = make_map(&mk, tt, 2, k, d_qk, rw.k, rw.zk, 128, true)) return s;
  if (sdpa_status_t s = make_map(&mv, tt, 2, v, d_v, rw.k, rw.zk, 128, true)) return s;

  FwdParams p{};
  p.B = static_cast<int>(b);
  p.H = static_cast<int>(h);
  p.H_kv = static_cast<int>(h_kv);
  p.S_q = static_cast<int>(s_q);
  p.S_kv = static_cast<int>(s_kv);
  p.scale_log2 = scale * kLog2e;
  set_window(mask, s_q, s_kv, &p);
  if (dropout_p > 0.0f && mask.keep_bits != nullptr) {  // bits drawn beforehand, [b, h, s_q, s_kv] frame
    p.keep_bits = mask.keep_bits;
    p.keep_words = (b * h * s_q * s_kv + 31) / 32;
  }
  if (dropout_p > 0.0f) p.keep_out = mask.keep_out;  // record the bits drawn here (checked above)
  p.bias = bias;
  p.dropout = dropout_p > 0.0f ? 1 : 0;
  p.drop_threshold = drop_threshold(dropout_p);
  p.keep_scale = 1.0f / (1.0f - dropout_p);
  p.seed_lo = static_cast<uint32_t>(seed);
  p.seed_hi = static_cast<uint32_t>(seed >> 32);
  p.offset_lo = static_cast<uint32_t>(offset);
  p.offset_hi = static_cast<uint32_t>(offset >> 32);
  p.o = o;
  p.lse = lse;
  p.seqstart_q = pk.seqstart_q;
  p.seqstart_k = pk.seqstart_k;
  p.rows_q = static_cast<int>(rw.q);
  p.rows_k = static_cast<int>(rw.k);
  p.fault = static_cast<uint32_t>(g_debug_fault.load());
  const uint64_t wait_ns = g_debug_wait_ns.load();
  p.wait_ns = wait_ns != 0 ? wait_ns : kWaitLimitNs;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // A record over a mask that hides no element (no causal mask or window,
  // batch mode) holds every bit of the frame: the mask kernel draws them at
  // full occupancy, faster than the softmax warps draw them between their
  // other work, and the forward then reads the record it would have written.
  if (p.keep_out != nullptr && pk.seqstart_q == nullptr && p.win_left < 0 && p.win_right < 0) {
    const int64_t total = b * h * s_q * s_kv;
    const cudaError_t me = launch_dropout_mask(total, p.drop_threshold, p.seed_lo, p.seed_hi, p.offset_lo,
                                               p.offset_hi, p.keep_out, st);
    if (me != cudaSuccess) return fail(SDPA_ERR_CUDA, "dropout mask launch", me);
    p.keep_bits = p.keep_out;
    p.keep_words = (total + 31) / 32;
    p.keep_out = nullptr;
  }
  if (sdpa_status_t s = error_word_ptr(&p.err)) return s;
  const cudaError_t e = bf16 ? launch_fwd_bf16(static_cast<int>(d_qk), static_cast<int>(d_v), mq, mk, mv, p, st)
                             : launch_fwd_fp16(static_cast<int>(d_qk), static_cast<int>(d_v), mq, mk, mv, p, st);
  return cuda_status(e, "forward kernel launch");
}


sdpa_status_t bwd_impl(int phases, int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                       int64_t d_qk, int64_t d_v, float scale, const Mask& mask, float dropout_p,
                       uint64_t seed, uint64_t offset, sdpa_dtype_t dtype, const void* q,
                       const void* k, const void* v, const float* bias, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       float* dbias, void* workspace, size_t workspace_bytes, void* stream,
                       const Packing& pk) {
  if ((phases & SDPA_BWD_ALL) == 0 || (phases & ~(SDPA_BWD_ALL | SDPA_BWD_DETERMINISTIC)) != 0)
    return fail(SDPA_ERR_INVALID_ARG, "phases");
  bool empty = false;
  if (sdpa_status_t s = check_sizes(b, h, s_q, s_kv, d_qk, d_v, dropout_p, dtype, &empty)) return s;
  if (!scale_ok(scale)) return fail(SDPA_ERR_INVALID_ARG, "scale must be finite");
  if (!kv_heads_ok(h, h_kv)) return fail(SDPA_ERR_INVALID_ARG, "h_kv must divide h");
  if (sdpa_status_t s = check_packing(pk, b, bias, &empty)) return s;
  if (sdpa_status_t s = check_alibi(mask, b, h)) return s;
  if (empty) return SDPA_OK;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return SDPA_ERR_INVALID_ARG;
  if ((bias == nullptr) != (dbias == nullptr)) return SDPA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (bias && !aligned16(bias)) || (dbias && !aligned16(dbias)))
    return SDPA_ERR_MISALIGNED;
  const size_t stat_bytes = pk.seqstart_q ? packed_stats_bytes(b, h, pk.total_q) : stats_bytes(b, h, s_q);
  // the fused backward's fp32 dQ accumulator follows the statistics (packed:
  // per head, over the packed rows); a packed call whose workspace holds only
  // the statistics runs the deterministic backward
  const size_t acc_bytes = pk.seqstart_q ? dq_acc_bytes(1, h, pk.total_q, d_qk) : dq_acc_bytes(b, h, s_q, d_qk);
  const bool fused = use_fused(phases, d_qk) &&
                     (pk.seqstart_q == nullptr || workspace_bytes >= stat_bytes + acc_bytes);
  const size_t need = stat_bytes + (fused ? acc_bytes : 0);
  if (workspace == nullptr || workspace_bytes < need) return SDPA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SDPA_ERR_MISALIGNED;
  // A split dK/dV when the group is large for the grid and the workspace has
  // the room sdpa_bwd_workspace_size_gqa asks for; else one CTA per key tile.
  int64_t kv_split = pk.seqstart_q ? 1 : dkdv_splits(b, h, h_kv, s_kv);
  if (kv_split > 1 && workspace_bytes < need + split_bytes(b, h, h_kv, s_kv, d_qk, d_v)) kv_split = 1;

  const bool bf16 = dtype == SDPA_BF16;
  const CUtensorMapDataType tt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  float* stats = static_cast<float*>(workspace);
  const Rows rw = rows_of(pk, b, h, h_kv, s_q, s_kv);
  const int di = static_cast<int>(d_qk), dvi = static_cast<int>(d_v);

  BwdParams p{};
  p.B = static_cast<int>(b);
  p.H = static_cast<int>(h);
  p.H_kv = static_cast<int>(h_kv);
  p.S_q = static_cast<int>(s_q);
  p.S_kv = static_cast<int>(s_kv);
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  set_window(mask, s_q, s_kv, &p);
  if (dropout_p > 0.0f && mask.keep_bits != nullptr) {  // bits drawn beforehand, [b, h, s_q, s_kv] frame
    p.keep_bits = mask.keep_bits;
    p.keep_words = (b * h * s_q * s_kv + 31) / 32;
  }
  p.bias = bias;
  p.dbias = dbias;
  p.dropout = dropout_p > 0.0f ? 1 : 0;
  p.drop_threshold = drop_threshold(dropout_p);
  p.keep_scale = 1.0f / (1.0f - dropout_p);
  p.seed_lo = static_cast<uint32_t>(seed);
  p.seed_hi = static_cast<uint32_t>(seed >> 32);
  p.offset_lo = static_cast<uint32_t>(offset);
  p.offset_hi = static_cast<uint32_t>(offset >> 32);
  p.stats = stats;
  p.S_pad = static_cast<int>(rw.stat_pad);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.seqstart_q = pk.seqstart_q;
  p.seqstart_k = pk.seqstart_k;
  p.rows_q = static_cast<int>(rw.q);
  p.rows_k = static_cast<int>(rw.k);
  p.kv_split = static_cast<int>(kv_split);
  // One key tile per (b, h) that every query tile meets (the tile range the
  // fused kernel walks for key tile 0 covers them all): each dQ row then has
  // a single contribution, written directly, and the accumulator, its zeroing
  // and the convert pass drop out. Batch mode only (packed lengths live on
  // the device), and not with split key tiles (whose drain warps hold 24
  // registers).
  bool dq_direct = false;
  if (fused && pk.seqstart_q == nullptr && s_kv <= 128 && kv_split <= 1) {
    const bool win = p.win_general || p.alibi != nullptr;  // the kernel instance's band
    const sdpa::Band bd = win ? sdpa::band_of(p.win_left, p.win_right, p.win_br, p.S_q, p.S_kv)
                              : sdpa::plain_band(p.win_right);
    const sdpa::TileRange r = sdpa::query_tiles_of_keys(win, bd, p.win_right, 0, 128, 128, p.S_q, p.S_kv);
    dq_direct = r.lo == 0 && r.hi == (p.S_q + 127) / 128 - 1;
  }
  p.dq_direct = dq_direct ? 1 : 0;
  if (fused && !dq_direct) {
    p.dq_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + stat_bytes);
    p.dq_tiles = static_cast<int>((rw.q + 127) / 128);
  }
  const int64_t dq_acc_elems = (fused && !dq_direct) ? rw.zq * p.dq_tiles * 128 * d_qk : 0;
  const int n_counters = kv_split > 1 ? static_cast<int>(((s_kv + 127) / 128) * b * h_kv) : 0;
  if (kv_split > 1) {
    uint8_t* extra = static_cast<uint8_t*>(workspace) + need;
    p.dkdv_count = reinterpret_cast<int*>(extra);
    p.dkdv_part = reinterpret_cast<float*>(extra + split_counter_bytes(b, h_kv, s_kv));
  }
  if (sdpa_status_t s = error_word_ptr(&p.err)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  cudaError_t e = cudaSuccess;
  if (phases & SDPA_BWD_PREPROCESS) {
    // dBias is zeroed here for the fused backward; the deterministic one zeroes
    // it in its dK/dV phase, on the dK/dV kernel's stream, so that the zero
    // pass runs beside the dQ kernel instead of ahead of both
    const int64_t dbias_elems = (bias && fused) ? h * s_q * s_kv : 0;
    e = launch_bwd_pre(bf16, o, dout, lse, stats, dbias, rw.zq, static_cast<int>(s_q), p.S_pad, p.rows_q,
                       pk.seqstart_q, static_cast<int>(b), dvi, dbias_elems, p.dkdv_count, n_counters,
                       p.dq_acc, dq_acc_elems, st);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "backward preprocess launch", e);
  }
  // Both main kernels requested: dK/dV on the side stream, forked after the
  // preprocess and joined back before the call returns (see SideStream). The
  // fused backward's convert pass reads what its main kernel accumulates, so
  // both stay on `stream`.
  SideStream side;
  const bool fork = !fused && (phases & SDPA_BWD_DKDV) && (phases & SDPA_BWD_DQ) &&
                    side_stream(&side) &&
                    cudaEventRecord(side.fork, st) == cudaSuccess &&
                    cudaStreamWaitEvent(side.stream, side.fork, 0) == cudaSuccess;
  const cudaStream_t st_dkdv = fork ? side.stream : st;
  auto join = [&]() {
    if (fork) {
      cudaEventRecord(side.join, side.stream);
      cudaStreamWaitEvent(st, side.join, 0);
    }
  };
  if (phases & SDPA_BWD_DKDV) {
    // key/value-stationary kernel: query tiles of 128 rows (64 at d_qk = 192)
    const uint32_t q_rows = d_qk <= 128 ? 128 : 64;
    CUtensorMap mq, mk, mv, mdo;
    sdpa_status_t ms = make_map(&mq, tt, 2, q, d_qk, rw.q, rw.zq, q_rows, true);
    if (!ms) ms = make_map(&mk, tt, 2, k, d_qk, rw.k, rw.zk, 128, true);
    if (!ms) ms = make_map(&mv, tt, 2, v, d_v, rw.k, rw.zk, 128, true);
    if (!ms) ms = make_map(&mdo, tt, 2, dout, d_v, rw.q, rw.zq, q_rows, true);
    // dK and dV leave either kernel by TMA stores, through maps of K's and
    // V's geometry
    CUtensorMap mdk, mdv;
    if (!ms) ms = make_map(&mdk, tt, 2, dk, d_qk, rw.k, rw.zk, 128, true);
    if (!ms) ms = make_map(&mdv, tt, 2, dv, d_v, rw.k, rw.zk, 128, true);
    if (ms) {
      join();
      return ms;
    }
    if (fused) {
      e = bf16 ? launch_bwd_fused_bf16(di, dvi, mq, mk, mv, mdo, mdk, mdv, p, st_dkdv)
               : launch_bwd_fused_fp16(di, dvi, mq, mk, mv, mdo, mdk, mdv, p, st_dkdv);
    } else {
      if (bias != nullptr) {  // dBias = 0 ahead of the kernel's fp32 reductions into it
        e = launch_bwd_pre(bf16, o, dout, lse, stats, dbias, 0, static_cast<int>(s_q), p.S_pad, p.rows_q,
                           nullptr, static_cast<int>(b), dvi, h * s_q * s_kv, nullptr, 0, nullptr, 0, st_dkdv);
        if (e != cudaSuccess) {
          join();
          return fail(SDPA_ERR_CUDA, "backward dBias zero pass launch", e);
        }
      }
      // the bias blocks by TMA where the kernel has room for them (d_qk 64
      // and 192: query tiles of 128 and 64 rows) and the rows are 16-byte
      // multiples; else the kernel reads them from global memory
      CUtensorMap mb{};
      p.bias_tma = 0;
      if (bias != nullptr && d_qk != 128 && s_kv % 4 == 0 &&
          encode_bias_map(&mb, bias, h, s_q, s_kv, 128, q_rows, false) == SDPA_OK)
        p.bias_tma = 1;
      e = bf16 ? launch_bwd_dkdv_bf16(di, dvi, mq, mk, mv, mdo, mb, mdk, mdv, p, st_dkdv)
               : launch_bwd_dkdv_fp16(di, dvi, mq, mk, mv, mdo, mb, mdk, mdv, p, st_dkdv);
    }
    if (e != cudaSuccess) {
      join();
      return fail(SDPA_ERR_CUDA, "backward dK/dV kernel launch", e);
    }
  }
  if ((phases & SDPA_BWD_DQ) && fused) {  // dQ = scale * dQacc in the io dtype
    if (!dq_direct) {
      e = launch_dq_convert(bf16, p.dq_acc, dq, rw.zq, static_cast<int>(rw.q), p.dq_tiles, di, scale, st);
      if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "backward dQ convert launch", e);
    }
  } else if (phases & SDPA_BWD_DQ) {
    CUtensorMap mq, mk, mv, mdo;
    sdpa_status_t ms = make_map(&mq, tt, 2, q, d_qk, rw.q, rw.zq, 128, true);
    if (!ms) ms = make_map(&mk, tt, 2, k, d_qk, rw.k, rw.zk, 128, true);
    if (!ms) ms = make_map(&mv, tt, 2, v, d_v, rw.k, rw.zk, 128, true);
    if (!ms) ms = make_map(&mdo, tt, 2, dout, d_v, rw.q, rw.zq, 128, true);
    CUtensorMap mdq;  // dQ leaves the kernel by TMA stores, through a map of Q's geometry
    if (!ms) ms = make_map(&mdq, tt, 2, dq, d_qk, rw.q, rw.zq, 128, true);
    if (ms) {
      join();
      return ms;
    }
    // the bias tiles by TMA where the kernel has room for them (d_qk 64 and
    // 192) and the rows are 16-byte multiples; else the kernel reads them
    // from global memory
    CUtensorMap mb{};
    p.bias_tma = 0;
    if (bias != nullptr && d_qk != 128 && s_kv % 4 == 0 &&
        encode_bias_map(&mb, bias, h, s_q, s_kv, 32, 128, true) == SDPA_OK)
      p.bias_tma = 1;
    e = bf16 ? launch_bwd_dq_bf16(di, dvi, mq, mk, mv, mdo, mb, mdq, p, st)
             : launch_bwd_dq_fp16(di, dvi, mq, mk, mv, mdo, mb, mdq, p, st);
    if (e != cudaSuccess) {
      join();
      return fail(SDPA_ERR_CUDA, "backward dQ kernel launch", e);
    }
  }
  join();
  return SDPA_OK;
}

}  // namespace

extern "C" {

const char* sdpa_status_string(sdpa_status_t s) {
  switch (s) {
    case SDPA_OK: return "SDPA_OK";
    case SDPA_ERR_INVALID_ARG: return "SDPA_ERR_INVALID_ARG: invalid argument";
    case SDPA_ERR_UNSUPPORTED: return "SDPA_ERR_UNSUPPORTED: unsupported configuration";
    case SDPA_ERR_MISALIGNED: return "SDPA_ERR_MISALIGNED: pointer not 16-byte aligned";
    case SDPA_ERR_WORKSPACE: return "SDPA_ERR_WORKSPACE: workspace missing or too small";
    case SDPA_ERR_CUDA: return "SDPA_ERR_CUDA: CUDA call failed";
    case SDPA_ERR_DEVICE_TIMEOUT: return "SDPA_ERR_DEVICE_TIMEOUT: a kernel wait ran out";
  }
  return "unknown sdpa status";
}

int sdpa_version(void) { return 10100; }

const char* sdpa_last_error(void) { return g_last_error; }

sdpa_status_t sdpa_debug_fault(int fault, uint64_t wait_limit_ns) {
  if (fault < 0 || fault > 1) return SDPA_ERR_INVALID_ARG;
  g_debug_fault.store(fault);
  g_debug_wait_ns.store(wait_limit_ns);
  return SDPA_OK;
}

int64_t sdpa_tile_ranges(int kernel, int64_t s_q, int64_t s_kv, int64_t window_left,
                         int64_t window_right, int bottom_right, int windowed, int query_rows,
                         int32_t* out, int64_t cap) {
  if (kernel < 0 || kernel > 2 || (query_rows != 64 && query_rows != 128) || s_q < 0 || s_kv < 0 ||
      s_q > kMaxSeq || s_kv > kMaxSeq || cap < 0 || (cap > 0 && out == nullptr))
    return -1;
  // the window as the launchers hand it to the kernels
  FwdParams w{};
  set_window(Mask{window_left, window_right, bottom_right}, s_q, s_kv, &w);
  const int S_q = static_cast<int>(s_q), S_kv = static_cast<int>(s_kv);
  const bool win = w.win_general != 0 || windowed != 0;
  const Band bd = win ? band_of(w.win_left, w.win_right, w.win_br, S_q, S_kv) : plain_band(w.win_right);
  constexpr int kTile = 128;  // forward and dQ query tiles; key tiles everywhere
  int64_t n = 0;
  auto emit = [&](int q0, int rows, int kt) {
    if (n < cap) {
      out[3 * n] = q0;
      out[3 * n + 1] = rows;
      out[3 * n + 2] = kt;
    }
    ++n;
  };
  if (kernel == 0) {  // forward: pairs of query tiles, key tiles from the diagonal down
    const int n_pairs = ((S_q + kTile - 1) / kTile + 1) / 2;
    for (int qt = 0; qt < n_pairs; ++qt) {
      const QueryPair qp = query_pair(qt, S_q, kTile);
      const TileRange kr[2] = {key_tiles_of_rows(bd, qp.q0, kTile, kTile, S_q, S_kv),
                               key_tiles_of_rows(bd, qp.lone ? S_q : qp.q0 + kTile, kTile, kTile, S_q, S_kv)};
      const FwdIters it = fwd_iters(kr[0], kr[1]);
      const IterSpan sp[2] = {fwd_tile_iters(kr[0], it), fwd_tile_iters(kr[1], it)};
      for (int j = 0; j < it.n_it; ++j)
        for (int t = 0; t < 2; ++t)
          if (sp[t].first <= j && j <= sp[t].last) emit(qp.q0 + t * kTile, kTile, it.khi - j);
    }
  } else if (kernel == 1) {  // key/value-stationary: a CTA per key tile
    for (int kt = 0; kt * kTile < S_kv; ++kt) {
      const TileRange qr = query_tiles_of_keys(win, bd, w.win_right, kt * kTile, kTile, query_rows, S_q, S_kv);
      for (int i = qr.lo; i <= qr.hi; ++i) emit(i * query_rows, query_rows, kt);
    }
  } else {  // query-stationary dQ: a CTA per query tile, key tiles from the diagonal down
    for (int q0 = 0; q0 < S_q; q0 += kTile) {
      const TileRange kr = win ? key_tiles_of_rows(bd, q0, kTile, kTile, S_q, S_kv)
                               : key_tiles_plain(w.win_right >= 0, q0, kTile, kTile, S_kv);
      for (int j = 0; j <= kr.hi - kr.lo; ++j) emit(q0, kTile, kr.hi - j);
    }
  }
  return n;
}

size_t sdpa_bwd_workspace_size_ex(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                                  int64_t d_qk, int64_t d_v, int deterministic) {
  bool empty = false;
  if (check_sizes(b, h, s_q, s_kv, d_qk, d_v, 0.0f, SDPA_BF16, &empty) != SDPA_OK) return 0;
  if (!kv_heads_ok(h, h_kv)) return 0;
  const int phases = SDPA_BWD_ALL | (deterministic ? SDPA_BWD_DETERMINISTIC : 0);
  const size_t base = stats_bytes(b, h, s_q) +
                      (use_fused(phases, d_qk) ? dq_acc_bytes(b, h, s_q, d_qk) : 0);
  return base + split_bytes(b, h, h_kv, s_kv, d_qk, d_v);
}

size_t sdpa_bwd_workspace_size_gqa(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                                   int64_t d_qk, int64_t d_v) {
  return sdpa_bwd_workspace_size_ex(b, h, h_kv, s_q, s_kv, d_qk, d_v, 0);
}

size_t sdpa_bwd_workspace_size(int64_t b, int64_t h, int64_t s_q, int64_t s_kv, int64_t d_qk,
                               int64_t d_v) {
  return sdpa_bwd_workspace_size_ex(b, h, h, s_q, s_kv, d_qk, d_v, 0);
}

sdpa_status_t sdpa_fwd_gqa(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                           int64_t d_qk, int64_t d_v, float scale, int is_causal, float dropout_p,
                           uint64_t seed, uint64_t offset, sdpa_dtype_t dtype, const void* q,
                           const void* k, const void* v, const float* bias, void* o, float* lse,
                           void* stream) {
  return fwd_impl(b, h, h_kv, s_q, s_kv, d_qk, d_v, scale, causal_mask(is_causal), dropout_p, seed,
                  offset, dtype, q, k, v, bias, o, lse, stream, Packing{});
}

sdpa_status_t sdpa_bwd_phases_gqa(int phases, int64_t b, int64_t h, int64_t h_kv, int64_t s_q,
                                  int64_t s_kv, int64_t d_qk, int64_t d_v, float scale,
                                  int is_causal, float dropout_p, uint64_t seed, uint64_t offset,
                                  sdpa_dtype_t dtype, const void* q, const void* k, const void* v,
                                  const float* bias, const void* o, const void* dout,
                                  const float* lse, void* dq, void* dk, void* dv, float* dbias,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(phases, b, h, h_kv, s_q, s_kv, d_qk, d_v, scale, causal_mask(is_causal), dropout_p,
                  seed, offset, dtype, q, k, v, bias, o, dout, lse, dq, dk, dv, dbias, workspace,
                  workspace_bytes, stream, Packing{});
}

// Packed sequences: b sequences, the i-th owning packed rows
// [seqstart_q[i], seqstart_q[i+1]) of the queries and [seqstart_k[i],
// seqstart_k[i+1]) of the keys of every head; max_seqlen_q / max_seqlen_k take
// the place of s_q / s_kv.
size_t sdpa_bwd_varlen_workspace_size(int64_t b, int64_t h, int64_t total_q) {
  if (b < 0 || h < 0 || total_q < 0 || total_q > kMaxSeq || b > (int64_t{1} << 24)) return 0;
  return packed_stats_bytes(b, h, total_q);
}

size_t sdpa_bwd_varlen_workspace_size_ex(int64_t b, int64_t h, int64_t total_q, int64_t d_qk,
                                         int deterministic) {
  if (h > (int64_t{1} << 24) || (d_qk != 64 && d_qk != 128 && d_qk != 192)) return 0;
  const size_t base = sdpa_bwd_varlen_workspace_size(b, h, total_q);
  if (base == 0) return 0;
  const int phases = SDPA_BWD_ALL | (deterministic ? SDPA_BWD_DETERMINISTIC : 0);
  return base + (use_fused(phases, d_qk) ? dq_acc_bytes(1, h, total_q, d_qk) : 0);
}

sdpa_status_t sdpa_fwd_varlen(int64_t b, int64_t h, int64_t h_kv, int64_t total_q, int64_t total_k,
                              int64_t max_seqlen_q, int64_t max_seqlen_k, int64_t d_qk, int64_t d_v,
                              float scale, int is_causal, float dropout_p, uint64_t seed,
                              uint64_t offset, sdpa_dtype_t dtype, const int32_t* seqstart_q,
                              const int32_t* seqstart_k, const void* q, const void* k, const void* v,
                              void* o, float* lse, void* stream) {
  const Packing pk{seqstart_q, seqstart_k, total_q, total_k};
  if (seqstart_q == nullptr || seqstart_k == nullptr) {
    if (b == 0 || h == 0 || total_q == 0 || total_k == 0) return SDPA_OK;
    return fail(SDPA_ERR_INVALID_ARG, "seqstart_q and seqstart_k are required");
  }
  return fwd_impl(b, h, h_kv, max_seqlen_q, max_seqlen_k, d_qk, d_v, scale, causal_mask(is_causal),
                  dropout_p, seed, offset, dtype, q, k, v, nullptr, o, lse, stream, pk);
}

sdpa_status_t sdpa_bwd_phases_varlen(int phases, int64_t b, int64_t h, int64_t h_kv, int64_t total_q,
                                     int64_t total_k, int64_t max_seqlen_q, int64_t max_seqlen_k,
                                     int64_t d_qk, int64_t d_v, float scale, int is_causal,
                                     float dropout_p, uint64_t seed, uint64_t offset,
                                     sdpa_dtype_t dtype, const int32_t* seqstart_q,
                                     const int32_t* seqstart_k, const void* q, const void* k,
                                     const void* v, const void* o, const void* dout,
                                     const float* lse, void* dq, void* dk, void* dv,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  const Packing pk{seqstart_q, seqstart_k, total_q, total_k};
  if (seqstart_q == nullptr || seqstart_k == nullptr) {
    if (b == 0 || h == 0 || total_q == 0 || total_k == 0) return SDPA_OK;
    return fail(SDPA_ERR_INVALID_ARG, "seqstart_q and seqstart_k are required");
  }
  return bwd_impl(phases, b, h, h_kv, max_seqlen_q, max_seqlen_k, d_qk, d_v, scale,
                  causal_mask(is_causal), dropout_p, seed, offset, dtype, q, k, v, nullptr, o, dout,
                  lse, dq, dk, dv, nullptr, workspace, workspace_bytes, stream, pk);
}

sdpa_status_t sdpa_bwd_varlen(int64_t b, int64_t h, int64_t h_kv, int64_t total_q, int64_t total_k,
                              int64_t max_seqlen_q, int64_t max_seqlen_k, int64_t d_qk, int64_t d_v,
                              float scale, int is_causal, float dropout_p, uint64_t seed,
                              uint64_t offset, sdpa_dtype_t dtype, const int32_t* seqstart_q,
                              const int32_t* seqstart_k, const void* q, const void* k, const void* v,
                              const void* o, const void* dout, const float* lse, void* dq, void* dk,
                              void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  return sdpa_bwd_phases_varlen(SDPA_BWD_ALL, b, h, h_kv, total_q, total_k, max_seqlen_q,
                                max_seqlen_k, d_qk, d_v, scale, is_causal, dropout_p, seed, offset,
                                dtype, seqstart_q, seqstart_k, q, k, v, o, dout, lse, dq, dk, dv,
                                workspace, workspace_bytes, stream);
}

// Local windows and the bottom-right alignment (batch and packed forms).
sdpa_status_t sdpa_fwd_ex(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                              int64_t d_qk, int64_t d_v, float scale, int64_t window_left,
                              int64_t window_right, int bottom_right, const float* alibi_slopes,
                              int64_t alibi_stride, const uint32_t* keep_bits, uint32_t* keep_bits_out,
                              float dropout_p, uint64_t seed,
                              uint64_t offset, sdpa_dtype_t dtype, const void* q, const void* k,
                              const void* v, const float* bias, void* o, float* lse, void* stream) {
  return fwd_impl(b, h, h_kv, s_q, s_kv, d_qk, d_v, scale,
                  Mask{window_left, window_right, bottom_right, alibi_slopes, alibi_stride, keep_bits,
                       keep_bits_out},
                  dropout_p, seed, offset, dtype, q, k, v, bias, o, lse, stream, Packing{});
}

sdpa_status_t sdpa_bwd_phases_ex(int phases, int64_t b, int64_t h, int64_t h_kv, int64_t s_q,
                                     int64_t s_kv, int64_t d_qk, int64_t d_v, float scale,
                                     int64_t window_left, int64_t window_right, int bottom_right,
                                     const float* alibi_slopes, int64_t alibi_stride, const uint32_t* keep_bits,
                                     float dropout_p, uint64_t seed, uint64_t offset,
                                     sdpa_dtype_t dtype, const void* q, const void* k, const void* v,
                                     const float* bias, const void* o, const void* dout,
                                     const float* lse, void* dq, void* dk, void* dv, float* dbias,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(phases, b, h, h_kv, s_q, s_kv, d_qk, d_v, scale,
                  Mask{window_left, window_right, bottom_right, alibi_slopes, alibi_stride, keep_bits},
                  dropout_p, seed, offset, dtype, q, k, v, bias, o, dout, lse, dq, dk, dv, dbias,
                  workspace, workspace_bytes, stream, Packing{});
}

sdpa_status_t sdpa_bwd_ex(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                              int64_t d_qk, int64_t d_v, float scale, int64_t window_left,
                              int64_t window_right, int bottom_right, const float* alibi_slopes,
                              int64_t alibi_stride, const uint32_t* keep_bits, float dropout_p, uint64_t seed,
                              uint64_t offset, sdpa_dtype_t dtype, const void* q, const void* k,
                              const void* v, const float* bias, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, float* dbias,
                              void* workspace, size_t workspace_bytes, void* stream) {
  return sdpa_bwd_phases_ex(SDPA_BWD_ALL, b, h, h_kv, s_q, s_kv, d_qk, d_v, scale, window_left,
                                window_right, bottom_right, alibi_slopes, alibi_stride, keep_bits, dropout_p,
                                seed, offset, dtype, q, k, v, bias, o, dout, lse, dq, dk, dv, dbias,
                                workspace, workspace_bytes, stream);
}

sdpa_status_t sdpa_fwd_varlen_ex(int64_t b, int64_t h, int64_t h_kv, int64_t total_q,
                                     int64_t total_k, int64_t max_seqlen_q, int64_t max_seqlen_k,
                                     int64_t d_qk, int64_t d_v, float scale, int64_t window_left,
                                     int64_t window_right, int bottom_right,
                                     const float* alibi_slopes, int64_t alibi_stride, const uint32_t* keep_bits,
                                     uint32_t* keep_bits_out, float dropout_p, uint64_t seed, uint64_t offset,
                                     sdpa_dtype_t dtype, const int32_t* seqstart_q,
                                     const int32_t* seqstart_k, const void* q, const void* k,
                                     const void* v, void* o, float* lse, void* stream) {
  const Packing pk{seqstart_q, seqstart_k, total_q, total_k};
  if (seqstart_q == nullptr || seqstart_k == nullptr) {
    if (b == 0 || h == 0 || total_q == 0 || total_k == 0) return SDPA_OK;
    return fail(SDPA_ERR_INVALID_ARG, "seqstart_q and seqstart_k are required");
  }
  return fwd_impl(b, h, h_kv, max_seqlen_q, max_seqlen_k, d_qk, d_v, scale,
                  Mask{window_left, window_right, bottom_right, alibi_slopes, alibi_stride, keep_bits,
                       keep_bits_out},
                  dropout_p, seed, offset, dtype, q, k, v, nullptr, o, lse, stream, pk);
}

sdpa_status_t sdpa_bwd_phases_varlen_ex(
    int phases, int64_t b, int64_t h, int64_t h_kv, int64_t total_q, int64_t total_k,
    int64_t max_seqlen_q, int64_t max_seqlen_k, int64_t d_qk, int64_t d_v, float scale,
    int64_t window_left, int64_t window_right, int bottom_right, const float* alibi_slopes,
    int64_t alibi_stride, const uint32_t* keep_bits, float dropout_p, uint64_t seed, uint64_t offset, sdpa_dtype_t dtype,
    const int32_t* seqstart_q, const int32_t* seqstart_k, const void* q, const void* k,
    const void* v, const void* o, const void* dout, const float* lse, void* dq, void* dk, void* dv,
    void* workspace, size_t workspace_bytes, void* stream) {
  const Packing pk{seqstart_q, seqstart_k, total_q, total_k};
  if (seqstart_q == nullptr || seqstart_k == nullptr) {
    if (b == 0 || h == 0 || total_q == 0 || total_k == 0) return SDPA_OK;
    return fail(SDPA_ERR_INVALID_ARG, "seqstart_q and seqstart_k are required");
  }
  return bwd_impl(phases, b, h, h_kv, max_seqlen_q, max_seqlen_k, d_qk, d_v, scale,
                  Mask{window_left, window_right, bottom_right, alibi_slopes, alibi_stride, keep_bits},
                  dropout_p, seed, offset, dtype, q, k, v, nullptr, o, dout, lse, dq, dk, dv,
                  nullptr, workspace, workspace_bytes, stream, pk);
}

sdpa_status_t sdpa_bwd_varlen_ex(int64_t b, int64_t h, int64_t h_kv, int64_t total_q,
                                     int64_t total_k, int64_t max_seqlen_q, int64_t max_seqlen_k,
                                     int64_t d_qk, int64_t d_v, float scale, int64_t window_left,
                                     int64_t window_right, int bottom_right,
                                     const float* alibi_slopes, int64_t alibi_stride, const uint32_t* keep_bits,
                                     float dropout_p, uint64_t seed, uint64_t offset,
                                     sdpa_dtype_t dtype, const int32_t* seqstart_q,
                                     const int32_t* seqstart_k, const void* q, const void* k,
                                     const void* v, const void* o, const void* dout,
                                     const float* lse, void* dq, void* dk, void* dv,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  return sdpa_bwd_phases_varlen_ex(SDPA_BWD_ALL, b, h, h_kv, total_q, total_k, max_seqlen_q,
                                       max_seqlen_k, d_qk, d_v, scale, window_left, window_right,
                                       bottom_right, alibi_slopes, alibi_stride, keep_bits, dropout_p, seed,
                                       offset, dtype, seqstart_q, seqstart_k, q, k, v, o, dout, lse,
                                       dq, dk, dv, workspace, workspace_bytes, stream);
}

sdpa_status_t sdpa_bwd_gqa(int64_t b, int64_t h, int64_t h_kv, int64_t s_q, int64_t s_kv,
                           int64_t d_qk, int64_t d_v, float scale, int is_causal, float dropout_p,
                           uint64_t seed, uint64_t offset, sdpa_dtype_t dtype, const void* q,
                           const void* k, const void* v, const float* bias, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           float* dbias, void* workspace, size_t workspace_bytes, void* stream) {
  return sdpa_bwd_phases_gqa(SDPA_BWD_ALL, b, h, h_kv, s_q, s_kv, d_qk, d_v, scale, is_causal,
                             dropout_p, seed, offset, dtype, q, k, v, bias, o, dout, lse, dq, dk,
                             dv, dbias, workspace, workspace_bytes, stream);
}

// The ungrouped entry points: every query head has its own K/V head.
sdpa_status_t sdpa_fwd(int64_t b, int64_t h, int64_t s_q, int64_t s_kv, int64_t d_qk, int64_t d_v,
                       float scale, int is_causal, float dropout_p, uint64_t seed, uint64_t offset,
                       sdpa_dtype_t dtype, const void* q, const void* k, const void* v,
                       const float* bias, void* o, float* lse, void* stream) {
  return sdpa_fwd_gqa(b, h, h, s_q, s_kv, d_qk, d_v, scale, is_causal, dropout_p, seed, offset,
                      dtype, q, k, v, bias, o, lse, stream);
}

sdpa_status_t sdpa_bwd_phases(int phases, int64_t b, int64_t h, int64_t s_q, int64_t s_kv,
                              int64_t d_qk, int64_t d_v, float scale, int is_causal,
                              float dropout_p, uint64_t seed, uint64_t offset, sdpa_dtype_t dtype,
                              const void* q, const void* k, const void* v, const float* bias,
                              const void* o, const void* dout, const float* lse, void* dq, void* dk,
                              void* dv, float* dbias, void* workspace, size_t workspace_bytes,
                              void* stream) {
  return sdpa_bwd_phases_gqa(phases, b, h, h, s_q, s_kv, d_qk, d_v, scale, is_causal, dropout_p,
                             seed, offset, dtype, q, k, v, bias, o, dout, lse, dq, dk, dv, dbias,
                             workspace, workspace_bytes, stream);
}

sdpa_status_t sdpa_bwd(int64_t b, int64_t h, int64_t s_q, int64_t s_kv, int64_t d_qk, int64_t d_v,
                       float scale, int is_causal, float dropout_p, uint64_t seed, uint64_t offset,
                       sdpa_dtype_t dtype, const void* q, const void* k, const void* v,
                       const float* bias, const void* o, const void* dout, const float* lse,
                       void* dq, void* dk, void* dv, float* dbias, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return sdpa_bwd_phases_gqa(SDPA_BWD_ALL, b, h, h, s_q, s_kv, d_qk, d_v, scale, is_causal,
                             dropout_p, seed, offset, dtype, q, k, v, bias, o, dout, lse, dq, dk,
                             dv, dbias, workspace, workspace_bytes, stream);
}

sdpa_status_t sdpa_dropout_mask(int64_t b, int64_t h, int64_t s_q, int64_t s_kv, float dropout_p,
                                uint64_t seed, uint64_t offset, uint32_t* bits, void* stream) {
  if (b < 0 || h < 0 || s_q < 0 || s_kv < 0) return SDPA_ERR_INVALID_ARG;
  if (!(dropout_p >= 0.0f && dropout_p < 1.0f)) return SDPA_ERR_INVALID_ARG;
  const int64_t total = b * h * s_q * s_kv;
  if (total == 0) return SDPA_OK;
  if (bits == nullptr) return SDPA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(bits) & 3u) != 0) return SDPA_ERR_MISALIGNED;
  return cuda_status(launch_dropout_mask(total, drop_threshold(dropout_p), static_cast<uint32_t>(seed),
                                         static_cast<uint32_t>(seed >> 32), static_cast<uint32_t>(offset),
                                         static_cast<uint32_t>(offset >> 32), bits,
                                         static_cast<cudaStream_t>(stream)),
                     "dropout mask launch");
}

sdpa_status_t sdpa_device_error(uint32_t* word, int clear) {
  uint32_t* dev_word = nullptr;
  if (sdpa_status_t s = error_word_ptr(&dev_word)) return s;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "cudaDeviceSynchronize", e);
  uint32_t host = 0;
  e = cudaMemcpy(&host, dev_word, sizeof(host), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "reading the error word", e);
  if (clear && host != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpy(dev_word, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "clearing the error word", e);
  }
  if (word) *word = host;
  return host ? SDPA_ERR_DEVICE_TIMEOUT : SDPA_OK;
}

}  // extern "C"
