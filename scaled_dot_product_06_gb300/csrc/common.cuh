// Device helpers and launch parameters shared by the attention kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace sdpa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
#define SDPA_NEG_INF (-__int_as_float(0x7f800000))

// Error-word site codes (bitwise OR of the sites whose wait ran out).
enum : uint32_t {
  kSiteFwdLoad = 1u << 0,
  kSiteFwdMma = 1u << 1,
  kSiteFwdSoftmax = 1u << 2,
  kSiteBwdLoad = 1u << 4,
  kSiteBwdMma = 1u << 5,
  kSiteBwdCompute = 1u << 6,
  kSiteDrain = 1u << 8,
  kSiteSmemAlign = 1u << 9,  // dynamic shared memory not 1024-byte aligned
};

struct FwdParams {
  int B, H, S_q, S_kv;
  int H_kv;                // K/V heads; query head h reads K/V head h / (H / H_kv)
  float scale_log2;        // softmax scale * log2(e)
  // Visible keys (CK's window_size_left / window_size_right and top-left /
  // bottom-right mask type): key j is visible to query i iff
  // i + off - win_left <= j <= i + off + win_right with off = S_kv - S_q (the
  // sequence's lengths) when win_br, else 0; a negative size leaves that side
  // unbounded. Causal is (-1, 0, 0); no mask (-1, -1, 0). See Band.
  int win_left, win_right, win_br;
  int win_general;         // 0: top-left, causal (win_right = 0) or unmasked (-1)
  // Dropout keep bits drawn beforehand (sdpa_dropout_mask's packing: bit
  // L % 32 of word L / 32, L the linear element index of the dropout rule) or
  // null to draw them here; keep_words is the array's length in words.
  const uint32_t* keep_bits;
  int64_t keep_words;
  // Record of the keep bits drawn here (same packing; null: none), for the
  // backward to read instead of drawing them again. Written only while
  // drawing (keep_bits null), whole words of a row (the host requires
  // S_kv % 32 == 0).
  uint32_t* keep_out;
  // ALiBi (null: none): score of (i, j) gets -alibi[b * alibi_stride + h] *
  // |j - i - off|, off = S_kv - S_q when alibi_br, else 0 (a top-left mask).
  // Handled by the kernels compiled for general windows.
  const float* alibi;
  int alibi_stride, alibi_br;
  const float* bias;       // [1, H, S_q, S_kv] fp32 or null
  int dropout;             // 0 / 1
  uint32_t drop_threshold; // drop iff draw < threshold
  float keep_scale;        // 1 / (1 - p)
  uint32_t seed_lo, seed_hi, offset_lo, offset_hi;
  void* o;                 // [B, H, S_q, D_v] io dtype
  float* lse;              // [B, H, S_q] natural-log logsumexp
  uint32_t* err;           // device error word
  // Packed sequences (both null in batch mode): sequence b owns rows
  // [seqstart_q[b], seqstart_q[b+1]) of every query head of Q, O and LSE and
  // rows [seqstart_k[b], seqstart_k[b+1]) of every K/V head of K and V. B is
  // then the number of sequences and S_q / S_kv the longest lengths, which
  // size the grid and stride the dropout index (see SeqSlice).
  const int* seqstart_q;
  const int* seqstart_k;
  int rows_q, rows_k;      // rows per head of the tensors: S_q / S_kv, or the packed totals
  // Test hook (sdpa_debug_fault): 1 = the producer issues no K/V loads, so
  // the MMA issuer's bounded wait runs out; wait_ns = limit of every wait.
  uint32_t fault;
  uint64_t wait_ns;
};

// Row statistics the backward kernels share, written by the preprocess kernel:
// for each (b, h) and each block of 64 query rows (S_q padded to a multiple
// of 128), 64 floats -LSE * log2(e) followed by 64 floats -D, D = rowsum(dO * O)
// (negated so dP - D is one fused multiply-add, also with the dropout factor).
// A tile of 64 or 128 query rows is thus one contiguous run of 512 or 1024
// bytes, fetched with one bulk copy. Rows past S_q hold -inf and 0.
__host__ __device__ __forceinline__ size_t stat_index(size_t bh, int S_pad, int q) {
  return (bh * static_cast<size_t>(S_pad) + static_cast<size_t>(q & ~63)) * 2 + static_cast<size_t>(q & 63);
}
__host__ __device__ __forceinline__ int stat_pad(int S_q) { return (S_q + 127) & ~127; }

// The visible keys of query row i are [i + lo, i + hi] (clamp to [0, S_kv)
// where used); an unbounded side is +-2^30. The host keeps sequence lengths
// below 2^29 and window sizes below S_q + S_kv (larger ones are unbounded),
// so every sum of a row or key index with lo or hi fits in an int.
constexpr int kUnbounded = 1 << 30;
struct Band {
  int lo, hi;
};
__host__ __device__ __forceinline__ Band band_of(int win_left, int win_right, int win_br, int S_q, int S_kv) {
  const int off = win_br ? S_kv - S_q : 0;
  return Band{win_left < 0 ? -kUnbounded : off - win_left, win_right < 0 ? kUnbounded : off + win_right};
}

// ---- tile ranges: which tiles each kernel walks. The kernels and the
// library's host-side range check (sdpa_tile_ranges) call these same
// functions, so a test of the one tests the other.
__host__ __device__ __forceinline__ int imin(int a, int b) {
#ifdef __CUDA_ARCH__
  return min(a, b);
#else
  return a < b ? a : b;
#endif
}
__host__ __device__ __forceinline__ int imax(int a, int b) {
#ifdef __CUDA_ARCH__
  return max(a, b);
#else
  return a > b ? a : b;
#endif
}

// The band of the plain kernels: top-left, causal when win_right >= 0.
__host__ __device__ __forceinline__ Band plain_band(int win_right) {
  return Band{-kUnbounded, win_right >= 0 ? 0 : kUnbounded};
}

// Tiles [lo, hi] of a range; lo > hi when empty.
struct TileRange {
  int lo, hi;
};

// Key tiles (bn keys each) holding a key that some row of [q0, q0 + rows)
// sees under the band; empty when q0 >= S_q or no row sees a key.
__host__ __device__ __forceinline__ TileRange key_tiles_of_rows(Band bd, int q0, int rows, int bn, int S_q,
                                                              int S_kv) {
  TileRange r{0, -1};
  if (q0 < S_q) {
    const int lo = imax(q0 + bd.lo, 0), hi = imin(imin(q0 + rows, S_q) - 1 + bd.hi, S_kv - 1);
    if (lo <= hi) r = TileRange{lo / bn, hi / bn};
  }
  return r;
}

// The same for the plain masks in closed form (the dQ kernel's plain
// instances): every key tile, or those up to the tile holding the last row's
// diagonal key under the causal mask.
__host__ __device__ __forceinline__ TileRange key_tiles_plain(bool causal, int q0, int rows, int bn, int S_kv) {
  const int n_all = (S_kv + bn - 1) / bn;
  return TileRange{0, (causal ? imin(n_all, (q0 + rows - 1) / bn + 1) : n_all) - 1};
}

// Query tiles (bm rows each) holding a row that sees some key of
// [k0, k0 + bn): under a general band (win), else the plain masks' closed
// form (from the diagonal tile down, or every tile).
__host__ __device__ __forceinline__ TileRange query_tiles_of_keys(bool win, Band bd, int win_right, int k0,
                                                                 int bn, int bm, int S_q, int S_kv) {
  if (win) {
    const int qlo = imax(k0 - bd.hi, 0), qhi = imin(imin(k0 + bn, S_kv) - 1 - bd.lo, S_q - 1);
    return qlo <= qhi ? TileRange{qlo / bm, qhi / bm} : TileRange{qlo / bm, qlo / bm - 1};
  }
  const int n_qt = (S_q + bm - 1) / bm;
  return TileRange{win_right >= 0 ? imin(n_qt, k0 / bm) : 0, n_qt - 1};
}

// The forward's pair of query tiles number qt of a sequence of S_q rows:
// tiles (0,1), (2,3), ... for an even tile count; tile 0 alone and then
// (1,2), (3,4), ... for an odd one, so the tile without a partner is the one
// with the fewest causal key tiles. q0 is the first row of the pair's tile 0.
struct QueryPair {
  int q0;
  bool lone;  // tile 1 of the pair does not exist
};
__host__ __device__ __forceinline__ QueryPair query_pair(int qt, int S_q, int bm) {
  const int n = (S_q + bm - 1) / bm;
  const bool odd = (n & 1) != 0;
  return QueryPair{(odd ? imax(2 * qt - 1, 0) : 2 * qt) * bm, odd && qt == 0};
}

// The forward's walk over a pair whose tiles see key tiles k0 and k1:
// iteration j (of n_it) visits key tile khi - j, from the diagonal down, and
// a query tile takes part in the iterations [first, last] of its own range
// (first > last when it sees no key).
struct FwdIters {
  int khi, n_it;
};
__host__ __device__ __forceinline__ FwdIters fwd_iters(TileRange k0, TileRange k1) {
  const bool has0 = k0.lo <= k0.hi, has1 = k1.lo <= k1.hi;
  const int khi = imax(k0.hi, k1.hi);
  return FwdIters{khi, (has0 || has1) ? khi - (has0 ? k0.lo : k1.lo) + 1 : 0};
}
struct IterSpan {
  int first, last;
};
__host__ __device__ __forceinline__ IterSpan fwd_tile_iters(TileRange k, FwdIters it) {
  return k.lo <= k.hi ? IterSpan{it.khi - k.hi, it.khi - k.lo} : IterSpan{it.n_it, -1};
}

// The band kept in shared memory and re-read where a loop needs it, so that
// it does not hold two registers through the loop (volatile: read each time).
__device__ __forceinline__ Band lds_band(const void* p) {
  int lo, hi;
  asm volatile("ld.shared.v2.s32 {%0, %1}, [%2];" : "=r"(lo), "=r"(hi) : "r"(smem_u32(p)));
  return Band{lo, hi};
}

// Packed sequences: the statistics of head z hold one block per sequence,
// sequence b's at row packed_stat_row(start_b, b) (start_b its first packed
// query row), padded to a multiple of 128 rows. start rounded up to 64 plus
// 192 per earlier sequence keeps the blocks disjoint (the next block begins at
// least len_b + 129 rows later) without a prefix sum, and packed_stat_pad
// rows per head hold them all for any start_b + len_b <= rows.
__host__ __device__ __forceinline__ int packed_stat_row(int start, int b) {
  return ((start + 63) & ~63) + 192 * b;
}
__host__ __device__ __forceinline__ int64_t packed_stat_pad(int64_t rows, int64_t n_seq) {
  return ((rows + 63) & ~int64_t{63}) + 192 * n_seq + 128;
}

// First row and length of packed sequence b, clamped so that any contents of
// seqstart stay inside [0, rows) and the length inside [0, max_len].
__device__ __forceinline__ int2 packed_rows(const int* seqstart, int rows, int max_len, int b) {
  const int s0 = min(max(__ldg(seqstart + b), 0), rows);
  const int s1 = min(max(__ldg(seqstart + b + 1), s0), rows);
  return make_int2(s0, min(s1 - s0, max_len));
}

// What one (sequence or batch entry) b of a call covers: its lengths, the
// packed rows of its first query and key, the tensor-map z of its query head
// 0 and K/V head 0 (z of head h = zq0 + h), and its first statistics row.
// In batch mode the rows of (b, h) form z = b * H + h; packed, z is the head.
struct SeqSlice {
  int len_q, len_k;
  int row_q, row_k;
  int zq0, zk0;
  int stat_row;
};
__device__ __forceinline__ SeqSlice seq_slice(const int* seqstart_q, const int* seqstart_k, int rows_q,
                                              int rows_k, int S_q, int S_kv, int H, int H_kv, int b) {
  if (seqstart_q == nullptr) return SeqSlice{S_q, S_kv, 0, 0, b * H, b * H_kv, 0};
  const int2 q = packed_rows(seqstart_q, rows_q, S_q, b);
  const int2 k = packed_rows(seqstart_k, rows_k, S_kv, b);
  return SeqSlice{q.y, k.y, q.x, k.x, 0, 0, packed_stat_row(q.x, b)};
}

// Order of the query tiles of the query-stationary kernels (forward, dQ):
// heads in groups of G, the largest divisor of H not above gmax, one group
// after another; within a group the causal tiles with the most key tiles first,
// across the group's heads; batch fastest (the batches of one head share
// Bias rows). The CTAs resident together then read the K and V of at most G
// heads (which stay in L2; with all heads in flight the forward and dQ read
// K and V 5-7 times from DRAM), while the grid still ends on its lightest
// tiles (one head after another would end on a head's heaviest tile).
struct QueryTile {
  int b, h, qt;
};
__device__ __forceinline__ QueryTile query_tile_order(int idx, int B, int H, int n_qt, int gmax) {
  int G = H < gmax ? H : gmax;
  while (H % G != 0) --G;
  const int b = idx % B;
  const int r = idx / B;
  const int g = r / (n_qt * G), w = r % (n_qt * G);
  return QueryTile{b, g * G + w % G, n_qt - 1 - w / G};
}

struct BwdParams {
  int B, H, S_q, S_kv;
  int H_kv;                // K/V heads; query head h reads K/V head h / (H / H_kv)
  float scale;             // softmax scale
  float scale_log2;        // scale * log2(e)
  int win_left, win_right, win_br;  // visible keys, as in FwdParams
  int win_general;
  const float* alibi;      // ALiBi slopes, as in FwdParams
  int alibi_stride, alibi_br;
  // Grouped K/V heads with a small grid: kv_split CTAs share a key tile, each
  // summing dK / dV over grp / kv_split query heads into fp32 partial rows
  // (dkdv_part, [tile][split][BN][d_qk + d_v]); the last of them to count
  // itself in (dkdv_count[tile]) adds the partials in split order and writes
  // dK / dV, so the result does not depend on which CTA finished last.
  int kv_split;
  float* dkdv_part;
  int* dkdv_count;
  const float* bias;       // [1, H, S_q, S_kv] or null
  float* dbias;            // [1, H, S_q, S_kv] or null (accumulated with atomics)
  int dropout;
  uint32_t drop_threshold;
  float keep_scale;
  uint32_t seed_lo, seed_hi, offset_lo, offset_hi;
  const float* stats;      // row statistics, see stat_index
  int S_pad;               // S_q rounded up to a multiple of 128
  void* dq;                // [B, H, S_q, D_qk]
  void* dk;                // [B, H, S_kv, D_qk]
  void* dv;                // [B, H, S_kv, D_v]
  uint32_t* err;
  const int* seqstart_q;   // packed sequences, as in FwdParams (null in batch mode)
  const int* seqstart_k;
  int rows_q, rows_k;
  const uint32_t* keep_bits;  // dropout keep bits drawn beforehand, as in FwdParams
  int64_t keep_words;
  // fp32 dQ accumulator of the fused backward (bwd_fused_kernel.cuh,
  // dq_acc_index): dq_tiles 128-row tiles per tensor-map z; null otherwise.
  float* dq_acc;
  int dq_tiles;
  // fused backward with one key tile per (b, h) that every query tile meets:
  // each dQ row has one contribution, which the drain writes to dq directly
  // (scaled, in the io dtype) with no accumulator and no convert pass
  int dq_direct;
  // the dQ kernel's bias tiles come by TMA into shared memory (the map
  // passed beside the operands' maps is valid): set where the bias is
  // present, its row is a multiple of 16 bytes and the buffer fits
  int bias_tma;
};

// ---------------------------------------------------------------- Philox4x32-10
// Restated from Salmon et al., "Parallel random numbers: as easy as 1, 2, 3"
// (SC'11): ten rounds of two 32x32->64 multiplies mixed into the counter,
// with the key bumped by the two Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += W0;
      k1 += W1;
    }
    const uint32_t hi0 = __umulhi(M0, c.x), lo0 = M0 * c.x;
    const uint32_t hi1 = __umulhi(M1, c.z), lo1 = M1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Keep flags of elements L0 .. L0 + 31 from packed keep bits (bit L % 32 of
// word L / 32): two words joined by a funnel shift; words past the array
// (elements past the problem, which callers mask anyway) read as 0.
__device__ __forceinline__ uint32_t keep_word(const uint32_t* bits, int64_t n_words, uint64_t L0) {
  const int64_t w = static_cast<int64_t>(L0 >> 5);
  const uint32_t sh = static_cast<uint32_t>(L0 & 31);
  const uint32_t lo = w < n_words ? __ldg(bits + w) : 0u;
  const uint32_t hi = (sh != 0 && w + 1 < n_words) ? __ldg(bits + w + 1) : 0u;
  return __funnelshift_r(lo, hi, sh);
}

// The four draws of linear-index group g (elements 4g .. 4g+3).
__device__ __forceinline__ uint4 dropout_draws(uint64_t g, uint32_t seed_lo, uint32_t seed_hi,
                                               uint32_t off_lo, uint32_t off_hi) {
  return philox4x32_10(make_uint4(off_lo, off_hi, static_cast<uint32_t>(g),
                                  static_cast<uint32_t>(g >> 32)),
                       seed_lo, seed_hi);
}

// ---------------------------------------------------------------- arithmetic
// Packed pairs of fp32 (sm_100 family f32x2 arithmetic): one instruction does
// two lanes' worth of FMA-pipe work, halving the issue slots the softmax and
// dS loops spend on it (the pipe throughput itself is unchanged).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2split(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Three-input max / min (sm_100 family): one instruction takes two more
// scores into a running maximum.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Largest (MIN: smallest) of x[0, N), N a multiple of 8, in four chains.
template <bool MIN, int N>
__device__ __forceinline__ float extreme_of(const float* x) {
  static_assert(N % 8 == 0, "extreme_of");
  auto f3 = [](float a, float b, float c) { return MIN ? fmin3(a, b, c) : fmax3(a, b, c); };
  float a0 = x[0], a1 = x[1], a2 = x[2], a3 = x[3];
#pragma unroll
  for (int i = 4; i < N - 4; i += 8) {
    a0 = f3(a0, x[i], x[i + 4]);
    a1 = f3(a1, x[i + 1], x[i + 5]);
    a2 = f3(a2, x[i + 2], x[i + 6]);
    a3 = f3(a3, x[i + 3], x[i + 7]);
  }
  a0 = f3(a0, a1, x[N - 4]);
  a2 = f3(a2, a3, x[N - 3]);
  return f3(a0, a2, f3(x[N - 2], x[N - 1], x[N - 1]));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
    return __bfloat1622float2(v);
  } else {
    __half2 v = *reinterpret_cast<__half2*>(&w);
    return __half22float2(v);
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Copies elements [e0, e0 + N) of row `row` of a 128-byte-swizzled K-major
// shared-memory tile (64-element boxes of `rows_per_box` rows, as TMA writes
// them) into the calling thread's TMEM lane at `taddr`, two elements per
// 32-bit column: the layout of an MMA A operand read from tensor memory.
// taddr must address column e0 / 2 of the thread's own lane. Caller waits with
// tmem_wait_st() before signalling the MMA issuer.
template <int N>
__device__ __forceinline__ void smem_row_to_tmem(const uint8_t* tile, int rows_per_box, int row,
                                                 int e0, uint32_t taddr) {
  static_assert(N % 32 == 0, "whole 16-column stores");
#pragma unroll
  for (int c = 0; c < N / 32; ++c) {
    uint32_t r[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = e0 + c * 32 + q * 8;
      const int chunk = (e & 63) >> 3;
      const uint4 v = *reinterpret_cast<const uint4*>(tile + (e >> 6) * rows_per_box * 128 +
                                                      row * 128 + ((chunk ^ (row & 7)) << 4));
      r[4 * q + 0] = v.x;
      r[4 * q + 1] = v.y;
      r[4 * q + 2] = v.z;
      r[4 * q + 3] = v.w;
    }
    tmem_st16(taddr + c * 16, r);
  }
}

// Records a failure detail for sdpa_last_error() on the calling thread.
void set_last_error(const char* msg);

// One-time per (kernel, device) launch preparation: raises the kernel's
// dynamic shared-memory limit to `smem` and, when regs > 0, checks that the
// compiled kernel uses exactly `regs` registers a thread. The result is
// cached, so later launches on the device skip these driver calls (they cost
// microseconds, which dominate small problems).
cudaError_t prepare_kernel(const void* kern, int smem, int regs);

// ---------------------------------------------------------------- launchers
// Defined in the per-dtype kernel translation units; return a CUDA error
// (cudaErrorInvalidValue for a head-size pair that has no kernel).
cudaError_t launch_fwd_bf16(int d_qk, int d_v, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, const FwdParams& p, cudaStream_t st);
cudaError_t launch_fwd_fp16(int d_qk, int d_v, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, const FwdParams& p, cudaStream_t st);
cudaError_t launch_bwd_dkdv_bf16(int d_qk, int d_v, const CUtensorMap& q, const CUtensorMap& k,
                                 const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& bias,
                                 const CUtensorMap& dk, const CUtensorMap& dv, const BwdParams& p,
                                 cudaStream_t st);
cudaError_t launch_bwd_dkdv_fp16(int d_qk, int d_v, const CUtensorMap& q, const CUtensorMap& k,
                                 const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& bias,
                                 const CUtensorMap& dk, const CUtensorMap& dv, const BwdParams& p,
                                 cudaStream_t st);
cudaError_t launch_bwd_dq_bf16(int d_qk, int d_v, const CUtensorMap& q, const CUtensorMap& k,
                               const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& bias,
                               const CUtensorMap& dq, const BwdParams& p,
                               cudaStream_t st);
cudaError_t launch_bwd_dq_fp16(int d_qk, int d_v, const CUtensorMap& q, const CUtensorMap& k,
                               const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& bias,
                               const CUtensorMap& dq, const BwdParams& p,
                               cudaStream_t st);
cudaError_t launch_bwd_fused_bf16(int d_qk, int d_v, const CUtensorMap& q, const CUtensorMap& k,
                                  const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& dk,
                                  const CUtensorMap& dv, const BwdParams& p, cudaStream_t st);
cudaError_t launch_bwd_fused_fp16(int d_qk, int d_v, const CUtensorMap& q, const CUtensorMap& k,
                                  const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& dk,
                                  const CUtensorMap& dv, const BwdParams& p, cudaStream_t st);
cudaError_t launch_bwd_pre(bool bf16, const void* o, const void* dout, const float* lse, float* stats,
                           float* dbias, int64_t z_count, int s_q, int s_pad, int rows,
                           const int* seqstart, int n_seq, int d_v, int64_t dbias_elems,
                           int* counters, int n_counters, float* dq_acc, int64_t dq_acc_elems,
                           cudaStream_t st);
cudaError_t launch_dq_convert(bool bf16, const float* dq_acc, void* dq, int64_t z_count, int rows,
                              int dq_tiles, int d_qk, float scale, cudaStream_t st);
cudaError_t launch_dropout_mask(int64_t total, uint32_t threshold, uint32_t seed_lo,
                                uint32_t seed_hi, uint32_t off_lo, uint32_t off_hi,
                                uint32_t* bits, cudaStream_t st);

}  // namespace sdpa
