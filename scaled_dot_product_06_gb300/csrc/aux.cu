// Memory-bound helper kernels of the backward pass and the dropout-mask hook.
//
// * bwd_pre: D = rowsum(dO * O) in fp32 (CK tile fmha_bwd_kernel.hpp,
//   FmhaBwdOGradDotOKernel; the D line of the header equations) next to
//   -LSE * log2(e), in the tiled row-statistics layout of stat_index, and zeroing
//   of dBias, which the key/value-stationary kernel accumulates into (oneDNN
//   sdpa micro.cpp, execute_backward: preprocess and fill of the f32
//   intermediates), and of the fused backward's fp32 dQ accumulator.
// * dq_convert: dQ = scale * dQacc rounded to the io dtype, the fused
//   backward's last step (CK tile fmha_bwd_kernel.hpp FmhaBwdConvertQGradKernel;
//   oneDNN sdpa micro.cpp's postprocess cast of the f32 dQ).
// * dropout_mask: the packed keep bits of the whole problem, drawn by the same
//   device Philox function the fused kernels use (oneDNN's dropout mask output
//   and CK's stored random values serve the same purpose).
#include "common.cuh"

namespace sdpa {

constexpr int kAuxThreads = 256;

static int aux_grid(int64_t work_items) {
  int64_t g = (work_items + kAuxThreads - 1) / kAuxThreads;
  const int64_t cap = 152 * 16;  // a few waves over 152 SMs, grid-stride beyond
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

// One group of DV/8 consecutive threads per row; each thread takes 8 elements.
// Walks the padded rows (s_pad per tensor-map z: (b, h) in batch mode, the head
// for packed sequences) so the padding of the statistics is written too: -inf
// and 0 there, as for a query row that sees no key. Packed, statistics row r
// of a head belongs to the last sequence whose block (packed_stat_row) starts
// at or before r; rows past that sequence's length are padding.
template <bool BF16>
__global__ void __launch_bounds__(kAuxThreads) bwd_pre_kernel(const uint4* __restrict__ o,
                                                              const uint4* __restrict__ dout,
                                                              const float* __restrict__ lse,
                                                              float* __restrict__ stats,
                                                              float4* __restrict__ dbias,
                                                              int64_t z_count, int s_q, int s_pad,
                                                              int rows, const int* __restrict__ seqstart,
                                                              int n_seq, int d_v, int64_t dbias_elems,
                                                              int* __restrict__ counters, int n_counters,
                                                              float4* __restrict__ dq_acc,
                                                              int64_t dq_acc_vec) {
  const int group = d_v / 8;  // 8 or 16 threads per row (power of two)
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int lane = threadIdx.x & 31, sub = lane % group;
  const int64_t rows_per_warp = 32 / group;
  const int64_t warp_id = tid / 32, nwarps = nthreads / 32;
  const int64_t prow_count = z_count * s_pad;
  // wbase is uniform across the warp, so every lane reaches every shuffle
  for (int64_t wbase = warp_id * rows_per_warp; wbase < prow_count; wbase += nwarps * rows_per_warp) {
    const int64_t prow = wbase + lane / group;  // padded row
    const int64_t z = prow / s_pad;
    const int r = static_cast<int>(prow - z * s_pad);
    int q = r, len = s_q;
    int64_t row = z * rows;  // row of O, dO and LSE of local row 0
    if (seqstart != nullptr && prow < prow_count) {
      int lo = 0, hi = n_seq - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (packed_stat_row(packed_rows(seqstart, rows, s_q, mid).x, mid) <= r)
          lo = mid;
        else
          hi = mid - 1;
      }
      const int2 sr = packed_rows(seqstart, rows, s_q, lo);
      q = r - packed_stat_row(sr.x, lo);
      len = sr.y;
      row += sr.x;
    }
    const bool live = prow < prow_count && q >= 0 && q < len;
    row += q;
    float acc = 0.f;
    if (live) {
      const uint4 a = o[row * group + sub];
      const uint4 c = dout[row * group + sub];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = unpack2<BF16>(aw[e]), y = unpack2<BF16>(cw[e]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
    for (int off = group / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, group);
    if (prow < prow_count && sub == 0) {
      const float L = live ? lse[row] : SDPA_NEG_INF;
      const size_t si = stat_index(static_cast<size_t>(z), s_pad, r);
      stats[si] = (L == SDPA_NEG_INF) ? SDPA_NEG_INF : -L * kLog2e;
      stats[si + 64] = -acc;
    }
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t dbias_vec = dbias_elems / 4;
  for (int64_t i = tid; i < dbias_vec; i += nthreads) dbias[i] = z;
  if (tid < (dbias_elems & 3)) reinterpret_cast<float*>(dbias)[dbias_vec * 4 + tid] = 0.f;
  for (int64_t i = tid; i < n_counters; i += nthreads) counters[i] = 0;  // split dK/dV tiles
  for (int64_t i = tid; i < dq_acc_vec; i += nthreads) dq_acc[i] = z;    // fused dQ accumulator
}

// dQ = scale * dQacc in the io dtype, transposed through shared memory so
// that both sides move whole lines: a block takes one 32-row slab of a
// 128-row tile of one z at a time, reads its D/4 column groups (each a
// 512-byte run of the tiled layout of dq_acc_index: per z and tile, per group
// of 4 columns, 128 rows of 16 bytes; one warp a run) into a row-major
// shared buffer, then writes whole dQ rows of the slab, D/8 consecutive
// threads a row, 16 bytes each.
template <bool BF16, int D>
__global__ void __launch_bounds__(kAuxThreads) dq_convert_kernel(const float4* __restrict__ acc,
                                                                 uint4* __restrict__ dq, int64_t z_count,
                                                                 int rows, int dq_tiles, float scale) {
  constexpr int G = D / 4;      // float4 column groups a row
  constexpr int LDV = G + 1;    // shared row stride in float4: 8 consecutive rows hit all 32 banks
  constexpr int C8 = D / 8;     // 16-byte output chunks a row
  __shared__ float4 slab_buf[32 * LDV];
  const int64_t n_slabs = z_count * dq_tiles * 4;
  for (int64_t sl = blockIdx.x; sl < n_slabs; sl += gridDim.x) {  // uniform over the block
    const int64_t zt = sl >> 2;  // z * dq_tiles + tile
    const int64_t z = zt / dq_tiles;
    const int row0 = static_cast<int>(zt - z * dq_tiles) * 128 + static_cast<int>(sl & 3) * 32;
    const float4* src = acc + zt * G * 128 + (sl & 3) * 32;
#pragma unroll
    for (int i = threadIdx.x; i < G * 32; i += kAuxThreads) slab_buf[(i & 31) * LDV + (i >> 5)] = src[(i >> 5) * 128 + (i & 31)];
    __syncthreads();
#pragma unroll
    for (int i = threadIdx.x; i < 32 * C8; i += kAuxThreads) {
      const int r = i / C8, c8 = i % C8;
      if (row0 + r < rows) {
        const float4 a = slab_buf[r * LDV + 2 * c8], b = slab_buf[r * LDV + 2 * c8 + 1];
        dq[(z * rows + row0 + r) * C8 + c8] =
            make_uint4(pack2<BF16>(a.x * scale, a.y * scale), pack2<BF16>(a.z * scale, a.w * scale),
                       pack2<BF16>(b.x * scale, b.y * scale), pack2<BF16>(b.z * scale, b.w * scale));
      }
    }
    __syncthreads();  // the buffer is read before the next slab overwrites it
  }
}

// Word w holds the keep bits of elements 32w .. 32w+31 (bit e = element 32w+e).
__global__ void __launch_bounds__(kAuxThreads) dropout_mask_kernel(int64_t total, uint32_t thr,
                                                                   uint32_t seed_lo, uint32_t seed_hi,
                                                                   uint32_t off_lo, uint32_t off_hi,
                                                                   uint32_t* __restrict__ bits) {
  const int64_t words = (total + 31) / 32;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < words; w += nthreads) {
    uint32_t out = 0;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint64_t grp = static_cast<uint64_t>(w) * 8 + g;
      const uint4 d = dropout_draws(grp, seed_lo, seed_hi, off_lo, off_hi);
      const uint32_t k = static_cast<uint32_t>(d.x >= thr) | (static_cast<uint32_t>(d.y >= thr) << 1) |
                         (static_cast<uint32_t>(d.z >= thr) << 2) | (static_cast<uint32_t>(d.w >= thr) << 3);
      out |= k << (4 * g);
    }
    const int64_t valid = total - w * 32;
    if (valid < 32) out &= (1u << valid) - 1u;
    bits[w] = out;
  }
}

cudaError_t launch_bwd_pre(bool bf16, const void* o, const void* dout, const float* lse, float* stats,
                           float* dbias, int64_t z_count, int s_q, int s_pad, int rows,
                           const int* seqstart, int n_seq, int d_v, int64_t dbias_elems,
                           int* counters, int n_counters, float* dq_acc, int64_t dq_acc_elems,
                           cudaStream_t st) {
  const int group = d_v / 8;
  const int64_t work = z_count * s_pad * group;
  const int64_t zero_work = (dbias_elems + dq_acc_elems) / 4;
  const int grid = aux_grid(work > zero_work ? work : zero_work);
  auto kern = bf16 ? bwd_pre_kernel<true> : bwd_pre_kernel<false>;
  kern<<<grid, kAuxThreads, 0, st>>>(static_cast<const uint4*>(o), static_cast<const uint4*>(dout), lse, stats,
                                      reinterpret_cast<float4*>(dbias), z_count, s_q, s_pad, rows, seqstart,
                                      n_seq, d_v, dbias_elems, counters, n_counters,
                                      reinterpret_cast<float4*>(dq_acc), dq_acc_elems / 4);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(bool bf16, const float* dq_acc, void* dq, int64_t z_count, int rows,
                              int dq_tiles, int d_qk, float scale, cudaStream_t st) {
  const int64_t slabs = z_count * dq_tiles * 4;
  const int grid = static_cast<int>(slabs < 152 * 8 ? slabs : 152 * 8);  // 8 resident blocks an SM
  auto kern = d_qk == 64 ? (bf16 ? dq_convert_kernel<true, 64> : dq_convert_kernel<false, 64>)
                         : (bf16 ? dq_convert_kernel<true, 128> : dq_convert_kernel<false, 128>);
  if (d_qk != 64 && d_qk != 128) return cudaErrorInvalidValue;
  if (slabs == 0) return cudaSuccess;
  kern<<<grid, kAuxThreads, 0, st>>>(reinterpret_cast<const float4*>(dq_acc), static_cast<uint4*>(dq),
                                     z_count, rows, dq_tiles, scale);
  return cudaGetLastError();
}

cudaError_t launch_dropout_mask(int64_t total, uint32_t threshold, uint32_t seed_lo, uint32_t seed_hi,
                                uint32_t off_lo, uint32_t off_hi, uint32_t* bits, cudaStream_t st) {
  const int64_t words = (total + 31) / 32;
  dropout_mask_kernel<<<aux_grid(words), kAuxThreads, 0, st>>>(total, threshold, seed_lo, seed_hi, off_lo,
                                                                off_hi, bits);
  return cudaGetLastError();
}

}  // namespace sdpa
