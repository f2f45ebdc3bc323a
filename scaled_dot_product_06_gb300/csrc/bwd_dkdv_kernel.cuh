// Attention backward, key/value-stationary half: dK, dV and dBias (sm_103a).
//
// Computes the dV, dS, dBias and dK lines of the equation block that opens CK
// tile's fmha_bwd_kernel.hpp: dV = P^T dO, dP = dO V^T, dS = P * (dP - D),
// dBias = dS, dK = dS^T Q * scale, with dropout entering as P~ = P * Z
// (Z = keep / (1 - p)) in dV and dS = P * (dP * Z - D). P is recomputed from
// the saved logsumexp, P = exp(S * scale + Bias - LSE), and D = rowsum(dO * O)
// comes from the preprocess kernel. dQ is produced by the query-stationary
// kernel in bwd_dq_kernel.cuh, so this kernel has no cross-CTA accumulation
// other than dBias.
//
// One CTA owns 128 key rows of one (b, h) (K_j and V_j stay resident) and
// loops over query tiles of BM rows (128, or 64 at d_qk = 192 where tensor
// memory is short). Every product keeps the 128 keys in the MMA's M dimension
// (the TMEM lanes):
//   S^T  = K Q_i^T      [128 x BM]  A = K,              B = Q_i (smem, K-major)
//   dP^T = V dO_i^T     [128 x BM]  A = V,              B = dO_i (smem, K-major)
//   dV  += P~^T dO_i    [128 x Dv]  A = P~^T (TMEM),    B = dO_i (smem, MN-major)
//   dK  += dS^T Q_i     [128 x Dk]  A = dS^T (TMEM),    B = Q_i (smem, MN-major)
// K and V are read from shared memory, or, when tensor memory has room for
// them next to the accumulators (d_qk = 64), copied once per CTA into TMEM so
// that S^T and dP^T read only their B operand from shared memory.
// Roles (BM/32 compute warpgroups, a producer warp and an MMA warp):
//   compute    warp w owns key rows 32*(w%4)..+31 (its TMEM lanes) and query
//              columns [32*hf, 32*hf + 32), hf = w/4, so each scheduler runs
//              BM/32 compute warps whose latencies hide one another.
//              Recomputes P^T, releasing the S^T columns as soon as they are
//              in registers; then writes P~^T and dS^T (io dtype, two per
//              column) over the 32 dP^T columns it reads, P~^T in the first
//              16 and dS^T in the second 16, and adds dS into dBias (fp32
//              atomics).
//   producer   TMA for K, V once and Q_i, dO_i through a 2-stage ring; the
//              row statistics of tile i (-LSE*log2e and D, one bulk copy)
//              ride with Q_i on its barrier and in its ring slot.
//   MMA        one lane issues, order per tile i: S^T(i+1) once S^T(i) is
//              in registers, dV(i), dK(i), dP^T(i+1). Tensor memory has no
//              room for a second S^T buffer, so P~^T must not stay in the S^T
//              columns (it would hold S^T(i+1) back until dV(i) had read it,
//              putting dV(i) + S^T(i+1) + the whole softmax on the per-tile
//              critical path). In the dP^T columns it is free of that: the
//              in-order tensor pipe finishes dV(i) before dP^T(i+1)
//              overwrites them. So the softmax of tile i overlaps S^T(i+1),
//              dS(i) overlaps dV(i), and the next softmax overlaps dK(i) and
//              dP^T(i+1).
// Tensor memory (512 columns): S^T [0,BM), dP^T [BM,2BM), dV [2BM,2BM+Dv),
// dK [2BM+Dv, 2BM+Dv+Dk), then K and V (two elements per column) if they fit.
// At the end the compute warps stage dV and dK in the Q / dO stages, idle by
// then, and one thread stores them by TMA.
#pragma once
#include <type_traits>

#include "common.cuh"

namespace sdpa {

template <int DQK, int DV>
struct DkdvCfg {
  static constexpr int DQK_ = DQK, DV_ = DV;
  static constexpr int BN = 128;                      // key rows per CTA
  static constexpr int BM = (DQK <= 128) ? 128 : 64;  // query rows per tile
  static constexpr int NQ = BM / 32;                  // compute warpgroups (32 query columns each)
  static constexpr int CW = BM / NQ;                  // query columns per compute thread
  static constexpr int NCT = 128 * NQ;                // compute threads
  static constexpr int STAGES = 2;
  static constexpr int K_BYTES = BN * DQK * 2;
  static constexpr int V_BYTES = BN * DV * 2;
  static constexpr int Q_BYTES = BM * DQK * 2;
  static constexpr int DO_BYTES = BM * DV * 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + K_BYTES;
  static constexpr int OFF_Q = OFF_V + V_BYTES;
  static constexpr int OFF_DO = OFF_Q + STAGES * Q_BYTES;
  static constexpr int STAT_BYTES = 2 * BM * 4;       // -LSE log2e and D of BM query rows
  static constexpr int OFF_ROW = OFF_DO + STAGES * DO_BYTES;  // [STAGES] row statistics
  // The bias block of a query tile ([BM query rows][BN keys] fp32, row-major,
  // so a warp's 32 keys of one query row are one 128-byte run), loaded by
  // TMA one tile ahead, where it fits (d_qk = 64 and 192; at d_qk = 128 the
  // bias is read from global memory).
  static constexpr int BIAS_BYTES = BM * BN * 4;
  static constexpr int OFF_BIAS = (OFF_ROW + STAGES * STAT_BYTES + 1023) & ~1023;
  static constexpr bool BIAS_TMA_OK = OFF_BIAS + BIAS_BYTES + 256 + 1024 <= 227 * 1024;
  static constexpr int OFF_BAR = BIAS_TMA_OK ? OFF_BIAS + BIAS_BYTES : OFF_ROW + STAGES * STAT_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr int THREADS = NCT + 64;            // + producer warp + MMA warp
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0, T_DP = BM, T_DV = 2 * BM, T_DK = 2 * BM + DV;
  // K and V, the operands every tile reuses, live in TMEM when they fit, so
  // S^T and dP^T take A from TMEM and read only Q_i / dO_i from shared memory.
  static constexpr uint32_t T_K = T_DK + DQK, T_V = T_K + DQK / 2;
  static constexpr bool OPS_IN_TMEM = T_V + DV / 2 <= 512;
  static_assert(T_DK + DQK <= 512, "tensor memory overflow");
  static_assert(SMEM <= 227 * 1024, "shared memory overflow");
  static_assert(DQK % 64 == 0 && DV % 64 == 0 && DV <= 128 && DQK <= 192, "head size");
  static_assert(CW == 32, "one 32-column TMEM load per compute thread and tile");
};

enum : int { AB_KV = 0, AB_QF, AB_DOF = AB_QF + 2, AB_QE = AB_DOF + 2, AB_S = AB_QE + 2, AB_SFREE,
             AB_P, AB_DP, AB_DSL, AB_DSH, AB_DKDV, AB_DRAIN, AB_OPS, AB_BF, AB_BE, AB_COUNT };

// Keep bits of key row k for the 32 query rows [row0, row0 + 32) of a tile.
// One Philox block covers four consecutive keys of one query row, i.e. the
// four lanes of a quad (lane 4g + w owns key 4g + w), so lane 4g + w draws the
// blocks of query rows row0 + 4r + w (r < 8) and the quad exchanges the bits.
// lin_quad is the linear index of (query row row0, first key of the quad).
// Returns m[src]: bit r = keep flag of query row row0 + 4r + src.
__device__ __forceinline__ void keep_bits_transposed(uint64_t lin_quad, int S_kv, int lane,
                                                     uint32_t thr, uint32_t seed_lo,
                                                     uint32_t seed_hi, uint32_t off_lo,
                                                     uint32_t off_hi, uint32_t (&m)[4]) {
  const int w = lane & 3;
  uint32_t a = 0;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const uint64_t L = lin_quad + static_cast<uint64_t>(4 * r + w) * S_kv;
    const uint4 d = dropout_draws(L >> 2, seed_lo, seed_hi, off_lo, off_hi);
    a |= (static_cast<uint32_t>(d.x >= thr) << r) | (static_cast<uint32_t>(d.y >= thr) << (8 + r)) |
         (static_cast<uint32_t>(d.z >= thr) << (16 + r)) | (static_cast<uint32_t>(d.w >= thr) << (24 + r));
  }
#pragma unroll
  for (int src = 0; src < 4; ++src) {
    const uint32_t x = __shfl_sync(0xffffffffu, a, (lane & ~3) | src);
    m[src] = (x >> (8 * w)) & 0xFFu;
  }
}

// Bit r of x to bit 4 r (r < 8).
__device__ __forceinline__ uint32_t spread4(uint32_t x) {
  x = (x | (x << 12)) & 0x000F000Fu;
  x = (x | (x << 6)) & 0x03030303u;
  return (x | (x << 3)) & 0x11111111u;
}

// Keep flags of one key for the 32 query rows [q0, q0 + 32) as one word, bit
// c = flag of query row q0 + c. The warp's lanes hold 32 consecutive keys
// key0 + lane. With keep bits drawn beforehand (sdpa_dropout_mask's packing,
// row-major: bit L % 32 of word L / 32), lane l reads the 32 flags of query
// row q0 + l for keys key0 .. key0 + 31 (one word, or two joined) and a warp
// bit-matrix transpose hands each lane its key's column;
// otherwise the flags are drawn (keep_bits_transposed) and their bits, which
// come grouped by query row modulo 4, are put in order.
// lin_q0_key0 is the linear element index of (q0, key0).
// The keep bits lane `lane` contributes to keep_flags_of_key: query row
// q0 + lane, keys key0 .. key0 + 31 (kernels may load it a tile early).
__device__ __forceinline__ uint32_t keep_row_word(const uint32_t* keep_bits, int64_t keep_words,
                                                  uint64_t lin_q0_key0, int S_kv, int lane) {
  return keep_word(keep_bits, keep_words, lin_q0_key0 + static_cast<uint64_t>(lane) * S_kv);
}
// The 32 words of a warp (lane l: keep_row_word of query row q0 + l) as a
// 32 x 32 bit matrix (row = lane, column = bit), transposed: bit c of the
// result is lane c's bit `lane`. Five rounds of the recursive block
// transpose: in round s the lanes l and l ^ s swap the off-diagonal s x s
// blocks of their 2s x 2s block (the lower lane's low column half moves up
// into the upper lane, the upper lane's high half down into the lower lane).
__device__ __forceinline__ uint32_t transpose_keep_words(uint32_t w, int lane) {
  uint32_t m = 0x0000FFFFu;  // columns in the low half of each 2s-column group
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1, m ^= (m << sh)) {
    const uint32_t o = __shfl_xor_sync(0xffffffffu, w, sh);
    w = (lane & sh) ? (((o >> sh) & m) | (w & ~m)) : ((w & m) | ((o & m) << sh));
  }
  return w;
}

__device__ __forceinline__ uint32_t keep_flags_of_key(const uint32_t* keep_bits, int64_t keep_words,
                                                      uint64_t lin_q0_key0, int S_kv, int lane,
                                                      uint32_t thr, uint32_t seed_lo, uint32_t seed_hi,
                                                      uint32_t off_lo, uint32_t off_hi) {
  if (keep_bits != nullptr)
    return transpose_keep_words(keep_row_word(keep_bits, keep_words, lin_q0_key0, S_kv, lane), lane);
  uint32_t m[4];
  keep_bits_transposed(lin_q0_key0 + (lane & ~3), S_kv, lane, thr, seed_lo, seed_hi, off_lo, off_hi, m);
  // m[src] bit r = flag of query row q0 + 4 r + src
  return spread4(m[0]) | (spread4(m[1]) << 1) | (spread4(m[2]) << 2) | (spread4(m[3]) << 3);
}

// Epilogue of a split key tile (BwdParams::kv_split > 1), run by all NCT
// compute threads: this CTA's fp32 dK / dV sums go to its partial rows
// [dK | dV]; after a fence, one atomic per key tile counts the CTA in, and the
// CTA that completes the count adds every split's partial rows in split order
// (the same sum whichever finishes last), scales dK, rounds, writes dK / dV
// and resets the counter. tl = TMEM base plus the warp's lane offset.
template <typename C, bool BF16>
__device__ __noinline__ void split_epilogue(float* dkdv_part, int* dkdv_count, int nsp, int tile,
                                            int sp, bool ready, bool kv_ok, int row, int hf,
                                            uint32_t tl, uint64_t rowi, float scale, void* dv,
                                            void* dk, volatile int* last_split) {
  constexpr int DQK = C::DQK_, DV = C::DV_, RW = DQK + DV;
  float* part0 = dkdv_part + static_cast<size_t>(tile) * nsp * (C::BN * RW);
  // tcgen05.ld is warp-collective: the loads run on the warp-uniform
  // condition (ready, hf), only the stores on the per-lane kv_ok
  if (ready && hf < 2) {
    float* dst = part0 + (static_cast<size_t>(sp) * C::BN + row) * RW + (hf == 0 ? DQK : 0);
    const uint32_t tcol = hf == 0 ? C::T_DV : C::T_DK;
    const int W = hf == 0 ? DV : DQK;
    for (int c = 0; c < W / 32; ++c) {
      uint32_t a[32];
      tmem_ld32(tl + tcol + c * 32, a);
      tmem_wait_ld();
      if (kv_ok) {
        float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          d4[e] = make_float4(__uint_as_float(a[4 * e]), __uint_as_float(a[4 * e + 1]),
                              __uint_as_float(a[4 * e + 2]), __uint_as_float(a[4 * e + 3]));
      }
    }
  }
  __threadfence();
  named_bar_sync(1, C::NCT);
  if (threadIdx.x == 0) *last_split = ready ? (atomicAdd(dkdv_count + tile, 1) == nsp - 1) : 0;
  named_bar_sync(1, C::NCT);
  if (!*last_split) return;
  __threadfence();
  if (kv_ok && hf < 2) {
    const int W = hf == 0 ? DV : DQK;
    const float mul = hf == 0 ? 1.0f : scale;
    const float* src = part0 + static_cast<size_t>(row) * RW + (hf == 0 ? DQK : 0);
    uint8_t* dst_row = static_cast<uint8_t*>(hf == 0 ? dv : dk) + rowi * W * 2;
    for (int c = 0; c < W / 8; ++c) {
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
      for (int s2 = 0; s2 < nsp; ++s2) {  // split order: the same sum whoever is last
        const float4* s4 = reinterpret_cast<const float4*>(src + static_cast<size_t>(s2) * C::BN * RW + c * 8);
        const float4 u = __ldcg(s4), w = __ldcg(s4 + 1);
        acc[0] += u.x; acc[1] += u.y; acc[2] += u.z; acc[3] += u.w;
        acc[4] += w.x; acc[5] += w.y; acc[6] += w.z; acc[7] += w.w;
      }
      reinterpret_cast<uint4*>(dst_row)[c] =
          make_uint4(pack2<BF16>(acc[0] * mul, acc[1] * mul), pack2<BF16>(acc[2] * mul, acc[3] * mul),
                     pack2<BF16>(acc[4] * mul, acc[5] * mul), pack2<BF16>(acc[6] * mul, acc[7] * mul));
    }
  }
  if (threadIdx.x == 0) dkdv_count[tile] = 0;  // ready for the next call
}

// DROP and BIAS are template parameters (not runtime branches) so the kernel
// without them is compiled alone: at 96 registers a thread (18 warps, five on
// some schedulers) the dropout body's keep bits would otherwise push the
// common path into spilling, and it carries no bias checks. WIN (a local
// window or the bottom-right alignment) likewise: the plain kernel masks only
// the top-left causal diagonal. SPLIT (kv_split > 1) likewise: its epilogue
// keeps the key tile's indices and the partial-row code out of the others.
template <int DQK, int DV, bool BF16, bool DROP, bool BIAS, bool WIN, bool SPLIT>
__global__ void __launch_bounds__(DkdvCfg<DQK, DV>::THREADS, 1)
    sdpa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmdO,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmdK,
                         const __grid_constant__ CUtensorMap tmdV, const BwdParams p) {
  using C = DkdvCfg<DQK, DV>;
  constexpr int BM = C::BM, CW = C::CW, NCT = C::NCT;
  // the bias of each query tile by TMA into shared memory (see DkdvCfg::OFF_BIAS)
  const bool bias_tma = BIAS && C::BIAS_TMA_OK && p.bias_tma != 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
  const uint32_t sQ = smem_u32(smem + C::OFF_Q), sdO = smem_u32(smem + C::OFF_DO);
  float* rowbuf = reinterpret_cast<float*>(smem + C::OFF_ROW);
  const uint32_t sB = smem_u32(smem + C::OFF_BIAS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + AB_COUNT);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  // dK / dV row of the tile's key 0, set at start-up and read by the epilogue
  // (kept out of the registers of the compute loop)
  uint64_t* key_row0 = bars + AB_COUNT + 1;
  Band* band_slot = reinterpret_cast<Band*>(bars + AB_COUNT + 2);  // see lds_band
  volatile int* last_split = reinterpret_cast<volatile int*>(bars + AB_COUNT + 3);
  // key tile index and split of this CTA for a split epilogue, set at start-up
  // (kept out of the registers of the compute loop)
  int* split_tile = reinterpret_cast<int*>(bars + AB_COUNT + 4);
  // the TMA stores of dK and dV: {key row of the tile in its tensor-map
  // plane, plane, staged (1) or written row by row (0)}
  int* out_slot = reinterpret_cast<int*>(bars + AB_COUNT + 5);
  static_assert((AB_COUNT + 7) * 8 <= 256, "barrier region");
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kLoadWarp = NCT / 32, kMmaWarp = NCT / 32 + 1;

  // ---- key tile of this CTA: K/V-head-major (one head's Q / dO stay in L2),
  // then the key tiles with the most query work first, batch fastest (the
  // batches of one head share Bias and dBias rows)
  // (with kv_split > 1, the splits of one key tile next to each other)
  const int n_kt = (p.S_kv + C::BN - 1) / C::BN;
  const int nsp = SPLIT ? p.kv_split : 1;
  const int b = static_cast<int>(blockIdx.x % p.B);
  const int rest = static_cast<int>(blockIdx.x / p.B);
  const int sp = rest % nsp;  // split: query heads [sp * gs, sp * gs + gs) of the group
  const int kt = (rest / nsp) % n_kt, hk = (rest / nsp) / n_kt;  // hk: K/V head
  const SeqSlice sl = seq_slice(p.seqstart_q, p.seqstart_k, p.rows_q, p.rows_k, p.S_q, p.S_kv, p.H,
                                p.H_kv, b);
  const int S_q = sl.len_q, S_kv = sl.len_k;  // this sequence's lengths
  const int zk = sl.zk0 + hk;                 // tensor-map z of the K/V head
  const int grp = p.H / p.H_kv;  // query heads sharing this K/V head
  const int gs = grp / nsp;      // of them, those this CTA sums over
  const int k0 = kt * C::BN;
  // A key tile past the end of a shorter packed sequence has nothing to do
  // (uniform over the CTA; never in batch mode).
  if (k0 >= S_kv) return;
  // query tiles [it0, it0 + n_per) holding a row that sees a key of this tile
  // (WIN: a general window; else top-left, causal when win_right >= 0)
  const Band bd = WIN ? band_of(p.win_left, p.win_right, p.win_br, S_q, S_kv) : plain_band(p.win_right);
  const TileRange qr_t = query_tiles_of_keys(WIN, bd, p.win_right, k0, C::BN, BM, S_q, S_kv);
  const int it0 = qr_t.lo, n_per = qr_t.hi - qr_t.lo + 1;
  // A key tile no query sees: its first split writes the zeros alone.
  if (SPLIT && n_per == 0 && sp != 0) return;
  // One loop over (query head of the split, query tile): iteration i visits
  // query head hk * grp + sp * gs + i / n_per and query tile it0 + i % n_per,
  // so dK and dV sum over the split's heads (the whole group when
  // kv_split = 1) inside tensor memory.
  const int n_it = n_per * gs;
  auto qhead = [&](int i) { return hk * grp + sp * gs + i / n_per; };
  auto qtile0 = [&](int i) { return (it0 + i % n_per) * BM; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < AB_COUNT; ++i)
      mbar_init(bar(i), (i == AB_SFREE || i == AB_P || i == AB_DSL || i == AB_DSH || i == AB_OPS ||
                         i == AB_BE)
                            ? static_cast<uint32_t>(NCT)
                            : 1u);
    *abort_flag = 0u;
    *key_row0 = static_cast<uint64_t>(zk) * p.rows_k + sl.row_k + k0;
    if (SPLIT) {
      split_tile[0] = (hk * n_kt + kt) * p.B + b;
      split_tile[1] = sp;
    }
    if (WIN) *band_slot = bd;
    out_slot[0] = sl.row_k + k0;
    out_slot[1] = zk;
    out_slot[2] = !SPLIT && (p.seqstart_k == nullptr || k0 + C::BN <= S_kv);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    if (bias_tma) tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmdK);
    tma_prefetch_desc(&tmdV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const ErrCtx ec{p.err, abort_flag};

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    int issued = 0, bias_issued = 0;
    if (n_it > 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(AB_KV), C::K_BYTES + C::V_BYTES);
#pragma unroll
        for (int c = 0; c < DQK / 64; ++c)
          tma_load_3d(sK + c * C::BN * 128, &tmK, bar(AB_KV), c * 64, sl.row_k + k0, zk);
#pragma unroll
        for (int c = 0; c < DV / 64; ++c)
          tma_load_3d(sV + c * C::BN * 128, &tmV, bar(AB_KV), c * 64, sl.row_k + k0, zk);
      }
      for (int i = 0; i < n_it; ++i) {
        const int s = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        const int q0 = qtile0(i);
        // the tile's bias first, as soon as the compute threads have read the
        // last tile's (early in that tile), so a whole tile hides its latency
        if (bias_tma) {
          if (!mbar_wait(bar(AB_BE), (i & 1) ^ 1, ec, kSiteBwdLoad, true, true)) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(AB_BF), C::BIAS_BYTES);
            tma_load_3d(sB, &tmB, bar(AB_BF), k0, q0, qhead(i));
          }
          bias_issued = i + 1;
        }
        if (!mbar_wait(bar(AB_QE + s), ph ^ 1, ec, kSiteBwdLoad, true, true)) break;
        const int zq = sl.zq0 + qhead(i);  // tensor-map z of the query head
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(AB_QF + s), C::Q_BYTES + C::STAT_BYTES);
#pragma unroll
          for (int c = 0; c < DQK / 64; ++c)
            tma_load_3d(sQ + s * C::Q_BYTES + c * BM * 128, &tmQ, bar(AB_QF + s), c * 64, sl.row_q + q0, zq);
          bulk_load(smem_u32(rowbuf) + s * C::STAT_BYTES, p.stats + stat_index(zq, p.S_pad, sl.stat_row + q0),
                    C::STAT_BYTES, bar(AB_QF + s));
          mbar_arrive_expect_tx(bar(AB_DOF + s), C::DO_BYTES);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_3d(sdO + s * C::DO_BYTES + c * BM * 128, &tmdO, bar(AB_DOF + s), c * 64, sl.row_q + q0, zq);
        }
        issued = i + 1;
      }
    }
    __syncwarp();
    if (*abort_flag && n_it > 0) {
      mbar_wait(bar(AB_KV), 0, ec, kSiteDrain, false);
      for (int i = 0; i < issued; ++i) {
        const uint32_t ph = (i >> 1) & 1;
        mbar_wait(bar(AB_QF + (i & 1)), ph, ec, kSiteDrain, false);
        mbar_wait(bar(AB_DOF + (i & 1)), ph, ec, kSiteDrain, false);
      }
      // one bias block at a time: only the last one can be in flight
      if (bias_issued > 0) mbar_wait(bar(AB_BF), (bias_issued - 1) & 1, ec, kSiteDrain, false);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16(128, BM, BF16, false, false);
    constexpr uint32_t kIdDV = idesc_f16(128, DV, BF16, false, true);
    constexpr uint32_t kIdDK = idesc_f16(128, DQK, BF16, false, true);
    const uint32_t tS = tbase + C::T_S, tDP = tbase + C::T_DP, tDV = tbase + C::T_DV,
                   tDK = tbase + C::T_DK;
    // Packed io-dtype operand columns of query rows [16kk, 16kk+16) within
    // the dP^T columns: each compute group wrote its CW queries, two per TMEM
    // column, P~^T at the start of the CW columns it read and dS^T CW/2 after.
    auto packed_col = [](int kk) -> uint32_t {
      return static_cast<uint32_t>(((kk * 16) / CW) * CW + ((kk * 16) % CW) / 2);
    };
    // base descriptors, advanced by constant offsets per instruction
    const uint64_t dK0 = sdesc_sw128(sK, 16, 1024), dV0 = sdesc_sw128(sV, 16, 1024);
    const uint64_t dQk0 = sdesc_sw128(sQ, 16, 1024), dOk0 = sdesc_sw128(sdO, 16, 1024);
    const uint64_t dQm0 = sdesc_sw128(sQ, BM * 128, 1024), dOm0 = sdesc_sw128(sdO, BM * 128, 1024);
    auto issue_s = [&](int s) {  // S^T = K Q^T
      const uint64_t dq = desc_adv(dQk0, s * C::Q_BYTES);
#pragma unroll
      for (int kk = 0; kk < DQK / 16; ++kk) {
        const uint64_t bq = desc_adv(dq, (kk >> 2) * (BM * 128) + (kk & 3) * 32);
        if constexpr (C::OPS_IN_TMEM)
          umma_ts_w(tS, tbase + C::T_K + kk * 8, bq, kIdS, kk > 0);
        else
          umma_ss_w(tS, desc_adv(dK0, (kk >> 2) * (C::BN * 128) + (kk & 3) * 32), bq, kIdS, kk > 0);
      }
    };
    auto issue_dp = [&](int s) {  // dP^T = V dO^T
      const uint64_t dob = desc_adv(dOk0, s * C::DO_BYTES);
#pragma unroll
      for (int kk = 0; kk < DV / 16; ++kk) {
        const uint64_t bo = desc_adv(dob, (kk >> 2) * (BM * 128) + (kk & 3) * 32);
        if constexpr (C::OPS_IN_TMEM)
          umma_ts_w(tDP, tbase + C::T_V + kk * 8, bo, kIdS, kk > 0);
        else
          umma_ss_w(tDP, desc_adv(dV0, (kk >> 2) * (C::BN * 128) + (kk & 3) * 32), bo, kIdS, kk > 0);
      }
    };
    // the whole warp runs the issue loop; one elected lane issues (umma_*_w)
    bool ok = n_it > 0;
    if (ok) ok = mbar_wait_w(bar(AB_KV), 0, ec, kSiteBwdMma);
    if (C::OPS_IN_TMEM && ok) ok = mbar_wait_w(bar(AB_OPS), 0, ec, kSiteBwdMma);
    if (ok) ok = mbar_wait_w(bar(AB_QF), 0, ec, kSiteBwdMma);
    if (ok) {
      tc_fence_after();
      issue_s(0);
      umma_commit_w(bar(AB_S));
      ok = mbar_wait_w(bar(AB_DOF), 0, ec, kSiteBwdMma);
    }
    if (ok) {
      tc_fence_after();
      issue_dp(0);
      umma_commit_w(bar(AB_DP));
    }
    for (int i = 0; ok && i < n_it; ++i) {
      const int s = i & 1, s1 = (i + 1) & 1;
      const uint32_t ph1 = ((i + 1) >> 1) & 1;
      if (i + 1 < n_it) {  // S^T(i+1) once the compute warps hold S^T(i) in registers
        if (!(ok = mbar_wait_w(bar(AB_SFREE), i & 1, ec, kSiteBwdMma))) break;
        if (!(ok = mbar_wait_w(bar(AB_QF + s1), ph1, ec, kSiteBwdMma))) break;
        tc_fence_after();
        issue_s(s1);
        umma_commit_w(bar(AB_S));
      }
      if (!(ok = mbar_wait_w(bar(AB_P), i & 1, ec, kSiteBwdMma))) break;
      tc_fence_after();
      {  // dV += P~^T dO_i
        const uint64_t dob = desc_adv(dOm0, s * C::DO_BYTES);
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          umma_ts_w(tDV, tDP + packed_col(kk), desc_adv(dob, kk * 2048), kIdDV, (i > 0 || kk > 0));
      }
      {  // dK += dS^T Q_i, the query steps of each group's first half of dS^T
         // as soon as it is written, the second half after
        const uint64_t dqb = desc_adv(dQm0, s * C::Q_BYTES);
        if (!(ok = mbar_wait_w(bar(AB_DSL), i & 1, ec, kSiteBwdMma))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BM / 16; kk += 2)
          umma_ts_w(tDK, tDP + packed_col(kk) + CW / 2, desc_adv(dqb, kk * 2048), kIdDK, (i > 0 || kk > 0));
        if (!(ok = mbar_wait_w(bar(AB_DSH), i & 1, ec, kSiteBwdMma))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 1; kk < BM / 16; kk += 2)
          umma_ts_w(tDK, tDP + packed_col(kk) + CW / 2, desc_adv(dqb, kk * 2048), kIdDK, 1u);
        umma_commit_w(bar(AB_QE + s));  // Q_i and dO_i are no longer read
      }
      if (i + 1 < n_it) {
        if (!(ok = mbar_wait_w(bar(AB_DOF + s1), ph1, ec, kSiteBwdMma))) break;
        tc_fence_after();
        issue_dp(s1);
        umma_commit_w(bar(AB_DP));
      }
    }
    if (ok) umma_commit_w(bar(AB_DKDV));
    umma_commit_w(bar(AB_DRAIN));
    mbar_wait(bar(AB_DRAIN), 0, ec, kSiteDrain, false);
  } else {
    // ------------------------------------------------------------ compute
    const int t = threadIdx.x;
    const int row = t & 127;  // key row within the tile = TMEM lane
    const int hf = t >> 7;    // query-column group
    const int kv = k0 + row;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool kv_ok = kv < S_kv;
    // This thread's 32 query columns lie in one 64-row block of the statistics
    // slot: 64 values -LSE*log2e (-inf for rows without keys), then 64 -D.
    const int stat_off = ((CW * hf) / 64) * 128 + (CW * hf) % 64;
    bool ok = true;
    if (C::OPS_IN_TMEM && n_it > 0) {  // K and V rows into this thread's TMEM lane
      ok = mbar_wait(bar(AB_KV), 0, ec, kSiteBwdCompute);
      if (ok && hf < 2) {  // the first two groups copy one half of the columns each
        smem_row_to_tmem<DQK / 2>(smem + C::OFF_K, C::BN, row, hf * (DQK / 2),
                                  tbase + lane_off + C::T_K + hf * (DQK / 4));
        smem_row_to_tmem<DV / 2>(smem + C::OFF_V, C::BN, row, hf * (DV / 2),
                                 tbase + lane_off + C::T_V + hf * (DV / 4));
        tmem_wait_st();
      }
      tc_fence_before();
      if (ok) mbar_arrive(bar(AB_OPS));
    }
    {
      const float zk = p.keep_scale;
      for (int i = 0; ok && i < n_it; ++i) {
        const int q0 = qtile0(i);
        const int h = qhead(i);          // query head
        const int bh = b * p.H + h;
        const int qc0 = q0 + CW * hf;  // first query row of this thread's columns
        const float* stat = rowbuf + (i & 1) * (2 * BM) + stat_off;
        const uint32_t nl2_s = smem_u32(stat), dd_s = smem_u32(stat + 64);
        // keep flags of this key for the thread's query columns (bit c: column c)
        uint32_t kw = 0xFFFFFFFFu;
        if constexpr (DROP)
          kw = keep_flags_of_key(p.keep_bits, p.keep_words,
                                 (static_cast<uint64_t>(bh) * p.S_q + qc0) * p.S_kv + k0 + (row & ~31),
                                 p.S_kv, lane, p.drop_threshold, p.seed_lo, p.seed_hi, p.offset_lo,
                                 p.offset_hi);
        auto zf = [&](int c) -> float {  // dropout factor of local column c
          if constexpr (DROP) return ((kw >> c) & 1u) ? zk : 0.f;
          return 1.0f;
        };
        // exponent in the log2 domain: S * scale * log2e - LSE * log2e (+ Bias * log2e)
        float pr[CW];
        if constexpr (BIAS) {
          // Bias of this key and the thread's queries (columns past S_q or a
          // missing key read 0): from the TMA block in shared memory (query
          // row 32 hf + c, key `row`: a warp reads 128 contiguous bytes a
          // column), else loaded from global memory before the wait so its
          // latency overlaps it
          if (bias_tma) {
            if (!(ok = mbar_wait(bar(AB_BF), i & 1, ec, kSiteBwdCompute))) break;
            const float* bcol = reinterpret_cast<const float*>(smem + C::OFF_BIAS) + (CW * hf) * C::BN + row;
#pragma unroll
            for (int c = 0; c < CW; ++c) pr[c] = bcol[c * C::BN];
            mbar_arrive(bar(AB_BE));
          } else {
            const float* bias_col =
                p.bias + (static_cast<size_t>(h) * p.S_q + qc0) * p.S_kv + (kv_ok ? kv : 0);
            const int lim = kv_ok ? min(CW, p.S_q - qc0) : 0;
#pragma unroll
            for (int c = 0; c < CW; ++c)
              pr[c] = (c < lim) ? __ldg(bias_col + static_cast<size_t>(c) * p.S_kv) : 0.f;
          }
        }
        if (!(ok = mbar_wait(bar(AB_S), i & 1, ec, kSiteBwdCompute))) break;
        // S^T(i) was issued after Q_i and the statistics landed; the wait on the
        // same barrier makes the statistics visible to this thread too
        if (!(ok = mbar_wait(bar(AB_QF + (i & 1)), (i >> 1) & 1, ec, kSiteBwdCompute))) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < CW / 32; ++c) {
          uint32_t a0[32];
          tmem_ld32(tbase + C::T_S + lane_off + CW * hf + 32 * c, a0);
          tmem_wait_ld();
          const uint64_t sc2 = f2(p.scale_log2, p.scale_log2);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 n4 = lds128(nl2_s + 16u * (8 * c + e4));
            uint64_t t01 = f2(n4.x, n4.y), t23 = f2(n4.z, n4.w);
            if constexpr (BIAS) {
              const uint64_t l2e = f2(kLog2e, kLog2e);
              const int b0 = 32 * c + 4 * e4;
              t01 = fma2(f2(pr[b0], pr[b0 + 1]), l2e, t01);
              t23 = fma2(f2(pr[b0 + 2], pr[b0 + 3]), l2e, t23);
            }
            const float2 x01 = f2split(fma2(f2(__uint_as_float(a0[4 * e4 + 0]), __uint_as_float(a0[4 * e4 + 1])),
                                            sc2, t01));
            const float2 x23 = f2split(fma2(f2(__uint_as_float(a0[4 * e4 + 2]), __uint_as_float(a0[4 * e4 + 3])),
                                            sc2, t23));
            pr[32 * c + 4 * e4 + 0] = x01.x;
            pr[32 * c + 4 * e4 + 1] = x01.y;
            pr[32 * c + 4 * e4 + 2] = x23.x;
            pr[32 * c + 4 * e4 + 3] = x23.y;
          }
        }
        tc_fence_before();
        mbar_arrive(bar(AB_SFREE));  // S^T(i) is in registers: S^T(i+1) may overwrite it
        // the thread's columns need masking where they cross S_q or an edge of
        // some key's window (a condition uniform over the warp)
        if constexpr (WIN) {
          if (p.alibi != nullptr) {  // ALiBi: -slope |j - i - off|, in the log2 domain
            const float ns = -__ldg(p.alibi + b * p.alibi_stride + h) * kLog2e;
            const float base = static_cast<float>(kv - qc0 - (p.alibi_br ? S_kv - S_q : 0));
#pragma unroll
            for (int c = 0; c < CW; ++c) pr[c] = fmaf(ns, fabsf(base - static_cast<float>(c)), pr[c]);
          }
          const Band wb = lds_band(band_slot);
          if ((qc0 < k0 + C::BN - 1 - wb.hi) || (qc0 + CW - 1 > k0 - wb.lo) || (qc0 + CW > S_q) ||
              !kv_ok) {
            // visible iff the key exists, the query exists and it lies in the key's window
            const int first = kv - wb.hi - qc0;  // visible local columns [first, lim)
            const int lim = kv_ok ? min(CW, min(S_q - 1, kv - wb.lo) + 1 - qc0) : 0;
#pragma unroll
            for (int c = 0; c < CW; ++c)
              if (c < first || c >= lim) pr[c] = SDPA_NEG_INF;
          }
        } else if ((p.win_right >= 0 && qc0 < k0 + C::BN - 1) || (qc0 + CW > S_q) || !kv_ok) {
          // visible iff the key exists, the query exists and (causal) key <= query
          const int first = p.win_right >= 0 ? kv - qc0 : 0;  // first visible local column
          const int lim = kv_ok ? min(CW, S_q - qc0) : 0;
#pragma unroll
          for (int c = 0; c < CW; ++c)
            if (c < first || c >= lim) pr[c] = SDPA_NEG_INF;
        }
#pragma unroll
        for (int c = 0; c < CW; ++c) pr[c] = ex2(pr[c]);
        if (!(ok = mbar_wait(bar(AB_DP), i & 1, ec, kSiteBwdCompute))) break;
        tc_fence_after();
        // The thread's 32 dP^T columns are handled in halves of 16 so that at
        // most half of dP^T is in registers next to P: the lower half is read,
        // P~^T (io dtype, two per column) goes over it at once, and dS of the
        // lower queries is formed; then the upper half is read and dS^T of all
        // 32 queries goes over it. dV reads P~^T from the first 16 columns of
        // each 32, dK reads dS^T from the second 16.
        const uint32_t tcol = tbase + C::T_DP + lane_off + CW * hf;
        float* dbias_col = (BIAS && kv_ok) ? p.dbias + (static_cast<size_t>(h) * p.S_q + qc0) * p.S_kv + kv
                                           : nullptr;
        // dS = P * (dP * Z - D) of local columns [c0, c0 + 16) into 8 packed
        // words, two columns per f32x2 instruction (dd holds -D)
        auto ds_half = [&](const uint32_t (&dp)[16], int c0, uint32_t* out) {
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 nd4 = lds128(dd_s + 16u * (c0 / 4 + e4));
            float ds[4];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int cc = c0 + 4 * e4 + 2 * h2;
              const uint64_t dp2 = f2(__uint_as_float(dp[4 * e4 + 2 * h2]), __uint_as_float(dp[4 * e4 + 2 * h2 + 1]));
              const uint64_t nd2 = h2 ? f2(nd4.z, nd4.w) : f2(nd4.x, nd4.y);
              const uint64_t t2 = fma2(dp2, f2(zf(cc), zf(cc + 1)), nd2);
              const float2 r = f2split(mul2(f2(pr[cc], pr[cc + 1]), t2));
              ds[2 * h2] = r.x;
              ds[2 * h2 + 1] = r.y;
            }
            if (BIAS && dbias_col != nullptr) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int cc = c0 + 4 * e4 + e;
                if (qc0 + cc < p.S_q) atomicAdd(dbias_col + static_cast<size_t>(cc) * p.S_kv, ds[e]);
              }
            }
            out[2 * e4] = pack2<BF16>(ds[0], ds[1]);
            out[2 * e4 + 1] = pack2<BF16>(ds[2], ds[3]);
          }
        };
        uint32_t pk[16];  // dS^T, packed
        {
          uint32_t lo[16], pw[16];
          tmem_ld16(tcol, lo);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) pw[e] = pack2<BF16>(pr[2 * e] * zf(2 * e), pr[2 * e + 1] * zf(2 * e + 1));
          tmem_st16(tcol, pw);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(AB_P));
          ds_half(lo, 0, pk);
        }
        {
          uint32_t hi[16];
          tmem_ld16(tcol + 16, hi);
          tmem_wait_ld();
          // dS^T of the first 16 queries over the upper half just read, so dK
          // can start on them while the second 16 are formed
          tmem_st8(tcol + 16, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(AB_DSL));
          ds_half(hi, 16, pk + 8);
        }
        tmem_st8(tcol + 24, pk + 8);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(AB_DSH));
      }
    }
    // ---- epilogue: dV and dK * scale (zeros for a key tile that no query
    // sees). Whole tiles, and the ragged last tile of an unpacked tensor (the
    // tensor maps drop its rows past the end), are staged in shared memory
    // and stored by TMA; a packed sequence's ragged tile is written row by
    // row, so that it stops at the sequence's end.
    const bool have = n_it > 0;
    const bool ready = have && ok && mbar_wait(bar(AB_DKDV), 0, ec, kSiteBwdCompute);
    if (!SPLIT && out_slot[2]) {
      // [dV | dK] lie side by side in tensor memory: column group hf takes its
      // 32-column chunks hf, hf + NQ, ... into 64-column boxes (dV's first)
      // with the 128-byte swizzle, in the Q / dO stages, idle once dK and dV
      // are complete
      constexpr int NCH = (DV + DQK) / 32;
      static_assert(NCH % C::NQ == 0 && DV % 64 == 0 && DQK % 64 == 0 &&
                        C::STAGES * (C::Q_BYTES + C::DO_BYTES) >= C::BN * (DV + DQK) * 2,
                    "staging of dK and dV");
      const bool write = !have || ready;
      if (ready) tc_fence_after();
      if (write) {
#pragma unroll 1
        for (int j = 0; j < NCH / C::NQ; ++j) {
          const int c = hf + C::NQ * j;
          const float mul = c * 32 < DV ? 1.0f : p.scale;
          const uint32_t dst = sQ + (c >> 1) * (C::BN * 128) + row * 128;
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {  // 16 columns: two 16-byte chunks
            uint32_t a[16];
            if (ready) {
              tmem_ld16(tbase + C::T_DV + lane_off + c * 32 + hc * 16, a);
              tmem_wait_ld();
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) a[e] = 0u;
            }
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              pk[e] = pack2<BF16>(__uint_as_float(a[2 * e]) * mul, __uint_as_float(a[2 * e + 1]) * mul);
#pragma unroll
            for (int e = 0; e < 2; ++e)
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                               dst + ((static_cast<uint32_t>(4 * (c & 1) + 2 * hc + e) ^ (row & 7)) << 4)),
                           "r"(pk[4 * e]), "r"(pk[4 * e + 1]), "r"(pk[4 * e + 2]), "r"(pk[4 * e + 3])
                           : "memory");
          }
        }
      }
      fence_proxy_async_smem();
      // stored only when every compute thread wrote its share
      if (named_bar_and(2, NCT, write) && threadIdx.x == 0) {
        const int r0 = out_slot[0], z = out_slot[1];
#pragma unroll
        for (int bx = 0; bx < DV / 64; ++bx) tma_store_3d(&tmdV, sQ + bx * (C::BN * 128), bx * 64, r0, z);
#pragma unroll
        for (int bx = 0; bx < DQK / 64; ++bx)
          tma_store_3d(&tmdK, sQ + (DV / 64 + bx) * (C::BN * 128), bx * 64, r0, z);
        bulk_commit_group();
        bulk_wait_group_read0();  // the boxes leave shared memory before the CTA does
      }
    } else if (SPLIT && have) {
      if (ready) tc_fence_after();
      split_epilogue<C, BF16>(p.dkdv_part, p.dkdv_count, nsp, split_tile[0], split_tile[1], ready,
                              kv_ok, row, hf, tbase + lane_off, *key_row0 + row, p.scale, p.dv,
                              p.dk, last_split);
    } else if (!have || ready) {
      if (ready) tc_fence_after();
      const size_t rowi = static_cast<size_t>(*key_row0) + (kv_ok ? row : 0);
      auto write_rows = [&](auto width_tag, uint32_t tcol, void* base, float mul) {
        constexpr int W = decltype(width_tag)::value;
        uint8_t* dst_row = static_cast<uint8_t*>(base) + rowi * W * 2;
#pragma unroll
        for (int c = 0; c < W / 32; ++c) {
          uint32_t a[32];
          if (ready) {
            tmem_ld32(tbase + tcol + lane_off + c * 32, a);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack2<BF16>(__uint_as_float(a[2 * e]) * mul, __uint_as_float(a[2 * e + 1]) * mul);
          if (kv_ok) {
            uint4* dst = reinterpret_cast<uint4*>(dst_row + c * 64);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        }
      };
      if (hf == 0)
        write_rows(std::integral_constant<int, DV>{}, C::T_DV, p.dv, 1.0f);
      else if (hf == 1)
        write_rows(std::integral_constant<int, DQK>{}, C::T_DK, p.dk, p.scale);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int DQK, int DV, bool BF16>
cudaError_t launch_bwd_dkdv_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                              const CUtensorMap& dout, const CUtensorMap& bias_map, const CUtensorMap& dk,
                              const CUtensorMap& dv, const BwdParams& p, cudaStream_t st) {
  using C = DkdvCfg<DQK, DV>;
  const bool bias = p.bias != nullptr;
  auto pick = [&](auto win, auto split) {
    constexpr bool W = decltype(win)::value, SP = decltype(split)::value;
    return p.dropout ? (bias ? sdpa_bwd_dkdv_kernel<DQK, DV, BF16, true, true, W, SP>
                             : sdpa_bwd_dkdv_kernel<DQK, DV, BF16, true, false, W, SP>)
                     : (bias ? sdpa_bwd_dkdv_kernel<DQK, DV, BF16, false, true, W, SP>
                             : sdpa_bwd_dkdv_kernel<DQK, DV, BF16, false, false, W, SP>);
  };
  const bool win = p.win_general || p.alibi != nullptr;
  auto kern = p.kv_split > 1 ? (win ? pick(std::true_type{}, std::true_type{})
                                    : pick(std::false_type{}, std::true_type{}))
                             : (win ? pick(std::true_type{}, std::false_type{})
                                    : pick(std::false_type{}, std::false_type{}));
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::SMEM, 0);
  if (e != cudaSuccess) return e;
  const int n_kt = (p.S_kv + C::BN - 1) / C::BN;
  const long long grid = static_cast<long long>(n_kt) * p.B * p.H_kv * p.kv_split;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, st>>>(q, k, v, dout, bias_map, dk, dv, p);
  return cudaGetLastError();
}

}  // namespace sdpa
