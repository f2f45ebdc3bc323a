// Attention backward in one key/value-stationary kernel: dK, dV, dBias and an
// fp32 dQ accumulator (sm_103a).
//
// Computes the dV .. dQ lines of the equation block that opens CK tile's
// fmha_bwd_kernel.hpp (dV = P^T dO, dP = dO V^T, dS = P * (dP - D),
// dBias = dS, dK = dS^T Q * scale, dQ = dS K * scale) the way that page's
// FmhaBwdDQDKDVKernel and oneDNN sdpa micro.cpp's backward kernel do: the CTA
// owning a key tile forms every product of its (query tile, key tile) pairs
// once, and adds its share of dQ into an fp32 accumulator in global memory
// (CK's dq_acc with atomic adds; oneDNN's f32 dQ scratchpad). A convert pass
// (aux.cu) then scales the accumulator and rounds it to the io dtype. Against
// the deterministic split (bwd_dkdv_kernel.cuh + bwd_dq_kernel.cuh) this
// forms 5 products per tile pair instead of 7, at the price of 4 * BM * d_qk
// bytes of fp32 reductions per pair and a dQ that depends on the order the
// reductions reach L2.
//
// One CTA owns 128 key rows of one (b, h) (K_j and V_j stay resident) and
// loops over query tiles of 128 rows. Products per tile i:
//   S^T  = K Q_i^T    [128 x 128]  A = K (smem or TMEM),  B = Q_i (K-major)
//   dP^T = V dO_i^T   [128 x 128]  A = V (smem or TMEM),  B = dO_i (K-major)
//   dV  += P~^T dO_i  [128 x Dv]   A = P~^T (TMEM),       B = dO_i (MN-major)
//   dQ_i = dS K       [128 x Dk]   A = dS (smem, MN-major), B = K (MN-major)
//   dK  += dS^T Q_i   [128 x Dk]   A = dS^T (smem, K-major), B = Q_i (MN-major)
// dS^T is written once, as an io-dtype [128 keys x 128 queries] tile in
// shared memory with the 128-byte swizzle: read K-major it is dK's A operand
// (keys in M), read MN-major the same bytes are dS, dQ's A operand (queries in
// M). dQ_i goes to global memory as fp32 vector reductions
// (red.global.add.v4.f32) into a tiled accumulator layout in which each warp
// instruction covers 512 contiguous bytes.
//
// Roles (24 warps):
//   compute   warps 0-15: warp w owns key rows 32*(w%4)..+31 (TMEM lanes) and
//             query columns [32*hf, 32*hf + 32), hf = w/4. Per tile: P^T from
//             S^T; then, reading dP^T over the same columns, P~^T (io dtype)
//             over the first 16 of them and dS into the shared dS^T tile (and
//             dBias).
//   producer  warp 16: TMA for K, V once; Q_i (with its row statistics) and
//             dO_i through a 2-stage ring.
//   MMA       warp 17: issue order per tile: dV(i) once P~^T(i) is written;
//             once dS(i) is written, S^T(i+1) (over the columns dP^T(i) and
//             P~^T(i) held) and dP^T(i+1) as soon as the compute warps hold
//             S^T(i+1) in registers (the two share their TMEM columns), then
//             dK(i). dQ(i) goes in the moment its columns are free (dQ(i-1)
//             read out) once dS(i) is written: the issuer checks for that
//             while it waits for anything else, since the reductions after
//             each dQ set the pace. The compute warps wait for dK(i) and
//             dQ(i) to have read the shared dS^T tile before writing dS(i+1)
//             into it.
//   drain     warps 20-23: warp 20 + r owns TMEM lanes 32 r..+31, the query
//             rows of dQ_i: it reads them out 16 columns at a time and adds
//             them into the accumulator with fp32 vector reductions. An SM
//             injects such reductions at ~22 bytes a cycle, so a tile's
//             4 * 128 * Dk bytes take about as long as its five products; in
//             warps of their own the reductions' queueing stalls none of the
//             compute warps, and with dQ_i in columns of its own they overlap
//             the next tile's products.
//   (warps 18, 19 idle.) Registers: launched at 80 a thread, the compute
//   warpgroups raise theirs to 96 (setmaxnreg), the producer/MMA warpgroup
//   drops to 56 (its base descriptors rebuilt at each use through
//   opaque_u64 instead of all held in registers) and the drain warpgroup to
//   40; in the split instances 72 and 24, with the descriptors held.
// Tensor memory (512 columns): S^T / dP^T / P~^T [0,128), dQ_i [128,128+Dk),
// dV [128+Dk, 128+Dk+Dv), dK after it, then K and V (two elements per column)
// when they fit (d = 64). At the end the compute warps stage dV and dK in the
// Q / dO stages, idle by then, and one thread stores them by TMA.
#pragma once
#include <type_traits>

#include "bwd_dkdv_kernel.cuh"

namespace sdpa {

template <int DQK, int DV>
struct FusedCfg {
  static constexpr int DQK_ = DQK, DV_ = DV;
  static constexpr int BN = 128;  // key rows per CTA
  static constexpr int BM = 128;  // query rows per tile
  static constexpr int CW = 32;   // query columns per compute thread
  static constexpr int NCT = 512; // compute threads (four warpgroups)
  static constexpr int NDT = 128; // drain threads (one warpgroup)
  static constexpr int K_BYTES = BN * DQK * 2;
  static constexpr int V_BYTES = BN * DV * 2;
  static constexpr int Q_BYTES = BM * DQK * 2;
  static constexpr int DO_BYTES = BM * DV * 2;
  static constexpr int DS_BYTES = BN * BM * 2;
  static constexpr int STAT_BYTES = 2 * BM * 4;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + K_BYTES;
  static constexpr int OFF_Q = OFF_V + V_BYTES;
  static constexpr int OFF_DO = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_DS = OFF_DO + 2 * DO_BYTES;
  static constexpr int OFF_ROW = OFF_DS + DS_BYTES;
  static constexpr int OFF_BAR = OFF_ROW + 2 * STAT_BYTES;
  // No alignment slack: the dynamic shared memory is declared 1024-aligned
  // and the kernel checks it (at d = 128 the layout leaves 768 bytes of the
  // 227 KB a CTA can have).
  static constexpr int SMEM = OFF_BAR + 256;
  static constexpr int THREADS = 768;  // 16 compute warps, producer, MMA, 2 idle, 4 drain
  static constexpr int kLoadWarp = 16, kMmaWarp = 17, kDrainWarp0 = 20;
  // registers: launched at REG_LAUNCH; compute warpgroups raise theirs, the
  // producer/MMA and drain warpgroups lower theirs, within the launch total
  static constexpr int REG_LAUNCH = 80, REG_COMPUTE = 96, REG_ISSUE = 56, REG_DRAIN = 40;
  // the split instances (grouped K/V heads over several CTAs per key tile)
  // keep plain descriptors and the issuer at 72: measured, the opaque form
  // there took the grouped workloads' kernel from 4.50 to 4.61 ms
  static constexpr int REG_ISSUE_SPLIT = 72, REG_DRAIN_SPLIT = 24;
  static_assert(4 * 128 * REG_COMPUTE + 128 * REG_ISSUE + 128 * REG_DRAIN == THREADS * REG_LAUNCH,
                "register split");
  static_assert(4 * 128 * REG_COMPUTE + 128 * REG_ISSUE_SPLIT + 128 * REG_DRAIN_SPLIT == THREADS * REG_LAUNCH,
                "register split");
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0, T_DQ = 128, T_DV = 128 + DQK, T_DK = T_DV + DV;
  static constexpr uint32_t T_K = T_DK + DQK, T_V = T_K + DQK / 2;
  static constexpr bool OPS_IN_TMEM = T_V + DV / 2 <= 512;
  static_assert(T_DK + DQK <= 512, "tensor memory overflow");
  static_assert(DQK % 16 == 0 && DQK <= 128, "dQ drained 16 columns at a time");
  static_assert(SMEM <= 232448, "shared memory overflow");
};

enum : int { FB_KV = 0, FB_QF, FB_DOF = FB_QF + 2, FB_QE = FB_DOF + 2, FB_S = FB_QE + 2, FB_SFREE,
             FB_DP, FB_P, FB_DS, FB_DQ, FB_DQFREE, FB_DSFREE, FB_DKDV, FB_DRAIN, FB_OPS, FB_COUNT };

// fp32 vector reduction into global memory (sm_90 and later).
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// Index (in floats) of columns [4 cg, 4 cg + 4) of accumulator row R of
// tensor-map z in the tiled dQ accumulator layout: per z, per 128-row tile,
// per group of 4 columns, the tile's 128 rows of 16 bytes each. A warp whose
// lanes hold 32 consecutive rows of one column group thus reduces into 512
// contiguous bytes.
__host__ __device__ __forceinline__ size_t dq_acc_index(size_t z, int dq_tiles, int dqk, int R, int cg) {
  return ((z * static_cast<size_t>(dq_tiles) + static_cast<size_t>(R >> 7)) * static_cast<size_t>(dqk / 4) +
          static_cast<size_t>(cg)) * 512 + static_cast<size_t>(R & 127) * 4;
}

template <int DQK, int DV, bool BF16, bool DROP, bool BIAS, bool WIN, bool SPLIT>
__global__ void __launch_bounds__(FusedCfg<DQK, DV>::THREADS, 1)
    sdpa_bwd_fused_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmdO,
                          const __grid_constant__ CUtensorMap tmdK,
                          const __grid_constant__ CUtensorMap tmdV, const BwdParams p) {
  using C = FusedCfg<DQK, DV>;
  constexpr int BM = C::BM, CW = C::CW, NCT = C::NCT;
  extern __shared__ __align__(1024) uint8_t fused_smem[];
  uint8_t* smem = fused_smem;
  // The layout has no room to realign: give up (error word) if the dynamic
  // shared memory does not start on a 1024-byte boundary.
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, kSiteSmemAlign);
    return;
  }
  const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
  const uint32_t sQ = smem_u32(smem + C::OFF_Q), sdO = smem_u32(smem + C::OFF_DO);
  const uint32_t sdS = smem_u32(smem + C::OFF_DS);
  float* rowbuf = reinterpret_cast<float*>(smem + C::OFF_ROW);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + FB_COUNT);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  uint64_t* key_row0 = bars + FB_COUNT + 1;  // dK / dV row of the tile's key 0
  Band* band_slot = reinterpret_cast<Band*>(bars + FB_COUNT + 2);  // see lds_band
  volatile int* last_split = reinterpret_cast<volatile int*>(bars + FB_COUNT + 3);
  int* split_tile = reinterpret_cast<int*>(bars + FB_COUNT + 4);
  // the TMA stores of dK and dV: {key row of the tile in its tensor-map
  // plane, plane, staged (1) or written row by row (0)}
  int* out_slot = reinterpret_cast<int*>(bars + FB_COUNT + 5);
  static_assert((FB_COUNT + 7) * 8 <= 256, "barrier region");
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kLoadWarp = C::kLoadWarp, kMmaWarp = C::kMmaWarp, kDrainWarp0 = C::kDrainWarp0;

  // ---- key tile of this CTA (the order of the dK/dV kernel): K/V-head-major,
  // key tiles with the most query work first, batch fastest
  const int n_kt = (p.S_kv + C::BN - 1) / C::BN;
  const int nsp = SPLIT ? p.kv_split : 1;
  const int b = static_cast<int>(blockIdx.x % p.B);
  const int rest = static_cast<int>(blockIdx.x / p.B);
  const int sp = rest % nsp;
  const int kt = (rest / nsp) % n_kt, hk = (rest / nsp) / n_kt;
  const SeqSlice sl = seq_slice(p.seqstart_q, p.seqstart_k, p.rows_q, p.rows_k, p.S_q, p.S_kv, p.H,
                                p.H_kv, b);
  const int S_q = sl.len_q, S_kv = sl.len_k;
  const int zk = sl.zk0 + hk;
  const int grp = p.H / p.H_kv;
  const int gs = grp / nsp;
  const int k0 = kt * C::BN;
  if (k0 >= S_kv) return;
  const Band bd = WIN ? band_of(p.win_left, p.win_right, p.win_br, S_q, S_kv) : plain_band(p.win_right);
  const TileRange qr_t = query_tiles_of_keys(WIN, bd, p.win_right, k0, C::BN, BM, S_q, S_kv);
  const int it0 = qr_t.lo, n_per = qr_t.hi - qr_t.lo + 1;
  if (SPLIT && n_per == 0 && sp != 0) return;
  const int n_it = n_per * gs;
  auto qhead = [&](int i) { return hk * grp + sp * gs + i / n_per; };
  auto qtile0 = [&](int i) { return (it0 + i % n_per) * BM; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < FB_COUNT; ++i)
      mbar_init(bar(i), (i == FB_SFREE || i == FB_P || i == FB_DS || i == FB_OPS)
                            ? static_cast<uint32_t>(NCT)
                            : (i == FB_DQFREE ? static_cast<uint32_t>(C::NDT) : 1u));
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
    tma_prefetch_desc(&tmdK);
    tma_prefetch_desc(&tmdV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const ErrCtx ec{p.err, abort_flag};

  if (warp >= kDrainWarp0) {
    // ------------------------------------------------------------ drain
    // (each warpgroup's register change directly precedes its own code, so
    // the compiler holds each role to its own budget)
    setmaxnreg_dec<SPLIT ? C::REG_DRAIN_SPLIT : C::REG_DRAIN>();
    // lanes of warp kDrainWarp0 + r: query rows 32 r .. 32 r + 31 of dQ_i
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    for (int i = 0; i < n_it; ++i) {
      if (!mbar_wait(bar(FB_DQ), i & 1, ec, kSiteBwdCompute)) break;
      tc_fence_after();
      const int qr = qtile0(i) + (warp & 3) * 32 + lane;  // local query row
      const bool live = qr < S_q;
      const int zr = sl.row_q + (live ? qr : 0);  // tensor row of the query
      if (!SPLIT && p.dq_direct) {  // the row's only contribution: dQ = scale * dQ_i, written out
        uint8_t* drow = static_cast<uint8_t*>(p.dq) +
                        (static_cast<size_t>(sl.zq0 + qhead(i)) * p.rows_q + zr) * DQK * 2;
#pragma unroll 1
        for (int c = 0; c < DQK / 16; ++c) {
          uint32_t a[16];
          tmem_ld16(tbase + C::T_DQ + lane_off + 16 * c, a);
          tmem_wait_ld();
          if (c == DQK / 16 - 1) {
            tc_fence_before();
            mbar_arrive(bar(FB_DQFREE));
          }
          if (live) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = pack2<BF16>(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
            uint4* dst = reinterpret_cast<uint4*>(drow + c * 32);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
        continue;
      }
      float* dst = p.dq_acc + dq_acc_index(static_cast<size_t>(sl.zq0 + qhead(i)), p.dq_tiles, DQK, zr, 0);
#pragma unroll 1
      for (int c = 0; c < DQK / 16; ++c) {
        uint32_t a[16];
        tmem_ld16(tbase + C::T_DQ + lane_off + 16 * c, a);
        tmem_wait_ld();
        if (c == DQK / 16 - 1) {  // dQ_i is out of tensor memory: dQ_{i+1} may come
          tc_fence_before();
          mbar_arrive(bar(FB_DQFREE));
        }
        if (live) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            red_add_v4(dst + static_cast<size_t>(4 * c + e) * 512, __uint_as_float(a[4 * e]),
                       __uint_as_float(a[4 * e + 1]), __uint_as_float(a[4 * e + 2]),
                       __uint_as_float(a[4 * e + 3]));
        }
      }
    }
  } else if (warp >= NCT / 32) {
    setmaxnreg_dec<SPLIT ? C::REG_ISSUE_SPLIT : C::REG_ISSUE>();
    if (warp == kLoadWarp) {
      // ---------------------------------------------------------- producer
      int issued = 0;
      if (n_it > 0) {
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(FB_KV), C::K_BYTES + C::V_BYTES);
#pragma unroll
          for (int c = 0; c < DQK / 64; ++c)
            tma_load_3d(sK + c * C::BN * 128, &tmK, bar(FB_KV), c * 64, sl.row_k + k0, zk);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_3d(sV + c * C::BN * 128, &tmV, bar(FB_KV), c * 64, sl.row_k + k0, zk);
        }
        for (int i = 0; i < n_it; ++i) {
          const int s = i & 1;
          const uint32_t ph = (i >> 1) & 1;
          if (!mbar_wait(bar(FB_QE + s), ph ^ 1, ec, kSiteBwdLoad, true, true)) break;
          const int q0 = qtile0(i);
          const int zq = sl.zq0 + qhead(i);
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(FB_QF + s), C::Q_BYTES + C::STAT_BYTES);
#pragma unroll
            for (int c = 0; c < DQK / 64; ++c)
              tma_load_3d(sQ + s * C::Q_BYTES + c * BM * 128, &tmQ, bar(FB_QF + s), c * 64, sl.row_q + q0, zq);
            bulk_load(smem_u32(rowbuf) + s * C::STAT_BYTES, p.stats + stat_index(zq, p.S_pad, sl.stat_row + q0),
                      C::STAT_BYTES, bar(FB_QF + s));
            mbar_arrive_expect_tx(bar(FB_DOF + s), C::DO_BYTES);
#pragma unroll
            for (int c = 0; c < DV / 64; ++c)
              tma_load_3d(sdO + s * C::DO_BYTES + c * BM * 128, &tmdO, bar(FB_DOF + s), c * 64, sl.row_q + q0, zq);
          }
          issued = i + 1;
        }
      }
      __syncwarp();
      if (*abort_flag && n_it > 0) {
        mbar_wait(bar(FB_KV), 0, ec, kSiteDrain, false);
        for (int i = 0; i < issued; ++i) {
          const uint32_t ph = (i >> 1) & 1;
          mbar_wait(bar(FB_QF + (i & 1)), ph, ec, kSiteDrain, false);
          mbar_wait(bar(FB_DOF + (i & 1)), ph, ec, kSiteDrain, false);
        }
      }
    } else if (warp == kMmaWarp) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdS = idesc_f16(128, BM, BF16, false, false);
      constexpr uint32_t kIdDV = idesc_f16(128, DV, BF16, false, true);
      constexpr uint32_t kIdDK = idesc_f16(128, DQK, BF16, false, true);
      constexpr uint32_t kIdDQ = idesc_f16(BM, DQK, BF16, true, true);
      const uint32_t tS = tbase + C::T_S, tDQ = tbase + C::T_DQ, tDV = tbase + C::T_DV,
                     tDK = tbase + C::T_DK;
      // P~^T of query rows [16kk, 16kk+16): group kk/2 wrote its 32 queries
      // into the first 16 of its 32 S^T / dP^T columns, two per column
      auto packed_col = [](int kk) -> uint32_t {
        return static_cast<uint32_t>((kk >> 1) * CW + (kk & 1) * 8);
      };
      const uint64_t dK0 = sdesc_sw128(sK, 16, 1024), dV0 = sdesc_sw128(sV, 16, 1024);
      const uint64_t dQk0 = sdesc_sw128(sQ, 16, 1024), dOk0 = sdesc_sw128(sdO, 16, 1024);
      const uint64_t dQm0 = sdesc_sw128(sQ, BM * 128, 1024), dOm0 = sdesc_sw128(sdO, BM * 128, 1024);
      // the dS^T tile: K-major (keys in M, 64-query boxes of 128 rows) for dK,
      // MN-major (queries in M, 16 KB between the two 64-query boxes) for dQ
      const uint64_t dSk0 = sdesc_sw128(sdS, 16, 1024), dSm0 = sdesc_sw128(sdS, C::BN * 128, 1024);
      const uint64_t dKm0 = sdesc_sw128(sK, C::BN * 128, 1024);  // K_j with d in N
      // the loop-invariant base descriptors (K, V, the dS^T tile) pass through
      // opaque_u64 at each product, so the issuer adds the constant offsets
      // where it issues instead of holding every descriptor in registers
      // (not in the split instances, see REG_ISSUE_SPLIT)
      auto opq = [](uint64_t d) { return SPLIT ? d : opaque_u64(d); };
      auto issue_s = [&](int s) {  // S^T = K Q^T
        const uint64_t dq = desc_adv(dQk0, s * C::Q_BYTES);
        const uint64_t dKb = opq(dK0);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint64_t bq = desc_adv(dq, (kk >> 2) * (BM * 128) + (kk & 3) * 32);
          if constexpr (C::OPS_IN_TMEM)
            umma_ts_w(tS, tbase + C::T_K + kk * 8, bq, kIdS, kk > 0);
          else
            umma_ss_w(tS, desc_adv(dKb, (kk >> 2) * (C::BN * 128) + (kk & 3) * 32), bq, kIdS, kk > 0);
        }
      };
      auto issue_dp = [&](int s) {  // dP^T = V dO^T, into the S^T columns
        const uint64_t dob = desc_adv(dOk0, s * C::DO_BYTES);
        const uint64_t dVb = opq(dV0);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint64_t bo = desc_adv(dob, (kk >> 2) * (BM * 128) + (kk & 3) * 32);
          if constexpr (C::OPS_IN_TMEM)
            umma_ts_w(tS, tbase + C::T_V + kk * 8, bo, kIdS, kk > 0);
          else
            umma_ss_w(tS, desc_adv(dVb, (kk >> 2) * (C::BN * 128) + (kk & 3) * 32), bo, kIdS, kk > 0);
        }
      };
      bool ok = n_it > 0;
      if (ok) ok = mbar_wait_w(bar(FB_KV), 0, ec, kSiteBwdMma);
      if (C::OPS_IN_TMEM && ok) ok = mbar_wait_w(bar(FB_OPS), 0, ec, kSiteBwdMma);
      if (ok) ok = mbar_wait_w(bar(FB_QF), 0, ec, kSiteBwdMma);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        umma_commit_w(bar(FB_S));
        ok = mbar_wait_w(bar(FB_SFREE), 0, ec, kSiteBwdMma);
      }
      if (ok) ok = mbar_wait_w(bar(FB_DOF), 0, ec, kSiteBwdMma);
      if (ok) {
        tc_fence_after();
        issue_dp(0);
        umma_commit_w(bar(FB_DP));
      }
      for (int i = 0; ok && i < n_it; ++i) {
        const int s = i & 1, s1 = (i + 1) & 1;
        const uint32_t ph1 = ((i + 1) >> 1) & 1;
        // dQ_i = dS K goes in as soon as dS(i) is written and the drain warps
        // have read dQ_{i-1} out of its columns: the reductions that follow it
        // set the pace, so once dS(i) is written the issuer offers dQ_i
        // whenever it would otherwise wait (try_dq(false) issues it only if
        // the columns are free; try_dq(true) waits for them).
        bool dq_in = false;
        auto try_dq = [&](bool block) -> bool {
          if (i > 0) {
            if (block) {
              if (!mbar_wait_w(bar(FB_DQFREE), (i - 1) & 1, ec, kSiteBwdMma)) return false;
            } else if (!__all_sync(0xffffffffu, mbar_try_wait(bar(FB_DQFREE), (i - 1) & 1))) {
              return true;  // not yet: nothing issued
            }
          }
          tc_fence_after();
          const uint64_t dSm = opq(dSm0), dKm = opq(dKm0);
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)
            umma_ss_w(tDQ, desc_adv(dSm, kk * 2048), desc_adv(dKm, kk * 2048), kIdDQ, kk > 0);
          umma_commit_w(bar(FB_DQ));
          dq_in = true;
          return true;
        };
        // bounded wait on phase ph of barrier b that offers dQ_i meanwhile
        auto wait_offering = [&](int b, uint32_t ph) -> bool {
          const uint64_t t0 = globaltimer_ns();
          for (uint32_t it = 0;; ++it) {
            if (__all_sync(0xffffffffu, mbar_try_wait(bar(b), ph))) return true;
            if (!dq_in) try_dq(false);
            if ((it & 63u) == 63u) {
              if (__any_sync(0xffffffffu, *ec.abort != 0u)) return false;
              if (globaltimer_ns() - t0 > ec.limit_ns) {
                if (elect_one_sync()) {
                  atomicOr(ec.err_word, kSiteBwdMma);
                  *ec.abort = 1u;
                }
                return false;
              }
            }
          }
        };
        if (!(ok = mbar_wait_w(bar(FB_P), i & 1, ec, kSiteBwdMma))) break;
        tc_fence_after();
        {  // dV += P~^T dO_i
          const uint64_t dob = desc_adv(dOm0, s * C::DO_BYTES);
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            umma_ts_w(tDV, tS + packed_col(kk), desc_adv(dob, kk * 2048), kIdDV, (i > 0 || kk > 0));
        }
        if (!(ok = mbar_wait_w(bar(FB_DS), i & 1, ec, kSiteBwdMma))) break;
        try_dq(false);
        if (i + 1 < n_it) {
          // S^T(i+1) over the columns P~^T(i) and dP^T(i) held: the pipe reads
          // P~^T(i) for dV(i) first, and the compute warps have read dP^T(i)
          if (!(ok = wait_offering(FB_QF + s1, ph1))) break;
          tc_fence_after();
          issue_s(s1);
          umma_commit_w(bar(FB_S));
          // dP^T(i+1) once the compute warps hold S^T(i+1) in registers
          if (!(ok = wait_offering(FB_SFREE, (i + 1) & 1))) break;
          if (!(ok = wait_offering(FB_DOF + s1, ph1))) break;
          tc_fence_after();
          issue_dp(s1);
          umma_commit_w(bar(FB_DP));
        }
        tc_fence_after();
        {  // dK += dS^T Q_i
          const uint64_t dqb = desc_adv(dQm0, s * C::Q_BYTES);
          const uint64_t dSk = opq(dSk0);
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            umma_ss_w(tDK, desc_adv(dSk, (kk >> 2) * (C::BN * 128) + (kk & 3) * 32),
                      desc_adv(dqb, kk * 2048), kIdDK, (i > 0 || kk > 0));
        }
        umma_commit_w(bar(FB_QE + s));  // Q_i and dO_i are no longer read
        if (!dq_in && !(ok = try_dq(true))) break;
        umma_commit_w(bar(FB_DSFREE));  // dK(i) and dQ(i) have read the dS^T tile
      }
      if (ok) umma_commit_w(bar(FB_DKDV));
      umma_commit_w(bar(FB_DRAIN));
      mbar_wait(bar(FB_DRAIN), 0, ec, kSiteDrain, false);
    }
  } else {
    // ------------------------------------------------------------ compute
    setmaxnreg_inc<C::REG_COMPUTE>();
    const int t = threadIdx.x;
    const int row = t & 127;  // key row within the tile = TMEM lane
    const int hf = t >> 7;    // query-column group
    const int kv = k0 + row;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool kv_ok = kv < S_kv;
    const int stat_off = ((CW * hf) / 64) * 128 + (CW * hf) % 64;
    // this thread's 64 bytes of each dS^T row: box hf/2, 16-byte chunks
    // 4 (hf & 1) .. +3, swizzled by the row
    const uint32_t ds_row = sdS + (hf >> 1) * (C::BN * 128) + row * 128;
    const int ds_c0 = 4 * (hf & 1);
    bool ok = true;
    if (C::OPS_IN_TMEM && n_it > 0) {  // K and V rows into this thread's TMEM lane
      ok = mbar_wait(bar(FB_KV), 0, ec, kSiteBwdCompute);
      if (ok && hf < 2) {
        smem_row_to_tmem<DQK / 2>(smem + C::OFF_K, C::BN, row, hf * (DQK / 2),
                                  tbase + lane_off + C::T_K + hf * (DQK / 4));
        smem_row_to_tmem<DV / 2>(smem + C::OFF_V, C::BN, row, hf * (DV / 2),
                                 tbase + lane_off + C::T_V + hf * (DV / 4));
        tmem_wait_st();
      }
      tc_fence_before();
      if (ok) mbar_arrive(bar(FB_OPS));
    }
    {
      const float zk = p.keep_scale;
      for (int i = 0; ok && i < n_it; ++i) {
        const int q0 = qtile0(i);
        const int h = qhead(i);
        const int bh = b * p.H + h;
        const int qc0 = q0 + CW * hf;
        const float* stat = rowbuf + (i & 1) * (2 * BM) + stat_off;
        const uint32_t nl2_s = smem_u32(stat), dd_s = smem_u32(stat + 64);
        // keep flags of this key for the thread's query columns (bit c: column
        // c), read from the keep bits drawn beforehand or drawn here
        uint32_t kw = 0xFFFFFFFFu;
        if constexpr (DROP)
          kw = keep_flags_of_key(p.keep_bits, p.keep_words,
                                 (static_cast<uint64_t>(bh) * p.S_q + qc0) * p.S_kv + k0 + (row & ~31),
                                 p.S_kv, lane, p.drop_threshold, p.seed_lo, p.seed_hi, p.offset_lo,
                                 p.offset_hi);
        auto zf = [&](int c) -> float {
          if constexpr (DROP) return ((kw >> c) & 1u) ? zk : 0.f;
          return 1.0f;
        };
        float pr[CW];
        if constexpr (BIAS) {
          const float* bias_col = p.bias + (static_cast<size_t>(h) * p.S_q + qc0) * p.S_kv + (kv_ok ? kv : 0);
          const int lim = kv_ok ? min(CW, p.S_q - qc0) : 0;
#pragma unroll
          for (int c = 0; c < CW; ++c) pr[c] = (c < lim) ? __ldg(bias_col + static_cast<size_t>(c) * p.S_kv) : 0.f;
        }
        if (!(ok = mbar_wait(bar(FB_S), i & 1, ec, kSiteBwdCompute))) break;
        if (!(ok = mbar_wait(bar(FB_QF + (i & 1)), (i >> 1) & 1, ec, kSiteBwdCompute))) break;
        tc_fence_after();
        const uint32_t tcs = tbase + C::T_S + lane_off + CW * hf;
        {
          uint32_t a0[32];
          tmem_ld32(tcs, a0);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(FB_SFREE));  // S^T(i) is in registers: dP^T(i) may take its columns
          const uint64_t sc2 = f2(p.scale_log2, p.scale_log2);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 n4 = lds128(nl2_s + 16u * e4);
            uint64_t t01 = f2(n4.x, n4.y), t23 = f2(n4.z, n4.w);
            if constexpr (BIAS) {
              const uint64_t l2e = f2(kLog2e, kLog2e);
              t01 = fma2(f2(pr[4 * e4], pr[4 * e4 + 1]), l2e, t01);
              t23 = fma2(f2(pr[4 * e4 + 2], pr[4 * e4 + 3]), l2e, t23);
            }
            const float2 x01 = f2split(fma2(f2(__uint_as_float(a0[4 * e4 + 0]), __uint_as_float(a0[4 * e4 + 1])),
                                            sc2, t01));
            const float2 x23 = f2split(fma2(f2(__uint_as_float(a0[4 * e4 + 2]), __uint_as_float(a0[4 * e4 + 3])),
                                            sc2, t23));
            pr[4 * e4 + 0] = x01.x;
            pr[4 * e4 + 1] = x01.y;
            pr[4 * e4 + 2] = x23.x;
            pr[4 * e4 + 3] = x23.y;
          }
        }
        if constexpr (WIN) {
          if (p.alibi != nullptr) {
            const float ns = -__ldg(p.alibi + b * p.alibi_stride + h) * kLog2e;
            const float base = static_cast<float>(kv - qc0 - (p.alibi_br ? S_kv - S_q : 0));
#pragma unroll
            for (int c = 0; c < CW; ++c) pr[c] = fmaf(ns, fabsf(base - static_cast<float>(c)), pr[c]);
          }
          const Band wb = lds_band(band_slot);
          if ((qc0 < k0 + C::BN - 1 - wb.hi) || (qc0 + CW - 1 > k0 - wb.lo) || (qc0 + CW > S_q) ||
              !kv_ok) {
            const int first = kv - wb.hi - qc0;
            const int lim = kv_ok ? min(CW, min(S_q - 1, kv - wb.lo) + 1 - qc0) : 0;
#pragma unroll
            for (int c = 0; c < CW; ++c)
              if (c < first || c >= lim) pr[c] = SDPA_NEG_INF;
          }
        } else if ((p.win_right >= 0 && qc0 < k0 + C::BN - 1) || (qc0 + CW > S_q) || !kv_ok) {
          const int first = p.win_right >= 0 ? kv - qc0 : 0;
          const int lim = kv_ok ? min(CW, S_q - qc0) : 0;
#pragma unroll
          for (int c = 0; c < CW; ++c)
            if (c < first || c >= lim) pr[c] = SDPA_NEG_INF;
        }
#pragma unroll
        for (int c = 0; c < CW; ++c) pr[c] = ex2(pr[c]);
        if (!(ok = mbar_wait(bar(FB_DP), i & 1, ec, kSiteBwdCompute))) break;
        tc_fence_after();
        float* dbias_col = (BIAS && kv_ok) ? p.dbias + (static_cast<size_t>(h) * p.S_q + qc0) * p.S_kv + kv
                                           : nullptr;
        // dS = P * (dP * Z - D) of local columns [c0, c0 + 16), packed into
        // the thread's dS^T row chunks c0/8 and c0/8 + 1 (dd holds -D)
        auto ds_half = [&](const uint32_t (&dp)[16], int c0) {
          uint32_t out[8];
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
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int chunk = ds_c0 + c0 / 8 + q;
            const uint32_t addr = ds_row + ((chunk ^ (row & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(out[4 * q]),
                         "r"(out[4 * q + 1]), "r"(out[4 * q + 2]), "r"(out[4 * q + 3])
                         : "memory");
          }
        };
        {  // the lower 16 dP^T columns, then P~^T (io dtype, two per column) over them
          uint32_t lo[16], pw[16];
          tmem_ld16(tcs, lo);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) pw[e] = pack2<BF16>(pr[2 * e] * zf(2 * e), pr[2 * e + 1] * zf(2 * e + 1));
          tmem_st16(tcs, pw);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(FB_P));
          // dQ(i-1) and dK(i-1), issued after dP^T(i), must have read the
          // dS^T tile before dS(i) goes into it
          if (i > 0 && !(ok = mbar_wait(bar(FB_DSFREE), (i - 1) & 1, ec, kSiteBwdCompute))) break;
          ds_half(lo, 0);
        }
        {
          uint32_t hi[16];
          tmem_ld16(tcs + 16, hi);
          tmem_wait_ld();
          ds_half(hi, 16);
        }
        // the dS^T tile is read by the tensor core (async proxy); the dP^T
        // columns are free for S^T(i+1)
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(FB_DS));
      }
    }
    // ---- epilogue: dV and dK * scale (zeros for a key tile that no query
    // sees). Whole tiles, and the ragged last tile of an unpacked tensor (the
    // tensor maps drop its rows past the end), are staged in shared memory
    // and stored by TMA; a packed sequence's ragged tile is written row by
    // row, so that it stops at the sequence's end.
    const bool have = n_it > 0;
    const bool ready = have && ok && mbar_wait(bar(FB_DKDV), 0, ec, kSiteBwdCompute);
    if (!SPLIT && out_slot[2]) {
      // [dV | dK] lie side by side in tensor memory: column group hf takes its
      // 32-column chunks hf, hf + 4, ... into 64-column boxes (dV's first) with
      // the 128-byte swizzle, in the Q / dO stages, idle once dK and dV are
      // complete
      constexpr int NCH = (DV + DQK) / 32;
      static_assert(NCH % 4 == 0 && 2 * (C::Q_BYTES + C::DO_BYTES) >= C::BN * (DV + DQK) * 2,
                    "staging of dK and dV");
      const bool write = !have || ready;
      if (ready) tc_fence_after();
      if (write) {
#pragma unroll 1
        for (int j = 0; j < NCH / 4; ++j) {
          const int c = hf + 4 * j;
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
      if (named_bar_and(1, NCT, write) && threadIdx.x == 0) {
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
cudaError_t launch_bwd_fused_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& dout, const CUtensorMap& dk, const CUtensorMap& dv,
                               const BwdParams& p, cudaStream_t st) {
  using C = FusedCfg<DQK, DV>;
  const bool bias = p.bias != nullptr;
  auto pick = [&](auto win, auto split) {
    constexpr bool W = decltype(win)::value, SP = decltype(split)::value;
    return p.dropout ? (bias ? sdpa_bwd_fused_kernel<DQK, DV, BF16, true, true, W, SP>
                             : sdpa_bwd_fused_kernel<DQK, DV, BF16, true, false, W, SP>)
                     : (bias ? sdpa_bwd_fused_kernel<DQK, DV, BF16, false, true, W, SP>
                             : sdpa_bwd_fused_kernel<DQK, DV, BF16, false, false, W, SP>);
  };
  const bool win = p.win_general || p.alibi != nullptr;
  auto kern = p.kv_split > 1 ? (win ? pick(std::true_type{}, std::true_type{})
                                    : pick(std::false_type{}, std::true_type{}))
                             : (win ? pick(std::true_type{}, std::false_type{})
                                    : pick(std::false_type{}, std::false_type{}));
  // The warpgroups' setmaxnreg shares add up to THREADS x REG_LAUNCH; had the
  // compiler given the kernel another launch register count, the compute
  // warpgroups' increase could never be granted, so refuse to launch then.
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::SMEM, C::REG_LAUNCH);
  if (e != cudaSuccess) return e;
  const int n_kt = (p.S_kv + C::BN - 1) / C::BN;
  const long long grid = static_cast<long long>(n_kt) * p.B * p.H_kv * p.kv_split;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, st>>>(q, k, v, dout, dk, dv, p);
  return cudaGetLastError();
}

}  // namespace sdpa
