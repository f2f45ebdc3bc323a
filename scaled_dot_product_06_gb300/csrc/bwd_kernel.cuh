// Fused attention backward for sm_103a (K/V-stationary), tcgen05 + TMA.
//
// Computes the backward half of the equation block that opens CK tile's
// fmha_bwd_kernel.hpp: dV = P^T dO, dP = dO V^T, dS = P * (dP - D),
// dBias = dS, dK = dS^T Q * scale, dQ = dS K * scale, with dropout entering as
// P~ = P * Z (Z = keep / (1 - p)) in dV and dS = P * (dP * Z - D). P is
// recomputed from the saved logsumexp, P = exp(S * scale + Bias - LSE).
// D = rowsum(dO * O) comes from the preprocess kernel, and dQ is accumulated in
// fp32 and scaled / cast by the convert kernel, as in the CK page's
// FmhaBwdOGradDotOKernel / FmhaBwdConvertQGradKernel split.
//
// One CTA owns 128 key rows of one (b, h) (K_j and V_j stay in shared memory)
// and loops over query tiles of 64 rows. All products are taken transposed so
// the 128 key rows sit in the MMA's M dimension (TMEM lanes):
//   S^T  = K Q_i^T          [128 x 64]   A = K (K-major),  B = Q_i (K-major)
//   dP^T = V dO_i^T         [128 x 64]   A = V (K-major),  B = dO_i (K-major)
//   dV  += P~^T dO_i        [128 x Dv]   A = P~^T in TMEM, B = dO_i (MN-major)
//   dK  += dS^T Q_i         [128 x Dk]   A = dS^T in smem, B = Q_i (MN-major)
//   dQ_i^T = K^T dS^T       [128 x 64]   A = K (MN-major), B = dS^T (MN-major),
//                                        one product per 128-wide slice of Dk
// Roles:
//   warps 0-7  compute, two warpgroups: warp w owns key rows 32*(w%4)..+31
//              (its TMEM lanes) and query columns [32*(w/4), +32) of each
//              tile. Recomputes P^T, writes P~^T into TMEM, forms dS^T, adds
//              it into dBias (fp32 atomics) and stores it to shared memory
//              (io dtype, 128-byte swizzle). Two warps per scheduler hide
//              each other's latencies.
//   warps 8-11 dQ drain: thread t owns TMEM lane t (a column of dQ); stages the
//              dQ_i^T slice in shared memory and reduce-adds it into the fp32
//              dQ accumulator with a TMA tensor reduce.
//   warp 12    TMA producer (K, V once; Q_i and dO_i through a 2-stage ring).
//   warp 13    MMA issuer (one lane).
// Tensor memory (512 columns): S^T [0,64) with P~^T over [0,16) and [32,48)
// (each warpgroup overwrites only columns it has already read), dP^T
// [64,128), dV [128,128+Dv), dK next, dQ^T slices after that.
#pragma once
#include <type_traits>

#include "common.cuh"

namespace sdpa {

template <int DQK, int DV>
struct BwdCfg {
  static constexpr int BN = 128;  // key rows per CTA
  static constexpr int BM = 64;   // query rows per iteration
  static constexpr int STAGES = 2;
  static constexpr int K_BYTES = BN * DQK * 2;
  static constexpr int V_BYTES = BN * DV * 2;
  static constexpr int Q_BYTES = BM * DQK * 2;
  static constexpr int DO_BYTES = BM * DV * 2;
  static constexpr int DS_BYTES = BN * BM * 2;
  static constexpr int NCH = (DQK > 128) ? 2 : 1;      // dQ^T slices of 128 lanes
  static constexpr int DQ_BUFS = (DQK > 128) ? 1 : 2;  // TMEM buffers for dQ^T slices
  static constexpr int DQ_STAGE_BYTES = ((DQK >= 128) ? 2 : 1) * BM * 64 * 4;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + K_BYTES;
  static constexpr int OFF_Q = OFF_V + V_BYTES;
  static constexpr int OFF_DO = OFF_Q + STAGES * Q_BYTES;
  static constexpr int OFF_DS = OFF_DO + STAGES * DO_BYTES;
  static constexpr int OFF_DQ = OFF_DS + DS_BYTES;
  static constexpr int OFF_ROW = OFF_DQ + DQ_STAGE_BYTES;  // 2 x 64 (-LSE log2e), 2 x 64 D
  static constexpr int OFF_BAR = OFF_ROW + 1024;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr int THREADS = 448;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0, T_DP = 64, T_DV = 128, T_DK = 128 + DV, T_DQ = T_DK + DQK;
  static_assert(T_DQ + DQ_BUFS * 64 <= 512, "tensor memory overflow");
  static_assert(SMEM <= 227 * 1024, "shared memory overflow");
  static_assert(DQK % 64 == 0 && DV % 64 == 0 && DV <= 128 && DQK <= 192, "head size");
};

constexpr int kLoadWarp = 12, kMmaWarp = 13;

enum : int { BB_KV = 0, BB_QF, BB_DOF = BB_QF + 2, BB_QE = BB_DOF + 2, BB_S = BB_QE + 2, BB_P,
             BB_DP, BB_DS, BB_DQF, BB_DQE = BB_DQF + 2, BB_DKDV = BB_DQE + 2, BB_DRAIN,
             BB_COUNT };

// Keep bits of key row k for the 32 query rows [row0, row0 + 32) of a tile.
// One Philox block covers four consecutive keys of one query row, i.e. the
// four lanes of a quad (lane 4g + w owns key 4g + w), so lane 4g + w draws the
// blocks of query rows row0 + 4r + w (r < 8) and the quad exchanges the bits.
// Returns m[src]: bit r = keep flag of query row row0 + 4r + src.
// lin_quad is the linear index of (query row row0, first key of the quad).
__device__ __forceinline__ void bwd_keep_bits(uint64_t lin_quad, int S_kv, int lane, uint32_t thr,
                                              uint32_t seed_lo, uint32_t seed_hi, uint32_t off_lo,
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

template <int DQK, int DV, bool BF16>
__global__ void __launch_bounds__(448, 1)
    sdpa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = BwdCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
  const uint32_t sQ = smem_u32(smem + C::OFF_Q), sdO = smem_u32(smem + C::OFF_DO);
  const uint32_t sdS = smem_u32(smem + C::OFF_DS), sDQ = smem_u32(smem + C::OFF_DQ);
  float* rowbuf = reinterpret_cast<float*>(smem + C::OFF_ROW);  // [2][64] nl2, [2][64] D
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + BB_COUNT);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- key tile of this CTA: head-major (one head's Q / dO / dQ stay in L2),
  // then key tiles with the most query work first, batch fastest (the batches
  // of one head share Bias and dBias rows)
  const int n_kt = (p.S_kv + C::BN - 1) / C::BN;
  const int b = static_cast<int>(blockIdx.x % p.B);
  const int rest = static_cast<int>(blockIdx.x / p.B);
  const int kt = rest % n_kt, h = rest / n_kt;
  const int bh = b * p.H + h;
  const int k0 = kt * C::BN;
  const int n_qt = (p.S_q + C::BM - 1) / C::BM;
  const int it0 = p.causal ? min(n_qt, k0 / C::BM) : 0;  // first query tile that sees a key here
  const int n_it = n_qt - it0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < BB_COUNT; ++i) {
      const uint32_t count = (i == BB_P || i == BB_DS) ? 256u
                             : (i == BB_DQE || i == BB_DQE + 1) ? 128u : 1u;
      mbar_init(bar(i), count);
    }
    *abort_flag = 0u;
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
    tma_prefetch_desc(&tmDQ);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const ErrCtx ec{p.err, abort_flag};

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    if (n_it > 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(BB_KV), C::K_BYTES + C::V_BYTES);
#pragma unroll
        for (int c = 0; c < DQK / 64; ++c)
          tma_load_3d(sK + c * C::BN * 128, &tmK, bar(BB_KV), c * 64, k0, bh);
#pragma unroll
        for (int c = 0; c < DV / 64; ++c)
          tma_load_3d(sV + c * C::BN * 128, &tmV, bar(BB_KV), c * 64, k0, bh);
      }
      for (int i = 0; i < n_it; ++i) {
        const int s = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!mbar_wait(bar(BB_QE + s), ph ^ 1, ec, kSiteBwdLoad)) break;
        const int q0 = (it0 + i) * C::BM;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(BB_QF + s), C::Q_BYTES);
#pragma unroll
          for (int c = 0; c < DQK / 64; ++c)
            tma_load_3d(sQ + s * C::Q_BYTES + c * C::BM * 128, &tmQ, bar(BB_QF + s), c * 64, q0, bh);
          mbar_arrive_expect_tx(bar(BB_DOF + s), C::DO_BYTES);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_3d(sdO + s * C::DO_BYTES + c * C::BM * 128, &tmdO, bar(BB_DOF + s), c * 64,
                        q0, bh);
        }
        issued = i + 1;
      }
    }
    __syncwarp();
    if (*abort_flag && n_it > 0) {
      mbar_wait(bar(BB_KV), 0, ec, kSiteDrain, false);
      for (int i = 0; i < issued; ++i) {
        const uint32_t ph = (i >> 1) & 1;
        mbar_wait(bar(BB_QF + (i & 1)), ph, ec, kSiteDrain, false);
        mbar_wait(bar(BB_DOF + (i & 1)), ph, ec, kSiteDrain, false);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16(128, 64, BF16, false, false);
    constexpr uint32_t kIdDV = idesc_f16(128, DV, BF16, false, true);
    constexpr uint32_t kIdDK = idesc_f16(128, DQK, BF16, false, true);
    constexpr uint32_t kIdDQ = idesc_f16(128, 64, BF16, true, true);
    const uint32_t tS = tbase + C::T_S, tDP = tbase + C::T_DP, tDV = tbase + C::T_DV,
                   tDK = tbase + C::T_DK, tDQ = tbase + C::T_DQ;
    bool ok = n_it > 0;
    auto issue_s = [&](int s) {  // S^T = K Q^T
      const uint32_t qb = sQ + s * C::Q_BYTES;
#pragma unroll
      for (int kk = 0; kk < DQK / 16; ++kk)
        umma_ss(tS, sdesc_sw128(sK + (kk >> 2) * (C::BN * 128) + (kk & 3) * 32, 16, 1024),
                sdesc_sw128(qb + (kk >> 2) * (C::BM * 128) + (kk & 3) * 32, 16, 1024), kIdS, kk > 0);
    };
    auto issue_dp = [&](int s) {  // dP^T = V dO^T
      const uint32_t ob = sdO + s * C::DO_BYTES;
#pragma unroll
      for (int kk = 0; kk < DV / 16; ++kk)
        umma_ss(tDP, sdesc_sw128(sV + (kk >> 2) * (C::BN * 128) + (kk & 3) * 32, 16, 1024),
                sdesc_sw128(ob + (kk >> 2) * (C::BM * 128) + (kk & 3) * 32, 16, 1024), kIdS, kk > 0);
    };
    if (ok) ok = mbar_wait(bar(BB_KV), 0, ec, kSiteBwdMma);
    if (ok) ok = mbar_wait(bar(BB_QF), 0, ec, kSiteBwdMma);
    if (ok) {
      tc_fence_after();
      if (lane == 0) {
        issue_s(0);
        umma_commit(bar(BB_S));
      }
      __syncwarp();
      ok = mbar_wait(bar(BB_DOF), 0, ec, kSiteBwdMma);
    }
    if (ok) {
      tc_fence_after();
      if (lane == 0) {
        issue_dp(0);
        umma_commit(bar(BB_DP));
      }
      __syncwarp();
    }
    for (int i = 0; ok && i < n_it; ++i) {
      const int s = i & 1, s1 = (i + 1) & 1;
      const uint32_t ph1 = ((i + 1) >> 1) & 1;
      if (!(ok = mbar_wait(bar(BB_P), i & 1, ec, kSiteBwdMma))) break;
      tc_fence_after();
      if (lane == 0) {  // dV += P~^T dO_i
        const uint32_t ob = sdO + s * C::DO_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          umma_ts(tDV, tS + (kk >> 1) * 32 + (kk & 1) * 8,
                  sdesc_sw128(ob + kk * 2048, C::BM * 128, 1024), kIdDV, (i > 0 || kk > 0));
      }
      __syncwarp();
      if (i + 1 < n_it) {
        if (!(ok = mbar_wait(bar(BB_QF + s1), ph1, ec, kSiteBwdMma))) break;
        tc_fence_after();
        if (lane == 0) {
          issue_s(s1);
          umma_commit(bar(BB_S));
        }
        __syncwarp();
      }
      if (!(ok = mbar_wait(bar(BB_DS), i & 1, ec, kSiteBwdMma))) break;
      tc_fence_after();
      if (lane == 0) {  // dK += dS^T Q_i
        const uint32_t qb = sQ + s * C::Q_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          umma_ss(tDK, sdesc_sw128(sdS + kk * 32, 16, 1024),
                  sdesc_sw128(qb + kk * 2048, C::BM * 128, 1024), kIdDK, (i > 0 || kk > 0));
      }
      __syncwarp();
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) {  // dQ_i^T slice c = K^T dS^T
        const int u = i * C::NCH + c, buf = u % C::DQ_BUFS;
        const uint32_t ph = (u / C::DQ_BUFS) & 1;
        if (!(ok = mbar_wait(bar(BB_DQE + buf), ph ^ 1, ec, kSiteBwdMma))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t ka = sK + (c == 0 ? 0 : 1) * (C::BN * 128);
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)
            umma_ss(tDQ + buf * 64, sdesc_sw128(ka + kk * 2048, C::BN * 128, 1024),
                    sdesc_sw128(sdS + kk * 2048, C::BN * 128, 1024), kIdDQ, kk > 0);
          umma_commit(bar(BB_DQF + buf));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) umma_commit(bar(BB_QE + s));
      __syncwarp();
      if (i + 1 < n_it) {
        if (!(ok = mbar_wait(bar(BB_DOF + s1), ph1, ec, kSiteBwdMma))) break;
        tc_fence_after();
        if (lane == 0) {
          issue_dp(s1);
          umma_commit(bar(BB_DP));
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      if (ok) umma_commit(bar(BB_DKDV));
      umma_commit(bar(BB_DRAIN));
    }
    __syncwarp();
    mbar_wait(bar(BB_DRAIN), 0, ec, kSiteDrain, false);
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ drain
    const int t = threadIdx.x - 256;  // TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float* stage = reinterpret_cast<float*>(smem + C::OFF_DQ);
    bool ok = true;
    for (int i = 0; ok && i < n_it; ++i) {
      const int q0 = (it0 + i) * C::BM;
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) {
        const int u = i * C::NCH + c, buf = u % C::DQ_BUFS;
        const uint32_t ph = (u / C::DQ_BUFS) & 1;
        if (!(ok = mbar_wait(bar(BB_DQF + buf), ph, ec, kSiteBwdDq))) break;
        tc_fence_after();
        uint32_t v0[32], v1[32];
        tmem_ld32(tbase + C::T_DQ + buf * 64 + lane_off, v0);
        tmem_ld32(tbase + C::T_DQ + buf * 64 + lane_off + 32, v1);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(BB_DQE + buf));
        // lane t holds column d = d_base + t of dQ_i for the 64 query rows
        const int d_base = (c == 0) ? 0 : 64;
        const int d = d_base + t;
        const bool valid = d < DQK && (c == 0 || t >= 64);
        const int gb_first = (c == 0) ? 0 : 2;  // first 64-wide box written by this slice
        if (t == 0) bulk_wait_group_read0();
        named_bar_sync(1, 128);
        if (valid) {
          float* col = stage + (d / 64 - gb_first) * (C::BM * 64) + (d & 63);
#pragma unroll
          for (int q = 0; q < 32; ++q) col[q * 64] = __uint_as_float(v0[q]);
#pragma unroll
          for (int q = 0; q < 32; ++q) col[(q + 32) * 64] = __uint_as_float(v1[q]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (t == 0) {
          const int gb_last = (c == 0) ? min(DQK, 128) / 64 - 1 : DQK / 64 - 1;
          for (int gb = gb_first; gb <= gb_last; ++gb)
            tma_reduce_add_3d(&tmDQ, sDQ + (gb - gb_first) * (C::BM * 64 * 4), gb * 64, q0, bh);
          bulk_commit_group();
        }
      }
    }
    if (t == 0) bulk_wait_group0();
  } else {
    // ------------------------------------------------------------ compute
    // Two warpgroups: warp w owns key rows 32*(w%4) .. +31 (its TMEM lanes)
    // and query columns [32*hf, 32*hf + 32) of each tile, hf = w / 4.
    const int t = threadIdx.x;
    const int row = t & 127;           // key row within the tile = TMEM lane
    const int hf = t >> 7;             // query-column half
    const int kv = k0 + row;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool kv_ok = kv < p.S_kv;
    float* nl2_buf = rowbuf;        // [2][64]  -LSE * log2(e) (-inf for rows without keys)
    float* d_buf = rowbuf + 128;    // [2][64]  D
    uint8_t* ds_row = smem + C::OFF_DS + row * 128;
    // Row statistics of query tile i: threads 0-63 read -LSE*log2e, threads
    // 64-127 read D. Tile i+1's values are fetched during tile i.
    auto fetch_row_stat = [&](int i) -> float {
      const int qr = (it0 + i) * C::BM + (t & 63);
      const size_t idx = static_cast<size_t>(bh) * p.S_q + qr;
      if (t < 64) {
        const float L = (qr < p.S_q) ? p.lse[idx] : SDPA_NEG_INF;
        return (L == SDPA_NEG_INF) ? SDPA_NEG_INF : -L * kLog2e;
      }
      return (qr < p.S_q) ? p.delta[idx] : 0.f;
    };
    auto store_row_stat = [&](int i, float v) {
      if (t < 128) rowbuf[(t < 64 ? 0 : 128) + (i & 1) * 64 + (t & 63)] = v;
    };
    bool ok = true;
    auto body = [&](auto drop_tag) {
      constexpr bool DROP = decltype(drop_tag)::value;
      const float zk = p.keep_scale;
      if (n_it > 0) store_row_stat(0, t < 128 ? fetch_row_stat(0) : 0.f);
      for (int i = 0; ok && i < n_it; ++i) {
        const int q0 = (it0 + i) * C::BM;
        const int qc0 = q0 + 32 * hf;  // first query row of this thread's columns
        named_bar_sync(2, 256);  // tile i's statistics are in shared memory
        const float4* nl2 = reinterpret_cast<const float4*>(nl2_buf + (i & 1) * 64 + 32 * hf);
        const float4* dd = reinterpret_cast<const float4*>(d_buf + (i & 1) * 64 + 32 * hf);
        const float next_stat = (t < 128 && i + 1 < n_it) ? fetch_row_stat(i + 1) : 0.f;
        uint32_t km[4] = {0xFFu, 0xFFu, 0xFFu, 0xFFu};
        if constexpr (DROP)
          bwd_keep_bits((static_cast<uint64_t>(bh) * p.S_q + qc0) * p.S_kv + k0 + (row & ~3), p.S_kv, lane,
                        p.drop_threshold, p.seed_lo, p.seed_hi, p.offset_lo, p.offset_hi, km);
        auto zf = [&](int c) -> float {
          if constexpr (DROP) return ((km[c & 3] >> (c >> 2)) & 1u) ? zk : 0.f;
          return 1.0f;
        };
        if (!(ok = mbar_wait(bar(BB_S), i & 1, ec, kSiteBwdCompute))) break;
        tc_fence_after();
        float pr[32];
        {
          uint32_t a0[32];
          tmem_ld32(tbase + C::T_S + lane_off + 32 * hf, a0);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) pr[c] = __uint_as_float(a0[c]);
        }
        const bool need_mask = (p.causal && qc0 < k0 + C::BN - 1) || (qc0 + 32 > p.S_q) ||
                               !kv_ok || (k0 + C::BN > p.S_kv);
        const float* bias_col =
            (p.bias != nullptr && kv_ok)
                ? p.bias + (static_cast<size_t>(h) * p.S_q + qc0) * p.S_kv + kv
                : nullptr;
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 n4 = nl2[c4];
          const float nv[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 4 * c4 + e;
            float x = fmaf(pr[c], p.scale_log2, nv[e]);
            if (bias_col != nullptr && qc0 + c < p.S_q)
              x = fmaf(__ldg(bias_col + static_cast<size_t>(c) * p.S_kv), kLog2e, x);
            if (need_mask && (!kv_ok || qc0 + c >= p.S_q || (p.causal && kv > qc0 + c)))
              x = SDPA_NEG_INF;
            pr[c] = ex2(x);
          }
        }
        {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = pack2<BF16>(pr[2 * c] * zf(2 * c), pr[2 * c + 1] * zf(2 * c + 1));
          tmem_st16(tbase + C::T_S + lane_off + 32 * hf, pk);  // P~^T over [32hf, 32hf+16)
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(bar(BB_P));
        if (!(ok = mbar_wait(bar(BB_DP), i & 1, ec, kSiteBwdCompute))) break;
        tc_fence_after();
        float dp[32];
        {
          uint32_t a0[32];
          tmem_ld32(tbase + C::T_DP + lane_off + 32 * hf, a0);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) dp[c] = __uint_as_float(a0[c]);
        }
        float* dbias_col =
            (p.dbias != nullptr && kv_ok)
                ? p.dbias + (static_cast<size_t>(h) * p.S_q + qc0) * p.S_kv + kv
                : nullptr;
#pragma unroll
        for (int chh = 0; chh < 4; ++chh) {
          float ds[8];
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const float4 d4 = dd[chh * 2 + g];
            const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = chh * 8 + g * 4 + e;
              ds[g * 4 + e] = pr[c] * (DROP ? fmaf(dp[c], zf(c), -dv4[e]) : dp[c] - dv4[e]);
            }
          }
          if (dbias_col != nullptr) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (qc0 + chh * 8 + e < p.S_q)
                atomicAdd(dbias_col + static_cast<size_t>(chh * 8 + e) * p.S_kv, ds[e]);
          }
          const int ch = 4 * hf + chh;  // 16-byte chunk = query columns 8ch .. 8ch+7
          *reinterpret_cast<uint4*>(ds_row + ((ch ^ (row & 7)) << 4)) =
              make_uint4(pack2<BF16>(ds[0], ds[1]), pack2<BF16>(ds[2], ds[3]),
                         pack2<BF16>(ds[4], ds[5]), pack2<BF16>(ds[6], ds[7]));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(BB_DS));
        if (i + 1 < n_it) store_row_stat(i + 1, next_stat);
      }
    };
    if (p.dropout)
      body(std::true_type{});
    else
      body(std::false_type{});
    // ---- epilogue: warps 0-3 write dV, warps 4-7 write dK * scale (zeros for
    // a key tile that no query sees)
    const bool have = n_it > 0;
    bool ready = have && ok && mbar_wait(bar(BB_DKDV), 0, ec, kSiteBwdCompute);
    if (have && !ready) ok = false;
    if (ok) {
      if (ready) tc_fence_after();
      const size_t rowi = static_cast<size_t>(bh) * p.S_kv + (kv_ok ? kv : 0);
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
      else
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
cudaError_t launch_bwd_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                         const CUtensorMap& dout, const CUtensorMap& dq, const BwdParams& p,
                         cudaStream_t st) {
  using C = BwdCfg<DQK, DV>;
  auto kern = sdpa_bwd_kernel<DQK, DV, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_kt = (p.S_kv + C::BN - 1) / C::BN;
  const long long grid = static_cast<long long>(n_kt) * p.B * p.H;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, st>>>(q, k, v, dout, dq, p);
  return cudaGetLastError();
}

}  // namespace sdpa
