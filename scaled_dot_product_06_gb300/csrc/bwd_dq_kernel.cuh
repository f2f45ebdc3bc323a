// Attention backward, query-stationary half: dQ (sm_103a).
//
// Computes the dQ line of the equation block that opens CK tile's
// fmha_bwd_kernel.hpp, dQ = dS K * scale with dS = P * (dP * Z - D),
// dP = dO V^T and P = exp(S * scale + Bias - LSE) recomputed from the saved
// logsumexp. Each CTA owns 128 query rows of one (b, h) and sums over the key
// tiles in a fixed order inside tensor memory, so dQ needs no cross-CTA
// accumulation and is bitwise reproducible. This trades the two extra
// products per tile (S and dP are also formed by the key/value-stationary
// kernel) for the fp32 atomics, accumulator buffer and convert kernel a fused
// backward needs.
//
// Per key tile j of 128 rows (keys in the N dimension, queries in the TMEM
// lanes):
//   S   = Q K_j^T     [128 x 128]  A = Q (smem, K-major),  B = K_j (K-major)
//   dP  = dO V_j^T    [128 x 128]  A = dO (smem, K-major), B = V_j (K-major)
//   dQ += dS K_j      [128 x Dk]   A = dS (TMEM),          B = K_j (MN-major)
// Roles (four compute warpgroups, a producer warp and an MMA warp):
//   compute    warp w owns query rows 32*(w%4)..+31 (its TMEM lanes) and key
//              columns [32*(w/4), +32) of each tile, so each scheduler runs
//              four compute warps whose latencies hide one another: P from S,
//              then dS (io dtype) written over the second half of the dP
//              columns it has read.
//   producer   TMA for Q, dO once and K_j, V_j through a ring.
//   MMA        the whole warp runs the issue loop, one elected lane issues.
// Tensor memory (512 columns): S [0,128), dP [128,256), dQ [256, 256+Dk),
// then Q and dO (two elements per column) when they fit (d_qk <= 128): the S
// and dP products then take A from TMEM and read only K_j / V_j from shared
// memory, which keeps the tensor core within the shared-memory read rate.
// At the end the compute warps stage dQ in Q's shared memory, idle by then,
// and one thread stores it by TMA.
#pragma once
#include <type_traits>

#include "common.cuh"

namespace sdpa {

template <int DQK, int DV>
struct DqCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int NQ = 4;             // compute warpgroups
  static constexpr int CW = BN / NQ;       // key columns per compute thread
  static constexpr int NCT = 128 * NQ;     // compute threads
  static constexpr int STAGES = (DQK <= 128) ? 2 : 1;
  static constexpr int Q_BYTES = BM * DQK * 2;
  static constexpr int DO_BYTES = BM * DV * 2;
  static constexpr int K_BYTES = BN * DQK * 2;
  static constexpr int V_BYTES = BN * DV * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + Q_BYTES;
  static constexpr int OFF_K = OFF_DO + DO_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * K_BYTES;
  // The bias tile of a key tile ([BM query rows][BN keys] fp32, four
  // 32-key column blocks of BM 128-byte rows, 128-byte swizzle), loaded by
  // TMA one tile ahead, where it fits beside the operands (d_qk = 64 and
  // 192; at d_qk = 128 the two K/V stages leave no room and the bias is read
  // from global memory).
  static constexpr int BIAS_BYTES = BM * BN * 4;
  static constexpr int OFF_BIAS = OFF_V + STAGES * V_BYTES;
  static constexpr bool BIAS_TMA_OK = OFF_BIAS + BIAS_BYTES + 256 + 1024 <= 227 * 1024;
  static constexpr int OFF_BAR = OFF_BIAS + (BIAS_TMA_OK ? BIAS_BYTES : 0);
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr int THREADS = NCT + 64;  // + producer warp + MMA warp
  static constexpr uint32_t TMEM_COLS = 512;
  // Two dP buffers where they fit next to the dQ accumulator and the Q / dO
  // operands (d_qk = 64): dS(j) stays in its dP buffer until dQ(j) has read
  // it, so with one buffer dP(j+1) queues behind dQ(j) and dQ(j) + dP(j+1) +
  // the dS step sit on the per-tile critical path; with two, dP(j+1) is
  // formed while tile j's softmax runs. At d_qk = 128 the second buffer would
  // cost the TMEM copies of Q and dO; measured on GB300, the S and dP products
  // then reading both operands from shared memory (and the K ring held longer)
  // cost more than the shorter chain saves (dQ 2.35 -> 2.94 ms at b1 h32
  // s16384 causal), so one buffer stays there.
  static constexpr int DPB = (128 + 2 * 128 + DQK + DQK / 2 + DV / 2 <= 512) ? 2 : 1;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 128 + 128 * DPB;
  // Q and dO, the operands every tile reuses, live in TMEM when they also fit,
  // so the S and dP products read only K_j / V_j from shared memory.
  static constexpr bool OPS_IN_TMEM = T_DQ + DQK + DQK / 2 + DV / 2 <= 512;
  static constexpr uint32_t T_Q = T_DQ + DQK, T_DO = T_Q + DQK / 2;
  static_assert(T_DQ + DQK <= 512, "tensor memory overflow");
  static_assert(DPB == 1 || STAGES == 2, "two dP buffers issue dP(j+1) before dQ(j)");
  static_assert(SMEM <= 227 * 1024, "shared memory overflow");
  static_assert(CW == 32, "one 32-column TMEM load per compute thread and tile");
};

enum : int { QB_Q = 0, QB_KF, QB_KE = QB_KF + 2, QB_VF = QB_KE + 2, QB_VE = QB_VF + 2,
             QB_S = QB_VE + 2, QB_SFREE, QB_DP, QB_DSL = QB_DP + 2, QB_DSH = QB_DSL + 2,
             QB_DONE = QB_DSH + 2, QB_DRAIN, QB_OPS, QB_BF, QB_BE, QB_COUNT };

// DROP, BIAS and WIN (a local window or the bottom-right alignment) are
// template parameters so the kernel without them is compiled alone and stays
// within 96 registers a thread without spilling.
template <int DQK, int DV, bool BF16, bool DROP, bool BIAS, bool WIN>
__global__ void __launch_bounds__(DqCfg<DQK, DV>::THREADS, 1)
    sdpa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmdQ, const BwdParams p) {
  using C = DqCfg<DQK, DV>;
  constexpr int BM = C::BM, BN = C::BN, CW = C::CW, ST = C::STAGES, NCT = C::NCT;
  // the bias of each key tile by TMA into shared memory (see DqCfg::OFF_BIAS)
  const bool bias_tma = BIAS && C::BIAS_TMA_OK && p.bias_tma != 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sQ = smem_u32(smem + C::OFF_Q), sdO = smem_u32(smem + C::OFF_DO);
  const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
  const uint32_t sB = smem_u32(smem + C::OFF_BIAS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + QB_COUNT);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  Band* band_slot = reinterpret_cast<Band*>(bars + QB_COUNT + 1);  // see lds_band
  // the TMA store of dQ: {query row of the tile in its tensor-map plane,
  // plane, staged (1) or written row by row (0)}
  int* out_slot = reinterpret_cast<int*>(bars + QB_COUNT + 2);
  static_assert((QB_COUNT + 4) * 8 <= 256, "barrier region");
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kLoadWarp = NCT / 32, kMmaWarp = NCT / 32 + 1;

  // ---- query tile of this CTA (order: query_tile_order, one head at a time:
  // measured at b1 h32 s16384 causal, dQ 2.08 ms one head per group, 2.13 ms
  // eight, 2.29 ms with every head in flight)
  const int n_qt = (p.S_q + BM - 1) / BM;
  const QueryTile qtile = query_tile_order(static_cast<int>(blockIdx.x), p.B, p.H, n_qt, 1);
  const int b = qtile.b, h = qtile.h, qt = qtile.qt;
  const int bh = b * p.H + h;  // (batch entry or sequence, head): the dropout index
  const SeqSlice sl = seq_slice(p.seqstart_q, p.seqstart_k, p.rows_q, p.rows_k, p.S_q, p.S_kv, p.H,
                                p.H_kv, b);
  const int S_q = sl.len_q, S_kv = sl.len_k;  // this sequence's lengths
  const int zq = sl.zq0 + h;                  // tensor-map z of the query head
  const int zk = sl.zk0 + h / (p.H / p.H_kv);  // and of its K/V head
  const int q0 = qt * BM;
  // key tiles [khi - n_kv + 1, khi] holding a key some row of the tile sees
  // (WIN: a general window; else top-left, causal when win_right >= 0)
  const Band bd = WIN ? band_of(p.win_left, p.win_right, p.win_br, S_q, S_kv) : plain_band(p.win_right);
  const TileRange kr = WIN ? key_tiles_of_rows(bd, q0, BM, BN, S_q, S_kv)
                           : key_tiles_plain(p.win_right >= 0, q0, BM, BN, S_kv);
  const int khi = kr.hi, n_kv = kr.hi - kr.lo + 1;
  // Uniform over the CTA: a tile past the end of a shorter packed sequence has
  // nothing to do, and rows that see no key (a sequence without keys, or the
  // window) have dQ = 0.
  if (q0 >= S_q) return;
  if (n_kv == 0) {
    const int row = q0 + static_cast<int>(threadIdx.x);
    if (threadIdx.x < BM && row < S_q) {
      const size_t ri = static_cast<size_t>(zq) * p.rows_q + sl.row_q + row;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.dq) + ri * DQK * 2);
#pragma unroll
      for (int v = 0; v < DQK / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  // Iteration j visits key tile n_kv - 1 - j: the CTAs of one head, resident
  // together, then start on different tiles (their own diagonal) instead of
  // all requesting tile 0 from L2 at once.

  if (threadIdx.x == 0) {
    for (int i = 0; i < QB_COUNT; ++i)
      mbar_init(bar(i), (i == QB_SFREE || i == QB_DSL || i == QB_DSL + 1 || i == QB_DSH ||
                         i == QB_DSH + 1 || i == QB_OPS || i == QB_BE)
                            ? static_cast<uint32_t>(NCT)
                            : 1u);
    *abort_flag = 0u;
    if (WIN) *band_slot = bd;
    out_slot[0] = sl.row_q + q0;
    out_slot[1] = zq;
    out_slot[2] = p.seqstart_q == nullptr || q0 + BM <= S_q;
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
    tma_prefetch_desc(&tmdQ);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const ErrCtx ec{p.err, abort_flag};

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    int issued = 0, bias_issued = 0;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(QB_Q), C::Q_BYTES + C::DO_BYTES);
#pragma unroll
      for (int c = 0; c < DQK / 64; ++c) tma_load_3d(sQ + c * BM * 128, &tmQ, bar(QB_Q), c * 64, sl.row_q + q0, zq);
#pragma unroll
      for (int c = 0; c < DV / 64; ++c) tma_load_3d(sdO + c * BM * 128, &tmdO, bar(QB_Q), c * 64, sl.row_q + q0, zq);
    }
    for (int j = 0; j < n_kv; ++j) {
      const int s = j % ST;
      const uint32_t ph = (j / ST) & 1;
      // the tile's bias first, as soon as the compute threads have read the
      // last tile's (early in that tile), so a whole tile hides its latency
      if (bias_tma) {
        if (!mbar_wait(bar(QB_BE), (j & 1) ^ 1, ec, kSiteBwdLoad, true, true)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(QB_BF), C::BIAS_BYTES);
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
            tma_load_3d(sB + c * (BM * 128), &tmB, bar(QB_BF), (khi - j) * BN + 32 * c, q0, h);
        }
        bias_issued = j + 1;
      }
      if (!mbar_wait(bar(QB_KE + s), ph ^ 1, ec, kSiteBwdLoad, true, true)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(QB_KF + s), C::K_BYTES);
#pragma unroll
        for (int c = 0; c < DQK / 64; ++c)
          tma_load_3d(sK + s * C::K_BYTES + c * BN * 128, &tmK, bar(QB_KF + s), c * 64, sl.row_k + (khi - j) * BN, zk);
      }
      if (!mbar_wait(bar(QB_VE + s), ph ^ 1, ec, kSiteBwdLoad, true, true)) {
        issued = 2 * j + 1;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(QB_VF + s), C::V_BYTES);
#pragma unroll
        for (int c = 0; c < DV / 64; ++c)
          tma_load_3d(sV + s * C::V_BYTES + c * BN * 128, &tmV, bar(QB_VF + s), c * 64, sl.row_k + (khi - j) * BN, zk);
      }
      issued = 2 * j + 2;
    }
    __syncwarp();
    if (*abort_flag) {
      mbar_wait(bar(QB_Q), 0, ec, kSiteDrain, false);
      for (int i = 0; i < issued; ++i) {
        const int j = i >> 1, s = j % ST;
        mbar_wait(bar(((i & 1) ? QB_VF : QB_KF) + s), (j / ST) & 1, ec, kSiteDrain, false);
      }
      // one bias tile at a time: only the last one can be in flight
      if (bias_issued > 0) mbar_wait(bar(QB_BF), (bias_issued - 1) & 1, ec, kSiteDrain, false);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16(128, BN, BF16, false, false);
    constexpr uint32_t kIdDQ = idesc_f16(128, DQK, BF16, false, true);
    const uint32_t tS = tbase + C::T_S, tDQ = tbase + C::T_DQ;
    // base descriptors, advanced by constant offsets per instruction
    const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024), dO0 = sdesc_sw128(sdO, 16, 1024);
    const uint64_t dK0 = sdesc_sw128(sK, 16, 1024), dV0 = sdesc_sw128(sV, 16, 1024);
    const uint64_t dKm0 = sdesc_sw128(sK, BN * 128, 1024);
    auto issue_s = [&](int j) {  // S = Q K_j^T
      const uint64_t dk = desc_adv(dK0, (j % ST) * C::K_BYTES);
#pragma unroll
      for (int kk = 0; kk < DQK / 16; ++kk) {
        const uint64_t bk = desc_adv(dk, (kk >> 2) * (BN * 128) + (kk & 3) * 32);
        if constexpr (C::OPS_IN_TMEM)
          umma_ts_w(tS, tbase + C::T_Q + kk * 8, bk, kIdS, kk > 0);
        else
          umma_ss_w(tS, desc_adv(dQ0, (kk >> 2) * (BM * 128) + (kk & 3) * 32), bk, kIdS, kk > 0);
      }
    };
    auto issue_dp = [&](int j) {  // dP = dO V_j^T into buffer j % DPB
      const uint32_t tDP = tbase + C::T_DP + 128 * (j % C::DPB);
      const uint64_t dv = desc_adv(dV0, (j % ST) * C::V_BYTES);
#pragma unroll
      for (int kk = 0; kk < DV / 16; ++kk) {
        const uint64_t bv = desc_adv(dv, (kk >> 2) * (BN * 128) + (kk & 3) * 32);
        if constexpr (C::OPS_IN_TMEM)
          umma_ts_w(tDP, tbase + C::T_DO + kk * 8, bv, kIdS, kk > 0);
        else
          umma_ss_w(tDP, desc_adv(dO0, (kk >> 2) * (BM * 128) + (kk & 3) * 32), bv, kIdS, kk > 0);
      }
    };
    // dS of keys [16kk, 16kk+16), packed two per column in the second half of
    // the CW dP columns each compute group read
    auto ds_col = [](int kk) -> uint32_t {
      return static_cast<uint32_t>(((kk * 16) / CW) * CW + CW / 2 + ((kk * 16) % CW) / 2);
    };
    // dQ += dS K_j, dS in dP buffer j % DPB: the key steps of each group's
    // first half of dS (even kk) as soon as it is written, then the second
    auto issue_dq = [&](int j, int half) {
      const uint32_t tDP = tbase + C::T_DP + 128 * (j % C::DPB);
      const uint64_t dk = desc_adv(dKm0, (j % ST) * C::K_BYTES);
#pragma unroll
      for (int kk = half; kk < BN / 16; kk += 2)
        umma_ts_w(tDQ, tDP + ds_col(kk), desc_adv(dk, kk * 2048), kIdDQ, (j > 0 || kk > 0));
    };
    // wait for one half of dS(j), then issue its dQ steps
    auto ds_then_dq = [&](int j, int half) {
      const int b = j % C::DPB;
      if (!mbar_wait_w(bar((half ? QB_DSH : QB_DSL) + b), (j / C::DPB) & 1, ec, kSiteBwdMma)) return false;
      tc_fence_after();
      issue_dq(j, half);
      return true;
    };
    auto wait_kv = [&](int which, int j) {
      return mbar_wait_w(bar(which + j % ST), (j / ST) & 1, ec, kSiteBwdMma);
    };
    // the whole warp runs the issue loop; one elected lane issues (umma_*_w)
    bool ok = mbar_wait_w(bar(QB_Q), 0, ec, kSiteBwdMma) && wait_kv(QB_KF, 0);
    if (C::OPS_IN_TMEM && ok) ok = mbar_wait_w(bar(QB_OPS), 0, ec, kSiteBwdMma);
    if (ok) {
      tc_fence_after();
      issue_s(0);
      umma_commit_w(bar(QB_S));
      ok = wait_kv(QB_VF, 0);
    }
    if (ok) {
      tc_fence_after();
      issue_dp(0);
      umma_commit_w(bar(QB_DP));
      umma_commit_w(bar(QB_VE + 0));
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      const bool more = j + 1 < n_kv;
      if constexpr (C::DPB == 2) {
        // S(j+1) and dP(j+1) (other buffer) while the compute warps work on tile j
        if (more) {
          if (!(ok = mbar_wait_w(bar(QB_SFREE), j & 1, ec, kSiteBwdMma) && wait_kv(QB_KF, j + 1))) break;
          tc_fence_after();
          issue_s(j + 1);
          umma_commit_w(bar(QB_S));
          if (!(ok = wait_kv(QB_VF, j + 1))) break;
          tc_fence_after();
          issue_dp(j + 1);
          umma_commit_w(bar(QB_DP + (j + 1) % 2));
          umma_commit_w(bar(QB_VE + (j + 1) % ST));
        }
        if (!(ok = ds_then_dq(j, 0) && ds_then_dq(j, 1))) break;
        umma_commit_w(bar(QB_KE + j % ST));
      } else {
        // one dP buffer: dP(j+1) goes after dQ(j), which reads dS(j) from it.
        // With two stages the next S is formed while the compute warps work on
        // tile j; with one stage K_{j+1} cannot land before dQ(j) frees K_j.
        if constexpr (ST > 1) {
          if (more) {
            if (!(ok = mbar_wait_w(bar(QB_SFREE), j & 1, ec, kSiteBwdMma) && wait_kv(QB_KF, j + 1))) break;
            tc_fence_after();
            issue_s(j + 1);
            umma_commit_w(bar(QB_S));
          }
        }
        if (!(ok = ds_then_dq(j, 0) && ds_then_dq(j, 1))) break;
        umma_commit_w(bar(QB_KE + j % ST));
        if constexpr (ST == 1) {
          if (more) {
            if (!(ok = mbar_wait_w(bar(QB_SFREE), j & 1, ec, kSiteBwdMma) && wait_kv(QB_KF, j + 1))) break;
            tc_fence_after();
            issue_s(j + 1);
            umma_commit_w(bar(QB_S));
          }
        }
        if (more) {
          if (!(ok = wait_kv(QB_VF, j + 1))) break;
          tc_fence_after();
          issue_dp(j + 1);
          umma_commit_w(bar(QB_DP));
          umma_commit_w(bar(QB_VE + (j + 1) % ST));
        }
      }
    }
    if (ok) umma_commit_w(bar(QB_DONE));
    umma_commit_w(bar(QB_DRAIN));
    mbar_wait(bar(QB_DRAIN), 0, ec, kSiteDrain, false);
  } else {
    // ------------------------------------------------------------ compute
    const int t = threadIdx.x;
    const int row = t & 127;  // query row within the tile = TMEM lane
    const int hf = t >> 7;    // key-column half
    const int qr = q0 + row;
    const bool row_ok = qr < S_q;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const size_t ridx = static_cast<size_t>(zq) * p.rows_q + sl.row_q + (row_ok ? qr : 0);
    // -LSE*log2e and D of this row (-inf and 0 past S_q: the tile never
    // reaches beyond the statistics' padding to 128 rows)
    const size_t sidx = stat_index(static_cast<size_t>(zq), p.S_pad, sl.stat_row + qr);
    const float nl2 = p.stats[sidx];
    const float nDrow = p.stats[sidx + 64];  // -D
    const float* bias_row =
        (BIAS && row_ok) ? p.bias + (static_cast<size_t>(h) * p.S_q + qr) * p.S_kv : nullptr;
    const bool bias_vec = (p.S_kv & 3) == 0;
    const uint64_t lin_row = (static_cast<uint64_t>(bh) * p.S_q + qr) * p.S_kv;
    bool ok = true;
    if constexpr (C::OPS_IN_TMEM) {  // Q and dO rows into this thread's TMEM lane
      ok = mbar_wait(bar(QB_Q), 0, ec, kSiteBwdCompute);
      if (ok && hf < 2) {  // the first two groups copy one half of the columns each
        smem_row_to_tmem<DQK / 2>(smem + C::OFF_Q, BM, row, hf * (DQK / 2),
                                  tbase + lane_off + C::T_Q + hf * (DQK / 4));
        smem_row_to_tmem<DV / 2>(smem + C::OFF_DO, BM, row, hf * (DV / 2),
                                 tbase + lane_off + C::T_DO + hf * (DV / 4));
        tmem_wait_st();
      }
      tc_fence_before();
      if (ok) mbar_arrive(bar(QB_OPS));
    }
    const float zk = p.keep_scale;
    for (int j = 0; ok && j < n_kv; ++j) {
      const int kc0 = (khi - j) * BN + CW * hf;  // first key of this thread's columns
      uint32_t keep = 0;                 // bit c: keep flag of local column c
      if (DROP && p.keep_bits != nullptr) {  // keep bits drawn beforehand
        keep = keep_word(p.keep_bits, p.keep_words, lin_row + kc0);
      } else if constexpr (DROP) {
#pragma unroll
        for (int g = 0; g < CW / 4; ++g) {
          const uint4 d = dropout_draws((lin_row + kc0) / 4 + g, p.seed_lo, p.seed_hi,
                                        p.offset_lo, p.offset_hi);
          const uint32_t k4 = static_cast<uint32_t>(d.x >= p.drop_threshold) |
                              (static_cast<uint32_t>(d.y >= p.drop_threshold) << 1) |
                              (static_cast<uint32_t>(d.z >= p.drop_threshold) << 2) |
                              (static_cast<uint32_t>(d.w >= p.drop_threshold) << 3);
          keep |= k4 << (4 * g);
        }
      }
      auto zf = [&](int c) -> float {
        if constexpr (DROP) return ((keep >> c) & 1u) ? zk : 0.f;
        return 1.0f;
      };
      // exponent in the log2 domain: S * scale * log2e - LSE * log2e (+ Bias * log2e)
      float pr[CW];
      if constexpr (BIAS) {
        // this row's Bias for the thread's keys (keys past S_kv or a missing
        // row read 0): from the TMA tile in shared memory, block hf, the
        // row's eight 16-byte chunks in their swizzled places; else loaded
        // from global memory before the wait so its latency overlaps it
        if (bias_tma) {
          if (!(ok = mbar_wait(bar(QB_BF), j & 1, ec, kSiteBwdCompute))) break;
          const uint32_t brow = sB + hf * (BM * 128) + row * 128;
#pragma unroll
          for (int c8 = 0; c8 < CW / 4; ++c8) {
            const float4 v = lds128(brow + ((c8 ^ (row & 7)) << 4));
            pr[4 * c8 + 0] = v.x;
            pr[4 * c8 + 1] = v.y;
            pr[4 * c8 + 2] = v.z;
            pr[4 * c8 + 3] = v.w;
          }
          mbar_arrive(bar(QB_BE));
        } else if (bias_row != nullptr && bias_vec && kc0 + CW <= p.S_kv) {
          const float4* b4 = reinterpret_cast<const float4*>(bias_row + kc0);
#pragma unroll
          for (int i = 0; i < CW / 4; ++i) {
            const float4 v = __ldg(b4 + i);
            pr[4 * i + 0] = v.x;
            pr[4 * i + 1] = v.y;
            pr[4 * i + 2] = v.z;
            pr[4 * i + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int c = 0; c < CW; ++c)
            pr[c] = (bias_row != nullptr && kc0 + c < p.S_kv) ? __ldg(bias_row + kc0 + c) : 0.f;
        }
      }
      if (!(ok = mbar_wait(bar(QB_S), j & 1, ec, kSiteBwdCompute))) break;
      tc_fence_after();
      {
        uint32_t a0[32];
        tmem_ld32(tbase + C::T_S + lane_off + CW * hf, a0);
        tmem_wait_ld();
        const uint64_t sc2 = f2(p.scale_log2, p.scale_log2), nl22 = f2(nl2, nl2);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          uint64_t t = nl22;
          if constexpr (BIAS) t = fma2(f2(pr[2 * e], pr[2 * e + 1]), f2(kLog2e, kLog2e), nl22);
          const float2 x = f2split(fma2(f2(__uint_as_float(a0[2 * e]), __uint_as_float(a0[2 * e + 1])), sc2, t));
          pr[2 * e] = x.x;
          pr[2 * e + 1] = x.y;
        }
      }
      tc_fence_before();
      mbar_arrive(bar(QB_SFREE));
      if constexpr (WIN) {
        if (p.alibi != nullptr) {  // ALiBi: -slope |j - i - off|, in the log2 domain
          const float ns = -__ldg(p.alibi + b * p.alibi_stride + h) * kLog2e;
          const float base = static_cast<float>(kc0 - qr - (p.alibi_br ? S_kv - S_q : 0));
#pragma unroll
          for (int c = 0; c < CW; ++c) pr[c] = fmaf(ns, fabsf(base + static_cast<float>(c)), pr[c]);
        }
        // the thread's columns need masking where they cross S_kv or an edge of
        // some row's window (a condition uniform over the warp)
        const Band wb = lds_band(band_slot);
        const bool need_mask = (kc0 + CW > S_kv) || (kc0 + CW - 1 > q0 + wb.hi) ||
                               (kc0 < q0 + BM - 1 + wb.lo) || !row_ok;
        if (need_mask) {
          const int first = qr + wb.lo;  // the row's visible keys, none past S_q
          const int last = row_ok ? min(S_kv - 1, qr + wb.hi) : -1;
#pragma unroll
          for (int c = 0; c < CW; ++c)
            if (kc0 + c < first || kc0 + c > last) pr[c] = SDPA_NEG_INF;
        }
      } else {
        const bool need_mask = (kc0 + CW > S_kv) || (p.win_right >= 0 && kc0 + CW - 1 > q0) || !row_ok;
        if (need_mask) {
          const int last = row_ok ? (p.win_right >= 0 ? min(S_kv - 1, qr) : S_kv - 1) : -1;
#pragma unroll
          for (int c = 0; c < CW; ++c)
            if (kc0 + c > last) pr[c] = SDPA_NEG_INF;
        }
      }
#pragma unroll
      for (int c = 0; c < CW; ++c) pr[c] = ex2(pr[c]);
      const int b = j % C::DPB;  // dP buffer of this tile
      if (!(ok = mbar_wait(bar(QB_DP + b), (j / C::DPB) & 1, ec, kSiteBwdCompute))) break;
      tc_fence_after();
      // dP in two halves of 16 columns (at most half of dP in registers next
      // to P); dS of all 32 keys goes over the upper half once it is read
      const uint32_t tcol = tbase + C::T_DP + 128 * b + lane_off + CW * hf;
      const uint64_t nD2 = f2(nDrow, nDrow);
      auto ds_half = [&](const uint32_t (&dp)[16], int c0, uint32_t* out) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int cc = c0 + 2 * e;
          const float d0 = __uint_as_float(dp[2 * e]), d1 = __uint_as_float(dp[2 * e + 1]);
          const float2 r = f2split(mul2(f2(pr[cc], pr[cc + 1]), fma2(f2(d0, d1), f2(zf(cc), zf(cc + 1)), nD2)));
          out[e] = pack2<BF16>(r.x, r.y);
        }
      };
      uint32_t pk[16];
      {
        uint32_t lo[16];
        tmem_ld16(tcol, lo);
        tmem_wait_ld();
        ds_half(lo, 0, pk);
      }
      {
        uint32_t hi[16];
        tmem_ld16(tcol + 16, hi);
        tmem_wait_ld();
        // dS of the first 16 keys over the upper half just read, so dQ can
        // start on them while the second 16 are formed
        tmem_st8(tcol + 16, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(QB_DSL + b));
        ds_half(hi, 16, pk + 8);
      }
      tmem_st8(tcol + 24, pk + 8);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(QB_DSH + b));
    }
    // ---- epilogue: dQ * scale. A tile whose rows all lie in its sequence,
    // or any tile of an unpacked tensor (the tensor map drops its rows past
    // the end), is staged in Q's shared memory (idle once dQ is complete) as
    // 64-column boxes with the 128-byte swizzle, each column group taking
    // every fourth 32-column chunk, and stored by TMA; a packed sequence's
    // ragged tile is written row by row, so that it stops at the sequence's
    // end.
    if (out_slot[2]) {
      const bool ready = ok && mbar_wait(bar(QB_DONE), 0, ec, kSiteBwdCompute);
      if (ready) {
        tc_fence_after();
#pragma unroll 1
        for (int c = hf; c < DQK / 32; c += C::NQ) {
          const uint32_t dst = sQ + (c >> 1) * (BM * 128) + row * 128;
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {  // 16 columns: two 16-byte chunks
            uint32_t a[16];
            tmem_ld16(tbase + C::T_DQ + lane_off + c * 32 + hc * 16, a);
            tmem_wait_ld();
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              pk[e] = pack2<BF16>(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
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
      if (named_bar_and(1, NCT, ready) && threadIdx.x == 0) {
        const int r0 = out_slot[0], z = out_slot[1];
#pragma unroll
        for (int bx = 0; bx < DQK / 64; ++bx) tma_store_3d(&tmdQ, sQ + bx * (BM * 128), bx * 64, r0, z);
        bulk_commit_group();
        bulk_wait_group_read0();  // the boxes leave shared memory before the CTA does
      }
    } else if (hf < 2 && ok && mbar_wait(bar(QB_DONE), 0, ec, kSiteBwdCompute)) {
      // the first two groups write half of the columns each
      tc_fence_after();
      constexpr int HW = DQK / 2;  // columns per thread
      uint8_t* dst_row = static_cast<uint8_t*>(p.dq) + ridx * DQK * 2 + hf * HW * 2;
#pragma unroll
      for (int c = 0; c < HW / 32; ++c) {
        uint32_t a[32];
        tmem_ld32(tbase + C::T_DQ + lane_off + hf * HW + c * 32, a);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack2<BF16>(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(dst_row + c * 64);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
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
cudaError_t launch_bwd_dq_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const CUtensorMap& bias_map, const CUtensorMap& dq,
                            const BwdParams& p, cudaStream_t st) {
  using C = DqCfg<DQK, DV>;
  const bool bias = p.bias != nullptr;
  auto pick = [&](auto win) {
    constexpr bool W = decltype(win)::value;
    return p.dropout ? (bias ? sdpa_bwd_dq_kernel<DQK, DV, BF16, true, true, W>
                             : sdpa_bwd_dq_kernel<DQK, DV, BF16, true, false, W>)
                     : (bias ? sdpa_bwd_dq_kernel<DQK, DV, BF16, false, true, W>
                             : sdpa_bwd_dq_kernel<DQK, DV, BF16, false, false, W>);
  };
  auto kern = (p.win_general || p.alibi != nullptr) ? pick(std::true_type{}) : pick(std::false_type{});
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::SMEM, 0);
  if (e != cudaSuccess) return e;
  const int n_qt = (p.S_q + C::BM - 1) / C::BM;
  const long long grid = static_cast<long long>(n_qt) * p.B * p.H;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, st>>>(q, k, v, dout, bias_map, dq, p);
  return cudaGetLastError();
}

}  // namespace sdpa
