// Fused attention forward for sm_103a: TMA-fed tiles, tcgen05 MMAs into tensor
// memory, fp32 online softmax with a saved natural-log logsumexp, in-kernel
// Philox4x32-10 dropout, optional fp32 additive bias and top-left causal mask.
//
// Computes, per (batch, head), the forward half of the equation block that
// opens CK tile's fmha_bwd_kernel.hpp: S = Q K^T, S' = S * scale,
// S'' = S' + Bias, P = softmax(S''), O = P V, with dropout applied to P before
// the product with V (keep / (1 - p)) and the softmax statistic returned as in
// PyTorch cudnn MHA.cpp run_cudnn_SDP_fprop (fp32 [b, h, s_q]).
//
// One CTA owns two tiles of 128 query rows (tile t = rows q0 + 128 t ..) of one
// (b, h), one CTA per SM, and walks the key/value tiles of 128 rows that either
// query tile sees, from the diagonal down. Each K_j / V_j tile is loaded once
// for both query tiles.
//   warpgroup 0, 1   softmax of query tile 0, 1: a thread owns one query row =
//                    TMEM lane. It reads S_t, applies scale, bias and mask in
//                    the exp2 domain, keeps a running max m and sum l, writes
//                    P_t (io dtype) over the first half of S_t's columns, and
//                    rescales O_t in TMEM when m has grown by more than 2^8
//                    since it was last used (otherwise the stale max is kept;
//                    P <= 256 is exact enough in fp32 / bf16).
//   warpgroup 2      warp 8: TMA producer (both Q tiles once; K_j and V_j
//                    through a ring). warp 9: MMA issuer; the whole warp runs
//                    the issue loop and one elected lane issues. Warps 10-11
//                    only give their registers away.
// MMA order per key tile j: O_0 += P_0(j) V_j, S_0(j+1), O_1 += P_1(j) V_j,
// S_1(j+1): while one warpgroup's softmax runs, the tensor core works for the
// other tile, so each softmax has two MMA groups' time before the tensor core
// waits for it. S_t(j+1) follows O_t's product in the in-order pipe, so it
// never overwrites P_t(j) before that product has read it.
// Tensor memory: S_0 [0,128), S_1 [128,256) (P_t aliases the first 64
// columns of S_t), O_0 [256, 256 + D_v), O_1 after it.
// Registers: launched at 168 a thread (384 threads); the producer/MMA
// warpgroup drops to 72 and the softmax warpgroups rise to 216, enough for a
// row's 128 scores without spilling: 2 x 128 x 216 + 128 x 72 = 384 x 168.
// With a bias (its 128 values per row loaded ahead of the scores) or dropout
// (the keep words) the softmax takes 224 and the issuing warpgroup 56, which
// it fits in when its descriptors are built at each issue (opaque_u64).
// GENERAL (an additive bias present), DROP (dropout) and WIN (a local window
// or the bottom-right alignment) are template parameters so the plain kernel
// is compiled without their registers. RAW (no bias or ALiBi, a nonzero
// scale) keeps the scores unscaled until the exponential, which takes the
// scale and the row max in one FMA per score; dropout leaves the softmax
// statistics alone (it zeroes entries of P after the exponentials), so it
// runs in the raw-score kernels too. Under dropout the kernel can also record
// the keep bits it draws (FwdParams::keep_out, sdpa_dropout_mask's packing),
// for the backward to read instead of drawing them again.
#pragma once
#include <type_traits>

#include "common.cuh"

namespace sdpa {

template <int DQK, int DV>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128;  // rows per query tile / key tile
  static constexpr int Q_BYTES = BM * DQK * 2;
  static constexpr int K_BYTES = BN * DQK * 2;
  static constexpr int V_BYTES = BN * DV * 2;
  // as many K/V stages as fit next to the two Q tiles (at most 3)
  static constexpr int AVAIL = 227 * 1024 - 2 * Q_BYTES - 256 - 1024;
  static constexpr int FIT = AVAIL / (K_BYTES + V_BYTES);
  static constexpr int STAGES = FIT >= 3 ? 3 : FIT;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * V_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + alignment slack
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0, T_O = 256;
  // measured with ptxas: the plain softmax needs ~210 registers and the MMA
  // issuer ~70; with a bias or dropout the softmax needs ~220, and the issuer
  // fits in 56 once its base descriptors are opaque
  static constexpr int REG_LAUNCH = 168, REG_SOFTMAX = 216, REG_OTHER = 72;
  static constexpr int REG_SOFTMAX_FLAGS = 224, REG_OTHER_FLAGS = 56;
  static_assert(STAGES >= 1 && SMEM <= 227 * 1024, "shared memory");
  static_assert(DQK % 64 == 0 && DV % 64 == 0 && DV <= 128, "unsupported head size");
  static_assert(2 * 128 * REG_SOFTMAX + 128 * REG_OTHER == THREADS * REG_LAUNCH, "register split");
  static_assert(2 * 128 * REG_SOFTMAX_FLAGS + 128 * REG_OTHER_FLAGS == THREADS * REG_LAUNCH,
                "register split");
};

// Barrier slots (the K/V ring has at most 3 stages).
enum : int { FB_Q = 0, FB_S, FB_P = FB_S + 2, FB_O = FB_P + 2, FB_DRAIN = FB_O + 2, FB_KF,
             FB_KE = FB_KF + 3, FB_VF = FB_KE + 3, FB_VE = FB_VF + 3, FB_COUNT = FB_VE + 3 };

template <int DQK, int DV, bool BF16, bool GENERAL, bool WIN, bool RAW, bool DROP>
__global__ void __launch_bounds__(384, 1)
    sdpa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<DQK, DV>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sQ = smem_u32(smem + C::OFF_Q);
  const uint32_t sK = smem_u32(smem + C::OFF_K);
  const uint32_t sV = smem_u32(smem + C::OFF_V);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + FB_COUNT);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  Band* band_slot = reinterpret_cast<Band*>(bars + FB_COUNT + 1);  // see lds_band
  static_assert((FB_COUNT + 2) * 8 <= 256, "barrier region");
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- query tiles of this CTA: query_tile_order over pairs of query tiles,
  // groups of up to 8 heads (one group's K/V stay in L2, the grid ends on its
  // lightest pairs)
  const int n_qt = (p.S_q + C::BM - 1) / C::BM;
  const int n_pairs = (n_qt + 1) / 2;
  const QueryTile qtile = query_tile_order(static_cast<int>(blockIdx.x), p.B, p.H, n_pairs, 8);
  const int b = qtile.b, h = qtile.h;
  const int bh = b * p.H + h;  // (batch entry or sequence, head): the dropout index
  const SeqSlice sl = seq_slice(p.seqstart_q, p.seqstart_k, p.rows_q, p.rows_k, p.S_q, p.S_kv, p.H,
                                p.H_kv, b);
  const int S_q = sl.len_q, S_kv = sl.len_k;  // this sequence's lengths
  const int zq = sl.zq0 + h;                  // tensor-map z of the query head
  const int zk = sl.zk0 + h / (p.H / p.H_kv);  // and of its K/V head
  // The ranges below are the arithmetic of query_pair, key_tiles_of_rows,
  // fwd_iters and fwd_tile_iters (common.cuh), which the library's host-side
  // range check (sdpa_tile_ranges) runs; they stay written out here because
  // calling those functions changed the compiled forward and cost 1.8% of
  // its time (measured, same box).
  // Pairs of query tiles: (0,1), (2,3), ... when the sequence has an even
  // number of tiles; with an odd number, tile 0 goes alone and the pairs are
  // (1,2), (3,4), ..., so the tile without a partner (which runs without the
  // other softmax group to overlap it) is the one with the fewest causal key
  // tiles, not the diagonal-most one that would end the grid.
  const int n_qt_seq = (S_q + C::BM - 1) / C::BM;
  const bool odd = (n_qt_seq & 1) != 0;
  const bool lone = odd && qtile.qt == 0;
  const int q0 = (odd ? max(2 * qtile.qt - 1, 0) : 2 * qtile.qt) * C::BM;  // first row of tile 0
  // (WIN: any window; else top-left, causal when win_right >= 0)
  const Band bd = WIN ? band_of(p.win_left, p.win_right, p.win_br, S_q, S_kv)
                          : Band{-kUnbounded, p.win_right >= 0 ? 0 : kUnbounded};
  // key tiles [klo_t, khi_t] query tile t sees: those holding a visible key of
  // one of its rows (none when the tile lies past S_q or no row sees a key)
  int klo0 = 0, khi0 = -1, klo1 = 0, khi1 = -1;
  auto tile_keys = [&](int t, int& klo, int& khi) {
    const int qs = q0 + t * C::BM;
    if ((t == 1 && lone) || qs >= S_q) return;
    const int lo = max(qs + bd.lo, 0), hi = min(min(qs + C::BM, S_q) - 1 + bd.hi, S_kv - 1);
    if (lo <= hi) {
      klo = lo / C::BN;
      khi = hi / C::BN;
    }
  };
  tile_keys(0, klo0, khi0);
  tile_keys(1, klo1, khi1);
  const int n_kv0 = khi0 - klo0 + 1, n_kv1 = khi1 - klo1 + 1;
  const bool has0 = n_kv0 > 0, has1 = n_kv1 > 0;
  // Iteration j visits key tile khi - j (from the diagonal down); query tile
  // t takes part in iterations [j0_t, j1_t]. The rows of tile 1 follow those
  // of tile 0, so its key range starts and ends no earlier.
  const int khi = max(khi0, khi1);
  const int n_it = (has0 || has1) ? khi - (has0 ? klo0 : klo1) + 1 : 0;
  const int j0_0 = has0 ? khi - khi0 : n_it, j1_0 = has0 ? khi - klo0 : -1;
  const int j0_1 = has1 ? khi - khi1 : n_it, j1_1 = has1 ? khi - klo1 : -1;

  // Nothing to compute (packed sequences only: a pair past the end of a
  // shorter sequence, or a sequence without keys, whose rows get O = 0 and
  // LSE = -inf as any query row that sees no key). Uniform over the CTA.
  if (n_it == 0) {
    const int row = q0 + static_cast<int>(threadIdx.x);
    if (threadIdx.x < (lone ? 1 : 2) * C::BM && row < S_q) {
      const size_t ri = static_cast<size_t>(zq) * p.rows_q + sl.row_q + row;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.o) + ri * DV * 2);
#pragma unroll
      for (int v = 0; v < DV / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
      p.lse[ri] = SDPA_NEG_INF;
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < FB_COUNT; ++i) mbar_init(bar(i), (i == FB_P || i == FB_P + 1) ? 128u : 1u);
    *abort_flag = 0u;
    if (WIN) *band_slot = bd;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const ErrCtx ec{p.err, abort_flag, p.wait_ns};

  // a bias or dropout moves registers from the issuing warpgroup to the softmax
  constexpr bool FLAGS = GENERAL || DROP;
  if (warp >= 8) {
    setmaxnreg_dec<FLAGS ? C::REG_OTHER_FLAGS : C::REG_OTHER>();
    if (warp == 8) {
      // ---------------------------------------------------------- producer
      int issued = 0;
      if (lane == 0 && n_it > 0) {
        mbar_arrive_expect_tx(bar(FB_Q), (has1 ? 2 : 1) * C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < DQK / 64; ++c) {
          tma_load_3d(sQ + c * C::BM * 128, &tmQ, bar(FB_Q), c * 64, sl.row_q + q0, zq);
          if (has1)
            tma_load_3d(sQ + C::Q_BYTES + c * C::BM * 128, &tmQ, bar(FB_Q), c * 64, sl.row_q + q0 + C::BM, zq);
        }
      }
      for (int j = 0; j < n_it; ++j) {
        const int s = j % ST;
        const uint32_t ph = (j / ST) & 1;
        const int kv0 = sl.row_k + (khi - j) * C::BN;
        if (!mbar_wait(bar(FB_KE + s), ph ^ 1, ec, kSiteFwdLoad, true, true)) break;
        if (p.fault == 1) break;  // test hook: K/V never arrive
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(FB_KF + s), C::K_BYTES);
#pragma unroll
          for (int c = 0; c < DQK / 64; ++c)
            tma_load_3d(sK + s * C::K_BYTES + c * C::BN * 128, &tmK, bar(FB_KF + s), c * 64, kv0, zk);
        }
        if (!mbar_wait(bar(FB_VE + s), ph ^ 1, ec, kSiteFwdLoad, true, true)) {
          issued = 2 * j + 1;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(FB_VF + s), C::V_BYTES);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_3d(sV + s * C::V_BYTES + c * C::BN * 128, &tmV, bar(FB_VF + s), c * 64, kv0, zk);
        }
        issued = 2 * j + 2;
      }
      __syncwarp();
      // Drain: every copy issued must land before the CTA can retire. On the
      // healthy path these phases completed long ago.
      if ((*abort_flag || p.fault != 0) && n_it > 0) {
        mbar_wait(bar(FB_Q), 0, ec, kSiteDrain, false);
        for (int i = 0; i < issued; ++i) {
          const int j = i >> 1, s = j % ST;
          const uint32_t ph = (j / ST) & 1;
          mbar_wait(bar(((i & 1) ? FB_VF : FB_KF) + s), ph, ec, kSiteDrain, false);
        }
      }
    } else if (warp == 9) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t kIdO = idesc_f16(128, DV, BF16, false, true);
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sK, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sV, C::BN * 128, 1024);
      uint32_t pph0 = 0, pph1 = 0;  // P phases consumed per query tile
      // base descriptors opaque where the issuer runs at 56 registers or the
      // ring has one stage (then nothing in them changes across iterations)
      constexpr bool OPQ = FLAGS || ST == 1;
      auto base = [](uint64_t d) { return OPQ ? opaque_u64(d) : d; };
      auto issue_s = [&](int t, int j) {  // S_t = Q_t K_j^T
        const uint64_t dQ = base(desc_adv(dQ0, t * C::Q_BYTES));
        const uint64_t dK = base(desc_adv(dK0, (j % ST) * C::K_BYTES));
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
          umma_ss_w(tbase + C::T_S + 128 * t, desc_adv(dQ, off), desc_adv(dK, off), kIdS, kk > 0);
        }
        umma_commit_w(bar(FB_S + t));
      };
      auto issue_pv = [&](int t, int j, bool first) {  // O_t += P_t V_j
        const uint64_t dV = base(desc_adv(dV0, (j % ST) * C::V_BYTES));
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          umma_ts_w(tbase + C::T_O + DV * t, tbase + C::T_S + 128 * t + kk * 8, desc_adv(dV, kk * 2048),
                    kIdO, (!first || kk > 0));
      };
      auto wait_k = [&](int j) { return mbar_wait_w(bar(FB_KF + j % ST), (j / ST) & 1, ec, kSiteFwdMma); };
      auto wait_v = [&](int j) { return mbar_wait_w(bar(FB_VF + j % ST), (j / ST) & 1, ec, kSiteFwdMma); };
      auto in0 = [&](int j) { return j >= j0_0 && j <= j1_0; };  // tile 0 uses key tile khi - j
      auto in1 = [&](int j) { return j >= j0_1 && j <= j1_1; };
      bool ok = n_it > 0 && mbar_wait_w(bar(FB_Q), 0, ec, kSiteFwdMma) && wait_k(0);
      if (ok) {
        tc_fence_after();
        if (in0(0)) issue_s(0, 0);
        if (in1(0)) issue_s(1, 0);
        umma_commit_w(bar(FB_KE + 0));
      }
      for (int j = 0; ok && j < n_it; ++j) {
        const bool more = j + 1 < n_it;
        if (!(ok = wait_v(j))) break;
        // query tile 0
        if (in0(j)) {
          if (!(ok = mbar_wait_w(bar(FB_P + 0), pph0, ec, kSiteFwdMma))) break;
          pph0 ^= 1u;
          tc_fence_after();
          issue_pv(0, j, j == j0_0);
        }
        if (more && in0(j + 1)) {
          if (!(ok = wait_k(j + 1))) break;
          tc_fence_after();
          issue_s(0, j + 1);
        }
        // query tile 1
        if (in1(j)) {
          if (!(ok = mbar_wait_w(bar(FB_P + 1), pph1, ec, kSiteFwdMma))) break;
          pph1 ^= 1u;
          tc_fence_after();
          issue_pv(1, j, j == j0_1);
        }
        if (more && in1(j + 1)) {
          if (!(ok = wait_k(j + 1))) break;
          tc_fence_after();
          issue_s(1, j + 1);
        }
        umma_commit_w(bar(FB_VE + j % ST));
        if (more) umma_commit_w(bar(FB_KE + (j + 1) % ST));
      }
      if (ok) {
        umma_commit_w(bar(FB_O + 0));
        umma_commit_w(bar(FB_O + 1));
      }
      umma_commit_w(bar(FB_DRAIN));
      mbar_wait(bar(FB_DRAIN), 0, ec, kSiteDrain, false);
    }
  } else {
    setmaxnreg_inc<FLAGS ? C::REG_SOFTMAX_FLAGS : C::REG_SOFTMAX>();
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;  // query tile of this warpgroup
    const int qt0 = q0 + t * C::BM;
    const int row = qt0 + (threadIdx.x & 127);
    const int n_kv = t == 0 ? n_kv0 : n_kv1;
    const int khi_t = WIN ? (t == 0 ? khi0 : khi1) : n_kv - 1;  // the plain masks start at key 0
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + C::T_S + 128 * t, tO = tbase + C::T_O + DV * t;
    const float sl2 = p.scale_log2;
    const bool row_ok = row < S_q;
    const float* bias_row = (GENERAL && p.bias != nullptr && row_ok)
                                ? p.bias + (static_cast<size_t>(h) * p.S_q + row) * p.S_kv
                                : nullptr;
    const bool bias_vec = (p.S_kv & 3) == 0;
    const uint64_t lin_row = (static_cast<uint64_t>(bh) * p.S_q + row) * p.S_kv;
    const uint64_t sl22 = f2(sl2, sl2);
    // RAW (no bias, dropout or ALiBi, a nonzero scale): the scores stay raw
    // until the exponential. A masked key takes the raw value that scales to
    // -inf, the row max is the largest raw score (the smallest under a
    // negative scale) times scale * log2e, which equals the largest scaled
    // score since rounding is monotonic, and P = 2^fma(S, scale * log2e, -m).
    static_assert(!(RAW && GENERAL), "raw scores have no additive terms");
    const float neg = (RAW && sl2 < 0.f) ? -SDPA_NEG_INF : SDPA_NEG_INF;  // masked score
    float m = SDPA_NEG_INF, l = 0.f;
    bool ok = true;
    for (int c = 0; c < n_kv; ++c) {
      const int k0 = (khi_t - c) * C::BN;  // key tiles from the diagonal down
      // scores in the log2 domain: S * scale * log2e (+ Bias * log2e)
      float x[128];
      if (GENERAL && bias_row != nullptr) {
        // the row's Bias, loaded before the wait so its latency overlaps it
        // (keys past S_kv read 0; they are masked below)
        if (bias_vec && k0 + C::BN <= p.S_kv) {
          const float4* b4 = reinterpret_cast<const float4*>(bias_row + k0);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float4 v = __ldg(b4 + i);
            x[4 * i + 0] = v.x;
            x[4 * i + 1] = v.y;
            x[4 * i + 2] = v.z;
            x[4 * i + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i) x[i] = (k0 + i < p.S_kv) ? __ldg(bias_row + k0 + i) : 0.f;
        }
      }
      // dropout keep flags of keys k0 .. k0 + 127 (word w: keys k0 + 32 w ..,
      // bit i: key k0 + 32 w + i, the packing of sdpa_dropout_mask), read or
      // drawn before the wait for the scores so the draws overlap it
      uint32_t kw[4] = {~0u, ~0u, ~0u, ~0u};
      if constexpr (DROP) {
        if (p.keep_bits != nullptr) {  // drawn beforehand
#pragma unroll
          for (int w = 0; w < 4; ++w) kw[w] = keep_word(p.keep_bits, p.keep_words, lin_row + k0 + 32 * w);
        } else {
          const uint64_t g0 = (lin_row + k0) >> 2;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint32_t acc = 0;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const uint4 d = dropout_draws(g0 + 8 * w + g, p.seed_lo, p.seed_hi, p.offset_lo, p.offset_hi);
              acc |= (static_cast<uint32_t>(d.x >= p.drop_threshold) << (4 * g)) |
                     (static_cast<uint32_t>(d.y >= p.drop_threshold) << (4 * g + 1)) |
                     (static_cast<uint32_t>(d.z >= p.drop_threshold) << (4 * g + 2)) |
                     (static_cast<uint32_t>(d.w >= p.drop_threshold) << (4 * g + 3));
            }
            kw[w] = acc;
          }
          if (p.keep_out != nullptr && row_ok) {
            // record them for the backward: whole words of this row only
            // (the host requires S_kv % 32 == 0 for a record)
            uint32_t* dst = p.keep_out + ((lin_row + k0) >> 5);
#pragma unroll
            for (int w = 0; w < 4; ++w)
              if (k0 + 32 * w < p.S_kv) dst[w] = kw[w];
          }
        }
      }
      if (!(ok = mbar_wait(bar(FB_S + t), c & 1, ec, kSiteFwdSoftmax))) break;
      tc_fence_after();
      if constexpr (GENERAL) {
        // a quarter at a time (the scores join the bias values held in x)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t rr[32];
          tmem_ld32(tS + lane_off + q * 32, rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t s2 = f2(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1]));
            float2 v;
            if (bias_row != nullptr)
              v = f2split(fma2(s2, sl22, mul2(f2(x[q * 32 + 2 * i], x[q * 32 + 2 * i + 1]), f2(kLog2e, kLog2e))));
            else
              v = f2split(mul2(s2, sl22));
            x[q * 32 + 2 * i] = v.x;
            x[q * 32 + 2 * i + 1] = v.y;
          }
        }
      } else {
        // the four quarters' loads in flight together, one wait
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32f(tS + lane_off + q * 32, x + q * 32);
        tmem_wait_ld();
        if constexpr (!RAW) {
#pragma unroll
          for (int i = 0; i < 128; i += 2) {
            const float2 v = f2split(mul2(f2(x[i], x[i + 1]), sl22));
            x[i] = v.x;
            x[i + 1] = v.y;
          }
        }
      }
      if constexpr (WIN && !RAW) {
        if (p.alibi != nullptr) {  // ALiBi: -slope |j - i - off|, in the log2 domain
          const float ns = -__ldg(p.alibi + b * p.alibi_stride + h) * kLog2e;
          const float base = static_cast<float>(k0 - row - (p.alibi_br ? S_kv - S_q : 0));
#pragma unroll
          for (int i = 0; i < 128; ++i) x[i] = fmaf(ns, fabsf(base + static_cast<float>(i)), x[i]);
        }
      }
      if constexpr (WIN) {
        // a tile needs masking where it crosses S_kv or an edge of some row's window
        const Band wb = lds_band(band_slot);
        if ((k0 + C::BN > S_kv) || (k0 + C::BN - 1 > qt0 + wb.hi) || (k0 < qt0 + C::BM - 1 + wb.lo)) {
          const int first = row + wb.lo, last = min(S_kv - 1, row + wb.hi);  // visible keys
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (k0 + i < first || k0 + i > last) x[i] = neg;
        }
      } else if ((k0 + C::BN > S_kv) || (p.win_right >= 0 && k0 + C::BN - 1 > qt0)) {
        const int lim = p.win_right >= 0 ? min(S_kv - 1, row) : S_kv - 1;  // last visible key
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (k0 + i > lim) x[i] = neg;
      }
      float mx;
      if (!RAW || sl2 > 0.f) {
        mx = extreme_of<false, 128>(x);
        if (RAW) mx *= sl2;
      } else {
        mx = extreme_of<true, 128>(x) * sl2;
      }
      // Rescale only when the max grew by more than 8 (a factor 256).
      const bool grow = mx > m + 8.0f;
      float alpha = 1.0f;
      if (grow) {
        alpha = ex2(m - mx);  // 0 when m was -inf
        m = mx;
      }
      // S_t(c) follows O_t's previous product in the pipe, so O_t is settled
      if (c > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int q = 0; q < DV / 16; ++q) {
          uint32_t rr[16];
          tmem_ld16(tO + lane_off + q * 16, rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
          tmem_st16(tO + lane_off + q * 16, rr);
        }
      }
      l *= alpha;
      const float mu = (m == SDPA_NEG_INF) ? 0.f : m;
      const uint64_t nm2 = f2(-mu, -mu);
      uint64_t sa = f2(0.f, 0.f), sb = f2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 128; i += 4) {
        const float2 a = f2split(RAW ? fma2(f2(x[i], x[i + 1]), sl22, nm2) : add2(f2(x[i], x[i + 1]), nm2));
        const float2 bq =
            f2split(RAW ? fma2(f2(x[i + 2], x[i + 3]), sl22, nm2) : add2(f2(x[i + 2], x[i + 3]), nm2));
        x[i] = ex2(a.x);
        x[i + 1] = ex2(a.y);
        x[i + 2] = ex2(bq.x);
        x[i + 3] = ex2(bq.y);
        sa = add2(sa, f2(x[i], x[i + 1]));
        sb = add2(sb, f2(x[i + 2], x[i + 3]));
      }
      {
        const float2 u = f2split(sa), w = f2split(sb);
        l += (u.x + u.y) + (w.x + w.y);
      }
      if constexpr (DROP) {  // dropout: zero the dropped entries of P
#pragma unroll
        for (int w = 0; w < 4; ++w) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (!((kw[w] >> i) & 1u)) x[32 * w + i] = 0.f;
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(x[q * 32 + 2 * i], x[q * 32 + 2 * i + 1]);
        tmem_st16(tS + lane_off + q * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(FB_P + t));
    }
    // ---- epilogue: O / l (times 1/(1-p) under dropout), LSE = m ln2 + ln l
    if (n_kv > 0 && ok && mbar_wait(bar(FB_O + t), 0, ec, kSiteFwdSoftmax)) {
      tc_fence_after();
      const float inv = (l > 0.f) ? (DROP ? p.keep_scale : 1.0f) / l : 0.f;
      const size_t ri = static_cast<size_t>(zq) * p.rows_q + sl.row_q + (row_ok ? row : 0);
      uint8_t* orow = static_cast<uint8_t*>(p.o) + ri * DV * 2;
#pragma unroll
      for (int q = 0; q < DV / 32; ++q) {
        uint32_t rr[32];
        tmem_ld32(tO + lane_off + q * 32, rr);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(rr[2 * i]) * inv, __uint_as_float(rr[2 * i + 1]) * inv);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + q * 64);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (row_ok)
        p.lse[ri] = (l > 0.f) ? fmaf(m, kLn2, __logf(l)) : SDPA_NEG_INF;
    } else if (n_kv == 0 && row_ok && !(t == 1 && lone)) {
      // no row of this tile sees a key (the other tile's rows do): O = 0, LSE = -inf
      // (a lone tile 0's partner rows belong to the next pair)
      const size_t ri = static_cast<size_t>(zq) * p.rows_q + sl.row_q + row;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.o) + ri * DV * 2);
#pragma unroll
      for (int v = 0; v < DV / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
      p.lse[ri] = SDPA_NEG_INF;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int DQK, int DV, bool BF16>
cudaError_t launch_fwd_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                         const FwdParams& p, cudaStream_t st) {
  using C = FwdCfg<DQK, DV>;
  const bool general = p.bias != nullptr;
  // raw scores (RAW) unless a bias, ALiBi or a zero scale; ALiBi and a zero
  // scale take the windowed kernel, which also runs the plain masks
  const bool raw = !general && p.alibi == nullptr && p.scale_log2 != 0.f;
  const bool win = p.win_general || p.alibi != nullptr || (!general && !raw);
  auto pick = [&](auto drop) {
    constexpr bool D = decltype(drop)::value;
    return general ? (win ? sdpa_fwd_kernel<DQK, DV, BF16, true, true, false, D>
                          : sdpa_fwd_kernel<DQK, DV, BF16, true, false, false, D>)
                   : !raw ? sdpa_fwd_kernel<DQK, DV, BF16, false, true, false, D>
                          : (win ? sdpa_fwd_kernel<DQK, DV, BF16, false, true, true, D>
                                 : sdpa_fwd_kernel<DQK, DV, BF16, false, false, true, D>);
  };
  auto kern = p.dropout ? pick(std::true_type{}) : pick(std::false_type{});
  // The warpgroups' setmaxnreg shares add up to exactly 384 x REG_LAUNCH; had
  // the compiler given the kernel another launch register count, the softmax
  // warpgroups' increase could never be granted, so refuse to launch then.
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::SMEM, C::REG_LAUNCH);
  if (e != cudaSuccess) return e;
  const int n_qt = (p.S_q + C::BM - 1) / C::BM;
  const long long grid = static_cast<long long>((n_qt + 1) / 2) * p.B * p.H;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, st>>>(q, k, v, p);
  return cudaGetLastError();
}

}  // namespace sdpa
