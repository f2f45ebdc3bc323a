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
// One CTA owns a tile of 128 query rows of one (b, h) and walks the key/value
// tiles of 128 rows:
//   warp 4       TMA producer: Q once, then K_j and V_j through a ring.
//   warp 5       MMA issuer (one lane): S = Q K_j^T into TMEM, then
//                O += P_j V_j with P_j read from TMEM.
//   warps 0-3    softmax: thread t owns query row t = TMEM lane t. It reads
//                S_j, applies scale, bias and mask in the exp2 domain, keeps a
//                running max m and sum l, writes P_j (io dtype) over the first
//                half of S_j's columns, and rescales O in TMEM when m has grown
//                by more than 2^8 since it was last used (otherwise the stale
//                max is kept; P <= 256 is exact enough in fp32 / bf16).
// Tensor memory: columns [0,128) hold S_j (P_j aliases [0,64)); columns
// [128, 128 + D_v) hold the O accumulator. Two CTAs share an SM when shared
// memory allows, so one CTA's softmax overlaps the other's MMAs.
#pragma once
#include "common.cuh"

namespace sdpa {

template <int DQK, int DV>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int STAGES = (DQK <= 64) ? 2 : (DQK <= 128 ? 1 : 2);
  static constexpr int Q_BYTES = BM * DQK * 2;
  static constexpr int K_BYTES = BN * DQK * 2;
  static constexpr int V_BYTES = BN * DV * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * V_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + alignment slack
  static constexpr int MIN_BLOCKS = (2 * SMEM <= 227 * 1024) ? 2 : 1;
  static constexpr int THREADS = 192;
  static constexpr uint32_t TMEM_COLS = 256;
  static_assert(DQK % 64 == 0 && DV % 64 == 0 && DV <= 128, "unsupported head size");
};

// Barrier slots.
enum : int { FB_Q = 0, FB_S, FB_P, FB_O, FB_DRAIN, FB_KF, FB_KE = FB_KF + 2, FB_VF = FB_KE + 2,
             FB_VE = FB_VF + 2, FB_COUNT = FB_VE + 2 };

template <int DQK, int DV, bool BF16>
__global__ void __launch_bounds__(192, FwdCfg<DQK, DV>::MIN_BLOCKS)
    sdpa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sQ = smem_u32(smem + C::OFF_Q);
  const uint32_t sK = smem_u32(smem + C::OFF_K);
  const uint32_t sV = smem_u32(smem + C::OFF_V);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + FB_COUNT);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- query tile of this CTA (order: query_tile_order, groups of up to 8
  // heads: measured at b1 h32 s16384 causal, 1.83 ms, against 1.98 ms one head
  // at a time, whose grid ends on a head's heaviest tiles)
  const int n_qt = (p.S_q + C::BM - 1) / C::BM;
  const QueryTile qtile = query_tile_order(static_cast<int>(blockIdx.x), p.B, p.H, n_qt, 8);
  const int b = qtile.b, h = qtile.h, qt = qtile.qt;
  const int bh = b * p.H + h;
  const int q0 = qt * C::BM;
  const int n_kv_all = (p.S_kv + C::BN - 1) / C::BN;
  const int n_kv = p.causal ? min(n_kv_all, (q0 + C::BM - 1) / C::BN + 1) : n_kv_all;
  // Iteration j visits key tile n_kv - 1 - j: the CTAs of one head, resident
  // together, then start on different tiles (their own diagonal) instead of
  // all requesting tile 0 from L2 at once.

  if (threadIdx.x == 0) {
    for (int i = 0; i < FB_COUNT; ++i) mbar_init(bar(i), i == FB_P ? 128u : 1u);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tS = tbase, tO = tbase + 128;
  const ErrCtx ec{p.err, abort_flag};

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(FB_Q), C::Q_BYTES);
#pragma unroll
      for (int c = 0; c < DQK / 64; ++c)
        tma_load_3d(sQ + c * C::BM * 128, &tmQ, bar(FB_Q), c * 64, q0, bh);
    }
    for (int j = 0; j < n_kv; ++j) {
      const int s = j % C::STAGES;
      const uint32_t ph = (j / C::STAGES) & 1;
      if (!mbar_wait(bar(FB_KE + s), ph ^ 1, ec, kSiteFwdLoad)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(FB_KF + s), C::K_BYTES);
#pragma unroll
        for (int c = 0; c < DQK / 64; ++c)
          tma_load_3d(sK + s * C::K_BYTES + c * C::BN * 128, &tmK, bar(FB_KF + s), c * 64,
                      (n_kv - 1 - j) * C::BN, bh);
      }
      if (!mbar_wait(bar(FB_VE + s), ph ^ 1, ec, kSiteFwdLoad)) {
        issued = 2 * j + 1;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(FB_VF + s), C::V_BYTES);
#pragma unroll
        for (int c = 0; c < DV / 64; ++c)
          tma_load_3d(sV + s * C::V_BYTES + c * C::BN * 128, &tmV, bar(FB_VF + s), c * 64,
                      (n_kv - 1 - j) * C::BN, bh);
      }
      issued = 2 * j + 2;
    }
    __syncwarp();
    // Drain: every copy issued must land before the CTA can retire. On the
    // healthy path these phases completed long ago.
    if (*abort_flag) {
      mbar_wait(bar(FB_Q), 0, ec, kSiteDrain, false);
      for (int i = 0; i < issued; ++i) {
        const int j = i >> 1, s = j % C::STAGES;
        const uint32_t ph = (j / C::STAGES) & 1;
        mbar_wait(bar(((i & 1) ? FB_VF : FB_KF) + s), ph, ec, kSiteDrain, false);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
    constexpr uint32_t kIdO = idesc_f16(128, DV, BF16, false, true);
    const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024);
    const uint64_t dK0 = sdesc_sw128(sK, 16, 1024);
    const uint64_t dV0 = sdesc_sw128(sV, C::BN * 128, 1024);
    // the whole warp runs the issue loop; one elected lane issues (umma_*_w)
    bool ok = mbar_wait_w(bar(FB_Q), 0, ec, kSiteFwdMma);
    for (int j = 0; ok && j < n_kv; ++j) {
      const int s = j % C::STAGES;
      const uint32_t ph = (j / C::STAGES) & 1;
      if (!(ok = mbar_wait_w(bar(FB_KF + s), ph, ec, kSiteFwdMma))) break;
      tc_fence_after();
      {
        const uint64_t dK = desc_adv(dK0, s * C::K_BYTES);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
          umma_ss_w(tS, desc_adv(dQ0, off), desc_adv(dK, off), kIdS, kk > 0);
        }
        umma_commit_w(bar(FB_S));
        umma_commit_w(bar(FB_KE + s));
      }
      if (!(ok = mbar_wait_w(bar(FB_P), j & 1, ec, kSiteFwdMma))) break;
      if (!(ok = mbar_wait_w(bar(FB_VF + s), ph, ec, kSiteFwdMma))) break;
      tc_fence_after();
      {
        const uint64_t dV = desc_adv(dV0, s * C::V_BYTES);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          umma_ts_w(tO, tS + kk * 8, desc_adv(dV, kk * 2048), kIdO, (j > 0 || kk > 0));
        umma_commit_w(bar(FB_VE + s));
      }
    }
    if (ok) umma_commit_w(bar(FB_O));
    umma_commit_w(bar(FB_DRAIN));
    mbar_wait(bar(FB_DRAIN), 0, ec, kSiteDrain, false);
  } else {
    // ------------------------------------------------------------ softmax
    const int t = threadIdx.x;  // 0..127 = TMEM lane = query row within the tile
    const int row = q0 + t;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    const bool row_ok = row < p.S_q;
    const float* bias_row =
        (p.bias != nullptr && row_ok) ? p.bias + (static_cast<size_t>(h) * p.S_q + row) * p.S_kv
                                      : nullptr;
    const bool bias_vec = (p.S_kv & 3) == 0;
    const uint64_t lin_row = (static_cast<uint64_t>(bh) * p.S_q + row) * p.S_kv;
    float m = SDPA_NEG_INF, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!(ok = mbar_wait(bar(FB_S), j & 1, ec, kSiteFwdSoftmax))) break;
      tc_fence_after();
      float x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t rr[32];
        tmem_ld32(tS + lane_off + c * 32, rr);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(rr[i]) * sl2;
      }
      const int k0 = (n_kv - 1 - j) * C::BN;  // key tiles from the diagonal down
      if (p.bias != nullptr) {
        if (bias_row != nullptr) {
          if (bias_vec && k0 + C::BN <= p.S_kv) {
            const float4* b4 = reinterpret_cast<const float4*>(bias_row + k0);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float4 v = __ldg(b4 + i);
              x[4 * i + 0] = fmaf(v.x, kLog2e, x[4 * i + 0]);
              x[4 * i + 1] = fmaf(v.y, kLog2e, x[4 * i + 1]);
              x[4 * i + 2] = fmaf(v.z, kLog2e, x[4 * i + 2]);
              x[4 * i + 3] = fmaf(v.w, kLog2e, x[4 * i + 3]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (k0 + i < p.S_kv) x[i] = fmaf(__ldg(bias_row + k0 + i), kLog2e, x[i]);
          }
        }
      }
      const bool need_mask = (k0 + C::BN > p.S_kv) || (p.causal && k0 + C::BN - 1 > q0);
      if (need_mask) {
        const int lim = p.causal ? min(p.S_kv - 1, row) : p.S_kv - 1;  // last visible key
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (k0 + i > lim) x[i] = SDPA_NEG_INF;
      }
      float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
      for (int i = 4; i < 128; i += 4) {
        mx0 = fmaxf(mx0, x[i]);
        mx1 = fmaxf(mx1, x[i + 1]);
        mx2 = fmaxf(mx2, x[i + 2]);
        mx3 = fmaxf(mx3, x[i + 3]);
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      // Rescale only when the max grew by more than 8 (a factor 256).
      const bool grow = mx > m + 8.0f;
      float alpha = 1.0f;
      if (grow) {
        alpha = ex2(m - mx);  // 0 when m was -inf
        m = mx;
      }
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int c = 0; c < DV / 16; ++c) {
          uint32_t rr[16];
          tmem_ld16(tO + lane_off + c * 16, rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
          tmem_st16(tO + lane_off + c * 16, rr);
        }
      }
      l *= alpha;
      const float mu = (m == SDPA_NEG_INF) ? 0.f : m;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int i = 0; i < 128; i += 4) {
        x[i] = ex2(x[i] - mu);
        x[i + 1] = ex2(x[i + 1] - mu);
        x[i + 2] = ex2(x[i + 2] - mu);
        x[i + 3] = ex2(x[i + 3] - mu);
        s0 += x[i];
        s1 += x[i + 1];
        s2 += x[i + 2];
        s3 += x[i + 3];
      }
      l += (s0 + s1) + (s2 + s3);
      if (p.dropout) {
        const uint64_t g0 = (lin_row + k0) >> 2;
#pragma unroll
        for (int g = 0; g < 32; ++g) {
          const uint4 w = dropout_draws(g0 + g, p.seed_lo, p.seed_hi, p.offset_lo, p.offset_hi);
          if (w.x < p.drop_threshold) x[4 * g + 0] = 0.f;
          if (w.y < p.drop_threshold) x[4 * g + 1] = 0.f;
          if (w.z < p.drop_threshold) x[4 * g + 2] = 0.f;
          if (w.w < p.drop_threshold) x[4 * g + 3] = 0.f;
        }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(x[c * 32 + 2 * i], x[c * 32 + 2 * i + 1]);
        tmem_st16(tS + lane_off + c * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(FB_P));
    }
    // ---- epilogue: O / l (times 1/(1-p) under dropout), LSE = m ln2 + ln l
    if (ok && mbar_wait(bar(FB_O), 0, ec, kSiteFwdSoftmax)) {
      tc_fence_after();
      const float inv = (l > 0.f) ? (p.dropout ? p.keep_scale : 1.0f) / l : 0.f;
      uint8_t* orow = static_cast<uint8_t*>(p.o) +
                      (static_cast<size_t>(bh) * p.S_q + (row_ok ? row : 0)) * DV * 2;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tO + lane_off + c * 32, rr);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(rr[2 * i]) * inv, __uint_as_float(rr[2 * i + 1]) * inv);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (row_ok)
        p.lse[static_cast<size_t>(bh) * p.S_q + row] = (l > 0.f) ? fmaf(m, kLn2, __logf(l)) : SDPA_NEG_INF;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int DQK, int DV, bool BF16>
cudaError_t launch_fwd_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                         const FwdParams& p, cudaStream_t st) {
  using C = FwdCfg<DQK, DV>;
  auto kern = sdpa_fwd_kernel<DQK, DV, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_qt = (p.S_q + C::BM - 1) / C::BM;
  const long long grid = static_cast<long long>(n_qt) * p.B * p.H;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, st>>>(q, k, v, p);
  return cudaGetLastError();
}

}  // namespace sdpa
