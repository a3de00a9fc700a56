// Head dimension 128: the same persistent, warp-specialised design as the
// D = 64 kernel (units of two query heads over one 128-row query tile, GQA
// reuse of every K/V tile, one thread per query row), re-balanced for the
// doubled MMA work and the 512-column TMEM budget:
//
//   TMEM   S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512); P_t is written
//          as bf16 pairs into columns [64,128) of S_t once the softmax holds
//          S_t(j) in registers.
//   MMA    per tile t (one issuing thread each):
//            S_t(0) = Q_t K_0^T;  then for every j:
//            O_t += P_t(j) V_j   (M=128, N=128, K=128; P from TMEM, V MN-major)
//            S_t(j+1) = Q_t K_{j+1}^T  (M=128, N=128, K=128, both from smem)
//          The MMAs of one thread run in issue order, so S_t(j+1) overwrites
//          P_t(j) only after PV_t(j) has read it; and the commit that signals
//          S_t(j+1) covers PV_t(j) too, so the softmax may rescale O_t as
//          soon as it sees S_t(j+1).  The two tiles' softmax phases
//          interleave on the tensor core.
//   smem   Q 2 x 32 KB (one buffer), K/V ring 2 x (32 + 32) KB with separate
//          empty barriers for K and V, 8 x 4 KB output staging slices.
//          Every 128-row x 128-column tile is two 64-column halves of 128-byte
//          swizzled rows (one TMA box each).
//   epilogue  two passes of 64 output columns per warp through its staging
//          slice and a TMA bulk tensor store.
//   E4M3 inputs (kFp8): Q and K tiles are 128 rows of 128 E4M3 bytes (one
//          TMA box, 128-byte swizzle, in the first half of each bf16 slot),
//          QK^T is four kind::f8f6f4 MMAs (K = 32) instead of eight; V comes
//          as bf16 values (exact) from the FP8 pre-pass, and the output is
//          multiplied by p.out_scale (the value scale).
#pragma once
#include "attention.cuh"

namespace tsk {
namespace d128 {

constexpr int kD = 128;
constexpr uint32_t kHalf = 128 * 64 * 2;    // 16 KB: 128 rows x 64 columns
constexpr uint32_t kTile = 2 * kHalf;       // 32 KB
constexpr int kStagesKV = 2;
constexpr uint32_t kSmemQ = 0;                                  // 2 tiles
constexpr uint32_t kSmemKV = 2 * kTile;                         // kStagesKV x (K, V)
constexpr uint32_t kSmemEpi = kSmemKV + kStagesKV * 2 * kTile;  // 8 x 4 KB
constexpr uint32_t kSmemBar = kSmemEpi + 8 * 4096;
constexpr uint32_t kSmemBytes = kSmemBar + 512 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

constexpr uint32_t kColS0 = 0, kColO0 = 256, kColP = 64;  // P at S_t + kColP

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescQK8 = idesc_e4m3_f32(128, 128);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);

enum : int {
  kBarQFull = 0,
  kBarQEmpty = 1,
  kBarKFull = 2,    // [2]
  kBarVFull = 4,    // [2]
  kBarKEmpty = 6,   // [2]
  kBarVEmpty = 8,   // [2]
  kBarSFull = 10,   // [2] per tile: S_t(j) computed (and every earlier MMA of t)
  kBarPFull = 12,   // [2] per tile: P_t(j) in TMEM (4 softmax warps)
  kBarODone = 14,   // [2] per tile: last PV of the unit completed
  kBarDrain = 16,   // [2]
  kBarNever = 18,
  kBarTurn = 19,    // [2] tile t may run its softmax step (4 arrivals of the other tile)
  kNumBars = 21
};
static_assert(8 * kNumBars + 8 <= 512, "barrier area");

// Descriptor of an MN-major operand whose N extent spans two 64-column
// halves `lbo` bytes apart (rows of 128 bytes, 128-byte swizzle); 8-row
// groups along K are 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// TMA producer (one thread).
template <int QS, bool kFp8>
__device__ __forceinline__ void role_producer(const Ctx& cx, const CUtensorMap* tmQ,
                                              const CUtensorMap* tmK, const CUtensorMap* tmV,
                                              const AttnParams& p) {
  uint32_t q_iter = 0, k_iss = 0, v_iss = 0;  // loads issued per buffer kind
  bool ok = true;
  TSK_TL_DECL;
  if (p.debug_stall) ok = mbar_wait(cx.bar(kBarNever), 0, 99, p, cx.abort);
  for (int ku = 0, u = cx.unit(0); u < cx.total_units && ok; u = cx.unit(++ku)) {
    const Unit w = decode_unit<QS>(p, u);
    if (q_iter >= 1) ok = mbar_wait(cx.bar(kBarQEmpty), (q_iter - 1) & 1, 1, p, cx.abort);
    if (!ok) break;
    mbar_arrive_expect_tx(cx.bar(kBarQFull), w.ntiles * (kFp8 ? kHalf : kTile));
    for (int t = 0; t < w.ntiles && ok; ++t) {
      const int h = tile_head<QS>(w, t), row = w.start + tile_q0<QS>(w, t);
      if (!TSK_IN_BOUNDS(p, cx.abort, h >= 0 && h < p.Hq && row >= 0 && row < p.q_rows, 41)) {
        ok = false;
        break;
      }
      for (int hf = 0; hf < (kFp8 ? 1 : 2); ++hf)
        tma_load_3d(cx.sbase + kSmemQ + t * kTile + hf * kHalf, tmQ, cx.bar(kBarQFull), 64 * hf,
                    h, row);
    }
    if (!ok) break;
    TSK_EV(20);
    ++q_iter;
    for (int j = 0; j < w.n_kv && ok; ++j) {
      const int pos0 = (w.kv_lo + j) * kTileN;  // key position of the tile's first key
      const int Lk = w.offset + w.len;
      {
        const int s = k_iss % kStagesKV;
        const uint32_t k = k_iss / kStagesKV;
        if (k >= 1) ok = mbar_wait(cx.bar(kBarKEmpty + s), (k - 1) & 1, 2, p, cx.abort);
        if (!ok) break;
        const uint32_t dst = cx.sbase + kSmemKV + s * 2 * kTile;
        if (!TSK_IN_BOUNDS(p, cx.abort,
                           w.g >= 0 && w.g < p.Hkv &&
                               (p.kv.page_size != 0 ||
                                (w.start_k + pos0 >= 0 && w.start_k + pos0 < p.kv_rows)),
                           42)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(cx.bar(kBarKFull + s), kFp8 ? kHalf : kTile);
        bool in = true;
        for (int hf = 0; hf < (kFp8 ? 1 : 2); ++hf)
          in = tma_load_key_rows(dst + hf * kHalf, tmK, cx.bar(kBarKFull + s), 64 * hf, w.g,
                                 p.kv, w.seq, w.start_k, pos0, Lk) && in;
        if (!TSK_IN_BOUNDS(p, cx.abort, in, 43)) {
          ok = false;
          break;
        }
        TSK_EV(21);
        ++k_iss;
      }
      {
        const int s = v_iss % kStagesKV;
        const uint32_t k = v_iss / kStagesKV;
        if (k >= 1) ok = mbar_wait(cx.bar(kBarVEmpty + s), (k - 1) & 1, 2, p, cx.abort);
        if (!ok) break;
        const uint32_t dst = cx.sbase + kSmemKV + s * 2 * kTile + kTile;
        mbar_arrive_expect_tx(cx.bar(kBarVFull + s), kTile);
        bool in = true;
        for (int hf = 0; hf < 2; ++hf)
          in = tma_load_key_rows(dst + hf * kHalf, tmV, cx.bar(kBarVFull + s), 64 * hf, w.g,
                                 p.kv, w.seq, w.start_k, pos0, Lk) && in;
        if (!TSK_IN_BOUNDS(p, cx.abort, in, 43)) {
          ok = false;
          break;
        }
        TSK_EV(22);
        ++v_iss;
      }
    }
  }
  // Drain: the last loads issued into every buffer (bounded, best effort).
  for (uint32_t i = (k_iss > kStagesKV ? k_iss - kStagesKV : 0); i < k_iss; ++i)
    mbar_wait<true>(cx.bar(kBarKFull + i % kStagesKV), (i / kStagesKV) & 1, 11, p, cx.abort);
  for (uint32_t i = (v_iss > kStagesKV ? v_iss - kStagesKV : 0); i < v_iss; ++i)
    mbar_wait<true>(cx.bar(kBarVFull + i % kStagesKV), (i / kStagesKV) & 1, 12, p, cx.abort);
  if (q_iter >= 1) mbar_wait<true>(cx.bar(kBarQFull), (q_iter - 1) & 1, 13, p, cx.abort);
}

// tcgen05.mma issuer for query tile t (one thread).  The release barriers
// (Q, K and V buffers) count one arrival per tile; in a unit with a single
// query tile the tile-1 issuer follows the fills and arrives without MMAs.
template <int QS, bool kFp8>
__device__ __forceinline__ void role_mma(const Ctx& cx, const AttnParams& p, int t) {
  uint32_t q_iter = 0, kv_iter = 0, p_cnt = 0;
  bool ok = true;
  TSK_TL_DECL;
  const uint32_t d_s = cx.tmem + kColS0 + 128 * t;
  const uint32_t d_o = cx.tmem + kColO0 + 128 * t;
  const uint32_t a_p = d_s + kColP;
  const uint32_t q_addr = cx.sbase + kSmemQ + t * kTile;
  for (int ku = 0, u = cx.unit(0); u < cx.total_units && ok; u = cx.unit(++ku)) {
    const Unit w = decode_unit<QS>(p, u);
    if (t >= w.ntiles) {
      // Idle in the unit: follow its Q and K/V fills and release them with
      // plain arrivals, so that no fill is replaced before both issuers have
      // seen it (no barrier runs two phases ahead of this thread).
      ok = mbar_wait(cx.bar(kBarQFull), q_iter & 1, 3, p, cx.abort);
      for (int j = 0; j < w.n_kv && ok; ++j) {
        const uint32_t cur = kv_iter + j;
        const int sc = cur % kStagesKV;
        ok = mbar_wait(cx.bar(kBarKFull + sc), (cur / kStagesKV) & 1, 4, p, cx.abort);
        if (ok) mbar_arrive(cx.bar(kBarKEmpty + sc));
        if (ok) ok = mbar_wait(cx.bar(kBarVFull + sc), (cur / kStagesKV) & 1, 7, p, cx.abort);
        if (ok) mbar_arrive(cx.bar(kBarVEmpty + sc));
      }
      if (!ok) break;
      mbar_arrive(cx.bar(kBarQEmpty));
      kv_iter += w.n_kv;
      ++q_iter;
      continue;
    }
    auto release = [&](int bar) { tc_commit(cx.bar(bar)); };
    auto issue_qk = [&](uint32_t it) {
      const int s = it % kStagesKV;
      const uint32_t kb = cx.sbase + kSmemKV + s * 2 * kTile;
      TSK_TRACE_T0(tr_is);
      if constexpr (kFp8) {
#pragma unroll
        for (int kk = 0; kk < kD / 32; ++kk)  // 32 E4M3 bytes per instruction
          mma_ss_f8(d_s, sdesc_sw128(q_addr + 32 * kk), sdesc_sw128(kb + 32 * kk), kIdescQK8,
                    kk > 0 ? 1u : 0u);
      } else {
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + 32 * (kk & 3);
          mma_ss(d_s, sdesc_sw128(q_addr + off), sdesc_sw128(kb + off), kIdescQK,
                 kk > 0 ? 1u : 0u);
        }
      }
      tc_commit(cx.bar(kBarSFull + t));
      release(kBarKEmpty + s);
      TSK_TRACE_ADD(18, tr_is);
      TSK_EV(12);
    };
    TSK_EV(13);
    ok = mbar_wait(cx.bar(kBarQFull), q_iter & 1, 3, p, cx.abort);
    if (ok) ok = mbar_wait(cx.bar(kBarKFull + kv_iter % kStagesKV), (kv_iter / kStagesKV) & 1, 4, p, cx.abort);
    if (!ok) break;
    tc_fence_after();
    issue_qk(kv_iter);
    if (w.n_kv == 1) release(kBarQEmpty);
    for (int j = 0; j < w.n_kv && ok; ++j) {
      const uint32_t cur = kv_iter + j;
      const int sc = cur % kStagesKV;
      ok = mbar_wait(cx.bar(kBarVFull + sc), (cur / kStagesKV) & 1, 7, p, cx.abort);
      if (ok) ok = mbar_wait(cx.bar(kBarPFull + t), p_cnt & 1, 8, p, cx.abort);
      if (!ok) break;
      ++p_cnt;
      TSK_EV(10);
      tc_fence_after();
      const uint32_t vb = cx.sbase + kSmemKV + sc * 2 * kTile + kTile;
      TSK_TRACE_T0(tr_ip);
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        mma_ts(d_o, a_p + 8 * kk, sdesc_sw128_mn(vb + 2048 * kk, kHalf), kIdescPV,
               (j > 0 || kk > 0) ? 1u : 0u);
      release(kBarVEmpty + sc);
      TSK_TRACE_ADD(19, tr_ip);
      TSK_EV(11);
      if (j + 1 < w.n_kv) {
        ok = mbar_wait(cx.bar(kBarKFull + (cur + 1) % kStagesKV), ((cur + 1) / kStagesKV) & 1, 6,
                       p, cx.abort);
        if (!ok) break;
        tc_fence_after();
        issue_qk(cur + 1);
        if (j + 2 == w.n_kv) release(kBarQEmpty);
      } else {
        tc_commit(cx.bar(kBarODone + t));
      }
    }
    if (!ok) break;
    kv_iter += w.n_kv;
    ++q_iter;
  }
  tc_commit(cx.bar(kBarDrain + t));
  mbar_wait<true>(cx.bar(kBarDrain + t), 0, 14, p, cx.abort);
}

// Softmax and epilogue of query tile t (one warpgroup, one thread per row).
template <int QS, bool kFp8>
__device__ __forceinline__ void role_softmax(const Ctx& cx, const AttnParams& p,
                                             const CUtensorMap* tmO, int warp, int lane) {
  const int t = (warp - kFirstSoftmaxWarp) >> 2;
  const int wq = warp & 3;
  const int r = wq * 32 + lane;
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const uint32_t tS = cx.tmem + lane_base + kColS0 + 128 * t;
  const uint32_t tO = cx.tmem + lane_base + kColO0 + 128 * t;
  const uint32_t slice = cx.sbase + kSmemEpi + (uint32_t)(4 * t + wq) * 4096u;
  const float sl2 = p.scale_log2;
  uint32_t s_cnt = 0, o_cnt = 0;
  uint32_t turn = 0;  // softmax steps taken in units with two query tiles
  bool ok = true;
  TSK_TL_DECL;
  for (int ku = 0, u = cx.unit(0); u < cx.total_units && ok; u = cx.unit(++ku)) {
    TSK_EV(7);
    int n_kv, kv_lo, diag0, pos;
    bool pair;  // two query tiles: their softmax steps alternate
    float m_used = -INFINITY, l = 0.f;
    {
      const Unit w = decode_unit<QS>(p, u);
      if (t >= w.ntiles) continue;
      pair = w.ntiles == 2;
      n_kv = w.n_kv;
      kv_lo = w.kv_lo;
      diag0 = w.offset + tile_q0<QS>(w, t);
      pos = diag0 + r;
      if (p.sinks) {
        if (TSK_IN_BOUNDS(p, cx.abort, tile_head<QS>(w, t) >= 0 && tile_head<QS>(w, t) < p.Hq, 44))
          m_used = __ldg(p.sinks + tile_head<QS>(w, t)) * 1.4426950408889634f;
        l = 1.f;
      }
    }
    for (int j = 0; j < n_kv; ++j) {
      ok = mbar_wait_warp(cx.bar(kBarSFull + t), s_cnt & 1, 9, p, cx.abort);
      if (!ok) break;
      ++s_cnt;
      TSK_EV(1);
      // Tiles take turns (the two warps of a sub-partition never run their
      // softmax at the same time): tile 1's step k follows tile 0's step k,
      // tile 0's step k+1 follows tile 1's step k.
      if (pair && (t == 1 || turn > 0)) {
        ok = mbar_wait_warp(cx.bar(kBarTurn + t), (t == 1 ? turn : turn - 1) & 1, 17, p, cx.abort);
        if (!ok) break;
      }
      TSK_EV(2);
      tc_fence_after();
      TSK_TRACE_T0(tr_ld);
      uint32_t sr[128];
      tmem_ld_32x32b_x32(tS + 0, sr + 0);
      tmem_ld_32x32b_x32(tS + 32, sr + 32);
      tmem_ld_32x32b_x32(tS + 64, sr + 64);
      tmem_ld_32x32b_x32(tS + 96, sr + 96);
      tmem_wait_ld();
      reg_fence<128>(sr);
      TSK_TRACE_ADD(20, tr_ld);
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      const int kbase = (kv_lo + j) * kTileN;
      TSK_TRACE_T0(tr_max);
      const bool edge = (kbase + kTileN - 1 > diag0) ||
                        (p.window > 0 && kbase < diag0 + kTileM - p.window);
      if (edge) {
        const ChunkMask cm = classify_chunks(diag0 + wq * 32, kbase, p.window);
        const int hi_c = pos - kbase;
        const int lo_c = p.window > 0 ? pos - p.window + 1 - kbase : -1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (cm.partial & (1u << k)) {
#pragma unroll
            for (int c = 32 * k; c < 32 * k + 32; ++c)
              s[c] = (c > hi_c || c < lo_c) ? -INFINITY : s[c];
          } else if (cm.none & (1u << k)) {
#pragma unroll
            for (int c = 32 * k; c < 32 * k + 32; ++c) s[c] = -INFINITY;
          }
        }
      }
      float m0 = s[0], m1 = s[1], m2 = s[2], m3 = s[3];
#pragma unroll
      for (int c = 4; c < 128; c += 8) {
        m0 = max3f(m0, s[c + 0], s[c + 1]);
        m1 = max3f(m1, s[c + 2], s[c + 3]);
        m2 = max3f(m2, s[c + 4], s[c + 5]);
        m3 = max3f(m3, s[c + 6], s[c + 7]);
      }
      const float m_tile = max3f(m0, m1, fmaxf(m2, m3)) * sl2;
      TSK_TRACE_ADD(21, tr_max);
      float alpha = 1.f;
      if (__any_sync(0xffffffffu, m_tile > m_used + kRescaleThreshold)) {
        if (m_tile > m_used) {
          alpha = ex2_approx(m_used - m_tile);  // m_used = -inf gives 0
          m_used = m_tile;
        }
      }
      l *= alpha;
      const float m_use = m_used == -INFINITY ? 0.f : m_used;
      TSK_TRACE_T0(tr_exp);
      uint32_t pk[64];
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      const uint64_t negm = f2_pack(-m_use, -m_use);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), sl2x2, negm), x0, x1);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        acc[c & 3] += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l += (acc[0] + acc[1]) + (acc[2] + acc[3]);
      TSK_TRACE_ADD(22, tr_exp);
      TSK_EV(3);
      // O_t is stable (the commit behind S_t(j) covers PV_t(j-1)); rescaled
      // after the exponentials, when the scores no longer occupy registers.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int hc = 0; hc < 4; ++hc) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tO + 32 * hc, o);
          tmem_wait_ld();
          reg_fence<32>(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st_32x32b_x32(tO + 32 * hc, o);
        }
      }
      TSK_TRACE_T0(tr_st);
      tmem_st_32x32b_x32(tS + kColP, pk);
      tmem_st_32x32b_x32(tS + kColP + 32, pk + 32);
      tmem_wait_st();
      TSK_TRACE_ADD(23, tr_st);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(cx.bar(kBarPFull + t));
        if (pair) mbar_arrive(cx.bar(kBarTurn + (t ^ 1)));
      }
      if (pair) ++turn;
      TSK_EV(4);
    }
    if (!ok) break;
    // ------------------------------------------------------------ epilogue
    const int per_tile = p.Hkv * p.HP;
    const int qi = u / per_tile;
    int4 e = ld_nc_v4_volatile(p.list + 2 * qi);  // {start, q0, kv_lo, len}
    const int g = (u - qi * per_tile) / p.HP;
    int h;
    if constexpr (QS != 0) {
      h = g * p.G;
      e.y += t * QS;  // first query row of this tile
    } else {
      h = g * p.G + 2 * (u - qi * per_tile - g * p.HP) + t;
    }
    ok = mbar_wait_warp(cx.bar(kBarODone + t), o_cnt & 1, 25, p, cx.abort);
    if (!ok) break;
    ++o_cnt;
    tc_fence_after();
    TSK_EV(5);
    TSK_TRACE_T0(tr_epi);
    const int row = e.y + r;
    const size_t orow = (size_t)(e.x + row) * p.Hq + h;
    // (rows past the sequence's end are neither stored nor checked)
    const bool row_ok = row < e.w && TSK_IN_BOUNDS(p, cx.abort, orow < (size_t)p.q_rows * p.Hq, 45);
    if (p.lse && row_ok) p.lse[orow] = (m_used + log2f(l)) * 0.69314718055994531f;
    float inv = rcp_approx(l);
    if constexpr (kFp8) inv *= p.out_scale;
    const bool staged = e.y + wq * 32 + 32 <= e.w;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t o[64];
      tmem_ld_32x32b_x32(tO + 64 * hf, o);
      tmem_ld_32x32b_x32(tO + 64 * hf + 32, o + 32);
      tmem_wait_ld();
      reg_fence<64>(o);
      uint32_t ob[32];
#pragma unroll
      for (int c = 0; c < 32; ++c)
        ob[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
      if (staged) {
        if (lane == 0) bulk_wait_group_read0();  // the previous store has read the slice
        __syncwarp();
        const uint32_t dst_row = slice + (uint32_t)lane * 128u;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_v4(dst_row + ((uint32_t)(c ^ (lane & 7)) << 4), ob[4 * c], ob[4 * c + 1],
                       ob[4 * c + 2], ob[4 * c + 3]);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0 && TSK_IN_BOUNDS(p, cx.abort,
                                       h < p.Hq && e.x + e.y + wq * 32 + 32 <= p.q_rows, 46)) {
          tma_store_3d(tmO, slice, 64 * hf, h, e.x + e.y + wq * 32);
          bulk_commit_group();
        }
      } else if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kD + 64 * hf);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          dst[c] = make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
      }
    }
    tc_fence_before();
    TSK_TRACE_ADD(28, tr_epi);
    TSK_EV(6);
  }
  if (lane == 0) bulk_wait_group0();  // every output store of this warp has completed
}

template <int QS, bool kFp8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    attention_fwd_d128_kernel(const __grid_constant__ CUtensorMap tmQ,
                              const __grid_constant__ CUtensorMap tmK,
                              const __grid_constant__ CUtensorMap tmV,
                              const __grid_constant__ CUtensorMap tmO,
                              const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Ctx cx;
  cx.sbase = smem_u32(smem);
  cx.bar0 = cx.sbase + kSmemBar;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemBar + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemBar + 8 * kNumBars + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(cx.bar(kBarQFull), 1);
    mbar_init(cx.bar(kBarQEmpty), 2);
    for (int s = 0; s < kStagesKV; ++s) {
      mbar_init(cx.bar(kBarKFull + s), 1);
      mbar_init(cx.bar(kBarVFull + s), 1);
      mbar_init(cx.bar(kBarKEmpty + s), 2);
      mbar_init(cx.bar(kBarVEmpty + s), 2);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(cx.bar(kBarSFull + i), 1);
      mbar_init(cx.bar(kBarPFull + i), kSoftmaxWarpsPerTile);
      mbar_init(cx.bar(kBarODone + i), 1);
      mbar_init(cx.bar(kBarDrain + i), 1);
    }
    mbar_init(cx.bar(kBarNever), 1);
    mbar_init(cx.bar(kBarTurn), kSoftmaxWarpsPerTile);
    mbar_init(cx.bar(kBarTurn + 1), kSoftmaxWarpsPerTile);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  trace_init();
  trace_cta_start();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *tmem_slot;
  cx.abort = smem_u32(const_cast<int*>(abort_flag));
  cx.total_units = p.ws[kWsNTiles] * p.Hkv * p.HP;
  cx.alternate = false;

  // Registers move from the producer/MMA warpgroup (96 each) to the softmax
  // warpgroups (200 each): 128 x 96 + 256 x 200 = 63,488 <= 384 x 168, the
  // launch's total.  (The split was chosen by measurement: the code ptxas
  // generates for the roles, and with it the step time, varies by up to 20%
  // between neighbouring splits.)
  if (warp < kFirstSoftmaxWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 96;");
    if (warp == 0 && lane == 0) d128::role_producer<QS, kFp8>(cx, &tmQ, &tmK, &tmV, p);
    else if (warp == 1 && lane == 0) d128::role_mma<QS, kFp8>(cx, p, 0);
    else if (warp == 2 && lane == 0) d128::role_mma<QS, kFp8>(cx, p, 1);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 200;");
    d128::role_softmax<QS, kFp8>(cx, p, &tmO, warp, lane);
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(cx.tmem, kTmemCols);
  }
  trace_flush();
  trace_cta_time();
}

}  // namespace d128
}  // namespace tsk
