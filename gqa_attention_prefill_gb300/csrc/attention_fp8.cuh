// FP8 (E4M3) Q, K, V with per-tensor scales, head dimension 64: the D = 64
// prefill design with 8-bit operands on the tensor cores.
//
//   QK^T   tcgen05.mma kind::f8f6f4, M=128, N=128, K=32 per instruction (two
//          per 64-column head); Q and K tiles are 128 rows of 64 bytes, stored
//          by TMA with the 64-byte swizzle.
//   PV     kind::f8f6f4 with P (E4M3, four per TMEM column) from TMEM and V^T
//          from shared memory: both operands K-major.  V^T tiles (64 rows of
//          128 keys) come from a transposed copy of V that fp8_vt_kernel
//          writes per query tile of the schedule (each sequence's keys start
//          on a 128-key boundary there, so every TMA box starts aligned;
//          key rows past a sequence's end are zero).
//   softmax as in the D = 64 kernel, with scale * q_scale * k_scale folded
//          into the exponent and P rounded to E4M3 (P <= 2^8 < 448);
//          O * v_scale / l in the epilogue.
// TMEM: S0 [0,128) S1 [128,256) O0 [256,320) O1 [320,384) P0 [384,416)
//       P1 [416,448).
#pragma once
#include "attention.cuh"

namespace tsk {
namespace fp8 {

constexpr uint32_t kQTile = 128 * 64;  // bytes: 128 rows x 64 E4M3
constexpr uint32_t kKTile = 128 * 64;
constexpr uint32_t kVTile = 64 * 128;  // V^T: 64 rows (d) x 128 keys
constexpr int kStages = 4;
constexpr uint32_t kSmemQ = 0;                                   // 2 buffers x 2 tiles
constexpr uint32_t kSmemKV = 4 * kQTile;                         // kStages x (K, V^T)
constexpr uint32_t kSmemEpi = kSmemKV + kStages * (kKTile + kVTile);  // 2 bf16 output tiles
constexpr uint32_t kEpiTile = 128 * 64 * 2;
constexpr uint32_t kSmemBar = kSmemEpi + 2 * kEpiTile;
constexpr uint32_t kSmemBytes = kSmemBar + 512 + 1024;
constexpr uint32_t kColS0 = 0, kColO0 = 256, kColP0 = 384;

// Barrier slots (this kernel's ring is deeper than the bf16 kernel's).
enum : int {
  kBarQFull = 0,                 // [2]
  kBarQEmpty = 2,                // [2]
  kBarKFull = 4,                 // [kStages]
  kBarVFull = 4 + kStages,       // [kStages]
  kBarKVEmpty = 4 + 2 * kStages,
  kBarSFull = 4 + 3 * kStages,   // [2]
  kBarSFree = 6 + 3 * kStages,   // [2]
  kBarPFull = 8 + 3 * kStages,   // [2]
  kBarPVDone = 10 + 3 * kStages, // [2]
  kBarDrain = 12 + 3 * kStages,  // [2]
  kBarNever = 14 + 3 * kStages,
  kNumBars = 15 + 3 * kStages
};
static_assert(8 * kNumBars + 8 <= 512, "barrier area");

// Instruction descriptor, kind::f8f6f4: E4M3 A and B, fp32 accumulation,
// both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdescQK = idesc_e4m3_f32(128, 128);
constexpr uint32_t kIdescPV = idesc_e4m3_f32(128, 64);

// Shared-memory descriptor: K-major rows of 64 bytes with the 64-byte swizzle
// (8-row groups 512 bytes apart).
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;   // leading-dimension byte offset (unused here)
  d |= (uint64_t)(512u >> 4) << 32;  // stride-dimension byte offset
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;            // swizzle mode: 64B
  return d;
}

__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Four fp32 values -> four E4M3 codes in one word (byte i = value i),
// round to nearest even, saturating.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

struct Fp8Params {
  AttnParams a;         // as the bf16 kernels (out, lse, list, ws, status, heads, window)
  const int* tile_off;  // [num_seqs + 1] query tiles before each sequence (schedule)
  float v_scale;
  // Extents checked by builds with -DTSK_DEBUG: sequences, V^T columns (keys).
  int num_seqs = 0;
  long long vt_cols = 0;
};

// Transposed V: vt[g][d][128 * i + r] = v[key r of query tile i][g][d] (zero
// past the sequence's end), for every query tile i of the schedule.
__global__ void __launch_bounds__(128)
    fp8_vt_kernel(const uint8_t* __restrict__ v, const int* __restrict__ cu,
                  const int* __restrict__ tile_off, const int* __restrict__ ws, int num_seqs,
                  int Hkv, uint8_t* __restrict__ vt, int64_t t_pad) {
  __shared__ __align__(16) uint8_t tile[128][64 + 16];
  const int i = blockIdx.x, g = blockIdx.y;
  if (i >= ws[kWsNTiles]) return;
#ifdef TSK_DEBUG
  if ((int64_t)(i + 1) * 128 > t_pad) {  // V^T too narrow for the tile list
    if (atomicCAS(const_cast<int*>(ws) + kWsStatus, 0, -9) == 0) {
      const_cast<int*>(ws)[kWsStatus + 1] = 50;
      const_cast<int*>(ws)[kWsStatus + 2] = (int)blockIdx.x;
    }
    return;
  }
#endif
  int lo = 0, hi = num_seqs - 1;  // the sequence owning tile i
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_off[mid] <= i) lo = mid;
    else hi = mid - 1;
  }
  const int s = lo;
  const int r = threadIdx.x;
  const int key = (i - tile_off[s]) * 128 + r;
  const int L = cu[s + 1] - cu[s];
  uint4 row[4] = {};
  if (key < L) {
    const uint4* src = reinterpret_cast<const uint4*>(v + ((size_t)(cu[s] + key) * Hkv + g) * 64);
#pragma unroll
    for (int c = 0; c < 4; ++c) row[c] = src[c];
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(&tile[r][16 * c]) = row[c];
  __syncthreads();
  // Thread t writes 64 keys of row d = t / 2 of the transposed tile.
  const int d = threadIdx.x >> 1, k0 = (threadIdx.x & 1) * 64;
  uint8_t* dst = vt + ((size_t)g * 64 + d) * t_pad + (size_t)i * 128 + k0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int kk = k0 + 16 * c + 4 * q;
      w[q] = (uint32_t)tile[kk][d] | ((uint32_t)tile[kk + 1][d] << 8) |
             ((uint32_t)tile[kk + 2][d] << 16) | ((uint32_t)tile[kk + 3][d] << 24);
    }
    *reinterpret_cast<uint4*>(dst + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__device__ __forceinline__ void role_producer(const Ctx& cx, const CUtensorMap* tmQ,
                                              const CUtensorMap* tmK, const CUtensorMap* tmVt,
                                              const Fp8Params& f) {
  const AttnParams& p = f.a;
  uint32_t q_iter = 0, kv_iter = 0;
  bool ok = true;
  if (p.debug_stall) ok = mbar_wait(cx.bar(kBarNever), 0, 99, p, cx.abort);
  for (int u = blockIdx.x; u < cx.total_units && ok; u += gridDim.x) {
    const Unit w = decode_unit(p, u);
    const int qb = q_iter & 1;
    if (q_iter >= 2) ok = mbar_wait(cx.bar(kBarQEmpty + qb), ((q_iter >> 1) & 1) ^ 1, 1, p, cx.abort);
    if (!ok) break;
    mbar_arrive_expect_tx(cx.bar(kBarQFull + qb), w.ntiles * kQTile);
    for (int t = 0; t < w.ntiles; ++t) {
      if (!TSK_IN_BOUNDS(p, cx.abort,
                         w.h0 + t < p.Hq && w.start + w.q0 >= 0 && w.start + w.q0 < p.q_rows, 41)) {
        ok = false;
        break;
      }
      tma_load_3d(cx.sbase + kSmemQ + (2 * qb + t) * kQTile, tmQ, cx.bar(kBarQFull + qb), 0,
                  w.h0 + t, w.start + w.q0);
    }
    if (!ok) break;
    ++q_iter;
    if (!TSK_IN_BOUNDS(p, cx.abort, w.seq >= 0 && w.seq < f.num_seqs, 47)) break;
    const int vt_tile0 = __ldg(f.tile_off + w.seq);  // the sequence's first tile in V^T
    for (int j = 0; j < w.n_kv; ++j, ++kv_iter) {
      const int s = kv_iter % kStages;
      const uint32_t k = kv_iter / kStages;
      if (k >= 1) ok = mbar_wait(cx.bar(kBarKVEmpty + s), (k - 1) & 1, 2, p, cx.abort);
      if (!ok) break;
      const int kt = w.kv_lo + j;
      const uint32_t kdst = cx.sbase + kSmemKV + s * (kKTile + kVTile);
      if (!TSK_IN_BOUNDS(p, cx.abort,
                         w.g < p.Hkv && w.start_k + kt * kTileN < p.kv_rows &&
                             (long long)(vt_tile0 + kt + 1) * 128 <= f.vt_cols,
                         42)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(cx.bar(kBarKFull + s), kKTile);
      tma_load_3d(kdst, tmK, cx.bar(kBarKFull + s), 0, w.g, w.start_k + kt * kTileN);
      mbar_arrive_expect_tx(cx.bar(kBarVFull + s), kVTile);
      tma_load_3d(kdst + kKTile, tmVt, cx.bar(kBarVFull + s), (vt_tile0 + kt) * 128, 0, w.g);
    }
  }
  for (uint32_t i = (kv_iter > kStages ? kv_iter - kStages : 0); i < kv_iter; ++i) {
    mbar_wait<true>(cx.bar(kBarKFull + i % kStages), (i / kStages) & 1, 11, p, cx.abort);
    mbar_wait<true>(cx.bar(kBarVFull + i % kStages), (i / kStages) & 1, 12, p, cx.abort);
  }
  for (uint32_t i = (q_iter > 2 ? q_iter - 2 : 0); i < q_iter; ++i)
    mbar_wait<true>(cx.bar(kBarQFull + (i & 1)), (i >> 1) & 1, 13, p, cx.abort);
}

// MMA issuer of query tile t (same protocol as the bf16 kernel).
__device__ __forceinline__ void role_mma(const Ctx& cx, const AttnParams& p, int t) {
  uint32_t q_iter = 0, kv_iter = 0, s_cnt = 0, p_cnt = 0;
  bool ok = true;
  const uint32_t d_s = cx.tmem + kColS0 + 128 * t;
  const uint32_t d_o = cx.tmem + kColO0 + 64 * t;
  const uint32_t a_p = cx.tmem + kColP0 + 32 * t;
  for (int u = blockIdx.x; u < cx.total_units && ok; u += gridDim.x) {
    const Unit w = decode_unit(p, u);
    const int qb = q_iter & 1;
    if (t >= w.ntiles) {
      kv_iter += w.n_kv;
      ++q_iter;
      continue;
    }
    const int commits = w.ntiles == 1 ? 2 : 1;
    ok = mbar_wait(cx.bar(kBarQFull + qb), (q_iter >> 1) & 1, 3, p, cx.abort);
    if (!ok) break;
    const uint32_t qaddr = cx.sbase + kSmemQ + (2 * qb + t) * kQTile;
    auto issue_s = [&](int stage) {
      const uint32_t b = cx.sbase + kSmemKV + stage * (kKTile + kVTile);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        mma_ss_f8(d_s, sdesc_sw64(qaddr + 32 * kk), sdesc_sw64(b + 32 * kk), kIdescQK,
                  kk > 0 ? 1u : 0u);
      tc_commit(cx.bar(kBarSFull + t));
      ++s_cnt;
    };
    {
      const int s0 = kv_iter % kStages;
      ok = mbar_wait(cx.bar(kBarKFull + s0), (kv_iter / kStages) & 1, 4, p, cx.abort);
      if (ok && s_cnt > 0) ok = mbar_wait(cx.bar(kBarSFree + t), (s_cnt - 1) & 1, 5, p, cx.abort);
      if (!ok) break;
      tc_fence_after();
      issue_s(s0);
    }
    for (int j = 0; j < w.n_kv && ok; ++j) {
      const uint32_t cur = kv_iter + j;
      const int sc = cur % kStages;
      if (j + 1 < w.n_kv) {
        const int sn = (cur + 1) % kStages;
        ok = mbar_wait(cx.bar(kBarKFull + sn), ((cur + 1) / kStages) & 1, 6, p, cx.abort);
        if (ok) ok = mbar_wait(cx.bar(kBarSFree + t), (s_cnt - 1) & 1, 5, p, cx.abort);
        if (!ok) break;
        tc_fence_after();
        issue_s(sn);
      }
      ok = mbar_wait(cx.bar(kBarVFull + sc), (cur / kStages) & 1, 7, p, cx.abort);
      if (ok) ok = mbar_wait(cx.bar(kBarPFull + t), p_cnt & 1, 8, p, cx.abort);
      if (!ok) break;
      tc_fence_after();
      const uint32_t vb = cx.sbase + kSmemKV + sc * (kKTile + kVTile) + kKTile;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // 32 keys per instruction
        mma_ts_f8(d_o, a_p + 8 * kk, sdesc_sw128(vb + 32 * kk), kIdescPV,
                  (j > 0 || kk > 0) ? 1u : 0u);
      tc_commit(cx.bar(kBarPVDone + t));
      ++p_cnt;
      for (int c = 0; c < commits; ++c) tc_commit(cx.bar(kBarKVEmpty + sc));
    }
    if (!ok) break;
    kv_iter += w.n_kv;
    for (int c = 0; c < commits; ++c) tc_commit(cx.bar(kBarQEmpty + qb));
    ++q_iter;
  }
  tc_commit(cx.bar(kBarDrain + t));
  mbar_wait<true>(cx.bar(kBarDrain + t), 0, 14, p, cx.abort);
}

__device__ __forceinline__ void role_softmax(const Ctx& cx, const Fp8Params& f,
                                             const CUtensorMap* tmO, int warp, int lane) {
  const AttnParams& p = f.a;
  const int t = (warp - kFirstSoftmaxWarp) >> 2;
  const int wq = warp & 3;
  const int r = wq * 32 + lane;
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const uint32_t tS = cx.tmem + lane_base + kColS0 + 128 * t;
  const uint32_t tO = cx.tmem + lane_base + kColO0 + 64 * t;
  const uint32_t tP = cx.tmem + lane_base + kColP0 + 32 * t;
  const uint32_t epi = cx.sbase + kSmemEpi + t * kEpiTile;
  const float sl2 = p.scale_log2;  // scale * q_scale * k_scale * log2(e)
  uint32_t s_cnt = 0, pv_cnt = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < cx.total_units && ok; u += gridDim.x) {
    int n_kv, kv_lo, diag0, pos;
    float m_used = -INFINITY, l = 0.f;
    {
      const Unit w = decode_unit(p, u);
      if (t >= w.ntiles) continue;
      n_kv = w.n_kv;
      kv_lo = w.kv_lo;
      diag0 = w.offset + w.q0;
      pos = diag0 + r;
      if (p.sinks) {
        if (TSK_IN_BOUNDS(p, cx.abort, w.h0 + t < p.Hq, 44))
          m_used = __ldg(p.sinks + w.h0 + t) * 1.4426950408889634f;
        l = 1.f;
      }
    }
    for (int j = 0; j < n_kv; ++j) {
      const int kt = kv_lo + j;
      ok = mbar_wait_warp(cx.bar(kBarSFull + t), s_cnt & 1, 9, p, cx.abort);
      if (!ok) break;
      ++s_cnt;
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld_32x32b_x128(tS, sr);
      tmem_wait_ld();
      reg_fence<128>(sr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(kBarSFree + t));
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      const int kbase = kt * kTileN;
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
      float alpha = 1.f;
      if (__any_sync(0xffffffffu, m_tile > m_used + kRescaleThreshold)) {
        if (m_tile > m_used) {
          alpha = ex2_approx(m_used - m_tile);
          m_used = m_tile;
        }
      }
      l *= alpha;
      const float m_use = m_used == -INFINITY ? 0.f : m_used;
      // p = 2^(s*sl2 - m) <= 2^8, rounded to E4M3 for the PV operand; row
      // sums in fp32.
      uint32_t pk[32];
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      const uint64_t negm = f2_pack(-m_use, -m_use);
      uint64_t acc2[2] = {0ull, 0ull};  // packed partial sums: one add per pair
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float x0, x1, x2, x3;
        f2_unpack(f2_fma(f2_pack(s[4 * c], s[4 * c + 1]), sl2x2, negm), x0, x1);
        f2_unpack(f2_fma(f2_pack(s[4 * c + 2], s[4 * c + 3]), sl2x2, negm), x2, x3);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
        acc2[0] = f2_add(acc2[0], f2_pack(p0, p1));
        acc2[1] = f2_add(acc2[1], f2_pack(p2, p3));
        pk[c] = pack_e4m3x4(p0, p1, p2, p3);
      }
      {
        float a0, a1, b0, b1;
        f2_unpack(acc2[0], a0, a1);
        f2_unpack(acc2[1], b0, b1);
        l += (a0 + b0) + (a1 + b1);
      }
      if (j > 0) {
        ok = mbar_wait_warp(cx.bar(kBarPVDone + t), pv_cnt & 1, 10, p, cx.abort);
        if (!ok) break;
        ++pv_cnt;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          uint32_t o[64];
          tmem_ld_32x32b_x64(tO, o);
          tmem_wait_ld();
          reg_fence<64>(o);
#pragma unroll
          for (int c = 0; c < 64; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st_32x32b_x64(tO, o);
        }
      }
      tmem_st_32x32b_x32(tP, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(kBarPFull + t));
    }
    if (!ok) break;
    // ------------------------------------------------------------ epilogue
    const int per_tile = p.Hkv * p.HP;
    const int qi = u / per_tile;
    const int4 e = ld_nc_v4_volatile(p.list + 2 * qi);  // {start, q0, kv_lo, len}
    const int g = (u - qi * per_tile) / p.HP;
    const int h = g * p.G + 2 * (u - qi * per_tile - g * p.HP) + t;
    ok = mbar_wait_warp(cx.bar(kBarPVDone + t), pv_cnt & 1, 25, p, cx.abort);
    if (!ok) break;
    ++pv_cnt;
    tc_fence_after();
    uint32_t o[64];
    tmem_ld_32x32b_x64(tO, o);
    tmem_wait_ld();
    reg_fence<64>(o);
    const float inv = f.v_scale * rcp_approx(l);
    uint32_t ob[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      float a, b;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * c]), __uint_as_float(o[2 * c + 1])),
                       f2_pack(inv, inv)),
                a, b);
      ob[c] = pack_bf16x2(a, b);
    }
    const int row = e.y + r;
    const size_t orow = (size_t)(e.x + row) * p.Hq + h;
    // (rows past the sequence's end are neither stored nor checked)
    const bool row_ok = row < e.w && TSK_IN_BOUNDS(p, cx.abort, orow < (size_t)p.q_rows * p.Hq, 45);
    if (p.lse && row_ok) p.lse[orow] = (m_used + lg2_approx(l)) * 0.69314718055994531f;
    if (e.y + wq * 32 + 32 <= e.w) {
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
      const uint32_t dst_row = epi + (uint32_t)r * 128u;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(dst_row + ((uint32_t)(c ^ (r & 7)) << 4), ob[4 * c], ob[4 * c + 1],
                     ob[4 * c + 2], ob[4 * c + 3]);
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0 && TSK_IN_BOUNDS(p, cx.abort,
                                     h < p.Hq && e.x + e.y + wq * 32 + 32 <= p.q_rows, 46)) {
        tma_store_3d(tmO, epi + (uint32_t)wq * 4096u, 0, h, e.x + e.y + wq * 32);
        bulk_commit_group();
      }
    } else if (row_ok) {
      uint4* dst = reinterpret_cast<uint4*>(p.out + orow * 64);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        dst[c] = make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
    }
    tc_fence_before();
  }
  if (lane == 0) bulk_wait_group0();
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ,
                             const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmVt,
                             const __grid_constant__ CUtensorMap tmO,
                             const __grid_constant__ Fp8Params f) {
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(cx.bar(kBarQFull + i), 1);
      mbar_init(cx.bar(kBarQEmpty + i), 2);
      mbar_init(cx.bar(kBarSFull + i), 1);
      mbar_init(cx.bar(kBarSFree + i), kSoftmaxWarpsPerTile);
      mbar_init(cx.bar(kBarPFull + i), kSoftmaxWarpsPerTile);
      mbar_init(cx.bar(kBarPVDone + i), 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(cx.bar(kBarKFull + s), 1);
      mbar_init(cx.bar(kBarVFull + s), 1);
      mbar_init(cx.bar(kBarKVEmpty + s), 2);
    }
    mbar_init(cx.bar(kBarDrain), 1);
    mbar_init(cx.bar(kBarDrain + 1), 1);
    mbar_init(cx.bar(kBarNever), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *tmem_slot;
  cx.abort = smem_u32(const_cast<int*>(abort_flag));
  cx.total_units = f.a.ws[kWsNTiles] * f.a.Hkv * f.a.HP;

  if (warp == 0 && lane == 0) fp8::role_producer(cx, &tmQ, &tmK, &tmVt, f);
  else if (warp == 1 && lane == 0) fp8::role_mma(cx, f.a, 0);
  else if (warp == 2 && lane == 0) fp8::role_mma(cx, f.a, 1);
  else if (warp >= kFirstSoftmaxWarp) fp8::role_softmax(cx, f, &tmO, warp, lane);

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(cx.tmem, kTmemCols);
  }
}

}  // namespace fp8
}  // namespace tsk
