// FP8 (E4M3) Q, K, V with per-tensor scales, head dimension 64.
//
//   QK^T   tcgen05.mma kind::f8f6f4, M=128, N=128, K=32 per instruction (two
//          per 64-column head): half the instructions and half the operand
//          bytes of the bf16 kernel's QK^T.  Q and K tiles are 128 rows of 64
//          bytes, stored by TMA with the 64-byte swizzle.
//   PV     kind::f16 exactly as in the bf16 kernel: P in bf16 from TMEM, V
//          from a bf16 copy of the E4M3 values that fp8_prep_kernel writes
//          (exact: an E4M3 value has at most four significant bits); v_scale
//          is applied in the epilogue.
//   softmax  the bf16 kernel's (role_softmax_causal) with scale * q_scale *
//          k_scale folded into the exponent, including its key-norm bound
//          (the norms of the E4M3 key rows come from fp8_prep_kernel too), so
//          the probabilities are bf16 and tiles may skip their row maximum.
// TMEM columns and mbarriers as in the bf16 kernel.
#pragma once
#include <cuda_fp16.h>

#include "attention.cuh"

namespace tsk {
namespace fp8 {

constexpr uint32_t kQTile = 128 * 64;  // bytes: 128 rows x 64 E4M3
constexpr uint32_t kKTile = 128 * 64;
constexpr uint32_t kVTile = kTileBytes;  // bf16 V: 128 rows x 128 bytes
constexpr uint32_t kStageBytes = kKTile + kVTile;
constexpr uint32_t kSmemQ = 0;                                   // 2 buffers x 2 tiles
constexpr uint32_t kSmemKV = 4 * kQTile;                         // kStages x (K, V)
constexpr uint32_t kSmemBar = kSmemKV + kStages * kStageBytes;   // barriers (< 512 B)
constexpr uint32_t kSmemEpi = kSmemBar + 1024;                   // 2 bf16 output tiles
constexpr uint32_t kSmemNorm = kSmemEpi + 2 * kTileBytes;        // key-norm bound per KV head
constexpr uint32_t kSmemBytes = kSmemNorm + 4 * kNormMaxHeads + 1024;

constexpr uint32_t kIdescQK = idesc_e4m3_f32(128, 128);

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

// The four E4M3 codes of w (byte i = element i) as floats, exactly (E4M3 ->
// f16 is exact; f16 -> f32 too).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float& x0, float& x1, float& x2,
                                              float& x3) {
  uint32_t h01, h23;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"((unsigned short)(w & 0xFFFFu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"((unsigned short)(w >> 16)));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h23));
  x0 = a.x;
  x1 = a.y;
  x2 = b.x;
  x3 = b.y;
}

// The E4M3 query tile: rows of 64 bytes, each within its own 64 bytes under the
// 64-byte swizzle (only the order of its four 16-byte chunks changes).
struct Layout {
  static constexpr uint32_t kQ = kSmemQ, kQTile = fp8::kQTile, kEpi = kSmemEpi, kNorm = kSmemNorm;
  static constexpr bool kScaleOut = true;  // (v_scale)
  static __device__ __forceinline__ float q_sq(uint32_t tile, int r) {
    const uint32_t qrow = tile + (uint32_t)r * 64u;
    float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = ld_shared_v4(qrow + 16u * (uint32_t)((k + (r >> 1)) & 3));
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x0, x1, x2, x3;
        e4m3x4_to_f32(wv[e], x0, x1, x2, x3);
        ss[0] = fmaf(x0, x0, ss[0]);
        ss[1] = fmaf(x1, x1, ss[1]);
        ss[2] = fmaf(x2, x2, ss[2]);
        ss[3] = fmaf(x3, x3, ss[3]);
      }
    }
    return (ss[0] + ss[1]) + (ss[2] + ss[3]);
  }
};

// V as bf16 ([rows, Hkv, D], rows = tokens; chunks_per_row = D / 16) and, if
// norms (D = 64), the per-KV-head maxima of the E4M3 key-row norms, in one
// pass: four threads per 64-byte key row, 16 codes each.
// The per-block maxima and the last block's reduction use the key-norm buffer
// and counter of the bf16 path (kn.out, ws[kWsNormCount]); with more than
// kNormMaxHeads KV heads only V is converted (the kernel then has no bound).
__global__ void __launch_bounds__(kSchedThreads, 1)
    fp8_prep_kernel(const uint8_t* __restrict__ k8, const uint8_t* __restrict__ v8,
                    long long rows, int heads, int chunks_per_row, bool norms,
                    uint4* __restrict__ vb, float* __restrict__ norm_out, int* __restrict__ ws) {
  __shared__ int s_max[kNormMaxHeads];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  const int blk = blockIdx.x, nblk = gridDim.x;
  // (norms: 64-byte key rows, at most kNormMaxHeads heads)
  for (int g = tid; g < heads && norms; g += kSchedThreads) s_max[g] = 0;
  __syncthreads();
  const long long total = rows * heads * chunks_per_row;  // 16-byte chunks
  const long long stride = (long long)nblk * kSchedThreads;
  const unsigned group = 0xFu << (tid & 28);  // the 4 lanes sharing this thread's row
  for (long long i = (long long)blk * kSchedThreads + tid; i < total; i += stride) {
    const uint4 kv = norms ? __ldg(reinterpret_cast<const uint4*>(k8) + i) : make_uint4(0, 0, 0, 0);
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(v8) + i);
    const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w}, vw[4] = {vv.x, vv.y, vv.z, vv.w};
    uint32_t ob[8];
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v0, v1, v2, v3;
      e4m3x4_to_f32(vw[e], v0, v1, v2, v3);
      ob[2 * e] = pack_bf16x2(v0, v1);  // (exact: at most four significant bits)
      ob[2 * e + 1] = pack_bf16x2(v2, v3);
      if (norms) {
        float k0, k1, k2, k3;
        e4m3x4_to_f32(kw[e], k0, k1, k2, k3);
        acc = fmaf(k0, k0, fmaf(k1, k1, fmaf(k2, k2, fmaf(k3, k3, acc))));
      }
    }
    vb[2 * i] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
    vb[2 * i + 1] = make_uint4(ob[4], ob[5], ob[6], ob[7]);
    if (!norms) continue;
    acc += __shfl_xor_sync(group, acc, 1);
    acc += __shfl_xor_sync(group, acc, 2);
    if ((tid & 3) == 0)  // (row index < 2^31: the host bounds tokens x heads)
      atomicMax(&s_max[(unsigned)(i >> 2) % (unsigned)heads], __float_as_int(sqrtf(acc)));
  }
  if (!norms) return;
  __syncthreads();
  for (int g = tid; g < heads; g += kSchedThreads)
    norm_out[blk * kNormMaxHeads + g] = __int_as_float(s_max[g]);
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&ws[kWsNormCount], 1) == nblk - 1;
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int g = tid; g < heads; g += kSchedThreads) s_max[g] = 0;
    __syncthreads();
    for (int i = tid; i < nblk * heads; i += kSchedThreads) {
      const int b = i / heads, g = i - b * heads;
      atomicMax(&s_max[g], __float_as_int(__ldcg(norm_out + b * kNormMaxHeads + g)));
    }
    __syncthreads();
    for (int g = tid; g < heads; g += kSchedThreads)
      norm_out[kNormBlocks * kNormMaxHeads + g] = __int_as_float(s_max[g]);
    if (tid == 0) ws[kWsNormCount] = 0;
  }
}

struct Fp8Params {
  AttnParams a;  // as the bf16 kernels (out, lse, list, ws, status, heads, window, knorm)
  float v_scale;
};

__device__ __forceinline__ void role_producer(const Ctx& cx, const CUtensorMap* tmQ,
                                              const CUtensorMap* tmK, const CUtensorMap* tmV,
                                              const AttnParams& p) {
  uint32_t q_iter = 0, kv_iter = 0;
  bool ok = true;
  if (p.debug_stall) ok = mbar_wait(cx.bar(kBarNever), 0, 99, p, cx.abort);
  for (int ku = 0, u = cx.unit(0); u < cx.total_units && ok; u = cx.unit(++ku)) {
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
    for (int j = 0; j < w.n_kv; ++j, ++kv_iter) {
      const int s = kv_iter % kStages;
      const uint32_t k = kv_iter / kStages;
      if (k >= 1) ok = mbar_wait(cx.bar(kBarKVEmpty + s), (k - 1) & 1, 2, p, cx.abort);
      if (!ok) break;
      const int row = w.start_k + (w.kv_lo + j) * kTileN;
      const uint32_t kdst = cx.sbase + kSmemKV + s * kStageBytes;
      if (!TSK_IN_BOUNDS(p, cx.abort, w.g < p.Hkv && row >= 0 && row < p.kv_rows, 42)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(cx.bar(kBarKFull + s), kKTile);
      tma_load_3d(kdst, tmK, cx.bar(kBarKFull + s), 0, w.g, row);
      mbar_arrive_expect_tx(cx.bar(kBarVFull + s), kVTile);
      tma_load_3d(kdst + kKTile, tmV, cx.bar(kBarVFull + s), 0, w.g, row);
    }
  }
  for (uint32_t i = (kv_iter > kStages ? kv_iter - kStages : 0); i < kv_iter; ++i) {
    mbar_wait<true>(cx.bar(kBarKFull + i % kStages), (i / kStages) & 1, 11, p, cx.abort);
    mbar_wait<true>(cx.bar(kBarVFull + i % kStages), (i / kStages) & 1, 12, p, cx.abort);
  }
  for (uint32_t i = (q_iter > 2 ? q_iter - 2 : 0); i < q_iter; ++i)
    mbar_wait<true>(cx.bar(kBarQFull + (i & 1)), (i >> 1) & 1, 13, p, cx.abort);
}

// MMA issuer of query tile t (the bf16 kernel's protocol and order).
__device__ __forceinline__ void role_mma(const Ctx& cx, const AttnParams& p, int t) {
  uint32_t q_iter = 0, kv_iter = 0, s_cnt = 0, p_cnt = 0;
  bool ok = true;
  const uint32_t d_s = cx.tmem + kColS0 + 128 * t;
  const uint32_t d_o = cx.tmem + kColO0 + 64 * t;
  const uint32_t a_p = cx.tmem + kColP0 + 64 * t;
  for (int ku = 0, u = cx.unit(0); u < cx.total_units && ok; u = cx.unit(++ku)) {
    const Unit w = decode_unit(p, u);
    const int qb = q_iter & 1;
    ok = mbar_wait(cx.bar(kBarQFull + qb), (q_iter >> 1) & 1, 3, p, cx.abort);
    if (!ok) break;
    if (t >= w.ntiles) {
      // idle in the unit: follow and release its K/V fills and its Q buffer
      for (int j = 0; j < w.n_kv && ok; ++j) {
        const uint32_t cur = kv_iter + j;
        const int sc = cur % kStages;
        ok = mbar_wait(cx.bar(kBarKFull + sc), (cur / kStages) & 1, 4, p, cx.abort);
        if (ok) ok = mbar_wait(cx.bar(kBarVFull + sc), (cur / kStages) & 1, 7, p, cx.abort);
        if (ok) mbar_arrive(cx.bar(kBarKVEmpty + sc));
      }
      if (!ok) break;
      mbar_arrive(cx.bar(kBarQEmpty + qb));
      kv_iter += w.n_kv;
      ++q_iter;
      continue;
    }
    const uint32_t qaddr = cx.sbase + kSmemQ + (2 * qb + t) * kQTile;
    auto issue_s = [&](int stage) {
      const uint32_t b = cx.sbase + kSmemKV + stage * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)  // 32 E4M3 elements per instruction
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
      const uint32_t vb = cx.sbase + kSmemKV + sc * kStageBytes + kKTile;
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        mma_ts(d_o, a_p + 8 * kk, sdesc_sw128(vb + 2048 * kk), kIdescPV,
               (j > 0 || kk > 0) ? 1u : 0u);
      tc_commit(cx.bar(kBarPVDone + t));
      ++p_cnt;
      tc_commit(cx.bar(kBarKVEmpty + sc));
    }
    if (!ok) break;
    kv_iter += w.n_kv;
    tc_commit(cx.bar(kBarQEmpty + qb));
    ++q_iter;
  }
  tc_commit(cx.bar(kBarDrain + t));
  mbar_wait<true>(cx.bar(kBarDrain + t), 0, 14, p, cx.abort);
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ,
                             const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV,
                             const __grid_constant__ CUtensorMap tmO,
                             const __grid_constant__ Fp8Params f) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const AttnParams& p = f.a;
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
      mbar_init(cx.bar(kBarQEmpty + i), 2 + 2 * kSoftmaxWarpsPerTile);  // issuers and softmax warps
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
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 3 && p.knorm)
    for (int g = lane; g < p.Hkv; g += 32) st_shared_f32(cx.sbase + kSmemNorm + 4u * g, __ldg(p.knorm + g));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *tmem_slot;
  cx.abort = smem_u32(const_cast<int*>(abort_flag));
  cx.total_units = p.ws[kWsNTiles] * p.Hkv * p.HP;
  cx.alternate = true;

  if (warp == 0 && lane == 0) fp8::role_producer(cx, &tmQ, &tmK, &tmV, p);
  else if (warp == 1 && lane == 0) fp8::role_mma(cx, p, 0);
  else if (warp == 2 && lane == 0) fp8::role_mma(cx, p, 1);
  else if (warp >= kFirstSoftmaxWarp)
    role_softmax_causal<0, Layout>(cx, p, &tmO, warp, lane, f.v_scale);

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
