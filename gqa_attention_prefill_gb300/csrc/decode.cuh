// Decode over a key/value cache: one new query token per sequence, at key
// position Lk - 1 (its own key is the last one in the cache), attending to
// key positions max(0, Lk - W) .. Lk - 1 with the sink of its head.
//
// The work is a stream over the cache (about 4 FLOP per byte for 8 query
// heads per KV head): the kernels are laid out for HBM bandwidth.
//   decode_check_kernel   validates cu_seqlens_k and clears the split counters
//                         (1 CTA)
//   decode_split_kernel   one CTA per (key split, KV head, block of <= 16 query
//                         heads of that KV head, sequence); 4 warps.  One thread
//                         streams 128-key K and V tiles into a 3-stage
//                         shared-memory ring with TMA (the prefill tensor maps);
//                         each warp takes 32 keys of every tile: S = Q K^T and
//                         O += P V are 16 x 8 x 16 warp MMAs (the query heads
//                         of the block are the 16 rows, padded with zeros), with
//                         an online base-2 softmax per row.  The four warps'
//                         states are merged in shared memory and the split's
//                         (m, l, O) written to a workspace.  The last CTA of a
//                         (sequence, KV head, head block) to finish (an atomic
//                         counter per triple) combines the splits' states and
//                         the sink (counted once) and writes bf16 out and the
//                         natural-log LSE.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"
#include "attention.cuh"

namespace tsk {
namespace dec {

constexpr int kThreads = 128;   // 4 warps
constexpr int kKeys = 128;      // keys per staged tile
constexpr int kRows = 16;       // query heads per CTA (MMA rows)

struct DecParams {
  const __nv_bfloat16* q;   // [num_seqs, Hq, D]
  const float* sinks;       // [Hq] or nullptr
  const int* cu_k;          // [num_seqs + 1]
  float* part;              // [splits][num_seqs][Hq][D + 2]: O (unnormalised), m, l
  int* counters;            // [num_seqs][Hkv][n_hb]: splits finished (cleared by the check)
  __nv_bfloat16* out;       // [num_seqs, Hq, D]
  float* lse;               // [num_seqs, Hq] or nullptr
  int* status;              // device status words (sticky error code first)
  const int* bad;           // this call's offset check: nonzero = compute nothing
  int num_seqs, Hq, Hkv, G, n_hb;  // n_hb = ceil(G / 16) query-head blocks per KV head
  int window;
  int splits, tiles_per_split;
  float scale_log2;         // scale * log2(e)
  unsigned long long timeout_ns;
  PagedKV kv;               // paged key/value cache, or kv.page_size == 0 (contiguous)
  int kv_rows = 0;          // rows of the k/v buffers (checked by builds with -DTSK_DEBUG)
};

template <int D>
__host__ __device__ constexpr uint32_t tile_bytes() { return kKeys * D * 2; }
// K/V ring depth: 3 x 32 KB for D = 64 (two CTAs per SM), 2 x 64 KB for D = 128.
template <int D>
__host__ __device__ constexpr int stages() { return D == 64 ? 3 : 2; }
// The four warps' final states are exchanged in the (then idle) ring.
template <int D>
__host__ __device__ constexpr uint32_t ring_bytes() { return stages<D>() * 2 * tile_bytes<D>(); }
template <int D>
__host__ __device__ constexpr uint32_t smem_bytes() { return ring_bytes<D>() + 256 + 1024; }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D (16x8 fp32) += A (16x16 bf16, row-major) * B (16x8 bf16, column-major).
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte address of 16-byte chunk `c` of row `r` in a tile of 128-byte rows
// written by TMA with the 128-byte swizzle (D = 128 tiles are two such
// 64-column halves, 128 rows each).
template <int D>
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int c) {
  const int half = c >> 3, cc = c & 7;
  return base + (uint32_t)half * (kKeys * 128) + (uint32_t)r * 128u + ((uint32_t)(cc ^ (r & 7)) << 4);
}

// cu_k must be 0 = cu_k[0] < cu_k[1] < ... with every length 1 .. max_k and
// cu_k[num_seqs] = total_k.  Writes this call's result to *bad and, on
// failure, TSK_ERR_BAD_SEQLENS (-8) to the sticky status word.  Also clears
// the n_counters split counters of this call.
__global__ void decode_check_kernel(const int* cu_k, int num_seqs, int total_k, int max_k,
                                    int* status, int* bad_out, PagedKV pg, int* counters,
                                    int n_counters) {
  for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0;
  bool bad = false;
  for (int s = threadIdx.x; s < num_seqs; s += blockDim.x) {
    const int a = cu_k[s], b = cu_k[s + 1];
    if (a < 0 || b < a + 1 || b - a > max_k || b > total_k) bad = true;
    else if (!pages_ok(pg, s, b - a)) bad = true;
  }
  if (threadIdx.x == 0 && (cu_k[0] != 0 || cu_k[num_seqs] != total_k)) bad = true;
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    *bad_out = bad ? 1 : 0;
    if (bad && atomicCAS(status, 0, -8) == 0) status[1] = 2000;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ DecParams p) {
  constexpr int KS = D / 16;      // k-steps of S = Q K^T
  constexpr int NT_O = D / 8;     // 8-column tiles of O
  constexpr int kStages = stages<D>();
  constexpr uint32_t kTile = tile_bytes<D>();
  static_assert(4 * kRows * (D + 2) * 4 <= ring_bytes<D>(), "state exchange fits the ring");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  float* red = reinterpret_cast<float*>(smem);  // [4 warps][16][D + 2], after the key loop
  const uint32_t bar_full = sbase + ring_bytes<D>(), bar_empty = bar_full + 8 * kStages;
  const uint32_t abort_addr = bar_full + 16 * kStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int g = blockIdx.y / p.n_hb, hb = blockIdx.y - g * p.n_hb;
  const int b = blockIdx.z;
  if (*reinterpret_cast<const volatile int*>(p.bad) != 0) return;  // offsets were rejected

  const int k0 = p.cu_k[b], Lk = p.cu_k[b + 1] - k0;
  const int lo = p.window > 0 ? max(0, Lk - p.window) : 0;  // first visible key position
  const int lo_al = lo - lo % kKeys;  // tiles start on multiples of 128 key positions
  const int t_begin = split * p.tiles_per_split;
  const int n_tiles_seq = (Lk - lo_al + kKeys - 1) / kKeys;
  const int t_end = min(n_tiles_seq, t_begin + p.tiles_per_split);
  const int nt = max(0, t_end - t_begin);  // tiles of this CTA
  const int h_lo = hb * kRows;             // first query head of the block within the group
  const int rows = min(kRows, p.G - h_lo);  // valid query heads in the block

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 4);
    }
    st_shared_volatile(abort_addr, 0);
    fence_mbar_init();
  }
  __syncthreads();

  struct P2 { int* status; unsigned long long timeout_ns; } pw{p.status, p.timeout_ns};
  bool ok = true;
  int issued = 0;  // tiles whose loads thread 0 has armed
  // Producer: thread 0 keeps kStages - 1 tiles ahead of the tile being consumed.
  auto issue = [&](int i) {  // tile i of this CTA into stage i % kStages
    const int s = i % kStages;
    if (i >= kStages) ok = ok && mbar_wait(bar_empty + 8 * s, ((i / kStages) - 1) & 1, 30, pw, abort_addr);
    if (!ok) return;
    const int pos0 = lo_al + (t_begin + i) * kKeys;
    if (!TSK_IN_BOUNDS(pw, abort_addr,
                       g < p.Hkv && (p.kv.page_size != 0 ||
                                     (k0 + pos0 >= 0 && k0 + pos0 < p.kv_rows)),
                       51)) {
      ok = false;
      return;
    }
    issued = i + 1;
    const uint32_t dst = sbase + (uint32_t)s * 2u * kTile;
    mbar_arrive_expect_tx(bar_full + 8 * s, 2 * kTile);
    bool in = true;
    for (int hf = 0; hf < D / 64; ++hf) {
      in = tma_load_key_rows(dst + hf * (kKeys * 128), &tmK, bar_full + 8 * s, 64 * hf, g, p.kv, b,
                             k0, pos0, Lk) && in;
      in = tma_load_key_rows(dst + kTile + hf * (kKeys * 128), &tmV, bar_full + 8 * s, 64 * hf, g,
                             p.kv, b, k0, pos0, Lk) && in;
    }
    if (!TSK_IN_BOUNDS(pw, abort_addr, in, 43)) ok = false;
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < kStages - 1 && i < nt; ++i) issue(i);

  // Q fragments (rows = query heads of the block, zero beyond `rows`).
  uint32_t qa[KS][4];
  {
    const int r0 = lane >> 2, r1 = r0 + 8, c = (lane & 3) * 2;
    const __nv_bfloat16* qb = p.q + ((size_t)b * p.Hq + (size_t)g * p.G + h_lo) * D;
    const bool q_ok =
        TSK_IN_BOUNDS(pw, abort_addr, b < p.num_seqs && g * p.G + h_lo + rows <= p.Hq, 52);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      auto ld = [&](int r, int col) -> uint32_t {
        return r < rows && q_ok ? *reinterpret_cast<const uint32_t*>(qb + (size_t)r * D + col) : 0u;
      };
      qa[ks][0] = ld(r0, 16 * ks + c);
      qa[ks][1] = ld(r1, 16 * ks + c);
      qa[ks][2] = ld(r0, 16 * ks + 8 + c);
      qa[ks][3] = ld(r1, 16 * ks + 8 + c);
    }
  }

  float o[NT_O][4];
#pragma unroll
  for (int i = 0; i < NT_O; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows lane/4 and lane/4 + 8
  const float sl2 = p.scale_log2;

  for (int i = 0; i < nt && ok; ++i) {
    if (threadIdx.x == 0 && i + kStages - 1 < nt) issue(i + kStages - 1);
    const int s = i % kStages;
    ok = __all_sync(0xffffffffu, ok && mbar_wait(bar_full + 8 * s, (i / kStages) & 1, 31, pw, abort_addr));
    if (!ok) break;
    const uint32_t kt = sbase + (uint32_t)s * 2u * kTile, vt = kt + kTile;
    const int key0 = lo_al + (t_begin + i) * kKeys + 32 * warp;  // key position of the warp's first key

    // S (16 x 32) = Q K^T for the warp's 32 keys.
    float sc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
      const int krow = 32 * warp + 8 * n + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < KS; ks += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(swz<D>(kt, krow, 2 * ks + (lane >> 3)), b0, b1, b2, b3);
        mma16816(sc[n], qa[ks], b0, b1);
        mma16816(sc[n], qa[ks + 1], b2, b3);
      }
    }
    // Mask keys outside [lo, Lk) (the tail of the last tile), scale to base 2.
    float mt0 = -INFINITY, mt1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < 4; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kp = key0 + 8 * n + (lane & 3) * 2 + e;
        const bool in = kp < Lk && kp >= lo;
        sc[n][e] = in ? sc[n][e] * sl2 : -INFINITY;
        sc[n][2 + e] = in ? sc[n][2 + e] * sl2 : -INFINITY;
        mt0 = fmaxf(mt0, sc[n][e]);
        mt1 = fmaxf(mt1, sc[n][2 + e]);
      }
    }
    mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, 1));
    mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, 2));
    mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, 1));
    mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, 2));
    const float mn0 = fmaxf(m0, mt0), mn1 = fmaxf(m1, mt1);
    const float a0 = mn0 == -INFINITY ? 1.f : ex2_approx(m0 - mn0);
    const float a1 = mn1 == -INFINITY ? 1.f : ex2_approx(m1 - mn1);
    const float u0 = mn0 == -INFINITY ? 0.f : mn0, u1 = mn1 == -INFINITY ? 0.f : mn1;
    m0 = mn0;
    m1 = mn1;
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int n = 0; n < NT_O; ++n) {
      o[n][0] *= a0;
      o[n][1] *= a0;
      o[n][2] *= a1;
      o[n][3] *= a1;
    }
    // P as A fragments of two 16-key steps (bf16); row sums in fp32.
    uint32_t pa[2][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const float p0 = ex2_approx(sc[n][0] - u0), p1 = ex2_approx(sc[n][1] - u0);
      const float p2 = ex2_approx(sc[n][2] - u1), p3 = ex2_approx(sc[n][3] - u1);
      const uint32_t x01 = pack_bf16x2(p0, p1), x23 = pack_bf16x2(p2, p3);
      l0 += p0 + p1;
      l1 += p2 + p3;
      pa[n >> 1][(n & 1) * 2 + 0] = x01;
      pa[n >> 1][(n & 1) * 2 + 1] = x23;
    }
    // O (16 x D) += P (16 x 32) V (32 x D).
#pragma unroll
    for (int kp = 0; kp < 2; ++kp) {
      const int vrow = 32 * warp + 16 * kp + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int n = 0; n < NT_O; n += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(swz<D>(vt, vrow, n + (lane >> 4)), b0, b1, b2, b3);
        mma16816(o[n], pa[kp], b0, b1);
        mma16816(o[n + 1], pa[kp], b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
  }
  // Every armed load must have landed before the ring is reused or the CTA
  // exits (after an abort some may not have been consumed).
  if (threadIdx.x == 0)
    for (int i = max(0, issued - kStages); i < issued; ++i)
      mbar_wait<true>(bar_full + 8 * (i % kStages), (i / kStages) & 1, 32, pw, abort_addr);
  __syncthreads();

  // Merge the four warps: row sums over the quad, then through shared memory.
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  {
    float* rw = red + (size_t)warp * kRows * (D + 2);
    const int r0 = lane >> 2, r1 = r0 + 8, c = (lane & 3) * 2;
#pragma unroll
    for (int n = 0; n < NT_O; ++n) {
      rw[r0 * (D + 2) + 8 * n + c] = o[n][0];
      rw[r0 * (D + 2) + 8 * n + c + 1] = o[n][1];
      rw[r1 * (D + 2) + 8 * n + c] = o[n][2];
      rw[r1 * (D + 2) + 8 * n + c + 1] = o[n][3];
    }
    if ((lane & 3) == 0) {
      rw[r0 * (D + 2) + D] = m0;
      rw[r0 * (D + 2) + D + 1] = l0;
      rw[r1 * (D + 2) + D] = m1;
      rw[r1 * (D + 2) + D + 1] = l1;
    }
  }
  __syncthreads();
  // 128 threads: thread t handles row t / 8 and columns (t % 8) * D/8 ...
  {
    const int r = threadIdx.x >> 3, part = threadIdx.x & 7;
    constexpr int per = D / 8;
    float mw[4], M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      mw[w] = red[((size_t)w * kRows + r) * (D + 2) + D];
      M = fmaxf(M, mw[w]);
    }
    float wt[4], L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      wt[w] = mw[w] == -INFINITY ? 0.f : ex2_approx(mw[w] - M);
      L += wt[w] * red[((size_t)w * kRows + r) * (D + 2) + D + 1];
    }
    if (r < rows && TSK_IN_BOUNDS(pw, abort_addr,
                                  split < p.splits && g * p.G + h_lo + r < p.Hq, 53)) {
      const int h = g * p.G + h_lo + r;
      float* dst = p.part + (((size_t)split * p.num_seqs + b) * p.Hq + h) * (D + 2);
#pragma unroll
      for (int j = 0; j < per; ++j) {
        const int col = part * per + j;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) acc += wt[w] * red[((size_t)w * kRows + r) * (D + 2) + col];
        dst[col] = acc;
      }
      if (part == 0) {
        dst[D] = M;
        dst[D + 1] = L;
      }
    }
  }

  // The last CTA of this (sequence, KV head, head block) to get here merges
  // the splits (release: each CTA's partial writes are fenced before its
  // count; acquire: the last one fences after it and reads around L1).
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    int prev = 0;
    if (TSK_IN_BOUNDS(pw, abort_addr, b < p.num_seqs && g < p.Hkv && hb < p.n_hb, 54))
      prev = atomicAdd(p.counters + ((size_t)b * p.Hkv + g) * p.n_hb + hb, 1);
    s_last = prev == p.splits - 1;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  {
    // 128 threads: eight per query head of the block, D / 8 columns each.
    const int r = threadIdx.x >> 3, part = threadIdx.x & 7;
    constexpr int per = D / 8;
    if (r < rows && TSK_IN_BOUNDS(pw, abort_addr, g * p.G + h_lo + r < p.Hq, 55)) {
      const int h = g * p.G + h_lo + r;
      const float sink2 = p.sinks ? p.sinks[h] * 1.4426950408889634f : -INFINITY;
      auto src_of = [&](int sp) {
        return p.part + (((size_t)sp * p.num_seqs + b) * p.Hq + h) * (D + 2);
      };
      float M = sink2;
      for (int sp = 0; sp < p.splits; ++sp) M = fmaxf(M, __ldcg(src_of(sp) + D));
      float Z = p.sinks ? ex2_approx(sink2 - M) : 0.f;
      float acc[per];
#pragma unroll
      for (int j = 0; j < per; ++j) acc[j] = 0.f;
      for (int sp = 0; sp < p.splits; ++sp) {
        const float* src = src_of(sp);
        const float ms = __ldcg(src + D);
        if (ms == -INFINITY) continue;
        const float wgt = ex2_approx(ms - M);
        Z += wgt * __ldcg(src + D + 1);
#pragma unroll
        for (int j = 0; j < per; ++j) acc[j] += wgt * __ldcg(src + part * per + j);
      }
      const float inv = 1.f / Z;
      __nv_bfloat16* o = p.out + ((size_t)b * p.Hq + h) * D + part * per;
#pragma unroll
      for (int j = 0; j < per; j += 2)
        *reinterpret_cast<uint32_t*>(o + j) = pack_bf16x2(acc[j] * inv, acc[j + 1] * inv);
      if (p.lse && part == 0) p.lse[(size_t)b * p.Hq + h] = (M + log2f(Z)) * 0.69314718055994531f;
    }
  }
}

}  // namespace dec
}  // namespace tsk
