// Persistent, warp-specialised causal GQA attention forward for sm_103a.
//
// One CTA per SM walks a static stride over the work units of the query-tile
// list, which the scheduler pre-pass sorted by cost (longest first).  A unit
// is (query tile of 128 rows, KV head g, head pair): two query heads of the
// same KV group over the same 128 tokens, so both share every K/V tile staged
// in shared memory (GQA reuse) and have identical key ranges.  With one query
// head per KV head (Hq == Hkv) a unit is instead two consecutive 128-row
// tiles of one head (list entries of 256 rows, key range the union of the
// two; a key tile only one tile needs is fully masked for the other and adds
// exact zeros), so that both query tiles of the CTA stay busy.  Roles:
//   warp 0        TMA producer: Q tiles (2 x 16 KB, double buffered) and a
//                 ring of kStages K/V stages (16 KB + 16 KB each)
//   warp 1        allocates TMEM; one lane issues tile 0's tcgen05.mma:
//                   S_0 = Q_0 K_j^T   (M=128, N=128, K=64, both K-major, smem)
//                   O_0 += P_0 V_j    (M=128, N=64,  K=128; P from TMEM, V MN-major)
//   warp 2        one lane issues tile 1's MMAs (same shapes)
//   warps 4..7    softmax + epilogue for query tile t=0 (one thread per row)
//   warps 8..11   softmax + epilogue for query tile t=1
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,320) O1 [320,384)
//               P0 [384,448) P1 [448,512)  (P is bf16, two per column)
// The issuer of tile t computes S_t(j+1) while the softmax of tile t works on
// S_t(j); the two tiles share the tensor core.
//
// Softmax (base 2): x = s * scale * log2(e).  The running maximum m and sum l
// start from the sink (m = sink*log2 e, l = 1) or from (-inf, 0) without one.
// The maximum used for exponentials is only raised when a tile's maximum
// exceeds it by more than kRescaleThreshold (then O and l are rescaled); so
// p <= 2^kRescaleThreshold.  The result is exact up to rounding because the
// same m enters numerator and denominator.  Only tiles that straddle the
// causal diagonal or the window's lower edge evaluate the mask; key tiles
// outside [kv_lo, diagonal] are never visited.  Every wait is bounded: on
// expiry the kernel records TSK_ERR_DEVICE_TIMEOUT, stops all roles, drains
// its copies and MMAs, frees TMEM and returns.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"
#include "schedule.cuh"

namespace tsk {

#ifndef TSK_KV_STAGES
#define TSK_KV_STAGES 3
#endif
#ifndef TSK_RESCALE_THRESHOLD
#define TSK_RESCALE_THRESHOLD 8.0f
#endif
constexpr int kStages = TSK_KV_STAGES;           // K/V ring depth
constexpr float kRescaleThreshold = TSK_RESCALE_THRESHOLD;  // log2 units
// A key tile of the causal kernel skips its row maximum when the bound on its
// scores lies within this much (log2 units) of the maximum in use: then every
// p <= 2^64.  With l kept below 2^32 between tiles (see the fast tile), a tile
// adds at most 128 * 2^64 to l, so |O| <= l max|v| stays finite for
// |v| < 2^56.
constexpr float kFastLag = 64.f;
struct SlowTile : std::true_type {};
struct FastTile : std::false_type {};
constexpr int kFirstSoftmaxWarp = 4;
constexpr int kSoftmaxWarpsPerTile = 4;
constexpr int kThreads = 32 * (kFirstSoftmaxWarp + 2 * kSoftmaxWarpsPerTile);
constexpr int kHeadDim = 64;
constexpr uint32_t kTileBytes = kTileM * kHeadDim * 2;  // 16 KB (also K/V tiles)
constexpr uint32_t kSmemQ = 0;                           // 2 buffers x 2 tiles
constexpr uint32_t kSmemKV = 4 * kTileBytes;             // kStages x (K, V)
constexpr uint32_t kSmemBar = kSmemKV + kStages * 2 * kTileBytes;  // barriers (< 512 B)
constexpr uint32_t kSmemEpi = kSmemBar + 1024;  // 2 output staging tiles
constexpr uint32_t kSmemNorm = kSmemEpi + 2 * kTileBytes;  // key-norm bound per KV head
// Dynamic shared memory per kernel variant, + 1 KB slack for the alignment.
constexpr uint32_t kSmemBytesCausal = kSmemNorm + 4 * kNormMaxHeads + 1024;
// (the small-window kernel has no key-norm bound; a second set of output
// staging tiles takes that region and more)
constexpr uint32_t kSmemBytesWindow = kSmemEpi + 4 * kTileBytes + 1024;
static_assert(kSmemBytesWindow <= 227 * 1024, "shared memory budget");

constexpr uint32_t kColS0 = 0, kColO0 = 256, kColP0 = 384;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 64, false, true);

struct AttnParams {
  const float* sinks;   // [Hq] or nullptr
  __nv_bfloat16* out;   // [T, Hq, 64]
  float* lse;           // [T, Hq] or nullptr
  const int4* list;     // sorted query tiles (two int4 per tile, see schedule.cuh)
  const int* ws;        // ws[kWsNTiles] = number of query tiles
  int* status;          // device status words
  int Hq, Hkv, G, HP;   // HP = ceil(G / 2) head pairs per KV head
  int window;
  float scale_log2;     // scale * log2(e)
  unsigned long long timeout_ns;
  int debug_stall;      // test hook: producer first waits on a barrier nothing signals
  PagedKV kv;           // paged key/value cache, or kv.page_size == 0 (contiguous)
  const float* knorm = nullptr;  // [Hkv] largest key-row norm per KV head, or nullptr
  // Extents checked by builds with -DTSK_DEBUG: rows of q/out, rows of the
  // k/v buffers (tokens, or slots of a paged pool), capacity of the tile list.
  int q_rows = 0, kv_rows = 0, max_tiles = 0;
  // Factor applied to the output (the value scale of E4M3 inputs; D = 128 kernel).
  float out_scale = 1.f;
};

// Barrier slots (8 bytes each) inside the barrier area.
enum : int {
  kBarQFull = 0,               // [2]
  kBarQEmpty = 2,              // [2]
  kBarKFull = 4,               // [kStages]
  kBarVFull = 4 + kStages,     // [kStages]
  kBarKVEmpty = 4 + 2 * kStages,
  kBarSFull = 4 + 3 * kStages,  // [2]
  kBarSFree = 6 + 3 * kStages,  // [2]
  kBarPFull = 8 + 3 * kStages,  // [2]
  kBarPVDone = 10 + 3 * kStages,  // [2]
  kBarDrain = 12 + 3 * kStages,  // [2] one per MMA issuer
  kBarNever = 14 + 3 * kStages,  // never signalled (stall injection)
  kNumBars = 15 + 3 * kStages
};
static_assert(8 * kNumBars + 8 <= 512, "barrier area");

// mbar_wait for warps whose every lane polls: the result is made warp-uniform
// so that the warp-collective tcgen05 instructions that follow never diverge.
template <class P>
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, int site, const P& p,
                                               uint32_t abort_saddr) {
  const bool ok = mbar_wait(bar, parity, site, p, abort_saddr);
  return __all_sync(0xffffffffu, ok);
}

struct Unit {
  int start, q0, kv_lo, len, n_kv, g, h0, ntiles;
  int start_k;  // first key row of the sequence (contiguous cache)
  int offset;   // Lk - Lq: key position of query row 0
  int seq;      // sequence index (block-table row of a paged cache)
};

// Unit u.  QS (a kernel template parameter) is the row offset between the
// unit's two query tiles: 0 when they are two heads over the same rows,
// kTileM when they are two row blocks of one head (Hq == Hkv).
template <int QS = 0>
__device__ __forceinline__ Unit decode_unit(const AttnParams& p, int u) {
  const int per_tile = p.Hkv * p.HP;
  int qi = u / per_tile;
  const int rem = u - qi * per_tile;
  if (!TSK_IN_BOUNDS(p, 0u, qi < p.max_tiles, 40)) qi = 0;  // (the unit is then wrong, the status says so)
  const int4 e = __ldg(p.list + 2 * qi);
  const int4 f = __ldg(p.list + 2 * qi + 1);
  Unit r;
  r.start = e.x;
  r.q0 = e.y;
  r.kv_lo = e.z;
  r.len = e.w;
  r.start_k = f.x;
  r.offset = f.y;
  r.n_kv = f.z;
  r.seq = f.w;
  r.g = rem / p.HP;
  const int hp = rem - r.g * p.HP;
  r.h0 = r.g * p.G + 2 * hp;
  r.ntiles = QS ? (r.q0 + QS < r.len ? 2 : 1) : ((2 * hp + 1 < p.G) ? 2 : 1);
  return r;
}

// Query head and first query row (relative to the sequence) of tile t of a unit.
template <int QS>
__device__ __forceinline__ int tile_head(const Unit& w, int t) {
  return w.h0 + (QS ? 0 : t);
}
template <int QS>
__device__ __forceinline__ int tile_q0(const Unit& w, int t) {
  return w.q0 + t * QS;
}

// The unit's sequence fields read again (volatile loads: not merged with the
// first read), so that they need no registers while a unit's key tiles run.
__device__ __forceinline__ int4 ld_nc_v4_volatile(const int4* a) {
  int4 v;
  asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(a));
  return v;
}


// TMA loads of the 128 cache rows holding key positions pos0 .. pos0 + 127 of
// sequence `seq` (Lk keys) from a paged cache into the 128-byte rows at `dst`,
// x = first of the 64 columns: one box per page chunk (min(page_size, 128)
// rows, at least 8: chunks start on 1024-byte boundaries, so the 128-byte
// swizzle is that of a single box); chunks past the sequence's last page
// re-read that page (their keys are masked).  Out of line: it is rare next to
// the contiguous case and stays out of the kernels' hot code.
// In builds with -DTSK_DEBUG a page outside the pool is not loaded and the
// function returns false.
__device__ __noinline__ bool tma_load_key_rows_paged(uint32_t dst, const CUtensorMap* tm,
                                                     uint32_t bar, int x, int head,
                                                     const PagedKV pg, int seq, int pos0, int Lk) {
  const int chunk = pg.page_size < 128 ? pg.page_size : 128;
  const int last_blk = (Lk - 1) / pg.page_size;
  bool in_pool = true;
  for (int c = 0; c < 128; c += chunk) {
    const int pos = pos0 + c;
    int blk = pos / pg.page_size;
    if (blk > last_blk) blk = last_blk;
    const int page = __ldg(pg.table + (size_t)seq * pg.max_blocks + blk);
#ifdef TSK_DEBUG
    if (page < 0 || page >= pg.num_pages || blk >= pg.max_blocks) {
      in_pool = false;
      continue;
    }
#endif
    tma_load_3d(dst + (uint32_t)c * 128u, tm, bar, x, head, page * pg.page_size + pos % pg.page_size);
  }
  return in_pool;
}

// The same for either cache layout; a contiguous cache (page_size 0) is one
// box at row row0 + pos0.
__device__ __forceinline__ bool tma_load_key_rows(uint32_t dst, const CUtensorMap* tm,
                                                  uint32_t bar, int x, int head, const PagedKV& pg,
                                                  int seq, int row0, int pos0, int Lk) {
  if (pg.page_size != 0) return tma_load_key_rows_paged(dst, tm, bar, x, head, pg, seq, pos0, Lk);
  tma_load_3d(dst, tm, bar, x, head, row0 + pos0);
  return true;
}

// State shared by the roles of one CTA.
struct Ctx {
  uint32_t sbase;   // 1 KB-aligned shared memory base (shared-window address)
  uint32_t bar0;    // first mbarrier
  uint32_t tmem;    // TMEM base address
  int total_units;
  uint32_t abort;   // shared address of the CTA's abort flag
  bool alternate;   // unit order (cta_unit)
  __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
  __device__ __forceinline__ int unit(int ku) const;
};

// The ku-th unit of this CTA.  The CTAs take the unit list in rounds of
// gridDim.x units.  With `alternate`, every other round runs in the opposite
// direction: the list is sorted by decreasing cost (key tiles), and with
// every round in the same direction the first CTAs get the dearer unit of
// each round that straddles a change of cost (4 x 4096 causal: the largest
// CTA total 3.5% above the mean, against 0.1% alternating; the causal D = 64
// kernels measured 1.5-2.3% faster).  The small-window kernel (units of
// equal cost; 1.4% slower alternating) and the D = 128 kernel (1-3% slower
// on 4 x 4096, 2% faster on one 32K sequence) keep one direction.  Every
// role of a CTA walks the same sequence; it increases with ku.
__device__ __forceinline__ int cta_unit(int ku, bool alternate) {
  const int g = (int)gridDim.x, b = (int)blockIdx.x;
  return ku * g + ((alternate && (ku & 1)) ? g - 1 - b : b);
}
__device__ __forceinline__ int Ctx::unit(int ku) const { return cta_unit(ku, alternate); }


// TMA producer (one thread).
template <int QS>
__device__ __forceinline__ void role_producer(const Ctx& cx, const CUtensorMap* tmQ,
                                           const CUtensorMap* tmK, const CUtensorMap* tmV,
                                           const AttnParams& p) {
  // ------------------------------------------------------------ producer
  uint32_t q_iter = 0, kv_iter = 0;
  bool ok = true;
  TSK_TL_DECL;
  if (p.debug_stall) ok = mbar_wait(cx.bar(kBarNever), 0, 99, p, cx.abort);
  for (int ku = 0, u = cx.unit(0); u < cx.total_units && ok; u = cx.unit(++ku)) {
    const Unit w = decode_unit<QS>(p, u);
    const int qb = q_iter & 1;
    if (q_iter >= 2) ok = mbar_wait(cx.bar(kBarQEmpty + qb), ((q_iter >> 1) & 1) ^ 1, 1, p, cx.abort);
    if (!ok) break;
    mbar_arrive_expect_tx(cx.bar(kBarQFull + qb), w.ntiles * kTileBytes);
    for (int t = 0; t < w.ntiles; ++t) {
      const int h = tile_head<QS>(w, t), row = w.start + tile_q0<QS>(w, t);
      if (!TSK_IN_BOUNDS(p, cx.abort, h >= 0 && h < p.Hq && row >= 0 && row < p.q_rows, 41)) {
        ok = false;
        break;
      }
      tma_load_3d(cx.sbase + kSmemQ + (2 * qb + t) * kTileBytes, tmQ, cx.bar(kBarQFull + qb), 0,
                  h, row);
    }
    if (!ok) break;
    ++q_iter;
    for (int j = 0; j < w.n_kv; ++j, ++kv_iter) {
      const int s = kv_iter % kStages;
      const uint32_t k = kv_iter / kStages;
      if (k >= 1) ok = mbar_wait(cx.bar(kBarKVEmpty + s), (k - 1) & 1, 2, p, cx.abort);
      if (!ok) break;
      TSK_EV(30);
      const int pos0 = (w.kv_lo + j) * kTileN;  // key position of the tile's first key
      const int Lk = w.offset + w.len;
      const uint32_t kdst = cx.sbase + kSmemKV + s * 2 * kTileBytes;
      if (!TSK_IN_BOUNDS(p, cx.abort,
                         w.g >= 0 && w.g < p.Hkv &&
                             (p.kv.page_size != 0 ||
                              (w.start_k + pos0 >= 0 && w.start_k + pos0 < p.kv_rows)),
                         42)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(cx.bar(kBarKFull + s), kTileBytes);
      bool in = tma_load_key_rows(kdst, tmK, cx.bar(kBarKFull + s), 0, w.g, p.kv, w.seq, w.start_k,
                                  pos0, Lk);
      mbar_arrive_expect_tx(cx.bar(kBarVFull + s), kTileBytes);
      in = tma_load_key_rows(kdst + kTileBytes, tmV, cx.bar(kBarVFull + s), 0, w.g, p.kv, w.seq,
                             w.start_k, pos0, Lk) && in;
      if (!TSK_IN_BOUNDS(p, cx.abort, in, 43)) {
        ok = false;
        break;
      }
    }
  }
  // Drain: wait for the last load issued into every buffer so that no
  // copy is still in flight when the CTA exits (bounded, best effort).
  for (uint32_t i = (kv_iter > kStages ? kv_iter - kStages : 0); i < kv_iter; ++i) {
    mbar_wait<true>(cx.bar(kBarKFull + i % kStages), (i / kStages) & 1, 11, p, cx.abort);
    mbar_wait<true>(cx.bar(kBarVFull + i % kStages), (i / kStages) & 1, 12, p, cx.abort);
  }
  for (uint32_t i = (q_iter > 2 ? q_iter - 2 : 0); i < q_iter; ++i)
    mbar_wait<true>(cx.bar(kBarQFull + (i & 1)), (i >> 1) & 1, 13, p, cx.abort);

}

// tcgen05.mma issuer (one thread).
// tcgen05.mma issuer for query tile t (one thread; tiles 0 and 1 have their
// own issuers, so a slow softmax of one tile never holds back the other's
// MMAs).  Per key tile j:
//   S_t(j+1) = Q_t K_{j+1}^T   once K_{j+1} is loaded and the softmax has read S_t(j)
//   O_t += P_t(j) V_j          once V_j is loaded and the softmax has written P_t(j)
// Each issuer releases a K/V stage (and the Q buffer) with its own commit, so
// those barriers count two arrivals (the Q buffer also counts the eight softmax
// warps); in a unit with one query tile the tile-1 issuer still waits for each
// of the unit's fills and releases it with a plain arrival, so that no fill is
// replaced before both issuers have seen it.
template <int QS>
__device__ __forceinline__ void role_mma(const Ctx& cx, const AttnParams& p, int t) {
  uint32_t q_iter = 0, kv_iter = 0, s_cnt = 0, p_cnt = 0;
  bool ok = true;
#define TSK_ISSUER_WAIT(bar, par, site) mbar_wait(bar, par, site, p, cx.abort)
#define TSK_MMA_SS(...) mma_ss(__VA_ARGS__)
#define TSK_MMA_TS(...) mma_ts(__VA_ARGS__)
#define TSK_COMMIT(bar) tc_commit(bar)
  TSK_TL_DECL;
  const uint32_t d_s = cx.tmem + kColS0 + 128 * t;
  const uint32_t d_o = cx.tmem + kColO0 + 64 * t;
  const uint32_t a_p = cx.tmem + kColP0 + 64 * t;
  for (int ku = 0, u = cx.unit(0); u < cx.total_units && ok; u = cx.unit(++ku)) {
    const Unit w = decode_unit<QS>(p, u);
    const int qb = q_iter & 1;
    ok = TSK_ISSUER_WAIT(cx.bar(kBarQFull + qb), (q_iter >> 1) & 1, 3);
    if (!ok) break;
    if (t >= w.ntiles) {
      // This tile is idle in the unit: follow the unit's K/V fills and release
      // them (and the Q buffer) like a present tile, so that no fill can be
      // replaced before this thread has seen it (no barrier ever runs two
      // phases ahead of it).
      for (int j = 0; j < w.n_kv && ok; ++j) {
        const uint32_t cur = kv_iter + j;
        const int sc = cur % kStages;
        ok = TSK_ISSUER_WAIT(cx.bar(kBarKFull + sc), (cur / kStages) & 1, 4);
        if (ok) ok = TSK_ISSUER_WAIT(cx.bar(kBarVFull + sc), (cur / kStages) & 1, 7);
        if (ok) mbar_arrive(cx.bar(kBarKVEmpty + sc));
      }
      if (!ok) break;
      mbar_arrive(cx.bar(kBarQEmpty + qb));
      kv_iter += w.n_kv;
      ++q_iter;
      continue;
    }
    const uint32_t qaddr = cx.sbase + kSmemQ + (2 * qb + t) * kTileBytes;
    auto issue_s = [&](int stage) {
      TSK_EV(21);
      TSK_TRACE_T0(tr_is);
      const uint32_t b = cx.sbase + kSmemKV + stage * 2 * kTileBytes;
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk)
        TSK_MMA_SS(d_s, sdesc_sw128(qaddr + 32 * kk), sdesc_sw128(b + 32 * kk), kIdescQK,
               kk > 0 ? 1u : 0u);
      TSK_COMMIT(cx.bar(kBarSFull + t));
      ++s_cnt;
      TSK_EV(22);
      TSK_TRACE_ADD(15, tr_is);
    };
    {  // S_t(0)
      const int s0 = kv_iter % kStages;
      ok = TSK_ISSUER_WAIT(cx.bar(kBarKFull + s0), (kv_iter / kStages) & 1, 4);
      if (ok && s_cnt > 0) ok = TSK_ISSUER_WAIT(cx.bar(kBarSFree + t), (s_cnt - 1) & 1, 5);
      if (!ok) break;
      tc_fence_after();
      issue_s(s0);
    }
    for (int j = 0; j < w.n_kv && ok; ++j) {
      const uint32_t cur = kv_iter + j;
      const int sc = cur % kStages;
      if (j + 1 < w.n_kv) {
        const int sn = (cur + 1) % kStages;
        TSK_EV(20);
        ok = TSK_ISSUER_WAIT(cx.bar(kBarKFull + sn), ((cur + 1) / kStages) & 1, 6);
        if (ok) ok = TSK_ISSUER_WAIT(cx.bar(kBarSFree + t), (s_cnt - 1) & 1, 5);
        if (!ok) break;
        tc_fence_after();
        issue_s(sn);
      }
      TSK_EV(23);
      ok = TSK_ISSUER_WAIT(cx.bar(kBarVFull + sc), (cur / kStages) & 1, 7);
      if (ok) ok = TSK_ISSUER_WAIT(cx.bar(kBarPFull + t), p_cnt & 1, 8);
      if (!ok) break;
      TSK_EV(24);
      tc_fence_after();
      const uint32_t b = cx.sbase + kSmemKV + sc * 2 * kTileBytes + kTileBytes;
      TSK_TRACE_T0(tr_ip);
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        TSK_MMA_TS(d_o, a_p + 8 * kk, sdesc_sw128(b + 2048 * kk), kIdescPV,
                   (j > 0 || kk > 0) ? 1u : 0u);
      TSK_COMMIT(cx.bar(kBarPVDone + t));
      ++p_cnt;
      TSK_EV(25);
      TSK_TRACE_ADD(16, tr_ip);
      TSK_COMMIT(cx.bar(kBarKVEmpty + sc));
    }
    if (!ok) break;
    kv_iter += w.n_kv;
    TSK_COMMIT(cx.bar(kBarQEmpty + qb));
    ++q_iter;
  }
  // Make sure none of this thread's MMAs is still running before TMEM is freed.
  TSK_COMMIT(cx.bar(kBarDrain + t));
  mbar_wait<true>(cx.bar(kBarDrain + t), 0, 14, p, cx.abort);
#undef TSK_ISSUER_WAIT
#undef TSK_MMA_SS
#undef TSK_MMA_TS
#undef TSK_COMMIT
}

// One tcgen05.mma issuer for both query tiles (the small-window kernel, whose
// units have few key tiles), in the order in which the softmax warpgroups
// usually free S and publish P: S_0(0), S_1(0), S_0(1), S_1(1), then per key
// tile j: PV_0(j), S_0(j+2), PV_1(j), S_1(j+2).  Any other order of those
// events only delays an MMA: each wait depends on MMAs issued before it.
// Its commits are the only arrivals on the stage and Q release barriers.
template <int QS>
__device__ __forceinline__ void role_mma_pair(const Ctx& cx, const AttnParams& p) {
  uint32_t q_iter = 0, kv_iter = 0;
  uint32_t s_cnt[2] = {0u, 0u}, p_cnt[2] = {0u, 0u};
  bool ok = true;
  TSK_TL_DECL;
  for (int ku = 0, u = cx.unit(0); u < cx.total_units && ok; u = cx.unit(++ku)) {
    const Unit w = decode_unit<QS>(p, u);
    const int qb = q_iter & 1;
    const int nt = w.ntiles;
    ok = mbar_wait(cx.bar(kBarQFull + qb), (q_iter >> 1) & 1, 3, p, cx.abort);
    if (!ok) break;
    auto issue_s = [&](int t, uint32_t kv) -> bool {
      const int st = kv % kStages;
      if (!mbar_wait(cx.bar(kBarKFull + st), (kv / kStages) & 1, 6, p, cx.abort)) return false;
      if (s_cnt[t] > 0 &&
          !mbar_wait(cx.bar(kBarSFree + t), (s_cnt[t] - 1) & 1, 5, p, cx.abort))
        return false;
      tc_fence_after();
      const uint32_t qaddr = cx.sbase + kSmemQ + (2 * qb + t) * kTileBytes;
      const uint32_t b = cx.sbase + kSmemKV + st * 2 * kTileBytes;
      const uint32_t d_s = cx.tmem + kColS0 + 128 * t;
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk)
        mma_ss(d_s, sdesc_sw128(qaddr + 32 * kk), sdesc_sw128(b + 32 * kk), kIdescQK,
               kk > 0 ? 1u : 0u);
      tc_commit(cx.bar(kBarSFull + t));
      ++s_cnt[t];
      return true;
    };
    auto issue_pv = [&](int t, uint32_t kv, int j) -> bool {
      const int st = kv % kStages;
      if (!mbar_wait(cx.bar(kBarVFull + st), (kv / kStages) & 1, 7, p, cx.abort)) return false;
      if (!mbar_wait(cx.bar(kBarPFull + t), p_cnt[t] & 1, 8, p, cx.abort)) return false;
      tc_fence_after();
      const uint32_t b = cx.sbase + kSmemKV + st * 2 * kTileBytes + kTileBytes;
      const uint32_t d_o = cx.tmem + kColO0 + 64 * t;
      const uint32_t a_p = cx.tmem + kColP0 + 64 * t;
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        mma_ts(d_o, a_p + 8 * kk, sdesc_sw128(b + 2048 * kk), kIdescPV,
               (j > 0 || kk > 0) ? 1u : 0u);
      tc_commit(cx.bar(kBarPVDone + t));
      ++p_cnt[t];
      return true;
    };
    const int n = w.n_kv;
    for (int t = 0; t < nt && ok; ++t) ok = issue_s(t, kv_iter);
    for (int t = 0; t < nt && ok && n > 1; ++t) ok = issue_s(t, kv_iter + 1);
    for (int j = 0; j < n && ok; ++j) {
      for (int t = 0; t < nt && ok; ++t) {
        ok = issue_pv(t, kv_iter + j, j);
        if (ok && j + 2 < n) ok = issue_s(t, kv_iter + j + 2);
      }
      if (ok) tc_commit(cx.bar(kBarKVEmpty + (kv_iter + j) % kStages));
    }
    if (!ok) break;
    kv_iter += n;
    tc_commit(cx.bar(kBarQEmpty + qb));
    ++q_iter;
  }
  tc_commit(cx.bar(kBarDrain));
  mbar_wait<true>(cx.bar(kBarDrain), 0, 14, p, cx.abort);
}

// Column chunks of a 128-key tile (32 keys each) classified for one warp:
// every row of the warp sees all keys of the chunk, none of them, or some.
struct ChunkMask {
  uint32_t none;     // bit k: chunk k masked for every row of the warp
  uint32_t partial;  // bit k: chunk k needs a per-element test
};

// Allowed keys of a query at key position `pos` (relative to the sequence's
// first key) in the key tile starting at `kbase`: columns c with lo_c <= c <=
// hi_c, where hi_c = pos - kbase and lo_c = pos - window + 1 - kbase
// (window > 0).  The warp's queries sit at row0 .. row0 + 31, so the bounds
// of its lanes 0 and 31 decide each chunk uniformly.
__device__ __forceinline__ ChunkMask classify_chunks(int row0, int kbase, int window) {
  ChunkMask m{0u, 0u};
  const int hi_min = row0 - kbase, hi_max = hi_min + 31;
  const int lo_min = window > 0 ? hi_min - window + 1 : -(1 << 30);
  const int lo_max = window > 0 ? lo_min + 31 : -(1 << 30);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int c0 = 32 * k, c1 = 32 * k + 31;
    if (c1 < lo_min || c0 > hi_max) m.none |= 1u << k;
    else if (!(c0 >= lo_max && c1 <= hi_min)) m.partial |= 1u << k;
  }
  return m;
}

// Softmax and epilogue of query tile t (one warpgroup, one thread per row),
// used for full causal attention and windows wider than kSmallWindowMax:
// each row's 128 scores are held in registers for one pass (maximum, then
// exponentials), edge tiles are masked per element, and each thread stores
// its output row directly.  L gives the shared-memory layout and the format of
// the query tile (bf16 here; E4M3 in the FP8 kernel, which also scales the
// output by out_scale).
struct Bf16Layout {
  static constexpr uint32_t kQ = kSmemQ, kQTile = kTileBytes, kEpi = kSmemEpi, kNorm = kSmemNorm;
  static constexpr bool kScaleOut = false;
  // Sum of squares of query row r of the (128-byte swizzled) bf16 tile at `tile`.
  static __device__ __forceinline__ float q_sq(uint32_t tile, int r) {
    // the row's 128 bytes (8 chunks of 16, permuted by the swizzle)
    const uint32_t qrow = tile + (uint32_t)r * 128u;
    float ss[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      // chunk k ^ (r & 7): the lanes of a warp spread over all 32 banks
      const uint4 v = ld_shared_v4(qrow + 16u * (uint32_t)(k ^ (r & 7)));
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(wv[e] << 16), hi = __uint_as_float(wv[e] & 0xFFFF0000u);
        ss[2 * e] = fmaf(lo, lo, ss[2 * e]);
        ss[2 * e + 1] = fmaf(hi, hi, ss[2 * e + 1]);
      }
    }
    return ((ss[0] + ss[1]) + (ss[2] + ss[3])) + ((ss[4] + ss[5]) + (ss[6] + ss[7]));
  }
};

template <int QS, class L = Bf16Layout>
__device__ __forceinline__ void role_softmax_causal(const Ctx& cx, const AttnParams& p,
                                                    const CUtensorMap* tmO, int warp, int lane,
                                                    float out_scale = 1.f) {
  const int t = (warp - kFirstSoftmaxWarp) >> 2;  // query tile of this warpgroup
  const int wq = warp & 3;          // TMEM lane quarter
  const int r = wq * 32 + lane;     // query row within the tile
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const uint32_t tS = cx.tmem + lane_base + kColS0 + 128 * t;
  const uint32_t tO = cx.tmem + lane_base + kColO0 + 64 * t;
  const uint32_t tP = cx.tmem + lane_base + kColP0 + 64 * t;
  const uint32_t epi = cx.sbase + L::kEpi + t * kTileBytes;
  const float sl2 = p.scale_log2;
  uint32_t s_cnt = 0, pv_cnt = 0, q_iter = 0;
  TSK_TL_DECL;
  TSK_TRACE_T0(tr_all);
  bool ok = true;
  // What the key loop needs from a unit (the epilogue reads the sequence
  // fields again: registers are the scarce resource here).  The next unit's
  // fields are loaded before a unit's epilogue, so that their latency passes
  // while the epilogue waits for the last PV.
  struct Fields {
    int n_kv, kv_lo, diag0, gk;
    float sink;  // sink * log2(e), or -inf
    float bq;    // bound on the row's scores (key-norm bound), or +inf
    bool active;
  };
  auto fetch = [&](int uu) {
    Fields f{0, 0, 0, 0, -INFINITY, INFINITY, false};
    if (uu < cx.total_units) {
      const Unit w = decode_unit<QS>(p, uu);
      f.active = t < w.ntiles;
      f.gk = w.g;
      f.n_kv = w.n_kv;
      f.kv_lo = w.kv_lo;
      f.diag0 = w.offset + tile_q0<QS>(w, t);  // key position of the tile's first query row
      if (p.sinks && f.active &&
          TSK_IN_BOUNDS(p, cx.abort, tile_head<QS>(w, t) >= 0 && tile_head<QS>(w, t) < p.Hq, 44))
        f.sink = __ldg(p.sinks + tile_head<QS>(w, t)) * 1.4426950408889634f;
    }
    return f;
  };
  // Q buffer handover of unit uu (the qi-th unit of this CTA): every softmax
  // warp takes part in every unit's (the release counts both issuers and all
  // eight softmax warps), so that no warp can fall two phases behind the Q
  // barriers.  A present tile reads its query rows first, for the bound on
  // x = s * scale * log2(e) over every key of a row: ||q|| times the largest
  // key norm of the KV head (Cauchy-Schwarz).  Done for the next unit before
  // a unit's epilogue, so that it overlaps the wait for the last PV.
  auto handover = [&](int uu, uint32_t qi, Fields& f) -> bool {
    if (uu >= cx.total_units) return true;
    const int qbb = qi & 1;
    TSK_EV(16);
    if (!mbar_wait_warp(cx.bar(kBarQFull + qbb), (qi >> 1) & 1, 17, p, cx.abort)) return false;
    TSK_EV(18);
    if (f.active && p.knorm) {
      const float sq = L::q_sq(cx.sbase + L::kQ + (2 * qbb + t) * L::kQTile, r);
      f.bq = sl2 * sqrtf(sq) * ld_shared_f32(cx.sbase + L::kNorm + 4u * (uint32_t)f.gk);
    }
    TSK_EV(19);
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.bar(kBarQEmpty + qbb));
    return true;
  };
  Fields nx = fetch(cx.unit(0));
  ok = handover(cx.unit(0), 0, nx);
  for (int ku = 0, u = cx.unit(0); u < cx.total_units && ok; u = cx.unit(++ku)) {
    TSK_EV(8);
    TSK_TRACE_T0(tr_dec);
    ++q_iter;  // (now the next unit's index)
    const Fields cf = nx;
    if (!cf.active) {
      nx = fetch(cx.unit(ku + 1));
      ok = handover(cx.unit(ku + 1), q_iter, nx);
      continue;
    }
    const int n_kv = cf.n_kv, kv_lo = cf.kv_lo, diag0 = cf.diag0;
    const int pos = diag0 + r;  // key position of this thread's query row
    float m_used = cf.sink, l = cf.sink == -INFINITY ? 0.f : 1.f;
    TSK_TRACE_ADD(24, tr_dec);
    const float bq = cf.bq;
    // One key tile.  A slow tile computes its row maximum and raises the
    // maximum in use, m_used, when the tile exceeds it by more than
    // kRescaleThreshold (p <= 2^8 then).  A fast tile skips the maximum and
    // keeps m_used, which the bound allows while bq - m_used <= kFastLag for
    // every row of the warp (p <= 2^40).  m_used only changes in slow tiles,
    // so once a tile is fast the rest of the unit is.
    auto step = [&](int j, auto slow_tag) -> bool {
      constexpr bool kSlow = decltype(slow_tag)::value;
      const int kt = kv_lo + j;
      TSK_EV(1);
      if (!mbar_wait_warp(cx.bar(kBarSFull + t), s_cnt & 1, j == 0 ? 26 : 9, p, cx.abort))
        return false;
      TSK_EV(2);
      ++s_cnt;
      tc_fence_after();
      TSK_TRACE_T0(tr_ld);
      uint32_t sr[128];
      tmem_ld_32x32b_x128(tS, sr);  // (one 128-column load: fewer instructions than four)
      tmem_wait_ld();
      reg_fence<128>(sr);
      TSK_TRACE_ADD(20, tr_ld);
      TSK_EV(3);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(kBarSFree + t));
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      const int kbase = kt * kTileN;
      const bool edge = (kbase + kTileN - 1 > diag0) ||
                        (p.window > 0 && kbase < diag0 + kTileM - p.window);
      TSK_TRACE_T0(tr_mask);
      if (edge) {
        // Only 32-key chunks partly visible to this warp need a per-element
        // test; chunks hidden from all of its rows are cleared whole.
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
      TSK_TRACE_ADD(27, tr_mask);
      float alpha = 1.f;
      if constexpr (kSlow) {
        // Row maximum: four independent chains of 3-input max.
        TSK_TRACE_T0(tr_max);
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
        if (__any_sync(0xffffffffu, m_tile > m_used + kRescaleThreshold)) {
          if (m_tile > m_used) {
            alpha = ex2_approx(m_used - m_tile);  // m_used = -inf gives 0
            m_used = m_tile;
          }
        }
        l *= alpha;
      } else {
        // Fast tiles keep m_used, so l (and O) grow with p <= 2^kFastLag.
        // Past 2^32, m_used moves up by l's binary exponent e: l and O are
        // multiplied by 2^-e exactly, and l stays above 1, so no term the sum
        // depends on underflows.
        if (__any_sync(0xffffffffu, l > 4294967296.f)) {
          const int e = l > 4294967296.f ? ((__float_as_int(l) >> 23) & 0xFF) - 127 : 0;
          alpha = __int_as_float((127 - e) << 23);  // 2^-e
          m_used += (float)e;
          l *= alpha;
        }
      }
      TSK_EV(4);
      const float m_use = m_used == -INFINITY ? 0.f : m_used;
      TSK_TRACE_T0(tr_exp);
      // p = 2^(s*scale*log2e - m): packed FMA on column pairs, exp2 per element,
      // packed partial sums, bf16x2 packing for TMEM.
      uint32_t pk[64];
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      const uint64_t negm = f2_pack(-m_use, -m_use);
      {
        // (row sums in two packed f32x2 accumulators: one add per pair)
        uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), sl2x2, negm), x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          acc2[c & 1] = f2_add(acc2[c & 1], f2_pack(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
        float a0, a1, b0, b1;
        f2_unpack(acc2[0], a0, a1);
        f2_unpack(acc2[1], b0, b1);
        l += (a0 + b0) + (a1 + b1);
      }
      TSK_TRACE_ADD(22, tr_exp);
      TSK_EV(5);
      if (j > 0) {
        // O_t is stable and P_t reusable once PV_t(j-1) has completed.
        if (!mbar_wait_warp(cx.bar(kBarPVDone + t), pv_cnt & 1, 10, p, cx.abort)) return false;
        TSK_EV(6);
        ++pv_cnt;
        tc_fence_after();
        {
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
      }
      TSK_TRACE_T0(tr_st);
      tmem_st_32x32b_x64(tP, pk);
      tmem_wait_st();
      TSK_TRACE_ADD(23, tr_st);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(kBarPFull + t));
      TSK_EV(7);
      return true;
    };
    int j = 0;
    // Tiles with the row maximum until the bound makes it unnecessary (with a
    // sink, usually none), then tiles without it.
    for (; j < n_kv && ok; ++j) {
      if (__all_sync(0xffffffffu, m_used != -INFINITY && bq - m_used <= kFastLag)) break;
      ok = step(j, SlowTile{});
    }
    for (; j < n_kv && ok; ++j) ok = step(j, FastTile{});
    if (!ok) break;
    nx = fetch(cx.unit(ku + 1));
    ok = handover(cx.unit(ku + 1), q_iter, nx);
    if (!ok) break;
    // ------------------------------------------------------------ epilogue
    TSK_EV(9);
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
    ok = mbar_wait_warp(cx.bar(kBarPVDone + t), pv_cnt & 1, 25, p, cx.abort);
    TSK_TRACE_T0(tr_epi);
    if (!ok) break;
    TSK_EV(10);
    ++pv_cnt;
    tc_fence_after();
    uint32_t o[64];
    tmem_ld_32x32b_x64(tO, o);
    tmem_wait_ld();
    reg_fence<64>(o);
    TSK_EV(12);
    float inv = rcp_approx(l);
    if constexpr (L::kScaleOut) inv *= out_scale;
    const uint64_t inv2 = f2_pack(inv, inv);
    uint32_t ob[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      float a, b;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * c]), __uint_as_float(o[2 * c + 1])), inv2),
                a, b);
      ob[c] = pack_bf16x2(a, b);
    }
    const int row = e.y + r;  // query row, relative to the sequence's first query
    const size_t orow = (size_t)(e.x + row) * p.Hq + h;
    // (rows past the sequence's end are neither stored nor checked)
    const bool row_ok = row < e.w && TSK_IN_BOUNDS(p, cx.abort, orow < (size_t)p.q_rows * p.Hq, 45);
    if (p.lse && row_ok) p.lse[orow] = (m_used + lg2_approx(l)) * 0.69314718055994531f;
    TSK_EV(13);
    if (e.y + wq * 32 + 32 <= e.w) {
      // The warp's 32 rows lie inside the sequence: stage them in this warp's
      // slice of the staging tile and store them with one TMA bulk store.
      if (lane == 0) bulk_wait_group_read0();  // the warp's previous store has read its slice
      __syncwarp();
      TSK_EV(14);
      const uint32_t dst_row = epi + (uint32_t)r * 128u;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(dst_row + ((uint32_t)(c ^ (r & 7)) << 4), ob[4 * c], ob[4 * c + 1],
                     ob[4 * c + 2], ob[4 * c + 3]);
      fence_proxy_async_shared();
      __syncwarp();
      TSK_EV(15);
      if (lane == 0 && TSK_IN_BOUNDS(p, cx.abort,
                                     h < p.Hq && e.x + e.y + wq * 32 + 32 <= p.q_rows, 46)) {
        tma_store_3d(tmO, epi + (uint32_t)wq * 4096u, 0, h, e.x + e.y + wq * 32);
        bulk_commit_group();
      }
    } else if (row_ok) {
      uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kHeadDim);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        dst[c] = make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
    }
    tc_fence_before();
    TSK_TRACE_ADD(28, tr_epi);
    TSK_EV(11);
  }
  if (lane == 0) bulk_wait_group0();  // every output store of this warp has completed
  TSK_TRACE_ADD(30, tr_all);
}

// Softmax and epilogue of query tile t (one warpgroup, one thread per row)
// for sliding windows of at most kSmallWindowMax keys, where every query tile
// visits only a few key tiles and per-tile costs dominate.  Each row's 128
// scores are processed as two 64-column halves; 32-key chunks are classified
// per warp so that only partly visible chunks pay a per-element mask.
// Epilogue: the row is normalised, packed to bf16 and written into the warp's
// 32-row slice of a 128-byte swizzled staging tile in shared memory; lane 0
// stores the slice with one TMA bulk tensor store (box 64 x 1 x 32).  Warps
// whose rows run past the end of their sequence (rows beyond it belong to the
// next sequence) use direct per-row stores instead.
template <int QS>
__device__ __forceinline__ void role_softmax_window(const Ctx& cx, const AttnParams& p,
                                                    const CUtensorMap* tmO, int warp, int lane) {
  const int t = (warp - kFirstSoftmaxWarp) >> 2;  // query tile of this warpgroup
  const int wq = warp & 3;                         // TMEM lane quarter
  const int r = wq * 32 + lane;                    // query row within the tile
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const uint32_t tS = cx.tmem + lane_base + kColS0 + 128 * t;
  const uint32_t tO = cx.tmem + lane_base + kColO0 + 64 * t;
  const uint32_t tP = cx.tmem + lane_base + kColP0 + 64 * t;
  const uint32_t epi = cx.sbase + kSmemEpi + t * kTileBytes;
  const float sl2 = p.scale_log2;
  uint32_t s_cnt = 0, pv_cnt = 0;
  uint32_t n_staged = 0;  // staged output stores of this warp (two staging buffers)
  TSK_TL_DECL;
  TSK_TRACE_T0(tr_all);
  bool ok = true;
  // The next unit and its sink are loaded before a unit's epilogue, so that
  // their latency passes while the epilogue waits for the last PV.
  auto fetch = [&](int uu, Unit& w, float& sink) {
    if (uu >= cx.total_units) return;
    w = decode_unit<QS>(p, uu);
    const int h = tile_head<QS>(w, t);
    sink = -INFINITY;
    if (t < w.ntiles && p.sinks && TSK_IN_BOUNDS(p, cx.abort, h >= 0 && h < p.Hq, 44))
      sink = __ldg(p.sinks + h) * 1.4426950408889634f;
  };
  Unit wn;
  float sink_n = -INFINITY;
  fetch(cx.unit(0), wn, sink_n);
  for (int ku = 0, u = cx.unit(0); u < cx.total_units && ok; u = cx.unit(++ku)) {
    TSK_EV(8);
    const Unit w = wn;
    const float sink = sink_n;
    if (t >= w.ntiles) {
      fetch(cx.unit(ku + 1), wn, sink_n);
      continue;
    }
    const int h = tile_head<QS>(w, t);
    const int q0t = tile_q0<QS>(w, t);  // first query row of this tile
    const int row = q0t + r;           // query row, relative to the sequence's first query
    const int pos = w.offset + row;    // its key position
    float m_used = sink, l = sink == -INFINITY ? 0.f : 1.f;
    for (int j = 0; j < w.n_kv; ++j) {
      const int kt = w.kv_lo + j;
      TSK_EV(1);
      ok = mbar_wait_warp(cx.bar(kBarSFull + t), s_cnt & 1, j == 0 ? 26 : 9, p, cx.abort);
      if (!ok) break;
      TSK_EV(2);
      ++s_cnt;
      tc_fence_after();
      const int kbase = kt * kTileN;
      const bool edge = (kbase + kTileN - 1 > w.offset + q0t) ||
                        (p.window > 0 && kbase < w.offset + q0t + kTileM - p.window);
      ChunkMask cm{0u, 0u};
      if (edge) cm = classify_chunks(w.offset + q0t + wq * 32, kbase, p.window);
      const int hi_c = pos - kbase;
      const int lo_c = p.window > 0 ? pos - p.window + 1 - kbase : -1;
      // The row's 128 scores are processed as two halves of 64 columns, so
      // that at most one half of scores and the packed P of the other are
      // held in registers at a time.
      float alpha = 1.f;      // factor for O (both halves' rescales)
      uint32_t pk[64];        // packed bf16 P of the row
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        TSK_TRACE_T0(tr_ld);
        uint32_t sr[64];
        tmem_ld_32x32b_x64(tS + 64 * hf, sr);
        tmem_wait_ld();
        reg_fence<64>(sr);
        TSK_TRACE_ADD(20, tr_ld);
        if (hf == 1) {
          // Both halves are in registers: the MMA may overwrite S_t.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(cx.bar(kBarSFree + t));
        }
        float sv[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = __uint_as_float(sr[c]);
        // Mask: only chunks (32 keys) partly visible to this warp need a
        // per-element test; chunks hidden from the whole warp are excluded
        // from the maximum and get p = 0 through their offset below.
        TSK_TRACE_T0(tr_mask);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int k = 2 * hf + kk;
          if (cm.partial & (1u << k)) {
#pragma unroll
            for (int c = 32 * kk; c < 32 * kk + 32; ++c)
              sv[c] = (64 * hf + c > hi_c || 64 * hf + c < lo_c) ? -INFINITY : sv[c];
          }
        }
        TSK_TRACE_ADD(27, tr_mask);
        TSK_TRACE_T0(tr_max);
        float mk[2];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const float* v = sv + 32 * kk;
          float a0 = v[0], a1 = v[1];
#pragma unroll
          for (int c = 2; c < 30; c += 4) {  // columns 2..29 of the chunk
            a0 = max3f(a0, v[c], v[c + 1]);
            a1 = max3f(a1, v[c + 2], v[c + 3]);
          }
          mk[kk] = max3f(a0, a1, fmaxf(v[30], v[31]));
          if (cm.none & (1u << (2 * hf + kk))) mk[kk] = -INFINITY;
        }
        const float m_half = fmaxf(mk[0], mk[1]) * sl2;
        TSK_TRACE_ADD(21, tr_max);
        // Raise the maximum in use only when this half exceeds it by more
        // than the threshold (then l, O and an already packed first half
        // are rescaled; p <= 2^threshold otherwise).
        if (__any_sync(0xffffffffu, m_half > m_used + kRescaleThreshold)) {
          float beta = 1.f;
          if (m_half > m_used) {
            beta = ex2_approx(m_used - m_half);  // m_used = -inf gives 0
            m_used = m_half;
          }
          l *= beta;
          alpha *= beta;
          if (hf == 1 && __any_sync(0xffffffffu, beta != 1.f)) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float lo = __uint_as_float(pk[c] << 16) * beta;
              const float hi = __uint_as_float(pk[c] & 0xFFFF0000u) * beta;
              pk[c] = pack_bf16x2(lo, hi);
            }
          }
        }
        const float m_use = m_used == -INFINITY ? 0.f : m_used;
        // p = 2^(s*scale*log2e - m): packed FMA on column pairs, exp2 per
        // element, packed partial sums, bf16x2 packing.
        TSK_TRACE_T0(tr_exp);
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        uint64_t negm[2];  // -m, or -inf for chunks hidden from the whole warp
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const float nm = (cm.none & (1u << (2 * hf + kk))) ? -INFINITY : -m_use;
          negm[kk] = f2_pack(nm, nm);
        }
        uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(sv[2 * c], sv[2 * c + 1]), sl2x2, negm[c >> 4]), x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          acc2[c & 1] = f2_add(acc2[c & 1], f2_pack(p0, p1));
          pk[32 * hf + c] = pack_bf16x2(p0, p1);
        }
        float a0, a1, b0, b1;
        f2_unpack(acc2[0], a0, a1);
        f2_unpack(acc2[1], b0, b1);
        l += (a0 + b0) + (a1 + b1);
        TSK_TRACE_ADD(22, tr_exp);
      }
      TSK_EV(5);
      if (j > 0) {
        // O_t is stable and P_t reusable once PV_t(j-1) has completed.
        ok = mbar_wait_warp(cx.bar(kBarPVDone + t), pv_cnt & 1, 10, p, cx.abort);
        if (!ok) break;
        TSK_EV(6);
        ++pv_cnt;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tO + 32 * hc, o);
            tmem_wait_ld();
            reg_fence<32>(o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st_32x32b_x32(tO + 32 * hc, o);
          }
        }
      }
      TSK_TRACE_T0(tr_st);
      tmem_st_32x32b_x64(tP, pk);
      tmem_wait_st();
      TSK_TRACE_ADD(23, tr_st);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.bar(kBarPFull + t));
      TSK_EV(7);
    }
    if (!ok) break;
    fetch(cx.unit(ku + 1), wn, sink_n);
    TSK_EV(9);
    // ------------------------------------------------------------ epilogue
    TSK_TRACE_T0(tr_epi);
    ok = mbar_wait_warp(cx.bar(kBarPVDone + t), pv_cnt & 1, 25, p, cx.abort);
    if (!ok) break;
    TSK_EV(10);
    ++pv_cnt;
    tc_fence_after();
    uint32_t o[64];
    tmem_ld_32x32b_x64(tO, o);
    tmem_wait_ld();
    reg_fence<64>(o);
    TSK_EV(12);
    const float inv = rcp_approx(l);
    const uint64_t inv2 = f2_pack(inv, inv);
    uint32_t ob[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      float a, b;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * c]), __uint_as_float(o[2 * c + 1])), inv2),
                a, b);
      ob[c] = pack_bf16x2(a, b);
    }
    const size_t orow = (size_t)(w.start + row) * p.Hq + h;
    // (rows past the sequence's end are neither stored nor checked)
    const bool row_ok = row < w.len && TSK_IN_BOUNDS(p, cx.abort, orow < (size_t)p.q_rows * p.Hq, 45);
    if (p.lse && row_ok) p.lse[orow] = (m_used + lg2_approx(l)) * 0.69314718055994531f;
    TSK_EV(13);
    if (q0t + wq * 32 + 32 <= w.len) {
      // The warp's 32 rows lie inside the sequence: stage them in this warp's
      // slice of the staging tile and store them with one TMA bulk store.
      // two staging buffers: the store that used this one (two units ago)
      // has read it once at most one store group is still reading
      const uint32_t epb = epi + ((n_staged++ & 1u) ? 2u * kTileBytes : 0u);
      if (lane == 0) bulk_wait_group_read1();
      __syncwarp();
      TSK_EV(14);
      const uint32_t dst_row = epb + (uint32_t)r * 128u;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(dst_row + ((uint32_t)(c ^ (r & 7)) << 4), ob[4 * c], ob[4 * c + 1],
                     ob[4 * c + 2], ob[4 * c + 3]);
      fence_proxy_async_shared();
      __syncwarp();
      TSK_EV(15);
      if (lane == 0 && TSK_IN_BOUNDS(p, cx.abort,
                                     h < p.Hq && w.start + q0t + wq * 32 + 32 <= p.q_rows, 46)) {
        tma_store_3d(tmO, epb + (uint32_t)wq * 4096u, 0, h, w.start + q0t + wq * 32);
        bulk_commit_group();
      }
    } else if (row_ok) {
      uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kHeadDim);
#pragma unroll
      for (int c = 0; c < 8; ++c) dst[c] = make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
    }
    tc_fence_before();
    TSK_TRACE_ADD(28, tr_epi);
    TSK_EV(11);
  }
  if (lane == 0) bulk_wait_group0();  // every output store of this warp has completed
  TSK_TRACE_ADD(30, tr_all);
}

// kSmallWindow selects the softmax role for 0 < window <= kSmallWindowMax.
constexpr int kSmallWindowMax = 512;

template <bool kSmallWindow, int QS>
__global__ void __launch_bounds__(kThreads, 1)
    attention_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(cx.bar(kBarQFull + i), 1);
      // one issuer; or one per tile plus the eight softmax warps
      mbar_init(cx.bar(kBarQEmpty + i), kSmallWindow ? 1 : 2 + 2 * kSoftmaxWarpsPerTile);
      mbar_init(cx.bar(kBarSFull + i), 1);
      mbar_init(cx.bar(kBarSFree + i), kSoftmaxWarpsPerTile);
      mbar_init(cx.bar(kBarPFull + i), kSoftmaxWarpsPerTile);
      mbar_init(cx.bar(kBarPVDone + i), 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(cx.bar(kBarKFull + s), 1);
      mbar_init(cx.bar(kBarVFull + s), 1);
      mbar_init(cx.bar(kBarKVEmpty + s), kSmallWindow ? 1 : 2);
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
  // Everything above overlaps the scheduler's tail; its outputs (the unit
  // list, the tile count, the key norms) are read only after this.
  griddep_wait();
  if (warp == 3 && p.knorm)
    for (int g = lane; g < p.Hkv; g += 32) st_shared_f32(cx.sbase + kSmemNorm + 4u * g, __ldg(p.knorm + g));
  trace_init();
  trace_cta_start();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cx.tmem = *tmem_slot;
  cx.abort = smem_u32(const_cast<int*>(abort_flag));
  cx.total_units = p.ws[kWsNTiles] * p.Hkv * p.HP;
  cx.alternate = !kSmallWindow;

  if (warp == 0 && lane == 0) role_producer<QS>(cx, &tmQ, &tmK, &tmV, p);
  else if (kSmallWindow && warp == 1 && lane == 0) role_mma_pair<QS>(cx, p);
  else if (!kSmallWindow && warp == 1 && lane == 0) role_mma<QS>(cx, p, 0);
  else if (!kSmallWindow && warp == 2 && lane == 0) role_mma<QS>(cx, p, 1);
  else if (warp >= kFirstSoftmaxWarp) {
    if constexpr (kSmallWindow) role_softmax_window<QS>(cx, p, &tmO, warp, lane);
    else role_softmax_causal<QS>(cx, p, &tmO, warp, lane);
  }

  // ------------------------------------------------------------------ teardown
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

}  // namespace tsk
