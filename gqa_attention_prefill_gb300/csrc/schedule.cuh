// Varlen scheduler pre-pass: one CTA turns the sequence offsets into the list
// of query tiles (entry_rows = 128 query rows of one sequence, or 256 when a
// work unit takes two consecutive 128-row tiles of one head), each with its
// key-tile range, sorted by cost (number of key tiles) in descending order, so that
// the persistent attention kernel hands out the longest work first
// (longest-processing-time order).  Sequence s has Lq = cu[s+1] - cu[s]
// queries and Lk = cu_k[s+1] - cu_k[s] >= Lq keys; query i sits at key
// position Lk - Lq + i (plain prefill: cu_k == cu).  It checks the offsets
// (start at 0, non-decreasing, end at the totals, Lk >= Lq); on failure it
// records TSK_ERR_BAD_SEQLENS and publishes an empty list.
#pragma once
#include <cstdint>

namespace tsk {

constexpr int kSchedThreads = 1024;
constexpr int kCostBins = 4096;  // costs >= kCostBins share the top bin
constexpr int kTileM = 128;      // query rows per tile
constexpr int kTileN = 128;      // keys per tile

// Workspace words (int32) at the head of the per-stream workspace.
constexpr int kWsStatus = 0;   // [0] error code, [1] site, [2] block
constexpr int kWsNTiles = 4;   // number of query tiles in the list
constexpr int kWsNormCount = 5;  // key-norm blocks finished (reset by the last one)
constexpr int kWsDecodeBad = 6;  // decode: this call's offset check
constexpr int kWsHeader = 8;   // ints; tile offsets follow, then the int4 list (16-B aligned)

// Key-norm pre-pass (extra blocks of the scheduler launch): the largest
// Euclidean norm of the key rows of every KV head, max_t ||k[t, g, :]||, which
// bounds every score of a query row q by ||q|| * max||k||.  Run for at most
// kNormMaxHeads KV heads by at most kNormBlocks blocks; its buffer holds
// kNormBlocks * kNormMaxHeads per-block maxima, then kNormMaxHeads results.
constexpr int kNormBlocks = 148;
constexpr int kNormMaxHeads = 256;
constexpr int kNormFloats = (kNormBlocks + 1) * kNormMaxHeads;

struct KeyNorms {
  const uint4* k;  // key rows: [rows, heads, D] bf16, or nullptr (no pre-pass)
  long long rows;  // rows of the key buffer (tokens, or pool slots of a paged cache)
  int heads, D;
  float* out;      // kNormFloats floats
};

// One query tile: two int4 per entry,
//   {start_q, q0, kv_lo, len_q}  query start row, first query row of the tile
//                                (relative to start_q), first key tile, Lq
//   {start_k, offset, n_kv, 0}   key start row, Lk - Lq, number of key tiles
constexpr int kTileEntryInts = 8;

// Key tiles [kv_lo, kv_lo + n_kv) the `rows` query rows starting at q0 need.
__device__ __forceinline__ int2 qtile_key_range(int q0, int len_q, int offset, int window,
                                                int rows = kTileM) {
  const int last = (q0 + rows - 1 < len_q - 1 ? q0 + rows - 1 : len_q - 1);
  const int kv_hi = (offset + last) / kTileN;
  int kv_lo = 0;
  if (window > 0) {
    const int lo = offset + q0 - window + 1;
    kv_lo = lo > 0 ? lo / kTileN : 0;
  }
  return make_int2(kv_lo, kv_hi - kv_lo + 1);
}

// Paged key/value cache (page_size > 0): sequence s's key position x lives in
// page block_table[s * max_blocks + x / page_size], slot x % page_size.
struct PagedKV {
  const int32_t* table;
  int max_blocks;
  int page_size;  // 0: contiguous cache
  int num_pages;
};

// True when sequence s (Lk keys) has a valid page for every key.
__device__ __forceinline__ bool pages_ok(const PagedKV& pg, int s, int Lk) {
  if (pg.page_size == 0) return true;
  const int nb = (Lk + pg.page_size - 1) / pg.page_size;
  if (nb > pg.max_blocks) return false;
  for (int i = 0; i < nb; ++i) {
    const int pgi = pg.table[(size_t)s * pg.max_blocks + i];
    if (pgi < 0 || pgi >= pg.num_pages) return false;
  }
  return true;
}

// Blocks 1.. of the scheduler launch: per-head maxima of key-row norms over
// a grid-stride share of the rows; the last block to finish reduces the
// per-block maxima and resets the counter.  Eight consecutive threads read
// the eight 16-byte chunks of one key row (D = 64), so a warp reads four
// whole rows, 512 contiguous bytes, per load; the eight partial sums of a row
// are combined with shuffles (a fixed order: the result does not depend on
// the number of blocks).  Norms are non-negative, so their bit patterns order
// like the values (shared-memory integer maxima); a NaN norm orders above
// every finite one and disables the bound for its head.
__device__ void key_norm_blocks(const KeyNorms& kn, int* __restrict__ ws, int* s_max,
                                int* s_last, int blk, int nblk) {
  const int tid = threadIdx.x;
  for (int g = tid; g < kn.heads; g += kSchedThreads) s_max[g] = 0;
  __syncthreads();
  // 16-byte chunks in all (8 per row); the stride keeps tid % 8 = chunk % 8, so
  // the eight threads of a row stay together in the loop.
  const long long total = kn.rows * kn.heads * 8;
  const long long stride = (long long)nblk * kSchedThreads;
  const unsigned group = 0xFFu << (tid & 24);  // the 8 lanes sharing this thread's row
  // kUnroll loads in flight per thread (enough bytes in flight to stream HBM)
  constexpr int kUnroll = 8;
  // KV head of chunk i: (i / 8) % heads, kept incrementally (no 64-bit division
  // in the loop): the stride is a multiple of 8 chunks.
  const int hs = (int)((stride >> 3) % kn.heads);
  int h0 = (int)((((long long)blk * kSchedThreads + tid) >> 3) % kn.heads);
  for (long long i0 = (long long)blk * kSchedThreads + tid; i0 < total; i0 += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = i0 + u * stride;
      v[u] = i < total ? __ldg(kn.k + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    int h = h0;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = i0 + u * stride;
      if (i >= total) break;  // (the same for the 8 lanes of a row)
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
        acc = fmaf(lo, lo, acc);
        acc = fmaf(hi, hi, acc);
      }
      acc += __shfl_xor_sync(group, acc, 1);
      acc += __shfl_xor_sync(group, acc, 2);
      acc += __shfl_xor_sync(group, acc, 4);
      if ((tid & 7) == 0) atomicMax(&s_max[h], __float_as_int(sqrtf(acc)));
      h += hs;
      if (h >= kn.heads) h -= kn.heads;
    }
    h0 = (int)((h0 + (long long)kUnroll * hs) % kn.heads);
  }
  __syncthreads();
  for (int g = tid; g < kn.heads; g += kSchedThreads)
    kn.out[blk * kNormMaxHeads + g] = __int_as_float(s_max[g]);
  __threadfence();
  __syncthreads();
  if (tid == 0) *s_last = atomicAdd(&ws[kWsNormCount], 1) == nblk - 1;
  __syncthreads();
  if (*s_last) {
    // every (block, head) maximum read by its own thread, reduced in shared memory
    __threadfence();
    for (int g = tid; g < kn.heads; g += kSchedThreads) s_max[g] = 0;
    __syncthreads();
    for (int i = tid; i < nblk * kn.heads; i += kSchedThreads) {
      const int b = i / kn.heads, g = i - b * kn.heads;
      atomicMax(&s_max[g], __float_as_int(__ldcg(kn.out + b * kNormMaxHeads + g)));
    }
    __syncthreads();
    for (int g = tid; g < kn.heads; g += kSchedThreads)
      kn.out[kNormBlocks * kNormMaxHeads + g] = __int_as_float(s_max[g]);
    if (tid == 0) ws[kWsNormCount] = 0;
  }
}

// The key-norm pre-pass alone (gridDim.x <= kNormBlocks blocks); ws[kWsNormCount]
// must be zero at launch (the last block resets it).
__global__ void __launch_bounds__(kSchedThreads, 1) key_norm_kernel(KeyNorms kn, int* ws) {
  __shared__ int s_max[kNormMaxHeads];
  __shared__ int s_last;
  key_norm_blocks(kn, ws, s_max, &s_last, blockIdx.x, gridDim.x);
}

// Exclusive prefix sum of v over the block (every thread calls it); *total
// receives the block's sum.  Warp shuffles, then one warp over the 32 warp sums.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  static_assert(kSchedThreads == 1024, "32 warps");
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int r = (wid ? s_warp[wid - 1] : 0) + x - v;
  *total = s_warp[31];
  __syncthreads();  // (s_warp is reused by the next call)
  return r;
}

// Sequences whose offsets the scheduler block keeps in shared memory; beyond
// this it reads them (and the tile offsets) from global memory.
constexpr int kSchedSmemSeqs = 2048;

__global__ void __launch_bounds__(kSchedThreads, 1)
    schedule_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_k,
                    int num_seqs, int total_tokens, int total_keys, int window,
                    int* __restrict__ ws, int* __restrict__ tile_off, int4* __restrict__ list,
                    int max_tiles, PagedKV pg, int entry_rows, KeyNorms kn) {
  __shared__ int s_hist[kCostBins];  // cost histogram, then the bins' write cursors
  __shared__ int s_cu[kSchedSmemSeqs + 1], s_cuk[kSchedSmemSeqs + 1], s_off[kSchedSmemSeqs + 1];
  __shared__ int s_warp[32];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  // The attention kernel may be launched now: it waits for this grid's
  // completion before it reads anything this grid writes.
  griddep_launch_dependents();
  if (blockIdx.x > 0) {
    key_norm_blocks(kn, ws, s_hist, &s_bad, blockIdx.x - 1, gridDim.x - 1);
    return;
  }
  const bool small = num_seqs <= kSchedSmemSeqs;
  if (tid == 0) {
    const int c0 = cu[0], k0 = cu_k[0];
    s_bad = (c0 != 0 || cu[num_seqs] != total_tokens || k0 != 0 || cu_k[num_seqs] != total_keys)
                ? 1 : 0;
    if (small) {
      s_cu[0] = c0;
      s_cuk[0] = k0;
    }
  }
  for (int i = tid; i < kCostBins; i += kSchedThreads) s_hist[i] = 0;
  __syncthreads();  // (s_bad is set before any thread can raise it)

  // Pass A: per-sequence tile counts -> exclusive prefix over sequences.
  int base = 0;
  for (int c0 = 0; c0 < num_seqs; c0 += kSchedThreads) {
    const int s = c0 + tid;
    int nt = 0;
    if (s < num_seqs) {
      const int a = cu[s], b = cu[s + 1], ak = cu_k[s], bk = cu_k[s + 1];
      if (small) {
        s_cu[s + 1] = b;
        s_cuk[s + 1] = bk;
      }
      int L = b - a;
      const int Lk = bk - ak;
      if (L < 0 || Lk < L || !pages_ok(pg, s, Lk)) {
        s_bad = 1;
        L = 0;
      }
      nt = (L + entry_rows - 1) / entry_rows;
    }
    int chunk_total;
    const int ex = block_exclusive_scan(nt, s_warp, &chunk_total);
    if (s < num_seqs) {
      tile_off[s] = base + ex;
      if (small) s_off[s] = base + ex;
    }
    base += chunk_total;
  }
  const int n_tiles = base;
  if (tid == 0) {
    tile_off[num_seqs] = n_tiles;
    if (small) s_off[num_seqs] = n_tiles;
  }
  __syncthreads();
  if (s_bad || n_tiles > max_tiles) {
    if (tid == 0) {
      ws[kWsNTiles] = 0;
      if (atomicCAS(&ws[kWsStatus], 0, -8) == 0) ws[kWsStatus + 1] = 1000;
    }
    return;
  }

  // Tile i belongs to the last sequence whose tile offset is <= i.
  auto off_at = [&](int s) { return small ? s_off[s] : tile_off[s]; };
  auto cu_at = [&](int s) { return small ? s_cu[s] : cu[s]; };
  auto cuk_at = [&](int s) { return small ? s_cuk[s] : cu_k[s]; };
  auto seq_of = [&](int i) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (off_at(mid) <= i) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  };
  // Pass B: cost histogram.
  for (int i = tid; i < n_tiles; i += kSchedThreads) {
    const int s = seq_of(i);
    const int qt = i - off_at(s);
    const int len = cu_at(s + 1) - cu_at(s);
    const int cost =
        qtile_key_range(qt * entry_rows, len, (cuk_at(s + 1) - cuk_at(s)) - len, window, entry_rows).y;
    atomicAdd(&s_hist[min(cost, kCostBins) - 1], 1);
  }
  __syncthreads();
  // Write cursors in descending cost order: bin b starts after all bins > b.
  {
    constexpr int per = kCostBins / kSchedThreads;
    int local[per];
    int sum = 0;
#pragma unroll
    for (int k = 0; k < per; ++k) {
      local[k] = s_hist[kCostBins - 1 - (tid * per + k)];
      sum += local[k];
    }
    int total;
    int run = block_exclusive_scan(sum, s_warp, &total);  // (its barriers order the reads above)
#pragma unroll
    for (int k = 0; k < per; ++k) {
      s_hist[kCostBins - 1 - (tid * per + k)] = run;
      run += local[k];
    }
  }
  __syncthreads();
  // Pass C: scatter.
  for (int i = tid; i < n_tiles; i += kSchedThreads) {
    const int s = seq_of(i);
    const int qt = i - off_at(s);
    const int q0 = qt * entry_rows;
    const int cs = cu_at(s), len = cu_at(s + 1) - cs;
    const int cks = cuk_at(s), offset = (cuk_at(s + 1) - cks) - len;
    const int2 kr = qtile_key_range(q0, len, offset, window, entry_rows);
    const int pos = atomicAdd(&s_hist[min(kr.y, kCostBins) - 1], 1);
    list[2 * pos] = make_int4(cs, q0, kr.x, len);
    list[2 * pos + 1] = make_int4(cks, offset, kr.y, s);
  }
  if (tid == 0) ws[kWsNTiles] = n_tiles;
}

}  // namespace tsk
