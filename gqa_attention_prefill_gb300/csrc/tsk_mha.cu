// Host side of the C ABI declared in include/tsk_mha.h: argument checks,
// TMA tensor-map encoding, the per-(device, stream) workspace, and the two
// launches (scheduler pre-pass, persistent attention kernel).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "tsk_mha.h"
#include "attention.cuh"
#include "attention_d128.cuh"
#include "decode.cuh"
#include "attention_fp8.cuh"
#include "schedule.cuh"
#include "probe.cuh"

namespace {

constexpr int32_t kVersion = 100;  // 0.1.0

struct Workspace {
  int* base = nullptr;   // header ints, tile offsets, tile list
  size_t bytes = 0;
  int max_tiles = 0;
  int max_seqs = 0;
  float* part = nullptr;  // decode: per-split partial states
  size_t part_bytes = 0;
  uint8_t* fp8_v = nullptr;  // FP8 prefill: V as bf16 values
  size_t fp8_v_bytes = 0;
};

struct DeviceState {
  bool checked = false;
  bool supported = false;
  int num_sms = 0;
  bool smem_set = false;
};

std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

// Host-buffer pipeline (tsk_mha_prefill_host), one per (device, caller
// stream): its own copy and compute streams and a grow-only device buffer
// that holds the call's inputs and outputs.
struct HostPipe {
  cudaStream_t h2d = nullptr, d2h = nullptr, comp[2] = {nullptr, nullptr};
  uint8_t* buf = nullptr;
  size_t cap = 0;
};
std::mutex g_pipe_mu;  // held for a whole tsk_mha_prefill_host call (never inside g_mu)
std::map<std::pair<int, cudaStream_t>, HostPipe> g_pipe;
std::map<int, DeviceState> g_dev;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool g_profile = false;
cudaEvent_t g_ev[3] = {nullptr, nullptr, nullptr};
int g_ev_dev = -1;
bool g_ev_recorded = false;

unsigned long long g_timeout_ns = 2000000000ull;  // bounded waits give up after 2 s
int g_debug_stall = 0;
#ifdef TSK_DEBUG
int g_debug_shrink = 0;  // rows taken off the checked extent of q/out
#endif

thread_local char g_last_error[256] = "";

void note_error(const char* where, cudaError_t e) {
  snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where, cudaGetErrorName(e),
           cudaGetErrorString(e));
}

tsk_status cuda_fail(cudaError_t e, const char* where = "CUDA call") {
  note_error(where, e);
  (void)cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? TSK_ERR_OOM : TSK_ERR_DEVICE;
}

tsk_status get_encoder() {
  if (g_encode) return TSK_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return TSK_ERR_DEVICE;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return TSK_OK;
}

// [T, H, D] bf16 viewed as a 3-D tensor (d, head, token); box = 64 x 1 x
// box_rows: rows of 128 bytes (64 of the D columns), stored with the 128-byte
// swizzle.  D = 128 rows are read as two boxes at d = 0 and d = 64.
tsk_status encode_thd(CUtensorMap* m, const void* ptr, int64_t T, int H, int D,
                      int box_rows = 128) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TSK_OK : TSK_ERR_DEVICE;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  auto x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

tsk_status check_device(int* dev_out, DeviceState** st_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail(cudaErrorNoDevice);
  DeviceState& st = g_dev[dev];
  if (!st.checked) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cuda_fail(cudaErrorInvalidDevice);
    st.supported = (major == 10 && minor == 3);
    st.checked = true;
  }
  if (!st.supported) return TSK_ERR_DEVICE;
  if (!st.smem_set) {
    constexpr int kQS = tsk::kTileM;  // units of two row blocks of one head
    cudaError_t e = cudaFuncSetAttribute(tsk::attention_fwd_kernel<false, 0>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)tsk::kSmemBytesCausal);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tsk::attention_fwd_kernel<true, 0>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tsk::kSmemBytesWindow);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tsk::attention_fwd_kernel<false, kQS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tsk::kSmemBytesCausal);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tsk::attention_fwd_kernel<true, kQS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tsk::kSmemBytesWindow);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tsk::d128::attention_fwd_d128_kernel<0>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tsk::d128::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tsk::d128::attention_fwd_d128_kernel<kQS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tsk::d128::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tsk::d128::attention_fwd_d128_kernel<0, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tsk::d128::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tsk::fp8::attention_fwd_fp8_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tsk::fp8::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tsk::dec::decode_split_kernel<64>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tsk::dec::smem_bytes<64>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tsk::dec::decode_split_kernel<128>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tsk::dec::smem_bytes<128>());
    if (e != cudaSuccess) return cuda_fail(e);
    st.smem_set = true;
  }
  *dev_out = dev;
  *st_out = &st;
  return TSK_OK;
}

tsk_status get_workspace(int dev, cudaStream_t stream, int max_tiles, int num_seqs,
                         Workspace** out) {
  Workspace& w = g_ws[{dev, stream}];
  if (w.base && w.max_tiles >= max_tiles && w.max_seqs >= num_seqs) {
    *out = &w;
    return TSK_OK;
  }
  int mt = max_tiles > w.max_tiles ? max_tiles : w.max_tiles;
  int ms = num_seqs > w.max_seqs ? num_seqs : w.max_seqs;
  mt = mt < 1024 ? 1024 : mt;
  ms = ms < 1024 ? 1024 : ms;
  size_t off_ints = ((size_t)tsk::kWsHeader + (size_t)ms + 1 + 3) & ~(size_t)3;
  size_t bytes = off_ints * 4 + (size_t)mt * 4 * tsk::kTileEntryInts + tsk::kNormFloats * 4;
  int* nb = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&nb), bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemsetAsync(nb, 0, bytes, stream);
  if (e != cudaSuccess) {
    cudaFreeAsync(nb, stream);
    return cuda_fail(e);
  }
  if (w.base) {
    // Carry a pending device error over to the new buffer, then retire the old one.
    cudaMemcpyAsync(nb, w.base, tsk::kWsHeader * 4, cudaMemcpyDeviceToDevice, stream);
    cudaFreeAsync(w.base, stream);
  }
  w.base = nb;
  w.bytes = bytes;
  w.max_tiles = mt;
  w.max_seqs = ms;
  *out = &w;
  return TSK_OK;
}

}  // namespace

extern "C" {

const char* tsk_status_string(tsk_status s) {
  switch (s) {
    case TSK_OK: return "ok";
    case TSK_ERR_INVALID_ARG: return "invalid argument";
    case TSK_ERR_UNSUPPORTED: return "unsupported shape or size";
    case TSK_ERR_ALIGNMENT: return "misaligned pointer";
    case TSK_ERR_DEVICE: return "device error or unsupported device (needs compute capability 10.3)";
    case TSK_ERR_OOM: return "out of device memory";
    case TSK_ERR_LAUNCH: return "kernel launch failed";
    case TSK_ERR_DEVICE_TIMEOUT: return "device-side bounded wait expired";
    case TSK_ERR_BAD_SEQLENS: return "cu_seqlens inconsistent with total_tokens";
    case TSK_ERR_BOUNDS: return "index or TMA coordinate out of bounds (debug build; access skipped)";
  }
  return "unknown status";
}

int32_t tsk_version(void) { return kVersion; }

const char* tsk_last_error(void) { return g_last_error; }

tsk_status tsk_debug_trace(unsigned long long* out, int32_t n) {
#ifdef TSK_TRACE
  if (!out || n <= 0) return TSK_ERR_INVALID_ARG;
  constexpr int kSites = 2 * tsk::kTraceSites;
  unsigned long long buf[kSites + tsk::kTraceCtas];
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(buf, tsk::g_tsk_trace, kSites * 8);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(buf + kSites, tsk::g_tsk_cta_ns, tsk::kTraceCtas * 8);
  if (e != cudaSuccess) return cuda_fail(e, "trace read");
  const int m = n < kSites + tsk::kTraceCtas ? n : kSites + tsk::kTraceCtas;
  for (int i = 0; i < m; ++i) out[i] = buf[i];
  unsigned long long zero[kSites] = {};
  e = cudaMemcpyToSymbol(tsk::g_tsk_trace, zero, sizeof zero);
  return e == cudaSuccess ? TSK_OK : cuda_fail(e, "trace clear");
#else
  (void)out;
  (void)n;
  return TSK_ERR_UNSUPPORTED;
#endif
}

tsk_status tsk_debug_timeline(unsigned long long* out, int32_t n) {
#ifdef TSK_TIMELINE
  if (!out || n <= 0) return TSK_ERR_INVALID_ARG;
  const size_t total = (size_t)tsk::kTlWarps * tsk::kTlCap;
  const size_t m = (size_t)n < total ? (size_t)n : total;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(out, tsk::g_tsk_tl, m * 8);
  if (e != cudaSuccess) return cuda_fail(e, "timeline read");
  static unsigned long long zero[tsk::kTlCap] = {};
  for (int w = 0; w < tsk::kTlWarps && e == cudaSuccess; ++w)
    e = cudaMemcpyToSymbol(tsk::g_tsk_tl, zero, sizeof zero, (size_t)w * sizeof zero);
  return e == cudaSuccess ? TSK_OK : cuda_fail(e, "timeline clear");
#else
  (void)out;
  (void)n;
  return TSK_ERR_UNSUPPORTED;
#endif
}

int32_t tsk_kernels_per_call(void) { return 2; }

// Exponential-unit throughput of the current device (one warm-up launch,
// then one launch timed with CUDA events on `stream`).
tsk_status tsk_bench_ex2_rate(double* ex2_per_second, tsk_stream_t stream_) {
  if (!ex2_per_second) return TSK_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = -1, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cuda_fail(cudaErrorNoDevice);
  constexpr int kIters = 1 << 14;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)
    return cuda_fail(cudaErrorUnknown, "tsk_bench_ex2_rate: events");
  tsk::ex2_rate_kernel<<<sms, tsk::kEx2ProbeThreads, 0, stream>>>(kIters / 8);
  cudaEventRecord(e0, stream);
  tsk::ex2_rate_kernel<<<sms, tsk::kEx2ProbeThreads, 0, stream>>>(kIters);
  cudaEventRecord(e1, stream);
  cudaError_t e = cudaEventSynchronize(e1);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess || !(ms > 0.f)) return cuda_fail(e, "tsk_bench_ex2_rate");
  *ex2_per_second = (double)sms * tsk::kEx2ProbeThreads * tsk::kEx2ProbeChains * kIters /
                    (ms * 1e-3);
  return TSK_OK;
}

}  // extern "C"

namespace {

// The attention kernel for head dimension D (64 or 128), the window and the
// unit layout (qstep: 0 = two heads of a group over the same rows, kTileM =
// two row blocks of one head).
// The D = 64 kernels follow the scheduler on the stream with programmatic
// stream serialisation: their CTAs may start (barrier set-up, TMEM
// allocation) while the scheduler finishes, and wait for its results on the
// device.
template <int QS>
void launch_attention_qs(int D, int window, int grid, const CUtensorMap& tq,
                         const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                         const tsk::AttnParams& p, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(tsk::kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (D == 128) {  // (an ordinary launch: 1.3% faster here than with the attribute)
    tsk::d128::attention_fwd_d128_kernel<QS>
        <<<grid, tsk::kThreads, tsk::d128::kSmemBytes, stream>>>(tq, tk, tv, to, p);
  } else if (window > 0 && window <= tsk::kSmallWindowMax) {
    cfg.dynamicSmemBytes = tsk::kSmemBytesWindow;
    cudaLaunchKernelEx(&cfg, tsk::attention_fwd_kernel<true, QS>, tq, tk, tv, to, p);
  } else {
    cfg.dynamicSmemBytes = tsk::kSmemBytesCausal;
    cudaLaunchKernelEx(&cfg, tsk::attention_fwd_kernel<false, QS>, tq, tk, tv, to, p);
  }
}
void launch_attention(int D, int window, int qstep, int grid, const CUtensorMap& tq,
                      const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                      const tsk::AttnParams& p, cudaStream_t stream) {
  if (qstep) launch_attention_qs<tsk::kTileM>(D, window, grid, tq, tk, tv, to, p, stream);
  else launch_attention_qs<0>(D, window, grid, tq, tk, tv, to, p, stream);
}

// The key-norm pre-pass (extra scheduler blocks) for a D = 64 prefill: the
// kernel bounds every score of a row by its query norm times the largest
// key norm of the KV head and skips the row maximum while that bound allows
// it (the D = 128 kernel keeps computing it: there the extra state of the
// bound spilled registers and cost 18-23%).  Returns the number of extra
// blocks (0: no bound; too many KV heads).
int key_norm_setup(tsk::KeyNorms* kn, const void* k, int64_t rows, int Hkv, int D, int window,
                   float* out) {
  *kn = tsk::KeyNorms{nullptr, 0, 0, 0, nullptr};
  // (the small-window softmax always computes its row maxima: no bound needed)
  if (D != 64 || Hkv > tsk::kNormMaxHeads || rows <= 0 ||
      (window > 0 && window <= tsk::kSmallWindowMax))
    return 0;
  *kn = tsk::KeyNorms{reinterpret_cast<const uint4*>(k), (long long)rows, Hkv, D, out};
  // about eight 16-byte chunks per thread (one round of loads), at most
  // kNormBlocks blocks
  const int64_t want = (rows * Hkv * 8 + 8 * tsk::kSchedThreads - 1) / (8 * tsk::kSchedThreads);
  return (int)(want < tsk::kNormBlocks ? (want < 1 ? 1 : want) : tsk::kNormBlocks);
}

// Shared by tsk_mha_prefill (cu_k == cu_q, total_keys == total_queries) and
// tsk_mha_prefill_kvcache.
// Host checks of a paged cache description; rows = cache rows it spans.
tsk_status check_paged(const int32_t* table, int32_t max_blocks, int32_t page_size,
                       int32_t num_pages, int32_t num_seqs, int32_t Hkv, int64_t* rows) {
  if (!table || max_blocks < 1 || num_pages < 1) return TSK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(table) & 3) != 0) return TSK_ERR_ALIGNMENT;
  if (page_size < 8 || page_size % 8 != 0 || (page_size % 128 != 0 && 128 % page_size != 0))
    return TSK_ERR_UNSUPPORTED;
  *rows = (int64_t)num_pages * page_size;
  if (*rows * Hkv >= ((int64_t)1 << 31) || (int64_t)num_seqs * max_blocks >= ((int64_t)1 << 31))
    return TSK_ERR_UNSUPPORTED;
  return TSK_OK;
}

tsk_status prefill_impl(const void* q, const void* k, const void* v, const float* sinks,
                        const int32_t* cu_q, const int32_t* cu_k, int32_t num_seqs,
                        int64_t total_q, int64_t total_k, int32_t Hq, int32_t Hkv, int32_t D,
                        int32_t window, float scale, void* out, float* lse,
                        cudaStream_t stream, const char* what, const int32_t* block_table = nullptr,
                        int32_t max_blocks = 0, int32_t page_size = 0, int32_t num_pages = 0,
                        const float* knorm_ext = nullptr) {
  // ---- host-only checks (no CUDA call before these pass)
  if (!q || !k || !v || !out || !cu_q || !cu_k) return TSK_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_q < 0 || total_k < 0 || Hq <= 0 || Hkv <= 0)
    return TSK_ERR_INVALID_ARG;
  if (total_k < total_q) return TSK_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return TSK_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || Hq % Hkv != 0) return TSK_ERR_UNSUPPORTED;
  if (num_seqs >= (1 << 24) || total_q * (int64_t)Hq >= ((int64_t)1 << 31) ||
      total_k * (int64_t)Hkv >= ((int64_t)1 << 31))
    return TSK_ERR_UNSUPPORTED;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; };
  if (!a16(q) || !a16(k) || !a16(v) || !a16(out)) return TSK_ERR_ALIGNMENT;
  if (!a4(cu_q) || !a4(cu_k) || (sinks && !a4(sinks)) || (lse && !a4(lse)))
    return TSK_ERR_ALIGNMENT;
  int64_t kv_rows = total_k;  // rows of the k and v buffers
  if (page_size != 0) {
    tsk_status pst = check_paged(block_table, max_blocks, page_size, num_pages, num_seqs, Hkv, &kv_rows);
    if (pst != TSK_OK) return pst;
  }
  const size_t qo_bytes = (size_t)total_q * Hq * D * 2;
  const size_t kv_bytes = (size_t)kv_rows * Hkv * D * 2;
  if (total_q > 0 && (overlaps(out, qo_bytes, q, qo_bytes) || overlaps(out, qo_bytes, k, kv_bytes) ||
                      overlaps(out, qo_bytes, v, kv_bytes)))
    return TSK_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_q == 0) return TSK_OK;
  const tsk::PagedKV pg{block_table, max_blocks, page_size, num_pages};
  const int kv_box = page_size != 0 && page_size < 128 ? page_size : 128;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = -1;
  DeviceState* ds = nullptr;
  tsk_status st = check_device(&dev, &ds);
  if (st != TSK_OK) return st;
  if ((st = get_encoder()) != TSK_OK) return st;

  const int64_t max_tiles64 = total_q / tsk::kTileM + num_seqs + 1;
  const int max_tiles = (int)max_tiles64;
  Workspace* ws = nullptr;
  if ((st = get_workspace(dev, stream, max_tiles, num_seqs, &ws)) != TSK_OK) return st;

  CUtensorMap tq, tk, tv, to;
  if ((st = encode_thd(&tq, q, total_q, Hq, D)) != TSK_OK) return st;
  if ((st = encode_thd(&tk, k, kv_rows, Hkv, D, kv_box)) != TSK_OK) return st;
  if ((st = encode_thd(&tv, v, kv_rows, Hkv, D, kv_box)) != TSK_OK) return st;
  if ((st = encode_thd(&to, out, total_q, Hq, D, 32)) != TSK_OK) return st;

  char name[112];
  snprintf(name, sizeof name, "%s[Hq=%d,Hkv=%d,D=%d,W=%d,nseq=%d,Tq=%lld,Tk=%lld]", what, Hq,
           Hkv, D, window, num_seqs, (long long)total_q, (long long)total_k);
  nvtxRangePushA(name);

  const size_t off_ints = ((size_t)tsk::kWsHeader + (size_t)ws->max_seqs + 1 + 3) & ~(size_t)3;
  int* tile_off = ws->base + tsk::kWsHeader;
  int4* list = reinterpret_cast<int4*>(ws->base + off_ints);

  const bool prof = g_profile;
  if (prof) {
    if (g_ev_dev != dev) {
      for (auto& e : g_ev) {
        if (e) cudaEventDestroy(e);
        e = nullptr;
      }
      for (auto& e : g_ev)
        if (cudaEventCreate(&e) != cudaSuccess) {
          nvtxRangePop();
          return TSK_ERR_DEVICE;
        }
      g_ev_dev = dev;
    }
    cudaEventRecord(g_ev[0], stream);
  }
  // With one query head per KV head, a unit takes two consecutive 128-row
  // tiles of one head (list entries of 256 rows); else two heads of a group.
  const int qstep = Hq == Hkv ? tsk::kTileM : 0;
  float* knorm = reinterpret_cast<float*>(ws->base + off_ints + (size_t)ws->max_tiles * tsk::kTileEntryInts);
  tsk::KeyNorms kn;
  // (knorm_ext: bounds the caller computed over a larger key set)
  const int norm_blocks = knorm_ext ? 0 : key_norm_setup(&kn, k, kv_rows, Hkv, D, window, knorm);
  if (knorm_ext) kn = tsk::KeyNorms{nullptr, 0, 0, 0, nullptr};
  tsk::schedule_kernel<<<1 + norm_blocks, tsk::kSchedThreads, 0, stream>>>(
      cu_q, cu_k, num_seqs, (int)total_q, (int)total_k, window, ws->base, tile_off, list,
      ws->max_tiles, pg, tsk::kTileM + qstep, kn);
  if (prof) cudaEventRecord(g_ev[1], stream);

  tsk::AttnParams p;
  p.sinks = sinks;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.list = list;
  p.ws = ws->base;
  p.status = ws->base + tsk::kWsStatus;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.HP = (p.G + 1) / 2;
  p.window = window;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = g_timeout_ns;
  p.debug_stall = g_debug_stall;
  p.kv = pg;
  p.q_rows = (int)total_q;
#ifdef TSK_DEBUG
  p.q_rows -= g_debug_shrink;
#endif
  p.kv_rows = (int)kv_rows;
  p.max_tiles = ws->max_tiles;
  p.knorm = knorm_ext ? knorm_ext
                      : norm_blocks ? knorm + tsk::kNormBlocks * tsk::kNormMaxHeads : nullptr;
  const int64_t units_bound = max_tiles64 * Hkv * p.HP;
  const int grid = (int)(units_bound < ds->num_sms ? units_bound : ds->num_sms);
  launch_attention(D, window, qstep, grid, tq, tk, tv, to, p, stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) note_error("attention kernel launch", e);
  if (prof) {
    cudaEventRecord(g_ev[2], stream);
    g_ev_recorded = true;
  }
  nvtxRangePop();
  return e == cudaSuccess ? TSK_OK : TSK_ERR_LAUNCH;
}

}  // namespace

extern "C" {

tsk_status tsk_mha_prefill(const void* q, const void* k, const void* v, const float* sinks,
                           const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                           int32_t Hq, int32_t Hkv, int32_t D, int32_t window, float scale,
                           void* out, float* lse, tsk_stream_t stream) {
  return prefill_impl(q, k, v, sinks, cu_seqlens, cu_seqlens, num_seqs, total_tokens,
                      total_tokens, Hq, Hkv, D, window, scale, out, lse,
                      reinterpret_cast<cudaStream_t>(stream), "tsk_mha_prefill");
}

tsk_status tsk_mha_prefill_kvcache(const void* q, const void* k, const void* v,
                                   const float* sinks, const int32_t* cu_seqlens_q,
                                   const int32_t* cu_seqlens_k, int32_t num_seqs,
                                   int64_t total_q, int64_t total_k, int32_t Hq, int32_t Hkv,
                                   int32_t D, int32_t window, float scale, void* out,
                                   float* lse, tsk_stream_t stream) {
  return prefill_impl(q, k, v, sinks, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                      Hq, Hkv, D, window, scale, out, lse,
                      reinterpret_cast<cudaStream_t>(stream), "tsk_mha_prefill_kvcache");
}

tsk_status tsk_mha_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                                 const float* sinks, const int32_t* cu_seqlens_q,
                                 const int32_t* cu_seqlens_k, const int32_t* block_table,
                                 int32_t max_blocks_per_seq, int32_t page_size, int32_t num_pages,
                                 int32_t num_seqs, int64_t total_q, int64_t total_k, int32_t Hq,
                                 int32_t Hkv, int32_t D, int32_t window, float scale, void* out,
                                 float* lse, tsk_stream_t stream) {
  if (page_size == 0) return TSK_ERR_UNSUPPORTED;
  return prefill_impl(q, k_pages, v_pages, sinks, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q,
                      total_k, Hq, Hkv, D, window, scale, out, lse,
                      reinterpret_cast<cudaStream_t>(stream), "tsk_mha_prefill_paged",
                      block_table, max_blocks_per_seq, page_size, num_pages);
}

tsk_status tsk_get_device_status(tsk_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TSK_ERR_DEVICE;
  auto it = g_ws.find({dev, stream});
  if (it == g_ws.end() || !it->second.base) return TSK_OK;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
  int hdr[4] = {0, 0, 0, 0};
  if (cudaMemcpy(hdr, it->second.base, sizeof hdr, cudaMemcpyDeviceToHost) != cudaSuccess)
    return cuda_fail(cudaErrorUnknown);
  if (hdr[0] != 0) {
    snprintf(g_last_error, sizeof g_last_error, "device status %d at site %d, block %d", hdr[0],
             hdr[1], hdr[2]);
    int zero[4] = {0, 0, 0, 0};
    cudaMemcpy(it->second.base, zero, sizeof zero, cudaMemcpyHostToDevice);
  }
  return (tsk_status)hdr[0];
}

tsk_status tsk_profile_enable(int enable) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_profile = enable != 0;
  return TSK_OK;
}

tsk_status tsk_profile_read(float* prepass_ms, float* attention_ms) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ev_recorded) return TSK_ERR_INVALID_ARG;
  if (cudaEventSynchronize(g_ev[2]) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
  float a = 0.f, b = 0.f;
  if (cudaEventElapsedTime(&a, g_ev[0], g_ev[1]) != cudaSuccess ||
      cudaEventElapsedTime(&b, g_ev[1], g_ev[2]) != cudaSuccess)
    return cuda_fail(cudaErrorUnknown);
  if (prepass_ms) *prepass_ms = a;
  if (attention_ms) *attention_ms = b;
  return TSK_OK;
}

tsk_status tsk_release(void) {
  std::lock_guard<std::mutex> plock(g_pipe_mu);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = -1;
  if ((!g_ws.empty() || !g_pipe.empty()) && cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceSynchronize();
  for (auto& kv : g_pipe) {
    HostPipe& hp = kv.second;
    cudaSetDevice(kv.first.first);  // (the device was synchronised above)
    if (hp.buf) cudaFree(hp.buf);
    for (cudaStream_t st : {hp.h2d, hp.d2h, hp.comp[0], hp.comp[1]}) {
      auto it = g_ws.find({kv.first.first, st});
      if (it != g_ws.end()) {
        if (it->second.base) cudaFree(it->second.base);
        if (it->second.part) cudaFree(it->second.part);
        if (it->second.fp8_v) cudaFree(it->second.fp8_v);
        g_ws.erase(it);
      }
      if (st) cudaStreamDestroy(st);
    }
  }
  g_pipe.clear();
  for (auto& kv : g_ws) {
    if (kv.second.base || kv.second.part) cudaSetDevice(kv.first.first);
    if (kv.second.base) cudaFree(kv.second.base);
    if (kv.second.part) cudaFree(kv.second.part);
    if (kv.second.fp8_v) cudaFree(kv.second.fp8_v);
  }
  if (dev >= 0) cudaSetDevice(dev);
  g_ws.clear();
  return TSK_OK;
}

// Test hook of builds with -DTSK_DEBUG: checks of later prefill calls use a
// q/out extent `rows` smaller than the real one.
tsk_status tsk_debug_shrink_extent(int32_t rows) {
#ifdef TSK_DEBUG
  std::lock_guard<std::mutex> lock(g_mu);
  if (rows < 0) return TSK_ERR_INVALID_ARG;
  g_debug_shrink = rows;
  return TSK_OK;
#else
  (void)rows;
  return TSK_ERR_UNSUPPORTED;
#endif
}

// Test hook: wait limit for later calls (0 = default 2 s) and stall injection.
tsk_status tsk_debug_set_wait(unsigned long long timeout_ns, int stall) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_timeout_ns = timeout_ns ? timeout_ns : 2000000000ull;
  g_debug_stall = stall ? 1 : 0;
  return TSK_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant.
//
// Some callers must not allocate device memory at call time: code running
// under an allocator they do not control (a serving engine that owns the
// whole memory pool), real-time paths where cudaMalloc's implicit
// synchronisation is unacceptable, or hosts that forbid allocation after
// start-up.  For them, tsk_mha_prefill_noalloc keeps its scratch (status
// words, per-sequence tile offsets, sorted query-tile list) in the
// file-scope array below, which every GPU that loads this library holds
// until the process exits.  Its device address is looked up once per device
// (cudaGetSymbolAddress on the first call made with that device current).
namespace {

constexpr int kNoAllocMaxSeqs = 16384;    // sequences per call
constexpr int kNoAllocMaxTiles = 49152;   // total_tokens/128 + num_seqs + 1, at most
constexpr size_t kNoAllocOffInts =
    ((size_t)tsk::kWsHeader + (size_t)kNoAllocMaxSeqs + 1 + 3) & ~(size_t)3;
constexpr size_t kNoAllocBytes = kNoAllocOffInts * 4 +
                                 (size_t)kNoAllocMaxTiles * 4 * tsk::kTileEntryInts +
                                 tsk::kNormFloats * 4;  // ~1.8 MB

static __device__ __align__(256) int g_noalloc_scratch[kNoAllocBytes / 4];

std::map<int, int*> g_noalloc_ptr;  // device -> device address of g_noalloc_scratch

}  // namespace

extern "C" tsk_status tsk_mha_prefill_noalloc(const void* q, const void* k, const void* v,
                                              const float* sinks, const int32_t* cu_seqlens,
                                              int32_t num_seqs, int64_t total_tokens, int32_t Hq,
                                              int32_t Hkv, int32_t D, int32_t window,
                                              float scale, void* out, float* lse,
                                              tsk_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // Same host-side checks as tsk_mha_prefill, plus the scratch limits.
  if (!q || !k || !v || !out || !cu_seqlens) return TSK_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_tokens < 0 || Hq <= 0 || Hkv <= 0) return TSK_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return TSK_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || Hq % Hkv != 0) return TSK_ERR_UNSUPPORTED;
  if (num_seqs >= (1 << 24) || total_tokens * (int64_t)Hq >= ((int64_t)1 << 31))
    return TSK_ERR_UNSUPPORTED;
  const int64_t max_tiles64 = total_tokens / tsk::kTileM + num_seqs + 1;
  if (num_seqs > kNoAllocMaxSeqs || max_tiles64 > kNoAllocMaxTiles) {
    snprintf(g_last_error, sizeof g_last_error,
             "tsk_mha_prefill_noalloc: problem exceeds the fixed scratch (num_seqs %d > %d or "
             "total_tokens/128 + num_seqs + 1 = %lld > %d)",
             num_seqs, kNoAllocMaxSeqs, (long long)max_tiles64, kNoAllocMaxTiles);
    return TSK_ERR_UNSUPPORTED;
  }
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; };
  if (!a16(q) || !a16(k) || !a16(v) || !a16(out)) return TSK_ERR_ALIGNMENT;
  if (!a4(cu_seqlens) || (sinks && !a4(sinks)) || (lse && !a4(lse))) return TSK_ERR_ALIGNMENT;
  const size_t qo_bytes = (size_t)total_tokens * Hq * D * 2;
  const size_t kv_bytes = (size_t)total_tokens * Hkv * D * 2;
  if (total_tokens > 0 && (overlaps(out, qo_bytes, q, qo_bytes) ||
                           overlaps(out, qo_bytes, k, kv_bytes) ||
                           overlaps(out, qo_bytes, v, kv_bytes)))
    return TSK_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_tokens == 0) return TSK_OK;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = -1;
  DeviceState* ds = nullptr;
  tsk_status st = check_device(&dev, &ds);
  if (st != TSK_OK) return st;
  if ((st = get_encoder()) != TSK_OK) return st;
  int*& scratch = g_noalloc_ptr[dev];
  if (!scratch) {
    // The array's name is a host-side stand-in; the device address must be
    // looked up with this device current.
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    scratch = static_cast<int*>(ptr);
  }

  CUtensorMap tq, tk, tv, to;
  if ((st = encode_thd(&tq, q, total_tokens, Hq, D)) != TSK_OK) return st;
  if ((st = encode_thd(&tk, k, total_tokens, Hkv, D)) != TSK_OK) return st;
  if ((st = encode_thd(&tv, v, total_tokens, Hkv, D)) != TSK_OK) return st;
  if ((st = encode_thd(&to, out, total_tokens, Hq, D, 32)) != TSK_OK) return st;

  int* tile_off = scratch + tsk::kWsHeader;
  int4* list = reinterpret_cast<int4*>(scratch + kNoAllocOffInts);
  // The array keeps the previous call's contents; the status words and the
  // tile count must start at zero.
  cudaError_t e = cudaMemsetAsync(scratch, 0, tsk::kWsHeader * sizeof(int), stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the no-alloc scratch header");
  const int qstep = Hq == Hkv ? tsk::kTileM : 0;  // see prefill_impl
  float* knorm = reinterpret_cast<float*>(scratch + kNoAllocOffInts +
                                          (size_t)kNoAllocMaxTiles * tsk::kTileEntryInts);
  tsk::KeyNorms kn;
  const int norm_blocks = key_norm_setup(&kn, k, total_tokens, Hkv, D, window, knorm);
  tsk::schedule_kernel<<<1 + norm_blocks, tsk::kSchedThreads, 0, stream>>>(
      cu_seqlens, cu_seqlens, num_seqs, (int)total_tokens, (int)total_tokens, window, scratch,
      tile_off, list, kNoAllocMaxTiles, tsk::PagedKV{nullptr, 0, 0, 0}, tsk::kTileM + qstep, kn);

  tsk::AttnParams p;
  p.sinks = sinks;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.list = list;
  p.ws = scratch;
  p.status = scratch + tsk::kWsStatus;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.HP = (p.G + 1) / 2;
  p.window = window;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = g_timeout_ns;
  p.debug_stall = 0;
  p.kv = tsk::PagedKV{nullptr, 0, 0, 0};
  p.q_rows = (int)total_tokens;
  p.kv_rows = (int)total_tokens;
  p.max_tiles = kNoAllocMaxTiles;
  p.knorm = norm_blocks ? knorm + tsk::kNormBlocks * tsk::kNormMaxHeads : nullptr;
  const int64_t units_bound = max_tiles64 * Hkv * p.HP;
  const int grid = (int)(units_bound < ds->num_sms ? units_bound : ds->num_sms);
  launch_attention(D, window, qstep, grid, tq, tk, tv, to, p, stream);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    note_error("attention kernel launch (no-alloc)", e);
    return TSK_ERR_LAUNCH;
  }
  return TSK_OK;
}

// Status words of the allocation-free call: the array holds those of the
// most recent call on the current device (each call clears them first).
extern "C" tsk_status tsk_noalloc_status(tsk_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return TSK_ERR_DEVICE;
    auto it = g_noalloc_ptr.find(dev);
    if (it == g_noalloc_ptr.end() || !it->second) return TSK_OK;  // no call on this device yet
    scratch = it->second;
  }
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "tsk_noalloc_status: stream synchronise");
  int hdr[4] = {0, 0, 0, 0};
  e = cudaMemcpy(hdr, scratch + tsk::kWsStatus, sizeof hdr, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "tsk_noalloc_status: read");
  if (hdr[0] != 0) {
    const int zero[4] = {0, 0, 0, 0};
    e = cudaMemcpy(scratch + tsk::kWsStatus, zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "tsk_noalloc_status: clear");
  }
  return (tsk_status)hdr[0];
}

// ---------------------------------------------------------------------------
// Decode over a key/value cache (one query token per sequence).
namespace {
tsk_status decode_impl(const void* q, const void* k, const void* v, const float* sinks,
                       const int32_t* cu_seqlens_k, int32_t num_seqs, int64_t total_k,
                       int32_t max_seqlen_k, int32_t Hq, int32_t Hkv, int32_t D, int32_t window,
                       float scale, void* out, float* lse, cudaStream_t stream, const char* what,
                       const int32_t* block_table, int32_t max_blocks, int32_t page_size,
                       int32_t num_pages) {
  if (!q || !k || !v || !out || !cu_seqlens_k) return TSK_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_k < 0 || Hq <= 0 || Hkv <= 0) return TSK_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return TSK_ERR_INVALID_ARG;
  if (num_seqs > 0 && (max_seqlen_k < 1 || (int64_t)max_seqlen_k > total_k ||
                       total_k < (int64_t)num_seqs))
    return TSK_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || Hq % Hkv != 0) return TSK_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || total_k * (int64_t)Hkv >= ((int64_t)1 << 31) ||
      (int64_t)num_seqs * Hq >= ((int64_t)1 << 31))
    return TSK_ERR_UNSUPPORTED;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; };
  if (!a16(q) || !a16(k) || !a16(v) || !a16(out)) return TSK_ERR_ALIGNMENT;
  if (!a4(cu_seqlens_k) || (sinks && !a4(sinks)) || (lse && !a4(lse))) return TSK_ERR_ALIGNMENT;
  int64_t kv_rows = total_k;
  if (page_size != 0) {
    tsk_status pst = check_paged(block_table, max_blocks, page_size, num_pages, num_seqs, Hkv, &kv_rows);
    if (pst != TSK_OK) return pst;
  }
  const size_t qo_bytes = (size_t)num_seqs * Hq * D * 2;
  const size_t kv_bytes = (size_t)kv_rows * Hkv * D * 2;
  if (num_seqs > 0 && (overlaps(out, qo_bytes, q, qo_bytes) || overlaps(out, qo_bytes, k, kv_bytes) ||
                       overlaps(out, qo_bytes, v, kv_bytes)))
    return TSK_ERR_INVALID_ARG;
  if (num_seqs == 0) return TSK_OK;
  const tsk::PagedKV pg{block_table, max_blocks, page_size, num_pages};
  const int kv_box = page_size != 0 && page_size < 128 ? page_size : 128;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = -1;
  DeviceState* ds = nullptr;
  tsk_status st = check_device(&dev, &ds);
  if (st != TSK_OK) return st;
  if ((st = get_encoder()) != TSK_OK) return st;
  Workspace* ws = nullptr;
  if ((st = get_workspace(dev, stream, 1024, 1024, &ws)) != TSK_OK) return st;

  // Key splits: enough CTAs for about two waves at the kernel's occupancy.
  const int G = Hq / Hkv;
  const int n_hb = (G + tsk::dec::kRows - 1) / tsk::dec::kRows;
  // Tiles start at multiples of 128 key positions, so a window's span can
  // touch one tile more than its length needs.
  const bool windowed = window > 0 && window < max_seqlen_k;
  const int span = windowed ? window : max_seqlen_k;
  const int n_tiles = (span + tsk::dec::kKeys - 1) / tsk::dec::kKeys + (windowed ? 1 : 0);
  // Among split counts from the smallest that gives two waves to four times
  // that, take the one with the least estimated time: waves of resident CTAs
  // x (tiles per CTA + 2), the 2 standing for a CTA's fixed cost (ring fill,
  // state merge, partial write) in tile loads (fewest splits on ties).
  const int64_t base_ctas = (int64_t)num_seqs * Hkv * n_hb;
  const int64_t slots = (int64_t)ds->num_sms * (D == 64 ? 2 : 1);  // resident CTAs
  int s_lo = (int)((2 * slots + base_ctas - 1) / base_ctas);
  s_lo = s_lo < 1 ? 1 : (s_lo > n_tiles ? n_tiles : s_lo);
  const int s_hi = 4 * s_lo < n_tiles ? 4 * s_lo : n_tiles;
  int splits = s_lo, tps = (n_tiles + s_lo - 1) / s_lo;
  double best = 1e300;
  for (int c = s_lo; c <= s_hi; ++c) {
    const int t = (n_tiles + c - 1) / c;
    const int sc = (n_tiles + t - 1) / t;  // splits that tile count really needs
    const int64_t waves = (base_ctas * sc + slots - 1) / slots;
    const double cost = (double)waves * (t + 2);
    if (cost < best - 1e-9) {
      best = cost;
      splits = sc;
      tps = t;
    }
  }

  // Partial states, then one split counter per (sequence, KV head, head block).
  const size_t part_floats = (size_t)splits * num_seqs * Hq * (D + 2);
  const int n_counters = num_seqs * Hkv * n_hb;
  const size_t need = part_floats * sizeof(float) + (size_t)n_counters * sizeof(int);
  if (ws->part_bytes < need) {
    float* nb = nullptr;
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&nb), need, stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode workspace");
    if (ws->part) cudaFreeAsync(ws->part, stream);
    ws->part = nb;
    ws->part_bytes = need;
  }

  CUtensorMap tk, tv;
  if ((st = encode_thd(&tk, k, kv_rows, Hkv, D, kv_box)) != TSK_OK) return st;
  if ((st = encode_thd(&tv, v, kv_rows, Hkv, D, kv_box)) != TSK_OK) return st;

  tsk::dec::DecParams p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(q);
  p.sinks = sinks;
  p.cu_k = cu_seqlens_k;
  p.part = ws->part;
  p.counters = reinterpret_cast<int*>(ws->part + part_floats);
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = ws->base + tsk::kWsStatus;
  p.bad = ws->base + tsk::kWsDecodeBad;
  p.num_seqs = num_seqs;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.n_hb = n_hb;
  p.window = window;
  p.splits = splits;
  p.tiles_per_split = tps;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = g_timeout_ns;
  p.kv = pg;
  p.kv_rows = (int)kv_rows;

  char name[160];
  snprintf(name, sizeof name, "%s[Hq=%d,Hkv=%d,D=%d,W=%d,nseq=%d,Tk=%lld,splits=%d]", what, Hq,
           Hkv, D, window, num_seqs, (long long)total_k, splits);
  nvtxRangePushA(name);
  const bool prof = g_profile;
  if (prof) {
    if (g_ev_dev != dev) {
      for (auto& e : g_ev) {
        if (e) cudaEventDestroy(e);
        e = nullptr;
      }
      for (auto& e : g_ev)
        if (cudaEventCreate(&e) != cudaSuccess) {
          nvtxRangePop();
          return TSK_ERR_DEVICE;
        }
      g_ev_dev = dev;
    }
    cudaEventRecord(g_ev[0], stream);
  }
  tsk::dec::decode_check_kernel<<<1, 1024, 0, stream>>>(cu_seqlens_k, num_seqs, (int)total_k,
                                                       max_seqlen_k, ws->base + tsk::kWsStatus,
                                                       ws->base + tsk::kWsDecodeBad, pg,
                                                       p.counters, n_counters);
  if (prof) cudaEventRecord(g_ev[1], stream);
  const dim3 grid(splits, Hkv * n_hb, num_seqs);
  if (D == 64)
    tsk::dec::decode_split_kernel<64><<<grid, tsk::dec::kThreads, tsk::dec::smem_bytes<64>(), stream>>>(tk, tv, p);
  else
    tsk::dec::decode_split_kernel<128><<<grid, tsk::dec::kThreads, tsk::dec::smem_bytes<128>(), stream>>>(tk, tv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) note_error("decode kernel launch", e);
  if (prof) {
    cudaEventRecord(g_ev[2], stream);
    g_ev_recorded = true;
  }
  nvtxRangePop();
  return e == cudaSuccess ? TSK_OK : TSK_ERR_LAUNCH;
}
}  // namespace

extern "C" tsk_status tsk_mha_decode_kvcache(const void* q, const void* k, const void* v,
                                             const float* sinks, const int32_t* cu_seqlens_k,
                                             int32_t num_seqs, int64_t total_k,
                                             int32_t max_seqlen_k, int32_t Hq, int32_t Hkv,
                                             int32_t D, int32_t window, float scale, void* out,
                                             float* lse, tsk_stream_t stream) {
  return decode_impl(q, k, v, sinks, cu_seqlens_k, num_seqs, total_k, max_seqlen_k, Hq, Hkv, D,
                     window, scale, out, lse, reinterpret_cast<cudaStream_t>(stream),
                     "tsk_mha_decode_kvcache", nullptr, 0, 0, 0);
}

extern "C" tsk_status tsk_mha_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                                           const float* sinks, const int32_t* cu_seqlens_k,
                                           const int32_t* block_table, int32_t max_blocks_per_seq,
                                           int32_t page_size, int32_t num_pages, int32_t num_seqs,
                                           int64_t total_k, int32_t max_seqlen_k, int32_t Hq,
                                           int32_t Hkv, int32_t D, int32_t window, float scale,
                                           void* out, float* lse, tsk_stream_t stream) {
  if (page_size == 0) return TSK_ERR_UNSUPPORTED;
  return decode_impl(q, k_pages, v_pages, sinks, cu_seqlens_k, num_seqs, total_k, max_seqlen_k,
                     Hq, Hkv, D, window, scale, out, lse, reinterpret_cast<cudaStream_t>(stream),
                     "tsk_mha_decode_paged", block_table, max_blocks_per_seq, page_size, num_pages);
}

// ---------------------------------------------------------------------------
// FP8 (E4M3) prefill, head dimension 64.
namespace {
// FP8 prefill over keys that may extend before the queries (cu_k == cu_q and
// total_k == total_q for plain prefill).
tsk_status prefill_fp8_impl(const void* q8, const void* k8, const void* v8, float q_scale,
                            float k_scale, float v_scale, const float* sinks,
                            const int32_t* cu_seqlens, const int32_t* cu_k, int32_t num_seqs,
                            int64_t total_tokens, int64_t total_k, int32_t Hq, int32_t Hkv,
                            int32_t D, int32_t window, float scale, void* out, float* lse,
                            cudaStream_t stream, const char* what) {
  if (!q8 || !k8 || !v8 || !out || !cu_seqlens || !cu_k) return TSK_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_tokens < 0 || total_k < 0 || Hq <= 0 || Hkv <= 0)
    return TSK_ERR_INVALID_ARG;
  for (float x : {scale, q_scale, k_scale, v_scale})
    if (!std::isfinite(x) || !(x > 0.f)) return TSK_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || Hq % Hkv != 0) return TSK_ERR_UNSUPPORTED;
  if (num_seqs >= (1 << 24) || total_tokens * (int64_t)Hq >= ((int64_t)1 << 31) ||
      total_k * (int64_t)Hkv * D >= ((int64_t)1 << 31) || total_k >= ((int64_t)1 << 31))
    return TSK_ERR_UNSUPPORTED;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; };
  if (!a16(q8) || !a16(k8) || !a16(v8) || !a16(out)) return TSK_ERR_ALIGNMENT;
  if (!a4(cu_seqlens) || !a4(cu_k) || (sinks && !a4(sinks)) || (lse && !a4(lse)))
    return TSK_ERR_ALIGNMENT;
  const size_t out_bytes = (size_t)total_tokens * Hq * D * 2;
  const size_t q_bytes = (size_t)total_tokens * Hq * D, kv_bytes = (size_t)total_k * Hkv * D;
  if (total_tokens > 0 && (overlaps(out, out_bytes, q8, q_bytes) ||
                           overlaps(out, out_bytes, k8, kv_bytes) ||
                           overlaps(out, out_bytes, v8, kv_bytes)))
    return TSK_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_tokens == 0) return TSK_OK;
  if (total_k < total_tokens) return TSK_ERR_INVALID_ARG;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = -1;
  DeviceState* ds = nullptr;
  tsk_status st = check_device(&dev, &ds);
  if (st != TSK_OK) return st;
  if ((st = get_encoder()) != TSK_OK) return st;
  const int64_t max_tiles64 = total_tokens / tsk::kTileM + num_seqs + 1;
  const int max_tiles = (int)max_tiles64;
  Workspace* ws = nullptr;
  if ((st = get_workspace(dev, stream, max_tiles, num_seqs, &ws)) != TSK_OK) return st;
  // V as bf16 values, [total_k, Hkv, D] (the PV operand).
  const size_t vb_need = (size_t)total_k * Hkv * D * 2;
  if (ws->fp8_v_bytes < vb_need) {
    uint8_t* nb = nullptr;
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&nb), vb_need, stream);
    if (e != cudaSuccess) return cuda_fail(e, "FP8 bf16 V buffer");
    if (ws->fp8_v) cudaFreeAsync(ws->fp8_v, stream);
    ws->fp8_v = nb;
    ws->fp8_v_bytes = vb_need;
  }

  CUtensorMap tq, tk, tv, to;
  {
    const cuuint64_t dq[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)total_tokens};
    const cuuint64_t sq[2] = {(cuuint64_t)D, (cuuint64_t)Hq * D};
    const cuuint64_t dk[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)total_k};
    const cuuint64_t sk[2] = {(cuuint64_t)D, (cuuint64_t)Hkv * D};
    // Q/K boxes: one whole row of D bytes x 1 head x 128 rows (the second box
    // dimension is the head); 64-byte rows use the 64-byte swizzle, 128-byte
    // rows the 128-byte one.
    cuuint32_t box[3] = {(cuuint32_t)D, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapSwizzle swz = D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    CUresult r = g_encode(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(q8),
                          const_cast<cuuint64_t*>(dq), const_cast<cuuint64_t*>(sq), box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS)
      r = g_encode(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(k8),
                   const_cast<cuuint64_t*>(dk), const_cast<cuuint64_t*>(sk), box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return TSK_ERR_DEVICE;
    if ((st = encode_thd(&tv, ws->fp8_v, total_k, Hkv, D)) != TSK_OK) return st;
    if ((st = encode_thd(&to, out, total_tokens, Hq, D, 32)) != TSK_OK) return st;
  }

  char name[112];
  snprintf(name, sizeof name, "%s[Hq=%d,Hkv=%d,W=%d,nseq=%d,T=%lld,Tk=%lld]", what, Hq, Hkv,
           window, num_seqs, (long long)total_tokens, (long long)total_k);
  nvtxRangePushA(name);
  const size_t off_ints = ((size_t)tsk::kWsHeader + (size_t)ws->max_seqs + 1 + 3) & ~(size_t)3;
  int* tile_off = ws->base + tsk::kWsHeader;
  int4* list = reinterpret_cast<int4*>(ws->base + off_ints);
  const bool prof = g_profile;
  if (prof) {
    if (g_ev_dev != dev) {
      for (auto& e : g_ev) {
        if (e) cudaEventDestroy(e);
        e = nullptr;
      }
      for (auto& e : g_ev)
        if (cudaEventCreate(&e) != cudaSuccess) {
          nvtxRangePop();
          return TSK_ERR_DEVICE;
        }
      g_ev_dev = dev;
    }
    cudaEventRecord(g_ev[0], stream);
  }
  tsk::schedule_kernel<<<1, tsk::kSchedThreads, 0, stream>>>(
      cu_seqlens, cu_k, num_seqs, (int)total_tokens, (int)total_k, window, ws->base,
      tile_off, list, ws->max_tiles, tsk::PagedKV{nullptr, 0, 0, 0}, tsk::kTileM,
      tsk::KeyNorms{nullptr, 0, 0, 0, nullptr});
  // bf16 V and, for D = 64, the E4M3 key-row norms (at most kNormBlocks
  // blocks, about four 16-byte chunks of each tensor per thread)
  float* knorm = reinterpret_cast<float*>(ws->base + off_ints + (size_t)ws->max_tiles * tsk::kTileEntryInts);
  const bool norms = D == 64 && Hkv <= tsk::kNormMaxHeads;
  const int chunks = D / 16;
  int prep_blocks = (int)((total_k * Hkv * chunks + 4 * tsk::kSchedThreads - 1) / (4 * tsk::kSchedThreads));
  prep_blocks = prep_blocks < 1 ? 1 : (prep_blocks > tsk::kNormBlocks ? tsk::kNormBlocks : prep_blocks);
  tsk::fp8::fp8_prep_kernel<<<prep_blocks, tsk::kSchedThreads, 0, stream>>>(
      reinterpret_cast<const uint8_t*>(k8), reinterpret_cast<const uint8_t*>(v8),
      (long long)total_k, Hkv, chunks, norms, reinterpret_cast<uint4*>(ws->fp8_v), knorm,
      ws->base);
  if (prof) cudaEventRecord(g_ev[1], stream);

  tsk::fp8::Fp8Params f;
  tsk::AttnParams& p = f.a;
  p.sinks = sinks;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.list = list;
  p.ws = ws->base;
  p.status = ws->base + tsk::kWsStatus;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.HP = (p.G + 1) / 2;
  p.window = window;
  p.scale_log2 = scale * q_scale * k_scale * 1.4426950408889634f;
  p.timeout_ns = g_timeout_ns;
  p.debug_stall = g_debug_stall;
  p.kv = tsk::PagedKV{nullptr, 0, 0, 0};
  p.q_rows = (int)total_tokens;
  p.kv_rows = (int)total_k;
  p.max_tiles = ws->max_tiles;
  p.knorm = norms ? knorm + tsk::kNormBlocks * tsk::kNormMaxHeads : nullptr;
  p.out_scale = v_scale;
  f.v_scale = v_scale;
  const int64_t units_bound = max_tiles64 * Hkv * p.HP;
  const int grid = (int)(units_bound < ds->num_sms ? units_bound : ds->num_sms);
  if (D == 64)
    tsk::fp8::attention_fwd_fp8_kernel<<<grid, tsk::kThreads, tsk::fp8::kSmemBytes, stream>>>(
        tq, tk, tv, to, f);
  else
    tsk::d128::attention_fwd_d128_kernel<0, true>
        <<<grid, tsk::kThreads, tsk::d128::kSmemBytes, stream>>>(tq, tk, tv, to, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) note_error("FP8 attention kernel launch", e);
  if (prof) {
    cudaEventRecord(g_ev[2], stream);
    g_ev_recorded = true;
  }
  nvtxRangePop();
  return e == cudaSuccess ? TSK_OK : TSK_ERR_LAUNCH;
}

// ---------------------------------------------------------------------------
}  // namespace

extern "C" tsk_status tsk_mha_prefill_fp8(const void* q8, const void* k8, const void* v8,
                                          float q_scale, float k_scale, float v_scale,
                                          const float* sinks, const int32_t* cu_seqlens,
                                          int32_t num_seqs, int64_t total_tokens, int32_t Hq,
                                          int32_t Hkv, int32_t D, int32_t window, float scale,
                                          void* out, float* lse, tsk_stream_t stream) {
  return prefill_fp8_impl(q8, k8, v8, q_scale, k_scale, v_scale, sinks, cu_seqlens, cu_seqlens,
                          num_seqs, total_tokens, total_tokens, Hq, Hkv, D, window, scale, out,
                          lse, reinterpret_cast<cudaStream_t>(stream), "tsk_mha_prefill_fp8");
}

extern "C" tsk_status tsk_mha_prefill_fp8_kvcache(
    const void* q8, const void* k8, const void* v8, float q_scale, float k_scale, float v_scale,
    const float* sinks, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
    int32_t num_seqs, int64_t total_q, int64_t total_k, int32_t Hq, int32_t Hkv, int32_t D,
    int32_t window, float scale, void* out, float* lse, tsk_stream_t stream) {
  return prefill_fp8_impl(q8, k8, v8, q_scale, k_scale, v_scale, sinks, cu_seqlens_q,
                          cu_seqlens_k, num_seqs, total_q, total_k, Hq, Hkv, D, window, scale,
                          out, lse, reinterpret_cast<cudaStream_t>(stream),
                          "tsk_mha_prefill_fp8_kvcache");
}

// ---------------------------------------------------------------------------
// Host buffers in, host buffers out: tsk_mha_prefill_host.
//
// The packed token stream is cut into chunks of consecutive tokens.  Chunk c
// covers tokens [t_c, t_{c+1}); for every sequence it touches, its queries
// are the sequence's rows inside the chunk and its keys are the sequence's
// rows from its start up to the chunk's end, which earlier chunks (and this
// one) have already copied to the device.  So each chunk is one prefill over
// a key/value cache (the same kernels as tsk_mha_prefill_kvcache), and the
// three stages overlap across chunks: the copy of chunk c+1's inputs, the
// attention of chunk c (two compute streams, so one chunk's tail overlaps the
// next chunk's start) and the copy of chunk c-1's outputs.
namespace {

__global__ void merge_status_kernel(int* dst, int* a, int* b) {
  int* const srcs[2] = {a, b};
  for (int j = 0; j < 2; ++j) {
    int* src = srcs[j];
    if (src == nullptr || src[tsk::kWsStatus] == 0) continue;
    if (dst[tsk::kWsStatus] == 0)
      for (int i = 0; i < 3; ++i) dst[tsk::kWsStatus + i] = src[tsk::kWsStatus + i];
    for (int i = 0; i < 3; ++i) src[tsk::kWsStatus + i] = 0;
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Chunk boundaries and, per chunk, the kvcache-call description.
struct HostChunk {
  int64_t t0, t1;      // token rows [t0, t1)
  int64_t k0;          // first key row: start of the chunk's first sequence
  int32_t nseq;        // sequences with at least one query row in the chunk
  size_t cu_off;       // index of the chunk's cu_q (nseq + 1) then cu_k (nseq + 1)
};

}  // namespace

extern "C" tsk_status tsk_mha_prefill_host(const void* q, const void* k, const void* v,
                                           const float* sinks, const int32_t* cu_seqlens,
                                           int32_t num_seqs, int64_t total_tokens, int32_t Hq,
                                           int32_t Hkv, int32_t D, int32_t window, float scale,
                                           void* out, float* lse, tsk_stream_t stream_) {
  // ---- host-only checks (the offsets are host memory here, so all of them)
  if (!q || !k || !v || !out || !cu_seqlens) return TSK_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_tokens < 0 || Hq <= 0 || Hkv <= 0) return TSK_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return TSK_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || Hq % Hkv != 0) return TSK_ERR_UNSUPPORTED;
  if (num_seqs >= (1 << 24) || total_tokens * (int64_t)Hq >= ((int64_t)1 << 31))
    return TSK_ERR_UNSUPPORTED;
  if (cu_seqlens[0] != 0 || (int64_t)cu_seqlens[num_seqs] != total_tokens)
    return TSK_ERR_INVALID_ARG;
  for (int32_t s = 0; s < num_seqs; ++s)
    if (cu_seqlens[s + 1] < cu_seqlens[s]) return TSK_ERR_INVALID_ARG;
  {
    const size_t qo = (size_t)total_tokens * Hq * D * 2, kvb = (size_t)total_tokens * Hkv * D * 2;
    if (total_tokens > 0 && (overlaps(out, qo, q, qo) || overlaps(out, qo, k, kvb) ||
                             overlaps(out, qo, v, kvb)))
      return TSK_ERR_INVALID_ARG;
  }
  if (num_seqs == 0 || total_tokens == 0) return TSK_OK;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  // ---- chunks: about sixteen, of at least min(T / 8, 4096) tokens (a chunk
  // of few query tiles loses more to its own launch and tail than the finer
  // overlap gains: one 32K sequence in sixteen chunks was 6.5% slower than in
  // eight, 32 ragged sequences 6.5% faster) and at least 2048.  A chunk ends at a
  // sequence end or 128 rows after a query-tile start of the sequence it
  // cuts, so that every query tile (and every warp's 32 rows) is the one
  // tsk_mha_prefill forms: the results are then bit for bit the same.
  const int64_t T = total_tokens;
  int64_t chunk = (T + 15) / 16;
  const int64_t floor8 = (T + 7) / 8 < 4096 ? (T + 7) / 8 : 4096;
  if (chunk < floor8) chunk = floor8;
  if (chunk < 2048) chunk = 2048;
  std::vector<HostChunk> chunks;
  std::vector<int32_t> cu_host;
  {
    int32_t s = 0, s1 = 0;
    for (int64_t t0 = 0, t1 = 0; t0 < T; t0 = t1) {
      t1 = t0 + chunk < T ? t0 + chunk : T;
      if (t1 < T) {
        while (cu_seqlens[s1 + 1] <= t1) ++s1;  // the sequence holding row t1
        const int64_t off = t1 - cu_seqlens[s1];
        if (off % tsk::kTileM != 0) {
          const int64_t up = cu_seqlens[s1] + (off / tsk::kTileM + 1) * tsk::kTileM;
          t1 = up < cu_seqlens[s1 + 1] ? up : cu_seqlens[s1 + 1];
        }
      }
      while (cu_seqlens[s + 1] <= t0) ++s;  // the sequence holding row t0
      HostChunk c{t0, t1, cu_seqlens[s], 0, cu_host.size()};
      std::vector<int32_t> cq{0}, ck{0};
      for (int32_t r = s; r < num_seqs && cu_seqlens[r] < t1; ++r) {
        const int64_t a = cu_seqlens[r] > t0 ? cu_seqlens[r] : t0;
        const int64_t b = cu_seqlens[r + 1] < t1 ? cu_seqlens[r + 1] : t1;
        if (b <= a) continue;  // empty sequence
        cq.push_back((int32_t)(b - t0));
        ck.push_back((int32_t)(b - c.k0));
      }
      c.nseq = (int32_t)cq.size() - 1;
      cu_host.insert(cu_host.end(), cq.begin(), cq.end());
      cu_host.insert(cu_host.end(), ck.begin(), ck.end());
      chunks.push_back(c);
    }
  }

  std::lock_guard<std::mutex> plock(g_pipe_mu);
  int dev = -1;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* ds = nullptr;
    tsk_status st = check_device(&dev, &ds);
    if (st != TSK_OK) return st;
  }
  HostPipe& hp = g_pipe[{dev, stream}];
  if (!hp.h2d) {
    for (cudaStream_t* st : {&hp.h2d, &hp.d2h, &hp.comp[0], &hp.comp[1]})
      if (cudaStreamCreateWithFlags(st, cudaStreamNonBlocking) != cudaSuccess)
        return cuda_fail(cudaErrorUnknown, "host pipeline streams");
  }

  // ---- device buffer: q, k, v, out, lse, sinks, chunk offsets
  const size_t q_bytes = (size_t)T * Hq * D * 2, kv_bytes = (size_t)T * Hkv * D * 2;
  const size_t lse_bytes = lse ? (size_t)T * Hq * 4 : 0, sink_bytes = sinks ? (size_t)Hq * 4 : 0;
  const size_t off_q = 0, off_k = align256(q_bytes), off_v = off_k + align256(kv_bytes),
               off_o = off_v + align256(kv_bytes), off_l = off_o + align256(q_bytes),
               off_s = off_l + align256(lse_bytes), off_c = off_s + align256(sink_bytes),
               off_n = off_c + align256(cu_host.size() * 4),
               need = off_n + align256((tsk::kNormFloats + 8) * 4);
  if (hp.cap < need) {
    if (hp.buf) {
      cudaStreamSynchronize(stream);  // earlier calls on this stream may still use it
      cudaFree(hp.buf);
      hp.buf = nullptr;
      hp.cap = 0;
    }
    if (cudaMalloc(reinterpret_cast<void**>(&hp.buf), need) != cudaSuccess)
      return cuda_fail(cudaErrorMemoryAllocation, "host pipeline buffer");
    hp.cap = need;
  }
  uint8_t* b = hp.buf;
  const size_t qrow = (size_t)Hq * D * 2, kvrow = (size_t)Hkv * D * 2;

  std::vector<cudaEvent_t> evs;
  auto event = [&]() {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return e;
    evs.push_back(e);
    return e;
  };
  tsk_status st = TSK_OK;
  cudaEvent_t ev_start = event(), ev_done = event();
  if (!ev_start || !ev_done) st = cuda_fail(cudaErrorUnknown, "host pipeline events");
  if (st == TSK_OK) {
    // Everything starts after the work already queued on the caller's stream
    // (earlier calls may still be reading the buffer).
    cudaEventRecord(ev_start, stream);
    for (cudaStream_t s2 : {hp.h2d, hp.d2h, hp.comp[0], hp.comp[1]})
      cudaStreamWaitEvent(s2, ev_start, 0);
    if (sinks) cudaMemcpyAsync(b + off_s, sinks, sink_bytes, cudaMemcpyHostToDevice, hp.h2d);
    cudaMemcpyAsync(b + off_c, cu_host.data(), cu_host.size() * 4, cudaMemcpyHostToDevice, hp.h2d);
    const float* d_sinks = sinks ? reinterpret_cast<const float*>(b + off_s) : nullptr;
    const int32_t* d_cu = reinterpret_cast<const int32_t*>(b + off_c);
    // The key-norm bound over all keys, as tsk_mha_prefill computes it, so
    // that every chunk makes the same choices and the results stay bit for
    // bit those of tsk_mha_prefill: K is copied whole first.
    tsk::KeyNorms kn;
    int* n_ws = reinterpret_cast<int*>(b + off_n);  // [kWsNormCount] counter, then the norms
    float* n_out = reinterpret_cast<float*>(b + off_n) + 8;
    const int nb = key_norm_setup(&kn, b + off_k, T, Hkv, D, window, n_out);
    const float* d_knorm = nb ? n_out + tsk::kNormBlocks * tsk::kNormMaxHeads : nullptr;
    if (nb) {
      cudaMemcpyAsync(b + off_k, k, T * kvrow, cudaMemcpyHostToDevice, hp.h2d);
      cudaMemsetAsync(n_ws, 0, 8 * sizeof(int), hp.h2d);
      tsk::key_norm_kernel<<<nb, tsk::kSchedThreads, 0, hp.h2d>>>(kn, n_ws);
    }
    for (size_t c = 0; c < chunks.size() && st == TSK_OK; ++c) {
      const HostChunk& ch = chunks[c];
      const int64_t n = ch.t1 - ch.t0;
      cudaEvent_t ev_in = event(), ev_out = event();
      if (!ev_in || !ev_out) {
        st = cuda_fail(cudaErrorUnknown, "host pipeline events");
        break;
      }
      const uint8_t* hq = static_cast<const uint8_t*>(q) + ch.t0 * qrow;
      const uint8_t* hk = static_cast<const uint8_t*>(k) + ch.t0 * kvrow;
      const uint8_t* hv = static_cast<const uint8_t*>(v) + ch.t0 * kvrow;
      cudaMemcpyAsync(b + off_q + ch.t0 * qrow, hq, n * qrow, cudaMemcpyHostToDevice, hp.h2d);
      if (!nb) cudaMemcpyAsync(b + off_k + ch.t0 * kvrow, hk, n * kvrow, cudaMemcpyHostToDevice, hp.h2d);
      cudaMemcpyAsync(b + off_v + ch.t0 * kvrow, hv, n * kvrow, cudaMemcpyHostToDevice, hp.h2d);
      cudaEventRecord(ev_in, hp.h2d);
      cudaStream_t cs = hp.comp[c & 1];
      cudaStreamWaitEvent(cs, ev_in, 0);
      if (ch.nseq > 0) {
        st = prefill_impl(b + off_q + ch.t0 * qrow, b + off_k + ch.k0 * kvrow,
                          b + off_v + ch.k0 * kvrow, d_sinks, d_cu + ch.cu_off,
                          d_cu + ch.cu_off + ch.nseq + 1, ch.nseq, n, ch.t1 - ch.k0, Hq, Hkv, D,
                          window, scale, b + off_o + ch.t0 * qrow,
                          lse ? reinterpret_cast<float*>(b + off_l) + ch.t0 * Hq : nullptr, cs,
                          "tsk_mha_prefill_host", nullptr, 0, 0, 0, d_knorm);
      }
      cudaEventRecord(ev_out, cs);
      cudaStreamWaitEvent(hp.d2h, ev_out, 0);
      cudaMemcpyAsync(static_cast<uint8_t*>(out) + ch.t0 * qrow, b + off_o + ch.t0 * qrow,
                      n * qrow, cudaMemcpyDeviceToHost, hp.d2h);
      if (lse)
        cudaMemcpyAsync(lse + ch.t0 * Hq, b + off_l + ch.t0 * Hq * 4, n * Hq * 4,
                        cudaMemcpyDeviceToHost, hp.d2h);
    }
    // The caller's stream continues once every copy back has finished (the
    // copy stream waited for both compute streams' chunks).
    cudaEventRecord(ev_done, hp.d2h);
    cudaStreamWaitEvent(stream, ev_done, 0);
    for (cudaStream_t s2 : {hp.h2d, hp.comp[0], hp.comp[1]}) {
      cudaEvent_t e = event();
      if (e) {
        cudaEventRecord(e, s2);
        cudaStreamWaitEvent(stream, e, 0);
      }
    }
    // Device-side errors of the chunks' kernels (bounded waits) move to the
    // caller stream's status words, where tsk_get_device_status reads them.
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace* ws = nullptr;
    if (get_workspace(dev, stream, 1024, 1024, &ws) == TSK_OK) {
      auto w0 = g_ws.find({dev, hp.comp[0]}), w1 = g_ws.find({dev, hp.comp[1]});
      int* a0 = w0 != g_ws.end() ? w0->second.base : nullptr;
      int* a1 = w1 != g_ws.end() ? w1->second.base : nullptr;
      merge_status_kernel<<<1, 1, 0, stream>>>(ws->base, a0, a1);
    }
  }
  for (cudaEvent_t e : evs) cudaEventDestroy(e);  // released once they complete
  cudaError_t e = cudaGetLastError();
  if (st == TSK_OK && e != cudaSuccess) {
    note_error("tsk_mha_prefill_host", e);
    st = TSK_ERR_LAUNCH;
  }
  return st;
}
