// Throughput probe of the exponential unit (ex2.approx.f32), used by the
// benchmark to state the roof of the softmax's exponentials next to the
// tensor-core and HBM roofs.  Not part of the attention path.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace tsk {

constexpr int kEx2ProbeThreads = 512;  // 16 warps per SM: four per sub-partition
constexpr int kEx2ProbeChains = 8;     // independent dependency chains per thread

__device__ float g_ex2_probe_sink;

// Each thread runs kEx2ProbeChains independent chains x <- 2^x - 1.5 (which
// stay inside [-1.5, 0]) for `iters` steps: one exponential and one add per
// step and chain, the add on another pipe.
__global__ void __launch_bounds__(kEx2ProbeThreads, 1) ex2_rate_kernel(int iters) {
  float x[kEx2ProbeChains];
#pragma unroll
  for (int i = 0; i < kEx2ProbeChains; ++i) x[i] = -0.01f * (float)((threadIdx.x + i) & 63);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kEx2ProbeChains; ++i) x[i] = ex2_approx(x[i]) - 1.5f;
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kEx2ProbeChains; ++i) s += x[i];
  if (s == 1234.5f) g_ex2_probe_sink = s;  // never true; keeps the chains live
}

}  // namespace tsk
