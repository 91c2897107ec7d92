// ra_ceil.cu -- microbenchmarks of the two non-tensor pipes the forward's
// online softmax leans on: the hardware exp2 (MUFU ex2) and fp32 FMA, scalar
// and packed f32x2.  They measure the ceilings that sit beside the tensor-core
// roofline: per allowed (query, key) pair the softmax issues one exp2 and a
// few fp32 operations, so these rates bound the pairs per second no matter how
// fast the tensor cores are.
//
// Each kernel runs one CTA per SM, 1024 threads, with kChains independent
// dependency chains per thread so the pipe, not latency, is the limit.  The
// CTA's first thread records the SM clock cycles (clock64) and nanoseconds
// (%globaltimer) its loop took; the host turns them into operations per SM
// per clock and per second.
#include <cuda_runtime.h>

#include <cstdint>

#include "ra_ptx.cuh"

namespace ra {
namespace {

constexpr int kCeilThreads = 1024;
constexpr int kChains = 8;

struct CeilTimes {
  long long cycles;
  unsigned long long ns;
};

// x <- 2^-x keeps every chain in [0.5, 1] (no overflow, no denormals)
__global__ void __launch_bounds__(kCeilThreads) ceil_ex2_kernel(float* sink, CeilTimes* t,
                                                                int iters) {
  float x[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j) x[j] = 0.5f + 0.01f * (float)((threadIdx.x + j) & 31);
  __syncthreads();
  const long long c0 = clock64();
  const uint64_t n0 = global_timer_ns();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) x[j] = ex2(-x[j]);
  }
  __syncthreads();
  const long long c1 = clock64();
  const uint64_t n1 = global_timer_ns();
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) acc += x[j];
  if (acc == 12345.0f) sink[threadIdx.x] = acc;  // keeps the chains alive
  if (threadIdx.x == 0) t[blockIdx.x] = CeilTimes{c1 - c0, n1 - n0};
}

// scalar fp32 FMA: x <- x * a + b with |a| < 1 (converges, stays finite)
__global__ void __launch_bounds__(kCeilThreads) ceil_ffma_kernel(float* sink, CeilTimes* t,
                                                                 int iters, float a, float b) {
  float x[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j) x[j] = 1.0f + 0.01f * (float)((threadIdx.x + j) & 31);
  __syncthreads();
  const long long c0 = clock64();
  const uint64_t n0 = global_timer_ns();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) x[j] = __fmaf_rn(x[j], a, b);
  }
  __syncthreads();
  const long long c1 = clock64();
  const uint64_t n1 = global_timer_ns();
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) acc += x[j];
  if (acc == 12345.0f) sink[threadIdx.x] = acc;
  if (threadIdx.x == 0) t[blockIdx.x] = CeilTimes{c1 - c0, n1 - n0};
}

// packed fp32x2 FMA: two lanes per instruction
__global__ void __launch_bounds__(kCeilThreads) ceil_ffma2_kernel(float* sink, CeilTimes* t,
                                                                  int iters, float a, float b) {
  uint64_t x[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j) {
    const float v = 1.0f + 0.01f * (float)((threadIdx.x + j) & 31);
    x[j] = f2_pack(v, v + 0.5f);
  }
  const uint64_t a2 = f2_pack(a, a), b2 = f2_pack(b, b);
  __syncthreads();
  const long long c0 = clock64();
  const uint64_t n0 = global_timer_ns();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) x[j] = f2_fma(x[j], a2, b2);
  }
  __syncthreads();
  const long long c1 = clock64();
  const uint64_t n1 = global_timer_ns();
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) acc += f2_lo(x[j]) + f2_hi(x[j]);
  if (acc == 12345.0f) sink[threadIdx.x] = acc;
  if (threadIdx.x == 0) t[blockIdx.x] = CeilTimes{c1 - c0, n1 - n0};
}

}  // namespace

// the kernels' sink and per-CTA timing records (library-owned, 20 KiB)
__device__ float g_ceil_sink[kCeilThreads];
__device__ CeilTimes g_ceil_times[1024];

// Runs the three microbenchmarks on the current device (synchronously, on its
// own stream) and fills `out`:
//   [0] ex2 per SM per clock        [1] ex2 per second (whole GPU)
//   [2] scalar FMA lanes / SM / clk [3] scalar FMA lanes per second
//   [4] f32x2 FMA lanes / SM / clk  [5] f32x2 FMA lanes per second
//   [6] SM clock during the runs (MHz, cycles / ns averaged)   [7] SMs
cudaError_t measure_ceilings(int sms, double* out) {
  float* sink = nullptr;
  CeilTimes* t = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&sink), g_ceil_sink);
  if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&t), g_ceil_times);
  if (e != cudaSuccess) return e;
  cudaStream_t s;
  e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) return e;
  const int iters = 4096;
  const double per_cta = (double)kCeilThreads * iters * kChains;
  CeilTimes host[1024];
  const int n = sms < 1024 ? sms : 1024;
  double mhz_sum = 0.0;
  for (int k = 0; k < 3 && e == cudaSuccess; ++k) {
    for (int rep = 0; rep < 2 && e == cudaSuccess; ++rep) {  // the first run warms up
      if (k == 0) ceil_ex2_kernel<<<n, kCeilThreads, 0, s>>>(sink, t, iters);
      if (k == 1) ceil_ffma_kernel<<<n, kCeilThreads, 0, s>>>(sink, t, iters, 0.999f, 0.001f);
      if (k == 2) ceil_ffma2_kernel<<<n, kCeilThreads, 0, s>>>(sink, t, iters, 0.999f, 0.001f);
      e = cudaGetLastError();
      if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    if (e != cudaSuccess) break;
    e = cudaMemcpy(host, t, sizeof(CeilTimes) * n, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) break;
    double cyc = 0.0, ns = 0.0;
    for (int i = 0; i < n; ++i) {
      cyc += (double)host[i].cycles;
      ns += (double)host[i].ns;
    }
    cyc /= n;
    ns /= n;
    const double lanes = (k == 2) ? 2.0 : 1.0;
    out[2 * k] = per_cta * lanes / cyc;
    out[2 * k + 1] = per_cta * lanes * n / (ns * 1e-9);
    mhz_sum += cyc / ns * 1e3;
  }
  out[6] = mhz_sum / 3.0;
  out[7] = (double)n;
  cudaStreamDestroy(s);
  return e;
}

}  // namespace ra
