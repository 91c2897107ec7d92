// ra_merge.cu -- merge of normalised partial attention results.
//
// The online-softmax fold of the mKernel overview page's Ring Attention row
// (table "Die fünf verschmolzenen Kerne"), written for partials that were each
// normalised by their own sum: lse = ln sum_k e^{lse_k},
// out = sum_k e^{lse_k - lse} O_k.  Pure streaming work (no reuse), so the
// kernel is organised for HBM bandwidth: each thread owns 8 consecutive
// elements of a row (one 16-byte bf16 vector), a grid-stride loop over a grid
// sized to the SM count, 16-byte loads and stores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ra_internal.h"

namespace ra {

// 8 consecutive elements of partial p (16-byte bf16 or 2 x 16-byte fp32
// loads, streamed: every byte is read exactly once) widened to fp32.
template <bool kFp32>
__device__ __forceinline__ void load8(const void* base, long long e0, float (&x)[8]) {
  if (kFp32) {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(base) + e0);
    const float4 a = __ldcs(src), b = __ldcs(src + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 a = __ldcs(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + e0));
    const uint32_t v[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(v[j] << 16);
      x[2 * j + 1] = __uint_as_float(v[j] & 0xFFFF0000u);
    }
  }
}

template <bool kFp32>
__global__ void __launch_bounds__(256) merge_kernel(const void* __restrict__ o_parts,
                                                    const float* __restrict__ lse_parts, int n,
                                                    __nv_bfloat16* __restrict__ out,
                                                    float* __restrict__ lse, long long rows, int H,
                                                    int S, int D) {
  constexpr int kBatch = 4;  // partials whose loads are in flight together
  const int per_row = D / 8;
  const int pr_shift = (per_row & (per_row - 1)) == 0 ? __ffs(per_row) - 1 : -1;
  const long long units = rows * per_row;
  const long long o_stride = rows * (long long)D;  // elements per partial
  const long long l_stride = rows;                 // B*H*S == rows
  for (long long w = blockIdx.x * (long long)blockDim.x + threadIdx.x; w < units;
       w += (long long)gridDim.x * blockDim.x) {
    // rows < 2^31 (checked on the host): 32-bit index arithmetic
    const unsigned row32 = (unsigned)(pr_shift >= 0 ? (w >> pr_shift) : w / per_row);  // [B,S,H]
    const long long row = row32;
    const int cpart = (int)(w - row * per_row);
    const unsigned h = row32 % (unsigned)H;
    const unsigned bs = row32 / (unsigned)H;
    const unsigned s = bs % (unsigned)S;
    const unsigned b = bs / (unsigned)S;
    const long long li = ((long long)b * H + h) * S + s;  // [B,H,S] order
    const long long e_row = row * D + cpart * 8;

    float M = -INFINITY;
    for (int p = 0; p < n; ++p) M = fmaxf(M, __ldg(lse_parts + p * l_stride + li));
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float L = -INFINITY;
    if (M != -INFINITY) {
      float Z = 0.0f;
      for (int p = 0; p < n; ++p) Z += expf(__ldg(lse_parts + p * l_stride + li) - M);
      L = M + logf(Z);
      for (int p0 = 0; p0 < n; p0 += kBatch) {
        float x[kBatch][8];
        float wgt[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const int p = p0 + q;
          const float lp = p < n ? __ldg(lse_parts + p * l_stride + li) : -INFINITY;
          wgt[q] = lp == -INFINITY ? 0.0f : expf(lp - L);  // an empty partial adds nothing
          if (lp != -INFINITY) load8<kFp32>(o_parts, p * o_stride + e_row, x[q]);
          else
#pragma unroll
            for (int j = 0; j < 8; ++j) x[q][j] = 0.0f;
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] += wgt[q] * x[q][j];
      }
    }
    uint32_t packed[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 t = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
      packed[j] = *reinterpret_cast<uint32_t*>(&t);
    }
    *reinterpret_cast<uint4*>(out + e_row) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if (lse && cpart == 0) lse[li] = L;
  }
}

cudaError_t launch_merge(const void* o_parts, int o_is_fp32, const float* lse_parts, int n,
                         void* out, float* lse, long long rows, int H, int S, int D, int grid,
                         cudaStream_t stream) {
  auto* o = static_cast<__nv_bfloat16*>(out);
  if (o_is_fp32)
    merge_kernel<true><<<grid, 256, 0, stream>>>(o_parts, lse_parts, n, o, lse, rows, H, S, D);
  else
    merge_kernel<false><<<grid, 256, 0, stream>>>(o_parts, lse_parts, n, o, lse, rows, H, S, D);
  return cudaGetLastError();
}

}  // namespace ra
