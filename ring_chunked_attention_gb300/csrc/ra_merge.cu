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

template <bool kFp32>
__global__ void __launch_bounds__(256) merge_kernel(const void* __restrict__ o_parts,
                                                    const float* __restrict__ lse_parts, int n,
                                                    __nv_bfloat16* __restrict__ out,
                                                    float* __restrict__ lse, long long rows, int H,
                                                    int S, int D) {
  const int per_row = D / 8;
  const long long units = rows * per_row;
  const long long o_stride = rows * (long long)D;  // elements per partial
  const long long l_stride = rows;                 // B*H*S == rows
  for (long long w = blockIdx.x * (long long)blockDim.x + threadIdx.x; w < units;
       w += (long long)gridDim.x * blockDim.x) {
    const long long row = w / per_row;  // [B,S,H] order
    const int cpart = (int)(w % per_row);
    const int h = (int)(row % H);
    const long long bs = row / H;
    const int s = (int)(bs % S);
    const long long b = bs / S;
    const long long li = (b * H + h) * S + s;  // [B,H,S] order

    float M = -INFINITY;
    for (int p = 0; p < n; ++p) M = fmaxf(M, __ldg(lse_parts + p * l_stride + li));
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float L = -INFINITY;
    if (M != -INFINITY) {
      float Z = 0.0f;
      for (int p = 0; p < n; ++p) Z += expf(__ldg(lse_parts + p * l_stride + li) - M);
      L = M + logf(Z);
      for (int p = 0; p < n; ++p) {
        const float lp = __ldg(lse_parts + p * l_stride + li);
        if (lp == -INFINITY) continue;
        const float wgt = expf(lp - L);
        const long long e0 = p * o_stride + row * D + cpart * 8;
        if (kFp32) {
          const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(o_parts) + e0);
          const float4 x0 = __ldg(src), x1 = __ldg(src + 1);
          acc[0] += wgt * x0.x; acc[1] += wgt * x0.y; acc[2] += wgt * x0.z; acc[3] += wgt * x0.w;
          acc[4] += wgt * x1.x; acc[5] += wgt * x1.y; acc[6] += wgt * x1.z; acc[7] += wgt * x1.w;
        } else {
          const uint4 x = __ldg(reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(o_parts) + e0));
          const uint32_t v[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[2 * j] += wgt * __uint_as_float(v[j] << 16);
            acc[2 * j + 1] += wgt * __uint_as_float(v[j] & 0xFFFF0000u);
          }
        }
      }
    }
    uint32_t packed[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 t = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
      packed[j] = *reinterpret_cast<uint32_t*>(&t);
    }
    *reinterpret_cast<uint4*>(out + row * D + cpart * 8) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
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
