// ra_merge.cu -- merge of normalised partial attention results.
//
// The online-softmax fold of the mKernel overview page's Ring Attention row
// (table "Die fünf verschmolzenen Kerne"), written for partials that were each
// normalised by their own sum: lse = ln sum_k e^{lse_k},
// out = sum_k e^{lse_k - lse} O_k.
//
// Pure streaming work (every byte is read once), so the kernel is organised
// for HBM bandwidth.  A CTA takes a tile of Ts consecutive sequence positions
// of one batch entry, every head: in [B, S, H] row order that is Ts*H
// consecutive rows, so the tile's D-vectors form one contiguous range in each
// partial.
//   1. The tile's n*H*Ts log-sum-exps are loaded into shared memory; for a
//      fixed (partial, head) the Ts positions are contiguous in [n, B, H, S],
//      so consecutive threads read consecutive words.
//   2. One thread per row turns them into weights e^{lse_k - lse} (in place)
//      and writes the row's lse.
//   3. The partials' D-vectors of the tile are streamed with 16-byte loads
//      (several partials' loads in flight per thread), weighted from shared
//      memory, summed in fp32 and stored as bf16 with 16-byte stores.
// Tiles are taken in a grid-stride loop over a grid of a few CTAs per SM.
// Shapes whose n*H lse values do not fit the shared-memory budget even at
// Ts = 1 use merge_rows_kernel, one thread per 8 elements of a row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ra_internal.h"

namespace ra {

namespace {

constexpr int kMergeThreads = 512;
constexpr int kMergeSmemFloats = 8192;  // 32 KiB of lse / weights per tile
constexpr int kMaxTileRows = 32;        // sequence positions per tile at most
// partials whose loads are in flight together (per thread): 8 x 16 bytes of
// bf16, or 4 x 32 bytes of fp32, within the 64 registers of two CTAs per SM
template <bool kFp32>
constexpr int load_batch() { return kFp32 ? 4 : 8; }

// 8 consecutive elements of one partial as loaded (16-byte streamed loads:
// every byte is read exactly once): bf16 in one 16-byte word, fp32 in two.
template <bool kFp32>
struct Raw8 {
  uint4 a, b;
};
template <>
struct Raw8<false> {
  uint4 a;
};

template <bool kFp32>
__device__ __forceinline__ void load8(const void* base, long long e0, Raw8<kFp32>& r) {
  if constexpr (kFp32) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const float*>(base) + e0);
    r.a = __ldcs(src);
    r.b = __ldcs(src + 1);
  } else {
    r.a = __ldcs(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + e0));
  }
}

// acc += w * (the 8 elements, widened exactly to fp32)
template <bool kFp32>
__device__ __forceinline__ void fma8(float (&acc)[8], float w, const Raw8<kFp32>& r) {
  if constexpr (kFp32) {
    const uint32_t v[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t] = fmaf(w, __uint_as_float(v[t]), acc[t]);
  } else {
    const uint32_t v[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[2 * j] = fmaf(w, __uint_as_float(v[j] << 16), acc[2 * j]);
      acc[2 * j + 1] = fmaf(w, __uint_as_float(v[j] & 0xFFFF0000u), acc[2 * j + 1]);
    }
  }
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
  uint32_t p[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __nv_bfloat162 t = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    p[j] = *reinterpret_cast<uint32_t*>(&t);
  }
  return make_uint4(p[0], p[1], p[2], p[3]);
}

// The weights of one row from its n log-sum-exps (lse_k = -inf: an empty
// partial, weight 0); returns the merged lse (-inf when every partial is empty).
__device__ __forceinline__ float row_weights(float* w, int n, int stride) {
  float M = -INFINITY;
  for (int p = 0; p < n; ++p) M = fmaxf(M, w[p * stride]);
  if (M == -INFINITY) {
    for (int p = 0; p < n; ++p) w[p * stride] = 0.0f;
    return -INFINITY;
  }
  float Z = 0.0f;
  for (int p = 0; p < n; ++p) Z += expf(w[p * stride] - M);
  const float L = M + logf(Z);
  for (int p = 0; p < n; ++p) {
    const float lp = w[p * stride];
    w[p * stride] = lp == -INFINITY ? 0.0f : expf(lp - L);
  }
  return L;
}

template <bool kFp32>
__global__ void __launch_bounds__(kMergeThreads, 2) merge_tiles_kernel(
    const void* __restrict__ o_parts, const float* __restrict__ lse_parts, int n,
    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int B, int H, int S, int D, int Ts,
    unsigned int* status, long long trim) {
  extern __shared__ float w_s[];  // [n][H][Ts]: lse of the tile, then the weights
  const int tiles_per_b = (S + Ts - 1) / Ts;
  const long long n_tiles = (long long)B * tiles_per_b;
  const long long rows = (long long)B * S * H;
  const long long o_stride = rows * D;  // elements per partial
  const long long lse_n = (long long)B * H * S;  // lse values per partial
  const int vec_per_row = D / 8;
  for (long long tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int b = (int)(tile / tiles_per_b);
    const int s0 = (int)(tile % tiles_per_b) * Ts;
    const int ts = min(Ts, S - s0);  // positions in this tile (the last one may be short)
    const int n_w = n * H * ts;
    // 1. the tile's lse values: index i = (p*H + h)*ts + j  <->  lse[p, b, h, s0 + j]
    for (int i = threadIdx.x; i < n_w; i += blockDim.x) {
      const int j = i % ts;
      const int ph = i / ts;  // p*H + h
      const int p = ph / H, h = ph % H;
      const long long li = (((long long)p * B + b) * H + h) * S + s0 + j;
      w_s[i] = in_bounds(li, 1, n * lse_n, trim, status) ? __ldg(lse_parts + li) : -INFINITY;
    }
    __syncthreads();
    // 2. weights per row (h, j), in place; the row's merged lse
    for (int r = threadIdx.x; r < H * ts; r += blockDim.x) {
      const float L = row_weights(w_s + r, n, H * ts);
      if (lse) {
        const int h = r / ts, j = r % ts;
        const long long li = ((long long)b * H + h) * S + s0 + j;
        if (in_bounds(li, 1, lse_n, trim, status)) lse[li] = L;
      }
    }
    __syncthreads();
    // 3. stream the D-vectors: vector v of the tile belongs to row
    //    (j, h) = (v / vec_per_row) in [position, head] order
    const long long e_base = ((long long)b * S + s0) * H * D;
    const int n_vec = ts * H * vec_per_row;
    for (int v = threadIdx.x; v < n_vec; v += blockDim.x) {
      const int row = v / vec_per_row;  // j*H + h
      const int j = row / H, h = row % H;
      const int wi = h * ts + j;        // this row's weight index inside a partial's [H][ts]
      const long long e = e_base + (long long)v * 8;
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      constexpr int kLoadBatch = load_batch<kFp32>();
      for (int p0 = 0; p0 < n; p0 += kLoadBatch) {
        Raw8<kFp32> x[kLoadBatch];
        float wg[kLoadBatch];
#pragma unroll
        for (int q = 0; q < kLoadBatch; ++q) {
          const int p = p0 + q;
          wg[q] = p < n ? w_s[p * H * ts + wi] : 0.0f;
          // an empty partial (weight 0) is not read
          if (wg[q] != 0.0f && in_bounds(p * o_stride + e, 8, n * o_stride, trim, status))
            load8<kFp32>(o_parts, p * o_stride + e, x[q]);
          else
            wg[q] = 0.0f;
        }
#pragma unroll
        for (int q = 0; q < kLoadBatch; ++q)
          if (wg[q] != 0.0f) fma8<kFp32>(acc, wg[q], x[q]);
      }
      if (in_bounds(e, 8, o_stride, trim, status)) *reinterpret_cast<uint4*>(out + e) = pack8(acc);
    }
    __syncthreads();  // the weights are rewritten by the next tile
  }
}

// One thread per 8 elements of a row, every lse read from global memory:
// for shapes whose n*H lse values of one position exceed the tile budget.
template <bool kFp32>
__global__ void __launch_bounds__(256) merge_rows_kernel(const void* __restrict__ o_parts,
                                                         const float* __restrict__ lse_parts, int n,
                                                         __nv_bfloat16* __restrict__ out,
                                                         float* __restrict__ lse, long long rows,
                                                         int H, int S, int D, unsigned int* status,
                                                         long long trim) {
  const int per_row = D / 8;
  const long long units = rows * per_row;
  const long long o_stride = rows * (long long)D;
  for (long long w = blockIdx.x * (long long)blockDim.x + threadIdx.x; w < units;
       w += (long long)gridDim.x * blockDim.x) {
    const long long row = w / per_row;  // [B,S,H] order
    const int cpart = (int)(w - row * per_row);
    const int h = (int)(row % H);
    const long long bs = row / H;
    const long long li = ((bs / S) * H + h) * S + bs % S;  // [B,H,S] order
    // a partial outside the buffers (bounds-checked builds only) counts as empty
    auto lse_of = [&](int p) {
      return in_bounds(p * rows + li, 1, n * rows, trim, status) ? __ldg(lse_parts + p * rows + li)
                                                                 : -INFINITY;
    };
    float M = -INFINITY;
    for (int p = 0; p < n; ++p) M = fmaxf(M, lse_of(p));
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float L = -INFINITY;
    if (M != -INFINITY) {
      float Z = 0.0f;
      for (int p = 0; p < n; ++p) Z += expf(lse_of(p) - M);
      L = M + logf(Z);
      for (int p = 0; p < n; ++p) {
        const float lp = lse_of(p);
        if (lp == -INFINITY) continue;
        if (!in_bounds(p * o_stride + row * D + cpart * 8, 8, n * o_stride, trim, status)) continue;
        Raw8<kFp32> x;
        load8<kFp32>(o_parts, p * o_stride + row * D + cpart * 8, x);
        fma8<kFp32>(acc, expf(lp - L), x);
      }
    }
    if (in_bounds(row * D + cpart * 8, 8, o_stride, trim, status))
      *reinterpret_cast<uint4*>(out + row * D + cpart * 8) = pack8(acc);
    if (lse && cpart == 0 && in_bounds(li, 1, rows, trim, status)) lse[li] = L;
  }
}

}  // namespace

cudaError_t launch_merge(const void* o_parts, int o_is_fp32, const float* lse_parts, int n,
                         void* out, float* lse, int B, int H, int S, int D, int sms,
                         unsigned int* status, long long trim, cudaStream_t stream) {
  auto* o = static_cast<__nv_bfloat16*>(out);
  const long long rows = (long long)B * S * H;
  const long long per_pos = (long long)n * H;  // lse values of one sequence position
  if (per_pos <= kMergeSmemFloats) {
    int Ts = (int)(kMergeSmemFloats / per_pos);
    if (Ts > kMaxTileRows) Ts = kMaxTileRows;
    if (Ts > S) Ts = S;
    const long long n_tiles = (long long)B * ((S + Ts - 1) / Ts);
    const long long cap = (long long)sms * 2;  // 2 resident CTAs of 512 threads per SM
    const int grid = (int)(n_tiles < cap ? n_tiles : cap);
    const size_t smem = (size_t)per_pos * Ts * sizeof(float);
    if (o_is_fp32)
      merge_tiles_kernel<true><<<grid, kMergeThreads, smem, stream>>>(o_parts, lse_parts, n, o, lse,
                                                                    B, H, S, D, Ts, status, trim);
    else
      merge_tiles_kernel<false><<<grid, kMergeThreads, smem, stream>>>(o_parts, lse_parts, n, o,
                                                                     lse, B, H, S, D, Ts, status,
                                                                     trim);
    return cudaGetLastError();
  }
  const long long units = rows * (D / 8);
  long long grid = (units + 255) / 256;
  if (grid > (long long)sms * 8) grid = (long long)sms * 8;
  if (o_is_fp32)
    merge_rows_kernel<true><<<(int)grid, 256, 0, stream>>>(o_parts, lse_parts, n, o, lse, rows, H,
                                                           S, D, status, trim);
  else
    merge_rows_kernel<false><<<(int)grid, 256, 0, stream>>>(o_parts, lse_parts, n, o, lse, rows, H,
                                                            S, D, status, trim);
  return cudaGetLastError();
}

}  // namespace ra
