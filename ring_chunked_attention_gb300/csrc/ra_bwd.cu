// ra_bwd.cu -- backward pass of the ring-chunked attention: dq, dk, dv for a
// given output gradient, on sm_103a tensor cores (tcgen05, tensor memory, TMA).
//
// The pages describe no backward pass.  What is computed is the gradient of
// the forward's definition (exact softmax attention), for one query row s of
// head h and a key t of its KV head g:
//   p_st    = exp(scale * q_s.k_t - lse_s)       (lse from the forward)
//   dp_st   = dout_s . v_t
//   delta_s = sum_d out_s[d] dout_s[d]            (= sum_t p_st dp_st)
//   ds_st   = p_st (dp_st - delta_s)
//   dq_s = scale sum_t ds_st k_t,  dk_t = scale sum_s ds_st q_s,  dv_t = sum_s p_st dout_s
// with dk, dv summed over the query heads of the GQA group.
//
// Three kernels, launched in order on one stream:
//   bwd_prep_kernel  -delta_s and -lse_s*log2(e) per query row (row sums,
//                    HBM-bound) into the caller's workspace;
//   bwd_dkdv_kernel  one 128-key tile of one KV head per work item: the K/V
//                    tiles stay in shared memory while the q/dout tiles of
//                    every query head of the group stream past; dk and dv
//                    accumulate in tensor memory;
//   bwd_dq_kernel    one 128-row query tile per work item: q/dout stay in
//                    shared memory while the K/V tiles stream past in the
//                    forward's ring order (own chunk first); dq accumulates in
//                    tensor memory.
// Every output element is written once (no atomics), so results are
// deterministic.  Splitting dq from dk/dv recomputes S and dP in both
// tensor-core kernels (7 tile MMAs per query/key tile pair instead of 5) in
// exchange for no fp32 dq scratch and no atomic traffic.
//
// CTA organisation of both tensor-core kernels (one persistent CTA per SM):
//   warps 0-3  elementwise work on columns 0-63 of every tile row, one
//              thread per TMEM lane (query row in the dq kernel, key row in
//              the dk/dv kernel), and half of the epilogue
//   warps 4-7  the same for columns 64-127 (nothing in the backward's
//              elementwise work reduces across a row, so the halves never
//              exchange data)
//   warp  8    TMA producer
//   warp  9    MMA issuer (one thread)
//   warps 10-11 idle (they complete the producer warpgroup)
// Registers are split with setmaxnreg as in the forward kernel: 168 per
// thread at launch, 200 for the elementwise warpgroups, 104 for the rest.
// Every wait is bounded as in the forward kernel: on timeout the CTA sets the
// status word, drains its copies and MMAs, frees tensor memory and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ra_internal.h"
#include "ra_ptx.cuh"
#include "ra_umma.cuh"

namespace ra {
namespace {

constexpr int kBwdThreads = 384;     // warps 10-11 idle: they complete the producer warpgroup
constexpr int kBwdComputeWarps = 8;  // two warpgroups, one half of every row each
constexpr int kBwdWarpTma = 8;
constexpr int kBwdWarpMma = 9;
// setmaxnreg split of the 168 registers a thread gets at launch
constexpr uint32_t kBwdLaunchRegs = 168, kBwdComputeRegs = 200, kBwdProducerRegs = 104;
static_assert(2 * 128 * kBwdComputeRegs + 128 * kBwdProducerRegs == kBwdThreads * kBwdLaunchRegs,
              "register split must use exactly the launch allocation");
constexpr int kT = 128;                // rows per tile (queries or keys)
constexpr int kBlk = 128 * 128;        // one [128 rows x 64 cols] bf16 block
constexpr uint32_t kBwdTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ MMAs
// D[128 x 128] = A[128 x DH] * B[128 x DH]^T, A and B K-major tiles.
template <int DH>
__device__ __forceinline__ void mma_nt(uint32_t tD, uint32_t a_lo, uint32_t b_lo) {
  constexpr uint32_t idesc = make_idesc(kT, kT, 0);
#pragma unroll
  for (int kk = 0; kk < DH / 16; ++kk) {
    const uint32_t off = (uint32_t)((kk >> 2) * kBlk + (kk & 3) * 32) >> 4;
    mma_ss_lh_e(tD, a_lo + off, kDescHiSw128, b_lo + off, kDescHiSw128, idesc, kk > 0 ? 1u : 0u);
  }
}

// D[128 x DH] (+)= A[128 x 128] (bf16 pairs in tensor memory) * B[128 x DH]
// (an MN-major tile in shared memory).  The A operand's K = 128 columns are
// 64 packed columns: contiguous at tA when kSplitA is false; otherwise the
// first 32 at tA and the last 32 at tA + 64 (each half of the elementwise
// work packs its 64 columns inside its own 64-column half of the source).
template <int DH, bool kSplitA>
__device__ __forceinline__ void mma_tn(uint32_t tD, uint32_t tA, uint32_t b_lo, bool accumulate) {
  constexpr uint32_t idesc = make_idesc(kT, DH, 1);
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk) {
    const uint32_t a_col = kSplitA ? (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8) : (uint32_t)(kk * 8);
    mma_ts_lh_e(tD, tA + a_col, b_lo + (uint32_t)(kk * (2048 >> 4)), kDescHiSw128, idesc,
                (accumulate || kk > 0) ? 1u : 0u);
  }
}

// ------------------------------------------------------------- waits
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      const BwdArgs& a) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, a.timeout_ns, a.status);
}

// Bounded wait taken by all 32 lanes of a warp; the vote makes the outcome
// warp-uniform.  Every warp waits this way: one lane polling while the others
// park at a __syncwarp cost the elementwise warps a divergent branch and a
// reconvergence per tile (GQA backward 10.0 against 9.4 ms, D = 64 58.3
// against 52.0 ms, bit-identical).
__device__ __forceinline__ bool bwait_all(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          const BwdArgs& a) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const bool ok = wait_slow(bar, parity, abort_flag, a.timeout_ns, a.status);
  return __all_sync(0xffffffffu, ok);
}

// every elementwise warp arrives once (from the lane elect.sync picks)
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  tc_fence_before();
  __syncwarp();
  mbar_arrive_e(bar);
}

// k-th work item of this CTA: snake order over rounds of gridDim.x items
__device__ __forceinline__ int bwd_item_index(int k) {
  const int G = gridDim.x, c = blockIdx.x;
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// ------------------------------------------------------- elementwise pieces
// p = exp2(x * scale*log2e - lse*log2e) for 32 scores of one row, in place
// (fp32 bit patterns).  kMask: zero every column c with c > lim (dq kernel,
// keys past the query row) or c < lim (dk/dv kernel, queries before the key
// row), selected by kKeyRows.  nl2 points at per-column values (dk/dv kernel)
// or is null with nl2x2 holding the row's value (dq kernel).
template <bool kMask, bool kKeyRows>
__device__ __forceinline__ void exp_chunk(uint32_t (&s)[32], int c0, int lim, uint64_t c2,
                                          uint64_t nl2x2, const float* nl2) {
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    uint64_t bias = nl2x2;
    if (nl2) bias = *reinterpret_cast<const uint64_t*>(nl2 + c0 + j);
    const uint64_t xs = f2_fma(f2_pack(__uint_as_float(s[j]), __uint_as_float(s[j + 1])), c2, bias);
    float p0 = ex2(f2_lo(xs)), p1 = ex2(f2_hi(xs));
    if (kMask) {
      if (kKeyRows) {
        p0 = (c0 + j < lim) ? 0.0f : p0;
        p1 = (c0 + j + 1 < lim) ? 0.0f : p1;
      } else {
        p0 = (c0 + j > lim) ? 0.0f : p0;
        p1 = (c0 + j + 1 > lim) ? 0.0f : p1;
      }
    }
    s[j] = __float_as_uint(p0);
    s[j + 1] = __float_as_uint(p1);
  }
}

// 32 weights -> 16 packed bf16 pairs
__device__ __forceinline__ void pack_chunk(const uint32_t (&p)[32], uint32_t (&pk)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(__uint_as_float(p[2 * j]), __uint_as_float(p[2 * j + 1]));
}

// ds = p (dp - delta) for 32 columns -> 16 packed bf16 pairs.  ndl: -delta per
// column (dk/dv kernel) or null with ndl2 holding the row's -delta (dq kernel);
// the sum dp + (-delta) is the subtraction.
__device__ __forceinline__ void ds_chunk(const uint32_t (&p)[32], const uint32_t (&dp)[32], int c0,
                                         uint64_t ndl2, const float* ndl, uint32_t (&pk)[16]) {
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    uint64_t nd = ndl2;
    if (ndl) nd = *reinterpret_cast<const uint64_t*>(ndl + c0 + j);
    const uint64_t d = f2_add(f2_pack(__uint_as_float(dp[j]), __uint_as_float(dp[j + 1])), nd);
    const uint64_t ds = f2_mul(f2_pack(__uint_as_float(p[j]), __uint_as_float(p[j + 1])), d);
    pk[j >> 1] = pack_bf16x2(f2_lo(ds), f2_hi(ds));
  }
}

// NC fp32 accumulator columns of this thread's TMEM lane -> bf16 in global
// memory at dst, times `mul` (the loads run whatever `ok` says: they are
// warp-collective; the stores only when it is true).
template <int NC>
__device__ __forceinline__ void store_row(uint32_t tAcc, float mul, __nv_bfloat16* dst, bool ok) {
  uint4* row = reinterpret_cast<uint4*>(dst);
#pragma unroll 1
  for (int c0 = 0; c0 < NC; c0 += 32) {
    uint32_t o[32];
    tmem_ld32(tAcc + c0, o);
    tmem_wait_ld_regs(o);
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      w[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * mul, __uint_as_float(o[2 * j + 1]) * mul);
#pragma unroll
    for (int j = 0; j < 4 && ok; ++j)
      row[c0 / 8 + j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
}

// ====================================================== row sums (prep)
// -delta_s = -sum_d out[s,d] dout[s,d] and -lse_s*log2(e), per query row.  DH/8
// threads per row, each reading 16 bytes of out and of dout.
template <int DH>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const BwdArgs a) {
  constexpr int per = DH / 8;
  const long long rows = (long long)a.B * a.S * a.H;  // [B,S,H] order
  const long long units = rows * per;
  const long long elems = rows * DH;  // elements of out and dout
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long w0 = (long long)blockIdx.x * blockDim.x + (threadIdx.x - lane); w0 < units;
       w0 += stride) {
    const long long w = w0 + lane;
    const bool active = w < units;
    const long long row = w / per;
    const int cpart = (int)(w - row * per);
    float acc = 0.0f;
    if (active && in_bounds(row * DH + cpart * 8, 8, elems, a.bounds_trim, a.status)) {
      const long long e0 = row * DH + cpart * 8;
      const uint4 o = __ldcs(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.out) + e0));
      const uint4 g = __ldcs(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.dout) + e0));
      const uint32_t ov[4] = {o.x, o.y, o.z, o.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc = fmaf(__uint_as_float(ov[j] << 16), __uint_as_float(gv[j] << 16), acc);
        acc = fmaf(__uint_as_float(ov[j] & 0xFFFF0000u), __uint_as_float(gv[j] & 0xFFFF0000u), acc);
      }
    }
#pragma unroll
    for (int o = per / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (active && cpart == 0) {
      const int h = (int)(row % a.H);
      const long long bs = row / a.H;
      const int s = (int)(bs % a.S);
      const long long b = bs / a.S;
      const long long li = (b * a.H + h) * a.S + s;
      if (in_bounds(li, 1, rows, a.bounds_trim, a.status)) {
        a.ndelta[li] = -acc;
        a.nlse2[li] = -a.lse[li] * kLog2e;
      }
    }
  }
}

// ============================================================ dk / dv
template <int DH>
struct KvLayout {
  static constexpr int DK = DH / 64;
  // q is read by the first MMA of a step (S^T) and by the last (dk); dout by
  // the second and third, so the q ring is one stage deeper than the dout
  // ring.  A dout stage also carries the step's 128 values of -lse*log2(e)
  // and -delta (bulk copies); they are first read after S^T of the step.
  static constexpr int ND = (DH == 128) ? 2 : 4;
  static constexpr int NQ = ND + 1;
  static constexpr int TILE = kT * DH * 2;
  static constexpr int DSTAGE = TILE + 1024;
  static constexpr int NL2_IN = TILE, DL_IN = TILE + 512;  // offsets inside a dout stage
  static constexpr int K_OFF = 0, V_OFF = TILE, Q_OFF = 2 * TILE;
  static constexpr int DO_OFF = Q_OFF + NQ * TILE;
  static constexpr int BAR_OFF = DO_OFF + ND * DSTAGE;
  static constexpr int KV_FULL = 0, KV_EMPTY = 1, Q_FULL = 2, Q_EMPTY = 2 + NQ,
                       DO_FULL = 2 + 2 * NQ, DO_EMPTY = 2 + 2 * NQ + ND,
                       S_FULL = 2 + 2 * NQ + 2 * ND, S_FREE = S_FULL + 1, DP_FULL = S_FULL + 2,
                       PDS_FULL = S_FULL + 3, ACC_DONE = S_FULL + 4, DONE = S_FULL + 5,
                       N_BARS = S_FULL + 6;
  static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;
  // no alignment slack: at D = 128 this layout uses all but ~0.8 KB of the
  // 227 KB a CTA can have, so the kernel requires (and checks) a 1024-byte
  // aligned dynamic shared memory base instead of rounding it up
  static constexpr int ALLOC = MISC_OFF + 16;
  // tensor memory columns: S^T, dP^T (then P^T and dS^T as bf16 pairs: in
  // each 64-column half, P^T in the first 32 columns and dS^T in the last
  // 32), dv, dk
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 256 + DH;
  __host__ __device__ static constexpr bool per_warp(int i) { return i == S_FREE || i == PDS_FULL; }
};
static_assert(KvLayout<128>::ALLOC <= 232448, "dk/dv shared memory layout exceeds 227 KB");

struct KvItem {
  int b, kvh, t;
};

__device__ __forceinline__ KvItem kv_item(const BwdArgs& a, int x) {
  const int groups = a.B * a.Hkv;
  KvItem it;
  it.t = x / groups;  // ascending: for causal the lowest key tiles carry the most queries
  const int g = x % groups;
  it.b = g / a.Hkv;
  it.kvh = g % a.Hkv;
  return it;
}

// (query head of the group, query tile) pairs of one dk/dv item, query tiles
// ascending inside each head; causal skips query tiles before the key tile.
struct KvCursor {
  int hh, j, j0, tiles;
  __device__ __forceinline__ void init(const BwdArgs& a, const KvItem& it) {
    j0 = a.causal ? it.t : 0;
    tiles = a.tiles;
    hh = 0;
    j = j0;
  }
  __device__ __forceinline__ void next() {
    if (++j == tiles) {
      j = j0;
      ++hh;
    }
  }
};

__device__ __forceinline__ int kv_steps(const BwdArgs& a, const KvItem& it) {
  return (a.H / a.Hkv) * (a.tiles - (a.causal ? it.t : 0));
}

template <int DH>
__device__ void dkdv_tma(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                         const CUtensorMap* tdo, const BwdArgs& a, uint32_t sbase,
                         volatile int* abort_flag) {
  using L = KvLayout<DH>;
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  const uint64_t pol_keep = l2_policy_evict_last();
  const uint64_t pol_once = l2_policy_evict_first();
  const int G = a.H / a.Hkv;
  uint32_t kv_cnt = 0, g = 0;  // g: steps whose q and dout copies were both issued
  uint32_t q_cnt = 0;          // q copies issued (g or g + 1)
  bool ok = true;
  for (int k = 0; ok; ++k) {
    if (k * (int)gridDim.x >= a.n_items) break;
    const int x = bwd_item_index(k);
    if (x >= a.n_items) continue;
    const KvItem it = kv_item(a, x);
    const int ns = kv_steps(a, it);
    if (kv_cnt > 0 && !bwait(bar(L::KV_EMPTY), (kv_cnt - 1) & 1, abort_flag, a)) break;
    mbar_arrive_expect_tx(bar(L::KV_FULL), 2 * L::TILE);
    const int krow = it.b * a.S + it.t * kT;
    for (int kb = 0; kb < L::DK; ++kb) {
      tma_load_3d(sbase + L::K_OFF + kb * kBlk, tk, bar(L::KV_FULL), kb * 64, it.kvh, krow, pol_once);
      tma_load_3d(sbase + L::V_OFF + kb * kBlk, tv, bar(L::KV_FULL), kb * 64, it.kvh, krow, pol_once);
    }
    ++kv_cnt;
    KvCursor cur;
    cur.init(a, it);
    for (int u = 0; u < ns; ++u, ++g, cur.next()) {
      const int sq = g % L::NQ, sd = g % L::ND;
      const int h = it.kvh * G + cur.hh;
      const int qrow = it.b * a.S + cur.j * kT;
      if (!bwait(bar(L::Q_EMPTY + sq), ((g / L::NQ) & 1) ^ 1, abort_flag, a)) { ok = false; break; }
      mbar_arrive_expect_tx(bar(L::Q_FULL + sq), L::TILE);
      for (int kb = 0; kb < L::DK; ++kb)
        tma_load_3d(sbase + L::Q_OFF + sq * L::TILE + kb * kBlk, tq, bar(L::Q_FULL + sq), kb * 64,
                    h, qrow, pol_keep);
      ++q_cnt;
      if (!bwait(bar(L::DO_EMPTY + sd), ((g / L::ND) & 1) ^ 1, abort_flag, a)) { ok = false; break; }
      const uint32_t stage = sbase + L::DO_OFF + sd * L::DSTAGE;
      const uint32_t fb = bar(L::DO_FULL + sd);
      mbar_arrive_expect_tx(fb, L::TILE + 1024);
      if (!(a.skip_first_load && g == 0))  // test hook: the stage then never completes
        for (int kb = 0; kb < L::DK; ++kb)
          tma_load_3d(stage + kb * kBlk, tdo, fb, kb * 64, h, qrow, pol_keep);
      size_t li = ((size_t)it.b * a.H + h) * a.S + (size_t)cur.j * kT;
      // outside the workspace (bounds-checked builds): copy from its start, so
      // that the stage's barrier still completes
      if (!in_bounds(li, kT, (size_t)a.B * a.H * a.S, a.bounds_trim, a.status)) li = 0;
      bulk_load(stage + L::NL2_IN, a.nlse2 + li, 512, fb);
      bulk_load(stage + L::DL_IN, a.ndelta + li, 512, fb);
    }
  }
  if (!ok) {  // let the copies in flight land before shared memory goes away
    if (kv_cnt > 0) wait_drain(bar(L::KV_FULL), (kv_cnt - 1) & 1, a.timeout_ns);
    // every issued copy, including a q copy whose dout partner was never issued
    for (uint32_t c = (q_cnt > (uint32_t)L::NQ ? q_cnt - L::NQ : 0); c < q_cnt; ++c)
      wait_drain(bar(L::Q_FULL + c % L::NQ), (c / L::NQ) & 1, a.timeout_ns);
    for (uint32_t c = (g > (uint32_t)L::ND ? g - L::ND : 0); c < g; ++c)
      wait_drain(bar(L::DO_FULL + c % L::ND), (c / L::ND) & 1, a.timeout_ns);
  }
}

// Issue order per step u of an item (S^T = K Q^T, dP^T = V dO^T):
//   S^T(u+1)            once the elementwise warps have read S^T(u)
//   dv += P^T(u) dO(u)  once P^T(u) and dS^T(u) are in tensor memory (both in
//   dk += dS^T(u) Q(u)  the dP^T columns)
//   dP^T(u+1)           after a tcgen05.shift of 8 of the dP^T columns: it
//                       rewrites the columns dv(u) and dk(u) read, and the PTX
//                       ISA orders two MMAs on different accumulators only
//                       through a commit and wait, or through operations it
//                       lists as executing in issue order: tcgen05.mma ->
//                       tcgen05.shift -> tcgen05.mma (same cta_group)
// so the next S^T runs on the tensor cores while the warps work on this step.
// The whole MMA warp runs the loop (waits by vote); an elected lane issues.
// Against the same loop in one lane without the commit wait before dP^T:
// 10.0 against 10.6 ms per call on the GQA workload, 58.7 against 69.7 ms at
// D = 64, bit-identical gradients.  The shift in place of that commit wait:
// D = 64 51.3 against 52.1 ms, bit-identical.
template <int DH>
__device__ void dkdv_mma(const BwdArgs& a, uint32_t sbase, uint32_t tmem,
                         volatile int* abort_flag) {
  using L = KvLayout<DH>;
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  const uint32_t tS = tmem + L::S_COL, tDP = tmem + L::DP_COL;
  const uint32_t tDV = tmem + L::DV_COL, tDK = tmem + L::DK_COL;
  const uint32_t k_lo = desc_lo(sbase + L::K_OFF, 16), v_lo = desc_lo(sbase + L::V_OFF, 16);
  const uint32_t q_lo0 = desc_lo(sbase + L::Q_OFF, 16);
  const uint32_t do_lo0 = desc_lo(sbase + L::DO_OFF, 16);
  const uint32_t q_mn0 = desc_lo(sbase + L::Q_OFF, kBlk);
  const uint32_t do_mn0 = desc_lo(sbase + L::DO_OFF, kBlk);
  constexpr uint32_t kQStageLo = (uint32_t)L::TILE >> 4, kDStageLo = (uint32_t)L::DSTAGE >> 4;
  uint32_t kv_cnt = 0, g = 0;
  bool ok = true;
  for (int k = 0; ok; ++k) {
    if (k * (int)gridDim.x >= a.n_items) break;
    const int x = bwd_item_index(k);
    if (x >= a.n_items) continue;
    const KvItem it = kv_item(a, x);
    const int ns = kv_steps(a, it);
    if (!bwait_all(bar(L::KV_FULL), kv_cnt & 1, abort_flag, a)) break;
    ++kv_cnt;
    {  // prologue: S^T(0), dP^T(0), once the previous step's S^T has been read
      const int sq = g % L::NQ, sd = g % L::ND;
      if (!bwait_all(bar(L::Q_FULL + sq), (g / L::NQ) & 1, abort_flag, a)) break;
      if (g > 0 && !bwait_all(bar(L::S_FREE), (g - 1) & 1, abort_flag, a)) break;
      tc_fence_after();
      mma_nt<DH>(tS, k_lo, q_lo0 + sq * kQStageLo);
      mma_commit_e(bar(L::S_FULL));
      if (!bwait_all(bar(L::DO_FULL + sd), (g / L::ND) & 1, abort_flag, a)) break;
      tc_fence_after();
      mma_nt<DH>(tDP, v_lo, do_lo0 + sd * kDStageLo);
      mma_commit_e(bar(L::DP_FULL));
    }
    for (int u = 0; u < ns; ++u, ++g) {
      const int sq = g % L::NQ, sd = g % L::ND;
      const bool more = u + 1 < ns;
      if (more) {
        const int sq1 = (g + 1) % L::NQ;
        if (!bwait_all(bar(L::S_FREE), g & 1, abort_flag, a)) { ok = false; break; }
        if (!bwait_all(bar(L::Q_FULL + sq1), ((g + 1) / L::NQ) & 1, abort_flag, a)) { ok = false; break; }
        tc_fence_after();
        mma_nt<DH>(tS, k_lo, q_lo0 + sq1 * kQStageLo);
        mma_commit_e(bar(L::S_FULL));
      }
      if (!bwait_all(bar(L::PDS_FULL), g & 1, abort_flag, a)) { ok = false; break; }
      tc_fence_after();
      mma_tn<DH, true>(tDV, tDP, do_mn0 + sd * kDStageLo, u > 0);
      mma_commit_e(bar(L::DO_EMPTY + sd));
      mma_tn<DH, true>(tDK, tDP + 32, q_mn0 + sq * kQStageLo, u > 0);
      mma_commit_e(bar(L::Q_EMPTY + sq));
      if (more) {
        const int sd1 = (g + 1) % L::ND;
        if (!bwait_all(bar(L::DO_FULL + sd1), ((g + 1) / L::ND) & 1, abort_flag, a)) { ok = false; break; }
        // dv(u) and dk(u) read P^T(u) and dS^T(u) from the dP^T columns that
        // dP^T(u+1) rewrites: a shift of 8 of those columns between them
        // orders the two (mma -> shift -> mma execute in issue order)
        tmem_shift_down_e(tDP);
        tc_fence_after();
        mma_nt<DH>(tDP, v_lo, do_lo0 + sd1 * kDStageLo);
        mma_commit_e(bar(L::DP_FULL));
      }
    }
    if (!ok) break;
    mma_commit_e(bar(L::ACC_DONE));
    mma_commit_e(bar(L::KV_EMPTY));
  }
  mma_commit_e(bar(L::DONE));
  wait_drain(bar(L::DONE), 0, a.timeout_ns);
}

template <int DH>
__device__ void dkdv_compute(const BwdArgs& a, uint32_t sbase, uint32_t tmem,
                             volatile int* abort_flag, const uint8_t* smem) {
  using L = KvLayout<DH>;
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  const int warp = threadIdx.x >> 5;
  const int r = threadIdx.x & 127;   // key row inside the tile == TMEM lane
  const int c0 = (warp >> 2) * 64;   // this warpgroup's half of the query columns
  const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
  const uint32_t tS = tmem + lb + L::S_COL + c0, tDP = tmem + lb + L::DP_COL + c0;
  const uint32_t tDV = tmem + lb + L::DV_COL, tDK = tmem + lb + L::DK_COL;
  const uint64_t c2 = f2_pack(a.scale_log2, a.scale_log2);
  uint32_t g = 0, n_done = 0;
  for (int k = 0;; ++k) {
    if (k * (int)gridDim.x >= a.n_items) break;
    const int x = bwd_item_index(k);
    if (x >= a.n_items) continue;
    const KvItem it = kv_item(a, x);
    const int ns = kv_steps(a, it);
    KvCursor cur;
    cur.init(a, it);
    for (int u = 0; u < ns; ++u, ++g, cur.next()) {
      const uint8_t* stage = smem + L::DO_OFF + (g % L::ND) * L::DSTAGE;
      const float* nl2 = reinterpret_cast<const float*>(stage + L::NL2_IN);
      const float* dl = reinterpret_cast<const float*>(stage + L::DL_IN);
      const bool diag = a.causal && cur.j == it.t;
      // the per-column arrays arrived by bulk copy with the step's dout tile:
      // acquire them through that stage's barrier
      if (!bwait_all(bar(L::DO_FULL + g % L::ND), (g / L::ND) & 1, abort_flag, a)) return;
      if (!bwait_all(bar(L::S_FULL), g & 1, abort_flag, a)) return;
      tc_fence_after();
      uint32_t sa[32], sb[32];
      tmem_ld32(tS + 0, sa);
      tmem_ld32(tS + 32, sb);
      tmem_wait_ld_regs(sa);
      tmem_wait_ld_regs(sb);
      warp_arrive(bar(L::S_FREE));
      // P^T: queries before this key row are masked on the diagonal tile
      if (diag) {
        exp_chunk<true, true>(sa, c0, r, c2, 0, nl2);
        exp_chunk<true, true>(sb, c0 + 32, r, c2, 0, nl2);
      } else {
        exp_chunk<false, true>(sa, c0, r, c2, 0, nl2);
        exp_chunk<false, true>(sb, c0 + 32, r, c2, 0, nl2);
      }
      // dS^T = P^T (dP^T - delta).  This half's 64 dP^T columns, once read,
      // take P^T (first 32) and dS^T (last 32) as bf16 pairs.
      if (!bwait_all(bar(L::DP_FULL), g & 1, abort_flag, a)) return;
      tc_fence_after();
      uint32_t va[32], vb[32], pk[16];
      tmem_ld32(tDP + 0, va);
      tmem_ld32(tDP + 32, vb);
      tmem_wait_ld_regs(va);
      tmem_wait_ld_regs(vb);
      pack_chunk(sa, pk);
      tmem_st16(tDP + 0, pk);
      pack_chunk(sb, pk);
      tmem_st16(tDP + 16, pk);
      ds_chunk(sa, va, c0, 0, dl, pk);
      tmem_st16(tDP + 32, pk);
      ds_chunk(sb, vb, c0 + 32, 0, dl, pk);
      tmem_st16(tDP + 48, pk);
      tmem_wait_st();
      warp_arrive(bar(L::PDS_FULL));
    }
    // epilogue: this warpgroup's half of the dv and dk rows of this key
    if (!bwait_all(bar(L::ACC_DONE), n_done & 1, abort_flag, a)) return;
    ++n_done;
    tc_fence_after();
    const size_t row = ((size_t)it.b * a.S + (size_t)it.t * kT + r) * a.Hkv + it.kvh;
    const int e0 = (warp >> 2) * (DH / 2);
    const bool ok = in_bounds(row * DH + e0, DH / 2, (size_t)a.B * a.S * a.Hkv * DH, a.bounds_trim,
                              a.status);
    store_row<DH / 2>(tDV + e0, 1.0f, static_cast<__nv_bfloat16*>(a.dv) + row * DH + e0, ok);
    store_row<DH / 2>(tDK + e0, a.scale, static_cast<__nv_bfloat16*>(a.dk) + row * DH + e0, ok);
    tc_fence_before();
  }
}

// ================================================================== dq
template <int DH>
struct DqLayout {
  static constexpr int DK = DH / 64;
  // K is read by the first and the last MMA of a step (S and dq), V only by
  // the second (dP), so the K ring is one stage deeper than the V ring
  static constexpr int NV = (DH == 128) ? 2 : 4;
  static constexpr int NK = NV + 1;
  static constexpr int TILE = kT * DH * 2;
  static constexpr int Q_OFF = 0, DO_OFF = TILE, K_OFF = 2 * TILE;
  static constexpr int V_OFF = K_OFF + NK * TILE;
  static constexpr int BAR_OFF = V_OFF + NV * TILE;
  static constexpr int QD_FULL = 0, QD_EMPTY = 1, K_FULL = 2, K_EMPTY = 2 + NK,
                       V_FULL = 2 + 2 * NK, V_EMPTY = 2 + 2 * NK + NV,
                       S_FULL = 2 + 2 * NK + 2 * NV,
                       S_FREE = S_FULL + 1, DP_FULL = S_FULL + 2, DP_FREE = S_FULL + 3,
                       DS_FULL = S_FULL + 4, DQ_DONE = S_FULL + 5, DONE = S_FULL + 6,
                       N_BARS = S_FULL + 7;
  static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;
  static constexpr int ALLOC = MISC_OFF + 16 + 1024;
  // tensor memory columns: S, dP, dS (bf16 pairs), dq
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DS_COL = 256, DQ_COL = 320;
  __host__ __device__ static constexpr bool per_warp(int i) {
    return i == S_FREE || i == DP_FREE || i == DS_FULL;
  }
};

struct DqItem {
  int b, h, kvh, j;
};

__device__ __forceinline__ DqItem dq_item(const BwdArgs& a, int x) {
  const int groups = a.B * a.H;
  const int qi = x / groups, g = x % groups;
  DqItem it;
  it.j = a.causal ? a.tiles - 1 - qi : qi;  // causal: heaviest rows first
  it.b = g / a.H;
  it.h = g % a.H;
  it.kvh = it.h / (a.H / a.Hkv);
  return it;
}

// Key tiles of one query tile in the forward's ring order: its own chunk
// first (up to the diagonal tile when causal), then the chunks below it,
// wrapping around for non-causal.
struct RingCursor {
  int kt, left, c, tpc, P;
  __device__ __forceinline__ void init(const BwdArgs& a, int j) {
    tpc = a.tpc;
    P = a.P;
    c = j / tpc;
    kt = c * tpc;
    left = a.causal ? j - kt + 1 : tpc;
  }
  __device__ __forceinline__ void next() {
    if (--left > 0) {
      ++kt;
      return;
    }
    c = (c == 0) ? P - 1 : c - 1;
    kt = c * tpc;
    left = tpc;
  }
};

template <int DH>
__device__ void dq_tma(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                       const CUtensorMap* tdo, const BwdArgs& a, uint32_t sbase,
                       volatile int* abort_flag) {
  using L = DqLayout<DH>;
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  const uint64_t pol_kv = l2_policy_evict_last();
  const uint64_t pol_q = l2_policy_evict_first();
  uint32_t qd_cnt = 0, kv_cnt = 0;  // kv_cnt: steps whose K and V copies were both issued
  uint32_t k_cnt = 0;               // K copies issued (kv_cnt or kv_cnt + 1)
  bool ok = true;
  for (int k = 0; ok; ++k) {
    if (k * (int)gridDim.x >= a.n_items) break;
    const int x = bwd_item_index(k);
    if (x >= a.n_items) continue;
    const DqItem it = dq_item(a, x);
    const int ns = a.causal ? it.j + 1 : a.tiles;
    if (qd_cnt > 0 && !bwait(bar(L::QD_EMPTY), (qd_cnt - 1) & 1, abort_flag, a)) break;
    mbar_arrive_expect_tx(bar(L::QD_FULL), 2 * L::TILE);
    const int qrow = it.b * a.S + it.j * kT;
    for (int kb = 0; kb < L::DK; ++kb) {
      tma_load_3d(sbase + L::Q_OFF + kb * kBlk, tq, bar(L::QD_FULL), kb * 64, it.h, qrow, pol_q);
      tma_load_3d(sbase + L::DO_OFF + kb * kBlk, tdo, bar(L::QD_FULL), kb * 64, it.h, qrow, pol_q);
    }
    ++qd_cnt;
    RingCursor cur;
    cur.init(a, it.j);
    for (int u = 0; u < ns; ++u, ++kv_cnt, cur.next()) {
      const int sk = kv_cnt % L::NK, sv = kv_cnt % L::NV;
      const int row = it.b * a.S + cur.kt * kT;
      if (!bwait(bar(L::K_EMPTY + sk), ((kv_cnt / L::NK) & 1) ^ 1, abort_flag, a)) { ok = false; break; }
      mbar_arrive_expect_tx(bar(L::K_FULL + sk), L::TILE);
      for (int kb = 0; kb < L::DK; ++kb)
        tma_load_3d(sbase + L::K_OFF + sk * L::TILE + kb * kBlk, tk, bar(L::K_FULL + sk), kb * 64,
                    it.kvh, row, pol_kv);
      ++k_cnt;
      if (!bwait(bar(L::V_EMPTY + sv), ((kv_cnt / L::NV) & 1) ^ 1, abort_flag, a)) { ok = false; break; }
      mbar_arrive_expect_tx(bar(L::V_FULL + sv), L::TILE);
      for (int kb = 0; kb < L::DK; ++kb)
        tma_load_3d(sbase + L::V_OFF + sv * L::TILE + kb * kBlk, tv, bar(L::V_FULL + sv), kb * 64,
                    it.kvh, row, pol_kv);
    }
  }
  if (!ok) {
    if (qd_cnt > 0) wait_drain(bar(L::QD_FULL), (qd_cnt - 1) & 1, a.timeout_ns);
    // every issued copy, including a K copy whose V partner was never issued
    for (uint32_t c = (k_cnt > (uint32_t)L::NK ? k_cnt - L::NK : 0); c < k_cnt; ++c)
      wait_drain(bar(L::K_FULL + c % L::NK), (c / L::NK) & 1, a.timeout_ns);
    for (uint32_t c = (kv_cnt > (uint32_t)L::NV ? kv_cnt - L::NV : 0); c < kv_cnt; ++c)
      wait_drain(bar(L::V_FULL + c % L::NV), (c / L::NV) & 1, a.timeout_ns);
  }
}

// Issue order per step u of an item (S = Q K^T, dP = dO V^T):
//   S(u+1)     once the elementwise warps have read S(u) into registers
//   dP(u+1)    once they have read dP(u)
//   dq += dS(u) K(u)   once dS(u) is in tensor memory
// so S and dP of the next step run on the tensor cores while the elementwise
// warps work on the current one.
template <int DH>
__device__ void dq_mma(const BwdArgs& a, uint32_t sbase, uint32_t tmem, volatile int* abort_flag) {
  using L = DqLayout<DH>;
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  const uint32_t tS = tmem + L::S_COL, tDP = tmem + L::DP_COL;
  const uint32_t tDS = tmem + L::DS_COL, tDQ = tmem + L::DQ_COL;
  const uint32_t q_lo = desc_lo(sbase + L::Q_OFF, 16), do_lo = desc_lo(sbase + L::DO_OFF, 16);
  const uint32_t k_lo0 = desc_lo(sbase + L::K_OFF, 16), v_lo0 = desc_lo(sbase + L::V_OFF, 16);
  const uint32_t k_mn0 = desc_lo(sbase + L::K_OFF, kBlk);  // K as the MN-major B of dq += dS K
  constexpr uint32_t kStageLo = (uint32_t)L::TILE >> 4;
  uint32_t qd_cnt = 0, c = 0, g = 0;
  bool ok = true;
  for (int k = 0; ok; ++k) {
    if (k * (int)gridDim.x >= a.n_items) break;
    const int x = bwd_item_index(k);
    if (x >= a.n_items) continue;
    const DqItem it = dq_item(a, x);
    const int ns = a.causal ? it.j + 1 : a.tiles;
    if (!bwait_all(bar(L::QD_FULL), qd_cnt & 1, abort_flag, a)) break;
    ++qd_cnt;
    {  // prologue: S(0), dP(0), once the previous item's last S and dP are read
      const int sk = c % L::NK, sv = c % L::NV;
      if (g > 0 && !bwait_all(bar(L::S_FREE), (g - 1) & 1, abort_flag, a)) break;
      if (!bwait_all(bar(L::K_FULL + sk), (c / L::NK) & 1, abort_flag, a)) break;
      tc_fence_after();
      mma_nt<DH>(tS, q_lo, k_lo0 + sk * kStageLo);
      mma_commit_e(bar(L::S_FULL));
      if (g > 0 && !bwait_all(bar(L::DP_FREE), (g - 1) & 1, abort_flag, a)) break;
      if (!bwait_all(bar(L::V_FULL + sv), (c / L::NV) & 1, abort_flag, a)) break;
      tc_fence_after();
      mma_nt<DH>(tDP, do_lo, v_lo0 + sv * kStageLo);
      mma_commit_e(bar(L::DP_FULL));
      mma_commit_e(bar(L::V_EMPTY + sv));
      if (ns == 1) mma_commit_e(bar(L::QD_EMPTY));
    }
    for (int u = 0; u < ns; ++u, ++g, ++c) {
      const int sk = c % L::NK;
      if (u + 1 < ns) {
        const int sk1 = (c + 1) % L::NK, sv1 = (c + 1) % L::NV;
        if (!bwait_all(bar(L::S_FREE), g & 1, abort_flag, a)) { ok = false; break; }
        if (!bwait_all(bar(L::K_FULL + sk1), ((c + 1) / L::NK) & 1, abort_flag, a)) { ok = false; break; }
        tc_fence_after();
        mma_nt<DH>(tS, q_lo, k_lo0 + sk1 * kStageLo);
        mma_commit_e(bar(L::S_FULL));
        if (!bwait_all(bar(L::DP_FREE), g & 1, abort_flag, a)) { ok = false; break; }
        if (!bwait_all(bar(L::V_FULL + sv1), ((c + 1) / L::NV) & 1, abort_flag, a)) { ok = false; break; }
        tc_fence_after();
        mma_nt<DH>(tDP, do_lo, v_lo0 + sv1 * kStageLo);
        mma_commit_e(bar(L::DP_FULL));
        mma_commit_e(bar(L::V_EMPTY + sv1));
        if (u + 2 == ns) mma_commit_e(bar(L::QD_EMPTY));  // last reads of q and dout issued
      }
      if (!bwait_all(bar(L::DS_FULL), g & 1, abort_flag, a)) { ok = false; break; }
      tc_fence_after();
      mma_tn<DH, false>(tDQ, tDS, k_mn0 + sk * kStageLo, u > 0);
      mma_commit_e(bar(L::DQ_DONE));
      mma_commit_e(bar(L::K_EMPTY + sk));
    }
  }
  mma_commit_e(bar(L::DONE));
  wait_drain(bar(L::DONE), 0, a.timeout_ns);
}

template <int DH>
__device__ void dq_compute(const BwdArgs& a, uint32_t sbase, uint32_t tmem,
                           volatile int* abort_flag) {
  using L = DqLayout<DH>;
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  const int warp = threadIdx.x >> 5;
  const int r = threadIdx.x & 127;  // query row inside the tile == TMEM lane
  const int c0 = (warp >> 2) * 64;  // this warpgroup's half of the key columns
  const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
  const uint32_t tS = tmem + lb + L::S_COL + c0, tDP = tmem + lb + L::DP_COL + c0;
  const uint32_t tDS = tmem + lb + L::DS_COL + c0 / 2, tDQ = tmem + lb + L::DQ_COL;
  const uint64_t c2 = f2_pack(a.scale_log2, a.scale_log2);
  uint32_t g = 0;
  for (int k = 0;; ++k) {
    if (k * (int)gridDim.x >= a.n_items) break;
    const int x = bwd_item_index(k);
    if (x >= a.n_items) continue;
    const DqItem it = dq_item(a, x);
    const int ns = a.causal ? it.j + 1 : a.tiles;
    const size_t li = ((size_t)it.b * a.H + it.h) * a.S + (size_t)it.j * kT + r;
    const bool li_ok = in_bounds(li, 1, (size_t)a.B * a.H * a.S, a.bounds_trim, a.status);
    const float nl2 = li_ok ? a.nlse2[li] : 0.0f, ndl = li_ok ? a.ndelta[li] : 0.0f;
    const uint64_t nl2x2 = f2_pack(nl2, nl2), ndl2 = f2_pack(ndl, ndl);
    RingCursor cur;
    cur.init(a, it.j);
    for (int u = 0; u < ns; ++u, ++g, cur.next()) {
      const bool diag = a.causal && cur.kt == it.j;
      if (!bwait_all(bar(L::S_FULL), g & 1, abort_flag, a)) return;
      tc_fence_after();
      uint32_t sa[32], sb[32];
      tmem_ld32(tS + 0, sa);
      tmem_ld32(tS + 32, sb);
      tmem_wait_ld_regs(sa);
      tmem_wait_ld_regs(sb);
      warp_arrive(bar(L::S_FREE));
      // P: keys past this query row are masked on the diagonal tile
      if (diag) {
        exp_chunk<true, false>(sa, c0, r, c2, nl2x2, nullptr);
        exp_chunk<true, false>(sb, c0 + 32, r, c2, nl2x2, nullptr);
      } else {
        exp_chunk<false, false>(sa, c0, r, c2, nl2x2, nullptr);
        exp_chunk<false, false>(sb, c0 + 32, r, c2, nl2x2, nullptr);
      }
      if (!bwait_all(bar(L::DP_FULL), g & 1, abort_flag, a)) return;
      // the previous step's dq MMA has read the dS columns
      if (g > 0 && !bwait_all(bar(L::DQ_DONE), (g - 1) & 1, abort_flag, a)) return;
      tc_fence_after();
      uint32_t va[32], vb[32], pk[16];
      tmem_ld32(tDP + 0, va);
      tmem_ld32(tDP + 32, vb);
      tmem_wait_ld_regs(va);
      tmem_wait_ld_regs(vb);
      warp_arrive(bar(L::DP_FREE));
      ds_chunk(sa, va, c0, ndl2, nullptr, pk);
      tmem_st16(tDS + 0, pk);
      ds_chunk(sb, vb, c0 + 32, ndl2, nullptr, pk);
      tmem_st16(tDS + 16, pk);
      tmem_wait_st();
      warp_arrive(bar(L::DS_FULL));
    }
    // epilogue: this warpgroup's half of the dq row = scale * accumulator
    if (!bwait_all(bar(L::DQ_DONE), (g - 1) & 1, abort_flag, a)) return;
    tc_fence_after();
    const size_t row = ((size_t)it.b * a.S + (size_t)it.j * kT + r) * a.H + it.h;
    const int e0 = (warp >> 2) * (DH / 2);
    store_row<DH / 2>(tDQ + e0, a.scale, static_cast<__nv_bfloat16*>(a.dq) + row * DH + e0,
                      in_bounds(row * DH + e0, DH / 2, (size_t)a.B * a.S * a.H * DH, a.bounds_trim,
                                a.status));
    tc_fence_before();
  }
}

// ============================================================ kernels
template <class L>
__device__ __forceinline__ void init_barriers(uint32_t sbase, volatile int* abort_flag) {
  for (int i = 0; i < L::N_BARS; ++i)
    mbar_init(sbase + L::BAR_OFF + 8u * i, L::per_warp(i) ? (uint32_t)kBwdComputeWarps : 1u);
  *abort_flag = 0;
  fence_barrier_init();
  fence_proxy_async_smem();
}

template <int DH>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do, const BwdArgs a) {
  using L = KvLayout<DH>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the layout has no room to round the base up: refuse (status word) and
  // return before any barrier or tensor memory is touched if it is not aligned
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusLayout);
    return;
  }
  uint8_t* smem = smem_raw;
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  if (threadIdx.x == 0) init_barriers<L>(sbase, abort_flag);
  if (warp == kBwdWarpTma && (threadIdx.x & 31) == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
  }
  if (warp == kBwdWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  if (warp < kBwdComputeWarps) {
    regs_inc<kBwdComputeRegs>();
    dkdv_compute<DH>(a, sbase, tmem, abort_flag, smem);
  } else {
    regs_dec<kBwdProducerRegs>();
    if (warp == kBwdWarpTma && (threadIdx.x & 31) == 0)
      dkdv_tma<DH>(&tm_q, &tm_k, &tm_v, &tm_do, a, sbase, abort_flag);
    else if (warp == kBwdWarpMma)
      dkdv_mma<DH>(a, sbase, tmem, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kBwdWarpMma) {
    __syncwarp();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

template <int DH>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdArgs a) {
  using L = DqLayout<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  if (threadIdx.x == 0) init_barriers<L>(sbase, abort_flag);
  if (warp == kBwdWarpTma && (threadIdx.x & 31) == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
  }
  if (warp == kBwdWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  if (warp < kBwdComputeWarps) {
    regs_inc<kBwdComputeRegs>();
    dq_compute<DH>(a, sbase, tmem, abort_flag);
  } else {
    regs_dec<kBwdProducerRegs>();
    if (warp == kBwdWarpTma && (threadIdx.x & 31) == 0)
      dq_tma<DH>(&tm_q, &tm_k, &tm_v, &tm_do, a, sbase, abort_flag);
    else if (warp == kBwdWarpMma)
      dq_mma<DH>(a, sbase, tmem, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kBwdWarpMma) {
    __syncwarp();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

// `prepared`: this kernel's per-device preparation state (see prepare_kernel)
template <class Kernel>
cudaError_t launch_tc(Kernel kernel, int smem, std::atomic<unsigned>* prepared, int grid,
                      cudaStream_t stream, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tv, const CUtensorMap& tdo, const BwdArgs& args) {
  const cudaError_t e = prepare_kernel(kernel, (int)kBwdLaunchRegs, smem, prepared);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kBwdThreads, smem, stream>>>(tq, tk, tv, tdo, args);
  return cudaGetLastError();
}

}  // namespace

// Scratch of the allocation-free backward entry point: -lse*log2(e) and
// -delta for up to kStaticBwdRows query rows (16 MiB), in the same
// [B,H,S] + [B,H,S] layout as a caller's workspace.  Every call on a device
// shares it; nothing in it needs clearing (the row-sum kernel writes every
// value the other two kernels read).
static __device__ __align__(256) float g_bwd_scratch[2 * kStaticBwdRows];

cudaError_t bwd_static_scratch(float** p) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(p), g_bwd_scratch);
}

cudaError_t launch_bwd_prep(int D, const BwdArgs& args, int grid, cudaStream_t stream) {
  if (D == 128)
    bwd_prep_kernel<128><<<grid, 256, 0, stream>>>(args);
  else
    bwd_prep_kernel<64><<<grid, 256, 0, stream>>>(args);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const BwdArgs& args,
                            int grid, cudaStream_t stream) {
  static std::atomic<unsigned> prepared128[kMaxPrepDevices], prepared64[kMaxPrepDevices];
  if (D == 128)
    return launch_tc(bwd_dkdv_kernel<128>, KvLayout<128>::ALLOC, prepared128, grid, stream, tq, tk,
                     tv, tdo, args);
  return launch_tc(bwd_dkdv_kernel<64>, KvLayout<64>::ALLOC, prepared64, grid, stream, tq, tk, tv,
                   tdo, args);
}

cudaError_t launch_bwd_dq(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const BwdArgs& args,
                          int grid, cudaStream_t stream) {
  static std::atomic<unsigned> prepared128[kMaxPrepDevices], prepared64[kMaxPrepDevices];
  if (D == 128)
    return launch_tc(bwd_dq_kernel<128>, DqLayout<128>::ALLOC, prepared128, grid, stream, tq, tk,
                     tv, tdo, args);
  return launch_tc(bwd_dq_kernel<64>, DqLayout<64>::ALLOC, prepared64, grid, stream, tq, tk, tv,
                   tdo, args);
}

}  // namespace ra
