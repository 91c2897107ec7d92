// ra_fwd.cu -- persistent, warp-specialised ring-chunked attention forward
// for sm_103a (tcgen05 tensor cores, tensor memory, TMA).
//
// Method: the "Ring Attention" row of the mKernel overview page (table "Die
// fünf verschmolzenen Kerne"): the key/value sequence is consumed block by
// block in ring order while the next block is being moved, and each block is
// folded into the exact softmax result with the FlashAttention online-softmax
// update.  On one GPU the "ring transfer" of the next block is the TMA
// staging of the next key/value tiles into shared memory, which runs ahead of
// the tensor cores across chunk boundaries without draining.
//
// CTA organisation (one CTA per SM, persistent over work items):
//   warps 0-3  softmax + correction + epilogue for query slot 0 (TMEM lanes 0-127)
//   warps 4-7  the same for query slot 1
//   warp  8    producer (one thread): claims the CTA's next work item at run
//              time and hands its id on, then TMA-loads the Q tiles and the
//              K/V tiles into an NS-stage ring
//   warp  9    MMA issuer (the whole warp runs the loop and waits; one
//              elected lane issues each tcgen05.mma and commit):
//              S_i = Q_i K^T and O_i += P_i V
//   warps 10-11 idle (they complete the producer warpgroup)
// Registers are split with setmaxnreg: the launch gives every thread 168
// (three warps per SM sub-partition); the two softmax warpgroups raise theirs
// to 200 so a thread can hold its whole 128-column score row, the producer
// warpgroup drops to 104 (2*128*200 + 128*104 = 384*168).
// A work item is two 128-row query tiles sharing one key/value stream (two
// heads of one GQA group, or two consecutive tiles of one head), so every
// K/V tile staged in shared memory feeds two MMAs.  Items are handed out
// longest first; a CTA claims its next one when it is about to be free.
//
// Tensor memory (512 columns x 128 lanes, fp32):
//   [  0,128) S_0   (P_0 as packed bf16 overwrites its first 64 columns)
//   [128,256) S_1   (P_1 likewise)
//   [256,256+W) O_0,  [256+W,256+2W) O_1   with W = D = 128, or W = 80 at
//   D = 64 (columns 64..79 hold the PV MMA's row sum of P)
//
// Every wait is bounded: on timeout the CTA raises a shared abort flag, sets
// the device status word, lets its in-flight copies and MMAs finish (bounded
// too), frees tensor memory and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ra_internal.h"
#include "ra_ptx.cuh"
#include "ra_umma.cuh"

namespace ra {

__device__ unsigned int g_status_word;
#ifdef RA_TRACE
__device__ unsigned long long g_trace[kTraceCtas * kTraceSlots];
#endif

// RA_TRACE builds: one role's counters into this CTA's trace slots (lane 0)
__device__ __forceinline__ void trace_store(const unsigned long long* arr, int n, int first) {
#ifdef RA_TRACE
  if ((threadIdx.x & 31) == 0 && blockIdx.x < kTraceCtas)
    for (int i = 0; i < n; ++i) g_trace[blockIdx.x * kTraceSlots + first + i] = arr[i];
#else
  (void)arr;
  (void)n;
  (void)first;
#endif
}
// work-item counters: per slot the next unclaimed item and the CTAs done
__device__ unsigned int g_item_ctr[2 * kItemCounterSlots];

constexpr int kThreads = 384;
// setmaxnreg split: ptxas allocates each role's code within its share, so the
// split decides the spills (200 / 104 left a few in the softmax code; 208 / 88
// leaves none in the paired kernels and was 0.5-0.9 % faster, bit-identical)
// The D = 64 kernel for single-tile items keeps 200 / 104 (ptxas: 8 bytes of
// spill stores, 368 of spill loads; 208 / 88 the same, 192 / 120 28 and 68).
constexpr uint32_t kLaunchRegs = 168, kSoftmaxRegs = 208, kProducerRegs = 88;
constexpr uint32_t kSoftmaxRegs64Single = 200, kProducerRegs64Single = 104;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kProducerRegs == kThreads * kLaunchRegs,
              "register split must use exactly the launch allocation");
static_assert(2 * 128 * kSoftmaxRegs64Single + 128 * kProducerRegs64Single == kThreads * kLaunchRegs,
              "register split must use exactly the launch allocation");
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile
constexpr uint32_t kTmemCols = 512;
// Work items are claimed at run time from a global counter (longest first) by
// the producer thread.  The softmax warps take their ids from a ring of this
// many entries in shared memory; the MMA thread reads each id from a word the
// producer writes before arming the barrier of the item's first query tile,
// which that thread waits for anyway.
constexpr int kItemRing = 4;
constexpr uint32_t kItemConsumers = 8;  // the eight softmax warps
// Reference-max policy of the online softmax.  The reference max m is
// refreshed only when a row's max grows by more than 2^8 (O is rescaled
// rarely), and on tiles after a row's first the max pass is skipped unless a
// weight grows past 2^30.  The dominant weight is then 2^(x - m) != 1, and its
// bf16 rounding would bias O / l, so O is normalised by the sum of the
// bf16-rounded weights, the ones the PV MMA used:
//  D = 128: the softmax adds them up (a second sum beside the exact one);
//  D = 64:  the PV MMA adds them up: it runs with N = D + 16 against a block of
//    ones in shared memory, so O's column D holds the row sum of P in fp32.
//    The extra columns cost no MMA time (an N = 64 MMA is bound by its issue
//    cost, not its execution) and fit in tensor memory.
template <int D>
struct SoftmaxPolicy {
  static constexpr float kRescaleThreshold = 8.0f;  // log2 units
  static constexpr bool kMmaRowSum = (D == 64);
};

template <int D>
struct Layout {
  static constexpr int DK = D / 64;                // 128-byte swizzle blocks per row
  static constexpr int NS = (D == 128) ? 2 : 5;    // K/V ring depth
  static constexpr int BLOCK = 128 * 128;          // one [128 rows x 64 cols] bf16 block
  static constexpr int TILE = kBM * D * 2;         // one 128-row tile, all D
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + 2 * TILE;
  static constexpr int V_OFF = K_OFF + NS * TILE;
  // row-sum columns of the PV MMA (D = 64): one 64-column block of bf16 ones
  static constexpr bool kRowSum = SoftmaxPolicy<D>::kMmaRowSum;
  // D = 128: per softmax warp a 4 KiB block that turns the warp's 32 output
  // rows (one 64-column half at a time) into whole 128-byte lines per store
  // D = 64 rows are 128 bytes: 2 KiB per warp holds 16 of its 32 rows at a time
  static constexpr bool kLineStores = true;
  static constexpr int EPI_BLOCK = (D == 128) ? 4096 : 2048;
  static constexpr int EPI_OFF = V_OFF + NS * TILE;
  static constexpr int ONES_OFF = EPI_OFF + 8 * EPI_BLOCK;
  static constexpr int OW = kRowSum ? D + 16 : D;  // O columns per slot
  static constexpr int BAR_OFF = ONES_OFF + (kRowSum ? BLOCK : 0);
  // barrier indices
  static constexpr int Q_FULL = 0, Q_EMPTY = 2, K_FULL = 4, K_EMPTY = 4 + NS, V_FULL = 4 + 2 * NS,
                       V_EMPTY = 4 + 3 * NS, S_FULL = 4 + 4 * NS, P_FULL = 6 + 4 * NS,
                       O_FREE = 8 + 4 * NS, DONE = 10 + 4 * NS, ITEM_FULL = 11 + 4 * NS,
                       ITEM_EMPTY = ITEM_FULL + kItemRing, N_BARS = ITEM_EMPTY + kItemRing;
  static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;
  static constexpr int ITEM_OFF = MISC_OFF + 16;  // kItemRing work-item ids (softmax warps)
  static constexpr int QID_OFF = ITEM_OFF + 4 * kItemRing;  // id of the item in query slot 0
  static constexpr int BYTES = QID_OFF + 4;
  static constexpr int ALLOC = BYTES + 1024;  // slack to align the base to 1024 B
  __host__ __device__ static constexpr uint32_t S_COL(int i) { return 128u * i; }
  // one query tile per item: S double-buffered (its second buffer in slot 1's
  // O columns) and P double-buffered in slot 1's S columns
  __host__ __device__ static constexpr uint32_t S1T_S_COL(uint32_t i) { return i ? 384u : 0u; }
  __host__ __device__ static constexpr uint32_t S1T_P_COL(uint32_t i) { return 128u + 64u * i; }
  __host__ __device__ static constexpr uint32_t O_COL(int i) { return 256u + (uint32_t)OW * i; }
};

struct Item {
  int b, kvh;
  int h[2];
  int qt[2];
  int valid1;
};

__device__ __forceinline__ Item decode_item(const FwdArgs& a, int x) {
  const int qi = x / a.groups, g = x % a.groups;
  const int q = a.causal ? (a.nq - 1 - qi) : qi;  // causal: heaviest rows first
  const int G = a.H / a.Hkv;
  Item it;
  if (a.mode == MODE_HEADS) {
    const int hp_per = G / 2;
    it.b = g / (a.Hkv * hp_per);
    const int r = g % (a.Hkv * hp_per);
    it.kvh = r / hp_per;
    it.h[0] = it.kvh * G + 2 * (r % hp_per);
    it.h[1] = it.h[0] + 1;
    it.qt[0] = it.qt[1] = q;
    it.valid1 = 1;
  } else {
    it.b = g / a.H;
    const int h = g % a.H;
    it.kvh = h / G;
    it.h[0] = it.h[1] = h;
    if (a.mode == MODE_QTILES) {
      it.qt[0] = 2 * q;
      it.qt[1] = 2 * q + 1;
      it.valid1 = 1;
    } else {
      it.qt[0] = it.qt[1] = q;
      it.valid1 = 0;
    }
  }
  return it;
}

// plain 32-bit shared-memory accesses for the work-item ids (ordered by the
// mbarrier arrive / wait that publishes them)
__device__ __forceinline__ void st_shared_i32(uint32_t addr, int v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_shared_i32(uint32_t addr) {
  int v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ int qmax_of(const Item& it) {
  return it.valid1 ? max(it.qt[0], it.qt[1]) : it.qt[0];
}

__device__ __forceinline__ int n_steps(const FwdArgs& a, const Item& it) {
  if (a.block) {  // key tiles 0.. of the block, up to the pair's last diagonal
    if (!a.causal) return a.tiles_k;
    const int n = a.q_tile0 + qmax_of(it) - a.k_tile0 + 1;
    return n < 0 ? 0 : (n > a.tiles_k ? a.tiles_k : n);
  }
  return a.causal ? qmax_of(it) + 1 : a.tiles;
}

// Walks the key tiles of one work item in ring order: chunks from the query
// tiles' own chunk i downwards (i, i-1, i-2, ..., wrapping for non-causal),
// tiles ascending inside a chunk; causal stops the own chunk at the diagonal
// tile and never visits chunks after i.  One division per item, none per step.
struct StepCursor {
  int kt;    // current key tile
  int left;  // tiles left in the current chunk, kt included
  int j;     // current chunk
  int tpc, P;
  __device__ __forceinline__ void init(const FwdArgs& a, const Item& it) {
    if (a.block) {  // one block: its key tiles in ascending order
      tpc = P = 1;
      j = 0;
      kt = 0;
      left = 1 << 30;
      return;
    }
    tpc = a.tpc;
    P = a.P;
    j = it.qt[0] / a.tpc;
    kt = j * tpc;
    left = a.causal ? qmax_of(it) - kt + 1 : tpc;
  }
  __device__ __forceinline__ void next() {
    if (--left > 0) {
      ++kt;
      return;
    }
    j = (j == 0) ? P - 1 : j - 1;
    kt = j * tpc;
    left = tpc;
  }
};

// Key tile of the item's last step.
__device__ __forceinline__ int last_tile(const FwdArgs& a, const Item& it) {
  if (a.block) return n_steps(a, it) - 1;
  const int ci = it.qt[0] / a.tpc;
  if (a.causal) return ci > 0 ? a.tpc - 1 : qmax_of(it);
  const int j = (ci + 1 == a.P) ? 0 : ci + 1;
  return j * a.tpc + a.tpc - 1;
}

// Query tile qt has allowed keys in key tile kt.
__device__ __forceinline__ bool needs_tile(const FwdArgs& a, int qt, int kt) {
  return !a.causal || a.k_tile0 + kt <= a.q_tile0 + qt;
}

// The key tile is the query tile's diagonal (causal only): mask keys past the row.
__device__ __forceinline__ bool is_diag(const FwdArgs& a, int qt, int kt) {
  return a.causal && a.k_tile0 + kt == a.q_tile0 + qt;
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, const FwdArgs& a) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, a.timeout_ns, a.status);
}

// Bounded wait taken by all 32 lanes of a warp; the vote makes the outcome
// (and so the branch that follows) warp-uniform.  Every warp that waits does
// it this way: a wait polled by one lane while the others park at a
// __syncwarp cost the softmax warps a divergent branch and a reconvergence per
// tile (the GQA workload: 3.30 against 3.07 ms, the D = 64 one 22.9 against
// 18.7 ms, bit-identical).
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         const FwdArgs& a) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const bool ok = wait_slow(bar, parity, abort_flag, a.timeout_ns, a.status);
  return __all_sync(0xffffffffu, ok);
}

// The k-th work item id of this CTA for a softmax warp (warp-collective call),
// from the ring the producer fills; -1 when the sequence has ended or a wait
// gave up.  The warp frees the ring entry at once.
template <int D>
__device__ __forceinline__ int next_item(const FwdArgs& a, uint32_t sbase, int k,
                                         volatile int* abort_flag) {
  using L = Layout<D>;
  const int rs = k % kItemRing;
  const uint32_t full = sbase + L::BAR_OFF + 8u * (L::ITEM_FULL + rs);
  const uint32_t empty = sbase + L::BAR_OFF + 8u * (L::ITEM_EMPTY + rs);
  if (!wait_all(full, (uint32_t)(k / kItemRing) & 1u, abort_flag, a)) return -1;
  const int x = ld_shared_i32(sbase + L::ITEM_OFF + 4 * rs);
  __syncwarp();
  mbar_arrive_e(empty);
  return x;
}

// ----------------------------------------------------------------- producer
template <int D>
__device__ void tma_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                         const FwdArgs& a, uint32_t sbase, volatile int* abort_flag) {
  using L = Layout<D>;
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  const uint64_t pol_kv = l2_policy_evict_last();
  const uint64_t pol_q = l2_policy_evict_first();
  uint32_t q_cnt[2] = {0, 0};
  uint32_t kv_cnt = 0;  // steps whose K and V copies were both issued
  uint32_t k_cnt = 0;   // K copies issued (kv_cnt or kv_cnt + 1)
  bool ok = true;
  // Work items are taken in order, longest first.  CTA c starts with item c;
  // the items after the first gridDim.x are claimed from the launch's counter.
  // The next claim is made when this thread reaches the current item's last
  // key/value step (three steps before it for paired items at D = 128): its
  // latency hides behind the consumers' remaining steps,
  // and an item goes to the CTA that is about to be free, so slower SMs claim
  // fewer items.
  const int first_claimed = (int)gridDim.x;
  int claim = (int)blockIdx.x;
  RA_TR_DECL(tr, 3);
  for (int k = 0; ok; ++k) {
    const int x = claim;
    const int rs = k % kItemRing;
    if (k >= kItemRing &&
        !wait_bounded(bar(L::ITEM_EMPTY + rs), (uint32_t)((k / kItemRing) - 1) & 1u, abort_flag, a)) {
      ok = false;
      break;
    }
    st_shared_i32(sbase + L::ITEM_OFF + 4 * rs, x < a.n_items ? x : -1);
    mbar_arrive(bar(L::ITEM_FULL + rs));  // release: the id is visible to whoever acquires it
    if (x >= a.n_items) {
      // the end, for the MMA thread: -1 in the slot-0 id word, through the
      // slot's barrier (one arrival, no bytes) once the slot is free
      if (q_cnt[0] > 0 &&
          !wait_bounded(bar(L::Q_EMPTY + 0), (q_cnt[0] - 1) & 1, abort_flag, a)) {
        ok = false;
        break;
      }
      st_shared_i32(sbase + L::QID_OFF, -1);
      mbar_arrive(bar(L::Q_FULL + 0));
      ++q_cnt[0];
      break;
    }
    const Item it = decode_item(a, x);
    const int ns = n_steps(a, it);
    if (ns == 0) {  // every key of the block is in the future of every row
      claim = first_claimed + (int)atomicAdd(a.item_ctr, 1u);
      continue;
    }
#pragma unroll
    for (int slot = 0; slot < 2 && ok; ++slot) {
      if (slot == 1 && !it.valid1) continue;
      RA_TR_NOW(tr_q);
      if (q_cnt[slot] > 0 &&
          !wait_bounded(bar(L::Q_EMPTY + slot), (q_cnt[slot] - 1) & 1, abort_flag, a)) {
        ok = false;
        break;
      }
      RA_TR_ADD(tr, 2, tr_q);
      if (slot == 0) st_shared_i32(sbase + L::QID_OFF, x);  // released by the arrive below
      mbar_arrive_expect_tx(bar(L::Q_FULL + slot), L::TILE);
      for (int kb = 0; kb < L::DK; ++kb)
        tma_load_3d(sbase + L::Q_OFF + slot * L::TILE + kb * L::BLOCK, tq, bar(L::Q_FULL + slot),
                    kb * 64, it.h[slot], it.b * a.S + it.qt[slot] * kBM, pol_q);
      ++q_cnt[slot];
    }
    StepCursor cur;
    cur.init(a, it);
    for (int u = 0; u < ns && ok; ++u, cur.next()) {
      const int kt = cur.kt;
      const int st = kv_cnt % L::NS;
      const uint32_t ph = (kv_cnt / L::NS) & 1;
      const int row = it.b * a.Sk + kt * kBN;
      // Paired items at D = 128 claim three steps before their end (the ring
      // is only two steps deep there), so that the next item's query tiles,
      // prefetched into L2 below, arrive before its copies are issued: GQA
      // 2.615 against 2.623 ms, long context 11.00 against 11.16 ms.
      const int claim_u = (D == 128 && a.mode != MODE_SINGLE) ? (ns > 3 ? ns - 3 : 0) : ns - 1;
      if (u == claim_u) {
        claim = first_claimed + (int)atomicAdd(a.item_ctr, 1u);  // the next item
        // Paired items at D = 128: the next item's query tiles go into L2 now;
        // their copies wait for this item's query slots and then find them
        // there.  GQA workload 2.613 against 2.643 ms, bit-identical; at
        // D = 64 (17.09 against 16.98 ms) and for one-tile items (S = 4096:
        // 0.0435 against 0.0420 ms) it was slower, so it is left out there.
        if (D == 128 && a.mode != MODE_SINGLE && claim < a.n_items) {
          const Item nx = decode_item(a, claim);
          for (int slot = 0; slot < (nx.valid1 ? 2 : 1); ++slot)
            for (int kb = 0; kb < L::DK; ++kb)
              tma_prefetch_3d(tq, kb * 64, nx.h[slot], nx.b * a.S + nx.qt[slot] * kBM);
        }
      }
      RA_TR_NOW(tr_k);
      if (!wait_bounded(bar(L::K_EMPTY + st), ph ^ 1, abort_flag, a)) { ok = false; break; }
      RA_TR_ADD(tr, 0, tr_k);
      mbar_arrive_expect_tx(bar(L::K_FULL + st), L::TILE);
      for (int kb = 0; kb < L::DK; ++kb)
        tma_load_3d(sbase + L::K_OFF + st * L::TILE + kb * L::BLOCK, tk, bar(L::K_FULL + st),
                    kb * 64, it.kvh, row, pol_kv);
      ++k_cnt;
      RA_TR_NOW(tr_v);
      if (!wait_bounded(bar(L::V_EMPTY + st), ph ^ 1, abort_flag, a)) { ok = false; break; }
      RA_TR_ADD(tr, 1, tr_v);
      mbar_arrive_expect_tx(bar(L::V_FULL + st), L::TILE);
      if (!(a.skip_value_load && kv_cnt == 0))
        for (int kb = 0; kb < L::DK; ++kb)
          tma_load_3d(sbase + L::V_OFF + st * L::TILE + kb * L::BLOCK, tv, bar(L::V_FULL + st),
                      kb * 64, it.kvh, row, pol_kv);
      ++kv_cnt;
    }
  }
#ifdef RA_TRACE
  trace_store(tr, 3, 28);
#endif
  // the last claim has returned (its value is used here) before this CTA can
  // count itself done and the last CTA resets the counter
  asm volatile("" ::"r"(claim));
  if (!ok) {
    // Let every copy this thread issued land before shared memory goes away:
    // wait (bounded) for the last armed phase of each full barrier.
    for (int slot = 0; slot < 2; ++slot)
      if (q_cnt[slot] > 0) wait_drain(bar(L::Q_FULL + slot), (q_cnt[slot] - 1) & 1, a.timeout_ns);
    // every issued copy, including a K copy whose V partner was never issued
    for (uint32_t c = (k_cnt > (uint32_t)L::NS ? k_cnt - L::NS : 0); c < k_cnt; ++c)
      wait_drain(bar(L::K_FULL + c % L::NS), (c / L::NS) & 1, a.timeout_ns);
    for (uint32_t c = (kv_cnt > (uint32_t)L::NS ? kv_cnt - L::NS : 0); c < kv_cnt; ++c)
      wait_drain(bar(L::V_FULL + c % L::NS), (c / L::NS) & 1, a.timeout_ns);
  }
}

// ---------------------------------------------------------------- MMA issuer
// P_i(u) is written over the first columns of S_i, so S_i(u+1) = Q_i K(u+1)^T
// must not start before O_i += P_i(u) V(u) has read them.  The PTX ISA orders
// two tcgen05.mma of one thread directly only when they share the accumulator
// (and shape); these two do not.  It lists other pairs of tcgen05 operations
// that execute in issue order, among them tcgen05.mma -> tcgen05.shift and
// tcgen05.shift -> tcgen05.mma (same cta_group), and it orders completion as
// observed through tcgen05.commit and an mbarrier wait.  The issue orders:
//   MMA_ORDER_BRIDGED (default): per key/value step u, for each slot in turn:
//     O_i += P_i(u) V(u); a tcgen05.shift of one 32-byte column block of S_i
//     that holds consumed scores (columns 64-71: not P, and rewritten by the
//     next S anyway); S_i(u+1).  PV -> shift -> S execute in issue order by
//     the two pairs above, so S_i(u+1) writes its columns after the PV has
//     read P, with no wait and no drain of the pipe.  GQA workload 2.80
//     against 3.15 ms for the commit-wait form, D = 64 18.1 against 18.5 ms,
//     bit-identical.
//   MMA_ORDER_STRICT: the same, with a wait for the PV's commit (O_FREE)
//     instead of the shift: ordered by completion; the tensor pipe drains once
//     per tile (the last PV MMA's execution plus the commit's round trip).
//   MMA_ORDER_GROUPED: both slots' PV products, then each slot's S after the
//     commit of its PV.  The wait for slot 0 overlaps slot 1's PV, so the pipe
//     does not drain, but the two slots' softmax warps run in phase and compete
//     for the same exp and issue slots: 3.21 against 3.15 ms (strict).
//   MMA_ORDER_INORDER: per slot, PV and the next S back to back with nothing
//     between, relying on the tensor pipe executing two MMAs with different
//     accumulators in issue order, which no document states; kept only to
//     measure against (2.72 ms on the GQA workload).
// The first S of an item still waits for the commit of the slot's last PV of
// the previous item (bridging it as well was slower: 18.6 against 18.1 ms at
// D = 64).
// A launch with one query tile per item (MODE_SINGLE) leaves slot 1 idle, so
// the kernel is built a second time (SINGLE = true) with a loop of its own
// (mma_role_single) that runs S two steps ahead in slot 1's free columns; the
// MMA order does not apply there.  S = 4096 workload (256 single-tile items):
// 0.0457 against 0.0534 ms for the form with one S buffer, bit-identical; the
// paired kernels are unchanged.
// The whole MMA warp runs the loop: every wait is taken by all 32 lanes
// (a vote makes its outcome warp-uniform), and each tcgen05.mma and
// tcgen05.commit is issued by the one lane elect.sync picks.  Measured against
// a loop run by a single lane (GQA workload, strict order): 3.43 against
// 3.48 ms, and 23.2 against 24.8 ms on the D = 64 workload, bit-identical
// outputs.  Back-to-back MMAs run at the pipe's rate however their operands
// are formed (a microbenchmark: 64 cycles per M128 N128 K16 MMA), so the time
// between MMA groups (waits, commits) is what the loop keeps short:
// descriptors are precomputed halves plus immediate offsets, and the step
// sequence comes from a division-free cursor.

// At D = 64 a group of MMAs is issued under one elect.sync (D = 64 17.14
// against 17.43 ms); at D = 128 each MMA has its own (grouped: GQA 2.733
// against 2.649 ms).  The same MMAs either way.
template <int D>
__device__ __forceinline__ void issue_s(uint32_t tS, uint32_t q_lo, uint32_t k_lo) {
  using L = Layout<D>;
  constexpr uint32_t idesc_s = make_idesc(kBM, kBN, 0);
  if constexpr (D == 64) {
    uint32_t qa[D / 16], kb[D / 16];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (uint32_t)((kk >> 2) * L::BLOCK + (kk & 3) * 32) >> 4;
      qa[kk] = q_lo + off;
      kb[kk] = k_lo + off;
    }
    mma_ss_group_e<D / 16>(tS, qa, kb, kDescHiSw128, idesc_s, 0u);
  } else {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (uint32_t)((kk >> 2) * L::BLOCK + (kk & 3) * 32) >> 4;
      mma_ss_lh_e(tS, q_lo + off, kDescHiSw128, k_lo + off, kDescHiSw128, idesc_s, kk > 0 ? 1u : 0u);
    }
  }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tP, uint32_t v_lo, bool accumulate) {
  constexpr uint32_t idesc_pv = make_idesc(kBM, Layout<D>::OW, 1);
  if constexpr (D == 64) {
    uint32_t pa[kBN / 16], vb[kBN / 16];
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk) {
      pa[kk] = tP + kk * 8;
      vb[kk] = v_lo + (uint32_t)(kk * (2048 >> 4));
    }
    mma_ts_group_e<kBN / 16>(tO, pa, vb, kDescHiSw128, idesc_pv, accumulate ? 1u : 0u);
  } else {
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk)
      mma_ts_lh_e(tO, tP + kk * 8, v_lo + (uint32_t)(kk * (2048 >> 4)), kDescHiSw128, idesc_pv,
                (accumulate || kk > 0) ? 1u : 0u);
  }
}

// A PV product and the commit of its completion to `bar`; at D = 64 under one
// elect.sync (the same instructions in the same order)
template <int D>
__device__ __forceinline__ void issue_pv_commit(uint32_t tO, uint32_t tP, uint32_t v_lo,
                                                bool accumulate, uint32_t bar) {
  if constexpr (D == 64) {
    constexpr uint32_t idesc_pv = make_idesc(kBM, Layout<D>::OW, 1);
    uint32_t pa[kBN / 16], vb[kBN / 16];
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk) {
      pa[kk] = tP + kk * 8;
      vb[kk] = v_lo + (uint32_t)(kk * (2048 >> 4));
    }
    mma_ts_group8_commit_e(tO, pa, vb, kDescHiSw128, idesc_pv, accumulate ? 1u : 0u, bar);
  } else {
    issue_pv<D>(tO, tP, v_lo, accumulate);
    mma_commit_e(bar);
  }
}

// The bridged order's next S: a tcgen05.shift of 8 consumed S columns, the S
// product and the commit of its completion to `bar`; at D = 64 under one
// elect.sync, after the fence (the same instructions in the same order)
template <int D>
__device__ __forceinline__ void issue_shift_s_commit(uint32_t shift_taddr, uint32_t tS,
                                                     uint32_t q_lo, uint32_t k_lo, uint32_t bar) {
  if constexpr (D == 64) {
    using L = Layout<D>;
    constexpr uint32_t idesc_s = make_idesc(kBM, kBN, 0);
    uint32_t qa[D / 16], kb[D / 16];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (uint32_t)((kk >> 2) * L::BLOCK + (kk & 3) * 32) >> 4;
      qa[kk] = q_lo + off;
      kb[kk] = k_lo + off;
    }
    tc_fence_after();
    mma_shift_ss_group4_commit_e(shift_taddr, tS, qa, kb, kDescHiSw128, idesc_s, bar);
  } else {
    tmem_shift_down_e(shift_taddr);
    tc_fence_after();
    issue_s<D>(tS, q_lo, k_lo);
    mma_commit_e(bar);
  }
}

// One query tile per item (slot 1 idle): S runs two steps ahead of PV.  The
// n-th S goes to buffer n % 2 and the softmax writes the n-th P to P buffer
// n % 2, so S(u+2) can start as soon as the softmax has handed over P(u), and
// the tensor cores compute it while the softmax works on S(u+1).  The slot's
// two S_FULL and two P_FULL barriers are one per buffer (a softmax warp can be
// a tile ahead of its warpgroup, never two).  Orders:
// S(u+2) rewrites S buffer u % 2 after PV(u) was issued and after P_FULL(u)
// (the softmax is done with S(u)); P(u+2) is written after S_FULL(u+2), whose
// commit follows PV(u); the softmax's rare O rescale at tile u+1 waits for
// the O_FREE commit of PV(u) itself.
template <int D>
__device__ void mma_role_single(const FwdArgs& a, uint32_t sbase, uint32_t tmem,
                                volatile int* abort_flag) {
  using L = Layout<D>;
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  const uint32_t tO0 = tmem + L::O_COL(0);
  const uint32_t q_lo0 = desc_lo(sbase + L::Q_OFF, 16);
  const uint32_t k_lo0 = desc_lo(sbase + L::K_OFF, 16);
  const uint32_t v_lo0 = desc_lo(sbase + L::V_OFF, L::kRowSum ? (uint32_t)(L::ONES_OFF - L::V_OFF) : L::BLOCK);
  constexpr uint32_t kStageLo = (uint32_t)L::TILE >> 4;
  auto v_desc = [&](int st) -> uint32_t {
    return L::kRowSum ? v_lo0 + st * kStageLo - ((st * kStageLo) << 16) : v_lo0 + st * kStageLo;
  };
  uint32_t s_cnt = 0;  // S products issued (the n-th into S buffer n % 2)
  uint32_t p_cnt = 0;  // PV products issued (the n-th reads P buffer n % 2)
  uint32_t q_cnt = 0;
  uint32_t c = 0;      // ring position of the current step
  bool ok = true;
  RA_TR_DECL(tr, 10);  // the same counter slots as the paired loop's
  RA_TR_NOW(tr_begin);
  while (ok) {
    RA_TR_NOW(tr_item);
    if (!wait_all(bar(L::Q_FULL + 0), q_cnt & 1, abort_flag, a)) break;
    ++q_cnt;
    const int x = ld_shared_i32(sbase + L::QID_OFF);
    if (x < 0) break;
    const Item it = decode_item(a, x);
    const int ns = n_steps(a, it);
    const int lim0 = a.causal ? a.q_tile0 + it.qt[0] - a.k_tile0 : INT_MAX;
    StepCursor cs;  // the step whose S is issued next
    cs.init(a, it);
    // S of the step cs points at, from K at ring position cpos
    auto issue_next_s = [&](uint32_t cpos) -> bool {
      const int st = cpos % L::NS;
      RA_TR_NOW(tr_k);
      if (!wait_all(bar(L::K_FULL + st), (cpos / L::NS) & 1, abort_flag, a)) return false;
      RA_TR_ADD(tr, 6, tr_k);
      if (cs.kt <= lim0) {
        RA_TR_NOW(tr_s);
        const uint32_t buf = s_cnt & 1u;
        tc_fence_after();
        issue_s<D>(tmem + L::S1T_S_COL(buf), q_lo0, k_lo0 + st * kStageLo);
        mma_commit_e(bar(L::S_FULL + (int)buf));
        RA_TR_ADD(tr, 3, tr_s);
        ++s_cnt;
      }
      mma_commit_e(bar(L::K_EMPTY + st));
      return true;
    };
    // prologue: S of steps 0 and 1
    if (!issue_next_s(c)) break;
    if (ns > 1) {
      cs.next();
      if (!issue_next_s(c + 1)) break;
    }
    if (ns <= 2) mma_commit_e(bar(L::Q_EMPTY + 0));  // the item's last S is issued
    StepCursor cp;  // the step whose PV is issued now
    cp.init(a, it);
    bool first = true;
    RA_TR_ADD(tr, 7, tr_item);
    RA_TR_INC(tr, 9);
    for (int u = 0; u < ns && ok; ++u, ++c, cp.next()) {
      const int st = c % L::NS;
      RA_TR_NOW(tr_w);
      if (!wait_all(bar(L::V_FULL + st), (c / L::NS) & 1, abort_flag, a)) { ok = false; break; }
      RA_TR_ADD(tr, 2, tr_w);
#ifdef RA_TRACE
      if (u == 0) RA_TR_ADD(tr, 8, tr_w);
#endif
      RA_TR_INC(tr, 4);
      if (cp.kt <= lim0) {
        // P_FULL per P buffer: a softmax warp may run a tile ahead of the
        // others (its next S is already there), so the arrivals of tile n and
        // n + 1 go to different barriers
        RA_TR_NOW(tr_p);
        if (!wait_all(bar(L::P_FULL + (int)(p_cnt & 1u)), (p_cnt >> 1) & 1u, abort_flag, a)) {
          ok = false;
          break;
        }
        RA_TR_ADD(tr, 0, tr_p);
        RA_TR_NOW(tr_i);
        tc_fence_after();
        issue_pv<D>(tO0, tmem + L::S1T_P_COL(p_cnt & 1u), v_desc(st), !first);
        mma_commit_e(bar(L::O_FREE + 0));
        RA_TR_ADD(tr, 1, tr_i);
        ++p_cnt;
        first = false;
      }
      mma_commit_e(bar(L::V_EMPTY + st));
      if (u + 2 < ns) {
        cs.next();
        if (!issue_next_s(c + 2)) { ok = false; break; }
        if (u + 3 == ns) mma_commit_e(bar(L::Q_EMPTY + 0));
      }
    }
  }
#ifdef RA_TRACE
  RA_TR_ADD(tr, 5, tr_begin);
  trace_store(tr, 8, 0);
  trace_store(tr + 8, 2, 24);
#endif
  // Every MMA this thread issued completes before tensor memory is freed.
  mma_commit_e(bar(L::DONE));
  wait_drain(bar(L::DONE), 0, a.timeout_ns);
}

template <int D, int ORDER>
__device__ void mma_role(const FwdArgs& a, uint32_t sbase, uint32_t tmem,
                         volatile int* abort_flag) {
  using L = Layout<D>;
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  const uint32_t tS0 = tmem + L::S_COL(0), tS1 = tmem + L::S_COL(1);
  const uint32_t tO0 = tmem + L::O_COL(0), tO1 = tmem + L::O_COL(1);
  const uint32_t q_lo0 = desc_lo(sbase + L::Q_OFF, 16);
  const uint32_t q_lo1 = desc_lo(sbase + L::Q_OFF + L::TILE, 16);
  const uint32_t k_lo0 = desc_lo(sbase + L::K_OFF, 16);
  const uint32_t v_lo0 = desc_lo(sbase + L::V_OFF, L::kRowSum ? (uint32_t)(L::ONES_OFF - L::V_OFF) : L::BLOCK);
  constexpr uint32_t kStageLo = (uint32_t)L::TILE >> 4;  // descriptor step between ring stages
  // V of ring stage st: start address st tiles on; with the row-sum columns its
  // second N block is the ones block, so the leading byte offset shrinks by a
  // tile per stage (it lives in bits 16..29 of the descriptor's low word)
  auto v_desc = [&](int st) -> uint32_t {
    return L::kRowSum ? v_lo0 + st * kStageLo - ((st * kStageLo) << 16) : v_lo0 + st * kStageLo;
  };
  uint32_t s_cnt0 = 0, s_cnt1 = 0;  // S MMAs issued per slot (== PV MMAs once a step is done)
  uint32_t q_cnt0 = 0, q_cnt1 = 0;
  uint32_t c = 0;                   // ring position of the current step
  bool ok = true;
  RA_TR_DECL(tr, 14);
  RA_TR_NOW(tr_begin);

  while (ok) {
    RA_TR_NOW(tr_item);
    // the next item with work: its id comes with its first query tile (-1: none left)
    RA_TR_NOW(tr_q);
    if (!wait_all(bar(L::Q_FULL + 0), q_cnt0 & 1, abort_flag, a)) break;
    ++q_cnt0;
    const int x = ld_shared_i32(sbase + L::QID_OFF);
    if (x < 0) break;
    const Item it = decode_item(a, x);
    const int ns = n_steps(a, it);
    if (it.valid1) {
      if (!wait_all(bar(L::Q_FULL + 1), q_cnt1 & 1, abort_flag, a)) break;
      ++q_cnt1;
    }
    RA_TR_ADD(tr, 10, tr_q);
    // slot i needs key tile kt iff kt <= lim_i (needs_tile's causal test,
    // taken once per item instead of per step; -1: the item has no slot 1)
    const int lim0 = a.causal ? a.q_tile0 + it.qt[0] - a.k_tile0 : INT_MAX;
    const int lim1 = !it.valid1 ? -1 : (a.causal ? a.q_tile0 + it.qt[1] - a.k_tile0 : INT_MAX);
    StepCursor nxt;  // the step whose S MMAs are issued next
    nxt.init(a, it);
    // prologue: S(0) for both slots
    {
      const int st = c % L::NS;
      if (!wait_all(bar(L::K_FULL + st), (c / L::NS) & 1, abort_flag, a)) break;
      if (nxt.kt <= lim0) {
        RA_TR_NOW(tr_o);
        if (s_cnt0 > 0 && !wait_all(bar(L::O_FREE + 0), (s_cnt0 - 1) & 1, abort_flag, a)) break;
        RA_TR_ADD(tr, 11, tr_o);
        tc_fence_after();
        issue_s<D>(tS0, q_lo0, k_lo0 + st * kStageLo);
        mma_commit_e(bar(L::S_FULL + 0));
        ++s_cnt0;
      }
      if (nxt.kt <= lim1) {
        RA_TR_NOW(tr_o);
        if (s_cnt1 > 0 && !wait_all(bar(L::O_FREE + 1), (s_cnt1 - 1) & 1, abort_flag, a)) break;
        RA_TR_ADD(tr, 11, tr_o);
        tc_fence_after();
        issue_s<D>(tS1, q_lo1, k_lo0 + st * kStageLo);
        mma_commit_e(bar(L::S_FULL + 1));
        ++s_cnt1;
      }
      mma_commit_e(bar(L::K_EMPTY + st));
      if (ns == 1) {
        mma_commit_e(bar(L::Q_EMPTY + 0));
        if (it.valid1) mma_commit_e(bar(L::Q_EMPTY + 1));
      }
    }
    bool first0 = true, first1 = true;
    RA_TR_ADD(tr, 7, tr_item);
    RA_TR_INC(tr, 9);
    for (int u = 0; u < ns && ok; ++u, ++c) {
      RA_TR_NOW(tr_top);
      const int st = c % L::NS;
      const bool n0 = nxt.kt <= lim0, n1 = nxt.kt <= lim1;
      const bool more = u + 1 < ns;
      if (more) nxt.next();
      const bool m0 = more && nxt.kt <= lim0, m1 = more && nxt.kt <= lim1;
      const int st1 = (c + 1) % L::NS;
      RA_TR_ADD(tr, 12, tr_top);
      RA_TR_NOW(tr_w);
      if (!wait_all(bar(L::V_FULL + st), (c / L::NS) & 1, abort_flag, a)) { ok = false; break; }
      RA_TR_ADD(tr, 2, tr_w);
#ifdef RA_TRACE
      if (u == 0) RA_TR_ADD(tr, 8, tr_w);
#endif
      RA_TR_INC(tr, 4);
      // K(u+1) is needed only by the next S products.  At D = 128 (a 2-deep
      // ring) it is waited for after slot 0's PV, which gives its copy that much
      // longer to land: GQA 2.72 against 2.81 ms.  At D = 64 the 5-deep ring has
      // it in place, and the later wait only lengthens the chain (18.6 against
      // 18.1 ms), so it stays at the top of the step there.
      constexpr bool kLateK = (D == 128 && ORDER == MMA_ORDER_BRIDGED);
      bool k_ready = !more;
      if (!kLateK) {
        if (more &&
            !wait_all(bar(L::K_FULL + st1), ((c + 1) / L::NS) & 1, abort_flag, a)) { ok = false; break; }
        k_ready = true;
      }
      if (ORDER == MMA_ORDER_GROUPED) {
        // both PV products, then each slot's next S once its PV has completed
        if (n0) {
          RA_TR_NOW(tr_p);
          if (!wait_all(bar(L::P_FULL + 0), (s_cnt0 - 1) & 1, abort_flag, a)) { ok = false; break; }
          RA_TR_ADD(tr, 0, tr_p);
          RA_TR_NOW(tr_i);
          tc_fence_after();
          issue_pv<D>(tO0, tS0, v_desc(st), !first0);
          mma_commit_e(bar(L::O_FREE + 0));
          RA_TR_ADD(tr, 1, tr_i);
          first0 = false;
        }
        if (n1) {
          RA_TR_NOW(tr_p);
          if (!wait_all(bar(L::P_FULL + 1), (s_cnt1 - 1) & 1, abort_flag, a)) { ok = false; break; }
          RA_TR_ADD(tr, 0, tr_p);
          RA_TR_NOW(tr_i);
          tc_fence_after();
          issue_pv<D>(tO1, tS1, v_desc(st), !first1);
          mma_commit_e(bar(L::O_FREE + 1));
          RA_TR_ADD(tr, 1, tr_i);
          first1 = false;
        }
        mma_commit_e(bar(L::V_EMPTY + st));
        if (m0) {
          // the PV just issued for slot 0 (the O_FREE commit of S tile s_cnt0)
          if (!wait_all(bar(L::O_FREE + 0), (s_cnt0 - 1) & 1, abort_flag, a)) { ok = false; break; }
          tc_fence_after();
          issue_s<D>(tS0, q_lo0, k_lo0 + st1 * kStageLo);
          mma_commit_e(bar(L::S_FULL + 0));
          ++s_cnt0;
        }
        if (m1) {
          if (s_cnt1 > 0 &&
              !wait_all(bar(L::O_FREE + 1), (s_cnt1 - 1) & 1, abort_flag, a)) { ok = false; break; }
          tc_fence_after();
          issue_s<D>(tS1, q_lo1, k_lo0 + st1 * kStageLo);
          mma_commit_e(bar(L::S_FULL + 1));
          ++s_cnt1;
        }
        if (more) mma_commit_e(bar(L::K_EMPTY + st1));
      } else {
        // slot 0: PV(u), then S(u+1)
        if (n0) {
          RA_TR_NOW(tr_p);
          if (!wait_all(bar(L::P_FULL + 0), (s_cnt0 - 1) & 1, abort_flag, a)) { ok = false; break; }
          RA_TR_ADD(tr, 0, tr_p);
          RA_TR_NOW(tr_i);
          tc_fence_after();
          issue_pv_commit<D>(tO0, tS0, v_desc(st), !first0, bar(L::O_FREE + 0));
          RA_TR_ADD(tr, 1, tr_i);
          first0 = false;
        }
        if (more && !k_ready) {
          RA_TR_NOW(tr_k);
          if (!wait_all(bar(L::K_FULL + st1), ((c + 1) / L::NS) & 1, abort_flag, a)) { ok = false; break; }
          RA_TR_ADD(tr, 6, tr_k);
          k_ready = true;
        }
        if (m0) {
          RA_TR_NOW(tr_s);
          if constexpr (ORDER == MMA_ORDER_BRIDGED) {
            issue_shift_s_commit<D>(tS0 + 64u, tS0, q_lo0, k_lo0 + st1 * kStageLo, bar(L::S_FULL + 0));
          } else {
            if (ORDER == MMA_ORDER_STRICT &&
                !wait_all(bar(L::O_FREE + 0), (s_cnt0 - 1) & 1, abort_flag, a)) { ok = false; break; }
            tc_fence_after();
            issue_s<D>(tS0, q_lo0, k_lo0 + st1 * kStageLo);
            mma_commit_e(bar(L::S_FULL + 0));
          }
          RA_TR_ADD(tr, 3, tr_s);
          ++s_cnt0;
        }
        // slot 1: PV(u), then S(u+1)
        if (n1) {
          RA_TR_NOW(tr_p);
          if (!wait_all(bar(L::P_FULL + 1), (s_cnt1 - 1) & 1, abort_flag, a)) { ok = false; break; }
          RA_TR_ADD(tr, 0, tr_p);
          RA_TR_NOW(tr_i);
          tc_fence_after();
          issue_pv_commit<D>(tO1, tS1, v_desc(st), !first1, bar(L::O_FREE + 1));
          RA_TR_ADD(tr, 1, tr_i);
          first1 = false;
        }
        if (m1) {
          RA_TR_NOW(tr_s);
          if constexpr (ORDER == MMA_ORDER_BRIDGED) {
            issue_shift_s_commit<D>(tS1 + 64u, tS1, q_lo1, k_lo0 + st1 * kStageLo, bar(L::S_FULL + 1));
          } else {
            if (ORDER == MMA_ORDER_STRICT && s_cnt1 > 0 &&
                !wait_all(bar(L::O_FREE + 1), (s_cnt1 - 1) & 1, abort_flag, a)) { ok = false; break; }
            tc_fence_after();
            issue_s<D>(tS1, q_lo1, k_lo0 + st1 * kStageLo);
            mma_commit_e(bar(L::S_FULL + 1));
          }
          RA_TR_ADD(tr, 3, tr_s);
          ++s_cnt1;
        }
        RA_TR_NOW(tr_end);
        if constexpr (D == 64) {
          mma_commit2_e(bar(L::V_EMPTY + st), bar(L::K_EMPTY + st1), more ? 1u : 0u);
        } else {
          mma_commit_e(bar(L::V_EMPTY + st));
          if (more) mma_commit_e(bar(L::K_EMPTY + st1));
        }
        RA_TR_ADD(tr, 13, tr_end);
      }
      if (u + 2 == ns) {  // the item's last S MMAs are issued: its Q tiles may be replaced
        mma_commit_e(bar(L::Q_EMPTY + 0));
        if (it.valid1) mma_commit_e(bar(L::Q_EMPTY + 1));
      }
    }
  }
#ifdef RA_TRACE
  RA_TR_ADD(tr, 5, tr_begin);
  trace_store(tr, 8, 0);
  trace_store(tr + 8, 2, 24);
  trace_store(tr + 10, 2, 26);
  trace_store(tr + 12, 2, 14);
#endif
  // Every MMA this thread issued completes before tensor memory is freed.
  mma_commit_e(bar(L::DONE));
  wait_drain(bar(L::DONE), 0, a.timeout_ns);
}

// ------------------------------------------------------ softmax / epilogue
// Row max of one 32-column chunk of raw scores (columns j0..j0+31); on the
// diagonal tile, columns past the row are masked out.
template <bool DIAG>
__device__ __forceinline__ float chunk_max(const uint32_t (&v)[32], int j0, int r, float mx) {
  float a0 = mx, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; j += 8) {
    float x[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      x[t] = __uint_as_float(v[j + t]);
      if (DIAG && j0 + j + t > r) x[t] = -INFINITY;
    }
    a0 = max3(a0, x[0], x[1]);
    a1 = max3(a1, x[2], x[3]);
    a2 = max3(a2, x[4], x[5]);
    a3 = max3(a3, x[6], x[7]);
  }
  return fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
}

// p = exp2(x*c - m) for one 32-column chunk; packs bf16 pairs into pk and
// accumulates the exact fp32 sum (for lse).  The sum of the rounded values
// that the PV product consumes (for the output normalisation) is taken later
// from the packed pairs, off the path to the PV product.
template <bool DIAG>
__device__ __forceinline__ void chunk_exp(const uint32_t (&v)[32], int j0, int r, uint64_t c2,
                                          uint64_t negm2, uint64_t& se0, uint64_t& se1,
                                          uint32_t (&pk)[16]) {
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const uint64_t xs = f2_fma(f2_pack(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), c2, negm2);
    float p0 = ex2(f2_lo(xs)), p1 = ex2(f2_hi(xs));
    if (DIAG) {
      p0 = (j0 + j > r) ? 0.0f : p0;
      p1 = (j0 + j + 1 > r) ? 0.0f : p1;
    }
    const uint32_t pr = pack_bf16x2(p0, p1);
    if ((j & 2) == 0) se0 = f2_add(se0, f2_pack(p0, p1));
    else se1 = f2_add(se1, f2_pack(p0, p1));
    pk[j >> 1] = pr;
  }
}

struct PackedRow {  // a row's 128 bf16 weights in pairs, by 32-column chunk
  uint32_t a[16], b[16], c[16], d[16];
};

// s_lo += low bf16 of p, s_hi += high bf16 of p (fp32 sums, round to nearest)
__device__ __forceinline__ void add_bf16_halves(uint32_t p, float& s_lo, float& s_hi) {
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %0;\n\t"
      "add.rn.f32.bf16 %1, hi, %1;\n\t}"
      : "+f"(s_lo), "+f"(s_hi)
      : "r"(p));
}

// Four running sums: even pairs' low and high halves, odd pairs' low and high
// halves, each a chain of fp32 additions in pair order
struct RoundedSums {
  float e_lo, e_hi, o_lo, o_hi;
};

__device__ __forceinline__ void rounded_sum_chunk(const uint32_t (&pk)[16], RoundedSums& s) {
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    add_bf16_halves(pk[i], s.e_lo, s.e_hi);
    add_bf16_halves(pk[i + 1], s.o_lo, s.o_hi);
  }
}

// fp32 sum of the row's bf16 weights: the normaliser of the output, which
// accumulates exactly these rounded values
__device__ __forceinline__ float rounded_sum(const PackedRow& pk) {
  RoundedSums s{0.0f, 0.0f, 0.0f, 0.0f};
  rounded_sum_chunk(pk.a, s);
  rounded_sum_chunk(pk.b, s);
  rounded_sum_chunk(pk.c, s);
  rounded_sum_chunk(pk.d, s);
  return (s.e_lo + s.o_lo) + (s.e_hi + s.o_hi);
}

struct RowState {
  float m;        // reference max (scaled, log2 units)
  float l_exact;  // sum of exp2(x - m) in fp32
  float l_round;  // sum of the bf16-rounded exp2(x - m)
};

// Rescale this row's O accumulator by alpha (warp-uniform call: the TMEM
// loads and stores are warp-collective; rows with alpha == 1 rewrite O unchanged).
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t tO, float alpha) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t o[32];
    tmem_ld32(tO + c0, o);
    tmem_wait_ld_regs(o);
#pragma unroll
    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
    tmem_st32(tO + c0, o);
  }
  if (Layout<D>::kRowSum) {  // the row-sum columns scale with O
    uint32_t o[16];
    tmem_ld16_wait(tO + D, o);
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
    tmem_st16(tO + D, o);
  }
}

// exp2 of one score row against reference m, into registers: bf16 weights
// packed in pairs and their exact fp32 sum (the scores stay in tensor memory).
template <bool DIAG>
__device__ __forceinline__ float exp_row(const uint32_t (&va)[32], const uint32_t (&vb)[32],
                                         const uint32_t (&vc)[32], const uint32_t (&vd)[32], int r,
                                         float c, float m, PackedRow& pk) {
  const uint64_t c2 = f2_pack(c, c);
  const uint64_t negm2 = f2_pack(-m, -m);
  uint64_t se0 = 0, se1 = 0;
  chunk_exp<DIAG>(va, 0, r, c2, negm2, se0, se1, pk.a);
  chunk_exp<DIAG>(vb, 32, r, c2, negm2, se0, se1, pk.b);
  chunk_exp<DIAG>(vc, 64, r, c2, negm2, se0, se1, pk.c);
  chunk_exp<DIAG>(vd, 96, r, c2, negm2, se0, se1, pk.d);
  const uint64_t se = f2_add(se0, se1);
  return f2_lo(se) + f2_hi(se);
}

template <bool DIAG>
__device__ __forceinline__ float row_max(const uint32_t (&va)[32], const uint32_t (&vb)[32],
                                         const uint32_t (&vc)[32], const uint32_t (&vd)[32], int r) {
  float mx = chunk_max<DIAG>(va, 0, r, -INFINITY);
  mx = chunk_max<DIAG>(vb, 32, r, mx);
  mx = chunk_max<DIAG>(vc, 64, r, mx);
  return chunk_max<DIAG>(vd, 96, r, mx);
}

// One S tile of one slot: bf16 P to tensor memory over the consumed S
// columns, the tile's exact sum into l; the packed weights are returned so
// that the caller can take their rounded sum once P has been handed over.
//
// The row's first tile sets the reference m to its max.  A later tile skips
// the max pass: the exps run against the current m, and the tile's exact sum
// tells whether any weight grew large (a tile sum <= 2^30 bounds every weight
// by 2^30: representable in bf16, and over T key tiles l stays below 2^30 T
// and O below 2^30 T max|v|, within fp32 while that is below 2^128; the
// result is exact for any m since l and O share it).  Only when some row
// of the warp exceeds that does the warp take the exact path, on the scores
// read again from tensor memory (P is stored only once the weights are
// accepted): row max, new reference where the max passed m + threshold, O
// rescale, exps again.
// pv_bar: the O_FREE barrier and the parity of the previous PV's commit, or
// 0 when every earlier PV is known complete (its commit preceded this S's)
template <int D, bool DIAG>
__device__ __forceinline__ bool softmax_tile(uint32_t tS, uint32_t tP, uint32_t tO, int r, float c,
                                             bool first, RowState& st, PackedRow& pk,
                                             uint32_t pv_bar, uint32_t pv_parity,
                                             volatile int* abort_flag, const FwdArgs& a) {
  constexpr float kSpecLimit = 1073741824.0f;  // 2^30
  float se;
  {
    uint32_t va[32], vb[32], vc[32], vd[32];
    tmem_ld128(tS, va, vb, vc, vd);
    tmem_wait_ld128(va, vb, vc, vd);
    if (first) st.m = row_max<DIAG>(va, vb, vc, vd, r) * c;
    se = exp_row<DIAG>(va, vb, vc, vd, r, c, st.m, pk);
  }
  // never taken on the first tile: its weights are at most 1
  if (__any_sync(0xffffffffu, !(se <= kSpecLimit))) {  // also catches inf
    // rare: the scores are read again from tensor memory (still there: P is
    // stored only once the weights are accepted)
    float mx = -INFINITY;
    if constexpr (D == 64) {
      // one load of the whole row for the max pass (D = 64 takes this path
      // more often: 18.3 against 18.6 ms with outlier keys)
      uint32_t wa[32], wb[32], wc[32], wd[32];
      tmem_ld32(tS + 0, wa);
      tmem_ld32(tS + 32, wb);
      tmem_ld32(tS + 64, wc);
      tmem_ld32(tS + 96, wd);
      tmem_wait_ld_regs(wa);
      tmem_wait_ld_regs(wb);
      tmem_wait_ld_regs(wc);
      tmem_wait_ld_regs(wd);
      mx = row_max<DIAG>(wa, wb, wc, wd, r);
    } else {
      uint32_t w[32];
      tmem_ld32(tS + 0, w); tmem_wait_ld_regs(w); mx = chunk_max<DIAG>(w, 0, r, mx);
      tmem_ld32(tS + 32, w); tmem_wait_ld_regs(w); mx = chunk_max<DIAG>(w, 32, r, mx);
      tmem_ld32(tS + 64, w); tmem_wait_ld_regs(w); mx = chunk_max<DIAG>(w, 64, r, mx);
      tmem_ld32(tS + 96, w); tmem_wait_ld_regs(w); mx = chunk_max<DIAG>(w, 96, r, mx);
    }
    mx *= c;
    // O is rescaled only when the max grows past the threshold (exact either
    // way: l and O always share the same m)
    float alpha = 1.0f;
    if (mx > st.m + SoftmaxPolicy<D>::kRescaleThreshold) {
      alpha = ex2(st.m - mx);
      st.m = mx;
      st.l_exact *= alpha;
      st.l_round *= alpha;
    }
    if (__any_sync(0xffffffffu, alpha != 1.0f)) {
      // O holds the previous PV's result once its commit has arrived
      if (pv_bar != 0u && !wait_all(pv_bar, pv_parity, abort_flag, a)) return false;
      tc_fence_after();
      rescale_o<D>(tO, alpha);
    }
    const uint64_t c2 = f2_pack(c, c);
    const uint64_t negm2 = f2_pack(-st.m, -st.m);
    uint64_t se0 = 0, se1 = 0;
    {
      uint32_t w[32];
      tmem_ld32(tS + 0, w); tmem_wait_ld_regs(w); chunk_exp<DIAG>(w, 0, r, c2, negm2, se0, se1, pk.a);
      tmem_ld32(tS + 32, w); tmem_wait_ld_regs(w); chunk_exp<DIAG>(w, 32, r, c2, negm2, se0, se1, pk.b);
      tmem_ld32(tS + 64, w); tmem_wait_ld_regs(w); chunk_exp<DIAG>(w, 64, r, c2, negm2, se0, se1, pk.c);
      tmem_ld32(tS + 96, w); tmem_wait_ld_regs(w); chunk_exp<DIAG>(w, 96, r, c2, negm2, se0, se1, pk.d);
    }
    const uint64_t sum = f2_add(se0, se1);
    se = f2_lo(sum) + f2_hi(sum);
  }
  tmem_st64(tP, pk.a, pk.b, pk.c, pk.d);
  st.l_exact += se;
  tmem_wait_st();
  return true;
}

template <int D, bool SINGLE>
__device__ void softmax_role(const FwdArgs& a, uint32_t sbase, uint32_t tmem,
                             volatile int* abort_flag) {
  using L = Layout<D>;
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = warp >> 2;
  const int r = threadIdx.x & 127;  // row inside the 128-row query tile == TMEM lane
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  const uint32_t tS_pair = tmem + lane_base + L::S_COL(slot);
  const uint32_t tO = tmem + lane_base + L::O_COL(slot);
  const float c = a.scale_log2;
  // buffer sizes in elements, for the bounds checks of RA_DEBUG builds
  const size_t out_n = (size_t)a.B * a.S * a.H * D, lse_n = (size_t)a.B * a.H * a.S;
  uint32_t n = 0;  // S tiles consumed so far by this slot
  RA_TR_DECL(tr, 6);

  for (int k = 0;; ++k) {
    const int x = next_item<D>(a, sbase, k, abort_flag);
    if (x < 0) break;
    const Item it = decode_item(a, x);
    if (slot == 1 && !it.valid1) continue;
    // this slot's query tile and head, selected once: indexing the item with
    // the run-time slot would place it in local memory
    const int my_qt = slot ? it.qt[1] : it.qt[0];
    const int my_h = slot ? it.h[1] : it.h[0];
    const int ns = n_steps(a, it);
    if (ns == 0 || !needs_tile(a, my_qt, 0)) {
      // block mode only: no key of the block is allowed for these rows
      const int srow = my_qt * kBM + r;
      const size_t e0 = (((size_t)it.b * a.S + srow) * a.H + my_h) * D;
      uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + e0);
      if (in_bounds(e0, D, out_n, a.bounds_trim, a.status)) {
#pragma unroll 1
        for (int j = 0; j < D / 8; ++j) orow[j] = make_uint4(0, 0, 0, 0);
      }
      const size_t li = ((size_t)it.b * a.H + my_h) * a.S + srow;
      if (a.lse && in_bounds(li, 1, lse_n, a.bounds_trim, a.status)) a.lse[li] = -INFINITY;
      continue;
    }
    // the slot's last step: the item's last one, or the one before it when
    // the slot does not need the last key tile (the second tile of a causal
    // pair in a one-chunk item)
    const int u_last = (ns > 1 && !needs_tile(a, my_qt, last_tile(a, it))) ? ns - 2 : ns - 1;
    StepCursor cur;
    cur.init(a, it);

    RowState st{-INFINITY, 0.0f, 0.0f};
    bool first = true;
    for (int u = 0; u < ns; ++u, cur.next()) {
      const int kt = cur.kt;
      if (!needs_tile(a, my_qt, kt)) continue;
      RA_TR_NOW(tr_0);
      // S_FULL: per slot; one query tile per item, per S buffer (n % 2)
      const int s_bar = SINGLE ? (int)(n & 1u) : slot;
      const uint32_t s_par = SINGLE ? (n >> 1) & 1u : n & 1u;
      if (!wait_all(bar(L::S_FULL + s_bar), s_par, abort_flag, a)) return;
      RA_TR_ADD(tr, 0, tr_0);
      RA_TR_NOW(tr_1);
      tc_fence_after();
      PackedRow pk;
      // one query tile per item: the n-th S and P in buffers n % 2; the
      // previous PV may still be running (see mma_role_single)
      const uint32_t tS = SINGLE ? tmem + lane_base + L::S1T_S_COL(n & 1u) : tS_pair;
      const uint32_t tP = SINGLE ? tmem + lane_base + L::S1T_P_COL(n & 1u) : tS_pair;
      const uint32_t pv_bar = (SINGLE && n > 0) ? bar(L::O_FREE + 0) : 0u;
      bool tile_ok;
      if (is_diag(a, my_qt, kt))
        tile_ok = softmax_tile<D, true>(tS, tP, tO, r, c, first, st, pk, pv_bar, (n - 1) & 1,
                                        abort_flag, a);
      else
        tile_ok = softmax_tile<D, false>(tS, tP, tO, r, c, first, st, pk, pv_bar, (n - 1) & 1,
                                         abort_flag, a);
      if (!tile_ok) return;
      // One query tile per item: the previous PV may still be running (its S
      // successor was issued two steps ahead).  Waiting for it here, before
      // this tile's P is handed over, keeps every O_FREE wait of the slot
      // within one phase of the barrier (the next PV cannot start before this
      // arrive), which is what a parity wait needs; the PV is usually long done.
      if (SINGLE && n > 0 && !wait_all(bar(L::O_FREE + 0), (n - 1) & 1, abort_flag, a)) return;
      tc_fence_before();
      __syncwarp();
      mbar_arrive_e(bar(L::P_FULL + (SINGLE ? (int)(n & 1u) : slot)));
      RA_TR_ADD(tr, 1, tr_1);
      RA_TR_NOW(tr_2);
      // the sum of the rounded weights is needed only by the epilogue: taken
      // here, while the tensor cores run this slot's PV and next S products
      // (with the row-sum columns the PV product sums them itself)
      if (!SoftmaxPolicy<D>::kMmaRowSum) st.l_round += rounded_sum(pk);
      ++n;
      first = false;
      RA_TR_ADD(tr, 2, tr_2);
      RA_TR_INC(tr, 3);

      if (u == u_last) {
        RA_TR_NOW(tr_e);
        // epilogue: wait for the last O_i += P_i V, then out = O / l, lse
        if (!wait_all(bar(L::O_FREE + slot), (n - 1) & 1, abort_flag, a)) return;
        tc_fence_after();
        const int srow = my_qt * kBM + r;
        const int h = my_h;
        float l_norm = st.l_round;
        if (Layout<D>::kRowSum) {  // the PV MMA's row sum of the rounded weights
          uint32_t ls[16];
          tmem_ld16_wait(tO + D, ls);
          l_norm = __uint_as_float(ls[0]);
        }
        const float inv_l = 1.0f / l_norm;
        if constexpr (Layout<D>::kLineStores) {
          // Each 64-column half of the warp's 32 rows goes through the warp's
          // block: lane i writes its row's 128 bytes (16-byte chunk c at
          // c ^ (i % 8), so a store touches every bank once per 8 lanes), then
          // each lane reads chunk (lane % 8) of row 4 j + lane / 8 and stores
          // it: 8 lanes cover one row's 128 contiguous bytes, a warp store 4
          // whole lines.
          const uint32_t blk = sbase + L::EPI_OFF + (uint32_t)warp * (uint32_t)L::EPI_BLOCK;
          const int row0 = my_qt * kBM + (r & ~31);  // the warp's first row
          __nv_bfloat16* obase = static_cast<__nv_bfloat16*>(a.out);
          if constexpr (D == 64) {
            // one 128-byte row per lane; 16 lanes' rows at a time
            uint32_t o[32], w[2][16];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              tmem_ld32(tO + part * 32, o);
              tmem_wait_ld_regs(o);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                w[part][j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv_l,
                                         __uint_as_float(o[2 * j + 1]) * inv_l);
            }
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              __syncwarp();  // the previous round has been read out of the block
              if ((lane >> 4) == half) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                  const uint32_t* src = &w[c >> 2][(c & 3) * 4];
                  st_shared_v4(blk + (lane & 15) * 128 + ((c ^ (lane & 7)) << 4), src[0], src[1],
                               src[2], src[3]);
                }
              }
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int row = 4 * j + (lane >> 3), c = lane & 7;
                const uint4 v = ld_shared_v4(blk + row * 128 + ((c ^ (row & 7)) << 4));
                const size_t e = (((size_t)it.b * a.S + row0 + 16 * half + row) * a.H + h) * D + c * 8;
                if (in_bounds(e, 8, out_n, a.bounds_trim, a.status))
                  *reinterpret_cast<uint4*>(obase + e) = v;
              }
            }
          }
#pragma unroll 1
          for (int hh = 0; hh < (D == 128 ? 2 : 0); ++hh) {
            uint32_t o[32], w[2][16];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              tmem_ld32(tO + hh * 64 + part * 32, o);
              tmem_wait_ld_regs(o);
              if constexpr (SINGLE) {
                // packed multiplies (the same roundings): S = 4096 workload
                // 0.0416-0.0422 against 0.0427-0.0437 ms; the paired kernel
                // measured slower with them (GQA 2.645 against 2.626 ms)
                const uint64_t inv2 = f2_pack(inv_l, inv_l);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  const uint64_t v =
                      f2_mul(f2_pack(__uint_as_float(o[2 * j]), __uint_as_float(o[2 * j + 1])), inv2);
                  w[part][j] = pack_bf16x2(f2_lo(v), f2_hi(v));
                }
              } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  w[part][j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv_l,
                                           __uint_as_float(o[2 * j + 1]) * inv_l);
              }
            }
            __syncwarp();  // the previous half has been read out of the block
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t* src = &w[c >> 2][(c & 3) * 4];
              st_shared_v4(blk + lane * 128 + ((c ^ (lane & 7)) << 4), src[0], src[1], src[2], src[3]);
            }
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int row = 4 * j + (lane >> 3), c = lane & 7;
              const uint4 v = ld_shared_v4(blk + row * 128 + ((c ^ (row & 7)) << 4));
              const size_t e = (((size_t)it.b * a.S + row0 + row) * a.H + h) * D + hh * 64 + c * 8;
              if (in_bounds(e, 8, out_n, a.bounds_trim, a.status))
                *reinterpret_cast<uint4*>(obase + e) = v;
            }
          }
        } else {
          const size_t e0 = (((size_t)it.b * a.S + srow) * a.H + h) * D;
          uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + e0);
          const bool row_ok = in_bounds(e0, D, out_n, a.bounds_trim, a.status);
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tO + c0, o);
            tmem_wait_ld_regs(o);
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              w[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv_l, __uint_as_float(o[2 * j + 1]) * inv_l);
#pragma unroll
            for (int j = 0; j < 4 && row_ok; ++j)
              orow[c0 / 8 + j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
          }
        }
        const size_t li = ((size_t)it.b * a.H + h) * a.S + srow;
        if (a.lse && in_bounds(li, 1, lse_n, a.bounds_trim, a.status))
          a.lse[li] = (st.m + log2f(st.l_exact)) * 0.69314718055994531f;
        tc_fence_before();
#ifdef RA_TRACE
        RA_TR_ADD(tr, 4, tr_e);
        RA_TR_INC(tr, 5);
        if ((warp & 3) == 0) trace_store(tr, 6, slot ? 16 : 8);
#endif
      }
    }
  }
}

template <int D, bool SINGLE>
__global__ void __launch_bounds__(kThreads, 1)
    ring_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::N_BARS; ++i) {
      const bool per_warp = (i == L::P_FULL || i == L::P_FULL + 1);
      const bool item_free = (i >= L::ITEM_EMPTY && i < L::ITEM_EMPTY + kItemRing);
      mbar_init(sbase + L::BAR_OFF + 8u * i, item_free ? kItemConsumers : (per_warp ? 4u : 1u));
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == kWarpTma && (threadIdx.x & 31) == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (L::kRowSum) {  // the B operand block of the row-sum columns: bf16 ones
    uint4* ones = reinterpret_cast<uint4*>(smem + L::ONES_OFF);
    for (int i = threadIdx.x; i < L::BLOCK / 16; i += kThreads)
      ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();  // visible to the tensor cores
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp < 8) {
    regs_inc<(D == 64 && SINGLE) ? kSoftmaxRegs64Single : kSoftmaxRegs>();
    softmax_role<D, SINGLE>(a, sbase, tmem, abort_flag);
  } else {
    regs_dec<(D == 64 && SINGLE) ? kProducerRegs64Single : kProducerRegs>();
    if (warp == kWarpTma) {
      if ((threadIdx.x & 31) == 0) tma_role<D>(&tm_q, &tm_k, &tm_v, a, sbase, abort_flag);
    } else if (warp == kWarpMma) {
      {
        if constexpr (SINGLE)
          mma_role_single<D>(a, sbase, tmem, abort_flag);
        else if (a.mma_order == MMA_ORDER_GROUPED)
          mma_role<D, MMA_ORDER_GROUPED>(a, sbase, tmem, abort_flag);
        else if (a.mma_order == MMA_ORDER_INORDER)
          mma_role<D, MMA_ORDER_INORDER>(a, sbase, tmem, abort_flag);
        else if (a.mma_order == MMA_ORDER_BRIDGED)
          mma_role<D, MMA_ORDER_BRIDGED>(a, sbase, tmem, abort_flag);
        else
          mma_role<D, MMA_ORDER_STRICT>(a, sbase, tmem, abort_flag);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
  // every claim of this CTA has returned (the producer used its last value
  // before the barrier above); the last CTA to get here resets the counter
  // for the next launch that uses this slot
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.item_ctr + 1, 1u) == gridDim.x - 1) {
      volatile unsigned int* ctr = a.item_ctr;
      ctr[0] = 0;
      ctr[1] = 0;
    }
  }
}

size_t fwd_smem_bytes(int D) {
  return D == 128 ? (size_t)Layout<128>::ALLOC : (size_t)Layout<64>::ALLOC;
}

template <int D, bool SINGLE>
static cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& args, int grid, cudaStream_t stream) {
  const int smem = Layout<D>::ALLOC;
  static std::atomic<unsigned> prepared[kMaxPrepDevices];
  const cudaError_t e = prepare_kernel(ring_attn_fwd_kernel<D, SINGLE>, (int)kLaunchRegs, smem, prepared);
  if (e != cudaSuccess) return e;
#ifdef RA_TRACE
  {  // traced builds: the counters describe this launch alone
    void* tr = nullptr;
    cudaError_t te = cudaGetSymbolAddress(&tr, g_trace);
    if (te == cudaSuccess) te = cudaMemsetAsync(tr, 0, sizeof(g_trace), stream);
    if (te != cudaSuccess) return te;
  }
#endif
  ring_attn_fwd_kernel<D, SINGLE><<<grid, kThreads, smem, stream>>>(tq, tk, tv, args);
  return cudaGetLastError();
}

cudaError_t launch_fwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& args, int grid, cudaStream_t stream) {
  const bool single = (args.mode == MODE_SINGLE);
  if (D == 128)
    return single ? launch_d<128, true>(tq, tk, tv, args, grid, stream)
                  : launch_d<128, false>(tq, tk, tv, args, grid, stream);
  return single ? launch_d<64, true>(tq, tk, tv, args, grid, stream)
                : launch_d<64, false>(tq, tk, tv, args, grid, stream);
}

cudaError_t item_counter_ptr(unsigned int** p) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(p), g_item_ctr);
}

cudaError_t trace_copy(unsigned long long* host, int n_ctas) {
#ifdef RA_TRACE
  if (n_ctas > kTraceCtas) n_ctas = kTraceCtas;
  return cudaMemcpyFromSymbol(host, g_trace, sizeof(unsigned long long) * kTraceSlots * n_ctas);
#else
  (void)host;
  (void)n_ctas;
  return cudaErrorNotSupported;
#endif
}

cudaError_t status_word_ptr(unsigned int** p) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(p), g_status_word);
}

cudaError_t read_and_clear_status(unsigned int* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_status_word, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_status_word, &zero, sizeof(unsigned int));
}

}  // namespace ra
