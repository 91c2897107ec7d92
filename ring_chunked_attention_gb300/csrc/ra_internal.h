// ra_internal.h -- declarations shared by the translation units of
// libringattn (host side only; not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace ra {

// How the two 128-row query tiles a CTA works on at a time are chosen.
enum PairMode : int {
  MODE_SINGLE = 0,  // one query tile; the second slot stays idle
  MODE_HEADS = 1,   // two query heads of the same KV head, same rows
  MODE_QTILES = 2,  // two consecutive 128-row tiles of one head, same chunk
};

// Issue order of the forward's MMA thread (see ra_fwd.cu, "MMA issuer").
enum MmaOrder : int {
  MMA_ORDER_STRICT = 0,   // per slot: PV, wait for its commit, next S
  MMA_ORDER_GROUPED = 1,  // both slots' PV, then each next S after its PV's commit
  MMA_ORDER_INORDER = 2,  // per slot: PV and next S back to back (relies on in-order execution)
  MMA_ORDER_BRIDGED = 3,  // per slot: PV, a tcgen05.shift of dead S columns, next S (default)
};

// Kernel arguments besides the three tensor maps (q, k, v).
struct FwdArgs {
  void* out;             // bf16 [B,S,H,D]
  float* lse;            // fp32 [B,H,S] or nullptr
  unsigned int* status;  // this device's sticky status word
  int B, H, Hkv, S, P;   // S: query rows per batch entry
  int Sk;                // key rows per batch entry (== S for the ring-chunked forward)
  int causal;
  int mode;              // PairMode
  int tiles;             // S / 128 (query tiles)
  int tiles_k;           // Sk / 128 (key tiles)
  int tpc;               // 128-row tiles per chunk (S / P / 128)
  int block;             // 0: ring-chunked forward over P chunks; 1: one query block
                         //    against one key/value block at the offsets below
  int q_tile0, k_tile0;  // block mode: global 128-row tile index of query / key row 0
  int groups;            // work items per query-tile index
  int nq;                // query-tile indices
  int n_items;           // groups * nq
  float scale_log2;      // scale * log2(e)
  unsigned long long timeout_ns;
  int skip_value_load;   // failure-path test hook
  int mma_order;         // MmaOrder: how S_i(u+1) is ordered after O_i += P_i(u) V
  unsigned int* item_ctr;  // this launch's work-item counter pair (next item, CTAs done), zero at launch
  long long bounds_trim;   // bounds-checked builds: elements at the end of every buffer that count
                           // as outside it (test hook; 0 normally)
};

// Kernel arguments of the backward pass besides the tensor maps (q, k, v, dout).
struct BwdArgs {
  const void* out;       // bf16 [B,S,H,D] forward output (row-sum kernel only)
  const void* dout;      // bf16 [B,S,H,D] gradient of the output
  const float* lse;      // fp32 [B,H,S] from the forward (natural log)
  float* nlse2;          // workspace fp32 [B,H,S]: -lse * log2(e)
  float* ndelta;         // workspace fp32 [B,H,S]: -sum_d out * dout
  void* dq;              // bf16 [B,S,H,D]
  void* dk;              // bf16 [B,S,Hkv,D]
  void* dv;              // bf16 [B,S,Hkv,D]
  unsigned int* status;  // this device's sticky status word
  int B, H, Hkv, S, P;
  int causal;
  int tiles;             // S / 128
  int tpc;               // 128-row tiles per ring chunk (S / P / 128)
  int n_items;           // work items of the kernel being launched
  float scale;           // multiplies dq and dk
  float scale_log2;      // scale * log2(e)
  unsigned long long timeout_ns;
  int skip_first_load;   // failure-path test hook: the dk/dv producer never issues
                         // its first dout-tile copy
  long long bounds_trim; // as FwdArgs::bounds_trim
};

// status word bits
constexpr unsigned int kStatusTimeout = 1u;
constexpr unsigned int kStatusLayout = 2u;  // a kernel found its shared memory base misaligned
constexpr unsigned int kStatusBounds = 4u;  // bounds-checked builds: an address outside its buffer

// Builds compiled with RA_DEBUG check every global address a kernel computes
// (the tensor-map copies are bounded by the hardware) against its buffer:
// when the element range [first, first + count) does not lie inside
// [0, extent - trim), the check sets kStatusBounds in the status word and the
// caller skips the access (a bulk copy reads element 0 instead, so that its
// barrier still completes).  trim is a test hook that makes the last elements
// of every buffer count as outside it.  Other builds compile the check away.
__device__ __forceinline__ bool in_bounds(size_t first, size_t count, size_t extent, long long trim,
                                          unsigned int* status) {
#ifdef RA_DEBUG
  if (extent >= (size_t)trim && first + count <= extent - (size_t)trim) return true;
  if (status) atomicOr(status, kStatusBounds);
  return false;
#else
  (void)first;
  (void)count;
  (void)extent;
  (void)trim;
  (void)status;
  return true;
#endif
}

// Per-role cycle counters of builds compiled with RA_TRACE (ra_trace_read):
// each CTA of the forward kernel keeps kTraceSlots clock64 sums in registers
// and stores them when its roles finish.  Other builds compile the counting
// away.  Slots: MMA warp 0 P waits, 1 PV issue, 2 V waits, 3 S issue,
// 4 steps, 5 role total, 6 late K waits, 7 item starts (Q waits and the first
// S); softmax slot 0 warp 0 at 8.., slot 1 (warp 4) at 16..: +0 S waits,
// +1 S to P hand-off, +2 after the hand-off, +3 tiles, +4 epilogues, +5 items;
// 24 V waits at an item's first step, 25 items, 26 Q waits and 27 waits for
// the previous item's last PV inside the item starts, 14 each step's top (up
// to its V wait) and 15 its closing commits (MMA warp, paired items);
// producer 28 K-stage waits, 29 V-stage waits, 30 Q-slot waits.
constexpr int kTraceSlots = 32;
constexpr int kTraceCtas = 1024;
#ifdef RA_TRACE
#define RA_TR_DECL(name, n) unsigned long long name[n] = {}
#define RA_TR_NOW(v) const long long v = clock64()
#define RA_TR_ADD(arr, i, v) ((arr)[i] += (unsigned long long)(clock64() - (v)))
#define RA_TR_INC(arr, i) ((arr)[i] += 1ull)
#else
#define RA_TR_DECL(name, n)
#define RA_TR_NOW(v)
#define RA_TR_ADD(arr, i, v)
#define RA_TR_INC(arr, i)
#endif
cudaError_t trace_copy(unsigned long long* host, int n_ctas);

// ra_fwd.cu
cudaError_t launch_fwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& args, int grid, cudaStream_t stream);
size_t fwd_smem_bytes(int D);
cudaError_t status_word_ptr(unsigned int** p);

// Host side: a tensor-core kernel's register count is checked (its setmaxnreg
// split is sized for exactly `regs` registers per thread at launch; any other
// allocation would make setmaxnreg.inc wait forever) and its dynamic
// shared-memory limit raised once per device and kernel.  Both persist on the
// function, so later launches, including launches recorded into a CUDA graph,
// make no attribute calls.  `prepared[dev]` holds the preparation epoch + 1;
// ra_shutdown starts a new epoch (after a device reset, call ra_shutdown).
constexpr int kMaxPrepDevices = 64;
extern std::atomic<unsigned> g_prep_epoch;

template <class Kernel>
inline cudaError_t prepare_kernel(Kernel kernel, int regs, int smem,
                                  std::atomic<unsigned>* prepared) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cache = dev >= 0 && dev < kMaxPrepDevices;
  const unsigned mark = g_prep_epoch.load(std::memory_order_acquire) + 1u;
  if (cache && prepared[dev].load(std::memory_order_acquire) == mark) return cudaSuccess;
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kernel);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != regs) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (cache) prepared[dev].store(mark, std::memory_order_release);
  return cudaSuccess;
}
// Work-item counter slots of the forward (2 words each).  Eager launches take
// the first kEagerCounterSlots in turn, so up to that many may run at once.  A
// launch recorded into a CUDA graph keeps its slot for every replay, so it
// takes one of the remaining slots, which is never handed out again in this
// process: no eager launch and no other captured launch can share it.
constexpr int kEagerCounterSlots = 64;
constexpr int kCapturedCounterSlots = 4032;
constexpr int kItemCounterSlots = kEagerCounterSlots + kCapturedCounterSlots;
cudaError_t item_counter_ptr(unsigned int** p);
cudaError_t read_and_clear_status(unsigned int* value);

// ra_bwd.cu
constexpr long long kStaticBwdRows = 1ll << 21;  // query rows B*H*S of the static scratch
cudaError_t bwd_static_scratch(float** p);       // its device address (cudaGetSymbolAddress)
cudaError_t launch_bwd_prep(int D, const BwdArgs& args, int grid, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const BwdArgs& args,
                            int grid, cudaStream_t stream);
cudaError_t launch_bwd_dq(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const BwdArgs& args,
                          int grid, cudaStream_t stream);

// ra_ceil.cu: ex2 and fp32 FMA rates of this device (see ra_measure_ceilings)
cudaError_t measure_ceilings(int sms, double* out);

// ra_merge.cu
// (status, trim: the bounds checks of RA_DEBUG builds)
cudaError_t launch_merge(const void* o_parts, int o_is_fp32, const float* lse_parts, int n,
                         void* out, float* lse, int B, int H, int S, int D, int sms,
                         unsigned int* status, long long trim, cudaStream_t stream);

}  // namespace ra
