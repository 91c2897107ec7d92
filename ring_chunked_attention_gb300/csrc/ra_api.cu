// ra_api.cu -- the C ABI of libringattn: argument validation, tensor-map
// encoding (cached), work decomposition and launch, status reporting.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "ra_internal.h"
#include "ringattn.h"

namespace {

thread_local int g_last_cuda_error = 0;

ra_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return RA_ERR_CUDA;
}

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s
std::mutex g_mu;

}  // namespace

namespace ra {
std::atomic<unsigned> g_prep_epoch{0};
}  // namespace ra

namespace {
unsigned long long g_timeout_ns = kDefaultTimeoutNs;
int g_skip_value_load = 0;
int g_mma_order = ra::MMA_ORDER_BRIDGED;  // ra::MmaOrder
int g_item_pairing = 0;  // 0 automatic, 1 always pair when the shape allows, 2 never pair
long long g_bounds_trim = 0;  // bounds-checked builds: test hook (ra_debug_set_bounds_trim)

// per-device facts, queried once
struct DeviceInfo {
  bool valid = false;
  bool sm103 = false;
  int sms = 0;
  unsigned int* status = nullptr;
  float* bwd_scratch = nullptr;  // the static scratch of ra_bwd_static on this device
  unsigned int* item_ctr = nullptr;  // the forward's work-item counter slots on this device
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];

// Which counter slot the next forward launch on a device takes.  Kept apart
// from DeviceInfo so that ra_shutdown does not restart the cycle: a launch
// still in flight after ra_shutdown keeps its slot to itself, and captured
// slots are never reused in this process.
struct SlotCursor {
  unsigned int eager = 0;     // eager launches so far (cycles through kEagerCounterSlots)
  unsigned int captured = 0;  // captured launches so far (each keeps its slot)
};
SlotCursor g_slots[kMaxDevices];

ra_status device_info(DeviceInfo** out, int* ordinal = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
  if (ordinal) *ordinal = dev;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.valid) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    unsigned int* st = nullptr;
    if ((e = ra::status_word_ptr(&st)) != cudaSuccess) return cuda_fail(e);
    float* scratch = nullptr;
    if ((e = ra::bwd_static_scratch(&scratch)) != cudaSuccess) return cuda_fail(e);
    unsigned int* ctr = nullptr;
    if ((e = ra::item_counter_ptr(&ctr)) != cudaSuccess) return cuda_fail(e);
    d.sm103 = (major == 10 && minor == 3);
    d.sms = sms;
    d.status = st;
    d.bwd_scratch = scratch;
    d.item_ctr = ctr;
    d.valid = true;
  }
  *out = &d;
  return RA_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

ra_status get_encoder(EncodeTiledFn* fn) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return cuda_fail(e);
    if (q != cudaDriverEntryPointSuccess || !p) return cuda_fail(cudaErrorSymbolNotFound);
    g_encode = reinterpret_cast<EncodeTiledFn>(p);
  }
  *fn = g_encode;
  return RA_OK;
}

// A [rows = B*S, heads, D] bf16 tensor read as 128-row x 64-column boxes,
// 128-byte swizzled (the layout the tensor-core descriptors expect).
struct MapKey {
  const void* ptr;
  long long rows;
  int heads, D;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && heads == o.heads && D == o.D;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  unsigned long long stamp;
  bool used;
};
constexpr int kMapCache = 32;
MapEntry g_maps[kMapCache];
unsigned long long g_stamp = 0;

ra_status tensor_map(const void* ptr, long long rows, int heads, int D, CUtensorMap* out) {
  const MapKey key{ptr, rows, heads, D};
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto& e : g_maps)
      if (e.used && e.key == key) {
        e.stamp = ++g_stamp;
        *out = e.map;
        return RA_OK;
      }
  }
  EncodeTiledFn enc = nullptr;
  ra_status st = get_encoder(&enc);
  if (st != RA_OK) return st;
  CUtensorMap m;
  std::memset(&m, 0, sizeof m);
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
  const cuuint32_t box[3] = {64, 1, 128};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  std::lock_guard<std::mutex> lock(g_mu);
  int victim = 0;
  for (int i = 0; i < kMapCache; ++i) {
    if (!g_maps[i].used) { victim = i; break; }
    if (g_maps[i].stamp < g_maps[victim].stamp) victim = i;
  }
  g_maps[victim] = MapEntry{key, m, ++g_stamp, true};
  *out = m;
  return RA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace {

// Shared tail of ra_fwd and ra_fwd_block: device check, tensor maps, work
// decomposition, launch.  Arguments are already validated.
ra_status launch_attention(const void* q, const void* k, const void* v, void* out, float* lse,
                           int B, int H, int Hkv, int Sq, int Sk, int D, int P, int causal,
                           float scale, int block, int q_tile0, int k_tile0, void* stream) {
  DeviceInfo* dev = nullptr;
  int ordinal = 0;
  ra_status st = device_info(&dev, &ordinal);
  if (st != RA_OK) return st;
  if (!dev->sm103) return RA_ERR_UNSUPPORTED;
  // a launch being recorded into a CUDA graph gets a counter slot of its own
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  cudaError_t ce = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &capture);
  if (ce != cudaSuccess) return cuda_fail(ce);
  const bool captured = capture != cudaStreamCaptureStatusNone;

  CUtensorMap tq, tk, tv;
  if ((st = tensor_map(q, (long long)B * Sq, H, D, &tq)) != RA_OK) return st;
  if ((st = tensor_map(k, (long long)B * Sk, Hkv, D, &tk)) != RA_OK) return st;
  if ((st = tensor_map(v, (long long)B * Sk, Hkv, D, &tv)) != RA_OK) return st;

  ra::FwdArgs a;
  std::memset(&a, 0, sizeof a);
  a.out = out;
  a.lse = lse;
  a.status = dev->status;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.S = Sq;
  a.Sk = Sk;
  a.P = P;
  a.causal = causal ? 1 : 0;
  a.tiles = Sq / 128;
  a.tiles_k = Sk / 128;
  a.tpc = block ? a.tiles_k : Sq / P / 128;
  a.block = block;
  a.q_tile0 = q_tile0;
  a.k_tile0 = k_tile0;
  const int G = H / Hkv;
  // two consecutive query tiles pair up only inside one ring chunk
  const bool pair_tiles = block ? (a.tiles % 2 == 0) : (a.tpc % 2 == 0);
  if (G % 2 == 0) {
    a.mode = ra::MODE_HEADS;
    a.groups = B * Hkv * (G / 2);
    a.nq = a.tiles;
  } else if (pair_tiles) {
    a.mode = ra::MODE_QTILES;
    a.groups = B * H;
    a.nq = a.tiles / 2;
  } else {
    a.mode = ra::MODE_SINGLE;
    a.groups = B * H;
    a.nq = a.tiles;
  }
  a.n_items = a.groups * a.nq;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  int pairing;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    a.timeout_ns = g_timeout_ns;
    a.skip_value_load = g_skip_value_load;
    a.mma_order = g_mma_order;
    a.bounds_trim = g_bounds_trim;
    pairing = g_item_pairing;
    // each eager launch takes the next of the eager slots (the kernel leaves
    // it at zero); a captured launch takes a captured slot that no other
    // launch will ever get
    SlotCursor& cur = g_slots[ordinal];
    int slot;
    if (captured) {
      if (cur.captured >= (unsigned)ra::kCapturedCounterSlots) return RA_ERR_UNSUPPORTED;
      slot = ra::kEagerCounterSlots + (int)cur.captured++;
    } else {
      slot = (int)(cur.eager++ % (unsigned)ra::kEagerCounterSlots);
    }
    a.item_ctr = dev->item_ctr + 2 * slot;
  }
  // With fewer paired items than SMs the heaviest pair is the critical path:
  // one query tile per item halves it and fills the SMs better.
  if (a.mode != ra::MODE_SINGLE && (pairing == 2 || (pairing == 0 && a.n_items < dev->sms))) {
    a.mode = ra::MODE_SINGLE;
    a.groups = B * H;
    a.nq = a.tiles;
    a.n_items = a.groups * a.nq;
  }
  const int grid = a.n_items < dev->sms ? a.n_items : dev->sms;
  cudaError_t e = ra::launch_fwd(D, tq, tk, tv, a, grid, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return RA_OK;
}

}  // namespace

extern "C" {

ra_status ra_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
                 int Hkv, int S, int D, int P, int causal, float scale, void* stream) {
  if (!q || !k || !v || !out) return RA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Hkv <= 0 || S <= 0 || D <= 0 || P <= 0) return RA_ERR_INVALID_ARG;
  if (H % Hkv != 0 || S % P != 0) return RA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return RA_ERR_INVALID_ARG;
  if (scale < 0.0f) return RA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return RA_ERR_UNSUPPORTED;
  if ((S / P) % 128 != 0) return RA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return RA_ERR_UNSUPPORTED;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return RA_ERR_UNSUPPORTED;
  // work-item ids, and the run-time claims past them, stay far inside int
  if ((long long)B * S >= (1ll << 31) || (long long)B * H * (S / 128) >= (1ll << 30))
    return RA_ERR_UNSUPPORTED;
  return launch_attention(q, k, v, out, lse, B, H, Hkv, S, S, D, P, causal, scale, 0, 0, 0,
                          stream);
}

ra_status ra_fwd_block(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                       int H, int Hkv, int Sq, int Sk, int D, long long q_pos0, long long k_pos0,
                       int causal, float scale, void* stream) {
  if (!q || !k || !v || !out) return RA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || D <= 0) return RA_ERR_INVALID_ARG;
  if (H % Hkv != 0 || q_pos0 < 0 || k_pos0 < 0) return RA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return RA_ERR_INVALID_ARG;
  if (scale < 0.0f) return RA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return RA_ERR_UNSUPPORTED;
  if (Sq % 128 != 0 || Sk % 128 != 0 || q_pos0 % 128 != 0 || k_pos0 % 128 != 0)
    return RA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return RA_ERR_UNSUPPORTED;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return RA_ERR_UNSUPPORTED;
  if ((long long)B * Sq >= (1ll << 31) || (long long)B * Sk >= (1ll << 31) ||
      (long long)B * H * (Sq / 128) >= (1ll << 30) || q_pos0 / 128 + Sq / 128 >= (1ll << 30) ||
      k_pos0 / 128 + Sk / 128 >= (1ll << 30))
    return RA_ERR_UNSUPPORTED;
  return launch_attention(q, k, v, out, lse, B, H, Hkv, Sq, Sk, D, 1, causal, scale, 1,
                          (int)(q_pos0 / 128), (int)(k_pos0 / 128), stream);
}

ra_status ra_merge_partials(const void* o_parts, int o_is_fp32, const float* lse_parts, int n,
                            void* out, float* lse, int B, int H, int S, int D, void* stream) {
  if (!o_parts || !lse_parts || !out) return RA_ERR_INVALID_ARG;
  if (n < 1 || B <= 0 || H <= 0 || S <= 0 || D <= 0) return RA_ERR_INVALID_ARG;
  if (D % 8 != 0) return RA_ERR_UNSUPPORTED;
  if (!aligned16(o_parts) || !aligned16(out)) return RA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(lse_parts) & 3u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return RA_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  ra_status st = device_info(&dev);
  if (st != RA_OK) return st;
  if (!dev->sm103) return RA_ERR_UNSUPPORTED;
  const long long rows = (long long)B * S * H;
  if (rows >= (1ll << 31)) return RA_ERR_UNSUPPORTED;
  long long trim;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    trim = g_bounds_trim;
  }
  cudaError_t e = ra::launch_merge(o_parts, o_is_fp32, lse_parts, n, out, lse, B, H, S, D,
                                   dev->sms, dev->status, trim, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return RA_OK;
}

unsigned long long ra_bwd_workspace_bytes(int B, int H, int S) {
  if (B <= 0 || H <= 0 || S <= 0) return 0;
  return (unsigned long long)B * (unsigned long long)H * (unsigned long long)S * 8ull;
}

}  // extern "C"

namespace {

// Checks shared by ra_bwd and ra_bwd_static (everything but the workspace).
ra_status check_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int S,
                    int D, int P, float scale) {
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return RA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Hkv <= 0 || S <= 0 || D <= 0 || P <= 0) return RA_ERR_INVALID_ARG;
  if (H % Hkv != 0 || S % P != 0) return RA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return RA_ERR_INVALID_ARG;
  if (scale < 0.0f) return RA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return RA_ERR_UNSUPPORTED;
  if ((S / P) % 128 != 0) return RA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return RA_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return RA_ERR_UNSUPPORTED;
  if ((long long)B * S >= (1ll << 31) || (long long)B * H * (S / 128) >= (1ll << 31))
    return RA_ERR_UNSUPPORTED;
  return RA_OK;
}

// Tensor maps, arguments and the three launches of the backward, with the
// per-row scratch at `ws` (8*B*H*S bytes).  Arguments are already checked.
ra_status launch_backward(DeviceInfo* dev, const void* q, const void* k, const void* v,
                          const void* out, const float* lse, const void* dout, void* dq, void* dk,
                          void* dv, float* ws, int B, int H, int Hkv, int S, int D, int P,
                          int causal, float scale, void* stream) {
  ra_status st;
  CUtensorMap tq, tk, tv, tdo;
  if ((st = tensor_map(q, (long long)B * S, H, D, &tq)) != RA_OK) return st;
  if ((st = tensor_map(k, (long long)B * S, Hkv, D, &tk)) != RA_OK) return st;
  if ((st = tensor_map(v, (long long)B * S, Hkv, D, &tv)) != RA_OK) return st;
  if ((st = tensor_map(dout, (long long)B * S, H, D, &tdo)) != RA_OK) return st;

  ra::BwdArgs a;
  std::memset(&a, 0, sizeof a);
  a.out = out;
  a.dout = dout;
  a.lse = lse;
  a.nlse2 = ws;
  a.ndelta = a.nlse2 + (size_t)B * H * S;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.status = dev->status;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.S = S;
  a.P = P;
  a.causal = causal ? 1 : 0;
  a.tiles = S / 128;
  a.tpc = S / P / 128;
  a.scale = scale;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    a.timeout_ns = g_timeout_ns;
    a.skip_first_load = g_skip_value_load;
    a.bounds_trim = g_bounds_trim;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long units = (long long)B * S * H * (D / 8);
  long long grid = (units + 255) / 256;
  if (grid > (long long)dev->sms * 8) grid = (long long)dev->sms * 8;
  cudaError_t e = ra::launch_bwd_prep(D, a, (int)grid, s);
  if (e != cudaSuccess) return cuda_fail(e);
  a.n_items = B * Hkv * a.tiles;
  e = ra::launch_bwd_dkdv(D, tq, tk, tv, tdo, a, a.n_items < dev->sms ? a.n_items : dev->sms, s);
  if (e != cudaSuccess) return cuda_fail(e);
  a.n_items = B * H * a.tiles;
  e = ra::launch_bwd_dq(D, tq, tk, tv, tdo, a, a.n_items < dev->sms ? a.n_items : dev->sms, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return RA_OK;
}

}  // namespace

extern "C" {

ra_status ra_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, void* workspace,
                 unsigned long long workspace_bytes, int B, int H, int Hkv, int S, int D, int P,
                 int causal, float scale, void* stream) {
  ra_status st = check_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, H, Hkv, S, D, P, scale);
  if (st != RA_OK) return st;
  if (!workspace || workspace_bytes < ra_bwd_workspace_bytes(B, H, S)) return RA_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return RA_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != RA_OK) return st;
  if (!dev->sm103) return RA_ERR_UNSUPPORTED;
  return launch_backward(dev, q, k, v, out, lse, dout, dq, dk, dv, static_cast<float*>(workspace),
                         B, H, Hkv, S, D, P, causal, scale, stream);
}

ra_status ra_bwd_static(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                        int H, int Hkv, int S, int D, int P, int causal, float scale,
                        void* stream) {
  ra_status st = check_bwd(q, k, v, out, lse, dout, dq, dk, dv, B, H, Hkv, S, D, P, scale);
  if (st != RA_OK) return st;
  if ((long long)B * H * S > ra::kStaticBwdRows) return RA_ERR_UNSUPPORTED;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != RA_OK) return st;
  if (!dev->sm103) return RA_ERR_UNSUPPORTED;
  return launch_backward(dev, q, k, v, out, lse, dout, dq, dk, dv, dev->bwd_scratch, B, H, Hkv, S,
                         D, P, causal, scale, stream);
}

ra_status ra_measure_ceilings(double* out) {
  if (!out) return RA_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  ra_status st = device_info(&dev);
  if (st != RA_OK) return st;
  if (!dev->sm103) return RA_ERR_UNSUPPORTED;
  const cudaError_t e = ra::measure_ceilings(dev->sms, out);
  return e == cudaSuccess ? RA_OK : cuda_fail(e);
}

ra_status ra_get_last_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int v = 0;
  e = ra::read_and_clear_status(&v);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v & ra::kStatusTimeout) return RA_ERR_TIMEOUT;
  if (v & ra::kStatusBounds) return RA_ERR_BOUNDS;
  return (v & ra::kStatusLayout) ? RA_ERR_UNSUPPORTED : RA_OK;
}

const char* ra_status_string(ra_status s) {
  switch (s) {
    case RA_OK: return "RA_OK";
    case RA_ERR_INVALID_ARG: return "RA_ERR_INVALID_ARG";
    case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED";
    case RA_ERR_CUDA: return "RA_ERR_CUDA";
    case RA_ERR_TIMEOUT: return "RA_ERR_TIMEOUT";
    case RA_ERR_BOUNDS: return "RA_ERR_BOUNDS";
  }
  return "RA_ERR_UNKNOWN";
}

int ra_last_cuda_error(void) { return g_last_cuda_error; }

int ra_version(void) { return (0 << 16) | (3 << 8) | 0; }

void ra_debug_set_fault(long long timeout_ns, int skip_value_load) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_timeout_ns = timeout_ns > 0 ? (unsigned long long)timeout_ns : kDefaultTimeoutNs;
  g_skip_value_load = skip_value_load ? 1 : 0;
}

void ra_debug_set_bounds_trim(long long elements) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_bounds_trim = elements > 0 ? elements : 0;
}

ra_status ra_trace_read(unsigned long long* out, int n_ctas) {
#ifdef RA_TRACE
  if (!out || n_ctas <= 0) return RA_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  e = ra::trace_copy(out, n_ctas);
  if (e != cudaSuccess) return cuda_fail(e);
  return RA_OK;
#else
  (void)out;
  (void)n_ctas;
  return RA_ERR_UNSUPPORTED;
#endif
}

int ra_debug_build(void) {
  int flags = 0;
#ifdef RA_DEBUG
  flags |= 1;
#endif
#ifdef RA_TRACE
  flags |= 2;
#endif
  return flags;
}

void ra_set_mma_order(int order) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_mma_order = (order == ra::MMA_ORDER_STRICT || order == ra::MMA_ORDER_GROUPED ||
                 order == ra::MMA_ORDER_INORDER)
                    ? order
                    : ra::MMA_ORDER_BRIDGED;
}

void ra_set_item_pairing(int policy) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_item_pairing = (policy == 1 || policy == 2) ? policy : 0;
}

void ra_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  ra::g_prep_epoch.fetch_add(1u, std::memory_order_acq_rel);  // kernels are prepared again
  for (auto& e : g_maps) e.used = false;
  for (auto& d : g_dev) d = DeviceInfo{};
  g_timeout_ns = kDefaultTimeoutNs;
  g_skip_value_load = 0;
  g_mma_order = ra::MMA_ORDER_BRIDGED;
  g_item_pairing = 0;
  g_bounds_trim = 0;
}

}  // extern "C"
