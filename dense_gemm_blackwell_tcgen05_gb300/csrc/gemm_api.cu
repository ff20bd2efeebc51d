// The C ABI (include/gemm_gb300.h): argument validation, per-device set-up,
// tensor-map encoding, kernel choice and the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gemm_gb300.h"
#include "gemm_host.h"
#include "kernel_common.cuh"

// The library's only device state: the watchdog status word (first error
// wins; cleared by gemm_last_status).
static __device__ unsigned long long g_status_word = 0ull;

namespace gb300 {
namespace {

constexpr int kMaxDevices = 128;

struct DeviceState {
  int state = 0;  // 0 = not yet set up, 1 = ready, < 0 = gemm_status_t failure
  int num_sms = 0;
  unsigned long long* status = nullptr;
};

std::mutex g_mu;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<int64_t> g_watchdog_ms{-1};
std::atomic<int> g_streamk_mode{kStreamKAuto};
std::atomic<int> g_tail_split{1};
std::atomic<int> g_edge_last{1};
std::atomic<uint32_t> g_streamk_epoch{0};
thread_local int t_last_cuda_error = 0;
thread_local int64_t t_stall_next = -1;   // one-shot watchdog test hook
thread_local int64_t t_schedule[7] = {0, 0, 0, 0, 0, 0, 0};

// Consumes the calling thread's pending stall request, if any.
uint32_t take_stall() {
  const int64_t v = t_stall_next;
  t_stall_next = -1;
  return v < 0 ? 0xFFFFFFFFu : static_cast<uint32_t>(v);
}

int64_t watchdog_ms() {
  int64_t v = g_watchdog_ms.load();
  if (v < 0) {
    int64_t def = 2000;
    if (const char* e = std::getenv("GEMM_WATCHDOG_MS")) {
      const long long x = std::atoll(e);
      if (x > 0) def = x;
    }
    int64_t expected = -1;
    g_watchdog_ms.compare_exchange_strong(expected, def);
    v = g_watchdog_ms.load();
  }
  return v;
}

// Current device: compute capability 10.3 required; SM count, the status
// word's device address and the tensor-map encoder are looked up once.
int current_device(LaunchCtx* ctx) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_devices[dev];
  if (d.state == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      d.state = GEMM_ERR_UNSUPPORTED_DEVICE;
    } else if (major != 10 || minor != 3) {
      d.state = GEMM_ERR_UNSUPPORTED_DEVICE;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
        cudaGetLastError();
        d.state = GEMM_ERR_LAUNCH;
      } else {
        d.status = static_cast<unsigned long long*>(p);
        d.num_sms = sms;
        d.state = 1;
      }
    }
    if (d.state == 1 && g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        d.state = GEMM_ERR_LAUNCH;
      } else {
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
    }
  }
  if (d.state != 1) return d.state;
  ctx->device = dev;
  ctx->num_sms = d.num_sms;
  ctx->status = d.status;
  return GEMM_OK;
}

// True when `p` is memory the current device can address (device or managed).
bool is_device_pointer(const void* p, int dev) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (attr.type == cudaMemoryTypeManaged) return true;
  return attr.type == cudaMemoryTypeDevice && attr.device == dev;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

// Shape and pitch checks shared by both element types (esize: operand bytes).
int check_shape(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                int64_t lda, int64_t ldb, int64_t ldd, int64_t esize) {
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (D == nullptr || ldd < N || ldd > (int64_t(1) << 36)) return GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(D) & 1u) != 0) return GEMM_ERR_ALIGNMENT;   // bf16 elements
  if (K == 0) return GEMM_OK;
  if (A == nullptr || B == nullptr || lda < K || ldb < K || lda > (int64_t(1) << 36) ||
      ldb > (int64_t(1) << 36))
    return GEMM_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || (lda * esize) % 16 != 0 || (ldb * esize) % 16 != 0)
    return GEMM_ERR_ALIGNMENT;
  return GEMM_OK;
}

// The TMA-store epilogue needs a 16-byte aligned D with a 16-byte multiple
// pitch, and N * 2 bytes a multiple of 16 as well: a tensor store clips its
// box against the row end only to 16-byte granularity, so a ragged N would
// also write the padding columns up to the next 16-byte boundary.
bool tma_store_ok(const void* D, int64_t N, int64_t ldd, bool direct) {
  return !direct && aligned16(D) && (ldd * 2) % 16 == 0 && (N * 2) % 16 == 0;
}

int64_t timeout_ns_for(int64_t K) {
  // The longest legitimate wait is about one tile's main loop; allow 64 ns per
  // k on top of the fixed limit (eight times a pessimistic per-SM rate).
  return watchdog_ms() * 1000000ll + K * 64ll;
}

// Every element of D, C and bias is accessed at its own alignment: the
// pointers must be multiples of their element sizes.  (Checked before any
// device work, like the shape.)
int check_epilogue_alignment(const gemm_epilogue_t* e, const void* D) {
  if (e == nullptr) return GEMM_OK;
  const uintptr_t osz = e->out_dtype == GEMM_DTYPE_F32 ? 4u : 2u;
  if ((reinterpret_cast<uintptr_t>(D) & (osz - 1)) != 0 ||
      (e->C != nullptr && (reinterpret_cast<uintptr_t>(e->C) & (osz - 1)) != 0) ||
      (e->bias != nullptr &&
       (reinterpret_cast<uintptr_t>(e->bias) & (e->bias_dtype == GEMM_DTYPE_F32 ? 3u : 1u)) != 0))
    return GEMM_ERR_ALIGNMENT;
  return GEMM_OK;
}

// Fills the fused-epilogue fields of `p` from `e` (NULL: the plain store).
// N, D and ldd are the call's; returns a gemm_status_t.
int parse_epilogue(const gemm_epilogue_t* e, int64_t N, const void* D, int64_t ldd, int device,
                   Problem& p) {
  if (e == nullptr) return GEMM_OK;
  if (e->reserved != 0 || (e->out_dtype != GEMM_DTYPE_BF16 && e->out_dtype != GEMM_DTYPE_F32) ||
      e->activation < GEMM_ACT_NONE || e->activation > GEMM_ACT_GELU)
    return GEMM_ERR_INVALID_ARG;
  uint32_t mode = static_cast<uint32_t>(e->activation) << kEpiActShift;
  if (e->out_dtype == GEMM_DTYPE_F32) mode |= kEpiOutF32;
  if (!(e->alpha == 1.0f)) mode |= kEpiAlpha;
  if (e->C != nullptr) {
    if (e->ldc < N || e->ldc > (int64_t(1) << 36) || !is_device_pointer(e->C, device) ||
        (e->C == D && e->ldc != ldd))
      return GEMM_ERR_INVALID_ARG;
    mode |= kEpiC;
  }
  if (e->bias != nullptr) {
    if ((e->bias_dtype != GEMM_DTYPE_BF16 && e->bias_dtype != GEMM_DTYPE_F32) ||
        !is_device_pointer(e->bias, device))
      return GEMM_ERR_INVALID_ARG;
    mode |= kEpiBias | (e->bias_dtype == GEMM_DTYPE_F32 ? kEpiBiasF32 : 0u);
  }
  p.epi_mode = mode;
  p.alpha = e->alpha;
  p.beta = e->beta;
  p.C = e->C;
  p.ldc = static_cast<uint64_t>(e->C != nullptr ? e->ldc : 0);
  p.bias = e->bias;
  return GEMM_OK;
}

}  // namespace

void note_cuda_error(cudaError_t e) { t_last_cuda_error = static_cast<int>(e); }

int streamk_mode() { return g_streamk_mode.load(); }

uint32_t plan_tail_split(uint64_t tiles, uint64_t resident) {
  if (g_tail_split.load() == 0 || tiles == 0 || resident == 0) return 0;
  // the tiles of the last round (all of them when there are fewer tiles than
  // clusters): cut in halves when the halves still fit in one round
  const uint64_t r = tiles % resident;
  return r != 0 && 2 * r <= resident ? static_cast<uint32_t>(r) : 0u;
}

uint32_t next_streamk_epoch() {
  uint32_t e = g_streamk_epoch.fetch_add(1) + 1;
  if (e == 0) e = g_streamk_epoch.fetch_add(1) + 1;   // 0 means "no partial yet"
  return e;
}

bool edge_last_enabled() { return g_edge_last.load() != 0; }

void note_schedule(uint32_t clusters, uint32_t cg, uint32_t dp_tiles, uint32_t sk_tiles,
                   uint32_t sk_unit, uint32_t half_tiles, uint32_t edge_last) {
  t_schedule[0] = clusters;
  t_schedule[1] = cg;
  t_schedule[2] = dp_tiles;
  t_schedule[3] = sk_tiles;
  t_schedule[4] = sk_unit;
  t_schedule[5] = half_tiles;
  t_schedule[6] = edge_last;
}

namespace {
// Encoded tensor maps are pure functions of their arguments, so a small
// per-thread direct-mapped cache saves the driver call on repeated shapes.
struct MapKey {
  const void* base;
  uint64_t inner, rows, pitch;
  uint32_t box_inner, box_rows;
  int dtype, swizzle;
  uint64_t dim2 = 0, pitch2 = 0;   // third dimension (0: a 2-D map)
  uint32_t box2 = 0;
  bool operator==(const MapKey& o) const {
    return base == o.base && inner == o.inner && rows == o.rows && pitch == o.pitch &&
           box_inner == o.box_inner && box_rows == o.box_rows && dtype == o.dtype &&
           swizzle == o.swizzle && dim2 == o.dim2 && pitch2 == o.pitch2 && box2 == o.box2;
  }
};
struct MapEntry {
  bool valid = false;
  MapKey key;
  CUtensorMap map;
};
constexpr int kMapCacheSize = 64;
thread_local MapEntry t_map_cache[kMapCacheSize];

uint32_t map_slot(const MapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
  h ^= (k.inner + 31 * k.rows + 131 * k.pitch + 1009ull * k.box_inner + 9176ull * k.box_rows +
        7ull * static_cast<uint64_t>(k.dtype) + 3ull * static_cast<uint64_t>(k.swizzle) +
        10007ull * k.dim2 + 37ull * k.pitch2 + 101ull * k.box2) *
       0xC2B2AE3D27D4EB4Full;
  return static_cast<uint32_t>(h >> 58) % kMapCacheSize;
}
}  // namespace

bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                   uint64_t rows, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle) {
  if (g_encode == nullptr) return false;
  const MapKey key{base, inner, rows, pitch_bytes, box_inner, box_rows, static_cast<int>(dtype),
                   static_cast<int>(swizzle)};
  MapEntry& slot = t_map_cache[map_slot(key)];
  if (slot.valid && slot.key == key) {
    *map = slot.map;
    return true;
  }
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = 100000 + static_cast<int>(r);
    return false;
  }
  slot.valid = true;
  slot.key = key;
  slot.map = *map;
  return true;
}

bool encode_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                   const uint64_t (&dims)[3], const uint64_t (&strides)[2], const uint32_t (&box)[3]) {
  if (g_encode == nullptr) return false;
  MapKey key{base, dims[0], dims[1], strides[0], box[0], box[1], static_cast<int>(dtype),
             static_cast<int>(CU_TENSOR_MAP_SWIZZLE_NONE)};
  key.dim2 = dims[2];
  key.pitch2 = strides[1];
  key.box2 = box[2];
  MapEntry& slot = t_map_cache[map_slot(key)];
  if (slot.valid && slot.key == key) {
    *map = slot.map;
    return true;
  }
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {strides[0], strides[1]};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, dtype, 3, const_cast<void*>(base), d, st, bx, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = 100000 + static_cast<int>(r);
    return false;
  }
  slot.valid = true;
  slot.key = key;
  slot.map = *map;
  return true;
}

}  // namespace gb300

using namespace gb300;

extern "C" {

static int bf16_impl(int variant, const void* A, const void* B, void* D, int64_t M, int64_t N,
                     int64_t K, int64_t lda, int64_t ldb, int64_t ldd, void* ws, int64_t ws_bytes,
                     const gemm_epilogue_t* epi, cudaStream_t stream) {
  const int base = variant & 0xFF;
  const bool direct = (variant & GEMM_VARIANT_DIRECT_STORE) != 0;
  if ((variant & ~(0xFF | GEMM_VARIANT_DIRECT_STORE)) != 0 || base > GEMM_VARIANT_SMALLK_TC)
    return GEMM_ERR_INVALID_ARG;
  const bool smallk = base == GEMM_VARIANT_SMALLK || base == GEMM_VARIANT_SMALLK_TC;
  if (smallk && (ws != nullptr || epi != nullptr || K > smallk_max_k())) return GEMM_ERR_INVALID_ARG;
  int rc = check_shape(A, B, D, M, N, K, lda, ldb, ldd, 2);
  if (rc == GEMM_OK && M != 0 && N != 0) rc = check_epilogue_alignment(epi, D);
  if (rc != GEMM_OK || M == 0 || N == 0) return rc;
  LaunchCtx ctx;
  if ((rc = current_device(&ctx)) != GEMM_OK) return rc;
  if (!is_device_pointer(D, ctx.device)) return GEMM_ERR_INVALID_ARG;
  Problem p = {};
  p.M = static_cast<uint32_t>(M);
  p.N = static_cast<uint32_t>(N);
  p.K = static_cast<uint32_t>(K);
  p.lda = static_cast<uint64_t>(lda);
  p.ldb = static_cast<uint64_t>(ldb);
  p.ldd = static_cast<uint64_t>(ldd);
  p.A = A;
  p.B = B;
  p.D = D;
  if ((rc = parse_epilogue(epi, N, D, ldd, ctx.device, p)) != GEMM_OK) return rc;
  if (p.epi_mode != 0 && base == GEMM_VARIANT_SYNC) return GEMM_ERR_INVALID_ARG;
  if (K == 0)
    return p.epi_mode != 0 ? launch_epilogue_only(p, ctx.num_sms, stream) : launch_zero_fill(p, stream);
  if (!is_device_pointer(A, ctx.device) || !is_device_pointer(B, ctx.device))
    return GEMM_ERR_INVALID_ARG;
  ctx.timeout_ns = static_cast<unsigned long long>(timeout_ns_for(K));
  p.stall_iter = take_stall();
  p.workspace = ws;
  p.workspace_bytes = ws_bytes > 0 ? static_cast<uint64_t>(ws_bytes) : 0u;
  if (ws != nullptr && (base == GEMM_VARIANT_SYNC || !is_device_pointer(ws, ctx.device)))
    return GEMM_ERR_INVALID_ARG;
  bool tma_store = tma_store_ok(D, N, ldd, direct) && !(p.epi_mode & kEpiOutF32);
  // A fused epilogue on the one-CTA kernel takes its masked-store build: the
  // library builds no fused TMA-store one-CTA kernel (see launch_ws.cuh).
  if (p.epi_mode != 0 &&
      (base == GEMM_VARIANT_1CTA || (base == GEMM_VARIANT_AUTO && M <= 128)))
    tma_store = false;
  // A launch that splits tiles along K sums the partial tiles in its epilogue
  // warps; the masked-store kernels have two epilogue groups against the
  // TMA-store kernels' one, which measured 11% faster on 1024x1024x16384.
  if (tma_store && ws != nullptr &&
      (base == GEMM_VARIANT_AUTO || base == GEMM_VARIANT_1CTA || base == GEMM_VARIANT_2CTA)) {
    const int cg = base == GEMM_VARIANT_1CTA ? 1 : base == GEMM_VARIANT_2CTA ? 2 : (M <= 128 ? 1 : 2);
    uint32_t sk_tiles = 0;
    if ((rc = bf16_streamk_split_tiles(cg, p, ctx, &sk_tiles)) != GEMM_OK) return rc;
    if (sk_tiles != 0) tma_store = false;
  }
  // Small K is a write of D: a small-K kernel unless the call needs the
  // persistent kernel's extras (an epilogue, a stream-K workspace).  The
  // tensor-core one writes D faster (3.2-3.6 TB/s against 2.5-2.7 at K = 8)
  // but costs about 6 us more to get going, so it takes outputs of 48 MB and
  // more (measured crossover about 46 MB).
  if (base == GEMM_VARIANT_AUTO && K <= smallk_max_k() && p.epi_mode == 0 && ws == nullptr) {
    if (static_cast<uint64_t>(M) * static_cast<uint64_t>(N) * 2 >= (48ull << 20))
      return launch_bf16_smallk_tc(p, ctx, stream);
    return launch_bf16_smallk(p, ctx.num_sms, stream);
  }
  switch (base) {
    case GEMM_VARIANT_SMALLK:
      return launch_bf16_smallk(p, ctx.num_sms, stream);
    case GEMM_VARIANT_SMALLK_TC:
      return launch_bf16_smallk_tc(p, ctx, stream);
    case GEMM_VARIANT_SYNC:
      return launch_bf16_sync(p, ctx, stream);
    case GEMM_VARIANT_1CTA:
      return launch_bf16_ws(1, tma_store, p, ctx, stream);
    case GEMM_VARIANT_AUTO:
      // One 128-row block of D: the pair's second CTA would multiply only
      // zero-filled rows, and the cluster launch costs about 2 us of latency.
      return launch_bf16_ws(M <= 128 ? 1 : 2, tma_store, p, ctx, stream);
    case GEMM_VARIANT_2CTA:
    default:
      return launch_bf16_ws(2, tma_store, p, ctx, stream);
  }
}

int gemm_bf16_variant(int variant, const void* A, const void* B, void* D, int64_t M, int64_t N,
                      int64_t K, int64_t lda, int64_t ldb, int64_t ldd, cudaStream_t stream) {
  return bf16_impl(variant, A, B, D, M, N, K, lda, ldb, ldd, nullptr, 0, nullptr, stream);
}

int gemm_bf16_streamk(int variant, const void* A, const void* B, void* D, int64_t M, int64_t N,
                      int64_t K, int64_t lda, int64_t ldb, int64_t ldd, void* workspace,
                      int64_t workspace_bytes, cudaStream_t stream) {
  if (workspace == nullptr) return GEMM_ERR_INVALID_ARG;
  return bf16_impl(variant, A, B, D, M, N, K, lda, ldb, ldd, workspace, workspace_bytes, nullptr,
                   stream);
}

int gemm_bf16_fused(int variant, const void* A, const void* B, void* D, int64_t M, int64_t N,
                    int64_t K, int64_t lda, int64_t ldb, int64_t ldd, const gemm_epilogue_t* epi,
                    cudaStream_t stream) {
  if ((variant & 0xFF) == GEMM_VARIANT_SYNC) return GEMM_ERR_INVALID_ARG;
  return bf16_impl(variant, A, B, D, M, N, K, lda, ldb, ldd, nullptr, 0, epi, stream);
}

int gemm_bf16(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
              int64_t lda, int64_t ldb, int64_t ldd, cudaStream_t stream) {
  return gemm_bf16_variant(GEMM_VARIANT_AUTO, A, B, D, M, N, K, lda, ldb, ldd, stream);
}

// sf_tiled: SFA/SFB hold the scale matrices in the tiled layout of
// gemm_mxfp8_tiled (ldsfa/ldsfb unused); else row-major with those pitches.
static int mxfp8_impl(int variant, const void* A, const void* B, const void* SFA,
                      const void* SFB, void* D, int64_t M, int64_t N, int64_t K, int64_t lda,
                      int64_t ldb, int64_t ldsfa, int64_t ldsfb, int64_t ldd, void* ws,
                      int64_t ws_bytes, const gemm_epilogue_t* epi, cudaStream_t stream,
                      bool sf_tiled = false) {
  const int base = variant & 0xFF;
  const bool direct = (variant & GEMM_VARIANT_DIRECT_STORE) != 0;
  if ((variant & ~(0xFF | GEMM_VARIANT_DIRECT_STORE)) != 0 || base > GEMM_VARIANT_2CTA)
    return GEMM_ERR_INVALID_ARG;
  int rc = check_shape(A, B, D, M, N, K, lda, ldb, ldd, 1);
  if (rc == GEMM_OK && M != 0 && N != 0) rc = check_epilogue_alignment(epi, D);
  if (rc != GEMM_OK || M == 0 || N == 0) return rc;
  if (K > 0 && sf_tiled) {
    // 512-byte chunks read by TMA: 16-byte aligned bases; each buffer's size
    // in 16-byte rows (32 per chunk) stays within a signed 32-bit count
    const int64_t kt = (K + 127) / 128;
    if (SFA == nullptr || SFB == nullptr || (M + 127) / 128 * kt * 32 > INT32_MAX ||
        (N + 127) / 128 * kt * 32 > INT32_MAX)
      return GEMM_ERR_INVALID_ARG;
    if (!aligned16(SFA) || !aligned16(SFB)) return GEMM_ERR_ALIGNMENT;
  } else if (K > 0) {
    const int64_t nblk = (K + 31) / 32;
    // Any pitch >= ceil(K/32) and any alignment: the launcher picks TMA or a
    // plain-load gather for the scale bytes.
    if (SFA == nullptr || SFB == nullptr || ldsfa < nblk || ldsfb < nblk ||
        ldsfa > (int64_t(1) << 36) || ldsfb > (int64_t(1) << 36))
      return GEMM_ERR_INVALID_ARG;
  }
  LaunchCtx ctx;
  if ((rc = current_device(&ctx)) != GEMM_OK) return rc;
  if (!is_device_pointer(D, ctx.device)) return GEMM_ERR_INVALID_ARG;
  Problem p = {};
  p.M = static_cast<uint32_t>(M);
  p.N = static_cast<uint32_t>(N);
  p.K = static_cast<uint32_t>(K);
  p.lda = static_cast<uint64_t>(lda);
  p.ldb = static_cast<uint64_t>(ldb);
  p.ldd = static_cast<uint64_t>(ldd);
  p.ldsfa = static_cast<uint64_t>(ldsfa);
  p.ldsfb = static_cast<uint64_t>(ldsfb);
  p.A = A;
  p.B = B;
  p.SFA = SFA;
  p.SFB = SFB;
  p.D = D;
  if ((rc = parse_epilogue(epi, N, D, ldd, ctx.device, p)) != GEMM_OK) return rc;
  if (K == 0)
    return p.epi_mode != 0 ? launch_epilogue_only(p, ctx.num_sms, stream) : launch_zero_fill(p, stream);
  if (!is_device_pointer(A, ctx.device) || !is_device_pointer(B, ctx.device) ||
      !is_device_pointer(SFA, ctx.device) || !is_device_pointer(SFB, ctx.device))
    return GEMM_ERR_INVALID_ARG;
  ctx.timeout_ns = static_cast<unsigned long long>(timeout_ns_for(K));
  p.stall_iter = take_stall();
  p.workspace = ws;
  p.workspace_bytes = ws_bytes > 0 ? static_cast<uint64_t>(ws_bytes) : 0u;
  if (ws != nullptr && !is_device_pointer(ws, ctx.device)) return GEMM_ERR_INVALID_ARG;
  // The automatic MXFP8 choice is the single-CTA kernel (the pair measures
  // slower), with the 32-column TMA-store epilogue where D allows it (same
  // four operand stages as the masked-store kernel; 0.5% faster at 8192^3).
  const bool tma_store = tma_store_ok(D, N, ldd, direct) && !(p.epi_mode & kEpiOutF32);
  // Tiled scales: the CTA pair unless one CTA is asked for.
  if (sf_tiled) return launch_mxf8t_ws(base == GEMM_VARIANT_1CTA ? 1 : 2, tma_store, p, ctx, stream);
  return launch_mxf8_ws(base == GEMM_VARIANT_2CTA ? 2 : 1, tma_store, p, ctx, stream);
}

int gemm_mxfp8_variant(int variant, const void* A, const void* B, const void* SFA,
                       const void* SFB, void* D, int64_t M, int64_t N, int64_t K, int64_t lda,
                       int64_t ldb, int64_t ldsfa, int64_t ldsfb, int64_t ldd,
                       cudaStream_t stream) {
  return mxfp8_impl(variant, A, B, SFA, SFB, D, M, N, K, lda, ldb, ldsfa, ldsfb, ldd, nullptr, 0,
                    nullptr, stream);
}

int gemm_mxfp8_fused(int variant, const void* A, const void* B, const void* SFA, const void* SFB,
                     void* D, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                     int64_t ldsfa, int64_t ldsfb, int64_t ldd, const gemm_epilogue_t* epi,
                     cudaStream_t stream) {
  return mxfp8_impl(variant, A, B, SFA, SFB, D, M, N, K, lda, ldb, ldsfa, ldsfb, ldd, nullptr, 0,
                    epi, stream);
}

int gemm_mxfp8_streamk(int variant, const void* A, const void* B, const void* SFA,
                       const void* SFB, void* D, int64_t M, int64_t N, int64_t K, int64_t lda,
                       int64_t ldb, int64_t ldsfa, int64_t ldsfb, int64_t ldd, void* workspace,
                       int64_t workspace_bytes, cudaStream_t stream) {
  if (workspace == nullptr) return GEMM_ERR_INVALID_ARG;
  return mxfp8_impl(variant, A, B, SFA, SFB, D, M, N, K, lda, ldb, ldsfa, ldsfb, ldd, workspace,
                    workspace_bytes, nullptr, stream);
}

int gemm_mxfp8_tiled(int variant, const void* A, const void* B, const void* SFA, const void* SFB,
                     void* D, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                     int64_t ldd, cudaStream_t stream) {
  return mxfp8_impl(variant, A, B, SFA, SFB, D, M, N, K, lda, ldb, 0, 0, ldd, nullptr, 0, nullptr,
                    stream, true);
}

int64_t gemm_streamk_workspace_bytes(int mxfp8, int variant) {
  LaunchCtx ctx;
  const int rc = current_device(&ctx);
  if (rc != GEMM_OK) return rc;
  const int base = variant & 0xFF;
  if (base > GEMM_VARIANT_2CTA) return GEMM_ERR_INVALID_ARG;
  KernelPlan k;
  const bool ok = mxfp8 ? plan_mxf8(base == GEMM_VARIANT_2CTA ? 2 : 1, false, &k)
                        : plan_bf16(base == GEMM_VARIANT_1CTA ? 1 : 2, false, &k);
  if (!ok) return GEMM_ERR_INVALID_ARG;
  return static_cast<int64_t>(static_cast<uint64_t>(ctx.num_sms) *
                              streamk_bytes_per_cta(static_cast<uint32_t>(k.tile_n)));
}

int gemm_mxfp8(const void* A, const void* B, const void* SFA, const void* SFB, void* D,
               int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldsfa,
               int64_t ldsfb, int64_t ldd, cudaStream_t stream) {
  return gemm_mxfp8_variant(GEMM_VARIANT_AUTO, A, B, SFA, SFB, D, M, N, K, lda, ldb, ldsfa, ldsfb,
                            ldd, stream);
}

int gemm_mxfp8_quantize(const float* X, int64_t rows, int64_t K, int64_t ldx, void* Q,
                        int64_t ldq, void* SF, int64_t ldsf, cudaStream_t stream) {
  if (rows < 0 || K < 0 || rows > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_ARG;
  if (rows == 0 || K == 0) return GEMM_OK;
  const int64_t nblk = (K + 31) / 32;
  if (X == nullptr || Q == nullptr || SF == nullptr || ldx < K || ldq < K || ldsf < nblk ||
      ldx > (int64_t(1) << 36) || ldq > (int64_t(1) << 36) || ldsf > (int64_t(1) << 36))
    return GEMM_ERR_INVALID_ARG;
  LaunchCtx ctx;
  int rc = current_device(&ctx);
  if (rc != GEMM_OK) return rc;
  if (!is_device_pointer(X, ctx.device) || !is_device_pointer(Q, ctx.device) ||
      !is_device_pointer(SF, ctx.device))
    return GEMM_ERR_INVALID_ARG;
  return launch_mxfp8_quantize(X, static_cast<uint32_t>(rows), static_cast<uint32_t>(K),
                               static_cast<uint64_t>(ldx), static_cast<uint8_t*>(Q),
                               static_cast<uint64_t>(ldq), static_cast<uint8_t*>(SF),
                               static_cast<uint64_t>(ldsf), false, ctx.num_sms, stream);
}

int gemm_mxfp8_quantize_tiled(const float* X, int64_t rows, int64_t K, int64_t ldx, void* Q,
                              int64_t ldq, void* SF, cudaStream_t stream) {
  if (rows < 0 || K < 0 || rows > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_ARG;
  if (rows == 0 || K == 0) return GEMM_OK;
  if (X == nullptr || Q == nullptr || SF == nullptr || ldx < K || ldq < K ||
      ldx > (int64_t(1) << 36) || ldq > (int64_t(1) << 36))
    return GEMM_ERR_INVALID_ARG;
  LaunchCtx ctx;
  int rc = current_device(&ctx);
  if (rc != GEMM_OK) return rc;
  if (!is_device_pointer(X, ctx.device) || !is_device_pointer(Q, ctx.device) ||
      !is_device_pointer(SF, ctx.device))
    return GEMM_ERR_INVALID_ARG;
  return launch_mxfp8_quantize(X, static_cast<uint32_t>(rows), static_cast<uint32_t>(K),
                               static_cast<uint64_t>(ldx), static_cast<uint8_t*>(Q),
                               static_cast<uint64_t>(ldq), static_cast<uint8_t*>(SF), 0, true,
                               ctx.num_sms, stream);
}

uint64_t gemm_last_status_word(cudaStream_t stream) {
  LaunchCtx ctx;
  if (current_device(&ctx) != GEMM_OK) return 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  unsigned long long w = 0;
  if (cudaMemcpyFromSymbol(&w, g_status_word, sizeof w) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return w;
}

int gemm_last_status(cudaStream_t stream) {
  LaunchCtx ctx;
  int rc = current_device(&ctx);
  if (rc != GEMM_OK) return rc;
  const cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_DEVICE_FAULT;
  }
  unsigned long long w = 0;
  if (cudaMemcpyFromSymbol(&w, g_status_word, sizeof w) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_DEVICE_FAULT;
  }
  if (w == 0) return GEMM_OK;
  const unsigned long long zero = 0;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_DEVICE_FAULT;
  }
  return (w >> 56) == kDevTimeout ? GEMM_ERR_TIMEOUT : GEMM_ERR_DEVICE_FAULT;
}

const char* gemm_status_string(int status) {
  switch (status) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_ALIGNMENT: return "operand alignment or pitch not supported by TMA";
    case GEMM_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103 (GB300)";
    case GEMM_ERR_LAUNCH: return "kernel launch or tensor-map encoding failed";
    case GEMM_ERR_TIMEOUT: return "device watchdog: a barrier wait timed out";
    case GEMM_ERR_DEVICE_FAULT: return "device fault reported by the stream";
    default: return "unknown status";
  }
}

int gemm_last_cuda_error(void) { return t_last_cuda_error; }

int gemm_set_streamk_mode(int mode) {
  if (mode < kStreamKAuto || mode > kStreamKNever) return GEMM_ERR_INVALID_ARG;
  return g_streamk_mode.exchange(mode);
}

int gemm_set_tail_split(int enable) {
  if (enable != 0 && enable != 1) return GEMM_ERR_INVALID_ARG;
  return g_tail_split.exchange(enable);
}

int gemm_set_edge_last(int enable) {
  if (enable != 0 && enable != 1) return GEMM_ERR_INVALID_ARG;
  return g_edge_last.exchange(enable);
}

int64_t gemm_tail_split_plan(int64_t tiles, int64_t resident) {
  if (tiles < 0 || resident < 0 || tiles > 0xFFFFFFFFll || resident > 0xFFFFFFFFll)
    return GEMM_ERR_INVALID_ARG;
  return plan_tail_split(static_cast<uint64_t>(tiles), static_cast<uint64_t>(resident));
}

int gemm_streamk_plan(int64_t tiles, int64_t resident, int64_t k_tiles, int64_t unit, int mode,
                      int64_t* out) {
  if (out == nullptr || tiles < 0 || resident < 1 || k_tiles < 0 || unit < 1 ||
      mode < kStreamKAuto || mode > kStreamKNever || tiles > 0x7FFFFFFF || resident > 0xFFFF ||
      k_tiles > 0x7FFFFFFF || unit > 0xFFFF)
    return GEMM_ERR_INVALID_ARG;
  if (tiles == 0 || k_tiles == 0) {
    out[0] = tiles;
    out[1] = 0;
    out[2] = 0;
    return GEMM_OK;
  }
  const StreamKPlan sp = plan_streamk(static_cast<uint64_t>(tiles), static_cast<uint64_t>(resident),
                                      static_cast<uint32_t>(k_tiles), static_cast<uint32_t>(unit), mode);
  out[0] = sp.dp_tiles;
  out[1] = sp.sk_tiles;
  out[2] = sp.clusters;
  return GEMM_OK;
}

int gemm_last_schedule(int64_t* out) {
  if (out == nullptr) return GEMM_ERR_INVALID_ARG;
  for (int i = 0; i < 7; ++i) out[i] = t_schedule[i];
  return GEMM_OK;
}

int gemm_debug_stall_next_launch(int64_t k_iteration) {
  if (k_iteration < 0 || k_iteration >= 0xFFFFFFFFll) return GEMM_ERR_INVALID_ARG;
  t_stall_next = k_iteration;
  return GEMM_OK;
}

int64_t gemm_set_watchdog_ms(int64_t ms) {
  const int64_t old = watchdog_ms();
  if (ms > 0) g_watchdog_ms.store(ms);
  return old;
}

int gemm_kernel_plan(int mxfp8, int variant, int32_t* stages, int32_t* smem_bytes,
                     int32_t* tmem_cols, int32_t* threads, int32_t* cluster, int32_t* tile_m,
                     int32_t* tile_n) {
  const int base = variant & 0xFF;
  const bool tma_store = (variant & GEMM_VARIANT_DIRECT_STORE) == 0;
  KernelPlan k;
  bool ok;
  if (mxfp8 == 2)
    ok = base <= GEMM_VARIANT_2CTA && plan_mxf8t(base == GEMM_VARIANT_1CTA ? 1 : 2, tma_store, &k);
  else if (mxfp8)
    ok = base <= GEMM_VARIANT_2CTA && plan_mxf8(base == GEMM_VARIANT_2CTA ? 2 : 1, tma_store, &k);
  else
    ok = plan_bf16(base == GEMM_VARIANT_AUTO ? 2 : base, tma_store, &k);
  if (!ok) return GEMM_ERR_INVALID_ARG;
  if (stages) *stages = k.stages;
  if (smem_bytes) *smem_bytes = k.smem_bytes;
  if (tmem_cols) *tmem_cols = k.tmem_cols;
  if (threads) *threads = k.threads;
  if (cluster) *cluster = k.cluster;
  if (tile_m) *tile_m = k.tile_m;
  if (tile_n) *tile_n = k.tile_n;
  return GEMM_OK;
}

}  // extern "C"
