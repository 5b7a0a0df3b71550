// lce_noalloc.cu -- ikbo_lce_forward_noalloc: the fused LCE for callers that
// must not allocate device memory.
//
// ikbo_lce_forward keeps its fp32 user partials and readiness flags in a
// plan that ikbo_plan_create fills with cudaMalloc.  Some callers cannot do
// that: their device memory belongs to another allocator (a framework's
// memory pool, a fixed per-process budget), or their request path may not
// call cudaMalloc / cudaFree, which can synchronise the whole device.  This
// entry point runs the same kernel with its scratch in a fixed-size array
// that the library itself declares in device memory, so nothing is
// allocated per call or per plan.
//
// The array is a file-scope static __device__ object: every GPU that loads
// the library holds its kNoallocScratchBytes until the process exits.  Its
// host-side name is only a stand-in, so the device address is fetched with
// cudaGetSymbolAddress, once per device, on the first call made while that
// device is current; make that first call before capturing any stream.
// All calls share the array and it keeps the last call's contents: each call
// first clears, on its stream, the words that must start at zero (status,
// readiness flags).  Calls that overlap on the GPU (two streams, or two host
// threads on one device) race on it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "ikbo.h"
#include "ikbo_internal.h"

namespace ikbo {
cudaError_t launch_lce(const CUtensorMap& tmU, const CUtensorMap& tmC, const CUtensorMap& tmWu,
                       const CUtensorMap& tmWc, const LceParams& p, int num_sms, cudaStream_t s, int* launches);
}  // namespace ikbo

using namespace ikbo;

namespace {

// 16 MiB: room for the user partials of n_users * N * D <= ~4.19 M fp32
// values (for example 80 users at N = 192, D = 256) plus their flags.
constexpr size_t kNoallocScratchBytes = size_t(16) << 20;
constexpr size_t kControlBytes = 256;  // [0] status bits, [1] flag-timeout word, [2] finished-CTA count
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_lce_scratch[kNoallocScratchBytes];

struct DeviceSlot {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_lce_scratch on this device
  int num_sms = 0;
  size_t max_smem = 0;
};

std::mutex g_mu;
DeviceSlot g_slots[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// bf16 tensor map, 128-byte swizzle, out-of-bounds elements read as zero.
bool tensor_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                const uint32_t* box) {
  EncodeTiledFn fn = encoder();
  if (!fn) return false;
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd, gs, bx,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// First call on a device (that device current): look up the scratch array's
// device address and the launch limits.  Returns the slot, or null.
DeviceSlot* device_slot(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  DeviceSlot* s = &g_slots[dev];
  if (s->ready) return s;
  void* ptr = nullptr;
  *err = cudaGetSymbolAddress(&ptr, g_lce_scratch);
  if (*err != cudaSuccess) return nullptr;
  int sms = 0, smem = 0, major = 0, minor = 0;
  if ((*err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
      (*err = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
      (*err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (*err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
    return nullptr;
  if (major != 10 || minor != 3) {
    *err = cudaErrorNoKernelImageForDevice;
    return nullptr;
  }
  s->scratch = static_cast<unsigned char*>(ptr);
  s->num_sms = sms;
  s->max_smem = static_cast<size_t>(smem);
  s->ready = true;
  return s;
}

}  // namespace

extern "C" ikbo_status_t ikbo_lce_forward_noalloc(const int32_t* d_map, int n_cand, int n_users, const void* U,
                                                  const void* C, const void* Wu, const void* Wc, const void* b,
                                                  void* Y, int K_u, int K_c, int D, int N, cudaStream_t stream) {
  if (!d_map || !U || !C || !Wu || !Wc || !Y) return IKBO_ERR_INVALID_ARG;
  if (n_cand < 1 || n_users < 1) return IKBO_ERR_INVALID_ARG;
  if (K_u < 1 || K_c < 1 || D < 1 || N < 1) return IKBO_ERR_UNSUPPORTED;
  if (!aligned16(U) || !aligned16(C) || !aligned16(Wu) || !aligned16(Wc) || !aligned16(Y) || (b && !aligned16(b)))
    return IKBO_ERR_INVALID_ARG;
  if (D % 8 != 0 || N % 8 != 0 || N > 256) return IKBO_ERR_UNSUPPORTED;

  LceParams lp;
  std::memset(&lp, 0, sizeof(lp));
  lp.n_cand = n_cand;
  lp.n_users = n_users;
  lp.K_u = K_u;
  lp.K_c = K_c;
  lp.D = D;
  lp.N = N;
  // shapes only here; the shared-memory limit is checked once the device is known
  if (!lce_configure(&lp, SIZE_MAX)) return IKBO_ERR_UNSUPPORTED;

  // scratch layout: control words | flags [n_users][n_dblk][NB] | partial [n_users][N][D] fp32
  const size_t flag_bytes = round256(sizeof(uint32_t) * lce_flag_count(lp));
  const size_t part_bytes = sizeof(float) * static_cast<size_t>(n_users) * N * D;
  if (kControlBytes + flag_bytes + part_bytes > kNoallocScratchBytes) return IKBO_ERR_UNSUPPORTED;

  DeviceSlot* slot = nullptr;
  {
    std::lock_guard<std::mutex> g(g_mu);
    cudaError_t e;
    slot = device_slot(&e);
    if (!slot) return IKBO_ERR_CUDA;
  }
  if (!lce_configure(&lp, slot->max_smem)) return IKBO_ERR_UNSUPPORTED;

  unsigned char* base = slot->scratch;
  lp.map = d_map;
  lp.bias = static_cast<const uint16_t*>(b);
  lp.U = static_cast<const uint16_t*>(U);
  lp.Wu = static_cast<const uint16_t*>(Wu);
  lp.Y = static_cast<uint16_t*>(Y);
  lp.status = reinterpret_cast<uint32_t*>(base);
  lp.timeout_epoch = reinterpret_cast<uint32_t*>(base) + 1;
  lp.done = reinterpret_cast<uint32_t*>(base) + 2;
  lp.flags = reinterpret_cast<uint32_t*>(base + kControlBytes);
  lp.partial = reinterpret_cast<float*>(base + kControlBytes + flag_bytes);
  lp.epoch = LCE_FLAG_READY;
  lp.debug = 0;
  lp.timeout_ns = 2000000000ull;

  CUtensorMap tmU, tmC, tmWu, tmWc;
  const uint64_t ud[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(K_u), static_cast<uint64_t>(n_users)};
  const uint64_t us[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(K_u) * D * 2};
  const uint64_t cd[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(K_c), static_cast<uint64_t>(n_cand)};
  const uint64_t cs[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(K_c) * D * 2};
  const uint32_t abox[3] = {64, LCE_BK, 1};
  const uint64_t wud[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K_u)};
  const uint64_t wcd[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K_c)};
  const uint64_t ws[1] = {static_cast<uint64_t>(N) * 2};
  const uint32_t wbox[2] = {64, LCE_BK};
  if (!tensor_map(&tmU, U, 3, ud, us, abox) || !tensor_map(&tmC, C, 3, cd, cs, abox) ||
      !tensor_map(&tmWu, Wu, 2, wud, ws, wbox) || !tensor_map(&tmWc, Wc, 2, wcd, ws, wbox))
    return IKBO_ERR_CUDA;

  // the control words and the readiness flags start at zero on every call
  // (an earlier call that did not finish cleanly may have left them set)
  if (cudaMemsetAsync(base, 0, kControlBytes + flag_bytes, stream) != cudaSuccess) return IKBO_ERR_CUDA;
  int launches = 0;
  if (launch_lce(tmU, tmC, tmWu, tmWc, lp, slot->num_sms, stream, &launches) != cudaSuccess) return IKBO_ERR_CUDA;
  return IKBO_OK;
}
