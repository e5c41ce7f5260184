// Index check that allocates nothing: ccu_conv1d_check_indices_noalloc.
//
// ccu_conv1d_check_indices needs a bitmap of one bit per cache slot, and expects the
// caller to provide that scratch. Some callers cannot: a plugin that reaches this library
// through a C function table with no handle on the host application's device allocator,
// or a serving loop whose owner forbids cudaMalloc between steps because it can
// synchronize the whole device and stall every other stream. For them the bitmap lives
// here, in a fixed array compiled into the library, and the caller passes only the
// indices and the status word.
//
// The array is a file-scope __device__ variable: every GPU on which the library's device
// code is loaded holds its 128 KB until the process exits. In host code its name is only
// a host-side stand-in, so the device address is looked up with cudaGetSymbolAddress with
// the device current. The lookup is repeated on every call whose stream is not being
// captured: after a cudaDeviceReset (or a release of the primary context) the device code
// is loaded again and the array may sit at another address. While a stream is being
// captured the address found by the last uncaptured call on the device is used instead,
// since the lookup may load device code, which a capture does not allow.
#include <mutex>

#include "ccu_conv1d.h"
#include "ccu_internal.cuh"

namespace {

constexpr int64_t kMaxSlots = CCU_CHECK_INDICES_NOALLOC_MAX_SLOTS;
constexpr int64_t kWords = (kMaxSlots + 31) / 32;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint32_t g_noalloc_bitmap[kWords];

std::mutex g_setup_mutex;
uint32_t *g_bitmap_addr[kMaxDevices] = {};  // device address of g_noalloc_bitmap, per device

// Failures are described in the library's per-thread message (ccu_conv1d_last_error).
ccu_status_t noalloc_fail(ccu_status_t st, const char *msg) {
  ccu::record_error(msg);
  return st;
}

// The bitmap's device address on the current device: looked up again unless `capturing`,
// in which case the address of the last uncaptured lookup on this device is returned
// (cudaErrorStreamCaptureUnsupported if there was none).
cudaError_t bitmap_on_current_device(bool capturing, uint32_t **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!capturing) {
    void *addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_noalloc_bitmap);
    if (e != cudaSuccess) return e;
    g_bitmap_addr[dev] = static_cast<uint32_t *>(addr);
  }
  if (g_bitmap_addr[dev] == nullptr) return cudaErrorStreamCaptureUnsupported;
  *out = g_bitmap_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

ccu_status_t ccu_conv1d_check_indices_noalloc(const int32_t *indices, int64_t N, int64_t S,
                                              int32_t *status_dev, ccu_stream_t stream) {
  ccu::record_error("");
  if (N < 0 || S < 0) return noalloc_fail(CCU_ERR_INVALID_ARGUMENT, "N and S must be >= 0");
  if (S > kMaxSlots)
    return noalloc_fail(CCU_ERR_NOT_IMPLEMENTED,
                        "S exceeds the 1048576 slots the built-in bitmap holds; use "
                        "ccu_conv1d_check_indices with a caller-provided bitmap");
  if (N == 0) return CCU_OK;
  if (indices == nullptr || status_dev == nullptr)
    return noalloc_fail(CCU_ERR_INVALID_ARGUMENT, "indices and status_dev must not be NULL");
  if (reinterpret_cast<uintptr_t>(indices) % 4 != 0 ||
      reinterpret_cast<uintptr_t>(status_dev) % 4 != 0)
    return noalloc_fail(CCU_ERR_INVALID_ARGUMENT, "indices and status_dev must be 4-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return noalloc_fail(CCU_ERR_CUDA, cudaGetErrorString(e));
  uint32_t *bitmap = nullptr;
  e = bitmap_on_current_device(cap != cudaStreamCaptureStatusNone, &bitmap);
  if (e != cudaSuccess)
    return noalloc_fail(CCU_ERR_CUDA,
                        "could not resolve the built-in bitmap on this device (while a stream is "
                        "captured, an earlier uncaptured call on the device is needed)");
  // The array keeps the previous call's bits: clear the words this call uses.
  const size_t bytes = (size_t)((S + 31) / 32) * sizeof(uint32_t);
  if (bytes > 0) e = cudaMemsetAsync(bitmap, 0, bytes, s);
  if (e == cudaSuccess) e = ccu::launch_check_indices(indices, N, S, bitmap, status_dev, s);
  if (e != cudaSuccess) return noalloc_fail(CCU_ERR_CUDA, cudaGetErrorString(e));
  return CCU_OK;
}

}  // extern "C"
