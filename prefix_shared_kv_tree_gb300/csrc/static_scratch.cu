// Fixed-size device scratch for pst_decode_attention_noalloc.
//
// The area is a file-scope device array, so it exists on every GPU that loads
// the library and stays there until the process exits.  Host code cannot use
// the array's name as a device address (on the host it only names a stand-in
// object); the device address is looked up here with cudaGetSymbolAddress,
// once per device, with that device made current for the lookup.
#include <mutex>

#include "pst_internal.h"

namespace pst {

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

cudaError_t static_scratch_address(int device, void** ptr) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  if (device < 0 || device >= kMaxDevices || ptr == nullptr) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[device] == nullptr) {
    int current = -1;
    cudaError_t e = cudaGetDevice(&current);
    if (e != cudaSuccess) return e;
    if (current != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_static_scratch);
    if (current != device) cudaSetDevice(current);
    if (e != cudaSuccess) return e;
    addr[device] = a;
  }
  *ptr = addr[device];
  return cudaSuccess;
}

}  // namespace pst
