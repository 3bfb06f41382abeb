// muon_step_noalloc: the Muon step for callers that must not allocate device
// memory themselves.  Some hosts hand this library only the tensors they own:
// an inference or training runtime whose memory is carved up once at start-up
// and which forbids cudaMalloc (or any allocating call) afterwards, a plugin
// that lives inside another framework's allocator, or code that runs where an
// allocation would synchronise the device.  Such callers cannot provide the
// step's scratch workspace, so this entry point uses a fixed array in device
// global memory instead.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library reserves it (MUON_STATIC_WORKSPACE_BYTES) until the process exits.
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress while
// that device is current, and caches it.  That first call should therefore
// come before any stream capture.  The step itself is the ordinary
// muon_step() on that address: nothing here calls cudaMalloc, cudaFree or an
// allocating library routine.
//
// All calls on a device share the one array and it keeps the previous call's
// contents.  No part of it needs to start at zero: the step writes every word
// it reads.  The kernels' status word sits at the start of the array;
// muon_check_status(h, NULL, stream) reads and clears it there.  Calls that
// overlap on the GPU -- on different streams, or from different host threads
// -- race on the array and must be serialised by the caller.
#include "muon.h"

#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "muon_internal.h"

namespace {

constexpr size_t kStaticBytes = (size_t)MUON_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_workspace[kStaticBytes];

std::mutex g_mutex;
void* g_address[kMaxDevices] = {};

}  // namespace

namespace muon {

// Device address of the array on `device`, looked up once per device (also
// used by muon_check_status to read the kernels' status word in it).
int static_workspace(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return (int)cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_address[device]) {
    *out = g_address[device];
    return cudaSuccess;
  }
  int old = -1;
  cudaError_t e = cudaGetDevice(&old);
  if (e != cudaSuccess) return (int)e;
  if (old != device && (e = cudaSetDevice(device)) != cudaSuccess) return (int)e;
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_static_workspace);
  if (old != device) cudaSetDevice(old);
  if (e != cudaSuccess) return (int)e;
  g_address[device] = ptr;
  *out = ptr;
  return cudaSuccess;
}

}  // namespace muon

extern "C" muon_status muon_step_noalloc(muon_handle h, const muon_matrix_desc* descs, int n, void* stream) {
  if (!h) return MUON_ERR_INVALID_ARG;
  size_t need = 0;
  muon_status st = muon_workspace_size(h, descs, n, &need);  // validates the descriptors
  if (st != MUON_OK) return st;
  const int device = muon::handle_device(h);
  if (need == 0 || device < 0) return muon_step(h, descs, n, nullptr, 0, stream);
  if (need > kStaticBytes) {
    muon::set_handle_error(h, "muon_step_noalloc: this batch needs " + std::to_string(need) +
                                  " bytes of workspace, more than the fixed " + std::to_string(kStaticBytes) +
                                  " bytes (MUON_STATIC_WORKSPACE_BYTES); use muon_step with a caller workspace");
    return MUON_ERR_WORKSPACE;
  }
  if (device >= kMaxDevices) {
    muon::set_handle_error(h, "muon_step_noalloc: device index beyond 63");
    return MUON_ERR_UNSUPPORTED;
  }
  void* ws = nullptr;
  const cudaError_t e = (cudaError_t)muon::static_workspace(device, &ws);
  if (e != cudaSuccess) {
    muon::set_handle_error(h, std::string("muon_step_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    return MUON_ERR_CUDA;
  }
  return muon_step(h, descs, n, ws, kStaticBytes, stream);
}
