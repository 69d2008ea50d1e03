// qli_run_static: the indexer for callers that cannot allocate device memory.
//
// Some callers have no way to allocate GPU memory when they call the
// indexer: a serving engine that has handed all free device memory to its
// KV-cache pool at start-up and runs with a fixed memory plan, or a plain C
// host program that links this library without any device allocator of its
// own. qli_run needs a caller-provided workspace; this entry point uses a
// fixed array compiled into the library instead, so such callers pass only
// their inputs and outputs.
//
// The array is a file-scope __device__ variable of QLI_STATIC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits. In host
// code its name is only a host-side stand-in, so its device address is looked
// up with cudaGetSymbolAddress, once per device, with that device current, on
// the first qli_run_static call made on that device; make that first call
// before any stream capture begins. Calls whose scratch need exceeds the
// array are rejected before anything is launched.
//
// All calls share the one array and it keeps whatever the previous call left
// there. No part of it needs to start at zero: the first kernel of every call
// resets the error word and the counter that later kernels accumulate into,
// and every other value is written before it is read. Two calls whose work
// overlaps on the GPU (for example on two streams) race on the array; order
// them on one stream.
#include <mutex>

#include "qli_internal.h"

namespace qli {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[QLI_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device (looked up once).
qli_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QLI_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return QLI_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return QLI_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return QLI_OK;
}

}  // namespace
}  // namespace qli

extern "C" qli_status qli_run_static(const qli_args* a, void* stream) {
  size_t need = 0;
  qli_status st = qli_workspace_size(a, &need);
  if (st != QLI_OK) return st;
  if (need > QLI_STATIC_SCRATCH_BYTES) return QLI_ERR_WORKSPACE_TOO_SMALL;
  if (a->T == 0) return QLI_OK;
  // the device check comes first, as in qli_run: on a GPU this library was
  // not built for, the symbol lookup would fail and leave a sticky error
  int sms = 0;
  st = qli::device_sms(&sms);
  if (st != QLI_OK) return st;
  void* scratch = nullptr;
  st = qli::static_scratch(&scratch);
  if (st != QLI_OK) return st;
  return qli_run(a, scratch, QLI_STATIC_SCRATCH_BYTES, stream);
}

// The error word sits at the start of the scratch, where every call's
// planning kernel resets it and later kernels OR their flags in.
extern "C" qli_status qli_read_static_device_error(uint32_t* host_word, void* stream) {
  if (host_word == nullptr) return QLI_ERR_INVALID_ARG;
  int sms = 0;
  qli_status st = qli::device_sms(&sms);
  if (st != QLI_OK) return st;
  void* scratch = nullptr;
  st = qli::static_scratch(&scratch);
  if (st != QLI_OK) return st;
  return qli_read_device_error(scratch, host_word, stream);
}
