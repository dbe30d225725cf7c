// Allocation-free variant of the forward pass.
//
// tpmlp_forward needs a caller-provided device workspace for its scratch data
// (the gathered sequence-parallel input and, in PARTIALS mode, the float32
// per-shard partial sums).  Some callers cannot provide one: their device
// memory is owned by a memory manager that does not let them allocate at the
// point of the call, or they run in a latency-critical loop where cudaMalloc's
// implicit device-wide synchronisation is not acceptable.  For them,
// tpmlp_forward_noalloc runs the same forward using a fixed scratch area that
// is compiled into this library: a file-scope __device__ array of
// TPMLP_NOALLOC_SCRATCH_BYTES (64 MiB).  Every GPU that loads the library holds
// that array until the process exits; the entry point itself calls no
// cudaMalloc, cudaFree or allocating library routine.
#include <mutex>

#include "internal.h"

namespace tpmlp {
namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(TPMLP_NOALLOC_SCRATCH_BYTES);

// The scratch area.  In host code this name is only a stand-in for the device
// symbol — its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[64] = {};
uint64_t g_scratch_gen[64] = {};  // the device context each address belongs to

// Device address of the scratch array in the current device's context.  The
// lookup runs on the first call in each context of a device — the first call
// on a device, and the first after the caller replaced its context (for
// example by cudaDeviceReset), since an address from a torn-down context must
// never reach a kernel.  Make that first call before any stream capture.
int scratch_address(void** out) {
  DeviceInfo* dev = nullptr;
  int rc = current_device(&dev);
  if (rc != TPMLP_OK) return rc;
  const int d = dev->device;
  if (d < 0 || d >= 64) return set_error(TPMLP_ERR_CUDA, "device ordinal out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[d] == nullptr || g_scratch_gen[d] != dev->generation) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(TPMLP_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
    g_scratch_addr[d] = p;
    g_scratch_gen[d] = dev->generation;
  }
  *out = g_scratch_addr[d];
  return TPMLP_OK;
}

}  // namespace
}  // namespace tpmlp

using namespace tpmlp;

extern "C" int tpmlp_forward_noalloc(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype, int act,
                                     int mode, const void* const* x, const void* w1, const void* w2, void* u, void* y,
                                     void* const* z, void* stream) {
  size_t need = 0;
  int rc = forward_workspace_bytes(s, b, h, f, tp, sp, dtype, act, mode, &need);
  if (rc != TPMLP_OK) return rc;
  if (need > kScratchBytes)
    return set_error(TPMLP_ERR_WORKSPACE,
                     "tpmlp_forward_noalloc: these sizes need " + std::to_string(need) +
                         " bytes of scratch but the built-in scratch holds " + std::to_string(kScratchBytes) +
                         " bytes; call tpmlp_forward with a caller workspace instead");
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != TPMLP_OK) return rc;
  // Nothing in the scratch needs to start at zero: the forward writes every
  // scratch byte it later reads (gathered input, partial sums) in the same call.
  return tpmlp_forward(s, b, h, f, tp, sp, dtype, act, mode, x, w1, w2, u, y, z, scratch, kScratchBytes, stream);
}
