// qlin_qmv_chain_static: qlin_qmv_chain for callers that cannot allocate
// device memory.
//
// qlin_qmv_chain needs a few hundred bytes of device scratch (one completion
// counter per link) that the caller normally allocates and passes in.  Some
// callers cannot do that: a plugin whose host framework owns every byte of
// device memory through its own pool and does not let extensions call
// cudaMalloc, or a deployment whose device memory budget is fixed at start-up
// with no allocation afterwards.  For them this entry point keeps the scratch
// in a file-scope static device array instead, so a call allocates nothing:
// no cudaMalloc, no cudaFree, no allocating library routine.
//
// Limits and sharing:
//   * at most QLIN_CHAIN_STATIC_MAX_LINKS links per call (the array holds one
//     32-bit counter per link); more is rejected with QLIN_ERR_INVALID_ARG;
//   * every GPU that loads the library holds its own copy of the array until
//     the process exits;
//   * all calls on a device share that one array: each call zeroes the
//     counters it uses on its stream before launching, but two calls whose
//     kernels overlap on the GPU (different streams, or no ordering between
//     them) race on the counters and give wrong results;
//   * the first call on each device looks the array's device address up
//     (cudaGetSymbolAddress, with that device current) and remembers it; make
//     that first call before any stream capture.

#include <mutex>

#include "qlin_internal.h"

namespace {

// counters of the links of one chain call: QLIN_CHAIN_STATIC_MAX_LINKS rounded
// up to the 256-byte workspace granularity of qlin_qmv_chain
constexpr int kStaticWords = (QLIN_CHAIN_STATIC_MAX_LINKS * 4 + 255) / 256 * 256 / 4;
static __device__ __align__(256) unsigned g_chain_static_scratch[kStaticWords];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" qlin_status qlin_qmv_chain_static(const void* x0, const qlin_link* links, int n_links,
                                             int bits, int group_size, qlin_dtype dtype,
                                             void* stream) {
  if (n_links < 1 || n_links > QLIN_CHAIN_STATIC_MAX_LINKS)
    return qlin::fail(QLIN_ERR_INVALID_ARG,
                      "qlin_qmv_chain_static: n_links=%d outside 1..%d (the static scratch holds "
                      "%d link counters)",
                      n_links, QLIN_CHAIN_STATIC_MAX_LINKS, QLIN_CHAIN_STATIC_MAX_LINKS);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return qlin::fail(QLIN_ERR_CUDA, "qlin_qmv_chain_static: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return qlin::fail(QLIN_ERR_UNSUPPORTED, "qlin_qmv_chain_static: device %d", dev);
  void* scratch = nullptr;
  {
    // set-up, once per device, with that device current: the array's name is
    // only a host-side stand-in; the kernel needs its device address
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_chain_static_scratch);
      if (e != cudaSuccess || !p)
        return qlin::fail(QLIN_ERR_CUDA, "qlin_qmv_chain_static: cudaGetSymbolAddress: %s",
                          cudaGetErrorString(e));
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  // the allocating entry point's own validation and launch, on the static
  // scratch (it zeroes the counters on the stream before launching)
  return qlin_qmv_chain(x0, links, n_links, bits, group_size, dtype, scratch,
                        sizeof(g_chain_static_scratch), stream);
}
