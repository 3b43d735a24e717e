// kvq_noalloc.cu -- kvq_decode_noalloc: the decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at decode time: a serving loop whose memory is fully reserved
// up front (any allocation there can fail or stall on a synchronising free), a plugin that runs
// inside another framework's allocator and must not take memory behind its back, or code that has
// no allocator handle at all.  They still own q, the pool and out, but cannot provide the split-K
// scratch that kvq_decode takes as `workspace`.  This entry point uses a fixed scratch array that
// lives in the library's own device memory instead.
//
// The scratch is a file-scope __device__ array of KVQ_NOALLOC_SCRATCH_BYTES.  Every GPU that loads
// the library keeps it until the process exits.  Host code cannot use the array's name as a device
// address (in host code it is only a host-side shadow symbol), so the first call on each device
// asks the runtime for the real address with cudaGetSymbolAddress, with that device current, and
// caches it.  All calls share the one array and it keeps the last call's contents: the status word
// and the split counters are cleared on every call (kvq_decode does that), and the split partials are
// always written before they are read.  Calls whose kernels overlap on the GPU (different streams, or different host
// threads without ordering) race on the array and give wrong results.
//
// The status word a decode leaves (a timed-out bounded wait, a block-table entry past the pool) lives in
// that array too, where the caller has no pointer to it; kvq_noalloc_status reads it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kvq.h"
#include "kvq_internal.h"

namespace kvq {
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
kvq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVQ_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return KVQ_ECUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return KVQ_OK;
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kvq_decode_noalloc(const void* q, const void* pool, const void* scales,
                                         const int32_t* block_table, int32_t max_pages_per_seq,
                                         const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                         float sm_scale, void* out, kvq_out_dtype out_dtype,
                                         const kvq_layout* layout, kvq_kind kind, void* stream) {
  const size_t need = kvq_decode_workspace_bytes(layout, batch, num_q_heads, max_pages_per_seq);
  if (need == 0) return KVQ_EINVAL;
  if (need > static_cast<size_t>(KVQ_NOALLOC_SCRATCH_BYTES)) return KVQ_EWORKSPACE;
  kvq_status st = kvq_device_check();
  if (st != KVQ_OK) return st;
  void* scratch = nullptr;
  st = kvq::scratch_address(&scratch);
  if (st != KVQ_OK) return st;
  return kvq_decode(q, pool, scales, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale, out,
                    out_dtype, scratch, static_cast<size_t>(KVQ_NOALLOC_SCRATCH_BYTES), layout, kind, stream);
}

extern "C" kvq_status kvq_noalloc_status(void* stream) {
  void* scratch = nullptr;
  const kvq_status st = kvq::scratch_address(&scratch);
  if (st != KVQ_OK) return st;
  return kvq_workspace_status(scratch, stream);
}
