// kvq_static.cu — kvq_decode_static: the INT2 decode step without a
// caller-supplied workspace.
//
// kvq_decode needs a workspace (rotated queries and split-K partials) that the
// caller allocates.  Some callers cannot do that: an integration whose
// attention-op signature has no workspace argument, or a serving process that
// reserves all device memory at start-up and forbids allocation on the decode
// path.  This entry point gives them the same computation with the scratch
// taken from one fixed array in device global memory that lives as long as the
// library is loaded.  It allocates nothing itself.
#include <stdint.h>

#include <atomic>

#include "kvq_internal.cuh"

namespace {

// Fixed scratch: every GPU that loads the library holds these bytes until the
// process exits.
constexpr size_t kStaticWsBytes = static_cast<size_t>(16) << 20;   // 16 MiB
static __device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_ws_addr[kMaxDevices] = {};

// Device address of g_static_ws on `dev` (current device), looked up once per
// device.  Threads that race on the first call all look up the same address
// and store the same value, so a relaxed load and store suffice.
int static_ws_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ECUDA;
  void* p = g_ws_addr[dev].load(std::memory_order_relaxed);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return KVQ_ECUDA;
    g_ws_addr[dev].store(p, std::memory_order_relaxed);
  }
  *out = p;
  return KVQ_OK;
}

}  // namespace

extern "C" int kvq_decode_static(kvq_handle* h, const void* pool, int num_pool_pages,
                                 const uint16_t* q, const int32_t* page_table, int max_pages,
                                 const int32_t* seq_lens, int batch, float* out, int num_splits,
                                 void* stream) {
  if (!h || batch < 1 || max_pages < 1 || num_splits < 0 || num_splits > kvq::kMaxSplits)
    return KVQ_EINVAL;
  int splits = num_splits;
  if (splits == 0) {
    // the automatic choice, lowered until its scratch fits the fixed array
    splits = kvq_auto_splits(h, batch, max_pages);
    while (splits > 1 && kvq_workspace_bytes(h, batch, splits) > kStaticWsBytes) --splits;
  }
  const size_t need = kvq_workspace_bytes(h, batch, splits);
  if (need == 0) return KVQ_EINVAL;
  if (need > kStaticWsBytes) return KVQ_ENOSPACE;   // batch x splits too large for 16 MiB
  // the symbol's address is per device: look it up with the handle's device current
  const int dev = kvq::handle_device(h);
  kvq::DeviceGuard dev_guard(dev);
  if (!dev_guard.ok()) return KVQ_ECUDA;
  void* ws = nullptr;
  const int rc = static_ws_address(dev, &ws);
  if (rc != KVQ_OK) return rc;
  return kvq_decode(h, pool, num_pool_pages, q, page_table, max_pages, seq_lens, batch, out, ws,
                    kStaticWsBytes, splits, stream);
}
