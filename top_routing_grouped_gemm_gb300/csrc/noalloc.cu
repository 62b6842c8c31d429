// moe_dispatch_noalloc: the dispatch step with its scratch memory built into the library.
//
// Some callers cannot hand the library a workspace: code that runs where the device memory
// is entirely owned by another allocator (a framework's caching pool that must not be
// bypassed, or a reservation that is already exhausted), and plugins that are given tensor
// pointers but no way to call cudaMalloc at all.  For them this entry point uses a fixed,
// file-scope device array as the dispatch scratch (per-slot ranks and per-chunk counts)
// instead of a caller workspace.  The array is part of the library image: every GPU that
// loads the library holds kNoallocScratchBytes of device memory for it until the process
// exits.
#include <mutex>

#include "moe_internal.h"
#include "route.h"

namespace {

constexpr size_t kNoallocScratchBytes = 8u << 20;  // 8 MiB

__device__ __align__(256) unsigned char g_dispatch_scratch[kNoallocScratchBytes];

// Device address of g_dispatch_scratch on the current device.  In host code the array's
// name is only a host-side stand-in, so the address is looked up once per device, with that
// device current, and cached.
int scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return MOE_OK;
}

inline size_t up256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

}  // namespace

extern "C" int moe_dispatch_noalloc(const moe_problem* p, const int32_t* topk_idx,
                                    const moe_bf16* x, int32_t* counts, int32_t* offsets,
                                    int32_t* slot_row, int32_t* row_slot,
                                    int32_t* n_kept_dropped, moe_bf16* x_perm,
                                    int32_t* dev_status, moe_stream_t stream) {
  using namespace moe;
  const size_t need = moe_dispatch_workspace_size(p);
  if (need == 0) return p == nullptr ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED;
  if (need > kNoallocScratchBytes) return MOE_ERR_WORKSPACE;
  if (!topk_idx || !x || !counts || !offsets || !slot_row || !row_slot || !n_kept_dropped ||
      !x_perm)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x_perm) & 15u))
    return MOE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  // Same carving as the workspace of moe_dispatch.  Both regions are fully written by the
  // counting kernel before they are read, so nothing needs clearing between calls.
  int32_t* local_rank = static_cast<int32_t*>(scratch);
  int32_t* chunk_cnt = reinterpret_cast<int32_t*>(
      static_cast<unsigned char*>(scratch) + up256(static_cast<size_t>(p->T) * p->k * 4));
  int capacity = -1;  // ceil(cf * T * k / E), as moe_dispatch computes it
  if (p->cap_den != 0) {
    const long long num = static_cast<long long>(p->cap_num) * p->T * p->k;
    const long long den = static_cast<long long>(p->cap_den) * p->E;
    const long long c = (num + den - 1) / den;
    capacity = c > (1ll << 30) ? (1 << 30) : static_cast<int>(c);
  }
  const int e = launch_dispatch(topk_idx, reinterpret_cast<const __nv_bfloat16*>(x), p->T, p->d,
                                p->E, p->k, capacity, counts, offsets, slot_row, row_slot,
                                n_kept_dropped, reinterpret_cast<__nv_bfloat16*>(x_perm),
                                local_rank, chunk_cnt, dev_status, stream);
  return e == 0 ? MOE_OK : MOE_ERR_CUDA;
}
