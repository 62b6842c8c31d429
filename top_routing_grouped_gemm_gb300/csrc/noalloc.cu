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

}  // namespace

extern "C" int moe_dispatch_noalloc(const moe_problem* p, const int32_t* topk_idx,
                                    const moe_bf16* x, int32_t* counts, int32_t* offsets,
                                    int32_t* slot_row, int32_t* row_slot,
                                    int32_t* n_kept_dropped, moe_bf16* x_perm,
                                    int32_t* dev_status, moe_stream_t stream) {
  using namespace moe;
  // the same argument rules as moe_dispatch: x_perm is optional (maps only), x is needed
  // only when x_perm is given
  const int st = check_problem(p);
  if (st != MOE_OK) return st;
  if (!topk_idx || !counts || !offsets || !slot_row || !row_slot || !n_kept_dropped)
    return MOE_ERR_INVALID_ARG;
  if (x_perm && !x) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x_perm) & 15u))
    return MOE_ERR_UNSUPPORTED;
  if (dispatch_ws(p) > kNoallocScratchBytes) return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int sa = scratch_address(&scratch);
  if (sa != MOE_OK) return sa;
  // Same carving as the workspace of moe_dispatch.  Both regions are fully written by the
  // counting kernel before they are read, so nothing needs clearing between calls.
  int32_t* local_rank = static_cast<int32_t*>(scratch);
  int32_t* chunk_cnt = reinterpret_cast<int32_t*>(
      static_cast<unsigned char*>(scratch) + up256(static_cast<size_t>(p->T) * p->k * 4));
  mark_before(MOE_KERNEL_DISPATCH, stream);
  const int e = launch_dispatch(topk_idx, reinterpret_cast<const __nv_bfloat16*>(x), p->T, p->d,
                                p->E, p->k, capacity_of(p), counts, offsets, slot_row, row_slot,
                                n_kept_dropped, reinterpret_cast<__nv_bfloat16*>(x_perm),
                                local_rank, chunk_cnt, dev_status, stream);
  mark_after(MOE_KERNEL_DISPATCH, stream);
  count_launches(4);
  return e == 0 ? MOE_OK : MOE_ERR_CUDA;
}
