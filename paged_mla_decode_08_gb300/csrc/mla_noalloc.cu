// mla_decode_noalloc: mla_decode with the library's own, fixed scratch.
//
// Who needs this.  mla_decode wants a caller-provided device workspace for
// the per-split partial results.  Some callers cannot obtain one: code that
// runs where allocating is not allowed or not wanted, e.g. a plugin that is
// handed only its input and output buffers by a host framework with its own
// memory manager, an allocation-free real-time or safety-checked serving loop,
// or a process whose memory is fully reserved up front.  For them this entry
// point takes the same inputs and outputs and uses a scratch array that lives
// in this file as a statically sized __device__ variable instead.
//
// Cost and limits.
//  - The array is MLA_NOALLOC_SCRATCH_BYTES (16 MiB: 127 split slots of 128
//    query rows with bf16 partials).  It is part of the
//    library's device image, so a device holds it from the moment this code is
//    loaded on it until the process exits.
//  - A plan whose workspace size exceeds the array is rejected with
//    MLA_ERR_WORKSPACE; use mla_decode with a larger caller buffer then.
//  - One array per device, shared by every call on that device.  It keeps
//    whatever the previous call left there; the decode reads nothing from it
//    that the same call did not write first, so no clearing is needed.  Calls
//    whose work overlaps on the GPU (different streams without ordering, or
//    several host threads) race on it and give wrong results: order them.
//  - The array's device address is looked up with cudaGetSymbolAddress, with
//    the device current, the first time a call runs under a given CUDA
//    context, and cached under that context's unique id (cuCtxGetId).  A
//    context made after cudaDeviceReset, or any other context, has another
//    id, so its first call looks the address up again instead of using a
//    dead one.  The first call in a context may load the library's module
//    there: make it before capturing the stream into a CUDA graph.
//  - Nothing here allocates: no cudaMalloc / cudaFree, no allocating library
//    routine.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mla_decode.h"
#include "mla_internal.h"

namespace mla {
int report_error(int code, const char* msg);
int require_sm103();
}

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
  static DriverFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return f;
}

// Unique id of the current context (never reused within the process), or 0.
unsigned long long current_context_id() {
  const DriverFns& f = driver_fns();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!f.get_current || !f.get_id || f.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// (context id, scratch address) pairs already looked up; a small ring
struct CacheEntry {
  unsigned long long ctx_id;
  void* ptr;
};
constexpr int kCacheEntries = 16;
std::mutex g_mu;
CacheEntry g_cache[kCacheEntries];
int g_next = 0;

// Device address of the scratch array in the current context, or nullptr
// with the error recorded.
void* scratch_address(int* rc) {
  const unsigned long long id = current_context_id();
  if (id != 0) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (const CacheEntry& e : g_cache)
      if (e.ctx_id == id) {
        *rc = MLA_OK;
        return e.ptr;
      }
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    *rc = mla::report_error(MLA_ERR_CUDA, "mla_decode_noalloc: cudaGetSymbolAddress of the scratch failed");
    return nullptr;
  }
  // the lookup made the runtime's context current if none was: cache under it
  const unsigned long long id_now = id != 0 ? id : current_context_id();
  if (id_now != 0) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_cache[g_next] = CacheEntry{id_now, p};
    g_next = (g_next + 1) % kCacheEntries;
  }
  *rc = MLA_OK;
  return p;
}

}  // namespace

extern "C" int mla_decode_noalloc(const mla_plan* plan, const void* q_nope, const void* q_pe, int num_tokens,
                                  int num_heads, const void* kv_pages, int kv_dtype, int64_t num_pages,
                                  int page_size, const int32_t* block_table, int bt_stride,
                                  const int32_t* seq_lens, float scale, float k_scale, void* out, float* lse,
                                  void* stream) {
  if (!plan) return mla::report_error(MLA_ERR_ARG, "plan is NULL");
  const int dev_rc = mla::require_sm103();  // before any lookup: a wrong device is MLA_ERR_UNSUPPORTED
  if (dev_rc != MLA_OK) return dev_rc;
  if (mla_plan_workspace_bytes(plan) > (size_t)MLA_NOALLOC_SCRATCH_BYTES)
    return mla::report_error(MLA_ERR_WORKSPACE,
                             "mla_decode_noalloc: the plan needs more scratch than the built-in 16 MiB "
                             "(mla_plan_workspace_bytes); call mla_decode with a caller workspace instead");
  int rc = MLA_OK;
  void* ws = scratch_address(&rc);
  if (!ws) return rc;
  return mla_decode(plan, q_nope, q_pe, num_tokens, num_heads, kv_pages, kv_dtype, num_pages, page_size,
                    block_table, bt_stride, seq_lens, scale, k_scale, out, lse, ws,
                    (size_t)MLA_NOALLOC_SCRATCH_BYTES, stream);
}
