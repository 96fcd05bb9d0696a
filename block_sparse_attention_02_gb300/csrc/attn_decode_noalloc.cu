// attn_decode_noalloc.cu -- paged decode attention for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// that runs inside a serving loop whose allocator is frozen after start-up,
// plugins of a host framework that owns every device allocation, or hooks that
// run where an allocation could synchronise the device.  This entry point
// runs the same kernels as msa_sparse_attn_decode, but its scratch (the
// per-split partial outputs and log-sum-exps) lives in one fixed array in
// device global memory that is part of the library image, so the call
// allocates nothing.
//
// The array is kNoallocScratchBytes large and stays resident on every device
// that loads the library until the process exits.  All calls share it: two
// calls whose kernels overlap on the GPU (different streams, or several host
// threads) race on it and must be serialised by the caller.  Each call clears
// the per-row counters it uses (cudaMemsetAsync) and writes every partial that
// the merge reads before reading it.
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "msa_internal.h"

namespace msa {
namespace {

constexpr size_t kNoallocScratchBytes = MSA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoallocScratchBytes];

// Device address of the array.  In host code the symbol itself is only a
// host-side handle; the device address comes from cudaGetSymbolAddress with
// the device current, and belongs to that device's current context.  It is
// looked up once per context: the cache entry of a device remembers the
// unique id of the context it was taken in (cuCtxGetId), so a context that was
// destroyed and created again (cudaDeviceReset) gets a fresh lookup instead of
// a stale address.  A failed lookup is not remembered: the next call tries
// again.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

constexpr int kMaxDevices = 64;
struct ScratchEntry {
  unsigned long long ctx_id = 0;   // 0: nothing cached
  void* ptr = nullptr;
};
ScratchEntry g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_fn_once;

// Unique id of the calling thread's current context, or 0 when there is none
// yet or the driver cannot say.
unsigned long long current_context_id() {
  std::call_once(g_ctx_fn_once, []() {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

msa_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MSA_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = current_context_id();
  if (id != 0 && g_scratch[dev].ctx_id == id) {
    *out = g_scratch[dev].ptr;
    return MSA_OK;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_decode_scratch);   // initialises the context if needed
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
  if (p == nullptr) return fail(MSA_ERR_CUDA, "decode scratch has no device address");
  // the context the address belongs to (now current, if the lookup created it)
  g_scratch[dev].ctx_id = current_context_id();
  g_scratch[dev].ptr = p;
  *out = p;
  return MSA_OK;
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_sparse_attn_decode_noalloc(const msa_decode_args* a, msa_stream_t stream) {
  // the checks of msa_sparse_attn_decode run first, before any CUDA call
  if (msa_status st = check_decode_args(a); st != MSA_OK) return st;
  const size_t need = msa_sparse_attn_decode_workspace_size(a);
  if (need > kNoallocScratchBytes) {
    char buf[256];
    std::snprintf(buf, sizeof(buf),
                  "decode needs %zu bytes of scratch (B*Hq*k*(D+1)*4 + B*Hkv*4 + 256) but the built-in array holds %zu; "
                  "use msa_sparse_attn_decode with a workspace",
                  need, kNoallocScratchBytes);
    return fail(MSA_ERR_WORKSPACE, buf);
  }
  void* scratch = nullptr;
  if (msa_status st = scratch_address(&scratch); st != MSA_OK) return st;
  // the shared array serves calls of every shape, so its counters are always cleared
  msa_decode_args cleared = *a;
  cleared.scratch_zeroed = 0;
  return msa_sparse_attn_decode(&cleared, scratch, kNoallocScratchBytes, stream);
}
