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
#include <cstdio>
#include <mutex>

#include "msa_internal.h"

namespace msa {
namespace {

constexpr size_t kNoallocScratchBytes = MSA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoallocScratchBytes];

// Device address of the array, looked up once per device with that device
// current.  In host code the symbol itself is only a host-side handle.
constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
cudaError_t g_scratch_err[kMaxDevices] = {};
std::once_flag g_scratch_once[kMaxDevices];

msa_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MSA_ERR_UNSUPPORTED, "device ordinal out of range");
  std::call_once(g_scratch_once[dev], [dev]() {
    void* p = nullptr;
    g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_decode_scratch);
    g_scratch_ptr[dev] = p;
  });
  if (g_scratch_err[dev] != cudaSuccess) return cuda_fail(g_scratch_err[dev], "cudaGetSymbolAddress(decode scratch)");
  if (g_scratch_ptr[dev] == nullptr) return fail(MSA_ERR_CUDA, "decode scratch has no device address");
  *out = g_scratch_ptr[dev];
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
