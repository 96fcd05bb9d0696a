// Prefill kernels are not built yet; the entry points report it.
#include "msa_internal.h"

namespace msa {
msa_status launch_index_prefill(const msa_index_args&, cudaStream_t) {
  return fail(MSA_ERR_UNSUPPORTED, "prefill index score is not built in this library");
}
msa_status launch_attn_prefill(const msa_prefill_args&, void*, size_t, cudaStream_t) {
  return fail(MSA_ERR_UNSUPPORTED, "prefill sparse attention is not built in this library");
}
size_t attn_prefill_workspace_size(const msa_prefill_args&, int64_t) { return 256; }
}  // namespace msa
