// msa_internal.h -- host-side plumbing shared by the MSA entry points and the
// kernel launchers: error text, device properties, tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "msa.h"

namespace msa {

// Thread-local last-error text; returns `st` for convenience.
msa_status fail(msa_status st, const std::string& why);
msa_status cuda_fail(cudaError_t e, const char* what);

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  size_t max_smem_optin = 0;
};
// Properties of the current device (cached per device).
msa_status current_device(DeviceInfo* info);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
// dims/strides in elements / bytes as the driver API expects: strides_bytes has rank-1 entries.
msa_status encode_tiled_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                            const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                            CUtensorMapSwizzle swizzle, const char* what);

// Launchers (validated arguments only).
msa_status launch_index_decode(const msa_index_args& a, cudaStream_t stream);
// Chunk scoring of S <= kChunkDecodeMaxS tokens per sequence over per-group
// index keys through the decode index kernel (B rows = the tokens' heads);
// index_chunk_tokens_ok tells whether a validated chunk call qualifies.
bool index_chunk_tokens_ok(const msa_index_args& a);
msa_status launch_index_chunk_tokens(const msa_index_args& a, cudaStream_t stream);
msa_status launch_index_prefill(const msa_index_args& a, cudaStream_t stream);
msa_status launch_topk(const msa_topk_args& a, cudaStream_t stream);
msa_status launch_page_table(const int32_t* sel, const int32_t* count, const int32_t* seq_pt,
                             int64_t max_pages, const int32_t* seq_len, int B, int Hkv, int k, int Bk,
                             int32_t* pt, int32_t* n, int32_t* last_len, int32_t* dev_err,
                             cudaStream_t stream, int S = 1, const int32_t* q_pos = nullptr);
msa_status launch_attn_decode(const msa_decode_args& a, float* o_part, float* lse_part, int32_t* counter,
                              cudaStream_t stream);
msa_status launch_lse_merge(const float* o_part, const float* lse_part, int64_t rows, int parts, int D,
                            void* O, float* LSE, int32_t* dev_err, cudaStream_t stream);
msa_status launch_lse_merge_bf16(const __nv_bfloat16* o_part, const float* lse_part, int64_t rows, int parts, int D,
                                 __nv_bfloat16* O, float* LSE, cudaStream_t stream);
msa_status launch_attn_prefill(const msa_prefill_args& a, void* ws, size_t ws_bytes, cudaStream_t stream);
msa_status launch_cache_append(const msa_append_args& a, cudaStream_t stream);
msa_status launch_dense_decode(const msa_dense_decode_args& a, void* ws, size_t ws_bytes, cudaStream_t stream);
size_t dense_decode_workspace_size(const msa_dense_decode_args& a);
msa_status launch_dense_prefill(const msa_dense_prefill_args& a, cudaStream_t stream);
// Host-side argument checks of msa_sparse_attn_decode (no CUDA call).
msa_status check_decode_args(const msa_decode_args* a);
size_t attn_prefill_workspace_size(const msa_prefill_args& a, int64_t chunk_queries);

constexpr int kBk = 128;
constexpr int kD = 128;
constexpr int kDI = 64;
constexpr int kMaxK = 64;
constexpr int kMaxHI = 4;
constexpr int kMaxG = 8;
constexpr int kMaxDecodeBatch = 4096;
constexpr int kChunkDecodeMaxS = 8;   // chunk attention through the decode kernel for S <= this
constexpr int kDenseMaxBatch = 1024;   // dense comparator: sequences per call
constexpr int kDenseMaxGrid = 256;     // dense decode: CTAs per launch (at most)

}  // namespace msa
