// api.cu -- the extern "C" entry points of libmsa: argument validation, error
// reporting and the sequence of kernel launches behind each call.
//
// Every check below runs on the host before anything touches the device, so a
// rejected call enqueues nothing.
#include <cudaTypedefs.h>

#include <cinttypes>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <string>

#include "msa_internal.h"

namespace msa {

namespace {
thread_local std::string g_last_error;

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;
}  // namespace

msa_status fail(msa_status st, const std::string& why) {
  g_last_error = why;
  return st;
}

msa_status cuda_fail(cudaError_t e, const char* what) {
  char buf[512];
  std::snprintf(buf, sizeof(buf), "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
  g_last_error = buf;
  return MSA_ERR_CUDA;
}

msa_status current_device(DeviceInfo* info) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MSA_ERR_UNSUPPORTED, "device ordinal out of range");
  cudaError_t init_err = cudaSuccess;
  std::call_once(g_dev_once[dev], [&]() {
    DeviceInfo d;
    d.device = dev;
    int v = 0;
    init_err = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    d.num_sms = v;
    if (init_err == cudaSuccess) init_err = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    d.max_smem_optin = static_cast<size_t>(v);
    if (init_err == cudaSuccess) g_dev[dev] = d;
  });
  if (init_err != cudaSuccess) return cuda_fail(init_err, "cudaDeviceGetAttribute");
  if (g_dev[dev].num_sms <= 0) return fail(MSA_ERR_CUDA, "device properties unavailable");
  *info = g_dev[dev];
  return MSA_OK;
}

msa_status encode_tiled_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                            const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                            CUtensorMapSwizzle swizzle, const char* what) {
  std::call_once(g_encode_once, []() {
    cudaDriverEntryPointQueryResult q;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&g_encode),
                                                    12000, cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess) g_encode = nullptr;
  });
  if (g_encode == nullptr) {
    if (g_encode_err != cudaSuccess) return cuda_fail(g_encode_err, "cuTensorMapEncodeTiled entry point");
    return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
  }
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[256];
    std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed for %s (CUresult %d)", what, static_cast<int>(r));
    return fail(MSA_ERR_INVALID_ARG, buf);
  }
  return MSA_OK;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A leading-dimension stride (elements) usable by TMA / 16-byte vector loads.
bool vec_stride_ok(int64_t s, int elem_bytes) {
  return s > 0 && (s * elem_bytes) % 16 == 0 && s * elem_bytes < (int64_t(1) << 40);
}

#define MSA_REQUIRE(cond, st, ...)                          \
  do {                                                      \
    if (!(cond)) {                                          \
      char _buf[384];                                       \
      std::snprintf(_buf, sizeof(_buf), __VA_ARGS__);       \
      return ::msa::fail(st, _buf);                         \
    }                                                       \
  } while (0)

msa_status check_common_shape(int Bk, int dI_or_D, int want, const char* name) {
  MSA_REQUIRE(Bk == kBk, MSA_ERR_UNSUPPORTED, "Bk = %d, only %d is supported", Bk, kBk);
  MSA_REQUIRE(dI_or_D == want, MSA_ERR_UNSUPPORTED, "%s = %d, only %d is supported", name, dI_or_D, want);
  return MSA_OK;
}

}  // namespace
}  // namespace msa

using namespace msa;

msa_status msa::check_decode_args(const msa_decode_args* a) {
  MSA_REQUIRE(a != nullptr, MSA_ERR_INVALID_ARG, "args is NULL");
  MSA_REQUIRE(a->B >= 0 && a->Hkv >= 1 && a->Hq >= 1, MSA_ERR_INVALID_ARG, "B = %d, Hq = %d, Hkv = %d", a->B, a->Hq,
              a->Hkv);
  MSA_REQUIRE(a->Hq % a->Hkv == 0 && a->Hq / a->Hkv <= kMaxG, MSA_ERR_UNSUPPORTED,
              "GQA ratio Hq/Hkv = %d/%d not in 1..%d", a->Hq, a->Hkv, kMaxG);
  if (msa_status st = check_common_shape(a->Bk, a->D, kD, "D"); st != MSA_OK) return st;
  MSA_REQUIRE(a->k >= 1 && a->k <= kMaxK, MSA_ERR_UNSUPPORTED, "k = %d, supported 1..%d", a->k, kMaxK);
  MSA_REQUIRE(a->Q && a->K_pool && a->V_pool && a->pt && a->n && a->last_len && a->O, MSA_ERR_INVALID_ARG,
              "Q, K_pool, V_pool, pt, n, last_len and O must be non-NULL");
  MSA_REQUIRE(aligned16(a->Q) && aligned16(a->K_pool) && aligned16(a->V_pool) && aligned16(a->O), MSA_ERR_INVALID_ARG,
              "Q, K_pool, V_pool and O must be 16-byte aligned");
  MSA_REQUIRE(a->num_pages >= 1 && a->num_pages < (int64_t(1) << 31), MSA_ERR_INVALID_ARG, "num_pages = %" PRId64,
              a->num_pages);
  for (int i = 0; i < 2; ++i)
    MSA_REQUIRE(vec_stride_ok(a->Q_stride[i], 2), MSA_ERR_INVALID_ARG,
                "Q_stride[%d] = %" PRId64 " must be a positive multiple of 8 elements", i, a->Q_stride[i]);
  for (int i = 0; i < 3; ++i)
    MSA_REQUIRE(vec_stride_ok(a->kv_stride[i], 2), MSA_ERR_INVALID_ARG,
                "kv_stride[%d] = %" PRId64 " must be a positive multiple of 8 elements", i, a->kv_stride[i]);
  return MSA_OK;
}

extern "C" {

int msa_version(void) { return 100; }

const char* msa_last_error_string(void) { return g_last_error.c_str(); }

const char* msa_status_string(msa_status s) {
  switch (s) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
    case MSA_ERR_DEVICE_CHECK: return "MSA_ERR_DEVICE_CHECK";
    case MSA_ERR_WORKSPACE: return "MSA_ERR_WORKSPACE";
  }
  return "MSA_ERR_UNKNOWN";
}

// ---------------------------------------------------------------------------
msa_status msa_index_score(const msa_index_args* a, msa_stream_t stream) {
  g_last_error.clear();
  MSA_REQUIRE(a != nullptr, MSA_ERR_INVALID_ARG, "args is NULL");
  MSA_REQUIRE(a->mode == MSA_MODE_PREFILL || a->mode == MSA_MODE_DECODE || a->mode == MSA_MODE_CHUNK,
              MSA_ERR_INVALID_ARG, "bad mode %d", static_cast<int>(a->mode));
  MSA_REQUIRE(a->B >= 0 && a->Hkv >= 1, MSA_ERR_INVALID_ARG, "B = %d, Hkv = %d", a->B, a->Hkv);
  if (msa_status st = check_common_shape(a->Bk, a->dI, kDI, "dI"); st != MSA_OK) return st;
  MSA_REQUIRE(a->HI >= 1 && a->HI <= kMaxHI, MSA_ERR_UNSUPPORTED, "HI = %d, supported 1..%d", a->HI, kMaxHI);
  MSA_REQUIRE(a->nb_stride >= 1, MSA_ERR_INVALID_ARG, "nb_stride = %d", a->nb_stride);
  MSA_REQUIRE(a->q_idx && a->w && a->k_idx && a->C, MSA_ERR_INVALID_ARG, "q_idx, w, k_idx and C must be non-NULL");
  MSA_REQUIRE(aligned16(a->q_idx) && aligned16(a->k_idx), MSA_ERR_INVALID_ARG,
              "q_idx and k_idx must be 16-byte aligned");
  if (a->mode == MSA_MODE_PREFILL || a->mode == MSA_MODE_CHUNK) {
    const bool chunk = a->mode == MSA_MODE_CHUNK;
    MSA_REQUIRE(a->S >= 0, MSA_ERR_INVALID_ARG, "S = %d", a->S);
    MSA_REQUIRE(a->nb_stride >= (a->S + a->Bk - 1) / a->Bk, MSA_ERR_INVALID_ARG, "nb_stride %d < ceil(S/Bk) = %d",
                a->nb_stride, (a->S + a->Bk - 1) / a->Bk);
    for (int i = 0; i < 4; ++i)
      MSA_REQUIRE(vec_stride_ok(a->q_idx_stride[i], 2), MSA_ERR_INVALID_ARG,
                  "q_idx_stride[%d] = %" PRId64 " must be a positive multiple of 8 elements", i, a->q_idx_stride[i]);
    // strides (b, s, g), or (page, g, t) for a chunk's page pool; a group
    // stride of 0: one index-key tensor for all KV groups
    const int gi = chunk ? 1 : 2;
    for (int i = 0; i < 3; ++i)
      MSA_REQUIRE(vec_stride_ok(a->k_idx_stride[i], 2) || (i == gi && a->k_idx_stride[i] == 0), MSA_ERR_INVALID_ARG,
                  "k_idx_stride[%d] = %" PRId64 " must be a positive multiple of 8 elements", i, a->k_idx_stride[i]);
    if (chunk) {
      MSA_REQUIRE(a->seq_pt && a->q_pos, MSA_ERR_INVALID_ARG, "chunk: seq_pt and q_pos must be non-NULL");
      MSA_REQUIRE(a->num_pages >= 1 && a->num_pages < (int64_t(1) << 31), MSA_ERR_INVALID_ARG,
                  "num_pages = %" PRId64, a->num_pages);
      MSA_REQUIRE(a->max_pages >= 1 && a->max_pages < (int64_t(1) << 31) / a->Bk, MSA_ERR_INVALID_ARG,
                  "max_pages = %" PRId64, a->max_pages);
      // no block lies past the page table, and with this bound the index score
      // and the top-k reject exactly the same sequences (a last own block at
      // or past nb_stride)
      MSA_REQUIRE(a->nb_stride <= a->max_pages, MSA_ERR_INVALID_ARG,
                  "chunk: nb_stride = %d exceeds max_pages = %" PRId64, a->nb_stride, a->max_pages);
    }
    for (int i = 0; i < 3; ++i)
      MSA_REQUIRE(a->w_stride[i] > 0 && a->C_stride[i] > 0, MSA_ERR_INVALID_ARG, "w / C strides must be positive");
    if (static_cast<int64_t>(a->B) * a->S == 0) return MSA_OK;
    return launch_index_prefill(*a, reinterpret_cast<cudaStream_t>(stream));
  }
  // decode
  MSA_REQUIRE(a->B <= kMaxDecodeBatch, MSA_ERR_UNSUPPORTED, "decode batch %d > %d", a->B, kMaxDecodeBatch);
  MSA_REQUIRE(a->seq_pt && a->seq_len, MSA_ERR_INVALID_ARG, "seq_pt and seq_len must be non-NULL");
  MSA_REQUIRE(a->num_pages >= 1 && a->num_pages < (int64_t(1) << 31), MSA_ERR_INVALID_ARG,
              "num_pages = %" PRId64, a->num_pages);
  MSA_REQUIRE(a->max_pages >= 1 && a->max_pages < (int64_t(1) << 31) / a->Bk, MSA_ERR_INVALID_ARG,
              "max_pages = %" PRId64, a->max_pages);
  for (int i = 0; i < 3; ++i) {
    // a group stride of 0: one index-key pool shared by all KV groups
    MSA_REQUIRE(vec_stride_ok(a->k_idx_stride[i], 2) || (i == 1 && a->k_idx_stride[i] == 0), MSA_ERR_INVALID_ARG,
                "k_idx_stride[%d] = %" PRId64 " must be a positive multiple of 8 elements", i, a->k_idx_stride[i]);
    MSA_REQUIRE(i == 2 || vec_stride_ok(a->q_idx_stride[i], 2), MSA_ERR_INVALID_ARG,
                "q_idx_stride[%d] = %" PRId64 " must be a positive multiple of 8 elements", i, a->q_idx_stride[i]);
  }
  MSA_REQUIRE(a->w_stride[0] > 0 && a->w_stride[1] > 0 && a->C_stride[0] > 0 && a->C_stride[1] > 0,
              MSA_ERR_INVALID_ARG, "w / C strides must be positive");
  if (a->sel != nullptr) {
    MSA_REQUIRE(a->k >= 1 && a->k <= kMaxK, MSA_ERR_UNSUPPORTED, "fused selection: k = %d, supported 1..%d", a->k,
                kMaxK);
    MSA_REQUIRE(a->count != nullptr && a->row_scratch != nullptr, MSA_ERR_INVALID_ARG,
                "fused selection needs count and row_scratch");
    MSA_REQUIRE(a->pt == nullptr || (a->n != nullptr && a->last_len != nullptr), MSA_ERR_INVALID_ARG,
                "fused page table needs n and last_len");
  }
  if (a->B == 0) return MSA_OK;
  return launch_index_decode(*a, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
msa_status msa_topk_blocks(const msa_topk_args* a, msa_stream_t stream) {
  g_last_error.clear();
  MSA_REQUIRE(a != nullptr, MSA_ERR_INVALID_ARG, "args is NULL");
  MSA_REQUIRE(a->mode == MSA_MODE_PREFILL || a->mode == MSA_MODE_DECODE || a->mode == MSA_MODE_CHUNK,
              MSA_ERR_INVALID_ARG, "bad mode");
  MSA_REQUIRE(a->Bk == kBk, MSA_ERR_UNSUPPORTED, "Bk = %d, only %d is supported", a->Bk, kBk);
  MSA_REQUIRE(a->k >= 1 && a->k <= kMaxK, MSA_ERR_UNSUPPORTED, "k = %d, supported 1..%d", a->k, kMaxK);
  MSA_REQUIRE(a->B >= 0 && a->Hkv >= 1 && a->nb_stride >= 1, MSA_ERR_INVALID_ARG, "B = %d, Hkv = %d, nb_stride = %d",
              a->B, a->Hkv, a->nb_stride);
  MSA_REQUIRE(a->C && a->sel && a->count, MSA_ERR_INVALID_ARG, "C, sel and count must be non-NULL");
  MSA_REQUIRE(a->C_stride[0] > 0 && a->C_stride[1] > 0, MSA_ERR_INVALID_ARG, "C strides must be positive");
  if (a->mode == MSA_MODE_PREFILL) {
    MSA_REQUIRE(a->S >= 0, MSA_ERR_INVALID_ARG, "S = %d", a->S);
    MSA_REQUIRE(a->C_stride[2] > 0, MSA_ERR_INVALID_ARG, "C strides must be positive");
    MSA_REQUIRE(a->nb_stride >= (a->S + a->Bk - 1) / a->Bk, MSA_ERR_INVALID_ARG, "nb_stride < ceil(S/Bk)");
    MSA_REQUIRE((a->S - 1) / a->Bk < 2048, MSA_ERR_UNSUPPORTED, "prefill rows with more than 2048 blocks");
  } else if (a->mode == MSA_MODE_CHUNK) {
    MSA_REQUIRE(a->S >= 0, MSA_ERR_INVALID_ARG, "S = %d", a->S);
    MSA_REQUIRE(a->C_stride[2] > 0, MSA_ERR_INVALID_ARG, "C strides must be positive");
    MSA_REQUIRE(a->q_pos != nullptr, MSA_ERR_INVALID_ARG, "q_pos must be non-NULL in chunk mode");
  } else {
    MSA_REQUIRE(a->seq_len != nullptr, MSA_ERR_INVALID_ARG, "seq_len must be non-NULL in decode");
  }
  return launch_topk(*a, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
msa_status msa_build_page_table(const int32_t* sel, const int32_t* count, const int32_t* seq_pt, int64_t max_pages,
                                const int32_t* seq_len, int B, int Hkv, int k, int Bk, int32_t* pt, int32_t* n,
                                int32_t* last_len, int32_t* dev_err, msa_stream_t stream) {
  g_last_error.clear();
  MSA_REQUIRE(B >= 0 && Hkv >= 1, MSA_ERR_INVALID_ARG, "B = %d, Hkv = %d", B, Hkv);
  MSA_REQUIRE(k >= 1 && k <= kMaxK, MSA_ERR_UNSUPPORTED, "k = %d, supported 1..%d", k, kMaxK);
  MSA_REQUIRE(Bk == kBk, MSA_ERR_UNSUPPORTED, "Bk = %d, only %d is supported", Bk, kBk);
  MSA_REQUIRE(max_pages >= 1, MSA_ERR_INVALID_ARG, "max_pages = %" PRId64, max_pages);
  MSA_REQUIRE(sel && count && seq_pt && seq_len && pt && n && last_len, MSA_ERR_INVALID_ARG,
              "all array arguments must be non-NULL");
  return launch_page_table(sel, count, seq_pt, max_pages, seq_len, B, Hkv, k, Bk, pt, n, last_len, dev_err,
                           reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------

size_t msa_sparse_attn_decode_workspace_size(const msa_decode_args* a) {
  if (a == nullptr || a->B < 0 || a->Hq < 1 || a->k < 1 || a->D < 1) return 0;
  const size_t parts = static_cast<size_t>(a->B) * a->Hq * a->k;
  const size_t rows = static_cast<size_t>(a->B) * (a->Hkv > 0 ? a->Hkv : 1);
  return parts * static_cast<size_t>(a->D) * 4 + parts * 4 + rows * 4 + 256;
}

msa_status msa_sparse_attn_decode(const msa_decode_args* a, void* ws, size_t ws_bytes, msa_stream_t stream) {
  g_last_error.clear();
  if (msa_status st = check_decode_args(a); st != MSA_OK) return st;
  const size_t need = msa_sparse_attn_decode_workspace_size(a);
  MSA_REQUIRE(ws != nullptr && ws_bytes >= need, MSA_ERR_WORKSPACE, "workspace %zu bytes, need %zu", ws_bytes, need);
  MSA_REQUIRE(aligned16(ws), MSA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (a->B == 0) return MSA_OK;
  float* o_part = static_cast<float*>(ws);
  const size_t parts = static_cast<size_t>(a->B) * a->Hq * a->k;
  float* lse_part = o_part + parts * a->D;
  int32_t* counter = reinterpret_cast<int32_t*>(lse_part + parts);
  return launch_attn_decode(*a, o_part, lse_part, counter, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
static msa_status check_prefill(const msa_prefill_args* a) {
  MSA_REQUIRE(a != nullptr, MSA_ERR_INVALID_ARG, "args is NULL");
  MSA_REQUIRE(a->mode == MSA_MODE_PREFILL || a->mode == MSA_MODE_CHUNK, MSA_ERR_INVALID_ARG,
              "mode %d: prefill attention takes PREFILL or CHUNK", static_cast<int>(a->mode));
  if (a->mode == MSA_MODE_CHUNK) {
    MSA_REQUIRE(a->seq_pt && a->q_pos, MSA_ERR_INVALID_ARG, "chunk: seq_pt and q_pos must be non-NULL");
    // the page id travels in the tile descriptor above two flag bits
    MSA_REQUIRE(a->num_pages >= 1 && a->num_pages <= (int64_t(1) << 29), MSA_ERR_INVALID_ARG,
                "num_pages = %" PRId64 ", supported 1..2^29", a->num_pages);
    MSA_REQUIRE(a->max_pages >= 1 && a->max_pages < (int64_t(1) << 31) / kBk, MSA_ERR_INVALID_ARG,
                "max_pages = %" PRId64, a->max_pages);
  }
  MSA_REQUIRE(a->B >= 0 && a->S >= 0 && a->Hkv >= 1 && a->Hq >= 1, MSA_ERR_INVALID_ARG,
              "B = %d, S = %d, Hq = %d, Hkv = %d", a->B, a->S, a->Hq, a->Hkv);
  MSA_REQUIRE(a->Hq % a->Hkv == 0 && a->Hq / a->Hkv <= kMaxG, MSA_ERR_UNSUPPORTED,
              "GQA ratio Hq/Hkv = %d/%d not in 1..%d", a->Hq, a->Hkv, kMaxG);
  if (msa_status st = check_common_shape(a->Bk, a->D, kD, "D"); st != MSA_OK) return st;
  MSA_REQUIRE(a->k >= 1 && a->k <= kMaxK, MSA_ERR_UNSUPPORTED, "k = %d, supported 1..%d", a->k, kMaxK);
  MSA_REQUIRE(a->Q && a->K && a->V && a->sel && a->count && a->O, MSA_ERR_INVALID_ARG,
              "Q, K, V, sel, count and O must be non-NULL");
  MSA_REQUIRE(aligned16(a->Q) && aligned16(a->K) && aligned16(a->V) && aligned16(a->O), MSA_ERR_INVALID_ARG,
              "Q, K, V and O must be 16-byte aligned");
  for (int i = 0; i < 3; ++i) {
    MSA_REQUIRE(vec_stride_ok(a->Q_stride[i], 2), MSA_ERR_INVALID_ARG,
                "Q_stride[%d] = %" PRId64 " must be a positive multiple of 8 elements", i, a->Q_stride[i]);
    MSA_REQUIRE(vec_stride_ok(a->K_stride[i], 2) && vec_stride_ok(a->V_stride[i], 2), MSA_ERR_INVALID_ARG,
                "K/V strides must be positive multiples of 8 elements");
  }
  MSA_REQUIRE(static_cast<int64_t>(a->B) * a->S < (int64_t(1) << 31), MSA_ERR_UNSUPPORTED, "B*S too large");
  return MSA_OK;
}

size_t msa_sparse_attn_prefill_workspace_size(const msa_prefill_args* a, int64_t chunk_queries) {
  if (a == nullptr || chunk_queries < 1) return 0;
  if (a->mode == MSA_MODE_CHUNK && a->max_pages < 1) return 0;
  return attn_prefill_workspace_size(*a, chunk_queries);
}

msa_status msa_sparse_attn_prefill(const msa_prefill_args* a, void* ws, size_t ws_bytes, msa_stream_t stream) {
  g_last_error.clear();
  if (msa_status st = check_prefill(a); st != MSA_OK) return st;
  const size_t need = attn_prefill_workspace_size(*a, 1);
  MSA_REQUIRE(ws != nullptr && ws_bytes >= need, MSA_ERR_WORKSPACE, "workspace %zu bytes, need at least %zu",
              ws_bytes, need);
  MSA_REQUIRE(aligned16(ws), MSA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (static_cast<int64_t>(a->B) * a->S == 0) return MSA_OK;
  return launch_attn_prefill(*a, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
static msa_status check_dense_decode(const msa_dense_decode_args* a) {
  MSA_REQUIRE(a != nullptr, MSA_ERR_INVALID_ARG, "args is NULL");
  MSA_REQUIRE(a->B >= 0 && a->B <= kDenseMaxBatch && a->Hkv >= 1 && a->Hq >= 1, MSA_ERR_INVALID_ARG,
              "B = %d (at most %d), Hq = %d, Hkv = %d", a->B, kDenseMaxBatch, a->Hq, a->Hkv);
  MSA_REQUIRE(a->Hq % a->Hkv == 0 && a->Hq / a->Hkv <= kMaxG, MSA_ERR_UNSUPPORTED,
              "GQA ratio Hq/Hkv = %d/%d not in 1..%d", a->Hq, a->Hkv, kMaxG);
  if (msa_status st = check_common_shape(a->Bk, a->D, kD, "D"); st != MSA_OK) return st;
  MSA_REQUIRE(a->Q && a->K_pool && a->V_pool && a->seq_pt && a->seq_len && a->O, MSA_ERR_INVALID_ARG,
              "Q, K_pool, V_pool, seq_pt, seq_len and O must be non-NULL");
  MSA_REQUIRE(aligned16(a->Q) && aligned16(a->K_pool) && aligned16(a->V_pool) && aligned16(a->O), MSA_ERR_INVALID_ARG,
              "Q, K_pool, V_pool and O must be 16-byte aligned");
  MSA_REQUIRE(a->num_pages >= 1 && a->num_pages < (int64_t(1) << 31), MSA_ERR_INVALID_ARG, "num_pages = %" PRId64,
              a->num_pages);
  MSA_REQUIRE(a->max_pages >= 1 && static_cast<int64_t>(a->B) * a->Hkv * a->max_pages < (int64_t(1) << 30),
              MSA_ERR_INVALID_ARG, "max_pages = %" PRId64 ": B * Hkv * max_pages must be below 2^30", a->max_pages);
  for (int i = 0; i < 2; ++i)
    MSA_REQUIRE(vec_stride_ok(a->Q_stride[i], 2), MSA_ERR_INVALID_ARG,
                "Q_stride[%d] = %" PRId64 " must be a positive multiple of 8 elements", i, a->Q_stride[i]);
  for (int i = 0; i < 3; ++i)
    MSA_REQUIRE(vec_stride_ok(a->kv_stride[i], 2), MSA_ERR_INVALID_ARG,
                "kv_stride[%d] = %" PRId64 " must be a positive multiple of 8 elements", i, a->kv_stride[i]);
  return MSA_OK;
}

size_t msa_dense_attn_decode_workspace_size(const msa_dense_decode_args* a) {
  if (a == nullptr || a->B < 0 || a->Hq < 1 || a->Hkv < 1 || a->max_pages < 1) return 0;
  return dense_decode_workspace_size(*a);
}

msa_status msa_dense_attn_decode(const msa_dense_decode_args* a, void* ws, size_t ws_bytes, msa_stream_t stream) {
  g_last_error.clear();
  if (msa_status st = check_dense_decode(a); st != MSA_OK) return st;
  const size_t need = dense_decode_workspace_size(*a);
  MSA_REQUIRE(ws != nullptr && ws_bytes >= need, MSA_ERR_WORKSPACE, "workspace %zu bytes, need %zu", ws_bytes, need);
  MSA_REQUIRE(aligned16(ws), MSA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (a->B == 0) return MSA_OK;
  return launch_dense_decode(*a, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

msa_status msa_dense_attn_prefill(const msa_dense_prefill_args* a, msa_stream_t stream) {
  g_last_error.clear();
  MSA_REQUIRE(a != nullptr, MSA_ERR_INVALID_ARG, "args is NULL");
  MSA_REQUIRE(a->B >= 0 && a->S >= 0 && a->Hkv >= 1 && a->Hq >= 1, MSA_ERR_INVALID_ARG,
              "B = %d, S = %d, Hq = %d, Hkv = %d", a->B, a->S, a->Hq, a->Hkv);
  MSA_REQUIRE(a->Hq % a->Hkv == 0 && a->Hq / a->Hkv <= kMaxG, MSA_ERR_UNSUPPORTED,
              "GQA ratio Hq/Hkv = %d/%d not in 1..%d", a->Hq, a->Hkv, kMaxG);
  MSA_REQUIRE(a->D == kD, MSA_ERR_UNSUPPORTED, "D = %d, only %d is supported", a->D, kD);
  MSA_REQUIRE(a->Q && a->K && a->V && a->O, MSA_ERR_INVALID_ARG, "Q, K, V and O must be non-NULL");
  MSA_REQUIRE(aligned16(a->Q) && aligned16(a->K) && aligned16(a->V) && aligned16(a->O), MSA_ERR_INVALID_ARG,
              "Q, K, V and O must be 16-byte aligned");
  for (int i = 0; i < 3; ++i)
    MSA_REQUIRE(vec_stride_ok(a->Q_stride[i], 2) && vec_stride_ok(a->K_stride[i], 2) && vec_stride_ok(a->V_stride[i], 2),
                MSA_ERR_INVALID_ARG, "Q/K/V strides must be positive multiples of 8 elements");
  MSA_REQUIRE(static_cast<int64_t>(a->B) * a->S < (int64_t(1) << 31), MSA_ERR_UNSUPPORTED, "B*S too large");
  if (static_cast<int64_t>(a->B) * a->S == 0) return MSA_OK;
  return launch_dense_prefill(*a, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
msa_status msa_lse_merge(const float* O_part, const float* LSE_part, int64_t rows, int parts, int D, void* O,
                         float* LSE, int32_t* dev_err, msa_stream_t stream) {
  g_last_error.clear();
  MSA_REQUIRE(rows >= 0, MSA_ERR_INVALID_ARG, "rows = %" PRId64, rows);
  MSA_REQUIRE(parts >= 1 && parts <= kMaxK, MSA_ERR_UNSUPPORTED, "parts = %d, supported 1..%d", parts, kMaxK);
  MSA_REQUIRE(D >= 4 && D <= 512 && D % 4 == 0, MSA_ERR_UNSUPPORTED, "D = %d, need a multiple of 4 in [4, 512]", D);
  MSA_REQUIRE(O_part && LSE_part && O, MSA_ERR_INVALID_ARG, "O_part, LSE_part and O must be non-NULL");
  MSA_REQUIRE(aligned16(O_part) && (reinterpret_cast<uintptr_t>(O) & 7u) == 0, MSA_ERR_INVALID_ARG,
              "O_part must be 16-byte and O 8-byte aligned");
  return launch_lse_merge(O_part, LSE_part, rows, parts, D, O, LSE, dev_err, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
msa_status msa_cache_append(const msa_append_args* a, msa_stream_t stream) {
  g_last_error.clear();
  MSA_REQUIRE(a != nullptr, MSA_ERR_INVALID_ARG, "args is NULL");
  MSA_REQUIRE(a->B >= 0 && a->Hkv >= 1, MSA_ERR_INVALID_ARG, "B = %d, Hkv = %d", a->B, a->Hkv);
  MSA_REQUIRE(a->Bk == kBk, MSA_ERR_UNSUPPORTED, "Bk = %d, supported %d", a->Bk, kBk);
  MSA_REQUIRE(a->D >= 8 && a->D % 8 == 0 && a->dI >= 8 && a->dI % 8 == 0, MSA_ERR_UNSUPPORTED,
              "D = %d, dI = %d: need positive multiples of 8", a->D, a->dI);
  MSA_REQUIRE(a->num_pages >= 1 && a->max_pages >= 1 && a->max_pages < (int64_t(1) << 31) / a->Bk,
              MSA_ERR_INVALID_ARG, "num_pages = %" PRId64 ", max_pages = %" PRId64, a->num_pages, a->max_pages);
  MSA_REQUIRE(a->K_new && a->V_new && a->kidx_new && a->K_pool && a->V_pool && a->kidx_pool && a->seq_pt && a->seq_len,
              MSA_ERR_INVALID_ARG, "tensor pointers must be non-NULL");
  MSA_REQUIRE(aligned16(a->K_new) && aligned16(a->V_new) && aligned16(a->kidx_new) && aligned16(a->K_pool) &&
                  aligned16(a->V_pool) && aligned16(a->kidx_pool),
              MSA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  for (int i = 0; i < 2; ++i)
    MSA_REQUIRE(vec_stride_ok(a->K_new_stride[i], 2) && vec_stride_ok(a->V_new_stride[i], 2) &&
                    (vec_stride_ok(a->kidx_new_stride[i], 2) || (i == 1 && a->kidx_new_stride[i] == 0)),
                MSA_ERR_INVALID_ARG, "new-token strides must be positive multiples of 8 elements");
  MSA_REQUIRE(a->T >= 0, MSA_ERR_INVALID_ARG, "T = %d", a->T);
  if (a->T > 1) {
    MSA_REQUIRE(static_cast<int64_t>(a->B) * a->T * a->Hkv < (int64_t(1) << 33), MSA_ERR_INVALID_ARG,
                "B*T*Hkv too large");
    for (int i = 0; i < 3; ++i)
      MSA_REQUIRE(vec_stride_ok(a->new_t_stride[i], 2), MSA_ERR_INVALID_ARG,
                  "new_t_stride[%d] = %" PRId64 " must be a positive multiple of 8 elements", i, a->new_t_stride[i]);
  }
  for (int i = 0; i < 3; ++i)
    MSA_REQUIRE(vec_stride_ok(a->kv_stride[i], 2) &&
                    (vec_stride_ok(a->kidx_stride[i], 2) || (i == 1 && a->kidx_stride[i] == 0)),
                MSA_ERR_INVALID_ARG, "pool strides must be positive multiples of 8 elements (k_idx: group stride 0 allowed)");
  if (a->B == 0) return MSA_OK;
  return launch_cache_append(*a, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
