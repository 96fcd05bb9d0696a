// cache_append.cu -- the step before a decode step: each sequence's current
// token (K, V and its index key) written into the 128-token paged caches.
//
// For sequence b of length L_b the new token sits at position L_b - 1, i.e. in
// slot t = (L_b - 1) % Bk of page seq_pt[b][(L_b - 1) / Bk] ("MiniMax M3
// preparado para inferencia en produccion", paragraph "MSA con paged
// attention": fixed-size pages; the token is in the cache before the step).
// With T tokens per sequence (a prefill chunk, draft tokens) token u sits at
// position L_b - T + u.  One warp per (b, u, g) copies the three rows with
// 16-byte accesses.
#include "msa_internal.h"

namespace msa {
namespace {

struct AppendParams {
  int B, Hkv, D, dI, Bk, T;
  const uint8_t* K_new;
  const uint8_t* V_new;
  const uint8_t* kidx_new;
  int64_t kn0, kn1, vn0, vn1, xn0, xn1;   // byte strides (b, g)
  int64_t knt, vnt, xnt;                  // byte strides of the token index u
  uint8_t* K_pool;
  uint8_t* V_pool;
  uint8_t* kidx_pool;
  int64_t kv0, kv1, kv2, x0, x1, x2;      // byte strides (page, g, t)
  int64_t num_pages;
  const int32_t* seq_pt;
  int64_t max_pages;
  const int32_t* seq_len;
  int32_t* dev_err;
};

__device__ __forceinline__ void copy_row(uint8_t* dst, const uint8_t* src, int bytes, int lane) {
  for (int o = lane * 16; o < bytes; o += 32 * 16)
    *reinterpret_cast<uint4*>(dst + o) = *reinterpret_cast<const uint4*>(src + o);
}

__global__ void __launch_bounds__(256) cache_append_kernel(const AppendParams p) {
  const int64_t wq = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (wq >= static_cast<int64_t>(p.B) * p.T * p.Hkv) return;
  const int lane = threadIdx.x & 31;
  const int g = static_cast<int>(wq % p.Hkv);
  const int64_t bu = wq / p.Hkv;
  const int u = static_cast<int>(bu % p.T), b = static_cast<int>(bu / p.T);
  const int L = p.seq_len[b];
  if (L < p.T || L < 1 || static_cast<int64_t>(L) > p.max_pages * p.Bk) {
    if (lane == 0 && g == 0 && u == 0 && p.dev_err != nullptr) atomicOr(p.dev_err, MSA_DEVERR_BAD_LEN);
    return;
  }
  const int pos = L - p.T + u;
  const int64_t page = p.seq_pt[b * p.max_pages + pos / p.Bk];
  if (page < 0 || page >= p.num_pages) {
    if (lane == 0 && g == 0 && p.dev_err != nullptr) atomicOr(p.dev_err, MSA_DEVERR_BAD_PAGE);
    return;
  }
  const int t = pos % p.Bk;
  copy_row(p.K_pool + page * p.kv0 + g * p.kv1 + t * p.kv2, p.K_new + b * p.kn0 + u * p.knt + g * p.kn1, p.D * 2,
           lane);
  copy_row(p.V_pool + page * p.kv0 + g * p.kv1 + t * p.kv2, p.V_new + b * p.vn0 + u * p.vnt + g * p.vn1, p.D * 2,
           lane);
  // one index-key pool shared by the groups (group stride 0): group 0 writes it
  if (p.x1 != 0 || g == 0)
    copy_row(p.kidx_pool + page * p.x0 + g * p.x1 + t * p.x2, p.kidx_new + b * p.xn0 + u * p.xnt + g * p.xn1,
             p.dI * 2, lane);
}

}  // namespace

msa_status launch_cache_append(const msa_append_args& a, cudaStream_t stream) {
  AppendParams p;
  p.B = a.B; p.Hkv = a.Hkv; p.D = a.D; p.dI = a.dI; p.Bk = a.Bk; p.T = a.T > 1 ? a.T : 1;
  p.K_new = static_cast<const uint8_t*>(a.K_new);
  p.V_new = static_cast<const uint8_t*>(a.V_new);
  p.kidx_new = static_cast<const uint8_t*>(a.kidx_new);
  p.kn0 = a.K_new_stride[0] * 2; p.kn1 = a.K_new_stride[1] * 2;
  p.vn0 = a.V_new_stride[0] * 2; p.vn1 = a.V_new_stride[1] * 2;
  p.xn0 = a.kidx_new_stride[0] * 2; p.xn1 = a.kidx_new_stride[1] * 2;
  p.knt = p.T > 1 ? a.new_t_stride[0] * 2 : 0;
  p.vnt = p.T > 1 ? a.new_t_stride[1] * 2 : 0;
  p.xnt = p.T > 1 ? a.new_t_stride[2] * 2 : 0;
  p.K_pool = static_cast<uint8_t*>(a.K_pool);
  p.V_pool = static_cast<uint8_t*>(a.V_pool);
  p.kidx_pool = static_cast<uint8_t*>(a.kidx_pool);
  p.kv0 = a.kv_stride[0] * 2; p.kv1 = a.kv_stride[1] * 2; p.kv2 = a.kv_stride[2] * 2;
  p.x0 = a.kidx_stride[0] * 2; p.x1 = a.kidx_stride[1] * 2; p.x2 = a.kidx_stride[2] * 2;
  p.num_pages = a.num_pages; p.seq_pt = a.seq_pt; p.max_pages = a.max_pages; p.seq_len = a.seq_len;
  p.dev_err = a.dev_err;
  const int64_t warps = static_cast<int64_t>(a.B) * p.T * a.Hkv;
  const unsigned grid = static_cast<unsigned>((warps + 7) / 8);
  cache_append_kernel<<<grid, 256, 0, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "cache_append_kernel launch");
  return MSA_OK;
}

}  // namespace msa
