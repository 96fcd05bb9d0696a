// topk.cu -- a2: per (query, KV group) block selection.
//
// Keep the query's own block plus the k-1 best earlier blocks, ranked by
// (score desc, block index asc); with at most k-1 earlier blocks keep them all
// ("MiniMax M3: Como la atencion dispersa hace practicos a los agentes de largo
// alcance", bullet "Costo predecible a cualquier longitud": k = 16 blocks,
// own block included).  The output row is ascending, own block last, padded
// with -1.
//
// Scores are mapped to order-preserving 32-bit keys (NaN lowest, -0 == +0);
// the composite key (key << 32 | ~j) makes every candidate distinct, so the
// selected set is unique.
//
// Short rows (<= 2048 candidates: all prefill rows, chunk rows of contexts up
// to 2049 blocks and short decode rows): one warp per row, the register
// algorithm of select_warp.cuh.
// Long rows: one 256-thread CTA per row; its warps select the best blocks of
// slices of the row, then the slices' picks are ranked together.
#include "msa_internal.h"
#include "msa_ptx.cuh"
#include "select_warp.cuh"

namespace msa {
namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kCtaThreads = 256;

__device__ __forceinline__ uint32_t order_key(float f) { return score_order_key(f); }
__device__ __forceinline__ uint64_t comp_key(uint32_t u, int j) {
  return (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(j));
}
__device__ __forceinline__ int comp_index(uint64_t K) { return select_key_index(K); }

struct RowInfo {
  const float* c;     // score row
  int own;            // own block = number of candidates
  int32_t* sel;
  int32_t* cnt;
  bool valid;
};

__device__ __forceinline__ RowInfo row_info(const msa_topk_args& a, int64_t row) {
  RowInfo r;
  if (a.mode != MSA_MODE_DECODE) {
    const int64_t g = row % a.Hkv, bs = row / a.Hkv;
    const int64_t s = bs % a.S, b = bs / a.S;
    r.c = a.C + b * a.C_stride[0] + s * a.C_stride[1] + g * a.C_stride[2];
    // a chunk's query s sits at position q_pos[b] + s; a chunk sequence is
    // rejected as a whole (as the index score does) when it starts before 0 or
    // its last query's own block is not below nb_stride
    const int64_t q0 = a.mode == MSA_MODE_CHUNK ? a.q_pos[b] : 0;
    const int64_t pos = q0 + s;
    r.valid = q0 >= 0 && (q0 + a.S - 1) / a.Bk < a.nb_stride;
    r.own = r.valid ? static_cast<int>(pos / a.Bk) : 0;
  } else {
    const int64_t g = row % a.Hkv, b = row / a.Hkv;
    r.c = a.C + b * a.C_stride[0] + g * a.C_stride[1];
    const int L = a.seq_len[b];
    r.valid = L >= 1 && (L - 1) / a.Bk < a.nb_stride;
    r.own = r.valid ? (L - 1) / a.Bk : 0;
  }
  r.sel = a.sel + row * a.k;
  r.cnt = a.count + row;
  return r;
}

// Rows with own <= k - 1 (and invalid rows): keep every earlier block.
__device__ __forceinline__ void write_all(const RowInfo& r, int k, int lane_or_tid, int stride) {
  for (int x = lane_or_tid; x < k; x += stride) r.sel[x] = (r.valid && x <= r.own) ? x : -1;
  if (lane_or_tid == 0) *r.cnt = r.valid ? r.own + 1 : 0;
}

// Rows are independent and each warp's row is latency-bound (its loads, then
// shuffles): the long-row variants are held to 64 registers so that four
// CTAs (32 rows) are in flight per SM instead of two.
template <int NPL>
__global__ void __launch_bounds__(kWarpsPerCta * 32, NPL >= 16 ? 4 : 1)
topk_warp_kernel(const msa_topk_args a, int64_t rows) {
  __shared__ uint64_t s_surv[kWarpsPerCta][kSelCap];
  __shared__ int s_pick[kWarpsPerCta][kMaxK];
  __shared__ int s_out[kWarpsPerCta][kMaxK];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + wid;
  if (row >= rows) return;
  RowInfo r = row_info(a, row);
  if (!r.valid && lane == 0) report(a.dev_err, MSA_DEVERR_BAD_LEN);
  const int m = a.k - 1;
  const int n = r.own;
  if (!r.valid || n <= m) {
    write_all(r, a.k, lane, 32);
    return;
  }
  warp_select<NPL>(r.c, n, m, s_surv[wid], s_pick[wid], s_out[wid]);
  for (int x = lane; x < a.k; x += 32) r.sel[x] = x < m ? s_out[wid][x] : (x == m ? n : -1);
  if (lane == 0) *r.cnt = m + 1;
}

// One CTA per long row, in two phases: the row is cut into at most kMaxSlices
// slices (of at most 1024 blocks when that leaves no more than one slice per
// warp, else 2048); each warp selects the best m of its slices with the
// register warp select into a pool (slot slice * m + y; 0 = empty, below every
// real key); then the pool's keys are ranked exactly and the m best are the
// picks.  The row's best m blocks are all in the pool: a block outside its
// slice's best m has m better blocks in that slice.  Rows of more than
// kMaxSlices * 2048 blocks take m rounds of block-wide arg-max below the
// previous pick instead.
constexpr int kMaxSlices = 32;
__global__ void __launch_bounds__(kCtaThreads, 1)
topk_cta_kernel(const msa_topk_args a, int64_t rows) {
  __shared__ uint64_t s_surv[kWarpsPerCta][kSelCap];
  __shared__ int s_wpick[kWarpsPerCta][kMaxK];
  __shared__ int s_wout[kWarpsPerCta][kMaxK];
  __shared__ uint64_t s_pool[kMaxSlices * (kMaxK - 1)];
  __shared__ uint64_t s_wmax[kCtaThreads / 32];
  __shared__ uint64_t s_best;
  __shared__ int s_pick[kMaxK];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int64_t row = blockIdx.x;
  if (row >= rows) return;
  RowInfo r = row_info(a, row);
  if (!r.valid && tid == 0) report(a.dev_err, MSA_DEVERR_BAD_LEN);
  const int m = a.k - 1;
  const int n = r.own;
  if (!r.valid || n <= m) {
    write_all(r, a.k, tid, kCtaThreads);
    return;
  }
  if (n <= kMaxSlices * 2048) {
    const int nslices = n <= kWarpsPerCta * 1024 ? (n + 1023) / 1024 : (n + 2047) / 2048;
    const int ssz = (n + nslices - 1) / nslices;     // <= 2048
    for (int sl = wid; sl < nslices; sl += kWarpsPerCta) {
      const int lo = sl * ssz, cnt = min(ssz, n - lo);
      int* out = s_wout[wid];
      int npick = m;
      if (cnt <= m) {
        for (int y = lane; y < cnt; y += 32) out[y] = y;
        npick = cnt;
      } else {
        warp_select_any(r.c + lo, cnt, m, s_surv[wid], s_wpick[wid], out);
      }
      __syncwarp();
      for (int y = lane; y < m; y += 32)
        s_pool[sl * m + y] = y < npick ? comp_key(order_key(r.c[lo + out[y]]), lo + out[y]) : 0ull;
      __syncwarp();
    }
    __syncthreads();
    const int npool = nslices * m;
    for (int x = tid; x < npool; x += kCtaThreads) {
      const uint64_t kx = s_pool[x];
      if (kx == 0ull) continue;
      int rank = 0;
      for (int y = 0; y < npool; ++y) rank += s_pool[y] > kx;
      if (rank < m) s_pick[rank] = comp_index(kx);
    }
    __syncthreads();
  } else {
    uint64_t prev = ~0ull;
    for (int t = 0; t < m; ++t) {
      uint64_t best = 0;
      for (int j = tid; j < n; j += kCtaThreads) {
        const uint64_t K = comp_key(order_key(r.c[j]), j);
        if (K < prev && K > best) best = K;
      }
      best = warp_max_u64(best);
      if (lane == 0) s_wmax[wid] = best;
      __syncthreads();
      if (wid == 0) {
        uint64_t v = lane < kCtaThreads / 32 ? s_wmax[lane] : 0ull;
        v = warp_max_u64(v);
        if (lane == 0) { s_pick[t] = comp_index(v); s_best = v; }
      }
      __syncthreads();
      prev = s_best;
    }
  }
  for (int t = tid; t < m; t += kCtaThreads) {
    const int jt = s_pick[t];
    int pos = 0;
    for (int y = 0; y < m; ++y) pos += s_pick[y] < jt;
    r.sel[pos] = jt;
  }
  if (tid == 0) {
    r.sel[m] = n;
    *r.cnt = m + 1;
  }
  for (int x = m + 1 + tid; x < a.k; x += kCtaThreads) r.sel[x] = -1;
}

template <int NPL>
msa_status launch_warp(const msa_topk_args& a, int64_t rows, cudaStream_t stream) {
  const int64_t grid = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
  topk_warp_kernel<NPL><<<static_cast<unsigned>(grid), kWarpsPerCta * 32, 0, stream>>>(a, rows);
  return MSA_OK;
}

}  // namespace

msa_status launch_topk(const msa_topk_args& a, cudaStream_t stream) {
  const int64_t rows = (a.mode != MSA_MODE_DECODE) ? static_cast<int64_t>(a.B) * a.S * a.Hkv
                                                   : static_cast<int64_t>(a.B) * a.Hkv;
  if (rows == 0) return MSA_OK;
  // the largest candidate count of any row (a chunk's rows: below nb_stride)
  const int64_t maxc = a.mode == MSA_MODE_PREFILL ? (a.S - 1) / a.Bk
                       : a.mode == MSA_MODE_CHUNK ? a.nb_stride - 1 : a.nb_stride;
  msa_status st = MSA_OK;
  if (maxc <= 32) st = launch_warp<1>(a, rows, stream);
  else if (maxc <= 64) st = launch_warp<2>(a, rows, stream);
  else if (maxc <= 128) st = launch_warp<4>(a, rows, stream);
  else if (maxc <= 256) st = launch_warp<8>(a, rows, stream);
  else if (maxc <= 512) st = launch_warp<16>(a, rows, stream);
  else if (maxc <= 1024) st = launch_warp<32>(a, rows, stream);
  else if (maxc <= 2048 && a.mode != MSA_MODE_DECODE) st = launch_warp<64>(a, rows, stream);
  else topk_cta_kernel<<<static_cast<unsigned>(rows), kCtaThreads, 0, stream>>>(a, rows);
  if (st != MSA_OK) return st;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "top-k kernel launch");
  return MSA_OK;
}

}  // namespace msa
