// page_table.cu -- a3: decode page table from the selected blocks.
//
// Fixed-page attention kernels want a page list per batch row, while MSA picks
// different blocks for every KV group; the selected blocks are therefore
// mapped to physical pages and the group dimension is flattened into the batch
// ("MiniMax M3 preparado para inferencia en produccion", paragraph "MSA con
// paged attention").  Row r = b * Hkv + g:
//     pt[r][s] = seq_pt[b][sel[b][g][s]]  (s < count),  n[r] = count,
//     last_len[r] = seq_len[b] - Bk * ((seq_len[b] - 1) / Bk).
// The same table serves a chunk of S queries per sequence (query s of
// sequence b at position q_pos[b] + s, i.e. length q_pos[b] + s + 1) with rows
// r = (b * S + s) * Hkv + g, so that the decode attention kernel can run a
// few queries per sequence (draft verification) in one launch.
#include "msa_internal.h"
#include "msa_ptx.cuh"

namespace msa {
namespace {

__global__ void page_table_kernel(const int32_t* __restrict__ sel, const int32_t* __restrict__ count,
                                  const int32_t* __restrict__ seq_pt, int64_t max_pages,
                                  const int32_t* __restrict__ seq_len, int B, int Hkv, int k, int Bk,
                                  int32_t* __restrict__ pt, int32_t* __restrict__ n, int32_t* __restrict__ last_len,
                                  int32_t* dev_err, int S, const int32_t* __restrict__ q_pos) {
  // rows r = (b * S + s) * Hkv + g; S = 1 without q_pos (one query per sequence)
  const int64_t total = static_cast<int64_t>(B) * S * Hkv * k;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = e / k;
    const int x = static_cast<int>(e % k);
    const int64_t bs = r / Hkv;
    const int b = static_cast<int>(bs / S);
    // the query's length: L_b, or for query s of a chunk its position + 1
    const int L = q_pos != nullptr ? q_pos[b] + static_cast<int>(bs % S) + 1 : seq_len[b];
    const int own = L >= 1 ? (L - 1) / Bk : -1;
    const int c = count[r];
    int32_t page = -1;
    if (x < c) {
      const int j = sel[e];
      if (j < 0 || j > own || j >= max_pages) {
        report(dev_err, MSA_DEVERR_BAD_SEL);
      } else {
        page = seq_pt[b * max_pages + j];
      }
    }
    pt[e] = page;
    if (x == 0) {
      n[r] = c;
      last_len[r] = L >= 1 ? L - Bk * own : 0;
    }
  }
}

}  // namespace

msa_status launch_page_table(const int32_t* sel, const int32_t* count, const int32_t* seq_pt, int64_t max_pages,
                             const int32_t* seq_len, int B, int Hkv, int k, int Bk, int32_t* pt, int32_t* n,
                             int32_t* last_len, int32_t* dev_err, cudaStream_t stream, int S, const int32_t* q_pos) {
  const int64_t total = static_cast<int64_t>(B) * S * Hkv * k;
  if (total == 0) return MSA_OK;
  const int threads = 256;
  const int64_t grid = std::min<int64_t>((total + threads - 1) / threads, 4096);
  page_table_kernel<<<static_cast<unsigned>(grid), threads, 0, stream>>>(sel, count, seq_pt, max_pages, seq_len, B,
                                                                        Hkv, k, Bk, pt, n, last_len, dev_err, S,
                                                                        q_pos);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "page_table_kernel launch");
  return MSA_OK;
}

}  // namespace msa
