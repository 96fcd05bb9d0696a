// select_warp.cuh -- exact top-m block selection of one score row by one warp.
//
// Order: score descending, then block index ascending (composite 64-bit key,
// see select_key in msa_ptx.cuh), so the selected set is unique.  Candidates
// j < n are held in registers, NPL per lane (n <= 32 * NPL).  A lower bound T0
// of the m-th largest key is the m-th largest of the 32 lane maxima (m <= 32);
// the survivors with key >= T0 (usually a few dozen) are compacted in index
// order into shared memory and ranked exactly.  More than kSelCap survivors
// (massive ties) take an exact successive arg-max over the registers.
// Used by the standalone top-k kernel and by the decode index kernel's fused
// selection ("MiniMax M3: Como la atencion dispersa hace practicos a los
// agentes de largo alcance", bullet "Costo predecible": k blocks per query and
// GQA group, own block included).
#pragma once

#include "msa_ptx.cuh"

namespace msa {

constexpr int kSelCap = 128;   // survivors ranked in shared memory per warp

// Writes the m best of crow[0..n) (n > m >= 1), ascending, to out[0..m).
// surv: kSelCap uint64 of shared memory, pick: m ints of shared memory, both
// private to the warp.  All 32 lanes call it.
template <int NPL>
__device__ __forceinline__ void warp_select(const float* crow, int n, int m, uint64_t* surv, int* pick, int* out) {
  const int lane = threadIdx.x & 31;
  uint32_t u[NPL];
  uint32_t lmax = 0;
  // every load first, then the keys: the loads stay in flight together
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int j = lane + 32 * i;
    u[i] = (j < n) ? __float_as_uint(__ldcg(crow + j)) : 0u;
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int j = lane + 32 * i;
    u[i] = (j < n) ? score_order_key(__uint_as_float(u[i])) : 0u;
    lmax = max(lmax, u[i]);
  }
  uint32_t T0 = 0;
  if (m <= 32) {
    uint32_t v = lmax;   // bitonic sort of the lane maxima, descending over lanes
#pragma unroll
    for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        const uint32_t o = __shfl_xor_sync(0xffffffffu, v, jj);
        const bool desc = (lane & kk) == 0;
        const bool lower = (lane & jj) == 0;
        v = (lower == desc) ? max(v, o) : min(v, o);
      }
    }
    T0 = __shfl_sync(0xffffffffu, v, m - 1);
  }
  int c = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int j = lane + 32 * i;
    const bool f = (j < n) && u[i] >= T0;
    const uint32_t mask = __ballot_sync(0xffffffffu, f);
    const int pos = c + __popc(mask & ((1u << lane) - 1u));
    if (f && pos < kSelCap) surv[pos] = (static_cast<uint64_t>(u[i]) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(j));
    c += __popc(mask);
  }
  __syncwarp();
  if (c <= kSelCap) {
    int outc = 0;   // exact rank of every survivor (index order); the m best have rank < m
    for (int base = 0; base < c; base += 32) {
      const int x = base + lane;
      bool pk = false;
      int jx = 0;
      if (x < c) {
        const uint64_t kx = surv[x];
        int rank = 0;
        for (int y = 0; y < c; ++y) rank += surv[y] > kx;
        pk = rank < m;
        jx = select_key_index(kx);
      }
      const uint32_t mask = __ballot_sync(0xffffffffu, pk);
      if (pk) out[outc + __popc(mask & ((1u << lane) - 1u))] = jx;
      outc += __popc(mask);
    }
  } else {
    uint64_t prev = ~0ull;   // m rounds of arg-max below the previous pick
    for (int t = 0; t < m; ++t) {
      uint64_t best = 0;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int j = lane + 32 * i;
        if (j < n) {
          const uint64_t key = (static_cast<uint64_t>(u[i]) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(j));
          if (key < prev && key > best) best = key;
        }
      }
      best = warp_max_u64(best);
      prev = best;
      if (lane == 0) pick[t] = select_key_index(best);
    }
    __syncwarp();
    for (int t = lane; t < m; t += 32) {   // ascending order by counting
      const int jt = pick[t];
      int pos = 0;
      for (int y = 0; y < m; ++y) pos += pick[y] < jt;
      out[pos] = jt;
    }
  }
  __syncwarp();
}

// Runtime dispatch on the candidate count (n <= 2048).
__device__ __forceinline__ void warp_select_any(const float* crow, int n, int m, uint64_t* surv, int* pick,
                                                int* out) {
  if (n <= 32) warp_select<1>(crow, n, m, surv, pick, out);
  else if (n <= 64) warp_select<2>(crow, n, m, surv, pick, out);
  else if (n <= 128) warp_select<4>(crow, n, m, surv, pick, out);
  else if (n <= 256) warp_select<8>(crow, n, m, surv, pick, out);
  else if (n <= 512) warp_select<16>(crow, n, m, surv, pick, out);
  else if (n <= 1024) warp_select<32>(crow, n, m, surv, pick, out);
  else warp_select<64>(crow, n, m, surv, pick, out);
}

}  // namespace msa
