// index_prefill.cu -- a1 (prefill): block scores of the Index Branch for every
// query of a causal prefill.
//
// For query i of sequence b, KV group g and every block j < i / Bk:
//     c_j = max_{t in block j} sum_{h < HI} w[b,i,g,h] * ReLU(q_idx[b,i,g,h] . k_idx[b,t,g])
// ("MiniMax M3: Como la atencion dispersa hace practicos a los agentes de largo
// alcance", MSA paragraph and caption; the formula is this library's).  The own
// block and later blocks are written -inf.
//
// This is a dense contraction on the tensor cores.  Work item = (b, g, query
// block qb): 128 queries against the qb earlier key blocks.  Items are paired
// (qb, nbq-1-qb) so every pair costs nbq-1 blocks, and a persistent CTA per SM
// takes pairs round-robin.
//   warp 0    TMA: the HI q_idx tiles of the item (128 queries x 64, one per
//             index head, double-buffered across items) and a 4-deep ring of
//             k_idx blocks (128 tokens x 64), all 128-byte swizzled;
//   warp 1    tcgen05: per key block, passes of two index heads:
//             D_h[query, token] = q_idx_h . k_idx  (M=128, N=128, K=64) for
//             both heads into a 256-column TMEM buffer, the two MMA chains
//             interleaved step by step (a single accumulation chain leaves the
//             tensor core waiting on its own results); two buffers;
//   warps 2-5 epilogue, thread = query: acc_t = sum_h w_h ReLU(D_h[t]) with
//             packed fp32 FMAs, carried across the passes in registers, then
//             the max over the block's 128 tokens, one store per (query, block).
#include "msa_internal.h"
#include "msa_ptx.cuh"

namespace msa {
namespace {

constexpr int kThreads = 192;
constexpr int kTile = 128 * 64 * 2;            // 16 KiB: 128 rows x 64 bf16
constexpr int kKStages = 4;
constexpr int kTmemCols = 512;
constexpr int kBufCols = 256;                  // one TMEM buffer: 2 heads x 128 tokens

struct Params {
  int B, S, Hkv, HI, nbq, nb_stride;
  const float* w;
  int64_t ws0, ws1, ws2;
  float* C;
  int64_t cs0, cs1, cs2;
  int32_t* dev_err;
};

struct Item {
  int b, g, qb;
};

// item t of pair p: pairs enumerate (b, g, pp) with qb in {pp, nbq-1-pp}
__device__ __forceinline__ int pair_items(const Params& p, int64_t pair, Item* it) {
  const int half = (p.nbq + 1) / 2;
  const int pp = static_cast<int>(pair % half);
  const int64_t bg = pair / half;
  const int g = static_cast<int>(bg % p.Hkv), b = static_cast<int>(bg / p.Hkv);
  it[0] = {b, g, pp};
  const int other = p.nbq - 1 - pp;
  if (other == pp) return 1;
  it[1] = {b, g, other};
  return 2;
}

__device__ __forceinline__ uint64_t pack2(float x, float y) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& x, float& y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__global__ void __launch_bounds__(kThreads, 1)
index_prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                     const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_a = smem;                              // [2][4] q_idx tiles
  uint8_t* s_k = smem + 2 * kMaxHI * kTile;         // [kKStages] k_idx blocks

  __shared__ __align__(8) uint64_t bar_afull[2], bar_aempty[2], bar_kfull[kKStages], bar_kempty[kKStages];
  __shared__ __align__(8) uint64_t bar_tfull[2], bar_tempty[2], bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_cst[128][33];   // block scores staged per query row, 32 blocks at a time

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_afull[i], 1); mbar_init(&bar_aempty[i], 1);
      mbar_init(&bar_tfull[i], 1); mbar_init(&bar_tempty[i], 4);
    }
    for (int i = 0; i < kKStages; ++i) { mbar_init(&bar_kfull[i], 1); mbar_init(&bar_kempty[i], 1); }
    mbar_init(&bar_drain, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&s_tmem, kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  const int64_t npairs = static_cast<int64_t>(p.B) * p.Hkv * ((p.nbq + 1) / 2);

  if (warp == 0) {
    // ===================== TMA producer =====================
    if (lane == 0) {
      int na = 0, nk = 0;
      bool ok = true;
      for (int64_t pr = blockIdx.x; pr < npairs && ok; pr += gridDim.x) {
        Item its[2];
        const int ni = pair_items(p, pr, its);
        for (int x = 0; x < ni && ok; ++x) {
          const Item it = its[x];
          if (it.qb == 0) continue;
          const int a = na & 1;
          if (!(ok = mbar_wait(&bar_aempty[a], ((na >> 1) & 1) ^ 1, abort_flag, p.dev_err))) break;
          mbar_arrive_expect_tx(&bar_afull[a], p.HI * kTile);
          for (int h = 0; h < p.HI; ++h)
            tma_load_5d(s_a + (a * kMaxHI + h) * kTile, &qmap, &bar_afull[a], 0, h, it.g, it.qb * kBk, it.b);
          ++na;
          for (int j = 0; j < it.qb; ++j) {
            const int st = nk % kKStages;
            if (!(ok = mbar_wait(&bar_kempty[st], ((nk / kKStages) & 1) ^ 1, abort_flag, p.dev_err))) break;
            mbar_arrive_expect_tx(&bar_kfull[st], kTile);
            tma_load_4d(s_k + st * kTile, &kmap, &bar_kfull[st], 0, it.g, j * kBk, it.b);
            ++nk;
          }
        }
      }
      if (*abort_flag) {  // let loads in flight land before the CTA exits
        for (int n = max(0, nk - kKStages); n < nk; ++n) {
          uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(&bar_kfull[n % kKStages], (n / kKStages) & 1) &&
                 global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
          }
        }
        for (int n = max(0, na - 2); n < na; ++n) {
          uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(&bar_afull[n & 1], (n >> 1) & 1) && global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ===================== tcgen05 issuer =====================
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
      const int npass = (p.HI + 1) / 2;
      int na = 0, nk = 0, nt = 0;
      bool ok = true;
      for (int64_t pr = blockIdx.x; pr < npairs && ok; pr += gridDim.x) {
        Item its[2];
        const int ni = pair_items(p, pr, its);
        for (int x = 0; x < ni && ok; ++x) {
          const Item it = its[x];
          if (it.qb == 0) continue;
          const int a = na & 1;
          if (!(ok = mbar_wait(&bar_afull[a], (na >> 1) & 1, abort_flag, p.dev_err))) break;
          const uint32_t abase = smem_u32(s_a + a * kMaxHI * kTile);
          for (int j = 0; j < it.qb && ok; ++j) {
            const int st = nk % kKStages;
            if (!(ok = mbar_wait(&bar_kfull[st], (nk / kKStages) & 1, abort_flag, p.dev_err))) break;
            const uint32_t kbase = smem_u32(s_k + st * kTile);
            for (int ps = 0; ps < npass; ++ps) {
              const int buf = nt & 1;
              if (!(ok = mbar_wait(&bar_tempty[buf], ((nt >> 1) & 1) ^ 1, abort_flag, p.dev_err))) break;
              tc_fence_after();
              const int h0 = 2 * ps, nh = min(2, p.HI - h0);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                for (int hh = 0; hh < nh; ++hh)
                  umma_bf16(tmem + buf * kBufCols + hh * 128, sdesc_sw128(abase + (h0 + hh) * kTile + 32 * kk, 16, 1024),
                            sdesc_sw128(kbase + 32 * kk, 16, 1024), idesc, kk > 0);
              umma_commit(&bar_tfull[buf]);
              ++nt;
            }
            umma_commit(&bar_kempty[st]);
            ++nk;
          }
          umma_commit(&bar_aempty[a]);
          ++na;
        }
      }
      umma_commit(&bar_drain);
      uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&bar_drain, 0) && global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
      }
    }
    __syncwarp();
  } else {
    // ===================== epilogue (warps 2..5), thread = query =====================
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    int nt = 0;
    bool ok = true;
    for (int64_t pr = blockIdx.x; pr < npairs && ok; pr += gridDim.x) {
      Item its[2];
      const int ni = pair_items(p, pr, its);
      for (int x = 0; x < ni && ok; ++x) {
        const Item it = its[x];
        const int i = it.qb * kBk + r;
        const bool valid = i < p.S;
        uint64_t w2[kMaxHI];
#pragma unroll
        for (int h = 0; h < kMaxHI; ++h) {
          const float wv = (valid && h < p.HI) ? p.w[it.b * p.ws0 + static_cast<int64_t>(i) * p.ws1 + it.g * p.ws2 + h]
                                               : 0.f;
          w2[h] = pack2(wv, wv);
        }
        // rows of this warp: queries it.qb*Bk + q*32 + rr, rr < 32
        const int row0 = it.qb * kBk + q * 32;
        auto flush = [&](int j0, int cnt) {   // coalesced: one 128-byte row segment per step
          __syncwarp();
          for (int rr = 0; rr < 32; ++rr) {
            if (row0 + rr < p.S && lane < cnt)
              p.C[it.b * p.cs0 + static_cast<int64_t>(row0 + rr) * p.cs1 + it.g * p.cs2 + j0 + lane] =
                  s_cst[q * 32 + rr][lane];
          }
          __syncwarp();
        };
        const int npass = (p.HI + 1) / 2;
        for (int j = 0; j < it.qb; ++j) {
          // acc[t/2] = sum over heads of w_h ReLU(D_h[query, t]) for t = 2e, 2e+1 (packed)
          uint64_t acc[64];
#pragma unroll
          for (int e = 0; e < 64; ++e) acc[e] = 0ull;
#pragma unroll
          for (int ps = 0; ps < (kMaxHI + 1) / 2; ++ps) {
            if (ps >= npass) break;
            const int buf = nt & 1;
            // warp-uniform decision: the TMEM loads below are warp-collective
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar_tfull[buf], (nt >> 1) & 1, abort_flag, p.dev_err))))
              break;
            tc_fence_after();
            const uint32_t base = tmem + lane_addr + buf * kBufCols;
            const bool two = 2 * ps + 1 < p.HI;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              uint32_t v[2][32];
              tmem_ld32(base + cc * 32, v[0]);
              if (two) tmem_ld32(base + 128 + cc * 32, v[1]);
              tmem_ld_wait();
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                if (hh == 1 && !two) break;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const uint64_t rl = pack2(fmaxf(__uint_as_float(v[hh][2 * e]), 0.f),
                                            fmaxf(__uint_as_float(v[hh][2 * e + 1]), 0.f));
                  acc[cc * 16 + e] = fma2(w2[2 * ps + hh], rl, acc[cc * 16 + e]);
                }
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_tempty[buf]);
            ++nt;
          }
          if (!ok) break;
          float m = -INFINITY;
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            float a0, a1, b0, b1;
            unpack2(acc[e], a0, a1);
            unpack2(acc[e + 1], b0, b1);
            m = max3(m, max3(a0, a1, b0), b1);
          }
          s_cst[r][j & 31] = m;
          if ((j & 31) == 31 || j == it.qb - 1) flush(j & ~31, (j & 31) + 1);
        }
        if (!ok) break;
        // -inf for the own block and every later entry, one row segment at a time
        for (int rr = 0; rr < 32; ++rr) {
          if (row0 + rr >= p.S) break;
          float* rowp = p.C + it.b * p.cs0 + static_cast<int64_t>(row0 + rr) * p.cs1 + it.g * p.cs2;
          for (int j = it.qb + lane; j < p.nb_stride; j += 32) rowp[j] = -INFINITY;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

msa_status launch_index_prefill(const msa_index_args& a, cudaStream_t stream) {
  DeviceInfo dev;
  if (msa_status st = current_device(&dev); st != MSA_OK) return st;
  // q_idx as 5-D (dI, h, g, s, b); box = one head of 128 queries
  CUtensorMap qmap, kmap;
  {
    const uint64_t dims[5] = {static_cast<uint64_t>(a.dI), static_cast<uint64_t>(a.HI), static_cast<uint64_t>(a.Hkv),
                              static_cast<uint64_t>(a.S), static_cast<uint64_t>(a.B)};
    const uint64_t strides[4] = {static_cast<uint64_t>(a.q_idx_stride[3]) * 2,
                                 static_cast<uint64_t>(a.q_idx_stride[2]) * 2,
                                 static_cast<uint64_t>(a.q_idx_stride[1]) * 2,
                                 static_cast<uint64_t>(a.q_idx_stride[0]) * 2};
    const uint32_t box[5] = {64, 1, 1, 128, 1};
    if (msa_status st = encode_tiled_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, a.q_idx, dims, strides, box,
                                         CU_TENSOR_MAP_SWIZZLE_128B, "q_idx");
        st != MSA_OK)
      return st;
  }
  {
    // k_idx as 4-D (dI, g, s, b); box = 128 tokens of one group
    const uint64_t dims[4] = {static_cast<uint64_t>(a.dI), static_cast<uint64_t>(a.Hkv), static_cast<uint64_t>(a.S),
                              static_cast<uint64_t>(a.B)};
    const uint64_t strides[3] = {static_cast<uint64_t>(a.k_idx_stride[2]) * 2,
                                 static_cast<uint64_t>(a.k_idx_stride[1]) * 2,
                                 static_cast<uint64_t>(a.k_idx_stride[0]) * 2};
    const uint32_t box[4] = {64, 1, 128, 1};
    if (msa_status st = encode_tiled_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.k_idx, dims, strides, box,
                                         CU_TENSOR_MAP_SWIZZLE_128B, "k_idx");
        st != MSA_OK)
      return st;
  }
  Params p;
  p.B = a.B; p.S = a.S; p.Hkv = a.Hkv; p.HI = a.HI;
  p.nbq = (a.S + kBk - 1) / kBk;
  p.nb_stride = a.nb_stride;
  p.w = a.w; p.ws0 = a.w_stride[0]; p.ws1 = a.w_stride[1]; p.ws2 = a.w_stride[2];
  p.C = a.C; p.cs0 = a.C_stride[0]; p.cs1 = a.C_stride[1]; p.cs2 = a.C_stride[2];
  p.dev_err = a.dev_err;
  const size_t smem = 1024 + (2 * kMaxHI + kKStages) * static_cast<size_t>(kTile);
  if (smem > dev.max_smem_optin) return fail(MSA_ERR_UNSUPPORTED, "prefill index score: not enough shared memory");
  cudaError_t e = cudaFuncSetAttribute(index_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(index_prefill)");
  const int64_t npairs = static_cast<int64_t>(a.B) * a.Hkv * ((p.nbq + 1) / 2);
  const int grid = static_cast<int>(std::min<int64_t>(dev.num_sms, std::max<int64_t>(npairs, 1)));
  index_prefill_kernel<<<grid, kThreads, smem, stream>>>(qmap, kmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "index_prefill_kernel launch");
  return MSA_OK;
}

}  // namespace msa
