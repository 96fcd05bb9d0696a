// dense_prefill.cu -- the dense comparator of a prefill layer: exact causal GQA
// attention of every query over every earlier token, with no index branch and
// no selection (flash attention on the 5th-generation tensor cores).
//
// The pages quote MSA's prefill speed only against dense attention ("MiniMax
// M3: Como la atencion dispersa hace practicos a los agentes de largo
// alcance", bullet "Rapido en produccion": 14.2x on H800; the M2-report
// article, section "MiniMax Sparse Attention (MSA) y escalado subcuadratico
// entrante": 9.7x at 1M tokens).  This kernel computes that baseline:
//     O[b, i, h] = sum_{t <= i} softmax_t(scale * Q[b, i, h] . K[b, t, g]) V[b, t, g],   g = h / G,
//     LSE[b, i, h] = ln sum_{t <= i} exp(scale * Q[b, i, h] . K[b, t, g]).
//
// An item is (b, g, 128-query tile qt, a pair of the group's query heads);
// both heads share the item's K/V stream (GQA), so every 128-token K/V block
// is loaded once per pair.  Items run heaviest first (qt descending), dealt
// round-robin to one persistent CTA per SM.  Per head ("slot", two per CTA):
//   S  = Q K_j^T   M = 128 queries, N = 128 keys, K = D   (TMEM, 128 columns)
//   softmax (thread = query row): block max, P = 2^(S*scale*log2e - m) written
//        back over S as bf16 pairs
//   O += P V_j     M = 128, N = D, K = 128 keys, P read from TMEM (128 columns)
// The running max m is updated lazily: O (in TMEM) and the running sum are
// rescaled only when a block's max exceeds m by more than 2^8, so P <= 256 and
// the result is exact whichever m is used.  The causal mask is applied in the
// diagonal block only.  Roles: warp 0 TMA (the pair's Q tiles once per item,
// a 2-deep K/V ring), warp 1 tcgen05 issuer (each slot's S and O issued as
// soon as their inputs are ready), warps 2-5 and 6-9 the two slots' softmax
// and epilogue.
#include <algorithm>

#include "msa_internal.h"
#include "msa_ptx.cuh"

namespace msa {
namespace {

constexpr int kHalf = 128 * 64 * 2;          // 16 KiB: 128 rows x 64 bf16
constexpr int kQTile = 2 * kHalf;            // 32 KiB: one head's 128 queries x D
constexpr int kKV = 4 * kHalf;               // 64 KiB: K0 K1 V0 V1
constexpr int kKVStages = 2;
constexpr int kThreads = 320;                // w0 TMA, w1 MMA, w2-5 slot 0, w6-9 slot 1
constexpr int kTmemCols = 512;               // per slot: S / P (128 columns) and O (128 columns)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;             // log2 of the largest P before the running max moves

struct Params {
  int B, S, Hq, Hkv, G, nq, npairs;
  int64_t n_items;
  float scale_log2;
  __nv_bfloat16* O;                          // [B, S, Hq, D] dense
  float* LSE;                                // [B, S, Hq] dense, or null
  int32_t* dev_err;
};

struct Item {
  int b, g, qt, h0, nh;                      // heads h0 .. h0 + nh - 1 (nh = 1 or 2)
};
// Items heaviest first: the query tile runs from the last to the first.
__device__ __forceinline__ Item item_of(const Params& p, int64_t it) {
  const int64_t per_tile = static_cast<int64_t>(p.B) * p.Hkv * p.npairs;
  Item x;
  x.qt = p.nq - 1 - static_cast<int>(it / per_tile);
  const int64_t rest = it % per_tile;
  const int pair = static_cast<int>(rest % p.npairs);
  const int64_t bg = rest / p.npairs;
  x.g = static_cast<int>(bg % p.Hkv);
  x.b = static_cast<int>(bg / p.Hkv);
  x.h0 = x.g * p.G + 2 * pair;
  x.nh = min(2, p.G - 2 * pair);
  return x;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h2);
}

__global__ void __launch_bounds__(kThreads, 1)
dense_prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_q = smem;                       // [2 heads] Q tiles
  uint8_t* s_kv = smem + 2 * kQTile;         // [kKVStages] K/V blocks

  __shared__ __align__(8) uint64_t bar_qfull, bar_qempty, bar_kvfull[kKVStages], bar_kvempty[kKVStages];
  __shared__ __align__(8) uint64_t bar_sfull[2], bar_pready[2], bar_ofull[2], bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bar_qfull, 1);
    mbar_init(&bar_qempty, 1);
    for (int i = 0; i < kKVStages; ++i) { mbar_init(&bar_kvfull[i], 1); mbar_init(&bar_kvempty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_sfull[i], 1); mbar_init(&bar_pready[i], 4); mbar_init(&bar_ofull[i], 1);
    }
    mbar_init(&bar_drain, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&s_tmem, kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // ===================== TMA producer =====================
    if (lane == 0) {
      int nit = 0, nkv = 0;
      bool ok = true;
      for (int64_t it = blockIdx.x; it < p.n_items && ok; it += gridDim.x, ++nit) {
        const Item x = item_of(p, it);
        // the pair's Q tiles, once the previous item's last S MMAs have read theirs
        if (!(ok = mbar_wait(&bar_qempty, (nit & 1) ^ 1, abort_flag, p.dev_err))) break;
        mbar_arrive_expect_tx(&bar_qfull, x.nh * kQTile);
        for (int hh = 0; hh < x.nh; ++hh) {
          tma_load_4d(s_q + hh * kQTile, &qmap, &bar_qfull, 0, x.h0 + hh, x.qt * 128, x.b);
          tma_load_4d(s_q + hh * kQTile + kHalf, &qmap, &bar_qfull, 64, x.h0 + hh, x.qt * 128, x.b);
        }
        for (int j = 0; j <= x.qt; ++j, ++nkv) {
          const int st = nkv % kKVStages;
          if (!(ok = mbar_wait(&bar_kvempty[st], ((nkv / kKVStages) & 1) ^ 1, abort_flag, p.dev_err))) break;
          uint8_t* kv = s_kv + st * kKV;
          mbar_arrive_expect_tx(&bar_kvfull[st], kKV);
          tma_load_4d(kv + 0 * kHalf, &kmap, &bar_kvfull[st], 0, x.g, j * 128, x.b);
          tma_load_4d(kv + 1 * kHalf, &kmap, &bar_kvfull[st], 64, x.g, j * 128, x.b);
          tma_load_4d(kv + 2 * kHalf, &vmap, &bar_kvfull[st], 0, x.g, j * 128, x.b);
          tma_load_4d(kv + 3 * kHalf, &vmap, &bar_kvfull[st], 64, x.g, j * 128, x.b);
        }
      }
      if (*abort_flag) {   // let loads in flight land before the CTA exits
        const uint64_t t0 = global_timer_ns();
        for (int i = max(0, nkv - kKVStages); i < nkv; ++i)
          while (!mbar_try_wait(&bar_kvfull[i % kKVStages], (i / kKVStages) & 1) &&
                 global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
          }
        if (nit > 0)
          while (!mbar_try_wait(&bar_qfull, (nit - 1) & 1) && global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
          }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ===================== tcgen05 issuer =====================
    // Per slot a state machine: S(j) needs the item's Q tiles (j = 0), K/V
    // block j and the slot's previous O MMA complete (S overwrites the P that
    // O read); O(j) needs P(j).  Whatever is ready is issued, O first.
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, 128, false, true);
      int64_t it = blockIdx.x;
      int nit = 0, kv_base = 0;          // items started; K/V ring index of the item's block 0
      Item x = it < p.n_items ? item_of(p, it) : Item{0, 0, 0, 0, 0};
      int js[2] = {0, 0}, jo[2] = {0, 0};       // next S / O block of each slot in the current item
      int ns[2] = {0, 0}, no[2] = {0, 0};       // S / O MMAs issued per slot (barrier phases)
      int s_last = 0, o_last = 0;               // slots whose last S / last O of the item is issued
      uint32_t spins = 0;
      uint64_t idle_since = 0;
      while (it < p.n_items) {
        bool progress = false;
        for (int s = 0; s < x.nh; ++s) {
          // ---- O(jo) of slot s
          if (jo[s] < js[s] && mbar_test_wait(&bar_pready[s], no[s] & 1)) {
            tc_fence_after();
            const int kvi = kv_base + jo[s];
            const uint32_t vb = smem_u32(s_kv + (kvi % kKVStages) * kKV + 2 * kHalf);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16_ts(tmem + s * 256 + 128, tmem + s * 256 + kk * 8, sdesc_sw128(vb + kk * 2048, kHalf, 1024),
                           idesc_o, (jo[s] > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&bar_ofull[s]);
            ++no[s];
            // the K/V block is free once every slot of the item has read it
            bool all = true;
            for (int s2 = 0; s2 < x.nh; ++s2) all = all && (s2 == s ? true : jo[s2] > jo[s]);
            if (all) umma_commit(&bar_kvempty[kvi % kKVStages]);
            if (++jo[s] > x.qt) ++o_last;
            progress = true;
          }
          // ---- S(js) of slot s
          if (js[s] <= x.qt && js[s] == jo[s]) {
            const int kvi = kv_base + js[s];
            const bool q_ok = js[s] > 0 || mbar_test_wait(&bar_qfull, nit & 1);
            const bool o_ok = no[s] == 0 || mbar_test_wait(&bar_ofull[s], (no[s] - 1) & 1);
            if (q_ok && o_ok && mbar_test_wait(&bar_kvfull[kvi % kKVStages], (kvi / kKVStages) & 1)) {
              tc_fence_after();
              const uint32_t qb = smem_u32(s_q + s * kQTile);
              const uint32_t kb = smem_u32(s_kv + (kvi % kKVStages) * kKV);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_bf16(tmem + s * 256, sdesc_sw128(qb + (kk >> 2) * kHalf + 32 * (kk & 3), 16, 1024),
                          sdesc_sw128(kb + (kk >> 2) * kHalf + 32 * (kk & 3), 16, 1024), idesc_s, kk > 0);
              umma_commit(&bar_sfull[s]);
              ++ns[s];
              if (++js[s] > x.qt && ++s_last == x.nh) umma_commit(&bar_qempty);   // Q tiles read by every slot
              progress = true;
            }
          }
        }
        if (o_last == x.nh) {          // the item's MMAs are all issued: next item
          kv_base += x.qt + 1;
          ++nit;
          it += gridDim.x;
          if (it < p.n_items) x = item_of(p, it);
          js[0] = js[1] = jo[0] = jo[1] = 0;
          s_last = o_last = 0;
          progress = true;
        }
        if (progress) {
          spins = 0;
        } else if ((++spins & 63u) == 0) {
          const uint64_t now = global_timer_ns();
          if (spins == 64) idle_since = now;
          if (*abort_flag) break;
          if (now - idle_since > MSA_WAIT_LIMIT_NS) {
            *abort_flag = 1;
            report(p.dev_err, MSA_DEVERR_TIMEOUT);
            break;
          }
        }
      }
      umma_commit(&bar_drain);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&bar_drain, 0) && global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
      }
    }
    __syncwarp();
  } else {
    // ===================== softmax + epilogue of slot s (thread = query row) =====================
    const int s = (warp - 2) >> 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t sbase = tmem + lane_addr + s * 256;     // S, then P (bf16 pairs) in its first 64 columns
    const uint32_t obase = sbase + 128;
    const float sc = p.scale_log2;
    int nS = 0, nO = 0;                                    // waits done on sfull / ofull of this slot
    bool alive = true;
    for (int64_t it = blockIdx.x; it < p.n_items && alive; it += gridDim.x) {
      const Item x = item_of(p, it);
      if (s >= x.nh) continue;                             // a single-head item: slot 1 idles
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j <= x.qt; ++j) {
        const bool ok_s = mbar_wait(&bar_sfull[s], nS & 1, abort_flag, p.dev_err);
        ++nS;
        if (!__all_sync(0xffffffffu, ok_s)) { alive = false; break; }
        tc_fence_after();
        // keys visible to row r in block j: all but in the diagonal block (c <= r)
        const int nvis = j < x.qt ? 128 : r + 1;
        float bm = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          tmem_ld32(sbase + cc * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (cc * 32 + e < nvis) bm = fmaxf(bm, __uint_as_float(v[e]));
        }
        bm *= sc;                                          // scale > 0: max of the scaled scores
        if (j == 0) {
          m = bm;
        } else if (bm > m + kRescale) {                    // rescale O and the sum to the new max
          const float alpha = fast_exp2(m - bm);
          l *= alpha;
          m = bm;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t v[32];
            tmem_ld32(obase + cc * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st32(obase + cc * 32, v);
          }
        }
        float lsum = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          tmem_ld32(sbase + cc * 32, v);
          tmem_ld_wait();
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 = (cc * 32 + e < nvis) ? fast_exp2(fmaf(__uint_as_float(v[e]), sc, -m)) : 0.f;
            const float p1 = (cc * 32 + e + 1 < nvis) ? fast_exp2(fmaf(__uint_as_float(v[e + 1]), sc, -m)) : 0.f;
            lsum += p0 + p1;
            pw[e >> 1] = pack_bf16x2(p0, p1);
          }
          tmem_st16(sbase + cc * 16, pw);                  // P columns 16 cc .. hold keys 32 cc ..
        }
        l += lsum;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_pready[s]);
      }
      if (!alive) break;
      // ---- epilogue: O(qt) complete -> O / l in bf16, LSE
      const bool ok_o = mbar_wait(&bar_ofull[s], (nO + x.qt) & 1, abort_flag, p.dev_err);
      nO += x.qt + 1;
      if (!__all_sync(0xffffffffu, ok_o)) break;
      tc_fence_after();
      const int i = x.qt * 128 + r;
      const float inv = 1.0f / l;
      __nv_bfloat16* orow = p.O + ((static_cast<int64_t>(x.b) * p.S + i) * p.Hq + x.h0 + s) * kD;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
        tmem_ld32(obase + cc * 32, v);
        tmem_ld_wait();
        if (i < p.S) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[e + 0]) * inv, __uint_as_float(v[e + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(v[e + 4]) * inv, __uint_as_float(v[e + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(v[e + 6]) * inv, __uint_as_float(v[e + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + cc * 32 + e) = w;
          }
        }
      }
      // the O loads above are complete (wait::ld) before this slot's next
      // pready arrive, which gates the next item's first O MMA into this slot
      tc_fence_before();
      if (i < p.S && p.LSE != nullptr)
        p.LSE[(static_cast<int64_t>(x.b) * p.S + i) * p.Hq + x.h0 + s] = (m + log2f(l)) * kLn2;
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

msa_status launch_dense_prefill(const msa_dense_prefill_args& a, cudaStream_t stream) {
  DeviceInfo dev;
  if (msa_status st = current_device(&dev); st != MSA_OK) return st;
  CUtensorMap qmap, kmap, vmap;
  {
    // Q as 4-D (d, h, s, b); box = 128 queries of one head, 64 columns
    const uint64_t dims[4] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(a.Hq), static_cast<uint64_t>(a.S),
                              static_cast<uint64_t>(a.B)};
    const uint64_t strides[3] = {static_cast<uint64_t>(a.Q_stride[2]) * 2, static_cast<uint64_t>(a.Q_stride[1]) * 2,
                                 static_cast<uint64_t>(a.Q_stride[0]) * 2};
    const uint32_t box[4] = {64, 1, 128, 1};
    if (msa_status st = encode_tiled_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.Q, dims, strides, box,
                                         CU_TENSOR_MAP_SWIZZLE_128B, "Q");
        st != MSA_OK)
      return st;
  }
  {
    // K, V as 4-D (d, g, s, b); box = 128 tokens of one group, 64 columns
    const uint64_t dims[4] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(a.Hkv), static_cast<uint64_t>(a.S),
                              static_cast<uint64_t>(a.B)};
    const uint32_t box[4] = {64, 1, 128, 1};
    const uint64_t ks[3] = {static_cast<uint64_t>(a.K_stride[2]) * 2, static_cast<uint64_t>(a.K_stride[1]) * 2,
                            static_cast<uint64_t>(a.K_stride[0]) * 2};
    const uint64_t vs[3] = {static_cast<uint64_t>(a.V_stride[2]) * 2, static_cast<uint64_t>(a.V_stride[1]) * 2,
                            static_cast<uint64_t>(a.V_stride[0]) * 2};
    if (msa_status st = encode_tiled_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.K, dims, ks, box,
                                         CU_TENSOR_MAP_SWIZZLE_128B, "K");
        st != MSA_OK)
      return st;
    if (msa_status st = encode_tiled_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.V, dims, vs, box,
                                         CU_TENSOR_MAP_SWIZZLE_128B, "V");
        st != MSA_OK)
      return st;
  }
  Params p;
  p.B = a.B; p.S = a.S; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = a.Hq / a.Hkv;
  p.nq = (a.S + 127) / 128;
  p.npairs = (p.G + 1) / 2;
  p.n_items = static_cast<int64_t>(p.nq) * a.B * a.Hkv * p.npairs;
  const float scale = a.softmax_scale > 0.f ? a.softmax_scale : 1.0f / sqrtf(static_cast<float>(a.D));
  p.scale_log2 = scale * kLog2e;
  p.O = static_cast<__nv_bfloat16*>(a.O);
  p.LSE = a.LSE;
  p.dev_err = a.dev_err;
  const size_t smem = 1024 + 2 * static_cast<size_t>(kQTile) + static_cast<size_t>(kKVStages) * kKV;
  if (smem > dev.max_smem_optin) return fail(MSA_ERR_UNSUPPORTED, "dense prefill: not enough shared memory");
  cudaError_t e = cudaFuncSetAttribute(dense_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(dense_prefill)");
  const int grid = static_cast<int>(std::min<int64_t>(dev.num_sms, p.n_items));
  dense_prefill_kernel<<<grid, kThreads, smem, stream>>>(qmap, kmap, vmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "dense_prefill_kernel launch");
  return MSA_OK;
}

}  // namespace msa
