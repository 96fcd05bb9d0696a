// attn_prefill.cu -- a3' + a4 + a6: causal sparse attention of a prefill,
// KV-block-major.
//
// Instead of walking queries and copying their selected KV blocks from HBM
// again and again, the outer loop walks KV blocks and the inner loop the
// queries that selected them; per-block partial outputs are recombined by a
// final log-sum-exp reduction ("MiniMax M3 preparado para inferencia en
// produccion", paragraph "KV-Block-Major").  Per query chunk:
//   1. count    how many (query, slot) pairs of the chunk selected each
//               (b, g, block j); empty slots get LSE_part = -inf;
//   2. scan     exclusive scan of the counts (CSR offsets) and of the number of
//               128-row tiles per block (rows = selecting queries x G heads);
//   3. fill     the CSR lists: entry = (query within chunk) * 64 + slot;
//   4. attend   persistent tcgen05 kernel over the tiles.  Per tile of 128
//               (query, head) rows of one (b, g, j): K_j and V_j are staged by
//               TMA once per block (double-buffered), the Q rows are gathered
//               with cp.async into a 128-byte-swizzled tile, then
//                 S = Q K_j^T                (M=128, N=128, K=D; TMEM)
//                 P = exp(S - rowmax), masked t <= i      (one thread per row)
//                 O = P V_j                  (V as the MN-major operand)
//               and each row writes its normalised partial O and
//               LSE = m + ln l for its (query, head, slot);
//   5. merge    the log-sum-exp merge kernel combines the k partials per
//               (query, head) into O (bf16) and LSE.
// Keys of block j seen by query i are t in [j*Bk, (j+1)*Bk) with t <= i.
#include "msa_internal.h"
#include "msa_ptx.cuh"

namespace msa {
namespace {

constexpr int kAttnThreads = 352;     // w0-1 Q gather + K/V TMA, w2-5 and w6-9 softmax/epilogue, w10 MMA
constexpr int kMmaWarp = 10;
constexpr int kHalf = 128 * 64 * 2;   // 16 KiB
constexpr int kQStage = 2 * kHalf;    // 32 KiB: 128 rows x 128 (Q, then P)
constexpr int kKV = 4 * kHalf;        // 64 KiB: K (2 halves) + V (2 halves)
constexpr int kTmemCols = 512;        // 2 slots x (S 128 + O 128)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct CsrParams {
  int S, Hkv, Hq, G, k, nb;
  int64_t q0;           // first flattened query (b*S + i) of the chunk
  int nq;               // queries in the chunk
  const int32_t* sel;
  const int32_t* count;
  int32_t* cnt;         // [n_items]
  int32_t* cursor;      // [n_items]
  int32_t* off;         // [n_items + 1]
  int32_t* tile_off;    // [n_items + 1]
  int32_t* list;
  float* lse_part;
  int32_t* dev_err;
};

// one thread per (query in chunk, group, slot)
__global__ void csr_count_kernel(const CsrParams p) {
  const int64_t total = static_cast<int64_t>(p.nq) * p.Hkv * p.k;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int s = static_cast<int>(e % p.k);
    const int64_t qg = e / p.k;
    const int g = static_cast<int>(qg % p.Hkv);
    const int qi = static_cast<int>(qg / p.Hkv);
    const int64_t bs = p.q0 + qi;
    const int b = static_cast<int>(bs / p.S), i = static_cast<int>(bs % p.S);
    const int c = p.count[bs * p.Hkv + g];
    bool live = false;
    if (s < c) {
      const int j = p.sel[(bs * p.Hkv + g) * p.k + s];
      if (j < 0 || j > i / kBk) {
        report(p.dev_err, MSA_DEVERR_BAD_SEL);
      } else {
        atomicAdd(&p.cnt[(static_cast<int64_t>(b) * p.Hkv + g) * p.nb + j], 1);
        live = true;
      }
    }
    if (!live) {
      for (int h = 0; h < p.G; ++h)
        p.lse_part[(static_cast<int64_t>(qi) * p.Hq + g * p.G + h) * p.k + s] = -INFINITY;
    }
  }
}

// single CTA: exclusive scans of counts and of tiles per item
__global__ void __launch_bounds__(1024) csr_scan_kernel(const CsrParams p, int64_t n_items) {
  __shared__ int64_t s_sum[32][2];
  const int tid = threadIdx.x;
  const int64_t per = (n_items + 1023) / 1024;
  const int64_t i0 = tid * per, i1 = min(n_items, i0 + per);
  int64_t c = 0, t = 0;
  for (int64_t x = i0; x < i1; ++x) {
    const int v = p.cnt[x];
    c += v;
    t += (static_cast<int64_t>(v) * p.G + 127) / 128;
  }
  // inclusive warp scans, then a scan of the 32 warp totals
  const int lane = tid & 31, wid = tid >> 5;
  int64_t ic = c, it = t;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t xc = __shfl_up_sync(0xffffffffu, ic, o);
    const int64_t xt = __shfl_up_sync(0xffffffffu, it, o);
    if (lane >= o) { ic += xc; it += xt; }
  }
  if (lane == 31) { s_sum[wid][0] = ic; s_sum[wid][1] = it; }
  __syncthreads();
  if (wid == 0) {
    int64_t wc = s_sum[lane][0], wt = s_sum[lane][1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t xc = __shfl_up_sync(0xffffffffu, wc, o);
      const int64_t xt = __shfl_up_sync(0xffffffffu, wt, o);
      if (lane >= o) { wc += xc; wt += xt; }
    }
    s_sum[lane][0] = wc;   // inclusive over warps
    s_sum[lane][1] = wt;
    if (lane == 31) {
      p.off[n_items] = static_cast<int32_t>(wc);
      p.tile_off[n_items] = static_cast<int32_t>(wt);
    }
  }
  __syncthreads();
  c = ic - c + (wid > 0 ? s_sum[wid - 1][0] : 0);   // exclusive prefix of this thread
  t = it - t + (wid > 0 ? s_sum[wid - 1][1] : 0);
  for (int64_t x = i0; x < i1; ++x) {
    const int v = p.cnt[x];
    p.off[x] = static_cast<int32_t>(c);
    p.cursor[x] = static_cast<int32_t>(c);
    p.tile_off[x] = static_cast<int32_t>(t);
    c += v;
    t += (static_cast<int64_t>(v) * p.G + 127) / 128;
  }
}

__global__ void csr_fill_kernel(const CsrParams p) {
  const int64_t total = static_cast<int64_t>(p.nq) * p.Hkv * p.k;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int s = static_cast<int>(e % p.k);
    const int64_t qg = e / p.k;
    const int g = static_cast<int>(qg % p.Hkv);
    const int qi = static_cast<int>(qg / p.Hkv);
    const int64_t bs = p.q0 + qi;
    const int b = static_cast<int>(bs / p.S), i = static_cast<int>(bs % p.S);
    const int c = p.count[bs * p.Hkv + g];
    if (s >= c) continue;
    const int j = p.sel[(bs * p.Hkv + g) * p.k + s];
    if (j < 0 || j > i / kBk) continue;
    const int pos = atomicAdd(&p.cursor[(static_cast<int64_t>(b) * p.Hkv + g) * p.nb + j], 1);
    p.list[pos] = qi * 64 + s;
  }
}

// ---------------------------------------------------------------------------
// attention over tiles
// ---------------------------------------------------------------------------

struct AttnParams {
  int S, Hq, Hkv, G, k, nb;
  int64_t q0;
  int64_t n_items;
  float scale_log2;
  const __nv_bfloat16* Q;
  int64_t qs0, qs1, qs2;
  const int32_t* off;
  const int32_t* tile_off;
  const int32_t* list;
  __nv_bfloat16* o_part;
  float* lse_part;
  int32_t* dev_err;
};

struct TileInfo {
  int item, b, g, j, row0, nrows, kvb, kv_new, kv_release, ebase;
};

__device__ __forceinline__ int64_t find_item(const AttnParams& p, int64_t t) {
  int64_t lo = 0, hi = p.n_items - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (p.tile_off[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// packed fp32 helpers and the hardware base-2 exponential
__device__ __forceinline__ uint64_t pack2f(float x, float y) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ void unpack2f(uint64_t v, float& x, float& y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool full) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(full ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kAttnThreads, 1)
attn_prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_kv = smem;                    // [2] x (K0 K1 V0 V1)
  uint8_t* s_q = smem + 2 * kKV;           // [2] x (Q then P), 128 rows x 128

  __shared__ __align__(8) uint64_t bar_qfull[2], bar_qempty[2], bar_kvfull[2], bar_kvempty[2];
  __shared__ __align__(8) uint64_t bar_sfull[2], bar_pready[2], bar_ofull[2], bar_tfree[2], bar_drain;
  __shared__ TileInfo s_info[2];
  __shared__ const __nv_bfloat16* s_rowsrc[2][128];
  __shared__ int2 s_rinfo[2][128];         // per tile row: query position i, partial row (-1: padding)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_fail[2], s_gfail[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_qfull[i], 32); mbar_init(&bar_qempty[i], 1);
      mbar_init(&bar_kvfull[i], 1); mbar_init(&bar_kvempty[i], 1);
      mbar_init(&bar_sfull[i], 1); mbar_init(&bar_pready[i], 4);
      mbar_init(&bar_ofull[i], 1); mbar_init(&bar_tfree[i], 4);
    }
    mbar_init(&bar_drain, 1);
    s_abort = 0;
    s_fail[0] = s_fail[1] = 0;
    s_gfail[0] = s_gfail[1] = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&s_tmem, kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;

  const int64_t total_tiles = p.tile_off[p.n_items];
  const int64_t per = (total_tiles + gridDim.x - 1) / gridDim.x;
  const int64_t t0 = min(total_tiles, static_cast<int64_t>(blockIdx.x) * per);
  const int64_t t1 = min(total_tiles, t0 + per);
  const int ntiles = static_cast<int>(t1 - t0);

  if (warp < 2) {
    // ===================== producers: warp gi owns Q stage gi (tiles n = gi mod 2) =====================
    // Each warp resolves its tile's rows (query, head, slot), gathers the Q rows,
    // waits for its own copies, fences them for the tensor core and releases the
    // stage; the two warps keep two gathers in flight.
    const int gi = warp;
    int64_t prev_item = -1;
    int kvn = 0, last_kv = -1;   // last K/V load issued by this warp
    // tiles of this CTA are contiguous: walk their items forward instead of searching
    int64_t item = ntiles > 0 ? find_item(p, t0) : 0;
    for (int n = 0; n < ntiles; ++n) {
      const int64_t t = t0 + n;
      while (p.tile_off[item + 1] <= t) ++item;
      const bool kv_new = item != prev_item;
      prev_item = item;
      if (kv_new) ++kvn;
      if ((n & 1) != gi) continue;
      const int st = gi;
      const int b = static_cast<int>(item / (static_cast<int64_t>(p.Hkv) * p.nb));
      const int g = static_cast<int>((item / p.nb) % p.Hkv);
      const int j = static_cast<int>(item % p.nb);
      const int ebase = p.off[item];
      const int rows_item = (p.off[item + 1] - ebase) * p.G;
      const int row0 = static_cast<int>(t - p.tile_off[item]) * 128;
      const int nrows = min(128, rows_item - row0);
      const int kvb = (kvn - 1) & 1;
      // rows of this tile (4 per lane), resolved before waiting for the stage
      const __nv_bfloat16* src[4];
      int2 ri[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int rr = lane + 32 * x;
        src[x] = nullptr;
        ri[x] = make_int2(0, -1);
        if (rr < nrows) {
          const int rho = row0 + rr;
          const int ent = p.list[ebase + rho / p.G];
          const int qi = ent >> 6;
          const int hq = g * p.G + rho % p.G;
          const int i = static_cast<int>((p.q0 + qi) % p.S);
          src[x] = p.Q + static_cast<int64_t>(b) * p.qs0 + static_cast<int64_t>(i) * p.qs1 +
                   static_cast<int64_t>(hq) * p.qs2;
          ri[x] = make_int2(i, (qi * p.Hq + hq) * p.k + (ent & 63));
        }
      }
      bool ok = true;
      if (lane == 0) {
        const bool release = (n + 1 == ntiles) || p.tile_off[item + 1] <= t + 1;
        ok = mbar_wait(&bar_qempty[st], ((n >> 1) & 1) ^ 1, abort_flag, p.dev_err);
        if (ok && kv_new) {
          ok = mbar_wait(&bar_kvempty[kvb], (((kvn - 1) >> 1) & 1) ^ 1, abort_flag, p.dev_err);
          if (ok) {
            uint8_t* kvbuf = s_kv + kvb * kKV;
            mbar_arrive_expect_tx(&bar_kvfull[kvb], kKV);
            tma_load_4d(kvbuf + 0 * kHalf, &kmap, &bar_kvfull[kvb], 0, g, j * kBk, b);
            tma_load_4d(kvbuf + 1 * kHalf, &kmap, &bar_kvfull[kvb], 64, g, j * kBk, b);
            tma_load_4d(kvbuf + 2 * kHalf, &vmap, &bar_kvfull[kvb], 0, g, j * kBk, b);
            tma_load_4d(kvbuf + 3 * kHalf, &vmap, &bar_kvfull[kvb], 64, g, j * kBk, b);
            last_kv = kvn - 1;
          }
        }
        s_info[st] = TileInfo{static_cast<int>(item), b, g, j, row0, nrows, kvb, kv_new ? 1 : 0, release ? 1 : 0,
                              ebase};
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;                      // the warp stops together
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        s_rowsrc[st][lane + 32 * x] = src[x];
        s_rinfo[st][lane + 32 * x] = ri[x];
      }
      __syncwarp();
      const uint32_t qbase = smem_u32(s_q + st * kQStage);
#pragma unroll 8
      for (int u = 0; u < 64; ++u) {
        const int idx = lane + 32 * u;     // 2048 chunks of 16 B
        const int rr = idx >> 4, c = idx & 15;
        const __nv_bfloat16* sp = s_rowsrc[st][rr];
        const uint32_t dst = qbase + (c >> 3) * kHalf + sw128_offset(rr, c & 7);
        cp_async16(dst, sp ? static_cast<const void*>(sp + c * 8) : static_cast<const void*>(p.Q), sp != nullptr);
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(&bar_qfull[st]);
      __syncwarp();                        // s_rowsrc[st] is rewritten two tiles later
    }
    if (*abort_flag && lane == 0 && last_kv >= 0) {   // let this warp's last K/V load land
      uint64_t tt = global_timer_ns();
      while (!mbar_try_wait(&bar_kvfull[last_kv & 1], (last_kv >> 1) & 1) &&
             global_timer_ns() - tt < MSA_WAIT_LIMIT_NS) {
      }
    }
  } else if (warp == kMmaWarp) {
    // ===================== tcgen05 issuer =====================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, 128, false, true);
      int kvn = 0;
      bool ok = true;
      auto issue_s = [&](int n) -> bool {
        const int st = n & 1, slot = n & 1;
        if (!mbar_wait(&bar_qfull[st], (n >> 1) & 1, abort_flag, p.dev_err)) return false;
        const TileInfo inf = s_info[st];
        if (inf.kv_new) {
          ++kvn;
          if (!mbar_wait(&bar_kvfull[inf.kvb], ((kvn - 1) >> 1) & 1, abort_flag, p.dev_err)) return false;
        }
        if (!mbar_wait(&bar_tfree[slot], ((n >> 1) & 1) ^ 1, abort_flag, p.dev_err)) return false;
        tc_fence_after();
        const uint32_t qb = smem_u32(s_q + st * kQStage);
        const uint32_t kb = smem_u32(s_kv + inf.kvb * kKV);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t o = (kk >> 2) * kHalf + 32 * (kk & 3);
          umma_bf16(tmem + slot * 256, sdesc_sw128(qb + o, 16, 1024), sdesc_sw128(kb + o, 16, 1024), idesc_s, kk > 0);
        }
        umma_commit(&bar_sfull[slot]);
        return true;
      };
      auto issue_o = [&](int n) -> bool {
        const int st = n & 1, slot = n & 1;
        if (!mbar_wait(&bar_pready[slot], (n >> 1) & 1, abort_flag, p.dev_err)) return false;
        tc_fence_after();
        const TileInfo inf = s_info[st];
        const uint32_t pb = smem_u32(s_q + st * kQStage);
        const uint32_t vb = smem_u32(s_kv + inf.kvb * kKV + 2 * kHalf);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t po = (kk >> 2) * kHalf + 32 * (kk & 3);
          umma_bf16(tmem + slot * 256 + 128, sdesc_sw128(pb + po, 16, 1024), sdesc_sw128(vb + kk * 2048, kHalf, 1024),
                    idesc_o, kk > 0);
        }
        umma_commit(&bar_ofull[slot]);
        umma_commit(&bar_qempty[st]);
        if (inf.kv_release) umma_commit(&bar_kvempty[inf.kvb]);
        return true;
      };
      if (ntiles > 0) ok = issue_s(0);
      for (int n = 0; n < ntiles && ok; ++n) {
        if (n + 1 < ntiles) ok = issue_s(n + 1);
        if (ok) ok = issue_o(n);
      }
      umma_commit(&bar_drain);
      uint64_t tt = global_timer_ns();
      while (!mbar_try_wait(&bar_drain, 0) && global_timer_ns() - tt < MSA_WAIT_LIMIT_NS) {
      }
    }
    __syncwarp();
  } else {
    // ===================== softmax + epilogue: warpgroup wg (warps 2-5 / 6-9) owns tiles n = wg mod 2 =====
    const int wg = (warp - 2) >> 2;
    const int bar_id = 1 + wg;
    const int q = warp & 3;
    const int r = q * 32 + lane;                     // tile row = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const int st = wg, slot = wg;
    for (int n = wg; n < ntiles; n += 2) {
      const uint32_t ph = (n >> 1) & 1;
      if (!mbar_wait(&bar_qfull[st], ph, abort_flag, p.dev_err)) s_fail[wg] = 1;
      named_bar_sync(bar_id, 128);
      if (s_fail[wg]) break;
      const int j = s_info[st].j;
      const int2 ri = s_rinfo[st][r];
      const bool valid = ri.y >= 0;
      // keys of this block visible to the row: t <= i
      const int nvis = valid ? min(kBk, ri.x - j * kBk + 1) : kBk;
      if (!mbar_wait(&bar_sfull[slot], ph, abort_flag, p.dev_err)) s_fail[wg] = 1;
      named_bar_sync(bar_id, 128);
      if (s_fail[wg]) break;
      tc_fence_after();
      const uint32_t sbase = tmem + lane_addr + slot * 256;
      uint8_t* prow = s_q + st * kQStage;
      const float sc = p.scale_log2;
      float m = -INFINITY, l = 0.f;
      // the branch must be warp-uniform: the TMEM loads inside are warp-collective
      if (__all_sync(0xffffffffu, nvis == kBk)) {
        // whole block visible to every row of the warp: no masking
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v[2][32];
          tmem_ld32(sbase + half * 64, v[0]);
          tmem_ld32(sbase + half * 64 + 32, v[1]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; e += 2) m = max3f(m, __uint_as_float(v[c][e]), __uint_as_float(v[c][e + 1]));
        }
        m *= sc;   // scale > 0: max of scaled scores
        uint64_t l2 = 0ull;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v[2][32];
          tmem_ld32(sbase + half * 64, v[0]);
          tmem_ld32(sbase + half * 64 + 32, v[1]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float p0 = fast_exp2(fmaf(__uint_as_float(v[c][e]), sc, -m));
              const float p1 = fast_exp2(fmaf(__uint_as_float(v[c][e + 1]), sc, -m));
              l2 = add2(l2, pack2f(p0, p1));
              pk[e >> 1] = pack_bf16x2(p0, p1);
            }
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const int ch = (half * 2 + c) * 4 + x;
              *reinterpret_cast<uint4*>(prow + (ch >> 3) * kHalf + sw128_offset(r, ch & 7)) =
                  make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
            }
          }
        }
        float la, lb;
        unpack2f(l2, la, lb);
        l = la + lb;
      } else {
        // some row of the warp sees only part of the block (its own block): keys t <= i
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          tmem_ld32(sbase + cc * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (cc * 32 + e < nvis) m = fmaxf(m, __uint_as_float(v[e]));
        }
        m *= sc;
        // same pairwise accumulation order as the unmasked path, so a fully
        // visible row gets identical bits whichever path its warp takes
        uint64_t l2 = 0ull;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          tmem_ld32(sbase + cc * 32, v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 = (cc * 32 + e < nvis) ? fast_exp2(fmaf(__uint_as_float(v[e]), sc, -m)) : 0.f;
            const float p1 = (cc * 32 + e + 1 < nvis) ? fast_exp2(fmaf(__uint_as_float(v[e + 1]), sc, -m)) : 0.f;
            l2 = add2(l2, pack2f(p0, p1));
            pk[e >> 1] = pack_bf16x2(p0, p1);
          }
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int ch = cc * 4 + x;
            *reinterpret_cast<uint4*>(prow + (ch >> 3) * kHalf + sw128_offset(r, ch & 7)) =
                make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
          }
        }
        float la, lb;
        unpack2f(l2, la, lb);
        l = la + lb;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pready[slot]);
      if (!mbar_wait(&bar_ofull[slot], ph, abort_flag, p.dev_err)) s_fail[wg] = 1;
      named_bar_sync(bar_id, 128);
      if (s_fail[wg]) break;
      tc_fence_after();
      const float inv = 1.0f / l;
      __nv_bfloat16* orow = p.o_part + static_cast<int64_t>(valid ? ri.y : 0) * kD;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
        tmem_ld32(sbase + 128 + cc * 32, v);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          const uint64_t inv2 = pack2f(inv, inv);
          for (int e = 0; e < 32; e += 8) {
            uint32_t w[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              float a, b;
              unpack2f(mul2(pack2f(__uint_as_float(v[e + 2 * x]), __uint_as_float(v[e + 2 * x + 1])), inv2), a, b);
              w[x] = pack_bf16x2(a, b);
            }
            *reinterpret_cast<uint4*>(orow + cc * 32 + e) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (valid) p.lse_part[ri.y] = (m + log2f(l)) * kLn2;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_tfree[slot]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

struct WsLayout {
  size_t cnt, cursor, off, tile_off, list, o_part, lse_part, total;
};

WsLayout ws_layout(const msa_prefill_args& a, int64_t cq) {
  const int64_t nb = (a.S + kBk - 1) / kBk;
  const int64_t n_items = static_cast<int64_t>(a.B) * a.Hkv * nb;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  WsLayout L;
  size_t o = 0;
  L.cnt = o; o = al(o + n_items * 4);
  L.cursor = o; o = al(o + n_items * 4);
  L.off = o; o = al(o + (n_items + 1) * 4);
  L.tile_off = o; o = al(o + (n_items + 1) * 4);
  L.list = o; o = al(o + static_cast<size_t>(cq) * a.Hkv * a.k * 4);
  L.o_part = o; o = al(o + static_cast<size_t>(cq) * a.Hq * a.k * kD * 2);   // bf16 partials
  L.lse_part = o; o = al(o + static_cast<size_t>(cq) * a.Hq * a.k * 4);
  L.total = o + 256;
  return L;
}

}  // namespace

size_t attn_prefill_workspace_size(const msa_prefill_args& a, int64_t chunk_queries) {
  return ws_layout(a, chunk_queries).total;
}

msa_status launch_attn_prefill(const msa_prefill_args& a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  DeviceInfo dev;
  if (msa_status st = current_device(&dev); st != MSA_OK) return st;
  const int64_t total_q = static_cast<int64_t>(a.B) * a.S;
  // largest chunk that fits the workspace
  int64_t lo = 1, hi = total_q;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) / 2;
    if (ws_layout(a, mid).total <= ws_bytes) lo = mid; else hi = mid - 1;
  }
  const int64_t cq = lo;
  const WsLayout L = ws_layout(a, cq);
  const int64_t nb = (a.S + kBk - 1) / kBk;
  const int64_t n_items = static_cast<int64_t>(a.B) * a.Hkv * nb;
  if (cq * 64 >= (int64_t(1) << 31) || cq * a.Hq * a.k >= (int64_t(1) << 31) || n_items >= (int64_t(1) << 31))
    return fail(MSA_ERR_UNSUPPORTED, "prefill attention: problem too large for 32-bit lists");
  uint8_t* w = static_cast<uint8_t*>(ws);

  CUtensorMap kmap, vmap;
  const uint64_t dims[4] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(a.Hkv), static_cast<uint64_t>(a.S),
                            static_cast<uint64_t>(a.B)};
  const uint32_t box[4] = {64, 1, 128, 1};
  {
    const uint64_t strides[3] = {static_cast<uint64_t>(a.K_stride[2]) * 2, static_cast<uint64_t>(a.K_stride[1]) * 2,
                                 static_cast<uint64_t>(a.K_stride[0]) * 2};
    if (msa_status st = encode_tiled_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.K, dims, strides, box,
                                         CU_TENSOR_MAP_SWIZZLE_128B, "K");
        st != MSA_OK)
      return st;
  }
  {
    const uint64_t strides[3] = {static_cast<uint64_t>(a.V_stride[2]) * 2, static_cast<uint64_t>(a.V_stride[1]) * 2,
                                 static_cast<uint64_t>(a.V_stride[0]) * 2};
    if (msa_status st = encode_tiled_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.V, dims, strides, box,
                                         CU_TENSOR_MAP_SWIZZLE_128B, "V");
        st != MSA_OK)
      return st;
  }
  const size_t smem = 1024 + 2 * static_cast<size_t>(kKV) + 2 * static_cast<size_t>(kQStage);
  if (smem > dev.max_smem_optin) return fail(MSA_ERR_UNSUPPORTED, "prefill attention: not enough shared memory");
  cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attn_prefill)");

  const int G = a.Hq / a.Hkv;
  const float scale = a.softmax_scale > 0.f ? a.softmax_scale : 1.0f / sqrtf(static_cast<float>(a.D));
  for (int64_t q0 = 0; q0 < total_q; q0 += cq) {
    const int nq = static_cast<int>(std::min<int64_t>(cq, total_q - q0));
    CsrParams c;
    c.S = a.S; c.Hkv = a.Hkv; c.Hq = a.Hq; c.G = G; c.k = a.k; c.nb = static_cast<int>(nb);
    c.q0 = q0; c.nq = nq;
    c.sel = a.sel; c.count = a.count;
    c.cnt = reinterpret_cast<int32_t*>(w + L.cnt);
    c.cursor = reinterpret_cast<int32_t*>(w + L.cursor);
    c.off = reinterpret_cast<int32_t*>(w + L.off);
    c.tile_off = reinterpret_cast<int32_t*>(w + L.tile_off);
    c.list = reinterpret_cast<int32_t*>(w + L.list);
    c.lse_part = reinterpret_cast<float*>(w + L.lse_part);
    c.dev_err = a.dev_err;
    e = cudaMemsetAsync(c.cnt, 0, n_items * 4, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(prefill counts)");
    const int64_t work = static_cast<int64_t>(nq) * a.Hkv * a.k;
    const int grid_w = static_cast<int>(std::min<int64_t>((work + 255) / 256, 8 * dev.num_sms));
    csr_count_kernel<<<grid_w, 256, 0, stream>>>(c);
    csr_scan_kernel<<<1, 1024, 0, stream>>>(c, n_items);
    csr_fill_kernel<<<grid_w, 256, 0, stream>>>(c);

    AttnParams p;
    p.S = a.S; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = G; p.k = a.k; p.nb = static_cast<int>(nb);
    p.q0 = q0; p.n_items = n_items;
    p.scale_log2 = scale * kLog2e;
    p.Q = static_cast<const __nv_bfloat16*>(a.Q);
    p.qs0 = a.Q_stride[0]; p.qs1 = a.Q_stride[1]; p.qs2 = a.Q_stride[2];
    p.off = c.off; p.tile_off = c.tile_off; p.list = c.list;
    p.o_part = reinterpret_cast<__nv_bfloat16*>(w + L.o_part);
    p.lse_part = c.lse_part;
    p.dev_err = a.dev_err;
    attn_prefill_kernel<<<dev.num_sms, kAttnThreads, smem, stream>>>(kmap, vmap, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "prefill attention launch");
    msa_status st = launch_lse_merge_bf16(p.o_part, p.lse_part, static_cast<int64_t>(nq) * a.Hq, a.k, kD,
                                          static_cast<__nv_bfloat16*>(a.O) + q0 * a.Hq * kD,
                                          a.LSE != nullptr ? a.LSE + q0 * a.Hq : nullptr, stream);
    if (st != MSA_OK) return st;
  }
  return MSA_OK;
}

}  // namespace msa
