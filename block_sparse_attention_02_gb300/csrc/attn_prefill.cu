// attn_prefill.cu -- a3' + a4 + a6: causal sparse attention of a prefill,
// KV-block-major.
//
// Instead of walking queries and copying their selected KV blocks from HBM
// again and again, the outer loop walks KV blocks and the inner loop the
// queries that selected them; per-block partial outputs are recombined by a
// final log-sum-exp reduction ("MiniMax M3 preparado para inferencia en
// produccion", paragraph "KV-Block-Major").  An item is one (b, g, block j);
// its entries are the queries that selected it.  A tile holds 16 entries of one
// item; entry e owns tile rows 8e .. 8e+7, of which the first G are its G query
// heads of group g (the rest are padding).  In shared memory entry e is one
// 2 KiB block: its 8 rows of columns 0-63, then of columns 64-127, each an
// 8-row 128-byte-swizzled atom, loaded by a single TMA box.  Per query chunk:
//   1. count    how many (query, slot) pairs of the chunk selected each item;
//               empty slots are marked in the slot map;
//   2. scan     CSR offsets, the number of tiles per item, and one descriptor
//               per tile (item, entries, ordinal of the item, first/last flags);
//   3. fill     the entry table in tile order (flattened query b*S+i of every
//               tile entry) and the slot map (query, g, slot) -> first row;
//   4. attend   persistent tcgen05 kernel over the tiles.  Per tile: K_j and
//               V_j are staged by TMA once per item (double-buffered), each
//               entry's query rows by one TMA box (three Q stages), then
//                 S = Q K_j^T                (M=128, N=128, K=D; TMEM)
//                 P = exp(S - rowmax), masked t <= i, written back to TMEM
//                 O = P V_j                  (P from TMEM, V as MN-major B)
//               and each valid row writes its normalised partial O (bf16) and
//               LSE = m + ln l at its tile row;
//   5. merge    per (query, head): the log-sum-exp merge of its k partials,
//               found through the slot map.
// Keys of block j seen by query i are t in [j*Bk, (j+1)*Bk) with t <= i.
// A chunk over a paged cache (MSA_MODE_CHUNK) differs only in where things
// are: query i of sequence b sits at position q_pos[b] + i (the causal limit),
// and block j of sequence b is page seq_pt[b][j] of the K/V pools (carried in
// the tile descriptor, so the producer needs no extra load).
#include <algorithm>

#include "msa_internal.h"
#include "msa_ptx.cuh"

namespace msa {
namespace {

constexpr int kProducerWarp = 0;      // w0: Q and K/V TMA
constexpr int kMmaWarp = 1;           // w1: tcgen05 issuer
constexpr int kSoftmax0 = 2;          // w2-5 and w6-9: softmax/epilogue warpgroups
constexpr int kAttnThreads = 10 * 32;
constexpr int kQStages = 3;
constexpr int kEntries = 16;          // queries (entries) per tile, 8 rows each
constexpr int kHalf = 128 * 64 * 2;   // 16 KiB: 128 rows x 64 bf16, 128-byte swizzled
constexpr int kQStage = 2 * kHalf;    // 32 KiB: 128 rows x 128
constexpr int kKV = 4 * kHalf;        // 64 KiB: K (2 halves) + V (2 halves)
constexpr int kEntryPart = 16 * 8 * 8; // bf16 elements reserved per entry's partial (16 chunks x G <= 8 rows x 8)
constexpr int kTmemCols = 512;        // 2 slots x (S/P 128 + O 128)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

constexpr int kTileFirst = 1;         // tile_info.w: first tile of its item
constexpr int kTileLast = 2;          //              last tile of its item
constexpr int kTilePageShift = 2;     //              page id of the block (chunk) above the flags

struct CsrParams {
  int S, Hkv, Hq, G, k, nb;
  int chunk;            // 1: queries at q_pos[b] + i, blocks are pages seq_pt[b][j]
  const int32_t* q_pos;
  const int32_t* seq_pt;
  int64_t max_pages, num_pages;
  int64_t q0;           // first flattened query (b*S + i) of the chunk
  int nq;               // queries in the chunk
  const int32_t* sel;
  const int32_t* count;
  int32_t* cnt;         // [n_items]
  int32_t* cursor;      // [n_items]
  int32_t* off;         // [n_items + 1]
  int32_t* tile_off;    // [n_items + 1]
  int32_t* ord;         // [n_items]: ordinal of the item among the non-empty ones
  int4* tile_info;      // [tiles]: item, entries, ordinal of the item, first/last flags
  int32_t* tile_q;      // [tiles * 16]: flattened query b*S+i of each tile entry
  int32_t* where;       // [nq, Hkv, k]: first tile row of the (query, g, slot) entry, -1 if empty
  int32_t* dev_err;
};

// Entry e of the chunk as (query in chunk, group, slot).  Lanes of a warp
// take 32 consecutive queries at the same (group, slot): neighbouring queries
// mostly select the same block there, so their counter updates combine into
// one atomic per distinct block (the hot blocks get one update per warp, not
// one per query).  `where` keeps the (query, group, slot) order.
struct CsrEntry {
  int64_t e;     // index into where[nq, Hkv, k]
  int64_t item;  // (b, g, j) item of the selected block, -1 if the slot is empty
  int64_t bs;    // flattened query b*S + i
  int page;      // chunk: page of the block
};
__device__ __forceinline__ CsrEntry csr_entry(const CsrParams& p, int64_t t, bool report_bad) {
  const int qi = static_cast<int>(t % p.nq);
  const int64_t rest = t / p.nq;
  const int g = static_cast<int>(rest % p.Hkv), s = static_cast<int>(rest / p.Hkv);
  CsrEntry x;
  x.e = (static_cast<int64_t>(qi) * p.Hkv + g) * p.k + s;
  x.bs = p.q0 + qi;
  x.item = -1;
  x.page = 0;
  const int b = static_cast<int>(x.bs / p.S), i = static_cast<int>(x.bs % p.S);
  if (s < p.count[x.bs * p.Hkv + g]) {
    const int j = p.sel[(x.bs * p.Hkv + g) * p.k + s];
    const int64_t pos = p.chunk ? static_cast<int64_t>(p.q_pos[b]) + i : i;
    if (j < 0 || pos < 0 || j > pos / kBk || j >= p.nb) {
      if (report_bad) report(p.dev_err, MSA_DEVERR_BAD_SEL);
    } else if (p.chunk) {
      const int page = p.seq_pt[b * p.max_pages + j];
      if (page < 0 || page >= p.num_pages) {
        if (report_bad) report(p.dev_err, MSA_DEVERR_BAD_PAGE);
      } else {
        x.item = (static_cast<int64_t>(b) * p.Hkv + g) * p.nb + j;
        x.page = page;
      }
    } else {
      x.item = (static_cast<int64_t>(b) * p.Hkv + g) * p.nb + j;
    }
  }
  return x;
}

__global__ void csr_count_kernel(const CsrParams p) {
  const int64_t total = static_cast<int64_t>(p.nq) * p.Hkv * p.k;
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // the loop is warp-uniform: every lane takes part in the match below
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); base < total;
       base += stride) {
    const int64_t t = base + lane;
    CsrEntry x{0, -1, 0, 0};
    if (t < total) x = csr_entry(p, t, true);
    const unsigned grp = __match_any_sync(0xffffffffu, static_cast<int>(x.item));
    if (x.item >= 0 && lane == __ffs(grp) - 1) atomicAdd(&p.cnt[x.item], __popc(grp));
    if (t < total && x.item < 0) p.where[x.e] = -1;
  }
}

__device__ __forceinline__ int tiles_of(int c) { return (c + kEntries - 1) / kEntries; }

// single CTA: exclusive scans of entries, tiles and non-empty items, one pass
// over tiles of 4096 items (4 consecutive items per thread, 16-byte loads and
// stores) with a block-wide scan per tile and a running carry.  Totals fit in
// int32: entries and tile rows are checked against 2^31 at launch.
constexpr int kScanThreads = 1024;
constexpr int kScanPer = 4;

__device__ __forceinline__ void scan_store4(int32_t* a, int64_t x0, int64_t n, const int (&v)[kScanPer]) {
  if (x0 + kScanPer <= n) {
    *reinterpret_cast<int4*>(a + x0) = make_int4(v[0], v[1], v[2], v[3]);
  } else {
#pragma unroll
    for (int u = 0; u < kScanPer; ++u)
      if (x0 + u < n) a[x0 + u] = v[u];
  }
}

__global__ void __launch_bounds__(kScanThreads) csr_scan_kernel(const CsrParams p, int64_t n_items) {
  __shared__ int s_sum[32][3];
  __shared__ int s_carry[3];                     // entries, tiles, non-empty items before this tile
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) s_carry[0] = s_carry[1] = s_carry[2] = 0;
  __syncthreads();
  for (int64_t base = 0; base < n_items; base += kScanThreads * kScanPer) {
    const int64_t x0 = base + static_cast<int64_t>(tid) * kScanPer;
    int v[kScanPer];
    if (x0 + kScanPer <= n_items) {
      const int4 q = *reinterpret_cast<const int4*>(p.cnt + x0);
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
#pragma unroll
      for (int u = 0; u < kScanPer; ++u) v[u] = x0 + u < n_items ? p.cnt[x0 + u] : 0;
    }
    int c = 0, t = 0, z = 0;
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      c += v[u];
      t += tiles_of(v[u]);
      z += v[u] > 0;
    }
    // inclusive scans within the warp, then over the 32 warp totals
    int ic = c, it = t, iz = z;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xc = __shfl_up_sync(0xffffffffu, ic, o);
      const int xt = __shfl_up_sync(0xffffffffu, it, o);
      const int xz = __shfl_up_sync(0xffffffffu, iz, o);
      if (lane >= o) { ic += xc; it += xt; iz += xz; }
    }
    if (lane == 31) { s_sum[wid][0] = ic; s_sum[wid][1] = it; s_sum[wid][2] = iz; }
    __syncthreads();
    if (wid == 0) {
      int wc = s_sum[lane][0], wt = s_sum[lane][1], wz = s_sum[lane][2];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int xc = __shfl_up_sync(0xffffffffu, wc, o);
        const int xt = __shfl_up_sync(0xffffffffu, wt, o);
        const int xz = __shfl_up_sync(0xffffffffu, wz, o);
        if (lane >= o) { wc += xc; wt += xt; wz += xz; }
      }
      s_sum[lane][0] = wc;   // inclusive over warps
      s_sum[lane][1] = wt;
      s_sum[lane][2] = wz;
    }
    __syncthreads();
    // exclusive prefixes of this thread's first item
    int pc = s_carry[0] + ic - c + (wid > 0 ? s_sum[wid - 1][0] : 0);
    int pt = s_carry[1] + it - t + (wid > 0 ? s_sum[wid - 1][1] : 0);
    int pz = s_carry[2] + iz - z + (wid > 0 ? s_sum[wid - 1][2] : 0);
    int o_c[kScanPer], o_t[kScanPer], o_z[kScanPer];
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      o_c[u] = pc; o_t[u] = pt; o_z[u] = pz;
      pc += v[u];
      pt += tiles_of(v[u]);
      pz += v[u] > 0;
    }
    scan_store4(p.off, x0, n_items, o_c);
    scan_store4(p.cursor, x0, n_items, o_c);
    scan_store4(p.tile_off, x0, n_items, o_t);
    scan_store4(p.ord, x0, n_items, o_z);
    __syncthreads();                             // every thread has read s_carry and s_sum
    if (tid == 0) {
      s_carry[0] += s_sum[31][0];
      s_carry[1] += s_sum[31][1];
      s_carry[2] += s_sum[31][2];
    }
    __syncthreads();
  }
  if (tid == 0) {
    p.off[n_items] = s_carry[0];
    p.tile_off[n_items] = s_carry[1];
  }
}

// Each entry claims its place in its item (lanes of one block in a warp
// claim consecutive places with one atomic) and writes the entry table and
// the slot map; the first entry of each tile writes the tile's descriptor.
__global__ void csr_fill_kernel(const CsrParams p) {
  const int64_t total = static_cast<int64_t>(p.nq) * p.Hkv * p.k;
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); base < total;
       base += stride) {
    const int64_t t = base + lane;
    CsrEntry x{0, -1, 0, 0};
    if (t < total) x = csr_entry(p, t, false);
    const unsigned grp = __match_any_sync(0xffffffffu, static_cast<int>(x.item));
    if (x.item >= 0) {   // no early exit: every lane reaches the next iteration's match together
      const int leader = __ffs(grp) - 1;
      int pos0 = 0;
      if (lane == leader) pos0 = atomicAdd(&p.cursor[x.item], __popc(grp));
      pos0 = __shfl_sync(grp, pos0, leader);
      const int pos = pos0 + __popc(grp & ((1u << lane) - 1u));
      const int64_t item = x.item;
      const int idx = pos - p.off[item];                                  // entry index within the item
      const int es = p.tile_off[item] * kEntries + idx;                   // entry slot in tile order
      p.tile_q[es] = static_cast<int>(x.bs);
      p.where[x.e] = es * 8;                                              // tile row of head 0
      if (idx % kEntries == 0) {
        const int c = p.off[item + 1] - p.off[item], u = idx / kEntries, nt = tiles_of(c);
        const int flags = (u == 0 ? kTileFirst : 0) | (u == nt - 1 ? kTileLast : 0) | (x.page << kTilePageShift);
        p.tile_info[es / kEntries] = make_int4(static_cast<int>(item), min(kEntries, c - idx), p.ord[item], flags);
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// attention over tiles
// ---------------------------------------------------------------------------

struct AttnParams {
  int S, Hkv, G, nb;
  int chunk;                 // 1: K/V are page pools, queries at q_pos[b] + i
  const int32_t* q_pos;
  int64_t n_items;
  float scale_log2;
  const int32_t* tile_off;   // tile_off[n_items] = number of tiles
  const int4* tile_info;
  const int32_t* tile_q;
  __nv_bfloat16* o_part;     // [tiles][16 entries][16 column chunks][G head rows][8] bf16, entries kEntryPart apart
  float* lse_part;           // [tiles * 128]
  int32_t* dev_err;
};

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

// streaming store (evict-first): the partials are read once, by the merge
__device__ __forceinline__ void st_cs_v4(void* ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__global__ void __launch_bounds__(kAttnThreads, 1)
attn_prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_kv = smem;                    // [2] x (K0 K1 V0 V1)
  uint8_t* s_q = smem + 2 * kKV;           // [kQStages] x Q tile

  __shared__ __align__(8) uint64_t bar_qfull[kQStages], bar_qempty[kQStages], bar_kvfull[2], bar_kvempty[2];
  __shared__ __align__(8) uint64_t bar_sfull[2], bar_pready[2], bar_ofull[2], bar_drain;
  __shared__ int s_kvinfo[kQStages];       // per Q stage: K/V buffer, new, release, phase (producer -> MMA)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // padding rows of a tile (no query) keep whatever the stage held; start from zeros
  for (int x = tid; x < kQStages * kQStage / 16; x += kAttnThreads)
    reinterpret_cast<uint4*>(s_q)[x] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (tid == 0) {
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&bar_qfull[i], 1);
      mbar_init(&bar_qempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_kvfull[i], 1); mbar_init(&bar_kvempty[i], 1);
      mbar_init(&bar_sfull[i], 1); mbar_init(&bar_pready[i], 4);
      mbar_init(&bar_ofull[i], 1);
    }
    mbar_init(&bar_drain, 1);
    s_abort = 0;
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

  if (warp == kProducerWarp) {
    // ===================== producer: Q boxes and K/V blocks by TMA =====================
    // Lane e loads the query rows of tile entry e (heads g*G .. g*G+7, both
    // column halves) into bytes 2048e.. of the stage; lane 0 also loads K_j, V_j
    // for the first tile of each item (in this CTA).
    const int ord0 = ntiles > 0 ? p.tile_info[t0].z : 0;
    constexpr uint32_t kQBytesPerEntry = 2048;   // full box, out-of-range heads included (zero-filled)
    int last_kv = -1, last_q = -1;
    // tile descriptors and entry queries, kPf tiles ahead (a ring in registers)
    constexpr int kPf = 4;
    int4 rti[kPf];
    int rbs[kPf];
#pragma unroll
    for (int x = 0; x < kPf; ++x) {
      rti[x] = make_int4(0, 0, 0, 0);
      rbs[x] = 0;
      if (x < ntiles) {
        rti[x] = p.tile_info[t0 + x];
        rbs[x] = lane < kEntries ? p.tile_q[(t0 + x) * kEntries + lane] : 0;   // entries past ti.y unused
      }
    }
    bool stop = false;
    for (int n0 = 0; n0 < ntiles && !stop; n0 += kPf) {
#pragma unroll
      for (int x = 0; x < kPf; ++x) {
        const int n = n0 + x;
        if (stop || n >= ntiles) break;
        const int4 ti = rti[x];
        const int bs = rbs[x];
        if (n + kPf < ntiles) {
          rti[x] = p.tile_info[t0 + n + kPf];
          rbs[x] = lane < kEntries ? p.tile_q[(t0 + n + kPf) * kEntries + lane] : 0;
        }
        const int item = ti.x, ne = ti.y, rel = ti.z - ord0;
        const int kvb = rel & 1;
        const bool kv_new = n == 0 || (ti.w & kTileFirst);
        const bool kv_rel = n + 1 == ntiles || (ti.w & kTileLast);
        const int b = static_cast<int>(item / (static_cast<int64_t>(p.Hkv) * p.nb));
        const int g = static_cast<int>((item / p.nb) % p.Hkv);
        const int j = static_cast<int>(item % p.nb);
        const int st = n % kQStages;
        bool ok = true;
        if (lane == 0) {
          ok = mbar_wait(&bar_qempty[st], ((n / kQStages) & 1) ^ 1, abort_flag, p.dev_err);
          if (ok && kv_new) {
            ok = mbar_wait(&bar_kvempty[kvb], ((rel >> 1) & 1) ^ 1, abort_flag, p.dev_err);
            if (ok) {
              uint8_t* kvbuf = s_kv + kvb * kKV;
              // contiguous K/V: (d, g, token, b); page pools: (d, token, g, page)
              const int x1 = p.chunk ? 0 : g, x2 = p.chunk ? g : j * kBk;
              const int x3 = p.chunk ? (ti.w >> kTilePageShift) : b;
              mbar_arrive_expect_tx(&bar_kvfull[kvb], kKV);
              tma_load_4d(kvbuf + 0 * kHalf, &kmap, &bar_kvfull[kvb], 0, x1, x2, x3);
              tma_load_4d(kvbuf + 1 * kHalf, &kmap, &bar_kvfull[kvb], 64, x1, x2, x3);
              tma_load_4d(kvbuf + 2 * kHalf, &vmap, &bar_kvfull[kvb], 0, x1, x2, x3);
              tma_load_4d(kvbuf + 3 * kHalf, &vmap, &bar_kvfull[kvb], 64, x1, x2, x3);
              last_kv = rel;
            }
          }
          if (ok) {
            s_kvinfo[st] = kvb | (kv_new ? 2 : 0) | (kv_rel ? 4 : 0) | (((rel >> 1) & 1) << 3);
            mbar_arrive_expect_tx(&bar_qfull[st], static_cast<uint32_t>(ne) * kQBytesPerEntry);
            last_q = n;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {                         // the warp stops together
          stop = true;
          break;
        }
        if (lane < ne) {
          const int qb_ = bs / p.S, qi_ = bs - qb_ * p.S;
          tma_load_5d(s_q + st * kQStage + lane * 2048, &qmap, &bar_qfull[st], 0, g * p.G, 0, qi_, qb_);
        }
        __syncwarp();
      }
    }
    if (*abort_flag && lane == 0) {        // let this warp's last loads land before the CTA exits
      const uint64_t tt = global_timer_ns();
      if (last_kv >= 0)
        while (!mbar_try_wait(&bar_kvfull[last_kv & 1], (last_kv >> 1) & 1) &&
               global_timer_ns() - tt < MSA_WAIT_LIMIT_NS) {
        }
      if (last_q >= 0)
        while (!mbar_try_wait(&bar_qfull[last_q % kQStages], (last_q / kQStages) & 1) &&
               global_timer_ns() - tt < MSA_WAIT_LIMIT_NS) {
        }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ===================== tcgen05 issuer =====================
    // S(n) and O(n) are issued as soon as their inputs are ready, O first:
    //   O(n) needs P(n) (pready); the warpgroup that arrives there has already
    //   read O(n-2) out of the slot's accumulator;
    //   S(n) needs Q(n), K_j, and O(n-2) issued: it overwrites the slot's S/P
    //   columns, from which O(n-2) reads P.  The MMAs of this one thread run
    //   in issue order, so O(n-2) has read its P operand before S(n) writes
    //   there, and S(n)'s commit (sfull) also covers O(n-2): the softmax
    //   warpgroup writes P(n) only after both.
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, 128, false, true);
      int ns = 0, no = 0;
      int kvinfo[2] = {0, 0};
      uint64_t idle_since = global_timer_ns();
      uint32_t spins = 0;
      while (no < ntiles) {
        bool progress = false;
        if (no < ns) {
          const int slot = no & 1;
          if (mbar_test_wait(&bar_pready[slot], (no >> 1) & 1)) {
            tc_fence_after();
            const int kv = kvinfo[slot];
            const uint32_t vb = smem_u32(s_kv + (kv & 1) * kKV + 2 * kHalf);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16_ts(tmem + slot * 256 + 128, tmem + slot * 256 + kk * 8,
                           sdesc_sw128(vb + kk * 2048, kHalf, 1024), idesc_o, kk > 0);
            umma_commit(&bar_ofull[slot]);
            if (kv & 4) umma_commit(&bar_kvempty[kv & 1]);
            ++no;
            progress = true;
          }
        }
        if (ns < ntiles && ns < no + 2) {
          const int st = ns % kQStages, slot = ns & 1;
          if (mbar_test_wait(&bar_qfull[st], (ns / kQStages) & 1)) {
            const int kv = s_kvinfo[st];
            if (!(kv & 2) || mbar_test_wait(&bar_kvfull[kv & 1], (kv >> 3) & 1)) {
              tc_fence_after();
              const uint32_t qb = smem_u32(s_q + st * kQStage);
              const uint32_t kb = smem_u32(s_kv + (kv & 1) * kKV);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                // Q: 8-row atoms 2048 B apart, column half at +1024; K: halves 16 KiB apart
                umma_bf16(tmem + slot * 256, sdesc_sw128(qb + (kk >> 2) * 1024 + 32 * (kk & 3), 16, 2048),
                          sdesc_sw128(kb + (kk >> 2) * kHalf + 32 * (kk & 3), 16, 1024), idesc_s, kk > 0);
              }
              umma_commit(&bar_sfull[slot]);
              umma_commit(&bar_qempty[st]);
              kvinfo[slot] = kv;
              ++ns;
              progress = true;
            }
          }
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
      const uint64_t tt = global_timer_ns();
      while (!mbar_try_wait(&bar_drain, 0) && global_timer_ns() - tt < MSA_WAIT_LIMIT_NS) {
      }
    }
    __syncwarp();
  } else {
    // ===================== softmax + epilogue: warpgroup wg owns TMEM slot wg (tiles n = wg mod 2) =====
    const int wg = (warp - kSoftmax0) >> 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;                     // tile row = TMEM lane
    const int e = r >> 3, h = r & 7;                 // entry of the row, head within the group
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const int slot = wg;
    const uint32_t sbase = tmem + lane_addr + slot * 256;   // S, then P (bf16 pairs) in its first 64 columns
    const float sc = p.scale_log2;
    int4 nti = make_int4(0, 0, 0, 0);
    int nbs = 0;
    if (wg < ntiles) {
      nti = p.tile_info[t0 + wg];
      nbs = p.tile_q[(t0 + wg) * kEntries + e];
    }
    for (int n = wg; n < ntiles; n += 2) {
      const int4 ti = nti;
      const int bs = nbs;
      if (n + 2 < ntiles) {
        nti = p.tile_info[t0 + n + 2];
        nbs = p.tile_q[(t0 + n + 2) * kEntries + e];
      }
      const uint32_t ph = (n >> 1) & 1;
      const int j = static_cast<int>(ti.x % p.nb);
      const bool valid = h < p.G && e < ti.y;
      // keys of this block visible to the row: t <= position of the query
      const int pos = bs % p.S + (p.chunk && valid ? __ldg(p.q_pos + bs / p.S) : 0);
      const int nvis = valid ? min(kBk, pos - j * kBk + 1) : kBk;
      const bool ok_s = mbar_wait(&bar_sfull[slot], ph, abort_flag, p.dev_err);
      if (!__all_sync(0xffffffffu, ok_s)) break;     // warp-uniform exit
      tc_fence_after();
      float m = -INFINITY, l = 0.f;
      // the branch must be warp-uniform: the TMEM loads and stores inside are warp-collective
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
          uint32_t pw[32];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float p0 = fast_exp2(fmaf(__uint_as_float(v[c][e]), sc, -m));
              const float p1 = fast_exp2(fmaf(__uint_as_float(v[c][e + 1]), sc, -m));
              l2 = add2(l2, pack2f(p0, p1));
              pw[16 * c + (e >> 1)] = pack_bf16x2(p0, p1);
            }
          }
          // P columns 32*half.. hold keys 64*half..: S columns already read
          tmem_st32(sbase + half * 32, pw);
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
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 = (cc * 32 + e < nvis) ? fast_exp2(fmaf(__uint_as_float(v[e]), sc, -m)) : 0.f;
            const float p1 = (cc * 32 + e + 1 < nvis) ? fast_exp2(fmaf(__uint_as_float(v[e + 1]), sc, -m)) : 0.f;
            l2 = add2(l2, pack2f(p0, p1));
            pw[e >> 1] = pack_bf16x2(p0, p1);
          }
          tmem_st16(sbase + cc * 16, pw);
        }
        float la, lb;
        unpack2f(l2, la, lb);
        l = la + lb;
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pready[slot]);
      const bool ok_o = mbar_wait(&bar_ofull[slot], ph, abort_flag, p.dev_err);
      if (!__all_sync(0xffffffffu, ok_o)) break;
      tc_fence_after();
      const float inv = 1.0f / l;
      const uint64_t inv2 = pack2f(inv, inv);
      const int64_t prow = (t0 + n) * 128 + r;
      // partial layout: one contiguous block of G * 256 bytes per tile entry
      // (a query's partial for this block, all its heads; entries 2 KiB
      // apart), [16-byte column chunk][head row] inside, no padding rows: the
      // merge reads each (query, slot) partial as exactly its G * 256 bytes
      // (with 8-row groups DRAM also fetched the two padding rows of every
      // 128-byte line)
      __nv_bfloat16* obase = p.o_part + ((t0 + n) * kEntries + e) * kEntryPart + h * 8;
      const int cstride = p.G * 8;                   // elements per 16-byte column chunk
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t v[2][32];
        tmem_ld32(sbase + 128 + hh * 64, v[0]);
        tmem_ld32(sbase + 128 + hh * 64 + 32, v[1]);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int e8 = 0; e8 < 32; e8 += 8) {
              uint32_t w4[4];
#pragma unroll
              for (int x = 0; x < 4; ++x) {
                float a0, a1;
                unpack2f(mul2(pack2f(__uint_as_float(v[c][e8 + 2 * x]), __uint_as_float(v[c][e8 + 2 * x + 1])), inv2),
                         a0, a1);
                w4[x] = pack_bf16x2(a0, a1);
              }
              const int chunk = hh * 8 + c * 4 + (e8 >> 3);
              st_cs_v4(obase + chunk * cstride, w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
      }
      // the loads above are complete (wait::ld): ordered before this
      // warpgroup's next pready arrive, which gates O(n+2) into this slot
      tc_fence_before();
      if (valid) __stcs(p.lse_part + prow, (m + log2f(l)) * kLn2);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// merge: O = sum_s e^{LSE_s - LSE} O_s, LSE = ln sum_s e^{LSE_s} over the k
// slots of each (query, head).  One warp per (query, group): lane L owns head
// h = L % 8 (idle if h >= G) and the column chunks c = L / 8 + 4x, x = 0..3,
// so that for each part and x the live lanes read chunks 4x .. 4x+3 of all G
// rows: one contiguous run of 4 * G * 16 bytes.
// ---------------------------------------------------------------------------

constexpr int kMergeWarps = 8;

struct MergeParams {
  int nq, Hq, Hkv, G, k;
  const __nv_bfloat16* o_part;
  const float* lse_part;
  const int32_t* where;
  __nv_bfloat16* O;      // chunk's first output row
  float* LSE;            // chunk's first LSE (or null)
};

__device__ __forceinline__ void fma8(float (&acc)[8], float w, uint4 raw) {
  const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
    acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
  }
}

// KMAX = 16 or 64 (k <= KMAX): lane (c0, h) also owns slots s = c0 + 4y.
template <int KMAX>
__global__ void __launch_bounds__(kMergeWarps * 32, 2) prefill_merge_kernel(const MergeParams p) {
  constexpr int SPL = KMAX / 4;              // slots per lane
  const int lane = threadIdx.x & 31;
  const int64_t wq = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (wq >= static_cast<int64_t>(p.nq) * p.Hkv) return;
  const int qi = static_cast<int>(wq / p.Hkv), g = static_cast<int>(wq % p.Hkv);
  const int h = lane & 7, c0 = lane >> 3;
  const bool live = h < p.G;
  const int32_t* wp = p.where + wq * p.k;
  int base[SPL];
  float wgt[SPL];
#pragma unroll
  for (int y = 0; y < SPL; ++y) base[y] = c0 + 4 * y < p.k ? wp[c0 + 4 * y] : -1;
#pragma unroll
  for (int y = 0; y < SPL; ++y) wgt[y] = live && base[y] >= 0 ? __ldcs(p.lse_part + base[y] + h) : -INFINITY;
  // this head's maximum and sum over its slots (the 4 lanes of head h)
  float m = -INFINITY;
#pragma unroll
  for (int y = 0; y < SPL; ++y) m = fmaxf(m, wgt[y]);
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
  float sum = 0.f;
#pragma unroll
  for (int y = 0; y < SPL; ++y) {
    wgt[y] = wgt[y] == -INFINITY ? 0.f : __expf(wgt[y] - m);
    sum += wgt[y];
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 8);
  sum += __shfl_xor_sync(0xffffffffu, sum, 16);
  // a head with no visible key (impossible for a valid selection) gets zeros, LSE = -inf
  const float inv = sum > 0.f ? 1.0f / sum : 0.f;
#pragma unroll
  for (int y = 0; y < SPL; ++y) wgt[y] *= inv;
  float acc[4][8];
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int z = 0; z < 8; ++z) acc[x][z] = 0.f;
  // slots 4y .. 4y+3 together: 16 loads of 16 B in flight per lane
#pragma unroll
  for (int y = 0; y < SPL; ++y) {
    if (4 * y >= p.k) break;
    uint4 raw[4][4];
    float w4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int src_lane = u * 8 + h;        // lane (c0 = u, h) owns slot 4y + u
      w4[u] = __shfl_sync(0xffffffffu, wgt[y], src_lane);
      const int b = __shfl_sync(0xffffffffu, base[y], src_lane);
      if (live && b >= 0 && w4[u] != 0.f) {
        const int64_t t = b >> 7, eb = (b & 127) >> 3;
        const int cstride = p.G * 8;         // [chunk][G head rows][8] per entry
        const __nv_bfloat16* src = p.o_part + (t * kEntries + eb) * kEntryPart + c0 * cstride + h * 8;
#pragma unroll
        for (int x = 0; x < 4; ++x) raw[u][x] = __ldcs(reinterpret_cast<const uint4*>(src + x * 4 * cstride));
      } else {
        w4[u] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (w4[u] != 0.f)
#pragma unroll
        for (int x = 0; x < 4; ++x) fma8(acc[x], w4[u], raw[u][x]);
  }
  if (live) {
    const int64_t orow = (static_cast<int64_t>(qi) * p.Hq + g * p.G + h) * kD;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      uint4 o;
      o.x = pack_bf16x2(acc[x][0], acc[x][1]);
      o.y = pack_bf16x2(acc[x][2], acc[x][3]);
      o.z = pack_bf16x2(acc[x][4], acc[x][5]);
      o.w = pack_bf16x2(acc[x][6], acc[x][7]);
      *reinterpret_cast<uint4*>(p.O + orow + (c0 + 4 * x) * 8) = o;
    }
    if (c0 == 0 && p.LSE != nullptr) p.LSE[qi * p.Hq + g * p.G + h] = sum > 0.f ? m + __logf(sum) : -INFINITY;
  }
}

struct WsLayout {
  size_t cnt, cursor, off, tile_off, ord, tile_info, tile_q, where, o_part, lse_part, total;
  int64_t max_tiles;
};

// Tiles of a chunk: sum over items of ceil(entries / 16)
//   <= entries / 16 + (non-empty items) + 1.
// Blocks per sequence: those of the prefill, or (chunk) the page-table width.
int64_t seq_blocks(const msa_prefill_args& a) {
  return a.mode == MSA_MODE_CHUNK ? a.max_pages : (a.S + kBk - 1) / kBk;
}

WsLayout ws_layout(const msa_prefill_args& a, int64_t cq) {
  const int64_t nb = seq_blocks(a);
  const int64_t n_items = static_cast<int64_t>(a.B) * a.Hkv * nb;
  const int64_t entries = cq * a.Hkv * a.k;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  WsLayout L;
  L.max_tiles = (entries + kEntries - 1) / kEntries + std::min(n_items, entries) + 1;
  const size_t rows = static_cast<size_t>(L.max_tiles) * 128;
  size_t o = 0;
  L.cnt = o; o = al(o + n_items * 4);
  L.cursor = o; o = al(o + n_items * 4);
  L.off = o; o = al(o + (n_items + 1) * 4);
  L.tile_off = o; o = al(o + (n_items + 1) * 4);
  L.ord = o; o = al(o + n_items * 4);
  L.tile_info = o; o = al(o + static_cast<size_t>(L.max_tiles) * 16);
  L.tile_q = o; o = al(o + static_cast<size_t>(L.max_tiles) * kEntries * 4);
  L.where = o; o = al(o + static_cast<size_t>(entries) * 4);
  L.o_part = o; o = al(o + rows * kD * 2);   // bf16 partials
  L.lse_part = o; o = al(o + rows * 4);
  L.total = o + 256;
  return L;
}

// A chunk of at most kChunkDecodeMaxS queries per sequence (a few decode
// tokens: draft verification) runs through the decode attention kernel
// instead: the rows (b, s, g), each with its own selected pages and last-page
// length, are a decode batch of B * S sequences, served in one launch after
// the page table (versus the per-chunk inversion, attention and merge of the
// KV-block-major path).  It needs Q dense over (b, s) and K, V with one set of
// strides; otherwise the KV-block-major path runs.
bool chunk_decode_path(const msa_prefill_args& a) {
  return a.mode == MSA_MODE_CHUNK && a.S <= kChunkDecodeMaxS && a.Q_stride[0] == a.S * a.Q_stride[1] &&
         a.K_stride[0] == a.V_stride[0] && a.K_stride[1] == a.V_stride[1] && a.K_stride[2] == a.V_stride[2];
}

struct ChunkDecodeWs {
  size_t pt, n, last_len, o_part, lse_part, counter, total;
};
ChunkDecodeWs chunk_decode_ws(const msa_prefill_args& a) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t rows = static_cast<size_t>(a.B) * a.S * a.Hkv;
  const size_t parts = static_cast<size_t>(a.B) * a.S * a.Hq * a.k;
  ChunkDecodeWs L;
  size_t o = 0;
  L.pt = o; o = al(o + rows * a.k * 4);
  L.n = o; o = al(o + rows * 4);
  L.last_len = o; o = al(o + rows * 4);
  L.o_part = o; o = al(o + parts * kD * 4);
  L.lse_part = o; o = al(o + parts * 4);
  L.counter = o; o = al(o + rows * 4);
  L.total = o + 256;
  return L;
}

msa_status launch_chunk_decode(const msa_prefill_args& a, void* ws, cudaStream_t stream) {
  const ChunkDecodeWs L = chunk_decode_ws(a);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* pt = reinterpret_cast<int32_t*>(w + L.pt);
  int32_t* n = reinterpret_cast<int32_t*>(w + L.n);
  int32_t* last_len = reinterpret_cast<int32_t*>(w + L.last_len);
  if (msa_status st = launch_page_table(a.sel, a.count, a.seq_pt, a.max_pages, nullptr, a.B, a.Hkv, a.k, kBk, pt, n,
                                        last_len, a.dev_err, stream, a.S, a.q_pos);
      st != MSA_OK)
    return st;
  msa_decode_args d{};
  d.B = a.B * a.S; d.Hq = a.Hq; d.Hkv = a.Hkv; d.D = a.D; d.Bk = a.Bk; d.k = a.k;
  d.softmax_scale = a.softmax_scale;
  d.Q = a.Q;
  d.Q_stride[0] = a.Q_stride[1];   // row (b, s) = b * S + s: Q is dense over (b, s)
  d.Q_stride[1] = a.Q_stride[2];
  d.K_pool = a.K; d.V_pool = a.V;
  for (int i = 0; i < 3; ++i) d.kv_stride[i] = a.K_stride[i];
  d.num_pages = a.num_pages;
  d.pt = pt; d.n = n; d.last_len = last_len;
  d.O = a.O; d.LSE = a.LSE; d.dev_err = a.dev_err;
  d.scratch_zeroed = 0;
  return launch_attn_decode(d, reinterpret_cast<float*>(w + L.o_part), reinterpret_cast<float*>(w + L.lse_part),
                            reinterpret_cast<int32_t*>(w + L.counter), stream);
}

}  // namespace

size_t attn_prefill_workspace_size(const msa_prefill_args& a, int64_t chunk_queries) {
  if (chunk_decode_path(a)) return chunk_decode_ws(a).total;
  return ws_layout(a, chunk_queries).total;
}

msa_status launch_attn_prefill(const msa_prefill_args& a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (chunk_decode_path(a)) return launch_chunk_decode(a, ws, stream);
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
  const int64_t nb = seq_blocks(a);
  const bool chunk = a.mode == MSA_MODE_CHUNK;
  const int64_t n_items = static_cast<int64_t>(a.B) * a.Hkv * nb;
  const int G = a.Hq / a.Hkv;
  if (L.max_tiles * 128 >= (int64_t(1) << 31) || cq * a.Hkv * a.k >= (int64_t(1) << 31) ||
      n_items >= (int64_t(1) << 31) || total_q >= (int64_t(1) << 31))
    return fail(MSA_ERR_UNSUPPORTED, "prefill attention: problem too large for 32-bit tile rows");
  uint8_t* w = static_cast<uint8_t*>(ws);

  CUtensorMap qmap, kmap, vmap;
  {
    // Q [B, S, Hq, D] seen as (64 columns, head, column half, i, b): one box =
    // 8 heads from g*G, both halves -> [half][head][64] in shared memory
    const uint64_t qdims[5] = {64, static_cast<uint64_t>(a.Hq), 2, static_cast<uint64_t>(a.S),
                               static_cast<uint64_t>(a.B)};
    const uint64_t qstrides[4] = {static_cast<uint64_t>(a.Q_stride[2]) * 2, 128,
                                  static_cast<uint64_t>(a.Q_stride[1]) * 2, static_cast<uint64_t>(a.Q_stride[0]) * 2};
    const uint32_t qbox[5] = {64, 8, 2, 1, 1};
    if (msa_status st = encode_tiled_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, a.Q, qdims, qstrides, qbox,
                                         CU_TENSOR_MAP_SWIZZLE_128B, "Q");
        st != MSA_OK)
      return st;
  }
  // contiguous K/V [B, S, Hkv, D] strides (b, s, g) as (d, g, s, b), box = 128
  // tokens of one group; page pools [pages, Hkv, Bk, D] strides (page, g, t) as
  // (d, t, g, page), box = one page of one group.  Both land in shared memory
  // as 128 rows of 64 columns.
  const uint64_t dims[4] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(chunk ? kBk : a.Hkv),
                            static_cast<uint64_t>(chunk ? a.Hkv : a.S),
                            static_cast<uint64_t>(chunk ? a.num_pages : a.B)};
  const uint32_t box[4] = {64, chunk ? 128u : 1u, chunk ? 1u : 128u, 1};
  // Strides (b, s, g) or (page, g, t): dims 1, 2, 3 take strides 2, 1, 0 either way.
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
  const size_t smem = 1024 + 2 * static_cast<size_t>(kKV) + kQStages * static_cast<size_t>(kQStage);
  if (smem > dev.max_smem_optin) return fail(MSA_ERR_UNSUPPORTED, "prefill attention: not enough shared memory");
  cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attn_prefill)");

  const float scale = a.softmax_scale > 0.f ? a.softmax_scale : 1.0f / sqrtf(static_cast<float>(a.D));
  for (int64_t q0 = 0; q0 < total_q; q0 += cq) {
    const int nq = static_cast<int>(std::min<int64_t>(cq, total_q - q0));
    CsrParams c;
    c.S = a.S; c.Hkv = a.Hkv; c.Hq = a.Hq; c.G = G; c.k = a.k; c.nb = static_cast<int>(nb);
    c.chunk = chunk; c.q_pos = a.q_pos; c.seq_pt = a.seq_pt; c.max_pages = a.max_pages; c.num_pages = a.num_pages;
    c.q0 = q0; c.nq = nq;
    c.sel = a.sel; c.count = a.count;
    c.cnt = reinterpret_cast<int32_t*>(w + L.cnt);
    c.cursor = reinterpret_cast<int32_t*>(w + L.cursor);
    c.off = reinterpret_cast<int32_t*>(w + L.off);
    c.tile_off = reinterpret_cast<int32_t*>(w + L.tile_off);
    c.ord = reinterpret_cast<int32_t*>(w + L.ord);
    c.tile_info = reinterpret_cast<int4*>(w + L.tile_info);
    c.tile_q = reinterpret_cast<int32_t*>(w + L.tile_q);
    c.where = reinterpret_cast<int32_t*>(w + L.where);
    c.dev_err = a.dev_err;
    e = cudaMemsetAsync(c.cnt, 0, n_items * 4, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(prefill counts)");
    const int64_t work = static_cast<int64_t>(nq) * a.Hkv * a.k;
    const int grid_w = static_cast<int>(std::min<int64_t>((work + 255) / 256, 8 * dev.num_sms));
    csr_count_kernel<<<grid_w, 256, 0, stream>>>(c);
    csr_scan_kernel<<<1, kScanThreads, 0, stream>>>(c, n_items);
    csr_fill_kernel<<<grid_w, 256, 0, stream>>>(c);

    AttnParams p;
    p.S = a.S; p.Hkv = a.Hkv; p.G = G; p.nb = static_cast<int>(nb);
    p.chunk = chunk; p.q_pos = a.q_pos;
    p.n_items = n_items;
    p.scale_log2 = scale * kLog2e;
    p.tile_off = c.tile_off; p.tile_info = c.tile_info; p.tile_q = c.tile_q;
    p.o_part = reinterpret_cast<__nv_bfloat16*>(w + L.o_part);
    p.lse_part = reinterpret_cast<float*>(w + L.lse_part);
    p.dev_err = a.dev_err;
    attn_prefill_kernel<<<dev.num_sms, kAttnThreads, smem, stream>>>(qmap, kmap, vmap, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "prefill attention launch");

    MergeParams mp;
    mp.nq = nq; mp.Hq = a.Hq; mp.Hkv = a.Hkv; mp.G = G; mp.k = a.k;
    mp.o_part = p.o_part; mp.lse_part = p.lse_part; mp.where = c.where;
    mp.O = static_cast<__nv_bfloat16*>(a.O) + q0 * a.Hq * kD;
    mp.LSE = a.LSE != nullptr ? a.LSE + q0 * a.Hq : nullptr;
    const int64_t mgrid = (static_cast<int64_t>(nq) * a.Hkv + kMergeWarps - 1) / kMergeWarps;
    if (a.k <= 16)
      prefill_merge_kernel<16><<<static_cast<unsigned>(mgrid), kMergeWarps * 32, 0, stream>>>(mp);
    else
      prefill_merge_kernel<64><<<static_cast<unsigned>(mgrid), kMergeWarps * 32, 0, stream>>>(mp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "prefill merge launch");
  }
  return MSA_OK;
}

}  // namespace msa
