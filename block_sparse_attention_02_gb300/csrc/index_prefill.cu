// index_prefill.cu -- a1 (prefill): block scores of the Index Branch for every
// query of a causal prefill.
//
// For query i of sequence b, KV group g and every block j < i / Bk:
//     c_j = max_{t in block j} sum_{h < HI} w[b,i,g,h] * ReLU(q_idx[b,i,g,h] . k_idx[b,t,g])
// ("MiniMax M3: Como la atencion dispersa hace practicos a los agentes de largo
// alcance", MSA paragraph and caption; the formula is this library's).  The own
// block and later blocks are written -inf.
//
// This is a dense contraction on the tensor cores.  An item is (b, g, query
// block qb of 64 queries); its queries share the own 128-token block qb / 2,
// so the item scores the key blocks j < qb / 2.  One pass = one key block:
//     D[t, (h, q)] = k_idx[t] . q_idx[q, h]    M = 128 tokens, N = 64 * HI
//                                              (heads x queries), K = 64
// With the tokens on M and the four heads side by side on N every MMA is
// N = 256 (the tensor core's full width), and the epilogue needs no state across
// passes: thread = token t forms s_t = sum_h w_h ReLU(D[t, (h, q)]) for its
// queries, the block max over tokens is one `redux.sync.max.f32` per warp and
// query plus a 4-warp combine in shared memory.
// A chunk over a paged cache (MSA_MODE_CHUNK) runs the same kernel: query s
// of sequence b sits at position q_pos[b] + s, key block j is page
// seq_pt[b][j] of the index-key pool, and an item whose 64 queries straddle a
// block boundary scores up to the later own block; each query's row then
// masks its own block to -inf when it is stored.
// When there are too few items to fill the GPU (short chunks: a few decode
// tokens per sequence), each item's key blocks are split into nsplit ranges
// scored by different CTAs (block scores are independent of each other).
// Items pair query block qb with nq-1-qb (constant cost per pair); a persistent
// CTA per SM takes pairs round-robin and runs two independent item streams
// ("slots") at once:
//   warp 0    TMA: per slot a q_idx tile (HI heads x 64 queries, one box per
//             head) and, in the merged pass order, a 6-deep ring of k_idx blocks
//             (128 tokens x 64), all 128-byte swizzled;
//   warp 1    tcgen05: per pass 4 MMAs into the slot's 256-column TMEM buffer;
//   warps 2-17: four epilogue warpgroups, two per slot, each reducing 32 of
//             the slot's 64 queries (TMEM loads of the next 8 queries in flight
//             while the current 8 are reduced).
#include "msa_internal.h"
#include "msa_ptx.cuh"

#include <type_traits>

namespace msa {
namespace {

constexpr int kQB = 64;                             // queries per item
constexpr int kHalves = 2;                          // epilogue warpgroups per slot (query halves)
constexpr int kQW = kQB / kHalves;                  // queries per epilogue warpgroup
constexpr int kThreads = 64 + 2 * kHalves * 128;    // w0 TMA, w1 MMA, then the epilogue warpgroups
constexpr int kKTile = 128 * 64 * 2;                // 16 KiB: one k_idx block
constexpr int kQHead = kQB * 64 * 2;                // 8 KiB: one head of a q_idx tile
constexpr int kQTile = kMaxHI * kQHead;             // 32 KiB
constexpr int kKStages = 6;
constexpr int kBufCols = 256;                       // TMEM per slot: HI x 64 columns
constexpr int kTmemCols = 512;
constexpr int kFlush = 8;                           // block scores staged per query before a store
constexpr int kStRow = kQB + 4;                     // staged row: one block's warp maxima for 64 queries (+4 pad)

struct Params {
  int B, S, Hkv, HI, nq, nb_stride;                 // nq = ceil(S / 64)
  int kgroups;                                      // 0: one k_idx shared by all groups (group stride 0)
  int chunk;                                        // 1: queries at q_pos[b] + s, paged index keys
  int nsplit;                                       // key-block ranges per item
  const int32_t* q_pos;                             // chunk: [B]
  const int32_t* seq_pt;                            // chunk: [B, max_pages]
  int64_t max_pages, num_pages;
  const float* w;
  int64_t ws0, ws1, ws2;
  float* C;
  int64_t cs0, cs1, cs2;
  int32_t* dev_err;
};

struct Item {
  int b, g, qb;
  int jb, je;                                       // this split's key blocks [jb, je)
  bool fill;                                        // last split (je = the item's block count): writes
                                                    // the -inf tail of the rows from je on
};

// CHUNK (a template parameter of everything below) selects the chunk mode:
// query positions, paged index keys and split items.  The prefill
// instantiations see nsplit = 1 and position 0 as constants.

// Position of query 0 of sequence b, or -1 when a chunk's q_pos[b] leaves the
// pages or the score rows (the sequence is then not scored).
template <bool CHUNK>
__device__ __forceinline__ int seq_pos0(const Params& p, int b) {
  if constexpr (!CHUNK) {
    return 0;
  } else {
    const int64_t q = p.q_pos[b];
    const int64_t last = q + p.S - 1;
    return (q < 0 || last >= p.max_pages * kBk || last / kBk >= p.nb_stride) ? -1 : static_cast<int>(q);
  }
}

// item `which` (0 or 1) of pair `pair`: pairs enumerate (b, g, pp, split r)
// with qb in {pp, nq-1-pp}; false when the pair has no such item.  The item
// scores the blocks before the own block of its last query; split r takes
// the r-th of nsplit equal ranges of them.
template <bool CHUNK>
__device__ __forceinline__ bool pair_item(const Params& p, int pair, int which, Item* it) {
  const int half = (p.nq + 1) / 2;
  const int nsplit = CHUNK ? p.nsplit : 1;
  const int r = pair % nsplit;
  const int rest = pair / nsplit;
  const int pp = rest % half;
  const int bg = rest / half;
  const int other = p.nq - 1 - pp;
  if (which == 1 && other == pp) return false;
  const int qb = which == 0 ? pp : other;
  const int b = bg / p.Hkv;
  const int pos0 = seq_pos0<CHUNK>(p, b);
  const int own = pos0 < 0 ? 0 : (pos0 + min(qb * kQB + kQB, p.S) - 1) / kBk;
  const int jb = static_cast<int>(static_cast<int64_t>(own) * r / nsplit);
  const int je = static_cast<int>(static_cast<int64_t>(own) * (r + 1) / nsplit);
  *it = {b, bg % p.Hkv, qb, jb, je, r == nsplit - 1};
  return true;
}

// The items of one slot: in the k-th pair of this CTA the slot takes item
// slot ^ (k & 1), so long and short items alternate between the slots.
struct Stream {
  int pr;          // next pair to look at
  int k;           // its ordinal in this CTA
  Item it;         // current item
  int j;           // next key block of the current item
  bool done;
};

// keep_empty: also stop at last splits with no key block to score (the
// epilogue still writes their -inf rows; the producer and the MMA warp skip
// them)
template <bool CHUNK>
__device__ __forceinline__ void stream_advance(const Params& p, Stream& s, int slot, int npairs,
                                               bool keep_empty) {
  for (;;) {
    if (s.pr >= npairs) {
      s.done = true;
      return;
    }
    Item it;
    const bool ok = pair_item<CHUNK>(p, s.pr, slot ^ (s.k & 1), &it);
    s.pr += gridDim.x;
    ++s.k;
    if (ok && (it.je > it.jb || (keep_empty && it.fill))) {
      s.it = it;
      s.j = it.jb;
      return;
    }
  }
}

template <bool CHUNK>
__device__ __forceinline__ void stream_init(const Params& p, Stream& s, int slot, int npairs, bool keep_empty) {
  s.pr = blockIdx.x;
  s.k = 0;
  s.done = false;
  stream_advance<CHUNK>(p, s, slot, npairs, keep_empty);
}

template <int N>
using SlotC = std::integral_constant<int, N>;

// One pass of stream `st` (slot SLOT): hand it to f(SlotC<SLOT>, item, j,
// first, last) and step the stream.  first/last = first/last pass of the item.
template <bool CHUNK, int SLOT, class F>
__device__ __forceinline__ bool stream_pass(const Params& p, Stream& st, int npairs, F& f) {
  const Item it = st.it;
  const int j = st.j;
  if (++st.j == it.je) stream_advance<CHUNK>(p, st, SLOT, npairs, false);
  return f(SlotC<SLOT>{}, it, j, j == it.jb, j == it.je - 1);
}

// The merged pass order of the producer and the MMA warp: the two slots'
// passes alternate while both have passes left.  The slot reaches f as a
// compile-time constant, so per-slot state and barrier addresses need no
// runtime selection, and both streams stay in registers.  Stops early when f
// returns false.
template <bool CHUNK, class F>
__device__ __forceinline__ void for_each_pass(const Params& p, int npairs, F&& f) {
  Stream s0, s1;
  stream_init<CHUNK>(p, s0, 0, npairs, false);
  stream_init<CHUNK>(p, s1, 1, npairs, false);
  bool turn = false;
  for (;;) {
    bool one;
    if (!s0.done && !s1.done) {
      one = turn;
      turn = !turn;
    } else if (!s0.done) {
      one = false;
    } else if (!s1.done) {
      one = true;
    } else {
      return;
    }
    if (!(one ? stream_pass<CHUNK, 1>(p, s1, npairs, f) : stream_pass<CHUNK, 0>(p, s0, npairs, f))) return;
  }
}

// Position in a ring of kKStages buffers: stage and the parity of its use.
struct Ring {
  int st = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next() {
    if (++st == kKStages) {
      st = 0;
      ph ^= 1u;
    }
  }
};

// The four K=16 steps of one pass, issued by one elected lane of a converged
// warp: D[d] = A[a] B[b]^T over K = 64 (descriptor start addresses advance by
// 32 bytes = 2 units per step inside the 128-byte swizzled rows).
__device__ __forceinline__ void umma_pass_elect(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\t"
      ".reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.ne.b32 f, %4, %4;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
      "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, t;\n\t}"
      ::"r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(0)
      : "memory");
}
// tcgen05.commit from one elected lane of a converged warp.
__device__ __forceinline__ void umma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// true in exactly one (the lowest) active lane of the warp
__device__ __forceinline__ bool elect_one() {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r));
  return r != 0;
}

// Named barrier over n threads that also returns the AND of `v` over them:
// every warp of an epilogue group leaves a pass with the same decision.
__device__ __forceinline__ bool named_bar_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Max of a float over the 32 lanes of the warp (exact: a max rounds nothing).
__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ uint64_t pack2(float x, float y) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& x, float& y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {   // two IEEE fmas
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// After tcgen05.wait::ld: ties the loaded registers to the wait so that no use
// of them is scheduled before it (emits no instruction).
__device__ __forceinline__ void regs_after_wait(uint32_t (&r)[8]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]));
}

constexpr int kCQ = 8;                               // queries per epilogue chunk
constexpr int kReluAlu = 2;                          // heads whose ReLU is a max; the others use x + |x|
constexpr int kNC = kQW / kCQ;                       // chunks per pass and warp

// FEW: a chunk of at most kCQ queries per sequence (a few decode tokens):
// only the first 8-query chunk of the first query half holds queries, so the
// epilogue loads and reduces that chunk alone.
template <int HI, bool CHUNK, bool FEW>
__global__ void __launch_bounds__(kThreads, 1)
index_prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                     const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_q = smem;                              // [2 slots] q_idx tiles: [head][64 queries][64]
  uint8_t* s_k = smem + 2 * kQTile;                 // [kKStages] k_idx blocks: [128 tokens][64]

  __shared__ __align__(8) uint64_t bar_qfull[2], bar_qempty[2], bar_kfull[kKStages], bar_kempty[kKStages];
  __shared__ __align__(8) uint64_t bar_tfull[2], bar_tempty[2], bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ __align__(16) float2 s_w[2][kQB / 2][kMaxHI];   // per slot: (w[2e][h], w[2e+1][h]) per query pair e
  // per slot, two alternating groups of kFlush blocks: each epilogue warp's
  // max over its 32 tokens, per block and query; combined over the 4 warps
  // when the group is stored
  __shared__ __align__(16) float s_stage[2][2][4][kFlush][kStRow];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_qfull[i], 1); mbar_init(&bar_qempty[i], 1);
      mbar_init(&bar_tfull[i], 1); mbar_init(&bar_tempty[i], 4 * kHalves);
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
  const int npairs = p.B * p.Hkv * ((p.nq + 1) / 2) * (CHUNK ? p.nsplit : 1);   // < 2^31, checked at launch

  if (warp == 0) {
    // ===================== TMA producer =====================
    // The whole warp runs the (warp-uniform) loop; one elected lane issues.
    const bool leader = elect_one();
    Ring kr;
    int n = 0, nql[2] = {0, 0};   // k blocks issued; q tiles issued per slot
    for_each_pass<CHUNK>(p, npairs, [&](auto slot_c, const Item& it, int j, bool first, bool) -> bool {
      constexpr int slot = decltype(slot_c)::value;
      if (first) {   // the item's q_idx tile into the slot's buffer, once its previous item is done
        if (!__all_sync(0xffffffffu, mbar_wait(&bar_qempty[slot], (nql[slot] & 1) ^ 1, abort_flag, p.dev_err)))
          return false;
        if (leader) {
          mbar_arrive_expect_tx(&bar_qfull[slot], HI * kQHead);
#pragma unroll
          for (int h = 0; h < HI; ++h)
            tma_load_5d(s_q + slot * kQTile + h * kQHead, &qmap, &bar_qfull[slot], 0, h, it.g, it.qb * kQB, it.b);
        }
        ++nql[slot];
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_kempty[kr.st], kr.ph ^ 1, abort_flag, p.dev_err))) return false;
      if (leader) {
        const int gk = p.kgroups ? it.g : 0;
        if constexpr (CHUNK) {
          // page of block j.  An id outside the pool is reported and not
          // loaded: the stage completes with a plain arrive, the MMA runs on
          // whatever the stage held, and the epilogue stores -inf for the block.
          const int page = p.seq_pt[it.b * p.max_pages + j];
          if (page < 0 || page >= p.num_pages) {
            report(p.dev_err, MSA_DEVERR_BAD_PAGE);
            mbar_arrive(&bar_kfull[kr.st]);
          } else {
            mbar_arrive_expect_tx(&bar_kfull[kr.st], kKTile);
            tma_load_4d(s_k + kr.st * kKTile, &kmap, &bar_kfull[kr.st], 0, 0, gk, page);
          }
        } else {
          mbar_arrive_expect_tx(&bar_kfull[kr.st], kKTile);
          tma_load_4d(s_k + kr.st * kKTile, &kmap, &bar_kfull[kr.st], 0, gk, j * kBk, it.b);
        }
      }
      kr.next();
      ++n;
      return true;
    });
    if (leader && *abort_flag) {  // let loads in flight land before the CTA exits
      const uint64_t t0 = global_timer_ns();
      for (int x = max(0, n - kKStages); x < n; ++x)
        while (!mbar_try_wait(&bar_kfull[x % kKStages], (x / kKStages) & 1) &&
               global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
        }
      for (int sl = 0; sl < 2; ++sl)
        if (nql[sl] > 0)
          while (!mbar_try_wait(&bar_qfull[sl], (nql[sl] - 1) & 1) && global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
          }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ===================== tcgen05 issuer (warp-uniform loop, one elected lane issues) =====================
    constexpr uint32_t idesc = idesc_bf16(128, kQB * HI, false, false);
    const uint64_t kdesc0 = sdesc_sw128(smem_u32(s_k), 16, 1024);
    const uint64_t qdesc0 = sdesc_sw128(smem_u32(s_q), 16, 1024);
    Ring kr;
    uint32_t qph[2] = {0, 0}, tph[2] = {0, 0};   // parities of the slots' qfull / tempty waits
    for_each_pass<CHUNK>(p, npairs, [&](auto slot_c, const Item&, int, bool first, bool last) -> bool {
      constexpr int slot = decltype(slot_c)::value;
      if (first) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bar_qfull[slot], qph[slot], abort_flag, p.dev_err))) return false;
        qph[slot] ^= 1u;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_kfull[kr.st], kr.ph, abort_flag, p.dev_err))) return false;
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_tempty[slot], tph[slot] ^ 1, abort_flag, p.dev_err))) return false;
      tph[slot] ^= 1u;
      tc_fence_after();
      // D[t, (h, q)] = k[t, :] . q[(h, q), :]; descriptor units are 16 bytes
      umma_pass_elect(tmem + slot * kBufCols, kdesc0 + static_cast<uint64_t>(kr.st * (kKTile >> 4)),
                      qdesc0 + static_cast<uint64_t>(slot * (kQTile >> 4)), idesc);
      umma_commit_elect(&bar_tfull[slot]);
      umma_commit_elect(&bar_kempty[kr.st]);
      if (last) umma_commit_elect(&bar_qempty[slot]);
      kr.next();
      return true;
    });
    if (elect_one()) {
      umma_commit(&bar_drain);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&bar_drain, 0) && global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
      }
    }
    __syncwarp();
  } else {
    // ===================== epilogue; thread = token =====================
    // warpgroup wg = (warp - 2) / 4 serves slot wg % 2 and the slot's queries
    // q0 .. q0 + 31 of every pass, q0 = 32 (wg / 2)
    const int wg = (warp - 2) >> 2;
    const int sl = wg & 1;
    const int q0 = (wg >> 1) * kQW;
    const int q4 = warp & 3;                          // TMEM lane quarter
    const int tw = tid - 64 - wg * 128;               // thread within the warpgroup
    const int bar_id = 1 + wg;
    const uint32_t base = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + sl * kBufCols + q0;
    Stream st;
    stream_init<CHUNK>(p, st, sl, npairs, true);
    int np = 0;
    bool ok = true;
    while (ok && !st.done) {
      const Item it = st.it;
      const int pos0 = seq_pos0<CHUNK>(p, it.b);    // -1: a rejected chunk sequence (no passes)
      if (pos0 < 0 && tw == 0 && it.qb == 0 && it.fill) report(p.dev_err, MSA_DEVERR_BAD_LEN);
      named_bar_sync(bar_id, 128);                    // the previous item's s_w / s_cst are no longer read
      if (tw < kQW) {
        const int i = it.qb * kQB + q0 + tw;
        const float* wp = p.w + it.b * p.ws0 + static_cast<int64_t>(i) * p.ws1 + it.g * p.ws2;
        float* sw = reinterpret_cast<float*>(&s_w[sl][(q0 + tw) >> 1][0]) + (tw & 1);
#pragma unroll
        for (int h = 0; h < HI; ++h) sw[2 * h] = i < p.S ? (h < kReluAlu ? wp[h] : 0.5f * wp[h]) : 0.f;
      }
      named_bar_sync(bar_id, 128);
      // -inf for every entry from the item's block count on (the last split
      // only; disjoint from the columns the passes below store)
      for (int rr = 0; rr < kQW / 4 && it.fill; ++rr) {
        const int i = it.qb * kQB + q0 + q4 * (kQW / 4) + rr;
        if (i >= p.S) break;
        float* rowp = p.C + it.b * p.cs0 + static_cast<int64_t>(i) * p.cs1 + it.g * p.cs2;
        for (int jj = it.je + lane; jj < p.nb_stride; jj += 32) rowp[jj] = -INFINITY;
      }
      for (int j = it.jb; j < it.je; ++j) {
        // warp-uniform decision: the TMEM loads below are warp-collective
        const bool got = __all_sync(0xffffffffu, mbar_wait(&bar_tfull[sl], np & 1, abort_flag, p.dev_err));
        if (got) tc_fence_after();
        float* red = &s_stage[sl][(j / kFlush) & 1][q4][j % kFlush][q0];
        // chunk c = queries 8c .. 8c+7; the TMEM loads of chunk c+1 are in flight
        // while chunk c is reduced
        uint32_t va[HI][kCQ], vb[HI][kCQ];
        auto load = [&](int c, uint32_t (&v)[HI][kCQ]) {
#pragma unroll
          for (int h = 0; h < HI; ++h) tmem_ld8(base + h * kQB + c * kCQ, v[h]);
        };
        auto wait = [&](uint32_t (&v)[HI][kCQ]) {
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < HI; ++h) regs_after_wait(v[h]);
        };
        auto reduce = [&](int c, uint32_t (&v)[HI][kCQ]) {
          // s_t = sum_h w_h ReLU(D[t, (h, q)]) for the chunk's 8 queries (two per fma.f32x2),
          // heads in order; then the max over this warp's 32 tokens
          float km[kCQ];
#pragma unroll
          for (int e = 0; e < kCQ / 2; ++e) {
            const float4* wq = reinterpret_cast<const float4*>(&s_w[sl][(q0 + c * kCQ) / 2 + e][0]);
            const float4 w01 = wq[0], w23 = wq[1];
            const float wx[4] = {w01.x, w01.z, w23.x, w23.z}, wy[4] = {w01.y, w01.w, w23.y, w23.w};
            uint64_t acc = 0ull;
#pragma unroll
            for (int h = 0; h < HI; ++h) {
              const float x0 = __uint_as_float(v[h][2 * e]), x1 = __uint_as_float(v[h][2 * e + 1]);
              // ReLU as a max (ALU pipe) for the first heads and as x + |x| against a
              // halved weight (FMA pipe) for the rest: (w / 2)(x + |x|) = w ReLU(x) exactly
              acc = h < kReluAlu ? fma2(pack2(wx[h], wy[h]), pack2(fmaxf(x0, 0.f), fmaxf(x1, 0.f)), acc)
                                 : fma2(pack2(wx[h], wy[h]), pack2(x0 + fabsf(x0), x1 + fabsf(x1)), acc);
            }
            float s0, s1;
            unpack2(acc, s0, s1);
            km[2 * e] = warp_max_f32(s0);
            km[2 * e + 1] = warp_max_f32(s1);
          }
          if (lane == 0) {
            float4* dst = reinterpret_cast<float4*>(red + c * kCQ);
            dst[0] = make_float4(km[0], km[1], km[2], km[3]);
            dst[1] = make_float4(km[4], km[5], km[6], km[7]);
          }
        };
        if constexpr (FEW) {
          if (got) {
            if (q0 == 0) {
              load(0, va);
              wait(va);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_tempty[sl]);
            if (q0 == 0) reduce(0, va);
          }
        } else if (got) {
          load(0, va);
          wait(va);
#pragma unroll
          for (int c = 0; c < kNC; c += 2) {
            load(c + 1, vb);
            reduce(c, va);
            wait(vb);
            if (c + 2 < kNC) {
              load(c + 2, va);
            } else {                                  // every load of the pass is done: free the buffer
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bar_tempty[sl]);
            }
            reduce(c + 1, vb);
            if (c + 2 < kNC) wait(va);
          }
        }
        // a warp that gave up waiting goes on (its later waits fail at once:
        // the abort flag is set) so that all four meet at the next store
        ok = ok && got;
        ++np;
        if (j % kFlush == kFlush - 1 || j == it.je - 1) {
          // all four warps' maxima of the group are staged, or some warp gave up
          if (!(ok = named_bar_and(bar_id, 128, ok))) break;
          // staged blocks j0 .. j (row = block mod kFlush, group (block / kFlush) mod 2)
          const int jal = j - j % kFlush, j0 = max(it.jb, jal), cnt = j - j0 + 1;
          const int jj = lane % kFlush, r4 = lane / kFlush;     // block and row of this lane
          const int x = j0 - jal + jj;
          const float(*stg)[kFlush][kStRow] = s_stage[sl][(j / kFlush) & 1];
          // a chunk's block whose page id is outside the pool was not loaded: -inf
          bool badpg = false;
          if constexpr (CHUNK) {
            if (jj < cnt) {
              const int pg = p.seq_pt[it.b * p.max_pages + j0 + jj];
              badpg = pg < 0 || pg >= p.num_pages;
            }
          }
#pragma unroll
          for (int rr = 0; rr < kQW / 4; rr += 32 / kFlush) {   // warp q4: query rows q0 + 8 q4 .. q0 + 8 q4 + 7
            const int qrow = q0 + q4 * (kQW / 4) + rr + r4;
            const int i = it.qb * kQB + qrow;
            // a query before the item's last own block has its own block among the passes: -inf
            if (i < p.S && jj < cnt) {
              const float v = fmaxf(fmaxf(stg[0][x][qrow], stg[1][x][qrow]), fmaxf(stg[2][x][qrow], stg[3][x][qrow]));
              p.C[it.b * p.cs0 + static_cast<int64_t>(i) * p.cs1 + it.g * p.cs2 + j0 + jj] =
                  (j0 + jj < (pos0 + i) / kBk && !badpg) ? v : -INFINITY;
            }
          }
        }
      }
      if (!ok) break;
      stream_advance<CHUNK>(p, st, sl, npairs, true);
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
  // a few tokens per sequence over per-group keys (draft verification,
  // multi-token decode): the decode kernel streams each page once for all of
  // them with two CTAs per SM
  if (index_chunk_tokens_ok(a)) return launch_index_chunk_tokens(a, stream);
  DeviceInfo dev;
  if (msa_status st = current_device(&dev); st != MSA_OK) return st;
  CUtensorMap qmap, kmap;
  {
    // q_idx as 5-D (dI, h, g, s, b); box = one head of 64 queries
    const uint64_t dims[5] = {static_cast<uint64_t>(a.dI), static_cast<uint64_t>(a.HI), static_cast<uint64_t>(a.Hkv),
                              static_cast<uint64_t>(a.S), static_cast<uint64_t>(a.B)};
    const uint64_t strides[4] = {static_cast<uint64_t>(a.q_idx_stride[3]) * 2,
                                 static_cast<uint64_t>(a.q_idx_stride[2]) * 2,
                                 static_cast<uint64_t>(a.q_idx_stride[1]) * 2,
                                 static_cast<uint64_t>(a.q_idx_stride[0]) * 2};
    const uint32_t box[5] = {64, 1, 1, kQB, 1};
    if (msa_status st = encode_tiled_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, a.q_idx, dims, strides, box,
                                         CU_TENSOR_MAP_SWIZZLE_128B, "q_idx");
        st != MSA_OK)
      return st;
  }
  const bool chunk = a.mode == MSA_MODE_CHUNK;
  if (chunk) {
    // index-key pool as 4-D (dI, t, g, page) with strides (page, g, t); box =
    // one page of one group.  A group stride of 0 becomes a g extent of 1.
    const bool shared = a.k_idx_stride[1] == 0;
    const uint64_t dims[4] = {static_cast<uint64_t>(a.dI), static_cast<uint64_t>(kBk),
                              static_cast<uint64_t>(shared ? 1 : a.Hkv), static_cast<uint64_t>(a.num_pages)};
    const uint64_t strides[3] = {static_cast<uint64_t>(a.k_idx_stride[2]) * 2,
                                 static_cast<uint64_t>(shared ? a.k_idx_stride[2] * kBk : a.k_idx_stride[1]) * 2,
                                 static_cast<uint64_t>(a.k_idx_stride[0]) * 2};
    const uint32_t box[4] = {64, kBk, 1, 1};
    if (msa_status st = encode_tiled_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.k_idx, dims, strides, box,
                                         CU_TENSOR_MAP_SWIZZLE_128B, "k_idx pool");
        st != MSA_OK)
      return st;
  } else {
    // k_idx as 4-D (dI, g, s, b); box = 128 tokens of one group.  A group
    // stride of 0 (one k_idx for all groups) becomes a g extent of 1.
    // (k_idx_stride is (b, s, g): the group stride is the last one)
    const bool shared = a.k_idx_stride[2] == 0;
    const uint64_t dims[4] = {static_cast<uint64_t>(a.dI), static_cast<uint64_t>(shared ? 1 : a.Hkv),
                              static_cast<uint64_t>(a.S), static_cast<uint64_t>(a.B)};
    const uint64_t strides[3] = {static_cast<uint64_t>(shared ? a.k_idx_stride[1] : a.k_idx_stride[2]) * 2,
                                 static_cast<uint64_t>(a.k_idx_stride[1]) * 2,
                                 static_cast<uint64_t>(a.k_idx_stride[0]) * 2};
    const uint32_t box[4] = {64, 1, kBk, 1};
    if (msa_status st = encode_tiled_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.k_idx, dims, strides, box,
                                         CU_TENSOR_MAP_SWIZZLE_128B, "k_idx");
        st != MSA_OK)
      return st;
  }
  Params p;
  p.B = a.B; p.S = a.S; p.Hkv = a.Hkv; p.HI = a.HI;
  p.nq = (a.S + kQB - 1) / kQB;
  p.kgroups = chunk ? a.k_idx_stride[1] != 0 : a.k_idx_stride[2] != 0;
  p.chunk = chunk;
  p.q_pos = a.q_pos; p.seq_pt = a.seq_pt; p.max_pages = a.max_pages; p.num_pages = a.num_pages;
  p.nb_stride = a.nb_stride;
  p.w = a.w; p.ws0 = a.w_stride[0]; p.ws1 = a.w_stride[1]; p.ws2 = a.w_stride[2];
  p.C = a.C; p.cs0 = a.C_stride[0]; p.cs1 = a.C_stride[1]; p.cs2 = a.C_stride[2];
  p.dev_err = a.dev_err;
  const size_t smem = 1024 + 2 * static_cast<size_t>(kQTile) + static_cast<size_t>(kKStages) * kKTile;
  if (smem > dev.max_smem_optin) return fail(MSA_ERR_UNSUPPORTED, "prefill index score: not enough shared memory");
  using Kern = void (*)(const CUtensorMap, const CUtensorMap, const Params);
  static constexpr Kern kPrefill[4] = {index_prefill_kernel<1, false, false>, index_prefill_kernel<2, false, false>,
                                       index_prefill_kernel<3, false, false>, index_prefill_kernel<4, false, false>};
  static constexpr Kern kChunk[4] = {index_prefill_kernel<1, true, false>, index_prefill_kernel<2, true, false>,
                                     index_prefill_kernel<3, true, false>, index_prefill_kernel<4, true, false>};
  static constexpr Kern kFew[4] = {index_prefill_kernel<1, true, true>, index_prefill_kernel<2, true, true>,
                                   index_prefill_kernel<3, true, true>, index_prefill_kernel<4, true, true>};
  const Kern kern = (!chunk ? kPrefill : a.S <= kCQ ? kFew : kChunk)[a.HI - 1];
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(index_prefill)");
  // Too few items for many per slot of every CTA: split each item's key
  // blocks into ranges of at least 16 blocks (the longest row has at most
  // max_own blocks before its own).  A chunk's items all have about the same
  // length (the cached prefix), so a few per slot leave the CTAs unevenly
  // loaded (3 or 4 pairs a CTA for an 8,192-query chunk of 8 KV groups);
  // about sixteen items per CTA keep the spread small.  (Prefill items, long and short
  // paired, are not split.)
  const int64_t items = static_cast<int64_t>(a.B) * a.Hkv * p.nq;
  const int64_t want = 16 * static_cast<int64_t>(dev.num_sms);
  const int64_t max_own = a.max_pages;
  p.nsplit = !chunk || items >= want
                  ? 1
                  : static_cast<int>(std::max<int64_t>(1, std::min((want + items - 1) / items, max_own / 16)));
  const int64_t npairs = static_cast<int64_t>(a.B) * a.Hkv * ((p.nq + 1) / 2) * p.nsplit;
  if (npairs >= (int64_t(1) << 31)) return fail(MSA_ERR_UNSUPPORTED, "prefill index score: too many query blocks");
  const int grid = static_cast<int>(std::min<int64_t>(dev.num_sms, std::max<int64_t>(npairs, 1)));
  kern<<<grid, kThreads, smem, stream>>>(qmap, kmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "index_prefill_kernel launch");
  return MSA_OK;
}

}  // namespace msa
