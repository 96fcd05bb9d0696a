// index_decode.cu -- a1 (decode): block scores of the Index Branch over a paged
// index-key cache.
//
// For every sequence b, KV group g and block j strictly before the query's own
// block ((L_b - 1) / Bk):
//     c_j = max_{t in block j} sum_{h < HI} w[b,g,h] * ReLU(q_idx[b,g,h] . k_idx_t)
// ("MiniMax M3: Como la atencion dispersa hace practicos a los agentes de largo
// alcance", MSA paragraph and caption: a light Index Branch scores the context
// in blocks; the formula is this library's, the pages give none.)
//
// This is an HBM stream: each (page, group) block of k_idx is 16 KiB, read
// once.  Two persistent CTAs per SM each walk a contiguous range of the
// flattened (b, g, j) items:
//   warp 0    TMA producer: one 4-D tiled load (128 tokens x 64 dims, 128-byte
//             swizzle) per block into a 6-deep shared-memory ring, page ids
//             fetched 32 at a time by the whole warp;
//   warp 1    tcgen05 issuer: D[t, h] = k_idx_t . q_idx_h as one M=128 (tokens)
//             x N=16 (index heads, zero-padded) x K=64 contraction (4 MMAs)
//             into one of 8 TMEM slots; it also stages q_idx of the current
//             (b, g) as the B operand (double-buffered);
//   warps 2-5 epilogue: thread = token; w-weighted ReLU sum over heads, max
//             over the block's 128 tokens, one fp32 store per block.
// With the optional fused selection, the CTA that completes a (b, g) row
// (per-row completion counter) then selects its top-k blocks and writes the
// row's page table, using the idle ring as scratch.
#include "msa_internal.h"
#include "msa_ptx.cuh"
#include "select_warp.cuh"

namespace msa {
namespace {

// Two CTAs per SM: one tcgen05 issue stream per CTA serialises on MMA latency,
// two overlap and keep the stream at the HBM rate.
constexpr int kCtasPerSm = 2;
constexpr int kStages = 6;
constexpr int kSlots = 8;
constexpr int kSlotCols = 16;
constexpr int kTmemCols = 128;
constexpr int kStageBytes = kBk * kDI * 2;   // 16 KiB
constexpr int kQTileBytes = 16 * kDI * 2;    // 2 KiB: 16 rows (HI used) x 64
// Shared-index variant (one k_idx pool for all KV groups): an item is (b, j),
// the B operand holds the index heads of all groups (g*HI + h, HI = 4,
// Hkv <= 8: 32 rows) and one M=128 x N=32 contraction scores every group.
constexpr int kSharedRows = 32;
constexpr int kSharedHI = 4;
constexpr int kThreads = 192;
// Partial-max buffers of the epilogue.  A warp can be at most kSlots items
// ahead of the slowest one (TMEM slots are released by all four), so twice
// that many buffers are never reused while still being read.
constexpr int kRedBufs = 2 * kSlots;

struct Params {
  int B, Hkv, HI, Bk;
  int S;                                  // multi-token mode: tokens per sequence (1 otherwise)
  const int32_t* q_pos;                   // multi-token mode: position of token 0 of sequence b
  int64_t qs_s, ws_s, cs_s;               // multi-token mode: q_idx, w and C strides of the token
  const __nv_bfloat16* q_idx;
  int64_t qs0, qs1, qs2;
  const float* w;
  int64_t ws0, ws1;
  int64_t num_pages;
  const int32_t* seq_pt;
  int64_t max_pages;
  const int32_t* seq_len;
  float* C;
  int64_t cs0, cs1;
  int nb_stride;
  int32_t* dev_err;
  // optional fused selection (a2) and page table (a3)
  int k;
  int32_t* sel;
  int32_t* count;
  int32_t* pt;
  int32_t* n_out;
  int32_t* last_len;
  int32_t* counter;
};

struct Walker {  // position in the flattened (b, g, j) item space
  int b, g, j;
};

__device__ __forceinline__ void walk_init(Walker& w, int64_t n, const int* pre, const int* own, int B, int Hkv) {
  // largest b with pre[b] <= n (pre is non-decreasing; items of b are [pre[b], pre[b+1]))
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= n) lo = mid; else hi = mid - 1;
  }
  int b = lo;
  while (b < B - 1 && pre[b + 1] <= n) ++b;   // skip sequences with no items
  int64_t rem = n - pre[b];
  w.b = b;
  w.g = static_cast<int>(rem / own[b]);
  w.j = static_cast<int>(rem % own[b]);
  (void)Hkv;
}

__device__ __forceinline__ void walk_next(Walker& w, const int* own, int B, int Hkv) {
  if (++w.j < own[w.b]) return;
  w.j = 0;
  if (++w.g < Hkv) return;
  w.g = 0;
  do { ++w.b; } while (w.b < B && own[w.b] == 0);
}

// Block-wide maximum of a uint64 over the kThreads threads of the CTA.
__device__ __forceinline__ uint64_t block_max_u64(uint64_t v, uint64_t* s_w) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  v = warp_max_u64(v);
  if (lane == 0) s_w[wid] = v;
  __syncthreads();
  if (wid == 0) {
    uint64_t x = lane < kThreads / 32 ? s_w[lane] : 0ull;
    x = warp_max_u64(x);
    if (lane == 0) s_w[kThreads / 32] = x;
  }
  __syncthreads();
  const uint64_t r = s_w[kThreads / 32];
  __syncthreads();
  return r;
}

// Writes the selection (a2) and, if requested, the page-table row (a3) of
// decode row (b, g): own block + the k-1 best earlier blocks by (score desc,
// index asc), ascending, -1 padded.  `valid` is false for a sequence whose
// length failed the checks (count 0).  All threads of the CTA call this.
__device__ void emit_row(const Params& p, int b, int g, int own, bool valid, const int* picks, int m_picked) {
  const int r = b * p.Hkv + g;
  const int tid = threadIdx.x;
  const int cnt = valid ? m_picked + 1 : 0;
  // entries from m_picked on: the own block, then -1 padding
  for (int x = m_picked + tid; x < p.k; x += kThreads) {
    const int j = (x == m_picked && valid) ? own : -1;
    p.sel[static_cast<int64_t>(r) * p.k + x] = j;
    if (p.pt != nullptr) p.pt[static_cast<int64_t>(r) * p.k + x] = j >= 0 ? p.seq_pt[b * p.max_pages + j] : -1;
  }
  // the picks, each placed at its rank in ascending order
  for (int t = tid; t < m_picked; t += kThreads) {
    const int jt = picks[t];
    int pos = 0;
    for (int y = 0; y < m_picked; ++y) pos += picks[y] < jt;
    p.sel[static_cast<int64_t>(r) * p.k + pos] = jt;
    if (p.pt != nullptr) p.pt[static_cast<int64_t>(r) * p.k + pos] = p.seq_pt[b * p.max_pages + jt];
  }
  if (tid == 0) {
    p.count[r] = cnt;
    if (p.pt != nullptr) {
      p.n_out[r] = cnt;
      const int L = p.seq_len[b];
      p.last_len[r] = valid ? L - p.Bk * own : 0;
    }
  }
}

// Exact top-(k-1) of the own_b earlier blocks of row (b, g), by m rounds of a
// block-wide arg-max below the previous pick; candidate keys are staged in
// shared memory when they fit, else re-read from C (L2) every round.
__device__ void select_row(const Params& p, int b, int g, int own, uint64_t* s_keys, int key_cap, uint64_t* s_w,
                           int* s_picks) {
  const int m = p.k - 1;
  if (own <= m) {
    for (int x = threadIdx.x; x < own; x += kThreads) s_picks[x] = x;
    __syncthreads();
    emit_row(p, b, g, own, true, s_picks, own);
    __syncthreads();
    return;
  }
  const float* crow = p.C + b * p.cs0 + g * p.cs1;
  const bool staged = own <= key_cap;
  if (staged) {
    for (int j = threadIdx.x; j < own; j += kThreads) s_keys[j] = select_key(__ldcg(crow + j), j);
    __syncthreads();
  }
  uint64_t prev = ~0ull;
  for (int t = 0; t < m; ++t) {
    uint64_t best = 0;
    for (int j = threadIdx.x; j < own; j += kThreads) {
      const uint64_t key = staged ? s_keys[j] : select_key(__ldcg(crow + j), j);
      if (key < prev && key > best) best = key;
    }
    best = block_max_u64(best, s_w);
    prev = best;
    if (threadIdx.x == 0) s_picks[t] = select_key_index(best);
  }
  __syncthreads();
  emit_row(p, b, g, own, true, s_picks, m);
  __syncthreads();
}

// Exact top-(k-1) of a long row (own > 2048 earlier blocks) in two phases:
// the row is cut into slices of at most 2048 blocks; each warp selects the best
// m of its slices with the register-based warp select into a pool (slot
// slice * m + y; 0 = empty, below every real key); then every thread ranks
// the pool's keys exactly and the m best are the picks.  The row's best m
// blocks are among the pool: a block outside its slice's best m has m better
// blocks in its own slice.  Falls back to select_row when the pool does not
// fit.  All threads of the CTA call this.
__device__ void select_long_row(const Params& p, int b, int g, int own, uint64_t* s_pool, int pool_cap,
                                uint64_t* s_surv, int (*s_wpick)[kMaxK], int (*s_wout)[kMaxK], int* s_final,
                                uint64_t* s_w) {
  const int m = p.k - 1;
  const int nslices = (own + 2047) / 2048;
  if (own <= m || static_cast<int64_t>(nslices) * m > pool_cap) {
    select_row(p, b, g, own, s_pool, pool_cap, s_w, s_final);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ssz = (own + nslices - 1) / nslices;     // <= 2048
  const float* crow = p.C + b * p.cs0 + g * p.cs1;
  for (int sl = warp; sl < nslices; sl += kThreads / 32) {
    const int lo = sl * ssz, n = min(ssz, own - lo);
    int* out = s_wout[warp];
    int npick = n;
    if (n <= m) {
      for (int y = lane; y < n; y += 32) out[y] = y;
    } else {
      warp_select_any(crow + lo, n, m, s_surv + warp * kSelCap, s_wpick[warp], out);
      npick = m;
    }
    __syncwarp();
    for (int y = lane; y < m; y += 32)
      s_pool[sl * m + y] = y < npick ? select_key(__ldcg(crow + lo + out[y]), lo + out[y]) : 0ull;
    __syncwarp();
  }
  __syncthreads();
  const int npool = nslices * m;
  for (int x = threadIdx.x; x < npool; x += kThreads) {
    const uint64_t kx = s_pool[x];
    if (kx == 0ull) continue;
    int rank = 0;
    for (int y = 0; y < npool; ++y) rank += s_pool[y] > kx;
    if (rank < m) s_final[rank] = select_key_index(kx);
  }
  __syncthreads();
  emit_row(p, b, g, own, true, s_final, m);
  __syncthreads();
}

// SHARED: one index-key pool for all groups, items (b, j), B rows (g, h).
// MQ (multi-token): S <= 8 tokens per sequence at positions q_pos[b] + s over
// per-group keys, items (b, g, j), B rows (s, h) with h < HI <= 4; token s
// keeps the blocks before its own, (q_pos[b] + s) / Bk.
template <bool SHARED, bool MQ>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
index_decode_kernel(const __grid_constant__ CUtensorMap kmap, const Params p) {
  constexpr bool WIDE = SHARED || MQ;                          // 32 B rows, 8 sums per token
  constexpr int QROWS = WIDE ? kSharedRows : 16;              // rows of the B operand (N)
  constexpr int SLOT = WIDE ? kSharedRows : kSlotCols;        // TMEM columns per slot
  constexpr int TCOLS = WIDE ? 2 * kTmemCols : kTmemCols;
  constexpr int QTILE = QROWS * kDI * 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_stage = smem;                                   // kStages x 16 KiB
  uint8_t* s_q = smem + kStages * kStageBytes;               // 2 q_idx tiles
  int* s_pre = reinterpret_cast<int*>(s_q + 2 * QTILE);      // B + 1
  int* s_own = s_pre + (p.B + 1);                             // B
  int* s_q0 = s_own + p.B;                                    // B (multi-token mode): q_pos, -1 if rejected
  // items per (b, j): one per group, or one for all groups with a shared index
  const int hkv_items = SHARED ? 1 : p.Hkv;

  __shared__ __align__(8) uint64_t bar_full[kStages], bar_empty[kStages];
  __shared__ __align__(8) uint64_t bar_tfull[kSlots], bar_tempty[kSlots];
  __shared__ __align__(8) uint64_t bar_qdone[2], bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ uint32_t s_red[kRedBufs][4][WIDE ? 8 : 1];
  __shared__ int s_cnt[kRedBufs];
  __shared__ int s_chunk[kThreads];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- per-sequence own blocks and the prefix over (b, g, j) items ----
  for (int b = tid; b < p.B; b += kThreads) {
    int own = 0;
    if constexpr (MQ) {
      // the items score the blocks before the last token's own block; a
      // sequence is rejected as a whole when its tokens start before 0 or the
      // last one leaves the pages or the score rows
      const int64_t q0 = p.q_pos[b], last = q0 + p.S - 1;
      const bool ok = q0 >= 0 && last < p.max_pages * p.Bk && last / p.Bk < p.nb_stride;
      if (!ok && blockIdx.x == 0) report(p.dev_err, MSA_DEVERR_BAD_LEN);
      own = ok ? static_cast<int>(last / p.Bk) : 0;
      s_q0[b] = ok ? static_cast<int>(q0) : -1;
    } else {
      const int L = p.seq_len[b];
      if (L < 1 || static_cast<int64_t>(L) > p.max_pages * p.Bk || (L - 1) / p.Bk >= p.nb_stride) {
        if (blockIdx.x == 0) report(p.dev_err, MSA_DEVERR_BAD_LEN);
      } else {
        own = (L - 1) / p.Bk;
      }
    }
    s_own[b] = own;
  }
  __syncthreads();
  {
    const int per = (p.B + kThreads - 1) / kThreads;
    const int b0 = tid * per, b1 = min(p.B, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += s_own[b] * hkv_items;
    s_chunk[tid] = sum;
    __syncthreads();
    if (tid == 0) {
      int run = 0;
      for (int t = 0; t < kThreads; ++t) { int v = s_chunk[t]; s_chunk[t] = run; run += v; }
      s_pre[p.B] = run;
    }
    __syncthreads();
    int run = s_chunk[tid];
    for (int b = b0; b < b1; ++b) { s_pre[b] = run; run += s_own[b] * hkv_items; }
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&bar_full[i], 1); mbar_init(&bar_empty[i], 1); }
    for (int i = 0; i < kSlots; ++i) { mbar_init(&bar_tfull[i], 1); mbar_init(&bar_tempty[i], 4); }
    mbar_init(&bar_qdone[0], 1); mbar_init(&bar_qdone[1], 1); mbar_init(&bar_drain, 1);
    s_abort = 0;
    for (int i = 0; i < kRedBufs; ++i) s_cnt[i] = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&s_tmem, TCOLS);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;

  // ---- -inf for the own block and everything after it ----
  {
    // rows (b, g), or (b, s, g) in multi-token mode (token s: from its own block on)
    const int64_t total = static_cast<int64_t>(p.B) * p.S * p.Hkv * p.nb_stride;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * kThreads + tid; e < total;
         e += static_cast<int64_t>(gridDim.x) * kThreads) {
      int j = static_cast<int>(e % p.nb_stride);
      int64_t r = e / p.nb_stride;
      const int g = static_cast<int>(r % p.Hkv);
      r /= p.Hkv;
      const int tk = static_cast<int>(r % p.S), b = static_cast<int>(r / p.S);
      if constexpr (MQ) {
        const int own_t = s_q0[b] < 0 ? 0 : (s_q0[b] + tk) / p.Bk;
        if (j >= own_t) p.C[b * p.cs0 + tk * p.cs_s + g * p.cs1 + j] = -INFINITY;
      } else {
        if (j >= s_own[b]) p.C[b * p.cs0 + g * p.cs1 + j] = -INFINITY;
      }
    }
  }
  if (!MQ && p.sel != nullptr && blockIdx.x == 0) {
    // rows with nothing to score: own block only (or nothing for a bad length)
    for (int r = tid; r < p.B * p.Hkv; r += kThreads) {
      const int b = r / p.Hkv;
      if (s_own[b] != 0) continue;
      const int L = p.seq_len[b];
      const bool valid = L >= 1 && static_cast<int64_t>(L) <= p.max_pages * p.Bk && (L - 1) / p.Bk < p.nb_stride;
      for (int x = 0; x < p.k; ++x) {
        const int j = (valid && x == 0) ? 0 : -1;
        p.sel[static_cast<int64_t>(r) * p.k + x] = j;
        if (p.pt != nullptr) p.pt[static_cast<int64_t>(r) * p.k + x] = j >= 0 ? p.seq_pt[b * p.max_pages] : -1;
      }
      p.count[r] = valid ? 1 : 0;
      if (p.pt != nullptr) {
        p.n_out[r] = valid ? 1 : 0;
        p.last_len[r] = valid ? L : 0;
      }
    }
  }

  const int64_t total_items = s_pre[p.B];
  const int64_t per_cta = (total_items + gridDim.x - 1) / gridDim.x;
  const int64_t lo = min(total_items, static_cast<int64_t>(blockIdx.x) * per_cta);
  const int64_t hi = min(total_items, lo + per_cta);
  const int count = static_cast<int>(hi - lo);

  if (warp == 0) {
    // ===================== TMA producer =====================
    // The page ids of the next 32 items are loaded by the 32 lanes at once, so
    // the TMA issue loop of lane 0 never waits on a global load.
    int issued = 0;
    bool ok = true;
    for (int base = 0; base < count && ok; base += 32) {
      const int nb = min(32, count - base);
      Walker w;
      int64_t page = -1;
      if (lane < nb) {
        walk_init(w, lo + base + lane, s_pre, s_own, p.B, hkv_items);
        page = p.seq_pt[w.b * p.max_pages + w.j];
      }
      for (int i = 0; i < nb; ++i) {
        const int64_t pg = __shfl_sync(0xffffffffu, page, i);
        const int g = __shfl_sync(0xffffffffu, w.g, i);
        if (lane == 0) {
          const int n = base + i;
          const int st = n % kStages;
          ok = mbar_wait(&bar_empty[st], ((n / kStages) & 1) ^ 1, abort_flag, p.dev_err);
          if (ok) {
            if (pg < 0 || pg >= p.num_pages) {
              mbar_arrive(&bar_full[st]);   // nothing to load; the epilogue reports the bad page
            } else {
              mbar_arrive_expect_tx(&bar_full[st], kStageBytes);
              tma_load_4d(s_stage + st * kStageBytes, &kmap, &bar_full[st], 0, 0, g, static_cast<int>(pg));
            }
            ++issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0 && *abort_flag) {  // drain loads still in flight before the CTA exits
      for (int n = max(0, issued - kStages); n < issued; ++n) {
        uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&bar_full[n % kStages], (n / kStages) & 1) &&
               global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
        }
      }
    }
  } else if (warp == 1) {
    // ===================== tcgen05 issuer =====================
    constexpr uint32_t idesc = idesc_bf16(128, QROWS, false, false);
    Walker it;
    if (count > 0) walk_init(it, lo, s_pre, s_own, p.B, hkv_items);
    int cur_b = -1, cur_g = -1, seg = -1;
    for (int n = 0; n < count; ++n) {
      const int st = n % kStages, slot = n % kSlots;
      if (it.b != cur_b || it.g != cur_g) {
        // new (b, g): stage its q_idx as the B operand in the other buffer
        if (lane == 0 && seg >= 0) umma_commit(&bar_qdone[seg & 1]);
        ++seg;
        const int buf = seg & 1;
        bool ok = true;
        if (seg >= 2 && lane == 0) ok = mbar_wait(&bar_qdone[buf], ((seg >> 1) - 1) & 1, abort_flag, p.dev_err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        uint8_t* qt = s_q + buf * QTILE;
        for (int c = lane; c < QROWS * 8; c += 32) {
          const int r = c >> 3, ch = c & 7;
          uint4 v = make_uint4(0, 0, 0, 0);
          if constexpr (SHARED) {   // row r = (group r / HI, head r % HI)
            if (r < p.Hkv * kSharedHI)
              v = *reinterpret_cast<const uint4*>(p.q_idx + it.b * p.qs0 + (r / kSharedHI) * p.qs1 +
                                                  (r % kSharedHI) * p.qs2 + ch * 8);
          } else if constexpr (MQ) {   // row r = (token r / 4, head r % 4)
            if (r / kSharedHI < p.S && r % kSharedHI < p.HI)
              v = *reinterpret_cast<const uint4*>(p.q_idx + it.b * p.qs0 + (r / kSharedHI) * p.qs_s + it.g * p.qs1 +
                                                  (r % kSharedHI) * p.qs2 + ch * 8);
          } else {
            if (r < p.HI)
              v = *reinterpret_cast<const uint4*>(p.q_idx + it.b * p.qs0 + it.g * p.qs1 + r * p.qs2 + ch * 8);
          }
          *reinterpret_cast<uint4*>(qt + sw128_offset(r, ch)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        cur_b = it.b;
        cur_g = it.g;
      }
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&bar_full[st], (n / kStages) & 1, abort_flag, p.dev_err) &&
             mbar_wait(&bar_tempty[slot], ((n / kSlots) & 1) ^ 1, abort_flag, p.dev_err);
        if (ok) {
          tc_fence_after();
          const uint32_t a0 = smem_u32(s_stage + st * kStageBytes);
          const uint32_t b0 = smem_u32(s_q + (seg & 1) * QTILE);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(tmem + slot * SLOT, sdesc_sw128(a0 + 32 * k, 16, 1024), sdesc_sw128(b0 + 32 * k, 16, 1024),
                      idesc, k > 0);
          umma_commit(&bar_empty[st]);
          umma_commit(&bar_tfull[slot]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      walk_next(it, s_own, p.B, hkv_items);
    }
    if (lane == 0) {  // every MMA issued by this thread is complete before TMEM is freed
      umma_commit(&bar_drain);
      uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&bar_drain, 0) && global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
      }
    }
    __syncwarp();
  } else {
    // ===================== epilogue (warps 2..5) =====================
    const int q = warp & 3;                       // TMEM lane quarter of this warp
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    Walker it;
    int64_t page_cur = 0;
    if (count > 0) {
      walk_init(it, lo, s_pre, s_own, p.B, hkv_items);
      page_cur = p.seq_pt[it.b * p.max_pages + it.j];
    }
    int cur_b = -1, cur_g = -1;
    constexpr int NW = WIDE ? kSharedRows : kMaxHI;     // weights: (g, h) or (token, h) pairs, or the HI heads
    constexpr int NG = WIDE ? 8 : 1;                    // groups (or tokens) scored per item
    float wv[NW];
#pragma unroll
    for (int c = 0; c < NW; ++c) wv[c] = 0.f;
    for (int n = 0; n < count; ++n) {
      const int slot = n % kSlots;
      // the next item's page id is loaded one item ahead, off the critical path
      Walker nxt = it;
      int64_t page_next = 0;
      if (n + 1 < count) {
        walk_next(nxt, s_own, p.B, hkv_items);
        page_next = p.seq_pt[nxt.b * p.max_pages + nxt.j];
      }
      if (it.b != cur_b || it.g != cur_g) {
#pragma unroll
        for (int c = 0; c < NW; ++c) {
          if constexpr (SHARED)
            wv[c] = c < p.Hkv * kSharedHI ? p.w[it.b * p.ws0 + (c / kSharedHI) * p.ws1 + c % kSharedHI] : 0.f;
          else if constexpr (MQ)
            wv[c] = c / kSharedHI < p.S && c % kSharedHI < p.HI
                        ? p.w[it.b * p.ws0 + (c / kSharedHI) * p.ws_s + it.g * p.ws1 + c % kSharedHI] : 0.f;
          else
            wv[c] = c < p.HI ? p.w[it.b * p.ws0 + it.g * p.ws1 + c] : 0.f;
        }
        cur_b = it.b;
        cur_g = it.g;
      }
      // the warp decides together: the TMEM load below is warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_tfull[slot], (n / kSlots) & 1, abort_flag, p.dev_err))) break;
      tc_fence_after();
      uint32_t wmax[NG];
      if constexpr (WIDE) {
        uint32_t v[kSharedRows];
        tmem_ld32(tmem + lane_addr + slot * SLOT, v);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_tempty[slot]);
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          float sg = 0.f;
#pragma unroll
          for (int h = 0; h < kSharedHI; ++h)
            sg = fmaf(wv[g * kSharedHI + h], fmaxf(__uint_as_float(v[g * kSharedHI + h]), 0.f), sg);
          wmax[g] = redux_max_u32(float_order_key(sg));
        }
      } else {
        uint32_t v[4];
        tmem_ld4(tmem + lane_addr + slot * SLOT, v);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_tempty[slot]);
        float sg = 0.f;
#pragma unroll
        for (int h = 0; h < kMaxHI; ++h) sg = fmaf(wv[h], fmaxf(__uint_as_float(v[h]), 0.f), sg);
        // warp max in one step on order-preserving integer keys
        wmax[0] = redux_max_u32(float_order_key(sg));
      }
      // cross-warp max without a barrier: the last of the four warps to arrive
      // combines the partial maxima and stores the block score(s), lane g
      // taking group g.
      const int rb = n % kRedBufs;
      int last = 0;
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < NG; ++g) s_red[rb][q][g] = wmax[g];
        __threadfence_block();
        last = atomicAdd(&s_cnt[rb], 1) == 3;
        if (last) {
          __threadfence_block();
          s_cnt[rb] = 0;
        }
      }
      __syncwarp();
      if (__shfl_sync(0xffffffffu, last, 0)) {
        const bool bad = page_cur < 0 || page_cur >= p.num_pages;
        if (bad && lane == 0) report(p.dev_err, MSA_DEVERR_BAD_PAGE);
        const int ng = SHARED ? p.Hkv : MQ ? p.S : 1;
        if (lane < ng) {
          const int g = WIDE ? lane : 0;
          const uint32_t mk = max(max(s_red[rb][0][g], s_red[rb][1][g]), max(s_red[rb][2][g], s_red[rb][3][g]));
          if constexpr (MQ) {
            // token g keeps the blocks before its own (the -inf fill covers the rest)
            if (it.j < (s_q0[it.b] + g) / p.Bk)
              p.C[it.b * p.cs0 + g * p.cs_s + it.g * p.cs1 + it.j] = bad ? -INFINITY : float_from_order_key(mk);
          } else {
            const int gg = SHARED ? g : it.g;
            p.C[it.b * p.cs0 + gg * p.cs1 + it.j] = bad ? -INFINITY : float_from_order_key(mk);
          }
        }
      }
      it = nxt;
      page_cur = page_next;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TCOLS);
  }

  // ---- fused selection: the CTA whose scores complete a (b, g) row selects it ----
  if (!MQ && p.sel != nullptr && !*abort_flag && count > 0) {
    __shared__ int s_nrows, s_nlong;
    // The TMA ring is idle now and holds the selection's scratch (static
    // shared memory would keep two CTAs of the shared-index variant from
    // fitting on one SM): survivors per warp at the start, the small arrays
    // at the end, staged keys in between.
    constexpr int kWarps = kThreads / 32;
    constexpr int kSmallBytes = 8 * (kWarps + 2) + 2 * kWarps * kMaxK * 4 + kMaxK * 4 + 2 * kThreads * 4;
    uint8_t* ring = s_stage;
    uint64_t* s_surv = reinterpret_cast<uint64_t*>(ring);                  // [warps][kSelCap]
    uint8_t* small = ring + kStages * kStageBytes - kSmallBytes;
    uint64_t* s_w = reinterpret_cast<uint64_t*>(small);                     // [warps + 1]
    int (*s_picks)[kMaxK] = reinterpret_cast<int (*)[kMaxK]>(small + 8 * (kWarps + 2));
    int (*s_out)[kMaxK] = s_picks + kWarps;
    int* s_final = reinterpret_cast<int*>(s_out + kWarps);                  // [kMaxK]
    int* s_rows = s_final + kMaxK;                                          // [kThreads]
    int* s_long = s_rows + kThreads;                                        // [kThreads]
    uint64_t* s_keys = reinterpret_cast<uint64_t*>(ring + kWarps * kSelCap * 8);
    const int key_cap = (kStages * kStageBytes - kWarps * kSelCap * 8 - kSmallBytes) / 8;
    const int m = p.k - 1;
    __threadfence();                                   // this CTA's scores, device-wide
    // this CTA's items cover the contiguous rows r_first .. r_last
    Walker wf, wl;
    walk_init(wf, lo, s_pre, s_own, p.B, hkv_items);
    walk_init(wl, hi - 1, s_pre, s_own, p.B, hkv_items);
    // with a shared index an item of sequence b counts toward all its groups' rows
    const int r_first = wf.b * p.Hkv + wf.g, r_last = wl.b * p.Hkv + (SHARED ? p.Hkv - 1 : wl.g);
    for (int base = r_first; base <= r_last; base += kThreads) {
      if (tid == 0) { s_nrows = 0; s_nlong = 0; }
      __syncthreads();
      const int r = base + tid;
      if (r <= r_last) {
        const int b = r / p.Hkv, g = r % p.Hkv;
        const int own = s_own[b];
        const int64_t row_start = s_pre[b] + (SHARED ? 0 : static_cast<int64_t>(g) * own);
        const int64_t mine64 = min(row_start + own, hi) - max(row_start, lo);
        if (own > 0 && mine64 > 0) {
          const int mine = static_cast<int>(mine64);
          if (atomicAdd(&p.counter[r], mine) + mine == own) {   // this CTA completed row r
            p.counter[r] = 0;                                   // no other CTA touches it again: leave it zero
            if (own <= 2048 || own <= m) s_rows[atomicAdd(&s_nrows, 1)] = r;
            else s_long[atomicAdd(&s_nlong, 1)] = r;
          }
        }
      }
      __syncthreads();
      __threadfence();                                 // scores written by other CTAs
      // short rows: one warp per row
      for (int x = warp; x < s_nrows; x += kThreads / 32) {
        const int rr = s_rows[x];
        const int b = rr / p.Hkv, g = rr % p.Hkv;
        const int own = s_own[b];
        const float* crow = p.C + b * p.cs0 + g * p.cs1;
        int* out = s_out[warp];
        int npick = own;
        if (own <= m) {
          for (int y = lane; y < own; y += 32) out[y] = y;
        } else {
          warp_select_any(crow, own, m, s_surv + warp * kSelCap, s_picks[warp], out);
          npick = m;
        }
        __syncwarp();
        for (int y = lane; y < p.k; y += 32) {
          const int j = y < npick ? out[y] : (y == npick ? own : -1);
          p.sel[static_cast<int64_t>(rr) * p.k + y] = j;
          if (p.pt != nullptr) p.pt[static_cast<int64_t>(rr) * p.k + y] = j >= 0 ? p.seq_pt[b * p.max_pages + j] : -1;
        }
        if (lane == 0) {
          p.count[rr] = npick + 1;
          if (p.pt != nullptr) {
            p.n_out[rr] = npick + 1;
            p.last_len[rr] = p.seq_len[b] - p.Bk * own;
          }
        }
        __syncwarp();
      }
      // long rows: the whole CTA
      for (int x = 0; x < s_nlong; ++x) {
        const int rr = s_long[x];
        select_long_row(p, rr / p.Hkv, rr % p.Hkv, s_own[rr / p.Hkv], s_keys, key_cap, s_surv, s_picks, s_out,
                        s_final, s_w);
      }
      __syncthreads();
    }
  }
}

}  // namespace

namespace {

msa_status launch_index_decode_impl(const msa_index_args& a, bool mq, cudaStream_t stream) {
  DeviceInfo dev;
  if (msa_status st = current_device(&dev); st != MSA_OK) return st;
  // k_idx pool as a 4-D tensor (dI, t, g, page) with a 64 x 128 x 1 x 1 box; a
  // group stride of 0 means one index pool shared by all groups (a g extent of 1)
  const bool shared = a.k_idx_stride[1] == 0;
  if (shared && (a.HI != kSharedHI || a.Hkv * a.HI > kSharedRows))
    return fail(MSA_ERR_UNSUPPORTED, "shared index keys (k_idx group stride 0): supported for HI = 4 and Hkv <= 8");
  CUtensorMap kmap;
  const uint64_t dims[4] = {static_cast<uint64_t>(a.dI), static_cast<uint64_t>(a.Bk),
                            static_cast<uint64_t>(shared ? 1 : a.Hkv), static_cast<uint64_t>(a.num_pages)};
  const uint64_t strides[3] = {static_cast<uint64_t>(a.k_idx_stride[2]) * 2,
                               static_cast<uint64_t>(shared ? a.k_idx_stride[2] * a.Bk : a.k_idx_stride[1]) * 2,
                               static_cast<uint64_t>(a.k_idx_stride[0]) * 2};
  const uint32_t box[4] = {64, 128, 1, 1};
  if (msa_status st = encode_tiled_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.k_idx, dims, strides, box,
                                       CU_TENSOR_MAP_SWIZZLE_128B, "k_idx page pool");
      st != MSA_OK)
    return st;

  Params p;
  p.B = a.B; p.Hkv = a.Hkv; p.HI = a.HI; p.Bk = a.Bk;
  p.q_idx = static_cast<const __nv_bfloat16*>(a.q_idx);
  p.w = a.w;
  p.num_pages = a.num_pages; p.seq_pt = a.seq_pt; p.max_pages = a.max_pages;
  p.C = a.C; p.nb_stride = a.nb_stride;
  p.dev_err = a.dev_err;
  if (mq) {   // chunk strides: q_idx (b, s, g, h), w and C (b, s, g)
    p.S = a.S; p.q_pos = a.q_pos; p.seq_len = nullptr;
    p.qs0 = a.q_idx_stride[0]; p.qs_s = a.q_idx_stride[1]; p.qs1 = a.q_idx_stride[2]; p.qs2 = a.q_idx_stride[3];
    p.ws0 = a.w_stride[0]; p.ws_s = a.w_stride[1]; p.ws1 = a.w_stride[2];
    p.cs0 = a.C_stride[0]; p.cs_s = a.C_stride[1]; p.cs1 = a.C_stride[2];
  } else {    // decode strides: q_idx (b, g, h), w and C (b, g)
    p.S = 1; p.q_pos = nullptr; p.seq_len = a.seq_len;
    p.qs0 = a.q_idx_stride[0]; p.qs_s = 0; p.qs1 = a.q_idx_stride[1]; p.qs2 = a.q_idx_stride[2];
    p.ws0 = a.w_stride[0]; p.ws_s = 0; p.ws1 = a.w_stride[1];
    p.cs0 = a.C_stride[0]; p.cs_s = 0; p.cs1 = a.C_stride[1];
  }
  p.k = a.k; p.sel = mq ? nullptr : a.sel; p.count = a.count; p.pt = a.pt; p.n_out = a.n; p.last_len = a.last_len;
  p.counter = a.row_scratch;
  // With one pool for all groups every group row of a sequence is completed
  // by the same CTA, which would select them one after another; rows of more
  // than 2048 blocks are therefore selected by the top-k kernel instead (one
  // CTA per row, all rows at once) and mapped by the page-table kernel: the
  // same outputs, two more launches.
  const bool select_after = !mq && shared && a.sel != nullptr && a.nb_stride > 2048;
  if (select_after) p.sel = nullptr;

  const size_t qtile = static_cast<size_t>(shared || mq ? kSharedRows : 16) * kDI * 2;
  const size_t smem = 1024 + kStages * kStageBytes + 2 * qtile + ((mq ? 3 : 2) * static_cast<size_t>(a.B) + 1) * 4;
  if (smem > dev.max_smem_optin) return fail(MSA_ERR_UNSUPPORTED, "decode index score: batch too large for shared memory");
  auto kern = mq ? index_decode_kernel<false, true>
                 : shared ? index_decode_kernel<true, false> : index_decode_kernel<false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(index_decode)");
  if (p.sel != nullptr && !a.scratch_zeroed) {   // otherwise zero by contract (and unused without p.sel)
    e = cudaMemsetAsync(p.counter, 0, static_cast<size_t>(a.B) * a.Hkv * sizeof(int32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(index row counters)");
  }
  // Two CTAs per SM, all resident at once: with the 1 KB the system keeps per
  // CTA, two fit up to B = 1024 with per-group keys and B = 256 with a shared
  // pool; a larger shared-pool batch runs the grid in two waves.
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(index_decode carveout)");
  const int grid = dev.num_sms * kCtasPerSm;
  kern<<<grid, kThreads, smem, stream>>>(kmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "index_decode_kernel launch");
  if (!select_after) return MSA_OK;
  msa_topk_args t{};
  t.mode = MSA_MODE_DECODE;
  t.B = a.B; t.S = 1; t.Hkv = a.Hkv; t.Bk = a.Bk; t.k = a.k;
  t.C = a.C; t.C_stride[0] = a.C_stride[0]; t.C_stride[1] = a.C_stride[1]; t.C_stride[2] = 0;
  t.nb_stride = a.nb_stride; t.seq_len = a.seq_len;
  t.sel = a.sel; t.count = a.count; t.dev_err = a.dev_err; t.q_pos = nullptr;
  if (msa_status st = launch_topk(t, stream); st != MSA_OK) return st;
  if (a.pt == nullptr) return MSA_OK;
  return launch_page_table(a.sel, a.count, a.seq_pt, a.max_pages, a.seq_len, a.B, a.Hkv, a.k, a.Bk, a.pt, a.n,
                           a.last_len, a.dev_err, stream);
}

}  // namespace

msa_status launch_index_decode(const msa_index_args& a, cudaStream_t stream) {
  return launch_index_decode_impl(a, false, stream);
}

bool index_chunk_tokens_ok(const msa_index_args& a) {
  return a.mode == MSA_MODE_CHUNK && a.S >= 1 && a.S <= kChunkDecodeMaxS && a.HI <= kSharedHI && a.dI == kDI &&
         a.k_idx_stride[1] != 0 && a.B <= kMaxDecodeBatch;
}

msa_status launch_index_chunk_tokens(const msa_index_args& a, cudaStream_t stream) {
  return launch_index_decode_impl(a, true, stream);
}

}  // namespace msa
