// dense_decode.cu -- the dense comparator of a decode step: exact GQA attention
// of one query per sequence over EVERY cached token of its paged K/V, with no
// index branch and no selection.
//
// The pages quote MSA's decode speed only against dense attention over the
// same cache ("MiniMax M3: Como la atencion dispersa hace practicos a los
// agentes de largo alcance", bullet "Rapido en produccion": 7.6x on H800; the
// M2-report article, section "MiniMax Sparse Attention (MSA) y escalado
// subcuadratico entrante": 15.6x at 1M tokens).  This kernel is that baseline
// built on the same machinery as the sparse decode kernel, so that the ratio
// can be measured on one GPU:
//     O[b, h] = sum_{t < L_b} softmax_t(scale * Q[b, h] . K[b, g, t]) V[b, g, t],  g = h / G.
//
// Work split (flash decoding): the pages of all rows r = b * Hkv + g are laid
// end to end, (b, g, j) in that order, and every CTA streams one contiguous
// range of that space (at least kMinPagesPerCta pages), so ragged batches are
// balanced without a host-side plan.  Per page the tcgen05 mapping is that of
// the sparse decode kernel (keys on M, the G heads on N):
//   MMA1  S^T[t][h] = K[t][:] . Q[h][:]    M = 128 keys, N = 16, K = 128
//   softmax: thread per key, per-head max / sum over the page, P^T in a
//            K-major B tile (bf16)
//   MMA2  O^T[d][h] = V^T[d][:] . P^T[:][h] M = 128, N = 16, K = 128 keys
// but instead of a partial per page, each softmax warpgroup keeps a running
// (max, sum, O) per head in registers (thread = d) over the pages it takes of
// a row, and writes one partial per (CTA, row, warpgroup) when the row ends.
// A per-row counter of processed pages tells the warpgroup that completes a
// row; it merges the row's partials with the log-sum-exp rule ("MiniMax M3
// preparado para inferencia en produccion", paragraph "KV-Block-Major").
#include <algorithm>
#include <cstdio>

#include "msa_internal.h"
#include "msa_ptx.cuh"

namespace msa {
namespace {

constexpr int kMinPagesPerCta = 32;   // a CTA's range is never shorter (bounds a row's partial count)
constexpr int kStages = 3;
constexpr int kHalf = 128 * 64 * 2;                    // 16 KiB: 128 rows x 64 bf16
constexpr int kQHalf = 16 * 64 * 2;                    // 2 KiB: 16 rows x 64 bf16
constexpr int kStageBytes = 4 * kHalf + 2 * kQHalf;    // K0 K1 V0 V1 Q0 Q1
constexpr int kPTile = 2 * kQHalf;                     // P^T: 16 rows x 128 keys
constexpr int kSlots = 2;
constexpr int kTmemCols = 64;
constexpr int kThreads = 320;   // w0 TMA, w1 MMA, w2-5 and w6-9 softmax/epilogue
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float fast_exp2(float x) {   // hardware 2^x (ex2.approx), 2^-inf = 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

struct Params {
  int B, Hq, Hkv, G;
  float scale_log2;
  int64_t num_pages, max_pages;
  const int32_t* seq_pt;                // [B, max_pages]
  const int32_t* seq_len;               // [B]
  int slots;                            // partial slots per (row, head)
  float* o_part;                        // [B*Hq][slots][D]
  float* lse_part;                      // [B*Hq][slots]
  int32_t* counter;                     // [B*Hkv] pages merged per row, zero on entry
  __nv_bfloat16* O;                     // [B, Hq, D]
  float* LSE;                           // [B, Hq] or null
  int32_t* dev_err;
};

// Position of flattened page u: sequence b, group g, page j of the row, and
// the row's page count np.  s_pref[b] = pages of the sequences before b (all
// groups); sequences without pages are skipped by the search.
struct Loc {
  int b, g, j, np;
};
__device__ __forceinline__ Loc locate(const int* s_pref, int B, int Hkv, int u) {
  int lo = 0, hi = B - 1;   // largest b with s_pref[b] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pref[mid] <= u) lo = mid; else hi = mid - 1;
  }
  // s_pref is non-decreasing; step over sequences with no pages at u
  while (s_pref[lo + 1] <= u) ++lo;
  Loc l;
  l.b = lo;
  l.np = (s_pref[lo + 1] - s_pref[lo]) / Hkv;
  const int off = u - s_pref[lo];
  l.g = off / l.np;
  l.j = off - l.g * l.np;
  return l;
}

__global__ void __launch_bounds__(kThreads, 1)
dense_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const __grid_constant__ CUtensorMap qmap, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_stage = smem;
  uint8_t* s_p = smem + kStages * kStageBytes;   // kSlots P^T tiles

  __shared__ __align__(8) uint64_t bar_full[kStages], bar_empty[kStages];
  __shared__ __align__(8) uint64_t bar_sfull[kSlots], bar_pready[kSlots], bar_ofull[kSlots], bar_sfree[kSlots];
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ __align__(16) float s_max[2][4][kMaxG];
  __shared__ __align__(16) float s_sum[2][4][kMaxG];
  __shared__ int s_pref[kDenseMaxBatch + 1];     // pages of sequences 0..b-1, all groups
  __shared__ int s_len[kDenseMaxBatch];          // sequence lengths
  __shared__ int s_lastw[2], s_fail[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- prefix of the page counts over the sequences (warp 0), lengths ----
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + lane;
      int L = 0, v = 0;
      if (b < p.B) {
        L = p.seq_len[b];
        const bool ok = L >= 1 && static_cast<int64_t>(L) <= p.max_pages * kBk;
        v = ok ? p.Hkv * ((L + kBk - 1) / kBk) : 0;
        s_len[b] = L;
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += x;
      }
      if (b < p.B) s_pref[b + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_pref[0] = 0;
  }
  __syncthreads();
  const int T = s_pref[p.B];
  const int per_cta = max(kMinPagesPerCta, (T + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x));
  const int lo = min(T, static_cast<int>(blockIdx.x) * per_cta);
  const int hi = min(T, lo + per_cta);
  const int cnt = hi - lo;

  // sequences with a length outside [1, max_pages * Bk]: O = 0, LSE = -inf
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    if (s_pref[b + 1] != s_pref[b]) continue;
    if (tid == 0) report(p.dev_err, MSA_DEVERR_BAD_LEN);
    for (int e = tid; e < p.Hq * (kD / 8); e += kThreads) {
      const int64_t row = static_cast<int64_t>(b) * p.Hq + e / (kD / 8);
      *reinterpret_cast<uint4*>(p.O + row * kD + (e % (kD / 8)) * 8) = make_uint4(0, 0, 0, 0);
      if (p.LSE != nullptr && e % (kD / 8) == 0) p.LSE[row] = -INFINITY;
    }
  }
  // this CTA's partial slots of every row it touches start empty (LSE -inf):
  // a warpgroup that gets no page of a row leaves its slot so
  if (cnt > 0) {
    const Loc a = locate(s_pref, p.B, p.Hkv, lo), z = locate(s_pref, p.B, p.Hkv, hi - 1);
    const int r0 = a.b * p.Hkv + a.g, r1 = z.b * p.Hkv + z.g;
    for (int e = tid; e < (r1 - r0 + 1) * p.G * 2; e += kThreads) {
      const int r = r0 + e / (p.G * 2), h = (e / 2) % p.G, w = e & 1;
      const int b = r / p.Hkv, g = r % p.Hkv;
      const int np = (s_pref[b + 1] - s_pref[b]) / p.Hkv;
      if (np == 0) continue;
      const int start = s_pref[b] + g * np;
      const int seg = static_cast<int>(blockIdx.x) - start / per_cta;
      p.lse_part[(static_cast<int64_t>(r) * p.G + h) * p.slots + 2 * seg + w] = -INFINITY;
    }
    __threadfence();
  }
  // P^T rows G..15 stay zero for the whole kernel
  for (int i = tid; i < kSlots * kPTile / 16; i += kThreads)
    reinterpret_cast<uint4*>(s_p)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) { mbar_init(&bar_full[i], 1); mbar_init(&bar_empty[i], 1); }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&bar_sfull[i], 1); mbar_init(&bar_pready[i], 4);
      mbar_init(&bar_ofull[i], 1); mbar_init(&bar_sfree[i], 4);
    }
    mbar_init(&bar_drain, 1);
    s_abort = 0;
    s_fail[0] = s_fail[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&s_tmem, kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // ===================== TMA producer (warp-uniform loop, lane 0 issues) =====================
    int n = 0;
    bool ok = true;
    for (int base = 0; base < cnt && ok; base += 32) {
      // lane l looks up the page id of unit base + l (one round trip for 32 pages)
      int pg = -1, bg = 0;
      if (base + lane < cnt) {
        const Loc l = locate(s_pref, p.B, p.Hkv, lo + base + lane);
        pg = p.seq_pt[static_cast<int64_t>(l.b) * p.max_pages + l.j];
        bg = l.b * p.Hkv + l.g;
      }
      for (int i = 0; i < 32 && base + i < cnt; ++i, ++n) {
        const int page = __shfl_sync(0xffffffffu, pg, i);
        const int r = __shfl_sync(0xffffffffu, bg, i);
        const int st = n % kStages;
        int go = 1;
        if (lane == 0) {
          go = mbar_wait(&bar_empty[st], ((n / kStages) & 1) ^ 1, abort_flag, p.dev_err);
          if (go) {
            const int b = r / p.Hkv, g = r % p.Hkv;
            uint8_t* sb = s_stage + st * kStageBytes;
            if (page < 0 || page >= p.num_pages) {   // not loaded: the softmax skips the page
              mbar_arrive(&bar_full[st]);
            } else {
              mbar_arrive_expect_tx(&bar_full[st], kStageBytes);
              tma_load_4d(sb + 0 * kHalf, &kmap, &bar_full[st], 0, 0, g, page);
              tma_load_4d(sb + 1 * kHalf, &kmap, &bar_full[st], 64, 0, g, page);
              tma_load_4d(sb + 2 * kHalf, &vmap, &bar_full[st], 0, 0, g, page);
              tma_load_4d(sb + 3 * kHalf, &vmap, &bar_full[st], 64, 0, g, page);
              tma_load_3d(sb + 4 * kHalf, &qmap, &bar_full[st], 0, g * p.G, b);
              tma_load_3d(sb + 4 * kHalf + kQHalf, &qmap, &bar_full[st], 64, g * p.G, b);
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, go, 0)) {
          ok = false;
          break;
        }
      }
    }
    if (lane == 0 && *abort_flag) {   // let loads in flight land before the CTA exits
      for (int i = max(0, n - kStages); i < n; ++i) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&bar_full[i % kStages], (i / kStages) & 1) &&
               global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ===================== tcgen05 issuer =====================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 16, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, 16, true, false);
      int ns = 0, no = 0;
      uint32_t spins = 0;
      uint64_t idle_since = 0;
      while (no < cnt) {
        bool progress = false;
        if (ns < cnt) {
          const int st = ns % kStages, slot = ns & 1;
          if (mbar_test_wait(&bar_full[st], (ns / kStages) & 1) &&
              mbar_test_wait(&bar_sfree[slot], ((ns >> 1) & 1) ^ 1)) {
            tc_fence_after();
            const uint32_t sb = smem_u32(s_stage + st * kStageBytes);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * kHalf + 32 * (kk & 3);
              const uint32_t qoff = 4 * kHalf + (kk >> 2) * kQHalf + 32 * (kk & 3);
              umma_bf16(tmem + slot * 32, sdesc_sw128(sb + off, 16, 1024), sdesc_sw128(sb + qoff, 16, 1024), idesc_s,
                        kk > 0);
            }
            umma_commit(&bar_sfull[slot]);
            ++ns;
            progress = true;
          }
        }
        if (no < ns) {
          const int st = no % kStages, slot = no & 1;
          if (mbar_test_wait(&bar_pready[slot], (no >> 1) & 1)) {
            tc_fence_after();
            const uint32_t sb = smem_u32(s_stage + st * kStageBytes);
            const uint32_t pb = smem_u32(s_p + slot * kPTile);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t voff = 2 * kHalf + kk * 2048;          // 16 keys per step
              const uint32_t poff = (kk >> 2) * kQHalf + 32 * (kk & 3);
              umma_bf16(tmem + slot * 32 + 16, sdesc_sw128(sb + voff, kHalf, 1024), sdesc_sw128(pb + poff, 16, 1024),
                        idesc_o, kk > 0);
            }
            umma_commit(&bar_ofull[slot]);
            umma_commit(&bar_empty[st]);
            ++no;
            progress = true;
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
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&bar_drain, 0) && global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
      }
    }
    __syncwarp();
  } else {
    // ===================== softmax + running accumulation: two warpgroups =====================
    // Warpgroup wg takes the pages n = wg (mod 2) of this CTA (TMEM slot wg).
    const int wg = (warp - 2) >> 2;
    const int bar_id = 1 + wg;
    const int q = warp & 3;
    const int t = q * 32 + lane;                 // key index (MMA1) / d index (MMA2)
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const int G = p.G;
    int cur_r = -1, cur_np = 0, cur_seg = 0, run_pages = 0, cur_start = 0;
    float M[kMaxG], Lsum[kMaxG], acc[kMaxG];
    // End of this warpgroup's run of pages of row cur_r: write its partial into
    // slot (2 * segment + wg), add its page count to the row counter; the
    // warpgroup that brings the count to the row's page count merges the row.
    auto flush = [&]() {
      if (cur_r < 0) return;
      const int slot = 2 * cur_seg + wg;
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) {
        if (h < G) {
          const int64_t row = static_cast<int64_t>(cur_r) * G + h;
          const bool any = Lsum[h] > 0.f;
          p.o_part[(row * p.slots + slot) * kD + t] = any ? acc[h] / Lsum[h] : 0.f;
          if (t == h) p.lse_part[row * p.slots + slot] = any ? (M[h] + log2f(Lsum[h])) * kLn2 : -INFINITY;
        }
      }
      __threadfence();
      named_bar_sync(bar_id, 128);
      if (t == 0) s_lastw[wg] = atomicAdd(&p.counter[cur_r], run_pages) + run_pages == cur_np;
      named_bar_sync(bar_id, 128);
      if (!s_lastw[wg]) return;
      __threadfence();
      // merge: the row's segments are the CTAs first..last that hold its pages
      const int first = cur_start / per_cta, last = (cur_start + cur_np - 1) / per_cta;
      const int ns = 2 * (last - first + 1);
      const int lq = t >> 5, ll = t & 31;       // warp lq merges heads lq and lq + 4; lane ll owns d = 4 ll ..
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = lq + 4 * hh;
        if (h >= G) break;                       // warp-uniform
        const int64_t row = static_cast<int64_t>(cur_r) * G + h;
        const float* lrow = p.lse_part + row * p.slots;
        const float* orow = p.o_part + row * p.slots * kD;
        float m = -INFINITY;
        for (int x = ll; x < ns; x += 32) m = fmaxf(m, __ldcg(lrow + x));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sum = 0.f;
        for (int x = ll; x < ns; x += 32) {
          const float l = __ldcg(lrow + x);
          sum += l == -INFINITY ? 0.f : __expf(l - m);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = sum > 0.f ? 1.0f / sum : 0.f;
        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int x0 = 0; x0 < ns; x0 += 8) {       // eight slots' loads in flight at once
          float lv[8];
          float4 v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) lv[i] = x0 + i < ns ? __ldcg(lrow + x0 + i) : -INFINITY;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            v[i] = lv[i] == -INFINITY ? make_float4(0.f, 0.f, 0.f, 0.f)
                                      : __ldcg(reinterpret_cast<const float4*>(orow + (x0 + i) * kD) + ll);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float wgt = lv[i] == -INFINITY ? 0.f : __expf(lv[i] - m) * inv;
            a4.x = fmaf(wgt, v[i].x, a4.x);
            a4.y = fmaf(wgt, v[i].y, a4.y);
            a4.z = fmaf(wgt, v[i].z, a4.z);
            a4.w = fmaf(wgt, v[i].w, a4.w);
          }
        }
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(a4.x, a4.y), hi2 = __floats2bfloat162_rn(a4.z, a4.w);
        *reinterpret_cast<uint2*>(p.O + row * kD + 4 * ll) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo2), *reinterpret_cast<uint32_t*>(&hi2));
        if (ll == 0 && p.LSE != nullptr) p.LSE[row] = sum > 0.f ? m + __logf(sum) : -INFINITY;
      }
      if (t == 0) p.counter[cur_r] = 0;          // ready for the next call
    };
    for (int n = wg; n < cnt; n += 2) {
      const Loc l = locate(s_pref, p.B, p.Hkv, lo + n);
      const int r = l.b * p.Hkv + l.g;
      const int page = p.seq_pt[static_cast<int64_t>(l.b) * p.max_pages + l.j];
      if (r != cur_r) {
        flush();
        cur_r = r;
        cur_np = l.np;
        cur_start = s_pref[l.b] + l.g * l.np;
        cur_seg = static_cast<int>(blockIdx.x) - cur_start / per_cta;
        run_pages = 0;
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) {
          M[h] = -INFINITY;
          Lsum[h] = 0.f;
          acc[h] = 0.f;
        }
      }
      const int valid = l.j == l.np - 1 ? s_len[l.b] - kBk * l.j : kBk;
      const int slot = wg;
      const uint32_t ph_slot = (n >> 1) & 1;
      // ---- S^T ready: the warpgroup decides together whether to go on
      if (!mbar_wait(&bar_sfull[slot], ph_slot, abort_flag, p.dev_err)) s_fail[wg] = 1;
      named_bar_sync(bar_id, 128);
      if (s_fail[wg]) break;
      tc_fence_after();
      uint32_t sv[8];
      tmem_ld8(tmem + lane_addr + slot * 32, sv);
      tmem_ld_wait();
      float z[kMaxG];
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) z[h] = (t < valid) ? __uint_as_float(sv[h]) * p.scale_log2 : -INFINITY;
      {
        float wm[kMaxG];
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) wm[h] = warp_max_f32(z[h]);
        if (lane == 0) {
          float4* d = reinterpret_cast<float4*>(&s_max[wg][q][0]);
          d[0] = make_float4(wm[0], wm[1], wm[2], wm[3]);
          d[1] = make_float4(wm[4], wm[5], wm[6], wm[7]);
        }
      }
      named_bar_sync(bar_id, 128);
      float mx[kMaxG];
#pragma unroll
      for (int h = 0; h < kMaxG; ++h)
        mx[h] = fmaxf(fmaxf(s_max[wg][0][h], s_max[wg][1][h]), fmaxf(s_max[wg][2][h], s_max[wg][3][h]));
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) z[h] = (t < valid) ? fast_exp2(z[h] - mx[h]) : 0.f;
      // per-head sums over the warp's 32 keys by a transposed butterfly
      {
        const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
        float u[4], w2[2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float send = b4 ? z[i] : z[i + 4], keep = b4 ? z[i + 4] : z[i];
          u[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float send = b3 ? u[i] : u[i + 2], keep = b3 ? u[i + 2] : u[i];
          w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        float x = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        if ((lane & 3) == 0) s_sum[wg][q][lane >> 2] = x;
      }
      uint8_t* pt_tile = s_p + slot * kPTile + (t >> 6) * kQHalf;
      const uint32_t tc = static_cast<uint32_t>(t & 63);
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) {
        if (h < G) {
          __nv_bfloat16 bv = __float2bfloat16_rn(z[h]);
          *reinterpret_cast<__nv_bfloat16*>(pt_tile + sw128_offset(h, tc >> 3) + (tc & 7) * 2) = bv;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pready[slot]);
      named_bar_sync(bar_id, 128);
      float lp[kMaxG];
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) lp[h] = (s_sum[wg][0][h] + s_sum[wg][1][h]) + (s_sum[wg][2][h] + s_sum[wg][3][h]);
      // ---- O^T ready
      if (!mbar_wait(&bar_ofull[slot], ph_slot, abort_flag, p.dev_err)) s_fail[wg] = 1;
      named_bar_sync(bar_id, 128);
      if (s_fail[wg]) break;
      tc_fence_after();
      uint32_t ov[8];
      tmem_ld8(tmem + lane_addr + slot * 32 + 16, ov);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_sfree[slot]);
      if (page < 0 || page >= p.num_pages) {      // not loaded: contributes nothing
        if (t == 0) report(p.dev_err, MSA_DEVERR_BAD_PAGE);
      } else {
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) {
          const float mn = fmaxf(M[h], mx[h]);
          const float a = fast_exp2(M[h] - mn), c = fast_exp2(mx[h] - mn);
          acc[h] = fmaf(acc[h], a, __uint_as_float(ov[h]) * c);
          Lsum[h] = fmaf(Lsum[h], a, lp[h] * c);
          M[h] = mn;
        }
      }
      ++run_pages;
    }
    if (!s_fail[wg]) flush();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Partial slots per (row, head): two per CTA whose range holds pages of the
// row, at most min(grid, ceil(max_pages / kMinPagesPerCta) + 1) CTAs.
int dense_slots(int64_t max_pages) {
  const int64_t span = std::min<int64_t>(kDenseMaxGrid, (max_pages + kMinPagesPerCta - 1) / kMinPagesPerCta + 1);
  return static_cast<int>(2 * span);
}

}  // namespace

size_t dense_decode_workspace_size(const msa_dense_decode_args& a) {
  const size_t slots = static_cast<size_t>(dense_slots(a.max_pages));
  const size_t rows = static_cast<size_t>(a.B) * a.Hq;
  return rows * slots * (static_cast<size_t>(kD) + 1) * 4 + static_cast<size_t>(a.B) * a.Hkv * 4 + 256;
}

msa_status launch_dense_decode(const msa_dense_decode_args& a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  DeviceInfo dev;
  if (msa_status st = current_device(&dev); st != MSA_OK) return st;
  const size_t need = dense_decode_workspace_size(a);
  if (ws == nullptr || ws_bytes < need) {
    char buf[160];
    std::snprintf(buf, sizeof(buf), "dense decode: workspace %zu bytes, need %zu", ws_bytes, need);
    return fail(MSA_ERR_WORKSPACE, buf);
  }
  CUtensorMap kmap, vmap, qmap;
  const uint64_t kv_dims[4] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(a.Bk), static_cast<uint64_t>(a.Hkv),
                               static_cast<uint64_t>(a.num_pages)};
  const uint64_t kv_strides[3] = {static_cast<uint64_t>(a.kv_stride[2]) * 2, static_cast<uint64_t>(a.kv_stride[1]) * 2,
                                  static_cast<uint64_t>(a.kv_stride[0]) * 2};
  const uint32_t kv_box[4] = {64, 128, 1, 1};
  if (msa_status st = encode_tiled_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.K_pool, kv_dims, kv_strides,
                                       kv_box, CU_TENSOR_MAP_SWIZZLE_128B, "K page pool");
      st != MSA_OK)
    return st;
  if (msa_status st = encode_tiled_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.V_pool, kv_dims, kv_strides,
                                       kv_box, CU_TENSOR_MAP_SWIZZLE_128B, "V page pool");
      st != MSA_OK)
    return st;
  const uint64_t q_dims[3] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(a.Hq), static_cast<uint64_t>(a.B)};
  const uint64_t q_strides[2] = {static_cast<uint64_t>(a.Q_stride[1]) * 2, static_cast<uint64_t>(a.Q_stride[0]) * 2};
  const uint32_t q_box[3] = {64, 16, 1};
  if (msa_status st = encode_tiled_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.Q, q_dims, q_strides, q_box,
                                       CU_TENSOR_MAP_SWIZZLE_128B, "Q");
      st != MSA_OK)
    return st;

  const int grid = std::min(dev.num_sms, kDenseMaxGrid);
  Params p;
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = a.Hq / a.Hkv;
  const float scale = a.softmax_scale > 0.f ? a.softmax_scale : 1.0f / sqrtf(static_cast<float>(a.D));
  p.scale_log2 = scale * kLog2e;
  p.num_pages = a.num_pages; p.max_pages = a.max_pages;
  p.seq_pt = a.seq_pt; p.seq_len = a.seq_len;
  p.slots = dense_slots(a.max_pages);
  float* o_part = static_cast<float*>(ws);
  const size_t parts = static_cast<size_t>(a.B) * a.Hq * p.slots;
  p.o_part = o_part;
  p.lse_part = o_part + parts * kD;
  p.counter = reinterpret_cast<int32_t*>(p.lse_part + parts);
  p.O = static_cast<__nv_bfloat16*>(a.O);
  p.LSE = a.LSE;
  p.dev_err = a.dev_err;

  const size_t smem = 1024 + static_cast<size_t>(kStages) * kStageBytes + kSlots * kPTile;
  if (smem > dev.max_smem_optin) return fail(MSA_ERR_UNSUPPORTED, "dense decode: not enough shared memory");
  cudaError_t e = cudaFuncSetAttribute(dense_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(dense_decode)");
  if (!a.scratch_zeroed) {
    e = cudaMemsetAsync(p.counter, 0, static_cast<size_t>(a.B) * a.Hkv * sizeof(int32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(dense decode row counters)");
  }
  dense_decode_kernel<<<grid, kThreads, smem, stream>>>(kmap, vmap, qmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "dense_decode_kernel launch");
  return MSA_OK;
}

}  // namespace msa
