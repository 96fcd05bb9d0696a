// attn_decode.cu -- a5 + a6: sparse attention of one decode step over the
// selected pages, the KV-group dimension flattened into the batch, with the
// log-sum-exp merge fused in.
//
// Row r = b * Hkv + g of the page table built from the selected blocks lists
// n[r] physical pages; the G query heads of group g attend to each page as an
// independent split of the softmax ("MiniMax M3 preparado para inferencia en
// produccion", paragraph "MSA con paged attention").  For unit (r, s):
//     z[h][t] = scale * Q[b, g*G + h] . K_page[t]      (t < valid tokens)
//     m_h = max_t z,  l_h = sum_t e^{z - m_h},  O_h = sum_t e^{z - m_h} V_t / l_h
//     O_part[(r*G + h), s] = O_h,   LSE_part[(r*G + h), s] = m_h + ln l_h
// and the CTA that finishes the last split of a row merges the row's partials
// (LSE = ln sum_s e^{LSE_s}, O = sum_s e^{LSE_s - LSE} O_s; paragraph
// "KV-Block-Major" of the same post) while they are still in L2.
//
// tcgen05 mapping (one TMEM slot of 32 columns per unit, two slots):
//   MMA1  S^T[t][h] = K[t][:] . Q[h][:]    M = 128 keys, N = 16 (heads, padded),
//                                          K = D = 128 (8 MMAs, both K-major)
//   softmax: one thread per key (TMEM lane), cross-warp max / sum per head,
//            P^T[h][t] (bf16) written into a K-major B tile
//   MMA2  O^T[d][h] = V^T[d][:] . P^T[:][h] M = 128 (d), N = 16, K = 128 keys;
//                                          V is the MN-major A operand
//   epilogue: one thread per d, coalesced fp32 partial rows.
// Warp 0 streams K, V (64 KiB) and the row's 16 Q rows by TMA into a 3-deep
// ring; warp 1 issues each unit's S and O MMAs as soon as their inputs are ready
// (polling both); warps 2-5 and 6-9 are two softmax/epilogue warpgroups
// taking alternate units, each with its own TMEM slot, and merge the rows
// they complete.
// Each CTA first copies its units' page ids and valid lengths into shared
// memory, so no role waits on a global load per unit.
#include "msa_internal.h"
#include "msa_ptx.cuh"

namespace msa {
namespace {

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
constexpr int kMaxUnits = 512;          // (row, page) units per CTA, kept in shared memory

__device__ __forceinline__ float fast_exp2(float x) {   // hardware 2^x (ex2.approx), 2^-inf = 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Max of a float over the 32 lanes of the warp (exact).
__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

struct Params {
  int B, Hq, Hkv, G, k;
  float scale_log2;
  int64_t num_pages;
  const int32_t* pt;
  const int32_t* n;
  const int32_t* last_len;
  float* o_part;
  float* lse_part;
  int32_t* counter;                     // [B*Hkv] splits finished per row, zero on entry
  __nv_bfloat16* O;                     // [B, Hq, D]
  float* LSE;                           // [B, Hq] or null
  int32_t* dev_err;
};

__global__ void __launch_bounds__(kThreads, 1)
attn_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
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
  __shared__ __align__(16) float s_max[2][4][kMaxG];   // per warpgroup and warp: per-head key maxima
  __shared__ __align__(16) float s_sum[2][4][kMaxG];   // and sums
  __shared__ int s_upage[kMaxUnits];    // physical page of each unit of this CTA
  __shared__ int s_uvalid[kMaxUnits];   // valid tokens of the page; 0 = no such split
  __shared__ int s_un[kMaxUnits];       // selected pages of the unit's row
  __shared__ int s_last[2], s_fail[2];
  __shared__ short s_live[kMaxUnits];         // offsets of the live units of this CTA, in order
  __shared__ int s_nlive;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t units = static_cast<int64_t>(p.B) * p.Hkv * p.k;
  const int64_t per_cta = (units + gridDim.x - 1) / gridDim.x;
  const int64_t lo = min(units, static_cast<int64_t>(blockIdx.x) * per_cta);
  const int64_t hi = min(units, lo + per_cta);

  // this CTA's units: page id, valid length and row size, read once
  for (int64_t u = lo + tid; u < hi; u += kThreads) {
    const int r = static_cast<int>(u / p.k), s = static_cast<int>(u % p.k);
    // the three loads are independent: one round trip to L2
    const int n_raw = p.n[r], page = p.pt[u], ll = p.last_len[r];
    const int nr = min(max(n_raw, 0), p.k);
    const bool live = s < nr;
    s_upage[u - lo] = live ? page : -1;
    s_uvalid[u - lo] = live ? (s == nr - 1 ? min(max(ll, 1), kBk) : kBk) : 0;
    s_un[u - lo] = nr;
    if (nr == 0 && s == 0) {   // a row with nothing selected: O = 0, LSE = -inf
      for (int h = 0; h < p.G; ++h) {
        const int64_t row = static_cast<int64_t>(r) * p.G + h;
        for (int d = 0; d < kD; d += 8) *reinterpret_cast<uint4*>(p.O + row * kD + d) = make_uint4(0, 0, 0, 0);
        if (p.LSE != nullptr) p.LSE[row] = -INFINITY;
      }
    }
  }
  __syncthreads();
  if (warp == 0) {   // compact the live units, in order
    int c = 0;
    const int cnt = static_cast<int>(hi - lo);
    for (int base = 0; base < cnt; base += 32) {
      const bool live = base + lane < cnt && s_uvalid[base + lane] > 0;
      const uint32_t m = __ballot_sync(0xffffffffu, live);
      if (live) s_live[c + __popc(m & ((1u << lane) - 1u))] = static_cast<short>(base + lane);
      c += __popc(m);
    }
    if (lane == 0) s_nlive = c;
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
    // ===================== TMA producer =====================
    if (lane == 0) {
      const int nlive = s_nlive;
      int n = 0;
      for (; n < nlive; ++n) {
        const int64_t u = lo + s_live[n];
        const int r = static_cast<int>(u / p.k);
        const int st = n % kStages;
        if (!mbar_wait(&bar_empty[st], ((n / kStages) & 1) ^ 1, abort_flag, p.dev_err)) break;
        const int64_t page = s_upage[u - lo];
        const int b = r / p.Hkv, g = r % p.Hkv;
        uint8_t* sb = s_stage + st * kStageBytes;
        if (page < 0 || page >= p.num_pages) {
          mbar_arrive(&bar_full[st]);
        } else {
          const int pg = static_cast<int>(page);
          mbar_arrive_expect_tx(&bar_full[st], kStageBytes);
          tma_load_4d(sb + 0 * kHalf, &kmap, &bar_full[st], 0, 0, g, pg);
          tma_load_4d(sb + 1 * kHalf, &kmap, &bar_full[st], 64, 0, g, pg);
          tma_load_4d(sb + 2 * kHalf, &vmap, &bar_full[st], 0, 0, g, pg);
          tma_load_4d(sb + 3 * kHalf, &vmap, &bar_full[st], 64, 0, g, pg);
          tma_load_3d(sb + 4 * kHalf, &qmap, &bar_full[st], 0, g * p.G, b);
          tma_load_3d(sb + 4 * kHalf + kQHalf, &qmap, &bar_full[st], 64, g * p.G, b);
        }
      }
      if (*abort_flag) {
        for (int i = max(0, n - kStages); i < n; ++i) {
          uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(&bar_full[i % kStages], (i / kStages) & 1) &&
                 global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ===================== tcgen05 issuer =====================
    // S of unit n (keys x heads) needs its stage loaded and its TMEM slot
    // (n mod 2) free; O of unit n needs P(n).  Both are polled and each MMA
    // group is issued as soon as its inputs are ready, so O(n) never waits
    // behind the load of unit n+1.
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 16, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, 16, true, false);
      const int nlive = s_nlive;
      int ns = 0, no = 0;
      uint32_t spins = 0;
      uint64_t idle_since = 0;
      while (no < nlive) {
        bool progress = false;
        if (ns < nlive) {
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
      uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&bar_drain, 0) && global_timer_ns() - t0 < MSA_WAIT_LIMIT_NS) {
      }
    }
    __syncwarp();
  } else {
    // ===================== softmax + epilogue: two warpgroups =====================
    // Warpgroup wg (warps 2-5 or 6-9) takes the units n = wg (mod 2), i.e. TMEM
    // slot wg, so two softmax chains run at once.
    const int wg = (warp - 2) >> 2;
    const int bar_id = 1 + wg;
    const int q = warp & 3;
    const int t = q * 32 + lane;                 // key index (MMA1) / d index (MMA2)
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const int G = p.G;
    const int nlive = s_nlive;
    int cur_r = -1, cur_nr = 0, seg_cnt = 0;
    // splits of row cur_r finished by this warpgroup are published in one step;
    // the warpgroup whose step completes the row merges the row's partials
    auto flush = [&]() {
      if (cur_r < 0) return;
      __threadfence();
      named_bar_sync(bar_id, 128);
      if (t == 0) s_last[wg] = atomicAdd(&p.counter[cur_r], seg_cnt) + seg_cnt == cur_nr;
      named_bar_sync(bar_id, 128);
      if (!s_last[wg]) return;
      __threadfence();
      const int r = cur_r, nr = cur_nr;
      // warp q merges heads q and q+4 (G <= 8); lane l owns d = 4l .. 4l+3.
      // A head's split LSEs (one per lane) and its first 16 partial rows
      // (float4 per lane) are loaded together; max, sum and weights by shuffles.
      const int lq = t >> 5, ll = t & 31;
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        const int h = lq + 4 * hi;
        if (h >= G) break;                     // warp-uniform
        const int64_t row = static_cast<int64_t>(r) * G + h;
        const float* lrow = p.lse_part + row * p.k;
        const float* orow = p.o_part + row * p.k * kD;
        const float l0 = ll < nr ? __ldcg(lrow + ll) : -INFINITY;
        const float l1 = ll + 32 < nr ? __ldcg(lrow + ll + 32) : -INFINITY;
        float4 v[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          v[x] = __ldcg(reinterpret_cast<const float4*>(orow + static_cast<int64_t>(min(x, nr - 1)) * kD) + ll);
        float m = fmaxf(l0, l1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float e0 = l0 == -INFINITY ? 0.f : __expf(l0 - m);
        const float e1 = l1 == -INFINITY ? 0.f : __expf(l1 - m);
        float sum = e0 + e1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = sum > 0.f ? 1.0f / sum : 0.f;
        const float w0 = e0 * inv, w1 = e1 * inv;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const float wgt = __shfl_sync(0xffffffffu, w0, x);   // 0 for x >= nr
          acc.x = fmaf(wgt, v[x].x, acc.x);
          acc.y = fmaf(wgt, v[x].y, acc.y);
          acc.z = fmaf(wgt, v[x].z, acc.z);
          acc.w = fmaf(wgt, v[x].w, acc.w);
        }
        for (int x = 16; x < nr; ++x) {        // k > 16
          const float wgt = __shfl_sync(0xffffffffu, x < 32 ? w0 : w1, x & 31);
          const float4 u = __ldcg(reinterpret_cast<const float4*>(orow + static_cast<int64_t>(x) * kD) + ll);
          acc.x = fmaf(wgt, u.x, acc.x);
          acc.y = fmaf(wgt, u.y, acc.y);
          acc.z = fmaf(wgt, u.z, acc.z);
          acc.w = fmaf(wgt, u.w, acc.w);
        }
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y), hi2 = __floats2bfloat162_rn(acc.z, acc.w);
        *reinterpret_cast<uint2*>(p.O + row * kD + 4 * ll) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo2), *reinterpret_cast<uint32_t*>(&hi2));
        if (ll == 0 && p.LSE != nullptr) p.LSE[row] = sum > 0.f ? m + __logf(sum) : -INFINITY;
      }
      if (t == 0) p.counter[r] = 0;           // ready for the next call
    };
    for (int n = wg; n < nlive; n += 2) {
      const int64_t u = lo + s_live[n];
      const int valid = s_uvalid[u - lo];
      const int r = static_cast<int>(u / p.k), s = static_cast<int>(u % p.k);
      if (r != cur_r) {
        flush();
        cur_r = r;
        cur_nr = s_un[u - lo];
        seg_cnt = 0;
      }
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
      // per-head maximum over this warp's 32 keys (exact), then over the 4 warps
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
      {
        const float4* m4 = reinterpret_cast<const float4*>(&s_max[wg][0][0]);
        const float4 a0 = m4[0], a1 = m4[1], b0 = m4[2], b1 = m4[3], c0 = m4[4], c1 = m4[5], d0 = m4[6], d1 = m4[7];
        mx[0] = fmaxf(fmaxf(a0.x, b0.x), fmaxf(c0.x, d0.x)); mx[1] = fmaxf(fmaxf(a0.y, b0.y), fmaxf(c0.y, d0.y));
        mx[2] = fmaxf(fmaxf(a0.z, b0.z), fmaxf(c0.z, d0.z)); mx[3] = fmaxf(fmaxf(a0.w, b0.w), fmaxf(c0.w, d0.w));
        mx[4] = fmaxf(fmaxf(a1.x, b1.x), fmaxf(c1.x, d1.x)); mx[5] = fmaxf(fmaxf(a1.y, b1.y), fmaxf(c1.y, d1.y));
        mx[6] = fmaxf(fmaxf(a1.z, b1.z), fmaxf(c1.z, d1.z)); mx[7] = fmaxf(fmaxf(a1.w, b1.w), fmaxf(c1.w, d1.w));
      }
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) z[h] = (t < valid) ? fast_exp2(z[h] - mx[h]) : 0.f;
      // per-head sums over the warp's 32 keys by a transposed butterfly: after
      // the xor-16/8/4 steps each lane carries one head (lane >> 2), then xor 2, 1
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
      // P^T[h][t] into the K-major B tile of this slot
      uint8_t* pt_tile = s_p + slot * kPTile + (t >> 6) * kQHalf;
      const uint32_t tc = static_cast<uint32_t>(t & 63);
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) {
        if (h < G) {
          __nv_bfloat16 b = __float2bfloat16_rn(z[h]);
          *reinterpret_cast<__nv_bfloat16*>(pt_tile + sw128_offset(h, tc >> 3) + (tc & 7) * 2) = b;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pready[slot]);
      named_bar_sync(bar_id, 128);
      float l[kMaxG], inv_l[kMaxG];
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) {
        l[h] = (s_sum[wg][0][h] + s_sum[wg][1][h]) + (s_sum[wg][2][h] + s_sum[wg][3][h]);
        inv_l[h] = __frcp_rn(l[h]);
      }
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
      const int64_t page = s_upage[u - lo];
      const bool bad = page < 0 || page >= p.num_pages;
      if (bad && t == 0) report(p.dev_err, MSA_DEVERR_BAD_PAGE);
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) {
        if (h < G) {
          const int64_t row = (static_cast<int64_t>(r) * G + h) * p.k + s;
          p.o_part[row * kD + t] = bad ? 0.f : __uint_as_float(ov[h]) * inv_l[h];
          if (t == h) p.lse_part[row] = bad ? -INFINITY : (mx[h] + log2f(l[h])) * kLn2;
        }
      }
      ++seg_cnt;
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

}  // namespace

msa_status launch_attn_decode(const msa_decode_args& a, float* o_part, float* lse_part, int32_t* counter,
                              cudaStream_t stream) {
  DeviceInfo dev;
  if (msa_status st = current_device(&dev); st != MSA_OK) return st;
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

  Params p;
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = a.Hq / a.Hkv; p.k = a.k;
  const float scale = a.softmax_scale > 0.f ? a.softmax_scale : 1.0f / sqrtf(static_cast<float>(a.D));
  p.scale_log2 = scale * kLog2e;
  p.num_pages = a.num_pages; p.pt = a.pt; p.n = a.n; p.last_len = a.last_len;
  p.o_part = o_part; p.lse_part = lse_part; p.dev_err = a.dev_err;
  p.counter = counter;
  p.O = static_cast<__nv_bfloat16*>(a.O);
  p.LSE = a.LSE;

  const size_t smem = 1024 + static_cast<size_t>(kStages) * kStageBytes + kSlots * kPTile;
  if (smem > dev.max_smem_optin) return fail(MSA_ERR_UNSUPPORTED, "decode attention: not enough shared memory");
  cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attn_decode)");
  const int64_t units = static_cast<int64_t>(a.B) * a.Hkv * a.k;
  const int64_t grid64 = std::max<int64_t>(std::min<int64_t>(dev.num_sms, units), (units + kMaxUnits - 1) / kMaxUnits);
  const int grid = static_cast<int>(std::max<int64_t>(grid64, 1));
  if (!a.scratch_zeroed) {   // otherwise zero by contract (every error-free call leaves them zero)
    e = cudaMemsetAsync(counter, 0, static_cast<size_t>(a.B) * a.Hkv * sizeof(int32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(decode row counters)");
  }
  attn_decode_kernel<<<grid, kThreads, smem, stream>>>(kmap, vmap, qmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode_kernel launch");
  return MSA_OK;
}

}  // namespace msa
