// lse_merge.cu -- a6: log-sum-exp merge of partial softmax results.
//
// The KV-block-major kernels compute partial outputs per block and recombine
// them with a final log-sum-exp based reduction ("MiniMax M3 preparado para
// inferencia en produccion", paragraph "KV-Block-Major"):
//     LSE = ln sum_p e^{LSE_p},   O = sum_p e^{LSE_p - LSE} O_p.
// One warp per output row; each lane owns float4 column groups.  Parts with
// LSE_p = -inf are empty and are neither weighted nor read.
#include "msa_internal.h"
#include "msa_ptx.cuh"

namespace msa {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// Partials are fp32 (public entry point, decode) or bf16 (prefill workspace).
template <typename TP>
__global__ void __launch_bounds__(kWarps * 32)
lse_merge_kernel(const TP* __restrict__ o_part, const float* __restrict__ lse_part, int64_t rows, int parts, int D,
                 __nv_bfloat16* __restrict__ O, float* __restrict__ LSE) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* lp = lse_part + row * parts;
  // two parts per lane cover parts <= 64
  const float l0 = lane < parts ? lp[lane] : -INFINITY;
  const float l1 = lane + 32 < parts ? lp[lane + 32] : -INFINITY;
  float m = fmaxf(l0, l1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __nv_bfloat16* orow = O + row * D;
  if (m == -INFINITY) {
    for (int c = lane * 4; c < D; c += 128) {
      *reinterpret_cast<uint2*>(orow + c) = make_uint2(0, 0);
    }
    if (lane == 0 && LSE != nullptr) LSE[row] = -INFINITY;
    return;
  }
  float sum = (l0 == -INFINITY ? 0.f : __expf(l0 - m)) + (l1 == -INFINITY ? 0.f : __expf(l1 - m));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float lse = m + __logf(sum);
  const float inv = 1.0f / sum;
  const TP* op = o_part + row * static_cast<int64_t>(parts) * D;
  for (int c = lane * 4; c < D; c += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int pi = 0; pi < parts; ++pi) {
      const float lpi = __shfl_sync(0xffffffffu, pi < 32 ? l0 : l1, pi & 31);
      if (lpi == -INFINITY) continue;
      const float wgt = __expf(lpi - m) * inv;
      const float4 v = load4(op + static_cast<int64_t>(pi) * D + c);
      acc.x = fmaf(wgt, v.x, acc.x);
      acc.y = fmaf(wgt, v.y, acc.y);
      acc.z = fmaf(wgt, v.z, acc.z);
      acc.w = fmaf(wgt, v.w, acc.w);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(orow + c) = packed;
  }
  if (lane == 0 && LSE != nullptr) LSE[row] = lse;
}

// bf16 partials, at most 16 parts, D = 128: one warp per row, every partial load
// of the row issued before any is used.
__global__ void __launch_bounds__(kWarps * 32)
lse_merge_bf16_k16_kernel(const __nv_bfloat16* __restrict__ o_part, const float* __restrict__ lse_part, int64_t rows,
                          int parts, __nv_bfloat16* __restrict__ O, float* __restrict__ LSE) {
  constexpr int D = 128;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float lv = lane < parts ? lse_part[row * parts + lane] : -INFINITY;
  const __nv_bfloat16* op = o_part + row * static_cast<int64_t>(parts) * D + lane * 4;
  uint2 raw[16];
#pragma unroll
  for (int pi = 0; pi < 16; ++pi) raw[pi] = pi < parts ? *reinterpret_cast<const uint2*>(op + pi * D) : make_uint2(0, 0);
  float m = lv;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __nv_bfloat16* orow = O + row * D + lane * 4;
  if (m == -INFINITY) {
    *reinterpret_cast<uint2*>(orow) = make_uint2(0, 0);
    if (lane == 0 && LSE != nullptr) LSE[row] = -INFINITY;
    return;
  }
  const float e = lv == -INFINITY ? 0.f : __expf(lv - m);
  float sum = e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float wgt = e / sum;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int pi = 0; pi < 16; ++pi) {
    const float wp = __shfl_sync(0xffffffffu, wgt, pi);
    if (pi < parts && wp != 0.f) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[pi].x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[pi].y));
      acc.x = fmaf(wp, a.x, acc.x);
      acc.y = fmaf(wp, a.y, acc.y);
      acc.z = fmaf(wp, b.x, acc.z);
      acc.w = fmaf(wp, b.y, acc.w);
    }
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  *reinterpret_cast<uint2*>(orow) = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  if (lane == 0 && LSE != nullptr) LSE[row] = m + __logf(sum);
}

}  // namespace

msa_status launch_lse_merge(const float* o_part, const float* lse_part, int64_t rows, int parts, int D, void* O,
                            float* LSE, int32_t* dev_err, cudaStream_t stream) {
  (void)dev_err;
  if (rows == 0) return MSA_OK;
  const int64_t grid = (rows + kWarps - 1) / kWarps;
  lse_merge_kernel<float><<<static_cast<unsigned>(grid), kWarps * 32, 0, stream>>>(
      o_part, lse_part, rows, parts, D, static_cast<__nv_bfloat16*>(O), LSE);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "lse_merge_kernel launch");
  return MSA_OK;
}

msa_status launch_lse_merge_bf16(const __nv_bfloat16* o_part, const float* lse_part, int64_t rows, int parts, int D,
                                 __nv_bfloat16* O, float* LSE, cudaStream_t stream) {
  if (rows == 0) return MSA_OK;
  const int64_t grid = (rows + kWarps - 1) / kWarps;
  if (parts <= 16 && D == 128)
    lse_merge_bf16_k16_kernel<<<static_cast<unsigned>(grid), kWarps * 32, 0, stream>>>(o_part, lse_part, rows, parts,
                                                                                      O, LSE);
  else
    lse_merge_kernel<__nv_bfloat16><<<static_cast<unsigned>(grid), kWarps * 32, 0, stream>>>(o_part, lse_part, rows,
                                                                                            parts, D, O, LSE);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "lse_merge_kernel<bf16> launch");
  return MSA_OK;
}

}  // namespace msa
