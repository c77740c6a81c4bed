// Log-sum-exp merge of per-chunk attention partials, for sm_103a.
//
// Per query row (the output_acc / logsumexp_acc accumulation of page
// "Ulysses与Ring-Attention序列并行技术详解", Ring-Attention part, taken per row
// with the empty accumulator at lse = -inf):
//   M = max_i lse_i,  w_i = exp(lse_i - M),  lse = M + ln(sum_i w_i),
//   O = sum_i w_i O_i / sum_i w_i;  no finite lse_i  ->  O = 0, lse = -inf.
//
// Memory-bound. D/4 threads own one row, each a float4 column slice, so a row
// of every partial is one coalesced 128-bit-per-thread read. The row's
// lse_i are read once (thread k holds parts k, k + D/4, ...), reduced with
// shuffles, and the weights are broadcast by shuffle; a partial with zero
// weight (lse_i = -inf) is never read. Partial reads use the streaming cache
// hint (read once). Grid-stride over rows, grid sized to the SM count.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kernels.h"

namespace seqattn {
namespace {

constexpr int kMergeThreads = 256;

template <int D, bool kBf16Out>
__global__ void __launch_bounds__(kMergeThreads)
    lse_merge_kernel(const float *o_parts, const float *lse_parts,
                     int P, long long nrows, void *o_out, float *lse_out) {
  constexpr int kTpr = D / 4;          // threads per row
  constexpr int kRowsPerWarp = 32 / kTpr;
  const int lane = threadIdx.x & 31;
  const int sub = lane % kTpr;         // float4 slot within the row
  const int grp = lane / kTpr;         // row slot within the warp
  const unsigned gmask = (kTpr == 32) ? 0xffffffffu : (0xffffu << (16 * grp));
  const long long warp_id = (static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * kMergeThreads) >> 5;

  for (long long row = warp_id * kRowsPerWarp + grp; row < nrows; row += n_warps * kRowsPerWarp) {
    // 1. M = max_i lse_i over the row's partials
    float mx = -INFINITY;
    for (int i = sub; i < P; i += kTpr) mx = fmaxf(mx, lse_parts[static_cast<long long>(i) * nrows + row]);
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(gmask, mx, off, kTpr));

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (mx != -INFINITY) {
      for (int i0 = 0; i0 < P; i0 += kTpr) {
        // this thread's weight for part i0 + sub
        const int mine = i0 + sub;
        const float li = mine < P ? lse_parts[static_cast<long long>(mine) * nrows + row] : -INFINITY;
        const float wi = (li == -INFINITY) ? 0.f : expf(li - mx);
        wsum += wi;
        const int cnt = min(kTpr, P - i0);
#pragma unroll 8
        for (int k = 0; k < cnt; ++k) {
          const float w = __shfl_sync(gmask, wi, k, kTpr);
          if (w != 0.f) {
            const float4 x = __ldcs(reinterpret_cast<const float4 *>(
                                        o_parts + (static_cast<long long>(i0 + k) * nrows + row) * D) +
                                    sub);
            acc.x = fmaf(w, x.x, acc.x);
            acc.y = fmaf(w, x.y, acc.y);
            acc.z = fmaf(w, x.z, acc.z);
            acc.w = fmaf(w, x.w, acc.w);
          }
        }
      }
#pragma unroll
      for (int off = kTpr / 2; off > 0; off >>= 1) wsum += __shfl_xor_sync(gmask, wsum, off, kTpr);
      const float inv = 1.f / wsum;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
    }
    if constexpr (kBf16Out) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 v = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
      reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(o_out) + row * D)[sub] = v;
    } else {
      reinterpret_cast<float4 *>(static_cast<float *>(o_out) + row * D)[sub] = acc;
    }
    if (sub == 0) lse_out[row] = (mx == -INFINITY) ? -INFINITY : mx + logf(wsum);
  }
}

template <int D, bool kBf16Out>
cudaError_t launch_merge_typed(const float *o_parts, const float *lse_parts, int P, long long nrows,
                               void *o, float *lse, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  constexpr int kRowsPerBlock = (kMergeThreads / 32) * (32 / (D / 4));
  long long blocks = (nrows + kRowsPerBlock - 1) / kRowsPerBlock;
  const long long cap = static_cast<long long>(sms) * (2048 / kMergeThreads);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  lse_merge_kernel<D, kBf16Out><<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(
      o_parts, lse_parts, P, nrows, o, lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lse_merge(const float *o_parts, const float *lse_parts, int P, long long nrows,
                             int D, void *o, bool bf16_out, float *lse, cudaStream_t stream) {
  if (D == 128) return bf16_out ? launch_merge_typed<128, true>(o_parts, lse_parts, P, nrows, o, lse, stream)
                                : launch_merge_typed<128, false>(o_parts, lse_parts, P, nrows, o, lse, stream);
  return bf16_out ? launch_merge_typed<64, true>(o_parts, lse_parts, P, nrows, o, lse, stream)
                  : launch_merge_typed<64, false>(o_parts, lse_parts, P, nrows, o, lse, stream);
}

}  // namespace seqattn
