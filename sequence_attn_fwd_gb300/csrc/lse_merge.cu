// Log-sum-exp merge of per-chunk attention partials, for sm_103a.
//
// Per query row (the output_acc / logsumexp_acc accumulation of page
// "Ulysses与Ring-Attention序列并行技术详解", Ring-Attention part, taken per row
// with the empty accumulator at lse = -inf):
//   M = max_i lse_i,  w_i = exp(lse_i - M),  lse = M + ln(sum_i w_i),
//   O = sum_i w_i O_i / sum_i w_i;  no finite lse_i  ->  O = 0, lse = -inf.
//
// Memory-bound. Main kernel (P <= 32): a warp owns 32 consecutive rows. Each
// lane reads the P lse values of one row (for each part, the warp's 32 reads
// are one coalesced 128-byte run), forms that row's normalised weights in
// registers and writes its lse. The warp then sweeps its 32 rows: D/4 lanes
// per row, one float4 column slice each, weights broadcast by shuffle, the P
// partial reads of a row issued together (a partial with lse_i = -inf is
// never read). Partial reads use the streaming cache hint (read once).
// Grid-stride over row groups, grid sized to the SM count. A row-at-a-time
// kernel covers P > 32.
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

// Up to 8 parts a row carries few loads, so more rows are kept in flight:
// four per warp step and three CTAs per SM (measured best on GB300 for 8
// parts; two and two for 16).
template <int kPMax>
constexpr int rows32_min_blocks() { return kPMax <= 8 ? 3 : 2; }

template <int D, bool kBf16Out, int kPMax>
__global__ void __launch_bounds__(kMergeThreads, rows32_min_blocks<kPMax>())
    lse_merge_rows32_kernel(const float *o_parts, const float *lse_parts, int P, long long nrows,
                            void *o_out, float *lse_out) {
  constexpr int kSlots = D / 4;            // float4 slices per row
  constexpr int kRowsPerStep = 32 / kSlots;  // rows a warp covers per step (1 or 2)
  const int lane = threadIdx.x & 31;
  const int sub = lane % kSlots;
  const int rsub = lane / kSlots;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * kMergeThreads) >> 5;

  for (long long base = warp_id * 32; base < nrows; base += n_warps * 32) {
    // this lane's row: its lse values, maximum, normalised weights, merged lse
    const long long my_row = base + lane;
    const bool my_valid = my_row < nrows;
    float w[kPMax];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPMax; ++i) {
      w[i] = (i < P && my_valid) ? lse_parts[static_cast<long long>(i) * nrows + my_row] : -INFINITY;
      mx = fmaxf(mx, w[i]);
    }
    float wsum = 0.f;
#pragma unroll
    for (int i = 0; i < kPMax; ++i) {
      w[i] = (w[i] == -INFINITY) ? 0.f : expf(w[i] - mx);
      wsum += w[i];
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int i = 0; i < kPMax; ++i) w[i] *= inv;
    // all of this row's lse_parts are in registers before the (possibly aliased) write
    if (my_valid) lse_out[my_row] = (mx == -INFINITY) ? -INFINITY : mx + logf(wsum);

    // the 32 rows' outputs: D/4 lanes per row (several rows' loads in flight when P is small)
#pragma unroll(kPMax <= 8 ? 4 : (kPMax <= 16 ? 2 : 1))
    for (int r = 0; r < 32; r += kRowsPerStep) {
      const int rr = r + rsub;
      const long long row = base + rr;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < kPMax; ++i) {
        const float wi = __shfl_sync(0xffffffffu, w[i], rr);
        if (wi != 0.f && row < nrows) {
          const float4 x = __ldcs(reinterpret_cast<const float4 *>(
                                      o_parts + (static_cast<long long>(i) * nrows + row) * D) +
                                  sub);
          acc.x = fmaf(wi, x.x, acc.x);
          acc.y = fmaf(wi, x.y, acc.y);
          acc.z = fmaf(wi, x.z, acc.z);
          acc.w = fmaf(wi, x.w, acc.w);
        }
      }
      if (row < nrows) {
        if constexpr (kBf16Out) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
          __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
          uint2 v = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
          reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(o_out) + row * D)[sub] = v;
        } else {
          reinterpret_cast<float4 *>(static_cast<float *>(o_out) + row * D)[sub] = acc;
        }
      }
    }
  }
}

template <int D, bool kBf16Out, int kPMax>
cudaError_t launch_rows32(const float *o_parts, const float *lse_parts, int P, long long nrows,
                          void *o, float *lse, int sms, cudaStream_t stream) {
  constexpr int kRowsPerBlock = (kMergeThreads / 32) * 32;
  long long blocks = (nrows + kRowsPerBlock - 1) / kRowsPerBlock;
  const long long cap = static_cast<long long>(sms) * (2048 / kMergeThreads);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  lse_merge_rows32_kernel<D, kBf16Out, kPMax>
      <<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(o_parts, lse_parts, P, nrows, o, lse);
  return cudaGetLastError();
}

template <int D, bool kBf16Out>
cudaError_t launch_merge_typed(const float *o_parts, const float *lse_parts, int P, long long nrows,
                               void *o, float *lse, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (P <= 8) return launch_rows32<D, kBf16Out, 8>(o_parts, lse_parts, P, nrows, o, lse, sms, stream);
  if (P <= 16) return launch_rows32<D, kBf16Out, 16>(o_parts, lse_parts, P, nrows, o, lse, sms, stream);
  if (P <= 32) return launch_rows32<D, kBf16Out, 32>(o_parts, lse_parts, P, nrows, o, lse, sms, stream);
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
