// Backward of blockwise attention for sm_103a (head dim 128, bf16): the
// gradients dQ, dK, dV for an output gradient dO, recomputing the scores
// tile by tile from Q, K and the forward's lse instead of storing the [S, S]
// probabilities (the backward the page "ms-swift集成FlashAttention 2/3，长文本
// 训练更高效" describes FlashAttention as recomputing block by block). With
// P = exp(scale * Q K^T - lse) and delta_i = <dO_i, O_i>:
//   dV = P^T dO,   dS = P * (dO V^T - delta),   dK = scale dS^T Q,   dQ = scale dS K.
// Included by attn_kernel.cu after the definition of the device error word.
//
// Three kernels:
//   delta       delta_i = <dO_i, O_i> per query row (memory-bound, a warp per row).
//   dK / dV     one CTA per 128-key tile of a (batch, KV head): K and V stay in
//               shared memory while the query tiles of every query head of the
//               GQA group stream through; S^T = K Q^T and dP^T = V dO^T land in
//               TMEM, two warpgroups (64 query columns each) form P^T and dS^T
//               as bf16 in TMEM, and dV += P^T dO, dK += dS^T Q accumulate in
//               TMEM (TS form, Q and dO as N-contiguous operands).
//   dQ          one CTA per 128-row query tile: Q and dO stay, the visible key
//               tiles stream through; S = Q K^T, dP = dO V^T, dS in TMEM, and
//               dQ += dS K.
// Both matrix kernels: warp 9 TMA producer, warp 8 MMA issuer (one thread),
// warps 0-7 the element-wise pass. Every wait is bounded.
#pragma once
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace seqattn {
namespace bwd {

constexpr int kD = 128;
constexpr int kRows = 128;                      // tile rows (keys or queries)
constexpr int kTileBytes = kRows * kD * 2;      // 32 KB: two 128-byte column blocks
constexpr int kColBlock = kRows * 128;          // 16 KB
constexpr int kStages = 4;                      // ring slots of 32 KB
constexpr int kThreads = 320;
constexpr int kMmaWarp = 8, kTmaWarp = 9;
constexpr float kLog2e = 1.4426950408889634f;

// barriers: stay_full, full[S], empty[S], st_full, pt_full, acc_done
constexpr int kNumBarriers = 1 + 2 * kStages + 3;
constexpr int kSmemBytes = 1024 + 2 * kTileBytes + kStages * kTileBytes + 2 * 2 * kRows * 4 +
                           8 * kNumBarriers + 16;

// Loads a 128 x 128 bf16 tile (two 64-column boxes) into `dst`.
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap *map, uint32_t bar, int row,
                                          int head) {
  tma_load_3d(dst, map, bar, 0, row, head);
  tma_load_3d(dst + kColBlock, map, bar, 64, row, head);
}

// S (or S^T) = A B^T over D = 128: A, B K-major tiles in shared memory.
__device__ __forceinline__ void mma_rows_dot(uint32_t d_tmem, uint32_t a, uint32_t b) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false);
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t off = (kk / 4) * kColBlock + (kk % 4) * 32;
    mma_ss(d_tmem, sw128_desc(a + off, 16, 1024), sw128_desc(b + off, 16, 1024), idesc,
           kk > 0 ? 1u : 0u);
  }
}

// acc (+)= A_tmem B: A = 128 x 128 bf16 in TMEM (contraction over its
// columns), B = 128 x 128 tile in shared memory whose rows are the contraction
// index (N-contiguous operand). A's 128 contraction elements are packed as
// bf16 pairs in two runs of 32 TMEM columns, at a_tmem and a_tmem + 64 (each
// element-wise warpgroup packs its 64 columns over the first half of its own).
__device__ __forceinline__ void mma_acc_tmem(uint32_t acc, uint32_t a_tmem, uint32_t b, bool first) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, kD, true);
#pragma unroll
  for (int kk = 0; kk < kRows / 16; ++kk)
    mma_ts(acc, a_tmem + (kk / 4) * 64 + (kk % 4) * 8, sw128_desc(b + kk * 2048, kColBlock, 1024),
           idesc, (first && kk == 0) ? 0u : 1u);
}

// One thread's row of a 128 x 128 fp32 TMEM accumulator, times `mul`, as bf16
// into global memory (one 256-byte row). Every lane of the warp takes part in
// the TMEM loads (they are warp-wide); only lanes with `valid` store.
__device__ __forceinline__ void store_acc_row(uint32_t taddr, float mul, __nv_bfloat16 *dst, bool valid) {
#pragma unroll 1
  for (int cb = 0; cb < kD / 32; ++cb) {
    uint32_t r[32];
    tmem_ld32(taddr + 32 * cb, r);
    tmem_ld_wait(r);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * i]) * mul,
                                               __uint_as_float(r[2 * i + 1]) * mul);
      pk[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    if (valid) {
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * cb);
#pragma unroll
      for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// ---------------------------------------------------------------- delta
__global__ void delta_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                             float *__restrict__ delta, long long nrows) {
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (long long r = warp; r < nrows; r += nwarps) {
    const uint2 a = reinterpret_cast<const uint2 *>(o + r * kD)[lane];
    const uint2 b = reinterpret_cast<const uint2 *>(dout + r * kD)[lane];
    const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 fa = __bfloat1622float2(pa[i]), fb = __bfloat1622float2(pb[i]);
      s = fmaf(fa.x, fb.x, s);
      s = fmaf(fa.y, fb.y, s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) delta[r] = s;
  }
}

// ---------------------------------------------------------------- dK / dV and dQ
// kDq = false: the dK / dV kernel (grid: key tiles x B*Hkv); kDq = true: the
// dQ kernel (grid: query tiles x B*Hq). "Stay" tiles are loaded once (K, V or
// Q, dO); "stream" tiles pass through the ring (Q_i, dO_i or K_j, V_j).
template <bool kDq>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sStay = smem;                       // [2][tile]: K, V (dK/dV) or Q, dO (dQ)
  uint8_t *sRing = smem + 2 * kTileBytes;      // [kStages][tile]
  float *sVec = reinterpret_cast<float *>(sRing + kStages * kTileBytes);  // [2 buffers][lse2 | delta][128]
  uint64_t *bars = reinterpret_cast<uint64_t *>(sVec + 2 * 2 * kRows);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBarriers);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const uint32_t bar0 = smem_addr(bars);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  const int kBarStay = 0, kBarFull = 1, kBarEmpty = 1 + kStages, kBarSt = 1 + 2 * kStages,
            kBarPt = kBarSt + 1, kBarAcc = kBarPt + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int *err = &g_device_error;
  const int S = p.S, group = p.Hq / p.Hkv;
  const int n_tiles = (S + kRows - 1) / kRows;
  const int tile = blockIdx.x;  // key tile (dK/dV) or query tile (dQ)
  const int head = blockIdx.y;  // b*Hkv + hkv (dK/dV) or b*Hq + hq (dQ)
  const int b = kDq ? head / p.Hq : head / p.Hkv;
  // dK/dV: iterations over (query head of the group, query tile >= this key
  // tile when causal); dQ: over key tiles <= this query tile when causal
  const int first_stream = (!kDq && p.causal) ? tile : 0;
  const int n_stream_tiles = kDq ? (p.causal ? tile + 1 : n_tiles) : n_tiles - first_stream;
  const int n_iter = kDq ? n_stream_tiles : group * n_stream_tiles;
  auto stream_of = [&](int it, int &row, int &q_head) {  // the streamed tile of iteration it
    if (kDq) {
      row = it * kRows;
      q_head = head;
    } else {
      row = (first_stream + it % n_stream_tiles) * kRows;
      q_head = b * p.Hq + (head % p.Hkv) * group + it / n_stream_tiles;
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarStay), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    mbar_init(bar(kBarSt), 1);
    mbar_init(bar(kBarPt), 8);  // one arrival per element-wise warp
    mbar_init(bar(kBarAcc), 1);
    *abort_flag = *reinterpret_cast<volatile int *>(err) != kErrNone;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;
  // TMEM: S or S^T [0,128) (then P / dS as bf16 pairs in columns [0,32) and [64,96)),
  // dP or dP^T [128,256), accumulators [256,384) and (dK/dV) [384,512)
  const uint32_t tS = tmem, tDP = tmem + 128, tAcc0 = tmem + 256, tAcc1 = tmem + 384;

  if (warp == kTmaWarp) {
    if (lane == 0 && !skip && n_iter > 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_do);
      mbar_arrive_expect_tx(bar(kBarStay), 2 * kTileBytes);
      if (kDq) {
        load_tile(smem_addr(sStay), &tm_q, bar(kBarStay), tile * kRows, head);
        load_tile(smem_addr(sStay + kTileBytes), &tm_do, bar(kBarStay), tile * kRows, head);
      } else {
        load_tile(smem_addr(sStay), &tm_k, bar(kBarStay), tile * kRows, head);
        load_tile(smem_addr(sStay + kTileBytes), &tm_v, bar(kBarStay), tile * kRows, head);
      }
      const int kv_head = kDq ? b * p.Hkv + (head % p.Hq) / group : head;
      int c = 0;
      bool ok = true;
      for (int it = 0; it < n_iter && ok; ++it) {
        int row, q_head;
        stream_of(it, row, q_head);
        for (int which = 0; which < 2; ++which, ++c) {  // Q_i then dO_i, or K_j then V_j
          const int slot = c % kStages;
          if (c >= kStages && !mbar_wait(bar(kBarEmpty + slot), ((c / kStages) - 1) & 1, abort_flag, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarFull + slot), kTileBytes);
          const CUtensorMap *map = kDq ? (which ? &tm_v : &tm_k) : (which ? &tm_do : &tm_q);
          load_tile(smem_addr(sRing + slot * kTileBytes), map, bar(kBarFull + slot), row,
                    kDq ? kv_head : q_head);
        }
      }
      mbar_drain(bar(kBarStay), 0, err);
      for (int i = max(0, c - kStages); i < c; ++i)
        mbar_drain(bar(kBarFull + i % kStages), (i / kStages) & 1, err);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0 && !skip && n_iter > 0) {
      const uint32_t stay0 = smem_addr(sStay), stay1 = stay0 + kTileBytes;
      const uint32_t ring = smem_addr(sRing);
      bool ok = mbar_wait(bar(kBarStay), 0, abort_flag, err);
      for (int it = 0; ok && it < n_iter; ++it) {
        const int c0 = 2 * it, c1 = 2 * it + 1;
        const int s0 = c0 % kStages, s1 = c1 % kStages;
        if (!mbar_wait(bar(kBarFull + s0), (c0 / kStages) & 1, abort_flag, err) ||
            !mbar_wait(bar(kBarFull + s1), (c1 / kStages) & 1, abort_flag, err))
          break;
        tc_fence_after();
        const uint32_t r0 = ring + s0 * kTileBytes, r1 = ring + s1 * kTileBytes;
        if (kDq) {
          mma_rows_dot(tS, stay0, r0);   // S = Q K_j^T
          mma_rows_dot(tDP, stay1, r1);  // dP = dO V_j^T
        } else {
          mma_rows_dot(tS, stay0, r0);   // S^T = K Q_i^T
          mma_rows_dot(tDP, stay1, r1);  // dP^T = V dO_i^T
        }
        mma_commit(bar(kBarSt));
        if (!mbar_wait(bar(kBarPt), it & 1, abort_flag, err)) break;
        tc_fence_after();
        if (kDq) {
          mma_acc_tmem(tAcc0, tS, r0, it == 0);   // dQ += dS K_j
        } else {
          mma_acc_tmem(tAcc0, tS, r1, it == 0);   // dV += P^T dO_i
          mma_acc_tmem(tAcc1, tDP, r0, it == 0);  // dK += dS^T Q_i
        }
        mma_commit(bar(kBarEmpty + s0));
        mma_commit(bar(kBarEmpty + s1));
      }
      mma_commit(bar(kBarAcc));
      mbar_drain(bar(kBarAcc), 0, err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ element-wise pass
    const int g = warp >> 2;                       // column half of this warpgroup
    const int row_in_tile = (warp & 3) * 32 + lane;  // TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int my_row = tile * kRows + row_in_tile;  // key (dK/dV) or query (dQ) of this thread
    const float c2 = p.scale * kLog2e;
    // dQ: this query row's lse (log2 units) and delta, once
    float row_lse2 = INFINITY, row_delta = 0.f;
    if (kDq && my_row < S) {
      row_lse2 = p.lse[static_cast<size_t>(head) * S + my_row] * kLog2e;
      row_delta = p.delta[static_cast<size_t>(head) * S + my_row];
    }
    bool ok = !skip;
    for (int it = 0; it < n_iter; ++it) {
      int srow, q_head;
      stream_of(it, srow, q_head);
      float *vec = sVec + (it & 1) * 2 * kRows;  // [lse2 | delta] of the streamed query tile
      if (!kDq) {
        const int t = threadIdx.x & 127;
        if (t < 64) {
          const int col = 64 * g + t, i = srow + col;
          vec[col] = (i < S) ? p.lse[static_cast<size_t>(q_head) * S + i] * kLog2e : INFINITY;
          vec[kRows + col] = (i < S) ? p.delta[static_cast<size_t>(q_head) * S + i] : 0.f;
        }
      }
      bool got = ok && mbar_wait(bar(kBarSt), it & 1, abort_flag, err);
      got = named_bar_and(1 + g, 128, __all_sync(0xffffffffu, got));  // also publishes vec
      if (!got) break;
      tc_fence_after();
      uint32_t pk_a[32], pk_b[32];  // bf16 pairs: P^T and dS^T (dK/dV) or dS (dQ)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int col0 = 64 * g + 32 * h;
        uint32_t sr[32], dr[32];
        tmem_ld32(tS + lane_off + col0, sr);
        tmem_ld32(tDP + lane_off + col0, dr);
        tmem_ld_wait(sr);
        tmem_ld_wait(dr);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float pv[2], dsv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col = col0 + e + u;
            const int other = srow + col;  // the query (dK/dV) or key (dQ) of this column
            int q_i, k_j;
            float lse2, dl;
            if (kDq) {
              q_i = my_row;
              k_j = other;
              lse2 = row_lse2;
              dl = row_delta;
            } else {
              q_i = other;
              k_j = my_row;
              lse2 = vec[col];
              dl = vec[kRows + col];
            }
            const bool vis = q_i < S && k_j < S && (!p.causal || k_j <= q_i);
            const float pr = vis ? ex2_approx(__uint_as_float(sr[e + u]) * c2 - lse2) : 0.f;
            pv[u] = pr;
            dsv[u] = pr * (__uint_as_float(dr[e + u]) - dl);
          }
          pk_a[16 * h + e / 2] = pack_bf16x2(pv[0], pv[1]);
          pk_b[16 * h + e / 2] = pack_bf16x2(dsv[0], dsv[1]);
        }
      }
      // the warpgroup's 64 columns become 32 TMEM columns of bf16 pairs, written
      // over the first half of its own columns (the other warpgroup may still
      // be reading its own)
      if (kDq) {
        tmem_st32(tS + lane_off + 64 * g, pk_b);  // dS over S
      } else {
        tmem_st32(tS + lane_off + 64 * g, pk_a);  // P^T over S^T
        tmem_st32(tDP + lane_off + 64 * g, pk_b); // dS^T over dP^T
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPt));
    }
    // ------------------------------------------------------------ epilogue
    bool done = ok && n_iter > 0 && mbar_wait(bar(kBarAcc), 0, abort_flag, err);
    done = __all_sync(0xffffffffu, done);
    tc_fence_after();
    // warp-uniform branches only around the TMEM loads; the row bound guards the stores
    const bool valid = my_row < S;
    const size_t row_off = static_cast<size_t>(head) * S + (valid ? my_row : 0);
    if (kDq) {
      if (g == 0) {  // dQ = scale dS K
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.dq) + row_off * kD;
        if (done) store_acc_row(tAcc0 + lane_off, p.scale, dst, valid);
        else if (valid) for (int d = 0; d < kD; ++d) dst[d] = __float2bfloat16(0.f);
      }
    } else {
      __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(g == 0 ? p.dv : p.dk) + row_off * kD;
      if (done) store_acc_row((g == 0 ? tAcc0 : tAcc1) + lane_off, g == 0 ? 1.f : p.scale, dst, valid);
      else if (valid) for (int d = 0; d < kD; ++d) dst[d] = __float2bfloat16(0.f);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace bwd
}  // namespace seqattn
