// Backward of blockwise attention for sm_103a (head dim 64 or 128, bf16): the
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
//               TMEM, four warpgroups (32 query columns each) form P^T and dS^T
//               as bf16 in TMEM, and dV += P^T dO, dK += dS^T Q accumulate in
//               TMEM (TS form, Q and dO as N-contiguous operands).
//   dQ          one CTA per 128-row query tile: Q and dO stay, the visible key
//               tiles stream through; S = Q K^T, dP = dO V^T, dS in TMEM, and
//               dQ += dS K.
// Both matrix kernels: warp 17 TMA producer, warp 16 MMA issuer (one thread),
// warps 0-15 the element-wise pass (four warpgroups of 32 columns each, in
// two phases per streamed tile: P from S, then dS from P and dP). The issuer
// orders each tile's products so that one tile's element-wise phases overlap
// its neighbours' products. Every wait is bounded.
#pragma once
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace seqattn {
namespace bwd {

constexpr int kRows = 128;                      // tile rows (keys or queries)
constexpr int kColBlock = kRows * 128;          // 16 KB: 128 rows of one 128-byte column block
constexpr int kThreads = 576;
constexpr int kMmaWarp = 16, kTmaWarp = 17;
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory plan for head dim D: tiles of 128 rows x D bf16 (D / 64
// column blocks), a 128 KB ring of them.
template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kTileBytes = kRows * D * 2;
  static constexpr int kStages = 131072 / kTileBytes;  // 4 slots of 32 KB or 8 of 16 KB
  // barriers: stay_full, full[S], empty[S / 2] (one per iteration's pair of
  // slots), st_full[2], pt_full[2], acc_done
  static constexpr int kNumBarriers = 1 + kStages + kStages / 2 + 5;
  static constexpr int kSmemBytes = 1024 + 2 * kTileBytes + kStages * kTileBytes + 2 * 2 * kRows * 4 +
                                    8 * kNumBarriers + 16;
};

// Loads a 128 x D bf16 tile (one 64-column box per column block) into `dst`.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap *map, uint32_t bar, int row,
                                          int head) {
#pragma unroll
  for (int cb = 0; cb < D / 64; ++cb) tma_load_3d(dst + cb * kColBlock, map, bar, 64 * cb, row, head);
}

// S (or S^T) = A B^T over D: A and B 128-row K-major tiles (N = 128: the
// full-rate shape; N = 64 halves are bound by shared-memory reads).
template <int D>
__device__ __forceinline__ void mma_rows_dot(uint32_t d_tmem, uint32_t a, uint32_t b) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * kColBlock + (kk % 4) * 32;
    mma_ss(d_tmem, sw128_desc(a + off, 16, 1024), sw128_desc(b + off, 16, 1024), idesc,
           kk > 0 ? 1u : 0u);
  }
}

// acc (+)= A_h B_h for contraction half h: A = 128 x 128 bf16 in TMEM
// (contraction over its columns), B = 128 x D tile in shared memory whose
// rows are the contraction index (N-contiguous operand); half h covers
// contraction elements [64h, 64h + 64). A's elements are packed as bf16 pairs:
// the element-wise warpgroup of columns [32c, 32c + 32) packs them over the
// first 16 of its own TMEM columns, so elements 16k..16k+15 sit in the 8
// columns at a_tmem + 32(k/2) + 8(k%2).
template <int D>
__device__ __forceinline__ void mma_acc_tmem(uint32_t acc, uint32_t a_tmem, uint32_t b, int h, bool first) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, true);
#pragma unroll
  for (int k4 = 0; k4 < 4; ++k4) {
    const int kk = 4 * h + k4;
    mma_ts(acc, a_tmem + 64 * h + 32 * (k4 >> 1) + 8 * (k4 & 1), sw128_desc(b + kk * 2048, kColBlock, 1024), idesc,
           (first && k4 == 0) ? 0u : 1u);
  }
}

// acc (+)= A B over the full contraction of 128 elements, A = 128 x 128 bf16
// in TMEM packed compactly (elements 16k..16k+15 in the 8 columns at
// a_tmem + 8k), B as for mma_acc_tmem.
template <int D>
__device__ __forceinline__ void mma_acc_compact(uint32_t acc, uint32_t a_tmem, uint32_t b, bool first) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, true);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts(acc, a_tmem + 8 * kk, sw128_desc(b + kk * 2048, kColBlock, 1024), idesc,
           (first && kk == 0) ? 0u : 1u);
}

// NC columns of one thread's row of an fp32 TMEM accumulator, times `mul`,
// as bf16 into global memory. Every lane of the warp takes part in the TMEM
// loads (they are warp-wide); only lanes with `valid` store.
template <int NC>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, float mul, __nv_bfloat16 *dst, bool valid) {
  static_assert(NC % 16 == 0, "16-column chunks");
#pragma unroll 1
  for (int cb = 0; cb < NC / 16; ++cb) {
    uint32_t r[16];
    tmem_ld16(taddr + 16 * cb, r);
    tmem_ld_wait(r);
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * i]) * mul,
                                               __uint_as_float(r[2 * i + 1]) * mul);
      pk[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    if (valid) {
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + 16 * cb);
#pragma unroll
      for (int i = 0; i < 2; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// ---------------------------------------------------------------- delta
// A warp per row; lane l reads elements [D/32 l, D/32 (l + 1)) of O and dO.
template <int D>
__global__ void delta_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                             float *__restrict__ delta, long long nrows) {
  using Vec = typename std::conditional<D == 128, uint2, uint32_t>::type;  // D / 32 bf16 per lane
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (long long r = warp; r < nrows; r += nwarps) {
    const Vec a = reinterpret_cast<const Vec *>(o + r * D)[lane];
    const Vec b = reinterpret_cast<const Vec *>(dout + r * D)[lane];
    const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < D / 64; ++i) {
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
template <int D, bool kDq>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int kTileBytes = C::kTileBytes, kStages = C::kStages, kNumBarriers = C::kNumBarriers;
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
  const int kBarStay = 0, kBarFull = 1, kBarEmpty = 1 + kStages, kBarSt = kBarEmpty + kStages / 2,
            kBarPt = kBarSt + 2, kBarAcc = kBarPt + 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int *err = &g_device_error;
  const int S = p.S, group = p.Hq / p.Hkv;
  const int n_tiles = (S + kRows - 1) / kRows;
  // tiles vary fastest, so the CTAs running together are tiles of one head
  // (they stream the same tiles of that head's group, shared in L2); the CTAs
  // with the most iterations come first: low key tiles (dK/dV), high query
  // tiles (causal dQ)
  const int head = blockIdx.y;  // b*Hkv + hkv (dK/dV) or b*Hq + hq (dQ)
  const int tile = (kDq && p.causal) ? n_tiles - 1 - static_cast<int>(blockIdx.x)
                                     : static_cast<int>(blockIdx.x);  // key or query tile
  const int b = kDq ? head / p.Hq : head / p.Hkv;
  // dK/dV: iterations over (query head of the group, query tile >= this key
  // tile when causal); dQ: over key tiles <= this query tile when causal
  const int first_stream = (!kDq && p.causal) ? tile : 0;
  const int n_stream_tiles = kDq ? (p.causal ? tile + 1 : n_tiles) : n_tiles - first_stream;
  const int n_iter = kDq ? n_stream_tiles : group * n_stream_tiles;
  // dK/dV streams the query tiles from the last one down, the group's query
  // heads innermost: every CTA of a KV head then reads the same (head, query
  // tile) at the same iteration until it reaches its own diagonal, so the
  // CTAs running together share each streamed tile in L2.
  auto stream_of = [&](int it, int &row, int &q_head) {  // the streamed tile of iteration it
    if (kDq) {
      row = it * kRows;
      q_head = head;
    } else {
      row = (n_tiles - 1 - it / group) * kRows;
      q_head = b * p.Hq + (head % p.Hkv) * group + it % group;
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarStay), 1);
    for (int s = 0; s < kStages; ++s) mbar_init(bar(kBarFull + s), 1);
    for (int s = 0; s < kStages / 2; ++s) mbar_init(bar(kBarEmpty + s), 1);
    mbar_init(bar(kBarSt), 1);      // S (or S^T) computed
    mbar_init(bar(kBarSt + 1), 1);  // dP (or dP^T) computed
    mbar_init(bar(kBarPt), 16);     // P^T in TMEM (dK/dV): one arrival per element-wise warp
    mbar_init(bar(kBarPt + 1), 16); // dS (or dS^T) in TMEM
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
  // dP or dP^T [128,256), accumulators [256,256+D) and (dK/dV) [256+D,256+2D)
  const uint32_t tS = tmem, tDP = tmem + 128, tAcc0 = tmem + 256, tAcc1 = tmem + 256 + D;
  const uint32_t tDS = tAcc1;  // dQ kernel: two 64-column buffers of packed dS (tAcc1 is dK/dV's)

  if (warp == kTmaWarp) {
    if (lane == 0 && !skip && n_iter > 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      tma_prefetch_map(&tm_do);
      mbar_arrive_expect_tx(bar(kBarStay), 2 * kTileBytes);
      if (kDq) {
        load_tile<D>(smem_addr(sStay), &tm_q, bar(kBarStay), tile * kRows, head);
        load_tile<D>(smem_addr(sStay + kTileBytes), &tm_do, bar(kBarStay), tile * kRows, head);
      } else {
        load_tile<D>(smem_addr(sStay), &tm_k, bar(kBarStay), tile * kRows, head);
        load_tile<D>(smem_addr(sStay + kTileBytes), &tm_v, bar(kBarStay), tile * kRows, head);
      }
      const int kv_head = kDq ? b * p.Hkv + (head % p.Hq) / group : head;
      int c = 0;
      bool ok = true;
      for (int it = 0; it < n_iter && ok; ++it) {
        int row, q_head;
        stream_of(it, row, q_head);
        // both slots of iteration it are free once iteration it - kStages / 2 is released
        const int pair = it % (kStages / 2), round = it / (kStages / 2);
        if (round > 0 && !mbar_wait(bar(kBarEmpty + pair), (round - 1) & 1, abort_flag, err)) break;
        for (int which = 0; which < 2; ++which, ++c) {  // Q_i then dO_i, or K_j then V_j
          const int slot = c % kStages;
          mbar_arrive_expect_tx(bar(kBarFull + slot), kTileBytes);
          const CUtensorMap *map = kDq ? (which ? &tm_v : &tm_k) : (which ? &tm_do : &tm_q);
          load_tile<D>(smem_addr(sRing + slot * kTileBytes), map, bar(kBarFull + slot), row,
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
      // Iteration it: S (or S^T) and dP (or dP^T) as N = 128 products, each on
      // its own barrier, so the element-wise warps form P while dP is still
      // being computed. dK/dV: dV += P^T dO as soon as P is in TMEM, then
      // the next S (it overwrites P^T, in issue order behind dV), then
      // dK += dS^T Q and the next dP. dQ: the next S as soon as the warps
      // have read S out, dQ += dS K once dS is in TMEM (double-buffered in
      // columns the dQ kernel has free), then the next dP. The element-wise
      // pass of one tile thus overlaps the products of its neighbours.
      auto full = [&](int it) {  // both tiles of iteration it have landed (no fence)
        const int c0 = 2 * it, c1 = 2 * it + 1;
        return mbar_wait(bar(kBarFull + c0 % kStages), (c0 / kStages) & 1, abort_flag, err) &&
               mbar_wait(bar(kBarFull + c1 % kStages), (c1 / kStages) & 1, abort_flag, err);
      };
      auto ring0 = [&](int it) { return ring + ((2 * it) % kStages) * kTileBytes; };
      auto ring1 = [&](int it) { return ring + ((2 * it + 1) % kStages) * kTileBytes; };
      // S = Q K_j^T, dP = dO V_j^T (or S^T = K Q_i^T, dP^T = V dO_i^T)
      auto scores_s = [&](int it) {
        mma_rows_dot<D>(tS, stay0, ring0(it));
        mma_commit(bar(kBarSt));
      };
      auto scores_dp = [&](int it) {
        mma_rows_dot<D>(tDP, stay1, ring1(it));
        mma_commit(bar(kBarSt + 1));
      };
      bool ok = mbar_wait(bar(kBarStay), 0, abort_flag, err) && full(0);
      if (ok) {
        scores_s(0);
        scores_dp(0);
      }
      for (int it = 0; ok && it < n_iter; ++it) {
        const bool more = it + 1 < n_iter;
        // P^T in TMEM (dK/dV), or S read out (dQ); then the next S, which
        // overwrites those columns, right behind the products that read them
        if (!mbar_wait(bar(kBarPt), it & 1, abort_flag, err) || (more && !full(it + 1))) break;
        tc_fence_after();
        if (!kDq) {  // dV += P^T dO_i
          mma_acc_tmem<D>(tAcc0, tS, ring1(it), 0, it == 0);
          mma_acc_tmem<D>(tAcc0, tS, ring1(it), 1, false);
        }
        if (more) scores_s(it + 1);
        if (!mbar_wait(bar(kBarPt + 1), it & 1, abort_flag, err)) break;
        tc_fence_after();
        if (kDq)  // dQ += dS K_j, dS in its own double-buffered columns
          mma_acc_compact<D>(tAcc0, tDS + 64 * (it & 1), ring0(it), it == 0);
        else {    // dK += dS^T Q_i
          mma_acc_tmem<D>(tAcc1, tDP, ring0(it), 0, it == 0);
          mma_acc_tmem<D>(tAcc1, tDP, ring0(it), 1, false);
        }
        mma_commit(bar(kBarEmpty + it % (kStages / 2)));
        if (more) scores_dp(it + 1);
      }
      mma_commit(bar(kBarAcc));
      mbar_drain(bar(kBarAcc), 0, err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ element-wise pass
    const int wg = warp >> 2;                        // element-wise warpgroup 0-3
    const int h = wg & 1;                            // 64-column half it serves
    const int c_base = 64 * h + 32 * (wg >> 1);      // its 32 columns of the tile
    const int row_in_tile = (warp & 3) * 32 + lane;  // TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int my_row = tile * kRows + row_in_tile;   // key (dK/dV) or query (dQ) of this thread
    const float c2 = p.scale * kLog2e;
    // dQ: this query row's lse (log2 units) and delta, once
    float row_lse2 = INFINITY, row_delta = 0.f;
    if (kDq && my_row < S) {
      row_lse2 = p.lse[static_cast<size_t>(head) * S + my_row] * kLog2e;
      row_delta = p.delta[static_cast<size_t>(head) * S + my_row];
    }
    // dK/dV: thread t < 32 of the warpgroup carries the lse (log2 units) and
    // delta of query column c_base + t of the streamed tile, loaded one
    // iteration ahead so that the load latency hides behind an iteration
    const int vec_col = c_base + (threadIdx.x & 127);
    const bool vec_thread = !kDq && (threadIdx.x & 127) < 32;
    float nxt_lse2 = INFINITY, nxt_delta = 0.f;
    auto load_vec = [&](int it) {
      int r, qh;
      stream_of(it, r, qh);
      const int i = r + vec_col;
      nxt_lse2 = (i < S) ? p.lse[static_cast<size_t>(qh) * S + i] * kLog2e : INFINITY;
      nxt_delta = (i < S) ? p.delta[static_cast<size_t>(qh) * S + i] : 0.f;
    };
    if (vec_thread && n_iter > 0) load_vec(0);
    bool ok = !skip;
    for (int it = 0; it < n_iter; ++it) {
      int srow, q_head;
      stream_of(it, srow, q_head);
      float *vec = sVec + (it & 1) * 2 * kRows;  // [lse2 | delta] of the streamed query tile
      if (vec_thread) {
        vec[vec_col] = nxt_lse2;
        vec[kRows + vec_col] = nxt_delta;
        if (it + 1 < n_iter) load_vec(it + 1);
      }
      // the mask matters only on tiles that cross the end of the sequence or
      // the causal diagonal
      const int base = tile * kRows;
      const bool need_mask = base + kRows > S || srow + kRows > S ||
                             (p.causal && (kDq ? srow + kRows > base : srow < base + kRows));
      bool got = ok && mbar_wait(bar(kBarSt), it & 1, abort_flag, err);
      got = named_bar_and(1 + wg, 128, __all_sync(0xffffffffu, got));  // also publishes vec
      if (!got) break;
      tc_fence_after();
      // Phase 1, once S is in TMEM: P for this thread's 32 columns (kept in
      // registers for dS); dK/dV writes it as bf16 pairs over the first 16 of
      // the warpgroup's columns (chunk c to c_base + 8c), which it has read.
      float pf[32];
      auto chunk_p = [&](auto mask_tag, int c) {
        constexpr bool kMask = decltype(mask_tag)::value;
        const int col0 = c_base + 16 * c;
        uint32_t sr[16];
        tmem_ld16(tS + lane_off + col0, sr);
        float lv[16];
        if (!kDq) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 a4 = reinterpret_cast<const float4 *>(vec + col0)[i];
            lv[4 * i] = a4.x, lv[4 * i + 1] = a4.y, lv[4 * i + 2] = a4.z, lv[4 * i + 3] = a4.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) lv[i] = row_lse2;
        }
        tmem_ld_wait(sr);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float pr = ex2_approx(__uint_as_float(sr[e]) * c2 - lv[e]);
          if (kMask) {
            const int other = srow + col0 + e;  // the query (dK/dV) or key (dQ) of this column
            const int q_i = kDq ? my_row : other, k_j = kDq ? other : my_row;
            if (!(q_i < S && k_j < S && (!p.causal || k_j <= q_i))) pr = 0.f;
          }
          pf[16 * c + e] = pr;
        }
        if (!kDq) {
          uint32_t pa[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) pa[e] = pack_bf16x2(pf[16 * c + 2 * e], pf[16 * c + 2 * e + 1]);
          tmem_st8(tS + lane_off + c_base + 8 * c, pa);  // P^T over S^T
        }
      };
      if (need_mask) {
        chunk_p(std::true_type{}, 0);
        chunk_p(std::true_type{}, 1);
      } else {
        chunk_p(std::false_type{}, 0);
        chunk_p(std::false_type{}, 1);
      }
      // P^T stored (dK/dV), or S read out (dQ): the issuer may overwrite S
      if (!kDq) tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPt));
      // Phase 2, once dP is in TMEM: dS = P (dP - delta), as bf16 pairs over
      // dP^T (dK/dV) or into the iteration's dS buffer (dQ, where P never
      // goes to TMEM)
      got = mbar_wait(bar(kBarSt + 1), it & 1, abort_flag, err);
      got = named_bar_and(1 + wg, 128, __all_sync(0xffffffffu, got));
      if (!got) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col0 = c_base + 16 * c;
        uint32_t dr[16];
        tmem_ld16(tDP + lane_off + col0, dr);
        float dl[16];
        if (!kDq) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 d4 = reinterpret_cast<const float4 *>(vec + kRows + col0)[i];
            dl[4 * i] = d4.x, dl[4 * i + 1] = d4.y, dl[4 * i + 2] = d4.z, dl[4 * i + 3] = d4.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) dl[i] = row_delta;
        }
        tmem_ld_wait(dr);
        uint32_t pb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          pb[e] = pack_bf16x2(pf[16 * c + 2 * e] * (__uint_as_float(dr[2 * e]) - dl[2 * e]),
                              pf[16 * c + 2 * e + 1] * (__uint_as_float(dr[2 * e + 1]) - dl[2 * e + 1]));
        if (kDq)  // dS packed compactly into the iteration's buffer (elements 16k.. at column 8k)
          tmem_st8(tDS + 64 * (it & 1) + lane_off + (c_base / 16 + c) * 8, pb);
        else      // dS^T over dP^T
          tmem_st8(tDP + lane_off + c_base + 8 * c, pb);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPt + 1));
    }
    // ------------------------------------------------------------ epilogue
    bool done = ok && n_iter > 0 && mbar_wait(bar(kBarAcc), 0, abort_flag, err);
    done = __all_sync(0xffffffffu, done);
    tc_fence_after();
    // warp-uniform branches only around the TMEM loads; the row bound guards the stores
    const bool valid = my_row < S;
    const size_t row_off = static_cast<size_t>(head) * S + (valid ? my_row : 0);
    if (kDq) {  // dQ = scale dS K: warpgroup w stores columns [D/4 w, D/4 (w + 1))
      constexpr int kNc = D / 4;
      __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.dq) + row_off * D + kNc * wg;
      if (done) store_acc_row<kNc>(tAcc0 + lane_off + kNc * wg, p.scale, dst, valid);
      else if (valid) for (int d = 0; d < kNc; ++d) dst[d] = __float2bfloat16(0.f);
    } else {  // warpgroups 0, 1: dV columns [0, D/2), [D/2, D); 2, 3: dK (times scale)
      constexpr int kNc = D / 2;
      const bool is_dk = wg >= 2;
      const int cofs = kNc * (wg & 1);
      __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(is_dk ? p.dk : p.dv) + row_off * D + cofs;
      if (done) store_acc_row<kNc>((is_dk ? tAcc1 : tAcc0) + lane_off + cofs, is_dk ? p.scale : 1.f, dst, valid);
      else if (valid) for (int d = 0; d < kNc; ++d) dst[d] = __float2bfloat16(0.f);
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
