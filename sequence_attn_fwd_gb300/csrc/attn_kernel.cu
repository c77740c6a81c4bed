// Blockwise exact attention forward for sm_103a.
//
// What it computes: for every query row, softmax(scale * q K^T) V over the
// visible keys and the row's log-sum-exp, tile by tile over K/V with a
// running maximum and normaliser, so the [S, S] scores never reach memory
// (the tiled online-softmax forward described on page "ms-swift集成
// FlashAttention 2/3，长文本训练更高效", section "FlashAttention 如何破局？
// 不只是融合内核": a block loads a Q tile, streams the matching K/V tiles
// through on-chip memory, keeps the max and normaliser up to date and writes
// only the output). With global offsets and fp32 output the same kernel
// produces the per-hop partial (O_i, lse_i) of Ring-Attention.
//
// How (one CTA = 256 query rows of one (batch, head), 320 threads):
//   warp 9      TMA producer: both Q tiles once, then K_j, V_j into a ring of
//               shared-memory slots (128-byte swizzle, 3-D tensor maps so
//               rows past the end of a head read as zero).
//   warp 8      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM (SS form)
//               and O_t += P_t V_j with P_t read from TMEM (TS form). The two
//               query tiles t = 0, 1 alternate so the tensor pipe works on one
//               tile while the other tile's softmax runs.
//   warps 0-7   two softmax warpgroups, one per query tile, one query row per
//               thread: load the row of S from TMEM, mask, update the running
//               max (in log2 units), exponentiate, write P (bf16) back over S
//               in TMEM, and rescale O in TMEM only when the max has grown by
//               more than 2^8 since the last rescale; finally O / l and lse.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [384,384+D).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace seqattn {

__device__ int g_device_error;  // set by a timed-out wait; read and cleared by the host

namespace {

constexpr int kRowsPerTile = 128;  // MMA M and KV tile length
constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kColBlockBytes = 128 * 128;  // 128 rows x 128 bytes (64 bf16) swizzle block
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows > 2^8

template <int D>
struct Cfg {
  static constexpr int kColBlocks = D / 64;
  static constexpr int kTileBytes = kRowsPerTile * D * 2;
  static constexpr int kStages = (D == 128) ? 4 : 8;
  static constexpr int kSmemQ = 2 * kTileBytes;
  static constexpr int kSmemRing = kStages * kTileBytes;
  // barriers: q, full[S], empty[S], s_full[2], p_full[2], o_full[2], mma_done
  static constexpr int kNumBarriers = 1 + 2 * kStages + 7;
  static constexpr int kSmemBytes = 1024 + kSmemQ + kSmemRing + 8 * kNumBarriers + 16;
};

// Per-tile number of KV tiles to visit (0 when the tile has no valid row or
// none of its rows sees any key).
__device__ __forceinline__ int kv_tiles_for(const AttnParams &p, int first_row) {
  const int n_all = (p.Skv + kRowsPerTile - 1) / kRowsPerTile;
  if (first_row >= p.Sq || n_all == 0) return 0;
  if (!p.causal) return n_all;
  const int last_row = min(first_row + kRowsPerTile - 1, p.Sq - 1);
  const long long max_key = p.q_off + last_row - p.kv_off;  // largest visible key index
  if (max_key < 0) return 0;
  const long long n = max_key / kRowsPerTile + 1;
  return n < n_all ? static_cast<int>(n) : n_all;
}

// Maximum of the 128 scores of a row (raw, before scaling).
__device__ __forceinline__ float row_max(const float *s) {
  float a = s[0], b = s[1], c = s[2], d = s[3];
#pragma unroll
  for (int i = 4; i < 124; i += 8) {
    a = fmax3(a, s[i], s[i + 1]);
    b = fmax3(b, s[i + 2], s[i + 3]);
    c = fmax3(c, s[i + 4], s[i + 5]);
    d = fmax3(d, s[i + 6], s[i + 7]);
  }
  a = fmax3(a, s[124], s[125]);
  b = fmax3(b, s[126], s[127]);
  return fmax3(fmaxf(a, b), c, d);
}

// P = 2^(s * c2 - m_ref) for the 128 scores of a row, packed as bf16 pairs
// (element 2i in the low half), returning the fp32 sum of the unrounded P.
// With kTrackMax the raw row maximum is found in the same pass.
template <bool kTrackMax>
__device__ __forceinline__ float exp_row(const float *s, float c2, float m_ref, uint32_t *pk,
                                         float *mx_out) {
  const uint64_t scale2 = f2_pack(c2, c2);
  const uint64_t neg_m2 = f2_pack(-m_ref, -m_ref);
  uint64_t sum_a = f2_pack(0.f, 0.f), sum_b = sum_a;
  float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
  for (int c = 0; c < 64; c += 2) {
    float x0, x1, x2, x3;
    f2_unpack(f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), scale2, neg_m2), x0, x1);
    f2_unpack(f2_fma(f2_pack(s[2 * c + 2], s[2 * c + 3]), scale2, neg_m2), x2, x3);
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
    sum_a = f2_add(sum_a, f2_pack(p0, p1));
    sum_b = f2_add(sum_b, f2_pack(p2, p3));
    if (kTrackMax) {
      ma = fmax3(ma, s[2 * c], s[2 * c + 1]);
      mb = fmax3(mb, s[2 * c + 2], s[2 * c + 3]);
    }
    __nv_bfloat162 h0 = __floats2bfloat162_rn(p0, p1);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(p2, p3);
    pk[c] = *reinterpret_cast<uint32_t *>(&h0);
    pk[c + 1] = *reinterpret_cast<uint32_t *>(&h1);
  }
  if (kTrackMax) *mx_out = fmaxf(ma, mb);
  float a0, a1, b0, b1;
  f2_unpack(sum_a, a0, a1);
  f2_unpack(sum_b, b0, b1);
  return (a0 + a1) + (b0 + b1);
}

template <int D, bool kF32Out>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem;                   // [tile][col block][128 rows][128 B]
  uint8_t *sRing = smem + C::kSmemQ;    // [slot][col block][128 rows][128 B]
  uint64_t *bars = reinterpret_cast<uint64_t *>(sRing + C::kSmemRing);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBarriers);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const uint32_t bar0 = smem_addr(bars);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  const int kBarQ = 0, kBarFull = 1, kBarEmpty = 1 + C::kStages, kBarSFull = 1 + 2 * C::kStages,
            kBarPFull = kBarSFull + 2, kBarOFull = kBarPFull + 2, kBarMmaDone = kBarOFull + 2;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;  // b * Hq + hq: heads of one GQA group are neighbours
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int hkv = hq / (p.Hq / p.Hkv);
  // causal: the longest query blocks (most KV tiles) are launched first
  const int qblock = p.causal ? (p.n_qblocks - 1 - static_cast<int>(blockIdx.y))
                              : static_cast<int>(blockIdx.y);
  const int row0 = qblock * 2 * kRowsPerTile;
  int *err = &g_device_error;

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPFull + t), 128);
      mbar_init(bar(kBarOFull + t), 1);
    }
    mbar_init(bar(kBarMmaDone), 1);
    // A timeout recorded by any earlier CTA or launch (and not yet cleared by
    // the host) makes this CTA skip its work: its rows come out as O = 0,
    // lse = -inf, and the host learns of it from the device error query.
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
  const int n_tiles[2] = {skip ? 0 : kv_tiles_for(p, row0), skip ? 0 : kv_tiles_for(p, row0 + kRowsPerTile)};
  const int n_max = max(n_tiles[0], n_tiles[1]);
  // TMEM column of S_t / P_t and of O_t for query tile t
  auto tS = [&](int t) -> uint32_t { return tmem + 128u * static_cast<uint32_t>(t); };
  auto tO = [&](int t) -> uint32_t { return tmem + 256u + 128u * static_cast<uint32_t>(t); };

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_max > 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      mbar_arrive_expect_tx(bar(kBarQ), 2 * C::kTileBytes);
      for (int t = 0; t < 2; ++t)
        for (int cb = 0; cb < C::kColBlocks; ++cb)
          tma_load_3d(smem_addr(sQ + (t * C::kColBlocks + cb) * kColBlockBytes), &tm_q, bar(kBarQ),
                      cb * 64, row0 + t * kRowsPerTile, bh);
      const int kv_head = b * p.Hkv + hkv;
      int c = 0;  // K_0, V_0, K_1, V_1, ... in the order the MMA issuer consumes them
      bool ok = true;
      for (int j = 0; j < n_max && ok; ++j) {
        for (int which = 0; which < 2; ++which, ++c) {
          const int slot = c % C::kStages;
          if (c >= C::kStages &&
              !mbar_wait(bar(kBarEmpty + slot), ((c / C::kStages) - 1) & 1, abort_flag, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarFull + slot), C::kTileBytes);
          const CUtensorMap *map = which ? &tm_v : &tm_k;
          for (int cb = 0; cb < C::kColBlocks; ++cb)
            tma_load_3d(smem_addr(sRing + (slot * C::kColBlocks + cb) * kColBlockBytes), map,
                        bar(kBarFull + slot), cb * 64, j * kRowsPerTile, kv_head);
        }
      }
      // Every copy issued must have landed before the CTA may exit.
      mbar_drain(bar(kBarQ), 0, err);
      for (int i = max(0, c - C::kStages); i < c; ++i)
        mbar_drain(bar(kBarFull + i % C::kStages), (i / C::kStages) & 1, err);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, true);
      const uint32_t q_base = smem_addr(sQ);
      const uint32_t ring_base = smem_addr(sRing);
      bool ok = n_max > 0 && mbar_wait(bar(kBarQ), 0, abort_flag, err);
      // Per KV step j: PV_0(j-1), S_0(j), PV_1(j-1), S_1(j). Both ring slots of
      // the step are waited for first (measured faster on GB300 than waiting
      // for each just before its first use); each slot is released by a commit
      // that fires when its last MMA completes.
      for (int j = 0; ok && j <= n_max; ++j) {
        const int cK = 2 * j, cV = 2 * j - 1;  // ring positions of K_j and V_{j-1}
        const int sK = cK % C::kStages, sV = (cV + C::kStages) % C::kStages;
        const uint32_t k_base = ring_base + sK * C::kTileBytes;
        const uint32_t v_base = ring_base + sV * C::kTileBytes;
        if (j < n_max && !mbar_wait(bar(kBarFull + sK), (cK / C::kStages) & 1, abort_flag, err)) break;
        if (j >= 1 && !mbar_wait(bar(kBarFull + sV), (cV / C::kStages) & 1, abort_flag, err)) break;
        tc_fence_after();
        for (int t = 0; t < 2 && ok; ++t) {
          const int nt = t ? n_tiles[1] : n_tiles[0];
          if (j >= 1 && j - 1 < nt) {
            // O_t += P_t V_{j-1}; P_t was written over S_t by the softmax warps
            if (!mbar_wait(bar(kBarPFull + t), (j - 1) & 1, abort_flag, err)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kRowsPerTile / 16; ++kk) {
              const uint64_t bdesc = sw128_desc(v_base + kk * 2048, kColBlockBytes, 1024);
              mma_ts(tO(t), tS(t) + kk * 8, bdesc, idesc_o, (j > 1 || kk > 0) ? 1u : 0u);
            }
            if (j - 1 == nt - 1) mma_commit(bar(kBarOFull + t));
            if (t == 1 || j - 1 >= n_tiles[1]) mma_commit(bar(kBarEmpty + sV));  // last use of V_{j-1}
          }
          if (j < nt) {
            // S_t = Q_t K_j^T
            const uint32_t qt = q_base + t * C::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk / 4) * kColBlockBytes + (kk % 4) * 32;
              mma_ss(tS(t), sw128_desc(qt + off, 16, 1024), sw128_desc(k_base + off, 16, 1024),
                     idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar(kBarSFull + t));
            if (t == 1 || j >= n_tiles[1]) mma_commit(bar(kBarEmpty + sK));  // last use of K_j
          }
        }
      }
      // All MMAs issued here must be complete before TMEM is released.
      mma_commit(bar(kBarMmaDone));
      mbar_drain(bar(kBarMmaDone), 0, err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;                       // query tile of this warpgroup
    const int row_in_tile = (warp & 3) * 32 + lane;  // TMEM lane = tile row
    const int row = row0 + t * kRowsPerTile + row_in_tile;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_addr = tS(t) + lane_off;
    const uint32_t o_addr = tO(t) + lane_off;
    const int n = t ? n_tiles[1] : n_tiles[0];
    const long long qpos = p.q_off + row;
    const long long tile_first_q = p.q_off + row0 + t * kRowsPerTile;
    const float c2 = p.scale_log2;
    float m = -INFINITY;  // running max of scale*log2(e)*s (the reference for P)
    float l = 0.f;        // running sum of P relative to m
    float m_grow = -INFINITY;  // candidate new reference from the latest tile
    bool ok = true;

    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + t), j & 1, abort_flag, err));
      if (!ok) break;
      tc_fence_after();
      const int kv0 = j * kRowsPerTile;
      const bool tail = kv0 + kRowsPerTile > p.Skv;
      const bool diag = p.causal && (p.kv_off + kv0 + kRowsPerTile - 1 > tile_first_q);
      int last = 127;  // last visible column of this row in the tile
      if (tail || diag) {
        long long lim = static_cast<long long>(p.Skv) - kv0 - 1;
        if (p.causal) {
          const long long c_lim = qpos - p.kv_off - kv0;
          lim = c_lim < lim ? c_lim : lim;
        }
        last = static_cast<int>(lim < -1 ? -1 : (lim > 127 ? 127 : lim));
      }
      // The row of S for this tile, masked (TMEM keeps S until P is written).
      auto load_scores = [&](uint32_t (&sr)[128]) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          tmem_ld32(s_addr + 32 * i, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * i]));
        tmem_ld_wait(sr);
        if (tail || diag) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > last) sr[c] = __float_as_uint(-INFINITY);
        }
      };
      uint32_t pk[64];
      float rowsum;
      {
        uint32_t sr[128];
        load_scores(sr);
        const float *s = reinterpret_cast<const float *>(sr);
        if (j == 0) {
          // no reference yet: the tile maximum first, then the exponentials
          m = row_max(s) * c2;
          rowsum = exp_row<false>(s, c2, (m == -INFINITY) ? 0.f : m, pk, nullptr);
        } else {
          // Exponentiate against the current reference while finding the tile
          // maximum; only if some row's maximum grew by more than 2^8 (rare
          // after the first tiles) is O rescaled and the pass redone.
          float mx;
          rowsum = exp_row<true>(s, c2, (m == -INFINITY) ? 0.f : m, pk, &mx);
          m_grow = fmaxf(m, mx * c2);
        }
      }
      if (j > 0) {
        const float m_new = m_grow;
        const bool grow = (m_new - m) > kRescaleThreshold;  // false while both are -inf
        if (__any_sync(0xffffffffu, grow)) {
          const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(m - m_new);
          m = m_new;
          l *= alpha;
          // O_t holds the sum through KV tile j-1: the MMA that produced it
          // completed before S_t for tile j was signalled.
#pragma unroll 1
          for (int cb = 0; cb < D / 32; ++cb) {
            uint32_t orr[32];
            tmem_ld32(o_addr + 32 * cb, orr);
            tmem_ld_wait(orr);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            tmem_st32(o_addr + 32 * cb, orr);
          }
          tmem_st_wait();
          uint32_t sr[128];
          load_scores(sr);
          rowsum = exp_row<false>(reinterpret_cast<const float *>(sr), c2,
                                  (m == -INFINITY) ? 0.f : m, pk, nullptr);
        }
      }
      l += rowsum;
      tmem_st32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + t));
    }

    // ------------------------------------------------------------ epilogue
    bool have_o = false;
    if (ok && n > 0) {
      have_o = __all_sync(0xffffffffu, mbar_wait(bar(kBarOFull + t), 0, abort_flag, err));
      tc_fence_after();
    }
    const bool row_valid = row < p.Sq;
    const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    const size_t row_index = static_cast<size_t>(bh) * p.Sq + row;
#pragma unroll 1
    for (int cb = 0; cb < D / 32; ++cb) {
      uint32_t orr[32];
      if (have_o) {
        tmem_ld32(o_addr + 32 * cb, orr);
        tmem_ld_wait(orr);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) orr[i] = 0u;
      }
      if (!row_valid) continue;
      if constexpr (kF32Out) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.o) + row_index * D + cb * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__uint_as_float(orr[4 * i]) * inv_l,
                               __uint_as_float(orr[4 * i + 1]) * inv_l,
                               __uint_as_float(orr[4 * i + 2]) * inv_l,
                               __uint_as_float(orr[4 * i + 3]) * inv_l);
      } else {
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(orr[2 * i]) * inv_l,
                                                   __uint_as_float(orr[2 * i + 1]) * inv_l);
          packed[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) + row_index * D +
                                               cb * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
      }
    }
    if (row_valid) p.lse[row_index] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kF32Out>
cudaError_t launch_typed(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const AttnParams &p, cudaStream_t stream) {
  auto kernel = attn_fwd_kernel<D, kF32Out>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(p.B * p.Hq), static_cast<unsigned>(p.n_qblocks));
  kernel<<<grid, kThreads, Cfg<D>::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(int D, bool f32_out, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const AttnParams &p, cudaStream_t stream) {
  if (D == 128) return f32_out ? launch_typed<128, true>(tq, tk, tv, p, stream)
                               : launch_typed<128, false>(tq, tk, tv, p, stream);
  return f32_out ? launch_typed<64, true>(tq, tk, tv, p, stream)
                 : launch_typed<64, false>(tq, tk, tv, p, stream);
}

cudaError_t read_and_clear_device_error(int *code) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace seqattn
