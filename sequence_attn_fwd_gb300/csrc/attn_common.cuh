// Pieces shared by the attention kernels: tile counting, the row maximum,
// the exponent pass, and the softmax + epilogue role of one query row.
#pragma once
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace seqattn {
namespace detail {

constexpr int kRowsPerTile = 128;  // MMA M and KV tile length
constexpr int kColBlockBytes = 128 * 128;  // 128 rows x 128 bytes (64 bf16) swizzle block
constexpr float kLn2 = 0.693147180559945309f;
// A row's P is formed against a lazily updated reference; the reference moves
// (and O is rescaled) only when the tile's P would sum to more than 2^8,
// which keeps every P at or below 2^8.
constexpr float kRescaleSum = 256.0f;

// The whole of a single problem as one block.
__host__ __device__ __forceinline__ BlockDesc whole_problem(const AttnParams &p) {
  return {0, 0, 0, p.q_off, p.kv_off, p.Sq, p.Skv, 0};
}

// Per-tile number of KV tiles to visit (0 when the tile has no valid row or
// none of its rows sees any key); first_row is the tile's first row within
// the block.
__device__ __forceinline__ int kv_tiles_for(const BlockDesc &b, int causal, int first_row) {
  const int n_all = (b.Skv + kRowsPerTile - 1) / kRowsPerTile;
  if (first_row >= b.Sq || n_all == 0) return 0;
  if (!causal) return n_all;
  const int last_row = min(first_row + kRowsPerTile - 1, b.Sq - 1);
  const long long max_key = b.q_pos + last_row - b.kv_pos;  // largest visible key index
  if (max_key < 0) return 0;
  const long long n = max_key / kRowsPerTile + 1;
  return n < n_all ? static_cast<int>(n) : n_all;
}
__device__ __forceinline__ int kv_tiles_for(const AttnParams &p, int first_row) {
  return kv_tiles_for(whole_problem(p), p.causal, first_row);
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

// 2^x for a pair of floats on the FMA pipe, offloading the MUFU unit (whose
// ex2 rate, 16 results per clock per SM, otherwise bounds the softmax):
// Cody-Waite style range reduction x = j + f with j = rint(x), found by adding
// and subtracting 1.5 * 2^23 (round-to-nearest), and f in [-1/2, 1/2]; 2^f by
// a degree-3 polynomial with p(0) = 1 whose other coefficients are the fit
// of least maximum relative error on [-1/2, 1/2] (a linear program over a
// uniform grid of 20,001 points, rounded to fp32; tests/test_exp2_fit.py
// re-runs it): 1.0e-4 in fp32 Horner form, far below the bf16 rounding of P;
// 2^j enters by adding j to the exponent field (the low bits of 1.5*2^23 + j,
// shifted by 23, are j << 23). x is clamped at -127 first: then every result
// is a non-negative float, and x = -inf gives +0 exactly (j = -127, f = 0,
// p = 1). Valid for x <= 127.
constexpr float kExp2C1 = 0x1.62f5fap-1f;
constexpr float kExp2C2 = 0x1.f00c4cp-3f;
constexpr float kExp2C3 = 0x1.c2a216p-5f;
__device__ __forceinline__ uint64_t exp2_poly_x2(uint64_t x) {
  float x0, x1;
  f2_unpack(x, x0, x1);
  const uint64_t xc = f2_pack(fmaxf(x0, -127.f), fmaxf(x1, -127.f));
  const uint64_t magic = f2_pack(12582912.f, 12582912.f);  // 1.5 * 2^23
  const uint64_t t = f2_add(xc, magic);                      // 1.5 * 2^23 + j
  const uint64_t j = f2_add(t, f2_pack(-12582912.f, -12582912.f));
  const uint64_t f = f2_fma(j, f2_pack(-1.f, -1.f), xc);    // x - j, exact
  uint64_t p = f2_fma(f, f2_pack(kExp2C3, kExp2C3), f2_pack(kExp2C2, kExp2C2));
  p = f2_fma(p, f, f2_pack(kExp2C1, kExp2C1));
  p = f2_fma(p, f, f2_pack(1.f, 1.f));
  float p0, p1, t0, t1;
  f2_unpack(p, p0, p1);
  f2_unpack(t, t0, t1);
  return f2_pack(__uint_as_float(__float_as_uint(p0) + (__float_as_uint(t0) << 23)),
                 __uint_as_float(__float_as_uint(p1) + (__float_as_uint(t1) << 23)));
}

// Of every 8 pairs of a row's exponentials, the kernel's kPoly take
// exp2_poly_x2 and the rest the MUFU ex2 (GB300's MUFU does 32 ex2 per clock
// per SM, so the softmax is bound by instruction issue rather than by the
// MUFU). The launch picks none for bf16 output, for e4m3 inputs and for fp32
// partials of blocks longer than kPolyMaxKeys, where every polynomial adds
// issue slots, and kPolyPairsShort for fp32 partials of short blocks, whose
// kernel measured faster with them (short items, where the fp32 epilogue's
// registers compete with the row's).
constexpr int kPolyPairsShort = 2;
constexpr int kPolyMaxKeys = 2048;

__device__ __forceinline__ uint64_t exp2_pair(uint64_t x, bool poly) {
  if (poly) return exp2_poly_x2(x);
  float a, b;
  f2_unpack(x, a, b);
  return f2_pack(ex2_approx(a), ex2_approx(b));
}

// P = 2^(s * c2 - m_ref) for the 128 scores of a row, packed as bf16 pairs
// (element 2i in the low half) or, with kFp8, as e4m3 quads, returning the
// fp32 sum of the unrounded P; kPoly of every 8 pairs take exp2_poly_x2.
template <bool kFp8, int kPoly>
__device__ __forceinline__ float exp_row(const float *s, float c2, float m_ref, uint32_t *pk) {
  const uint64_t scale2 = f2_pack(c2, c2);
  const uint64_t neg_m2 = f2_pack(-m_ref, -m_ref);
  uint64_t sum_a = f2_pack(0.f, 0.f), sum_b = sum_a;
#pragma unroll
  for (int q = 0; q < 64; q += 2) {  // pairs q and q + 1: elements 2q .. 2q + 3
    const uint64_t pa = exp2_pair(f2_fma(f2_pack(s[2 * q], s[2 * q + 1]), scale2, neg_m2),
                                  (q % 8) < kPoly);
    const uint64_t pb = exp2_pair(f2_fma(f2_pack(s[2 * q + 2], s[2 * q + 3]), scale2, neg_m2),
                                  ((q + 1) % 8) < kPoly);
    sum_a = f2_add(sum_a, pa);
    sum_b = f2_add(sum_b, pb);
    float p0, p1, p2, p3;
    f2_unpack(pa, p0, p1);
    f2_unpack(pb, p2, p3);
    if constexpr (kFp8) {  // four e4m3 per 32-bit TMEM column, element 4i in the low byte
      pk[q / 2] = pack_e4m3x2(p0, p1) | (pack_e4m3x2(p2, p3) << 16);
    } else {
      __nv_bfloat162 h0 = __floats2bfloat162_rn(p0, p1);
      __nv_bfloat162 h1 = __floats2bfloat162_rn(p2, p3);
      pk[q] = *reinterpret_cast<uint32_t *>(&h0);
      pk[q + 1] = *reinterpret_cast<uint32_t *>(&h1);
    }
  }
  float a0, a1, b0, b1;
  f2_unpack(sum_a, a0, a1);
  f2_unpack(sum_b, b0, b1);
  return (a0 + a1) + (b0 + b1);
}


// A block of query rows none of which sees a key: lse = -inf and, unless the
// caller asked to skip them, O = 0. The rows of one head are contiguous in
// memory, so the zero fill is one coalesced run of 16-byte stores by the
// `nthreads` threads taking part (tid = 0 .. nthreads - 1).
template <int D, bool kF32Out>
__device__ __forceinline__ void write_empty_rows(const AttnParams &p, const BlockDesc &blk, int bh,
                                                 int row_begin, int nrows, int tid, int nthreads) {
  const int rows = min(nrows, blk.Sq - row_begin);
  if (rows <= 0) return;
  const size_t base = static_cast<size_t>(bh) * p.o_rows + blk.o_row + row_begin;
  for (int i = tid; i < rows; i += nthreads) p.lse[base + i] = -INFINITY;
  if (p.skip_empty) return;
  const size_t n16 = static_cast<size_t>(rows) * D * (kF32Out ? 4 : 2) / 16;
  uint4 *dst = reinterpret_cast<uint4 *>(static_cast<char *>(p.o) + base * D * (kF32Out ? 4 : 2));
  for (size_t i = tid; i < n16; i += nthreads) dst[i] = make_uint4(0u, 0u, 0u, 0u);
}

// How a warpgroup's epilogue writes its 128-row O tile. With a tensor map the
// tile leaves through shared memory: each thread puts its row's 128-byte slice
// of a column chunk into its warp's quarter of a 128-byte-swizzled staging
// buffer (conflict-free), and lane 0 of the warp stores that quarter (32 rows)
// with TMA, so global writes are whole lines instead of one 16-byte piece of
// 32 different rows per warp store. Without a map each thread stores its own
// row.
struct EpilogueStore {
  const CUtensorMap *map;  // O as [heads][rows][D], box 128 bytes x 32 rows x 1, 128-byte swizzle
  uint32_t stage;          // shared address of this warpgroup's 16 KB staging buffer (1024-byte aligned)
  int named_bar;           // barrier id private to the warpgroup (128 threads)
  int head;                // third map coordinate, b * Hq + hq
};

// Softmax and epilogue for one query row (one thread; a warp covers 32 rows
// of a 128-row tile, TMEM lane = tile row).
//   s_addr / o_addr   TMEM address of this row's S (later P) and O columns
//   n                 KV tiles this tile visits; bar_sfull / bar_ofull are the
//                     mbarriers the MMA issuer commits when S(j) / the final O
//                     are ready; signal_p() tells it P(j) is in TMEM (called by
//                     every thread after its tcgen05 stores are fenced).
//   step_base         S(j) completes phase step_base + j of bar_sfull (a CTA
//                     that works through several tiles keeps counting)
//   ofull_parity      parity of the bar_ofull phase that marks this tile's O
// Returns false if the pipeline was aborted.
template <int D, bool kF32Out, typename SignalP, bool kFp8, int kPoly>
__device__ __forceinline__ bool softmax_row(const AttnParams &p, const BlockDesc &blk, int row,
                                            int tile_first_row, int n,
                                            uint32_t s_addr, uint32_t o_addr, uint32_t bar_sfull,
                                            uint32_t bar_ofull, int step_base,
                                            uint32_t ofull_parity, size_t row_index,
                                            volatile int *abort_flag, int *err,
                                            const EpilogueStore &store, SignalP signal_p) {
    const long long qpos = blk.q_pos + row;
    const long long tile_first_q = blk.q_pos + tile_first_row;
    const float c2 = p.scale_log2;
    float m = -INFINITY;  // running max of scale*log2(e)*s (the reference for P)
    float l = 0.f;        // running sum of P relative to m
    bool ok = true;

    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar_sfull, static_cast<uint32_t>(step_base + j) & 1u, abort_flag, err));
      if (!ok) break;
      tc_fence_after();
      const int kv0 = j * kRowsPerTile;
      const bool tail = kv0 + kRowsPerTile > blk.Skv;
      const bool diag = p.causal && (blk.kv_pos + kv0 + kRowsPerTile - 1 > tile_first_q);
      int last = 127;  // last visible column of this row in the tile
      if (tail || diag) {
        long long lim = static_cast<long long>(blk.Skv) - kv0 - 1;
        if (p.causal) {
          const long long c_lim = qpos - blk.kv_pos - kv0;
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
      uint32_t sr[128];
      load_scores(sr);
      float rowsum;
      if (j == 0) {
        // no reference yet: the tile maximum first, then the exponentials
        m = row_max(reinterpret_cast<const float *>(sr)) * c2;
        rowsum = exp_row<kFp8, kPoly>(reinterpret_cast<const float *>(sr), c2,
                                      (m == -INFINITY) ? 0.f : m, pk);
      } else {
        // Exponentiate against the current reference. A row sum of at most
        // 2^8 bounds every P by 2^8 (the bf16 P and the fp32 sums stay in
        // range); only otherwise (rare after the first tiles), or while the
        // row has no reference yet, is the tile maximum found, O rescaled and
        // the pass redone.
        rowsum = exp_row<kFp8, kPoly>(reinterpret_cast<const float *>(sr), c2,
                                      (m == -INFINITY) ? 0.f : m, pk);
        const bool big = !(rowsum <= kRescaleSum) || (m == -INFINITY && rowsum > 0.f);
        if (__any_sync(0xffffffffu, big)) {
          // the tile maximum, 32 columns at a time (few live registers)
          float mx = -INFINITY;
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            uint32_t x[32];
            tmem_ld32(s_addr + 32 * cb, x);
            tmem_ld_wait(x);
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (!(tail || diag) || 32 * cb + c <= last) mx = fmaxf(mx, __uint_as_float(x[c]));
          }
          const float m_new = fmaxf(m, mx * c2);
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
          load_scores(sr);
          rowsum = exp_row<kFp8, kPoly>(reinterpret_cast<const float *>(sr), c2,
                                        (m == -INFINITY) ? 0.f : m, pk);
        }
      }
      l += rowsum;
      tmem_st32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      if constexpr (!kFp8) tmem_st32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      tmem_st_wait();
      tc_fence_before();
      signal_p();
    }

    // ------------------------------------------------------------ epilogue
    bool have_o = false;
    if (ok && n > 0) {
      have_o = __all_sync(0xffffffffu, mbar_wait(bar_ofull, ofull_parity, abort_flag, err));
      tc_fence_after();
    }
    const bool row_valid = row < blk.Sq;
    const bool write_o = row_valid && !(p.skip_empty && l == 0.f);
    float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    if constexpr (kFp8) inv_l *= p.o_scale;  // dequantisation of V
    bool via_tma = store.map != nullptr;
    if (via_tma) {
      // Whole-box stores need the final O on every row, no row that must stay
      // unwritten (skip_empty rows before the chunk's first key), and a box
      // that ends inside the block or at the end of the tensor (the map clips
      // there; elsewhere the box would spill into the next block's rows).
      const bool keep_rows = p.skip_empty && p.causal && (blk.q_pos + tile_first_row < blk.kv_pos);
      const bool box_fits = tile_first_row < blk.Sq &&
                            (tile_first_row + kRowsPerTile <= blk.Sq || blk.o_row + blk.Sq == p.o_rows);
      via_tma = named_bar_and(store.named_bar, 128, have_o) && !keep_rows && box_fits;
    }
    if (via_tma) {
      // Each warp stores its own 32 rows from its own quarter of the
      // warpgroup's staging buffer (4 KB), so only warp-level syncs are needed
      // between writing the buffer and the TMA store that reads it.
      constexpr int kChunkCols = kF32Out ? 32 : 64;  // 128 bytes of a row
      constexpr int kChunks = D / kChunkCols;
      const bool wleader = (threadIdx.x & 31) == 0;
      const uint32_t row_in_tile = static_cast<uint32_t>(row - tile_first_row);
      const uint32_t warp_row0 = row_in_tile & ~31u;
      const uint32_t swz = row_in_tile & 7u;
      const uint32_t wbuf = store.stage + warp_row0 * 128u;
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c) {
        uint32_t v[32];
        if constexpr (kF32Out) {
          tmem_ld32(o_addr + 32 * c, v);
          tmem_ld_wait(v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * inv_l);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t orr[32];
            tmem_ld32(o_addr + 64 * c + 32 * h, orr);
            tmem_ld_wait(orr);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(orr[2 * i]) * inv_l,
                                                        __uint_as_float(orr[2 * i + 1]) * inv_l);
              v[16 * h + i] = *reinterpret_cast<uint32_t *>(&b2);
            }
          }
        }
        // the previous box this warp stored from its quarter (the previous
        // chunk's, or the last one of its previous tile) must have been read
        // out of it; waiting here rather than after each tile's last store
        // keeps that read off the path to the next tile's softmax
        if (wleader) bulk_wait_group_read<0>();
        __syncwarp();
        const uint32_t dst = wbuf + (row_in_tile & 31u) * 128u;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          st_shared_v4(dst + ((static_cast<uint32_t>(k) ^ swz) << 4), v[4 * k], v[4 * k + 1],
                       v[4 * k + 2], v[4 * k + 3]);
        fence_proxy_async_shared();
        __syncwarp();
        if (wleader) {
          // O is written once and not read back by this kernel: let it leave
          // L2 ahead of the K and V tiles other items still read
          tma_store_3d_hint(store.map, wbuf, c * kChunkCols,
                            static_cast<int>(blk.o_row + tile_first_row + warp_row0), store.head,
                            l2_policy_evict_first());
          bulk_commit_group();
        }
      }
      // The last stores may still be reading the buffer: the next tile's first
      // chunk waits for them, and the caller waits for every store before the
      // CTA exits.
      if (row_valid) p.lse[row_index] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
      return true;  // every thread of the warpgroup had the final O
    }
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
      if (!write_o) continue;
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
    const bool done = ok && (n == 0 || have_o);
    // a caller that goes on to another tile needs the same answer on every
    // thread of the warpgroup
    return store.map != nullptr ? named_bar_and(store.named_bar, 128, done) : done;
}

}  // namespace detail
}  // namespace seqattn
