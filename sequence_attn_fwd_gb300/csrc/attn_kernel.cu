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
// How (one CTA = 256 query rows of one (batch, head), 352 threads):
//   warp 9      TMA producer: both Q tiles once, then K_j, V_j into a ring of
//               shared-memory slots (128-byte swizzle, 3-D tensor maps so
//               rows past the end of a head read as zero).
//   warps 8, 10 MMA issuers, one thread each, warp 8 for query tile 0 and
//               warp 10 for tile 1: S_t = Q_t K_j^T into TMEM (SS form) and
//               O_t += P_t V_j with P_t read from TMEM (TS form). Their bursts
//               alternate through a shared turn counter (tile 0, tile 1, tile
//               0, ...), so the tensor pipe works on one tile while the other
//               tile's softmax runs, and each issuer's barrier waits and
//               commits overlap the other's MMAs: a lone issuer spent about
//               40 % of every KV step in those, with the tensor pipe idle.
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
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include <type_traits>

#include "attn_common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace seqattn {

__device__ int g_device_error;  // set by a timed-out wait; read and cleared by the host

namespace {

using namespace detail;

constexpr int kThreads = 352;
constexpr int kMmaWarp = 8;   // MMA issuer of query tile 0 (also allocates TMEM)
constexpr int kTmaWarp = 9;
constexpr int kMmaWarp1 = 10;  // MMA issuer of query tile 1

template <int D, bool kFp8 = false>
struct Cfg {
  static constexpr int kElemBytes = kFp8 ? 1 : 2;              // bf16 or e4m3 operands
  static constexpr int kColBlocks = D * kElemBytes / 128;        // 128-byte column blocks of a row
  static constexpr int kColBlockElems = 128 / kElemBytes;
  static constexpr int kTileBytes = kRowsPerTile * D * kElemBytes;
  static constexpr int kStages = 131072 / kTileBytes;            // a 128 KB K/V ring
  static constexpr int kSmemQ = 2 * kTileBytes;
  static constexpr int kSmemRing = kStages * kTileBytes;
  static constexpr int kStageBytes = 16384;  // epilogue staging box of one softmax warpgroup
  static constexpr int kSmemStage = 2 * kStageBytes;
  // barriers: q_full, q_empty, full[S], empty[S], s_full[2], p_full[2], o_full[2], mma_done
  static constexpr int kNumBarriers = 2 + 2 * kStages + 7;
  static constexpr int kSmemBytes =
      1024 + kSmemQ + kSmemRing + kSmemStage + 8 * kNumBarriers + 16;
};
static_assert(Cfg<128>::kSmemBytes <= 232448 && Cfg<64>::kSmemBytes <= 232448 &&
                  Cfg<128, true>::kSmemBytes <= 232448,
              "shared memory per CTA");

// Work item k of a launch: 256 query rows of one (batch, head) of one block of
// the launch's table. Within a block, items are numbered with the head
// fastest; causal launches number the longest query rows (most KV tiles) first.
struct Item {
  int blk;   // block of the table
  int bh;    // b * Hq + hq
  int row0;  // first query row within the block
};
// The i-th item of this CTA. Items are dealt in rounds of gridDim.x, one per
// CTA, in alternating direction, so that with causal cost falling along the
// numbering every CTA's total stays within one item of every other's.
__device__ __forceinline__ long long item_index(long long i) {
  const long long G = gridDim.x;
  return i * G + ((i & 1) ? (G - 1 - blockIdx.x) : blockIdx.x);
}
// A single problem (attn_fwd, attn_partial): its one block is built from p, so
// the geometry folds into parameter reads.
struct SingleProblem {
  int unused;
};

__device__ __forceinline__ long long n_items_of(const AttnParams &, const BlockTable &tbl) {
  return tbl.item_start[tbl.n];
}
__device__ __forceinline__ BlockDesc block_of(const AttnParams &p, const SingleProblem &, int) {
  return whole_problem(p);
}
__device__ __forceinline__ BlockDesc block_of(const AttnParams &, const BlockTable &tbl, int blk) {
  return tbl.b[blk];
}
// Single problems: the heads come in chunks of p.heads_per_chunk (whole GQA
// groups, sized on the host so that a chunk's K and V stay in L2), and within
// a chunk the items are numbered with the head fastest, so that the query
// heads of a KV head run side by side and every K / V tile is read from DRAM
// about once. Every chunk but the last is padded with empty items to whole
// rounds of gridDim.x, so that a chunk's light last items and the next
// chunk's heavy first ones never share a round (the padding items have no
// rows: every role skips them).
__device__ __forceinline__ long long chunk_items(const AttnParams &p, long long heads, long long &hc) {
  hc = p.heads_per_chunk > 0 && p.heads_per_chunk < heads ? p.heads_per_chunk : heads;
  const long long G = gridDim.x;
  return (hc * p.n_qblocks + G - 1) / G * G;  // a full chunk's items with its padding
}
__device__ __forceinline__ long long n_items_of(const AttnParams &p, const SingleProblem &) {
  const long long heads = static_cast<long long>(p.B) * p.Hq;
  long long hc;
  const long long per_chunk = chunk_items(p, heads, hc);
  const long long n_chunks = (heads + hc - 1) / hc;
  return (n_chunks - 1) * per_chunk + (heads - (n_chunks - 1) * hc) * p.n_qblocks;
}
__device__ __forceinline__ Item item_of(const AttnParams &p, const SingleProblem &, long long k, int &) {
  const long long heads = static_cast<long long>(p.B) * p.Hq;
  long long hc;
  const long long per_chunk = chunk_items(p, heads, hc);
  const long long c = k / per_chunk;
  const long long h0 = c * hc;
  const long long hn = heads - h0 < hc ? heads - h0 : hc;  // the last chunk may be short
  const long long r = k - c * per_chunk;
  if (r >= hn * p.n_qblocks) return {0, 0, p.n_qblocks * 2 * kRowsPerTile};  // padding: no rows
  const int qi = static_cast<int>(r / hn);
  const int qblock = p.causal ? p.n_qblocks - 1 - qi : qi;
  return {0, static_cast<int>(h0 + r % hn), qblock * 2 * kRowsPerTile};
}
// `cur` is the caller's cursor: the block of its previous item. A CTA's items
// come in increasing order, so the block of item k (the last one with
// item_start <= k) is found by scanning on from there, usually in no step.
__device__ __forceinline__ Item item_of(const AttnParams &p, const BlockTable &tbl, long long k, int &cur) {
  int lo = cur;
  while (lo + 1 < tbl.n && tbl.item_start[lo + 1] <= k) ++lo;
  cur = lo;
  const long long local = k - tbl.item_start[lo];
  const long long heads = static_cast<long long>(p.B) * p.Hq;
  const int qi = static_cast<int>(local / heads);
  const int n_qb = (tbl.b[lo].Sq + 2 * kRowsPerTile - 1) / (2 * kRowsPerTile);
  const int qblock = p.causal ? n_qb - 1 - qi : qi;
  return {lo, static_cast<int>(local % heads), qblock * 2 * kRowsPerTile};
}
// Blocks sharing their query rows: items number 256-row query blocks of the
// shared rows with the head fastest, longest first when causal; every block
// of the table is a segment of each item.
__device__ __forceinline__ long long n_items_of(const AttnParams &p, const SegTable &tbl) {
  return static_cast<long long>(p.B) * p.Hq * ((tbl.b[0].Sq + 2 * kRowsPerTile - 1) / (2 * kRowsPerTile));
}
__device__ __forceinline__ Item item_of(const AttnParams &p, const SegTable &tbl, long long k, int &) {
  const long long heads = static_cast<long long>(p.B) * p.Hq;
  const int qi = static_cast<int>(k / heads);
  const int n_qb = (tbl.b[0].Sq + 2 * kRowsPerTile - 1) / (2 * kRowsPerTile);
  const int qblock = p.causal ? n_qb - 1 - qi : qi;
  return {0, static_cast<int>(k % heads), qblock * 2 * kRowsPerTile};
}
// Segments of an item: one (its block) except with a SegTable.
__device__ __forceinline__ int n_segs_of(const SingleProblem &) { return 1; }
__device__ __forceinline__ int n_segs_of(const BlockTable &) { return 1; }
__device__ __forceinline__ int n_segs_of(const SegTable &tbl) { return tbl.n; }
__device__ __forceinline__ BlockDesc seg_block(const AttnParams &p, const SingleProblem &t, const Item &, int) {
  return block_of(p, t, 0);
}
__device__ __forceinline__ BlockDesc seg_block(const AttnParams &p, const BlockTable &t, const Item &it, int) {
  return block_of(p, t, it.blk);
}
__device__ __forceinline__ BlockDesc seg_block(const AttnParams &, const SegTable &t, const Item &, int s) {
  return t.b[s];
}

// kFp8: Q, K in e4m3 with K-major tiles, V given transposed ([heads][D][keys],
// so its tiles are K-major too), P rounded to e4m3 in TMEM (one instantiation:
// D = 128, bf16 output, single problem).
template <int D, bool kF32Out, typename Table, bool kFp8, int kPoly>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, const AttnParams p,
                    const __grid_constant__ Table tbl) {
  using C = Cfg<D, kFp8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem;                          // [tile][col block][128 rows][128 B]
  uint8_t *sRing = smem + C::kSmemQ;           // [slot][col block][128 rows][128 B]
  uint8_t *sStage = sRing + C::kSmemRing;      // [warpgroup][16 KB]
  uint64_t *bars = reinterpret_cast<uint64_t *>(sStage + C::kSmemStage);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBarriers);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *turn = reinterpret_cast<volatile int *>(tmem_slot + 2);  // next MMA burst slot

  const uint32_t bar0 = smem_addr(bars);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  const int kBarQFull = 0, kBarQEmpty = 1, kBarFull = 2, kBarEmpty = 2 + C::kStages,
            kBarSFull = 2 + 2 * C::kStages, kBarPFull = kBarSFull + 2, kBarOFull = kBarPFull + 2,
            kBarMmaDone = kBarOFull + 2;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int *err = &g_device_error;
  const long long n_items = n_items_of(p, tbl);

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 2);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 2);  // released by both issuers
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPFull + t), 4);  // one arrival per softmax warp
      mbar_init(bar(kBarOFull + t), 1);
    }
    mbar_init(bar(kBarMmaDone), 2);
    // A timeout recorded by any earlier CTA or launch (and not yet cleared by
    // the host) makes this CTA skip its work: its rows come out as O = 0,
    // lse = -inf, and the host learns of it from the device error query.
    *abort_flag = *reinterpret_cast<volatile int *>(err) != kErrNone;
    *turn = 0;
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
  // Single problems and block tables take the loops without segments (one a
  // work item); tables of blocks sharing their query rows the segmented ones.
  constexpr bool kSeg = std::is_same<Table, SegTable>::value;
  static_assert(!(kSeg && kFp8), "segmented items load V in the bf16 layout only");
  const int n_segs = n_segs_of(tbl);
  // KV tiles query tile t of an item visits in segment sg (0: none of its rows sees a key)
  auto tiles = [&](const Item &it, int sg, int t) -> int {
    return skip ? 0 : kv_tiles_for(seg_block(p, tbl, it, sg), p.causal, it.row0 + t * kRowsPerTile);
  };
  auto seg_max = [&](const Item &it, int sg) { return max(tiles(it, sg, 0), tiles(it, sg, 1)); };
  // TMEM column of S_t / P_t and of O_t for query tile t
  auto tS = [&](int t) -> uint32_t { return tmem + 128u * static_cast<uint32_t>(t); };
  auto tO = [&](int t) -> uint32_t { return tmem + 256u + 128u * static_cast<uint32_t>(t); };

  // The CTA works through items item_index(0), item_index(1), ...; each role
  // walks the same sequence, and within an item its segments (one, except
  // with a SegTable), and skips those with no visible key. Barrier phases run
  // on across items: the Q buffer by loaded item, the K/V ring by ring
  // position, S/P by KV step of each query tile, O by segment of each query
  // tile.
  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !skip) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      // K and V are read again by every query block and head of their group:
      // kept in L2 ahead of Q, which each item reads once
      const uint64_t pol_keep = l2_policy_evict_last(), pol_stream = l2_policy_evict_first();
      int c = 0;   // K_0, V_0, K_1, V_1, ... of every item, in the order the MMA issuer consumes them
      int nq = 0;  // Q tile pairs loaded
      bool ok = true;
      if constexpr (!kSeg) {
        int cur_blk = 0;  // block of the previous item (block tables)
        for (long long i = 0, k = item_index(0); k < n_items && ok; k = item_index(++i)) {
          const Item it = item_of(p, tbl, k, cur_blk);
          const int n_max = seg_max(it, 0);
          if (n_max == 0) continue;
          // the previous item's S MMAs must be done reading the Q buffer
          if (nq > 0 && !mbar_wait(bar(kBarQEmpty), (nq - 1) & 1, abort_flag, err)) break;
          mbar_arrive_expect_tx(bar(kBarQFull), 2 * C::kTileBytes);
          const BlockDesc blk = block_of(p, tbl, it.blk);
          const int q_row = static_cast<int>(blk.q_row) + it.row0;
          const int kv_row = static_cast<int>(blk.kv_row);
          for (int t = 0; t < 2; ++t)
            for (int cb = 0; cb < C::kColBlocks; ++cb)
              tma_load_3d_hint(smem_addr(sQ + (t * C::kColBlocks + cb) * kColBlockBytes), &tm_q,
                               bar(kBarQFull), cb * C::kColBlockElems, q_row + t * kRowsPerTile, it.bh,
                               pol_stream);
          ++nq;
          const int b = it.bh / p.Hq, hq = it.bh % p.Hq;
          const int kv_head = b * p.Hkv + hq / (p.Hq / p.Hkv);
          for (int j = 0; j < n_max && ok; ++j) {
            for (int which = 0; which < 2; ++which, ++c) {
              const int slot = c % C::kStages;
              if (c >= C::kStages &&
                  !mbar_wait(bar(kBarEmpty + slot), ((c / C::kStages) - 1) & 1, abort_flag, err)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(bar(kBarFull + slot), C::kTileBytes);
              if (kFp8 && which) {
                // V^T tile j: the 128 keys of the tile along x, all D rows (one box at D = 128)
                tma_load_3d_hint(smem_addr(sRing + slot * C::kTileBytes), &tm_v, bar(kBarFull + slot),
                                 kv_row + j * kRowsPerTile, 0, kv_head, pol_keep);
              } else {
                const CUtensorMap *map = which ? &tm_v : &tm_k;
                for (int cb = 0; cb < C::kColBlocks; ++cb)
                  tma_load_3d_hint(smem_addr(sRing + (slot * C::kColBlocks + cb) * kColBlockBytes), map,
                                   bar(kBarFull + slot), cb * C::kColBlockElems, kv_row + j * kRowsPerTile,
                                   kv_head, pol_keep);
              }
            }
          }
        }
      } else {
        int cur_blk = 0;  // block of the previous item (block tables)
        for (long long i = 0, k = item_index(0); k < n_items && ok; k = item_index(++i)) {
          const Item it = item_of(p, tbl, k, cur_blk);
          bool any = false;
          for (int sg = 0; sg < n_segs && !any; ++sg) any = seg_max(it, sg) > 0;
          if (!any) continue;
          // the previous item's S MMAs must be done reading the Q buffer
          if (nq > 0 && !mbar_wait(bar(kBarQEmpty), (nq - 1) & 1, abort_flag, err)) break;
          mbar_arrive_expect_tx(bar(kBarQFull), 2 * C::kTileBytes);
          const int q_row = static_cast<int>(seg_block(p, tbl, it, 0).q_row) + it.row0;
          for (int t = 0; t < 2; ++t)
            for (int cb = 0; cb < C::kColBlocks; ++cb)
              tma_load_3d_hint(smem_addr(sQ + (t * C::kColBlocks + cb) * kColBlockBytes), &tm_q,
                               bar(kBarQFull), cb * C::kColBlockElems, q_row + t * kRowsPerTile, it.bh,
                               pol_stream);
          ++nq;
          const int b = it.bh / p.Hq, hq = it.bh % p.Hq;
          const int kv_head = b * p.Hkv + hq / (p.Hq / p.Hkv);
          for (int sg = 0; sg < n_segs && ok; ++sg) {  // each segment's K/V tiles in turn
            const int n_max = seg_max(it, sg);
            const int kv_row = static_cast<int>(seg_block(p, tbl, it, sg).kv_row);
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
                  tma_load_3d_hint(smem_addr(sRing + (slot * C::kColBlocks + cb) * kColBlockBytes), map,
                                   bar(kBarFull + slot), cb * C::kColBlockElems, kv_row + j * kRowsPerTile,
                                   kv_head, pol_keep);
              }
            }
          }
        }
      }
      // Every copy issued must have landed before the CTA may exit (only the
      // last Q load and the last ring fills can still be in flight).
      if (nq > 0) mbar_drain(bar(kBarQFull), (nq - 1) & 1, err);
      for (int i = max(0, c - C::kStages); i < c; ++i)
        mbar_drain(bar(kBarFull + i % C::kStages), (i / C::kStages) & 1, err);
    }
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kMmaWarp1) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing thread per query tile t, so that one tile's barrier waits
    // and commits overlap the other tile's MMAs. Both consume every K/V ring
    // slot of an item (each releases it once: the empty barriers count two
    // arrivals); a tile that does not use a slot's tile waits for it to land
    // before releasing it, so that its release always counts toward the
    // phase the slot is in.
    const int t = (warp == kMmaWarp) ? 0 : 1;
    if (lane == 0 && !skip) {
      constexpr uint32_t idesc_s = kFp8 ? idesc_e4m3_f32(128, 128) : idesc_bf16_f32(128, 128, false);
      constexpr uint32_t idesc_o = kFp8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(128, D, true);
      constexpr int kKSteps = D * C::kElemBytes / 32;  // 32-byte K steps of S = Q K^T
      const uint32_t qt = smem_addr(sQ) + t * C::kTileBytes;
      const uint32_t ring_base = smem_addr(sRing);
      const uint32_t s_col = tS(t), o_col = tO(t);
      int c = 0;             // ring position of the item's K_0
      int nq = 0;            // Q tile pairs consumed
      int g = 0;             // KV steps done by this tile over earlier items
      bool ok = true;
      int base = 0;          // burst slots of earlier items
      if constexpr (!kSeg) {
        int cur_blk = 0;  // block of the previous item (block tables)
        for (long long i = 0, k = item_index(0); k < n_items && ok; k = item_index(++i)) {
          const Item it = item_of(p, tbl, k, cur_blk);
          const int nt = tiles(it, 0, t);
          const int n_max = seg_max(it, 0);
          if (n_max == 0) continue;
          if (!mbar_wait(bar(kBarQFull), nq & 1, abort_flag, err)) break;
          ++nq;
          if (nt == 0) mma_commit(bar(kBarQEmpty));  // this tile reads nothing of Q
          // Burst slots alternate between the tiles: (step j, tile t) is slot
          // base + 2 j + t. A tile waits for its data before its slot comes up
          // and makes its commits after handing the slot on, so that its
          // waits and commits overlap the other tile's MMAs.
          for (int j = 0; ok && j <= n_max; ++j) {
            const int cK = c + 2 * j, cV = c + 2 * j - 1;  // ring positions of K_j and V_{j-1}
            const int sK = cK % C::kStages, sV = (cV + C::kStages) % C::kStages;
            const int cV2 = cK + 1, sV2 = cV2 % C::kStages;  // V_j
            const uint32_t k_base = ring_base + sK * C::kTileBytes;
            const uint32_t v_base = ring_base + sV * C::kTileBytes;
            const bool has_pv = j >= 1 && j - 1 < nt, has_s = j < nt, unused = !has_s && j < n_max;
            // the data first (usually there already), the softmax's P last
            if ((has_s || unused) && !mbar_wait(bar(kBarFull + sK), (cK / C::kStages) & 1, abort_flag, err)) {
              ok = false;
              break;
            }
            if (unused && !mbar_wait(bar(kBarFull + sV2), (cV2 / C::kStages) & 1, abort_flag, err)) {
              ok = false;
              break;
            }
            if (has_pv && (!mbar_wait(bar(kBarFull + sV), (cV / C::kStages) & 1, abort_flag, err) ||
                           !mbar_wait(bar(kBarPFull + t), (g + j - 1) & 1, abort_flag, err))) {
              ok = false;
              break;
            }
            const int slot = base + 2 * j + t;
            if (!wait_turn(turn, slot, abort_flag, err)) {
              ok = false;
              break;
            }
            if (has_pv) {
              // O_t += P_t V_{j-1}; P_t was written over S_t by the softmax
              // warps. For j = 1 this overwrites O_t: the warpgroup read the
              // previous item's O_t before it signalled this P.
              tc_fence_after();
              if constexpr (kFp8) {
#pragma unroll
                for (int kk = 0; kk < kRowsPerTile / 32; ++kk)
                  mma_ts_e4m3(o_col, s_col + kk * 8, sw128_desc(v_base + kk * 32, 16, 1024), idesc_o,
                              (j > 1 || kk > 0) ? 1u : 0u);
              } else {
                // descriptor start fields advance by 2048 / 16 per 16 keys
                const uint64_t vd = sw128_desc(v_base, kColBlockBytes, 1024);
                mma_ts(o_col, s_col, vd, idesc_o, j > 1 ? 1u : 0u);
#pragma unroll
                for (int kk = 1; kk < kRowsPerTile / 16; ++kk)
                  mma_ts(o_col, s_col + kk * 8, vd + static_cast<uint64_t>(kk * 128), idesc_o, 1u);
              }
            }
            if (has_s) {
              // S_t = Q_t K_j^T
              const uint64_t qd = sw128_desc(qt, 16, 1024), kd = sw128_desc(k_base, 16, 1024);
#pragma unroll
              for (int kk = 0; kk < kKSteps; ++kk) {
                const uint64_t off = static_cast<uint64_t>(((kk / 4) * kColBlockBytes + (kk % 4) * 32) >> 4);
                if constexpr (kFp8)
                  mma_ss_e4m3(s_col, qd + off, kd + off, idesc_s, kk > 0 ? 1u : 0u);
                else
                  mma_ss(s_col, qd + off, kd + off, idesc_s, kk > 0 ? 1u : 0u);
              }
            }
            *turn = slot + 1;
            if (has_s) mma_commit(bar(kBarSFull + t));
            if (has_pv) {
              if (j - 1 == nt - 1) mma_commit(bar(kBarOFull + t));
              mma_commit(bar(kBarEmpty + sV));  // this tile's last use of V_{j-1}
            }
            if (has_s) {
              mma_commit(bar(kBarEmpty + sK));  // this tile's use of K_j
              if (j == nt - 1) mma_commit(bar(kBarQEmpty));  // this tile's last read of Q
            }
            if (unused) {  // K_j and V_j are not visible to this tile
              mma_commit(bar(kBarEmpty + sK));
              mma_commit(bar(kBarEmpty + sV2));
            }
          }
          c += 2 * n_max;
          g += nt;
          base += 2 * (n_max + 1);
        }
      } else {
        int cur_blk = 0;  // block of the previous item (block tables)
        for (long long i = 0, k = item_index(0); k < n_items && ok; k = item_index(++i)) {
          const Item it = item_of(p, tbl, k, cur_blk);
          bool any = false;
          int last_sg = -1;  // this tile's last segment with a KV tile: its last S reads Q
          for (int sg = 0; sg < n_segs; ++sg) {
            any |= seg_max(it, sg) > 0;
            if (tiles(it, sg, t) > 0) last_sg = sg;
          }
          if (!any) continue;
          if (!mbar_wait(bar(kBarQFull), nq & 1, abort_flag, err)) break;
          ++nq;
          if (last_sg < 0) mma_commit(bar(kBarQEmpty));  // this tile reads nothing of Q
          for (int sg = 0; sg < n_segs && ok; ++sg) {  // the segments in turn, Q staying
            const int nt = tiles(it, sg, t);
            const int n_max = seg_max(it, sg);
            if (n_max == 0) continue;
            // Burst slots alternate between the tiles: (step j, tile t) is slot
            // base + 2 j + t. A tile waits for its data before its slot comes up
            // and makes its commits after handing the slot on, so that its
            // waits and commits overlap the other tile's MMAs.
            for (int j = 0; ok && j <= n_max; ++j) {
              const int cK = c + 2 * j, cV = c + 2 * j - 1;  // ring positions of K_j and V_{j-1}
              const int sK = cK % C::kStages, sV = (cV + C::kStages) % C::kStages;
              const int cV2 = cK + 1, sV2 = cV2 % C::kStages;  // V_j
              const uint32_t k_base = ring_base + sK * C::kTileBytes;
              const uint32_t v_base = ring_base + sV * C::kTileBytes;
              const bool has_pv = j >= 1 && j - 1 < nt, has_s = j < nt, unused = !has_s && j < n_max;
              // the data first (usually there already), the softmax's P last
              if ((has_s || unused) && !mbar_wait(bar(kBarFull + sK), (cK / C::kStages) & 1, abort_flag, err)) {
                ok = false;
                break;
              }
              if (unused && !mbar_wait(bar(kBarFull + sV2), (cV2 / C::kStages) & 1, abort_flag, err)) {
                ok = false;
                break;
              }
              if (has_pv && (!mbar_wait(bar(kBarFull + sV), (cV / C::kStages) & 1, abort_flag, err) ||
                             !mbar_wait(bar(kBarPFull + t), (g + j - 1) & 1, abort_flag, err))) {
                ok = false;
                break;
              }
              const int slot = base + 2 * j + t;
              if (!wait_turn(turn, slot, abort_flag, err)) {
                ok = false;
                break;
              }
              if (has_pv) {
                // O_t += P_t V_{j-1}; P_t was written over S_t by the softmax
                // warps. For j = 1 this overwrites O_t: the warpgroup read the
                // previous segment's O_t before it signalled this P.
                tc_fence_after();
                if constexpr (kFp8) {
#pragma unroll
                  for (int kk = 0; kk < kRowsPerTile / 32; ++kk)
                    mma_ts_e4m3(o_col, s_col + kk * 8, sw128_desc(v_base + kk * 32, 16, 1024), idesc_o,
                                (j > 1 || kk > 0) ? 1u : 0u);
                } else {
                  // descriptor start fields advance by 2048 / 16 per 16 keys
                  const uint64_t vd = sw128_desc(v_base, kColBlockBytes, 1024);
                  mma_ts(o_col, s_col, vd, idesc_o, j > 1 ? 1u : 0u);
#pragma unroll
                  for (int kk = 1; kk < kRowsPerTile / 16; ++kk)
                    mma_ts(o_col, s_col + kk * 8, vd + static_cast<uint64_t>(kk * 128), idesc_o, 1u);
                }
              }
              if (has_s) {
                // S_t = Q_t K_j^T
                const uint64_t qd = sw128_desc(qt, 16, 1024), kd = sw128_desc(k_base, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kKSteps; ++kk) {
                  const uint64_t off = static_cast<uint64_t>(((kk / 4) * kColBlockBytes + (kk % 4) * 32) >> 4);
                  if constexpr (kFp8)
                    mma_ss_e4m3(s_col, qd + off, kd + off, idesc_s, kk > 0 ? 1u : 0u);
                  else
                    mma_ss(s_col, qd + off, kd + off, idesc_s, kk > 0 ? 1u : 0u);
                }
              }
              *turn = slot + 1;
              if (has_s) mma_commit(bar(kBarSFull + t));
              if (has_pv) {
                if (j - 1 == nt - 1) mma_commit(bar(kBarOFull + t));
                mma_commit(bar(kBarEmpty + sV));  // this tile's last use of V_{j-1}
              }
              if (has_s) {
                mma_commit(bar(kBarEmpty + sK));  // this tile's use of K_j
                if (j == nt - 1 && sg == last_sg) mma_commit(bar(kBarQEmpty));  // its last read of Q
              }
              if (unused) {  // K_j and V_j are not visible to this tile
                mma_commit(bar(kBarEmpty + sK));
                mma_commit(bar(kBarEmpty + sV2));
              }
            }
            c += 2 * n_max;
            g += nt;
            base += 2 * (n_max + 1);
          }
        }
      }
      // All MMAs issued here must be complete before TMEM is released.
      mma_commit(bar(kBarMmaDone));
      mbar_drain(bar(kBarMmaDone), 0, err);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax + epilogue
    const int t = warp >> 2;                         // query tile of this warpgroup
    const int row_in_tile = (warp & 3) * 32 + lane;  // TMEM lane = tile row
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t pfull = bar(kBarPFull + t);
    const uint32_t stage = smem_addr(sStage + t * C::kStageBytes);
    if constexpr (!kSeg) {
      int g = 0;       // KV steps of this tile over earlier items
      uint32_t u = 0;  // earlier items in which this tile visited a KV tile
      int cur_blk = 0;  // block of the previous item (block tables)
      for (long long i = 0, k = item_index(0); k < n_items; k = item_index(++i)) {
        const Item it = item_of(p, tbl, k, cur_blk);
        const BlockDesc blk = block_of(p, tbl, it.blk);
        const int out_head = blk.part * p.B * p.Hq + it.bh;  // head of O / lse written
        const int tile_first = it.row0 + t * kRowsPerTile;
        const int n = tiles(it, 0, t);
        if (n == 0) {
          write_empty_rows<D, kF32Out>(p, blk, out_head, tile_first, kRowsPerTile,
                                       threadIdx.x & 127, 128);
          continue;
        }
        const int row = tile_first + row_in_tile;
        const EpilogueStore store{&tm_o, stage, 1 + t, out_head};
        auto signal_p = [&] {
          __syncwarp();
          if (lane == 0) mbar_arrive(pfull);  // one arrival per warp
        };
        const bool ok = softmax_row<D, kF32Out, decltype(signal_p), kFp8, kPoly>(
            p, blk, row, tile_first, n, tS(t) + lane_off, tO(t) + lane_off, bar(kBarSFull + t),
            bar(kBarOFull + t), g, u & 1u,
            static_cast<size_t>(out_head) * p.o_rows + static_cast<size_t>(blk.o_row + row),
            abort_flag, err, store, signal_p);
        g += n;
        ++u;
        if (!ok) break;  // the same on every thread of the warpgroup
      }
    } else {
      int g = 0;       // KV steps of this tile over earlier segments
      uint32_t u = 0;  // earlier segments in which this tile visited a KV tile
      int cur_blk = 0;  // block of the previous item (block tables)
      bool ok = true;
      for (long long i = 0, k = item_index(0); k < n_items && ok; k = item_index(++i)) {
        const Item it = item_of(p, tbl, k, cur_blk);
        for (int sg = 0; sg < n_segs && ok; ++sg) {  // each segment's partial in turn
          const BlockDesc blk = seg_block(p, tbl, it, sg);
          const int out_head = blk.part * p.B * p.Hq + it.bh;  // head of O / lse written
          const int tile_first = it.row0 + t * kRowsPerTile;
          const int n = tiles(it, sg, t);
          if (n == 0) {
            write_empty_rows<D, kF32Out>(p, blk, out_head, tile_first, kRowsPerTile,
                                         threadIdx.x & 127, 128);
            continue;
          }
          const int row = tile_first + row_in_tile;
          const EpilogueStore store{&tm_o, stage, 1 + t, out_head};
          auto signal_p = [&] {
            __syncwarp();
            if (lane == 0) mbar_arrive(pfull);  // one arrival per warp
          };
          // a failed segment ends both loops, the same on every thread of the warpgroup
          ok = softmax_row<D, kF32Out, decltype(signal_p), kFp8, kPoly>(
              p, blk, row, tile_first, n, tS(t) + lane_off, tO(t) + lane_off, bar(kBarSFull + t),
              bar(kBarOFull + t), g, u & 1u,
              static_cast<size_t>(out_head) * p.o_rows + static_cast<size_t>(blk.o_row + row),
              abort_flag, err, store, signal_p);
          g += n;
          ++u;
        }
      }
    }
    // the epilogue's last TMA stores (issued by lane 0 of each warp): read out
    // of shared memory and written to global memory before the CTA's shared
    // memory goes away
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Number of SMs of the current device (read once per device).
int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 1;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int D, bool kF32Out, typename Table, bool kFp8, int kPoly>
cudaError_t launch_typed(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const CUtensorMap &to, const AttnParams &p, const Table &tbl,
                         long long n_items, cudaStream_t stream) {
  auto kernel = attn_fwd_kernel<D, kF32Out, Table, kFp8, kPoly>;
  constexpr int kSmem = Cfg<D, kFp8>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  if (n_items == 0) return cudaSuccess;
  // persistent: one CTA per SM (or per work item, if there are fewer)
  const long long grid = n_items < sm_count() ? n_items : sm_count();
  kernel<<<static_cast<unsigned>(grid), kThreads, kSmem, stream>>>(tq, tk, tv, to, p, tbl);
  return cudaGetLastError();
}

// bf16 output: every exponential on the MUFU. fp32 partials: kPolyPairsShort
// of every 8 pairs on the FMA pipe, unless some block is longer than
// kPolyMaxKeys. Segment tables (the partials of short blocks) come with fp32
// output only.
template <int D, typename Table>
cudaError_t launch_out(bool f32_out, bool long_keys, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &to, const AttnParams &p,
                       const Table &tbl, long long n_items, cudaStream_t stream) {
  if constexpr (std::is_same<Table, SegTable>::value) {
    if (!f32_out || long_keys) return cudaErrorInvalidValue;
  } else {
    if (!f32_out) return launch_typed<D, false, Table, false, 0>(tq, tk, tv, to, p, tbl, n_items, stream);
    if (long_keys) return launch_typed<D, true, Table, false, 0>(tq, tk, tv, to, p, tbl, n_items, stream);
  }
  return launch_typed<D, true, Table, false, kPolyPairsShort>(tq, tk, tv, to, p, tbl, n_items, stream);
}

template <typename Table>
cudaError_t launch_dispatch(int D, bool f32_out, bool long_keys, const CUtensorMap &tq,
                            const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &to,
                            const AttnParams &p, const Table &tbl, long long n_items,
                            cudaStream_t stream) {
  if (D == 128) return launch_out<128>(f32_out, long_keys, tq, tk, tv, to, p, tbl, n_items, stream);
  return launch_out<64>(f32_out, long_keys, tq, tk, tv, to, p, tbl, n_items, stream);
}

}  // namespace
}  // namespace seqattn

#include "attn_bwd.cuh"

namespace seqattn {

int device_sm_count() { return sm_count(); }

cudaError_t launch_attention(int D, bool f32_out, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const CUtensorMap &to, const AttnParams &p,
                             cudaStream_t stream) {
  return launch_dispatch(D, f32_out, p.Skv > kPolyMaxKeys, tq, tk, tv, to, p, SingleProblem{0},
                         static_cast<long long>(p.B) * p.Hq * p.n_qblocks, stream);
}

cudaError_t launch_attention_fp8(const CUtensorMap &tq, const CUtensorMap &tk,
                                 const CUtensorMap &tvt, const CUtensorMap &to,
                                 const AttnParams &p, cudaStream_t stream) {
  return launch_typed<128, false, SingleProblem, true, 0>(
      tq, tk, tvt, to, p, SingleProblem{0}, static_cast<long long>(p.B) * p.Hq * p.n_qblocks, stream);
}

cudaError_t launch_attention_blocks(int D, bool f32_out, const CUtensorMap &tq,
                                    const CUtensorMap &tk, const CUtensorMap &tv,
                                    const CUtensorMap &to, const AttnParams &p,
                                    const BlockTable &tbl, cudaStream_t stream) {
  bool long_keys = false;
  for (int i = 0; i < tbl.n; ++i) long_keys = long_keys || tbl.b[i].Skv > kPolyMaxKeys;
  return launch_dispatch(D, f32_out, long_keys, tq, tk, tv, to, p, tbl, tbl.item_start[tbl.n], stream);
}

cudaError_t launch_attention_segments(int D, bool f32_out, const CUtensorMap &tq,
                                      const CUtensorMap &tk, const CUtensorMap &tv,
                                      const CUtensorMap &to, const AttnParams &p,
                                      const SegTable &tbl, cudaStream_t stream) {
  bool long_keys = false;
  for (int i = 0; i < tbl.n; ++i) long_keys = long_keys || tbl.b[i].Skv > kPolyMaxKeys;
  const long long items = static_cast<long long>(p.B) * p.Hq * ((tbl.b[0].Sq + 255) / 256);
  return launch_dispatch(D, f32_out, long_keys, tq, tk, tv, to, p, tbl, items, stream);
}

namespace {

template <int D>
cudaError_t launch_bwd_typed(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const CUtensorMap &tdo, const void *o, const void *dout, float *delta,
                             const BwdParams &p, cudaStream_t stream) {
  const long long nrows = static_cast<long long>(p.B) * p.Hq * p.S;
  if (nrows == 0) return cudaSuccess;
  long long blocks = (nrows + 7) / 8;  // 8 warps of 256 threads, a row per warp
  const long long cap = static_cast<long long>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  bwd::delta_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(o), static_cast<const __nv_bfloat16 *>(dout), delta, nrows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned n_tiles = static_cast<unsigned>((p.S + bwd::kRows - 1) / bwd::kRows);
  constexpr int kSmem = bwd::BwdCfg<D>::kSmemBytes;
  for (int dq = 0; dq < 2; ++dq) {
    auto kernel = dq ? bwd::attn_bwd_kernel<D, true> : bwd::attn_bwd_kernel<D, false>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid(n_tiles, static_cast<unsigned>(p.B * (dq ? p.Hq : p.Hkv)));
    kernel<<<grid, bwd::kThreads, kSmem, stream>>>(tq, tk, tv, tdo, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_attention_bwd(int D, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const CUtensorMap &tdo, const void *o, const void *dout,
                                 float *delta, const BwdParams &p, cudaStream_t stream) {
  return D == 64 ? launch_bwd_typed<64>(tq, tk, tv, tdo, o, dout, delta, p, stream)
                 : launch_bwd_typed<128>(tq, tk, tv, tdo, o, dout, delta, p, stream);
}

// A one-CTA kernel waiting on an mbarrier that nothing ever arrives at, with
// a short limit: the wait gives up exactly as a stuck attention pipeline's
// would, recording the timeout in the device error word.
__global__ void expire_wait_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_addr(&bar), 0, &abort_flag, &g_device_error, limit_ns);
}

cudaError_t launch_expire_wait(unsigned timeout_us, cudaStream_t stream) {
  expire_wait_kernel<<<1, 32, 0, stream>>>(static_cast<unsigned long long>(timeout_us) * 1000ull);
  return cudaGetLastError();
}

// Element pairs (2i, 2i + 1) through exp2_pair; an odd last element pairs with itself.
__global__ void exp2_probe_kernel(const float *x, float *y, long long n, bool poly) {
  const long long i = 2 * (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float a = x[i], b = (i + 1 < n) ? x[i + 1] : a;
  float ra, rb;
  f2_unpack(exp2_pair(f2_pack(a, b), poly), ra, rb);
  y[i] = ra;
  if (i + 1 < n) y[i + 1] = rb;
}

cudaError_t launch_exp2_probe(const float *x, float *y, long long n, bool poly,
                              cudaStream_t stream) {
  const long long pairs = (n + 1) / 2;
  const long long blocks = (pairs + 255) / 256;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  exp2_probe_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, y, n, poly);
  return cudaGetLastError();
}

cudaError_t read_and_clear_device_error(int *code) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace seqattn
