// Blockwise exact attention forward on SM pairs (head dim 128), sm_103a.
//
// Same computation as attn_fwd_kernel (the tiled online-softmax forward of
// page "ms-swift集成FlashAttention 2/3，长文本训练更高效", section
// "FlashAttention 如何破局？不只是融合内核"), mapped onto 2-SM tcgen05 MMAs so
// that each SM receives half of every K/V tile:
//
//   cluster of two CTAs (ranks 0, 1) = 512 query rows of one (batch, head).
//   MMA group g (g = 0, 1) is M = 256 rows [row0 + 256 g, +256): its first 128
//   rows live in CTA 0, the next 128 in CTA 1 (Q tile, S, P and O in each
//   CTA's own shared memory / TMEM).
//   S_g = Q_g K_j^T: B split along N, so CTA r holds keys [64 r, 64 r + 64) of
//   KV tile j (a 16 KB half tile, both 64-column blocks).
//   O_g += P_g V_j: B split along N = head dim, so CTA r holds column block r
//   of V_j (128 keys x 64 dims, 16 KB).
//   Per KV step each SM therefore loads 32 KB instead of 64 KB and its tensor
//   core reads half the B operand bytes from shared memory.
//
// Roles (320 threads per CTA):
//   warp 9   both CTAs: TMA producer for its own Q tiles and K/V halves, into a
//            ring of 8 16-KB slots; completion lands on its own barriers.
//   warp 8   CTA 0: the MMA issuer for the pair (cta_group::2), committing to
//            barriers in both CTAs by multicast. CTA 1: forwards each of its
//            load completions to CTA 0 with a remote mbarrier arrive.
//   warps 0-7 both CTAs: softmax + epilogue for the CTA's own two 128-row tiles
//            (one per MMA group); P-ready is one arrival per warp on CTA 0's
//            barrier (remote from CTA 1).
// The two halves of a group differ by 128 rows, so under causal masking the
// first half visits at most one KV tile it cannot see (fully masked, P = 0).

namespace seqattn {
namespace pair2sm {

using namespace detail;

constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kD = 128;
constexpr int kQTileBytes = kRowsPerTile * kD * 2;  // 32 KB
constexpr int kSlotBytes = 16384;                   // half a K or V tile
constexpr int kKHalfColBlock = 64 * 128;            // 64 keys x 128 B
constexpr int kStages = 8;
// q, q_peer, full[S], full_peer[S], empty[S], s_full[2], p_full[2], o_full[2], mma_done
constexpr int kNumBarriers = 2 + 3 * kStages + 7;
constexpr int kSmemBytes = 1024 + 2 * kQTileBytes + kStages * kSlotBytes + 8 * kNumBarriers + 16;
constexpr int kRowsPerCluster = 512;

template <bool kF32Out>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_fwd_2sm_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const AttnParams p,
                        long long n_work) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem;                      // [group][col block][128 rows][128 B]
  uint8_t *sRing = smem + 2 * kQTileBytes;  // [slot] 16 KB
  uint64_t *bars = reinterpret_cast<uint64_t *>(sRing + kStages * kSlotBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBarriers);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const long long work = static_cast<long long>(blockIdx.y) +
                         static_cast<long long>(blockIdx.z) * gridDim.y;
  if (work >= n_work) return;  // both CTAs of the cluster leave together

  const uint32_t bar0 = smem_addr(bars);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  constexpr int kBarQ = 0, kBarQPeer = 1, kBarFull = 2, kBarFullPeer = 2 + kStages,
                kBarEmpty = 2 + 2 * kStages, kBarSFull = 2 + 3 * kStages, kBarPFull = kBarSFull + 2,
                kBarOFull = kBarPFull + 2, kBarMmaDone = kBarOFull + 2;

  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int BH = p.B * p.Hq;
  const int bh = static_cast<int>(work % BH);
  const int qb_raw = static_cast<int>(work / BH);
  // causal: the longest query blocks first; heads of one GQA group adjacent
  const int qb = p.causal ? (p.n_qblocks - 1 - qb_raw) : qb_raw;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int hkv = hq / (p.Hq / p.Hkv);
  const int row0 = qb * kRowsPerCluster;
  int *err = &g_device_error;

  // No row of the cluster's 512 sees a key: both CTAs reach the same decision
  // and leave before any cluster-wide operation.
  {
    bool any = false;
    for (int r = 0; r < kRowsPerCluster; r += kRowsPerTile) any = any || kv_tiles_for(p, row0 + r) > 0;
    if (!any) {
      for (int g = 0; g < 2; ++g)
        write_empty_rows<kD, kF32Out>(p, whole_problem(p), bh,
                                      row0 + 256 * g + kRowsPerTile * static_cast<int>(rank),
                                      kRowsPerTile, threadIdx.x, blockDim.x);
      return;
    }
  }

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    mbar_init(bar(kBarQPeer), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarFullPeer + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(bar(kBarSFull + g), 1);
      mbar_init(bar(kBarPFull + g), 8);  // one arrival per softmax warp of both CTAs
      mbar_init(bar(kBarOFull + g), 1);
    }
    mbar_init(bar(kBarMmaDone), 1);
    // the even CTA decides for the pair whether a recorded timeout skips the work
    *abort_flag = leader ? (*reinterpret_cast<volatile int *>(err) != kErrNone) : 0;
    fence_barrier_init();
  }
  cluster_sync();  // every barrier of both CTAs exists before any remote arrival
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_addr(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip =
      ld_shared_cluster_u32(mapa_shared(smem_addr(const_cast<int *>(abort_flag)), 0)) != 0;
  int n_grp[2];
  for (int g = 0; g < 2; ++g) {
    const int first = row0 + 256 * g;
    n_grp[g] = skip ? 0 : max(kv_tiles_for(p, first), kv_tiles_for(p, first + kRowsPerTile));
  }
  const int n_max = max(n_grp[0], n_grp[1]);
  auto tS = [&](int g) -> uint32_t { return tmem + 128u * static_cast<uint32_t>(g); };
  auto tO = [&](int g) -> uint32_t { return tmem + 256u + 128u * static_cast<uint32_t>(g); };

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0 && n_max > 0) {
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      tma_prefetch_map(&tm_v);
      mbar_arrive_expect_tx(bar(kBarQ), 2 * kQTileBytes);
      for (int g = 0; g < 2; ++g)
        for (int cb = 0; cb < 2; ++cb)
          tma_load_3d(smem_addr(sQ + g * kQTileBytes + cb * kColBlockBytes), &tm_q, bar(kBarQ),
                      cb * 64, row0 + 256 * g + kRowsPerTile * static_cast<int>(rank), bh);
      const int kv_head = b * p.Hkv + hkv;
      int c = 0;  // K_0, V_0, K_1, V_1, ...
      bool ok = true;
      for (int j = 0; j < n_max && ok; ++j) {
        for (int which = 0; which < 2; ++which, ++c) {
          const int slot = c % kStages;
          if (c >= kStages &&
              !mbar_wait(bar(kBarEmpty + slot), ((c / kStages) - 1) & 1, abort_flag, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarFull + slot), kSlotBytes);
          const uint32_t dst = smem_addr(sRing + slot * kSlotBytes);
          if (which == 0) {  // keys [64 r, 64 r + 64) of K_j, both column blocks
            for (int cb = 0; cb < 2; ++cb)
              tma_load_3d(dst + cb * kKHalfColBlock, &tm_k, bar(kBarFull + slot), cb * 64,
                          j * kRowsPerTile + 64 * static_cast<int>(rank), kv_head);
          } else {  // column block r of V_j
            tma_load_3d(dst, &tm_v, bar(kBarFull + slot), 64 * static_cast<int>(rank),
                        j * kRowsPerTile, kv_head);
          }
        }
      }
      mbar_drain(bar(kBarQ), 0, err);
      for (int i = max(0, c - kStages); i < c; ++i)
        mbar_drain(bar(kBarFull + i % kStages), (i / kStages) & 1, err);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- MMA issuer (CTA 0)
      constexpr uint32_t idesc_s = idesc_bf16_f32(256, 128, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(256, kD, true);
      const uint32_t q_base = smem_addr(sQ);
      const uint32_t ring_base = smem_addr(sRing);
      bool ok = n_max > 0 && mbar_wait(bar(kBarQ), 0, abort_flag, err) &&
                mbar_wait_cluster(bar(kBarQPeer), 0, abort_flag, err);
      for (int j = 0; ok && j <= n_max; ++j) {
        const int cK = 2 * j, cV = 2 * j - 1;
        const int sK = cK % kStages, sV = (cV + kStages) % kStages;
        const uint32_t k_base = ring_base + sK * kSlotBytes;
        const uint32_t v_base = ring_base + sV * kSlotBytes;
        if (j < n_max && !(mbar_wait(bar(kBarFull + sK), (cK / kStages) & 1, abort_flag, err) &&
                           mbar_wait_cluster(bar(kBarFullPeer + sK), (cK / kStages) & 1,
                                             abort_flag, err)))
          break;
        if (j >= 1 && !(mbar_wait(bar(kBarFull + sV), (cV / kStages) & 1, abort_flag, err) &&
                        mbar_wait_cluster(bar(kBarFullPeer + sV), (cV / kStages) & 1, abort_flag,
                                          err)))
          break;
        tc_fence_after();
        for (int g = 0; g < 2 && ok; ++g) {
          const int ng = g ? n_grp[1] : n_grp[0];
          if (j >= 1 && j - 1 < ng) {
            // O_g += P_g V_{j-1}
            if (!mbar_wait_cluster(bar(kBarPFull + g), (j - 1) & 1, abort_flag, err)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kRowsPerTile / 16; ++kk)
              mma_ts_pair(tO(g), tS(g) + kk * 8, sw128_desc(v_base + kk * 2048, kColBlockBytes, 1024),
                          idesc_o, (j > 1 || kk > 0) ? 1u : 0u);
            if (j - 1 == ng - 1) mma_commit_pair(bar(kBarOFull + g), 3);
            if (g == 1 || j - 1 >= n_grp[1]) mma_commit_pair(bar(kBarEmpty + sV), 3);
          }
          if (j < ng) {
            // S_g = Q_g K_j^T
            const uint32_t qg = q_base + g * kQTileBytes;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t off_a = (kk / 4) * kColBlockBytes + (kk % 4) * 32;
              const uint32_t off_b = (kk / 4) * kKHalfColBlock + (kk % 4) * 32;
              mma_ss_pair(tS(g), sw128_desc(qg + off_a, 16, 1024),
                          sw128_desc(k_base + off_b, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit_pair(bar(kBarSFull + g), 3);
            if (g == 1 || j >= n_grp[1]) mma_commit_pair(bar(kBarEmpty + sK), 3);
          }
        }
      }
      // All MMAs issued here must be complete before either CTA releases memory.
      mma_commit_pair(bar(kBarMmaDone), 1);
      mbar_drain(bar(kBarMmaDone), 0, err);
    } else if (lane == 0 && n_max > 0) {
      // ---------------------------------------------------------- forwarder (CTA 1)
      if (mbar_wait(bar(kBarQ), 0, abort_flag, err)) {
        mbar_arrive_remote(mapa_shared(bar(kBarQPeer), 0));
        for (int c = 0; c < 2 * n_max; ++c) {
          const int slot = c % kStages;
          if (!mbar_wait(bar(kBarFull + slot), (c / kStages) & 1, abort_flag, err)) break;
          mbar_arrive_remote(mapa_shared(bar(kBarFullPeer + slot), 0));
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int g = warp >> 2;
    const int tile_first = row0 + 256 * g + kRowsPerTile * static_cast<int>(rank);
    const int row = tile_first + (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t pfull_local = bar(kBarPFull + g);
    const uint32_t pfull_leader = mapa_shared(pfull_local, 0);
    softmax_row<kD, kF32Out>(p, whole_problem(p), row, tile_first, g ? n_grp[1] : n_grp[0],
                             tS(g) + lane_off, tO(g) + lane_off, bar(kBarSFull + g),
                             bar(kBarOFull + g), 0, 0u, static_cast<size_t>(bh) * p.o_rows + row,
                             abort_flag, err,
                             EpilogueStore{nullptr, 0u, 0, 0}, [&] {
                               __syncwarp();
                               if (lane == 0) {
                                 if (leader)
                                   mbar_arrive(pfull_local);
                                 else
                                   mbar_arrive_remote(pfull_leader);
                               }
                             });
  }

  tc_fence_before();
  cluster_sync();  // the pair's MMAs and remote arrivals are all complete
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
  cluster_sync();
}

template <bool kF32Out>
cudaError_t launch_pair(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        AttnParams p, cudaStream_t stream) {
  auto kernel = attn_fwd_2sm_kernel<kF32Out>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  p.n_qblocks = (p.Sq + kRowsPerCluster - 1) / kRowsPerCluster;
  const long long n_work = static_cast<long long>(p.n_qblocks) * p.B * p.Hq;
  const long long gy = n_work < 65535 ? n_work : 65535;
  const long long gz = (n_work + gy - 1) / gy;
  if (gz > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid(2, static_cast<unsigned>(gy), static_cast<unsigned>(gz));
  kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p, n_work);
  return cudaGetLastError();
}

}  // namespace pair2sm
}  // namespace seqattn
