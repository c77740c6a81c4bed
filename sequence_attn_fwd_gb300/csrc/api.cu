// C-ABI entry points of libseqattn.so (declared in include/seqattn.h):
// argument validation, TMA tensor-map construction and kernel launch. No
// entry point allocates device memory or synchronises, except the explicit
// device-error query.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/seqattn.h"
#include "kernels.h"

namespace {

std::atomic<int> g_last_cuda_error{0};

int cuda_fail(cudaError_t e) {
  g_last_cuda_error.store(static_cast<int>(e));
  return ATTN_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 3-D bf16 view [heads][rows][D] with the head stride given in elements; box
// 64 x box_rows x 1 with 128-byte swizzle. Rows past `rows` read as zero.
bool make_map(CUtensorMap *map, const void *base, int D, long long rows, long long heads,
              long long head_stride, unsigned box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2u,
                           static_cast<cuuint64_t>(head_stride) * 2u};
  cuuint32_t box[3] = {64u, box_rows, 1u};
  cuuint32_t estride[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view [heads][rows][D] of the output (fp32 or bf16, rows contiguous per
// head); box 128 bytes x 32 rows x 1 (the rows of one warp) with 128-byte
// swizzle, for TMA stores.
bool make_out_map(CUtensorMap *map, void *base, int D, long long rows, long long heads,
                  bool f32) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const unsigned es = f32 ? 4u : 2u;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * es,
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(D) * es};
  cuuint32_t box[3] = {128u / es, 32u, 1u};  // 128 bytes x the 32 rows of one warp
  cuuint32_t estride[3] = {1u, 1u, 1u};
  return fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base,
            dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool scale_ok(float scale) { return isfinite(scale) && scale > 0.f; }

// Heads per item chunk of a single problem: whole GQA groups whose K and V
// (Skv rows each, elem_bytes per element) fit in 32 MB of L2 together, at
// least one group.
int heads_per_chunk(int B, int Hq, int Hkv, long long Skv, int D, int elem_bytes) {
  const long long group = Hq / Hkv;
  const long long kv_bytes = 2LL * (Skv > 0 ? Skv : 1) * D * elem_bytes;  // K and V of one KV head
  long long groups = (32LL << 20) / kv_bytes;
  if (groups < 1) groups = 1;
  const long long heads = static_cast<long long>(B) * Hq;
  const long long hc = groups * group;
  return static_cast<int>(hc < heads ? hc : heads);
}

// 3-D byte view [heads][rows][cols] of e4m3 data (rows contiguous), box
// 128 x 128 x 1 with 128-byte swizzle.
bool make_map_u8(CUtensorMap *map, const void *base, long long cols, long long rows, long long heads) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols),
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(cols)};
  cuuint32_t box[3] = {128u, 128u, 1u};
  cuuint32_t estride[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr long long kMaxRowsPerHead = 1ll << 30;  // keeps every row index within int range

int run_attention(const void *q, const void *k, const void *v, long long q_off, long long kv_off,
                  long long kv_head_stride, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
                  int Skv, int D, int causal, float scale, bool f32_out, bool skip_empty,
                  cudaStream_t stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv < 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (Sq > kMaxRowsPerHead || Skv > kMaxRowsPerHead) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
  if ((Sq + 255ll) / 256 > 65535) return ATTN_ERR_UNSUPPORTED;
  if (kv_head_stride == 0) kv_head_stride = static_cast<long long>(Skv) * D;
  if (kv_head_stride < static_cast<long long>(Skv) * D || kv_head_stride % 8 != 0)
    return ATTN_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0) return ATTN_OK;  // nothing to compute
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return ATTN_ERR_INVALID_ARG;

  CUtensorMap tq, tk, tv, to;
  // An empty key set still needs well-formed maps; no KV tile is ever loaded.
  const long long kv_rows = Skv > 0 ? Skv : 1;
  if (!make_map(&tq, q, D, Sq, static_cast<long long>(B) * Hq, static_cast<long long>(Sq) * D) ||
      !make_map(&tk, k, D, kv_rows, static_cast<long long>(B) * Hkv, kv_head_stride) ||
      !make_map(&tv, v, D, kv_rows, static_cast<long long>(B) * Hkv, kv_head_stride) ||
      !make_out_map(&to, o, D, Sq, static_cast<long long>(B) * Hq, f32_out))
    return cuda_fail(cudaErrorInvalidValue);

  seqattn::AttnParams p;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Skv = Skv;
  p.q_off = q_off;
  p.kv_off = kv_off;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal;
  p.n_qblocks = (Sq + 255) / 256;
  p.skip_empty = skip_empty ? 1 : 0;
  p.o_rows = Sq;
  p.o_scale = 1.f;
  p.heads_per_chunk = heads_per_chunk(B, Hq, Hkv, Skv, D, 2);
  cudaError_t e = seqattn::launch_attention(D, f32_out, tq, tk, tv, to, p, stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// Attention over a list of blocks (row ranges of packed [heads][rows][D]
// tensors), launched in tables of at most kMaxLaunchBlocks blocks. The caller
// has validated shapes, pointers and ranges.
int run_blocks(const void *q, const void *k, const void *v, void *o, float *lse,
               const std::vector<seqattn::BlockDesc> &blocks, int B, int Hq, int Hkv,
               long long q_rows, long long kv_rows, long long o_rows, int n_parts, int D,
               int causal, float scale, bool f32_out, bool skip_empty, cudaStream_t stream) {
  if (blocks.empty() || B == 0) return ATTN_OK;
  CUtensorMap tq, tk, tv, to;
  const long long heads = static_cast<long long>(B) * Hq, kv_heads = static_cast<long long>(B) * Hkv;
  const long long o_heads = heads * n_parts;
  if (!make_map(&tq, q, D, q_rows > 0 ? q_rows : 1, heads, (q_rows > 0 ? q_rows : 1) * D) ||
      !make_map(&tk, k, D, kv_rows > 0 ? kv_rows : 1, kv_heads, (kv_rows > 0 ? kv_rows : 1) * D) ||
      !make_map(&tv, v, D, kv_rows > 0 ? kv_rows : 1, kv_heads, (kv_rows > 0 ? kv_rows : 1) * D) ||
      !make_out_map(&to, o, D, o_rows > 0 ? o_rows : 1, o_heads, f32_out))
    return cuda_fail(cudaErrorInvalidValue);
  seqattn::AttnParams p{};
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal;
  p.skip_empty = skip_empty ? 1 : 0;
  p.o_rows = o_rows;
  p.o_scale = 1.f;
  // Short blocks that all share their query rows (the key chunks of a ring
  // pass, up to kSegMaxKeys keys each) run as the segments of each work item:
  // Q is loaded once for all of them and each chunk's first scores follow the
  // previous chunk's last product, which pays where an item's fixed cost is a
  // large part of its work. Longer chunks keep the block table, whose items
  // run one chunk after another and so keep a chunk's K and V in L2, where
  // segments would stream the K and V of every chunk at once; so do lists
  // whose shared rows make fewer items than the GPU has SMs, where one item a
  // block keeps more SMs busy.
  constexpr int kSegMaxKeys = 2048;
  bool shared_q = f32_out && blocks.size() >= 2 && blocks[0].Sq > 0 &&
                  heads * ((blocks[0].Sq + 255) / 256) >= seqattn::device_sm_count();
  for (const auto &b : blocks)
    shared_q = shared_q && b.q_row == blocks[0].q_row && b.o_row == blocks[0].o_row &&
               b.q_pos == blocks[0].q_pos && b.Sq == blocks[0].Sq && b.Skv <= kSegMaxKeys;
  if (shared_q) {
    for (size_t first = 0; first < blocks.size(); first += seqattn::kMaxLaunchBlocks) {
      seqattn::SegTable tbl{};
      const size_t n = std::min(blocks.size() - first, static_cast<size_t>(seqattn::kMaxLaunchBlocks));
      tbl.n = static_cast<int>(n);
      for (size_t i = 0; i < n; ++i) tbl.b[i] = blocks[first + i];
      cudaError_t e = seqattn::launch_attention_segments(D, f32_out, tq, tk, tv, to, p, tbl, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return ATTN_OK;
  }
  for (size_t first = 0; first < blocks.size(); first += seqattn::kMaxLaunchBlocks) {
    seqattn::BlockTable tbl{};
    const size_t n = std::min(blocks.size() - first, static_cast<size_t>(seqattn::kMaxLaunchBlocks));
    tbl.n = static_cast<int>(n);
    long long items = 0;
    for (size_t i = 0; i < n; ++i) {
      tbl.b[i] = blocks[first + i];
      tbl.item_start[i] = items;
      items += heads * ((blocks[first + i].Sq + 255) / 256);
    }
    tbl.item_start[n] = items;
    cudaError_t e = seqattn::launch_attention_blocks(D, f32_out, tq, tk, tv, to, p, tbl, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return ATTN_OK;
}

// Checks shared by the block entry points; blocks must lie inside the tensors
// and the output rows of blocks of the same part must not overlap.
int check_blocks(const std::vector<seqattn::BlockDesc> &blocks, long long q_rows, long long kv_rows,
                 long long o_rows, int n_parts) {
  if (q_rows < 0 || kv_rows < 0 || o_rows < 0 || q_rows > kMaxRowsPerHead ||
      kv_rows > kMaxRowsPerHead || o_rows > kMaxRowsPerHead || n_parts < 1)
    return ATTN_ERR_INVALID_ARG;
  std::vector<std::pair<std::pair<int, long long>, long long>> outs;
  for (const auto &b : blocks) {
    if (b.Sq < 0 || b.Skv < 0 || b.q_row < 0 || b.kv_row < 0 || b.o_row < 0) return ATTN_ERR_INVALID_ARG;
    if (b.part < 0 || b.part >= n_parts) return ATTN_ERR_INVALID_ARG;
    if (b.q_row + b.Sq > q_rows || b.kv_row + b.Skv > kv_rows || b.o_row + b.Sq > o_rows)
      return ATTN_ERR_INVALID_ARG;
    if (b.q_pos < -kMaxRowsPerHead * 4 || b.q_pos > kMaxRowsPerHead * 4 ||
        b.kv_pos < -kMaxRowsPerHead * 4 || b.kv_pos > kMaxRowsPerHead * 4)
      return ATTN_ERR_INVALID_ARG;
    if (b.Sq > 0) outs.push_back({{b.part, b.o_row}, b.o_row + b.Sq});
  }
  std::sort(outs.begin(), outs.end());
  for (size_t i = 1; i < outs.size(); ++i)
    if (outs[i].first.first == outs[i - 1].first.first && outs[i].first.second < outs[i - 1].second)
      return ATTN_ERR_INVALID_ARG;  // overlapping outputs
  return ATTN_OK;
}

int check_common(const void *q, const void *k, const void *v, const void *o, const float *lse, int B,
                 int Hq, int Hkv, int D, int causal, float scale) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
             const void *dout, float *delta, void *dq, void *dk, void *dv, int B, int Hq, int Hkv,
             int S, int D, int causal, float scale, attn_stream_t stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || S < 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (S > kMaxRowsPerHead) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq > 65535) return ATTN_ERR_UNSUPPORTED;  // heads along the grid's y
  if (B == 0 || S == 0) return ATTN_OK;
  const void *ptrs16[] = {q, k, v, o, dout, dq, dk, dv};
  for (const void *ptr : ptrs16)
    if (!ptr || !aligned16(ptr)) return ATTN_ERR_INVALID_ARG;
  if (!lse || !delta || (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(delta) & 3u))
    return ATTN_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv, tdo;
  const long long heads = static_cast<long long>(B) * Hq, kv_heads = static_cast<long long>(B) * Hkv;
  const long long hs = static_cast<long long>(S) * D;
  if (!make_map(&tq, q, D, S, heads, hs) || !make_map(&tk, k, D, S, kv_heads, hs) ||
      !make_map(&tv, v, D, S, kv_heads, hs) || !make_map(&tdo, dout, D, S, heads, hs))
    return cuda_fail(cudaErrorInvalidValue);
  seqattn::BwdParams p{};
  p.lse = lse;
  p.delta = delta;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.S = S;
  p.scale = scale;
  p.causal = causal;
  cudaError_t e = seqattn::launch_attention_bwd(D, tq, tk, tv, tdo, o, dout, delta, p,
                                                reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

int attn_fwd_fp8(const void *q8, const void *k8, const void *vt8, void *o, float *lse, int B, int Hq,
                 int Hkv, int S, int D, int causal, float scale, float q_scale, float k_scale,
                 float v_scale, attn_stream_t stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || S < 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!scale_ok(scale) || !scale_ok(q_scale) || !scale_ok(k_scale) || !scale_ok(v_scale))
    return ATTN_ERR_INVALID_ARG;
  if (D != 128) return ATTN_ERR_UNSUPPORTED;
  if (S % 16 != 0) return ATTN_ERR_UNSUPPORTED;  // V^T rows of S bytes must be 16-byte multiples
  if (S > kMaxRowsPerHead || (S + 255ll) / 256 > 65535) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || S == 0) return ATTN_OK;
  if (!q8 || !k8 || !vt8 || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return ATTN_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tvt, to;
  const long long heads = static_cast<long long>(B) * Hq, kv_heads = static_cast<long long>(B) * Hkv;
  if (!make_map_u8(&tq, q8, D, S, heads) || !make_map_u8(&tk, k8, D, S, kv_heads) ||
      !make_map_u8(&tvt, vt8, S, D, kv_heads) || !make_out_map(&to, o, D, S, heads, false))
    return cuda_fail(cudaErrorInvalidValue);
  seqattn::AttnParams p{};
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = S;
  p.Skv = S;
  p.q_off = 0;
  p.kv_off = 0;
  p.scale_log2 = scale * q_scale * k_scale * 1.4426950408889634f;
  p.causal = causal;
  p.n_qblocks = (S + 255) / 256;
  p.skip_empty = 0;
  p.o_rows = S;
  p.o_scale = v_scale;
  p.heads_per_chunk = heads_per_chunk(B, Hq, Hkv, S, D, 1);
  cudaError_t e = seqattn::launch_attention_fp8(tq, tk, tvt, to, p, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

int attn_partial_blocks(const void *q, const void *k, const void *v, float *o_part, float *lse_part,
                        const attn_block *blocks, int n_blocks, int B, int Hq, int Hkv,
                        long long q_rows, long long kv_rows, long long o_rows, int n_parts, int D,
                        int causal, float scale, int flags, attn_stream_t stream) {
  if (flags & ~ATTN_PARTIAL_SKIP_EMPTY) return ATTN_ERR_INVALID_ARG;
  if (n_blocks < 0 || (n_blocks > 0 && !blocks)) return ATTN_ERR_INVALID_ARG;
  if (n_blocks == 0 || B == 0) return (B < 0) ? ATTN_ERR_INVALID_ARG : ATTN_OK;
  int st = check_common(q, k, v, o_part, lse_part, B, Hq, Hkv, D, causal, scale);
  if (st != ATTN_OK) return st;
  std::vector<seqattn::BlockDesc> bl(static_cast<size_t>(n_blocks));
  for (int i = 0; i < n_blocks; ++i)
    bl[i] = {blocks[i].q_row, blocks[i].kv_row, blocks[i].o_row, blocks[i].q_pos, blocks[i].kv_pos,
             blocks[i].Sq, blocks[i].Skv, blocks[i].part};
  st = check_blocks(bl, q_rows, kv_rows, o_rows, n_parts);
  if (st != ATTN_OK) return st;
  if (static_cast<long long>(B) * Hq * n_parts > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
  return run_blocks(q, k, v, o_part, lse_part, bl, B, Hq, Hkv, q_rows, kv_rows, o_rows, n_parts, D,
                    causal, scale, true, (flags & ATTN_PARTIAL_SKIP_EMPTY) != 0,
                    reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                    const long long *cu_seqlens_q, const long long *cu_seqlens_k, int nseq, int Hq,
                    int Hkv, int D, int causal, float scale, attn_stream_t stream) {
  if (nseq < 0 || (nseq > 0 && (!cu_seqlens_q || !cu_seqlens_k))) return ATTN_ERR_INVALID_ARG;
  if (nseq == 0) return ATTN_OK;
  if (cu_seqlens_q[0] != 0 || cu_seqlens_k[0] != 0) return ATTN_ERR_INVALID_ARG;
  std::vector<seqattn::BlockDesc> bl(static_cast<size_t>(nseq));
  for (int s = 0; s < nseq; ++s) {
    const long long sq = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
    const long long sk = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
    if (sq < 0 || sk < 0 || sq > kMaxRowsPerHead || sk > kMaxRowsPerHead) return ATTN_ERR_INVALID_ARG;
    // causal: aligned at the bottom right (query row i of a sequence sees keys j <= i + sk - sq)
    bl[s] = {cu_seqlens_q[s], cu_seqlens_k[s], cu_seqlens_q[s], sk - sq, 0, static_cast<int>(sq),
             static_cast<int>(sk), 0};
  }
  const long long total_q = cu_seqlens_q[nseq], total_k = cu_seqlens_k[nseq];
  if (total_q == 0) return ATTN_OK;
  int st = check_common(q, k, v, o, lse, 1, Hq, Hkv, D, causal, scale);
  if (st != ATTN_OK) return st;
  st = check_blocks(bl, total_q, total_k, total_q, 1);
  if (st != ATTN_OK) return st;
  return run_blocks(q, k, v, o, lse, bl, 1, Hq, Hkv, total_q, total_k, total_q, 1, D, causal, scale,
                    false, false, reinterpret_cast<cudaStream_t>(stream));
}


int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
             int Hkv, int S, int D, int causal, float scale, attn_stream_t stream) {
  return run_attention(q, k, v, 0, 0, 0, o, lse, B, Hq, Hkv, S, S, D, causal, scale, false, false,
                       reinterpret_cast<cudaStream_t>(stream));
}

int attn_partial(const void *q, const void *k_chunk, const void *v_chunk, long long q_off,
                 long long kv_off, long long kv_head_stride, float *o_part, float *lse_part,
                 int B, int Hq, int Hkv, int Sq, int Skv, int D, int causal, float scale, int flags,
                 attn_stream_t stream) {
  if (flags & ~ATTN_PARTIAL_SKIP_EMPTY) return ATTN_ERR_INVALID_ARG;
  return run_attention(q, k_chunk, v_chunk, q_off, kv_off, kv_head_stride, o_part, lse_part, B, Hq,
                       Hkv, Sq, Skv, D, causal, scale, true, (flags & ATTN_PARTIAL_SKIP_EMPTY) != 0,
                       reinterpret_cast<cudaStream_t>(stream));
}

int lse_merge(const float *o_parts, const float *lse_parts, int P, void *o, int o_dtype,
              float *lse, int B, int H, int S, int D, attn_stream_t stream) {
  if (P < 1 || B < 0 || H <= 0 || S < 0) return ATTN_ERR_INVALID_ARG;
  if (o_dtype != ATTN_BF16 && o_dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  const long long nrows = static_cast<long long>(B) * H * S;
  if (nrows == 0) return ATTN_OK;
  if (!o_parts || !lse_parts || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return ATTN_ERR_INVALID_ARG;
  cudaError_t e = seqattn::launch_lse_merge(o_parts, lse_parts, P, nrows, D, o, o_dtype == ATTN_BF16,
                                            lse, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

int attn_query_device_error(attn_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int code = 0;
  e = seqattn::read_and_clear_device_error(&code);
  if (e != cudaSuccess) return cuda_fail(e);
  return code == 0 ? ATTN_OK : ATTN_ERR_TIMEOUT;
}

const char *attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape or head dimension";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int attn_last_cuda_error(void) { return g_last_cuda_error.load(); }

int attn_debug_exp2(const float *x, float *y, long long n, int poly, attn_stream_t stream) {
  if (n < 0 || (poly != 0 && poly != 1)) return ATTN_ERR_INVALID_ARG;
  if (n == 0) return ATTN_OK;
  if (!x || !y) return ATTN_ERR_INVALID_ARG;
  cudaError_t e = seqattn::launch_exp2_probe(x, y, n, poly != 0, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

int attn_debug_expire_wait(unsigned timeout_us, attn_stream_t stream) {
  if (timeout_us == 0 || timeout_us > 1000000u) return ATTN_ERR_INVALID_ARG;
  cudaError_t e = seqattn::launch_expire_wait(timeout_us, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Ring forward with library-owned scratch, for callers that cannot allocate.
//
// Some callers of this library must not, or cannot, call cudaMalloc: code
// embedded in a host application whose own allocator has already reserved
// nearly all device memory (a raw allocation would fail or fragment it), and
// latency-sensitive loops where cudaMalloc/cudaFree are unacceptable because
// they can synchronise the whole device. attn_ring_fwd_static serves them: the
// fp32 per-chunk partials that ring_attn_fwd keeps in caller memory live here
// in one fixed device array instead. Every GPU that loads this library holds
// the array (kRingScratchBytes) until the process exits.
//
// In host code `g_ring_scratch` is only a host-side stand-in for the device
// symbol; its device address comes from cudaGetSymbolAddress, looked up once
// per device (with that device current) on the first call there.
static __device__ __align__(256) unsigned char g_ring_scratch[SEQATTN_RING_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_ring_scratch_mutex;
void *g_ring_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on first use).
int ring_scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_ring_scratch_mutex);
  if (!g_ring_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_ring_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_ring_scratch_ptr[dev] = p;
  }
  *out = g_ring_scratch_ptr[dev];
  return ATTN_OK;
}

size_t align_up_256(size_t n) { return (n + 255u) & ~static_cast<size_t>(255u); }

}  // namespace

extern "C" int attn_ring_fwd_static(const void *q, const void *k, const void *v, void *o,
                                    float *lse, int B, int Hq, int Hkv, int S, int D, int P,
                                    int causal, float scale, attn_stream_t stream) {
  if (P < 1 || S < 0 || B < 0 || Hq <= 0) return ATTN_ERR_INVALID_ARG;
  if (S % P != 0) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(B) * Hq * S;
  if (rows == 0) return ATTN_OK;
  // partials: o_parts fp32 [P, B, Hq, S, D], then lse_parts fp32 [P, B, Hq, S]
  const size_t o_bytes = align_up_256(static_cast<size_t>(P) * rows * D * sizeof(float));
  const size_t l_bytes = align_up_256(static_cast<size_t>(P) * rows * sizeof(float));
  if (o_bytes + l_bytes > static_cast<size_t>(SEQATTN_RING_SCRATCH_BYTES)) return ATTN_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  int st = ring_scratch_address(&scratch);
  if (st != ATTN_OK) return st;
  float *o_parts = static_cast<float *>(scratch);
  float *lse_parts = reinterpret_cast<float *>(static_cast<unsigned char *>(scratch) + o_bytes);
  // Every partial element the merge reads is written by the hops of this same
  // call: each hop writes every lse, and the O rows of every row with a finite
  // lse (rows a chunk cannot see get lse = -inf and are never read), so
  // nothing left in the array by an earlier call needs clearing.
  const int C = S / P;
  for (int j = 0; j < P; ++j) {
    const size_t kv_offset = static_cast<size_t>(j) * C * D;  // elements: chunk j of every head
    st = attn_partial(q, static_cast<const unsigned char *>(k) + kv_offset * 2,
                      static_cast<const unsigned char *>(v) + kv_offset * 2, 0,
                      static_cast<long long>(j) * C, static_cast<long long>(S) * D,
                      o_parts + static_cast<size_t>(j) * rows * D, lse_parts + static_cast<size_t>(j) * rows,
                      B, Hq, Hkv, S, C, D, causal, scale, ATTN_PARTIAL_SKIP_EMPTY, stream);
    if (st != ATTN_OK) return st;
  }
  return lse_merge(o_parts, lse_parts, P, o, ATTN_BF16, lse, B, Hq, S, D, stream);
}

namespace {

// Byte offsets inside the workspace of attn_ring_fwd_host, each part 256-byte aligned.
struct HostLayout {
  size_t q, k, v, o_parts, lse_parts, o, lse, total;
};

bool host_layout(int B, int Hq, int Hkv, int S, int D, int P, HostLayout *L) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || S < 0 || (D != 64 && D != 128) || P < 1 || P > 64) return false;
  const size_t rows = static_cast<size_t>(B) * Hq * S, kv_rows = static_cast<size_t>(B) * Hkv * S;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up_256(off + bytes);
    return at;
  };
  L->q = take(rows * D * 2);
  L->k = take(kv_rows * D * 2);
  L->v = take(kv_rows * D * 2);
  L->o_parts = take(P > 1 ? static_cast<size_t>(P) * rows * D * sizeof(float) : 0);
  L->lse_parts = take(P > 1 ? static_cast<size_t>(P) * rows * sizeof(float) : 0);
  L->o = take(rows * D * 2);
  L->lse = take(rows * sizeof(float));
  L->total = off;
  return true;
}

// One non-blocking copy stream per device, created on the first call there.
std::mutex g_copy_stream_mutex;
cudaStream_t g_copy_stream[kMaxDevices] = {};

int copy_stream(cudaStream_t *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_copy_stream_mutex);
  if (!g_copy_stream[dev]) {
    cudaStream_t s = nullptr;
    e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e);
    g_copy_stream[dev] = s;
  }
  *out = g_copy_stream[dev];
  return ATTN_OK;
}

// `waiter` waits for the work queued on `signaller` so far.
cudaError_t stream_wait(cudaStream_t waiter, cudaStream_t signaller) {
  cudaEvent_t ev = nullptr;
  cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return e;
  e = cudaEventRecord(ev, signaller);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(waiter, ev, 0);
  const cudaError_t d = cudaEventDestroy(ev);  // released once the event completes
  return e != cudaSuccess ? e : d;
}

}  // namespace

extern "C" size_t attn_ring_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int S, int D, int P) {
  HostLayout L;
  return host_layout(B, Hq, Hkv, S, D, P, &L) ? L.total : 0;
}

extern "C" int attn_ring_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                                  void *workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int S,
                                  int D, int P, int causal, float scale, attn_stream_t stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || S < 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (P < 1 || P > 64 || S % P != 0) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (S > kMaxRowsPerHead) return ATTN_ERR_UNSUPPORTED;
  HostLayout L;
  if (!host_layout(B, Hq, Hkv, S, D, P, &L)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || S == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse || !workspace) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < L.total) return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream), cs = nullptr;
  int rc = copy_stream(&cs);
  if (rc != ATTN_OK) return rc;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  unsigned char *qd = ws + L.q, *kd = ws + L.k, *vd = ws + L.v;
  float *o_parts = reinterpret_cast<float *>(ws + L.o_parts), *lse_parts = reinterpret_cast<float *>(ws + L.lse_parts);
  void *od = ws + L.o;
  float *lsed = reinterpret_cast<float *>(ws + L.lse);
  const size_t rows = static_cast<size_t>(B) * Hq * S;
  const size_t head_bytes = static_cast<size_t>(S) * D * 2;  // one head's K or V rows
  const int C = S / P;
  const size_t chunk_bytes = static_cast<size_t>(C) * D * 2;
  // the uploads start after the work queued on `stream` before this call
  cudaError_t e = stream_wait(cs, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(qd, q, rows * D * 2, cudaMemcpyHostToDevice, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  for (int j = 0; j < P; ++j) {
    // chunk j of every (batch, KV head): B*Hkv rows of chunk_bytes, head_bytes apart
    const size_t off = static_cast<size_t>(j) * chunk_bytes;
    e = cudaMemcpy2DAsync(kd + off, head_bytes, static_cast<const unsigned char *>(k) + off, head_bytes,
                          chunk_bytes, static_cast<size_t>(B) * Hkv, cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(vd + off, head_bytes, static_cast<const unsigned char *>(v) + off, head_bytes,
                            chunk_bytes, static_cast<size_t>(B) * Hkv, cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = stream_wait(st, cs);  // chunk j (and Q) on the device
    if (e != cudaSuccess) return cuda_fail(e);
    if (P > 1) {
      rc = attn_partial(qd, kd + off, vd + off, 0, static_cast<long long>(j) * C, static_cast<long long>(S) * D,
                        o_parts + static_cast<size_t>(j) * rows * D, lse_parts + static_cast<size_t>(j) * rows,
                        B, Hq, Hkv, S, C, D, causal, scale, ATTN_PARTIAL_SKIP_EMPTY, stream);
      if (rc != ATTN_OK) return rc;
    }
  }
  rc = P > 1 ? lse_merge(o_parts, lse_parts, P, od, ATTN_BF16, lsed, B, Hq, S, D, stream)
             : attn_fwd(qd, kd, vd, od, lsed, B, Hq, Hkv, S, D, causal, scale, stream);
  if (rc != ATTN_OK) return rc;
  e = cudaMemcpyAsync(o, od, rows * D * 2, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(lse, lsed, rows * sizeof(float), cudaMemcpyDeviceToHost, st);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}
