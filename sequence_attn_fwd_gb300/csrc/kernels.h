// Host-side interface between the C-ABI layer (api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace seqattn {

// Parameters of one attention launch (attn_fwd or attn_partial).
struct AttnParams {
  void *o;            // [B, Hq, Sq, D] bf16 (attn_fwd) or fp32 (attn_partial)
  float *lse;         // [B, Hq, Sq]
  int B, Hq, Hkv, Sq, Skv;
  long long q_off, kv_off;  // global positions of query row 0 and key 0
  float scale_log2;   // softmax scale times log2(e)
  int causal;
  int n_qblocks;      // ceil(Sq / 256): two 128-row query tiles per CTA
  int skip_empty;     // rows that see no key: write lse = -inf only, leave O untouched
  long long o_rows;   // rows per head of O and lse (Sq for a single problem)
  float o_scale;      // e4m3 attention: the V scale applied to O (1 otherwise)
  int heads_per_chunk;  // single problems: items come in chunks of this many consecutive
                        // heads (whole GQA groups), all query blocks of a chunk before the next
};

// One block of attention: the queries in rows [q_row, q_row + Sq) of Q (per
// head) against the keys and values in rows [kv_row, kv_row + Skv) of K / V,
// written to rows [o_row, o_row + Sq) of part `part` of O and lse (O viewed as
// [parts][B * Hq heads][rows][D]). q_pos / kv_pos are the global positions of
// query row 0 and key 0 (the causal mask compares them).
struct BlockDesc {
  long long q_row, kv_row, o_row;
  long long q_pos, kv_pos;
  int Sq, Skv;
  int part;
};

// The blocks of one launch, passed by value in the kernel parameters.
// item_start[i] is the first work item of block i (items: B * Hq heads times
// ceil(Sq / 256) query blocks per block), item_start[n] the total.
constexpr int kMaxLaunchBlocks = 64;
struct BlockTable {
  int n;
  long long item_start[kMaxLaunchBlocks + 1];
  BlockDesc b[kMaxLaunchBlocks];
};

// Blocks that share their query rows (q_row, o_row, q_pos and Sq equal to
// block 0's), such as the key chunks of a ring pass: a work item is 256 of
// those rows of one (batch, head) taken against every block in turn, each
// block a segment of the item with its own partial, Q loaded once.
struct SegTable {
  int n;
  BlockDesc b[kMaxLaunchBlocks];
};

// Number of SMs of the current device (read once per device).
int device_sm_count();

// Tensor maps are 3-D views [heads][rows][D] built by the caller: q, k, v of
// bf16 data, box 64 columns x 128 rows x 1; o of the output type (fp32 when
// f32_out, else bf16), box 128 bytes x 32 rows x 1 (one warp's rows); all with
// 128-byte swizzle.
cudaError_t launch_attention(int D, bool f32_out, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                             const CUtensorMap &tm_v, const CUtensorMap &tm_o, const AttnParams &p,
                             cudaStream_t stream);

// Backward (head dim 64 or 128): gradients of a forward whose O and lse are given.
struct BwdParams {
  const float *lse;    // [B*Hq, S] natural log (the forward's)
  const float *delta;  // [B*Hq, S] workspace: <dO_i, O_i>, written by the first kernel
  void *dq, *dk, *dv;  // bf16 [B*Hq, S, D], [B*Hkv, S, D] x 2
  int B, Hq, Hkv, S;
  float scale;         // softmax scale
  int causal;
};

// delta, then dK / dV (grid: key tiles x B*Hkv), then dQ (grid: query tiles x
// B*Hq); maps over bf16 [heads][S][D], box 64 x 128 x 1, 128-byte swizzle.
cudaError_t launch_attention_bwd(int D, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                 const CUtensorMap &tm_v, const CUtensorMap &tm_do,
                                 const void *o, const void *dout, float *delta,
                                 const BwdParams &p, cudaStream_t stream);

// e4m3 attention (D = 128, bf16 O): tq / tk over e4m3 [heads][S][128] with
// box 128 x 128 x 1, tvt over V^T e4m3 [kv heads][128][S] with box 128 (keys)
// x 128 x 1, all 128-byte swizzle; p.scale_log2 includes the Q and K scales,
// p.o_scale is the V scale.
cudaError_t launch_attention_fp8(const CUtensorMap &tq, const CUtensorMap &tk,
                                 const CUtensorMap &tvt, const CUtensorMap &to,
                                 const AttnParams &p, cudaStream_t stream);

// The single-SM persistent kernel over a table of blocks (row ranges of the
// maps' row dimension; p's Sq / Skv / q_off / kv_off / n_qblocks are unused).
cudaError_t launch_attention_blocks(int D, bool f32_out, const CUtensorMap &tm_q,
                                    const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                    const CUtensorMap &tm_o, const AttnParams &p,
                                    const BlockTable &tbl, cudaStream_t stream);

// The same kernel over a table of blocks that share their query rows (see
// SegTable; p's Sq / Skv / q_off / kv_off / n_qblocks are unused): fp32
// partials of blocks of at most 2048 keys (anything else is refused with
// cudaErrorInvalidValue).
cudaError_t launch_attention_segments(int D, bool f32_out, const CUtensorMap &tm_q,
                                      const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                      const CUtensorMap &tm_o, const AttnParams &p,
                                      const SegTable &tbl, cudaStream_t stream);

cudaError_t launch_lse_merge(const float *o_parts, const float *lse_parts, int P, long long nrows,
                             int D, void *o, bool bf16_out, float *lse, cudaStream_t stream);

// One CTA waits on an mbarrier nothing arrives at until timeout_us runs out.
cudaError_t launch_expire_wait(unsigned timeout_us, cudaStream_t stream);

// y[i] = 2^x[i] by the softmax's exponential routine (polynomial or MUFU).
cudaError_t launch_exp2_probe(const float *x, float *y, long long n, bool poly,
                              cudaStream_t stream);

// Reads and clears the device error word (after the caller synchronised).
cudaError_t read_and_clear_device_error(int *code);

}  // namespace seqattn
