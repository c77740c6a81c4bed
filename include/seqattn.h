/*
 * seqattn -- blockwise exact attention and log-sum-exp merge for GB300 (sm_103a).
 *
 * C ABI of libseqattn.so. Every entry point takes plain device pointers and
 * sizes, enqueues its kernels on the caller's CUDA stream and returns a status
 * code; nothing is thrown across this boundary and no call synchronises,
 * except attn_query_device_error().
 *
 * Common conventions
 *   Layout     Q and O are [B, Hq, S, D], K and V are [B, Hkv, S, D], lse is
 *              [B, Hq, S]; all row-major with D innermost (the [B, H, L, D]
 *              layout of the listings on page "Ulysses与Ring-Attention序列并行
 *              技术详解").
 *   GQA        query head hq reads KV head hq / (Hq / Hkv); Hq % Hkv == 0.
 *   scale      multiplies Q K^T before the softmax; pass 1/sqrt(D) for the
 *              pages' scaling. Must be finite and > 0.
 *   lse        natural logarithm of the softmax normaliser of each query row:
 *              lse = ln(sum_j exp(scale * q . k_j)) over the visible keys.
 *   Masking    with causal != 0, query row r (global position q_off + r) sees
 *              key j (global position kv_off + j) iff kv_off + j <= q_off + r.
 *              A row that sees no key gets O = 0 and lse = -inf.
 *   Ownership  all buffers are allocated and owned by the caller; the library
 *              allocates no device memory. Pointers must be 16-byte aligned.
 *   Inputs     must be finite (inf/NaN inputs give unspecified outputs).
 *   Empty      B == 0, S == 0 (or Sq == 0) is a valid no-op returning ATTN_OK.
 *   Errors     invalid arguments return ATTN_ERR_INVALID_ARG or
 *              ATTN_ERR_UNSUPPORTED before anything is launched; a failed launch
 *              returns ATTN_ERR_CUDA (the cudaError_t is kept for
 *              attn_last_cuda_error()). Device-side waits are bounded: a wait
 *              that runs out records a code that attn_query_device_error()
 *              reports as ATTN_ERR_TIMEOUT.
 */
#ifndef SEQATTN_H
#define SEQATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or stride */
    ATTN_ERR_UNSUPPORTED = 2, /* head dim other than 64 or 128, shape past limits */
    ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
    ATTN_ERR_TIMEOUT = 4      /* a device-side wait ran out (see attn_query_device_error) */
} attn_status;

typedef enum { ATTN_BF16 = 0, ATTN_F32 = 1 } attn_dtype;

/*
 * attn_fwd -- exact attention softmax(scale * Q K^T) V in one pass, computed
 * tile by tile over K/V with a running maximum and normaliser (the tiled
 * online-softmax forward of page "ms-swift集成FlashAttention 2/3，长文本训练
 * 更高效", section "FlashAttention 如何破局？不只是融合内核"); the scores never
 * reach memory.
 *
 *   q    bf16 [B, Hq, S, D]            k, v  bf16 [B, Hkv, S, D]
 *   o    bf16 [B, Hq, S, D] (output)   lse   fp32 [B, Hq, S] (output)
 *   D    64 or 128.  causal: 0 or 1 (q_off = kv_off = 0).
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
             int Hkv, int S, int D, int causal, float scale, attn_stream_t stream);

/*
 * attn_partial -- attention of a block of queries against one chunk of keys
 * and values: the per-hop partial result of Ring-Attention (page
 * "Ulysses与Ring-Attention序列并行技术详解", Ring-Attention part: each hop
 * attends the local queries to the K/V chunk just received). The result is
 * normalised within the chunk and carries its own lse, ready for lse_merge.
 *
 *   q         bf16 [B, Hq, Sq, D], contiguous.
 *   k_chunk, v_chunk  bf16; key t of KV head (b, h) is the D contiguous values at
 *             k_chunk + ((b*Hkv + h) * kv_head_stride + t*D). kv_head_stride is
 *             in elements; 0 means Skv*D (a contiguous [B,Hkv,Skv,D] chunk). A
 *             chunk of a larger [B,Hkv,S,D] tensor is passed without a copy as
 *             k + j0*D with kv_head_stride = S*D. Must be a multiple of 8.
 *   q_off, kv_off  global positions of query row 0 and key 0 (used by causal).
 *   o_part    fp32 [B, Hq, Sq, D] (output, normalised by the chunk's softmax
 *             sum; rows that see no key of the chunk are 0).
 *   lse_part  fp32 [B, Hq, Sq] (output; -inf where the row sees no key).
 *   flags     0, or ATTN_PARTIAL_SKIP_EMPTY: rows that see no key of the chunk
 *             get lse_part = -inf and their o_part row is left unwritten (its
 *             previous contents stay). lse_merge never reads such rows, so a
 *             ring loop feeding lse_merge can skip those writes.
 */
#define ATTN_PARTIAL_SKIP_EMPTY 1
int attn_partial(const void *q, const void *k_chunk, const void *v_chunk, long long q_off,
                 long long kv_off, long long kv_head_stride, float *o_part, float *lse_part,
                 int B, int Hq, int Hkv, int Sq, int Skv, int D, int causal, float scale, int flags,
                 attn_stream_t stream);

/*
 * lse_merge -- combine P partial results per query row in log space (the
 * output_acc / logsumexp_acc accumulation of page "Ulysses与Ring-Attention序列
 * 并行技术详解", Ring-Attention part, read per row with an empty accumulator
 * at lse = -inf):
 *     M = max_i lse_i,  w_i = exp(lse_i - M),  lse = M + ln(sum_i w_i),
 *     O = sum_i w_i O_i / sum_i w_i;   all lse_i = -inf  ->  O = 0, lse = -inf.
 * Partials with lse_i = -inf are not read.
 *
 *   o_parts   fp32 [P, B, H, S, D]     lse_parts  fp32 [P, B, H, S]
 *   o         [B, H, S, D], bf16 or fp32 per o_dtype (output). With ATTN_F32 it
 *             may be o_parts itself (part 0), merged in place.
 *   lse       fp32 [B, H, S] (output; may be lse_parts itself).
 *   P >= 1, D 64 or 128.
 */
int lse_merge(const float *o_parts, const float *lse_parts, int P, void *o, int o_dtype,
              float *lse, int B, int H, int S, int D, attn_stream_t stream);

/* Synchronises `stream`, then returns ATTN_OK, or ATTN_ERR_TIMEOUT if a kernel
 * recorded a timed-out wait since the last query (the record is cleared), or
 * ATTN_ERR_CUDA if the synchronisation failed. */
int attn_query_device_error(attn_stream_t stream);

/* Static English text for a status code. */
const char *attn_status_string(int status);

/* The cudaError_t of the most recent ATTN_ERR_CUDA (0 if none). */
int attn_last_cuda_error(void);

/*
 * attn_debug_expire_wait -- test hook for the bounded-wait path (no
 * counterpart on the pages). Enqueues a one-CTA kernel that waits on an
 * mbarrier nothing ever arrives at; after timeout_us (1 .. 1e6) the wait gives
 * up the same way a stuck attention pipeline's wait does: it records a
 * timeout in the device error word. Until attn_query_device_error() reports
 * and clears it, later attention launches skip their work (every row comes
 * out as O = 0, lse = -inf). Faults nothing; the context stays usable.
 */
int attn_debug_expire_wait(unsigned timeout_us, attn_stream_t stream);

/*
 * attn_debug_exp2 -- test hook for the softmax exponentials (no counterpart on
 * the pages): y[i] = 2^x[i] computed by the same device code the attention
 * kernels use, the FMA-pipe polynomial (poly = 1) or the MUFU ex2 (poly = 0).
 * x, y: device fp32 arrays of n elements (owned by the caller). Asynchronous
 * on `stream`. ATTN_ERR_INVALID_ARG for n < 0, a null pointer with n > 0, or
 * poly other than 0 / 1.
 */
int attn_debug_exp2(const float *x, float *y, long long n, int poly, attn_stream_t stream);

/*
 * attn_block -- one block of attention over row ranges of packed tensors
 * (heads outermost, rows contiguous per head, D innermost): the queries in
 * rows [q_row, q_row + Sq) of every head of Q against the keys and values in
 * rows [kv_row, kv_row + Skv) of K / V, written to rows [o_row, o_row + Sq) of
 * part `part` of O and lse. q_pos / kv_pos are the global sequence positions of the block's
 * query row 0 and key 0: under the causal mask query i sees key j iff
 * kv_pos + j <= q_pos + i (the masking of page "Ulysses与Ring-Attention序列并行
 * 技术详解", Ring-Attention part, at global positions; a row that sees no key
 * gets O = 0, lse = -inf).
 */
typedef struct {
  long long q_row, kv_row, o_row;
  long long q_pos, kv_pos;
  int Sq, Skv;
  int part;
} attn_block;

/*
 * attn_partial_blocks -- several attn_partial blocks in one persistent launch
 * (per 64 blocks): e.g. the blocks one Ring-Attention device computes at one
 * hop, or every chunk of a ring pass at once.
 *   q         bf16 [B, Hq, q_rows, D];  k, v  bf16 [B, Hkv, kv_rows, D]
 *   o_part    fp32 [n_parts, B, Hq, o_rows, D];  lse_part fp32 [n_parts, B, Hq, o_rows]
 *             (the layout lse_merge reads); block b writes part b.part
 *   blocks    host array of n_blocks attn_block (read during the call only)
 *   flags     0 or ATTN_PARTIAL_SKIP_EMPTY (as for attn_partial)
 * Each block's O rows are normalised within the block (a partial, merged by
 * lse_merge). Rows of K / V past a block's end, up to the next multiple of
 * 128, are read and masked: they must hold finite values (they do when they
 * belong to other blocks or to the same tensor). Blocks must lie inside the
 * tensors, 0 <= part < n_parts, and the output rows of blocks of the same
 * part must not overlap, else
 * ATTN_ERR_INVALID_ARG (as for bad shapes, pointers or alignment); head dims
 * other than 64 / 128: ATTN_ERR_UNSUPPORTED. Device pointers owned by the
 * caller; asynchronous on `stream`.
 */
int attn_partial_blocks(const void *q, const void *k, const void *v, float *o_part,
                        float *lse_part, const attn_block *blocks, int n_blocks, int B, int Hq,
                        int Hkv, long long q_rows, long long kv_rows, long long o_rows,
                        int n_parts, int D, int causal, float scale, int flags,
                        attn_stream_t stream);

/*
 * attn_fwd_varlen -- attention over packed variable-length sequences (the
 * packing of page "ms-swift集成FlashAttention 2/3，长文本训练更高效": sequences
 * concatenated without padding, attention kept within each sequence).
 *   q, o       bf16 [Hq, total_q, D]   (sequence s in rows cu_seqlens_q[s] ..)
 *   k, v       bf16 [Hkv, total_k, D]  (rows cu_seqlens_k[s] ..)
 *   lse        fp32 [Hq, total_q]      (natural log)
 *   cu_seqlens_q / cu_seqlens_k  host int64 arrays of nseq + 1 entries, starting
 *              at 0, non-decreasing; total_q / total_k are their last entries
 * Causal masks are aligned at the bottom right of each sequence: query row i
 * of a sequence sees key j iff j <= i + Skv_s - Sq_s (the usual mask when
 * Sq_s == Skv_s). Sequences with no query rows are skipped; rows that see no
 * key get O = 0, lse = -inf. Errors as for attn_partial_blocks.
 */
int attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                    const long long *cu_seqlens_q, const long long *cu_seqlens_k, int nseq, int Hq,
                    int Hkv, int D, int causal, float scale, attn_stream_t stream);

/*
 * attn_fwd_fp8 -- attention with e4m3 (FP8) Q, K, V and per-tensor scales (the
 * FP8 attention of FlashAttention-3, page "ms-swift集成FlashAttention 2/3，
 * 长文本训练更高效"): with q = q_scale * Q8, k = k_scale * K8, v = v_scale * V8,
 * softmax(scale * q k^T) v and its lse, as attn_fwd. Both products run on the
 * e4m3 tensor cores with fp32 accumulation; P is rounded to e4m3 before P V
 * (the normaliser l is summed from the unrounded P).
 *   q8      e4m3 [B, Hq, S, 128]; k8  e4m3 [B, Hkv, S, 128]
 *   vt8     e4m3 [B, Hkv, 128, S]  (V transposed: keys contiguous)
 *   o       bf16 [B, Hq, S, 128];  lse  fp32 [B, Hq, S] (natural log)
 * Head dim 128 only and S a multiple of 16 (else ATTN_ERR_UNSUPPORTED); scales
 * finite and positive, aligned pointers (else ATTN_ERR_INVALID_ARG). Device
 * pointers owned by the caller; asynchronous on `stream`.
 */
int attn_fwd_fp8(const void *q8, const void *k8, const void *vt8, void *o, float *lse, int B, int Hq,
                 int Hkv, int S, int D, int causal, float scale, float q_scale, float k_scale,
                 float v_scale, attn_stream_t stream);

/*
 * attn_bwd -- gradients of attention (dQ, dK, dV) for the output gradient dO,
 * recomputing the scores tile by tile from Q, K and the forward's lse (the
 * backward FlashAttention recomputes block by block, page "ms-swift集成
 * FlashAttention 2/3，长文本训练更高效"):
 *   P = exp(scale Q K^T - lse),  delta_i = <dO_i, O_i>,
 *   dV = P^T dO,  dS = P * (dO V^T - delta),  dK = scale dS^T Q,  dQ = scale dS K,
 * dK and dV summed over the query heads of each GQA group.
 *   q, o, dout  bf16 [B, Hq, S, D];  k, v  bf16 [B, Hkv, S, D]
 *   lse         fp32 [B, Hq, S] from attn_fwd (natural log)
 *   delta       fp32 [B, Hq, S] workspace (written, then read)
 *   dq          bf16 [B, Hq, S, D];  dk, dv  bf16 [B, Hkv, S, D]  (outputs)
 * D in {64, 128}, S <= 2^30 and B * Hq <= 65535 (else ATTN_ERR_UNSUPPORTED); bad
 * shapes, scale, pointers or alignment: ATTN_ERR_INVALID_ARG. Device pointers
 * owned by the caller; asynchronous on `stream`.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
             const void *dout, float *delta, void *dq, void *dk, void *dv, int B, int Hq, int Hkv,
             int S, int D, int causal, float scale, attn_stream_t stream);

/*
 * attn_ring_fwd_host_workspace_bytes -- bytes of device workspace that
 * attn_ring_fwd_host needs for these sizes (device copies of Q, K, V, the
 * fp32 partials when P > 1, and O and lse), or 0 for invalid sizes.
 */
size_t attn_ring_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int S, int D, int P);

/*
 * attn_ring_fwd_host -- the ring-emulated forward from host buffers to host
 * buffers: the Ring-Attention pass of the page "Ulysses与Ring-Attention序列
 * 并行技术详解" with each hop's K/V chunk arriving over the host link. Q and
 * then every K/V chunk are copied to the device on an internal copy stream;
 * chunk j's attn_partial starts on `stream` as soon as chunk j has arrived, so
 * the copies of later chunks overlap it; then lse_merge and the copies of O
 * and lse back to the host, on `stream`. P = 1: one attn_fwd after the copies.
 *   q, k, v   host bf16 [B, Hq, S, D], [B, Hkv, S, D], [B, Hkv, S, D]
 *             (page-locked, or the copies cannot overlap anything)
 *   o, lse    host bf16 [B, Hq, S, D], fp32 [B, Hq, S] (outputs, page-locked
 *             likewise)
 *   workspace device memory, 256-byte aligned, at least
 *             attn_ring_fwd_host_workspace_bytes(B, Hq, Hkv, S, D, P) bytes,
 *             owned by the caller; no other call may use it at the same time.
 * Asynchronous: the call returns once everything is queued; o and lse hold
 * the result when `stream` reaches the end of the call. The uploads of a call
 * wait for the work queued on `stream` before it (and so for an earlier call
 * on that stream that used the same workspace); a caller that alternates two
 * (stream, workspace, o/lse) sets overlaps one call's uploads with the
 * previous call's compute and downloads. Host-side inputs must stay unchanged,
 * and outputs unread, until then.
 * Rules as attn_fwd (D 64 or 128), plus 1 <= P <= 64 and S % P == 0. Errors as
 * attn_fwd; ATTN_ERR_INVALID_ARG also for a null pointer or a workspace that is
 * too small or misaligned. Chunk j's partial is attn_partial with
 * ATTN_PARTIAL_SKIP_EMPTY, so results equal those of the device-side ring with
 * one attn_partial per chunk.
 */
int attn_ring_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, void *workspace,
                       size_t workspace_bytes, int B, int Hq, int Hkv, int S, int D, int P, int causal,
                       float scale, attn_stream_t stream);

/* Size of the library's fixed scratch array used by attn_ring_fwd_static. */
#define SEQATTN_RING_SCRATCH_BYTES (64ull << 20) /* 64 MiB */

/*
 * attn_ring_fwd_static -- the ring-emulated forward (keys split into P equal
 * chunks, one attn_partial per chunk, then lse_merge into bf16 o and fp32 lse),
 * with the fp32 partials kept in a fixed device array owned by the library
 * instead of in memory the caller provides. The source pages have no
 * counterpart to this entry point; it exists for callers that must not or
 * cannot allocate device memory themselves: code inside a host application
 * whose allocator already holds nearly all device memory, or latency-sensitive
 * loops that cannot afford cudaMalloc/cudaFree (which may synchronise the
 * device). It allocates nothing.
 *
 *   q  bf16 [B, Hq, S, D]; k, v bf16 [B, Hkv, S, D]; o bf16 [B, Hq, S, D];
 *   lse fp32 [B, Hq, S]. S % P == 0. Other rules as attn_fwd.
 *   Limit: P * B * Hq * S * (D + 1) * 4 bytes (each part rounded up to 256 B)
 *   must fit in SEQATTN_RING_SCRATCH_BYTES; larger problems are rejected with
 *   ATTN_ERR_UNSUPPORTED before anything is launched.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture on the device. Every call on a device shares the one array: calls
 *   whose kernels overlap on the GPU (different streams, no ordering between
 *   them) race on it and give wrong results. Each call writes every partial
 *   element it reads, so the contents left by an earlier call do no harm.
 */
int attn_ring_fwd_static(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                         int Hq, int Hkv, int S, int D, int P, int causal, float scale,
                         attn_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SEQATTN_H */
