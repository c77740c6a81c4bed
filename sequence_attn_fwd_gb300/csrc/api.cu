// C-ABI entry points of libseqattn.so (declared in include/seqattn.h):
// argument validation, TMA tensor-map construction and kernel launch. No
// entry point allocates device memory or synchronises, except the explicit
// device-error query.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

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
// 64 x 128 x 1 with 128-byte swizzle. Rows past `rows` read as zero.
bool make_map(CUtensorMap *map, const void *base, int D, long long rows, long long heads,
              long long head_stride) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2u,
                           static_cast<cuuint64_t>(head_stride) * 2u};
  cuuint32_t box[3] = {64u, 128u, 1u};
  cuuint32_t estride[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool scale_ok(float scale) { return isfinite(scale) && scale > 0.f; }

constexpr long long kMaxRowsPerHead = 1ll << 30;  // keeps every row index within int range

int run_attention(const void *q, const void *k, const void *v, long long q_off, long long kv_off,
                  long long kv_head_stride, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
                  int Skv, int D, int causal, float scale, bool f32_out, cudaStream_t stream) {
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

  CUtensorMap tq, tk, tv;
  // An empty key set still needs well-formed maps; no KV tile is ever loaded.
  const long long kv_rows = Skv > 0 ? Skv : 1;
  if (!make_map(&tq, q, D, Sq, static_cast<long long>(B) * Hq, static_cast<long long>(Sq) * D) ||
      !make_map(&tk, k, D, kv_rows, static_cast<long long>(B) * Hkv, kv_head_stride) ||
      !make_map(&tv, v, D, kv_rows, static_cast<long long>(B) * Hkv, kv_head_stride))
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
  cudaError_t e = seqattn::launch_attention(D, f32_out, tq, tk, tv, p, stream);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
             int Hkv, int S, int D, int causal, float scale, attn_stream_t stream) {
  return run_attention(q, k, v, 0, 0, 0, o, lse, B, Hq, Hkv, S, S, D, causal, scale, false,
                       reinterpret_cast<cudaStream_t>(stream));
}

int attn_partial(const void *q, const void *k_chunk, const void *v_chunk, long long q_off,
                 long long kv_off, long long kv_head_stride, float *o_part, float *lse_part,
                 int B, int Hq, int Hkv, int Sq, int Skv, int D, int causal, float scale,
                 attn_stream_t stream) {
  return run_attention(q, k_chunk, v_chunk, q_off, kv_off, kv_head_stride, o_part, lse_part, B, Hq,
                       Hkv, Sq, Skv, D, causal, scale, true, reinterpret_cast<cudaStream_t>(stream));
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

}  // extern "C"
