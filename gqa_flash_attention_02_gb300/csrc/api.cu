// C ABI of the library (declared in include/gqa_attn.h): argument
// validation, the per-(device, stream) workspace, TMA tensor-map encoding and
// dispatch to the kernels. No torch types cross this boundary.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include "gqa_attn.h"
#include "gqa_internal.h"

using namespace gqa;

namespace {

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = e;
  cudaGetLastError();  // clear the sticky-free error state for this thread
  return GQA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ workspace

struct WsKey {
  int dev;
  cudaStream_t stream;
  bool operator<(const WsKey &o) const {
    return dev != o.dev ? dev < o.dev : reinterpret_cast<uintptr_t>(stream) < reinterpret_cast<uintptr_t>(o.stream);
  }
};

std::mutex g_ws_mutex;
std::map<WsKey, Workspace> g_ws;
std::map<int, int> g_num_sms;

int device_sms(int dev) {
  std::lock_guard<std::mutex> lk(g_ws_mutex);
  auto it = g_num_sms.find(dev);
  if (it != g_num_sms.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  g_num_sms[dev] = n;
  return n;
}

// Returns the workspace of (current device, stream) with at least
// `partials_bytes` of partials space and `counters` zeroed decode counters;
// creates or grows it stream-ordered.
int get_workspace(cudaStream_t stream, size_t partials_bytes, Workspace **out,
                  size_t counters = 0, size_t units = 0) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  std::lock_guard<std::mutex> lk(g_ws_mutex);
  Workspace &ws = g_ws[WsKey{dev, stream}];
  if (ws.ctl == nullptr) {
    void *p = nullptr;
    e = cudaMallocAsync(&p, kCtlInts * sizeof(int), stream);
    if (e != cudaSuccess) {
      g_ws.erase(WsKey{dev, stream});
      cudaGetLastError();
      return GQA_ERR_OOM;
    }
    e = cudaMemsetAsync(p, 0, kCtlInts * sizeof(int), stream);
    if (e != cudaSuccess) return cuda_fail(e);
    ws.ctl = static_cast<int *>(p);
  }
  if (partials_bytes > ws.partials_bytes) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap != cudaStreamCaptureStatusNone)
      return GQA_ERR_OOM;  // cannot grow while capturing: warm up outside the capture first
    if (ws.partials) cudaFreeAsync(ws.partials, stream);
    ws.partials = nullptr;
    ws.partials_bytes = 0;
    void *p = nullptr;
    // grow geometrically so a sweep of shapes does not reallocate each call
    size_t want = partials_bytes < (1u << 20) ? (1u << 20) : partials_bytes + partials_bytes / 4;
    e = cudaMallocAsync(&p, want, stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return GQA_ERR_OOM;
    }
    ws.partials = static_cast<float *>(p);
    ws.partials_bytes = want;
  }
  if (counters > ws.counters_len) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap != cudaStreamCaptureStatusNone)
      return GQA_ERR_OOM;
    if (ws.counters) cudaFreeAsync(ws.counters, stream);
    ws.counters = nullptr;
    ws.counters_len = 0;
    void *p = nullptr;
    const size_t want = counters < 4096 ? 4096 : counters + counters / 4;
    e = cudaMallocAsync(&p, want * sizeof(int), stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return GQA_ERR_OOM;
    }
    e = cudaMemsetAsync(p, 0, want * sizeof(int), stream);
    if (e != cudaSuccess) return cuda_fail(e);
    ws.counters = static_cast<int *>(p);
    ws.counters_len = want;
  }
  if (units > ws.units_len) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap != cudaStreamCaptureStatusNone)
      return GQA_ERR_OOM;
    if (ws.units) cudaFreeAsync(ws.units, stream);
    ws.units = nullptr;
    ws.units_len = 0;
    void *p = nullptr;
    const size_t want = units < 4096 ? 4096 : units + units / 4;
    e = cudaMallocAsync(&p, want * sizeof(int4), stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return GQA_ERR_OOM;
    }
    ws.units = static_cast<int4 *>(p);
    ws.units_len = want;
  }
  *out = &ws;
  return GQA_OK;
}

// ------------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cudaGetLastError();
  });
  return g_encode;
}

// bf16 tensor viewed as [planes][rows][d]; box = 64 columns x box_rows rows,
// 128-byte swizzle, zero fill outside the tensor.
bool encode_bf16_3d(CUtensorMap *map, const void *base, int d, long rows, long planes,
                    int box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 tensor [tokens][heads][d] viewed for TMA as (column, head, token) with
// boxes of 64 columns x 1 head x box_rows tokens: in shared memory such a box
// is box_rows rows of 128 bytes, the layout of a [planes][rows][d] box.
bool encode_bf16_thd(CUtensorMap *map, const void *base, int d, long heads, long tokens,
                     int box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(heads) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64u, 1u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 tensor viewed as [planes][rows][d] with a row and a plane stride
// (elements; d contiguous); boxes of 64 columns x box_rows rows, 128-byte
// swizzle, zero fill outside.
bool encode_bf16_3d_strided(CUtensorMap *map, const void *base, int d, long rows, long planes,
                            long long s_row, long long s_plane, int box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(s_row) * 2, static_cast<cuuint64_t>(s_plane) * 2};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 tensor indexed [batch][head][row][d] with the given strides (elements;
// d contiguous) for TMA as (column, row, head, batch): boxes of 64 columns x
// box_rows rows, 128-byte swizzle, zero fill outside (so columns past d and
// rows past `rows` read as zero).
bool encode_bf16_4d(CUtensorMap *map, const void *base, int d, long rows, long heads, long batch,
                    long long s_row, long long s_head, long long s_batch, int box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(s_row) * 2, static_cast<cuuint64_t>(s_head) * 2,
                           static_cast<cuuint64_t>(s_batch) * 2};
  cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(box_rows), 1u, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 8-bit tensor (an fp8 K/V cache) viewed as [planes][rows][d] bytes; box =
// d bytes x box_rows rows with the d-byte swizzle (128 B for d = 128, 64 B
// for d = 64), zero fill outside the tensor.
// fp8 cache [planes][rows][d] bytes; boxes of box_cols (the kernel's width,
// 64 or 128 >= d: zeros past d) x box_rows, swizzled as the kernel reads them.
bool encode_u8_3d(CUtensorMap *map, const void *base, int d, long rows, long planes, int box_cols,
                  int box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d),
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(d)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   box_cols == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

namespace gqa {
// Shared with the other host-side translation units of the library.
bool encode_tensor_map_bf16_thd(CUtensorMap *map, const void *base, int d, long heads,
                                long tokens, int box_rows) {
  return encode_bf16_thd(map, base, d, heads, tokens, box_rows);
}
bool encode_tensor_map_bf16_3d(CUtensorMap *map, const void *base, int d, long rows, long planes,
                               int box_rows) {
  return encode_bf16_3d(map, base, d, rows, planes, box_rows);
}
}  // namespace gqa

namespace {

// ------------------------------------------------------------------ validation

constexpr long long kMaxElems = (1ll << 31) - 1;

int check_prefill_args(const void *q, const void *k, const void *v, const void *o, int B, int H_q,
                       int H_kv, int N_q, int N_kv, int d, int causal, float scale) {
  if (!q || !k || !v || !o) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return GQA_ERR_INVALID_ARG;
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || N_q <= 0 || N_kv <= 0 || d <= 0) return GQA_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (causal && N_q > N_kv) return GQA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H_q * N_q * d > kMaxElems ||
      static_cast<long long>(B) * H_kv * N_kv * d > kMaxElems)
    return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

int check_decode_args(const void *q, const void *kc, const void *vc, const int *seqlens,
                      const void *o, int B, int H_q, int H_kv, int max_len, int d, float scale) {
  if (!q || !kc || !vc || !seqlens || !o) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(o)) return GQA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seqlens) & 3u) != 0) return GQA_ERR_INVALID_ARG;
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || max_len <= 0 || d <= 0) return GQA_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (max_len > (1 << 20)) return GQA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H_kv * max_len * d > kMaxElems ||
      static_cast<long long>(B) * H_q * d > kMaxElems)
    return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

bool d_supported_simt(int d) { return d == 32 || d == 64 || d == 96 || d == 128; }

}  // namespace

namespace {
int decode_bf16(const void *q, const void *k_cache, const void *v_cache, const int *seqlens,
                void *o, float *lse, int B, int H_q, int H_kv, int max_len, int d, float scale,
                int chunk_tokens, cudaStream_t stream, const int *seqlens_first = nullptr) {
  int rc = check_decode_args(q, k_cache, v_cache, seqlens, o, B, H_q, H_kv, max_len, d, scale);
  if (rc != GQA_OK) return rc;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return GQA_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 96 && d != 128 && d != 256) return GQA_ERR_UNSUPPORTED;
  if (!decode_units_fit(B, H_q, H_kv, max_len)) return GQA_ERR_UNSUPPORTED;
  if (chunk_tokens != 0 &&
      (chunk_tokens < 0 || chunk_tokens % kDecodeChunkUnit != 0 || chunk_tokens > kDecodeChunkMax))
    return GQA_ERR_INVALID_ARG;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const int grid = decode_grid(B, H_q, H_kv, max_len, d, device_sms(dev), chunk_tokens);
  Workspace *ws = nullptr;
  rc = get_workspace(stream, decode_partials_bytes(B, H_q, H_kv, d, grid), &ws,
                     decode_planes(B, H_q, H_kv));
  if (rc != GQA_OK) return rc;
  CUtensorMap tq, tk, tv;
  if (!encode_bf16_3d(&tq, q, d, static_cast<long>(B) * H_q, 1, kDecodeHeads) ||
      !encode_bf16_3d(&tk, k_cache, d, max_len, static_cast<long>(B) * H_kv, decode_box_rows(d)) ||
      !encode_bf16_3d(&tv, v_cache, d, max_len, static_cast<long>(B) * H_kv, decode_box_rows(d)))
    return cuda_fail(cudaErrorInvalidValue);
  e = launch_decode_bf16(tq, tk, tv, q, seqlens, o, lse, ws->partials, ws->counters, B, H_q, H_kv,
                         max_len, d, scale, grid, ws->ctl + kCtlErr, stream, seqlens_first);
  return e == cudaSuccess ? GQA_OK : cuda_fail(e);
}
}  // namespace

namespace {
// Dense prefill with the caller's strides (elements; d contiguous): the
// tensor maps are 4-D (column, row, head, batch), so any batch and head
// strides work, e.g. slices of a fused QKV buffer.
bool d_supported_tc(int d) { return d == 32 || d == 64 || d == 96 || d == 128 || d == 256; }

bool strides_ok(long long sb, long long sh, long long sn, int d) {
  // TMA wants 16-byte multiples; rows must not overlap within a head
  return sb > 0 && sh > 0 && sn >= d && sb % 8 == 0 && sh % 8 == 0 && sn % 8 == 0;
}

int fwd_dense(const void *q, long long q_sb, long long q_sh, long long q_sn, const void *k,
              long long k_sb, long long k_sh, long long k_sn, const void *v, long long v_sb,
              long long v_sh, long long v_sn, void *o, long long o_sb, long long o_sh,
              long long o_sn, float *lse, int B, int H_q, int H_kv, int N_q, int N_kv, int d,
              int causal, float scale, cudaStream_t stream) {
  int rc = check_prefill_args(q, k, v, o, B, H_q, H_kv, N_q, N_kv, d, causal, scale);
  if (rc != GQA_OK) return rc;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return GQA_ERR_INVALID_ARG;
  if (!d_supported_tc(d)) return GQA_ERR_UNSUPPORTED;
  if (!strides_ok(q_sb, q_sh, q_sn, d) || !strides_ok(k_sb, k_sh, k_sn, d) ||
      !strides_ok(v_sb, v_sh, v_sn, d) || !strides_ok(o_sb, o_sh, o_sn, d))
    return GQA_ERR_INVALID_ARG;
  const PrefillPlan plan = make_prefill_plan(B, H_q, H_kv, N_q, N_kv, causal, d == 256);
  Workspace *ws = nullptr;
  rc = get_workspace(stream, 0, &ws);
  if (rc != GQA_OK) return rc;
  // When each batch's heads follow one another at the head stride (packed
  // and row-padded layouts), the heads of all batches form one run of
  // planes and 3-D maps serve (column, row, batch * H + head); other views
  // take 4-D maps (column, row, head, batch).
  const bool plane_uniform =
      q_sb == q_sh * H_q && k_sb == k_sh * H_kv && v_sb == v_sh * H_kv;
  CUtensorMap tq, tk, tv;
  bool enc_ok;
  if (plane_uniform)
    enc_ok = encode_bf16_3d_strided(&tq, q, d, N_q, static_cast<long>(B) * H_q, q_sn, q_sh, kTileM) &&
             encode_bf16_3d_strided(&tk, k, d, N_kv, static_cast<long>(B) * H_kv, k_sn, k_sh, kTileN) &&
             encode_bf16_3d_strided(&tv, v, d, N_kv, static_cast<long>(B) * H_kv, v_sn, v_sh, kTileN);
  else
    enc_ok = encode_bf16_4d(&tq, q, d, N_q, H_q, B, q_sn, q_sh, q_sb, kTileM) &&
             encode_bf16_4d(&tk, k, d, N_kv, H_kv, B, k_sn, k_sh, k_sb, kTileN) &&
             encode_bf16_4d(&tv, v, d, N_kv, H_kv, B, v_sn, v_sh, v_sb, kTileN);
  if (!enc_ok) return cuda_fail(cudaErrorInvalidValue);
  int dev = 0;
  cudaGetDevice(&dev);
  const OutView ov{o_sb, o_sh, o_sn, d, plane_uniform ? 0 : 1};
  cudaError_t e = launch_prefill_tc(tq, tk, tv, o, ov, lse, plan, scale, ws->ctl, device_sms(dev),
                                    stream);
  return e == cudaSuccess ? GQA_OK : cuda_fail(e);
}
}  // namespace

extern "C" {

int gqa_attn_fwd_lse(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                     int H_q, int H_kv, int N_q, int N_kv, int d, int causal, float scale,
                     cudaStream_t stream) {
  const long long nq = N_q, nk = N_kv, dd = d;
  return fwd_dense(q, nq * dd * H_q, nq * dd, dd, k, nk * dd * H_kv, nk * dd, dd, v,
                   nk * dd * H_kv, nk * dd, dd, o, nq * dd * H_q, nq * dd, dd, lse, B, H_q, H_kv,
                   N_q, N_kv, d, causal, scale, stream);
}

int gqa_attn_fwd_strided(const void *q, long long q_sb, long long q_sh, long long q_sn,
                         const void *k, long long k_sb, long long k_sh, long long k_sn,
                         const void *v, long long v_sb, long long v_sh, long long v_sn, void *o,
                         long long o_sb, long long o_sh, long long o_sn, int B, int H_q, int H_kv,
                         int N_q, int N_kv, int d, int causal, float scale, cudaStream_t stream) {
  return fwd_dense(q, q_sb, q_sh, q_sn, k, k_sb, k_sh, k_sn, v, v_sb, v_sh, v_sn, o, o_sb, o_sh,
                   o_sn, nullptr, B, H_q, H_kv, N_q, N_kv, d, causal, scale, stream);
}

}  // extern "C"

namespace {
// Ragged batch (cu_* given) or equal lengths uni_q / uni_k ([B][N][H][d],
// cu_* null), packed token-major: the plan kernel, then the prefill kernel.
int fwd_packed(const void *q, const void *k, const void *v, void *o, float *lse, const int *cu_q,
               const int *cu_k, int uni_q, int uni_k, int B, int H_q, int H_kv, int total_q,
               int total_k, int d, int causal, float scale, cudaStream_t stream) {
  if (!q || !k || !v || !o) return GQA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return GQA_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return GQA_ERR_INVALID_ARG;
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || total_q < 0 || total_k < 0 || d <= 0)
    return GQA_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 96 && d != 128 && d != 256) return GQA_ERR_UNSUPPORTED;
  if (B > kVarlenMaxB) return GQA_ERR_UNSUPPORTED;
  if (static_cast<long long>(total_q) * H_q * d > kMaxElems ||
      static_cast<long long>(total_k) * H_kv * d > kMaxElems)
    return GQA_ERR_UNSUPPORTED;
  if (total_q == 0) return GQA_OK;  // no query rows: nothing to compute
  if (total_k == 0) return GQA_ERR_INVALID_ARG;  // rows with no keys
  const int tpu = d == 256 ? 1 : 2;  // one query tile per unit at head dim 256
  const long long most = varlen_max_units(B, H_q, H_kv, total_q, tpu);
  if (most > (1ll << 30)) return GQA_ERR_UNSUPPORTED;
  Workspace *ws = nullptr;
  int rc = get_workspace(stream, 0, &ws, 0, static_cast<size_t>(most));
  if (rc != GQA_OK) return rc;
  CUtensorMap tq, tk, tv;
  if (!encode_bf16_thd(&tq, q, d, H_q, total_q, kTileM) ||
      !encode_bf16_thd(&tk, k, d, H_kv, total_k, kTileN) ||
      !encode_bf16_thd(&tv, v, d, H_kv, total_k, kTileN))
    return cuda_fail(cudaErrorInvalidValue);
  VarlenArgs va;
  va.cu_q = cu_q;
  va.cu_k = cu_k;
  va.uni_q = uni_q;
  va.uni_k = uni_k;
  va.units = ws->units;
  va.B = B;
  va.H_q = H_q;
  va.H_kv = H_kv;
  va.group = H_q / H_kv;
  va.causal = causal ? 1 : 0;
  va.total_q = total_q;
  va.total_k = total_k;
  va.tpu = tpu;
  cudaError_t e = launch_varlen_plan(va, ws->units, ws->ctl, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  int dev = 0;
  cudaGetDevice(&dev);
  const OutView ov{0, d, static_cast<long long>(H_q) * d, d, 0};  // [total_q][H_q][d]
  e = launch_prefill_tc_varlen(tq, tk, tv, o, ov, lse, va, scale, ws->ctl, device_sms(dev), stream);
  return e == cudaSuccess ? GQA_OK : cuda_fail(e);
}
}  // namespace

extern "C" {

int gqa_attn_fwd_varlen_lse(const void *q, const void *k, const void *v, void *o, float *lse,
                            const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int H_q,
                            int H_kv, int total_q, int total_k, int d, int causal, float scale,
                            cudaStream_t stream) {
  if (!cu_seqlens_q || !cu_seqlens_k) return GQA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u) != 0)
    return GQA_ERR_INVALID_ARG;
  return fwd_packed(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, 0, 0, B, H_q, H_kv, total_q,
                    total_k, d, causal, scale, stream);
}

int gqa_attn_fwd_bshd(const void *q, const void *k, const void *v, void *o, int B, int H_q,
                      int H_kv, int N_q, int N_kv, int d, int causal, float scale,
                      cudaStream_t stream) {
  if (B <= 0 || N_q <= 0 || N_kv <= 0) return GQA_ERR_INVALID_ARG;
  if (causal && N_q > N_kv) return GQA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * N_q > INT32_MAX || static_cast<long long>(B) * N_kv > INT32_MAX)
    return GQA_ERR_UNSUPPORTED;
  return fwd_packed(q, k, v, o, nullptr, nullptr, nullptr, N_q, N_kv, B, H_q, H_kv, B * N_q,
                    B * N_kv, d, causal, scale, stream);
}

int gqa_attn_fwd_varlen(const void *q, const void *k, const void *v, void *o,
                        const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int H_q, int H_kv,
                        int total_q, int total_k, int d, int causal, float scale,
                        cudaStream_t stream) {
  return gqa_attn_fwd_varlen_lse(q, k, v, o, nullptr, cu_seqlens_q, cu_seqlens_k, B, H_q, H_kv,
                                 total_q, total_k, d, causal, scale, stream);
}

int gqa_attn_fwd(const void *q, const void *k, const void *v, void *o, int B, int H_q, int H_kv,
                 int N_q, int N_kv, int d, int causal, float scale, cudaStream_t stream) {
  return gqa_attn_fwd_lse(q, k, v, o, nullptr, B, H_q, H_kv, N_q, N_kv, d, causal, scale, stream);
}

int gqa_attn_fwd_f32(const void *q, const void *k, const void *v, void *o, int B, int H_q,
                     int H_kv, int N_q, int N_kv, int d, int causal, float scale,
                     cudaStream_t stream) {
  int rc = check_prefill_args(q, k, v, o, B, H_q, H_kv, N_q, N_kv, d, causal, scale);
  if (rc != GQA_OK) return rc;
  if (!d_supported_simt(d)) return GQA_ERR_UNSUPPORTED;
  Workspace *ws = nullptr;
  rc = get_workspace(stream, 0, &ws);
  if (rc != GQA_OK) return rc;
  cudaError_t e = launch_attn_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                                  static_cast<const float *>(v), static_cast<float *>(o), B, H_q,
                                  H_kv, N_q, N_kv, d, causal, scale, nullptr, N_kv,
                                  ws->ctl + kCtlErr, stream);
  return e == cudaSuccess ? GQA_OK : cuda_fail(e);
}

int gqa_attn_decode_chunked(const void *q, const void *k_cache, const void *v_cache,
                            const int *seqlens, void *o, int B, int H_q, int H_kv, int max_len,
                            int d, float scale, int chunk_tokens, cudaStream_t stream) {
  return decode_bf16(q, k_cache, v_cache, seqlens, o, nullptr, B, H_q, H_kv, max_len, d, scale,
                     chunk_tokens, stream);
}

int gqa_attn_decode(const void *q, const void *k_cache, const void *v_cache, const int *seqlens,
                    void *o, int B, int H_q, int H_kv, int max_len, int d, float scale,
                    cudaStream_t stream) {
  return decode_bf16(q, k_cache, v_cache, seqlens, o, nullptr, B, H_q, H_kv, max_len, d, scale, 0,
                     stream);
}

int gqa_attn_decode_lse(const void *q, const void *k_cache, const void *v_cache,
                        const int *seqlens, void *o, float *lse, int B, int H_q, int H_kv,
                        int max_len, int d, float scale, cudaStream_t stream) {
  return decode_bf16(q, k_cache, v_cache, seqlens, o, lse, B, H_q, H_kv, max_len, d, scale, 0,
                     stream);
}

int gqa_attn_decode_f32(const void *q, const void *k_cache, const void *v_cache,
                        const int *seqlens, void *o, int B, int H_q, int H_kv, int max_len, int d,
                        float scale, cudaStream_t stream) {
  int rc = check_decode_args(q, k_cache, v_cache, seqlens, o, B, H_q, H_kv, max_len, d, scale);
  if (rc != GQA_OK) return rc;
  if (!d_supported_simt(d)) return GQA_ERR_UNSUPPORTED;
  Workspace *ws = nullptr;
  rc = get_workspace(stream, 0, &ws);
  if (rc != GQA_OK) return rc;
  // decode = prefill form with one query row and per-sequence key counts
  cudaError_t e = launch_attn_f32(static_cast<const float *>(q), static_cast<const float *>(k_cache),
                                  static_cast<const float *>(v_cache), static_cast<float *>(o), B,
                                  H_q, H_kv, 1, max_len, d, 0, scale, seqlens, max_len,
                                  ws->ctl + kCtlErr, stream);
  return e == cudaSuccess ? GQA_OK : cuda_fail(e);
}

int gqa_attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                 const float *lse, void *dq, void *dk, void *dv, int B, int H_q, int H_kv, int N_q,
                 int N_kv, int d, int causal, float scale, cudaStream_t stream) {
  int rc = check_prefill_args(q, k, v, o, B, H_q, H_kv, N_q, N_kv, d, causal, scale);
  if (rc != GQA_OK) return rc;
  if (!dout || !lse || !dq || !dk || !dv) return GQA_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return GQA_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 96 && d != 128) return GQA_ERR_UNSUPPORTED;
  const long long units = static_cast<long long>(B) * H_kv * ((N_kv + kTileN - 1) / kTileN) +
                          static_cast<long long>(B) * H_q * ((N_q + kTileM - 1) / kTileM);
  if (units > INT32_MAX) return GQA_ERR_UNSUPPORTED;
  Workspace *ws = nullptr;
  rc = get_workspace(stream, bwd_workspace_bytes(B, H_q, N_q), &ws);
  if (rc != GQA_OK) return rc;
  CUtensorMap tq, tk, tv, tdo;
  if (!encode_bf16_3d(&tq, q, d, N_q, static_cast<long>(B) * H_q, kTileM) ||
      !encode_bf16_3d(&tdo, dout, d, N_q, static_cast<long>(B) * H_q, kTileM) ||
      !encode_bf16_3d(&tk, k, d, N_kv, static_cast<long>(B) * H_kv, kTileN) ||
      !encode_bf16_3d(&tv, v, d, N_kv, static_cast<long>(B) * H_kv, kTileN))
    return cuda_fail(cudaErrorInvalidValue);
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e = launch_attn_bwd(tq, tk, tv, tdo, o, dout, lse, ws->partials, dq, dk, dv, B, H_q,
                                  H_kv, N_q, N_kv, d, causal, scale, device_sms(dev),
                                  ws->ctl + kCtlErr, stream);
  return e == cudaSuccess ? GQA_OK : cuda_fail(e);
}

namespace {
// Decode against a one-byte cache (e4m3 or int8 codes, per-K/V-head scales):
// checks, workspace, maps, launch.
int decode_byte_cache(bool int8, const void *q, const void *k_cache, const void *v_cache,
                      const float *k_scale, const float *v_scale, const int *seqlens, void *o,
                      float *lse, int B, int H_q, int H_kv, int max_len, int d, float scale,
                      cudaStream_t stream) {
  int rc = check_decode_args(q, k_cache, v_cache, seqlens, o, B, H_q, H_kv, max_len, d, scale);
  if (rc != GQA_OK) return rc;
  if (!k_scale || !v_scale || (reinterpret_cast<uintptr_t>(k_scale) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(v_scale) & 3u) != 0)
    return GQA_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return GQA_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 96 && d != 128) return GQA_ERR_UNSUPPORTED;
  if (!decode_units_fit(B, H_q, H_kv, max_len)) return GQA_ERR_UNSUPPORTED;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const int grid = decode_grid(B, H_q, H_kv, max_len, d, device_sms(dev), 0);
  Workspace *ws = nullptr;
  rc = get_workspace(stream, decode_partials_bytes(B, H_q, H_kv, d, grid), &ws,
                     decode_planes(B, H_q, H_kv));
  if (rc != GQA_OK) return rc;
  CUtensorMap tq, tk, tv;
  if (!encode_bf16_3d(&tq, q, d, static_cast<long>(B) * H_q, 1, kDecodeHeads) ||
      !encode_u8_3d(&tk, k_cache, d, max_len, static_cast<long>(B) * H_kv, d <= 64 ? 64 : 128,
                    kDecodeByteUnit) ||
      !encode_u8_3d(&tv, v_cache, d, max_len, static_cast<long>(B) * H_kv, d <= 64 ? 64 : 128,
                    kDecodeByteUnit))
    return cuda_fail(cudaErrorInvalidValue);
  e = (int8 ? launch_decode_int8 : launch_decode_fp8)(tq, tk, tv, q, seqlens, o, lse, ws->partials,
                                                      ws->counters, B, H_q, H_kv, max_len, d, scale,
                                                      k_scale, v_scale, grid, ws->ctl + kCtlErr,
                                                      stream);
  return e == cudaSuccess ? GQA_OK : cuda_fail(e);
}
}  // namespace

int gqa_attn_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                        const float *k_scale, const float *v_scale, const int *seqlens, void *o,
                        float *lse, int B, int H_q, int H_kv, int max_len, int d, float scale,
                        cudaStream_t stream) {
  return decode_byte_cache(false, q, k_cache, v_cache, k_scale, v_scale, seqlens, o, lse, B, H_q,
                           H_kv, max_len, d, scale, stream);
}

int gqa_attn_decode_int8(const void *q, const void *k_cache, const void *v_cache,
                         const float *k_scale, const float *v_scale, const int *seqlens, void *o,
                         float *lse, int B, int H_q, int H_kv, int max_len, int d, float scale,
                         cudaStream_t stream) {
  return decode_byte_cache(true, q, k_cache, v_cache, k_scale, v_scale, seqlens, o, lse, B, H_q,
                           H_kv, max_len, d, scale, stream);
}

const char *gqa_attn_status_string(int status) {
  switch (status) {
    case GQA_OK: return "GQA_OK";
    case GQA_ERR_INVALID_ARG: return "GQA_ERR_INVALID_ARG: invalid argument (null/misaligned pointer, non-positive size, H_q not a multiple of H_kv, non-finite scale)";
    case GQA_ERR_UNSUPPORTED: return "GQA_ERR_UNSUPPORTED: unsupported configuration (head dim, causal with N_q > N_kv, or size limit)";
    case GQA_ERR_CUDA: {
      thread_local char buf[160];
      snprintf(buf, sizeof(buf), "GQA_ERR_CUDA: %s", cudaGetErrorName(g_last_cuda_error));
      return buf;
    }
    case GQA_ERR_DEVICE_TIMEOUT: return "GQA_ERR_DEVICE_TIMEOUT: a bounded device-side wait ran out";
    case GQA_ERR_OOM: return "GQA_ERR_OOM: workspace allocation failed (or would grow during stream capture)";
    case GQA_ERR_BAD_SEQLEN: return "GQA_ERR_BAD_SEQLEN: a seqlens entry was outside [0, max_len]";
    default: return "unknown gqa_status";
  }
}

int gqa_attn_get_device_error(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  int *ctl = nullptr, *counters = nullptr;
  size_t counters_len = 0;
  {
    std::lock_guard<std::mutex> lk(g_ws_mutex);
    auto it = g_ws.find(WsKey{dev, stream});
    if (it == g_ws.end()) return GQA_OK;  // nothing ever ran on this stream
    ctl = it->second.ctl;
    counters = it->second.counters;
    counters_len = it->second.counters_len;
  }
  int word = 0;
  e = cudaMemcpyAsync(&word, ctl + kCtlErr, sizeof(int), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctl + kCtlErr, 0, sizeof(int), stream);
  if (e == cudaSuccess && (word & kErrTimeout)) {
    // a pipeline that gave up may have left the work counter armed
    e = cudaMemsetAsync(ctl + kCtlWork, 0, 2 * sizeof(int), stream);
    if (e == cudaSuccess && counters != nullptr)
      e = cudaMemsetAsync(counters, 0, counters_len * sizeof(int), stream);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if (word & kErrTimeout) return GQA_ERR_DEVICE_TIMEOUT;
  if (word & kErrBadSeqlen) return GQA_ERR_BAD_SEQLEN;
  return GQA_OK;
}

int gqa_attn_prefill_plan(int B, int H_q, int H_kv, int N_q, int N_kv, int causal, int unit,
                          int *out) {
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || N_q <= 0 || N_kv <= 0 || H_q % H_kv != 0) return -1;
  if (causal && N_q > N_kv) return -1;
  const PrefillPlan plan = make_prefill_plan(B, H_q, H_kv, N_q, N_kv, causal);
  if (out != nullptr && unit >= 0 && unit < plan.total_units) {
    const Unit w = decode_unit(plan, unit);
    out[0] = w.b;
    out[1] = w.h_kv;
    for (int t = 0; t < 2; ++t) {
      out[2 + 3 * t] = w.t[t].h_q;
      out[3 + 3 * t] = w.t[t].q_tile;
      out[4 + 3 * t] = w.t[t].kv_blocks;
    }
  }
  return plan.total_units;
}

int gqa_attn_selftest_wait_timeout(int timeout_us, cudaStream_t stream) {
  if (timeout_us < 1 || timeout_us > 100000) return GQA_ERR_INVALID_ARG;
  Workspace *ws = nullptr;
  int rc = get_workspace(stream, 0, &ws);
  if (rc != GQA_OK) return rc;
  cudaError_t e = launch_wait_timeout_selftest(timeout_us, ws->ctl + kCtlErr, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return gqa_attn_get_device_error(stream);
}

int gqa_attn_selftest_decode_early_lengths(const void *q, const void *k_cache,
                                           const void *v_cache, const int *seqlens,
                                           const int *seqlens_early, void *o, float *lse, int B,
                                           int H_q, int H_kv, int max_len, int d, float scale,
                                           cudaStream_t stream) {
  if (seqlens_early == nullptr || (reinterpret_cast<uintptr_t>(seqlens_early) & 3u) != 0)
    return GQA_ERR_INVALID_ARG;
  return decode_bf16(q, k_cache, v_cache, seqlens, o, lse, B, H_q, H_kv, max_len, d, scale, 0,
                     stream, seqlens_early);
}

void gqa_attn_shutdown(void) {
  std::lock_guard<std::mutex> lk(g_ws_mutex);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto &kv : g_ws) {
    cudaSetDevice(kv.first.dev);
    cudaDeviceSynchronize();
    if (kv.second.partials) cudaFree(kv.second.partials);
    if (kv.second.counters) cudaFree(kv.second.counters);
    if (kv.second.units) cudaFree(kv.second.units);
    if (kv.second.ctl) cudaFree(kv.second.ctl);
  }
  g_ws.clear();
  cudaSetDevice(cur);
  cudaGetLastError();
}

}  // extern "C"
