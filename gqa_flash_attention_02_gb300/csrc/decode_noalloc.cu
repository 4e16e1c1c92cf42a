// gqa_attn_decode_noalloc: the split-KV decode for callers that must not
// allocate device memory.
//
// The regular decode entry point grows a per-stream workspace on demand
// (cudaMallocAsync) for its split partials and merge counters. Some callers
// cannot allow that: a serving loop that runs inside a fixed, pre-reserved
// memory budget, where a new allocation may fail or fragment the pool; a
// latency-critical path where an allocation call may synchronise the
// device; or a process whose device memory is owned by another allocator
// that forbids raw allocations. This entry point runs the same decode kernel
// but takes its scratch from a fixed-size array in the library's own device
// memory, so a call allocates nothing.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "gqa_attn.h"
#include "gqa_internal.h"

namespace {

// Scratch layout (bytes): split partials | merge counters | error word.
constexpr size_t kPartialsMax = 4u << 20;           // 4 MiB of fp32 partials
constexpr size_t kCountersMax = 16384;              // (b, h_kv, head group) planes
constexpr size_t kCountersOff = kPartialsMax;
constexpr size_t kErrOff = kCountersOff + kCountersMax * sizeof(int);
constexpr size_t kScratchBytes = kErrOff + 256;

// Lives on every GPU that loads the library until the process exits. Host
// code must not pass this name to a kernel: on the host it is only a
// stand-in; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).
cudaError_t scratch_for_current_device(unsigned char **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<unsigned char *>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int gqa_attn_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                       const int *seqlens, void *o, int B, int H_q, int H_kv,
                                       int max_len, int d, float scale, cudaStream_t stream) {
  using namespace gqa;
  // same argument checks as gqa_attn_decode (validation runs before any CUDA call)
  if (!q || !k_cache || !v_cache || !seqlens || !o) return GQA_ERR_INVALID_ARG;
  auto misaligned = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (misaligned(q) || misaligned(k_cache) || misaligned(v_cache) || misaligned(o) ||
      (reinterpret_cast<uintptr_t>(seqlens) & 3u) != 0)
    return GQA_ERR_INVALID_ARG;
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || max_len <= 0 || d <= 0 || H_q % H_kv != 0)
    return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 96 && d != 128 && d != 256) return GQA_ERR_UNSUPPORTED;
  if (!decode_units_fit(B, H_q, H_kv, max_len)) return GQA_ERR_UNSUPPORTED;
  if (max_len > (1 << 20) ||
      static_cast<long long>(B) * H_kv * max_len * d > (1ll << 31) - 1)
    return GQA_ERR_UNSUPPORTED;

  // The partials need one slot per CTA plus one per plane: shrink the grid
  // until they fit the fixed scratch.
  int dev = 0, sms = 1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return GQA_ERR_CUDA;
  const size_t planes = decode_planes(B, H_q, H_kv);
  const size_t slot_bytes = decode_partials_bytes(B, H_q, H_kv, d, 1) / (planes + 1);
  const size_t max_slots = kPartialsMax / slot_bytes;
  if (planes >= max_slots || planes > kCountersMax)
    return GQA_ERR_UNSUPPORTED;  // beyond the fixed scratch: use gqa_attn_decode instead
  int grid = decode_grid(B, H_q, H_kv, max_len, d, sms, 0);
  if (static_cast<size_t>(grid) > max_slots - planes) grid = static_cast<int>(max_slots - planes);

  unsigned char *scratch = nullptr;
  e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess) return GQA_ERR_CUDA;
  float *partials = reinterpret_cast<float *>(scratch);
  int *counters = reinterpret_cast<int *>(scratch + kCountersOff);
  int *err_word = reinterpret_cast<int *>(scratch + kErrOff);
  // the array keeps the previous call's contents: zero what must start at zero
  e = cudaMemsetAsync(counters, 0, planes * sizeof(int), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(err_word, 0, sizeof(int), stream);
  if (e != cudaSuccess) return GQA_ERR_CUDA;

  CUtensorMap tq, tk, tv;
  if (!encode_tensor_map_bf16_3d(&tq, q, d, static_cast<long>(B) * H_q, 1, kDecodeHeads) ||
      !encode_tensor_map_bf16_3d(&tk, k_cache, d, max_len, static_cast<long>(B) * H_kv,
                                 decode_box_rows(d)) ||
      !encode_tensor_map_bf16_3d(&tv, v_cache, d, max_len, static_cast<long>(B) * H_kv,
                                 decode_box_rows(d)))
    return GQA_ERR_CUDA;
  e = launch_decode_bf16(tq, tk, tv, q, seqlens, o, nullptr, partials, counters, B, H_q, H_kv, max_len, d,
                         scale, grid, err_word, stream);
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}
