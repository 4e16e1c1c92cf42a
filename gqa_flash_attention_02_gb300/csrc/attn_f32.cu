// fp32 SIMT attention: the full-precision path (fp32 in, fp32 math, fp32
// out, no tensor cores) for both the prefill and the decode form.
//
// Design: a CTA of 4 warps owns 16 query rows of one (b, h_q); K/V rows of
// the mapped head h_kv = h_q / (H_q/H_kv) are staged 32 at a time in shared
// memory and shared by the 16 rows (the key-tile reuse of the BootstrapAI
// evolution log's collab-007 "Kernel 3 cooperative"). Each lane scores one
// key of the tile against the row, the warp reduces max and sum with
// shuffles and updates the running (max, sum, output) state: the online
// softmax of collab-005 "Kernel 2 tiling". The K tile is padded by one float
// per row so the 32 lanes reading one column hit 32 different banks
// (collab "Kernel 4 padded smem").
#include <cuda_runtime.h>
#include <math.h>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {

namespace {

constexpr int kRowsPerCta = 16;
constexpr int kRowsPerWarp = 4;
constexpr int kKeyTile = 32;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// seqlens == nullptr: prefill form, every (b) has N_kv keys and the K/V head
// stride is N_kv rows. seqlens != nullptr: decode form (N_q == 1), batch b
// has seqlens[b] keys and the K/V head stride is kv_cap rows.
template <int D>
__global__ void __launch_bounds__(128) attn_f32_kernel(
    const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
    float *__restrict__ o, int H_q, int H_kv, int N_q, int N_kv, int causal, float scale,
    const int *__restrict__ seqlens, int kv_cap, int *err_word) {
  constexpr int EPT = D / 32;  // elements of a row per lane
  __shared__ float qs[kRowsPerCta][D];
  __shared__ float ks[kKeyTile][D + 1];
  __shared__ float vs[kKeyTile][D];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h_q = blockIdx.y, b = blockIdx.z;
  const int h_kv = h_q / (H_q / H_kv);
  const int row0 = blockIdx.x * kRowsPerCta;

  int n_kv = N_kv;
  bool bad = false;
  if (seqlens != nullptr) {
    n_kv = seqlens[b];
    if (n_kv < 0 || n_kv > kv_cap) {
      bad = true;
      if (tid == 0 && h_q == 0) record_error(err_word, kErrBadSeqlen);
      n_kv = 0;
    }
  }
  const int off = n_kv - N_q;  // bottom-right causal alignment
  const size_t kv_head = (static_cast<size_t>(b) * H_kv + h_kv) * static_cast<size_t>(kv_cap);
  const float *kh = k + kv_head * D;
  const float *vh = v + kv_head * D;
  const float *qh = q + (static_cast<size_t>(b) * H_q + h_q) * static_cast<size_t>(N_q) * D;
  float *oh = o + (static_cast<size_t>(b) * H_q + h_q) * static_cast<size_t>(N_q) * D;

  for (int i = tid; i < kRowsPerCta * D; i += blockDim.x) {
    const int r = i / D, c = i % D;
    qs[r][c] = (row0 + r < N_q) ? qh[static_cast<size_t>(row0 + r) * D + c] : 0.f;
  }

  // keys any row of this CTA can see
  int last_row = row0 + kRowsPerCta - 1;
  if (last_row > N_q - 1) last_row = N_q - 1;
  int kmax = n_kv;
  if (causal) kmax = min(n_kv, max(0, last_row + off + 1));

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][EPT];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) acc[i][e] = 0.f;
  }

  for (int base = 0; base < kmax; base += kKeyTile) {
    __syncthreads();
    for (int i = tid; i < kKeyTile * D; i += blockDim.x) {
      const int r = i / D, c = i % D;
      const bool in = base + r < kmax;  // rows past the visible range are never read
      ks[r][c] = in ? kh[static_cast<size_t>(base + r) * D + c] : 0.f;
      vs[r][c] = in ? vh[static_cast<size_t>(base + r) * D + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int rl = warp * kRowsPerWarp + i;
      const int row = row0 + rl;
      if (row >= N_q) continue;
      const int kvis = causal ? min(n_kv, max(0, row + off + 1)) : n_kv;
      if (base >= kvis) continue;  // warp-uniform
      const int key = base + lane;
      float s = 0.f;
#pragma unroll 8
      for (int c = 0; c < D; ++c) s = fmaf(qs[rl][c], ks[lane][c], s);
      s = (key < kvis) ? s * scale : -INFINITY;
      const float m_new = fmaxf(m[i], warp_max(s));
      const float alpha = expf(m[i] - m_new);  // 0 on the first visible tile
      const float p = (key < kvis) ? expf(s - m_new) : 0.f;
      l[i] = l[i] * alpha + warp_sum(p);
#pragma unroll
      for (int e = 0; e < EPT; ++e) acc[i][e] *= alpha;
#pragma unroll 4
      for (int j = 0; j < kKeyTile; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int e = 0; e < EPT; ++e) acc[i][e] = fmaf(pj, vs[j][lane + 32 * e], acc[i][e]);
      }
      m[i] = m_new;
    }
  }

#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int row = row0 + warp * kRowsPerWarp + i;
    if (row >= N_q) continue;
    const float inv = (l[i] > 0.f && !bad) ? 1.f / l[i] : 0.f;
#pragma unroll
    for (int e = 0; e < EPT; ++e) oh[static_cast<size_t>(row) * D + lane + 32 * e] = acc[i][e] * inv;
  }
}

}  // namespace

cudaError_t launch_attn_f32(const float *q, const float *k, const float *v, float *o, int B,
                            int H_q, int H_kv, int N_q, int N_kv, int d, int causal, float scale,
                            const int *seqlens, int kv_row_capacity, int *err_word,
                            cudaStream_t stream) {
  dim3 grid((N_q + kRowsPerCta - 1) / kRowsPerCta, H_q, B);
  dim3 block(128);
  const int cap = seqlens ? kv_row_capacity : N_kv;
  switch (d) {
    case 32:
      attn_f32_kernel<32><<<grid, block, 0, stream>>>(q, k, v, o, H_q, H_kv, N_q, N_kv, causal,
                                                      scale, seqlens, cap, err_word);
      break;
    case 64:
      attn_f32_kernel<64><<<grid, block, 0, stream>>>(q, k, v, o, H_q, H_kv, N_q, N_kv, causal,
                                                      scale, seqlens, cap, err_word);
      break;
    case 96:
      attn_f32_kernel<96><<<grid, block, 0, stream>>>(q, k, v, o, H_q, H_kv, N_q, N_kv, causal,
                                                      scale, seqlens, cap, err_word);
      break;
    case 128:
      attn_f32_kernel<128><<<grid, block, 0, stream>>>(q, k, v, o, H_q, H_kv, N_q, N_kv, causal,
                                                       scale, seqlens, cap, err_word);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gqa
