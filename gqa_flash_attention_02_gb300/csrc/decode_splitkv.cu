// Single-token GQA decode against a bf16 K/V cache: split-KV partials and a
// log-sum-exp combine.
//
// The decode step reads every valid cache row once and does ~2 FLOPs per
// byte, so it is bound by HBM bandwidth (kaispace.site, prefill-vs-decode
// note). The cache is cut into fixed-size chunks ("splits", the
// split-sequence cached attention of the microLLM-rocm optimisation log,
// Experiments 282-284) so that B * H_kv * splits CTAs fill all SMs even at
// small batch; ragged lengths balance themselves because splits past
// seqlens[b] exit at once.
//
// One CTA = one (b, h_kv, split). It serves ALL g = H_q / H_kv query heads
// of the group from one read of its K and V chunk (no K/V replication,
// microLLM-rocm Experiment 044 / BootstrapAI collab-014 "Kernel 9 GQA"):
//   1. TMA copies the K chunk and the V chunk (128-byte swizzled panels of
//      64 columns) into shared memory; V streams in while K is scored.
//   2. Thread r scores cache row r against the g query vectors (fp32 FMA,
//      q pre-scaled by scale*log2(e) and broadcast from shared memory).
//   3. Per head: block max, p = 2^(s - m), block sum.
//   4. O_partial[h][c] = sum_r p[h][r] V[r][c], with each thread owning a
//      column pair over a slice of rows, then a shared-memory reduction.
//   5. (m, l, O_partial) go to the workspace; a second kernel merges the
//      splits of each (b, h_q):  M = max m_i, L = sum 2^(m_i - M) l_i,
//      O = sum 2^(m_i - M) O_i / L.
#include <cuda_runtime.h>
#include <math.h>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {

namespace {

constexpr int kThreads = 128;
constexpr int kMaxGroup = 8;  // query heads scored per pass over the K chunk

// Byte offset of element (row, col) of a [rows][D] bf16 chunk stored as
// D/64 panels of rows x 128 B with the TMA 128-byte swizzle (16-byte unit
// index XOR row % 8).
template <int C>
__device__ __forceinline__ uint32_t swz_offset(int row, int col) {
  const int panel = col >> 6;
  const int byte_in_line = (col & 63) * 2;
  const int unit = byte_in_line >> 4;
  return static_cast<uint32_t>(panel * C * 128 + row * 128 + ((unit ^ (row & 7)) << 4) +
                               (byte_in_line & 15));
}

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

template <int D, int C>
struct DecodeSmem {
  static constexpr int kChunkBytes = C * D * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kChunkBytes;
  static constexpr int kOffQ = 2 * kChunkBytes;                   // float [kMaxGroup][D]
  static constexpr int kOffP = kOffQ + kMaxGroup * D * 4;         // float [C][kMaxGroup]
  static constexpr int kOffRed = kOffP + C * kMaxGroup * 4;       // float [4][kMaxGroup]
  static constexpr int kRS = kThreads / (D / 2);                  // row slices in PV
  static constexpr int kOffO = kOffRed + 4 * kMaxGroup * 4;       // float [kRS][kMaxGroup][D]
  static constexpr int kOffBar = kOffO + kRS * kMaxGroup * D * 4; // 2 mbarriers
  static constexpr int kBytes = kOffBar + 16;
  static constexpr int kAlloc = kBytes + 1024;                    // room to align to 1 KB
};

template <int D, int C>
__global__ void __launch_bounds__(kThreads) decode_splitkv_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __nv_bfloat16 *__restrict__ q, const int *__restrict__ seqlens,
    float *__restrict__ part_o, float *__restrict__ part_ml, int H_q, int H_kv, int max_len,
    int n_splits, float scale_log2, int *err_word) {
  using L = DecodeSmem<D, C>;
  constexpr int RPT = (C + kThreads - 1) / kThreads;  // score rows per thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_k = smem_addr(smem + L::kOffK);
  const uint32_t s_v = smem_addr(smem + L::kOffV);
  float *qf = reinterpret_cast<float *>(smem + L::kOffQ);
  float *ps = reinterpret_cast<float *>(smem + L::kOffP);
  float *red = reinterpret_cast<float *>(smem + L::kOffRed);
  float *ored = reinterpret_cast<float *>(smem + L::kOffO);
  const uint32_t bar_k = smem_addr(smem + L::kOffBar);
  const uint32_t bar_v = bar_k + 8;

  const int split = blockIdx.x, h_kv = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int group = H_q / H_kv;

  const int len = seqlens[b];
  if (len < 0 || len > max_len) {
    if (tid == 0 && split == 0 && h_kv == 0) record_error(err_word, kErrBadSeqlen);
    return;
  }
  const int s0 = split * C;
  if (s0 >= len) return;
  const int n = min(C, len - s0);
  const int kv_plane = b * H_kv + h_kv;

  if (tid == 0) {
    mbar_init(bar_k, 1);
    mbar_init(bar_v, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_k, L::kChunkBytes);
#pragma unroll
    for (int p = 0; p < D / 64; ++p) tma_load_3d(s_k + p * C * 128, &tm_k, bar_k, p * 64, s0, kv_plane);
    mbar_arrive_expect_tx(bar_v, L::kChunkBytes);
#pragma unroll
    for (int p = 0; p < D / 64; ++p) tma_load_3d(s_v + p * C * 128, &tm_v, bar_v, p * 64, s0, kv_plane);
  }

  bool ok = mbar_wait(bar_k, 0, nullptr);
  ok = mbar_wait(bar_v, 0, nullptr) && ok;  // both copies have landed before any exit
  if (!__syncthreads_and(ok)) {             // CTA-uniform exit on a timeout
    if (tid == 0) record_error(err_word, kErrTimeout);
    return;
  }

  for (int hg = 0; hg < group; hg += kMaxGroup) {
    const int G = min(kMaxGroup, group - hg);
    const int hq0 = h_kv * group + hg;
    __syncthreads();  // previous pass done with qf / ps / ored
    for (int i = tid; i < kMaxGroup * D; i += kThreads) {
      const int h = i / D, c = i % D;
      qf[i] = (h < G) ? __bfloat162float(q[(static_cast<size_t>(b) * H_q + hq0 + h) * D + c]) *
                            scale_log2
                      : 0.f;
    }
    __syncthreads();

    // ---- scores: thread owns rows tid, tid + 128, ...
    float s[RPT][kMaxGroup];
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) {
      const int r = tid + rr * kThreads;
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h) s[rr][h] = 0.f;
      if (r < n) {
#pragma unroll 2
        for (int c8 = 0; c8 < D / 8; ++c8) {
          const uint4 raw = *reinterpret_cast<const uint4 *>(smem + L::kOffK +
                                                               swz_offset<C>(r, c8 * 8));
          float kf[8];
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            kf[2 * e] = __uint_as_float(w[e] << 16);
            kf[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
          }
#pragma unroll
          for (int h = 0; h < kMaxGroup; ++h) {
            if (h < G) {
              const float4 qa = *reinterpret_cast<const float4 *>(qf + h * D + c8 * 8);
              const float4 qb = *reinterpret_cast<const float4 *>(qf + h * D + c8 * 8 + 4);
              float a = s[rr][h];
              a = fmaf(qa.x, kf[0], a); a = fmaf(qa.y, kf[1], a);
              a = fmaf(qa.z, kf[2], a); a = fmaf(qa.w, kf[3], a);
              a = fmaf(qb.x, kf[4], a); a = fmaf(qb.y, kf[5], a);
              a = fmaf(qb.z, kf[6], a); a = fmaf(qb.w, kf[7], a);
              s[rr][h] = a;
            }
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) s[rr][h] = -INFINITY;
      }
    }

    // ---- per-head max over the chunk
    float mh[kMaxGroup];
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      float x = s[0][h];
#pragma unroll
      for (int rr = 1; rr < RPT; ++rr) x = fmaxf(x, s[rr][h]);
      x = warp_max(x);
      if (lane == 0) red[warp * kMaxGroup + h] = x;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h)
      mh[h] = fmaxf(fmaxf(red[h], red[kMaxGroup + h]), fmaxf(red[2 * kMaxGroup + h], red[3 * kMaxGroup + h]));
    __syncthreads();  // red reused for the sums

    // ---- p = 2^(s - m), per-head sums
    float lsum[kMaxGroup];
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) lsum[h] = 0.f;
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) {
      const int r = tid + rr * kThreads;
      if (r < C) {
        float pv[kMaxGroup];
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) {
          pv[h] = (r < n && h < G) ? ex2(s[rr][h] - mh[h]) : 0.f;
          lsum[h] += pv[h];
        }
        float4 *dst = reinterpret_cast<float4 *>(ps + r * kMaxGroup);
        dst[0] = make_float4(pv[0], pv[1], pv[2], pv[3]);
        dst[1] = make_float4(pv[4], pv[5], pv[6], pv[7]);
      }
    }
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      const float x = warp_sum(lsum[h]);
      if (lane == 0) red[warp * kMaxGroup + h] = x;
    }
    __syncthreads();

    // ---- O_partial = P V : thread owns a column pair over a slice of rows
    {
      constexpr int CP = D / 2;        // column pairs
      constexpr int RS = kThreads / CP;  // row slices
      constexpr int RPS = (C + RS - 1) / RS;
      const int cp = tid % CP, slice = tid / CP;
      const int r_begin = slice * RPS;
      const int r_end = min(n, r_begin + RPS);
      float acc[kMaxGroup][2];
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h) acc[h][0] = acc[h][1] = 0.f;
      for (int r = r_begin; r < r_end; ++r) {
        const uint32_t w =
            *reinterpret_cast<const uint32_t *>(smem + L::kOffV + swz_offset<C>(r, 2 * cp));
        const float v0 = __uint_as_float(w << 16), v1 = __uint_as_float(w & 0xffff0000u);
        const float4 pa = *reinterpret_cast<const float4 *>(ps + r * kMaxGroup);
        const float4 pb = *reinterpret_cast<const float4 *>(ps + r * kMaxGroup + 4);
        const float pr[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) {
          acc[h][0] = fmaf(pr[h], v0, acc[h][0]);
          acc[h][1] = fmaf(pr[h], v1, acc[h][1]);
        }
      }
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h) {
        float2 *dst = reinterpret_cast<float2 *>(ored + (slice * kMaxGroup + h) * D + 2 * cp);
        *dst = make_float2(acc[h][0], acc[h][1]);
      }
    }
    __syncthreads();

    // ---- write (m, l, O_partial) for each head of this pass
    for (int i = tid; i < G * D; i += kThreads) {
      const int h = i / D, c = i % D;
      float x = 0.f;
#pragma unroll
      for (int sl = 0; sl < L::kRS; ++sl) x += ored[(sl * kMaxGroup + h) * D + c];
      const size_t slot = (static_cast<size_t>(b) * H_q + hq0 + h) * n_splits + split;
      part_o[slot * D + c] = x;
    }
    if (tid < G) {
      const int h = tid;
      const size_t slot = (static_cast<size_t>(b) * H_q + hq0 + h) * n_splits + split;
      const float l = red[h] + red[kMaxGroup + h] + red[2 * kMaxGroup + h] + red[3 * kMaxGroup + h];
      part_ml[slot * 2 + 0] = mh[h];
      part_ml[slot * 2 + 1] = l;
    }
  }
}

// One CTA of D threads per (b, h_q): merges the splits that saw keys.
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(
    const float *__restrict__ part_o, const float *__restrict__ part_ml,
    const int *__restrict__ seqlens, __nv_bfloat16 *__restrict__ o, int H_q, int max_len,
    int n_splits, int chunk) {
  const int bh = blockIdx.x;
  const int b = bh / H_q;
  const int c = threadIdx.x;
  const int len = seqlens[b];
  __nv_bfloat16 *dst = o + static_cast<size_t>(bh) * D + c;
  if (len <= 0 || len > max_len) {  // empty or invalid sequence: O = 0
    *dst = __float2bfloat16_rn(0.f);
    return;
  }
  const int ns = (len + chunk - 1) / chunk;
  const float *ml = part_ml + static_cast<size_t>(bh) * n_splits * 2;
  const float *po = part_o + static_cast<size_t>(bh) * n_splits * D;
  float M = -INFINITY;
  for (int i = 0; i < ns; ++i) M = fmaxf(M, ml[2 * i]);
  float acc = 0.f, Lsum = 0.f;
  for (int i = 0; i < ns; ++i) {
    const float w = ex2(ml[2 * i] - M);
    Lsum = fmaf(w, ml[2 * i + 1], Lsum);
    acc = fmaf(w, po[static_cast<size_t>(i) * D + c], acc);
  }
  *dst = __float2bfloat16_rn(acc / Lsum);
}

template <int D, int C>
cudaError_t launch_decode_dc(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const void *q,
                             const int *seqlens, void *o, float *partials, int B, int H_q,
                             int H_kv, int max_len, float scale, int *err_word,
                             cudaStream_t stream) {
  using L = DecodeSmem<D, C>;
  static bool configured = false;  // attribute is per device; harmless to repeat
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_splitkv_kernel<D, C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int n_splits = (max_len + C - 1) / C;
  float *part_o = partials;
  float *part_ml = partials + static_cast<size_t>(B) * H_q * n_splits * D;
  const float scale_log2 = scale * 1.4426950408889634f;
  dim3 grid(n_splits, H_kv, B);
  decode_splitkv_kernel<D, C><<<grid, kThreads, L::kAlloc, stream>>>(
      tm_k, tm_v, static_cast<const __nv_bfloat16 *>(q), seqlens, part_o, part_ml, H_q, H_kv,
      max_len, n_splits, scale_log2, err_word);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<D><<<B * H_q, D, 0, stream>>>(part_o, part_ml, seqlens,
                                                      static_cast<__nv_bfloat16 *>(o), H_q,
                                                      max_len, n_splits, C);
  return cudaGetLastError();
}

}  // namespace

size_t decode_partials_bytes(int B, int H_q, int max_len, int d, int chunk) {
  const size_t n_splits = (static_cast<size_t>(max_len) + chunk - 1) / chunk;
  return static_cast<size_t>(B) * H_q * n_splits * (static_cast<size_t>(d) + 2) * sizeof(float);
}

int decode_default_chunk(int B, int H_kv, int max_len, int num_sms) {
  // Prefer long chunks (fewer partials to merge) as long as the grid still
  // offers about two CTAs per SM.
  for (int c : {128, 64}) {
    const long ctas = static_cast<long>(B) * H_kv * ((max_len + c - 1) / c);
    if (ctas >= 2L * num_sms) return c;
  }
  return 32;
}

cudaError_t launch_decode_bf16(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const void *q,
                               const int *seqlens, void *o, float *partials, int B, int H_q,
                               int H_kv, int max_len, int d, float scale, int chunk,
                               int *err_word, cudaStream_t stream) {
#define GQA_DECODE_CASE(DD, CC)                                                              \
  if (d == DD && chunk == CC)                                                                \
    return launch_decode_dc<DD, CC>(tm_k, tm_v, q, seqlens, o, partials, B, H_q, H_kv,      \
                                    max_len, scale, err_word, stream);
  GQA_DECODE_CASE(64, 32)
  GQA_DECODE_CASE(64, 64)
  GQA_DECODE_CASE(64, 128)
  GQA_DECODE_CASE(64, 256)
  GQA_DECODE_CASE(128, 32)
  GQA_DECODE_CASE(128, 64)
  GQA_DECODE_CASE(128, 128)
  GQA_DECODE_CASE(128, 256)
#undef GQA_DECODE_CASE
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- self-test

namespace {
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, int *err_word) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(a, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Nobody arrives: the wait must give up by itself and report it.
  if (!mbar_wait(a, 0, nullptr, limit_ns) && threadIdx.x == 0) record_error(err_word, kErrTimeout);
}
}  // namespace

cudaError_t launch_wait_timeout_selftest(int timeout_us, int *err_word, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(timeout_us) * 1000ull,
                                                     err_word);
  return cudaGetLastError();
}

}  // namespace gqa
