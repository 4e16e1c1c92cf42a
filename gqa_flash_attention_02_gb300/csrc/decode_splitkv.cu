// Single-token GQA decode against a bf16 K/V cache: split-KV with the
// log-sum-exp merge done in the same kernel.
//
// The decode step reads every valid cache row once and does about 3 FLOPs
// per byte at the workload's group size, so it is bound by HBM bandwidth
// (kaispace.site, prefill-vs-decode note). The cache of each (b, h_kv) is cut
// into fixed-size splits (the split-sequence cached attention of the
// microLLM-rocm optimisation log, Experiments 282-284) so that B * H_kv *
// splits CTAs cover all SMs even at small batch; ragged lengths balance
// themselves because splits past seqlens[b] exit at once.
//
// One CTA = one (b, h_kv, split), 4 warps. It serves ALL g = H_q / H_kv
// query heads of the group from a single read of its K/V rows (no K/V
// replication: microLLM-rocm Experiment 044, BootstrapAI collab-014
// "Kernel 9 GQA"):
//   * TMA streams 64-row K and V sub-blocks (128-byte swizzled 64-column
//     panels) through a multi-stage shared-memory ring, so loads for later
//     sub-blocks are in flight while earlier ones are consumed.
//   * Warp w takes rows [16w, 16w+16) of each sub-block. The group's query
//     heads (padded to 16) times those rows is a dense contraction over d:
//     S = Q K^T and O += P V run on mma.sync (bf16 in, fp32 accumulate) from
//     ldmatrix fragments, which keeps the kernel's instruction count far
//     below its memory time. Softmax (online, exp2 with the scale folded
//     in) runs on the fragments in registers.
//   * The 4 warps' (m, l, O) states merge in shared memory. A sequence that
//     fits in one split writes its output directly; otherwise each split
//     writes (m, l, O) to the workspace and the LAST split to finish
//     (atomic counter per (b, h_kv), no waiting) merges them:
//         M = max m_i,  L = sum 2^(m_i - M) l_i,  O = sum 2^(m_i - M) O_i / L.
#include <cuda_runtime.h>
#include <math.h>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {

namespace {

constexpr int kThreads = 128;
constexpr int kSub = 64;     // cache rows per sub-block (16 per warp)
constexpr int kHeads = 16;   // query heads per pass (mma M)

// Byte offset of (row, 16-byte unit u) inside a [rows][D] bf16 tile stored
// as D/64 panels of `rows` x 128 B with the TMA 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int row, int u, int rows) {
  return static_cast<uint32_t>((u >> 3) * rows * 128 + row * 128 + (((u & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8, fp32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int D, int NSTG>
struct DecodeSmem {
  static constexpr int kTile = kSub * D * 2;            // one K or V sub-block
  static constexpr int kStage = 2 * kTile;               // K then V
  static constexpr int kOffStage = 0;
  static constexpr int kRingBytes = NSTG * kStage;
  // merge area (reuses the ring once the sweep is done)
  static constexpr int kMergeO = 4 * kHeads * D * 4;     // float [4 warps][16][D]
  static constexpr int kMergeML = 4 * kHeads * 2 * 4;    // float [4][16][2]
  static constexpr int kRegion = kRingBytes > kMergeO + kMergeML ? kRingBytes : kMergeO + kMergeML;
  static constexpr int kOffBar = kRegion;                // NSTG mbarriers
  static constexpr int kOffFlag = kOffBar + NSTG * 8;    // int: "this CTA merges"
  static constexpr int kBytes = kOffFlag + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

struct DecodeParams {
  const __nv_bfloat16 *q;
  const int *seqlens;
  __nv_bfloat16 *o;
  float *part;     // [B][H_q][splits][D + 2]: O (unnormalised), m, l
  int *counters;   // [B][H_kv], zero between launches
  int *err_word;
  int H_q, H_kv, max_len, n_splits, chunk;
  float scale_log2;
};

template <int D, int NSTG>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                          const __grid_constant__ CUtensorMap tm_v,
                                                          const DecodeParams prm) {
  using L = DecodeSmem<D, NSTG>;
  constexpr int NT = D / 8;  // n-tiles of O per warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t bars = s_base + L::kOffBar;
  volatile int *merge_flag = reinterpret_cast<volatile int *>(smem + L::kOffFlag);

  const int split = blockIdx.x, h_kv = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int group = prm.H_q / prm.H_kv;

  const int len = prm.seqlens[b];
  if (len < 0 || len > prm.max_len) {
    if (tid == 0 && split == 0 && h_kv == 0) record_error(prm.err_word, kErrBadSeqlen);
    if (split == 0) {  // the sequence's output is defined as 0
      for (int i = tid; i < group * D; i += kThreads)
        prm.o[(static_cast<size_t>(b) * prm.H_q + h_kv * group) * D + i] = __float2bfloat16_rn(0.f);
    }
    return;
  }
  const int n_split_b = (len + prm.chunk - 1) / prm.chunk;
  if (len == 0) {
    if (split == 0)
      for (int i = tid; i < group * D; i += kThreads)
        prm.o[(static_cast<size_t>(b) * prm.H_q + h_kv * group) * D + i] = __float2bfloat16_rn(0.f);
    return;
  }
  if (split >= n_split_b) return;
  const int r0 = split * prm.chunk;
  const int n = min(prm.chunk, len - r0);  // rows of this split
  const int nsub = (n + kSub - 1) / kSub;
  const int plane = b * prm.H_kv + h_kv;

  if (tid == 0) {
    for (int s = 0; s < NSTG; ++s) mbar_init(bars + 8 * s, 1);
    fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int i) {  // TMA for sub-block i into stage i % NSTG (thread 0)
    const int st = i % NSTG;
    const uint32_t dst = s_base + L::kOffStage + st * L::kStage;
    mbar_arrive_expect_tx(bars + 8 * st, L::kStage);
#pragma unroll
    for (int p = 0; p < D / 64; ++p) {
      tma_load_3d(dst + p * kSub * 128, &tm_k, bars + 8 * st, p * 64, r0 + i * kSub, plane);
      tma_load_3d(dst + L::kTile + p * kSub * 128, &tm_v, bars + 8 * st, p * 64, r0 + i * kSub,
                  plane);
    }
  };
  if (tid == 0)
    for (int i = 0; i < NSTG && i < nsub; ++i) issue(i);

  bool ok = true;
  // Each pass serves up to 16 query heads of the group.
  for (int hg = 0; hg < group && ok; hg += kHeads) {
    const int G = min(kHeads, group - hg);
    const int hq0 = h_kv * group + hg;
    // Q fragments (A operand, 16 heads x D): thread holds rows lane/4 and
    // lane/4 + 8, columns 2*(lane%4) + {0,1} and + 8, for each 16-wide k-step.
    uint32_t qa[D / 16][4];
    {
      const int r_lo = lane >> 2, r_hi = r_lo + 8, c = 2 * (lane & 3);
      const uint32_t *qlo = reinterpret_cast<const uint32_t *>(
          prm.q + (static_cast<size_t>(b) * prm.H_q + hq0 + r_lo) * D);
      const uint32_t *qhi = reinterpret_cast<const uint32_t *>(
          prm.q + (static_cast<size_t>(b) * prm.H_q + hq0 + r_hi) * D);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qa[ks][0] = r_lo < G ? __ldg(qlo + (ks * 16 + c) / 2) : 0u;
        qa[ks][1] = r_hi < G ? __ldg(qhi + (ks * 16 + c) / 2) : 0u;
        qa[ks][2] = r_lo < G ? __ldg(qlo + (ks * 16 + c + 8) / 2) : 0u;
        qa[ks][3] = r_hi < G ? __ldg(qhi + (ks * 16 + c + 8) / 2) : 0u;
      }
    }
    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

    for (int i = 0; i < nsub; ++i) {
      const int st = i % NSTG;
      // fills of this stage before this one: per pass the ring restarts at
      // stage 0 and stage st is filled ceil((nsub - st) / NSTG) times
      const int fills = (hg / kHeads) * ((nsub - st + NSTG - 1) / NSTG) + i / NSTG;
      const uint32_t phase = static_cast<uint32_t>(fills & 1);
      if (!__syncthreads_and(mbar_wait(bars + 8 * st, phase, nullptr))) { ok = false; break; }
      const uint32_t kt = s_base + L::kOffStage + st * L::kStage;
      const uint32_t vt = kt + L::kTile;
      const int rows_here = min(kSub, n - i * kSub);  // valid rows in this sub-block
      const int wrow = warp * 16;                     // this warp's first row
      if (rows_here < kSub) {
        // rows past the sequence (other sequences' data or NaN padding) must
        // not reach P.V: zero this warp's invalid V rows
        for (int idx = lane; idx < 16 * (D / 8); idx += 32) {
          const int r = wrow + idx / (D / 8), u = idx % (D / 8);
          if (r >= rows_here)
            *reinterpret_cast<uint4 *>(smem + (vt - s_base) + swz(r, u, kSub)) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // ---- S = Q K^T for this warp's 16 rows (two n-tiles of 8 keys)
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      {
        // lanes 0-7: keys 0-7 unit 2ks; 8-15: keys 0-7 unit 2ks+1;
        // 16-23: keys 8-15 unit 2ks; 24-31: keys 8-15 unit 2ks+1
        const int key = wrow + (lane & 7) + ((lane >> 4) << 3);
        const int uo = (lane >> 3) & 1;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kt + swz(key, 2 * ks + uo, kSub), b0, b1, b2, b3);
          mma_bf16(s0, qa[ks], b0, b1);
          mma_bf16(s1, qa[ks], b2, b3);
        }
      }
      // ---- online softmax on the fragments: rows (heads) lane/4 and lane/4+8
      const int kc = wrow + 2 * (lane & 3);  // key of s?[0]; s?[1] is kc+1; s1 adds 8
      const float sl2 = prm.scale_log2;
      float x[8] = {s0[0] * sl2, s0[1] * sl2, s1[0] * sl2, s1[1] * sl2,
                    s0[2] * sl2, s0[3] * sl2, s1[2] * sl2, s1[3] * sl2};
      const int keys[4] = {kc, kc + 1, kc + 8, kc + 9};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (keys[e] >= rows_here) { x[e] = -INFINITY; x[4 + e] = -INFINITY; }
      }
      float mx_lo = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      float mx_hi = fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7]));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      // a warp whose 16 rows are all past the sequence sees mn = -inf: skip
      const float a_lo = (mn_lo == -INFINITY) ? 1.f : ex2(m_lo - mn_lo);
      const float a_hi = (mn_hi == -INFINITY) ? 1.f : ex2(m_hi - mn_hi);
      float p[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p[e] = (mn_lo == -INFINITY) ? 0.f : ex2(x[e] - mn_lo);
        p[4 + e] = (mn_hi == -INFINITY) ? 0.f : ex2(x[4 + e] - mn_hi);
      }
      l_lo = l_lo * a_lo + ((p[0] + p[1]) + (p[2] + p[3]));
      l_hi = l_hi * a_hi + ((p[4] + p[5]) + (p[6] + p[7]));
      m_lo = mn_lo;
      m_hi = mn_hi;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        acc[t][0] *= a_lo; acc[t][1] *= a_lo;
        acc[t][2] *= a_hi; acc[t][3] *= a_hi;
      }
      // P as the A operand (16 heads x 16 keys): keys 0-7 from n-tile 0, 8-15 from n-tile 1
      const uint32_t pa[4] = {pack_bf16x2(p[0], p[1]), pack_bf16x2(p[4], p[5]),
                              pack_bf16x2(p[2], p[3]), pack_bf16x2(p[6], p[7])};
      // ---- O += P V (V rows = k, d = n): transposed ldmatrix of 8x8 blocks
      {
        // lanes 0-7: keys 0-7 unit u; 8-15: keys 8-15 unit u; 16-23: keys 0-7 unit u+1;
        // 24-31: keys 8-15 unit u+1  -> {b0,b1} for d-tile u and {b0,b1} for u+1
        const int key = wrow + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int uo = lane >> 4;
#pragma unroll
        for (int u = 0; u < NT; u += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vt + swz(key, u + uo, kSub), b0, b1, b2, b3);
          mma_bf16(acc[u], pa, b0, b1);
          mma_bf16(acc[u + 1], pa, b2, b3);
        }
      }
      // all warps are done with this stage: refill it with sub-block i + NSTG
      __syncthreads();
      if (tid == 0 && i + NSTG < nsub) {
        fence_proxy_async_smem();  // generic-proxy writes (V zeroing) before the TMA overwrite
        issue(i + NSTG);
      }
    }
    if (!ok) break;

    // ---- merge the 4 warps' states in shared memory (the ring is idle now)
    float *mo = reinterpret_cast<float *>(smem);                    // [4][16][D]
    float *mml = reinterpret_cast<float *>(smem + L::kMergeO);      // [4][16][2]
    {
      const int r_lo = lane >> 2, r_hi = r_lo + 8;
      // quad-reduce l across the 4 threads sharing a row
      float ll = l_lo, lh = l_hi;
      ll += __shfl_xor_sync(0xffffffffu, ll, 1);
      ll += __shfl_xor_sync(0xffffffffu, ll, 2);
      lh += __shfl_xor_sync(0xffffffffu, lh, 1);
      lh += __shfl_xor_sync(0xffffffffu, lh, 2);
      if ((lane & 3) == 0) {
        mml[(warp * 16 + r_lo) * 2 + 0] = m_lo;
        mml[(warp * 16 + r_lo) * 2 + 1] = ll;
        mml[(warp * 16 + r_hi) * 2 + 0] = m_hi;
        mml[(warp * 16 + r_hi) * 2 + 1] = lh;
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int col = t * 8 + 2 * (lane & 3);
        *reinterpret_cast<float2 *>(mo + (warp * 16 + r_lo) * D + col) = make_float2(acc[t][0], acc[t][1]);
        *reinterpret_cast<float2 *>(mo + (warp * 16 + r_hi) * D + col) = make_float2(acc[t][2], acc[t][3]);
      }
    }
    __syncthreads();
    const bool single = (n_split_b == 1);
    for (int idx = tid; idx < G * D; idx += kThreads) {
      const int h = idx / D, c = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, mml[(w * 16 + h) * 2]);
      float Lsum = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = mml[(w * 16 + h) * 2];
        const float wgt = (mw == -INFINITY) ? 0.f : ex2(mw - M);
        Lsum = fmaf(wgt, mml[(w * 16 + h) * 2 + 1], Lsum);
        O = fmaf(wgt, mo[(w * 16 + h) * D + c], O);
      }
      const size_t row = static_cast<size_t>(b) * prm.H_q + hq0 + h;
      if (single) {
        prm.o[row * D + c] = __float2bfloat16_rn(O / Lsum);
      } else {
        float *dst = prm.part + (row * prm.n_splits + split) * (D + 2);
        dst[c] = O;
        if (c == 0) {
          dst[D] = M;
          dst[D + 1] = Lsum;
        }
      }
    }
    __syncthreads();  // merge area free again (next pass reloads the ring)
    if (hg + kHeads < group) {
      // another pass over the same rows: restart the ring
      if (tid == 0)
        for (int i = 0; i < NSTG && i < nsub; ++i) issue(i);
    }
  }
  if (!ok) {
    if (tid == 0) record_error(prm.err_word, kErrTimeout);
    return;
  }
  if (n_split_b == 1) return;

  // ---- the last split of (b, h_kv) to finish merges all of them
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int *ctr = prm.counters + plane;
    const int prev = atomicAdd(ctr, 1);
    const bool last = (prev == n_split_b - 1);
    if (last) atomicExch(ctr, 0);  // re-arm for the next launch
    *merge_flag = last ? 1 : 0;
  }
  __syncthreads();
  if (!*merge_flag) return;
  __threadfence();
  for (int idx = tid; idx < group * D; idx += kThreads) {
    const int h = idx / D, c = idx % D;
    const size_t row = static_cast<size_t>(b) * prm.H_q + h_kv * group + h;
    const float *src = prm.part + row * prm.n_splits * (D + 2);
    float M = -INFINITY;
    for (int sp = 0; sp < n_split_b; ++sp) M = fmaxf(M, __ldcg(src + sp * (D + 2) + D));
    float Lsum = 0.f, O = 0.f;
    for (int sp = 0; sp < n_split_b; ++sp) {
      const float *pp = src + sp * (D + 2);
      const float wgt = ex2(__ldcg(pp + D) - M);
      Lsum = fmaf(wgt, __ldcg(pp + D + 1), Lsum);
      O = fmaf(wgt, __ldcg(pp + c), O);
    }
    prm.o[row * D + c] = __float2bfloat16_rn(O / Lsum);
  }
}

template <int D, int NSTG>
cudaError_t launch_decode_d(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const void *q,
                            const int *seqlens, void *o, float *partials, int *counters, int B,
                            int H_q, int H_kv, int max_len, float scale, int chunk, int *err_word,
                            cudaStream_t stream) {
  using L = DecodeSmem<D, NSTG>;
  static unsigned configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(configured & (1u << dev))) {
    e = cudaFuncSetAttribute(decode_kernel<D, NSTG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kAlloc);
    if (e != cudaSuccess) return e;
    if (dev < 32) configured |= 1u << dev;
  }
  DecodeParams prm;
  prm.q = static_cast<const __nv_bfloat16 *>(q);
  prm.seqlens = seqlens;
  prm.o = static_cast<__nv_bfloat16 *>(o);
  prm.part = partials;
  prm.counters = counters;
  prm.err_word = err_word;
  prm.H_q = H_q;
  prm.H_kv = H_kv;
  prm.max_len = max_len;
  prm.chunk = chunk;
  prm.n_splits = (max_len + chunk - 1) / chunk;
  prm.scale_log2 = scale * 1.4426950408889634f;
  dim3 grid(prm.n_splits, H_kv, B);
  decode_kernel<D, NSTG><<<grid, kThreads, L::kAlloc, stream>>>(tm_k, tm_v, prm);
  return cudaGetLastError();
}

}  // namespace

size_t decode_partials_bytes(int B, int H_q, int max_len, int d, int chunk) {
  const size_t n_splits = (static_cast<size_t>(max_len) + chunk - 1) / chunk;
  return static_cast<size_t>(B) * H_q * n_splits * (static_cast<size_t>(d) + 2) * sizeof(float);
}

int decode_default_chunk(int B, int H_kv, int max_len, int num_sms) {
  // Longest split (fewest partials to merge) that still offers about four
  // CTAs per SM when every sequence is full length.
  for (int c : {512, 256, 128}) {
    const long ctas = static_cast<long>(B) * H_kv * ((max_len + c - 1) / c);
    if (ctas >= 4L * num_sms) return c;
  }
  return 64;
}

cudaError_t launch_decode_bf16(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const void *q,
                               const int *seqlens, void *o, float *partials, int *counters, int B,
                               int H_q, int H_kv, int max_len, int d, float scale, int chunk,
                               int *err_word, cudaStream_t stream) {
  if (chunk % kSub != 0 || chunk <= 0) return cudaErrorInvalidValue;
  if (d == 64)
    return launch_decode_d<64, 4>(tm_k, tm_v, q, seqlens, o, partials, counters, B, H_q, H_kv,
                                  max_len, scale, chunk, err_word, stream);
  if (d == 128)
    return launch_decode_d<128, 3>(tm_k, tm_v, q, seqlens, o, partials, counters, B, H_q, H_kv,
                                   max_len, scale, chunk, err_word, stream);
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
