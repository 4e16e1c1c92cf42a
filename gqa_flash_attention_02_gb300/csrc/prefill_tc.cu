// bf16 GQA prefill attention on the sm_103a tensor cores.
//
// What it computes: O = softmax(scale * Q K^T [+ causal mask]) V per query
// head h_q against K/V head h_kv = h_q / (H_q/H_kv) (BootstrapAI evolution
// log, collab-014 "Kernel 9 GQA"), bf16 in, fp32 accumulation, bf16 out.
//
// How (GB300-first; the pages' sm_89 kernels are prior art only):
//   * Persistent grid of one CTA per SM pulling work units from an atomic
//     counter (the persistent-kernel entry of the BootstrapAI evolution log),
//     in heavy-first causal order. A unit = two 128-row query tiles of the
//     same K/V group, so every K/V block loaded serves two query tiles (and,
//     when g is even, two query heads of the group at the same q_tile).
//   * Warp roles (the producer/consumer split of the log's warp-specialised
//     kernel, re-done with mbarriers instead of spinning flags):
//       warps 0-3  softmax + epilogue for query tile 0 (thread = query row)
//       warps 4-7  softmax + epilogue for query tile 1
//       warp  8    TMA producer: Q tiles and a ring of K/V blocks
//       warp  9    tcgen05 MMA issuer (and tensor-memory owner)
//   * Tensor memory (512 columns): S_t = Q_t K^T in columns [128t, 128t+128)
//     as fp32; P_t (bf16, packed in pairs) overwrites the upper half of S_t;
//     O_t accumulates in columns [256 + t*D, 256 + (t+1)*D).
//   * S = Q K^T: tcgen05.mma kind::f16, A = Q (smem, K-major), B = K (smem,
//     K-major), M = N = 128. O += P V: A = P from tensor memory, B = V (smem,
//     MN-major), M = 128, N = D. Tiles are TMA-copied with the 128-byte
//     swizzle the MMA descriptors expect.
//   * Online softmax (BootstrapAI collab-005 "Kernel 2 tiling") in fp32
//     registers with exp2 and the scale folded into the exponent. The
//     running maximum is only raised when it grows by more than 2^8, so O is
//     rescaled in tensor memory rarely; the result is unchanged because O and
//     the running sum always use the same reference maximum.
//   * Every wait is bounded: a stuck pipeline records kErrTimeout in the
//     workspace error word and unwinds instead of hanging the GPU.
#include <cuda_runtime.h>
#include <math.h>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {

namespace {

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows > 2^8

template <int D>
struct TcLayout {
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row bf16 tile
  static constexpr int kPanelBytes = 128 * 128;   // 128 rows x 64 columns
  static constexpr int kStages = (D == 128) ? 4 : 8;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kTileBytes;
  static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
  // barrier indices
  static constexpr int kQFull = 0, kQEmpty = 2, kSFull = 4, kPFull = 6, kOFull = 8,
                       kOEmpty = 10, kSchedFull = 12, kSchedEmpty = 14, kDrain = 16,
                       kKVFull = 17, kKVEmpty = 17 + kStages;
  static constexpr int kNumBars = 17 + 2 * kStages;
  static constexpr int kOffSched = kOffBar + kNumBars * 8;
  static constexpr int kOffTmem = kOffSched + 8;
  static constexpr int kOffAbort = kOffTmem + 4;
  static constexpr int kBytes = kOffAbort + 4;
  static constexpr int kAlloc = kBytes + 1024;
};

struct TcParams {
  __nv_bfloat16 *o;
  PrefillPlan plan;
  float scale_log2;
  int *ctl;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const TcParams prm) {
  using L = TcLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t bars = s_base + L::kOffBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  volatile int *sched = reinterpret_cast<volatile int *>(smem + L::kOffSched);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffTmem);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffAbort);

  const PrefillPlan &plan = prm.plan;
  int *err_word = prm.ctl + kCtlErr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::kQFull + t), 1);
      mbar_init(bar(L::kQEmpty + t), 1);
      mbar_init(bar(L::kSFull + t), 1);
      mbar_init(bar(L::kPFull + t), 128);
      mbar_init(bar(L::kOFull + t), 1);
      mbar_init(bar(L::kOEmpty + t), 128);
      mbar_init(bar(L::kSchedFull + t), 1);
      mbar_init(bar(L::kSchedEmpty + t), 9);  // MMA lane + 8 softmax warps
    }
    mbar_init(bar(L::kDrain), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kKVFull + s), 1);
      mbar_init(bar(L::kKVEmpty + s), 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    *abort_flag = 1;
    record_error(err_word, kErrTimeout);
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0, kv_it = 0, vc[2] = {0, 0};
      while (true) {
        const int u = atomicAdd(prm.ctl + kCtlWork, 1);
        const int slot = it & 1;
        if (!mbar_wait(bar(L::kSchedEmpty + slot), ((it >> 1) & 1) ^ 1, abort_flag)) { fail(); break; }
        sched[slot] = u;
        mbar_arrive(bar(L::kSchedFull + slot));
        ++it;
        if (u >= plan.total_units) break;
        const Unit w = decode_unit(plan, u);
        const int nb = max(w.t[0].kv_blocks, w.t[1].kv_blocks);
        bool ok = true;
        for (int t = 0; t < 2 && ok; ++t) {
          if (w.t[t].kv_blocks == 0) continue;
          if (!mbar_wait(bar(L::kQEmpty + t), (vc[t] & 1) ^ 1, abort_flag)) { ok = false; break; }
          ++vc[t];
          const uint32_t dst = s_base + L::kOffQ + t * L::kTileBytes;
          mbar_arrive_expect_tx(bar(L::kQFull + t), L::kTileBytes);
#pragma unroll
          for (int p = 0; p < D / 64; ++p)
            tma_load_3d(dst + p * L::kPanelBytes, &tm_q, bar(L::kQFull + t), p * 64,
                        w.t[t].q_tile * kTileM, w.b * plan.H_q + w.t[t].h_q);
        }
        const int kv_plane = w.b * plan.H_kv + w.h_kv;
        for (int j = 0; j < nb && ok; ++j) {
          for (int kind = 0; kind < 2; ++kind) {  // K_j then V_j
            const int st = kv_it % L::kStages;
            const uint32_t ph = (kv_it / L::kStages) & 1;
            if (!mbar_wait(bar(L::kKVEmpty + st), ph ^ 1, abort_flag)) { ok = false; break; }
            const uint32_t dst = s_base + L::kOffKV + st * L::kTileBytes;
            mbar_arrive_expect_tx(bar(L::kKVFull + st), L::kTileBytes);
#pragma unroll
            for (int p = 0; p < D / 64; ++p)
              tma_load_3d(dst + p * L::kPanelBytes, kind ? &tm_v : &tm_k, bar(L::kKVFull + st),
                          p * 64, j * kTileN, kv_plane);
            ++kv_it;
          }
        }
        if (!ok) { fail(); break; }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
      int it = 0, kv_it = 0, vc[2] = {0, 0};
      uint32_t pcnt[2] = {0, 0};
      bool ok = true;

      auto issue_qk = [&](int t, int st) {
        const uint32_t qa = s_base + L::kOffQ + t * L::kTileBytes;
        const uint32_t kb = s_base + L::kOffKV + st * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kPanelBytes + (kk & 3) * 32;
          mma_ss(tmem + 128u * t, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                 idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int st, bool accumulate) {
        const uint32_t vb = s_base + L::kOffKV + st * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)
          mma_ts(tmem + 256u + D * t, tmem + 128u * t + 64u + kk * 8, sdesc_sw128(vb + kk * 2048, L::kPanelBytes, 1024),
                 idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
      };
      auto wait_kv = [&](int &st) -> bool {
        st = kv_it % L::kStages;
        const uint32_t ph = (kv_it / L::kStages) & 1;
        ++kv_it;
        return mbar_wait(bar(L::kKVFull + st), ph, abort_flag);
      };
      // PV for tile t over block jb (all checks on the caller's side).
      auto do_pv = [&](int t, int jb, int st) -> bool {
        if (jb == 0 && !mbar_wait(bar(L::kOEmpty + t), (vc[t] & 1) ^ 1, abort_flag)) return false;
        if (!mbar_wait(bar(L::kPFull + t), pcnt[t] & 1, abort_flag)) return false;
        ++pcnt[t];
        tc_fence_after_sync();
        issue_pv(t, st, jb > 0);
        return true;
      };

      while (ok) {
        const int slot = it & 1;
        if (!mbar_wait(bar(L::kSchedFull + slot), (it >> 1) & 1, abort_flag)) { ok = false; break; }
        const int u = sched[slot];
        mbar_arrive(bar(L::kSchedEmpty + slot));
        ++it;
        if (u >= plan.total_units) break;
        const Unit w = decode_unit(plan, u);
        const int nbt[2] = {w.t[0].kv_blocks, w.t[1].kv_blocks};
        const int nb = max(nbt[0], nbt[1]);
        for (int t = 0; t < 2 && ok; ++t)
          if (nbt[t] > 0 && !mbar_wait(bar(L::kQFull + t), vc[t] & 1, abort_flag)) ok = false;
        if (!ok) break;
        // block 0: S_t = Q_t K_0^T
        int st_k, st_v;
        if (!wait_kv(st_k)) { ok = false; break; }
        tc_fence_after_sync();
        for (int t = 0; t < 2; ++t) {
          if (nbt[t] == 0) continue;
          issue_qk(t, st_k);
          tc_commit(bar(L::kSFull + t));
          if (nbt[t] == 1) tc_commit(bar(L::kQEmpty + t));
        }
        // blocks 1..nb-1: O_t += P_t V_{j-1}, then S_t = Q_t K_j^T
        for (int j = 1; j < nb && ok; ++j) {
          tc_commit(bar(L::kKVEmpty + st_k));  // K_{j-1} no longer read after this point
          if (!wait_kv(st_v) || !wait_kv(st_k)) { ok = false; break; }
          tc_fence_after_sync();
          for (int t = 0; t < 2 && ok; ++t) {
            if (j - 1 < nbt[t]) {
              if (!do_pv(t, j - 1, st_v)) { ok = false; break; }
              if (j - 1 == nbt[t] - 1) tc_commit(bar(L::kOFull + t));
            }
            if (j < nbt[t]) {
              issue_qk(t, st_k);
              tc_commit(bar(L::kSFull + t));
              if (j == nbt[t] - 1) tc_commit(bar(L::kQEmpty + t));
            }
          }
          tc_commit(bar(L::kKVEmpty + st_v));
        }
        if (!ok) break;
        // last block: O_t += P_t V_{nb-1}
        tc_commit(bar(L::kKVEmpty + st_k));
        if (!wait_kv(st_v)) { ok = false; break; }
        tc_fence_after_sync();
        for (int t = 0; t < 2 && ok; ++t) {
          if (nbt[t] != nb) continue;
          if (!do_pv(t, nb - 1, st_v)) { ok = false; break; }
          tc_commit(bar(L::kOFull + t));
        }
        tc_commit(bar(L::kKVEmpty + st_v));
        for (int t = 0; t < 2; ++t)
          if (nbt[t] > 0) ++vc[t];
      }
      if (!ok) fail();
      // Drain: every tcgen05 operation issued above has completed.
      tc_commit(bar(L::kDrain));
      mbar_wait(bar(L::kDrain), 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int t = warp >> 2;                       // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;        // row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tm_s = tmem + lane_off + t * 128u;
    const uint32_t tm_p = tm_s + 64u;
    const uint32_t tm_o = tmem + lane_off + 256u + t * D;
    const float sl2 = prm.scale_log2;
    int it = 0, vc = 0;
    uint32_t scnt = 0;
    bool ok = true;
    while (ok) {
      const int slot = it & 1;
      if (!mbar_wait(bar(L::kSchedFull + slot), (it >> 1) & 1, abort_flag)) { ok = false; break; }
      const int u = sched[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kSchedEmpty + slot));
      ++it;
      if (u >= plan.total_units) break;
      const Unit w = decode_unit(plan, u);
      const int nbt = w.t[t].kv_blocks;
      if (nbt == 0) continue;
      const int q_row = w.t[t].q_tile * kTileM + row;
      // last visible key of this row (inclusive)
      int lim = plan.N_kv - 1;
      if (plan.causal) lim = min(lim, q_row + plan.kv_offset);
      float m_ref = -INFINITY;  // reference maximum, log2-scaled units
      float l_sum = 0.f;
      for (int j = 0; j < nbt; ++j) {
        if (!mbar_wait(bar(L::kSFull + t), scnt & 1, abort_flag)) { ok = false; break; }
        ++scnt;
        __syncwarp();  // tcgen05.ld/st below are warp-collective
        tc_fence_after_sync();
        uint32_t sr[128];
        tmem_ld128_wait(tm_s, sr);
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        const int kbase = j * kTileN;
        if (__any_sync(0xffffffffu, kbase + kTileN - 1 > lim)) {
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (kbase + c > lim) ? -INFINITY : s[c];
        }
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int c = 4; c < 128; c += 4) {
          mx0 = fmaxf(mx0, s[c]);
          mx1 = fmaxf(mx1, s[c + 1]);
          mx2 = fmaxf(mx2, s[c + 2]);
          mx3 = fmaxf(mx3, s[c + 3]);
        }
        const float m_blk = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
        // Raise the reference maximum only when it grows by more than 2^8
        // (always on the first block, whose O is overwritten anyway).
        float alpha = 1.f;
        const bool raise = (j == 0) || (m_blk > m_ref + kRescaleThreshold);
        if (raise) {
          const float m_new = fmaxf(m_ref, m_blk);
          alpha = (j == 0) ? 0.f : ex2(m_ref - m_new);
          m_ref = m_new;
        }
        __syncwarp();
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t ov[32];
            tmem_ld32_wait(tm_o + c0, ov);
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st32(tm_o + c0, ov);
          }
        }
        const float neg_m = -m_ref;
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float p0 = ex2(fmaf(s[h * 64 + 2 * c], sl2, neg_m));
            const float p1 = ex2(fmaf(s[h * 64 + 2 * c + 1], sl2, neg_m));
            ls0 += p0;
            ls1 += p1;
            pk[c] = pack_bf16x2(p0, p1);
          }
          tmem_st32(tm_p + h * 32u, pk);
        }
        tmem_st_wait();
        l_sum = l_sum * alpha + (ls0 + ls1);
        tc_fence_before_sync();
        mbar_arrive(bar(L::kPFull + t));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16 -> global
      if (!mbar_wait(bar(L::kOFull + t), vc & 1, abort_flag)) { ok = false; break; }
      ++vc;
      __syncwarp();
      tc_fence_after_sync();
      const float inv_l = 1.f / l_sum;
      __nv_bfloat16 *dst =
          prm.o + ((static_cast<size_t>(w.b) * plan.H_q + w.t[t].h_q) * plan.N_q + q_row) * D;
      const bool store = q_row < plan.N_q;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        __syncwarp();
        tmem_ld32_wait(tm_o + c0, ov);
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack_bf16x2(__uint_as_float(ov[2 * c]) * inv_l,
                              __uint_as_float(ov[2 * c + 1]) * inv_l);
        if (store) {
          uint4 *g = reinterpret_cast<uint4 *>(dst + c0);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            g[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
      tc_fence_before_sync();
      mbar_arrive(bar(L::kOEmpty + t));
    }
    if (!ok) fail();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0) {
    // The last CTA to finish re-arms the work counter for the next launch.
    __threadfence();
    const int done = atomicAdd(prm.ctl + kCtlDone, 1);
    if (done == static_cast<int>(gridDim.x) - 1) {
      atomicExch(prm.ctl + kCtlWork, 0);
      atomicExch(prm.ctl + kCtlDone, 0);
    }
  }
}

template <int D>
cudaError_t launch_d(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                     void *o, const PrefillPlan &plan, float scale, int *ctl, int num_sms,
                     cudaStream_t stream) {
  using L = TcLayout<D>;
  static unsigned configured = 0;  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 32 && !(configured & (1u << dev))) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kAlloc);
    if (e != cudaSuccess) return e;
    configured |= 1u << dev;
  }
  TcParams prm;
  prm.o = static_cast<__nv_bfloat16 *>(o);
  prm.plan = plan;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.ctl = ctl;
  const int grid = min(num_sms, plan.total_units);
  prefill_tc_kernel<D><<<grid, kThreads, L::kAlloc, stream>>>(tm_q, tm_k, tm_v, prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, void *o, const PrefillPlan &plan, int d,
                              float scale, int *ctl, int num_sms, cudaStream_t stream) {
  if (d == 64) return launch_d<64>(tm_q, tm_k, tm_v, o, plan, scale, ctl, num_sms, stream);
  if (d == 128) return launch_d<128>(tm_q, tm_k, tm_v, o, plan, scale, ctl, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gqa
