// Attention backward on the sm_103a tensor cores: dQ, dK and dV of
// O = softmax(scale Q K^T [+ causal mask]) V, with the GQA reduction of dK
// and dV over the query heads of a group (microLLM-rocm optimisation log,
// Experiments 051-057: causal GQA attention backward with row recompute and
// the softmax backward). bf16 in, fp32 accumulation, bf16 out.
//
// Per query row i of head h_q (K/V head h_kv = h_q / g), from the forward's
// per-row log-sum-exp lse_i:
//   P_ij  = exp(scale q_i.k_j - lse_i)          (row recompute)
//   D_i   = sum_c dO_ic O_ic
//   dP_ij = dO_i . v_j,     dS_ij = P_ij (dP_ij - D_i)
//   dQ_i  = scale sum_j dS_ij k_j
//   dK_j  = scale sum_{h_q of the group} sum_i dS_ij q_i
//   dV_j  =       sum_{h_q of the group} sum_i P_ij dO_i
//
// Two launches:
//   * bwd_prep_kernel: -D_i and -lse_i in log2 units into a workspace
//     padded to whole 128-row tiles (pad rows: 0 and -inf, so P = 0 there);
//     negated so that x = s scale log2(e) - lse and dP - D are single
//     packed fp32 operations.
//   * bwd_kernel: one grid with two kinds of CTA, one work unit each.
//     - dK/dV units (b, h_kv, 128-key block), first: K and V of the block
//       stay in shared memory; the CTA sweeps every query head of the group
//       and every query tile that sees the block, so the GQA reduction
//       happens in the tensor-memory accumulators, in a fixed order (no
//       atomics: the result is deterministic). Per (head, tile) t, with the
//       key rows as tensor-memory lanes, and per query half h of the tile:
//         S^T_h = K Q_th^T, dP^T_h = V dO_th^T  (tcgen05, N = 64, A and B
//                                               from shared memory)
//         P^T_h, dS^T_h  (4 warps, fp32, written back as bf16 over S^T_h
//                         and dP^T_h)
//         dV += P^T_h dO_th, dK += dS^T_h Q_th  (tcgen05, K = 64, A from
//                                                tensor memory)
//       The two halves have their own barriers and warps, so the products
//       of one half run while the softmax warps of the other half work;
//       the K-steps reach dV and dK in the same order as one K = 128
//       product would. Q_t, dO_t and the tile's lse / D arrive through a
//       two-stage TMA ring.
//     - dQ units (b, h_q, 128-row query tile), heaviest tiles first: Q and
//       dO stay in shared memory, K/V blocks stream through two TMA rings
//       (K blocks stay until their dQ product completes, V blocks only
//       until their dP product does):
//         S = Q K_j^T, dP = dO V_j^T; dS (8 warps); dQ += dS K_j.
//       S and dP have their own tensor-memory columns apart from dS, so the
//       next block's two products run while the softmax warps work on dS.
//   Tensor memory (512 columns): dK/dV units S^T [0,128), dP^T [128,256),
//   dV [256, 256+D), dK [256+D, 256+2D); dQ units S [0,128), dP [128,256),
//   dS [256,320), dQ [320, 320+D).
//   Warps 0-7 compute P and dS (warps w and w+4 share the lanes of warp
//   w % 4 and take one half of the 128 columns each: in dK/dV units, one
//   query half each) and store the results;
//   warp 8 issues the TMA loads, warp 9 the tcgen05 products. Every wait is
//   bounded: a stuck pipeline records kErrTimeout and unwinds.
#include <cuda_runtime.h>
#include <math.h>

#include <type_traits>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {

namespace {

constexpr int kThreads = 320;
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTmemCols = 512;

// barrier indices (both kinds of unit use the same slots)
enum {
  kInFull = 0,  // Q and dO (dQ units) or K and V (dK/dV units) loaded
  kSFull,       // S and dP products complete
  kSFree,       // softmax warps have read S and dP (dQ units)
  kDsFull,      // softmax warps have written dS (and P^T)
  kDsFree,      // the product reading dS has completed (dQ units)
  kAccFull,     // the accumulator is final
  kDrain,
  kRingFull0 = 8,
  kRingEmpty0 = 16,
  kSFull1 = 24,   // dK/dV units: S^T and dP^T of query half 1 complete
  kDsFull1,       // dK/dV units: P^T and dS^T of query half 1 written
  kNumBars
};

template <int D>
struct BwdLayout {
  static constexpr int kTile = kTileM * D * 2;    // 128 rows x D bf16
  static constexpr int kPanel = 128 * 128;        // 128 rows x 64 columns
  // dQ units: K and V blocks in rings of their own; a K block is read until
  // its dQ product completes, a V block only until its dP product does
  static constexpr int kRingK = D == 128 ? 3 : 5, kRingV = D == 128 ? 2 : 3;
  static constexpr int kRing = kRingK + kRingV;
  // dQ units: Q | dO | K/V ring
  static constexpr int kOffQ = 0, kOffDO = kTile, kOffRing = 2 * kTile;
  static constexpr int kEndQ = kOffRing + kRing * kTile;
  // dK/dV units: K | V | 2 stages of (Q, dO) | 2 stages of (lse[128], D[128])
  static constexpr int kOffK = 0, kOffV = kTile, kOffStage = 2 * kTile;
  static constexpr int kOffVec = kOffStage + 4 * kTile;
  static constexpr int kEndKV = kOffVec + 2 * 2 * kTileM * 4;
  static constexpr int kOffBar = kEndQ > kEndKV ? kEndQ : kEndKV;
  static constexpr int kOffTmem = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmem + 4;
  static constexpr int kBytes = kOffAbort + 4;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kRing <= kRingEmpty0 - kRingFull0, "ring barriers");
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

struct BwdParams {
  __nv_bfloat16 *dq, *dk, *dv;
  const float *lse2;   // [B*H_q][nq_pad]: -lse in log2 units, -inf on pad rows
  const float *delta;  // [B*H_q][nq_pad]: -D_i, 0 on pad rows
  int B, H_q, H_kv, N_q, N_kv, group, n_qt, n_kt, nq_pad, causal, kv_offset;
  int n_kv_units;      // blocks [0, n_kv_units) are dK/dV units, the rest dQ units
  float scale, scale_log2;
  int *err_word;
};

// 8 fp32 products of two 16-byte bf16 vectors, summed
__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b) {
  const __nv_bfloat162 *x = reinterpret_cast<const __nv_bfloat162 *>(&a);
  const __nv_bfloat162 *y = reinterpret_cast<const __nv_bfloat162 *>(&b);
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 u = __bfloat1622float2(x[k]), v = __bfloat1622float2(y[k]);
    s = fmaf(u.x, v.x, s);
    s = fmaf(u.y, v.y, s);
  }
  return s;
}

// -D_i = -sum_c dO_ic O_ic and -lse_i * log2(e), for every row of the padded
// [B*H_q][nq_pad] layout; 8 lanes per row, each over D/8 contiguous columns.
// OD: the head dim, the row stride of o, dO, dQ, dK, dV and the columns
// stored (<= D; the TMA boxes read zeros past it, so at d = 32 and 96 the
// 64- and 128-column kernels compute on zero-padded tiles).
template <int D, int OD>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *o,
                                                       const __nv_bfloat16 *dout,
                                                       const float *lse, float *lse2,
                                                       float *delta, int rows, int N_q,
                                                       int nq_pad) {
  // o, dO and lse may come from the previous kernel of the stream
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31, sub = lane & 7;
  const long long total = static_cast<long long>(rows) * nq_pad;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long r0 = (static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 4;
       r0 < total; r0 += warps * 4) {
    const long long r = r0 + (lane >> 3);
    const long long bh = r / nq_pad;
    const int i = static_cast<int>(r - bh * nq_pad);
    const bool valid = r < total && i < N_q;
    float acc = 0.f;
    if (valid) {
      const size_t base = (static_cast<size_t>(bh) * N_q + i) * OD + sub * (D / 8);
#pragma unroll
      for (int c = 0; c < D / 8; c += 8)
        if (sub * (D / 8) + c < OD)  // columns past the head dim do not exist
          acc += dot8_bf16(__ldg(reinterpret_cast<const uint4 *>(o + base + c)),
                           __ldg(reinterpret_cast<const uint4 *>(dout + base + c)));
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (sub == 0 && r < total) {
      float l2 = -INFINITY;  // pad rows (and a row with no visible key): P = 0
      if (valid) {
        const float l = __ldg(lse + static_cast<size_t>(bh) * N_q + i);
        if (l != -INFINITY) l2 = l * -1.4426950408889634f;
      }
      delta[r] = valid ? -acc : 0.f;
      lse2[r] = l2;
    }
  }
}

template <int D, int OD>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const BwdParams prm) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  // offset (not integer) arithmetic on smem_raw keeps the pointer in the
  // shared window, so accesses through it compile to shared-memory loads
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t s_base = smem_addr(smem);
  auto bar = [&](int i) -> uint32_t { return s_base + L::kOffBar + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffTmem);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffAbort);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool kv_unit = static_cast<int>(blockIdx.x) < prm.n_kv_units;

  // ---- the unit
  int b, h_kv, h_q = 0, qt = 0, kb = 0, qt_first = 0, ntq = 0, n_iter;
  if (kv_unit) {
    // key blocks ascending: under the causal mask the first blocks are seen
    // by the most query tiles, so the heaviest units start first
    const int groups = prm.B * prm.H_kv;
    kb = static_cast<int>(blockIdx.x) / groups;
    const int bh = static_cast<int>(blockIdx.x) - kb * groups;
    b = bh / prm.H_kv;
    h_kv = bh - b * prm.H_kv;
    if (prm.causal) {
      // the first query row that sees key kb*128 (bottom-right alignment)
      const int first_row = kb * kTileN - prm.kv_offset;
      qt_first = first_row > 0 ? first_row / kTileM : 0;
    }
    ntq = max(0, prm.n_qt - qt_first);
    n_iter = prm.group * ntq;  // (query head, query tile) pairs, head-major
  } else {
    const int u = static_cast<int>(blockIdx.x) - prm.n_kv_units;
    const int heads = prm.B * prm.H_q;
    const int rank = u / heads;
    qt = prm.n_qt - 1 - rank;  // later query tiles see more keys: heaviest first
    const int bh = u - rank * heads;
    b = bh / prm.H_q;
    h_q = bh - b * prm.H_q;
    h_kv = h_q / prm.group;
    n_iter = prm.n_kt;
    if (prm.causal) {
      const int last_row = min((qt + 1) * kTileM, prm.N_q) - 1;
      n_iter = min(prm.n_kt, (last_row + prm.kv_offset) / kTileN + 1);
    }
  }

  if (tid == 0) {
    mbar_init(bar(kInFull), 1);
    mbar_init(bar(kSFull), 1);
    mbar_init(bar(kSFree), kSoftmaxWarps);
    mbar_init(bar(kDsFull), kv_unit ? kSoftmaxWarps / 2 : kSoftmaxWarps);
    mbar_init(bar(kSFull1), 1);
    mbar_init(bar(kDsFull1), kSoftmaxWarps / 2);
    mbar_init(bar(kDsFree), 1);
    mbar_init(bar(kAccFull), 1);
    mbar_init(bar(kDrain), 1);
    for (int s = 0; s < L::kRing; ++s) {
      mbar_init(bar(kRingFull0 + s), 1);
      mbar_init(bar(kRingEmpty0 + s), 1);
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
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // D and lse come from the prep kernel just before this one
  grid_dependency_wait();
  grid_launch_dependents();

  auto fail = [&]() {
    *abort_flag = 1;
    record_error(prm.err_word, kErrTimeout);
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      const int plane_kv = b * prm.H_kv + h_kv;
      if (!kv_unit) {
        const int plane_q = b * prm.H_q + h_q;
        mbar_arrive_expect_tx(bar(kInFull), 2 * L::kTile);
#pragma unroll
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d(s_base + L::kOffQ + p * L::kPanel, &tm_q, bar(kInFull), p * 64,
                      qt * kTileM, plane_q);
          tma_load_3d(s_base + L::kOffDO + p * L::kPanel, &tm_do, bar(kInFull), p * 64,
                      qt * kTileM, plane_q);
        }
        // K_j and V_j, each through its own ring
        for (int j = 0; j < n_iter && ok; ++j) {
#pragma unroll
          for (int kind = 0; kind < 2; ++kind) {
            const int n = kind ? L::kRingV : L::kRingK;
            const int slot = (kind ? L::kRingK : 0) + j % n;
            if (!mbar_wait(bar(kRingEmpty0 + slot), ((j / n) & 1) ^ 1, abort_flag)) {
              ok = false;
              break;
            }
            const uint32_t dst = s_base + L::kOffRing + slot * L::kTile;
            mbar_arrive_expect_tx(bar(kRingFull0 + slot), L::kTile);
#pragma unroll
            for (int p = 0; p < D / 64; ++p)
              tma_load_3d(dst + p * L::kPanel, kind ? &tm_v : &tm_k, bar(kRingFull0 + slot), p * 64,
                          j * kTileN, plane_kv);
          }
        }
      } else {
        mbar_arrive_expect_tx(bar(kInFull), 2 * L::kTile);
#pragma unroll
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d(s_base + L::kOffK + p * L::kPanel, &tm_k, bar(kInFull), p * 64, kb * kTileN,
                      plane_kv);
          tma_load_3d(s_base + L::kOffV + p * L::kPanel, &tm_v, bar(kInFull), p * 64, kb * kTileN,
                      plane_kv);
        }
        // per (head, query tile): Q_t, dO_t, and the tile's lse and D
        for (int t = 0; t < n_iter && ok; ++t) {
          const int st = t & 1;
          if (!mbar_wait(bar(kRingEmpty0 + st), ((t >> 1) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const int hq = h_kv * prm.group + t / ntq, qtt = qt_first + t % ntq;
          const int plane_q = b * prm.H_q + hq;
          const uint32_t dst = s_base + L::kOffStage + st * 2 * L::kTile;
          mbar_arrive_expect_tx(bar(kRingFull0 + st), 2 * L::kTile + 2 * kTileM * 4);
#pragma unroll
          for (int p = 0; p < D / 64; ++p) {
            tma_load_3d(dst + p * L::kPanel, &tm_q, bar(kRingFull0 + st), p * 64, qtt * kTileM,
                        plane_q);
            tma_load_3d(dst + L::kTile + p * L::kPanel, &tm_do, bar(kRingFull0 + st), p * 64,
                        qtt * kTileM, plane_q);
          }
          // rows of the padded workspace: 512-byte aligned runs
          const size_t vec = static_cast<size_t>(plane_q) * prm.nq_pad + qtt * kTileM;
          const uint32_t vdst = s_base + L::kOffVec + st * 2 * kTileM * 4;
          bulk_load(vdst, prm.lse2 + vec, kTileM * 4, bar(kRingFull0 + st));
          bulk_load(vdst + kTileM * 4, prm.delta + vec, kTileM * 4, bar(kRingFull0 + st));
        }
      }
      if (!ok) fail();
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
    constexpr uint32_t kHi = sdesc_hi_sw128(1024);
    bool ok = true;
    // d = A B^T over D: A and B 128 x D tiles, K-major, 128-byte swizzled panels
    auto mma_ss = [&](uint32_t d, uint32_t a_lo, uint32_t b_lo) {
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off =
              static_cast<uint32_t>(((kk >> 2) * L::kPanel + (kk & 3) * 32) >> 4);
          mma_ss_w(d, a_lo + off, kHi, b_lo + off, kHi, idesc_ss, kk > 0 ? 1u : 0u);
        }
      }
      __syncwarp();
    };
    // d (+)= A B over 128: A from tensor memory as bf16 pairs (K-steps 0-3
    // at columns a_lo + 8 kk, 4-7 at a_hi + 8 (kk - 4)), B a 128 x D tile
    // read MN-major
    auto mma_ts = [&](uint32_t d, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, bool acc) {
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t a = kk < 4 ? a_lo + 8u * kk : a_hi + 8u * (kk - 4);
          mma_ts_w(d, a, b_lo + 128u * kk, kHi, idesc_acc, (acc || kk > 0) ? 1u : 0u);
        }
      }
      __syncwarp();
    };
    auto commit = [&](int i) {
      if (elect_one()) tc_commit(bar(i));
      __syncwarp();
    };
    if (!kv_unit) {
      const uint32_t q_lo = sdesc_lo(s_base + L::kOffQ, 16);
      const uint32_t do_lo = sdesc_lo(s_base + L::kOffDO, 16);
      const uint32_t ring_lo = sdesc_lo(s_base + L::kOffRing, 16);
      const uint32_t ring_mn = sdesc_lo(s_base + L::kOffRing, L::kPanel);
      const uint32_t tS = tmem, tDP = tmem + 128, tDS = tmem + 256, tDQ = tmem + 320;
      ok = mbar_wait_warp(bar(kInFull), 0, abort_flag);
      int st_k_prev = 0;
      for (int j = 0; j < n_iter && ok; ++j) {
        const int st_k = j % L::kRingK, st_v = L::kRingK + j % L::kRingV;
        if (!mbar_wait_warp(bar(kRingFull0 + st_k), (j / L::kRingK) & 1, abort_flag) ||
            !mbar_wait_warp(bar(kRingFull0 + st_v), (j / L::kRingV) & 1, abort_flag)) {
          ok = false;
          break;
        }
        // S and dP of the previous block have been read by the softmax warps
        if (j > 0 && !mbar_wait_warp(bar(kSFree), (j - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        mma_ss(tS, q_lo, ring_lo + static_cast<uint32_t>((st_k * L::kTile) >> 4));
        mma_ss(tDP, do_lo, ring_lo + static_cast<uint32_t>((st_v * L::kTile) >> 4));
        commit(kSFull);
        commit(kRingEmpty0 + st_v);  // V_j is not read again
        if (j > 0) {
          // dQ += dS_{j-1} K_{j-1}
          if (!mbar_wait_warp(bar(kDsFull), (j - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          mma_ts(tDQ, tDS, tDS + 32, ring_mn + static_cast<uint32_t>((st_k_prev * L::kTile) >> 4),
                 j > 1);
          commit(kDsFree);
          commit(kRingEmpty0 + st_k_prev);
        }
        st_k_prev = st_k;
      }
      if (ok && n_iter > 0) {
        if (!mbar_wait_warp(bar(kDsFull), (n_iter - 1) & 1, abort_flag)) {
          ok = false;
        } else {
          tc_fence_after_sync();
          mma_ts(tDQ, tDS, tDS + 32, ring_mn + static_cast<uint32_t>((st_k_prev * L::kTile) >> 4),
                 n_iter > 1);
          commit(kRingEmpty0 + st_k_prev);
        }
      }
      if (ok) commit(kAccFull);
    } else {
      const uint32_t k_lo = sdesc_lo(s_base + L::kOffK, 16);
      const uint32_t v_lo = sdesc_lo(s_base + L::kOffV, 16);
      const uint32_t tST = tmem, tDPT = tmem + 128, tDV = tmem + 256, tDK = tmem + 256 + D;
      constexpr uint32_t idesc_half = idesc_bf16_f32(128, 64, false, false);
      // S^T and dP^T of query half h of stage st: N = 64, B rows [64h, 64h+64)
      auto issue_s = [&](int st, int h) {
        const uint32_t stq = s_base + L::kOffStage + st * 2 * L::kTile + h * 64 * 128;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off =
                static_cast<uint32_t>(((kk >> 2) * L::kPanel + (kk & 3) * 32) >> 4);
            mma_ss_w(tST + 64u * h, k_lo + off, kHi, sdesc_lo(stq, 16) + off, kHi, idesc_half,
                     kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off =
                static_cast<uint32_t>(((kk >> 2) * L::kPanel + (kk & 3) * 32) >> 4);
            mma_ss_w(tDPT + 64u * h, v_lo + off, kHi, sdesc_lo(stq + L::kTile, 16) + off, kHi,
                     idesc_half, kk > 0 ? 1u : 0u);
          }
        }
        __syncwarp();
        commit(h ? kSFull1 : kSFull);
      };
      // dV += P^T dO and dK += dS^T Q over query half h (K = 64): P^T and
      // dS^T sit in the first 32 columns of that half's S^T and dP^T
      auto issue_acc = [&](int st, int h, bool acc) {
        const uint32_t stq = s_base + L::kOffStage + st * 2 * L::kTile;
        const uint32_t do_mn = sdesc_lo(stq + L::kTile, L::kPanel);
        const uint32_t q_mn = sdesc_lo(stq, L::kPanel);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts_w(tDV, tST + 64u * h + 8u * kk, do_mn + 128u * (4 * h + kk), kHi, idesc_acc,
                     (acc || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts_w(tDK, tDPT + 64u * h + 8u * kk, q_mn + 128u * (4 * h + kk), kHi, idesc_acc,
                     (acc || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
      };
      ok = mbar_wait_warp(bar(kInFull), 0, abort_flag);
      if (ok && n_iter > 0) {
        ok = mbar_wait_warp(bar(kRingFull0), 0, abort_flag);
        if (ok) {
          tc_fence_after_sync();
          issue_s(0, 0);
          issue_s(0, 1);
        }
      }
      // the halves alternate so that one half's products run while the
      // softmax warps of the other half work
      for (int t = 0; t < n_iter && ok; ++t) {
        const int st = t & 1;
        for (int h = 0; h < 2 && ok; ++h) {
          if (!mbar_wait_warp(bar(h ? kDsFull1 : kDsFull), t & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_acc(st, h, t > 0 || h > 0);
          if (h == 1) commit(kRingEmpty0 + st);  // Q_t, dO_t and the vectors are free
          if (t + 1 < n_iter) {
            if (h == 0) {
              if (!mbar_wait_warp(bar(kRingFull0 + (st ^ 1)), ((t + 1) >> 1) & 1, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
            }
            issue_s(st ^ 1, h);
          }
        }
      }
      if (ok) commit(kAccFull);
    }
    if (!ok && lane == 0) fail();
    // every tcgen05 operation issued above has completed
    commit(kDrain);
    mbar_wait_warp(bar(kDrain), 0, nullptr);
  } else {
    // ------------------------------------------------------------ softmax warps
    const int half = warp >> 2;                 // which 64 of the 128 columns
    const int row = (warp & 3) * 32 + lane;     // tensor-memory lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = prm.scale_log2;
    bool ok = true;
    auto arrive = [&](int i) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(i));
    };
    // an accumulator row: D/2 columns from tensor memory, times mul, to bf16 at dst
    // half h of a row: columns [h D/2, (h+1) D/2), of which those below OD
    // exist in memory
    auto store_half_row = [&](uint32_t taddr, __nv_bfloat16 *dst, int half, float mul, bool store,
                              bool zero) {
      uint32_t v[D / 2];
      if constexpr (D == 128)
        tmem_ld64_wait(taddr, v);
      else
        tmem_ld32_wait(taddr, v);
      if (!store) return;
      uint4 *g = reinterpret_cast<uint4 *>(dst);
#pragma unroll
      for (int c = 0; c < D / 2; c += 8) {
        if (OD < D && half * (D / 2) + c >= OD) continue;  // columns past the head dim
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          w[k] = zero ? 0u
                      : pack_bf16x2(__uint_as_float(v[c + 2 * k]) * mul,
                                    __uint_as_float(v[c + 2 * k + 1]) * mul);
        g[c / 8] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    };
    if (!kv_unit) {
      // thread = query row i; columns = keys
      const int i = qt * kTileM + row;
      const size_t vrow = static_cast<size_t>(b * prm.H_q + h_q) * prm.nq_pad + i;
      // -lse_i log2(e) and -D_i, as pairs for the packed fp32 operations
      const float nl2 = __ldg(prm.lse2 + vrow), nd = __ldg(prm.delta + vrow);
      const float2 nl2v = make_float2(nl2, nl2), ndv = make_float2(nd, nd);
      const float2 sl2v = make_float2(sl2, sl2);
      int lim = prm.N_kv - 1;  // last visible key (bottom-right causal)
      if (prm.causal) lim = min(lim, i + prm.kv_offset);
      for (int j = 0; j < n_iter; ++j) {
        if (!mbar_wait_warp(bar(kSFull), j & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t sv[64], pv[64];
        tmem_ld64_wait(tmem + lane_off + half * 64u, sv);
        tmem_ld64_wait(tmem + lane_off + 128u + half * 64u, pv);
        tc_fence_before_sync();
        arrive(kSFree);
        const int kbase = j * kTileN + half * 64;
        // columns c > cut of this half are past the last visible key
        const int cut = lim - kbase;
        uint32_t pk[32];
        // dS for the 64 columns; kMasked only on blocks that reach past a
        // row's last visible key (a warp-uniform choice, so the common
        // blocks carry no per-element compare)
        auto make_ds = [&](auto masked) {
          constexpr bool kMasked = decltype(masked)::value;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            float2 p = ffma2(make_float2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])),
                             sl2v, nl2v);
            p.x = ex2(p.x);
            p.y = ex2(p.y);
            if constexpr (kMasked) {
              p.x = 2 * c > cut ? 0.f : p.x;
              p.y = 2 * c + 1 > cut ? 0.f : p.y;
            }
            const float2 ds = fmul2(
                p, fadd2(make_float2(__uint_as_float(pv[2 * c]), __uint_as_float(pv[2 * c + 1])), ndv));
            pk[c] = pack_bf16x2(ds.x, ds.y);
          }
        };
        if (__any_sync(0xffffffffu, cut < 63))
          make_ds(std::true_type{});
        else
          make_ds(std::false_type{});
        // dS's columns are free once the previous block's dQ product completed
        if (j > 0 && !mbar_wait_warp(bar(kDsFree), (j - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        tmem_st32(tmem + lane_off + 256u + half * 32u, pk);
        tmem_st_wait();
        tc_fence_before_sync();
        arrive(kDsFull);
      }
      if (ok) {
        if (!mbar_wait_warp(bar(kAccFull), 0, abort_flag)) {
          ok = false;
        } else {
          tc_fence_after_sync();
          __nv_bfloat16 *dst = prm.dq +
                               (static_cast<size_t>(b * prm.H_q + h_q) * prm.N_q + i) * OD + half * (D / 2);
          store_half_row(tmem + lane_off + 320u + half * (D / 2), dst, half, prm.scale, i < prm.N_q,
                         n_iter == 0);
        }
      }
    } else {
      // thread = key row j; columns = query rows of the tile
      const int j = kb * kTileN + row;
      const float4 *vec = reinterpret_cast<const float4 *>(smem + L::kOffVec);
      for (int t = 0; t < n_iter; ++t) {
        const int st = t & 1, qtt = qt_first + t % ntq;
        if (!mbar_wait_warp(bar(half ? kSFull1 : kSFull), t & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t sv[64], pv[64];
        tmem_ld64_wait(tmem + lane_off + half * 64u, sv);
        tmem_ld64_wait(tmem + lane_off + 128u + half * 64u, pv);
        const float4 *lse2v = vec + st * 64 + half * 16;  // this half's 64 rows
        const float4 *dltv = lse2v + 32;
        // key j is visible to query row i iff j <= i + kv_offset: here the
        // columns c < cut are not
        const int cut = j - (qtt * kTileM + half * 64) - prm.kv_offset;
        uint32_t ppk[32], dpk[32];
        // P^T and dS^T for the 64 columns; kMasked only on tiles that cross
        // the causal diagonal (a warp-uniform choice, so the common tiles
        // carry no per-element compare)
        auto make_p_ds = [&](auto masked) {
          constexpr bool kMasked = decltype(masked)::value;
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            const float4 l4 = lse2v[c4], d4 = dltv[c4];  // -lse log2(e) and -D
            float2 p[2], ds[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = 4 * c4 + 2 * e;
              p[e] = ffma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])),
                           make_float2(sl2, sl2), e ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y));
              p[e].x = ex2(p[e].x);
              p[e].y = ex2(p[e].y);
              if constexpr (kMasked) {
                p[e].x = c < cut ? 0.f : p[e].x;
                p[e].y = c + 1 < cut ? 0.f : p[e].y;
              }
              ds[e] = fmul2(p[e], fadd2(make_float2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])),
                                        e ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y)));
            }
            ppk[2 * c4] = pack_bf16x2(p[0].x, p[0].y);
            ppk[2 * c4 + 1] = pack_bf16x2(p[1].x, p[1].y);
            dpk[2 * c4] = pack_bf16x2(ds[0].x, ds[0].y);
            dpk[2 * c4 + 1] = pack_bf16x2(ds[1].x, ds[1].y);
          }
        };
        if (prm.causal && __any_sync(0xffffffffu, cut > 0))
          make_p_ds(std::true_type{});
        else
          make_p_ds(std::false_type{});
        // P^T over S^T and dS^T over dP^T, in this half's own columns
        tmem_st32(tmem + lane_off + half * 64u, ppk);
        tmem_st32(tmem + lane_off + 128u + half * 64u, dpk);
        tmem_st_wait();
        tc_fence_before_sync();
        arrive(half ? kDsFull1 : kDsFull);
      }
      if (ok) {
        if (!mbar_wait_warp(bar(kAccFull), 0, abort_flag)) {
          ok = false;
        } else {
          tc_fence_after_sync();
          const size_t at = (static_cast<size_t>(b * prm.H_kv + h_kv) * prm.N_kv + j) * OD + half * (D / 2);
          const bool store = j < prm.N_kv, zero = n_iter == 0;
          store_half_row(tmem + lane_off + 256u + half * (D / 2), prm.dv + at, half, 1.f, store, zero);
          store_half_row(tmem + lane_off + 256u + D + half * (D / 2), prm.dk + at, half, prm.scale, store,
                         zero);
        }
      }
    }
    if (!ok) fail();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int OD>
cudaError_t launch_bwd_d(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                         const CUtensorMap &tm_do, const void *o, const void *dout,
                         const float *lse, float *work, void *dq, void *dk, void *dv, int B,
                         int H_q, int H_kv, int N_q, int N_kv, int causal, float scale,
                         int num_sms, int *err_word, cudaStream_t stream) {
  using L = BwdLayout<D>;
  static unsigned configured = 0;  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(configured & (1u << dev))) {
    e = cudaFuncSetAttribute(bwd_kernel<D, OD>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    if (dev < 32) configured |= 1u << dev;
  }
  const int n_qt = (N_q + kTileM - 1) / kTileM, n_kt = (N_kv + kTileN - 1) / kTileN;
  const int nq_pad = n_qt * kTileM;
  const int rows = B * H_q;
  float *lse2 = work;
  float *delta = work + static_cast<size_t>(rows) * nq_pad;
  // prep: 32 rows per 256-thread block (4 per warp)
  const long long prep_rows = static_cast<long long>(rows) * nq_pad;
  long long prep_grid = (prep_rows + 31) / 32;
  if (prep_grid > 8LL * num_sms) prep_grid = 8LL * num_sms;
  e = launch_programmatic(bwd_prep_kernel<D, OD>, static_cast<int>(prep_grid), 256, 0, stream,
                          static_cast<const __nv_bfloat16 *>(o),
                          static_cast<const __nv_bfloat16 *>(dout), lse, lse2, delta, rows, N_q,
                          nq_pad);
  if (e != cudaSuccess) return e;
  BwdParams prm;
  prm.dq = static_cast<__nv_bfloat16 *>(dq);
  prm.dk = static_cast<__nv_bfloat16 *>(dk);
  prm.dv = static_cast<__nv_bfloat16 *>(dv);
  prm.lse2 = lse2;
  prm.delta = delta;
  prm.B = B;
  prm.H_q = H_q;
  prm.H_kv = H_kv;
  prm.N_q = N_q;
  prm.N_kv = N_kv;
  prm.group = H_q / H_kv;
  prm.n_qt = n_qt;
  prm.n_kt = n_kt;
  prm.nq_pad = nq_pad;
  prm.causal = causal ? 1 : 0;
  prm.kv_offset = N_kv - N_q;
  prm.n_kv_units = B * H_kv * n_kt;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.err_word = err_word;
  const long long grid = static_cast<long long>(prm.n_kv_units) + static_cast<long long>(B) * H_q * n_qt;
  return launch_programmatic(bwd_kernel<D, OD>, static_cast<int>(grid), kThreads, L::kAlloc, stream,
                             tm_q, tm_k, tm_v, tm_do, prm);
}

}  // namespace

size_t bwd_workspace_bytes(int B, int H_q, int N_q) {
  const size_t nq_pad = static_cast<size_t>((N_q + kTileM - 1) / kTileM) * kTileM;
  return 2 * static_cast<size_t>(B) * H_q * nq_pad * sizeof(float);
}

cudaError_t launch_attn_bwd(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                            const CUtensorMap &tm_v, const CUtensorMap &tm_do, const void *o,
                            const void *dout, const float *lse, float *work, void *dq, void *dk,
                            void *dv, int B, int H_q, int H_kv, int N_q, int N_kv, int d,
                            int causal, float scale, int num_sms, int *err_word,
                            cudaStream_t stream) {
  // head dims 32 and 96 run the 64- and 128-column kernels on zero-padded tiles
#define GQA_BWD(D_, OD_)                                                                     \
  launch_bwd_d<D_, OD_>(tm_q, tm_k, tm_v, tm_do, o, dout, lse, work, dq, dk, dv, B, H_q, H_kv, \
                        N_q, N_kv, causal, scale, num_sms, err_word, stream)
  switch (d) {
    case 32: return GQA_BWD(64, 32);
    case 64: return GQA_BWD(64, 64);
    case 96: return GQA_BWD(128, 96);
    case 128: return GQA_BWD(128, 128);
    default: return cudaErrorInvalidValue;
  }
#undef GQA_BWD
}

}  // namespace gqa
