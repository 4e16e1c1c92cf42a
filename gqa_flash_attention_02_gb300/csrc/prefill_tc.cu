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
//       warps 10-11 idle (they complete the third warpgroup, which gives
//                   its registers to the two softmax warpgroups)
//   * Tensor memory (512 columns): S_t = Q_t K^T in columns [128t, 128t+128)
//     as fp32; P_t (bf16, packed in pairs) overwrites the upper half of S_t;
//     O_t accumulates in columns [256 + t*D, 256 + (t+1)*D).
//   * S = Q K^T: tcgen05.mma kind::f16, A = Q (smem, K-major), B = K (smem,
//     K-major), M = N = 128. O += P V: A = P from tensor memory, B = V (smem,
//     MN-major), M = 128, N = D. Tiles are TMA-copied with the 128-byte
//     swizzle the MMA descriptors expect.
//   * Online softmax (BootstrapAI collab-005 "Kernel 2 tiling") in fp32
//     registers with exp2 and the scale folded into the exponent. The
//     running maximum is only raised when it grows by more than 2^4 (2^8
//     with fp32 exponentials), so O is rescaled in tensor memory rarely; the
//     result is unchanged because O and the running sum always use the same
//     reference maximum.
//   * Every wait is bounded: a stuck pipeline records kErrTimeout in the
//     workspace error word and unwinds instead of hanging the GPU.
//   * Ragged batches (prompts of different lengths packed token-major,
//     [total][H][d], with per-sequence offsets; the pages' batched prompt
//     prefill, microLLM-rocm optimisation log, Experiment 101) run the same
//     body as prefill_varlen_kernel: a one-block plan kernel first lists the
//     units heaviest first, the producer decodes each unit once and hands the
//     other roles a descriptor, and the masks and stores follow each
//     sequence's own lengths (bottom-right causal inside the sequence).
#include <cuda_runtime.h>
#include <math.h>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {

namespace {

constexpr int kThreads = 384;  // three warpgroups
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// Register split (per thread). The block is launched with kLaunchRegs per
// thread (65536 / 384 rounded down to a multiple of 8); setmaxnreg can only
// move registers WITHIN that launch allocation, so the three warpgroups'
// shares must sum to at most 3 * kLaunchRegs, or setmaxnreg.inc waits
// forever. The producer/MMA warpgroup gives registers back so each softmax
// thread can keep a full 128-column row of S in registers.
constexpr int kLaunchRegs = 168;
constexpr int kRegsLow = 104;
constexpr int kRegsHigh = 200;
static_assert(kRegsLow + 2 * kRegsHigh <= 3 * kLaunchRegs,
              "register split exceeds the launch allocation: setmaxnreg.inc would never return");
static_assert(kRegsLow % 8 == 0 && kRegsHigh % 8 == 0 && kRegsLow >= 24 && kRegsHigh <= 256,
              "setmaxnreg counts must be multiples of 8 in [24, 256]");
constexpr int kTmemCols = 512;
// A ragged-batch unit as the producer decodes it for the other roles:
// b, h_kv, then (h_q, q_tile, key blocks) of tile 0 and of tile 1, then the
// sequence's first query token, query length, first key token, key length.
constexpr int kDescInts = 16;
enum { kDB = 0, kDHkv, kDT0, kDT1 = kDT0 + 3, kDQ0 = kDT1 + 3, kDLenQ, kDK0, kDLenK };
template <int D>
struct TcLayout {
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row bf16 tile
  static constexpr int kPanelBytes = 128 * 128;   // 128 rows x 64 columns
  // At D = 256 a tile's S and O fill the 512 tensor-memory columns, so a
  // unit is one query tile, and one Q tile and two K/V tiles fill the
  // shared memory.
  static constexpr int kQTiles = D == 256 ? 1 : 2;
  static constexpr int kStages = D == 256 ? 2 : (D == 128 ? 5 : 8);  // K or V tiles in the ring
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kQTiles * kTileBytes;
  static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
  // barrier indices
  // P arrives in two halves: kPFull for keys 0-63 of a block, kPFullB for 64-127
  // (at D = 64 only kPFullB is used, for the whole block)
  static constexpr int kQFull = 0, kQEmpty = 2, kSFull = 4, kPFull = 6, kOFull = 8,
                       kOEmpty = 10, kSchedFull = 12, kSchedEmpty = 14, kDrain = 16,
                       kPFullB = 17, kKVFull = 19, kKVEmpty = 19 + kStages;
  // clusters: the leader hands each unit index it draws to the other CTAs
  // (kXFull, in those CTAs) and learns when they have read it (kXEmpty, in
  // the leader)
  static constexpr int kXFull = 19 + 2 * kStages, kXEmpty = kXFull + 2;
  // d = 64 (P in columns of its own): S_t consumed by the softmax (the next
  // S may overwrite it) and P_t consumed by the P V of the block (the next
  // P may overwrite it)
  static constexpr int kSEmpty = kXEmpty + 2, kPEmpty = kSEmpty + 2;
  static constexpr int kNumBars = kPEmpty + 2;
  static constexpr int kOffSched = kOffBar + kNumBars * 8;
  static constexpr int kOffX = kOffSched + 8;  // two slots of the leader's hand-out
  static constexpr int kOffTmem = kOffX + 8;
  static constexpr int kOffAbort = kOffTmem + 4;
  // ragged batches: the decoded unit of each schedule slot (kDescInts ints)
  static constexpr int kOffDesc = (kOffAbort + 4 + 15) / 16 * 16;
  static constexpr int kBytes = kOffDesc + 2 * kDescInts * 4;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

// Extreme of a 128-column score row in eight independent chains of
// three-input max: the maximum, or with kMin the minimum (as minus the
// maximum of the negated values; the negation folds into the instruction).
template <bool kMin>
__device__ __forceinline__ float row_extreme(const float (&s)[128]) {
  auto v = [&](int c) { return kMin ? -s[c] : s[c]; };
  float mx[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    mx[k] = fmax3(v(16 * k), v(16 * k + 1), v(16 * k + 2));
#pragma unroll
    for (int c = 3; c < 15; c += 2) mx[k] = fmax3(mx[k], v(16 * k + c), v(16 * k + c + 1));
    mx[k] = fmaxf(mx[k], v(16 * k + 15));
  }
  const float r = fmaxf(fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), mx[6]), mx[7]);
  return kMin ? -r : r;
}

struct TcParams {
  __nv_bfloat16 *o;
  float *lse;     // per row natural-log sum of exp(scale q.k), or null: [B][H_q][N_q]
                  // (dense) or [H_q][total_q] (ragged batch)
  int o_align32;  // every row of O starts on a 32-byte boundary (base and strides)
  OutView ov;     // O's strides (elements) and the columns stored (the head dim)
  int tma4;       // dense q/k/v maps are 4-D (column, row, head, batch); else 3-D
                  // (column, row, batch * heads + head) for plane-uniform strides
  PrefillPlan plan;
  VarlenArgs va;  // ragged batches only
  float scale_log2;
  int *ctl;
};

// The kernel body. kLse: also write each row's log-sum-exp (a separate
// instantiation, so the plain kernel carries none of its code). kVarlen: a
// ragged batch packed token-major ([total][H][d]), its units taken from the
// plan kernel's list; it is launched as its own kernel, prefill_varlen_kernel.
template <int D, bool kLse, bool kVarlen, int kC>
__device__ __forceinline__ void prefill_body(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                             const CUtensorMap &tm_v, const TcParams &prm) {
  using L = TcLayout<D>;
  // At D = 128 the P of a block is handed over in two halves, so the PV over
  // the first 64 keys overlaps the exponentials of the other 64; at D = 64
  // the PV is short and the extra hand-over costs more than it hides.
  constexpr bool kSplitP = D == 128;
  // At d = 64 the tensor memory holds, per tile, S (128 columns), O (64) and
  // P (64, bf16 pairs) side by side: the next block's S is computed while
  // the softmax still works on this block's, instead of after its P V (at
  // d = 128 P overwrites half of S: 2 x (128 + 128) columns fill the 512).
  constexpr bool kSepP = D == 64;
  constexpr uint32_t kPCol = 384;  // P_t at columns [384 + 64 t, 448 + 64 t) when kSepP
  // P's exponentials are fp32 (ex2) at every head dim. (Two per
  // special-function instruction on bf16 pairs, with the exponent input
  // rounded to bf16, measured no faster at D = 128 -- the special-function
  // pipe takes twice as long per pair instruction -- and less accurate.)
  // The running (reference) maximum is only raised, and O rescaled, when a
  // row's maximum grows past it by more than this many log2 units; until
  // then exponents up to this bound are allowed (weights up to 2^8, exact
  // enough in fp32 and in P's bf16). On iid N(0,1) inputs the bound is
  // crossed in about 0.1 % of (warp, key block) steps after the first block.
  constexpr float kRescaleThreshold = 8.0f;
  constexpr float kRescaleBound = 256.0f;  // 2^threshold
  extern __shared__ uint8_t smem_raw[];
  // offset (not integer) arithmetic on smem_raw keeps the pointer in the
  // shared window, so accesses through it compile to shared-memory loads
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t s_base = smem_addr(smem);
  const uint32_t bars = s_base + L::kOffBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  volatile int *sched = reinterpret_cast<volatile int *>(smem + L::kOffSched);
  volatile int *sdesc = reinterpret_cast<volatile int *>(smem + L::kOffDesc);
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
      mbar_init(bar(L::kPFullB + t), 128);
      mbar_init(bar(L::kOFull + t), 1);
      mbar_init(bar(L::kOEmpty + t), 128);
      mbar_init(bar(L::kSchedFull + t), 1);
      mbar_init(bar(L::kSchedEmpty + t), 9);  // MMA lane + 8 softmax warps
      mbar_init(bar(L::kSEmpty + t), 128);
      mbar_init(bar(L::kPEmpty + t), 1);
    }
    mbar_init(bar(L::kDrain), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kKVFull + s), 1);
      mbar_init(bar(L::kKVEmpty + s), kC);  // every CTA of the cluster releases it
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kXFull + s), 1);
      mbar_init(bar(L::kXEmpty + s), kC > 1 ? kC - 1 : 1);
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
  // the other CTAs' barriers are initialised before anything reaches them
  if constexpr (kC > 1) cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // cluster: this CTA's rank, and unit u of the cluster's unit cu
  constexpr int csize = kC;
  const uint32_t crank = csize > 1 ? cluster_ctarank() : 0u;
  const uint16_t cmask = static_cast<uint16_t>((1u << csize) - 1u);
  const int groups_all = plan.B * plan.H_kv;
  auto unit_of = [&](int cu) {
    const int m = cu / groups_all;
    return (csize * m + static_cast<int>(crank)) * groups_all + (cu - m * groups_all);
  };
  if constexpr (!kVarlen) {
    // While the previous grid finishes, warm L2 with the first tiles of
    // unit blockIdx.x: the counter hands out the first units about one per
    // CTA, so together the CTAs cover the first wave's Q tiles and first K/V
    // blocks, whichever CTA takes each unit.
    if (warp == kProducerWarp && lane == 0 &&
        static_cast<int>(blockIdx.x) / csize < plan.total_units / csize) {
      const Unit w = decode_unit(plan, unit_of(static_cast<int>(blockIdx.x) / csize));
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (w.t[t].kv_blocks > 0)
          for (int p = 0; p < D / 64; ++p)
            if (prm.tma4)
              tma_prefetch_l2_4d(&tm_q, p * 64, w.t[t].q_tile * kTileM, w.t[t].h_q, w.b);
            else
              tma_prefetch_l2_3d(&tm_q, p * 64, w.t[t].q_tile * kTileM, w.b * plan.H_q + w.t[t].h_q);
      const int nb = min(2, max(w.t[0].kv_blocks, w.t[1].kv_blocks));
      for (int j = 0; j < nb; ++j)
        for (int p = 0; p < D / 64; ++p) {
          if (prm.tma4) {
            tma_prefetch_l2_4d(&tm_k, p * 64, j * kTileN, w.h_kv, w.b);
            tma_prefetch_l2_4d(&tm_v, p * 64, j * kTileN, w.h_kv, w.b);
          } else {
            tma_prefetch_l2_3d(&tm_k, p * 64, j * kTileN, w.b * plan.H_kv + w.h_kv);
            tma_prefetch_l2_3d(&tm_v, p * 64, j * kTileN, w.b * plan.H_kv + w.h_kv);
          }
        }
    }
  }
  // Everything above only set up this CTA. Global reads (inputs, the work
  // counter) come after the previous grid of the stream has completed.
  grid_dependency_wait();
  grid_launch_dependents();

  auto fail = [&]() {
    *abort_flag = 1;
    record_error(err_word, kErrTimeout);
  };

  if (warp >= 8) {
  regs_dealloc<kRegsLow>();
  // Both roles below run warp-uniform control flow on all 32 lanes (so the
  // descriptor and index arithmetic lives in the uniform datapath); only the
  // TMA / tcgen05 instructions themselves are issued by one elected lane.
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    int it = 0, kv_it = 0, vc0 = 0, vc1 = 0;
    bool ok = true;
    // units to take: the dense plan's count, or the plan kernel's list length
    // (written before this grid's dependency wait returned)
    int total_units = plan.total_units;
    if constexpr (kVarlen) total_units = __ldcg(prm.ctl + kCtlVarlenUnits);
    // A CTA's first unit is unit blockIdx.x, taken without an atomic (the
    // heaviest units go to the first CTAs); the counter hands out units
    // grid, grid + 1, ... after that. Every CTA's last fetch fails, so the
    // fetches number max(total, grid) + (successful ones) and the one that
    // draws max(total, grid) - 1 is the grid's last: it re-arms the counter
    // for the next launch (which reads it only after this grid completes).
    // Clusters (dense batches only): the same with cluster units (the g / 2
    // units of one (b, h_kv, q_tile)) and clusters in place of units and
    // CTAs; the leader draws, hands the index to the other CTAs, and each
    // CTA takes its own unit of the cluster unit.
    const int grid = static_cast<int>(gridDim.x) / csize;
    const int my = static_cast<int>(blockIdx.x) / csize;
    const int total_cu = total_units / csize;
    bool first = true;
    int xit = 0;
    while (ok) {
      int u = 0;
      if (first && my < total_cu) {
        u = my;
      } else if (crank == 0) {
        int c = 0;
        if (lane == 0) {
          c = atomicAdd(prm.ctl + kCtlWork, 1);
          if (c == max(total_cu, grid) - 1) st_relaxed_gpu(prm.ctl + kCtlWork, 0);
        }
        u = grid + __shfl_sync(0xffffffffu, c, 0);
        if (csize > 1) {
          const int xs = xit & 1;
          // the other CTAs have read this slot's previous index
          if (xit >= 2 && !mbar_wait_warp(bar(L::kXEmpty + xs), ((xit >> 1) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          if (lane > 0 && lane < csize) {
            const uint32_t r = static_cast<uint32_t>(lane);
            st_shared_remote(map_shared_rank(s_base + L::kOffX + 4 * xs, r), u);
            mbar_arrive_remote(map_shared_rank(bar(L::kXFull + xs), r));
          }
          __syncwarp();
          ++xit;
        }
      } else {
        const int xs = xit & 1;
        bool got = mbar_try_wait_cluster(bar(L::kXFull + xs), (xit >> 1) & 1);
        const uint64_t t0 = global_timer_ns();
        while (!got && !*abort_flag && global_timer_ns() - t0 < kWaitLimitNs)
          got = mbar_try_wait_cluster(bar(L::kXFull + xs), (xit >> 1) & 1);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        u = *reinterpret_cast<volatile int *>(smem + L::kOffX + 4 * xs);
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(map_shared_rank(bar(L::kXEmpty + xs), 0));
        ++xit;
      }
      first = false;
      // this CTA's unit of the cluster unit (the unit itself without clusters)
      if (u < total_cu) u = unit_of(u);
      else u = total_units;
      const int slot = it & 1;
      Unit w;
      int q0 = 0, len_q = 0, k0 = 0, len_k = 0;
      if (u < total_units) {
        if constexpr (kVarlen) {
          // the listed unit: sequence b, K/V head, pair of query tiles (one
          // tile at head dim 256)
          const int4 un = __ldcg(prm.va.units + u);
          const int g = prm.va.group;
          w.b = un.x;
          w.h_kv = un.y;
          q0 = varlen_start(prm.va.cu_q, prm.va.uni_q, w.b);
          len_q = varlen_start(prm.va.cu_q, prm.va.uni_q, w.b + 1) - q0;
          k0 = varlen_start(prm.va.cu_k, prm.va.uni_k, w.b);
          len_k = varlen_start(prm.va.cu_k, prm.va.uni_k, w.b + 1) - k0;
          const int n_qt = (len_q + kTileM - 1) / kTileM;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int f = L::kQTiles * un.z + t;
            if (t < L::kQTiles && f < g * n_qt) {
              w.t[t].q_tile = n_qt - 1 - f / g;
              w.t[t].h_q = w.h_kv * g + f % g;
              w.t[t].kv_blocks = varlen_kv_blocks(len_q, len_k, prm.va.causal, w.t[t].q_tile);
            } else {
              w.t[t].q_tile = w.t[t].h_q = -1;
              w.t[t].kv_blocks = 0;
            }
          }
        } else {
          w = decode_unit(plan, u);
        }
      }
      if (!mbar_wait_warp(bar(L::kSchedEmpty + slot), ((it >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
      __syncwarp();
      if (lane == 0) {
        sched[slot] = u < total_units ? u : -1;  // -1: no more work
        if constexpr (kVarlen) {
          volatile int *dsc = sdesc + kDescInts * slot;
          dsc[kDB] = w.b;
          dsc[kDHkv] = w.h_kv;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            dsc[kDT0 + 3 * t] = w.t[t].h_q;
            dsc[kDT0 + 3 * t + 1] = w.t[t].q_tile;
            dsc[kDT0 + 3 * t + 2] = w.t[t].kv_blocks;
          }
          dsc[kDQ0] = q0;
          dsc[kDLenQ] = len_q;
          dsc[kDK0] = k0;
          dsc[kDLenK] = len_k;
        }
        mbar_arrive(bar(L::kSchedFull + slot));
      }
      ++it;
      if (u >= total_units) break;
      const int nb = max(w.t[0].kv_blocks, w.t[1].kv_blocks);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const UnitTile tt = t ? w.t[1] : w.t[0];
        int &vc = t ? vc1 : vc0;
        if (!ok || tt.kv_blocks == 0) continue;
        if (!mbar_wait_warp(bar(L::kQEmpty + t), (vc & 1) ^ 1, abort_flag)) { ok = false; continue; }
        ++vc;
        __syncwarp();
        if (elect_one()) {
          const uint32_t dst = s_base + L::kOffQ + t * L::kTileBytes;
          mbar_arrive_expect_tx(bar(L::kQFull + t), L::kTileBytes);
#pragma unroll
          for (int p = 0; p < D / 64; ++p) {
            if constexpr (kVarlen)  // [total_q][H_q][d]: (column, head, token)
              tma_load_3d(dst + p * L::kPanelBytes, &tm_q, bar(L::kQFull + t), p * 64, tt.h_q,
                          q0 + tt.q_tile * kTileM);
            else if (prm.tma4)  // [B][H_q][N_q][d] with the caller's strides: (column, row, head, batch)
              tma_load_4d(dst + p * L::kPanelBytes, &tm_q, bar(L::kQFull + t), p * 64,
                          tt.q_tile * kTileM, tt.h_q, w.b);
            else  // (column, row, batch * H_q + head)
              tma_load_3d(dst + p * L::kPanelBytes, &tm_q, bar(L::kQFull + t), p * 64,
                          tt.q_tile * kTileM, w.b * plan.H_q + tt.h_q);
          }
        }
        __syncwarp();
      }
      for (int j = 0; j < nb && ok; ++j) {
#pragma unroll
        for (int kind = 0; kind < 2; ++kind) {  // K_j then V_j
          if (!ok) continue;
          const int st = kv_it % L::kStages;
          const uint32_t ph = (kv_it / L::kStages) & 1;
          if (!mbar_wait_warp(bar(L::kKVEmpty + st), ph ^ 1, abort_flag)) { ok = false; continue; }
          __syncwarp();
          if (elect_one()) {
            const uint32_t dst = s_base + L::kOffKV + st * L::kTileBytes;
            mbar_arrive_expect_tx(bar(L::kKVFull + st), L::kTileBytes);
#pragma unroll
            for (int p = 0; p < D / 64; ++p) {
              if constexpr (kVarlen) {  // [total_k][H_kv][d]: (column, head, token)
                tma_load_3d(dst + p * L::kPanelBytes, kind ? &tm_v : &tm_k, bar(L::kKVFull + st),
                            p * 64, w.h_kv, k0 + j * kTileN);
              } else if (csize > 1) {
                // the cluster's CTAs share the block's 64-column panels out
                // and multicast each to all of them (their stage st, their
                // barrier, whose expected bytes count the whole block)
                if (p % csize != static_cast<int>(crank)) continue;
                if (prm.tma4)
                  tma_load_4d_mc(dst + p * L::kPanelBytes, kind ? &tm_v : &tm_k, bar(L::kKVFull + st),
                                 p * 64, j * kTileN, w.h_kv, w.b, cmask);
                else
                  tma_load_3d_mc(dst + p * L::kPanelBytes, kind ? &tm_v : &tm_k, bar(L::kKVFull + st),
                                 p * 64, j * kTileN, w.b * plan.H_kv + w.h_kv, cmask);
              } else if (prm.tma4) {
                tma_load_4d(dst + p * L::kPanelBytes, kind ? &tm_v : &tm_k, bar(L::kKVFull + st),
                            p * 64, j * kTileN, w.h_kv, w.b);
              } else {
                tma_load_3d(dst + p * L::kPanelBytes, kind ? &tm_v : &tm_k, bar(L::kKVFull + st),
                            p * 64, j * kTileN, w.b * plan.H_kv + w.h_kv);
              }
            }
          }
          __syncwarp();
          ++kv_it;
        }
      }
    }
    if (!ok && lane == 0) fail();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
    // Descriptor words: the high word (stride 1024 B, version, 128-byte
    // swizzle) is shared by every operand; low words are base + constant.
    constexpr uint32_t kDescHi = sdesc_hi_sw128(1024);
    const uint32_t q_lo0 = sdesc_lo(s_base + L::kOffQ, 16);
    const uint32_t kv_lo0 = sdesc_lo(s_base + L::kOffKV, 16);
    const uint32_t v_lo0 = sdesc_lo(s_base + L::kOffKV, L::kPanelBytes);
    int it = 0, kv_it = 0, vc0 = 0, vc1 = 0;
    uint32_t pc0 = 0, pc1 = 0;
    uint32_t sc0 = 0, sc1 = 0;  // S issued per tile (d = 64: their reads by the softmax gate the next)
    bool ok = true;

    auto issue_qk = [&](int t, int st) {
      const uint32_t a_lo = q_lo0 + static_cast<uint32_t>(t * L::kTileBytes >> 4);
      const uint32_t b_lo = kv_lo0 + static_cast<uint32_t>(st * L::kTileBytes >> 4);
      const uint32_t d = tmem + 128u * t;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K-step kk: panel kk/4 (64 columns each), 32 bytes per step inside it
          const uint32_t off = static_cast<uint32_t>(((kk >> 2) * L::kPanelBytes + (kk & 3) * 32) >> 4);
          mma_ss_w(d, a_lo + off, kDescHi, b_lo + off, kDescHi, idesc_qk, kk > 0 ? 1u : 0u);
        }
      }
      __syncwarp();
    };
    // O_t += P_t V over keys [64 half, 64 half + 64) of the block
    auto issue_pv = [&](int t, int st, bool accumulate, int half) {
      const uint32_t b_lo = v_lo0 + static_cast<uint32_t>(st * L::kTileBytes >> 4);
      const uint32_t d = tmem + 256u + D * t;
      const uint32_t a = kSepP ? tmem + kPCol + 64u * t : tmem + 128u * t + 64u;
      if (elect_one()) {
#pragma unroll
        for (int k4 = 0; k4 < kTileN / 32; ++k4) {  // 16 key rows (2048 B) per K-step
          const int kk = half * (kTileN / 32) + k4;
          mma_ts_w(d, a + kk * 8, b_lo + kk * 128, kDescHi, idesc_pv,
                   (accumulate || kk > 0) ? 1u : 0u);
        }
      }
      __syncwarp();
    };
    auto commit = [&](int b) {
      if (elect_one()) tc_commit(bar(b));
      __syncwarp();
    };
    // a K/V stage is free once every CTA of the cluster has read it
    auto release_kv = [&](int st) {
      if (elect_one()) {
        if (csize > 1)
          tc_commit_mc(bar(L::kKVEmpty + st), cmask);
        else
          tc_commit(bar(L::kKVEmpty + st));
      }
      __syncwarp();
    };
    auto wait_kv = [&](int &st) -> bool {
      st = kv_it % L::kStages;
      const uint32_t ph = (kv_it / L::kStages) & 1;
      ++kv_it;
      return mbar_wait_warp(bar(L::kKVFull + st), ph, abort_flag);
    };
    // PV for tile t over block jb (all checks on the caller's side): the
    // first half of the keys as soon as their P is in tensor memory, the
    // second half while nothing else waits.
    auto do_pv = [&](int t, int jb, int st) -> bool {
      const int vc = t ? vc1 : vc0;
      uint32_t &pc = t ? pc1 : pc0;
      if (jb == 0 && !mbar_wait_warp(bar(L::kOEmpty + t), (vc & 1) ^ 1, abort_flag)) return false;
      if (kSplitP) {
        if (!mbar_wait_warp(bar(L::kPFull + t), pc & 1, abort_flag)) return false;
        tc_fence_after_sync();
        issue_pv(t, st, jb > 0, 0);
      }
      if (!mbar_wait_warp(bar(L::kPFullB + t), pc & 1, abort_flag)) return false;
      ++pc;
      tc_fence_after_sync();
      if (!kSplitP) issue_pv(t, st, jb > 0, 0);
      issue_pv(t, st, true, 1);
      return true;
    };

    while (ok) {
      const int slot = it & 1;
      if (!mbar_wait_warp(bar(L::kSchedFull + slot), (it >> 1) & 1, abort_flag)) { ok = false; break; }
      const int u = sched[slot];
      int nbt0 = 0, nbt1 = 0;
      if constexpr (kVarlen) {  // read before the slot is released
        nbt0 = sdesc[kDescInts * slot + kDT0 + 2];
        nbt1 = sdesc[kDescInts * slot + kDT1 + 2];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kSchedEmpty + slot));
      ++it;
      if (u < 0) break;
      if constexpr (!kVarlen) {
        const Unit w = decode_unit(plan, u);
        nbt0 = w.t[0].kv_blocks;
        nbt1 = w.t[1].kv_blocks;
      }
      const int nb = max(nbt0, nbt1);
      if (nbt0 > 0 && !mbar_wait_warp(bar(L::kQFull + 0), vc0 & 1, abort_flag)) ok = false;
      if (ok && nbt1 > 0 && !mbar_wait_warp(bar(L::kQFull + 1), vc1 & 1, abort_flag)) ok = false;
      if (!ok) break;
      int st_k, st_v;
      if constexpr (kSepP) {
        // S_t[j] as soon as the softmax has read S_t[j-1] (and K_j is in),
        // P V of block j-1 once P_t[j-1] is complete; per block the two
        // tiles' S go first, as the softmax reads S long before its P.
        auto s_free = [&](int t) -> bool {  // the softmax has read this tile's previous S
          uint32_t &sc = t ? sc1 : sc0;
          const bool r = sc == 0 || mbar_wait_warp(bar(L::kSEmpty + t), (sc - 1) & 1, abort_flag);
          ++sc;
          return r;
        };
        if (!wait_kv(st_k)) { ok = false; break; }
        __syncwarp();
        tc_fence_after_sync();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nbt = t ? nbt1 : nbt0;
          if (!ok || nbt == 0) continue;
          if (!s_free(t)) { ok = false; continue; }
          tc_fence_after_sync();
          issue_qk(t, st_k);
          commit(L::kSFull + t);
          if (nbt == 1) commit(L::kQEmpty + t);
        }
        for (int j = 1; j < nb && ok; ++j) {
          release_kv(st_k);  // K_{j-1} no longer read after this point
          if (!wait_kv(st_v) || !wait_kv(st_k)) { ok = false; break; }
          __syncwarp();
          tc_fence_after_sync();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int nbt = t ? nbt1 : nbt0;
            if (!ok || j >= nbt) continue;
            if (!s_free(t)) { ok = false; continue; }
            tc_fence_after_sync();
            issue_qk(t, st_k);
            commit(L::kSFull + t);
            if (j == nbt - 1) commit(L::kQEmpty + t);
          }
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int nbt = t ? nbt1 : nbt0;
            if (!ok || j - 1 >= nbt) continue;
            if (!do_pv(t, j - 1, st_v)) { ok = false; continue; }
            commit(j - 1 == nbt - 1 ? L::kOFull + t : L::kPEmpty + t);
          }
          release_kv(st_v);
        }
        if (!ok) break;
        release_kv(st_k);
        if (!wait_kv(st_v)) { ok = false; break; }
        __syncwarp();
        tc_fence_after_sync();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nbt = t ? nbt1 : nbt0;
          if (!ok || nbt != nb) continue;
          if (!do_pv(t, nb - 1, st_v)) { ok = false; continue; }
          commit(L::kOFull + t);
        }
        release_kv(st_v);
      } else {
        // block 0: S_t = Q_t K_0^T
        if (!wait_kv(st_k)) { ok = false; break; }
        __syncwarp();
        tc_fence_after_sync();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nbt = t ? nbt1 : nbt0;
          if (nbt == 0) continue;
          issue_qk(t, st_k);
          commit(L::kSFull + t);
          if (nbt == 1) commit(L::kQEmpty + t);
        }
        // blocks 1..nb-1: O_t += P_t V_{j-1}, then S_t = Q_t K_j^T
        for (int j = 1; j < nb && ok; ++j) {
          release_kv(st_k);  // K_{j-1} no longer read after this point
          if (!wait_kv(st_v) || !wait_kv(st_k)) { ok = false; break; }
          __syncwarp();
          tc_fence_after_sync();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int nbt = t ? nbt1 : nbt0;
            if (!ok) continue;
            if (j - 1 < nbt) {
              if (!do_pv(t, j - 1, st_v)) { ok = false; continue; }
              if (j - 1 == nbt - 1) commit(L::kOFull + t);
            }
            if (j < nbt) {
              issue_qk(t, st_k);
              commit(L::kSFull + t);
              if (j == nbt - 1) commit(L::kQEmpty + t);
            }
          }
          release_kv(st_v);
        }
        if (!ok) break;
        // last block: O_t += P_t V_{nb-1}
        release_kv(st_k);
        if (!wait_kv(st_v)) { ok = false; break; }
        __syncwarp();
        tc_fence_after_sync();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nbt = t ? nbt1 : nbt0;
          if (!ok || nbt != nb) continue;
          if (!do_pv(t, nb - 1, st_v)) { ok = false; continue; }
          commit(L::kOFull + t);
        }
        release_kv(st_v);
      }
      if (nbt0 > 0) ++vc0;
      if (nbt1 > 0) ++vc1;
    }
    if (!ok && lane == 0) fail();
    // Drain: every tcgen05 operation issued above has completed.
    commit(L::kDrain);
    mbar_wait_warp(bar(L::kDrain), 0, nullptr);
  }
  } else {
    regs_alloc<kRegsHigh>();
    // ------------------------------------------------------------ softmax / epilogue
    const int t = warp >> 2;                       // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;        // row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tm_s = tmem + lane_off + t * 128u;
    const uint32_t tm_p = kSepP ? tmem + lane_off + kPCol + 64u * t : tm_s + 64u;
    const uint32_t tm_o = tmem + lane_off + 256u + t * D;
    const float sl2 = prm.scale_log2;
    // a masked score: whatever the sign of the scale, it scales to -inf
    // (the host never passes a zero scale_log2)
    const float s_masked = sl2 >= 0.f ? -INFINITY : INFINITY;
    int it = 0, vc = 0;
    uint32_t scnt = 0;
    uint32_t pwc = 0;  // d = 64: P V completions waited for (one per block after a unit's first)
    bool ok = true;
    while (ok) {
      const int slot = it & 1;
      if (!mbar_wait_warp(bar(L::kSchedFull + slot), (it >> 1) & 1, abort_flag)) { ok = false; break; }
      const int u = sched[slot];
      // this warpgroup's tile: (b, h_q, q_tile, key blocks); the sequence's
      // query and key lengths and (ragged batches) first query token
      int b = 0, h_q = 0, q_tile = 0, nbt = 0, q0 = 0, len_q = plan.N_q, len_k = plan.N_kv;
      if constexpr (kVarlen) {  // read before the slot is released
        const volatile int *dsc = sdesc + kDescInts * slot;
        b = dsc[kDB];
        h_q = dsc[kDT0 + 3 * t];
        q_tile = dsc[kDT0 + 3 * t + 1];
        nbt = dsc[kDT0 + 3 * t + 2];
        q0 = dsc[kDQ0];
        len_q = dsc[kDLenQ];
        len_k = dsc[kDLenK];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kSchedEmpty + slot));
      ++it;
      if (u < 0) break;
      if constexpr (!kVarlen) {
        const Unit w = decode_unit(plan, u);
        const UnitTile mine = t ? w.t[1] : w.t[0];  // select, not a runtime index
        b = w.b;
        h_q = mine.h_q;
        q_tile = mine.q_tile;
        nbt = mine.kv_blocks;
      }
      if (nbt == 0) continue;
      const int q_row = q_tile * kTileM + row;
      // last visible key of this row (inclusive; bottom-right causal)
      int lim = len_k - 1;
      if (plan.causal) lim = min(lim, q_row + len_k - len_q);
      float m_ref = -INFINITY;  // reference maximum, log2-scaled units
      float l_sum = 0.f;
      for (int j = 0; j < nbt; ++j) {
        if (!mbar_wait_warp(bar(L::kSFull + t), scnt & 1, abort_flag)) { ok = false; break; }
        ++scnt;
        __syncwarp();  // tcgen05.ld/st below are warp-collective
        tc_fence_after_sync();
        uint32_t sr[128];
        tmem_ld128_wait(tm_s, sr);
        if constexpr (kSepP) {
          // S_t is in registers: the next block's S may overwrite it
          tc_fence_before_sync();
          mbar_arrive(bar(L::kSEmpty + t));
        }
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        const int kbase = j * kTileN;
        if (__any_sync(0xffffffffu, kbase + kTileN - 1 > lim)) {
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (kbase + c > lim) ? s_masked : s[c];
        }
        // P = 2^(S * scale*log2e - m) for the 64 columns of half h, with
        // packed fp32 ops, stored to tensor memory as bf16 pairs; returns the
        // half's row sum. (P of half 0 overwrites S columns 64-95, which are
        // already in registers.)
        auto make_half = [&](int h, float m) -> float {
          const float2 sl2v = make_float2(sl2, sl2);
          const float2 negm = make_float2(-m, -m);
          // The row sum adds the very bf16 weights P.V uses (so O is an
          // exact weighted average of V whatever their rounding), widened
          // inside mixed-precision adds; eight partial sums keep the
          // dependency chains short.
          float lsum[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) lsum[i] = 0.f;
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x = ffma2(make_float2(s[h * 64 + 2 * c], s[h * 64 + 2 * c + 1]), sl2v, negm);
            pk[c] = pack_bf16x2(ex2(x.x), ex2(x.y));
            add_bf16x2_to(lsum[2 * (c & 3)], lsum[2 * (c & 3) + 1], pk[c]);
          }
          tmem_st32(tm_p + h * 32u, pk);
          return ((lsum[0] + lsum[1]) + (lsum[2] + lsum[3])) + ((lsum[4] + lsum[5]) + (lsum[6] + lsum[7]));
        };
        // row maximum of s * scale * log2e: the maximum of s for a
        // non-negative scale, its minimum for a negative one
        auto row_max = [&]() -> float {
          return (sl2 >= 0.f ? row_extreme<false>(s) : row_extreme<true>(s)) * sl2;
        };
        // halves computed before the row maximum is known: the first one
        // when P is handed over in halves, else both
        constexpr int kEarly = kSplitP ? 1 : 2;
        if constexpr (kSepP) {
          // P_t[j-1] has been read by its P V before this block's P
          // overwrites it (and O, last written by that P V, may be rescaled
          // below)
          if (j > 0) {
            if (!mbar_wait_warp(bar(L::kPEmpty + t), pwc & 1, abort_flag)) { ok = false; break; }
            ++pwc;
            tc_fence_after_sync();
          }
        }
        float alpha = 1.f, sum = 0.f;
        if (j == 0) {
          m_ref = row_max();  // first block: its O is overwritten, nothing to rescale
          alpha = 0.f;
#pragma unroll
          for (int h = 0; h < kEarly; ++h) sum += make_half(h, m_ref);
        } else {
          // Speculate that the reference maximum still holds (it only moves
          // when the row maximum grows by more than the threshold): the exponentials
          // do not wait for the block maximum.
#pragma unroll
          for (int h = 0; h < kEarly; ++h) sum += make_half(h, m_ref);
          // When the whole block's weights are in `sum` (P handed over in one
          // piece), each weight is at most their sum: if no row's sum
          // exceeds 2^threshold, no row's block maximum exceeds the
          // reference by more than the threshold, and the maximum need not
          // be computed (measured 160.5 -> 152.5 us on the d = 64 long
          // sequence, 13.0 -> 12.5 us on the sweep). Otherwise, and when P
          // goes in halves, the maximum decides.
          const bool maybe = kSplitP || __any_sync(0xffffffffu, sum > kRescaleBound);
          const float m_blk = maybe ? row_max() : m_ref;
          const bool raise = m_blk > m_ref + kRescaleThreshold;
          if (__any_sync(0xffffffffu, raise)) {
            // rare: some row's maximum jumped; redo this warp's early halves
            // with the raised maxima (rows that did not jump keep theirs,
            // alpha = 1) and rescale O before any of this block's PV. O_t
            // was last written by the PV of block j-1, which completed
            // before S_t[j] was committed (d = 64: before kPEmpty, waited
            // for above).
            if (raise) {
              alpha = ex2(m_ref - m_blk);
              m_ref = m_blk;
            }
            tmem_st_wait();
            sum = 0.f;
#pragma unroll
            for (int h = 0; h < kEarly; ++h) sum += make_half(h, m_ref);
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t ov[32];
              tmem_ld32_wait(tm_o + c0, ov);
#pragma unroll
              for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
              tmem_st32(tm_o + c0, ov);
            }
          }
        }
        if (kSplitP) {
          tmem_st_wait();
          tc_fence_before_sync();
          mbar_arrive(bar(L::kPFull + t));  // PV over keys 0-63 may start
          sum += make_half(1, m_ref);
        }
        tmem_st_wait();
        l_sum = l_sum * alpha + sum;
        tc_fence_before_sync();
        mbar_arrive(bar(L::kPFullB + t));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16 -> global
      if (!mbar_wait_warp(bar(L::kOFull + t), vc & 1, abort_flag)) { ok = false; break; }
      ++vc;
      __syncwarp();
      tc_fence_after_sync();
      const float inv_l = 1.f / l_sum;
      // O row: [B][H_q][N_q][D] dense, [total_q][H_q][D] ragged (rows past
      // the sequence belong to the next one and are not stored)
      // (o_sn is the token stride for ragged batches, the row stride otherwise)
      long long o_at;
      size_t lse_at;
      if constexpr (kVarlen) {
        o_at = static_cast<long long>(q0 + q_row) * prm.ov.sn + static_cast<long long>(h_q) * prm.ov.sh;
        lse_at = static_cast<size_t>(h_q) * prm.va.total_q + q0 + q_row;
      } else {
        o_at = static_cast<long long>(b) * prm.ov.sb + static_cast<long long>(h_q) * prm.ov.sh +
               static_cast<long long>(q_row) * prm.ov.sn;
        lse_at = (static_cast<size_t>(b) * plan.H_q + h_q) * plan.N_q + q_row;
      }
      __nv_bfloat16 *dst = prm.o + o_at;
      const bool store = q_row < len_q;
      // log-sum-exp of the row in natural-log units: l is relative to
      // 2^m_ref with m_ref in log2 units of scale * q.k
      if (kLse && store) prm.lse[lse_at] = (m_ref + log2f(l_sum)) * 0.6931471805599453f;
      // The row of O in tensor-memory loads of up to 128 columns; O_t is
      // free for the next unit's PV once the last has completed
      constexpr int kChunk = D > 128 ? 128 : D;
#pragma unroll 1
      for (int cb = 0; cb < D; cb += kChunk) {
        uint32_t ov[kChunk];
        __syncwarp();
        if constexpr (kChunk == 128)
          tmem_ld128_wait(tm_o + cb, ov);
        else
          tmem_ld64_wait(tm_o + cb, ov);
        if (cb + kChunk == D) {
          tc_fence_before_sync();
          mbar_arrive(bar(L::kOEmpty + t));
        }
#pragma unroll
        for (int c0 = 0; c0 < kChunk; c0 += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = pack_bf16x2(__uint_as_float(ov[c0 + 2 * c]) * inv_l,
                                __uint_as_float(ov[c0 + 2 * c + 1]) * inv_l);
          if (store && cb + c0 < prm.ov.d) {  // columns past the head dim are padding
            // a lane writes its own row: whole 32-byte sectors when O allows
            if (prm.o_align32) {
              st_global_v8(dst + cb + c0, pk);
              st_global_v8(dst + cb + c0 + 16, pk + 8);
            } else {
              uint4 *g = reinterpret_cast<uint4 *>(dst + cb + c0);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                g[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
            }
          }
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
  // no CTA leaves while another of its cluster may still reach its shared
  // memory (multicast loads, barrier arrivals)
  if constexpr (kC > 1) cluster_sync();
}

// [B][H][N][d] batches of equal lengths
// (kC CTAs per cluster: a cluster works on the g / 2 units of one (b, h_kv,
// q_tile), every K/V block multicast to all of them)
template <int D, bool kLse, int kC>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const TcParams prm) {
  prefill_body<D, kLse, false, kC>(tm_q, tm_k, tm_v, prm);
}

// ragged batches packed token-major
template <int D, bool kLse>
__global__ void __launch_bounds__(kThreads, 1) prefill_varlen_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const TcParams prm) {
  prefill_body<D, kLse, true, 1>(tm_q, tm_k, tm_v, prm);
}

template <int D, bool kLse, bool kVarlen, int kC>
constexpr auto prefill_entry() {
  if constexpr (kVarlen)
    return prefill_varlen_kernel<D, kLse>;
  else
    return prefill_tc_kernel<D, kLse, kC>;
}

template <int D, bool kLse, bool kVarlen, int kC>
cudaError_t launch_d(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                     void *o, const OutView &ov, float *lse, const PrefillPlan &plan,
                     const VarlenArgs &va, int grid, float scale, int *ctl, cudaStream_t stream) {
  using L = TcLayout<D>;
  static unsigned configured = 0;  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(configured & (1u << dev))) {
    // The register split is only safe if the compiled kernel is launched
    // with at least kLaunchRegs registers per thread; refuse otherwise.
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, prefill_entry<D, kLse, kVarlen, kC>());
    if (e != cudaSuccess) return e;
    if (attr.numRegs < kLaunchRegs || attr.maxThreadsPerBlock < kThreads)
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(prefill_entry<D, kLse, kVarlen, kC>(),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    if (dev < 32) configured |= 1u << dev;
  }
  TcParams prm;
  prm.o = static_cast<__nv_bfloat16 *>(o);
  prm.lse = lse;
  prm.o_align32 = ((reinterpret_cast<uintptr_t>(o) | static_cast<uintptr_t>(ov.sb * 2) |
                     static_cast<uintptr_t>(ov.sh * 2) | static_cast<uintptr_t>(ov.sn * 2)) & 31u) == 0
                       ? 1
                       : 0;
  prm.ov = ov;
  prm.tma4 = ov.tma4;
  prm.plan = plan;
  prm.va = va;
  // A zero scale (uniform weights over the visible keys) is taken as a
  // tiny one of the same effect: the kernel scales masked scores (+-inf)
  // by it, and inf * 0 would be NaN. Any |s| below 1e8 then gives an
  // exponent within 2^-70 of zero, so every weight is exactly 1 in bf16.
  float sl2 = scale * 1.4426950408889634f;
  if (fabsf(sl2) < 1e-30f) sl2 = sl2 < 0.f ? -1e-30f : 1e-30f;
  prm.scale_log2 = sl2;
  prm.ctl = ctl;
  if constexpr (kC > 1)
    return launch_programmatic_cluster(prefill_entry<D, kLse, kVarlen, kC>(), grid, kThreads,
                                       L::kAlloc, kC, stream, tm_q, tm_k, tm_v, prm);
  return launch_programmatic(prefill_entry<D, kLse, kVarlen, kC>(), grid, kThreads, L::kAlloc,
                             stream, tm_q, tm_k, tm_v, prm);
}

// Head dims 32 and 64 run the D = 64 kernel, 96 and 128 the D = 128 one: the
// TMA boxes are 64 columns wide and read zeros past the head dim, so the
// extra columns of Q and K add nothing to S and those of V leave zero
// columns in O, which the epilogue does not store.
template <bool kVarlen, int kC>
cudaError_t launch_dc(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                      void *o, const OutView &ov, float *lse, const PrefillPlan &plan,
                      const VarlenArgs &va, int grid, float scale, int *ctl, cudaStream_t stream) {
  const bool with_lse = lse != nullptr;
  if (ov.d == 32 || ov.d == 64)
    return with_lse ? launch_d<64, true, kVarlen, kC>(tm_q, tm_k, tm_v, o, ov, lse, plan, va, grid,
                                                      scale, ctl, stream)
                    : launch_d<64, false, kVarlen, kC>(tm_q, tm_k, tm_v, o, ov, lse, plan, va,
                                                       grid, scale, ctl, stream);
  if (ov.d == 96 || ov.d == 128)
    return with_lse ? launch_d<128, true, kVarlen, kC>(tm_q, tm_k, tm_v, o, ov, lse, plan, va,
                                                       grid, scale, ctl, stream)
                    : launch_d<128, false, kVarlen, kC>(tm_q, tm_k, tm_v, o, ov, lse, plan, va,
                                                        grid, scale, ctl, stream);
  if constexpr (kC == 1) {
    if (ov.d == 256)  // one query tile per unit (the plan says so)
      return with_lse ? launch_d<256, true, kVarlen, 1>(tm_q, tm_k, tm_v, o, ov, lse, plan, va,
                                                        grid, scale, ctl, stream)
                      : launch_d<256, false, kVarlen, 1>(tm_q, tm_k, tm_v, o, ov, lse, plan, va,
                                                         grid, scale, ctl, stream);
  }
  return cudaErrorInvalidValue;
}

template <bool kVarlen>
cudaError_t launch_any(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                       void *o, const OutView &ov, float *lse, const PrefillPlan &plan,
                       const VarlenArgs &va, int grid, int csize, float scale, int *ctl,
                       cudaStream_t stream) {
  if constexpr (!kVarlen) {
    if (csize == 2)
      return launch_dc<false, 2>(tm_q, tm_k, tm_v, o, ov, lse, plan, va, grid, scale, ctl, stream);
    if (csize == 4)
      return launch_dc<false, 4>(tm_q, tm_k, tm_v, o, ov, lse, plan, va, grid, scale, ctl, stream);
  }
  return launch_dc<kVarlen, 1>(tm_q, tm_k, tm_v, o, ov, lse, plan, va, grid, scale, ctl, stream);
}

// ------------------------------------------------------------ ragged-batch plan
//
// One block. Per sequence b: check the offsets, then count its units,
// H_kv * ceil(g * n_qt / 2) (n_qt = ceil(len_q / 128)); number the units b by
// b, and (h_kv fastest) the pairs of each sequence heaviest first. Then a
// counting sort on each unit's key blocks (the larger of its two tiles')
// lists them most first, so the atomic counter hands out the heaviest units
// first across all sequences. The order inside one block count is not fixed;
// which CTA computes a unit does not change its result.
constexpr int kPlanThreads = 1024;

// Exclusive prefix of one value per thread over the block (thread order);
// `total` receives the block's sum. Every thread must call it.
__device__ __forceinline__ int block_exclusive_scan(int v, int *s_warp, int &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? s_warp[warp - 1] : 0);
  total = s_warp[kPlanThreads / 32 - 1];
  __syncthreads();  // s_warp may be reused
  return excl;
}

// Dynamic shared memory of the plan kernel for B sequences.
inline size_t plan_smem_bytes(int B) {
  return (3 * static_cast<size_t>(B) + 1 + kVarlenMaxBlocks + 1) * sizeof(int);
}

__global__ void __launch_bounds__(kPlanThreads) varlen_plan_kernel(const VarlenArgs va, int4 *units,
                                                                   int *ctl) {
  extern __shared__ int plan_smem[];
  int *s_pre = plan_smem;            // [B + 1] units of the sequences before b
  int *s_lq = s_pre + va.B + 1;      // [B] query length (0: no units)
  int *s_lk = s_lq + va.B;           // [B] key length
  int *s_bin = s_lk + va.B;          // [kVarlenMaxBlocks + 1] per key-block count
  __shared__ int s_warp[kPlanThreads / 32];
  __shared__ int s_max_nb;
  const int tid = threadIdx.x;
  // the previous grid of the stream may still read the list or write the offsets
  grid_dependency_wait();
  grid_launch_dependents();
  if (tid == 0) s_max_nb = 0;
  __syncthreads();
  // ---- units per sequence (kPer consecutive sequences per thread); a
  // sequence with bad offsets gets none
  const int kPer = (va.B + kPlanThreads - 1) / kPlanThreads;
  int local = 0;
  for (int k = 0; k < kPer; ++k) {
    const int b = tid * kPer + k;
    if (b >= va.B) break;
    const int q0 = varlen_start(va.cu_q, va.uni_q, b), q1 = varlen_start(va.cu_q, va.uni_q, b + 1);
    const int k0 = varlen_start(va.cu_k, va.uni_k, b), k1 = varlen_start(va.cu_k, va.uni_k, b + 1);
    const int len_q = q1 - q0, len_k = k1 - k0;
    const int n_kt = (len_k + kTileN - 1) / kTileN;
    const bool ok = q0 >= 0 && q1 >= q0 && q1 <= va.total_q && k0 >= 0 && k1 >= k0 &&
                    k1 <= va.total_k && (len_q == 0 || len_k > 0) &&
                    (!va.causal || len_k >= len_q) && n_kt <= kVarlenMaxBlocks;
    if (!ok) record_error(ctl + kCtlErr, kErrBadSeqlen);
    const int lq = ok ? len_q : 0;
    s_lq[b] = lq;
    s_lk[b] = len_k;
    if (lq > 0) {
      local += va.H_kv * ((va.group * ((lq + kTileM - 1) / kTileM) + va.tpu - 1) / va.tpu);
      atomicMax(&s_max_nb, n_kt);
    }
  }
  int total = 0;
  int run = block_exclusive_scan(local, s_warp, total);
  for (int k = 0; k < kPer; ++k) {
    const int b = tid * kPer + k;
    if (b >= va.B) break;
    s_pre[b] = run;
    if (s_lq[b] > 0)
      run += va.H_kv * ((va.group * ((s_lq[b] + kTileM - 1) / kTileM) + va.tpu - 1) / va.tpu);
  }
  if (tid == 0) s_pre[va.B] = total;
  const int max_nb = s_max_nb;
  for (int i = tid; i <= max_nb; i += kPlanThreads) s_bin[i] = 0;
  __syncthreads();
  // unit x -> (b, h_kv, pair (or tile, when tpu = 1), key blocks)
  auto unit_at = [&](int x) -> int4 {
    int lo = 0, hi = va.B - 1;  // last b with s_pre[b] <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pre[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const int b = lo, r = x - s_pre[b];
    const int len_q = s_lq[b], len_k = s_lk[b];
    const int n_qt = (len_q + kTileM - 1) / kTileM;
    const int pair = r / va.H_kv;
    int nb = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int f = va.tpu * pair + t;
      if (t < va.tpu && f < va.group * n_qt)
        nb = max(nb, varlen_kv_blocks(len_q, len_k, va.causal, n_qt - 1 - f / va.group));
    }
    return make_int4(b, r % va.H_kv, pair, nb);
  };
  // ---- counting sort on key blocks, most first
  for (int x = tid; x < total; x += kPlanThreads) atomicAdd(&s_bin[unit_at(x).w], 1);
  __syncthreads();
  // each thread takes kb consecutive bins in descending block count
  const int kb = (max_nb + 1 + kPlanThreads - 1) / kPlanThreads;
  int mine = 0;
  for (int i = 0; i < kb; ++i) {
    const int nb = max_nb - (tid * kb + i);
    if (nb >= 0) mine += s_bin[nb];
  }
  int dummy = 0;
  int at = block_exclusive_scan(mine, s_warp, dummy);
  for (int i = 0; i < kb; ++i) {
    const int nb = max_nb - (tid * kb + i);
    if (nb >= 0) {
      const int c = s_bin[nb];
      s_bin[nb] = at;
      at += c;
    }
  }
  if (tid == 0) ctl[kCtlVarlenUnits] = total;
  __syncthreads();
  for (int x = tid; x < total; x += kPlanThreads) {
    const int4 un = unit_at(x);
    units[atomicAdd(&s_bin[un.w], 1)] = un;
  }
}

}  // namespace

cudaError_t launch_prefill_tc(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, void *o, const OutView &ov, float *lse,
                              const PrefillPlan &plan, float scale, int *ctl, int num_sms,
                              cudaStream_t stream) {
  const VarlenArgs none = {};
  // Pairs of tiles from a group of 4 or 8 query heads run in clusters of
  // g / 2 CTAs, one pair per CTA, so that each K/V block is read once for
  // the whole group and multicast to all of them. A cluster's work unit is
  // then g / 2 times a pair's, which costs balance when there are few units
  // per SM: measured on the LLaMA-3-8B layer (256 pairs, 1.7 per cluster of
  // 2) the clustered schedule took 32.3 us against 31.4 us; with 1024 pairs
  // (B = 4, 16/4 heads, N = 4096) it took 160.4 us against 162.0 us. So
  // clusters are used from four pairs per SM up.
  const int csize = plan.total_units >= 4 * num_sms ? cluster_size_for(plan, ov.d) : 1;
  int grid = min(num_sms, plan.total_units);
  if (csize > 1) grid = max(csize, grid / csize * csize);
  return launch_any<false>(tm_q, tm_k, tm_v, o, ov, lse, plan, none, grid, csize, scale, ctl,
                           stream);
}

cudaError_t launch_varlen_plan(const VarlenArgs &va, int4 *units, int *ctl, cudaStream_t stream) {
  const size_t smem = plan_smem_bytes(va.B);
  static unsigned configured = 0;  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(configured & (1u << dev))) {
    e = cudaFuncSetAttribute(varlen_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(plan_smem_bytes(kVarlenMaxB)));
    if (e != cudaSuccess) return e;
    if (dev < 32) configured |= 1u << dev;
  }
  return launch_programmatic(varlen_plan_kernel, 1, kPlanThreads, smem, stream, va, units, ctl);
}

cudaError_t launch_prefill_tc_varlen(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                     const CUtensorMap &tm_v, void *o, const OutView &ov,
                                     float *lse, const VarlenArgs &va, float scale, int *ctl,
                                     int num_sms, cudaStream_t stream) {
  // the schedule fields the kernel reads; the unit count comes from the plan kernel
  PrefillPlan plan = make_prefill_plan(1, va.H_q, va.H_kv, 1, 1, va.causal);
  // the kernel takes L::kQTiles query tiles per listed unit
  if (va.tpu != (ov.d == 256 ? 1 : 2)) return cudaErrorInvalidValue;
  const long long most = varlen_max_units(va.B, va.H_q, va.H_kv, va.total_q, va.tpu);
  const int grid = static_cast<int>(most < num_sms ? (most < 1 ? 1 : most) : num_sms);
  return launch_any<true>(tm_q, tm_k, tm_v, o, ov, lse, plan, va, grid, 1, scale, ctl, stream);
}

}  // namespace gqa
