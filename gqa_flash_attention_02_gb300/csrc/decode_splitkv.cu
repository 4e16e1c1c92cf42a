// Single-token GQA decode against a bf16 K/V cache: a persistent,
// row-balanced split-KV kernel with the log-sum-exp merge in the same launch.
//
// The decode step reads every valid cache row once and does about 3 FLOPs
// per byte at the workload's group size, so it is bound by HBM bandwidth
// (kaispace.site, prefill-vs-decode note). What keeps HBM busy is a steady
// stream of bytes in flight on every SM. So the valid cache rows of all
// sequences are cut into 64-row units -- (b, h_kv, head group, sub-block),
// in that order -- and a persistent grid of a few CTAs per SM takes equal
// contiguous ranges of units. Each CTA streams its range through a TMA ring
// without stopping at sequence boundaries, so ragged lengths balance
// themselves and every SM reads about the same number of bytes. A range that
// covers part of a sequence produces a partial result: this is the
// split-sequence cached attention of the microLLM-rocm optimisation log
// (Experiments 282-284) with the splits chosen by row balance.
//
// A (b, h_kv, head group) "plane" serves up to 16 query heads of the group
// from ONE read of its K/V rows (no K/V replication: microLLM-rocm Experiment
// 044, BootstrapAI collab-014 "Kernel 9 GQA"). Per CTA:
//   * warp 4 is the producer: it walks the same unit sequence and issues the
//     TMA loads (K then V, 128-byte swizzled 64-column panels) into a ring of
//     stages, refilling a stage once the four MMA warps have released it;
//   * warps 0-3 take rows [16w, 16w+16) of each unit. The group's query
//     heads (padded to 16) times those rows is a dense contraction over d:
//     S = Q K^T and O += P V run on mma.sync (bf16 in, fp32 accumulate) from
//     ldmatrix fragments, with an online softmax (exp2, scale folded in) on
//     the register fragments;
//   * at the end of a plane's run the four warps leave their (m, l, O) in
//     shared memory and go on with the next unit; warp 5 (epilogue) merges
//     them. A run that covers the whole plane writes O, otherwise it writes a
//     partial and the last run of the plane to finish (atomic counter,
//     nobody waits) merges the partials:
//         M = max m_i,  L = sum 2^(m_i - M) l_i,  O = sum 2^(m_i - M) O_i / L.
//     The CTA's last run is merged by the MMA warps themselves.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "gqa_device.cuh"
#include "gqa_internal.h"

namespace gqa {

namespace {

constexpr int kMmaWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kEpilogueWarp = 5;
constexpr int kThreads = 32 * (kMmaWarps + 2);
// At head dim 256 a warp's 16-head x d fp32 accumulator would not fit in
// its registers, so two MMA warps share each 16-row group of a unit: both
// compute the group's S over all 256 dims and each keeps O for its 128
// columns. Elsewhere each MMA warp has its own rows and all d columns.
template <int D>
constexpr int kDimSplitOf = D == 256 ? 2 : 1;
// Cache rows per unit: 16 per row group of a bf16 cache (64 rows, or 32 at
// d = 256), 32 per MMA warp of a one-byte cache (128 rows), so a unit is 16 KB
// of K and of V at d = 128 and 256 alike, and each MMA warp's share of a
// stage's rows holds its accumulator fragments when it hands a run to the
// epilogue warp.
template <int D, bool kByte>
constexpr int kSubFor = kByte ? 128 : 64 / kDimSplitOf<D>;
constexpr int kHeads = kDecodeHeads;  // query heads per plane (mma M)

// A K/V cache box, read once per launch: loaded with an L2 evict-first
// policy, so the stream does not push out of L2 what is read back later in
// the launch (the query rows, the split partials the merges read).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_load_3d_stream(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                   int c0, int c1, int c2, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
      : "memory");
}
// Fewest units a CTA takes: fewer, longer runs (each run ends in a merge
// step and a plane spans at most nsub / kMinUnits + 2 CTAs); no CTA range
// is ever empty.
constexpr int kMinUnits = 4;
constexpr int kLenCache = 1024;  // sequence lengths kept in shared memory
constexpr int kEpRun = 1, kEpStop = 2;  // epilogue queue entry kinds
constexpr int kCtasPerSm = 1;    // the balanced partition assumes one resident wave

// Byte offset of (row, 16-byte unit u) inside a [rows][D] bf16 tile stored
// as D/64 panels of `rows` x 128 B with the TMA 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int row, int u, int rows) {
  return static_cast<uint32_t>((u >> 3) * rows * 128 + row * 128 + (((u & 7) ^ (row & 7)) << 4));
}

// Byte offset of 16-byte chunk c of row `row` in a one-byte tile of D-byte rows
// as TMA writes it: the 128-byte swizzle (D = 128) XORs the chunk index with
// row % 8, the 64-byte swizzle (D = 64) with (row / 2) % 4, so the 8 rows
// of an ldmatrix read fall in different banks.
template <int D>
__device__ __forceinline__ uint32_t swz8(int row, int c) {
  const int x = D == 128 ? (row & 7) : ((row >> 1) & 3);
  return static_cast<uint32_t>(row * D + ((c ^ x) << 4));
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

// The same with f16 operands (P.V over a one-byte cache: e4m3 and int8 widen to f16
// exactly, and P <= 1 keeps 11 significant bits in f16).
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two e4m3 values (low byte first) widened to an f16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// Two one-byte cache codes (the low 16 bits of v, low byte first) widened
// to an f16 pair, exactly. e4m3: the conversion instruction. int8: the byte
// with its sign bit flipped (x + 128, in 0..255) becomes the low mantissa
// bits of an f16 of exponent 10 (unit spacing on [1024, 2048)), i.e. the
// value 1152 + x, and subtracting 1152 leaves x.
template <bool kI8>
__device__ __forceinline__ uint32_t byte2_to_f16x2(uint32_t v) {
  if constexpr (kI8) {
    const uint32_t r = __byte_perm(v, 0u, 0x4140u) ^ 0x64806480u;
    uint32_t out;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(out) : "r"(r), "r"(0x64806480u));
    return out;
  } else {
    return e4m3x2_to_f16x2(static_cast<uint16_t>(v & 0xffffu));
  }
}

// An f16 pair holding one-byte cache values (e4m3, or integers in
// [-128, 127]) as a bf16 pair, exactly (at most 8 significant bits and
// exponents within both formats' ranges).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
  return pack_bf16x2(f.x, f.y);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// Barrier among the four MMA warps only (producer and epilogue keep going).
__device__ __forceinline__ void mma_warps_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kMmaWarps) : "memory");
}

template <int D, int NSTG, bool kByte>
struct DecodeSmem {
  static constexpr int kSub = kSubFor<D, kByte>;
  static constexpr int kDimSplit = kDimSplitOf<D>;
  static constexpr int kTile = kSub * D * (kByte ? 1 : 2);  // one K or V unit
  static constexpr int kQTile = kHeads * D * 2;  // the plane's 16 query rows
  static constexpr int kStage = 2 * kTile + kQTile;
  static constexpr int kRingBytes = NSTG * kStage;
  // A merged run state: O rows [16][kRow] (unnormalised), m[16], l[16].
  static constexpr int kRow = D + 4;  // padded: fragment stores spread over banks
  static constexpr int kStateFloats = kHeads * kRow + 2 * kHeads;
  static constexpr int kStateBytes = kStateFloats * 4;
  // At the end of the CTA's last run the four MMA warps merge their
  // (m, l, O) fragments through two slots of 32 lanes x (D/8 * 4
  // accumulators + m_lo, m_hi, l_lo, l_hi) in the stage of the run's last
  // unit and keep the merged state there, behind the slots.
  static constexpr int kLaneFloats = D / 8 / kDimSplit * 4 + 4;
  static constexpr int kTreeBytes = 2 * 32 * kLaneFloats * 4;
  static_assert(kTreeBytes + kStateBytes <= kStage, "run-end scratch");
  // A run that ends before the CTA's last unit is finished by the epilogue
  // warp: each MMA warp leaves its accumulator fragments in the K/V rows of
  // its row group in its columns of the stage (16 K and 16 V rows: 2 D /
  // kDimSplit bytes per lane) and its (m, l) in the stage's side buffer.
  static_assert(32 * (D / 8 / kDimSplit) * 4 * 4 ==
                    2 * (kSub * kDimSplit / kMmaWarps) * (D / kDimSplit) * (kByte ? 1 : 2),
                "fragments fill the warp's rows");
  static constexpr int kOffML = kRingBytes;                  // [NSTG][4 warps][32 lanes] float4
  static constexpr int kOffEp = kOffML + NSTG * kMmaWarps * 32 * 16;  // epilogue's merged state
  static constexpr int kOffQueue = kOffEp + kStateBytes;     // [NSTG] run entries of 16 ints
  static constexpr int kOffMeta = kOffQueue + NSTG * 64;     // per stage: b, pib, s, len,
                                                             // c_first, c_last, -, -
  static constexpr int kOffLen = kOffMeta + NSTG * 32;
  static constexpr int kOffBar = kOffLen + kLenCache * 4;  // full, empty, ep_full [NSTG]
  static constexpr int kOffInfo = kOffBar + 3 * NSTG * 8;
  static constexpr int kBytes = kOffInfo + 32;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kStage % 1024 == 0 && kStateBytes % 16 == 0 && kOffBar % 8 == 0, "alignment");
};

struct DecodeParams {
  const __nv_bfloat16 *q;
  const int *seqlens;
  const int *seqlens_first;  // read before the dependency wait: seqlens (a decoy only in the self-test)
  __nv_bfloat16 *o;
  float *lse;      // [B][H_q] natural-log sum of exp(scale q.k), or null
  float *part;     // [(grid + planes)] slots of O [16][D] (unnormalised), m [16], l [16]
  int *counters;   // [planes], zero between launches (the last merger re-arms it)
  int *err_word;
  const float *k_scale, *v_scale;  // one-byte caches: per K/V head dequantisation scales
  int B, H_q, H_kv, max_len, nhg;  // nhg = query-head groups of 16 per K/V head
  float scale_log2;
};

__device__ __forceinline__ int seq_len(const DecodeParams &prm, const int *s_len, int b) {
  return b < kLenCache ? s_len[b] : __ldg(prm.seqlens + b);
}

// Units of a sequence of length len for each of its planes (0 for a length
// outside [1, max_len]).
template <int kSub>
__device__ __forceinline__ int units_for(const DecodeParams &prm, int len) {
  return (len <= 0 || len > prm.max_len) ? 0 : (len + kSub - 1) / kSub;
}

// Position in the unit sequence: sequence b, plane pib inside it (h_kv-major,
// then head group), unit s inside the plane (nsub units per plane).
struct Pos {
  int b, pib, s, nsub;
};

template <int kSub>
__device__ __forceinline__ void advance(const DecodeParams &prm, const int *s_len,
                                        int planes_per_b, Pos &p) {
  if (++p.s < p.nsub) return;
  p.s = 0;
  if (++p.pib < planes_per_b) return;
  p.pib = 0;
  do {
    ++p.b;
    p.nsub = (p.b < prm.B) ? units_for<kSub>(prm, seq_len(prm, s_len, p.b)) : 1;  // past the end only at termination
  } while (p.b < prm.B && p.nsub == 0);
}

// Balanced partition of U units over G CTAs: the first r = U % G CTAs take
// q + 1 = U / G + 1 units, the others q.
struct Split {
  int q, r;
};

__device__ __forceinline__ int split_first(const Split &sp, int c) {
  return c * sp.q + min(c, sp.r);
}

__device__ __forceinline__ int owner_of(int u, const Split &sp) {
  const int t = sp.r * (sp.q + 1);
  return u < t ? u / (sp.q + 1) : sp.r + (u - t) / sp.q;
}

// Where CTA c starts when B <= 128 (warp-wide; lane holds the lengths of
// sequences 32k + lane): total units U, effective grid G (every CTA takes at
// least kMinUnits units), and the CTA's first unit as (sequence sb, plane
// spib, unit ss of the plane's snsub); sb = B when the CTA has none.
struct Start {
  int U, G, sb, spib, ss, snsub;
};

template <int kSub>
__device__ __forceinline__ Start locate_start(const DecodeParams &prm, const int (&len)[4],
                                              int lane, int c, int planes_per_b) {
  Start st{0, 1, prm.B, 0, 0, 1};
  int n_first[4], before_first[4];  // units of sequence 32k + lane and units before it
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int b = 32 * k + lane;
    const int n = b < prm.B ? units_for<kSub>(prm, len[k]) : 0;
    const int x = n * planes_per_b;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    n_first[k] = n;
    before_first[k] = st.U + incl - x;
    st.U += __shfl_sync(0xffffffffu, incl, 31);
  }
  st.G = max(1, min(static_cast<int>(gridDim.x), st.U / kMinUnits));
  const Split sp{st.U / st.G, st.U % st.G};
  const int u0 = (c < st.G) ? split_first(sp, c) : st.U;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int b = 32 * k + lane, x = n_first[k] * planes_per_b;
    const unsigned hit = __ballot_sync(
        0xffffffffu, b < prm.B && x > 0 && u0 >= before_first[k] && u0 < before_first[k] + x);
    if (hit && st.sb == prm.B) {
      const int src = __ffs(hit) - 1;
      const int bef = __shfl_sync(0xffffffffu, before_first[k], src);
      const int nn = __shfl_sync(0xffffffffu, n_first[k], src);
      const int off = u0 - bef;
      st.sb = 32 * k + src;
      st.spib = off / nn;
      st.ss = off % nn;
      st.snsub = nn;
    }
  }
  return st;
}

// Merges another (m, l, acc) state into this one for one row: returns the
// weights of the old and the new accumulator.
__device__ __forceinline__ void merge_row(float &m, float &l, float m2, float l2, float &w1,
                                          float &w2) {
  const float M = fmaxf(m, m2);
  w1 = (m == -INFINITY) ? 0.f : ex2(m - M);
  w2 = (m2 == -INFINITY) ? 0.f : ex2(m2 - M);
  l = fmaf(w1, l, w2 * l2);
  m = M;
}

// Folds the parts j = 0, 1, ..., nparts - 1 of a plane, in that order, for
// the (head, 4 columns) items it = t, t + nt, ... < Gh * D / 4 and writes O:
//   M' = max(M, m_j),  L' = 2^(M-M') L + 2^(m_j-M') l_j,
//   O' = 2^(M-M') O + 2^(m_j-M') O_j,  O = O' / L' at the end.
// Part j lives in partial slot pbase + j * kSlot, except part jself, the
// calling CTA's own state, which self(k, it, O, m, l) supplies for the k-th
// item of a group. lse_plane (if not null) receives each head's
// log-sum-exp. Every item's arithmetic is the same whichever CTA or
// warp runs it, so the result does not depend on who merges. kBatch parts'
// loads are in flight together.
template <int D, bool kByte, int kItems, int kBatch, typename SelfFn>
__device__ __forceinline__ void merge_parts(const float *pbase, int nparts, int jself, SelfFn self,
                                            int Gh, __nv_bfloat16 *o_plane, float *lse_plane,
                                            int t, int nt, float v_mul, int od) {
  constexpr int kQuads = D / 4;
  constexpr int kSlot = kHeads * (D + 2);
  const int items = Gh * kQuads;
  for (int base = t; base < items; base += nt * kItems) {
    float Mr[kItems], Lr[kItems];
    float4 Ar[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      Mr[k] = -INFINITY;
      Lr[k] = 0.f;
      Ar[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int j0 = 0; j0 < nparts; j0 += kBatch) {
      float4 v[kBatch][kItems];
      float mj[kBatch][kItems], lj[kBatch][kItems];
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
        const int j = j0 + jj;
        const float *pp = pbase + static_cast<size_t>(j) * kSlot;
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
          const int it = base + nt * k, h = it / kQuads;
          const bool ok = j < nparts && it < items;
          if (ok && j == jself) {
            self(k, it, v[jj][k], mj[jj][k], lj[jj][k]);
          } else if (ok) {
            v[jj][k] = __ldcg(reinterpret_cast<const float4 *>(pp) + it);
            mj[jj][k] = __ldcg(pp + kHeads * D + h);
            lj[jj][k] = __ldcg(pp + kHeads * D + kHeads + h);
          } else {
            v[jj][k] = make_float4(0.f, 0.f, 0.f, 0.f);
            mj[jj][k] = -INFINITY;
            lj[jj][k] = 0.f;
          }
        }
      }
#pragma unroll
      for (int jj = 0; jj < kBatch; ++jj) {
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
          float wa, wb;
          merge_row(Mr[k], Lr[k], mj[jj][k], lj[jj][k], wa, wb);
          Ar[k] = make_float4(fmaf(wa, Ar[k].x, wb * v[jj][k].x), fmaf(wa, Ar[k].y, wb * v[jj][k].y),
                              fmaf(wa, Ar[k].z, wb * v[jj][k].z), fmaf(wa, Ar[k].w, wb * v[jj][k].w));
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int it = base + nt * k;
      if (it < items) {
        const int h = it / kQuads, q4 = it % kQuads;
        const float il = v_mul / Lr[k];
        if constexpr (kByte) {
          // fragment columns 4q4 .. 4q4+3 are columns 4(q4 % 2) .. +3 of
          // n-tile q4 / 2, i.e. dims 16 (t / 2) + (t % 2) + 2 n (see write_o_row)
          const int t = q4 >> 1, base = 16 * (t >> 1) + (t & 1) + 8 * (q4 & 1);
          if (16 * (t >> 1) < od) {  // 16-dim chunks past the head dim are padding
            __nv_bfloat16 *row = o_plane + h * od + base;
            row[0] = __float2bfloat16_rn(Ar[k].x * il);
            row[2] = __float2bfloat16_rn(Ar[k].y * il);
            row[4] = __float2bfloat16_rn(Ar[k].z * il);
            row[6] = __float2bfloat16_rn(Ar[k].w * il);
          }
        } else {
          if (4 * q4 < od)  // columns past the head dim are padding
            *reinterpret_cast<uint2 *>(o_plane + h * od + 4 * q4) =
                make_uint2(pack_bf16x2(Ar[k].x * il, Ar[k].y * il), pack_bf16x2(Ar[k].z * il, Ar[k].w * il));
        }
        // the head's log-sum-exp (M, L are in log2 units of scale * q.k)
        if (lse_plane != nullptr && q4 == 0) lse_plane[h] = (Mr[k] + log2f(Lr[k])) * 0.6931471805599453f;
      }
    }
  }
}

// Writes one head's row of O (times il, as bf16) from accumulator
// fragments: entries e0, e0 + 1 of each n-tile are the lane's columns cc,
// cc + 1 of the tile. With a one-byte cache n-tile 2ch holds the even dims of the
// 16-dim chunk ch and n-tile 2ch + 1 its odd dims (the order P.V produces
// them in), so the lane's four values are dims 16ch + 2cc .. 16ch + 2cc + 3.
// (bf16 cache at d = 256: the NTW n-tiles of one warp's columns from col0.)
template <int D, bool kByte, int NTW = D / 8>
__device__ __forceinline__ void write_o_row(__nv_bfloat16 *dst, const float (&A)[NTW][4], int e0,
                                            int cc, float il, int od, int col0 = 0) {
  if constexpr (kByte) {
#pragma unroll
    for (int ch = 0; ch < D / 16; ++ch)
      if (16 * ch < od)  // 16-dim chunks past the head dim are padding
        *reinterpret_cast<uint2 *>(dst + 16 * ch + 2 * cc) =
          make_uint2(pack_bf16x2(A[2 * ch][e0] * il, A[2 * ch + 1][e0] * il),
                     pack_bf16x2(A[2 * ch][e0 + 1] * il, A[2 * ch + 1][e0 + 1] * il));
  } else {
#pragma unroll
    for (int t = 0; t < NTW; ++t)
      if (col0 + t * 8 < od)  // columns past the head dim are padding
        *reinterpret_cast<uint32_t *>(dst + col0 + t * 8 + cc) =
            pack_bf16x2(A[t][e0] * il, A[t][e0 + 1] * il);
  }
}

// float4 index, inside a stage, of MMA warp w's accumulator n-tile t (plus
// the lane) when the warp hands a run to the epilogue warp: the K and V rows
// of the stage that only warp w reads hold exactly its 32 lanes x D/8
// float4, lane-contiguous per n-tile (no bank conflicts). bf16 cache: rows
// [16w, 16w+16) of each 64-column panel of K then V; one-byte cache: rows
// [32w, 32w+32) of K (n-tiles 0 .. D/16-1), then of V. At d = 256 warp w
// has row group r = w % 2 and column half h = w / 2: rows [16r, 16r+16) of
// K panels 2h, 2h+1, then of the same V panels (its 16 n-tiles; the K rows
// are free once both warps of the group have computed their S).
template <int D, bool kByte>
__device__ __forceinline__ int frag_slot(int w, int t) {
  constexpr int NT = D / 8;
  constexpr int kSub = kSubFor<D, kByte>;
  if constexpr (D == 256) {
    constexpr int kRowGroups = kMmaWarps / kDimSplitOf<D>;
    const int c = t >> 2;  // 2 KB chunk: K (c < 2) or V panel 2h + (c & 1)
    const int panel = (c >> 1) * (D / 64) + (w / kRowGroups) * 2 + (c & 1);
    return panel * kSub * 8 + (w % kRowGroups) * 16 * 8 + (t & 3) * 32;
  } else if constexpr (kByte) {
    constexpr int kRowsF4 = (kSub / kMmaWarps) * D / 16;  // float4 of a warp's rows of one tile
    return (t < NT / 2 ? 0 : kSub * D / 16) + w * kRowsF4 + (t % (NT / 2)) * 32;
  } else {
    return (t >> 2) * kSub * 8 + w * 16 * 8 + (t & 3) * 32;
  }
}

// OD: the head dim, O's row stride and the columns stored (<= D; the TMA
// boxes read zeros past it, as for the prefill's padded head dims).
template <int D, int NSTG, bool kByte, int OD, bool kI8>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const DecodeParams prm) {
  using L = DecodeSmem<D, NSTG, kByte>;
  constexpr int kSub = L::kSub;
  constexpr int kDimSplit = L::kDimSplit;    // MMA warps per row group
  constexpr int kRowGroups = kMmaWarps / kDimSplit;
  constexpr int kRows = kSub / kRowGroups;   // rows of a unit per row group
  constexpr int NT = D / 8;                  // n-tiles of O
  constexpr int NTW = NT / kDimSplit;        // n-tiles of O per MMA warp
  constexpr int DW = D / kDimSplit;          // columns of O per MMA warp
  constexpr int kSlot = kHeads * (D + 2);    // floats per partial slot
  constexpr int kQuads = D / 4;              // float4 column groups per head
  constexpr int kPer = kHeads * kQuads / (32 * kMmaWarps);  // state items per MMA thread
  constexpr int kMergeItems = kPer < 4 ? kPer : 4;  // merge items in flight per MMA thread
  constexpr int kEpPer = kHeads * kQuads / 32;              // merge items per epilogue lane
  extern __shared__ uint8_t smem_raw[];
  // offset (not integer) arithmetic on smem_raw keeps the pointer in the
  // shared window, so accesses through it compile to shared-memory loads
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t s_base = smem_addr(smem);
  const uint32_t full = s_base + L::kOffBar;
  const uint32_t empty = full + 8 * NSTG;
  const uint32_t ep_full = empty + 8 * NSTG;  // [NSTG]: a run queued for the epilogue warp
  int *queue = reinterpret_cast<int *>(smem + L::kOffQueue);
  float4 *side_ml = reinterpret_cast<float4 *>(smem + L::kOffML);
  volatile int *info = reinterpret_cast<volatile int *>(smem + L::kOffInfo);
  int *s_len = reinterpret_cast<int *>(smem + L::kOffLen);
  int *stage_meta = reinterpret_cast<int *>(smem + L::kOffMeta);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const int group = prm.H_q / prm.H_kv;
  const int planes_per_b = prm.H_kv * prm.nhg;

  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == kEpilogueWarp && lane == 0) {
    for (int s = 0; s < NSTG; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, kMmaWarps);
    }
    for (int e = 0; e < NSTG; ++e) mbar_init(ep_full + 8 * e, kMmaWarps);
    fence_barrier_init();
  }
  // While the previous grid finishes (it may still be writing the inputs),
  // warp 0 works out the CTA's start from a first read of the lengths (B <=
  // 128) and prefetches the CTA's first units of K and V into L2: four with
  // a bf16 cache, two with a one-byte cache (where four measured slower).
  // The walk over planes reads the first read's lengths, put in shared
  // memory for it and rewritten after the wait. The start stands only if a
  // read after the dependency wait finds the same lengths; a prefetch never
  // changes what is read.
  const bool few_b = prm.B <= 128;
  int spec_len[4];
  Start spec{};
  if (warp == 0) {
    if (few_b) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int b = 32 * k + lane;
        spec_len[k] = b < prm.B ? __ldcg(prm.seqlens_first + b) : 0;
      }
      spec = locate_start<kSub>(prm, spec_len, lane, c, planes_per_b);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (32 * k + lane < prm.B) s_len[32 * k + lane] = spec_len[k];
      __syncwarp();
      if (lane == 0 && c < spec.G && spec.sb < prm.B) {
        const Split sp{spec.U / spec.G, spec.U % spec.G};
        const int n = min(kByte ? 2 : 4, sp.q + (c < sp.r ? 1 : 0));
        Pos p{spec.sb, spec.spib, spec.ss, spec.snsub};
        for (int i = 0; i < n && p.b < prm.B; ++i) {
          const int plane_kv = p.b * prm.H_kv + p.pib / prm.nhg;
#pragma unroll
          for (int q = 0; q < (kByte ? 1 : D / 64); ++q) {
            tma_prefetch_l2_3d(&tm_k, q * 64, p.s * kSub, plane_kv);
            tma_prefetch_l2_3d(&tm_v, q * 64, p.s * kSub, plane_kv);
          }
          advance<kSub>(prm, s_len, planes_per_b, p);
        }
      }
    } else {
      for (int b = 32 * lane; b < prm.B; b += 32 * 32) prefetch_l2(prm.seqlens + b);
    }
  }
  // Global reads (inputs, partials, counters) come after the previous grid
  // of the stream has completed; the next grid may start setting up.
  grid_dependency_wait();
  grid_launch_dependents();
  // ---- warp 0 (B <= 128): the lengths again, and the start unless they changed
  if (warp == 0 && few_b) {
    int len[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int b = 32 * k + lane;
      len[k] = b < prm.B ? __ldcg(prm.seqlens + b) : 0;
    }
    const bool same = __all_sync(0xffffffffu, len[0] == spec_len[0] && len[1] == spec_len[1] &&
                                                  len[2] == spec_len[2] && len[3] == spec_len[3]);
    const Start st = same ? spec : locate_start<kSub>(prm, len, lane, c, planes_per_b);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int b = 32 * k + lane;
      if (b < prm.B && b < kLenCache) s_len[b] = len[k];
      if (b < prm.B && (len[k] < 0 || len[k] > prm.max_len) && c == 0)
        record_error(prm.err_word, kErrBadSeqlen);
    }
    __syncwarp();
    if (lane == 0) {
      info[0] = st.U;
      info[1] = st.sb;
      info[2] = st.spib;
      info[3] = st.ss;
      info[5] = st.G;
      info[6] = st.snsub;
    }
  }
  // ---- warp 0 (B > 128): lengths (128 per pass, loads in flight together,
  // the first kLenCache kept in shared memory), total units and this CTA's
  // start
  if (warp == 0 && !few_b) {
    int U = 0;
    for (int b0 = 0; b0 < prm.B; b0 += 128) {
      int len[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int b = b0 + 32 * k + lane;
        len[k] = (b < prm.B) ? __ldg(prm.seqlens + b) : 0;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int b = b0 + 32 * k + lane;
        if (b < prm.B && b < kLenCache) s_len[b] = len[k];
        if (b < prm.B && (len[k] < 0 || len[k] > prm.max_len) && c == 0)
          record_error(prm.err_word, kErrBadSeqlen);
        const int n = units_for<kSub>(prm, len[k]);
        const int x = n * planes_per_b;
        int incl = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        U += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    __syncwarp();
    // effective grid: every CTA takes at least kMinUnits units
    const int G = max(1, min(static_cast<int>(gridDim.x), U / kMinUnits));
    const Split sp{U / G, U % G};
    const int u0 = (c < G) ? split_first(sp, c) : U;
    // locate u0: the sequence whose units contain it, then the plane and unit
    int sb = prm.B, spib = 0, ss = 0, snsub = 1;
    auto found = [&](unsigned hit, int b0, int before, int n) {
      const int src = __ffs(hit) - 1;
      const int bef = __shfl_sync(0xffffffffu, before, src);
      const int nn = __shfl_sync(0xffffffffu, n, src);
      const int off = u0 - bef;
      sb = b0 + src;
      spib = off / nn;
      ss = off % nn;
      snsub = nn;
    };
    {
      int cum = 0;
      for (int b0 = 0; b0 < prm.B && sb == prm.B; b0 += 32) {
        const int b = b0 + lane;
        const int n = (b < prm.B) ? units_for<kSub>(prm, seq_len(prm, s_len, b)) : 0;
        const int x = n * planes_per_b;
        int incl = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int before = cum + incl - x;  // units before sequence b
        const unsigned hit =
            __ballot_sync(0xffffffffu, b < prm.B && x > 0 && u0 >= before && u0 < before + x);
        if (hit) found(hit, b0, before, n);
        cum += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (lane == 0) {
      info[0] = U;
      info[1] = sb;
      info[2] = spib;
      info[3] = ss;
      info[5] = G;
      info[6] = snsub;
    }
  }
  __syncthreads();
  const int U = info[0];
  const int G = info[5];
  if (c >= G) return;
  if (warp < kMmaWarps) {
    // a sequence with no rows (or a rejected length) gets a zero output,
    // written by CTA b % G
    for (int b = c; b < prm.B; b += G) {
      if (units_for<kSub>(prm, seq_len(prm, s_len, b)) != 0) continue;
      uint4 *ob = reinterpret_cast<uint4 *>(prm.o + static_cast<size_t>(b) * prm.H_q * OD);
      for (int idx = tid; idx < prm.H_q * OD / 8; idx += 32 * kMmaWarps) ob[idx] = make_uint4(0, 0, 0, 0);
      if (prm.lse != nullptr)
        for (int h = tid; h < prm.H_q; h += 32 * kMmaWarps) prm.lse[static_cast<size_t>(b) * prm.H_q + h] = -INFINITY;
    }
  }
  if (U == 0) return;
  const Split sp{U / G, U % G};
  const int u0 = split_first(sp, c);
  const int n_units = sp.q + (c < sp.r ? 1 : 0);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Walks the CTA's units; per unit it leaves (b, pib, s, len) and the
    // first and last CTA of the unit's plane in the stage's metadata (the
    // owners take two divisions: off the MMA warps' path) and loads K, V and
    // the plane's 16 query rows with one completion barrier.
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      Pos p{info[1], info[2], info[3], info[6]};
      int c_first = 0, c_last = 0;
      for (int i = 0; i < n_units; ++i) {
        if (i == 0 || p.s == 0) {
          const int plane_first = u0 + i - p.s;  // global unit of (plane, s = 0)
          c_first = owner_of(plane_first, sp);
          c_last = owner_of(plane_first + p.nsub - 1, sp);
        }
        const int st = i % NSTG;
        if (i >= NSTG && !mbar_wait(empty + 8 * st, ((i / NSTG) & 1) ^ 1, nullptr)) {
          record_error(prm.err_word, kErrTimeout);
          break;
        }
        int *meta = stage_meta + 8 * st;
        meta[0] = p.b;
        meta[1] = p.pib;
        meta[2] = p.s;
        meta[3] = seq_len(prm, s_len, p.b);
        meta[4] = c_first;
        meta[5] = c_last;
        const int h_kv = p.pib / prm.nhg, hg = p.pib - h_kv * prm.nhg;
        const int plane_kv = p.b * prm.H_kv + h_kv;
        const uint32_t dst = s_base + st * L::kStage;
        mbar_arrive_expect_tx(full + 8 * st, L::kStage);
        if constexpr (kByte) {
          // one box of kSub rows x D bytes each (unswizzled)
          tma_load_3d_stream(dst, &tm_k, full + 8 * st, 0, p.s * kSub, plane_kv, pol);
          tma_load_3d_stream(dst + L::kTile, &tm_v, full + 8 * st, 0, p.s * kSub, plane_kv, pol);
        } else {
#pragma unroll
          for (int q = 0; q < D / 64; ++q) {
            tma_load_3d_stream(dst + q * kSub * 128, &tm_k, full + 8 * st, q * 64, p.s * kSub,
                               plane_kv, pol);
            tma_load_3d_stream(dst + L::kTile + q * kSub * 128, &tm_v, full + 8 * st, q * 64,
                               p.s * kSub, plane_kv, pol);
          }
        }
        // the plane's 16 query rows come with every unit (an L2 hit after the
        // first), so the MMA warps keep no Q fragments across units
        const int row = p.b * prm.H_q + h_kv * group + hg * kHeads;
#pragma unroll
        for (int q = 0; q < D / 64; ++q)
          tma_load_3d(dst + 2 * L::kTile + q * kHeads * 128, &tm_q, full + 8 * st, q * 64, row, 0);
        advance<kSub>(prm, s_len, planes_per_b, p);
      }
    }
    return;
  }

  if (warp == kEpilogueWarp) {
    // ------------------------------------------------------------ epilogue
    // Finishes the runs that end before the CTA's last unit, so the MMA
    // warps go on streaming meanwhile. Per queued run it folds the MMA
    // warps' (m, l, O) states, in warp order (per column half at d = 256,
    // over the half's two row groups), from the run's last stage (then
    // releases the stage), and either writes O (the run is the whole plane)
    // or publishes a partial: the state goes to slot c + plane, then (fence)
    // the plane's unit counter; the run that completes the count merges the
    // plane's parts. A run whose count is already complete when it starts
    // merges without publishing.
    float *so = reinterpret_cast<float *>(smem + L::kOffEp);
    float *sm = so + kHeads * L::kRow, *sl = sm + kHeads;
    const int r_lo = lane >> 2, r_hi = r_lo + 8, cc = 2 * (lane & 3);
    for (int k = 0;; ++k) {
      const int qk = k % NSTG;
      if (!mbar_wait_warp(ep_full + 8 * qk, (k / NSTG) & 1, nullptr)) {
        if (lane == 0) record_error(prm.err_word, kErrTimeout);
        return;
      }
      const int *qe = queue + 16 * qk;
      if (qe[0] == kEpStop) return;
      const int b = qe[1], hq0 = qe[2], Gh = qe[3], plane = qe[4], c_first = qe[5],
                c_last = qe[6], run_units = qe[7], nsub = qe[8], split = qe[9], st = qe[10];
      // A first look at the plane's unit counter, its latency hidden behind
      // the fold below (relaxed: a fence orders what it allows to be read).
      int done = 0;
      if (split && lane == 0) done = ld_relaxed_gpu(prm.counters + plane);
      __nv_bfloat16 *o_plane = prm.o + (static_cast<size_t>(b) * prm.H_q + hq0) * OD;
      float *lse_plane = prm.lse == nullptr ? nullptr : prm.lse + static_cast<size_t>(b) * prm.H_q + hq0;
      const float4 *frag = reinterpret_cast<const float4 *>(smem + st * L::kStage) + lane;
      float A[NTW][4];
      float m_lo, m_hi, l_lo, l_hi;
      // one pass per column share (d = 256: two), each over its row groups
#pragma unroll
      for (int h = 0; h < kDimSplit; ++h) {
        m_lo = m_hi = -INFINITY;
        l_lo = l_hi = 0.f;
#pragma unroll
        for (int t = 0; t < NTW; ++t) A[t][0] = A[t][1] = A[t][2] = A[t][3] = 0.f;
#pragma unroll
        for (int r = 0; r < kRowGroups; ++r) {
          const int w = r + kRowGroups * h;
          const float4 ml = side_ml[(st * kMmaWarps + w) * 32 + lane];
          float w1l, w2l, w1h, w2h;
          merge_row(m_lo, l_lo, ml.x, ml.z, w1l, w2l);
          merge_row(m_hi, l_hi, ml.y, ml.w, w1h, w2h);
#pragma unroll
          for (int t = 0; t < NTW; ++t) {
            const float4 v = frag[frag_slot<D, kByte>(w, t)];
            A[t][0] = fmaf(w1l, A[t][0], w2l * v.x);
            A[t][1] = fmaf(w1l, A[t][1], w2l * v.y);
            A[t][2] = fmaf(w1h, A[t][2], w2h * v.z);
            A[t][3] = fmaf(w1h, A[t][3], w2h * v.w);
          }
        }
        if (h == kDimSplit - 1) {
          // the stage is free for the producer again
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive_cnt(empty + 8 * st, kMmaWarps);
        }
        // full row sums: the four lanes of a quad hold different keys
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
        if (!split) {
          // the run is the whole plane: write O / l
          const float vm = kByte ? __ldg(prm.v_scale + (plane % planes_per_b) / prm.nhg) : 1.f;
          const float il = vm / l_lo, ih = vm / l_hi;
          if (r_lo < Gh) write_o_row<D, kByte, NTW>(o_plane + r_lo * OD, A, 0, cc, il, OD, h * DW);
          if (r_hi < Gh) write_o_row<D, kByte, NTW>(o_plane + r_hi * OD, A, 2, cc, ih, OD, h * DW);
          if (h == 0 && lse_plane != nullptr && (lane & 3) == 0) {
            // log-sum-exp per head (m, l in log2 units of scale * q.k)
            if (r_lo < Gh) lse_plane[r_lo] = (m_lo + log2f(l_lo)) * 0.6931471805599453f;
            if (r_hi < Gh) lse_plane[r_hi] = (m_hi + log2f(l_hi)) * 0.6931471805599453f;
          }
        } else {
#pragma unroll
          for (int t = 0; t < NTW; ++t) {
            *reinterpret_cast<float2 *>(so + r_lo * L::kRow + h * DW + t * 8 + cc) = make_float2(A[t][0], A[t][1]);
            *reinterpret_cast<float2 *>(so + r_hi * L::kRow + h * DW + t * 8 + cc) = make_float2(A[t][2], A[t][3]);
          }
        }
      }
      if (!split) continue;
      if ((lane & 3) == 0) {
        sm[r_lo] = m_lo;
        sl[r_lo] = l_lo;
        sm[r_hi] = m_hi;
        sl[r_hi] = l_hi;
      }
      __syncwarp();
      bool last = __shfl_sync(0xffffffffu, done, 0) + run_units == nsub;
      // the first look is relaxed: a fence then orders the reads it allows
      if (last) fence_acq_rel_gpu();
      if (!last) {
        float4 *dst = reinterpret_cast<float4 *>(prm.part + static_cast<size_t>(c + plane) * kSlot);
#pragma unroll
        for (int k2 = 0; k2 < kEpPer; ++k2) {
          const int it = lane + 32 * k2;
          dst[it] = *reinterpret_cast<const float4 *>(so + (it / kQuads) * L::kRow + 4 * (it % kQuads));
        }
        if (lane < kHeads) {
          reinterpret_cast<float *>(dst)[kHeads * D + lane] = sm[lane];
          reinterpret_cast<float *>(dst)[kHeads * D + kHeads + lane] = sl[lane];
        }
        // the count publishes the part (release, for the warp's stores
        // before the barrier) and, for the run that completes it, acquires
        // the other parts
        __syncwarp();
        int prev = 0;
        if (lane == 0) prev = atom_add_acq_rel_gpu(prm.counters + plane, run_units);
        last = __shfl_sync(0xffffffffu, prev, 0) + run_units == nsub;
      }
      if (last) {
        __syncwarp();
        auto self = [&](int, int it, float4 &v, float &m, float &l) {
          const int h = it / kQuads;
          v = *reinterpret_cast<const float4 *>(so + h * L::kRow + 4 * (it % kQuads));
          m = sm[h];
          l = sl[h];
        };
        merge_parts<D, kByte, 6, 4>(prm.part + static_cast<size_t>(c_first + plane) * kSlot,
                             c_last - c_first + 1, c - c_first, self, Gh, o_plane, lse_plane, lane, 32,
                             kByte ? __ldg(prm.v_scale + (plane % planes_per_b) / prm.nhg) : 1.f, OD);
        // re-arm for the next launch (every other count of the plane was
        // observed before this store)
        if (lane == 0) st_relaxed_gpu(prm.counters + plane, 0);
      }
      __syncwarp();  // every lane is done with the state buffer
    }
  }

  // -------------------------------------------------------------- MMA warps
  const int wgrp = warp % kRowGroups;   // this warp's row group
  const int whalf = warp / kRowGroups;  // and its share of the columns (d = 256)
  const int wrow = wgrp * kRows;        // this warp's first row in a unit
  int seg_first_i = 0;
  int ep_k = 0;  // runs queued for the epilogue warp so far
  int counter_seen = 0, counter_seen2 = 0;  // the last run's looks at its plane counter
  struct FinalRun {
    int plane = -1, c_first, c_last, run_units, nsub, Gh;
    float vmul;
    __nv_bfloat16 *o_plane;
    float *lse_plane;
    float *state;
  } fin;
  float acc[NTW][4];
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

  for (int i = 0; i < n_units; ++i) {
    const int st = i % NSTG;
    if (!mbar_wait_warp(full + 8 * st, (i / NSTG) & 1, nullptr)) {
      if (lane == 0) record_error(prm.err_word, kErrTimeout);
      break;  // every MMA warp times out on the same phase
    }
    const int *meta = stage_meta + 8 * st;
    const int b = meta[0], pib = meta[1], s = meta[2], len = meta[3];
    const int nsub = (len + kSub - 1) / kSub;
    const int h_kv = pib / prm.nhg, hg = pib - h_kv * prm.nhg;
    const int Gh = min(kHeads, group - hg * kHeads);  // query heads in this plane
    const int hq0 = h_kv * group + hg * kHeads;
    const uint32_t kt = s_base + st * L::kStage;
    const uint32_t vt = kt + L::kTile;
    if (i == 0 || s == 0) {
      // a new run
      seg_first_i = i;
      // The CTA's last run reads its plane's unit counter now; the value is
      // used at the run's end (a fence then orders the reads it allows), so
      // the load's latency hides behind the run's units.
      if (warp == 0 && lane == 0 && i + (nsub - s) >= n_units)
        counter_seen = ld_relaxed_gpu(prm.counters + b * planes_per_b + pib);
      counter_seen2 = 0;
#pragma unroll
      for (int t = 0; t < NTW; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
      m_lo = m_hi = -INFINITY;
      l_lo = l_hi = 0.f;
    }
    if (warp == 0 && lane == 0 && i == n_units - 3 && i > seg_first_i && i + (nsub - s) >= n_units)
      counter_seen2 = ld_relaxed_gpu(prm.counters + b * planes_per_b + pib);  // a later look
    const int rows_here = min(kSub, len - s * kSub);  // valid rows in this unit
    // one-byte caches: the K/V head's scales (K's folds into the exponent scale)
    const float sl2 = kByte ? prm.scale_log2 * __ldg(prm.k_scale + h_kv) : prm.scale_log2;
#pragma unroll 1
    for (int grp = 0; grp < kRows / 16; ++grp) {
    const int r0 = wrow + 16 * grp;  // first row of this 16-row group in the unit
    // ---- S = Q K^T for the group's 16 rows (two n-tiles of 8 keys)
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t qt = kt + 2 * L::kTile;
    const bool lo_ok = (lane >> 2) < Gh, hi_ok = (lane >> 2) + 8 < Gh;
    if constexpr (kByte) {
      // The one-byte K rows are read as 8x8 matrices of 16-bit pairs: lane l gets
      // key row l/4 of a matrix and bytes 4(l%4)..+3, the dims 4t..4t+3 (t =
      // l%4) of a 16-dim chunk. Widened to two bf16 pairs they are the B
      // fragment of one k16 step under a permutation of the contraction
      // index (k 2t,2t+1 <-> dims 4t,4t+1; k 2t+8,2t+9 <-> dims 4t+2,4t+3),
      // and Q's A fragment is read under the same permutation (8 bytes of
      // dims 4t..4t+3 per row), so S is unchanged. Matrices: keys 0-7 and
      // 8-15 of the group x chunks 2cp and 2cp+1.
      const int mat = lane >> 3;
      const int key = r0 + (lane & 7) + ((mat >> 1) << 3);
      const int t = lane & 3, g = lane >> 2;
#pragma unroll
      for (int cp = 0; cp < D / 32; ++cp) {
        uint32_t r[4];
        ldsm_x4(kt + swz8<D>(key, 2 * cp + (mat & 1)), r[0], r[1], r[2], r[3]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // chunk 2cp + h
          const int ch = 2 * cp + h;
          uint32_t qa[4];
          const uint2 lo = *reinterpret_cast<const uint2 *>(smem + (qt - s_base) +
                                                            swz(g, 2 * ch + (t >> 1), kHeads) + 8 * (t & 1));
          const uint2 hi = *reinterpret_cast<const uint2 *>(smem + (qt - s_base) +
                                                            swz(g + 8, 2 * ch + (t >> 1), kHeads) + 8 * (t & 1));
          qa[0] = lo_ok ? lo.x : 0u;
          qa[2] = lo_ok ? lo.y : 0u;
          qa[1] = hi_ok ? hi.x : 0u;
          qa[3] = hi_ok ? hi.y : 0u;
          const uint32_t k0 = r[h], k1 = r[2 + h];  // keys 0-7, keys 8-15
          mma_bf16(s0, qa, f16x2_to_bf16x2(byte2_to_f16x2<kI8>(k0)),
                   f16x2_to_bf16x2(byte2_to_f16x2<kI8>(k0 >> 16)));
          mma_bf16(s1, qa, f16x2_to_bf16x2(byte2_to_f16x2<kI8>(k1)),
                   f16x2_to_bf16x2(byte2_to_f16x2<kI8>(k1 >> 16)));
        }
      }
    } else {
      // A (16 heads x 16 of D) from the stage's Q tile: ldmatrix lanes 0-15
      // address rows 0-15 at a k-step's first 8 columns, lanes 16-31 the
      // next 8; rows past the group are zero. B (K^T): lanes 0-7 keys 0-7
      // unit 2ks; 8-15 keys 0-7 unit 2ks+1; 16-23 keys 8-15 unit 2ks;
      // 24-31 keys 8-15 unit 2ks+1.
      const int key = r0 + (lane & 7) + ((lane >> 4) << 3);
      const int uo = (lane >> 3) & 1;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t qa[4], b0, b1, b2, b3;
        ldsm_x4(qt + swz(lane & 15, 2 * ks + (lane >> 4), kHeads), qa[0], qa[1], qa[2], qa[3]);
        if (!lo_ok) qa[0] = qa[2] = 0u;
        if (!hi_ok) qa[1] = qa[3] = 0u;
        ldsm_x4(kt + swz(key, 2 * ks + uo, kSub), b0, b1, b2, b3);
        mma_bf16(s0, qa, b0, b1);
        mma_bf16(s1, qa, b2, b3);
      }
    }
    // ---- online softmax on the fragments: rows (heads) lane/4 and lane/4+8
    const int kc = r0 + 2 * (lane & 3);  // key of s?[0]; s?[1] is kc+1; s1 adds 8
    float x[8] = {s0[0] * sl2, s0[1] * sl2, s1[0] * sl2, s1[1] * sl2,
                  s0[2] * sl2, s0[3] * sl2, s1[2] * sl2, s1[3] * sl2};
    const int keys[4] = {kc, kc + 1, kc + 8, kc + 9};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (keys[e] >= rows_here) {
        x[e] = -INFINITY;
        x[4 + e] = -INFINITY;
      }
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
    float pr[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      pr[e] = (mn_lo == -INFINITY) ? 0.f : ex2(x[e] - mn_lo);
      pr[4 + e] = (mn_hi == -INFINITY) ? 0.f : ex2(x[4 + e] - mn_hi);
    }
    l_lo = l_lo * a_lo + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
    l_hi = l_hi * a_hi + ((pr[4] + pr[5]) + (pr[6] + pr[7]));
    m_lo = mn_lo;
    m_hi = mn_hi;
#pragma unroll
    for (int t = 0; t < NTW; ++t) {
      acc[t][0] *= a_lo;
      acc[t][1] *= a_lo;
      acc[t][2] *= a_hi;
      acc[t][3] *= a_hi;
    }
    // ---- O += P V (V rows = k, d = n): transposed ldmatrix of 8x8 blocks
    if constexpr (kByte) {
      // P as f16 (16 heads x 16 keys). The one-byte V rows are read transposed
      // as 16-bit pairs: lane l gets keys 2t, 2t+1 of a matrix at bytes
      // 2c, 2c+1 (c = l/4), i.e. two dims of a 16-dim chunk for two keys;
      // one byte permute splits them into the key pairs of dim 2c and of dim
      // 2c+1, widened to f16 pairs: B fragments of two n-tiles, one holding
      // the chunk's even dims, the other its odd dims (the accumulator's
      // column order that the final O stores undo). Keys 8-15 of the group
      // are rows past the sequence when r0 + 8 >= rows_here: P is 0 there,
      // and any NaN bytes are replaced by zero before they reach the MMA.
      const uint32_t pa[4] = {pack_f16x2(pr[0], pr[1]), pack_f16x2(pr[4], pr[5]),
                              pack_f16x2(pr[2], pr[3]), pack_f16x2(pr[6], pr[7])};
      const int key = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
      const int t = lane & 3;
      const bool dead0 = r0 + 2 * t >= rows_here, dead1 = r0 + 2 * t + 1 >= rows_here;
      const bool dead8 = r0 + 8 + 2 * t >= rows_here, dead9 = r0 + 9 + 2 * t >= rows_here;
#pragma unroll
      for (int cp = 0; cp < D / 32; ++cp) {
        uint32_t r[4];
        ldsm_x4_t(vt + swz8<D>(key, 2 * cp + (lane >> 4)), r[0], r[1], r[2], r[3]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ch = 2 * cp + h;
          // keys 0-7 (r[2h]) and 8-15 (r[2h+1]); zero the bytes of keys past the sequence
          uint32_t lo = r[2 * h], hi = r[2 * h + 1];
          lo = (dead0 ? 0u : (lo & 0x0000ffffu)) | (dead1 ? 0u : (lo & 0xffff0000u));
          hi = (dead8 ? 0u : (hi & 0x0000ffffu)) | (dead9 ? 0u : (hi & 0xffff0000u));
          const uint32_t plo = __byte_perm(lo, 0, 0x3120), phi = __byte_perm(hi, 0, 0x3120);
          mma_f16(acc[2 * ch], pa, byte2_to_f16x2<kI8>(plo), byte2_to_f16x2<kI8>(phi));
          mma_f16(acc[2 * ch + 1], pa, byte2_to_f16x2<kI8>(plo >> 16), byte2_to_f16x2<kI8>(phi >> 16));
        }
      }
    } else {
      // P as the A operand (16 heads x 16 keys): keys 0-7 from n-tile 0, 8-15 from n-tile 1
      const uint32_t pa[4] = {pack_bf16x2(pr[0], pr[1]), pack_bf16x2(pr[4], pr[5]),
                              pack_bf16x2(pr[2], pr[3]), pack_bf16x2(pr[6], pr[7])};
      // lanes 0-7: keys 0-7 unit u; 8-15: keys 8-15 unit u; 16-23: keys 0-7 unit u+1;
      // 24-31: keys 8-15 unit u+1  -> {b0,b1} for d-tile u and {b0,b1} for u+1
      const int key = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
      const int uo = lane >> 4;
      // Rows past the sequence (other sequences' data or NaN padding) must
      // not reach P.V: their P is 0, and their V values are cleared in the
      // fragments (b0, b2: keys 2t, 2t+1 of the group; b1, b3: keys 2t+8,
      // 2t+9; t = lane % 4; the lower half of a pair is the lower key).
      const bool partial = r0 + 16 > rows_here;  // warp-uniform
      const int k2 = r0 + 2 * (lane & 3);
      const uint32_t keep_lo = (k2 < rows_here ? 0x0000ffffu : 0u) | (k2 + 1 < rows_here ? 0xffff0000u : 0u);
      const uint32_t keep_hi = (k2 + 8 < rows_here ? 0x0000ffffu : 0u) | (k2 + 9 < rows_here ? 0xffff0000u : 0u);
#pragma unroll
      for (int u = 0; u < NTW; u += 2) {  // the warp's n-tiles (8 columns each)
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vt + swz(key, whalf * NTW + u + uo, kSub), b0, b1, b2, b3);
        if (partial) {
          b0 &= keep_lo;
          b2 &= keep_lo;
          b1 &= keep_hi;
          b3 &= keep_hi;
        }
        mma_bf16(acc[u], pa, b0, b1);
        mma_bf16(acc[u + 1], pa, b2, b3);
      }
    }
    }  // 16-row groups

    const bool final_run = (i == n_units - 1);
    if (!final_run && s != nsub - 1) {
      // release the stage to the producer
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + 8 * st);
      continue;
    }
    // ---- the run ends here; stage st stays held
    // (the stage's metadata stays until the stage is released)
    const int c_first = meta[4], c_last = meta[5];
    const bool split = c_first != c_last;
    const int plane = b * planes_per_b + pib;
    const int run_units = i - seg_first_i + 1;
    if (!final_run) {
      // Hand the run to the epilogue warp and go on streaming. The warp's
      // fragments go to the K and V rows of the stage that only this warp
      // reads (lane-contiguous float4 per n-tile: no bank conflicts), its
      // (m, l) to the stage's side buffer; the epilogue warp releases the
      // stage. The queue cannot overrun: every queued run holds a stage.
      const int qk = ep_k % NSTG;
      if constexpr (kDimSplit > 1) {
        // the group's K rows hold both its warps' fragments: both must be
        // done with their S (named barriers 2, 3: one per row group)
        if (wgrp == 0)
          asm volatile("bar.sync 2, %0;" ::"n"(32 * kDimSplit) : "memory");
        else
          asm volatile("bar.sync 3, %0;" ::"n"(32 * kDimSplit) : "memory");
      } else {
        __syncwarp();  // the warp's reads of its rows are done
      }
      float4 *rows = reinterpret_cast<float4 *>(smem + st * L::kStage) + lane;
#pragma unroll
      for (int t = 0; t < NTW; ++t)
        rows[frag_slot<D, kByte>(warp, t)] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
      side_ml[(st * kMmaWarps + warp) * 32 + lane] = make_float4(m_lo, m_hi, l_lo, l_hi);
      if (warp == 0 && lane == 0) {
        int *qe = queue + 16 * qk;
        qe[0] = kEpRun;
        qe[1] = b;
        qe[2] = hq0;
        qe[3] = Gh;
        qe[4] = plane;
        qe[5] = c_first;
        qe[6] = c_last;
        qe[7] = run_units;
        qe[8] = nsub;
        qe[9] = split ? 1 : 0;
        qe[10] = st;
      }
      fence_proxy_async_smem();  // before the TMA that refills the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(ep_full + 8 * qk);
      ++ep_k;
      continue;
    }
    // The CTA's last run: the four warps merge their (m, l, O) fragments
    // in the held stage (a lane with the same lane of another warp holds the
    // same heads and columns): warps 2,3 -> 0,1, then warp 1 -> warp 0. At
    // d = 256 the second row group's warps hand their states to the first's
    // (warp 1 -> 0, 3 -> 2), and warps 0 and 2 finish a column half each.
    float *tree = reinterpret_cast<float *>(smem + st * L::kStage);
    float *mine = tree + lane * L::kLaneFloats;
    auto put = [&](int slot) {
      float *dst = mine + slot * 32 * L::kLaneFloats;
#pragma unroll
      for (int t = 0; t < NTW; ++t)
        *reinterpret_cast<float4 *>(dst + 4 * t) = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
      *reinterpret_cast<float4 *>(dst + 4 * NTW) = make_float4(m_lo, m_hi, l_lo, l_hi);
    };
    auto take = [&](int slot) {
      const float *src = mine + slot * 32 * L::kLaneFloats;
      const float4 ml = *reinterpret_cast<const float4 *>(src + 4 * NTW);
      float w1l, w2l, w1h, w2h;
      merge_row(m_lo, l_lo, ml.x, ml.z, w1l, w2l);
      merge_row(m_hi, l_hi, ml.y, ml.w, w1h, w2h);
#pragma unroll
      for (int t = 0; t < NTW; ++t) {
        const float4 a = *reinterpret_cast<const float4 *>(src + 4 * t);
        acc[t][0] = fmaf(w1l, acc[t][0], w2l * a.x);
        acc[t][1] = fmaf(w1l, acc[t][1], w2l * a.y);
        acc[t][2] = fmaf(w1h, acc[t][2], w2h * a.z);
        acc[t][3] = fmaf(w1h, acc[t][3], w2h * a.w);
      }
    };
    mma_warps_sync();  // every warp is done reading stage st
    if constexpr (kRowGroups == 4) {
      if (warp >= 2) put(warp - 2);
      mma_warps_sync();
      if (warp < 2) take(warp);
      mma_warps_sync();
      if (warp == 1) put(0);
      mma_warps_sync();
    } else {
      if (wgrp == 1) put(whalf);
      mma_warps_sync();
    }
    __nv_bfloat16 *o_plane = prm.o + (static_cast<size_t>(b) * prm.H_q + hq0) * OD;
    float *lse_plane = prm.lse == nullptr ? nullptr : prm.lse + static_cast<size_t>(b) * prm.H_q + hq0;
    // a split run's merged state stays behind the tree slots in the stage
    float *state = tree + L::kTreeBytes / 4;
    float *st_m = state + kHeads * L::kRow, *st_l = st_m + kHeads;
    if (wgrp == 0) {
      take(kRowGroups == 4 ? 0 : whalf);
      // full row sums: the four lanes of a quad hold different keys
      l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
      l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
      l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
      l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
      const int r_lo = lane >> 2, r_hi = r_lo + 8, cc = 2 * (lane & 3);
      if (!split) {
        // this run is the whole plane: write O / l
        const float vm = kByte ? __ldg(prm.v_scale + h_kv) : 1.f;
        const float il = vm / l_lo, ih = vm / l_hi;
        if (r_lo < Gh) write_o_row<D, kByte, NTW>(o_plane + r_lo * OD, acc, 0, cc, il, OD, whalf * DW);
        if (r_hi < Gh) write_o_row<D, kByte, NTW>(o_plane + r_hi * OD, acc, 2, cc, ih, OD, whalf * DW);
        if (whalf == 0 && lse_plane != nullptr && (lane & 3) == 0) {
          // log-sum-exp per head (m, l in log2 units of scale * q.k)
          if (r_lo < Gh) lse_plane[r_lo] = (m_lo + log2f(l_lo)) * 0.6931471805599453f;
          if (r_hi < Gh) lse_plane[r_hi] = (m_hi + log2f(l_hi)) * 0.6931471805599453f;
        }
      } else {
#pragma unroll
        for (int t = 0; t < NTW; ++t) {
          *reinterpret_cast<float2 *>(state + r_lo * L::kRow + whalf * DW + t * 8 + cc) =
              make_float2(acc[t][0], acc[t][1]);
          *reinterpret_cast<float2 *>(state + r_hi * L::kRow + whalf * DW + t * 8 + cc) =
              make_float2(acc[t][2], acc[t][3]);
        }
        if (whalf == 0 && (lane & 3) == 0) {
          st_m[r_lo] = m_lo;
          st_l[r_lo] = l_lo;
          st_m[r_hi] = m_hi;
          st_l[r_hi] = l_hi;
        }
        if (warp == 0 && lane == 0) {
          // If every other run of the plane had counted in (their partials
          // published before their count) when one of the early looks at the
          // counter was made, this run is the last one and merges without
          // publishing its own part.
          const bool direct = max(counter_seen, counter_seen2) + run_units == nsub;
          if (direct) fence_acq_rel_gpu();
          info[4] = direct ? 1 : 0;
        }
      }
    }
    if (split) {
      // the CTA's last run leaves the loop with its merged state in shared
      // memory; it is published and merged below, outside the loop, so the
      // loop's registers stay low
      fin.plane = plane;
      fin.c_first = c_first;
      fin.c_last = c_last;
      fin.run_units = run_units;
      fin.nsub = nsub;
      fin.Gh = Gh;
      fin.vmul = kByte ? __ldg(prm.v_scale + h_kv) : 1.f;
      fin.o_plane = o_plane;
      fin.lse_plane = lse_plane;
      fin.state = state;
    }
    break;
  }
  if (fin.plane >= 0) {
    // ---- the CTA's last run, part of a plane other CTAs share
    const int plane = fin.plane, c_first = fin.c_first, c_last = fin.c_last;
    const int run_units = fin.run_units, nsub = fin.nsub, Gh = fin.Gh;
    __nv_bfloat16 *o_plane = fin.o_plane;
    float *lse_plane = fin.lse_plane;
    float *state = fin.state;
    float *st_m = state + kHeads * L::kRow, *st_l = st_m + kHeads;
    mma_warps_sync();  // the run's state is in shared memory
    bool last = info[4] != 0;
    if (!last) {
      // publish the state to slot c + plane (coalesced, all MMA threads),
      // then count the plane's units done: the run that completes the
      // count merges (no CTA range is empty, so every owner takes part)
      float *dst = prm.part + static_cast<size_t>(c + plane) * kSlot;
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int it = tid + 32 * kMmaWarps * k;
        reinterpret_cast<float4 *>(dst)[it] =
            *reinterpret_cast<const float4 *>(state + (it / kQuads) * L::kRow + 4 * (it % kQuads));
      }
      if (tid < kHeads) {
        dst[kHeads * D + tid] = st_m[tid];
        dst[kHeads * D + kHeads + tid] = st_l[tid];
      }
      // the count publishes the part (release, for the stores of all MMA
      // threads before the barrier) and, for the run that completes it,
      // acquires the other parts
      mma_warps_sync();
      if (tid == 0)
        info[4] = atom_add_acq_rel_gpu(prm.counters + plane, run_units) + run_units == nsub ? 1 : 0;
      mma_warps_sync();
      last = info[4] != 0;
    }
    if (last) {
      // ---- the plane's last run: merge the parts of CTAs c_first..c_last
      // (CTA cs in slot cs + plane; this CTA's own part in shared memory;
      // the acquiring thread passed a barrier with the others since)
      auto self = [&](int, int it, float4 &v, float &m, float &l) {
        const int h = it / kQuads;
        v = *reinterpret_cast<const float4 *>(state + h * L::kRow + 4 * (it % kQuads));
        m = st_m[h];
        l = st_l[h];
      };
      merge_parts<D, kByte, kMergeItems, 4>(prm.part + static_cast<size_t>(c_first + plane) * kSlot,
                              c_last - c_first + 1, c - c_first, self, Gh, o_plane, lse_plane, tid,
                              32 * kMmaWarps, fin.vmul, OD);
      // re-arm for the next launch (every other count of the plane was
      // observed before this store)
      if (tid == 0) st_relaxed_gpu(prm.counters + plane, 0);
    }
  }
  // tell the epilogue warp that no more runs follow (every queued run holds
  // a stage, so the entry's previous use has been consumed)
  const int qk = ep_k % NSTG;
  if (warp == 0 && lane == 0) queue[16 * qk] = kEpStop;
  __syncwarp();
  if (lane == 0) mbar_arrive(ep_full + 8 * qk);
}

template <int D, int NSTG, bool kByte, int OD, bool kI8 = false>
cudaError_t launch_decode_d(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                            const CUtensorMap &tm_v, const void *q, const int *seqlens, void *o,
                            float *lse, float *partials, int *counters, int B, int H_q, int H_kv,
                            int max_len, float scale, int grid, int *err_word,
                            const float *k_scale, const float *v_scale, cudaStream_t stream,
                            const int *seqlens_first = nullptr) {
  using L = DecodeSmem<D, NSTG, kByte>;
  static_assert(L::kAlloc <= 227 * 1024, "shared memory");
  static unsigned configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 32 || !(configured & (1u << dev))) {
    e = cudaFuncSetAttribute(decode_kernel<D, NSTG, kByte, OD, kI8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    if (dev < 32) configured |= 1u << dev;
  }
  DecodeParams prm;
  prm.q = static_cast<const __nv_bfloat16 *>(q);
  prm.seqlens = seqlens;
  prm.seqlens_first = seqlens_first != nullptr ? seqlens_first : seqlens;
  prm.o = static_cast<__nv_bfloat16 *>(o);
  prm.lse = lse;
  prm.part = partials;
  prm.counters = counters;
  prm.err_word = err_word;
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  prm.B = B;
  prm.H_q = H_q;
  prm.H_kv = H_kv;
  prm.max_len = max_len;
  prm.nhg = decode_head_groups(H_q, H_kv);
  prm.scale_log2 = scale * 1.4426950408889634f;
  return launch_programmatic(decode_kernel<D, NSTG, kByte, OD, kI8>, grid, kThreads, L::kAlloc, stream, tm_q,
                             tm_k, tm_v, prm);
}

}  // namespace

int decode_head_groups(int H_q, int H_kv) { return (H_q / H_kv + kHeads - 1) / kHeads; }

size_t decode_partials_bytes(int B, int H_q, int H_kv, int d, int grid) {
  const size_t planes = static_cast<size_t>(B) * H_kv * decode_head_groups(H_q, H_kv);
  const size_t D = d <= 64 ? 64 : (d <= 128 ? 128 : 256);  // the kernel's head dim (32, 96 padded)
  return (static_cast<size_t>(grid) + planes) * kHeads * (D + 2) * sizeof(float);
}

size_t decode_planes(int B, int H_q, int H_kv) {
  return static_cast<size_t>(B) * H_kv * decode_head_groups(H_q, H_kv);
}

bool decode_units_fit(int B, int H_q, int H_kv, int max_len) {
  const long long units = static_cast<long long>(decode_planes(B, H_q, H_kv)) *
                          ((static_cast<long long>(max_len) + kDecodeMinUnit - 1) / kDecodeMinUnit);
  return units <= (1ll << 30);
}

int decode_grid(int B, int H_q, int H_kv, int max_len, int d, int num_sms, int chunk) {
  (void)d;
  // Rows of all planes if every sequence were full length; the real count is
  // known on the device only, so this is an upper bound.
  const long long rows = static_cast<long long>(decode_planes(B, H_q, H_kv)) * max_len;
  long long g;
  if (chunk > 0) {
    g = (rows + chunk - 1) / chunk;
  } else {
    g = static_cast<long long>(num_sms) * kCtasPerSm;
  }
  if (g > 65535) g = 65535;
  return g < 1 ? 1 : static_cast<int>(g);
}

cudaError_t launch_decode_bf16(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                               const CUtensorMap &tm_v, const void *q, const int *seqlens, void *o,
                               float *lse, float *partials, int *counters, int B, int H_q,
                               int H_kv, int max_len, int d, float scale, int grid,
                               int *err_word, cudaStream_t stream, const int *seqlens_first) {
  if (grid <= 0 || !decode_units_fit(B, H_q, H_kv, max_len)) return cudaErrorInvalidValue;
  // head dims 32 and 96 run the 64- and 128-column kernels on zero-padded boxes
#define GQA_DECODE_BF16(D_, NSTG_, OD_)                                                      \
  launch_decode_d<D_, NSTG_, false, OD_>(tm_q, tm_k, tm_v, q, seqlens, o, lse, partials,       \
                                         counters, B, H_q, H_kv, max_len, scale, grid, err_word, \
                                         nullptr, nullptr, stream, seqlens_first)
  switch (d) {
    case 32: return GQA_DECODE_BF16(64, 8, 32);
    case 64: return GQA_DECODE_BF16(64, 8, 64);
    case 96: return GQA_DECODE_BF16(128, 5, 96);
    case 128: return GQA_DECODE_BF16(128, 5, 128);
    case 256: return GQA_DECODE_BF16(256, 4, 256);
    default: return cudaErrorInvalidValue;
  }
#undef GQA_DECODE_BF16
}

namespace {
template <bool kI8>
cudaError_t launch_decode_byte(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                               const CUtensorMap &tm_v, const void *q, const int *seqlens, void *o,
                               float *lse, float *partials, int *counters, int B, int H_q,
                               int H_kv, int max_len, int d, float scale, const float *k_scale,
                               const float *v_scale, int grid, int *err_word, cudaStream_t stream) {
  if (grid <= 0 || !decode_units_fit(B, H_q, H_kv, max_len)) return cudaErrorInvalidValue;
  // head dims 32 and 96 run the 64- and 128-column kernels on zero-padded boxes
#define GQA_DECODE_BYTE(D_, NSTG_, OD_)                                                       \
  launch_decode_d<D_, NSTG_, true, OD_, kI8>(tm_q, tm_k, tm_v, q, seqlens, o, lse, partials,    \
                                             counters, B, H_q, H_kv, max_len, scale, grid,      \
                                             err_word, k_scale, v_scale, stream)
  switch (d) {
    case 32: return GQA_DECODE_BYTE(64, 8, 32);
    case 64: return GQA_DECODE_BYTE(64, 8, 64);
    case 96: return GQA_DECODE_BYTE(128, 5, 96);
    case 128: return GQA_DECODE_BYTE(128, 5, 128);
    default: return cudaErrorInvalidValue;
  }
#undef GQA_DECODE_BYTE
}
}  // namespace

cudaError_t launch_decode_fp8(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, const void *q, const int *seqlens, void *o,
                              float *lse, float *partials, int *counters, int B, int H_q,
                              int H_kv, int max_len, int d, float scale, const float *k_scale,
                              const float *v_scale, int grid, int *err_word, cudaStream_t stream) {
  return launch_decode_byte<false>(tm_q, tm_k, tm_v, q, seqlens, o, lse, partials, counters, B, H_q,
                                   H_kv, max_len, d, scale, k_scale, v_scale, grid, err_word, stream);
}

cudaError_t launch_decode_int8(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                               const CUtensorMap &tm_v, const void *q, const int *seqlens, void *o,
                               float *lse, float *partials, int *counters, int B, int H_q,
                               int H_kv, int max_len, int d, float scale, const float *k_scale,
                               const float *v_scale, int grid, int *err_word, cudaStream_t stream) {
  return launch_decode_byte<true>(tm_q, tm_k, tm_v, q, seqlens, o, lse, partials, counters, B, H_q,
                                  H_kv, max_len, d, scale, k_scale, v_scale, grid, err_word, stream);
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
