// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stdint.h>

#ifdef __CUDACC__
#define GQA_HD __host__ __device__ __forceinline__
#else
#define GQA_HD inline
#endif

#ifdef __CUDACC__
#include <cuda_runtime.h>

#include <utility>
#endif

namespace gqa {

#ifdef __CUDACC__
// Launches `kernel` with programmatic stream serialisation: it may begin
// while the previous grid of the stream is finishing. The kernels launched
// this way call grid_dependency_wait() before reading anything earlier work
// may have written, so stream order is kept.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kernel)(KArgs...), int grid, int block, size_t smem,
                                cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same in thread-block clusters of `cluster` consecutive CTAs (grid a
// multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic_cluster(void (*kernel)(KArgs...), int grid, int block, size_t smem,
                                        int cluster, cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
#endif

// Bits of the device error word kept in each workspace.
constexpr int kErrTimeout = 1 << 0;
constexpr int kErrBadSeqlen = 1 << 1;

constexpr int kTileM = 128;  // query rows per tile
constexpr int kTileN = 128;  // key rows per K/V block
// Dense prefill units hold one query tile instead of two when pairs would
// number fewer than this (the SM count of a GB300).
constexpr int kSingleTileUnitsBelow = 148;

// ------------------------------------------------------------------------
// Persistent prefill schedule.
//
// A (b, h_kv) group owns g = H_q / H_kv query heads, each cut into
// n_qt = ceil(N_q / 128) query tiles. Within a group the g * n_qt tiles are
// listed heaviest first (q_tile descending -- later tiles see more keys
// under the causal mask -- and head ascending within one q_tile) and paired
// consecutively: a unit is two query tiles of the same group, so ONE stream
// of K/V blocks feeds both. When g is even the two tiles share their q_tile
// (identical causal extent). Units are numbered pair-rank-major across all
// groups, so unit order is heavy-first globally; an atomic counter hands
// them out (the persistent-kernel entry's global work queue, BootstrapAI
// evolution log).
// ------------------------------------------------------------------------
struct PrefillPlan {
  int B, H_q, H_kv, N_q, N_kv, causal;
  int group;           // g
  int n_qt, n_kt;      // query tiles per head, key blocks per head
  int tiles_per_group; // g * n_qt
  int tpu;             // query tiles per unit: 2, or 1 for problems too small to fill the GPU
  int pairs_per_group; // units per group: ceil(tiles_per_group / tpu)
  int total_units;     // B * H_kv * pairs_per_group
  int kv_offset;       // N_kv - N_q (bottom-right causal alignment)
};

struct UnitTile {
  int h_q, q_tile, kv_blocks;  // kv_blocks == 0 -> no tile
};

struct Unit {
  int b, h_kv;
  UnitTile t[2];
};

// single_tiles: one tile per unit whatever the size (head dim 256, where one
// tile's S and O fill the tensor memory).
GQA_HD PrefillPlan make_prefill_plan(int B, int H_q, int H_kv, int N_q, int N_kv, int causal,
                                     int single_tiles = 0) {
  PrefillPlan p;
  p.B = B; p.H_q = H_q; p.H_kv = H_kv; p.N_q = N_q; p.N_kv = N_kv; p.causal = causal ? 1 : 0;
  p.group = H_q / H_kv;
  p.n_qt = (N_q + kTileM - 1) / kTileM;
  p.n_kt = (N_kv + kTileN - 1) / kTileN;
  p.tiles_per_group = p.group * p.n_qt;
  // Two tiles per unit share every K/V block load; but when pairing leaves
  // fewer units than the GPU has SMs, single tiles run twice as many CTAs
  // (each SM then works on one tile at full speed instead of idling).
  const int pairs = (p.tiles_per_group + 1) / 2;
  p.tpu = (single_tiles || static_cast<long long>(B) * H_kv * pairs < kSingleTileUnitsBelow) ? 1 : 2;
  p.pairs_per_group = (p.tiles_per_group + p.tpu - 1) / p.tpu;
  p.total_units = B * H_kv * p.pairs_per_group;
  p.kv_offset = N_kv - N_q;
  return p;
}

// CTAs per cluster of the dense prefill: g / 2 when units pair the tiles of
// a group of 4 or 8 query heads (head dims up to 128; ranks c*m .. c*m+c-1
// are then the g tiles of one q_tile), else 1.
GQA_HD int cluster_size_for(const PrefillPlan &p, int d) {
  return (p.tpu == 2 && d <= 128 && (p.group == 4 || p.group == 8)) ? p.group / 2 : 1;
}

// Number of key blocks query tile `qt` must visit.
GQA_HD int kv_blocks_for_tile(const PrefillPlan &p, int qt) {
  if (!p.causal) return p.n_kt;
  int last_row = (qt + 1) * kTileM - 1;
  if (last_row > p.N_q - 1) last_row = p.N_q - 1;
  const int last_key = last_row + p.kv_offset;  // >= 0 because N_kv >= N_q
  int nb = last_key / kTileN + 1;
  return nb < p.n_kt ? nb : p.n_kt;
}

GQA_HD Unit decode_unit(const PrefillPlan &p, int u) {
  Unit w;
  const int groups = p.B * p.H_kv;
  const int rank = u / groups;
  const int bh = u - rank * groups;
  w.b = bh / p.H_kv;
  w.h_kv = bh - w.b * p.H_kv;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int f = p.tpu * rank + s;
    if (s < p.tpu && f < p.tiles_per_group) {
      const int qt = p.n_qt - 1 - f / p.group;
      w.t[s].h_q = w.h_kv * p.group + (f % p.group);
      w.t[s].q_tile = qt;
      w.t[s].kv_blocks = kv_blocks_for_tile(p, qt);
    } else {
      w.t[s].h_q = -1;
      w.t[s].q_tile = -1;
      w.t[s].kv_blocks = 0;
    }
  }
  return w;
}

// ------------------------------------------------------------------------
// Workspace: per (device, stream). Layout of the control block (ints):
//   [0] device error word   [1] work counter   [2] CTAs finished
//   [3] units listed by the ragged-batch plan kernel
// ------------------------------------------------------------------------
constexpr int kCtlErr = 0;
constexpr int kCtlWork = 1;
constexpr int kCtlDone = 2;
constexpr int kCtlVarlenUnits = 3;
constexpr int kCtlInts = 64;

struct Workspace {
  int *ctl = nullptr;        // kCtlInts ints, zeroed at creation
  float *partials = nullptr; // split-KV decode partials
  size_t partials_bytes = 0;
  int *counters = nullptr;   // split-KV decode: splits finished per (b, h_kv); re-armed by the kernel
  size_t counters_len = 0;
  int4 *units = nullptr;     // ragged-batch prefill: the plan kernel's unit list
  size_t units_len = 0;
};

// ------------------------------------------------------------------------
// Ragged-batch (varlen) prefill. B sequences packed token-major:
// q / o [total_q][H_q][d] and k / v [total_k][H_kv][d]; sequence b owns the
// query tokens [cu_q[b], cu_q[b+1]) and the key tokens [cu_k[b], cu_k[b+1]),
// causal alignment bottom-right within each sequence. A one-block plan
// kernel checks the offsets and lists the units -- (b, h_kv, pair of query
// tiles), the tiles of each sequence paired heaviest first as in the dense
// schedule -- sorted by key blocks, most first; the persistent kernel's
// producer takes units from that list through the atomic counter.
// ------------------------------------------------------------------------
constexpr int kVarlenMaxB = 4096;       // sequences per call
constexpr int kVarlenMaxBlocks = 4096;  // 128-row key blocks per sequence

struct VarlenArgs {
  const int *cu_q, *cu_k;  // device int32 [B + 1]; null: every sequence has uni_q / uni_k rows
  const int4 *units;       // the plan kernel's list: {b, h_kv, pair, key blocks}
  int B, H_q, H_kv, group, causal, total_q, total_k;
  int uni_q, uni_k;        // the lengths when cu_q / cu_k are null ([B][N][H][d] batches)
  int tpu;                 // query tiles per listed unit: 2, or 1 at head dim 256
};

// First row of sequence b: from the offsets, or b * n for equal lengths.
GQA_HD int varlen_start(const int *cu, int n, int b) {
#ifdef __CUDA_ARCH__
  return cu ? __ldg(cu + b) : b * n;
#else
  return cu ? cu[b] : b * n;
#endif
}

// Units a call can list at most (workspace sizing): every sequence's query
// tiles, paired (tpu = 2) or one by one (tpu = 1), for each K/V head.
GQA_HD long long varlen_max_units(int B, int H_q, int H_kv, long long total_q, int tpu = 2) {
  const long long group = H_q / H_kv;
  const long long tiles = total_q / kTileM + B;  // sum over b of ceil(len_q / 128)
  if (tpu == 1) return static_cast<long long>(H_kv) * group * tiles;
  return static_cast<long long>(H_kv) * ((group * tiles + B) / 2 + B);
}

// Key blocks query tile qt of a sequence (len_q, len_k) visits.
GQA_HD int varlen_kv_blocks(int len_q, int len_k, int causal, int qt) {
  const int n_kt = (len_k + kTileN - 1) / kTileN;
  if (!causal) return n_kt;
  int last_row = (qt + 1) * kTileM - 1;
  if (last_row > len_q - 1) last_row = len_q - 1;
  const int nb = (last_row + len_k - len_q) / kTileN + 1;  // len_k >= len_q: never negative
  return nb < n_kt ? nb : n_kt;
}

// Where the prefill kernels write O: strides in elements (batch, head, row;
// for ragged batches `sn` is the token stride and `sb` unused) and the head
// dim d, the columns stored (the kernel's D may pad it with zero columns).
struct OutView {
  long long sb, sh, sn;
  int d;
  int tma4;  // dense prefill: q/k/v tensor maps are 4-D (column, row, head, batch)
};

// Launchers (return a cudaError_t; arguments already validated).
// lse: optional per-row log-sum-exp output (null: not written). For the
// dense prefill tm_q, tm_k, tm_v are 4-D maps (column, row, head, batch)
// with 64-column x 128-row boxes.
cudaError_t launch_prefill_tc(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, void *o, const OutView &ov, float *lse,
                              const PrefillPlan &plan, float scale, int *ctl, int num_sms,
                              cudaStream_t stream);

// The varlen plan kernel (one block) writes the unit list to `units` and its
// length to ctl[kCtlVarlenUnits]; bad offsets set kErrBadSeqlen in
// ctl[kCtlErr] and the sequence is left out. The prefill kernel then reads
// q, k, v through THD tensor maps: [total][H][d] with 128-token boxes.
cudaError_t launch_varlen_plan(const VarlenArgs &va, int4 *units, int *ctl, cudaStream_t stream);
cudaError_t launch_prefill_tc_varlen(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                     const CUtensorMap &tm_v, void *o, const OutView &ov,
                                     float *lse, const VarlenArgs &va, float scale, int *ctl,
                                     int num_sms, cudaStream_t stream);

cudaError_t launch_attn_f32(const float *q, const float *k, const float *v, float *o, int B,
                            int H_q, int H_kv, int N_q, int N_kv, int d, int causal, float scale,
                            const int *seqlens, int kv_row_capacity, int *err_word,
                            cudaStream_t stream);

// Decode: the valid cache rows are cut into 64-row units (one TMA box; 32
// rows at head dim 256) and balanced over a persistent grid; a CTA's run
// over part of a (b, h_kv, head group) plane leaves a partial result merged
// in the same launch.
constexpr int kDecodeChunkUnit = 64;    // rows per unit (the TMA box height)
constexpr int kDecodeMinUnit = 32;      // the smallest unit (head dim 256)
// Rows of the K/V TMA box (= rows per unit) of a bf16 cache at head dim d.
GQA_HD int decode_box_rows(int d) { return d == 256 ? kDecodeMinUnit : kDecodeChunkUnit; }
constexpr int kDecodeHeads = 16;        // query heads per plane (the Q box height)
constexpr int kDecodeChunkMax = 2048;   // largest rows-per-CTA sizing hint
int decode_head_groups(int H_q, int H_kv);                     // query heads per K/V head / 16, rounded up
size_t decode_planes(int B, int H_q, int H_kv);                // merge counters needed
size_t decode_partials_bytes(int B, int H_q, int H_kv, int d, int grid);
// CTAs to launch: `chunk` > 0 sizes the grid as (upper bound of rows) / chunk;
// 0 gives one wave of resident CTAs.
int decode_grid(int B, int H_q, int H_kv, int max_len, int d, int num_sms, int chunk);
// False when the unit count of the largest case would not fit the kernel's
// 32-bit unit indices.
bool decode_units_fit(int B, int H_q, int H_kv, int max_len);
// tm_q views q as [1][B * H_q][d] with 16-row boxes; tm_k / tm_v view the
// caches as [B * H_kv][max_len][d] with 64-row boxes. seqlens_first: the
// lengths read before the grid-dependency wait to start early (null: the
// same array as seqlens; anything else only in the self-test).
cudaError_t launch_decode_bf16(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                               const CUtensorMap &tm_v, const void *q, const int *seqlens, void *o,
                               float *lse, float *partials, int *counters, int B, int H_q,
                               int H_kv, int max_len, int d, float scale, int grid,
                               int *err_word, cudaStream_t stream,
                               const int *seqlens_first = nullptr);

// The same decode over a one-byte cache, fp8 (e4m3) or int8 codes: tm_k /
// tm_v view the caches as [B * H_kv][max_len][d] bytes with boxes of 64 (d
// <= 64) or 128 bytes x 128 rows (kDecodeByteUnit), swizzled by the box
// width; k_scale / v_scale are the per-K/V-head dequantisation scales
// (device fp32 [H_kv]).
constexpr int kDecodeByteUnit = 128;
cudaError_t launch_decode_fp8(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                              const CUtensorMap &tm_v, const void *q, const int *seqlens, void *o,
                              float *lse, float *partials, int *counters, int B, int H_q,
                              int H_kv, int max_len, int d, float scale, const float *k_scale,
                              const float *v_scale, int grid, int *err_word, cudaStream_t stream);
cudaError_t launch_decode_int8(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                               const CUtensorMap &tm_v, const void *q, const int *seqlens, void *o,
                               float *lse, float *partials, int *counters, int B, int H_q,
                               int H_kv, int max_len, int d, float scale, const float *k_scale,
                               const float *v_scale, int grid, int *err_word, cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(int timeout_us, int *err_word, cudaStream_t stream);

// Attention backward: workspace floats for the per-row lse (log2 units) and
// D = rowsum(dO * O), both padded to whole 128-row query tiles; tm_q / tm_do
// view q / dO as [B*H_q][N_q][d], tm_k / tm_v view k / v as
// [B*H_kv][N_kv][d], all with 128-row boxes.
size_t bwd_workspace_bytes(int B, int H_q, int N_q);
cudaError_t launch_attn_bwd(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                            const CUtensorMap &tm_v, const CUtensorMap &tm_do, const void *o,
                            const void *dout, const float *lse, float *work, void *dq, void *dk,
                            void *dv, int B, int H_q, int H_kv, int N_q, int N_kv, int d,
                            int causal, float scale, int num_sms, int *err_word,
                            cudaStream_t stream);

// bf16 tensor viewed as [planes][rows][d] for TMA: boxes of 64 columns x
// box_rows rows, 128-byte swizzle, zero fill outside. False on failure.
bool encode_tensor_map_bf16_3d(CUtensorMap *map, const void *base, int d, long rows, long planes,
                               int box_rows);
// bf16 tensor [tokens][heads][d] (token-major) for TMA: boxes of 64 columns
// x 1 head x box_rows tokens, laid out in shared memory like a box_rows-row
// tile of the [planes][rows][d] view. False on failure.
bool encode_tensor_map_bf16_thd(CUtensorMap *map, const void *base, int d, long heads,
                                long tokens, int box_rows);

}  // namespace gqa
