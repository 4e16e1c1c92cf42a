/*
 * gqa_attn.h -- C ABI of the GB300 (sm_103a) grouped-query attention library.
 *
 * Operation (both forms):  O = softmax(scale * Q K^T [+ causal mask]) V,
 * where query head h_q reads K/V head h_kv = h_q / (H_q / H_kv). With
 * H_kv == H_q this is multi-head attention, with H_kv == 1 multi-query
 * attention, anything in between grouped-query attention.
 *   - Head mapping and the MHA/GQA/MQA unification: BootstrapAI evolution log,
 *     collab-014 "Kernel 9 GQA".
 *   - Prefill is compute-bound, single-token decode against a K/V cache is
 *     memory-bound: kaispace.site, the "prefill vs decode / chunked prefill"
 *     note; cached GQA decode with per-row lengths and a bf16 cache:
 *     microLLM-rocm optimisation log, Experiments 064-065.
 *   - Split-sequence decode with a merge of partial results: microLLM-rocm
 *     optimisation log, Experiments 282-284.
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers to contiguous row-major arrays
 *     owned by the caller, at least 16-byte aligned. The library never frees,
 *     retains or reallocates them.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream):
 *     outputs are valid once the stream has synchronised.
 *   - Precision: the unsuffixed entry points take bf16 inputs, accumulate in
 *     fp32 on the tensor cores (prefill) or CUDA cores (decode), and write
 *     bf16 output. The `_f32` siblings take and write fp32 with fp32 math
 *     throughout (no TF32).
 *   - Causal alignment is bottom-right: query row i sees key j iff
 *     j <= i + (N_kv - N_q) (per sequence for ragged batches). With
 *     N_q == N_kv this is the ordinary lower triangle. causal with
 *     N_q > N_kv is rejected (GQA_ERR_UNSUPPORTED).
 *   - `scale` is used as given (typically 1/sqrt(d)); it must be finite.
 *   - The library owns a small per-(device, stream) workspace (the scheduler
 *     counters, the device error word, the split-KV partials and the
 *     ragged-batch unit list). It grows
 *     on demand with stream-ordered allocation and is released by
 *     gqa_attn_shutdown(). Calls on DIFFERENT streams use different
 *     workspaces and may run concurrently.
 *   - Errors are returned as a gqa_status code before anything is launched;
 *     nothing is launched when a call fails validation. Faults detected on
 *     the device (a bounded wait that ran out, a seqlen outside
 *     [0, max_len], bad ragged-batch offsets) are recorded in the
 *     workspace's error word and reported
 *     by gqa_attn_get_device_error(). No kernel traps or asserts.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gqa_status {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARG = 1,    /* dims <= 0, H_q % H_kv != 0, non-finite scale,
                                   null or misaligned pointer */
    GQA_ERR_UNSUPPORTED = 2,    /* head dim not supported by the call; causal with N_q > N_kv;
                                   a size beyond the documented limits */
    GQA_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
    GQA_ERR_DEVICE_TIMEOUT = 4, /* a bounded device-side wait ran out */
    GQA_ERR_OOM = 5,            /* the workspace could not be grown */
    GQA_ERR_BAD_SEQLEN = 6      /* the device saw seqlens[b] < 0 or > max_len */
} gqa_status;

/*
 * Prefill attention, bf16 in / bf16 out, fp32 accumulation (tcgen05 tensor
 * cores, TMEM accumulators, TMA-staged tiles, persistent tile scheduler).
 *   q : [B][H_q][N_q][d]  bf16      k, v : [B][H_kv][N_kv][d]  bf16
 *   o : [B][H_q][N_q][d]  bf16 (written)
 *   d in {32, 64, 96, 128, 256} (32 and 96 run the 64- and 128-column
 *   kernels on tiles the TMA pads with zero columns; at 256 one query
 *   tile's S and O fill the tensor memory, so each CTA works on one tile
 *   at a time); 1 <= B*H_q*N_q*d < 2^31 elements per tensor.
 * Pages: BootstrapAI evolution log, collab-014 "Kernel 9 GQA" (semantics),
 * and the persistent-kernel entry (atomic work counter over tiles).
 */
int gqa_attn_fwd(const void *q, const void *k, const void *v, void *o,
                 int B, int H_q, int H_kv, int N_q, int N_kv, int d,
                 int causal, float scale, cudaStream_t stream);

/*
 * gqa_attn_fwd that also returns each query row's log-sum-exp,
 *   lse[b][h_q][i] = ln( sum_j exp(scale * q_i . k_j) )  over the visible keys,
 * as fp32 [B][H_q][N_q] (device pointer, 4-byte aligned, caller-owned). It
 * lets a caller merge this result with attention over other keys
 * (O = sum_p exp(lse_p - M) O_p / sum_p exp(lse_p - M), M = max_p lse_p).
 * All other arguments, layouts and errors as gqa_attn_fwd.
 * Pages: microLLM-rocm optimisation log, Experiments 282-284 (split-sequence
 * attention carries each part's (max, sum) to a log-sum-exp merge).
 */
int gqa_attn_fwd_lse(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int H_q, int H_kv, int N_q, int N_kv, int d,
                     int causal, float scale, cudaStream_t stream);

/*
 * gqa_attn_fwd on tensors with arbitrary batch, head and row strides, so a
 * view needs no copy (for example q, k and v sliced out of a fused QKV
 * projection's [B][N][H_q + 2 H_kv][d] output, or a [B][N][H][d] layout).
 * Element (b, h, i, c) of q is at q + b*q_sb + h*q_sh + i*q_sn + c; the same
 * for k, v (head index h_kv, row j) and o. Strides are in elements, the head
 * dim is contiguous; every stride must be a positive multiple of 8 (16
 * bytes, a rule of the TMA tensor maps) and each row stride at least d. o
 * must not overlap q, k or v. d in {32, 64, 96, 128, 256}; everything else
 * as gqa_attn_fwd (which is this call with the packed strides).
 * Pages: microLLM-rocm optimisation log, Experiments 202-206 (attention on
 * the token-major BTHD layout without strided copies).
 */
int gqa_attn_fwd_strided(const void *q, long long q_sb, long long q_sh, long long q_sn,
                         const void *k, long long k_sb, long long k_sh, long long k_sn,
                         const void *v, long long v_sb, long long v_sh, long long v_sn,
                         void *o, long long o_sb, long long o_sh, long long o_sn,
                         int B, int H_q, int H_kv, int N_q, int N_kv, int d,
                         int causal, float scale, cudaStream_t stream);

/*
 * Ragged-batch ("varlen") prefill: B sequences of different lengths packed
 * token-major, one call. bf16 in / bf16 out, fp32 accumulation, same kernel
 * design as gqa_attn_fwd.
 *   q : [total_q][H_q][d]  bf16     k, v : [total_k][H_kv][d]  bf16
 *   o : [total_q][H_q][d]  bf16 (written for every token some sequence owns)
 *   cu_seqlens_q, cu_seqlens_k : device int32 [B + 1], 4-byte aligned:
 *       sequence b owns query tokens [cu_seqlens_q[b], cu_seqlens_q[b+1])
 *       and key tokens [cu_seqlens_k[b], cu_seqlens_k[b+1]).
 *   Causal alignment is bottom-right inside each sequence: its query row i
 *   sees its key j iff j <= i + (len_k - len_q).
 *   d in {32, 64, 96, 128, 256} (at 256 each work unit holds one query
 *   tile instead of two); 1 <= B <= 4096; each of total_q*H_q*d,
 *   total_k*H_kv*d below 2^31; at most 4096 blocks of 128 keys per sequence.
 * The offsets live on the device, so the library checks them there: a
 * sequence whose offsets are decreasing, outside [0, total], with keys
 * missing (len_q > 0 with len_k == 0, or len_k < len_q when causal) or longer
 * than the key limit is skipped (its o rows are left as they were) and
 * GQA_ERR_BAD_SEQLEN is recorded (gqa_attn_get_device_error). total_q == 0
 * returns GQA_OK without launching. Two kernels are launched: a one-block
 * plan (lists the work units, heaviest first) and the prefill kernel.
 * Pages: microLLM-rocm optimisation log, Experiment 101 (prompts batched
 * into one prefill) and Experiment 062 (prefill into the cache);
 * BootstrapAI evolution log, collab-014 "Kernel 9 GQA" (semantics).
 */
int gqa_attn_fwd_varlen(const void *q, const void *k, const void *v, void *o,
                        const int *cu_seqlens_q, const int *cu_seqlens_k,
                        int B, int H_q, int H_kv, int total_q, int total_k, int d,
                        int causal, float scale, cudaStream_t stream);

/*
 * gqa_attn_fwd_varlen that also returns each query row's log-sum-exp as
 * fp32 [H_q][total_q] (lse[h][t] for the token t of head h; device pointer,
 * 4-byte aligned, caller-owned). Everything else as gqa_attn_fwd_varlen.
 */
int gqa_attn_fwd_varlen_lse(const void *q, const void *k, const void *v, void *o, float *lse,
                            const int *cu_seqlens_q, const int *cu_seqlens_k,
                            int B, int H_q, int H_kv, int total_q, int total_k, int d,
                            int causal, float scale, cudaStream_t stream);

/*
 * gqa_attn_fwd for token-major batches: q, o are [B][N_q][H_q][d] and k, v
 * [B][N_kv][H_kv][d] bf16 (the layout of a fused QKV projection's output).
 * It is the ragged-batch path with every sequence of length N_q / N_kv (no
 * offset arrays), so it launches the same two kernels as
 * gqa_attn_fwd_varlen. B <= 4096; causal with N_q > N_kv is rejected
 * (GQA_ERR_UNSUPPORTED); everything else as gqa_attn_fwd.
 */
int gqa_attn_fwd_bshd(const void *q, const void *k, const void *v, void *o,
                      int B, int H_q, int H_kv, int N_q, int N_kv, int d,
                      int causal, float scale, cudaStream_t stream);

/*
 * Same operation in fp32: q, k, v, o are float arrays with the layouts of
 * gqa_attn_fwd. SIMT FMA kernel (online softmax, warp-shuffle reductions);
 * d in {32, 64, 96, 128}.
 * Pages: BootstrapAI evolution log, collab-005 "Kernel 2 tiling" (online
 * softmax over key tiles) and collab-014 "Kernel 9 GQA".
 */
int gqa_attn_fwd_f32(const void *q, const void *k, const void *v, void *o,
                     int B, int H_q, int H_kv, int N_q, int N_kv, int d,
                     int causal, float scale, cudaStream_t stream);

/*
 * Single-token decode against a bf16 K/V cache: persistent split-KV with the
 * log-sum-exp merge of the splits in the same launch; bf16 output, fp32
 * math.
 *   q       : [B][H_q][d] bf16         o : [B][H_q][d] bf16 (written)
 *   k_cache, v_cache : [B][H_kv][max_len][d] bf16; rows [0, seqlens[b]) are
 *             valid, later rows are never read into the result
 *   seqlens : [B] int32 on the device, each in [0, max_len]; a sequence of
 *             length 0 yields O = 0. Out-of-range values make the call
 *             record GQA_ERR_BAD_SEQLEN (read with gqa_attn_get_device_error)
 *             and leave that sequence's output at 0.
 *   d in {32, 64, 96, 128, 256} (32 and 96 run the 64- and 128-column
 *   kernels on tiles the TMA pads with zero columns; at 256 two warps share
 *   each 16-row group of a 32-row unit, 128 columns each); max_len <= 1 << 20;
 *   at most 2^30 row units (B * H_kv * ceil(H_q / H_kv / 16) *
 *   ceil(max_len / 32)), else GQA_ERR_UNSUPPORTED.
 * Pages: microLLM-rocm optimisation log, Experiments 064-065 (batched cached
 * GQA decode, bf16 cache with fp32 accumulation) and 282-284 (split-sequence
 * cached attention).
 */
int gqa_attn_decode(const void *q, const void *k_cache, const void *v_cache,
                    const int *seqlens, void *o,
                    int B, int H_q, int H_kv, int max_len, int d,
                    float scale, cudaStream_t stream);

/*
 * gqa_attn_decode that also returns each query head's log-sum-exp,
 *   lse[b][h_q] = ln( sum_{j < seqlens[b]} exp(scale * q . k_j) ),
 * as fp32 [B][H_q] (device pointer, 4-byte aligned, caller-owned); -inf for
 * a sequence with no rows. Other arguments as gqa_attn_decode.
 * Pages: microLLM-rocm optimisation log, Experiments 282-284.
 */
int gqa_attn_decode_lse(const void *q, const void *k_cache, const void *v_cache,
                        const int *seqlens, void *o, float *lse,
                        int B, int H_q, int H_kv, int max_len, int d,
                        float scale, cudaStream_t stream);

/*
 * gqa_attn_decode with an explicit work split. The valid cache rows are
 * cut into 64-row units and balanced over a grid of CTAs; `chunk_tokens`
 * (a multiple of 64 in [64, 2048]) sizes that grid as
 * ceil(B * H_kv * ceil(g / 16) * max_len / chunk_tokens) CTAs, g = H_q / H_kv,
 * so smaller values split each sequence into more partial results. 0 picks
 * one wave of resident CTAs (the default). The result is the same operation
 * for every value, up to fp32 rounding. Other values: GQA_ERR_INVALID_ARG.
 */
int gqa_attn_decode_chunked(const void *q, const void *k_cache,
                            const void *v_cache, const int *seqlens, void *o,
                            int B, int H_q, int H_kv, int max_len, int d,
                            float scale, int chunk_tokens, cudaStream_t stream);

/*
 * Decode against an fp8 K/V cache: the cache holds OCP FP8 E4M3 values
 * (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest 448, codes
 * 0x7F / 0xFF are NaN, no infinities), one byte each, and the value a byte
 * stands for is its e4m3 value times the scale of its K/V head:
 *   K[b][h][j][c] = e4m3(k_cache[b][h][j][c]) * k_scale[h]   (likewise V)
 *   q       : [B][H_q][d] bf16         o : [B][H_q][d] bf16 (written)
 *   k_cache, v_cache : [B][H_kv][max_len][d] bytes (16-byte aligned)
 *   k_scale, v_scale : device fp32 [H_kv], 4-byte aligned, finite
 *   seqlens : as gqa_attn_decode (rows [0, seqlens[b]) are valid; later rows
 *             are never used, whatever their bytes)
 *   lse     : optional fp32 [B][H_q] log-sum-exp as gqa_attn_decode_lse, or
 *             NULL
 * Same kernel design as gqa_attn_decode (persistent split-KV with the merge
 * in the same launch), streaming half the cache bytes: units of 128 rows;
 * each MMA warp widens its rows of K to bf16 (Q K^T on bf16 pairs, exact
 * widening) and of V to f16 (P V on f16 pairs, exact widening), fp32
 * accumulation; k_scale multiplies the exponent scale, v_scale the output.
 * d in {32, 64, 96, 128} (32 and 96 run the 64- and 128-column kernels on
 * boxes that read zeros past d); limits and errors as gqa_attn_decode.
 * Pages: microLLM-rocm optimisation log, Experiment 065 (the K/V cache
 * stored narrower than fp32 with fp32 accumulation) and Experiments 354 and
 * 359 (an 8-bit cache read fused into decode attention).
 */
int gqa_attn_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                        const float *k_scale, const float *v_scale, const int *seqlens,
                        void *o, float *lse,
                        int B, int H_q, int H_kv, int max_len, int d,
                        float scale, cudaStream_t stream);

/*
 * Decode against an int8 K/V cache: the cache holds one-byte two's-complement
 * codes (-128 .. 127), and the value a byte stands for is its integer times
 * the scale of its K/V head:
 *   K[b][h][j][c] = int8(k_cache[b][h][j][c]) * k_scale[h]   (likewise V)
 * Arguments, layouts, limits and errors as gqa_attn_decode_fp8 (k_cache,
 * v_cache: [B][H_kv][max_len][d] bytes, 16-byte aligned; d in {32, 64, 96,
 * 128}). Same kernel as the fp8 cache; each MMA warp widens its rows
 * exactly: the byte, sign bit flipped, becomes the low mantissa bits of the
 * f16 1024, minus 1152 (K then to bf16, V kept in f16).
 * Pages: microLLM-rocm optimisation log, Experiments 352 and 354 (a
 * one-byte tensor with an explicit scale, read and widened inside the
 * decode kernel) and Experiment 065 (the K/V cache narrower than the
 * arithmetic).
 */
int gqa_attn_decode_int8(const void *q, const void *k_cache, const void *v_cache,
                         const float *k_scale, const float *v_scale, const int *seqlens,
                         void *o, float *lse,
                         int B, int H_q, int H_kv, int max_len, int d,
                         float scale, cudaStream_t stream);

/*
 * Decode in fp32 (q, caches and o are float arrays, layouts as
 * gqa_attn_decode); d in {32, 64, 96, 128}.
 */
int gqa_attn_decode_f32(const void *q, const void *k_cache, const void *v_cache,
                        const int *seqlens, void *o,
                        int B, int H_q, int H_kv, int max_len, int d,
                        float scale, cudaStream_t stream);

/*
 * gqa_attn_decode for callers that must not allocate device memory. The
 * pages describe no counterpart: this is a deployment variant of the same
 * operation. gqa_attn_decode grows a per-stream workspace with
 * cudaMallocAsync; a serving loop confined to a pre-reserved memory budget,
 * a latency-critical path where an allocation may synchronise the device, or
 * a process whose device memory belongs to another allocator cannot allow
 * that. This entry point calls no allocation routine: its scratch (split
 * partials and merge counters) is a fixed 4 MiB + 64 KiB array in the
 * library's own device memory, present on every GPU that loads the library
 * until the process exits.
 *   - Arguments, layouts and results as gqa_attn_decode (same kernel), with
 *     the grid trimmed so the partials fit: (grid + P) * 16 * (D + 2) * 4
 *     bytes <= 4 MiB, where P = B * H_kv * ceil(H_q / H_kv / 16) <= 16384
 *     and D is the kernel's head dim (64 for d <= 64, 128 for d <= 128,
 *     else 256).
 *     Larger problems return GQA_ERR_UNSUPPORTED (use gqa_attn_decode).
 *   - The first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call uses the same array and clears the parts that must start at
 *     zero; calls that overlap on the GPU (different streams, or different
 *     host threads) race on it and must be serialised by the caller.
 *   - Sequences whose seqlens entry is outside [0, max_len] get O = 0. This
 *     entry point does not report device-side errors: its error word lives
 *     in the scratch array and is cleared on every call, and
 *     gqa_attn_get_device_error() reads the per-stream workspaces of the
 *     other entry points, not this array. A bounded wait that ran out here
 *     (which leaves O incomplete) is therefore not reported either.
 */
int gqa_attn_decode_noalloc(const void *q, const void *k_cache,
                            const void *v_cache, const int *seqlens, void *o,
                            int B, int H_q, int H_kv, int max_len, int d,
                            float scale, cudaStream_t stream);

/*
 * Attention backward (bf16 in / bf16 out, fp32 accumulation on the tensor
 * cores): the gradients of O = softmax(scale Q K^T [+ causal mask]) V with
 * respect to q, k and v, given dO = dL/dO.
 *   q, o, dout, dq : [B][H_q][N_q][d] bf16     k, v, dk, dv : [B][H_kv][N_kv][d] bf16
 *   lse : fp32 [B][H_q][N_q], the per-row log-sum-exp that gqa_attn_fwd_lse
 *         returned with o for the same q, k, v, causal and scale (device
 *         pointer, 4-byte aligned).
 *   dq, dk, dv are written in full (every element), and must not overlap
 *   the inputs. dK and dV of a K/V head are the sums over the H_q / H_kv
 *   query heads that read it (the GQA reduction), accumulated in a fixed
 *   order: the result is deterministic for a given input.
 *   Causal alignment, size limits and errors as gqa_attn_fwd; d in {32, 64,
 *   96, 128} (32 and 96 run the 64- and 128-column kernels on tiles the TMA
 *   pads with zero columns).
 * Three kernels are launched: a small one for D_i = sum_c dO_ic O_ic and
 * the lse in log2 units (kept in the stream's workspace), then one grid of
 * dK/dV units (per K/V head and 128-key block, looping over the group's
 * query heads) and dQ units (per query head and 128-row tile).
 * Pages: microLLM-rocm optimisation log, Experiments 051-057 (causal GQA
 * attention backward: row recompute, softmax backward, dK/dV reduction over
 * the query heads of a group).
 */
int gqa_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                 const void *dout, const float *lse, void *dq, void *dk, void *dv,
                 int B, int H_q, int H_kv, int N_q, int N_kv, int d,
                 int causal, float scale, cudaStream_t stream);

/* Human-readable text for a gqa_status (never NULL; static storage). For
 * GQA_ERR_CUDA it includes the last CUDA error name seen by this thread. */
const char *gqa_attn_status_string(int status);

/*
 * Synchronises `stream`, reads and clears the device error word of that
 * stream's workspace on the current device, and returns GQA_OK,
 * GQA_ERR_DEVICE_TIMEOUT or GQA_ERR_BAD_SEQLEN (timeout wins when both are
 * set), or GQA_ERR_CUDA if the synchronisation itself failed.
 */
int gqa_attn_get_device_error(cudaStream_t stream);

/*
 * Work plan of the persistent prefill scheduler, for inspection and tests
 * (host only, no CUDA call). A unit is the pair of 128-row query tiles that
 * one CTA processes against one K/V stream. Units are handed out by an
 * atomic counter in index order; units with more visible key blocks come
 * first (heavy-first causal order).
 * This is the plan for head dims up to 128 (at 256 every unit is one tile).
 * Returns the number of units, or -1 for invalid sizes. When `unit` is in
 * range, writes out[0..7] = {b, h_kv, h_q0, q_tile0, kv_blocks0,
 * h_q1, q_tile1, kv_blocks1}; the second tile has kv_blocks1 == 0 (and
 * h_q1 = q_tile1 = -1) when the unit holds only one tile.
 */
int gqa_attn_prefill_plan(int B, int H_q, int H_kv, int N_q, int N_kv,
                          int causal, int unit, int *out);

/*
 * Failure-detection self-test: launches a kernel that waits on an mbarrier
 * nobody arrives at, with a limit of `timeout_us` microseconds (1..100000),
 * then returns the result of gqa_attn_get_device_error(stream), which is
 * GQA_ERR_DEVICE_TIMEOUT when the bounded wait works. Nothing else runs in
 * that kernel, so the context stays usable.
 */
int gqa_attn_selftest_wait_timeout(int timeout_us, cudaStream_t stream);

/*
 * Self-test of the decode's early start: gqa_attn_decode_lse, except that
 * the lengths the kernel reads before its grid-dependency wait (to locate
 * each CTA's first unit and prefetch it into L2 while the previous grid
 * finishes) come from `seqlens_early` (device int32 [B], 4-byte aligned)
 * instead of `seqlens`. In normal use both reads see the same array; a
 * preceding kernel that is still writing the lengths makes them differ, and
 * then the start is worked out again from `seqlens`. With a decoy here the
 * outputs must equal gqa_attn_decode_lse's for `seqlens`, bit for bit.
 * Errors as gqa_attn_decode_lse, plus GQA_ERR_INVALID_ARG for a null or
 * misaligned `seqlens_early`.
 */
int gqa_attn_selftest_decode_early_lengths(const void *q, const void *k_cache,
                                           const void *v_cache, const int *seqlens,
                                           const int *seqlens_early, void *o, float *lse,
                                           int B, int H_q, int H_kv, int max_len, int d,
                                           float scale, cudaStream_t stream);

/* Frees every library-owned workspace on every device (synchronising the
 * streams they belong to first). Safe to call more than once. */
void gqa_attn_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
