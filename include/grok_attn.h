/*
 * grok_attn.h - C ABI of the GB300 (sm_103a) Grok-1 grouped-query attention core.
 *
 * The operation is the self-attention core of Grok-1 as quoted in the Grok-1
 * code-reading guide (yingwang.github.io/grok-1/):
 *   ch. 4 "model.py close reading I: RMSNorm, RoPE, GQA Attention"
 *     §4.3 / §4.3.1  rotate_half and RotaryEmbedding (RoPE, base 10000, NeoX pairing)
 *     §4.4           RoPE on K and Q before the KV-cache write; update_into; memory mask
 *     §4.5.2         GQA: 48 query heads, 8 KV heads, query head h uses KV head h / 6;
 *                    logits * attn_output_multiplier (1/sqrt(128)); 30 * tanh(x / 30)
 *     §4.5.3         where(mask, logits, -1e30); softmax over keys in fp32
 *     §4.5.4         weighted sum of V, heads flattened in order h = 6 g + r
 *   ch. 6 "model.py close reading II"
 *     §6.4.2         causal (tril) x key-padding mask; decode masks through the memory mask
 *     §6.6 / §6.6.1  KVMemory(k, v, step): caches [B, Tmax, 8, 128] bf16, per-sequence step;
 *                    continuous batching (a new request takes a finished sequence's slot)
 *     §6.6.2         paged KV cache (pages allocated only when used)
 *
 * Calls by group:
 *   attention core      grok_rope_kv_append, grok_rope_kv_append_table, grok_rope_cos_sin,
 *                       grok_attn_prefill,
 *                       grok_attn_prefill_workspace(_min), grok_attn_prefill_ws,
 *                       grok_attn_decode_workspace, grok_attn_decode, grok_attn_combine,
 *                       grok_attn_decode_step_static, grok_attn_decode_step(_workspace)
 *   projections         grok_qkv_project, grok_linear, grok_dequant_int8,
 *                       grok_linear_int8(_workspace), grok_qkv_workspace, grok_qkv_rope_append,
 *                       grok_qkv_rope_append_table
 *   runtime             grok_prefill_pipe_create / _submit / _wait / _destroy
 *   paged cache         grok_rope_kv_append_paged, grok_attn_prefill_paged, grok_attn_prefill_ws_paged,
 *                       grok_attn_decode_paged, grok_qkv_rope_append_paged
 *   continuous batching grok_kv_insert_slot
 *   diagnostics         grok_abi_version, grok_last_error, grok_selftest_bounded_wait
 *
 * Conventions for every call:
 *   - bf16 tensors are passed as grok_bf16 (uint16_t storage), row-major with the
 *     innermost dimension contiguous and no padding:
 *       q, q_rot, out  [B, T, 48, 128]      k, v  [B, T, 8, 128]
 *       cache_k/v      [B, Tmax, 8, 128]
 *   - every pointer argument is a DEVICE pointer owned by the caller (except
 *     the host buffers of the prefill pipeline); the library never frees or
 *     retains caller memory, and every pointer to a bf16 tensor must be 16-byte
 *     aligned (32-byte for the outputs of the projection, Linear and dequant
 *     calls below, which are written with 32-byte stores).
 *   - no call allocates device memory except grok_prefill_pipe_create, which
 *     allocates the pipeline's buffers once (freed by grok_prefill_pipe_destroy).
 *     Scratch space is a caller-owned workspace whose size a *_workspace call
 *     gives, or, for grok_attn_decode_step_static, a static array of the library.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream); every call
 *     is asynchronous on it and returns after enqueueing its kernels.
 *   - errors found on the host (null or misaligned pointers, bad sizes) return
 *     GROK_ERR_INVALID_ARG before anything is launched; a failed CUDA call or
 *     launch returns GROK_ERR_CUDA, or GROK_ERR_DEVICE_FAULT when the error is
 *     a sticky one that has left the CUDA context unusable (an earlier kernel's
 *     illegal address, say: every later call then reports it).
 *     grok_last_error() then describes it (thread-local).
 *   - errors that depend on device data (positions, lengths) or a bounded wait
 *     that gave up are OR-ed into *dev_status (a device int32 the caller zeroes;
 *     NULL disables reporting) as GROK_DEV_* bits. The kernels never trap or
 *     hang; a sequence whose integers are invalid is skipped (its outputs and
 *     cache rows are left untouched).
 *   - positions must stay below GROK_MAX_POSITION (the fp32 RoPE chain is exact
 *     and bit-reproducible there).
 */
#ifndef GROK_ATTN_H
#define GROK_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 2: GROK_DECODE_SPLIT went from 512 to 1024 keys (decode workspace sizes changed) */
#define GROK_ATTN_ABI_VERSION 2

#define GROK_N_Q_HEADS 48
#define GROK_N_KV_HEADS 8
#define GROK_HEAD_DIM 128
#define GROK_MAX_POSITION 65536
/* keys per decode split (one partial result per split) */
#define GROK_DECODE_SPLIT 1024

typedef uint16_t grok_bf16;

typedef enum {
  GROK_OK = 0,
  GROK_ERR_INVALID_ARG = 1,
  GROK_ERR_UNSUPPORTED = 2,  /* no sm_103 device, or a size this build does not cover */
  GROK_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed; the context is still usable */
  GROK_ERR_DEVICE_FAULT = 4  /* a sticky device error (illegal address or instruction, misaligned
                                address, launch failure, uncorrectable ECC or NVLink error, ...):
                                the CUDA context is dead and every later call fails the same way;
                                the process must be restarted to use the GPU again */
} grok_status;

/* bits OR-ed into *dev_status by the kernels */
#define GROK_DEV_BAD_START 0x1   /* start_pos[b] < 0, start_pos[b] + T > Tmax, or > GROK_MAX_POSITION */
#define GROK_DEV_BAD_VALID 0x2   /* valid_len[b] outside [1, T] */
#define GROK_DEV_BAD_KV_LEN 0x4  /* kv_len[b] outside [1, Tmax] */
#define GROK_DEV_TIMEOUT 0x8     /* a bounded wait inside a kernel gave up */
#define GROK_DEV_BAD_PAGE 0x10   /* a block-table entry the paged calls need lies outside [0, n_pages) */

/* Tokens per page of the paged KV cache (one prefill key tile). */
#define GROK_PAGE_TOKENS 128

/* ABI version this library was built with (GROK_ATTN_ABI_VERSION). */
int grok_abi_version(void);

/* Message describing the last non-OK status returned on this thread. */
const char* grok_last_error(void);

/*
 * The status this library returns when a CUDA runtime call fails with
 * `cuda_error` (a cudaError_t value): GROK_OK for cudaSuccess,
 * GROK_ERR_DEVICE_FAULT for the errors that leave the context unusable,
 * GROK_ERR_CUDA for the rest. Host only; touches no device.
 */
grok_status grok_cuda_error_status(int cuda_error);

/*
 * RoPE on Q and K, then the KV-cache append (ch. 4 §4.3.1, §4.4).
 *
 * For sequence b and new token i (position p = start_pos[b] + i), every query
 * head and every KV head is rotated pairwise (feature j with feature j + 64):
 *   inv_freq[j] = 1 / RN32(10000^(j/64)),  phase = RN32(p * inv_freq[j]),
 *   c = RN32(cos(phase)), s = RN32(sin(phase)) (fp64 evaluation),
 *   x'[j] = RN32(RN32(x[j] c) - RN32(x[j+64] s)),
 *   x'[j+64] = RN32(RN32(x[j+64] c) + RN32(x[j] s)), rounded to bf16 (nearest even).
 * Rotated Q goes to q_rot; rotated K and raw V are written to cache rows
 * [start_pos[b], start_pos[b] + T) of sequence b; no other cache row is touched.
 *   q [B,T,48,128], k, v [B,T,8,128] in; start_pos [B] int32 (device);
 *   q_rot [B,T,48,128] out (may not alias q); cache_k, cache_v [B,Tmax,8,128] in/out.
 * The caller advances its step counter by T afterwards (new_step = step + T).
 */
grok_status grok_rope_kv_append(const grok_bf16* q, const grok_bf16* k, const grok_bf16* v,
                                const int32_t* start_pos, int B, int T, int Tmax, grok_bf16* q_rot,
                                grok_bf16* cache_k, grok_bf16* cache_v, int32_t* dev_status, void* stream);

/*
 * grok_rope_kv_append with the (cos, sin) pairs read from a table instead of
 * evaluated per token. The values depend only on the position (ch. 4 §4.3.1),
 * so one table, filled once by grok_rope_cos_sin(0, tab_positions, cos_tab,
 * sin_tab), serves every layer and every step of a model: the per-layer
 * append then does no transcendental work. Same bits as grok_rope_kv_append.
 *   cos_tab, sin_tab: device float[tab_positions * 64] (position p, frequency j
 *   at p * 64 + j), 16-byte aligned; positions start_pos[b] + T must not exceed
 *   tab_positions (else GROK_DEV_BAD_START and the sequence is skipped).
 * Other arguments as for grok_rope_kv_append.
 */
grok_status grok_rope_kv_append_table(const grok_bf16* q, const grok_bf16* k, const grok_bf16* v,
                                      const int32_t* start_pos, int B, int T, int Tmax, const float* cos_tab,
                                      const float* sin_tab, int tab_positions, grok_bf16* q_rot, grok_bf16* cache_k,
                                      grok_bf16* cache_v, int32_t* dev_status, void* stream);

/*
 * The fp32 RoPE table the append uses (ch. 4 §4.3.1: phase = t * inv_freq,
 * cos and sin of it): cos_out[i * 64 + j] and sin_out[i * 64 + j] for position
 * first_position + i and frequency j < 64, i < n_positions; each value is the
 * correctly rounded fp32 cos / sin of the fp32 phase RN32(p * inv_freq[j]).
 * cos_out, sin_out: device float[n_positions * 64]. Positions < GROK_MAX_POSITION.
 */
grok_status grok_rope_cos_sin(int first_position, int n_positions, float* cos_out, float* sin_out, void* stream);

/*
 * Prefill attention of T new tokens per sequence over the appended cache
 * (ch. 4 §4.5.2-§4.5.4, ch. 6 §6.4.2).
 *
 * Query i of sequence b (cache position start_pos[b] + i) attends cache row j iff
 *   j <= start_pos[b] + i  and  j < start_pos[b] + valid_len[b];
 * logits = (q_rot . k) / sqrt(128), capped as 30 tanh(x / 30), softmax over the
 * visible rows, output = sum of weights x v, rounded to bf16. Padding query rows
 * (i >= valid_len[b]) are computed too. Query head h reads KV head h / 6.
 *   q_rot [B,T,48,128]; cache_k, cache_v [B,Tmax,8,128]; start_pos [B] int32;
 *   valid_len [B] int32 or NULL (= T for every sequence); out [B,T,48,128].
 * Requires T <= Tmax and T, Tmax >= 1.
 */
grok_status grok_attn_prefill(const grok_bf16* q_rot, const grok_bf16* cache_k, const grok_bf16* cache_v,
                              const int32_t* start_pos, const int32_t* valid_len, int B, int T, int Tmax,
                              grok_bf16* out, int32_t* dev_status, void* stream);

/*
 * Prefill with fp16 softmax weights (same operation, arguments and results as
 * grok_attn_prefill; ch. 4 §4.5.3 casts the softmax weights to the value dtype
 * before the weighted sum, which this call does in fp16 instead of bf16, so
 * each P V product runs once instead of twice). Each row's weights are taken
 * relative to a reference set from its first key tile (its largest weight
 * there is 2^-8) and rounded once to fp16; V is read from an fp16 copy that
 * the call first writes into `workspace` (rows [0, start_pos[b] + T) of each
 * sequence rounded to nearest fp16, then zeros to the next multiple of 128).
 * Items (128 query rows x 2 heads) whose weights could leave fp16's range (a
 * row's weight sum reaching 65504), and every item of a sequence holding a
 * finite |v| >= 65520, are listed in the workspace and recomputed by a second
 * pass with bf16 weights from the bf16 cache, so every finite input is
 * handled; results then equal grok_attn_prefill's for those items.
 *   workspace: caller-owned device memory, 256-byte aligned, of at least
 *   grok_attn_prefill_workspace_min(B, Tmax) bytes (B * round_up(Tmax, 128) *
 *   2 KB for the V copy plus a header of about B * Tmax / 128 * 864 bytes).
 *   grok_attn_prefill_workspace(B, Tmax) adds, for the current device, room
 *   for the key-range split (SM count x 130 KB, about 20 MB on 152 SMs; none
 *   when Tmax < 1921): when a call has fewer than two work items (128 query
 *   rows x 2 heads) per SM, the items left for the last round (all of them
 *   when there are fewer items than SMs) have their key tiles shared among up
 *   to 4 work units of at least 8 tiles each, run by a second pass; each
 *   unit's unnormalised output (fp32) goes to the workspace and the item's
 *   last unit to finish adds them in unit order and writes the output. The
 *   bits then do not depend on scheduling, but differ from an unsplit call's
 *   within the same tolerance. With less workspace than that the call runs
 *   unsplit. Calls that overlap on the GPU need separate workspaces.
 *   reuse_v_half: 0 = convert rows [0, start_pos[b] + T) (the call is self-
 *   contained). 1 = convert only rows [start_pos[b], start_pos[b] + T): rows
 *   below start_pos[b] must already be in this workspace from earlier calls
 *   over the same caches (for example the previous chunks of a chunked
 *   prefill), and no other call may have written those cache rows since (a
 *   decode step's append, a slot insertion); a sequence once found to hold V
 *   beyond fp16 stays on the bf16 path until a call with 0.
 */
grok_status grok_attn_prefill_workspace(int B, int Tmax, size_t* bytes);
grok_status grok_attn_prefill_workspace_min(int B, int Tmax, size_t* bytes);
grok_status grok_attn_prefill_ws(const grok_bf16* q_rot, const grok_bf16* cache_k, const grok_bf16* cache_v,
                                 const int32_t* start_pos, const int32_t* valid_len, int B, int T, int Tmax,
                                 grok_bf16* out, void* workspace, size_t workspace_bytes, int reuse_v_half,
                                 int32_t* dev_status, void* stream);

/*
 * Bytes of device workspace grok_attn_decode needs for B sequences and a cache
 * of Tmax rows (fp32 partial sums per split of GROK_DECODE_SPLIT keys), and the
 * number of splits per sequence. Either output pointer may be NULL.
 */
grok_status grok_attn_decode_workspace(int B, int Tmax, size_t* bytes, int* max_splits);

/*
 * One decode step, split-K part (ch. 4 §4.4.1; ch. 6 §6.4.2: the new token
 * attends every cache row below step + 1, which the memory mask selects).
 *
 * For sequence b the single query q_rot[b] (its own K/V already appended at
 * row kv_len[b] - 1) is scored against cache rows [0, kv_len[b]) in splits of
 * GROK_DECODE_SPLIT rows. Each split writes, per query head, the sums
 *   l = sum_j exp(c_j - 30),  o = sum_j exp(c_j - 30) v_j
 * (c = capped logit; 30 bounds every capped logit, so no running maximum is
 * needed) into `workspace`. grok_attn_combine finishes the step.
 *   q_rot [B,48,128]; cache_k, cache_v [B,Tmax,8,128]; kv_len [B] int32 (device);
 *   workspace: device buffer of at least grok_attn_decode_workspace bytes,
 *   256-byte aligned, owned by the caller.
 */
grok_status grok_attn_decode(const grok_bf16* q_rot, const grok_bf16* cache_k, const grok_bf16* cache_v,
                             const int32_t* kv_len, int B, int Tmax, void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, void* stream);

/*
 * Decode step, combine part: out[b, h] = (sum over splits of o) / (sum over
 * splits of l), rounded to bf16. Reads the workspace written by
 * grok_attn_decode with the same B, Tmax and kv_len. workspace_bytes is the
 * size of that workspace, checked against grok_attn_decode_workspace(B, Tmax)
 * before anything is launched (the pages' interface has no workspace; the
 * size travels with the pointer so that a short buffer is an argument error,
 * not an out-of-bounds read). If grok_attn_decode set a bit in *dev_status
 * (a bounded wait that gave up skips a split's writes), out is undefined.
 *   out [B,48,128] bf16.
 */
grok_status grok_attn_combine(const void* workspace, size_t workspace_bytes, const int32_t* kv_len, int B,
                              int Tmax, grok_bf16* out, int32_t* dev_status, void* stream);

/*
 * Failure-detection self-test. Every wait inside the pipelined kernels is
 * bounded: after a clock-cycle limit it ORs GROK_DEV_TIMEOUT into *dev_status,
 * raises its CTA's abort flag so the other waiting warps leave too, and the
 * kernel returns without trapping. This call runs that machinery on a
 * one-CTA kernel whose two barriers nothing ever completes: warp 0 waits
 * limit_cycles and gives up, warp 1 (limit 1000x longer) must leave through
 * the abort flag. Afterwards *dev_status has GROK_DEV_TIMEOUT and
 * flags[0] = flags[1] = 2 (device int32[2]). limit_cycles in [1, 4e9].
 */
grok_status grok_selftest_bounded_wait(int32_t* dev_status, int32_t* flags, long long limit_cycles, void* stream);

/* Size of the library's static decode workspace (bytes). */
#define GROK_STATIC_WORKSPACE_BYTES (16u << 20)

/*
 * A whole decode step (grok_attn_decode then grok_attn_combine) that
 * allocates nothing and takes no workspace. The pages have no counterpart:
 * this call exists for callers that cannot allocate device memory, such as a
 * plugin whose host framework owns all device memory, or a serving loop whose
 * memory is planned up front and may not call cudaMalloc (which can
 * synchronise the device) between steps.
 *
 * The split-K partial sums go to a static device array of
 * GROK_STATIC_WORKSPACE_BYTES; shapes whose workspace (grok_attn_decode_workspace)
 * is larger are rejected with GROK_ERR_INVALID_ARG. CUDA loads the library's
 * device code lazily by default (CUDA_MODULE_LOADING=LAZY), so the array is
 * reserved on a device when the library's code is first used there, possibly
 * by the first call of this function, and held until the process exits. The
 * first call on a device also looks up the array's device address
 * (cudaGetSymbolAddress) with that device current. So make one warm-up call on
 * each device at initialisation, before the memory plan is fixed and before
 * any stream capture; later calls allocate nothing.
 * All calls share the one array: calls that overlap on the GPU (different
 * streams, or different host threads on the same device) race and give wrong
 * results; calls ordered on one stream are safe. Nothing needs clearing: each
 * call that completes writes every partial sum it reads. If *dev_status comes
 * back nonzero (a bad kv_len, or a bounded wait that gave up), out is undefined
 * for this call and may hold values computed from an earlier call's partial
 * sums. Arguments and results are those of grok_attn_decode + grok_attn_combine:
 *   q_rot [B,48,128]; cache_k, cache_v [B,Tmax,8,128]; kv_len [B] int32; out [B,48,128].
 */
grok_status grok_attn_decode_step_static(const grok_bf16* q_rot, const grok_bf16* cache_k, const grok_bf16* cache_v,
                                         const int32_t* kv_len, int B, int Tmax, grok_bf16* out,
                                         int32_t* dev_status, void* stream);

/*
 * One whole decode step in one call (ch. 4 §4.4 and §4.4.1: the new token's
 * K and V are rotated and written into the cache at step[b], then attention
 * over rows [0, step[b]] with the memory mask):
 *   grok_rope_kv_append(q, k, v, start_pos, B, T = 1, Tmax, ...), then
 *   grok_attn_decode and grok_attn_combine with kv_len[b] = start_pos[b] + 1.
 * Same bits as those three calls. The decode and combine are launched as
 * programmatic dependents of the kernel before them: each may start while its
 * predecessor finishes, and the decode loads the cache rows the append does
 * not write before it waits for the append.
 *   q [B,48,128], k, v [B,8,128] bf16; start_pos [B] int32 (the new token's
 *   position, 0 <= start_pos[b] < Tmax); cache_k, cache_v [B,Tmax,8,128];
 *   out [B,48,128] bf16. workspace: caller-owned device memory, 256-byte
 *   aligned, of at least grok_attn_decode_step_workspace(B, Tmax) bytes (it
 *   holds q_rot and the split partials). Errors as for the three calls.
 */
grok_status grok_attn_decode_step_workspace(int B, int Tmax, size_t* bytes);
grok_status grok_attn_decode_step(const grok_bf16* q, const grok_bf16* k, const grok_bf16* v,
                                  const int32_t* start_pos, int B, int Tmax, grok_bf16* cache_k, grok_bf16* cache_v,
                                  void* workspace, size_t workspace_bytes, grok_bf16* out, int32_t* dev_status,
                                  void* stream);

/*
 * Q/K/V projection (code-reading guide ch. 4 §4.1 Linear, §4.5.1 Q/K/V
 * projection): the three bias-free Linears of the attention call as one
 * product with the weights side by side.
 *   x [M, 6144] bf16 (M = B*T rows, row b*T + i), w [6144, 8192] bf16 in the
 *   pages' [input, output] layout: columns h*128 + d are query head h,
 *   6144 + g*128 + d key head g, 7168 + g*128 + d value head g.
 * fp32 accumulation on the tensor cores, one rounding to bf16 per output.
 *
 * grok_qkv_project: y [M, 8192] = x . w. dev_status is unused (nullable).
 * grok_qkv_rope_append: the projection fused with grok_rope_kv_append. q heads
 *   are rotated into q_rot [B,T,48,128]; k heads are rotated and v heads copied
 *   into rows [start_pos[b], start_pos[b]+T) of cache_k / cache_v
 *   [B,Tmax,8,128]. Bits equal grok_rope_kv_append applied to the bf16
 *   projection. workspace: caller-owned device memory of at least
 *   grok_qkv_workspace(B, T) bytes (a per-step cos/sin table), 16-byte aligned.
 *   A sequence whose start_pos[b] + T > Tmax (or start < 0) sets
 *   GROK_DEV_BAD_START and none of its rows are written.
 * All pointers device-resident and 16-byte aligned; the outputs (y; q_rot,
 * cache_k, cache_v) 32-byte aligned. Work is asynchronous on stream.
 */
grok_status grok_qkv_project(const grok_bf16* x, const grok_bf16* w, int M, grok_bf16* y, int32_t* dev_status,
                             void* stream);

/*
 * A bias-free Linear (ch. 4 §4.1) on the same tensor-core kernel:
 * y [M, N] = x [M, K] . w [K, N], bf16, fp32 accumulation, one rounding.
 * K must be a positive multiple of 64 and N of 256 or of 192; 1 <= M <= 2^30. Row-major
 * device tensors, x and w 16-byte aligned, y 32-byte aligned. Serves the output projection (ch. 4 §4.5.4:
 * attention output [B*T, 48*128] head-major . W_o [6144, 6144]) and each
 * tensor-parallel rank's share of it (the rows of W_o for the rank's heads,
 * K = 6144 / ranks; the ranks' partial outputs are summed by the caller).
 * grok_qkv_project is grok_linear with K = 6144, N = 8192.
 */
grok_status grok_linear(const grok_bf16* x, const grok_bf16* w, int M, int K, int N, grok_bf16* y, int32_t* dev_status,
                        void* stream);

/*
 * Int8 weight-only Linear (ch. 4 §4.1 Linear with QuantizedWeight8bit, §4.1.1):
 * weight int8 [K, N] (row-major, the pages' [input, output] layout) with one
 * fp32 scale per output column, scales [N].
 * grok_dequant_int8: w16 [K, N] bf16 = bf16(fp32(w8 * scales[n])): an fp32
 *   multiply rounded to fp32, then rounded to nearest even bf16 (the pages'
 *   astype(scales.dtype) * scales, then astype(bf16)). N a multiple of 16.
 * grok_linear_int8: y [M, N] = x [M, K] . dequant(w8, scales): the weight is
 *   dequantized into the caller's workspace (at least
 *   grok_linear_int8_workspace(K, N) bytes, K*N bf16) and then multiplied by
 *   grok_linear (so K % 64 == 0, N % 256 == 0 or N % 192 == 0). For prefill-sized M the
 *   product is tensor-bound and the one pass over the weight costs a few
 *   percent; the workspace may be reused across calls with the same weight.
 *   For decode-sized M (M <= 32, K a multiple of 512) the weight is instead
 *   read once and dequantized on chip, the same per-element rounding: clusters
 *   of 8 CTAs split K and add their partial sums in a fixed order, so the bits
 *   do not depend on scheduling. The workspace is not touched then (it must
 *   still be passed).
 * All pointers device-resident and 16-byte aligned; w16, the workspace and y
 * 32-byte aligned. Asynchronous on stream.
 */
grok_status grok_dequant_int8(const int8_t* w8, const float* scales, int K, int N, grok_bf16* w16, void* stream);
grok_status grok_linear_int8_workspace(int K, int N, size_t* bytes);
grok_status grok_linear_int8(const grok_bf16* x, const int8_t* w8, const float* scales, int M, int K, int N,
                             grok_bf16* y, void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);
grok_status grok_qkv_workspace(int B, int T, size_t* bytes);
/*
 * grok_qkv_rope_append with cos/sin read from a table of positions
 * [0, tab_positions) (grok_rope_cos_sin(0, tab_positions, ...), filled once
 * and shared by every layer and step) instead of a per-call table: no table
 * kernel and no workspace. Same bits as grok_qkv_rope_append. A sequence whose
 * positions start_pos[b] + T exceed Tmax or tab_positions sets
 * GROK_DEV_BAD_START and none of its rows are written. cos_tab, sin_tab:
 * device float[tab_positions * 64], 16-byte aligned.
 */
grok_status grok_qkv_rope_append_table(const grok_bf16* x, const grok_bf16* w, const int32_t* start_pos, int B,
                                       int T, int Tmax, const float* cos_tab, const float* sin_tab, int tab_positions,
                                       grok_bf16* q_rot, grok_bf16* cache_k, grok_bf16* cache_v, int32_t* dev_status,
                                       void* stream);
grok_status grok_qkv_rope_append(const grok_bf16* x, const grok_bf16* w, const int32_t* start_pos, int B, int T,
                                 int Tmax, grok_bf16* q_rot, grok_bf16* cache_k, grok_bf16* cache_v, void* workspace,
                                 size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * Host-buffer prefill pipeline. The pages feed the attention core from a model
 * on the same device and have no counterpart; this runtime object is for
 * callers whose q, k, v arrive in host memory and whose output goes back there
 * (a serving front end). A pipeline owns device double buffers and three CUDA
 * streams (host-to-device copies, kernels, device-to-host copies), so the
 * copies of one step overlap the kernels of the steps before and after it.
 *
 * grok_prefill_pipe_create: B, T, Tmax as for grok_rope_kv_append and
 *   grok_attn_prefill. cache_k, cache_v are the caller's device caches
 *   [B,Tmax,8,128] bf16 (16-byte aligned): every step appends to them and
 *   attends over them, and they must stay allocated until destroy. Allocates
 *   about B*T*(5*48 + 4*8)*128*2 bytes of device memory on the current device,
 *   plus grok_attn_prefill_workspace(B, Tmax) bytes and a Tmax * 512-byte
 *   cos/sin table, which the pipeline uses from then on. *pipe receives the handle.
 * grok_prefill_pipe_submit: queue one step. Copy q [B,T,48,128], k and v
 *   [B,T,8,128], start_pos [B] and valid_len [B] (NULL: every token valid) from
 *   host memory; run grok_rope_kv_append_table (with a cos/sin table of
 *   positions [0, Tmax) made at create) then grok_attn_prefill_ws; copy the output
 *   [B,T,48,128] to host memory at out. Returns once the work is queued. The
 *   host buffers must stay valid, the inputs unchanged and the output unread
 *   until the next grok_prefill_pipe_wait. Page-locked host memory
 *   (cudaHostAlloc, cudaHostRegister) lets the copies overlap; pageable memory
 *   works but serialises them. Steps run in submission order. Argument errors
 *   are returned before anything is queued.
 * grok_prefill_pipe_wait: block until every queued step has finished.
 *   *dev_status (nullable) receives the OR of the steps' device status words
 *   (GROK_DEV_* bits, 0 when every sequence's integers were valid); the word is
 *   then cleared.
 * grok_prefill_pipe_destroy: wait, then free everything. NULL is ignored.
 * One host thread at a time may use a pipeline.
 */
typedef struct grok_prefill_pipe grok_prefill_pipe;
grok_status grok_prefill_pipe_create(int B, int T, int Tmax, grok_bf16* cache_k, grok_bf16* cache_v,
                                     grok_prefill_pipe** pipe);
grok_status grok_prefill_pipe_submit(grok_prefill_pipe* pipe, const grok_bf16* q, const grok_bf16* k,
                                     const grok_bf16* v, const int32_t* start_pos, const int32_t* valid_len,
                                     grok_bf16* out);
grok_status grok_prefill_pipe_wait(grok_prefill_pipe* pipe, int32_t* dev_status);
grok_status grok_prefill_pipe_destroy(grok_prefill_pipe* pipe);

/*
 * Paged KV cache (code-reading guide ch. 6 "model.py close reading II": §6.6
 * preallocates the cache at (B, 8192, 8, 128); §6.6.1 gives every sequence its
 * own step counter so sequences can join and leave a batch independently;
 * §6.6.2 notes that serving systems store the cache in token pages that are
 * allocated only when used, which Grok-1's code does not do). These calls are
 * the contiguous calls above with the cache rows looked up through a block
 * table; the arithmetic, and so every result bit, is the same as for a
 * contiguous cache holding the same keys and values.
 *
 * Layout: k_pool, v_pool [n_pages, GROK_PAGE_TOKENS, 8, 128] bf16, 16-byte
 * aligned, owned by the caller. block_table [B, max_pages] int32 (device):
 * position p of sequence b lives in row p % GROK_PAGE_TOKENS of page
 * block_table[b * max_pages + p / GROK_PAGE_TOKENS]. A sequence's capacity is
 * max_pages * GROK_PAGE_TOKENS (it plays the part of Tmax, at most
 * GROK_MAX_POSITION). Pages may be shared between sequences and listed in any
 * order; table entries past what a call touches are never read, so unused
 * entries may hold anything. Every table entry a call reads must lie in
 * [0, n_pages): otherwise the call sets GROK_DEV_BAD_PAGE, reads page 0 in
 * its place (results for that sequence are then meaningless) and the append
 * skips that token's cache write (its q_rot is still written).
 *
 * grok_rope_kv_append_paged: grok_rope_kv_append writing rows
 *   [start_pos[b], start_pos[b] + T) of sequence b through the table.
 * grok_attn_prefill_paged: grok_attn_prefill reading keys [0, start_pos[b] +
 *   valid_len[b]) of sequence b through the table.
 * grok_attn_prefill_ws_paged: grok_attn_prefill_ws over the pools: K is read
 *   through the table, and the call's fp16 copy of V (in the workspace, sized
 *   by grok_attn_prefill_workspace(B, max_pages * GROK_PAGE_TOKENS)) is made
 *   through the table, contiguous per sequence; reuse_v_half as for
 *   grok_attn_prefill_ws. Bits equal grok_attn_prefill_ws over a contiguous
 *   cache holding the same keys and values.
 * grok_attn_decode_paged: grok_attn_decode reading keys [0, kv_len[b]) through
 *   the table; workspace sized by grok_attn_decode_workspace(B, max_pages *
 *   GROK_PAGE_TOKENS) and combined with grok_attn_combine(..., Tmax = max_pages
 *   * GROK_PAGE_TOKENS, ...).
 * grok_qkv_rope_append_paged: grok_qkv_rope_append (the projection fused with
 *   RoPE and the append) writing the k and v rows through the table; the
 *   workspace is sized by grok_qkv_workspace(B, T); q_rot and the pools must
 *   be 32-byte aligned, as for grok_qkv_rope_append.
 * Argument errors (null pointers, misaligned tensors, n_pages < 1,
 * max_pages < 1, sizes past the limits above) return GROK_ERR_INVALID_ARG with
 * nothing launched.
 */
grok_status grok_rope_kv_append_paged(const grok_bf16* q, const grok_bf16* k, const grok_bf16* v,
                                      const int32_t* start_pos, int B, int T, grok_bf16* q_rot, grok_bf16* k_pool,
                                      grok_bf16* v_pool, int n_pages, const int32_t* block_table, int max_pages,
                                      int32_t* dev_status, void* stream);
grok_status grok_attn_prefill_paged(const grok_bf16* q_rot, const grok_bf16* k_pool, const grok_bf16* v_pool,
                                    int n_pages, const int32_t* block_table, int max_pages,
                                    const int32_t* start_pos, const int32_t* valid_len, int B, int T,
                                    grok_bf16* out, int32_t* dev_status, void* stream);
grok_status grok_attn_prefill_ws_paged(const grok_bf16* q_rot, const grok_bf16* k_pool, const grok_bf16* v_pool,
                                       int n_pages, const int32_t* block_table, int max_pages,
                                       const int32_t* start_pos, const int32_t* valid_len, int B, int T,
                                       grok_bf16* out, void* workspace, size_t workspace_bytes, int reuse_v_half,
                                       int32_t* dev_status, void* stream);
grok_status grok_attn_decode_paged(const grok_bf16* q_rot, const grok_bf16* k_pool, const grok_bf16* v_pool,
                                   int n_pages, const int32_t* block_table, int max_pages, const int32_t* kv_len,
                                   int B, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                   void* stream);
grok_status grok_qkv_rope_append_paged(const grok_bf16* x, const grok_bf16* w, const int32_t* start_pos, int B,
                                       int T, grok_bf16* q_rot, grok_bf16* k_pool, grok_bf16* v_pool, int n_pages,
                                       const int32_t* block_table, int max_pages, void* workspace, size_t ws_bytes,
                                       int32_t* dev_status, void* stream);

/*
 * Continuous-batching slot insertion (code-reading guide ch. 6 §6.6.1: every
 * sequence has its own step, so a finished sequence's batch slot can be handed
 * to a new request; the runner inserts the new sequence's memory into slot i
 * along the batch axis, for the k and v caches and the step).
 *
 * grok_kv_insert_slot copies rows [0, n_rows) of one sequence's caches src_k,
 * src_v [src_rows, 8, 128] into rows [0, n_rows) of slot `slot` of the batch
 * caches cache_k, cache_v [B, Tmax, 8, 128] (all bf16, device, 16-byte
 * aligned, caller-owned), and sets step[slot] = step_value when step (device
 * int32 [B], e.g. the start_pos / kv_len array of the next call) is not NULL.
 * Rows >= n_rows of the slot are left as they are: attention never reads rows
 * at or beyond a sequence's step, so n_rows >= step_value gives the results of
 * replacing the whole slot. The source rows must not overlap the slot.
 * Argument errors return GROK_ERR_INVALID_ARG with nothing launched; one kernel
 * launch otherwise (none when n_rows == 0 and step is NULL).
 * With a paged cache (GROK_PAGE_TOKENS) no copy is needed: the new sequence's
 * pages are named in its row of the block table.
 */
grok_status grok_kv_insert_slot(grok_bf16* cache_k, grok_bf16* cache_v, int B, int Tmax, int slot,
                                const grok_bf16* src_k, const grok_bf16* src_v, int src_rows, int n_rows,
                                int32_t* step, int step_value, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GROK_ATTN_H */
