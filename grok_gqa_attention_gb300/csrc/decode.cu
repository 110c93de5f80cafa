// K3: split-K decode attention, K4: combine.
//
// Grok-1 code-reading guide, ch. 4 "model.py close reading I", §4.4.1 (a decode
// step attends every cache row already written; the memory mask does the
// masking) and §4.5.2-§4.5.4 (GQA logits, 1/sqrt(128), soft cap, fp32
// softmax, weighted sum of V); ch. 6 "model.py close reading II", §6.4.2.
//
// Memory-bound: one step streams K and V of every used cache row once
// (512 bytes per row per KV head). Grid = (KV group, sequence, split); a CTA
// of 4 warps streams GROK_DECODE_SPLIT rows of one (sequence, group) through a
// 3-stage TMA ring of 64-row tiles and keeps the group's 6 query heads as a
// 16-row mma.sync operand (rows 6..15 zero): per 16 rows a warp computes
// S = Q K^T (m16n8k16, fp32 accumulate), the capped weights relative to the
// fixed reference logit 30 (no running maximum is needed because every capped
// logit is below 30), and O += P_hi V + P_lo V with P split into two bf16
// halves. Each split writes its unnormalised O and row sum l; the combine
// kernel adds the splits and divides.
#include <mutex>

#include "common.cuh"
#include "host.cuh"

namespace grok {

constexpr int kDecThreads = 128;
constexpr int kDecKeysPerStage = 64;
constexpr int kDecStages = 3;
constexpr int kDecBox = kDecKeysPerStage * 128;  // [64 rows][64 bf16] = 8 KB
constexpr int kDecStageBytes = 4 * kDecBox;      // K halves then V halves
constexpr int kDecSmem = kDecStages * kDecStageBytes + 1024 + 256;
constexpr int kDecSplit = GROK_DECODE_SPLIT;
static_assert(kDecSplit % kDecKeysPerStage == 0, "split must be whole stages");

struct DecWs {
  float* o;  // [B][8][n_split][6][128]
  float* l;  // [B][8][n_split][6]
};

__host__ __device__ inline size_t dec_o_floats(int B, int n_split) {
  return size_t(B) * kKVHeads * n_split * kGroup * kD;
}
__host__ __device__ inline size_t dec_ws_bytes(int B, int n_split) {
  const size_t o = dec_o_floats(B, n_split) * 4;
  const size_t l = size_t(B) * kKVHeads * n_split * kGroup * 4;
  return ((o + 255) & ~size_t(255)) + ((l + 255) & ~size_t(255));
}
__host__ __device__ inline DecWs dec_ws(void* base, int B, int n_split) {
  DecWs w;
  w.o = reinterpret_cast<float*>(base);
  w.l = reinterpret_cast<float*>(reinterpret_cast<char*>(base) +
                                 ((dec_o_floats(B, n_split) * 4 + 255) & ~size_t(255)));
  return w;
}

__global__ void __launch_bounds__(kDecThreads) decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                             const __grid_constant__ CUtensorMap tm_v,
                                                             const uint32_t* __restrict__ q_rot,
                                                             const int32_t* __restrict__ kv_len, int kv_add,
                                                             int Tmax, int n_split, DecWs ws, PageMap pm,
                                                             int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kDecStages * kDecStageBytes);
  uint64_t* empty = full + kDecStages;
  int* abort_flag = reinterpret_cast<int*>(empty + kDecStages);
  volatile int* abort = abort_flag;

  // A dependent combine may be scheduled as soon as every CTA has started.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // split is the slowest grid dimension: the splits past a sequence's length, which
  // leave at once, come after every split with work
  const int g = blockIdx.x, b = blockIdx.y, split = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long L_ = (long long)__ldg(kv_len + b) + kv_add;
  const int L = L_ < 1 || L_ > Tmax ? 0 : int(L_);
  if (L < 1) {
    if (split == 0 && g == 0 && tid == 0) report(status, GROK_DEV_BAD_KV_LEN);
    return;
  }
  const int k0 = split * kDecSplit;
  if (k0 >= L) return;  // this split has no rows; the combine does not read it
  const int k1 = min(k0 + kDecSplit, L);
  const int n_st = (k1 - k0 + kDecKeysPerStage - 1) / kDecKeysPerStage;

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  // The first stages of the ring. When this grid is the programmatic dependent
  // of the append that wrote the newest row (kv_add = 1: rows < L - 1 are older
  // than that grid and complete), the stages that cannot hold row L - 1 are
  // loaded before waiting for it; the rest, q_rot included, after.
  auto load_stage = [&](int s) {
    uint8_t* base = smem + s * kDecStageBytes;
    const int key0 = k0 + s * kDecKeysPerStage;
    int row, bc;
    kv_coord(pm, b, key0, row, bc, status);  // a 64-key tile never straddles a page
    mbar_arrive_expect_tx(&full[s], kDecStageBytes);
    tma_load_4d(base, &tm_k, &full[s], 0, g, row, bc);
    tma_load_4d(base + kDecBox, &tm_k, &full[s], 64, g, row, bc);
    tma_load_4d(base + 2 * kDecBox, &tm_v, &full[s], 0, g, row, bc);
    tma_load_4d(base + 3 * kDecBox, &tm_v, &full[s], 64, g, row, bc);
  };
  auto early = [&](int s) { return kv_add == 1 && k0 + (s + 1) * kDecKeysPerStage <= L - 1; };
  if (tid == 0)
    for (int s = 0; s < kDecStages && s < n_st; ++s)
      if (early(s)) load_stage(s);
  asm volatile("griddepcontrol.wait;" ::: "memory");  // no-op unless launched as a dependent
  if (tid == 0)
    for (int s = 0; s < kDecStages && s < n_st; ++s)
      if (!early(s)) load_stage(s);

  // Q of the group's 6 heads as the A operand (rows lane/4; rows >= 6 and the
  // upper 8 rows are zero). A fragment: a0 = (row, k 2t..2t+1), a2 = (row, k 2t+8..).
  const int qrow = lane >> 2, t4 = lane & 3;
  uint32_t qa[8][2];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    if (qrow < kGroup) {
      const uint32_t* qh = q_rot + ((size_t)b * kQHeads + g * kGroup + qrow) * (kD / 2);
      qa[kk][0] = __ldg(qh + kk * 8 + t4);
      qa[kk][1] = __ldg(qh + kk * 8 + 4 + t4);
    } else {
      qa[kk][0] = 0u;
      qa[kk][1] = 0u;
    }
  }
  __syncthreads();

  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float lsum = 0.f;
  const uint32_t sbase = smem_u32(smem);
  bool ok = true;

  for (int it = 0; it < n_st; ++it) {
    const int st = it % kDecStages;
    ok = mbar_wait(&full[st], (it / kDecStages) & 1, abort, status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    const uint32_t kb = sbase + st * kDecStageBytes;
    const uint32_t vb = kb + 2 * kDecBox;
    const int key_base = k0 + it * kDecKeysPerStage + warp * 16;  // this warp's 16 rows
    if (key_base < k1) {
      // S[16 heads x 16 keys] = Q K^T over d = 128
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int mi = lane >> 3, mr = lane & 7;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int row = warp * 16 + (mi >> 1) * 8 + mr;
        const int col = (kk & 3) * 16 + (mi & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + (kk >> 2) * kDecBox + sw128_offset(row, col), b0, b1, b2, b3);
        const uint32_t a[4] = {qa[kk][0], 0u, qa[kk][1], 0u};
        mma_bf16_16816(s[0], a, b0, b1);
        mma_bf16_16816(s[1], a, b2, b3);
      }
      // weights: row qrow, keys key_base + 8n + 2 t4 + e
      float w[2][2];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key_base + 8 * n + 2 * t4 + e;
          const float x = capped_weight_precise(s[n][e]);
          w[n][e] = (qrow < kGroup && key < k1) ? x : 0.f;
          lsum += w[n][e];
        }
      uint32_t phi[4], plo[4];
      split_bf16x2(w[0][0], w[0][1], phi[0], plo[0]);
      split_bf16x2(w[1][0], w[1][1], phi[2], plo[2]);
      phi[1] = phi[3] = plo[1] = plo[3] = 0u;
      const bool tail = key_base + 16 > k1;  // rows past k1 may hold anything
      // O[16 x 128] += P[16 x 16] V[16 x 128]
#pragma unroll
      for (int np = 0; np < 8; ++np) {  // pairs of 8-wide d tiles
        const int row = warp * 16 + (mi & 1) * 8 + mr;
        const int col = (np & 3) * 16 + (mi >> 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + (np >> 2) * kDecBox + sw128_offset(row, col), b0, b1, b2, b3);
        if (tail) {
          // b0/b2 hold rows 2t4, 2t4+1; b1/b3 rows 8 + 2t4, 9 + 2t4 (low half = first row)
          const int r0 = key_base + 2 * t4, r1 = key_base + 8 + 2 * t4;
          const uint32_t m0 = (r0 < k1 ? 0x0000FFFFu : 0u) | (r0 + 1 < k1 ? 0xFFFF0000u : 0u);
          const uint32_t m1 = (r1 < k1 ? 0x0000FFFFu : 0u) | (r1 + 1 < k1 ? 0xFFFF0000u : 0u);
          b0 &= m0;
          b2 &= m0;
          b1 &= m1;
          b3 &= m1;
        }
        mma_bf16_16816(o[2 * np], phi, b0, b1);
        mma_bf16_16816(o[2 * np], plo, b0, b1);
        mma_bf16_16816(o[2 * np + 1], phi, b2, b3);
        mma_bf16_16816(o[2 * np + 1], plo, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    // refill this stage with the tile kDecStages ahead
    if (tid == 0 && it + kDecStages < n_st) {
      if (mbar_wait(&empty[st], (it / kDecStages) & 1, abort, status)) {
        uint8_t* base = smem + st * kDecStageBytes;
        const int key0 = k0 + (it + kDecStages) * kDecKeysPerStage;
        int row, bc;
        kv_coord(pm, b, key0, row, bc, status);
        mbar_arrive_expect_tx(&full[st], kDecStageBytes);
        tma_load_4d(base, &tm_k, &full[st], 0, g, row, bc);
        tma_load_4d(base + kDecBox, &tm_k, &full[st], 64, g, row, bc);
        tma_load_4d(base + 2 * kDecBox, &tm_v, &full[st], 0, g, row, bc);
        tma_load_4d(base + 3 * kDecBox, &tm_v, &full[st], 64, g, row, bc);
      }
    }
  }
  // Every issued copy must land before the shared memory is reused or released.
  if (tid == 0) {
    volatile int never = 0;
    const int issued = n_st;  // tiles 0..n_st-1 were all issued unless an abort cut the refill short
    for (int t = max(0, issued - kDecStages); t < issued; ++t)
      mbar_wait(&full[t % kDecStages], (t / kDecStages) & 1, &never, status);
  }
  __syncthreads();
  if (*abort) return;

  // row sums: the 4 lanes of a row hold disjoint keys
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
  // cross-warp reduction through shared memory (the ring is idle now)
  float* red = reinterpret_cast<float*>(smem);          // [4 warps][6 rows][128]
  float* lred = red + 4 * kGroup * kD;                  // [4 warps][6 rows]
  if (qrow < kGroup) {
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      red[(warp * kGroup + qrow) * kD + 8 * n + 2 * t4] = o[n][0];
      red[(warp * kGroup + qrow) * kD + 8 * n + 2 * t4 + 1] = o[n][1];
    }
    if (t4 == 0) lred[warp * kGroup + qrow] = lsum;
  }
  __syncthreads();
  const size_t part = ((size_t)b * kKVHeads + g) * n_split + split;
  for (int e = tid; e < kGroup * kD; e += kDecThreads) {
    const float v = red[e] + red[kGroup * kD + e] + red[2 * kGroup * kD + e] + red[3 * kGroup * kD + e];
    ws.o[part * kGroup * kD + e] = v;
  }
  if (tid < kGroup) ws.l[part * kGroup + tid] = lred[tid] + lred[kGroup + tid] + lred[2 * kGroup + tid] +
                                              lred[3 * kGroup + tid];
}

__global__ void __launch_bounds__(192) combine_kernel(const DecWs ws, const int32_t* __restrict__ kv_len,
                                                      int kv_add, int Tmax, int n_split, uint2* __restrict__ out,
                                                      int32_t* status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the partials of a decode grid this one depends on
  const int g = blockIdx.x, b = blockIdx.y;
  const long long L_ = (long long)__ldg(kv_len + b) + kv_add;
  const int L = L_ < 1 || L_ > Tmax ? 0 : int(L_);
  if (L < 1) {
    if (g == 0 && threadIdx.x == 0) report(status, GROK_DEV_BAD_KV_LEN);
    return;
  }
  const int r = threadIdx.x >> 5;          // head within the group
  const int d = (threadIdx.x & 31) * 4;    // 4 features per thread
  const int ns = (L + kDecSplit - 1) / kDecSplit;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  const size_t part0 = ((size_t)b * kKVHeads + g) * n_split;
  for (int s = 0; s < ns; ++s) {
    const float4 v = *reinterpret_cast<const float4*>(ws.o + ((part0 + s) * kGroup + r) * kD + d);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
    l += ws.l[(part0 + s) * kGroup + r];
  }
  const float inv = 1.0f / l;
  const int h = g * kGroup + r;
  out[((size_t)b * kQHeads + h) * (kD / 4) + d / 4] =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

}  // namespace grok

using namespace grok;

extern "C" grok_status grok_attn_decode_workspace(int B, int Tmax, size_t* bytes, int* max_splits) {
  if (B < 1 || Tmax < 1 || Tmax > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_workspace: need B >= 1, 1 <= Tmax <= %d",
                GROK_MAX_POSITION);
  const int ns = (Tmax + kDecSplit - 1) / kDecSplit;
  if (bytes) *bytes = dec_ws_bytes(B, ns);
  if (max_splits) *max_splits = ns;
  return GROK_OK;
}

static grok_status decode_args(const void* ws, size_t ws_bytes, const int32_t* kv_len, int B, int Tmax,
                               const char* who) {
  if (!ws || !kv_len) return fail(GROK_ERR_INVALID_ARG, "%s: null pointer", who);
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(GROK_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  if (B < 1 || Tmax < 1 || Tmax > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "%s: need B >= 1, 1 <= Tmax <= %d", who, GROK_MAX_POSITION);
  const int ns = (Tmax + kDecSplit - 1) / kDecSplit;
  if (ws_bytes < dec_ws_bytes(B, ns))
    return fail(GROK_ERR_INVALID_ARG, "%s: workspace of %zu bytes is smaller than the %zu needed", who, ws_bytes,
                dec_ws_bytes(B, ns));
  return GROK_OK;
}

// pdl: launch as the programmatic dependent of the kernel before it on the
// stream (the decode step's append); kv_add: kv_len[b] + kv_add keys.
static grok_status decode_launch(const grok_bf16* q_rot, const grok_bf16* k_src, const grok_bf16* v_src,
                                 uint64_t kv_rows, uint64_t kv_seqs, PageMap pm, const int32_t* kv_len, int kv_add,
                                 int B, int Tmax, void* workspace, int32_t* dev_status, void* stream,
                                 bool pdl = false) {
  grok_status st;
  int sms = 0;
  if ((st = device_sm_count(&sms)) != GROK_OK) return st;
  const int ns = (Tmax + kDecSplit - 1) / kDecSplit;
  CUtensorMap tk, tv;
  const uint64_t dims[4] = {kD, kKVHeads, kv_rows, kv_seqs};
  const uint64_t strides[3] = {kD * 2, uint64_t(kKVHeads) * kD * 2, kv_rows * kKVHeads * kD * 2};
  const uint32_t box[4] = {64, 1, kDecKeysPerStage, 1};
  if ((st = encode_tmap_bf16_4d(&tk, k_src, dims, strides, box)) != GROK_OK) return st;
  if ((st = encode_tmap_bf16_4d(&tv, v_src, dims, strides, box)) != GROK_OK) return st;
  static bool attr_set[kMaxDevices] = {};  // per device; idempotent: every thread would set the same value
  int dev = 0;
  if ((st = device_index(&dev)) != GROK_OK) return st;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
    if (e != cudaSuccess) return fail(cuda_status(e), "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kKVHeads, B, ns);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = kDecSmem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel, tk, tv, reinterpret_cast<const uint32_t*>(q_rot), kv_len,
                                     kv_add, Tmax, ns, dec_ws(workspace, B, ns), pm, dev_status);
  if (e != cudaSuccess) return fail(cuda_status(e), "decode launch: %s", cudaGetErrorString(e));
  return check_launch("decode");
}

static grok_status combine_launch(const void* workspace, const int32_t* kv_len, int kv_add, int B, int Tmax,
                                  grok_bf16* out, int32_t* dev_status, void* stream, bool pdl = false) {
  const int ns = (Tmax + kDecSplit - 1) / kDecSplit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kKVHeads, B);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel, dec_ws(const_cast<void*>(workspace), B, ns), kv_len,
                                     kv_add, Tmax, ns, reinterpret_cast<uint2*>(out), dev_status);
  if (e != cudaSuccess) return fail(cuda_status(e), "combine launch: %s", cudaGetErrorString(e));
  return check_launch("combine");
}

extern "C" grok_status grok_attn_decode(const grok_bf16* q_rot, const grok_bf16* cache_k,
                                        const grok_bf16* cache_v, const int32_t* kv_len, int B, int Tmax,
                                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                        void* stream) {
  if (!q_rot || !cache_k || !cache_v) return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode: null pointer");
  if (!aligned16(q_rot) || !aligned16(cache_k) || !aligned16(cache_v))
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode: bf16 tensors must be 16-byte aligned");
  grok_status st = decode_args(workspace, workspace_bytes, kv_len, B, Tmax, "grok_attn_decode");
  if (st != GROK_OK) return st;
  return decode_launch(q_rot, cache_k, cache_v, uint64_t(Tmax), uint64_t(B), PageMap{nullptr, 0, 0}, kv_len, 0, B,
                       Tmax, workspace, dev_status, stream);
}

extern "C" grok_status grok_attn_decode_paged(const grok_bf16* q_rot, const grok_bf16* k_pool,
                                              const grok_bf16* v_pool, int n_pages, const int32_t* block_table,
                                              int max_pages, const int32_t* kv_len, int B, void* workspace,
                                              size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (!q_rot || !k_pool || !v_pool || !block_table)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_paged: null pointer");
  if (!aligned16(q_rot) || !aligned16(k_pool) || !aligned16(v_pool))
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_paged: bf16 tensors must be 16-byte aligned");
  if (n_pages < 1 || max_pages < 1 || (long long)n_pages * GROK_PAGE_TOKENS > (1LL << 31))
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_paged: need n_pages, max_pages >= 1 (n_pages=%d, max_pages=%d)",
                n_pages, max_pages);
  const long long Tmax = (long long)max_pages * GROK_PAGE_TOKENS;
  if (Tmax > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_paged: max_pages * %d must be <= %d", GROK_PAGE_TOKENS,
                GROK_MAX_POSITION);
  grok_status st = decode_args(workspace, workspace_bytes, kv_len, B, int(Tmax), "grok_attn_decode_paged");
  if (st != GROK_OK) return st;
  return decode_launch(q_rot, k_pool, v_pool, uint64_t(n_pages) * GROK_PAGE_TOKENS, 1,
                       PageMap{block_table, max_pages, n_pages}, kv_len, 0, B, int(Tmax), workspace, dev_status,
                       stream);
}

extern "C" grok_status grok_attn_combine(const void* workspace, size_t workspace_bytes, const int32_t* kv_len,
                                         int B, int Tmax, grok_bf16* out, int32_t* dev_status, void* stream) {
  if (!out) return fail(GROK_ERR_INVALID_ARG, "grok_attn_combine: null pointer");
  if (!aligned16(out)) return fail(GROK_ERR_INVALID_ARG, "grok_attn_combine: out must be 16-byte aligned");
  grok_status st = decode_args(workspace, workspace_bytes, kv_len, B, Tmax, "grok_attn_combine");
  if (st != GROK_OK) return st;
  int sms = 0;
  if ((st = device_sm_count(&sms)) != GROK_OK) return st;
  return combine_launch(workspace, kv_len, 0, B, Tmax, out, dev_status, stream);
}

// ----------------------------------------------------------------------------
// Decode step with library-owned scratch, for callers that may not allocate.
//
// Some callers cannot hand this library a workspace: a host framework that
// owns every byte of device memory and gives its plugins no allocator, or a
// serving loop whose memory plan is fixed up front and where cudaMalloc, which
// may synchronise the device and take milliseconds, is not allowed between
// steps. For them the split-K partial sums live in this file-scope array.
// CUDA loads device code lazily by default, so a device reserves the array
// when the library's code is first used on it (possibly by the first call of
// grok_attn_decode_step_static) and holds it until the process exits; callers
// make one warm-up call per device before fixing their memory plan.
static __device__ __align__(256) unsigned char g_static_ws[GROK_STATIC_WORKSPACE_BYTES];

namespace {

// Device address of g_static_ws on each device. In host code the symbol itself
// is only a host-side stand-in, so the address must come from the runtime.
std::mutex g_static_mu;
void* g_static_ptr[64] = {nullptr};

grok_status static_ws_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(cuda_status(e), "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(GROK_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess || !p)
      return fail(cuda_status(e), "cudaGetSymbolAddress(static workspace): %s", cudaGetErrorString(e));
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return GROK_OK;
}

}  // namespace

extern "C" grok_status grok_attn_decode_step_static(const grok_bf16* q_rot, const grok_bf16* cache_k,
                                                    const grok_bf16* cache_v, const int32_t* kv_len, int B,
                                                    int Tmax, grok_bf16* out, int32_t* dev_status,
                                                    void* stream) {
  if (B < 1 || Tmax < 1 || Tmax > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_step_static: need B >= 1, 1 <= Tmax <= %d",
                GROK_MAX_POSITION);
  const int ns = (Tmax + kDecSplit - 1) / kDecSplit;
  const size_t need = dec_ws_bytes(B, ns);
  if (need > sizeof(g_static_ws))
    return fail(GROK_ERR_INVALID_ARG,
                "grok_attn_decode_step_static: B=%d, Tmax=%d needs %zu bytes of scratch, more than the %zu "
                "bytes of the library's static workspace (use grok_attn_decode with a caller workspace)",
                B, Tmax, need, sizeof(g_static_ws));
  void* ws = nullptr;
  grok_status st = static_ws_address(&ws);
  if (st != GROK_OK) return st;
  // Every partial sum the combine reads is written by the decode launch just
  // before it, so the scratch needs no clearing between calls. (A decode CTA
  // whose bounded wait gives up skips its writes and reports GROK_DEV_TIMEOUT;
  // the output is then undefined, as documented.)
  if ((st = grok_attn_decode(q_rot, cache_k, cache_v, kv_len, B, Tmax, ws, need, dev_status, stream)) != GROK_OK)
    return st;
  return grok_attn_combine(ws, need, kv_len, B, Tmax, out, dev_status, stream);
}

// ----------------------------------------------------------------------------
// One whole decode step as a chain of programmatic dependents: append (the new
// token's RoPE and cache write), split-K decode, combine. Each kernel may start
// while the one before it finishes; the decode loads the cache stages that
// cannot hold the new row before it waits for the append, the combine waits
// for the decode. The append is launched normally, so everything written on the
// stream before the call (the caches, start_pos) is complete when the decode
// starts.
static size_t step_q_bytes(int B) { return (size_t(B) * kQHeads * kD * sizeof(grok_bf16) + 255) & ~size_t(255); }

extern "C" grok_status grok_attn_decode_step_workspace(int B, int Tmax, size_t* bytes) {
  if (!bytes) return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_step_workspace: null pointer");
  if (B < 1 || Tmax < 1 || Tmax > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_step_workspace: need B >= 1, 1 <= Tmax <= %d",
                GROK_MAX_POSITION);
  *bytes = step_q_bytes(B) + dec_ws_bytes(B, (Tmax + kDecSplit - 1) / kDecSplit);
  return GROK_OK;
}

extern "C" grok_status grok_attn_decode_step(const grok_bf16* q, const grok_bf16* k, const grok_bf16* v,
                                             const int32_t* start_pos, int B, int Tmax, grok_bf16* cache_k,
                                             grok_bf16* cache_v, void* workspace, size_t workspace_bytes,
                                             grok_bf16* out, int32_t* dev_status, void* stream) {
  if (!q || !k || !v || !start_pos || !cache_k || !cache_v || !workspace || !out)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_step: null pointer");
  if (!aligned16(out)) return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_step: out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_step: workspace must be 256-byte aligned");
  size_t need = 0;
  grok_status st = grok_attn_decode_step_workspace(B, Tmax, &need);
  if (st != GROK_OK) return st;
  if (workspace_bytes < need)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_decode_step: workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, need);
  grok_bf16* q_rot = static_cast<grok_bf16*>(workspace);
  void* dws = static_cast<char*>(workspace) + step_q_bytes(B);
  if ((st = grok_rope_kv_append(q, k, v, start_pos, B, 1, Tmax, q_rot, cache_k, cache_v, dev_status, stream)) !=
      GROK_OK)
    return st;
  if ((st = decode_launch(q_rot, cache_k, cache_v, uint64_t(Tmax), uint64_t(B), PageMap{nullptr, 0, 0}, start_pos, 1,
                          B, Tmax, dws, dev_status, stream, true)) != GROK_OK)
    return st;
  return combine_launch(dws, start_pos, 1, B, Tmax, out, dev_status, stream, true);
}
