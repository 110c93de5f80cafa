// K1: RoPE on Q and K fused with the KV-cache append.
//
// Grok-1 code-reading guide, ch. 4 "model.py close reading I": §4.3 rotate_half
// (NeoX pairing of feature j with j + 64), §4.3.1 RotaryEmbedding (fp32 phase
// t * inv_freq, x * cos + rotate_half(x) * sin, cast to bf16), §4.4 (K and Q
// rotated with offset = step before the cache write; V written unrotated;
// update_into at step[b]).
//
// A team of 1, 2, 4 or 8 warps handles one token (b, i) (more warps per token
// when there are few tokens): each warp loads its share of the token's 48
// query heads and 8 key heads (128-bit loads of 8 bf16 of the first half and
// the matching 8 of the second half) and of its 8 value heads, evaluates the
// 64 (cos, sin) pairs of the token's position in fp64 (rounded to fp32) while
// those loads are in flight, then rotates and stores. The rotation uses
// separately rounded fp32 multiplies and adds (no FMA contraction), so the
// result is bit-for-bit the fp32 chain.
//
// Memory-bound: per token it reads 14 KB (q, k, v) and writes 14 KB.
//
// Table variant (kTab, grok_rope_kv_append_table): the (cos, sin) pairs are
// read from a table of positions [0, n) that grok_rope_cos_sin filled once
// (the values depend only on the position, so one table serves every layer
// and step), instead of being evaluated per token: 512 bytes of L2-resident
// table per token in place of 64 fp64 cos/sin evaluations. The table holds
// the same fp32 values the evaluation gives, so the bits are the same.
#include "common.cuh"
#include "host.cuh"
#include "rope_math.cuh"

namespace grok {

constexpr int kRopeThreads = 128;

__device__ __forceinline__ void rotate8(const uint4& x1, const uint4& x2, const float* c, const float* s,
                                        uint4& y1, uint4& y2) {
  const uint32_t a[4] = {x1.x, x1.y, x1.z, x1.w};
  const uint32_t b[4] = {x2.x, x2.y, x2.z, x2.w};
  uint32_t o1[4], o2[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float a0 = bf16lo_to_f32(a[w]), a1 = bf16hi_to_f32(a[w]);
    const float b0 = bf16lo_to_f32(b[w]), b1 = bf16hi_to_f32(b[w]);
    const float c0 = c[2 * w], c1 = c[2 * w + 1], s0 = s[2 * w], s1 = s[2 * w + 1];
    // x'[j] = x[j] cos - x[j+64] sin ; x'[j+64] = x[j+64] cos + x[j] sin
    const float y1a = __fadd_rn(__fmul_rn(a0, c0), -__fmul_rn(b0, s0));
    const float y1b = __fadd_rn(__fmul_rn(a1, c1), -__fmul_rn(b1, s1));
    const float y2a = __fadd_rn(__fmul_rn(b0, c0), __fmul_rn(a0, s0));
    const float y2b = __fadd_rn(__fmul_rn(b1, c1), __fmul_rn(a1, s1));
    o1[w] = pack_bf16x2(y1a, y1b);
    o2[w] = pack_bf16x2(y2a, y2b);
  }
  y1 = make_uint4(o1[0], o1[1], o1[2], o1[3]);
  y2 = make_uint4(o2[0], o2[1], o2[2], o2[3]);
}

// A team of `team` warps (1, 2, 4 or 8) per token, grid-stride over tokens
// with no CTA-wide barrier. Warp w of the team takes the rotation units (8
// pairs of one head) and value units whose index m satisfies m % team == w: it
// issues all their loads first, then evaluates the token's 64 (cos, sin) pairs
// in fp64 into its own shared-memory slice while the loads are in flight (the
// fp64 work, slow on this part, overlaps the memory latency instead of
// preceding it), then rotates and stores. Large batches use one warp per
// token; a handful of tokens (a decode step) spreads each token over eight
// warps.
constexpr int kRopeWarps = kRopeThreads / 32;

template <int team, bool kTab>
__global__ void __launch_bounds__(kRopeThreads) rope_kv_append_kernel(
    const uint4* __restrict__ q, const uint4* __restrict__ k, const uint4* __restrict__ v,
    const int32_t* __restrict__ start_pos, int B, int T, int Tmax, uint4* __restrict__ q_rot,
    uint4* __restrict__ cache_k, uint4* __restrict__ cache_v, PageMap pm, const float4* __restrict__ cos_tab,
    const float4* __restrict__ sin_tab, int tab_n, int32_t* status) {
  // A kernel launched as this grid's programmatic dependent (the decode step's
  // split-K decode) may start at once; it waits for this grid before reading
  // what it writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float s_inv[64];
  __shared__ float s_cos[kRopeWarps][64];
  __shared__ float s_sin[kRopeWarps][64];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (!kTab) {
    if (tid < 64) s_inv[tid] = rope_inv_freq(tid);
    __syncthreads();
  }
  const long long ntok = (long long)B * T;
  const long long gw = (long long)blockIdx.x * kRopeWarps + warp;
  const int member = int(gw % team);
  const long long n_teams = (long long)gridDim.x * kRopeWarps / team;
  for (long long tok = gw / team; tok < ntok; tok += n_teams) {
    const int b = int(tok / T);
    const int i = int(tok - (long long)b * T);
    const int s0 = __ldg(start_pos + b);
    const bool ok = s0 >= 0 && (long long)s0 + T <= Tmax && (long long)s0 + T <= (kTab ? tab_n : GROK_MAX_POSITION);
    if (!ok) {  // uniform over the warp
      if (lane == 0 && i == 0 && member == 0) report(status, GROK_DEV_BAD_START);
      continue;
    }
    const int pos = s0 + i;
    // cache row of (b, pos): contiguous b * Tmax + pos, paged page * 128 + pos % 128; a
    // token whose page id is out of range still gets its q_rot but no cache write
    size_t row = (size_t)b * Tmax + pos;
    bool kv_ok = true;
    if (pm.table) {
      const int pg = __ldg(pm.table + (size_t)b * pm.max_pages + pos / GROK_PAGE_TOKENS);
      kv_ok = pg >= 0 && pg < pm.n_pages;
      if (!kv_ok && lane == 0 && member == 0) report(status, GROK_DEV_BAD_PAGE);
      row = (size_t)(kv_ok ? pg : 0) * GROK_PAGE_TOKENS + pos % GROK_PAGE_TOKENS;
    }
    const uint4* qsrc = q + (size_t)tok * kQHeads * 16;
    const uint4* ksrc = k + (size_t)tok * kKVHeads * 16;
    uint4* qdst = q_rot + (size_t)tok * kQHeads * 16;
    uint4* kdst = cache_k + row * kKVHeads * 16;
    // 56 heads x 8 pair groups = 448 rotation units: unit u = head * 8 + c (pairs 8c .. 8c+7)
    uint4 x1[14], x2[14];
#pragma unroll
    for (int m = 0; m < 14; ++m) {
      if (m % team != member) continue;
      const int u = lane + 32 * m, head = u >> 3, c = u & 7;
      const uint4* src = head < kQHeads ? qsrc + head * 16 : ksrc + (head - kQHeads) * 16;
      x1[m] = __ldg(src + c);
      x2[m] = __ldg(src + c + 8);
    }
    uint4 vv[4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
      if (m % team == member) vv[m] = __ldg(v + (size_t)tok * (kKVHeads * 16) + lane + 32 * m);
    // Every unit of this lane rotates pairs 8c .. 8c+7 with c = lane % 8.
    float tc[8], ts[8];
    if (kTab) {
      const size_t t0 = (size_t)pos * 16 + 2 * (lane & 7);  // float4 index of (pos, 8c)
      const float4 c0 = __ldg(cos_tab + t0), c1 = __ldg(cos_tab + t0 + 1);
      const float4 d0 = __ldg(sin_tab + t0), d1 = __ldg(sin_tab + t0 + 1);
      tc[0] = c0.x, tc[1] = c0.y, tc[2] = c0.z, tc[3] = c0.w, tc[4] = c1.x, tc[5] = c1.y, tc[6] = c1.z, tc[7] = c1.w;
      ts[0] = d0.x, ts[1] = d0.y, ts[2] = d0.z, ts[3] = d0.w, ts[4] = d1.x, ts[5] = d1.y, ts[6] = d1.z, ts[7] = d1.w;
    } else {
      __syncwarp();  // the previous token's table is no longer read
      rope_cos_sin(__fmul_rn(float(pos), s_inv[lane]), s_cos[warp][lane], s_sin[warp][lane]);
      rope_cos_sin(__fmul_rn(float(pos), s_inv[lane + 32]), s_cos[warp][lane + 32], s_sin[warp][lane + 32]);
      __syncwarp();
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        tc[e] = s_cos[warp][8 * (lane & 7) + e];
        ts[e] = s_sin[warp][8 * (lane & 7) + e];
      }
    }
#pragma unroll
    for (int m = 0; m < 14; ++m) {
      if (m % team != member) continue;
      const int u = lane + 32 * m, head = u >> 3, c = u & 7;
      if (head >= kQHeads && !kv_ok) continue;
      uint4 y1, y2;
      rotate8(x1[m], x2[m], tc, ts, y1, y2);
      uint4* dst = head < kQHeads ? qdst + head * 16 : kdst + (head - kQHeads) * 16;
      dst[c] = y1;
      dst[c + 8] = y2;
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
      if (m % team == member && kv_ok) cache_v[row * (kKVHeads * 16) + lane + 32 * m] = vv[m];
  }
}

// The fp32 table the append kernel uses: entry (p, j) for positions
// [p0, p0 + n) and frequencies j < 64.
__global__ void rope_table_kernel(int p0, int n, float* __restrict__ cos_out, float* __restrict__ sin_out) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)n * 64) return;
  const int j = int(idx & 63);
  const int pos = p0 + int(idx >> 6);
  float c, s;
  rope_cos_sin(__fmul_rn(float(pos), rope_inv_freq(j)), c, s);
  cos_out[idx] = c;
  sin_out[idx] = s;
}

}  // namespace grok

using namespace grok;

static grok_status append_launch(const grok_bf16* q, const grok_bf16* k, const grok_bf16* v,
                                 const int32_t* start_pos, int B, int T, int Tmax, grok_bf16* q_rot,
                                 grok_bf16* cache_k, grok_bf16* cache_v, PageMap pm, int32_t* dev_status,
                                 void* stream, const char* name, const float* cos_tab = nullptr,
                                 const float* sin_tab = nullptr, int tab_n = 0) {
  if (!q || !k || !v || !start_pos || !q_rot || !cache_k || !cache_v)
    return fail(GROK_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_rot) || !aligned16(cache_k) ||
      !aligned16(cache_v))
    return fail(GROK_ERR_INVALID_ARG, "%s: bf16 tensors must be 16-byte aligned", name);
  if (B < 1 || T < 1 || Tmax < 1 || T > Tmax || T > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "%s: need B >= 1, 1 <= T <= Tmax (B=%d T=%d Tmax=%d)", name, B, T, Tmax);
  if (q == q_rot) return fail(GROK_ERR_INVALID_ARG, "%s: q_rot may not alias q", name);
  int sms = 0;
  grok_status st = device_sm_count(&sms);
  if (st != GROK_OK) return st;
  const long long ntok = (long long)B * T;
  // warps per token: as many as keep about four resident CTAs' worth of warps per SM busy, up to 8
  int team = 1;
  while (team < 8 && ntok * team * 2 <= (long long)sms * 4 * kRopeWarps) team *= 2;
  const long long want = (ntok * team + kRopeWarps - 1) / kRopeWarps;
  const bool tab = cos_tab != nullptr;
  // The table variant takes one token per team and leaves the balancing to the
  // CTA scheduler (a fixed grid striding over the tokens left a last round in
  // which a third of the warps had no token: B8 T2048 96.6 -> 89.3 us). The
  // evaluating variant (254 registers, two CTAs per SM) keeps its grid of at
  // most 8 CTAs per SM striding over the tokens.
  const long long cap = tab ? (1ll << 30) : (long long)sms * 8;
  const int grid = int(want < cap ? want : cap);
  auto kernel = tab ? (team == 8   ? rope_kv_append_kernel<8, true>
                       : team == 4 ? rope_kv_append_kernel<4, true>
                       : team == 2 ? rope_kv_append_kernel<2, true>
                                   : rope_kv_append_kernel<1, true>)
                    : (team == 8   ? rope_kv_append_kernel<8, false>
                       : team == 4 ? rope_kv_append_kernel<4, false>
                       : team == 2 ? rope_kv_append_kernel<2, false>
                                   : rope_kv_append_kernel<1, false>);
  // Few tokens (a decode step): the SMs' shared-memory split is set for the
  // decode kernel that may join them, not for this kernel's 2 KB.
  static bool carve_set[kMaxDevices] = {};  // per device; idempotent: every thread would set the same values
  int dev = 0;
  if ((st = device_index(&dev)) != GROK_OK) return st;
  if (!carve_set[dev]) {
    for (auto kf : {rope_kv_append_kernel<8, false>, rope_kv_append_kernel<4, false>, rope_kv_append_kernel<2, false>,
                    rope_kv_append_kernel<8, true>, rope_kv_append_kernel<4, true>, rope_kv_append_kernel<2, true>}) {
      cudaError_t e = cudaFuncSetAttribute(kf, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           int(cudaSharedmemCarveoutMaxShared));
      if (e != cudaSuccess) return fail(cuda_status(e), "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    }
    carve_set[dev] = true;
  }
  kernel<<<grid, kRopeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(q), reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v),
      start_pos, B, T, Tmax, reinterpret_cast<uint4*>(q_rot), reinterpret_cast<uint4*>(cache_k),
      reinterpret_cast<uint4*>(cache_v), pm, reinterpret_cast<const float4*>(cos_tab),
      reinterpret_cast<const float4*>(sin_tab), tab_n, dev_status);
  return check_launch("rope_kv_append");
}

extern "C" grok_status grok_rope_kv_append_table(const grok_bf16* q, const grok_bf16* k, const grok_bf16* v,
                                                 const int32_t* start_pos, int B, int T, int Tmax,
                                                 const float* cos_tab, const float* sin_tab, int tab_positions,
                                                 grok_bf16* q_rot, grok_bf16* cache_k, grok_bf16* cache_v,
                                                 int32_t* dev_status, void* stream) {
  if (!cos_tab || !sin_tab) return fail(GROK_ERR_INVALID_ARG, "grok_rope_kv_append_table: null table");
  if (!aligned16(cos_tab) || !aligned16(sin_tab))
    return fail(GROK_ERR_INVALID_ARG, "grok_rope_kv_append_table: tables must be 16-byte aligned");
  if (tab_positions < 1 || tab_positions > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "grok_rope_kv_append_table: need 1 <= tab_positions <= %d", GROK_MAX_POSITION);
  return append_launch(q, k, v, start_pos, B, T, Tmax, q_rot, cache_k, cache_v, PageMap{nullptr, 0, 0}, dev_status,
                       stream, "grok_rope_kv_append_table", cos_tab, sin_tab, tab_positions);
}

extern "C" grok_status grok_rope_kv_append(const grok_bf16* q, const grok_bf16* k, const grok_bf16* v,
                                           const int32_t* start_pos, int B, int T, int Tmax, grok_bf16* q_rot,
                                           grok_bf16* cache_k, grok_bf16* cache_v, int32_t* dev_status,
                                           void* stream) {
  return append_launch(q, k, v, start_pos, B, T, Tmax, q_rot, cache_k, cache_v, PageMap{nullptr, 0, 0}, dev_status,
                       stream, "grok_rope_kv_append");
}

extern "C" grok_status grok_rope_kv_append_paged(const grok_bf16* q, const grok_bf16* k, const grok_bf16* v,
                                                 const int32_t* start_pos, int B, int T, grok_bf16* q_rot,
                                                 grok_bf16* k_pool, grok_bf16* v_pool, int n_pages,
                                                 const int32_t* block_table, int max_pages, int32_t* dev_status,
                                                 void* stream) {
  if (!block_table) return fail(GROK_ERR_INVALID_ARG, "grok_rope_kv_append_paged: null block table");
  if (n_pages < 1 || max_pages < 1 || (long long)n_pages * GROK_PAGE_TOKENS > (1LL << 31) ||
      (long long)max_pages * GROK_PAGE_TOKENS > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG,
                "grok_rope_kv_append_paged: need n_pages, max_pages >= 1, max_pages * %d <= %d "
                "(n_pages=%d max_pages=%d)",
                GROK_PAGE_TOKENS, GROK_MAX_POSITION, n_pages, max_pages);
  return append_launch(q, k, v, start_pos, B, T, max_pages * GROK_PAGE_TOKENS, q_rot, k_pool, v_pool,
                       PageMap{block_table, max_pages, n_pages}, dev_status, stream, "grok_rope_kv_append_paged");
}

extern "C" grok_status grok_rope_cos_sin(int first_position, int n_positions, float* cos_out, float* sin_out,
                                         void* stream) {
  if (!cos_out || !sin_out) return fail(GROK_ERR_INVALID_ARG, "grok_rope_cos_sin: null pointer");
  if (first_position < 0 || n_positions < 1 || (long long)first_position + n_positions > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "grok_rope_cos_sin: positions must lie in [0, %d)", GROK_MAX_POSITION);
  int sms = 0;
  grok_status st = device_sm_count(&sms);
  if (st != GROK_OK) return st;
  const long long total = (long long)n_positions * 64;
  rope_table_kernel<<<unsigned((total + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      first_position, n_positions, cos_out, sin_out);
  return check_launch("rope_table");
}
