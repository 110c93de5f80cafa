// K1: RoPE on Q and K fused with the KV-cache append.
//
// Grok-1 code-reading guide, ch. 4 "model.py close reading I": §4.3 rotate_half
// (NeoX pairing of feature j with j + 64), §4.3.1 RotaryEmbedding (fp32 phase
// t * inv_freq, x * cos + rotate_half(x) * sin, cast to bf16), §4.4 (K and Q
// rotated with offset = step before the cache write; V written unrotated;
// update_into at step[b]).
//
// One CTA iteration handles one token (b, i): 64 threads evaluate the 64
// (cos, sin) pairs of its position in fp64 and round them to fp32; then the
// CTA streams the token's 48 query heads and 8 key heads (128-bit loads of 8
// bf16 of the first half and the matching 8 of the second half) and its 8
// value heads. The rotation uses separately rounded fp32 multiplies and adds
// (no FMA contraction), so the result is bit-for-bit the fp32 chain.
//
// Memory-bound: per token it reads 14 KB (q, k, v) and writes 14 KB.
#include "common.cuh"
#include "host.cuh"

namespace grok {

constexpr int kRopeThreads = 128;
constexpr int kRopeUnits = (kQHeads + kKVHeads) * 8;  // 8 groups of 8 pairs per head
constexpr int kVUnits = kKVHeads * kD / 8;             // uint4 units of V per token

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

__global__ void __launch_bounds__(kRopeThreads) rope_kv_append_kernel(
    const uint4* __restrict__ q, const uint4* __restrict__ k, const uint4* __restrict__ v,
    const int32_t* __restrict__ start_pos, int B, int T, int Tmax, uint4* __restrict__ q_rot,
    uint4* __restrict__ cache_k, uint4* __restrict__ cache_v, int32_t* status) {
  __shared__ float s_inv[64];
  __shared__ float s_cos[64];
  __shared__ float s_sin[64];
  const int tid = threadIdx.x;
  if (tid < 64) {
    // inv_freq[j] = 1 / RN32(10000^(2j/128)): fp64 power rounded once, fp32 division
    const float p32 = __double2float_rn(pow(10000.0, double(tid) / 64.0));
    s_inv[tid] = __fdiv_rn(1.0f, p32);
  }
  const long long ntok = (long long)B * T;
  for (long long tok = blockIdx.x; tok < ntok; tok += gridDim.x) {
    const int b = int(tok / T);
    const int i = int(tok - (long long)b * T);
    const int s0 = start_pos[b];
    const bool ok = s0 >= 0 && (long long)s0 + T <= Tmax && (long long)s0 + T <= GROK_MAX_POSITION;
    if (!ok) {  // uniform over the CTA
      if (tid == 0 && i == 0) report(status, GROK_DEV_BAD_START);
      continue;
    }
    const int pos = s0 + i;
    __syncthreads();  // previous token's table no longer in use (and s_inv ready)
    if (tid < 64) {
      const float ph = __fmul_rn(float(pos), s_inv[tid]);
      double sd, cd;
      sincos(double(ph), &sd, &cd);
      s_cos[tid] = __double2float_rn(cd);
      s_sin[tid] = __double2float_rn(sd);
    }
    __syncthreads();
    const size_t row = (size_t)b * Tmax + pos;
    for (int u = tid; u < kRopeUnits + kVUnits; u += kRopeThreads) {
      if (u < kRopeUnits) {
        const int head = u >> 3, c = u & 7;  // pairs j = 8c .. 8c+7
        const uint4* src;
        uint4* dst;
        if (head < kQHeads) {
          src = q + ((size_t)tok * kQHeads + head) * 16;
          dst = q_rot + ((size_t)tok * kQHeads + head) * 16;
        } else {
          const int g = head - kQHeads;
          src = k + ((size_t)tok * kKVHeads + g) * 16;
          dst = cache_k + (row * kKVHeads + g) * 16;
        }
        const uint4 x1 = __ldg(src + c);
        const uint4 x2 = __ldg(src + c + 8);
        uint4 y1, y2;
        rotate8(x1, x2, s_cos + 8 * c, s_sin + 8 * c, y1, y2);
        dst[c] = y1;
        dst[c + 8] = y2;
      } else {
        const int w = u - kRopeUnits;
        cache_v[row * (kKVHeads * 16) + w] = __ldg(v + (size_t)tok * (kKVHeads * 16) + w);
      }
    }
  }
}

}  // namespace grok

using namespace grok;

extern "C" grok_status grok_rope_kv_append(const grok_bf16* q, const grok_bf16* k, const grok_bf16* v,
                                           const int32_t* start_pos, int B, int T, int Tmax, grok_bf16* q_rot,
                                           grok_bf16* cache_k, grok_bf16* cache_v, int32_t* dev_status,
                                           void* stream) {
  if (!q || !k || !v || !start_pos || !q_rot || !cache_k || !cache_v)
    return fail(GROK_ERR_INVALID_ARG, "grok_rope_kv_append: null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_rot) || !aligned16(cache_k) ||
      !aligned16(cache_v))
    return fail(GROK_ERR_INVALID_ARG, "grok_rope_kv_append: bf16 tensors must be 16-byte aligned");
  if (B < 1 || T < 1 || Tmax < 1 || T > Tmax || T > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "grok_rope_kv_append: need B >= 1, 1 <= T <= Tmax (B=%d T=%d Tmax=%d)", B,
                T, Tmax);
  if (q == q_rot) return fail(GROK_ERR_INVALID_ARG, "grok_rope_kv_append: q_rot may not alias q");
  int sms = 0;
  grok_status st = device_sm_count(&sms);
  if (st != GROK_OK) return st;
  const long long ntok = (long long)B * T;
  const int grid = int(ntok < (long long)sms * 16 ? ntok : (long long)sms * 16);
  rope_kv_append_kernel<<<grid, kRopeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(q), reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v),
      start_pos, B, T, Tmax, reinterpret_cast<uint4*>(q_rot), reinterpret_cast<uint4*>(cache_k),
      reinterpret_cast<uint4*>(cache_v), dev_status);
  return check_launch("rope_kv_append");
}
