// Continuous-batching slot insertion: a new sequence's cache rows go into one
// batch slot of the batch cache, and the slot's step is set.
//
// Grok-1 code-reading guide, ch. 6 "model.py close reading II", §6.6.1: each
// sequence of a batch has its own int32 step, so a finished sequence's slot can
// be given to a new request; the runner inserts the new sequence's memory into
// slot i with a dynamic update along the batch axis, for the k and v caches and
// the step. The kernels never read cache rows at or beyond a sequence's step,
// so copying the used rows [0, n_rows) is equivalent to replacing the slot.
//
// One launch copies K and V with 128-bit loads and stores over a grid-stride
// loop (memory-bound: 4 KiB per row) and writes the step.
#include "common.cuh"
#include "host.cuh"

namespace grok {

constexpr int kSlotThreads = 256;

__global__ void __launch_bounds__(kSlotThreads) insert_slot_kernel(const uint4* __restrict__ src_k,
                                                                   const uint4* __restrict__ src_v,
                                                                   uint4* __restrict__ dst_k,
                                                                   uint4* __restrict__ dst_v, long long n16,
                                                                   int32_t* step, int slot, int step_value) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 k = __ldg(src_k + i), v = __ldg(src_v + i);
    dst_k[i] = k;
    dst_v[i] = v;
  }
  if (step && blockIdx.x == 0 && threadIdx.x == 0) step[slot] = step_value;
}

}  // namespace grok

using namespace grok;

extern "C" grok_status grok_kv_insert_slot(grok_bf16* cache_k, grok_bf16* cache_v, int B, int Tmax, int slot,
                                           const grok_bf16* src_k, const grok_bf16* src_v, int src_rows,
                                           int n_rows, int32_t* step, int step_value, void* stream) {
  if (!cache_k || !cache_v || !src_k || !src_v) return fail(GROK_ERR_INVALID_ARG, "grok_kv_insert_slot: null pointer");
  if (!aligned16(cache_k) || !aligned16(cache_v) || !aligned16(src_k) || !aligned16(src_v))
    return fail(GROK_ERR_INVALID_ARG, "grok_kv_insert_slot: bf16 tensors must be 16-byte aligned");
  if (B < 1 || Tmax < 1 || Tmax > GROK_MAX_POSITION || slot < 0 || slot >= B || src_rows < 0 || n_rows < 0 ||
      n_rows > src_rows || n_rows > Tmax || (step && (step_value < 0 || step_value > Tmax)))
    return fail(GROK_ERR_INVALID_ARG,
                "grok_kv_insert_slot: need 0 <= slot < B, 0 <= n_rows <= min(src_rows, Tmax), Tmax <= %d and "
                "0 <= step_value <= Tmax (B=%d Tmax=%d slot=%d src_rows=%d n_rows=%d step_value=%d)",
                GROK_MAX_POSITION, B, Tmax, slot, src_rows, n_rows, step_value);
  const size_t row = size_t(GROK_N_KV_HEADS) * GROK_HEAD_DIM;  // bf16 per cache row
  const grok_bf16* dk = cache_k + size_t(slot) * Tmax * row;
  const grok_bf16* dv = cache_v + size_t(slot) * Tmax * row;
  const size_t bytes = size_t(n_rows) * row * sizeof(grok_bf16);
  auto overlaps = [bytes](const void* a, const void* b) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bytes && y < x + bytes;
  };
  if (bytes && (overlaps(dk, src_k) || overlaps(dv, src_v) || overlaps(dk, src_v) || overlaps(dv, src_k)))
    return fail(GROK_ERR_INVALID_ARG, "grok_kv_insert_slot: the source rows overlap the slot");
  if (n_rows == 0 && !step) return GROK_OK;
  int sms = 0;
  grok_status st = device_sm_count(&sms);
  if (st != GROK_OK) return st;
  const long long n16 = (long long)n_rows * (long long)(row * sizeof(grok_bf16) / 16);
  long long blocks = (n16 + kSlotThreads - 1) / kSlotThreads;
  if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
  if (blocks < 1) blocks = 1;
  insert_slot_kernel<<<unsigned(blocks), kSlotThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(src_k), reinterpret_cast<const uint4*>(src_v),
      reinterpret_cast<uint4*>(const_cast<grok_bf16*>(dk)), reinterpret_cast<uint4*>(const_cast<grok_bf16*>(dv)),
      n16, step, slot, step_value);
  return check_launch("insert_slot");
}
