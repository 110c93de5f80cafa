// Host-buffer prefill pipeline: grok_rope_kv_append_table (with a cos/sin table
// of positions [0, Tmax) computed once at create) + grok_attn_prefill_ws (the
// prefill with fp16 softmax weights) fed from host memory, with the copies of
// one step overlapping the kernels of the steps around it.
//
// Three streams: host-to-device copies, kernels, device-to-host copies. Inputs
// and outputs are double-buffered on the device (two slots, used alternately);
// q_rot is shared because every kernel runs in order on the kernel stream.
// Ordering per slot, by events:
//   copy-in of step n   waits for the kernels of step n-2 (they read the slot's inputs)
//   kernels of step n   wait for the copy-in of step n, and for the copy-out of
//                       step n-2 (they overwrite the slot's output)
//   copy-out of step n  waits for the kernels of step n
#include "host.cuh"

struct grok_prefill_pipe {
  int dev = 0, B = 0, T = 0, Tmax = 0;
  grok_bf16* cache_k = nullptr;
  grok_bf16* cache_v = nullptr;
  cudaStream_t s_in = nullptr, s_run = nullptr, s_out = nullptr;
  struct Slot {
    grok_bf16 *q = nullptr, *k = nullptr, *v = nullptr, *out = nullptr;
    int32_t *start = nullptr, *valid = nullptr;
    cudaEvent_t in_done = nullptr, run_done = nullptr, out_done = nullptr;
    bool used = false;
  } slot[2];
  grok_bf16* q_rot = nullptr;
  void* pf_ws = nullptr;      // grok_attn_prefill_ws workspace (used in kernel-stream order)
  float* cos_tab = nullptr;   // RoPE table of positions [0, Tmax)
  float* sin_tab = nullptr;
  size_t pf_ws_bytes = 0;
  int32_t* status = nullptr;  // OR of every step's device status since the last wait
  long long submitted = 0;
};

namespace grok {
namespace {

// Makes the pipeline's device current for the lifetime of the guard.
struct DeviceGuard {
  int prev = -1;
  cudaError_t err = cudaSuccess;
  explicit DeviceGuard(int dev) {
    err = cudaGetDevice(&prev);
    if (err == cudaSuccess && prev != dev) err = cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

size_t q_bytes(const grok_prefill_pipe* p) { return size_t(p->B) * p->T * GROK_N_Q_HEADS * GROK_HEAD_DIM * sizeof(grok_bf16); }
size_t kv_bytes(const grok_prefill_pipe* p) { return size_t(p->B) * p->T * GROK_N_KV_HEADS * GROK_HEAD_DIM * sizeof(grok_bf16); }

void release(grok_prefill_pipe* p) {
  for (auto& s : p->slot) {
    cudaFree(s.q);
    cudaFree(s.k);
    cudaFree(s.v);
    cudaFree(s.out);
    cudaFree(s.start);
    cudaFree(s.valid);
    if (s.in_done) cudaEventDestroy(s.in_done);
    if (s.run_done) cudaEventDestroy(s.run_done);
    if (s.out_done) cudaEventDestroy(s.out_done);
  }
  cudaFree(p->q_rot);
  cudaFree(p->pf_ws);
  cudaFree(p->cos_tab);
  cudaFree(p->sin_tab);
  cudaFree(p->status);
  if (p->s_in) cudaStreamDestroy(p->s_in);
  if (p->s_run) cudaStreamDestroy(p->s_run);
  if (p->s_out) cudaStreamDestroy(p->s_out);
  delete p;
}

grok_status cuda_fail(const char* what, cudaError_t e) {
  return fail(cuda_status(e), "grok_prefill_pipe: %s: %s", what, cudaGetErrorString(e));
}

}  // namespace
}  // namespace grok

using namespace grok;

extern "C" grok_status grok_prefill_pipe_create(int B, int T, int Tmax, grok_bf16* cache_k, grok_bf16* cache_v,
                                                grok_prefill_pipe** pipe) {
  if (!pipe || !cache_k || !cache_v) return fail(GROK_ERR_INVALID_ARG, "grok_prefill_pipe_create: null pointer");
  *pipe = nullptr;
  if (B < 1 || T < 1 || Tmax < 1 || T > Tmax || Tmax > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG,
                "grok_prefill_pipe_create: need B >= 1, 1 <= T <= Tmax <= %d (B=%d T=%d Tmax=%d)", GROK_MAX_POSITION,
                B, T, Tmax);
  if (!aligned16(cache_k) || !aligned16(cache_v))
    return fail(GROK_ERR_INVALID_ARG, "grok_prefill_pipe_create: caches must be 16-byte aligned");
  int sms = 0;
  grok_status st = device_sm_count(&sms);
  if (st != GROK_OK) return st;
  grok_prefill_pipe* p = new grok_prefill_pipe;
  p->B = B;
  p->T = T;
  p->Tmax = Tmax;
  p->cache_k = cache_k;
  p->cache_v = cache_v;
  cudaError_t e = cudaGetDevice(&p->dev);
  const size_t nq = q_bytes(p), nkv = kv_bytes(p), ni = size_t(B) * sizeof(int32_t);
  for (auto& s : p->slot) {
    if (e == cudaSuccess) e = cudaMalloc(&s.q, nq);
    if (e == cudaSuccess) e = cudaMalloc(&s.k, nkv);
    if (e == cudaSuccess) e = cudaMalloc(&s.v, nkv);
    if (e == cudaSuccess) e = cudaMalloc(&s.out, nq);
    if (e == cudaSuccess) e = cudaMalloc(&s.start, ni);
    if (e == cudaSuccess) e = cudaMalloc(&s.valid, ni);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.in_done, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.run_done, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.out_done, cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaMalloc(&p->q_rot, nq);
  if (e == cudaSuccess && (st = grok_attn_prefill_workspace(B, Tmax, &p->pf_ws_bytes)) != GROK_OK) {
    release(p);
    return st;
  }
  if (e == cudaSuccess) e = cudaMalloc(&p->pf_ws, p->pf_ws_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&p->cos_tab, size_t(Tmax) * 64 * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&p->sin_tab, size_t(Tmax) * 64 * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&p->status, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(p->status, 0, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->s_run, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    release(p);
    return cuda_fail("create", e);
  }
  if ((st = grok_rope_cos_sin(0, Tmax, p->cos_tab, p->sin_tab, p->s_run)) != GROK_OK) {
    release(p);
    return st;
  }
  *pipe = p;
  return GROK_OK;
}

extern "C" grok_status grok_prefill_pipe_submit(grok_prefill_pipe* p, const grok_bf16* q, const grok_bf16* k,
                                                const grok_bf16* v, const int32_t* start_pos,
                                                const int32_t* valid_len, grok_bf16* out) {
  if (!p || !q || !k || !v || !start_pos || !out)
    return fail(GROK_ERR_INVALID_ARG, "grok_prefill_pipe_submit: null pointer");
  DeviceGuard guard(p->dev);
  if (guard.err != cudaSuccess) return cuda_fail("set device", guard.err);
  auto& s = p->slot[p->submitted & 1];
  const size_t nq = q_bytes(p), nkv = kv_bytes(p), ni = size_t(p->B) * sizeof(int32_t);
  cudaError_t e = cudaSuccess;
  // copy-in: the slot's inputs are free once the kernels of its previous step ran
  if (s.used) e = cudaStreamWaitEvent(p->s_in, s.run_done, 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(s.q, q, nq, cudaMemcpyHostToDevice, p->s_in);
  if (e == cudaSuccess) e = cudaMemcpyAsync(s.k, k, nkv, cudaMemcpyHostToDevice, p->s_in);
  if (e == cudaSuccess) e = cudaMemcpyAsync(s.v, v, nkv, cudaMemcpyHostToDevice, p->s_in);
  if (e == cudaSuccess) e = cudaMemcpyAsync(s.start, start_pos, ni, cudaMemcpyHostToDevice, p->s_in);
  if (e == cudaSuccess && valid_len) e = cudaMemcpyAsync(s.valid, valid_len, ni, cudaMemcpyHostToDevice, p->s_in);
  if (e == cudaSuccess) e = cudaEventRecord(s.in_done, p->s_in);
  // kernels: after the copy-in, and after the slot's previous output left the device
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p->s_run, s.in_done, 0);
  if (e == cudaSuccess && s.used) e = cudaStreamWaitEvent(p->s_run, s.out_done, 0);
  if (e != cudaSuccess) return cuda_fail("enqueue copy-in", e);
  grok_status st = grok_rope_kv_append_table(s.q, s.k, s.v, s.start, p->B, p->T, p->Tmax, p->cos_tab, p->sin_tab,
                                             p->Tmax, p->q_rot, p->cache_k, p->cache_v, p->status, p->s_run);
  if (st != GROK_OK) return st;
  st = grok_attn_prefill_ws(p->q_rot, p->cache_k, p->cache_v, s.start, valid_len ? s.valid : nullptr, p->B, p->T,
                            p->Tmax, s.out, p->pf_ws, p->pf_ws_bytes, 0, p->status, p->s_run);
  if (st != GROK_OK) return st;
  e = cudaEventRecord(s.run_done, p->s_run);
  // copy-out
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p->s_out, s.run_done, 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(out, s.out, nq, cudaMemcpyDeviceToHost, p->s_out);
  if (e == cudaSuccess) e = cudaEventRecord(s.out_done, p->s_out);
  if (e != cudaSuccess) return cuda_fail("enqueue copy-out", e);
  s.used = true;
  ++p->submitted;
  return GROK_OK;
}

extern "C" grok_status grok_prefill_pipe_wait(grok_prefill_pipe* p, int32_t* dev_status) {
  if (!p) return fail(GROK_ERR_INVALID_ARG, "grok_prefill_pipe_wait: null pipeline");
  DeviceGuard guard(p->dev);
  if (guard.err != cudaSuccess) return cuda_fail("set device", guard.err);
  cudaError_t e = cudaStreamSynchronize(p->s_in);
  if (e == cudaSuccess) e = cudaStreamSynchronize(p->s_run);
  if (e == cudaSuccess) e = cudaStreamSynchronize(p->s_out);
  int32_t bits = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&bits, p->status, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && bits != 0) e = cudaMemset(p->status, 0, sizeof(int32_t));
  if (e != cudaSuccess) return cuda_fail("wait", e);
  if (dev_status) *dev_status = bits;
  return GROK_OK;
}

extern "C" grok_status grok_prefill_pipe_destroy(grok_prefill_pipe* p) {
  if (!p) return GROK_OK;
  grok_status st = grok_prefill_pipe_wait(p, nullptr);
  {
    DeviceGuard guard(p->dev);
    release(p);
  }
  return st;
}
