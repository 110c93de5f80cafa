// Host-side helpers shared by the entry points: thread-local error text,
// argument checks, device capability and TMA tensor-map encoding.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "grok_attn.h"

namespace grok {

// Record a message for grok_last_error() and return `s`.
grok_status fail(grok_status s, const char* fmt, ...);

// Status for a failed CUDA runtime call: GROK_ERR_DEVICE_FAULT for the sticky
// errors that leave the context unusable, GROK_ERR_CUDA otherwise.
grok_status cuda_status(cudaError_t e);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Outputs written with 32-byte stores (st.global.v8.b32) need 32-byte alignment.
inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// The current device must be compute capability 10.3; returns its SM count.
grok_status device_sm_count(int* sm_count);

// Index of the current device, for one-time setup that must be repeated on
// every device (function attributes live in each device's context).
constexpr int kMaxDevices = 64;
grok_status device_index(int* dev);

// Launch-error check after a kernel launch.
grok_status check_launch(const char* what);

// 4-D bf16 tensor map, 128-byte swizzle, zero fill out of bounds.
// dims innermost first; strides in bytes for dims 1..3.
grok_status encode_tmap_bf16_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                                const uint64_t strides[3], const uint32_t box[4]);
// The same for fp16 elements.
grok_status encode_tmap_f16_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                               const uint64_t strides[3], const uint32_t box[4]);

// 2-D uint8 tensor map (dims innermost first, row stride in bytes), no
// swizzle, zero fill out of bounds.
grok_status encode_tmap_u8_2d(CUtensorMap* map, const void* base, const uint64_t dims[2], uint64_t row_stride,
                              const uint32_t box[2]);

// Small-M int8 weight-only Linear (int8_small.cu): shape rule and launch.
bool small_int8_ok(int M, int K, int N);
grok_status linear_int8_small(const grok_bf16* x, const int8_t* w8, const float* scales, int M, int K, int N,
                              grok_bf16* y, int32_t* dev_status, void* stream);

}  // namespace grok
