// Small-M int8 weight-only Linear (decode-sized batches, M <= 32):
//   y [M, N] = x [M, K] . dequant(w8 [K, N], scales [N])
// Grok-1 code-reading guide, ch. 4 "model.py close reading I": §4.1 Linear with
// QuantizedWeight8bit, §4.1.1 (int8 weight, one fp32 scale per output column,
// dequantized as astype(scales.dtype) * scales, then astype(bf16)).
//
// At decode sizes the product is bound by reading the int8 weight once (1 byte
// per element, 50 MB for the Q/K/V shape); x is tiny and stays in L2.
//
// Grid: (8, N / 256) in clusters of 8 CTAs along K. CTA (r, nb) owns output
// columns [256 nb, 256 nb + 256) and weight rows [r K/8, (r+1) K/8). Each
// weight row slice is 256 contiguous bytes, and 2 CTAs fit per SM, so the
// whole grid of the Q/K/V shape (256 CTAs) is resident at once and every CTA
// streams its own 196 KB.
//
// Per CTA (8 warps): a 3-stage ring of 64-row stages loaded by TMA, each
// holding the stage's weight tile [64 rows x 256 bytes] and x tile
// [16 MT rows x 64 bf16] (rows >= M are zero-filled by TMA; 128-byte swizzle).
// Per stage:
//   1. every warp loads the stage's A fragments of x (ldmatrix) into registers;
//   2. all 256 threads dequantize the weight tile into a bf16 tile in shared
//      memory, each element exactly as grok_dequant_int8 does it: the byte is
//      turned into a float by placing it in the mantissa of 2^23 (byte permute)
//      and subtracting 2^23 + 128, multiplied by its column scale with one
//      fp32 rounding, then rounded to nearest-even bf16;
//   3. a CTA barrier; the stage is free and thread 0 refills it with TMA;
//   4. warp w multiplies the tile's columns [32 w, 32 w + 32) (mma.sync
//      m16n8k16, B fragments by ldmatrix.trans), accumulating in fp32;
//   5. a CTA barrier before the next stage overwrites the bf16 tile.
// The 8 CTAs of a cluster then add their partial sums through distributed
// shared memory in a fixed rank order (so results do not depend on
// scheduling): CTA r sums columns [32 r, 32 r + 32) of all 8 partials, rounds
// to bf16 and writes them.
#include "common.cuh"
#include "host.cuh"

namespace grok {

constexpr int kI8Cluster = 8;                      // CTAs along K
constexpr int kI8Cols = 256;                       // output columns per CTA
constexpr int kI8Rows = 64;                        // weight rows per stage
constexpr int kI8Stages = 3;
constexpr int kI8Threads = 256;
constexpr int kI8XBytes = 32 * kI8Rows * 2;        // x tile (room for 32 rows)
constexpr int kI8WBytes = kI8Rows * kI8Cols;       // int8 weight tile, 16 KB
constexpr int kI8StageBytes = kI8XBytes + kI8WBytes;
constexpr int kI8TileRow = kI8Cols * 2 + 16;       // bf16 tile row: 512 bytes + 16 of padding
constexpr int kI8Tile = kI8Rows * kI8TileRow;
constexpr int kI8Smem = kI8Stages * kI8StageBytes + kI8Tile + 64 + 1024;
static_assert(32 * kI8Cols * 4 <= kI8Stages * kI8StageBytes, "partial sums must fit in the ring");

// 2-d tile load; the map must have been encoded with rank 2 (the instruction's
// dimensionality must equal the map's rank).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

// Four signed bytes -> four exact floats: byte b + 128 placed in the low
// mantissa bits of 2^23, minus 2^23 + 128.
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float (&f)[4]) {
  const uint32_t u = w ^ 0x80808080u;
  const uint64_t bias = f2_pack(8388736.0f, 8388736.0f);
  float a, b, c, d;
  f2_unpack(f2_sub(f2_pack(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)),
                           __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541))),
                   bias),
            a, b);
  f2_unpack(f2_sub(f2_pack(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)),
                           __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543))),
                   bias),
            c, d);
  f[0] = a, f[1] = b, f[2] = c, f[3] = d;
}

template <int MT>
__global__ void __cluster_dims__(kI8Cluster, 1, 1) __launch_bounds__(kI8Threads, 2)
    linear_int8_small_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                             const float* __restrict__ scales, int M, int K, int N, uint32_t* __restrict__ y,
                             int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tile = smem + kI8Stages * kI8StageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(tile + kI8Tile);
  int* abort_flag = reinterpret_cast<int*>(full + kI8Stages);
  volatile int* abort = abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = blockIdx.x;  // position in the cluster = K slice
  const int n0 = blockIdx.y * kI8Cols;
  const int rows = K / kI8Cluster;
  const int k_first = rank * rows;
  const int n_st = rows / kI8Rows;
  constexpr uint32_t kStageTx = uint32_t(16 * MT * kI8Rows * 2 + kI8WBytes);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kI8Stages; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_w);
  }
  __syncthreads();
  auto load_stage = [&](int it) {
    uint8_t* base = smem + (it % kI8Stages) * kI8StageBytes;
    const int k = k_first + it * kI8Rows;
    mbar_arrive_expect_tx(&full[it % kI8Stages], kStageTx);
    tma_load_4d(base, &tm_x, &full[it % kI8Stages], k, 0, 0, 0);  // x's map is 4-d (rows, 1, 1)
    tma_load_2d(base + kI8XBytes, &tm_w, &full[it % kI8Stages], n0, k);
  };
  if (threadIdx.x == 0)
    for (int it = 0; it < kI8Stages && it < n_st; ++it) load_stage(it);

  // this lane's 8 dequant columns 8 lane .. 8 lane + 7 and their scales
  float sc[8];
  {
    const float4* s4 = reinterpret_cast<const float4*>(scales + n0 + 8 * lane);
    const float4 a = __ldg(s4), b = __ldg(s4 + 1);
    sc[0] = a.x, sc[1] = a.y, sc[2] = a.z, sc[3] = a.w, sc[4] = b.x, sc[5] = b.y, sc[6] = b.z, sc[7] = b.w;
  }
  float acc[MT][4][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
  const int mi = lane >> 3, mr = lane & 7;
  const uint32_t tile_s = smem_u32(tile);
  int issued = min(kI8Stages, n_st);  // stages whose copies were started (thread 0's count)
  int consumed = 0;                    // stages whose copies landed (every thread's count)

  for (int it = 0; it < n_st; ++it) {
    const int st = it % kI8Stages;
    const bool ok = __syncthreads_and(mbar_wait(&full[st], (it / kI8Stages) & 1, abort, status));
    if (!ok) break;
    ++consumed;
    const uint8_t* xs = smem + st * kI8StageBytes;
    const uint8_t* ws = xs + kI8XBytes;
    // 1. A fragments of x: k steps kk of 16, rows mt*16 + (0..15)
    uint32_t a[4][MT][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        ldsm_x4(smem_u32(xs) + sw128_offset(mt * 16 + (mi & 1) * 8 + mr, kk * 16 + (mi >> 1) * 8), a[kk][mt][0],
                a[kk][mt][1], a[kk][mt][2], a[kk][mt][3]);
    // 2. dequantize: warp w rows 8w .. 8w+7, lane columns 8 lane .. +7
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      const int row = warp * 8 + rr;
      const uint2 raw = *reinterpret_cast<const uint2*>(ws + row * kI8Cols + 8 * lane);
      float f[2][4];
      i8x4_to_f32(raw.x, f[0]);
      i8x4_to_f32(raw.y, f[1]);
      uint32_t pk[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float p0, p1;
        f2_unpack(f2_mul(f2_pack(f[q >> 1][2 * (q & 1)], f[q >> 1][2 * (q & 1) + 1]),
                         f2_pack(sc[2 * q], sc[2 * q + 1])),
                  p0, p1);
        pk[q] = pack_bf16x2(p0, p1);
      }
      *reinterpret_cast<uint4*>(tile + row * kI8TileRow + 16 * lane) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    __syncthreads();
    // 3. the stage is consumed: refill it
    if (threadIdx.x == 0 && it + kI8Stages < n_st) {
      load_stage(it + kI8Stages);
      ++issued;
    }
    // 4. products for this warp's 32 columns
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int row = kk * 16 + (mi & 1) * 8 + mr, col = warp * 32 + np * 16 + (mi >> 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(tile_s + row * kI8TileRow + col * 2, b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma_bf16_16816(acc[mt][2 * np], a[kk][mt], b0, b1);
          mma_bf16_16816(acc[mt][2 * np + 1], a[kk][mt], b2, b3);
        }
      }
    }
    __syncthreads();  // 5. the tile is read before the next stage's dequant
  }
  // Copies still in flight (only after a wait gave up) land before the ring is reused.
  if (threadIdx.x == 0) {
    volatile int never = 0;
    for (int t = consumed; t < issued; ++t) mbar_wait(&full[t % kI8Stages], (t / kI8Stages) & 1, &never, status);
  }
  __syncthreads();
  // Partial sums into the ring: part[row][col], rows 0 .. 16 MT - 1, 256 columns.
  float* part = reinterpret_cast<float*>(smem);
  {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          part[(mt * 16 + g + 8 * (e >> 1)) * kI8Cols + warp * 32 + nt * 8 + 2 * t + (e & 1)] = acc[mt][nt][e];
  }
  cluster_sync();  // every CTA's partial sums are in its shared memory
  // CTA `rank` finishes columns [32 rank, 32 rank + 32): pairs of columns, rows < M
  for (int o = threadIdx.x; o < 16 * MT * 16; o += kI8Threads) {
    const int row = o / 16, col = 32 * rank + 2 * (o % 16);
    if (row < M) {
      const uint32_t local = smem_u32(part + row * kI8Cols + col);
      float v0 = 0.f, v1 = 0.f;
#pragma unroll
      for (int q = 0; q < kI8Cluster; ++q) {  // fixed order
        const float2 v = ld_dsmem_f2(dsmem_addr(local, uint32_t(q)));
        v0 += v.x;
        v1 += v.y;
      }
      y[(size_t(row) * N + n0 + col) / 2] = pack_bf16x2(v0, v1);
    }
  }
  cluster_sync();  // no CTA leaves while another reads its shared memory
}

bool small_int8_ok(int M, int K, int N) {
  return M >= 1 && M <= 32 && K % (kI8Cluster * kI8Rows) == 0 && N % kI8Cols == 0;
}

grok_status linear_int8_small(const grok_bf16* x, const int8_t* w8, const float* scales, int M, int K, int N,
                              grok_bf16* y, int32_t* dev_status, void* stream) {
  const int mt = M <= 16 ? 1 : 2;
  CUtensorMap tx, tw;
  grok_status st;
  {
    const uint64_t dims[4] = {uint64_t(K), uint64_t(M), 1, 1};
    const uint64_t strides[3] = {uint64_t(K) * 2, uint64_t(K) * 2 * M, uint64_t(K) * 2 * M};
    const uint32_t box[4] = {uint32_t(kI8Rows), uint32_t(16 * mt), 1, 1};
    if ((st = encode_tmap_bf16_4d(&tx, x, dims, strides, box)) != GROK_OK) return st;
  }
  {
    const uint64_t dims[2] = {uint64_t(N), uint64_t(K)};
    const uint32_t box[2] = {uint32_t(kI8Cols), uint32_t(kI8Rows)};
    if ((st = encode_tmap_u8_2d(&tw, w8, dims, uint64_t(N), box)) != GROK_OK) return st;
  }
  static bool attr_set[kMaxDevices][2] = {};  // per device and instance; idempotent
  int dev = 0;
  if ((st = device_index(&dev)) != GROK_OK) return st;
  auto kernel = mt == 1 ? linear_int8_small_kernel<1> : linear_int8_small_kernel<2>;
  if (!attr_set[dev][mt - 1]) {
    // two CTAs per SM need the largest shared-memory carveout
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kI8Smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return fail(cuda_status(e), "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    attr_set[dev][mt - 1] = true;
  }
  kernel<<<dim3(kI8Cluster, unsigned(N / kI8Cols)), kI8Threads, kI8Smem, static_cast<cudaStream_t>(stream)>>>(
      tx, tw, scales, M, K, N, reinterpret_cast<uint32_t*>(y), dev_status);
  return check_launch("linear_int8_small");
}

}  // namespace grok
