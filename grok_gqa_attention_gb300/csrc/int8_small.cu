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
// columns [256 nb, 256 nb + 256) and weight rows [r K/8, (r+1) K/8); each
// weight row slice is 256 contiguous bytes. Two CTAs fit per SM, so the whole
// grid of the Q/K/V shape (256 CTAs) is resident at once.
//
// Per CTA, three roles that run concurrently:
//   warp 9     TMA producers: lane 0 streams the weight through a 3-stage
//              ring of 64-row tiles [64 rows x 256 bytes], lane 1 the matching
//              x tiles [16 MT rows x 64 bf16] (rows >= M zero-filled; 128-byte
//              swizzle) through a 4-stage ring. Weight stages are released as
//              soon as the converters hold their bytes in registers, x stages
//              when the products that read them complete, so the weight stream
//              never waits for the tensor core.
//   warps 0-7  dequantize: each thread copies its 8 x 8 weight bytes of a stage
//              to registers and releases the stage, then converts them into a
//              2-stage ring of bf16 tiles [32 k x 256 n], stored as the
//              MN-major, 128-byte-swizzled A operand (four 64-column blocks).
//              Each element exactly as grok_dequant_int8 does it: the byte is
//              turned into a float by placing it in the mantissa of 2^23 (byte
//              permute) and subtracting 2^23 + 128, multiplied by its column
//              scale with one fp32 rounding, then rounded to nearest-even bf16.
//   warp 8     tcgen05.mma issuer (one lane) and TMEM owner: D[n, m] +=
//              W^T[n, k] x^T[k, m] per 128-column half, M = 128 (n), N = 16 MT
//              (m), K = 16, fp32 accumulators in TMEM (64 columns).
// Then warps 0-7 read D (warp w: columns half w / 4, TMEM lanes 32 (w % 4),
// i.e. columns [32 w, 32 w + 32) of the block). CTA r of the cluster finishes
// columns [32 r, 32 r + 32): once every CTA's products are complete (a cluster
// barrier; the A rings then serve as receive buffers), warp w of each CTA
// stores its partial sums straight into CTA w's shared memory, in the slot of
// its own rank, and after a second barrier each CTA adds the 8 slots in rank
// order (so results do not depend on scheduling), rounds to bf16 and writes.
// Remote stores need no round trip, unlike reading the other CTAs' partials.
#include "common.cuh"
#include "host.cuh"

namespace grok {

constexpr int kI8Cluster = 8;                      // CTAs along K
constexpr int kI8Cols = 256;                       // output columns per CTA
constexpr int kI8Rows = 64;                        // weight rows per TMA stage
constexpr int kI8Stages = 3;                       // weight ring
constexpr int kI8XStages = 4;                      // x ring
constexpr int kI8ARows = 32;                       // k rows per bf16 A tile
constexpr int kI8AStages = 2;
constexpr int kI8DqWarps = 8;
constexpr int kI8Threads = (kI8DqWarps + 2) * 32;  // + MMA warp + producer warp
constexpr int kI8XBytes = 32 * kI8Rows * 2;        // x tile (room for 32 rows), 1024-byte aligned
constexpr int kI8WBytes = kI8Rows * kI8Cols;       // int8 weight tile, 16 KB
constexpr int kI8ABlock = kI8ARows * 128;          // [32 k][64 n] bf16, 128-byte swizzled
constexpr int kI8ABytes = 4 * kI8ABlock;           // 256 columns
constexpr int kI8XOff = kI8Stages * kI8WBytes;     // x ring after the weight ring
constexpr int kI8AOff = kI8XOff + kI8XStages * kI8XBytes;
constexpr int kI8Data = kI8AOff + kI8AStages * kI8ABytes;
constexpr int kI8Smem = kI8Data + 256 + 1024;
static_assert(kI8Cluster * 32 * 32 * 4 <= kI8AStages * kI8ABytes, "received partial sums must fit in the A ring");

struct I8Bars {
  uint64_t w_full[kI8Stages], w_empty[kI8Stages];
  uint64_t x_full[kI8XStages], x_empty[kI8XStages];
  uint64_t a_full[kI8AStages], a_empty[kI8AStages];
  uint64_t d_full, mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(I8Bars) <= 256, "barrier block");
static_assert(kI8XOff % 1024 == 0 && kI8AOff % 1024 == 0, "swizzled tiles need 1024-byte alignment");

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  // the map must have been encoded with rank 2 (the instruction's dimensionality equals the map's rank)
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

__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
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
  uint8_t* sA = smem + kI8AOff;
  I8Bars* bars = reinterpret_cast<I8Bars*>(smem + kI8Data);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = blockIdx.x;  // position in the cluster = K slice
  const int n0 = blockIdx.y * kI8Cols;
  const int k_first = rank * (K / kI8Cluster);
  const int n_st = K / kI8Cluster / kI8Rows;
  constexpr uint32_t kXTx = uint32_t(16 * MT * kI8Rows * 2);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kI8Stages; ++s) {
      mbar_init(&bars->w_full[s], 1);
      mbar_init(&bars->w_empty[s], kI8DqWarps * 32);  // every converter thread holds its bytes
    }
    for (int s = 0; s < kI8XStages; ++s) {
      mbar_init(&bars->x_full[s], 1);
      mbar_init(&bars->x_empty[s], 1);  // the products that read the tile completed
    }
    for (int s = 0; s < kI8AStages; ++s) {
      mbar_init(&bars->a_full[s], kI8DqWarps * 32);
      mbar_init(&bars->a_empty[s], 1);
    }
    mbar_init(&bars->d_full, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kI8DqWarps) {
    tmem_alloc(&bars->tmem_base, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Launched as a programmatic dependent: the setup above (and the CTA launch)
  // overlaps the previous kernel's tail on the stream. Nothing in global memory
  // is read or written before the wait, so stream order holds for every operand.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t tmem = bars->tmem_base;
  uint32_t d[32];     // converter warps: the accumulator's 32 columns of this warp
  bool done = false;  // converter warps: every product completed (no wait gave up)

  if (warp == kI8DqWarps + 1) {
    // ------------------------------------------------------------ TMA producers
    if (lane == 0) {  // weight tiles
      prefetch_tmap(&tm_w);
      int it = 0;
      for (; it < n_st; ++it) {
        const int st = it % kI8Stages;
        if (!mbar_wait(&bars->w_empty[st], ((it / kI8Stages) & 1) ^ 1, abort, status)) break;
        mbar_arrive_expect_tx(&bars->w_full[st], kI8WBytes);
        tma_load_2d(smem + st * kI8WBytes, &tm_w, &bars->w_full[st], n0, k_first + it * kI8Rows);
      }
      // copies still in flight (only after a wait gave up) land before the CTA exits
      volatile int never = 0;
      for (int t = max(0, it - kI8Stages); t < it; ++t)
        mbar_wait(&bars->w_full[t % kI8Stages], (t / kI8Stages) & 1, &never, status);
    } else if (lane == 1) {  // x tiles
      prefetch_tmap(&tm_x);
      int it = 0;
      for (; it < n_st; ++it) {
        const int st = it % kI8XStages;
        if (!mbar_wait(&bars->x_empty[st], ((it / kI8XStages) & 1) ^ 1, abort, status)) break;
        mbar_arrive_expect_tx(&bars->x_full[st], kXTx);
        tma_load_4d(smem + kI8XOff + st * kI8XBytes, &tm_x, &bars->x_full[st], k_first + it * kI8Rows, 0, 0,
                    0);  // x's map is 4-d (rows, 1, 1)
      }
      volatile int never = 0;
      for (int t = max(0, it - kI8XStages); t < it; ++t)
        mbar_wait(&bars->x_full[t % kI8XStages], (t / kI8XStages) & 1, &never, status);
    }
  } else if (warp == kI8DqWarps) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one();
    // A: MN-major (n contiguous), 64-column blocks kI8ABlock apart, 8-row groups 1024 apart
    const uint64_t ad = make_sdesc_sw128(smem_u32(sA), kI8ABlock, 1024);
    // B = x^T: K-major (rows of x), 8-row groups 1024 apart
    const uint64_t xd = make_sdesc_sw128(smem_u32(smem), 16, 1024);
    constexpr uint32_t idesc = make_idesc_bf16(128, 16 * MT, 0) | (1u << 15);  // A MN-major
    bool ok = true;
    for (int it = 0; ok && it < n_st; ++it) {
      const int st = it % kI8XStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->x_full[st], (it / kI8XStages) & 1, abort, status))) break;
      for (int hs = 0; hs < kI8Rows / kI8ARows; ++hs) {
        const int q = it * (kI8Rows / kI8ARows) + hs, a = q % kI8AStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->a_full[a], (q / kI8AStages) & 1, abort, status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int nh = 0; nh < 2; ++nh)
#pragma unroll
            for (int kk = 0; kk < kI8ARows / 16; ++kk) {
              const uint64_t adesc = ad + uint64_t((a * kI8ABytes + nh * 2 * kI8ABlock + kk * 2048) >> 4);
              const uint64_t bdesc =
                  xd + uint64_t((kI8XOff + st * kI8XBytes + (hs * (kI8ARows / 16) + kk) * 32) >> 4);
              umma_ss(tmem + nh * 32, adesc, bdesc, idesc, (it > 0 || hs > 0 || kk > 0) ? 1u : 0u);
            }
          umma_commit(&bars->a_empty[a]);
          if (hs == kI8Rows / kI8ARows - 1) umma_commit(&bars->x_empty[st]);  // the x tile is read
        }
        __syncwarp();
      }
    }
    if (leader) {
      umma_commit(&bars->d_full);
      umma_commit(&bars->mma_done);
    }
    __syncwarp();
    volatile int never = 0;
    mbar_wait(&bars->mma_done, 0, &never, status);
  } else {
    // ------------------------------------------------------------ converters
    float sc[8];  // this lane's columns 8 lane .. 8 lane + 7
    {
      const float4* s4 = reinterpret_cast<const float4*>(scales + n0 + 8 * lane);
      const float4 u = __ldg(s4), v = __ldg(s4 + 1);
      sc[0] = u.x, sc[1] = u.y, sc[2] = u.z, sc[3] = u.w, sc[4] = v.x, sc[5] = v.y, sc[6] = v.z, sc[7] = v.w;
    }
    // where this lane's 8 columns go in an A tile row: 64-column block lane / 8, 16-byte chunk lane % 8
    const int blk = lane >> 3, chunk = lane & 7;
    bool ok = true;
    for (int it = 0; ok && it < n_st; ++it) {
      const int st = it % kI8Stages;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->w_full[st], (it / kI8Stages) & 1, abort, status))) break;
      // rows warp + 8 i of the stage, i = 0..7
      const uint8_t* ws = smem + st * kI8WBytes;
      uint2 raw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) raw[i] = *reinterpret_cast<const uint2*>(ws + (warp + 8 * i) * kI8Cols + 8 * lane);
      mbar_arrive(&bars->w_empty[st]);
      for (int hs = 0; hs < kI8Rows / kI8ARows; ++hs) {
        const int q = it * (kI8Rows / kI8ARows) + hs, a = q % kI8AStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->a_empty[a], ((q / kI8AStages) & 1) ^ 1, abort, status))) {
          ok = false;
          break;
        }
        uint8_t* at = sA + a * kI8ABytes + blk * kI8ABlock;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = warp + 8 * i;  // k row within the A tile (rows of raw[4 hs + i])
          const uint2 r2 = raw[4 * hs + i];
          float f[2][4];
          i8x4_to_f32(r2.x, f[0]);
          i8x4_to_f32(r2.y, f[1]);
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float p0, p1;
            f2_unpack(f2_mul(f2_pack(f[e >> 1][2 * (e & 1)], f[e >> 1][2 * (e & 1) + 1]),
                             f2_pack(sc[2 * e], sc[2 * e + 1])),
                      p0, p1);
            pk[e] = pack_bf16x2(p0, p1);
          }
          *reinterpret_cast<uint4*>(at + row * 128 + ((chunk ^ (row & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async_smem();  // the generic-proxy stores become visible to the tensor core
        mbar_arrive(&bars->a_full[a]);
      }
    }
    // D: this warp's 32 columns (32 warp + lane of the block), rows m < 16 MT
    done = __all_sync(0xffffffffu, mbar_wait(&bars->d_full, 0, abort, status));
    tc_fence_after();
    tmem_ld32(tmem + (uint32_t((warp & 3) * 32) << 16) + (warp >> 2) * 32, d);
    tmem_wait_ld_dep(d);
  }
  tc_fence_before();
  cluster_sync();  // every CTA's products are complete: its A ring may receive partial sums
  if (warp < kI8DqWarps && done) {
    // recv[src][m][c] (columns 32 w + c of the block) in CTA w = warp, slot src = this CTA
    const uint32_t dst = dsmem_addr(smem_u32(sA) + uint32_t((rank * 32 * 32 + lane) * 4), uint32_t(warp));
#pragma unroll
    for (int m = 0; m < 16 * MT; ++m) st_dsmem_f32(dst + uint32_t(m * 32 * 4), __uint_as_float(d[m]));
  }
  cluster_sync();  // every partial sum has landed
  if (warp < kI8DqWarps) {
    const float* recv = reinterpret_cast<const float*>(sA);
    // CTA `rank` finishes columns [32 rank, 32 rank + 32): pairs of columns, rows < M
    for (int o = threadIdx.x; o < 16 * MT * 16; o += kI8DqWarps * 32) {
      const int row = o / 16, c = 2 * (o % 16);
      if (row < M) {
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int q = 0; q < kI8Cluster; ++q) {  // fixed order
          const float2 v = *reinterpret_cast<const float2*>(recv + (q * 32 + row) * 32 + c);
          v0 += v.x;
          v1 += v.y;
        }
        y[(size_t(row) * N + n0 + 32 * rank + c) / 2] = pack_bf16x2(v0, v1);
      }
    }
  }
  if (warp == kI8DqWarps) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kI8Cluster, unsigned(N / kI8Cols));
  cfg.blockDim = dim3(kI8Threads);
  cfg.dynamicSmemBytes = kI8Smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see the kernel's griddepcontrol.wait
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, kernel, tx, tw, scales, M, K, N, reinterpret_cast<uint32_t*>(y), dev_status);
  if (e != cudaSuccess) return fail(cuda_status(e), "linear_int8_small launch: %s", cudaGetErrorString(e));
  return check_launch("linear_int8_small");
}

}  // namespace grok
