// Q/K/V projection on the 5th-generation tensor cores, optionally fused with
// RoPE and the KV-cache append.
//
// Grok-1 code-reading guide, ch. 4 "model.py close reading I": §4.1 Linear
// (weight [input_size, output_size], out = dot(x, w) in the input dtype),
// §4.5.1 Q/K/V projection (three bias-free Linears, 6144 -> 48 x 128, 8 x 128,
// 8 x 128, reshaped head-major), §4.3.1 RotaryEmbedding and §4.4 (rotate Q and
// K at offset = step, write rotated K and raw V into the cache at step).
//
// One GEMM: Y [M, 8192] = X [M, 6144] . W [6144, 8192], W = [W_q | W_k | W_v]
// side by side, M = B * T rows (b * T + i). bf16 operands, fp32 accumulation
// in TMEM, one rounding to bf16 per output. Output column h*128 + d is query
// head h, 6144 + g*128 + d key head g, 7168 + g*128 + d value head g.
// The same kernel with the plain epilogue is the general bias-free Linear
// (grok_linear: any K that is a multiple of 64, N of 256 or of 192), which also
// serves the output projection [M, 6144] . W_o [6144, 6144] and each
// tensor-parallel rank's head slice of it.
//
// Persistent kernel, one CTA per SM, 10 warps:
//   warp 0      TMA producer: per 64-wide K block two X boxes [128 rows x 64]
//               and four W boxes [64 rows x 64 columns] (64 KB; three, 56 KB,
//               with 192-column tiles) into a 3-stage ring
//   warp 1      TMEM owner and MMA issuer (converged; one fixed lane issues)
//   warps 2-9   epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31, one output
//               row per thread; of the two warps on a lane quarter, warps 2-5
//               take the first half of every head's features (fused: 0..31
//               with their rotation partners 64..95), warps 6-9 the second
// Tile = 256 rows x 256 columns (two heads; the plain epilogue also runs 256 x
// 192 tiles, see qkv_stage_bytes), as two 128-row halves that share
// each staged W block: tcgen05.mma M=128, N=256, K=16 per half, A = X
// (K-major), B = W (N-contiguous rows, MN-major), both 128-byte swizzled. The
// halves accumulate in TMEM columns 0..255 and 256..511. Sharing W between the
// halves is what keeps the MMAs fed: a 128-row tile needs 48 KB per 512 MMA
// cycles from L2 (94 B/cycle per SM), more than an SM's TMA stream delivers,
// the 256-row tile 64 KB per 1024 cycles. The epilogue drains half 0 while
// half 1's last products run, and the next tile's half-0 products start while
// half 1 is drained. Tiles go in groups of sixteen 256-row blocks by all the
// column blocks, so the tiles in flight share X and W in L2.
//
// Epilogues: plain (write Y) or fused (q heads: RoPE -> q_rot; k heads: RoPE
// -> cache_k at row start_pos[b] + i, or at its page of a paged pool; v heads
// -> cache_v). The rotation is the
// one of rope_kv_append (separately rounded fp32 products and sum of the bf16
// value and the fp32 cos / sin; scalar instructions, since ptxas may fuse a
// packed f32x2 multiply into the add that consumes it) with cos / sin taken
// from a table: per position (grok_qkv_rope_append_table), or per token row,
// filled by qkv_table_kernel with the shared fp64 routine. The projection is
// that kernel's programmatic dependent launch: its main loop runs while the
// table is computed, and its epilogue waits for the table grid. The half's
// epilogue holds back the next tile's products, so it stages the table through
// shared memory (coalesced loads; see kQkvTabWarpBytes) and splits each row
// over two warps: with per-row table loads it cost 50 us over the plain
// epilogue, staged and split 27 us.
#include "common.cuh"
#include "host.cuh"
#include "rope_math.cuh"

namespace grok {

constexpr int kQkvK = 6144;                 // model size
constexpr int kQkvN = 8192;                 // 48 * 128 + 2 * 8 * 128
constexpr int kQkvBM = 256, kQkvBK = 64;  // tile: two 128-row MMA halves
constexpr int kQkvHM = 128;                               // rows per MMA and per X box
constexpr int kQkvStages = 3;
constexpr int kQkvThreads = 320;
constexpr int kQkvEpiThreads = 256;  // warps 2-9
constexpr int kQkvGroupM = 16;  // 256-row blocks per tile group (8: 1 % slower, 32: 1-2 % slower)
constexpr int kQkvABox = kQkvHM * kQkvBK * 2;               // 16 KB: one half's X block
constexpr int kQkvABytes = 2 * kQkvABox;                    // 32 KB
constexpr int kQkvBBox = kQkvBK * 64 * 2;                   // 8 KB: 64 K rows x 64 columns
// The plain epilogue also runs with 192-column tiles (BN): for N = 6144 (the
// output projection) 256-row x 256-column tiles leave a last round of 8 tiles
// on 152 SMs (768 tiles, 0.84 of the rounds busy), 192-column ones fill 0.96
// (1024 tiles).
template <int BN>
__host__ __device__ constexpr int qkv_stage_bytes() { return kQkvABytes + (BN / 64) * kQkvBBox; }   // 64 KB (256), 56 KB (192)
// N the plain epilogue takes: whole 256- or 192-column tiles
constexpr bool linear_n_ok(int N) { return N >= 192 && (N % 256 == 0 || N % 192 == 0); }

struct QkvBars {
  uint64_t full[kQkvStages], empty[kQkvStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
// Fused epilogue: each epilogue warp stages its 32 rows' cos / sin for 16
// features at a time (4 KB) in shared memory. A row's slice is 64 contiguous
// bytes of the table, so a warp that loads its own row per thread touches 32
// lines per load (32 L1 wavefronts); staged, a load reads eight whole row
// slices (4 wavefronts), and the tile's two heads share them.
constexpr int kQkvTabWarpBytes = 4096;
constexpr int kQkvTabBytes = 8 * kQkvTabWarpBytes;
constexpr int qkv_smem(bool fused, int bn) {
  return kQkvStages * (kQkvABytes + (bn / 64) * kQkvBBox) + (fused ? kQkvTabBytes : 0) + int(sizeof(QkvBars)) + 1024;
}

struct QkvParams {
  int M, K, N, T, Tmax, n_mtiles, n_ntiles, k_blocks, n_tiles;
  const int32_t* start_pos;     // fused epilogue only
  const float* cos_tab;         // [M][64] per token row, or [tab_n][64] per position (tab_n > 0)
  const float* sin_tab;
  int tab_n;                    // > 0: the tables hold positions [0, tab_n), indexed by position
  uint4* y;                     // plain: [M][N]
  uint4* q_rot;                 // fused: [B][T][48][128]
  uint4* cache_k;               // fused: [B][Tmax][8][128]
  uint4* cache_v;
  PageMap pm;                   // fused: cache rows through a block table (null: contiguous)
  int32_t* status;
};

__device__ __forceinline__ void qkv_tile(const QkvParams& p, int t, int& m, int& n) {
  const int per_group = kQkvGroupM * p.n_ntiles;
  const int g = t / per_group, r = t % per_group;
  const int gm = min(kQkvGroupM, p.n_mtiles - g * kQkvGroupM);
  m = g * kQkvGroupM + r % gm;
  n = r / gm;
}

// cos / sin of every row's position for the fused epilogue (row = b * T + i,
// position start_pos[b] + i); rows of an invalid sequence are left unset. Each
// thread evaluates kQkvTabPer frequencies of one row at a time, independent
// fp64 chains that keep the fp64 pipe fed, over a grid-stride loop. The
// projection kernel is launched as this kernel's programmatic dependent: it may
// start at once, and only its epilogue waits for the table. The table grid is
// one small block per SM so that the projection's persistent CTAs fit beside
// it (a grid sized to the work fills every SM's registers, and the projection
// could then only start as the table drained).
constexpr int kQkvTabPer = 4;
constexpr int kQkvTabThreads = 128;

__global__ void __launch_bounds__(kQkvTabThreads) qkv_table_kernel(const int32_t* __restrict__ start_pos, int M,
                                                                     int T, int Tmax, float* __restrict__ cos_tab,
                                                                     float* __restrict__ sin_tab, int32_t* status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float s_inv[64];  // the 64 inverse frequencies, once per block (each is an fp64 power)
  if (threadIdx.x < 64) s_inv[threadIdx.x] = rope_inv_freq(threadIdx.x);
  __syncthreads();
  const long long total = (long long)M * (64 / kQkvTabPer);
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {   // one (row, group of frequencies)
    const int row = int(idx / (64 / kQkvTabPer)), j0 = int(idx % (64 / kQkvTabPer)) * kQkvTabPer;
    const int b = row / T, i = row % T;
    const int s = __ldg(start_pos + b);
    if (s < 0 || (long long)s + T > Tmax) {
      if (i == 0 && j0 == 0) report(status, GROK_DEV_BAD_START);
      continue;
    }
    float c[kQkvTabPer], sn[kQkvTabPer];
#pragma unroll
    for (int u = 0; u < kQkvTabPer; ++u) rope_cos_sin(__fmul_rn(float(s + i), s_inv[j0 + u]), c[u], sn[u]);
    float4* cp = reinterpret_cast<float4*>(cos_tab + (size_t)row * 64 + j0);
    float4* sp = reinterpret_cast<float4*>(sin_tab + (size_t)row * 64 + j0);
    *cp = make_float4(c[0], c[1], c[2], c[3]);
    *sp = make_float4(sn[0], sn[1], sn[2], sn[3]);
  }
}

__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t* r) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// 32 accumulator columns -> 16 packed bf16 pairs (round to nearest even).
__device__ __forceinline__ void qkv_round32(const uint32_t (&a)[32], uint32_t (&o)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) o[e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
}

// RoPE on one pair of features (x1: d, d+1 as packed bf16; x2: d+64, d+65):
// x1' = x1 cos - x2 sin, x2' = x2 cos + x1 sin, every product and sum rounded
// to fp32 separately, then to bf16.
__device__ __forceinline__ void qkv_rotate2(uint32_t& x1, uint32_t& x2, float c0, float c1, float s0, float s1) {
  const float a0 = bf16lo_to_f32(x1), a1 = bf16hi_to_f32(x1);
  const float b0 = bf16lo_to_f32(x2), b1 = bf16hi_to_f32(x2);
  const float y1a = __fadd_rn(__fmul_rn(a0, c0), -__fmul_rn(b0, s0));
  const float y1b = __fadd_rn(__fmul_rn(a1, c1), -__fmul_rn(b1, s1));
  const float y2a = __fadd_rn(__fmul_rn(b0, c0), __fmul_rn(a0, s0));
  const float y2b = __fadd_rn(__fmul_rn(b1, c1), __fmul_rn(a1, s1));
  x1 = pack_bf16x2(y1a, y1b);
  x2 = pack_bf16x2(y2a, y2b);
}

// The warp's cos / sin staging (4 KB: cos [32 rows][16 features] then sin),
// 16-byte piece q of row j at j * 64 + 16 (q ^ ((j >> 1) & 3)), so that the
// stores (4 lanes per row) and the row reads (lane l: row l) hit distinct banks.
__device__ __forceinline__ uint32_t qkv_tab_off(int j, int q) {
  return uint32_t(j * 64 + ((q ^ ((j >> 1) & 3)) << 4));
}

// Coalesced loads of the warp's rows' table slice for features f0 .. f0+15
// into v (cos in v[0..3], sin in v[4..7]): load k takes rows 8k .. 8k+7, four
// lanes per row. trow / ok: this lane's table row and whether it is rotated.
__device__ __forceinline__ void qkv_tab_load(const QkvParams& p, int trow, bool ok, int f0, int lane,
                                             float4 (&v)[8]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = 8 * k + (lane >> 2), q = lane & 3;
    const int tr = __shfl_sync(0xffffffffu, trow, j);
    const bool okj = __shfl_sync(0xffffffffu, ok ? 1 : 0, j) != 0;
    const size_t off = (size_t)tr * 64 + f0 + q * 4;
    v[k] = okj ? __ldg(reinterpret_cast<const float4*>(p.cos_tab + off)) : make_float4(0.f, 0.f, 0.f, 0.f);
    v[4 + k] = okj ? __ldg(reinterpret_cast<const float4*>(p.sin_tab + off)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__device__ __forceinline__ void qkv_tab_store(uint8_t* tab, int lane, const float4 (&v)[8]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = 8 * k + (lane >> 2), q = lane & 3;
    *reinterpret_cast<float4*>(tab + qkv_tab_off(j, q)) = v[k];
    *reinterpret_cast<float4*>(tab + 2048 + qkv_tab_off(j, q)) = v[4 + k];
  }
}

// RoPE on this lane's row for the 16 staged features (x1, packed bf16) and
// their partners 64 further on (x2).
__device__ __forceinline__ void qkv_rotate16_staged(uint32_t (&x1)[8], uint32_t (&x2)[8], const uint8_t* tab,
                                                    int lane) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 c4 = *reinterpret_cast<const float4*>(tab + qkv_tab_off(lane, q));
    const float4 s4 = *reinterpret_cast<const float4*>(tab + 2048 + qkv_tab_off(lane, q));
    qkv_rotate2(x1[2 * q], x2[2 * q], c4.x, c4.y, s4.x, s4.y);
    qkv_rotate2(x1[2 * q + 1], x2[2 * q + 1], c4.z, c4.w, s4.z, s4.w);
  }
}

// 32 lanes x 32 bit, 16 consecutive columns into r[0..15].
__device__ __forceinline__ void qkv_tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

template <bool kFused, int BN>
__global__ void __launch_bounds__(kQkvThreads, 1)
    qkv_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, const QkvParams p) {
  static_assert(BN == 256 || (!kFused && BN == 192), "tile width: two heads (fused), or 192 plain");
  constexpr int kStageBytes = qkv_stage_bytes<BN>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  QkvBars* bars = reinterpret_cast<QkvBars*>(smem + kQkvStages * kStageBytes + (kFused ? kQkvTabBytes : 0));
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQkvStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->acc_full[s], 1);
      mbar_init(&bars->acc_empty[s], kQkvEpiThreads);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x) {
        int m, n;
        qkv_tile(p, t, m, n);
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const int st = it % kQkvStages;
          if (!mbar_wait(&bars->empty[st], ((it / kQkvStages) & 1) ^ 1, abort, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + st * kStageBytes;
          mbar_arrive_expect_tx(&bars->full[st], kStageBytes);
          tma_load_4d(sa, &tm_x, &bars->full[st], kb * kQkvBK, m * kQkvBM, 0, 0);
          tma_load_4d(sa + kQkvABox, &tm_x, &bars->full[st], kb * kQkvBK, m * kQkvBM + kQkvHM, 0, 0);
#pragma unroll
          for (int c = 0; c < BN / 64; ++c)
            tma_load_4d(sa + kQkvABytes + c * kQkvBBox, &tm_w, &bars->full[st], n * BN + c * 64, kb * kQkvBK, 0, 0);
        }
      }
      // Drain: copies still in flight (only after an abort) land before the CTA exits.
      volatile int never = 0;
      for (int u = max(0, it - kQkvStages); u < it; ++u)
        mbar_wait(&bars->full[u % kQkvStages], (u / kQkvStages) & 1, &never, p.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one();
    constexpr uint32_t idesc = make_idesc_bf16(kQkvHM, BN, 1);
    int it = 0, tc = 0;
    bool ok = true;
    // TMEM: half 0 of the tile accumulates in columns 0..255, half 1 in 256..511.
    // The epilogue drains half 0 first: the next tile's half-0 products start
    // while half 1 is still being read out.
    for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++tc) {
      const uint32_t par = uint32_t(tc & 1) ^ 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->acc_empty[0], par, abort, p.status))) break;
      tc_fence_after();
      for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
        const int st = it % kQkvStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->full[st], (it / kQkvStages) & 1, abort, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + st * kStageBytes);
        const uint64_t bdesc = make_sdesc_sw128(sa + kQkvABytes, kQkvBBox, 1024);
        if (leader) {
          const uint64_t adesc = make_sdesc_sw128(sa, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 64 in steps of 16: A +32 B, B +16 rows (2048 B)
            umma_ss(tmem, adesc + uint64_t((kk * 32) >> 4), bdesc + uint64_t((kk * 2048) >> 4), idesc,
                    (kb > 0 || kk > 0) ? 1u : 0u);
          if (kb == p.k_blocks - 1) umma_commit(&bars->acc_full[0]);
        }
        __syncwarp();
        if (kb == 0) {
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->acc_empty[1], par, abort, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (leader) {
          const uint64_t adesc = make_sdesc_sw128(sa + kQkvABox, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss(tmem + BN, adesc + uint64_t((kk * 32) >> 4), bdesc + uint64_t((kk * 2048) >> 4), idesc,
                    (kb > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars->empty[st]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) umma_commit(&bars->acc_full[1]);
      __syncwarp();
    }
    // No MMA may still be running when TMEM is released.
    if (leader) umma_commit(&bars->mma_done);
    __syncwarp();
    volatile int never = 0;
    mbar_wait(&bars->mma_done, 0, &never, p.status);
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int part = (warp - 2) >> 2;  // 0: features 0..31 (+64) of each head, 1: 32..63 (+64)
    const int r = quad * 32 + lane;
    const uint32_t tlane = uint32_t(quad * 32) << 16;
    // The fused epilogue reads the cos / sin table of the kernel launched just
    // before this one: wait for that grid (a no-op without a prerequisite).
    if (kFused) asm volatile("griddepcontrol.wait;" ::: "memory");
    int tc = 0;
    for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++tc) {
      int m, n;
      qkv_tile(p, t, m, n);
      bool ok_all = true;
      for (int hf = 0; hf < 2; ++hf) {   // the tile's two 128-row halves, half 0 first
      const int row = m * kQkvBM + hf * kQkvHM + r;
      const bool live = row < p.M;
      // Fused: the row's destinations, and the first table slice's loads, ahead
      // of the accumulator wait (the warp is idle until then).
      int b = 0, i = 0, s = 0, trow = 0;
      bool write = false, kv_write = false;
      size_t crow = 0;
      const bool rotate = kFused && n < (kQHeads + kKVHeads) * kD / BN;  // query and key columns
      float4 tv[8];
      if (kFused) {
        b = row / p.T;
        i = row % p.T;
        s = live ? __ldg(p.start_pos + b) : 0;
        write = live && s >= 0 && (long long)s + p.T <= p.Tmax && (p.tab_n == 0 || (long long)s + p.T <= p.tab_n);
        // with a position table no table kernel runs to report a bad start: the epilogue does
        // (once, from the first column tile)
        if (n == 0 && live && i == 0 && !write && p.tab_n > 0) report(p.status, GROK_DEV_BAD_START);
        trow = write ? (p.tab_n > 0 ? s + i : row) : 0;  // table row of this token
        // cache row of position s + i: contiguous b * Tmax + s + i; paged page * 128 + (s + i) % 128
        crow = (size_t)b * p.Tmax + s + i;
        kv_write = write;
        if (p.pm.table && write) {
          const int pos = s + i;
          const int pg = __ldg(p.pm.table + (size_t)b * p.pm.max_pages + pos / GROK_PAGE_TOKENS);
          kv_write = pg >= 0 && pg < p.pm.n_pages;
          if (!kv_write) report(p.status, GROK_DEV_BAD_PAGE);
          crow = (size_t)(kv_write ? pg : 0) * GROK_PAGE_TOKENS + pos % GROK_PAGE_TOKENS;
        }
        if (rotate) qkv_tab_load(p, trow, write, 32 * part, lane, tv);
      }
      const bool ok = mbar_wait(&bars->acc_full[hf], tc & 1, abort, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok_all = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem + tlane + hf * BN;
      if (!kFused) {
        uint8_t* dst = reinterpret_cast<uint8_t*>(p.y) + ((size_t)row * p.N + n * BN) * 2;
        constexpr int kChunks = BN / 64;  // 32-column chunks per part
#pragma unroll
        for (int c = kChunks * part; c < kChunks * part + kChunks; ++c) {
          uint32_t a[32], o[16];
          tmem_ld32(acc + c * 32, a);
          tmem_wait_ld_dep(a);
          qkv_round32(a, o);
          if (live) {
            st_global_v8(dst + c * 64, o);
            st_global_v8(dst + c * 64 + 32, o + 8);
          }
        }
      } else {
        uint8_t* tab = smem + kQkvStages * kStageBytes + (warp - 2) * kQkvTabWarpBytes;
#pragma unroll 1
        for (int pc = 0; pc < 2; ++pc) {   // features f0 .. f0+15 paired with 64+f0 ..
          const int f0 = 32 * part + 16 * pc;
          if (rotate) {
            qkv_tab_store(tab, lane, tv);
            __syncwarp();
            if (pc == 0) qkv_tab_load(p, trow, write, f0 + 16, lane, tv);  // the next slice, while this one is used
          }
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {   // the tile's two heads share the slice
            const int col = n * BN + hh * kD;   // first output column of the head
            uint8_t* dst;
            const bool store = col < kQHeads * kD ? write : kv_write;
            if (col < kQHeads * kD) {
              dst = reinterpret_cast<uint8_t*>(p.q_rot) + ((size_t)row * kQHeads * kD + col) * 2;
            } else if (col < (kQHeads + kKVHeads) * kD) {
              const int g = (col - kQHeads * kD) / kD;
              dst = reinterpret_cast<uint8_t*>(p.cache_k) + ((crow * kKVHeads + g) * kD) * 2;
            } else {
              const int g = (col - (kQHeads + kKVHeads) * kD) / kD;
              dst = reinterpret_cast<uint8_t*>(p.cache_v) + ((crow * kKVHeads + g) * kD) * 2;
            }
            uint32_t a[32], x1[8], x2[8];
            qkv_tmem_ld16(acc + hh * kD + f0, a);
            qkv_tmem_ld16(acc + hh * kD + 64 + f0, a + 16);
            tmem_wait_ld_dep(a);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              x1[e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
              x2[e] = pack_bf16x2(__uint_as_float(a[16 + 2 * e]), __uint_as_float(a[16 + 2 * e + 1]));
            }
            if (rotate && write) qkv_rotate16_staged(x1, x2, tab, lane);
            if (store) {
              st_global_v8(dst + f0 * 2, x1);
              st_global_v8(dst + 128 + f0 * 2, x2);
            }
          }
          if (rotate) __syncwarp();  // every lane's reads of the slice before it is overwritten
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->acc_empty[hf]);
      }
      if (!ok_all) break;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Int8 weight-only quantisation (ch. 4 §4.1, §4.1.1 QuantizedWeight8bit): the
// weight is int8 [K, N] with one fp32 scale per output column, dequantized as
// an fp32 product rounded to fp32, then rounded to bf16 (the pages' order:
// astype(scales.dtype) * scales, then astype(bf16)).
// Each thread owns one 16-column chunk of the weight (its 16 scales stay in
// registers) and walks down the rows of its column, four rows per pass with
// all four loads issued before any converts; each chunk's 16 bf16 go out as
// one 32-byte store. Grid: (column blocks, row groups). Memory-bound: 1 byte
// read and 2 written per weight.
constexpr int kDqThreads = 128;
constexpr int kDqRows = 4;

__device__ __forceinline__ void dequant16r(uint4 raw, const float (&sc)[16], uint4* dst) {
  const uint32_t word[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t out[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float f[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int v = int(word[q] << (24 - 8 * b)) >> 24;  // sign-extended byte b
      f[b] = __fmul_rn(float(v), sc[4 * q + b]);
    }
    out[2 * q] = pack_bf16x2(f[0], f[1]);
    out[2 * q + 1] = pack_bf16x2(f[2], f[3]);
  }
  st_global_v8(dst, out);  // one 32-byte store (w16 is 32-byte aligned)
}

__global__ void __launch_bounds__(kDqThreads) dequant_int8_kernel(const uint4* __restrict__ w8,
                                                                  const float4* __restrict__ scales, int K, int N,
                                                                  uint4* __restrict__ w16) {
  const int per_row = N / 16;
  const int cc = blockIdx.x * kDqThreads + threadIdx.x;  // column chunk
  if (cc >= per_row) return;
  float sc[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = __ldg(scales + cc * 4 + q);
    sc[4 * q] = v.x, sc[4 * q + 1] = v.y, sc[4 * q + 2] = v.z, sc[4 * q + 3] = v.w;
  }
  for (int r0 = blockIdx.y * kDqRows; r0 < K; r0 += gridDim.y * kDqRows) {
    uint4 raw[kDqRows];
#pragma unroll
    for (int u = 0; u < kDqRows; ++u)
      if (r0 + u < K) raw[u] = __ldg(w8 + (size_t)(r0 + u) * per_row + cc);
#pragma unroll
    for (int u = 0; u < kDqRows; ++u)
      if (r0 + u < K) dequant16r(raw[u], sc, w16 + 2 * ((size_t)(r0 + u) * per_row + cc));
  }
}


grok_status qkv_launch(bool fused, const grok_bf16* x, const grok_bf16* w, int M, int K, int N, QkvParams& prm,
                       void* stream, bool after_table = true) {
  int sms = 0;
  grok_status st = device_sm_count(&sms);
  if (st != GROK_OK) return st;
  CUtensorMap tx, tw;
  {
    const uint64_t dims[4] = {uint64_t(K), uint64_t(M), 1, 1};
    const uint64_t strides[3] = {uint64_t(K) * 2, uint64_t(K) * 2 * M, uint64_t(K) * 2 * M};
    const uint32_t box[4] = {uint32_t(kQkvBK), uint32_t(kQkvHM), 1, 1};
    if ((st = encode_tmap_bf16_4d(&tx, x, dims, strides, box)) != GROK_OK) return st;
  }
  {
    const uint64_t dims[4] = {uint64_t(N), uint64_t(K), 1, 1};
    const uint64_t strides[3] = {uint64_t(N) * 2, uint64_t(N) * 2 * K, uint64_t(N) * 2 * K};
    const uint32_t box[4] = {64, uint32_t(kQkvBK), 1, 1};
    if ((st = encode_tmap_bf16_4d(&tw, w, dims, strides, box)) != GROK_OK) return st;
  }
  prm.M = M;
  prm.K = K;
  prm.N = N;
  prm.k_blocks = K / kQkvBK;
  prm.n_mtiles = (M + kQkvBM - 1) / kQkvBM;
  // tile width: 256 columns (two heads; the fused epilogue needs it), or for the
  // plain epilogue 192 when that keeps more of the rounds of tiles busy
  int bn = 256;
  if (!fused && N % 192 == 0) {
    auto busy = [&](int w) {
      const long long tiles = (long long)prm.n_mtiles * (N / w);
      const long long rounds = (tiles + sms - 1) / sms;
      return double(tiles) / double(rounds * sms);
    };
    if (N % 256 != 0 || busy(192) > busy(256) + 1e-9) bn = 192;
  }
  prm.n_ntiles = N / bn;
  prm.n_tiles = prm.n_mtiles * prm.n_ntiles;
  const int grid = prm.n_tiles < sms ? prm.n_tiles : sms;
  auto kernel = fused ? qkv_kernel<true, 256> : bn == 192 ? qkv_kernel<false, 192> : qkv_kernel<false, 256>;
  const int kind = fused ? 1 : bn == 192 ? 2 : 0;
  static bool attr_set[kMaxDevices][3] = {};  // per device and kernel instance; idempotent
  int dev = 0;
  if ((st = device_index(&dev)) != GROK_OK) return st;
  if (!attr_set[dev][kind]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, qkv_smem(fused, bn));
    if (e != cudaSuccess) return fail(cuda_status(e), "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    attr_set[dev][kind] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kQkvThreads);
  cfg.dynamicSmemBytes = qkv_smem(fused, bn);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap the table kernel before it
  attr[0].val.programmaticStreamSerializationAllowed = (fused && after_table) ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tx, tw, prm);
  if (e != cudaSuccess) return fail(cuda_status(e), "qkv launch: %s", cudaGetErrorString(e));
  return check_launch("qkv");
}

}  // namespace grok

using namespace grok;

extern "C" grok_status grok_linear(const grok_bf16* x, const grok_bf16* w, int M, int K, int N, grok_bf16* y,
                                   int32_t* dev_status, void* stream) {
  if (!x || !w || !y) return fail(GROK_ERR_INVALID_ARG, "grok_linear: null pointer");
  if (!aligned16(x) || !aligned16(w) || !aligned32(y))
    return fail(GROK_ERR_INVALID_ARG, "grok_linear: x and w must be 16-byte aligned, y 32-byte aligned");
  if (M < 1 || M > (1 << 30) || K < kQkvBK || K % kQkvBK != 0 || !linear_n_ok(N))
    return fail(GROK_ERR_INVALID_ARG,
                "grok_linear: need 1 <= M <= 2^30, K a positive multiple of %d, N of 256 or of 192 (M=%d K=%d N=%d)",
                kQkvBK, M, K, N);
  QkvParams prm = {};
  prm.T = 1;
  prm.Tmax = 1;
  prm.y = reinterpret_cast<uint4*>(y);
  prm.status = dev_status;
  return qkv_launch(false, x, w, M, K, N, prm, stream);
}

extern "C" grok_status grok_qkv_project(const grok_bf16* x, const grok_bf16* w, int M, grok_bf16* y,
                                        int32_t* dev_status, void* stream) {
  return grok_linear(x, w, M, kQkvK, kQkvN, y, dev_status, stream);
}

extern "C" grok_status grok_qkv_workspace(int B, int T, size_t* bytes) {
  if (!bytes) return fail(GROK_ERR_INVALID_ARG, "grok_qkv_workspace: null pointer");
  if (B < 1 || T < 1) return fail(GROK_ERR_INVALID_ARG, "grok_qkv_workspace: need B, T >= 1");
  *bytes = size_t(B) * T * 64 * 2 * sizeof(float);
  return GROK_OK;
}

static grok_status qkv_rope_append_launch(const grok_bf16* x, const grok_bf16* w, const int32_t* start_pos, int B,
                                          int T, int Tmax, grok_bf16* q_rot, grok_bf16* cache_k, grok_bf16* cache_v,
                                          PageMap pm, void* workspace, size_t ws_bytes, int32_t* dev_status,
                                          void* stream, const char* name) {
  if (!x || !w || !start_pos || !q_rot || !cache_k || !cache_v || !workspace)
    return fail(GROK_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(x) || !aligned16(w) || !aligned32(q_rot) || !aligned32(cache_k) || !aligned32(cache_v) ||
      !aligned16(workspace))
    return fail(GROK_ERR_INVALID_ARG, "%s: x, w and the workspace must be 16-byte aligned, q_rot and the caches "
                "32-byte aligned", name);
  if (B < 1 || T < 1 || Tmax < 1 || T > Tmax || Tmax > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "%s: need B >= 1, 1 <= T <= Tmax <= %d (B=%d T=%d Tmax=%d)", name,
                GROK_MAX_POSITION, B, T, Tmax);
  size_t need = 0;
  grok_qkv_workspace(B, T, &need);
  if (ws_bytes < need) return fail(GROK_ERR_INVALID_ARG, "%s: workspace of %zu bytes, need %zu", name, ws_bytes, need);
  const long long M = (long long)B * T;
  if (M > (1LL << 30)) return fail(GROK_ERR_INVALID_ARG, "%s: B * T too large", name);
  QkvParams prm = {};
  prm.T = T;
  prm.Tmax = Tmax;
  prm.start_pos = start_pos;
  prm.cos_tab = static_cast<const float*>(workspace);
  prm.sin_tab = prm.cos_tab + M * 64;
  prm.q_rot = reinterpret_cast<uint4*>(q_rot);
  prm.cache_k = reinterpret_cast<uint4*>(cache_k);
  prm.cache_v = reinterpret_cast<uint4*>(cache_v);
  prm.pm = pm;
  prm.status = dev_status;
  int sms = 0;
  grok_status st0 = device_sm_count(&sms);
  if (st0 != GROK_OK) return st0;
  const long long total = M * (64 / kQkvTabPer);
  const long long want = (total + kQkvTabThreads - 1) / kQkvTabThreads;
  const unsigned tab_grid = unsigned(want < sms ? want : sms);
  // An SM's shared-memory / L1 split is set for the blocks it runs: with the
  // default split for this small-smem kernel, the projection's CTAs could not
  // join its SMs before the table blocks finished.
  static bool tab_attr_set[kMaxDevices] = {};  // per device; idempotent
  int dev = 0;
  if ((st0 = device_index(&dev)) != GROK_OK) return st0;
  if (!tab_attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(qkv_table_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         int(cudaSharedmemCarveoutMaxShared));
    if (e != cudaSuccess) return fail(cuda_status(e), "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    tab_attr_set[dev] = true;
  }
  qkv_table_kernel<<<tab_grid, kQkvTabThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      start_pos, int(M), T, Tmax, const_cast<float*>(prm.cos_tab), const_cast<float*>(prm.sin_tab), dev_status);
  grok_status st = check_launch("qkv table");
  if (st != GROK_OK) return st;
  return qkv_launch(true, x, w, int(M), kQkvK, kQkvN, prm, stream);
}

// The fused projection with cos/sin from a table of positions [0, tab_n)
// (grok_rope_cos_sin(0, tab_n)): no per-call table kernel and no workspace.
extern "C" grok_status grok_qkv_rope_append_table(const grok_bf16* x, const grok_bf16* w, const int32_t* start_pos,
                                                  int B, int T, int Tmax, const float* cos_tab, const float* sin_tab,
                                                  int tab_positions, grok_bf16* q_rot, grok_bf16* cache_k,
                                                  grok_bf16* cache_v, int32_t* dev_status, void* stream) {
  const char* name = "grok_qkv_rope_append_table";
  if (!x || !w || !start_pos || !q_rot || !cache_k || !cache_v || !cos_tab || !sin_tab)
    return fail(GROK_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(x) || !aligned16(w) || !aligned32(q_rot) || !aligned32(cache_k) || !aligned32(cache_v) ||
      !aligned16(cos_tab) || !aligned16(sin_tab))
    return fail(GROK_ERR_INVALID_ARG, "%s: x, w and the tables must be 16-byte aligned, q_rot and the caches "
                "32-byte aligned", name);
  if (B < 1 || T < 1 || Tmax < 1 || T > Tmax || Tmax > GROK_MAX_POSITION || tab_positions < 1 ||
      tab_positions > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "%s: need B >= 1, 1 <= T <= Tmax <= %d, 1 <= tab_positions <= %d", name,
                GROK_MAX_POSITION, GROK_MAX_POSITION);
  const long long M = (long long)B * T;
  if (M > (1LL << 30)) return fail(GROK_ERR_INVALID_ARG, "%s: B * T too large", name);
  QkvParams prm = {};
  prm.T = T;
  prm.Tmax = Tmax;
  prm.start_pos = start_pos;
  prm.cos_tab = cos_tab;
  prm.sin_tab = sin_tab;
  prm.tab_n = tab_positions;
  prm.q_rot = reinterpret_cast<uint4*>(q_rot);
  prm.cache_k = reinterpret_cast<uint4*>(cache_k);
  prm.cache_v = reinterpret_cast<uint4*>(cache_v);
  prm.pm = PageMap{nullptr, 0, 0};
  prm.status = dev_status;
  return qkv_launch(true, x, w, int(M), kQkvK, kQkvN, prm, stream, false);
}

extern "C" grok_status grok_qkv_rope_append(const grok_bf16* x, const grok_bf16* w, const int32_t* start_pos, int B,
                                            int T, int Tmax, grok_bf16* q_rot, grok_bf16* cache_k, grok_bf16* cache_v,
                                            void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  return qkv_rope_append_launch(x, w, start_pos, B, T, Tmax, q_rot, cache_k, cache_v, PageMap{nullptr, 0, 0},
                                workspace, ws_bytes, dev_status, stream, "grok_qkv_rope_append");
}

extern "C" grok_status grok_qkv_rope_append_paged(const grok_bf16* x, const grok_bf16* w, const int32_t* start_pos,
                                                  int B, int T, grok_bf16* q_rot, grok_bf16* k_pool,
                                                  grok_bf16* v_pool, int n_pages, const int32_t* block_table,
                                                  int max_pages, void* workspace, size_t ws_bytes,
                                                  int32_t* dev_status, void* stream) {
  if (!block_table) return fail(GROK_ERR_INVALID_ARG, "grok_qkv_rope_append_paged: null block table");
  if (n_pages < 1 || max_pages < 1 || (long long)n_pages * GROK_PAGE_TOKENS > (1LL << 31) ||
      (long long)max_pages * GROK_PAGE_TOKENS > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG,
                "grok_qkv_rope_append_paged: need n_pages, max_pages >= 1, max_pages * %d <= %d "
                "(n_pages=%d max_pages=%d)",
                GROK_PAGE_TOKENS, GROK_MAX_POSITION, n_pages, max_pages);
  return qkv_rope_append_launch(x, w, start_pos, B, T, max_pages * GROK_PAGE_TOKENS, q_rot, k_pool, v_pool,
                                PageMap{block_table, max_pages, n_pages}, workspace, ws_bytes, dev_status, stream,
                                "grok_qkv_rope_append_paged");
}

extern "C" grok_status grok_dequant_int8(const int8_t* w8, const float* scales, int K, int N, grok_bf16* w16,
                                         void* stream) {
  if (!w8 || !scales || !w16) return fail(GROK_ERR_INVALID_ARG, "grok_dequant_int8: null pointer");
  if (!aligned16(w8) || !aligned16(scales) || !aligned32(w16))
    return fail(GROK_ERR_INVALID_ARG, "grok_dequant_int8: w8 and scales must be 16-byte aligned, w16 32-byte aligned");
  if (K < 1 || N < 16 || N % 16 != 0)
    return fail(GROK_ERR_INVALID_ARG, "grok_dequant_int8: need K >= 1 and N a positive multiple of 16 (K=%d N=%d)", K,
                N);
  int sms = 0;
  grok_status st = device_sm_count(&sms);
  if (st != GROK_OK) return st;
  const int per_row = N / 16;
  const int col_blocks = (per_row + kDqThreads - 1) / kDqThreads;
  // about 16 resident blocks of kDqThreads per SM in total, each walking its rows
  long long row_groups = ((long long)sms * 16 + col_blocks - 1) / col_blocks;
  const long long max_groups = ((long long)K + kDqRows - 1) / kDqRows;
  if (row_groups > max_groups) row_groups = max_groups;
  if (row_groups > 65535) row_groups = 65535;
  dequant_int8_kernel<<<dim3(unsigned(col_blocks), unsigned(row_groups)), kDqThreads, 0,
                        static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(w8), reinterpret_cast<const float4*>(scales), K, N,
      reinterpret_cast<uint4*>(w16));
  return check_launch("dequant_int8");
}

extern "C" grok_status grok_linear_int8_workspace(int K, int N, size_t* bytes) {
  if (!bytes) return fail(GROK_ERR_INVALID_ARG, "grok_linear_int8_workspace: null pointer");
  if (K < 1 || N < 1) return fail(GROK_ERR_INVALID_ARG, "grok_linear_int8_workspace: need K, N >= 1");
  *bytes = size_t(K) * N * sizeof(grok_bf16);
  return GROK_OK;
}

extern "C" grok_status grok_linear_int8(const grok_bf16* x, const int8_t* w8, const float* scales, int M, int K,
                                        int N, grok_bf16* y, void* workspace, size_t ws_bytes, int32_t* dev_status,
                                        void* stream) {
  if (!workspace) return fail(GROK_ERR_INVALID_ARG, "grok_linear_int8: null workspace");
  if (!aligned32(workspace) || !aligned32(y))
    return fail(GROK_ERR_INVALID_ARG, "grok_linear_int8: the workspace and y must be 32-byte aligned");
  if (ws_bytes < size_t(K) * N * sizeof(grok_bf16))
    return fail(GROK_ERR_INVALID_ARG, "grok_linear_int8: workspace of %zu bytes, need %zu", ws_bytes,
                size_t(K) * N * sizeof(grok_bf16));
  // grok_linear's shape rules first, so that nothing is queued for a call it would reject
  if (M < 1 || M > (1 << 30) || K < kQkvBK || K % kQkvBK != 0 || !linear_n_ok(N))
    return fail(GROK_ERR_INVALID_ARG,
                "grok_linear_int8: need 1 <= M <= 2^30, K a positive multiple of %d, N of 256 or of 192 (M=%d K=%d "
                "N=%d)",
                kQkvBK, M, K, N);
  // Decode-sized M: one pass over the int8 weight, dequantized in shared memory
  // (int8_small.cu).
  if (small_int8_ok(M, K, N)) {
    if (!x || !w8 || !scales) return fail(GROK_ERR_INVALID_ARG, "grok_linear_int8: null pointer");
    if (!aligned16(x) || !aligned16(w8) || !aligned16(scales))
      return fail(GROK_ERR_INVALID_ARG, "grok_linear_int8: x, w8 and scales must be 16-byte aligned");
    int sms = 0;
    grok_status st0 = device_sm_count(&sms);
    if (st0 != GROK_OK) return st0;
    return linear_int8_small(x, w8, scales, M, K, N, y, dev_status, stream);
  }
  grok_bf16* w16 = static_cast<grok_bf16*>(workspace);
  grok_status st = grok_dequant_int8(w8, scales, K, N, w16, stream);
  if (st != GROK_OK) return st;
  return grok_linear(x, w16, M, K, N, y, dev_status, stream);
}
