// K2: prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Grok-1 code-reading guide, ch. 4 "model.py close reading I": §4.5.2 (GQA
// logits, query head h reads KV head h / 6, multiplier 1/sqrt(128), soft cap
// 30 tanh(x / 30)), §4.5.3 (mask, softmax over keys in fp32), §4.5.4 (weighted
// sum of V); ch. 6 "model.py close reading II", §6.4.2 (causal x padding mask).
//
// Work item = (sequence b, 128-row query tile, KV group g, pair of query heads
// of that group). One persistent CTA per SM walks the items in a snake order
// over rounds of gridDim.x items (heaviest first; odd rounds reversed), which
// evens out the causal work per CTA. Both heads of an item read the same K/V
// tiles, so every K/V tile staged in shared memory by TMA feeds two heads; the
// three head pairs of a group run in neighbouring CTAs and meet the same tiles
// in L2.
//
// Four independent chains per CTA. Each 128-key tile of each head is handled
// as two 64-key halves, and each (head, half) is its own chain:
//   S_h = Q K_h^T (64 TMEM columns) -> softmax -> P_h over S_h ->
//   O += P_h V_h, then at once S_h of the next tile = Q K_h'^T
// so one half's softmax overlaps the other half's products. The next tile's
// first product is issued right after the previous P V that read the same
// columns (the tensor pipe runs one thread's MMAs in order).
//
// Warp roles (608 threads):
//   warp 0      TMA producer: Q tiles of both heads, then K and V tiles in two
//               separate 2-stage rings
//   warp 1      TMEM owner and MMA issuer of head slot 0
//   warp 18     MMA issuer of head slot 1 (on another SMSP). Each issuer warp
//               runs converged through its barrier waits and one fixed lane
//               issues the MMAs and commits; the two issuers do not coordinate,
//               so one's waits are covered by the other's products.
//   warps 2-9   softmax + epilogue for head slot 0: warps 2-5 own half 0 (key
//               columns 0..63 of each tile, output features 0..63), warps 6-9
//               half 1 (warp w reads TMEM lanes 32 (w % 4) .. +31, so four
//               consecutive warps cover rows 0..127)
//   warps 10-17 the same for head slot 1
// The two halves of a row add their partial row sums through shared memory.
// TMEM (512 columns): per slot, S in 128 fp32 columns (half h in 64h..64h+63)
// and O in 128. The softmax warps overwrite S in place with P as two bf16
// halves (hi, lo) that sum to P to ~2^-16; O += P_hi V + P_lo V reads them
// straight from TMEM.
//
// Softmax without a running maximum: every capped logit is below 30, so the
// weights exp(c - 30) lie in (e^-60, 1] and fp32 holds them and their sums
// with full relative precision. O therefore accumulates across all key tiles
// with no rescaling; the epilogue divides by the row sum once. The weight's
// tanh runs on the special-function unit; its exp2 does too for half of the
// columns and runs as a polynomial on the FMA pipe for the other half, which
// balances the two pipes.
//
// Keys beyond the last visible row of an item's final tile may hold anything
// (including NaN): the softmax gives them weight 0 by selection and the softmax
// warps zero those rows of the staged V tile before the PV product reads it.
//
// fp16 mode (kF16, grok_attn_prefill_ws): P is rounded once to fp16 (11-bit
// significand, enough for the weights' precision) and P V is one product per
// 16 keys instead of two, with V read as fp16 from a copy in the caller's
// workspace (both operands of a kind::f16 product have one type). fp16's
// exponent range cannot hold weights relative to the fixed reference 30, so
// each row takes its own reference from its item's first key tile: the two
// warps of a quadrant exchange their 64-key maxima once per item, and
// m = 30 log2(e) tanh(y_max) + 8 (log2 units) puts the row's largest weight of
// that tile at 2^-8. Later tiles whose logits rise above it by up to 2^24
// (about 16.6 on the capped-logit scale) still fit fp16; a row whose weight sum
// reaches 65504 (or any non-finite sum) puts its item on a fallback list in the
// workspace, and so does every item of a sequence whose V does not fit fp16.
// The bf16 mode of this kernel then recomputes exactly the listed items.
//
// Split pass (kSplit, fp16 mode): when a call has fewer than two items per SM,
// the items of the ragged last round run in a second launch, each shared among
// up to four units over consecutive key tiles. A unit writes its unnormalised
// O, row sums and references to the workspace; the item's last unit to finish
// (a per-item counter) adds the parts in part order and writes the output.
#include <algorithm>

#include "common.cuh"
#include "host.cuh"

namespace grok {

constexpr int kPfThreads = 608;
constexpr int kPfRows = 128;   // query rows per tile (MMA M)
constexpr int kPfKeys = 128;   // keys per K/V tile (MMA N for Q K^T, K for P V)
constexpr int kPfStages = 2;
constexpr int kBox = 128 * 128;             // [128 rows][64 bf16], 128-byte swizzled
constexpr int kQBytes = 2 * 2 * kBox;       // two heads, two 64-wide halves of d
constexpr int kTileBytes = 2 * kBox;        // one K or V tile: two 64-wide halves of d
constexpr int kPfData = kQBytes + 2 * kPfStages * kTileBytes;
constexpr int kPfSeqCache = 512;  // sequences whose start / valid length are staged in shared memory
constexpr float kPfHeadroom = 8.0f;  // fp16 mode: log2 gap between a row's reference and its first-tile maximum
constexpr int kPfMaxParts = 4;       // key-range split: most units one item's key tiles are shared among
constexpr int kPfMinPartTiles = 8;   // key-range split: fewest key tiles per unit

struct PfBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kPfStages], k_empty[kPfStages], v_full[kPfStages], v_empty[kPfStages];
  uint64_t s_full[2][2], p_full[2][2], o_full[2], o_empty[2];  // [slot][half]
  uint64_t mma_done;
  uint64_t lsum_ready[2];  // both halves of a slot posted their partial row sums
  uint64_t epi_done[2];    // the slot's eight epilogue warps' output stores have read their staging
  uint64_t xbar[2][4];     // fp16 mode: [slot][quad] both warps of a quadrant posted their first-tile maxima
  uint64_t split_in[2];    // key-range split: the slot's eight epilogue warps wrote their unit's part
  uint64_t split_out[2];   // key-range split: the unit is counted (split_last is set)
  int split_last[2];       // key-range split: this unit is its item's last to finish (it adds the parts)
  int split_over[2];       // key-range split: some row of this unit reached fp16's range
  float xmax[2][4][2][32];   // [slot][quad][half][lane]
  float lsum[2][2][2][128];  // [item parity][slot][half][row]
  int seq_start[kPfSeqCache], seq_valid[kPfSeqCache], seq_vflag[kPfSeqCache];
  uint32_t tmem_base;
  int abort;
};
constexpr int kPfSmem = kPfData + int(sizeof(PfBars)) + 1024;

struct PfParams {
  int B, T, Tmax, n_qt, n_items;
  PageMap pm;  // K/V addressing (contiguous cache or paged pool)
  const int32_t* start_pos;
  const int32_t* valid_len;
  int32_t* status;
  // fp16 mode: per-sequence "V does not fit fp16" flags and the fallback list it appends to
  const int32_t* v_flags;
  int32_t* fb_count;
  int32_t* fb_list;
  int fb_cap;
  // bf16 mode over a list of items only (the fallback pass): item_list[0 .. *item_count)
  const int32_t* item_list;
  const int32_t* item_count;
  int n_units;  // work units of this pass (items, or in the split pass units of items)
  // key-range split pass (fp16 mode): items [item_base, item_base + n_units / n_parts),
  // each shared among n_parts units (unit = (item - item_base) * n_parts + part)
  int item_base, n_parts;
  float4* part_o;     // [unit][slot][half][16 feature quads][128 rows]: the unit's unnormalised O
  float2* part_lm;    // [unit][slot][128 rows]: (row sum, reference) of the unit
  int32_t* part_cnt;  // [item - item_base][slot]: units finished; zero at the start of the call
};

struct PfItem {
  int item;         // the item this unit computes (part of)
  int part, parts;  // key-range split: this unit's part and the item's number of parts (1: whole item)
  int j0;           // first key tile of the unit
  int b, qt, g, hp;
  int s, n;     // start position, valid length
  int kv_end;   // keys [0, kv_end) are visible to some row of the tile
  int n_kv;     // key tiles to visit from j0 (0: skip the unit)
  int n_sub;    // 64-key halves of those tiles that hold a visible key
  int bad;      // GROK_DEV_* bits when the sequence's integers are invalid
  bool redirect;  // fp16 mode: the sequence's V does not fit fp16; the fallback pass computes the item
};

// The item a CTA takes in round rd (-1 when there is none): rounds of gridDim.x
// items, odd rounds in reverse CTA order, so the heavy items of one round and
// the light items of the next land on the same CTA.
template <bool kList>
__device__ __forceinline__ int pf_item_index(const PfParams& p, int rd) {
  const int k = (rd & 1) ? int(gridDim.x) - 1 - int(blockIdx.x) : int(blockIdx.x);
  const long long idx = (long long)rd * gridDim.x + k;
  if (kList) {
    const int n = min(__ldg(p.item_count), p.fb_cap);
    return idx < n ? __ldg(p.item_list + idx) : -1;
  }
  return idx < p.n_units ? int(idx) : -1;
}

// Decode work unit `unit`. Outside the split pass a unit is a whole item.
template <bool kF16, bool kSplit>
__device__ __forceinline__ PfItem pf_item(const PfParams& p, const PfBars* bars, int unit) {
  PfItem it;
  const int item = kSplit ? p.item_base + unit / p.n_parts : unit;
  it.item = item;
  it.part = kSplit ? unit % p.n_parts : 0;
  it.parts = 1;
  it.j0 = 0;
  it.hp = item % 3;
  int rest = item / 3;
  it.g = rest % kKVHeads;
  rest /= kKVHeads;
  it.b = rest % p.B;
  it.qt = p.n_qt - 1 - rest / p.B;  // heaviest (last) query tiles first
  int vflag = 0;
  if (it.b < kPfSeqCache) {
    it.s = bars->seq_start[it.b];
    it.n = bars->seq_valid[it.b];
    if (kF16) vflag = bars->seq_vflag[it.b];
  } else {
    it.s = __ldg(p.start_pos + it.b);
    it.n = p.valid_len ? __ldg(p.valid_len + it.b) : p.T;
    if (kF16) vflag = __ldg(p.v_flags + it.b);
  }
  it.bad = 0;
  it.redirect = false;
  if (it.s < 0 || (long long)it.s + p.T > p.Tmax) it.bad |= GROK_DEV_BAD_START;
  if (it.n < 1 || it.n > p.T) it.bad |= GROK_DEV_BAD_VALID;
  if (it.bad) {
    it.kv_end = 0;
    it.n_kv = 0;
    it.n_sub = 0;
    return it;
  }
  if (kF16 && vflag) {
    it.redirect = true;
    it.kv_end = 0;
    it.n_kv = 0;
    it.n_sub = 0;
    return it;
  }
  const int last_row = min(it.qt * kPfRows + kPfRows, p.T);  // rows [qt*128, last_row)
  it.kv_end = min(it.s + last_row, it.s + it.n);
  it.n_sub = (it.kv_end + 63) / 64;
  it.n_kv = (it.n_sub + 1) / 2;
  if (kSplit) {
    // part k of `parts` takes key tiles [k n_kv / parts, (k + 1) n_kv / parts),
    // at least kPfMinPartTiles each
    const int parts = max(1, min(p.n_parts, it.n_kv / kPfMinPartTiles));
    it.parts = parts;
    if (it.part >= parts) {
      it.n_kv = 0;
      it.n_sub = 0;
      return it;
    }
    const int j0 = it.part * it.n_kv / parts, j1 = (it.part + 1) * it.n_kv / parts;
    it.j0 = j0;
    it.n_sub = min(2 * j1, it.n_sub) - 2 * j0;
    it.n_kv = j1 - j0;
  }
  return it;
}

// Append an item to the fallback list (duplicates are harmless: the fallback
// pass would compute the same bits twice).
__device__ __forceinline__ void pf_fallback(const PfParams& p, int item) {
  const int k = atomicAdd(p.fb_count, 1);
  if (k < p.fb_cap) p.fb_list[k] = item;
}

// Instruction descriptor, kind::f16 with fp16 A and B, fp32 D.
__host__ __device__ constexpr uint32_t make_idesc_f16(int M, int N, int b_mn_major) {
  return (1u << 4) | (uint32_t(b_mn_major) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// MMA issue. The issuing thread shares its SMSP with busy softmax warps, so the
// per-instruction work is kept to a descriptor add: the 64-bit descriptors of
// the first K-step are built once and later steps add their byte offset / 16
// to the start-address field (no carry: shared addresses are below 2^18).
constexpr uint64_t kQSlotDesc = uint64_t((2 * kBox) >> 4);   // descriptor step between the slots' Q tiles
constexpr uint64_t kStageDesc = uint64_t(kTileBytes >> 4);    // descriptor step between ring stages

__device__ __forceinline__ void pf_issue_qk(uint32_t d, uint64_t qdesc, uint64_t kdesc) {
  constexpr uint32_t idesc = make_idesc_bf16(kPfRows, kPfKeys, 0);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {  // K = 128 in steps of 16
    const uint64_t off = uint64_t(((kk >> 2) * kBox + (kk & 3) * 32) >> 4);
    umma_ss(d, qdesc + off, kdesc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// Q K^T for one 64-key half of a K tile (kdesc already points at its first row).
__device__ __forceinline__ void pf_issue_qk_half(uint32_t d, uint64_t qdesc, uint64_t kdesc) {
  constexpr uint32_t idesc = make_idesc_bf16(kPfRows, 64, 0);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint64_t off = uint64_t(((kk >> 2) * kBox + (kk & 3) * 32) >> 4);
    umma_ss(d, qdesc + off, kdesc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V over the keys 64h .. 64h+63 of a tile: P as bf16 hi + lo (two
// products per 16 keys), or, in fp16 mode, P and V fp16 (one product).
template <bool kF16>
__device__ __forceinline__ void pf_issue_pv_half(uint32_t d, uint32_t pbase, uint64_t vdesc, int h, bool accumulate) {
  constexpr uint32_t idesc = kF16 ? make_idesc_f16(kPfRows, kD, 1) : make_idesc_bf16(kPfRows, kD, 1);
#pragma unroll
  for (int k4 = 0; k4 < 4; ++k4) {
    const int kk = 4 * h + k4;
    const uint32_t pcol = (kk >> 1) * 32 + (kk & 1) * 8;
    const uint64_t b = vdesc + uint64_t((kk * 2048) >> 4);
    umma_ts(d, pbase + pcol, b, idesc, (accumulate || k4 > 0) ? 1u : 0u);
    if (!kF16) umma_ts(d, pbase + pcol + 16, b, idesc, 1u);
  }
}

// tanh(y) for a pair of |y| <= 1.5 on the FMA pipe instead of the special-
// function unit: the odd polynomial y + y^3 Q(y^2), Q of degree 5, fitted here
// for absolute error on [0, 1.5] by Lawson's iteratively reweighted least
// squares (which converges to the minimax fit), then rounded to fp32: maximum
// absolute error 3.0e-6 including the fp32 steps (tanh.approx: 7.8e-6). The
// caller checks the range: beyond it the polynomial leaves [-1, 1] quickly.
constexpr float kTanhPolyRange = 1.5f;
__device__ __forceinline__ uint64_t tanh_poly_f2(uint64_t y) {
  const uint64_t z = f2_mul(y, y);
  const uint64_t yz = f2_mul(y, z);
  uint64_t q = f2_fma(f2_pack(0x1.38efe80p-12f, 0x1.38efe80p-12f), z, f2_pack(-0x1.999c920p-9f, -0x1.999c920p-9f));
  q = f2_fma(q, z, f2_pack(0x1.f398040p-7f, 0x1.f398040p-7f));
  q = f2_fma(q, z, f2_pack(-0x1.9526880p-5f, -0x1.9526880p-5f));
  q = f2_fma(q, z, f2_pack(0x1.0ddb2e0p-3f, 0x1.0ddb2e0p-3f));
  q = f2_fma(q, z, f2_pack(-0x1.55208c0p-2f, -0x1.55208c0p-2f));
  return f2_fma(yz, q, y);
}

// Column pairs of a 32-key chunk whose exp2 runs on the FMA pipe (bit e: pair
// e); the rest use the special-function unit, which also evaluates every tanh.
// Half is best in both modes (fp16 mode: 0.668 ms with half, 0.706 with three
// quarters, 0.747 with all on prefill_b1_t8192).
constexpr uint32_t kPolyPairs = 0x3333;

// For a chunk whose logits all lie in the tanh polynomial's range, per mode:
// the column pairs whose tanh runs as that polynomial on the FMA pipe, and the
// pairs whose exp2 does (the rest on the special-function unit). Measured on
// prefill_b1_t8192: fp16 mode 0.661 ms with half the tanh on the polynomial and
// every exp2 on the special-function unit, against 0.666 with the plain split
// above (0.674-0.679 with a quarter, 0.690 / 0.710 / 0.780 with five eighths,
// three quarters, all). bf16 mode has the FMA pipe busier (the lo half of P):
// every split tried was slower there (0.765-0.85 against 0.750), so it has none.
constexpr uint32_t kTanhPolyPairsBf16 = 0x0000, kTanhPolyExp2PairsBf16 = 0x0000;
constexpr uint32_t kTanhPolyPairsF16 = 0x5555, kTanhPolyExp2PairsF16 = 0x0000;
// Raw logit bound of the polynomial's range |s * kY| <= kTanhPolyRange.
constexpr float kTanhPolyRaw = kTanhPolyRange / kY;

// S -> P for one 32-key chunk c of one row (this thread's TMEM lane): weights
// 2^(30 log2(e) tanh(y) - mref) (mref = 30 log2(e): exp(capped logit - 30)),
// zero where masked, accumulated into the row sum and returned as bf16 hi/lo
// halves for the caller to write back over S (keys 32c..32c+31: hi in columns
// 32c..32c+15, lo in 32c+16..32c+31), or in fp16 mode as fp16 pairs (hi only).
// kTanhPoly (fp16 mode, every logit of the warp's chunk within kTanhPolyRaw):
// the tanh of the pairs in kTanhPolyPairs is the FMA-pipe polynomial.
template <bool kMask, bool kF16, bool kTanhPoly>
__device__ __forceinline__ void pf_softmax_chunk(const uint32_t (&sv)[32], int c, int rel, float mref, float& l0,
                                                 float& l1, uint32_t (&hi)[16], uint32_t (&lo)[16]) {
  // The arithmetic of capped_weight and split_bf16x2, two columns at a time
  // with packed f32x2 instructions; the exp2 of the pairs in the exp2 mask is
  // the FMA-pipe polynomial instead of ex2.approx.
  constexpr uint32_t exp2_pairs = !kTanhPoly ? kPolyPairs : kF16 ? kTanhPolyExp2PairsF16 : kTanhPolyExp2PairsBf16;
  constexpr uint32_t tanh_pairs = !kTanhPoly ? 0u : kF16 ? kTanhPolyPairsF16 : kTanhPolyPairsBf16;
  const uint64_t y2 = f2_pack(kY, kY), t2 = f2_pack(kT, kT), mt2 = f2_pack(-mref, -mref);
  uint64_t l = f2_pack(l0, l1);
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    float y0, y1, x0, x1;
    const uint64_t y = f2_mul(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), y2);
    uint64_t t;
    if ((tanh_pairs >> e) & 1) {
      t = tanh_poly_f2(y);
    } else {
      f2_unpack(y, y0, y1);
      t = f2_pack(tanh_approx(y0), tanh_approx(y1));
    }
    const uint64_t x = f2_fma(t, t2, mt2);
    float w0, w1;
    if ((exp2_pairs >> e) & 1) {
      exp2_poly_f2(x, w0, w1);
    } else {
      f2_unpack(x, x0, x1);
      w0 = ex2_approx(x0);
      w1 = ex2_approx(x1);
    }
    if (kMask) {
      w0 = (c * 32 + 2 * e <= rel) ? w0 : 0.f;
      w1 = (c * 32 + 2 * e + 1 <= rel) ? w1 : 0.f;
    }
    const uint64_t w = f2_pack(w0, w1);
    l = f2_add(l, w);
    if (kF16) {
      hi[e] = pack_f16x2(w0, w1);
    } else {
      hi[e] = pack_bf16x2(w0, w1);
      float r0, r1;
      f2_unpack(f2_sub(w, f2_pack(bf16lo_to_f32(hi[e]), bf16hi_to_f32(hi[e]))), r0, r1);
      lo[e] = pack_bf16x2(r0, r1);
    }
  }
  f2_unpack(l, l0, l1);
}

// Largest raw logit among this thread's visible keys of 32 logits starting at
// key column c0 of the tile (-inf if none).
template <bool kMask>
__device__ __forceinline__ float pf_rowmax32(const uint32_t (&a)[32], int c0, int rel) {
  float mx = -INFINITY;
#pragma unroll
  for (int e = 0; e < 32; ++e) mx = (!kMask || c0 + e <= rel) ? fmaxf(mx, __uint_as_float(a[e])) : mx;
  return mx;
}

// One warp's half of a tile: key columns 64 half .. 64 half + 63 of its rows,
// in two 32-column chunks (a TMEM load returns in ~30 cycles, so no prefetch).
template <bool kMask, bool kF16>
__device__ __forceinline__ void pf_softmax_half(uint32_t trow, int half, int rel, float mref, float& l0, float& l1) {
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int c = 2 * half + cc;
    uint32_t a[32];
    uint32_t hi[16], lo[16];
    tmem_ld32(trow + c * 32, a);
    tmem_wait_ld_dep(a);
    constexpr uint32_t tanh_pairs = kF16 ? kTanhPolyPairsF16 : kTanhPolyPairsBf16;
    if (tanh_pairs != 0 && !kMask) {
      // The polynomial form only when every logit of the warp's chunk in its
      // columns is in its range (a warp-uniform choice; fmaxf skips a NaN
      // logit, which stays NaN through the polynomial as through tanh.approx).
      // Only whole-visible chunks take it, so that keys behind a mask, whatever
      // the cache holds there, cannot change which form the visible ones get.
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if ((tanh_pairs >> e) & 1)
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(a[2 * e])), fabsf(__uint_as_float(a[2 * e + 1]))));
      if (__all_sync(0xffffffffu, m <= kTanhPolyRaw)) {
        pf_softmax_chunk<kMask, kF16, true>(a, c, rel, mref, l0, l1, hi, lo);
      } else {
        pf_softmax_chunk<kMask, kF16, false>(a, c, rel, mref, l0, l1, hi, lo);
      }
    } else {
      pf_softmax_chunk<kMask, kF16, false>(a, c, rel, mref, l0, l1, hi, lo);
    }
    tmem_st16(trow + c * 32, hi);
    if (!kF16) tmem_st16(trow + c * 32 + 16, lo);
  }
}

// Largest raw logit among this thread's visible keys of the half's 64 (-inf if none).
template <bool kMask>
__device__ __forceinline__ float pf_rowmax_half(uint32_t trow, int half, int rel) {
  float mx = -INFINITY;
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    uint32_t a[32];
    tmem_ld32(trow + (2 * half + cc) * 32, a);
    tmem_wait_ld_dep(a);
    mx = fmaxf(mx, pf_rowmax32<kMask>(a, (2 * half + cc) * 32, rel));
  }
  return mx;
}

// Split-pass epilogue of one epilogue warp (slot, half, quad) for a unit whose
// item is shared among `parts` units: the unit's unnormalised O (the warp's 32
// rows x 64 features) and, from half 0, the rows' sums and references go to
// the workspace; one thread per slot then counts the unit, and the item's last
// unit to finish adds every part in part order (so the result does not depend
// on which unit finishes last) and stages the output rows. Returns 1 when this
// warp staged output rows, 0 when it has none to write, -1 when a bounded wait
// gave up. Out of line: its registers stay out of the softmax loop's.
__device__ __noinline__ int pf_split_epilogue(const PfParams& p, PfBars* bars, volatile int* abort, int unit,
                                              int item, int parts, int slot, int half, int quad, int lane,
                                              uint32_t trow, float lt, float mref, bool over, uint8_t* stage,
                                              uint32_t parity) {
  const int r = quad * 32 + lane;
  const size_t su = size_t(unit) * 2 + slot;
  float4* po = p.part_o + (su * 2 + half) * (16 * kPfRows) + r;
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    uint32_t ov[32];
    tmem_ld32(trow + 128 + half * 64 + cc * 32, ov);
    tmem_wait_ld_dep(ov);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      po[(cc * 8 + q) * kPfRows] = make_float4(__uint_as_float(ov[4 * q]), __uint_as_float(ov[4 * q + 1]),
                                               __uint_as_float(ov[4 * q + 2]), __uint_as_float(ov[4 * q + 3]));
  }
  if (half == 0) p.part_lm[su * kPfRows + r] = make_float2(lt, mref);
  tc_fence_before();
  mbar_arrive(&bars->o_empty[slot]);  // O is read: the next unit's products may overwrite it
  __threadfence();                    // this thread's part is visible before the item's count moves
  __syncwarp();
  if (lane == 0) {
    if (over) atomicOr(&bars->split_over[slot], 1);
    mbar_arrive(&bars->split_in[slot]);
  }
  if (half == 0 && quad == 0 && lane == 0) {
    // one thread per slot counts the unit once all eight warps wrote theirs
    int last = 0;
    if (mbar_wait(&bars->split_in[slot], parity, abort, p.status)) {
      __threadfence();
      last = atomicAdd(p.part_cnt + item * 2 + slot, 1) == parts - 1;
      if (bars->split_over[slot]) pf_fallback(p, p.item_base + item);  // the fallback pass recomputes the item
      bars->split_over[slot] = 0;
    }
    bars->split_last[slot] = last;
    mbar_arrive(&bars->split_out[slot]);
  }
  if (!mbar_wait(&bars->split_out[slot], parity, abort, p.status)) return -1;
  if (!bars->split_last[slot]) return 0;
  __threadfence();
  // Part k's weights are 2^(t - m_k) (m_k its reference); on the common
  // reference mx they are scaled by 2^(m_k - mx) <= 1.
  const size_t su0 = size_t(item) * p.n_parts * 2 + slot;  // part 0 of the item, this slot
  float2 lm[kPfMaxParts];
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < kPfMaxParts; ++k)
    if (k < parts) {
      lm[k] = __ldcg(p.part_lm + (su0 + 2 * k) * kPfRows + r);
      mx = fmaxf(mx, lm[k].y);
    }
  float fk[kPfMaxParts];
  float lsum = 0.f;
#pragma unroll
  for (int k = 0; k < kPfMaxParts; ++k)
    if (k < parts) {
      fk[k] = ex2_approx(lm[k].y - mx);
      lsum = fmaf(lm[k].x, fk[k], lsum);
    }
  const float inv_l = 1.0f / lsum;
#pragma unroll 2
  for (int c = 0; c < 8; ++c) {  // 16-byte chunk c of the row's 64 output features (8 bf16)
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
    for (int k = 0; k < kPfMaxParts; ++k)
      if (k < parts) {
        const float4* pk4 = p.part_o + ((su0 + 2 * k) * 2 + half) * (16 * kPfRows) + r;
        const float4 v0 = __ldcg(pk4 + (2 * c) * kPfRows), v1 = __ldcg(pk4 + (2 * c + 1) * kPfRows);
        acc[0] = fmaf(v0.x, fk[k], acc[0]);
        acc[1] = fmaf(v0.y, fk[k], acc[1]);
        acc[2] = fmaf(v0.z, fk[k], acc[2]);
        acc[3] = fmaf(v0.w, fk[k], acc[3]);
        acc[4] = fmaf(v1.x, fk[k], acc[4]);
        acc[5] = fmaf(v1.y, fk[k], acc[5]);
        acc[6] = fmaf(v1.z, fk[k], acc[6]);
        acc[7] = fmaf(v1.w, fk[k], acc[7]);
      }
    *reinterpret_cast<uint4*>(stage + r * 128 + ((c ^ (r & 7)) << 4)) =
        make_uint4(pack_bf16x2(acc[0] * inv_l, acc[1] * inv_l), pack_bf16x2(acc[2] * inv_l, acc[3] * inv_l),
                   pack_bf16x2(acc[4] * inv_l, acc[5] * inv_l), pack_bf16x2(acc[6] * inv_l, acc[7] * inv_l));
  }
  return 1;
}

// kF16: fp16 mode; kList: bf16 mode over the fallback list only; kSplit:
// fp16 mode over units that share their items' key tiles (the split pass).
template <bool kF16, bool kList, bool kSplit>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const PfParams p) {
  // (tm_v: bf16 V of the cache, or in fp16 mode the fp16 copy of V in the workspace)
  extern __shared__ uint8_t smem_raw[];
  // The fallback pass runs as a programmatic dependent of the fp16 pass: wait
  // for that grid's writes (the list, the outputs it replaces). A no-op otherwise.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kQBytes;                           // K ring
  uint8_t* sV = sK + kPfStages * kTileBytes;              // V ring
  PfBars* bars = reinterpret_cast<PfBars*>(smem + kPfData);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 2);
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 2);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s][0], 1);
      mbar_init(&bars->s_full[s][1], 1);
      mbar_init(&bars->p_full[s][0], 128);
      mbar_init(&bars->p_full[s][1], 128);
      mbar_init(&bars->o_full[s], 1);
      mbar_init(&bars->o_empty[s], 256);
      mbar_init(&bars->lsum_ready[s], 256);
      mbar_init(&bars->epi_done[s], 8);
      for (int q = 0; q < 4; ++q) mbar_init(&bars->xbar[s][q], 64);
      mbar_init(&bars->split_in[s], 8);
      mbar_init(&bars->split_out[s], 1);
      bars->split_over[s] = 0;
    }
    mbar_init(&bars->mma_done, 2);
    bars->abort = 0;
    fence_barrier_init();
  }
  // Every role reads each item's sequence integers; stage them once.
  for (int b = threadIdx.x; b < p.B && b < kPfSeqCache; b += blockDim.x) {
    bars->seq_start[b] = __ldg(p.start_pos + b);
    bars->seq_valid[b] = p.valid_len ? __ldg(p.valid_len + b) : p.T;
    if (kF16) bars->seq_vflag[b] = __ldg(p.v_flags + b);
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_o);
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
      int kv_it = 0, q_it = 0;
      for (int rd = 0, item; (item = pf_item_index<kList>(p, rd)) >= 0; ++rd) {
        const PfItem it = pf_item<kF16, kSplit>(p, bars, item);
        if (it.n_kv == 0) continue;
        if (!mbar_wait(&bars->q_empty, (q_it & 1) ^ 1, abort, p.status)) break;
        mbar_arrive_expect_tx(&bars->q_full, kQBytes);
        for (int hs = 0; hs < 2; ++hs) {
          const int h = it.g * kGroup + it.hp * 2 + hs;
          for (int half = 0; half < 2; ++half)
            tma_load_4d(sQ + (hs * 2 + half) * kBox, &tm_q, &bars->q_full, half * 64, h, it.qt * kPfRows, it.b);
        }
        ++q_it;
        bool ok = true;
        for (int j = 0; j < it.n_kv; ++j, ++kv_it) {
          const int st = kv_it % kPfStages;
          const uint32_t par = ((kv_it / kPfStages) & 1) ^ 1;
          if (!mbar_wait(&bars->k_empty[st], par, abort, p.status)) {
            ok = false;
            break;
          }
          int krow, kb;
          kv_coord(p.pm, it.b, (it.j0 + j) * kPfKeys, krow, kb, p.status);  // a tile is one page when paged
          mbar_arrive_expect_tx(&bars->k_full[st], kTileBytes);
          tma_load_4d(sK + st * kTileBytes, &tm_k, &bars->k_full[st], 0, it.g, krow, kb);
          tma_load_4d(sK + st * kTileBytes + kBox, &tm_k, &bars->k_full[st], 64, it.g, krow, kb);
          if (!mbar_wait(&bars->v_empty[st], par, abort, p.status)) {
            ok = false;
            break;
          }
          // fp16 mode reads V from the copy in the workspace, contiguous per
          // sequence whether or not the cache is paged
          const int vrow = kF16 ? (it.j0 + j) * kPfKeys : krow, vb = kF16 ? it.b : kb;
          mbar_arrive_expect_tx(&bars->v_full[st], kTileBytes);
          tma_load_4d(sV + st * kTileBytes, &tm_v, &bars->v_full[st], 0, it.g, vrow, vb);
          tma_load_4d(sV + st * kTileBytes + kBox, &tm_v, &bars->v_full[st], 64, it.g, vrow, vb);
        }
        if (!ok) break;
      }
      // Drain: copies still in flight (only after an abort) land before the CTA exits.
      volatile int never = 0;
      for (int t = max(0, kv_it - kPfStages); t < kv_it; ++t) {
        mbar_wait(&bars->k_full[t % kPfStages], (t / kPfStages) & 1, &never, p.status);
        mbar_wait(&bars->v_full[t % kPfStages], (t / kPfStages) & 1, &never, p.status);
      }
      if (q_it > 0) mbar_wait(&bars->q_full, (q_it - 1) & 1, &never, p.status);
    }
  } else if (warp == 1 || warp == 18) {
    // ------------------------------------------------------------ MMA issuers (one warp per slot)
    // The warp runs converged through the waits; one fixed lane issues every
    // MMA and commit (a commit tracks the MMAs of the thread that issues it).
    const bool leader = elect_one();
    const int slot = warp == 1 ? 0 : 1;
    const uint32_t s_tm = tmem + slot * 256, o_tm = s_tm + 128;
    const uint64_t qd = make_sdesc_sw128(smem_u32(sQ), 16, 1024) + slot * kQSlotDesc;
    const uint64_t kd = make_sdesc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t vd = make_sdesc_sw128(smem_u32(sV), kBox, 1024);
    int kv_it = 0, q_it = 0, item_it = 0;
    int pc0 = 0, pc1 = 0;  // P hand-overs consumed per half (p_full parity)
    bool ok = true;
    for (int rd = 0, item; ok && (item = pf_item_index<kList>(p, rd)) >= 0; ++rd) {
      const PfItem it = pf_item<kF16, kSplit>(p, bars, item);
      if (it.n_kv == 0) continue;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->q_full, q_it & 1, abort, p.status))) break;
      {
        const int st = kv_it % kPfStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->k_full[st], (kv_it / kPfStages) & 1, abort, p.status))) break;
        tc_fence_after();
        if (leader) {
          if (it.n_sub >= 2)
            pf_issue_qk(s_tm, qd, kd + st * kStageDesc);
          else
            pf_issue_qk_half(s_tm, qd, kd + st * kStageDesc);
          umma_commit(&bars->s_full[slot][0]);
          if (it.n_sub >= 2) umma_commit(&bars->s_full[slot][1]);
          // (the last tile's K and V stages are handed back by the epilogue, which
          // stages the output in them)
          if (it.n_kv > 1) umma_commit(&bars->k_empty[st]);
          if (it.n_sub <= 2) umma_commit(&bars->q_empty);  // Q is read by no later product
        }
        __syncwarp();
        // The first tile's other inputs, waited while that product runs.
        const bool w = mbar_wait(&bars->v_full[st], (kv_it / kPfStages) & 1, abort, p.status) &&
                       (it.n_sub <= 2 || mbar_wait(&bars->k_full[(kv_it + 1) % kPfStages], ((kv_it + 1) / kPfStages) & 1, abort, p.status)) &&
                       mbar_wait(&bars->o_empty[slot], (item_it & 1) ^ 1, abort, p.status);
        if (!__all_sync(0xffffffffu, w)) break;
      }
      for (int u = 0; u < it.n_sub; ++u) {
        const int h = u & 1, j = u >> 1;
        const int cur = kv_it + j;
        const int st = cur % kPfStages, stn = (cur + 1) % kPfStages;
        const bool qk_next = u + 2 < it.n_sub;
        const bool tile_end = h == 1 || u == it.n_sub - 1;
        // V of tile j and K of tile j + 1 were waited for earlier (item start or
        // the middle of the previous tile's second step); only P is waited here.
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->p_full[slot][h], uint32_t(h ? pc1 : pc0) & 1, abort, p.status))) {
          ok = false;
          break;
        }
        if (h) ++pc1; else ++pc0;
        tc_fence_after();
        if (leader) pf_issue_pv_half<kF16>(o_tm, s_tm, vd + st * kStageDesc, h, u > 0);
        __syncwarp();
        if (h == 1 && u + 1 < it.n_sub) {
          // inputs of the next tile's steps: its V and the K after it
          const bool w = mbar_wait(&bars->v_full[stn], ((cur + 1) / kPfStages) & 1, abort, p.status) &&
                         (u + 3 >= it.n_sub || mbar_wait(&bars->k_full[st], ((cur + 2) / kPfStages) & 1, abort, p.status));
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (leader) {
          if (qk_next) {
            pf_issue_qk_half(s_tm + 64 * h, qd, kd + stn * kStageDesc + uint64_t((8192 * h) >> 4));
            umma_commit(&bars->s_full[slot][h]);
            // The item's last Q K^T: the producer may load the next item's Q
            // while the remaining P V products and the epilogue run.
            if (u + 3 == it.n_sub) umma_commit(&bars->q_empty);
          }
          if (tile_end && j + 1 < it.n_kv) {  // not the item's last tile
            umma_commit(&bars->v_empty[st]);
            if (j + 2 < it.n_kv) umma_commit(&bars->k_empty[stn]);
          }
          if (u == it.n_sub - 1) umma_commit(&bars->o_full[slot]);
        }
        __syncwarp();
      }
      kv_it += it.n_kv;
      ++q_it;
      ++item_it;
    }
    // No MMA may still be running when TMEM is released.
    if (leader) umma_commit(&bars->mma_done);
    __syncwarp();
    volatile int never = 0;
    mbar_wait(&bars->mma_done, 0, &never, p.status);
  } else if (warp >= 2 && warp <= 17) {
    // ------------------------------------------------------------ softmax + epilogue
    const int slot = (warp - 2) >> 3;
    const int half = ((warp - 2) >> 2) & 1;    // key columns / output features 64 half ..
    const int quad = warp & 3;                 // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;            // query row within the tile
    const uint32_t trow = tmem + (uint32_t(quad * 32) << 16) + slot * 256;
    int tile_cnt = 0, item_it = 0, sub_cnt = 0, xch_cnt = 0, split_cnt = 0;
    for (int rd = 0, item; (item = pf_item_index<kList>(p, rd)) >= 0; ++rd) {
      const PfItem it = pf_item<kF16, kSplit>(p, bars, item);
      if (it.n_kv == 0) {
        if (it.part == 0 && slot == 0 && half == 0 && r == 0) {
          if (it.bad) report(p.status, it.bad);
          if (kF16 && it.redirect) pf_fallback(p, it.item);
        }
        continue;
      }
      const int i = it.qt * kPfRows + r;
      // last visible key of this row, counted from the unit's first key
      const int lim = min(it.s + i, it.s + it.n - 1) - it.j0 * kPfKeys;
      float l0 = 0.f, l1 = 0.f;
      float mref = kT;  // bf16 mode: the fixed reference logit 30 (30 log2(e) in log2 units)
      bool ok = true;
      for (int u = half; u < it.n_sub; u += 2) {
        const int j = u >> 1;
        ok = mbar_wait(&bars->s_full[slot][half], sub_cnt & 1, abort, p.status);
        ++sub_cnt;
        if (!__all_sync(0xffffffffu, ok)) {  // leave together: the TMEM ops below are warp-collective
          ok = false;
          break;
        }
        tc_fence_after();
        const int rel = lim - j * kPfKeys;       // columns c <= rel are visible
        // The choice must be warp-uniform: the TMEM loads and stores inside
        // are warp-collective (.sync.aligned).
        const bool unmasked = __all_sync(0xffffffffu, rel >= 64 * half + 63);
        if (kF16 && j == 0) {
          // fp16 mode: the row's reference from the unit's first tile (both halves)
          float mx = unmasked ? pf_rowmax_half<false>(trow, half, rel) : pf_rowmax_half<true>(trow, half, rel);
          if (it.n_sub >= 2) {
            bars->xmax[slot][quad][half][lane] = mx;
            mbar_arrive(&bars->xbar[slot][quad]);
            const bool w = mbar_wait(&bars->xbar[slot][quad], xch_cnt & 1, abort, p.status);
            ++xch_cnt;
            if (!__all_sync(0xffffffffu, w)) {
              ok = false;
              break;
            }
            mx = fmaxf(mx, bars->xmax[slot][quad][half ^ 1][lane]);
          }
          // Key 0 is visible to every row, so mx is finite, except in a split
          // unit after an item's first: rows with no visible key in it (all
          // their weights zero) keep a finite reference through the clamp.
          mref = kT * tanh_approx((kSplit ? fmaxf(mx, -1.0e30f) : mx) * kY) + kPfHeadroom;
        }
        if (unmasked)
          pf_softmax_half<false, kF16>(trow, half, rel, mref, l0, l1);
        else
          pf_softmax_half<true, kF16>(trow, half, rel, mref, l0, l1);
        if (!kF16 && u == it.n_sub - 1) {
          // Zero the V rows of the last tile that lie beyond every visible key.
          // Both slots do it (same zeros) before handing over their P, since
          // each slot's PV product may be issued first.
          const int first_dead = it.kv_end - (it.j0 + j) * kPfKeys;
          const int st = (tile_cnt + j) % kPfStages;
          // The tile's V may still be landing: for a half-0 step the issuer has
          // not waited for it yet, and the zeros must not be overwritten by it.
          const bool vw = mbar_wait(&bars->v_full[st], ((tile_cnt + j) / kPfStages) & 1, abort, p.status);
          if (!__all_sync(0xffffffffu, vw)) {
            ok = false;
            break;
          }
          if (r >= first_dead) {
            uint4* v0 = reinterpret_cast<uint4*>(sV + st * kTileBytes + r * 128);
            uint4* v1 = reinterpret_cast<uint4*>(sV + st * kTileBytes + kBox + r * 128);
            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              v0[q] = z;
              v1[q] = z;
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[slot][half]);
      }
      if (!ok) break;
      tile_cnt += it.n_kv;
      // row sum of both halves (double-buffered by item parity)
      bars->lsum[item_it & 1][slot][half][r] = l0 + l1;
      mbar_arrive(&bars->lsum_ready[slot]);
      // Epilogue: O / l -> bf16 for this half's 64 output features, staged in
      // shared memory (128-byte swizzled, as TMA expects) and written by TMA, so
      // the scattered rows do not pass through the load/store unit. The staging
      // buffers are the item's last K stage (slot 0) and V stage (slot 1): every
      // product of both slots has read them once both slots' O are complete.
      ok = mbar_wait(&bars->lsum_ready[slot], item_it & 1, abort, p.status) &&
           mbar_wait(&bars->o_full[0], item_it & 1, abort, p.status) &&
           mbar_wait(&bars->o_full[1], item_it & 1, abort, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const float lt = bars->lsum[item_it & 1][slot][0][r] + bars->lsum[item_it & 1][slot][1][r];
      const int h = it.g * kGroup + it.hp * 2 + slot;
      const int st_last = (tile_cnt - 1) % kPfStages;
      uint8_t* stage = (slot == 0 ? sK : sV) + st_last * kTileBytes + half * kBox;
      bool store = true;  // this warp's output rows are staged
      if (!kSplit || it.parts == 1) {
        // fp16 mode: a weight sum that reached fp16's range means some weight may
        // have overflowed: the fallback pass recomputes the item (a half-0 warp
        // of each quadrant reports; duplicates are harmless)
        if (kF16 && half == 0 && __any_sync(0xffffffffu, !(lt < 65504.0f)) && lane == 0) pf_fallback(p, it.item);
        const float inv_l = 1.0f / lt;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t ov[32];
          tmem_ld32(trow + 128 + half * 64 + cc * 32, ov);
          tmem_wait_ld_dep(ov);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = cc * 4 + q;  // 16-byte chunk of the row's 128 bytes
            *reinterpret_cast<uint4*>(stage + r * 128 + ((c ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
        tc_fence_before();
        mbar_arrive(&bars->o_empty[slot]);  // O is read: the next item's products may overwrite it
      } else {
        const int res =
            pf_split_epilogue(p, bars, abort, item, it.item - p.item_base, it.parts, slot, half, quad, lane, trow, lt,
                              mref, __any_sync(0xffffffffu, !(lt < 65504.0f)), stage, uint32_t(split_cnt & 1));
        ++split_cnt;
        if (!__all_sync(0xffffffffu, res >= 0)) break;
        store = res > 0;
      }
      if (store) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int row0 = it.qt * kPfRows + quad * 32;
        if (store && row0 < p.T) {
          tma_store_4d(&tm_o, stage + quad * 32 * 128, half * 64, h, row0, it.b);
          bulk_commit_group();
          bulk_wait_read_all();
        }
        mbar_arrive(&bars->epi_done[slot]);
        // One thread per slot hands the two staging stages back to the producer
        // once all eight of the slot's stores have read them (each stage needs
        // one hand-back from each slot).
        if (half == 0 && quad == 2) {
          if (mbar_wait(&bars->epi_done[slot], item_it & 1, abort, p.status)) {
            mbar_arrive(&bars->k_empty[st_last]);
            mbar_arrive(&bars->v_empty[st_last]);
          }
        }
      }
      __syncwarp();
      ++item_it;
    }
    if (lane == 0) bulk_wait_all();  // output stores complete before the CTA exits
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------------------
// fp16 mode pre-pass: the fp16 copy of V. For sequence b with a valid start s,
// rows [0, s + T) of the cache (contiguous, or through the block table) are
// rounded to nearest fp16 and rows [s + T, round_up(s + T, 128)) are zeroed, so
// every key tile the fp16 pass reads is finite. A finite |v| >= 65520 (beyond
// fp16) sets v_flags[b]: the fp16 pass then hands all of that sequence's items
// to the fallback pass.
__global__ void __launch_bounds__(256) v_to_half_kernel(const uint4* __restrict__ cache_v, PageMap pm,
                                                        const int32_t* start_pos, int T, int Tmax, int vh_rows,
                                                        int from_start, uint4* __restrict__ vh, int32_t* v_flags,
                                                        int32_t* zero, int n_zero, int32_t* status) {
  // the key-range split's per-item counters start at zero
  if (blockIdx.y == 0)
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x) zero[i] = 0;
  const int b = blockIdx.y;
  const int s = __ldg(start_pos + b);
  if (s < 0 || (long long)s + T > Tmax) return;  // the attention passes skip this sequence
  const int rows = s + T, rows_pad = min(vh_rows, (rows + kPfKeys - 1) / kPfKeys * kPfKeys);
  const int first = from_start ? s : 0;  // rows below `first` are already converted (reuse)
  constexpr int kChunks = kKVHeads * kD / 8;  // 16-byte chunks (8 values) per row
  bool over = false;
  for (long long e = (long long)first * kChunks + (long long)blockIdx.x * blockDim.x + threadIdx.x;
       e < (long long)rows_pad * kChunks; e += (long long)gridDim.x * blockDim.x) {
    const int row = int(e / kChunks), ch = int(e % kChunks);
    uint4 out = make_uint4(0, 0, 0, 0);
    if (row < rows) {
      int src_row, src_b;
      kv_coord(pm, b, row, src_row, src_b, status);  // (row, b) contiguous, (page row, 0) paged
      const size_t rows_per_seq = pm.table ? size_t(0) : size_t(Tmax);
      const uint4 in = __ldg(cache_v + ((size_t)src_b * rows_per_seq + src_row) * kChunks + ch);
      const uint32_t w[4] = {in.x, in.y, in.z, in.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = bf16lo_to_f32(w[q]), c = bf16hi_to_f32(w[q]);
        over |= (fabsf(a) >= 65520.f && fabsf(a) != INFINITY) || (fabsf(c) >= 65520.f && fabsf(c) != INFINITY);
        o[q] = pack_f16x2(a, c);
      }
      out = make_uint4(o[0], o[1], o[2], o[3]);
    }
    vh[((size_t)b * vh_rows + row) * kChunks + ch] = out;
  }
  if (__any_sync(0xffffffffu, over) && (threadIdx.x & 31) == 0) atomicOr(v_flags + b, 1);
}

}  // namespace grok

using namespace grok;

// Extra inputs of the fp16 mode and of the fallback pass.
struct PfExtra {
  bool f16 = false;                 // fp16 mode: v_half holds the fp16 copy of V, [B][vh_rows][8][128]
  const void* v_half = nullptr;
  int vh_rows = 0;
  const int32_t* v_flags = nullptr;
  int32_t* fb_count = nullptr;      // fallback list (written by the fp16 pass, read by the fallback pass)
  int32_t* fb_list = nullptr;
  int fb_cap = 0;
  bool fallback = false;            // bf16 mode over the listed items only, launched as a dependent
  int n_units = -1;                 // units of this pass (-1: every item, whole)
  bool split = false;               // fp16 split pass: items [item_base, ...) shared among n_parts units each
  int item_base = 0, n_parts = 1;
  float4* part_o = nullptr;
  float2* part_lm = nullptr;
  int32_t* part_cnt = nullptr;
};

static grok_status prefill_launch(const grok_bf16* q_rot, const grok_bf16* k_src, const grok_bf16* v_src,
                                  uint64_t kv_rows, uint64_t kv_seqs, PageMap pm, const int32_t* start_pos,
                                  const int32_t* valid_len, int B, int T, int Tmax, grok_bf16* out, int32_t* dev_status,
                                  void* stream, const PfExtra& ex = PfExtra()) {
  int sms = 0;
  grok_status st = device_sm_count(&sms);
  if (st != GROK_OK) return st;

  CUtensorMap tq, tk, tv, to;
  const uint32_t box[4] = {64, 1, 128, 1};
  {
    const uint64_t dims[4] = {kD, kQHeads, uint64_t(T), uint64_t(B)};
    const uint64_t strides[3] = {kD * 2, uint64_t(kQHeads) * kD * 2, uint64_t(T) * kQHeads * kD * 2};
    if ((st = encode_tmap_bf16_4d(&tq, q_rot, dims, strides, box)) != GROK_OK) return st;
    const uint32_t obox[4] = {64, 1, 32, 1};  // one epilogue warp's 32 rows x 64 features
    if ((st = encode_tmap_bf16_4d(&to, out, dims, strides, obox)) != GROK_OK) return st;
  }
  {
    const uint64_t dims[4] = {kD, kKVHeads, kv_rows, kv_seqs};
    const uint64_t strides[3] = {kD * 2, uint64_t(kKVHeads) * kD * 2, kv_rows * kKVHeads * kD * 2};
    if ((st = encode_tmap_bf16_4d(&tk, k_src, dims, strides, box)) != GROK_OK) return st;
    if (ex.f16) {
      const uint64_t hdims[4] = {kD, kKVHeads, uint64_t(ex.vh_rows), uint64_t(B)};
      const uint64_t hstrides[3] = {kD * 2, uint64_t(kKVHeads) * kD * 2, uint64_t(ex.vh_rows) * kKVHeads * kD * 2};
      if ((st = encode_tmap_f16_4d(&tv, ex.v_half, hdims, hstrides, box)) != GROK_OK) return st;
    } else if ((st = encode_tmap_bf16_4d(&tv, v_src, dims, strides, box)) != GROK_OK) {
      return st;
    }
  }
  PfParams prm;
  prm.B = B;
  prm.T = T;
  prm.Tmax = Tmax;
  prm.pm = pm;
  prm.n_qt = (T + kPfRows - 1) / kPfRows;
  prm.n_items = prm.n_qt * B * kKVHeads * 3;
  prm.start_pos = start_pos;
  prm.valid_len = valid_len;
  prm.status = dev_status;
  prm.v_flags = ex.v_flags;
  prm.fb_count = ex.fb_count;
  prm.fb_list = ex.fb_list;
  prm.fb_cap = ex.fb_cap;
  prm.item_list = ex.fallback ? ex.fb_list : nullptr;
  prm.item_count = ex.fallback ? ex.fb_count : nullptr;
  prm.n_units = ex.n_units >= 0 ? ex.n_units : prm.n_items;
  prm.item_base = ex.split ? ex.item_base : 0;
  prm.n_parts = ex.split ? ex.n_parts : 1;
  prm.part_o = ex.part_o;
  prm.part_lm = ex.part_lm;
  prm.part_cnt = ex.part_cnt;

  static bool attr_set[kMaxDevices][4] = {};  // per device and kernel instance; idempotent
  int dev = 0;
  grok_status dst = device_index(&dev);
  if (dst != GROK_OK) return dst;
  const int mode = ex.split ? 3 : ex.f16 ? 1 : ex.fallback ? 2 : 0;
  auto kernel = mode == 3   ? prefill_kernel<true, false, true>
                : mode == 1 ? prefill_kernel<true, false, false>
                : mode == 2 ? prefill_kernel<false, true, false>
                            : prefill_kernel<false, false, false>;
  if (!attr_set[dev][mode]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    if (e != cudaSuccess) return fail(cuda_status(e), "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    attr_set[dev][mode] = true;
  }
  // The fallback pass does not know how many items it has (the list is on the
  // device), so it takes one CTA per SM; it is a programmatic dependent of the
  // fp16 pass, so its launch overlaps that pass's tail, and it waits for the
  // whole fp16 grid (griddepcontrol.wait) before reading the list.
  const int grid = ex.fallback ? sms : (prm.n_units < sms ? prm.n_units : sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPfThreads);
  cfg.dynamicSmemBytes = kPfSmem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = ex.fallback ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, prm);
  if (e != cudaSuccess) return fail(cuda_status(e), "prefill launch: %s", cudaGetErrorString(e));
  return check_launch("prefill");
}

extern "C" grok_status grok_attn_prefill(const grok_bf16* q_rot, const grok_bf16* cache_k,
                                         const grok_bf16* cache_v, const int32_t* start_pos,
                                         const int32_t* valid_len, int B, int T, int Tmax, grok_bf16* out,
                                         int32_t* dev_status, void* stream) {
  if (!q_rot || !cache_k || !cache_v || !start_pos || !out)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill: null pointer");
  if (!aligned16(q_rot) || !aligned16(cache_k) || !aligned16(cache_v) || !aligned16(out))
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill: bf16 tensors must be 16-byte aligned");
  if (B < 1 || T < 1 || Tmax < 1 || T > Tmax || Tmax > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill: need B >= 1, 1 <= T <= Tmax <= %d (B=%d T=%d Tmax=%d)",
                GROK_MAX_POSITION, B, T, Tmax);
  return prefill_launch(q_rot, cache_k, cache_v, uint64_t(Tmax), uint64_t(B), PageMap{nullptr, 0, 0}, start_pos,
                        valid_len, B, T, Tmax, out, dev_status, stream);
}

extern "C" grok_status grok_attn_prefill_paged(const grok_bf16* q_rot, const grok_bf16* k_pool,
                                               const grok_bf16* v_pool, int n_pages, const int32_t* block_table,
                                               int max_pages, const int32_t* start_pos, const int32_t* valid_len,
                                               int B, int T, grok_bf16* out, int32_t* dev_status, void* stream) {
  if (!q_rot || !k_pool || !v_pool || !block_table || !start_pos || !out)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill_paged: null pointer");
  if (!aligned16(q_rot) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill_paged: bf16 tensors must be 16-byte aligned");
  const long long Tmax = (long long)max_pages * GROK_PAGE_TOKENS;
  if (B < 1 || T < 1 || n_pages < 1 || max_pages < 1 || T > Tmax || Tmax > GROK_MAX_POSITION ||
      (long long)n_pages * GROK_PAGE_TOKENS > (1LL << 31))
    return fail(GROK_ERR_INVALID_ARG,
                "grok_attn_prefill_paged: need B, T, n_pages, max_pages >= 1, T <= max_pages * %d <= %d "
                "(B=%d T=%d max_pages=%d n_pages=%d)",
                GROK_PAGE_TOKENS, GROK_MAX_POSITION, B, T, max_pages, n_pages);
  return prefill_launch(q_rot, k_pool, v_pool, uint64_t(n_pages) * GROK_PAGE_TOKENS, 1,
                        PageMap{block_table, max_pages, n_pages}, start_pos, valid_len, B, T, int(Tmax), out,
                        dev_status, stream);
}

// ----------------------------------------------------------------------------
// Prefill with fp16 softmax weights (grok_attn_prefill_ws). Workspace layout:
//   int32 v_flags[B], fb_count, fb_list[fb_cap]  (padded to 256 bytes)
//   fp16 V copy [B][round_up(Tmax, 128)][8][128]
//   optional, for the key-range split (at most one unit per SM):
//     int32 part_cnt[sms][2] (padded to 256 bytes), float2 part_lm[sms][2][128],
//     float4 part_o[sms][2][2][16][128]
static int ws_vh_rows(int Tmax) { return (Tmax + kPfKeys - 1) / kPfKeys * kPfKeys; }
static int prefill_items(int B, int T) { return B * ((T + kPfRows - 1) / kPfRows) * kKVHeads * 3; }

// The key-range split. With fewer than two work items per SM, the items left
// for the ragged last round (all of them when there are fewer items than SMs)
// would hold their SMs while the rest idle: 192 equal items of a chunk over a
// long cache on 152 SMs keep 40 SMs for two items. Those items are instead
// shared among P = min(4, SMs / items) units each, run by a second pass, and
// combined by each item's last unit to finish (at most one unit per SM, so the
// partial outputs take at most SMs x 130 KB). Only caches of 16 key tiles or
// more qualify, since a unit holds at least 8 tiles.
static bool split_allowed(int Tmax) { return (Tmax + kPfKeys - 1) / kPfKeys >= 2 * kPfMinPartTiles; }
static size_t split_cnt_bytes(int sms) { return (size_t(sms) * 2 * sizeof(int32_t) + 255) & ~size_t(255); }
static size_t split_lm_bytes(int sms) { return size_t(sms) * 2 * kPfRows * sizeof(float2); }
static size_t split_area_bytes(int sms) {
  return split_cnt_bytes(sms) + split_lm_bytes(sms) + size_t(sms) * 2 * 2 * 16 * kPfRows * sizeof(float4);
}
static int ws_fb_cap(int B, int Tmax) {
  // items of the largest call (T = Tmax); each may be listed by up to 8
  // quadrant warps of the fp16 pass (split items: once per slot by each of up
  // to 4 units) plus once for its sequence's V
  return 9 * ((Tmax + kPfRows - 1) / kPfRows) * B * kKVHeads * 3;
}
static size_t ws_header_bytes(int B, int Tmax) {
  return ((size_t(B) + 1 + size_t(ws_fb_cap(B, Tmax))) * sizeof(int32_t) + 255) & ~size_t(255);
}

// The part every call needs: the header and the fp16 V copy.
static size_t ws_base_bytes(int B, int Tmax) {
  return ws_header_bytes(B, Tmax) + size_t(B) * ws_vh_rows(Tmax) * kKVHeads * kD * 2;
}

extern "C" grok_status grok_attn_prefill_workspace_min(int B, int Tmax, size_t* bytes) {
  if (!bytes) return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill_workspace_min: null pointer");
  if (B < 1 || Tmax < 1 || Tmax > GROK_MAX_POSITION || (long long)B * ws_vh_rows(Tmax) > (1LL << 31))
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill_workspace_min: need B >= 1, 1 <= Tmax <= %d",
                GROK_MAX_POSITION);
  *bytes = ws_base_bytes(B, Tmax);
  return GROK_OK;
}

extern "C" grok_status grok_attn_prefill_workspace(int B, int Tmax, size_t* bytes) {
  grok_status st = grok_attn_prefill_workspace_min(B, Tmax, bytes);
  if (st != GROK_OK || !split_allowed(Tmax)) return st;
  int sms = 0;
  if ((st = device_sm_count(&sms)) != GROK_OK) return st;
  *bytes += split_area_bytes(sms);
  return GROK_OK;
}

// The fp16-weight prefill over a contiguous cache or a paged pool (pm), its
// arguments already checked: V pre-pass, whole items, the split pass, then the
// bf16 fallback pass over the listed items.
static grok_status prefill_ws_run(const grok_bf16* q_rot, const grok_bf16* k_src, const grok_bf16* v_src,
                                  uint64_t kv_rows, uint64_t kv_seqs, PageMap pm, const int32_t* start_pos,
                                  const int32_t* valid_len, int B, int T, int Tmax, grok_bf16* out, void* workspace,
                                  size_t workspace_bytes, int reuse_v_half, int32_t* dev_status, void* stream,
                                  const char* what) {
  size_t need = 0;
  grok_status st = grok_attn_prefill_workspace_min(B, Tmax, &need);
  if (st != GROK_OK) return st;
  if (workspace_bytes < need)
    return fail(GROK_ERR_INVALID_ARG, "%s: workspace of %zu bytes is smaller than the %zu needed", what,
                workspace_bytes, need);
  int sms = 0;
  if ((st = device_sm_count(&sms)) != GROK_OK) return st;
  // items [0, n_whole) run whole; the rest, if the split applies, n_parts units each
  const int n_items = prefill_items(B, T);
  int n_whole = n_items, n_parts = 1;
  if (n_items < 2 * sms && split_allowed(Tmax) && workspace_bytes >= need + split_area_bytes(sms)) {
    const int rest = n_items % sms;
    const int parts = rest > 0 ? std::min(kPfMaxParts, sms / rest) : 1;
    if (parts > 1) {
      n_whole = n_items - rest;
      n_parts = parts;
    }
  }
  const int n_split = n_items - n_whole;
  char* split_area = static_cast<char*>(workspace) + need;
  const int vh_rows = ws_vh_rows(Tmax);
  int32_t* v_flags = static_cast<int32_t*>(workspace);
  int32_t* fb_count = v_flags + B;
  int32_t* fb_list = fb_count + 1;
  void* vh = static_cast<char*>(workspace) + ws_header_bytes(B, Tmax);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // the list count, and unless the copy is reused the overflow flags (reused: they persist)
  cudaError_t e = reuse_v_half ? cudaMemsetAsync(fb_count, 0, sizeof(int32_t), s)
                               : cudaMemsetAsync(v_flags, 0, (size_t(B) + 1) * sizeof(int32_t), s);
  if (e != cudaSuccess) return fail(cuda_status(e), "cudaMemsetAsync: %s", cudaGetErrorString(e));
  {
    const long long per_seq = (long long)(reuse_v_half ? ((T + 2 * kPfKeys - 1) / kPfKeys * kPfKeys) : vh_rows) *
                              (kKVHeads * kD / 8);
    long long bx = (per_seq + 255) / 256;
    const long long cap = ((long long)sms * 8 + B - 1) / B;  // about 8 blocks per SM in all
    if (bx > cap) bx = cap;
    if (bx < 1) bx = 1;
    v_to_half_kernel<<<dim3(unsigned(bx), unsigned(B)), 256, 0, s>>>(
        reinterpret_cast<const uint4*>(v_src), pm, start_pos, T, Tmax, vh_rows, reuse_v_half ? 1 : 0,
        static_cast<uint4*>(vh), v_flags, reinterpret_cast<int32_t*>(split_area), 2 * n_split, dev_status);
    if ((st = check_launch("v_to_half")) != GROK_OK) return st;
  }
  PfExtra ex;
  ex.f16 = true;
  ex.v_half = vh;
  ex.vh_rows = vh_rows;
  ex.v_flags = v_flags;
  ex.fb_count = fb_count;
  ex.fb_list = fb_list;
  ex.fb_cap = ws_fb_cap(B, Tmax);
  if (n_whole > 0) {
    ex.n_units = n_whole;
    if ((st = prefill_launch(q_rot, k_src, v_src, kv_rows, kv_seqs, pm, start_pos,
                             valid_len, B, T, Tmax, out, dev_status, stream, ex)) != GROK_OK)
      return st;
  }
  if (n_split > 0) {
    ex.split = true;
    ex.item_base = n_whole;
    ex.n_parts = n_parts;
    ex.n_units = n_split * n_parts;
    ex.part_cnt = reinterpret_cast<int32_t*>(split_area);
    ex.part_lm = reinterpret_cast<float2*>(split_area + split_cnt_bytes(sms));
    ex.part_o = reinterpret_cast<float4*>(split_area + split_cnt_bytes(sms) + split_lm_bytes(sms));
    if ((st = prefill_launch(q_rot, k_src, v_src, kv_rows, kv_seqs, pm, start_pos,
                             valid_len, B, T, Tmax, out, dev_status, stream, ex)) != GROK_OK)
      return st;
  }
  ex.split = false;
  ex.n_units = -1;
  ex.f16 = false;
  ex.fallback = true;
  return prefill_launch(q_rot, k_src, v_src, kv_rows, kv_seqs, pm, start_pos,
                        valid_len, B, T, Tmax, out, dev_status, stream, ex);
}


extern "C" grok_status grok_attn_prefill_ws(const grok_bf16* q_rot, const grok_bf16* cache_k,
                                            const grok_bf16* cache_v, const int32_t* start_pos,
                                            const int32_t* valid_len, int B, int T, int Tmax, grok_bf16* out,
                                            void* workspace, size_t workspace_bytes, int reuse_v_half,
                                            int32_t* dev_status, void* stream) {
  if (!q_rot || !cache_k || !cache_v || !start_pos || !out || !workspace)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill_ws: null pointer");
  if (!aligned16(q_rot) || !aligned16(cache_k) || !aligned16(cache_v) || !aligned16(out))
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill_ws: bf16 tensors must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill_ws: workspace must be 256-byte aligned");
  if (B < 1 || T < 1 || Tmax < 1 || T > Tmax || Tmax > GROK_MAX_POSITION)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill_ws: need B >= 1, 1 <= T <= Tmax <= %d (B=%d T=%d Tmax=%d)",
                GROK_MAX_POSITION, B, T, Tmax);
  return prefill_ws_run(q_rot, cache_k, cache_v, uint64_t(Tmax), uint64_t(B), PageMap{nullptr, 0, 0}, start_pos,
                        valid_len, B, T, Tmax, out, workspace, workspace_bytes, reuse_v_half, dev_status, stream,
                        "grok_attn_prefill_ws");
}

extern "C" grok_status grok_attn_prefill_ws_paged(const grok_bf16* q_rot, const grok_bf16* k_pool,
                                                  const grok_bf16* v_pool, int n_pages, const int32_t* block_table,
                                                  int max_pages, const int32_t* start_pos, const int32_t* valid_len,
                                                  int B, int T, grok_bf16* out, void* workspace,
                                                  size_t workspace_bytes, int reuse_v_half, int32_t* dev_status,
                                                  void* stream) {
  if (!q_rot || !k_pool || !v_pool || !block_table || !start_pos || !out || !workspace)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill_ws_paged: null pointer");
  if (!aligned16(q_rot) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill_ws_paged: bf16 tensors must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(GROK_ERR_INVALID_ARG, "grok_attn_prefill_ws_paged: workspace must be 256-byte aligned");
  const long long Tmax = (long long)max_pages * GROK_PAGE_TOKENS;
  if (B < 1 || T < 1 || n_pages < 1 || max_pages < 1 || T > Tmax || Tmax > GROK_MAX_POSITION ||
      (long long)n_pages * GROK_PAGE_TOKENS > (1LL << 31))
    return fail(GROK_ERR_INVALID_ARG,
                "grok_attn_prefill_ws_paged: need B, T, n_pages, max_pages >= 1, T <= max_pages * %d <= %d "
                "(B=%d T=%d max_pages=%d n_pages=%d)",
                GROK_PAGE_TOKENS, GROK_MAX_POSITION, B, T, max_pages, n_pages);
  return prefill_ws_run(q_rot, k_pool, v_pool, uint64_t(n_pages) * GROK_PAGE_TOKENS, 1,
                        PageMap{block_table, max_pages, n_pages}, start_pos, valid_len, B, T, int(Tmax), out,
                        workspace, workspace_bytes, reuse_v_half, dev_status, stream, "grok_attn_prefill_ws_paged");
}
