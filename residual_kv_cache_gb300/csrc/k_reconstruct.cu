// k_reconstruct.cu - fused read path (ResidualKV notes §2.5 boxed equation
// KV_hat = f_d(z~) + mean with f_d(z) = z W_d; §2.4 z~ = q Delta + min; §2.1 the
// restored pre-RoPE key is rotated at the token's own position; §2.7 only the selected
// tokens are restored).
//
// Work unit = (tile of 128 selected tokens, 128 output columns = one head for D = 128,
// two for D = 64).  A CTA owns a contiguous range of units (with several problems in one
// launch: every gridDim-th token tile, each with all its units), so consecutive units
// share the token tile.  Two loader warps stage each later token tile of the CTA in shared
// memory while the previous tile is restored: per row its record (validity, k_i,
// position, pool rows of its references), its extremes and, for code rows of at most
// 128 bytes, its codes.  Per token tile, the 512 epilogue threads (four warpgroups; the
// threads of TMEM lane r own token row r):
//   1. dequantise the row's codes in fp32 (z~ = q * Delta + min, Delta = (max - min) /
//      (2^b - 1)) and store bf16 z~ straight into tensor memory, where the tensor core
//      reads the A operand (two bf16 per 32-bit column); with d_c <= 256 z~ has two
//      buffers, so the next tile's goes in while the tensor core still reads this one's;
//   2. build the row's RoPE cos/sin for its 16 column pairs (float64-built two-level
//      tables, angle addition in fp32) into shared memory.
// Per unit, a TMA ring streams W_d^T tiles (the B operand) and one thread issues
// tcgen05.mma into one of two TMEM accumulators.  The epilogue warps prefetch, one unit
// ahead, exactly the reference bytes they will read (32 rows x 16 column pairs x <= 4
// references, 16-byte cp.async copies): the two warps that read the two halves of the
// same 32-byte sectors share one shared-memory slot per reference, one copying the x
// sectors and the other the y sectors, and meet at a named barrier per reference.  Each
// epilogue thread then sums its row's references (exact in fp32), adds the sum / k_i to
// its accumulator row (one fma for k_i = 1, 2, 4, where the scaling is exact; the
// correctly rounded s / 3 for k_i = 3), rotates the K columns and stores its 16 + 16 K
// or V values straight from registers, one 32-byte store per 16 bf16 values (a whole
// sector of the row); rows past the selection are not stored.
//
// Back-to-back launches overlap: every CTA lets the next launch of the stream start its
// CTAs as SMs free up, and a thread waits for the previous grid to complete only before
// its first output store, so one launch's first-tile setup (dependent loads of
// selections, slots and codes, dequantisation) hides behind the previous launch's last
// CTAs.  Nothing else this kernel reads is written by it.
//
// Per unit an SM pulls 256 d_c bytes of W_d^T and up to 64 KB of reference rows from L2;
// the tensor core finishes a unit's MMAs well within the epilogue's time, so the kernel
// is bound by the epilogue's dependent chains and the first tile's setup, not by the
// tensor core or by HBM.
//
// Restore fused into the sparse layer's attention (§2.7: o = softmax(q K_hat^T / sqrt(D))
// V_hat over the selected tokens; D = 128, bf16 K_hat / V_hat).  The same kernel,
// instantiated with kAttend, orders its units as (K head h, V head h) pairs of a token
// tile and keeps the restored rows on chip:
//   * the K unit's epilogue writes its bf16 K_hat rows into a shared-memory tile
//     (token-major, 128-byte swizzle), and the MMA thread computes the tile's scores
//     S = K_hat Q^T into the K accumulator's first 16 columns, Q holding the scaled query
//     rows of the head's group as bf16 high and low parts (q / sqrt(D) = hi + lo to
//     within 2^-16 relative), so that the tensor core's products stay exact;
//   * the epilogue reads each row's scores, takes the tile's maximum m and the weights
//     p = exp(s - m) per query head (rows past the selection weigh nothing; computed in
//     base 2, log2(e) folded into the query scale), writes m and l = sum p per (tile,
//     query head) to global memory, and puts p into a second tile as bf16 high and low
//     parts;
//   * the V unit's epilogue writes its V_hat rows transposed (dimension-major) into the
//     first tile, and the MMA thread computes V_hat^T P into the V accumulator's first
//     16 columns: per dimension d and query head, sum over the tile's tokens of p v_d;
//   * a merge kernel combines the tiles of each query head: M = max m, L = sum l 2^(m-M),
//     o = sum o_tile 2^(m - M) / L.
// No restored row is written to global memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_common.cuh"

namespace rkv {
namespace {

// 20 warps: 0 TMEM + W_d^T producer, 1 MMA, 2..3 loaders, 4..19 epilogue.
// The register file is split over the four SM sub-partitions, so 18 or 20 warps both
// cap a thread at 96 registers.
constexpr int kReconThreads = 640;
constexpr int kEpiWarpR = 4;                 // first epilogue warp
constexpr int kNT = 128;                     // output columns per unit
constexpr uint32_t kBBytes = kNT * 128;      // one 64-wide k-block of W_d^T rows
constexpr uint32_t kPlaneBytes = kTileM * 32;            // one 32-byte sector per tile row
constexpr uint32_t kGBytes = 2 * 4 * 2 * kPlaneBytes;    // [group pair][ref][x|y] planes
constexpr uint32_t kCSBytes = 4 * 8 * kTileM * 16;   // cos/sin: 4 groups x 8 float4 x 128 rows
constexpr uint32_t kBarBytes = 1024;            // mbarriers, TMEM slot; from +512 the
                                               // fused read's reduction slots
constexpr int kRecInts = 8;                  // staged row record: flags, pos, pool rows 0..3, seq
constexpr int kLoadWarp0 = 2;                // warps 2..3 stage the CTA's later tiles
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol = 2 * kNT;          // z~ after the two accumulators
constexpr int kMaxStages = 8;
// Extra cost of a token-tile change inside a CTA's range (staging the next tile's z~ and
// cos/sin while the tensor core drains), in quarter units.
#ifndef RKV_TILE_CHANGE_COST4
#define RKV_TILE_CHANGE_COST4 10
#endif
constexpr int kTileChangeCost4 = RKV_TILE_CHANGE_COST4;
// restore + attention: K_hat / V_hat^T tile (two 64-column swizzle atoms of 128 rows),
// the weight tile P and the pair's query tile (16 rows x 128 bf16 each)
constexpr uint32_t kKVBytes = 2 * kTileM * 128;
constexpr uint32_t kRowTile16 = 16 * 128;            // one swizzle atom of a 16-row tile
constexpr uint32_t kPBytes = 2 * kRowTile16;
constexpr uint32_t kAttendBytes = kKVBytes + 2 * kPBytes;
constexpr int kGroupBar0 = 9;     // named barriers 9..12: the four warps of one epilogue group
constexpr int kHalfBar0 = 13;     // 13, 14: the eight warps of groups 0-1, 2-3

struct ReconArgs {
  const int32_t* seq;
  const int32_t* pos;
  int n_sel;
  int n_tiles;   // 2d_k / 128
  int units;
  int b_stages;
  const uint8_t* codes;
  const uint32_t* meta;
  const int32_t* ref_idx;
  const uint8_t* pool8;
  const float2* rope_lo;
  const float2* rope_hi;
  void* k_out;
  void* v_out;
  int out_f32;
  int B, T_cap, R_cap, topk, dkv, dk, dc, D, G, bits, code_bytes;
  int zbufs;          // z~ buffers in TMEM: 2 when d_c <= 256, else 1
  int stage_codes;    // later tiles' codes are staged in shared memory (code_bytes <= 256)
  int chunk_mask;     // swizzle of a staged code row's 16-byte chunks: chunk c ^ (row & mask)
  int* status;
  // restore + attention only
  const float* q;     // [N gq][D] fp32 decode queries; query head h gq + g reads head h
  int gq;             // query heads per key/value head (<= 8)
  float q_scale;      // log2(e) / sqrt(D): scores in base-2 units, s' = s log2(e)
  float* part_m;      // [tiles][N gq] each token tile's maximum score s'
  float* part_l;      // [tiles][N gq] sum of 2^(s' - m) over the tile
  float* part_o;      // [tiles][N gq][D] sum of 2^(s' - m) v over the tile
};

// One 32-byte store (eight 32-bit words) to a 32-byte aligned global address.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat16 lo = __float2bfloat16_rn(a), hi = __float2bfloat16_rn(b);
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// Byte offset of bf16 element (r, c) in a K-major tile stored with the 128-byte swizzle:
// 64-column atoms `atom` bytes apart, 128-byte rows, 16-byte chunk (c % 64) / 8 of row r
// at position chunk ^ (r % 8).
__device__ __forceinline__ uint32_t sw128_off(int r, int c, uint32_t atom) {
  return (uint32_t)(c >> 6) * atom + (uint32_t)r * 128u +
         ((uint32_t)(((c & 63) >> 3) ^ (r & 7)) << 4) + (uint32_t)(c & 7) * 2u;
}

// s[i] += value of FP8 byte i of v (16 bytes); exact in fp32 for <= 4 addends (their
// bits span 2^-9 .. 2^11).
__device__ __forceinline__ void fp8x16_add(uint4 v, float* s) {
  fp8x4_add(v.x, s[0], s[1], s[2], s[3]);
  fp8x4_add(v.y, s[4], s[5], s[6], s[7]);
  fp8x4_add(v.z, s[8], s[9], s[10], s[11]);
  fp8x4_add(v.w, s[12], s[13], s[14], s[15]);
}

// z~ = q * Delta + min of code groups g0 .. g0 + g_per - 1 (at most four) of one row into
// TMEM at zaddr + 16 g; mt[i] holds the group's (min, max) as two f16, cw[i] its packed
// codes.  An invalid row decodes to zeros.
__device__ __forceinline__ void dequant_groups(const ReconArgs& a, bool valid, const uint32_t* mt,
                                               const uint4* cw, int g0, int g_per, uint32_t zaddr) {
  // Codes become floats without integer-to-float conversions: a code q placed in the
  // low mantissa bits under the exponent of 2^23 reads as the float 2^23 + q exactly,
  // and one subtraction leaves q.  z~ = RN(RN(q * Delta) + min), two columns at a time.
  const int levels = (1 << a.bits) - 1;
  const uint64_t two23 = f32x2_pack(8388608.0f, 8388608.0f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (i >= g_per) break;
    const int g = g0 + i;
    float lo = __half2float(__ushort_as_half((unsigned short)(mt[i] & 0xFFFFu)));
    const float hi = __half2float(__ushort_as_half((unsigned short)(mt[i] >> 16)));
    float delta = __fdiv_rn(__fsub_rn(hi, lo), (float)levels);
    if (!valid) lo = 0.f, delta = 0.f;              // an invalid row decodes to zeros
    const uint64_t dd = f32x2_pack(delta, delta);
    const uint32_t w4[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
    uint32_t o[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      uint32_t t0, t1;                               // 2^23 + q of coordinates 2e, 2e + 1
      if (a.bits == 4) {
        // word e/4 holds coordinates 8 (e/4) + n in nibble n: the even nibbles of a
        // word are its bytes' low halves, the odd nibbles their high halves
        const uint32_t w = w4[e >> 2];
        const uint32_t sel = 0x7650u + (uint32_t)(e & 3);
        t0 = __byte_perm(w & 0x0F0F0F0Fu, 0x4B000000u, sel);
        t1 = __byte_perm((w >> 4) & 0x0F0F0F0Fu, 0x4B000000u, sel);
      } else {
        const int k = 2 * e;
        t0 = ((w4[k >> 4] >> (2 * (k & 15))) & 3u) | 0x4B000000u;
        t1 = ((w4[k >> 4] >> (2 * (k & 15) + 2)) & 3u) | 0x4B000000u;
      }
      const uint64_t q = f32x2_sub(f32x2_pack(__uint_as_float(t0), __uint_as_float(t1)), two23);
      // the addition stays scalar: ptxas contracts a packed multiply followed by a
      // packed add into one fused multiply-add, which rounds once instead of twice
      float m0, m1;
      f32x2_unpack(f32x2_mul(q, dd), m0, m1);
      o[e] = pack_bf16x2(__fadd_rn(m0, lo), __fadd_rn(m1, lo));
    }
    tmem_st16(zaddr + 16u * (uint32_t)g, o);
  }
}

// The inputs that belong to one restore problem: its selection, storage and status
// word.  A launch restores one problem, or several contexts' selections at once
// (reconstruct_multi_kernel), whose token tiles it numbers one after the other.
struct ProbView {
  const int32_t* seq;
  const int32_t* pos;
  int n_sel;
  const uint8_t* codes;
  const uint32_t* meta;
  const int32_t* ref_idx;
  int* status;
};

struct ReconProblems {
  int n;
  int tile0[kReconMaxProblems + 1];   // first token tile of each problem; [n] = all tiles
  const int32_t* seq[kReconMaxProblems];
  const int32_t* pos[kReconMaxProblems];
  int n_sel[kReconMaxProblems];
  const uint8_t* codes[kReconMaxProblems];
  const uint32_t* meta[kReconMaxProblems];
  const int32_t* ref_idx[kReconMaxProblems];
  const uint8_t* pool8[kReconMaxProblems];
  void* k_out[kReconMaxProblems];
  void* v_out[kReconMaxProblems];
  int* status[kReconMaxProblems];
};

struct ReconMaps {
  CUtensorMap tmW[kReconMaxProblems];   // each problem's W_d^T
};

// Problem of token tile T (tiles of problem i are [tile0[i], tile0[i + 1])).
__device__ __forceinline__ int problem_of(const ReconProblems& mp, int T) {
  int i = 0;
  while (i + 1 < mp.n && T >= mp.tile0[i + 1]) ++i;
  return i;
}

// Per-tile state of one epilogue thread's token row, packed into two registers.
struct RowState {
  int flags;    // bit 0: the row has a readable code and a first reference; bits 1..4:
                // reference t is a valid slot; bits 5..: k_i
  int pos;      // the token's position (RoPE)
  __device__ __forceinline__ bool valid() const { return flags & 1; }
  __device__ __forceinline__ bool has_ref(int t) const { return (flags >> (1 + t)) & 1; }
  __device__ __forceinline__ int kcnt() const { return flags >> 5; }
};

// A row's state, the pool rows of its references 0..3 (-1 where there is none) and the
// sequence and position of the same row of the next tile (-1 past the selection).
struct TileRow {
  RowState st;
  int r[4];
  int nx_s, nx_p;
};

// The row `row` of token tile m, whose sequence and position s_, p_ the caller has
// already loaded: its metadata and references, and its share of code groups
// [g0, g0 + g_per) dequantised (z~ = q * Delta + min in fp32, bf16 into TMEM at
// zaddr + 16 g; zeros for an invalid row).  Raises the device flags for bad selections.
// With `next`, also loads the next tile's sequence and position of the row, so that the
// next call starts with independent loads.
__device__ __forceinline__ TileRow tile_setup(const ReconArgs& a, const ProbView& v, int m,
                                              int row, int wg, int g0, int g_per,
                                              uint32_t zaddr, int s_, int p_, bool next) {
  TileRow tr;
  RowState& st = tr.st;
  const int64_t gi = (int64_t)m * kTileM + row;
  const bool in_sel = gi < v.n_sel;
  st.pos = 0;
  bool in_range = false;
  int64_t dst = 0;
  if (in_sel) {
    if (s_ < 0 || s_ >= a.B || p_ < 0 || p_ >= a.T_cap) {
      if (wg == 0) atomicOr(v.status, RKV_FLAG_BAD_INDEX);
    } else {
      in_range = true;
      dst = (int64_t)s_ * a.T_cap + p_;
      st.pos = p_;
    }
  }
  // one round trip: slots, extremes and codes together
  int32_t sl[4] = {-1, -1, -1, -1};
  uint32_t mt[4] = {0u, 0u, 0u, 0u};
  uint4 cw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) cw[i] = make_uint4(0u, 0u, 0u, 0u);
  const uint8_t* crow = v.codes + dst * a.code_bytes;
  if (in_range) {
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (t < a.topk) sl[t] = v.ref_idx[dst * a.topk + t];
    if (a.bits != 16) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i < g_per) {
          const int g = g0 + i;
          mt[i] = v.meta[dst * a.G + g];
          if (a.bits == 4) {
            cw[i] = *reinterpret_cast<const uint4*>(crow + (int64_t)g * 16);
          } else {
            const uint2 v = *reinterpret_cast<const uint2*>(crow + (int64_t)g * 8);
            cw[i] = make_uint4(v.x, v.y, 0u, 0u);
          }
        }
      }
    }
  }
  {
    const int64_t gn = gi + kTileM;
    const bool nx = next && gn < v.n_sel;
    tr.nx_s = nx ? v.seq[gn] : -1;
    tr.nx_p = nx ? v.pos[gn] : -1;
  }
  int kcnt = 0;
  bool valid = false;
#pragma unroll
  for (int t = 0; t < 4; ++t) tr.r[t] = -1;
  if (in_range) {
    if (sl[0] < 0 && wg == 0) atomicOr(v.status, RKV_FLAG_UNWRITTEN);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (sl[t] >= a.R_cap && wg == 0) atomicOr(v.status, RKV_FLAG_BAD_SLOT);
      if (sl[t] >= 0 && sl[t] < a.R_cap) {
        tr.r[t] = s_ * a.R_cap + sl[t];
        ++kcnt;
      }
    }
    valid = tr.r[0] >= 0 && kcnt > 0;
  }
  if (!valid) {
    kcnt = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) tr.r[t] = -1;
  }
  st.flags = (valid ? 1 : 0) | (kcnt << 5);
#pragma unroll
  for (int t = 0; t < 4; ++t) st.flags |= (tr.r[t] >= 0 ? 1 : 0) << (1 + t);
  // dequantise this row's share of code groups straight into TMEM
  if (a.bits == 16) {
    for (int g = g0; g < g0 + g_per; ++g) {
      uint32_t o[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = valid ? reinterpret_cast<const uint4*>(crow + (int64_t)g * 64)[q]
                              : make_uint4(0u, 0u, 0u, 0u);
        o[4 * q] = v.x, o[4 * q + 1] = v.y, o[4 * q + 2] = v.z, o[4 * q + 3] = v.w;
      }
      tmem_st16(zaddr + 16u * (uint32_t)g, o);
    }
  } else {
    dequant_groups(a, valid, mt, cw, g0, g_per, zaddr);
  }
  tmem_st_wait();
  return tr;
}

// Row `row` of token tile m staged for the epilogue by a loader thread: its record
// (flags as in RowState, position, pool rows of references 0..3 or -1, sequence), its
// extremes and, with a.stage_codes, its packed codes (16-byte chunks, chunk c stored at
// c ^ (row & a.chunk_mask)).  Raises the device flags for bad selections.
__device__ __forceinline__ void stage_row(const ReconArgs& a, const ProbView& v, int m, int row,
                                          int* rec, uint32_t* smeta, uint8_t* scodes) {
  const int64_t gi = (int64_t)m * kTileM + row;
  const bool in_sel = gi < v.n_sel;
  const int s_ = in_sel ? v.seq[gi] : -1;
  const int p_ = in_sel ? v.pos[gi] : -1;
  bool in_range = false;
  int64_t dst = 0;
  if (in_sel) {
    if (s_ < 0 || s_ >= a.B || p_ < 0 || p_ >= a.T_cap) {
      atomicOr(v.status, RKV_FLAG_BAD_INDEX);
    } else {
      in_range = true;
      dst = (int64_t)s_ * a.T_cap + p_;
    }
  }
  int32_t sl[4] = {-1, -1, -1, -1};
  if (in_range) {
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (t < a.topk) sl[t] = v.ref_idx[dst * a.topk + t];
  }
  int r[4] = {-1, -1, -1, -1};
  int kcnt = 0;
  if (in_range) {
    if (sl[0] < 0) atomicOr(v.status, RKV_FLAG_UNWRITTEN);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (sl[t] >= a.R_cap) atomicOr(v.status, RKV_FLAG_BAD_SLOT);
      if (sl[t] >= 0 && sl[t] < a.R_cap) {
        r[t] = s_ * a.R_cap + sl[t];
        ++kcnt;
      }
    }
  }
  const bool valid = in_range && r[0] >= 0 && kcnt > 0;
  if (!valid) {
    kcnt = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) r[t] = -1;
  }
  int flags = (valid ? 1 : 0) | (kcnt << 5);
#pragma unroll
  for (int t = 0; t < 4; ++t) flags |= (r[t] >= 0 ? 1 : 0) << (1 + t);
  if (valid) {
    if (a.bits != 16)
      for (int g = 0; g < a.G; ++g) smeta[row * a.G + g] = v.meta[dst * a.G + g];
    if (a.stage_codes) {
      const uint8_t* crow = v.codes + dst * a.code_bytes;
      uint8_t* srow = scodes + row * a.code_bytes;
      for (int c = 0; c < a.code_bytes / 16; ++c)
        cp_async16(srow + ((c ^ (row & a.chunk_mask)) << 4), crow + 16 * c);
    }
  }
  reinterpret_cast<int4*>(rec)[0] = make_int4(flags, in_range ? p_ : 0, r[0], r[1]);
  reinterpret_cast<int4*>(rec)[1] = make_int4(r[2], r[3], in_range ? s_ : 0, 0);
}

// First unit of CTA b's contiguous range (b = grid gives `units`).  The ranges split a
// cost of one per unit plus cost4 / 4 per token-tile boundary crossed inside
// a range evenly over the grid: each tile after the first carries that extra cost ahead
// of its first unit, and a cut falling there starts the next range on the tile.
__device__ __forceinline__ int range_start(int b, int grid, int units, int n_tiles, int cost4) {
  const int64_t tc = 4 * (int64_t)n_tiles + cost4;
  const int64_t total = (int64_t)(units / n_tiles) * tc - cost4;
  const int64_t c = (int64_t)b * total / grid + cost4;
  const int64_t t = c / tc;
  const int64_t off4 = c - t * tc - cost4;
  const int64_t u = t * n_tiles + (off4 <= 0 ? 0 : off4 / 4);
  return (int)(u < units ? u : units);
}

// Output column tile of unit j of a token tile: j itself, or with kAttend the pairs
// (K head j / 2, V head j / 2).
template <bool kAttend>
__device__ __forceinline__ int unit_col(int j, int n_tiles) {
  if constexpr (kAttend) return (j & 1) ? (n_tiles >> 1) + (j >> 1) : (j >> 1);
  return j;
}

// The kernel body.  tmWs: W_d^T's tensor map (one per problem with kMulti); mp: the
// problems of a multi-problem launch (unused otherwise: a's pointers are the problem).
template <bool kAttend, bool kMulti>
__device__ __forceinline__ void restore_body(const CUtensorMap* tmWs, const ReconArgs& a,
                                             const ReconProblems* mp) {
  extern __shared__ uint8_t smem_raw[];
  // problem of a token tile, its inputs, and the tile's index within the problem
  auto view = [&](int pi) -> ProbView {
    if constexpr (kMulti)
      return ProbView{mp->seq[pi], mp->pos[pi], mp->n_sel[pi], mp->codes[pi],
                      mp->meta[pi], mp->ref_idx[pi], mp->status[pi]};
    else
      return ProbView{a.seq, a.pos, a.n_sel, a.codes, a.meta, a.ref_idx, a.status};
  };
  auto tile_local = [&](int T, int& pi) -> int {
    if constexpr (kMulti) {
      pi = problem_of(*mp, T);
      return T - mp->tile0[pi];
    } else {
      pi = 0;
      return T;
    }
  };
  uint8_t* smem = align1024(smem_raw);
  const int nkb = a.dc / kTileK;
  uint8_t* sB = smem;                                       // b_stages x W_d^T k-block
  // restore + attention: K_hat / V_hat^T tile, weight tile, query tile
  uint8_t* sKV = sB + a.b_stages * kBBytes;
  uint8_t* sP = sKV + kKVBytes;
  uint8_t* sQ = sP + kPBytes;
  uint8_t* sG = kAttend ? sQ + kPBytes : sKV;               // per-warp reference slots
  float4* sCS = reinterpret_cast<float4*>(sG + kGBytes);
  int* sRec = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(sCS) + kCSBytes);  // staged tile
  uint32_t* sMeta = reinterpret_cast<uint32_t*>(sRec + kTileM * kRecInts);
  uint8_t* sCodes = reinterpret_cast<uint8_t*>(sMeta + kTileM * a.G);
  uint64_t* full = reinterpret_cast<uint64_t*>(
      sCodes + (a.stage_codes ? ((kTileM * a.code_bytes + 127) & ~127) : 0));
  uint64_t* empty = full + a.b_stages;
  uint64_t* tfull = empty + a.b_stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* afull = tempty + 2;                             // z~ of a tile is in TMEM
  uint64_t* afree = afull + 1;                              // the MMAs of a tile are done
  uint64_t* staged = afree + 1;                             // the next tile is staged
  uint64_t* sfree = staged + 1;                             // the staged tile has been read
  uint64_t* kready = sfree + 1;       // restore + attention: K_hat (and the queries) staged
  uint64_t* sdone = kready + 1;       //   the scores are in TMEM
  uint64_t* vready = sdone + 1;       //   V_hat^T and the weights staged
  uint64_t* odone = vready + 1;       //   V_hat^T P is in TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(odone + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* sRed = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 512);  // [4][16]

  const int warp = threadIdx.x >> 5;
  pdl_launch_dependents();
  // The CTA's units, in order.  One problem: a contiguous range, cost-balanced (with
  // kAttend cut between pairs).  Several problems (kMulti): every gridDim-th token tile,
  // each tile's units in a row, so that the CTAs work through the problems together and
  // the L2 holds one or two problems' pools and weights at a time rather than all.
  constexpr int kSpan = kAttend ? 2 : 1;
  int u_first = 0, u_count = 0, t_count = 0;          // first unit; units and tiles
  if constexpr (kMulti) {
    const int tiles = a.units / a.n_tiles, b = (int)blockIdx.x, gs = (int)gridDim.x;
    t_count = tiles > b ? (tiles - b + gs - 1) / gs : 0;
    u_count = t_count * a.n_tiles;
  } else {
    u_first = kSpan * range_start(blockIdx.x, gridDim.x, a.units / kSpan, a.n_tiles / kSpan,
                                  kTileChangeCost4 / kSpan);
    const int u_last = kSpan * range_start(blockIdx.x + 1, gridDim.x, a.units / kSpan,
                                           a.n_tiles / kSpan, kTileChangeCost4 / kSpan);
    u_count = u_last - u_first;
    t_count = u_count > 0 ? (u_last - 1) / a.n_tiles - u_first / a.n_tiles + 1 : 0;
  }
  auto unit_at = [&](int k) -> int {                  // the CTA's k-th unit
    if constexpr (kMulti)
      return ((int)blockIdx.x + (k / a.n_tiles) * (int)gridDim.x) * a.n_tiles + k % a.n_tiles;
    else
      return u_first + k;
  };
  auto tile_at = [&](int j) -> int {                  // the CTA's j-th token tile
    if constexpr (kMulti)
      return (int)blockIdx.x + j * (int)gridDim.x;
    else
      return u_first / a.n_tiles + j;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.b_stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 16);
    }
    mbar_init(afull, 16);
    mbar_init(afree, 1);
    mbar_init(staged, 2 * 64);       // 64 loader threads: a plain and a copy-completion arrival
    mbar_init(sfree, 16);
    mbar_init(kready, 16);
    mbar_init(sdone, 1);
    mbar_init(vready, 16);
    mbar_init(odone, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(tmWs);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer: W_d^T tiles
    if (elect_one()) {
      Ring ring;
      uint32_t issued = 0, issued_phase = 0;             // bit s: stage s used / its phase
      bool ok = true;
      int pw = 0;                                        // problem of unit u
      for (int k = 0; k < u_count && ok; ++k) {
        const int u = unit_at(k);
        const int n = unit_col<kAttend>(u % a.n_tiles, a.n_tiles);
        if constexpr (kMulti)
          while (pw + 1 < mp->n && u / a.n_tiles >= mp->tile0[pw + 1]) ++pw;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[ring.stage], ring.phase ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[ring.stage], kBBytes);
          tma_load_2d(sB + ring.stage * kBBytes, tmWs + pw, &full[ring.stage], kb * kTileK, n * kNT);
          issued |= 1u << ring.stage;
          issued_phase = (issued_phase & ~(1u << ring.stage)) | (ring.phase << ring.stage);
          ring.next(a.b_stages);
        }
      }
      if (!ok)
        for (int s = 0; s < a.b_stages; ++s)
          if ((issued >> s) & 1u) drain_wait(&full[s], (issued_phase >> s) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (A from TMEM)
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTileM, kNT);
      Ring ring;
      int acc = 0;
      uint32_t acc_phase = 0, a_phase = 0;
      int cur_m = -1, tt = -1;
      uint32_t zoff = 0;
      bool ok = true, any = false;
      int last_stage = 0;
      uint32_t last_phase = 0;
      // restore + attention: a pair's products of two 128 x 128 shared-memory tiles with a
      // 16-row tile (scores K_hat Q^T, then V_hat^T P), 16 accumulator columns each
      bool pend_o = false, small_last = false;
      uint32_t s_phase = 0, o_phase = 0, small_par = 0;
      uint64_t* small_bar = sdone;
      auto pair_mma = [&](uint32_t d, const uint8_t* A, const uint8_t* B) {
        constexpr uint32_t idesc16 = idesc_bf16_f32(kTileM, 16);
        const uint32_t a0 = smem_u32(A), b0 = smem_u32(B);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k)
            umma_bf16(d, sdesc_sw128(a0 + kb * (kTileM * 128) + k * 32),
                      sdesc_sw128(b0 + kb * kRowTile16 + k * 32), idesc16, (kb | k) != 0 ? 1u : 0u);
      };
      for (int k = 0; k < u_count && ok; ++k) {
        const int u = unit_at(k);
        const int m = u / a.n_tiles;
        if (m != cur_m) {
          // with one z~ buffer, the previous tile's z~ may be overwritten once its MMAs
          // are done
          if (cur_m >= 0 && a.zbufs == 1) umma_commit(afree);
          ++tt;
          zoff = (uint32_t)((tt % a.zbufs) * (a.dc / 2));
          if (!mbar_wait(afull, a_phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          a_phase ^= 1u;
          cur_m = m;
        }
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + acc * kNT;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[ring.stage], ring.phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b0 = smem_u32(sB + ring.stage * kBBytes);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k)
            umma_bf16_ta(d, tmem + kACol + zoff + (uint32_t)(kb * (kTileK / 2) + k * 8),
                         sdesc_sw128(b0 + k * 32), idesc, (kb | k) != 0 ? 1u : 0u);
          umma_commit(&empty[ring.stage]);
          any = true;
          last_stage = ring.stage;
          last_phase = ring.phase;
          ring.next(a.b_stages);
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        small_last = false;
        if constexpr (kAttend) {
          if (acc == 0) {
            // the next pair's K unit is issued: the previous pair's V_hat^T P next
            if (pend_o) {
              if (!mbar_wait(vready, o_phase, abort_flag, a.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              pair_mma(tmem + kNT, sKV, sP);
              umma_commit(odone);
              small_bar = odone, small_par = o_phase, small_last = true;
              o_phase ^= 1u;
              pend_o = false;
            }
          } else {
            // the pair's scores, once its K_hat rows (and the queries) are staged
            if (!mbar_wait(kready, s_phase, abort_flag, a.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            pair_mma(tmem, sKV, sQ);
            umma_commit(sdone);
            small_bar = sdone, small_par = s_phase, small_last = true;
            s_phase ^= 1u;
            pend_o = true;
          }
        }
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if constexpr (kAttend) {
        if (ok && pend_o) {
          if (mbar_wait(vready, o_phase, abort_flag, a.status)) {
            tc_fence_after();
            pair_mma(tmem + kNT, sKV, sP);
            umma_commit(odone);
            small_bar = odone, small_par = o_phase, small_last = true;
          } else {
            ok = false;
          }
        }
      }
      // MMAs complete in issue order: waiting for the last commit drains them all
      if (!ok && any) {
        if (small_last)
          drain_wait(small_bar, small_par);
        else
          drain_wait(&empty[last_stage], last_phase);
      }
    }
  } else if (warp < kEpiWarpR) {
    // ------------------------------------------------ loaders: the CTA's later tiles
    // (records, extremes, codes) staged in shared memory one tile ahead, so that a tile
    // change costs the epilogue no global round trip
    const int l = (int)threadIdx.x - 32 * kLoadWarp0;
    {
      uint32_t free_phase = 0;
      for (int j = 1; j < t_count; ++j) {
        const int m = tile_at(j);
        if (j > 1) {
          if (!mbar_wait(sfree, free_phase, abort_flag, a.status)) break;
          free_phase ^= 1u;
        }
        int pl;
        const int ml = tile_local(m, pl);
        const ProbView v = view(pl);
        stage_row(a, v, ml, l, sRec + l * kRecInts, sMeta, sCodes);
        stage_row(a, v, ml, l + 64, sRec + (l + 64) * kRecInts, sMeta, sCodes);
        cp_async_arrive_noinc(staged);
        mbar_arrive(staged);
      }
    }
    cp_async_wait_all();                               // no copy may outlive the CTA
  } else {
    // Four groups of four consecutive warps (warps 4..19).  Warp w reads TMEM lanes
    // [32 (w % 4), +32), so every group owns the same 128 rows; group g takes 16 of each
    // unit's 64 column pairs and a quarter of each row's code groups.
    const int ew = warp & 3;
    const int wg = (warp - kEpiWarpR) >> 2;
    const int row = ew * 32 + (int)lane_id();        // TMEM lane = tile row
    const uint32_t lane_base = (uint32_t)(ew * 32) << 16;
    const int P = a.D / 2;                           // pairs per head
    const int slot0 = 16 * wg;                       // first of this group's 16 pair slots
    const int hl = slot0 / P, j0 = slot0 % P;        // head within the unit, first pair
    const int xcol = hl * a.D + j0, ycol = xcol + P; // unit-local columns of x and y
    // Groups 2p and 2p+1 read the two 16-byte halves of the same 32-byte sectors of each
    // reference row (x columns, and y columns), so they share reference slots: plane
    // (ref t, x|y) of pair p holds one whole sector per tile row, the halves swapped on
    // every other group of four rows so that a warp's 16-byte reads hit distinct banks.
    // Per reference, the warp of group 2p copies the x sectors and the warp of group 2p+1
    // the y sectors of their 32 rows (two lanes per row, one instruction per 16 rows, so
    // each sector is fetched once); the two warps meet at named barrier 1 + ew + 4p.
    const int half = wg & 1;                           // this group's half of a sector
    const int bar_id = 1 + ew + 4 * (wg >> 1);
    const int xsec = xcol - 16 * half;                 // the pair's sectors (32-aligned)
    uint8_t* pslots = sG + (uint32_t)(wg >> 1) * (4 * 2 * kPlaneBytes);
    const uint32_t rd_off = (uint32_t)row * 32 + (uint32_t)((half ^ ((row >> 2) & 1)) * 16);
    const int cl = (int)lane_id();
    const int cp_r0 = ew * 32 + (cl >> 1);             // copies rows cp_r0 and cp_r0 + 16
    uint8_t* cp_dst0 = pslots + half * kPlaneBytes + (uint32_t)cp_r0 * 32 +
                       (uint32_t)(((cl & 1) ^ ((cp_r0 >> 2) & 1)) * 16);
    const int cp_off = (half ? xsec + P : xsec) + 16 * (cl & 1);
    // kMulti: bits 0..7 the problem of the current tile, bits 8..15 the problem the
    // thread's reference copies in flight are for (the next tile's, from its set-up on)
    int pp = 0;
    const uint32_t zaddr = tmem + lane_base + kACol;  // this thread's z~ columns (buffer 0)
    const int g0 = wg * a.G / 4;                     // this group's code groups [g0, g0+g_per)
    const int g_per = (wg + 1) * a.G / 4 - g0;
    float4* cs_row = sCS + wg * 8 * kTileM + row;    // entry i at cs_row[i * kTileM]

    // z~ of tile m into TMEM (the caller has made sure the tensor core is done with the
    // previous tile), then one arrival per warp on afull.
    int cp0[4], cp1[4];                               // pool rows this lane copies (per tile)
    int nx_s = -1, nx_p = -1;                         // the row of the next tile
    auto setup_a = [&](int m, const ProbView& v) -> RowState {
      const TileRow tr = tile_setup(a, v, m, row, wg, g0, g_per, zaddr, nx_s, nx_p, false);
      tc_fence_before();
      __syncwarp();
      if (lane_id() == 0) mbar_arrive(afull);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        cp0[t] = __shfl_sync(0xffffffffu, tr.r[t], cl >> 1);
        cp1[t] = __shfl_sync(0xffffffffu, tr.r[t], (cl >> 1) + 16);
      }
      return tr.st;
    };

    // z~ of the staged tile into z~ buffer zb (its previous tile's MMAs are done), the
    // row state and this lane's copy rows from the records, then one arrival per warp on
    // afull (the tensor core may start the tile) and on sfree (the loaders may restage).
    uint32_t staged_phase = 0;
    auto setup_s = [&](int zb, RowState& st, int ps) -> bool {
      const uint8_t* codes_s = a.codes;                // the staged tile's problem's codes
      if constexpr (kMulti) codes_s = mp->codes[ps];
      const bool w = mbar_wait(staged, staged_phase, abort_flag, a.status);
      bool wa = __all_sync(0xffffffffu, w);
      if constexpr (kAttend) wa = bar_red_and(kHalfBar0 + (wg >> 1), 256, wa);
      if (!wa) return false;
      staged_phase ^= 1u;
      const int* rec = sRec + row * kRecInts;
      st.flags = rec[0];
      st.pos = rec[1];
      const bool valid = st.valid();
      const uint32_t za = zaddr + (uint32_t)(zb * (a.dc / 2));
      const uint8_t* srow = sCodes + row * a.code_bytes;
      if (a.bits == 16) {
        const uint8_t* crow = codes_s + ((int64_t)rec[6] * a.T_cap + rec[1]) * a.code_bytes;
        for (int g = g0; g < g0 + g_per; ++g) {
          uint32_t o[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (valid)
              v = a.stage_codes
                      ? *reinterpret_cast<const uint4*>(srow + (((4 * g + q) ^ (row & a.chunk_mask)) << 4))
                      : reinterpret_cast<const uint4*>(crow + (int64_t)g * 64)[q];
            o[4 * q] = v.x, o[4 * q + 1] = v.y, o[4 * q + 2] = v.z, o[4 * q + 3] = v.w;
          }
          tmem_st16(za + 16u * (uint32_t)g, o);
        }
      } else {
        const uint8_t* crow = codes_s + ((int64_t)rec[6] * a.T_cap + rec[1]) * a.code_bytes;
        uint32_t mt[4] = {0u, 0u, 0u, 0u};
        uint4 cw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          cw[i] = make_uint4(0u, 0u, 0u, 0u);
          if (i < g_per && valid) {
            const int g = g0 + i;
            mt[i] = sMeta[row * a.G + g];
            if (a.bits == 4) {
              cw[i] = a.stage_codes
                          ? *reinterpret_cast<const uint4*>(srow + ((g ^ (row & a.chunk_mask)) << 4))
                          : *reinterpret_cast<const uint4*>(crow + (int64_t)g * 16);
            } else {
              const uint2 v = a.stage_codes
                                  ? *reinterpret_cast<const uint2*>(
                                        srow + (((g >> 1) ^ (row & a.chunk_mask)) << 4) + 8 * (g & 1))
                                  : *reinterpret_cast<const uint2*>(crow + (int64_t)g * 8);
              cw[i] = make_uint4(v.x, v.y, 0u, 0u);
            }
          }
        }
        dequant_groups(a, valid, mt, cw, g0, g_per, za);
      }
      tmem_st_wait();
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        cp0[t] = sRec[cp_r0 * kRecInts + 2 + t];
        cp1[t] = sRec[(cp_r0 + 16) * kRecInts + 2 + t];
      }
      tc_fence_before();
      __syncwarp();
      if (lane_id() == 0) {
        mbar_arrive(afull);
        mbar_arrive(sfree);
      }
      return true;
    };

    // cos/sin of the row's 16 pairs at its own position, into shared memory
    auto setup_cs = [&](int p) {
      const float4* th = reinterpret_cast<const float4*>(a.rope_hi + (int64_t)(p >> 9) * P + j0);
      const float4* tl = reinterpret_cast<const float4*>(a.rope_lo + (int64_t)(p & (kRopeLo - 1)) * P + j0);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 hv = __ldg(th + i), lv = __ldg(tl + i);
        float4 o;
        o.x = hv.x * lv.x - hv.y * lv.y;    // cos(A + B), pair 2i
        o.y = hv.y * lv.x + hv.x * lv.y;    // sin(A + B)
        o.z = hv.z * lv.z - hv.w * lv.w;    // pair 2i + 1
        o.w = hv.w * lv.z + hv.z * lv.w;
        cs_row[i * kTileM] = o;
      }
    };

    // One commit group per (unit, reference) and one empty group per unit: copy this
    // warp's sectors of reference t of unit column block n_next into its plane; nothing
    // when `active` is false or a row has no such reference.  Five groups per unit, so
    // that exactly three are always younger than the one waited for.
    auto issue_ref = [&](int n_next, bool active, int t) {
      if (active) {
        const int p0 = cp0[t], p1 = cp1[t];
        uint8_t* dst = cp_dst0 + (uint32_t)(t * 2) * kPlaneBytes;
        const uint8_t* pool = a.pool8;
        if constexpr (kMulti) pool = mp->pool8[(pp >> 8) & 0xff];
        const uint8_t* src = pool + cp_off + n_next * kNT;
        if (p0 >= 0) cp_async16(dst, src + (int64_t)p0 * a.dkv);
        if (p1 >= 0) cp_async16(dst + 16 * 32, src + (int64_t)p1 * a.dkv);
      }
      cp_async_commit();
    };

    RowState cur, nxt;
    bool waited = false;                               // previous grid complete (first store)
    int acc = 0;
    uint32_t acc_phase = 0, afree_phase = 0;
    int cur_m = -1, tt = 0;
    bool ok = true;
    uint32_t s_phase = 0, o_phase = 0;                // restore + attention
    // A wait that gives up makes the warp leave the unit loop, together with every warp
    // it meets at a named barrier.  Without kAttend that is the pair sharing reference
    // slots: the two vote.  With kAttend the four warps of a group also meet in the
    // softmax, which joins groups 0 and 1 (and 2 and 3) through their pairs: the eight
    // warps of each half vote together.  The two halves share no barrier.
    const int vote_id = kAttend ? kHalfBar0 + (wg >> 1) : bar_id;
    const int vote_n = kAttend ? 256 : 64;
    // V_hat^T P of the pair whose V unit is uv: lane d of the V accumulator, column g +
    // column gq + g = sum over the tile's tokens of p v_d; then the accumulator is free.
    auto finish_o = [&](int uv) -> bool {
      if (!bar_red_and(vote_id, vote_n, warp_wait(odone, o_phase, abort_flag, a.status))) return false;
      o_phase ^= 1u;
      tc_fence_after();
      const int gA = wg, gB = wg + 4;
      const bool hasA = gA < a.gq, hasB = gB < a.gq;
      const uint32_t tO = tmem + lane_base + kNT;
      uint32_t oa = 0u, oa2 = 0u, ob = 0u, ob2 = 0u;
      if (hasA) oa = tmem_ld1(tO + gA), oa2 = tmem_ld1(tO + a.gq + gA);
      if (hasB) ob = tmem_ld1(tO + gB), ob2 = tmem_ld1(tO + a.gq + gB);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane_id() == 0) mbar_arrive(&tempty[1]);
      const int64_t qh0 =
          ((int64_t)(uv / a.n_tiles) * (a.dk / a.D) + ((uv % a.n_tiles) >> 1)) * a.gq;
      float* po = a.part_o + qh0 * a.D + row;
      if (hasA) po[(int64_t)gA * a.D] = __uint_as_float(oa) + __uint_as_float(oa2);
      if (hasB) po[(int64_t)gB * a.D] = __uint_as_float(ob) + __uint_as_float(ob2);
      return true;
    };
    int k_done = 0;                                    // == u_count unless the loop broke off
    for (; k_done < u_count && ok; ++k_done) {
      const int u = unit_at(k_done);
      // the next unit (meaningful while k_done + 1 < u_count)
      const int u_next = kMulti ? unit_at(k_done + 1) : u + 1;
      const int m = u / a.n_tiles, n = unit_col<kAttend>(u % a.n_tiles, a.n_tiles);
      if (m != cur_m) {
        if (cur_m < 0) {
          int p0 = 0, ml = m;
          if constexpr (kMulti) {
            ml = tile_local(m, p0);
            pp = p0 | (p0 << 8);
          }
          const ProbView v = view(p0);
          const int64_t gi = (int64_t)ml * kTileM + row;
          nx_s = gi < v.n_sel ? v.seq[gi] : -1;
          nx_p = gi < v.n_sel ? v.pos[gi] : -1;
          cur = setup_a(ml, v);
#pragma unroll
          for (int t = 0; t < 4; ++t) issue_ref(n, true, t);   // the first unit's copies
        } else {
          cur = nxt;                                   // z~ already set up before the last unit
          if constexpr (kMulti) pp = ((pp >> 8) & 0xff) * 0x101;
          ++tt;
        }
        cur_m = m;
        setup_cs(cur.pos);
      }
      // Last unit of its tile: set up the next tile (staged by the loaders) so the MMAs
      // go on while this unit's epilogue runs; with one z~ buffer, once the tensor core
      // is done with this tile.  From here on every copy this thread issues is for the
      // next tile.
      if (k_done + 1 < u_count && u_next / a.n_tiles != m) {
        if (a.zbufs == 1) {
          // both warps of the pair leave together, so neither waits at a barrier alone
          if (!bar_red_and(vote_id, vote_n, warp_wait(afree, afree_phase, abort_flag, a.status))) break;
          afree_phase ^= 1u;
        }
        int pn = 0;
        if constexpr (kMulti) pn = problem_of(*mp, u_next / a.n_tiles);
        if (!setup_s((tt + 1) % a.zbufs, nxt, pn)) break;
        if constexpr (kMulti) pp = (pp & 0xff) | (pn << 8);   // this unit's copies are the next tile's
      }
      const bool more = k_done + 1 < u_count;
      const int n_next = unit_col<kAttend>(u_next % a.n_tiles, a.n_tiles);
      const int c0 = n * kNT + hl * a.D;               // first KV_hat column of the head
      const bool is_k = c0 < a.dk;
      // ---- mean of the references: wait for this unit's copies of reference t (both
      // warps' halves), read it; reference t-1 has then been read by both warps, so its
      // plane takes the next unit's copy
      float mx[16], my[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) mx[i] = 0.f, my[i] = 0.f;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        cp_async_wait<3>();
        bar_sync(bar_id, 64);
        if (cur.has_ref(t)) {
          const uint8_t* pt = pslots + (uint32_t)(t * 2) * kPlaneBytes + rd_off;
          fp8x16_add(*reinterpret_cast<const uint4*>(pt), mx);
          fp8x16_add(*reinterpret_cast<const uint4*>(pt + kPlaneBytes), my);
        }
        if (t > 0)
          issue_ref(n_next, more && t - 1 < a.topk, t - 1);
        else
          cp_async_commit();
      }
      // mean = sum / k_i.  For k_i = 1, 2, 4 the scaling is exact, so it folds into the
      // accumulator add below: one fma, RN(acc + sum / k_i), the same value as rounding
      // the exact mean's sum with acc.  For k_i = 3 the sum is divided here (correctly
      // rounded) and added with scale 1.  Rows without references keep zeros.
      float kinv = 1.0f;
      if (cur.kcnt() == 3) {
#pragma unroll
        for (int i = 0; i < 16; ++i) mx[i] = div3_rn(mx[i]), my[i] = div3_rn(my[i]);
      } else {
        kinv = cur.kcnt() == 2 ? 0.5f : (cur.kcnt() == 4 ? 0.25f : 1.0f);
      }
      // ---- accumulator row; the pair's vote also tells that both warps have read
      // reference 3, whose plane then takes the next unit's copy
      if (!bar_red_and(vote_id, vote_n, warp_wait(&tfull[acc], acc_phase, abort_flag, a.status))) break;
      issue_ref(n_next, more && 3 < a.topk, 3);
      tc_fence_after();
      {
        const uint32_t tacc = tmem + lane_base + (uint32_t)(acc * kNT);
        uint32_t xr[16], yr[16];
        tmem_ld16(tacc + xcol, xr);
        tmem_ld16(tacc + ycol, yr);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          mx[i] = __fmaf_rn(mx[i], kinv, __uint_as_float(xr[i]));
          my[i] = __fmaf_rn(my[i], kinv, __uint_as_float(yr[i]));
        }
      }
      // the accumulator is free as soon as it has been read (with kAttend, once the
      // pair's product in its first columns has been read)
      if constexpr (!kAttend) {
        tc_fence_before();
        __syncwarp();
        if (lane_id() == 0) mbar_arrive(&tempty[acc]);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      if (is_k) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 cs = cs_row[i * kTileM];
          const float x0 = mx[2 * i], y0 = my[2 * i], x1 = mx[2 * i + 1], y1 = my[2 * i + 1];
          mx[2 * i] = x0 * cs.x - y0 * cs.y;
          my[2 * i] = y0 * cs.x + x0 * cs.y;
          mx[2 * i + 1] = x1 * cs.z - y1 * cs.w;
          my[2 * i + 1] = y1 * cs.z + x1 * cs.w;
        }
      }
      if (!cur.valid()) {
#pragma unroll
        for (int i = 0; i < 16; ++i) mx[i] = 0.f, my[i] = 0.f;
      }
      if constexpr (kAttend) {
        // ---- attention over the tile (ResidualKV notes §2.7 output equation).  Each
        // tensor-core round trip overlaps the epilogue's next piece of restore work: the
        // scores of pair p run while its V_hat rows are built, its V_hat^T P while the
        // next pair's K_hat rows are built.
        const int et = (int)threadIdx.x - 32 * kEpiWarpR;
        const int h = (u % a.n_tiles) >> 1;             // key/value head of the pair
        const bool live = (int64_t)m * kTileM + row < a.n_sel;
        if (is_k) {
          // the head's query rows (loads in flight while the previous pair is finished)
          float2 qv[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int i = et + 512 * j, r16 = i >> 6, d = 2 * (i & 63);
            qv[j] = make_float2(0.f, 0.f);
            if (r16 < 2 * a.gq) {
              const int g = r16 < a.gq ? r16 : r16 - a.gq;
              qv[j] = *reinterpret_cast<const float2*>(a.q + ((int64_t)h * a.gq + g) * a.D + d);
            }
          }
          if (!waited) {
            // the queries and the partial sums may belong to the previous launch's merge
            pdl_wait_previous_grid();
            waited = true;
            // the weight tile's rows past 2 gq stay zero
            for (int i = et; i < (int)(kPBytes / 16); i += 512)
              reinterpret_cast<uint4*>(sP)[i] = make_uint4(0u, 0u, 0u, 0u);
          } else if (!finish_o(u - 1)) {
            break;                                      // the previous pair's V_hat^T P
          }
          // query tile: row g < gq the bf16 high part of q_g / sqrt(D), row gq + g the low
          // part (the exact remainder, rounded), other rows zero
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int i = et + 512 * j, r16 = i >> 6, d = 2 * (i & 63);
            const float q0 = qv[j].x * a.q_scale, q1 = qv[j].y * a.q_scale;
            const float h0 = __bfloat162float(__float2bfloat16_rn(q0));
            const float h1 = __bfloat162float(__float2bfloat16_rn(q1));
            const uint32_t wv = r16 < a.gq ? pack_bf16x2(h0, h1) : pack_bf16x2(q0 - h0, q1 - h1);
            *reinterpret_cast<uint32_t*>(sQ + sw128_off(r16, d, kRowTile16)) = wv;
          }
          // K_hat row into the token-major tile: x values (dimensions j0 ..) in the first
          // 64-column atom, y values (j0 + 64 ..) in the second
          {
            uint32_t wx[8], wy[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              wx[i] = pack_bf16x2(mx[2 * i], mx[2 * i + 1]);
              wy[i] = pack_bf16x2(my[2 * i], my[2 * i + 1]);
            }
            const int cx = j0 >> 3, sw = row & 7;
            uint8_t* k0 = sKV + (uint32_t)row * 128u;
            uint8_t* k1 = k0 + kTileM * 128;
            *reinterpret_cast<uint4*>(k0 + ((cx ^ sw) << 4)) = make_uint4(wx[0], wx[1], wx[2], wx[3]);
            *reinterpret_cast<uint4*>(k0 + (((cx + 1) ^ sw) << 4)) = make_uint4(wx[4], wx[5], wx[6], wx[7]);
            *reinterpret_cast<uint4*>(k1 + ((cx ^ sw) << 4)) = make_uint4(wy[0], wy[1], wy[2], wy[3]);
            *reinterpret_cast<uint4*>(k1 + (((cx + 1) ^ sw) << 4)) = make_uint4(wy[4], wy[5], wy[6], wy[7]);
          }
          tc_fence_before();                            // the K accumulator has been read
          fence_proxy_async_smem();                     // the tiles are visible to the MMA
          __syncwarp();
          if (lane_id() == 0) mbar_arrive(kready);
        } else {
          // the pair's scores: S[:, g] + S[:, gq + g] = K_hat (q_hi + q_lo) / sqrt(D)
          if (!bar_red_and(vote_id, vote_n, warp_wait(sdone, s_phase, abort_flag, a.status))) break;
          s_phase ^= 1u;
          tc_fence_after();
          const int gA = wg, gB = wg + 4;               // this group's query heads
          const bool hasA = gA < a.gq, hasB = gB < a.gq;  // uniform over the group
          const uint32_t tS = tmem + lane_base;
          uint32_t sa = 0u, sa2 = 0u, sb = 0u, sb2 = 0u;
          if (hasA) sa = tmem_ld1(tS + gA), sa2 = tmem_ld1(tS + a.gq + gA);
          if (hasB) sb = tmem_ld1(tS + gB), sb2 = tmem_ld1(tS + a.gq + gB);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane_id() == 0) mbar_arrive(&tempty[0]);
          if (hasA) {
            const int64_t qh0 = ((int64_t)m * (a.dk / a.D) + h) * a.gq;  // (tile, head h gq)
            const float s0 = live ? __uint_as_float(sa) + __uint_as_float(sa2) : -INFINITY;
            const float s1 = live && hasB ? __uint_as_float(sb) + __uint_as_float(sb2) : -INFINITY;
            float* red = sRed + wg * 16;                // [max A | max B | sum A | sum B][4 warps]
            float m0 = s0, m1 = s1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
              m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
            }
            if (lane_id() == 0) red[ew] = m0, red[4 + ew] = m1;
            bar_sync(kGroupBar0 + wg, 128);
            m0 = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
            m1 = fmaxf(fmaxf(red[4], red[5]), fmaxf(red[6], red[7]));
            // exp(s - m) in base 2: 2^(s' - m') with s' = s log2(e) (folded into q)
            const float p0 = live ? ex2_approx(s0 - m0) : 0.f;
            const float p1 = live && hasB ? ex2_approx(s1 - m1) : 0.f;
            float l0 = p0, l1 = p1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              l0 += __shfl_xor_sync(0xffffffffu, l0, o);
              l1 += __shfl_xor_sync(0xffffffffu, l1, o);
            }
            if (lane_id() == 0) red[8 + ew] = l0, red[12 + ew] = l1;
            // weights as bf16 high + low parts: rows g and gq + g of P, column = token
            const float pa = __bfloat162float(__float2bfloat16_rn(p0));
            const float pb = __bfloat162float(__float2bfloat16_rn(p1));
            *reinterpret_cast<__nv_bfloat16*>(sP + sw128_off(gA, row, kRowTile16)) = __float2bfloat16_rn(pa);
            *reinterpret_cast<__nv_bfloat16*>(sP + sw128_off(a.gq + gA, row, kRowTile16)) =
                __float2bfloat16_rn(p0 - pa);
            if (hasB) {
              *reinterpret_cast<__nv_bfloat16*>(sP + sw128_off(gB, row, kRowTile16)) = __float2bfloat16_rn(pb);
              *reinterpret_cast<__nv_bfloat16*>(sP + sw128_off(a.gq + gB, row, kRowTile16)) =
                  __float2bfloat16_rn(p1 - pb);
            }
            bar_sync(kGroupBar0 + wg, 128);
            if (ew == 0 && lane_id() == 0) {
              a.part_m[qh0 + gA] = m0;
              a.part_l[qh0 + gA] = (red[8] + red[9]) + (red[10] + red[11]);
              if (hasB) {
                a.part_m[qh0 + gB] = m1;
                a.part_l[qh0 + gB] = (red[12] + red[13]) + (red[14] + red[15]);
              }
            }
          }
          // V_hat row transposed into the dimension-major tile (the scores are done with
          // the K_hat rows): element (d, token) at row d, token chunk (token & 63) / 8
          // swizzled with d, atom token / 64
          {
            const int e = row & 63, c = e >> 3;
            uint8_t* vb = sKV + (uint32_t)(row >> 6) * (kTileM * 128) + (uint32_t)(e & 7) * 2;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int dx = xcol + i, dy = ycol + i;
              *reinterpret_cast<__nv_bfloat16*>(vb + dx * 128 + ((c ^ (dx & 7)) << 4)) =
                  __float2bfloat16_rn(mx[i]);
              *reinterpret_cast<__nv_bfloat16*>(vb + dy * 128 + ((c ^ (dy & 7)) << 4)) =
                  __float2bfloat16_rn(my[i]);
            }
          }
          tc_fence_before();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane_id() == 0) mbar_arrive(vready);
        }
        continue;
      }
      // ---- output: 32-byte stores straight from registers (the row's 16 x values, then
      // its 16 y values); K/V may be the previous launch's outputs, so each thread waits
      // for the previous grid before its first store
      if (!waited) {
        pdl_wait_previous_grid();
        waited = true;
      }
      int64_t grow = (int64_t)m * kTileM + row;
      int nsel_cur = a.n_sel;
      void* kb_cur = a.k_out;
      void* vb_cur = a.v_out;
      if constexpr (kMulti) {
        const int pc = pp & 0xff;
        grow -= (int64_t)mp->tile0[pc] * kTileM;
        nsel_cur = mp->n_sel[pc], kb_cur = mp->k_out[pc], vb_cur = mp->v_out[pc];
      }
      if (grow < nsel_cur) {
        const int64_t o0 = grow * a.dk + (is_k ? c0 : c0 - a.dk) + j0;
        void* base = is_k ? kb_cur : vb_cur;
        if (a.out_f32) {
          float* o = static_cast<float*>(base) + o0;
          st_global_v8(o, reinterpret_cast<const uint32_t*>(mx));
          st_global_v8(o + 8, reinterpret_cast<const uint32_t*>(mx + 8));
          st_global_v8(o + P, reinterpret_cast<const uint32_t*>(my));
          st_global_v8(o + P + 8, reinterpret_cast<const uint32_t*>(my + 8));
        } else {
          uint32_t wx[8], wy[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            wx[i] = pack_bf16x2(mx[2 * i], mx[2 * i + 1]);
            wy[i] = pack_bf16x2(my[2 * i], my[2 * i + 1]);
          }
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(base) + o0;
          st_global_v8(o, wx);
          st_global_v8(o + P, wy);
        }
      }
    }
    if constexpr (kAttend) {
      if (ok && k_done == u_count && u_count > 0) finish_o(unit_at(u_count - 1));
    }
    cp_async_wait<0>();                                // no copy may outlive the CTA
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool kAttend>
__global__ void __launch_bounds__(kReconThreads, 1)
    reconstruct_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ ReconArgs a) {
  restore_body<kAttend, false>(&tmW, a, nullptr);
}

// Several contexts' selections in one launch: a's dimensions, tables and wait status
// are shared, mp holds each problem's inputs and outputs, mm its W_d^T map.
__global__ void __launch_bounds__(kReconThreads, 1)
    reconstruct_multi_kernel(const __grid_constant__ ReconMaps mm, const __grid_constant__ ReconArgs a,
                             const __grid_constant__ ReconProblems mp) {
  restore_body<false, true>(mm.tmW, a, &mp);
}

}  // namespace

// The restore's arguments and shared-memory size for a selection of n_sel >= 1 tokens;
// `attend_bytes` of shared memory are set aside before the reference slots.
static cudaError_t recon_setup(rkv_ctx* c, const int32_t* seq, const int32_t* pos, int n_sel,
                               size_t attend_bytes, ReconArgs* ap, size_t* smem_out) {
  const Dims& d = c->d;
  // staged tile: records, extremes and (rows of at most 128 bytes) codes
  const bool stage_codes = d.code_bytes <= 128;
  const size_t stage = (size_t)kTileM * kRecInts * 4 + (size_t)kTileM * d.G * 4 +
                       (stage_codes ? (((size_t)kTileM * d.code_bytes + 127) & ~(size_t)127) : 0);
  const size_t fixed = 1024 + attend_bytes + kCSBytes + kGBytes + stage + kBarBytes;
  int b_stages = (int)((232448 - fixed) / kBBytes);
  if (b_stages > kMaxStages) b_stages = kMaxStages;
  if (b_stages < 2) return cudaErrorInvalidConfiguration;
  *smem_out = fixed + (size_t)b_stages * kBBytes;
  ReconArgs& a = *ap;
  a = ReconArgs{};
  a.seq = seq;
  a.pos = pos;
  a.n_sel = n_sel;
  a.n_tiles = d.dkv / kNT;
  const int m_tiles = (n_sel + kTileM - 1) / kTileM;
  a.units = m_tiles * a.n_tiles;
  a.b_stages = b_stages;
  a.codes = static_cast<const uint8_t*>(c->st.codes);
  a.meta = static_cast<const uint32_t*>(c->st.meta);
  a.ref_idx = c->st.ref_idx;
  a.pool8 = static_cast<const uint8_t*>(c->st.pool_fp8);
  a.rope_lo = c->rope_lo;
  a.rope_hi = c->rope_hi;
  a.out_f32 = d.out_f32;
  a.B = d.B;
  a.T_cap = d.T_cap;
  a.R_cap = d.R_cap;
  a.topk = d.topk;
  a.dkv = d.dkv;
  a.dk = d.dk;
  a.dc = d.dc;
  a.D = d.D;
  a.G = d.G;
  a.bits = d.bits;
  a.code_bytes = d.code_bytes;
  a.zbufs = 2 * kNT + d.dc <= (int)kTmemCols ? 2 : 1;     // d_c / 2 TMEM columns per buffer
  a.stage_codes = stage_codes ? 1 : 0;
  {
    const int chunks = d.code_bytes / 16;
    const int low = chunks & -chunks;                         // largest power of two dividing it
    a.chunk_mask = (low < 8 ? low : 8) - 1;
  }
  a.status = c->status;
  return cudaSuccess;
}

template <bool kAttend>
static cudaError_t recon_launch(rkv_ctx* c, const ReconArgs& a, size_t smem, int grid,
                                int* smem_set, const char* name, cudaStream_t s) {
  // the kernel's shared-memory limit is raised once per context (on its device)
  cudaError_t e = cudaSuccess;
  if (*smem_set < (int)smem) {
    e = cudaFuncSetAttribute(reconstruct_kernel<kAttend>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    *smem_set = (int)smem;
  }
  cudaEvent_t ev;
  timing_begin(c, name, s, &ev);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(kReconThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  e = cudaLaunchKernelEx(&lc, reconstruct_kernel<kAttend>, c->tm_wd, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  timing_end(c, name, s, ev);
  return e;
}

cudaError_t launch_reconstruct(rkv_ctx* c, const int32_t* seq, const int32_t* pos, int n_sel,
                               void* k_out, void* v_out, cudaStream_t s) {
  if (n_sel <= 0) return cudaSuccess;
  ReconArgs a;
  size_t smem = 0;
  cudaError_t e = recon_setup(c, seq, pos, n_sel, 0, &a, &smem);
  if (e != cudaSuccess) return e;
  a.k_out = k_out;
  a.v_out = v_out;
  const int grid = a.units < c->num_sms ? a.units : c->num_sms;
  return recon_launch<false>(c, a, smem, grid, &c->recon_smem, "rkv_reconstruct_kernel", s);
}

cudaError_t launch_reconstruct_multi(rkv_ctx* const* cs, int n, const int32_t* const* seqs,
                                     const int32_t* const* poss, const int32_t* n_sels,
                                     void* const* k_outs, void* const* v_outs, cudaStream_t s) {
  ReconProblems mp{};                 // launch parameters (copied when the kernel is launched)
  ReconMaps mm;
  rkv_ctx* c0 = cs[0];
  mp.n = n;
  int tiles = 0, first = -1;
  for (int i = 0; i < n; ++i) {
    mp.tile0[i] = tiles;
    tiles += (n_sels[i] + kTileM - 1) / kTileM;
    mp.seq[i] = seqs[i];
    mp.pos[i] = poss[i];
    mp.n_sel[i] = n_sels[i];
    mp.codes[i] = static_cast<const uint8_t*>(cs[i]->st.codes);
    mp.meta[i] = static_cast<const uint32_t*>(cs[i]->st.meta);
    mp.ref_idx[i] = cs[i]->st.ref_idx;
    mp.pool8[i] = static_cast<const uint8_t*>(cs[i]->st.pool_fp8);
    mp.k_out[i] = k_outs[i];
    mp.v_out[i] = v_outs[i];
    mp.status[i] = cs[i]->status;
    mm.tmW[i] = cs[i]->tm_wd;
    if (first < 0 && n_sels[i] > 0) first = i;
  }
  mp.tile0[n] = tiles;
  if (tiles == 0) return cudaSuccess;
  ReconArgs a;
  size_t smem = 0;
  cudaError_t e = recon_setup(c0, seqs[first], poss[first], n_sels[first], 0, &a, &smem);
  if (e != cudaSuccess) return e;
  a.units = tiles * a.n_tiles;
  a.k_out = k_outs[first];
  a.v_out = v_outs[first];
  if (c0->multi_smem < (int)smem) {
    e = cudaFuncSetAttribute(reconstruct_multi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    c0->multi_smem = (int)smem;
  }
  const int grid = a.units < c0->num_sms ? a.units : c0->num_sms;
  cudaEvent_t ev;
  timing_begin(c0, "rkv_reconstruct_multi_kernel", s, &ev);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(kReconThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  e = cudaLaunchKernelEx(&lc, reconstruct_multi_kernel, mm, a, mp);
  if (e == cudaSuccess) e = cudaGetLastError();
  timing_end(c0, "rkv_reconstruct_multi_kernel", s, ev);
  return e;
}

cudaError_t launch_restore_attend(rkv_ctx* c, const int32_t* seq, const int32_t* pos, int n_sel,
                                  const float* q, int n_q_heads, float* out, cudaStream_t s) {
  const Dims& d = c->d;
  if (n_sel <= 0) return cudaSuccess;
  const size_t attend = kAttendBytes;
  ReconArgs a;
  size_t smem = 0;
  cudaError_t e = recon_setup(c, seq, pos, n_sel, attend, &a, &smem);
  if (e != cudaSuccess) return e;
  const int gq = n_q_heads / d.N;
  const int m_tiles = (n_sel + kTileM - 1) / kTileM;
  a.q = q;
  a.gq = gq;
  a.q_scale = (float)(1.4426950408889634 / sqrt((double)d.D));   // log2(e) / sqrt(D)
  a.part_m = c->fa_ws;
  a.part_l = a.part_m + (size_t)m_tiles * n_q_heads;
  a.part_o = a.part_l + (size_t)m_tiles * n_q_heads;
  const int pairs = a.units / 2;
  const int grid = pairs < c->num_sms ? pairs : c->num_sms;
  e = recon_launch<true>(c, a, smem, grid, &c->fused_smem, "rkv_restore_attend_kernel", s);
  if (e != cudaSuccess) return e;
  return launch_attend_merge(c, a.part_m, a.part_l, a.part_o, m_tiles, n_q_heads, out, s);
}

}  // namespace rkv
